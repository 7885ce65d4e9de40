// Shared device helpers for the sm_103a kernels: geometry, bounded mbarrier
// waits, TMA (cp.async.bulk.tensor), and tcgen05 (TMEM alloc / MMA / ld / st).
// All inline PTX follows the public PTX ISA.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sda {

// ----------------------------------------------------------------------------
// Status latch (one word per device, see status.cu).  Bits record what went
// wrong on the device; the host reads and clears it.
enum : unsigned {
  kStatusWaitTimeout = 1u,  // a bounded wait ran out
  kStatusBadIndex = 2u,     // a block_idx entry outside [0, n_b), or repeated in its row
  kStatusRange = 4u,        // an input value outside fp16's finite range met an fp16 conversion
};

// Bounded waits give up after this many nanoseconds of %globaltimer.
#ifndef SDA_WAIT_LIMIT_NS
#define SDA_WAIT_LIMIT_NS 2000000000ull
#endif

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------
// Tile geometry: block I of an (nT, nH, nW) tiling, row r inside a bt x bh x bw
// tile ordered (tt, hh, ww).
struct Geom {
  int T, H, W, bt, bh, bw, nT, nH, nW, nb, bs;
};

__host__ __device__ __forceinline__ void block_origin(const Geom& g, int I, int& t0, int& h0, int& w0) {
  int iw = I % g.nW;
  int ih = (I / g.nW) % g.nH;
  int it = I / (g.nW * g.nH);
  t0 = it * g.bt;
  h0 = ih * g.bh;
  w0 = iw * g.bw;
}

// Raster token index of row r of block I, or -1 when the row is outside the grid.
__host__ __device__ __forceinline__ int block_row_token(const Geom& g, int I, int r) {
  int t0, h0, w0;
  block_origin(g, I, t0, h0, w0);
  int ww = r % g.bw;
  int hh = (r / g.bw) % g.bh;
  int tt = r / (g.bw * g.bh);
  int t = t0 + tt, h = h0 + hh, w = w0 + ww;
  if (t >= g.T || h >= g.H || w >= g.W) return -1;
  return (t * g.H + h) * g.W + w;
}

__host__ __device__ __forceinline__ bool block_is_full(const Geom& g, int I) {
  int t0, h0, w0;
  block_origin(g, I, t0, h0, w0);
  return t0 + g.bt <= g.T && h0 + g.bh <= g.H && w0 + g.bw <= g.W;
}

// Bit c set when row (col0 + c) of block I lies inside the grid, c = 0..31.
// Out of line on purpose: it runs only for clipped edge tiles and keeps the
// unrolled inner loops that call it small.
__device__ __noinline__ inline uint32_t block_rows_mask32(const Geom& g, int I, int col0) {
  uint32_t m = 0;
  for (int c = 0; c < 32; ++c) m |= (block_row_token(g, I, col0 + c) >= 0 ? 1u : 0u) << c;
  return m;
}

// ----------------------------------------------------------------------------
// Shared-memory addresses and mbarriers.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// One bounded test of the phase; the thread may be suspended by the hardware for
// up to kSuspendHintNs while the phase is incomplete (it resumes as soon as the
// phase completes), so waiting warps do not spin on the issue slots.
constexpr uint32_t kSuspendHintNs = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase.  A phase that has already completed costs about
// 50 cycles here against about 85 through mbar_try_wait, whose suspend hint makes
// even a satisfied wait slower; pipelines mostly find their barriers complete.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// SDA_WAIT_LIMIT_NS, latches kStatusWaitTimeout into *status, raises the CTA's
// abort flag and returns false; callers then stop issuing work.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* status,
                                          volatile int* abort_flag, uint64_t limit_ns = SDA_WAIT_LIMIT_NS) {
  if (mbar_test(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7u) == 7u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(status, kStatusWaitTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Release/acquire counters in shared memory: a cheaper hand-off than an mbarrier
// when the waiter usually finds the count already reached (one shared load).
__device__ __forceinline__ void count_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned count_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
// Whole warp: wait until *p >= target (bounded like mbar_wait); the same result on every lane.
__device__ __forceinline__ bool warp_wait_count(const unsigned* p, unsigned target, unsigned* status,
                                                volatile int* abort_flag) {
  if (__all_sync(0xffffffffu, count_acquire(p) >= target)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (__all_sync(0xffffffffu, count_acquire(p) >= target)) return true;
    if ((it & 63u) == 63u) {
      const bool stop = *abort_flag != 0 || globaltimer_ns() - t0 > SDA_WAIT_LIMIT_NS;
      if (__any_sync(0xffffffffu, stop)) {
        if ((threadIdx.x & 31) == 0 && !*abort_flag) {
          atomicOr(status, kStatusWaitTimeout);
          *abort_flag = 1;
        }
        return false;
      }
    }
  }
}

// ----------------------------------------------------------------------------
// TMA (bulk tensor copies).  Destination/source shared addresses are CTA-local.
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, const void* src, int c0, int c1, int c2,
                                             int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

// Plain (untiled) bulk copy global -> shared; both addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make generic-proxy shared-memory writes visible to the async proxy (TMA, MMA).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Named barrier among `nthreads` threads (multiple of 32), id 1..15.
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns the AND of `v` over the participating threads,
// so a group can take a decision (continue or stop) uniformly.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %3, 0;\n\t"
      "bar.red.and.pred p, %1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 layout).  swz: 0 none, 2 = 128B,
// 4 = 64B, 6 = 32B.  lbo/sbo in bytes.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // fixed 0b001 in bits 46..48
  d |= (uint64_t)(swz & 7u) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
// a_mn / b_mn: operand stored MN-major (1) instead of K-major (0).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                       // D format f32
         | (1u << 7)                     // A format bf16
         | (1u << 10)                    // B format bf16
         | ((uint32_t)a_mn << 15)        //
         | ((uint32_t)b_mn << 16)        //
         | ((uint32_t)(N >> 3) << 17)    //
         | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor for kind::f16 with fp16 A/B and fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                       // D format f32 (A, B format fields 0 = f16)
         | ((uint32_t)a_mn << 15)        //
         | ((uint32_t)b_mn << 16)        //
         | ((uint32_t)(N >> 3) << 17)    //
         | ((uint32_t)(M >> 4) << 24);
}

// tcgen05.mma (kind::f16, one CTA): D[tmem] (+)= A * B with A from shared memory
// (mma_ss_by) or from TMEM (mma_ts_by), B from shared memory; tcgen05.commit arrives on
// an mbarrier once every tcgen05 operation the issuing thread started has completed.
//
// Warp-converged issue.  Every lane of the MMA warp runs the issue loop with the
// same operands; only the lane whose `leader` is nonzero issues.  The leader is
// elected once (elect_leader) and reused, so the lane that issues the MMAs is the
// lane that commits them.  Keeping the loop converged lets the operands live in
// warp-uniform registers: the issue rate then matches the tensor pipe instead of
// being limited by per-instruction operand moves.
__device__ __forceinline__ uint32_t elect_leader() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred;
}

__device__ __forceinline__ void mma_ss_by(uint32_t leader, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 e, %5, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accum), "r"(leader)
      : "memory");
}

__device__ __forceinline__ void mma_ts_by(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 e, %5, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accum), "r"(leader)
      : "memory");
}

__device__ __forceinline__ void mma_commit_by(uint32_t leader, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\tsetp.ne.b32 e, %1, 0;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar)),
      "r"(leader)
      : "memory");
}

// Bounded wait by a whole warp; the result is the same on every lane.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned* status, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// As tmem_ld32, and also the maximum of the 32 loaded fp32 values of this thread
// (the reducing form of the TMEM load); call tmem_wait_ld before using either.
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31]), "=f"(mx)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------------------
// Small math helpers.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// d = fma(a, b, c) on two fp32 lanes at once (the packed FP32 FMA of sm_100 and later).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d, ua, ub, uc;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ua) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ub) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(uc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(ua), "l"(ub), "l"(uc));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}

// a * b and a + b on two fp32 lanes at once (round to nearest, as the scalar forms).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t d, ua, ub;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ua) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ub) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(ua), "l"(ub));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t d, ua, ub;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ua) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ub) : "f"(b.x), "f"(b.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(ua), "l"(ub));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}

// The two bf16 of a 32-bit word as fp32 (low half first).
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// Max of the loaded values whose column bit is set in v0 (u0) or v1 (u1).
__device__ __forceinline__ float masked_max64(uint32_t v0, uint32_t v1, const uint32_t (&u0)[32],
                                              const uint32_t (&u1)[32]) {
  float m = -INFINITY;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    if ((v0 >> c) & 1u) m = fmaxf(m, __uint_as_float(u0[c]));
    if ((v1 >> c) & 1u) m = fmaxf(m, __uint_as_float(u1[c]));
  }
  return m;
}

// Byte offset of element (row, col) of a 128 x ncols 16-bit tile in the tensor
// cores' unswizzled K-major operand layout: 8x8 core matrices (8 rows x 16
// bytes, rows contiguous), K-adjacent core matrices 128 bytes apart (LBO),
// 8-row groups ncols*16 bytes apart (SBO).
__host__ __device__ __forceinline__ uint32_t coremat_offset(int row, int col, int ncols) {
  return (uint32_t)((row >> 3) * (ncols >> 3) * 128 + (col >> 3) * 128 + (row & 7) * 16 + (col & 7) * 2);
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` inside a 128B-swizzled
// tile whose rows are 128 bytes (the TMA SWIZZLE_128B pattern).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}

}  // namespace sda
