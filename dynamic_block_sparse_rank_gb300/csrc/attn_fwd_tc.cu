// Block-sparse flash-attention forward on the 5th-generation tensor cores.
//
// "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT
// Training", section 4 (stage 2): attention is computed only on the key blocks
// the predictor kept.  For row i of query block I and the kept key blocks J
// with kb_begin <= J < kb_end:  S = scale Q K^T,  LSE_i = log sum_j exp(S_ij),
// O_i = sum_j exp(S_ij - LSE_i) v_j.  The key range and the query-block mask
// give the per-partition states of "DiTango: Cost-Effective Parallel Diffusion
// Generation with Selective Attention State Reuse".
//
// Two operand types.  The inference forward reads the caller's bf16 Q, K, V
// and splits P into two bf16 terms for the P V product.  The training forward reads fp16
// copies of Q, K, V (exact for bf16 values inside fp16's range) and rounds P
// to fp16, eight times finer, and also writes O in fp32: the backward then
// takes D_i = dO_i . O_i from that O, which is close enough to the exact
// sum_j P_ij dP_ij that no correction pass is needed.
//
// One CTA per (query block, head); 12 warps:
//   warps 0, 2  TMA producers: Q once and the K tiles of each kept block
//               (warp 0), the V tiles (warp 2), through separate rings (the
//               tile box *is* the space-time tile, so no token reordering pass
//               exists).
//   warp 1      TMEM owner and MMA issuer (converged warp, one elected lane):
//               S_j = Q K_j^T (Q from TMEM) into one of two TMEM S buffers, up
//               to two blocks ahead of the softmax; once P_j is ready, O += P_j
//               V_j with P_j read from TMEM (in bf16 twice, P_hi then P_lo),
//               then S_{j+2} into the buffer P_j leaves.
//   warps 4-11  copy Q from its tile into TMEM once, then softmax: two warps
//               per query row quarter (thread = row = TMEM lane), each owning
//               64 of the 128 key columns; the pair swaps
//               its half-row maxima at a named barrier.  Online softmax in
//               base 2 with a lazy rescale: O and the sums are rescaled only
//               when the row max grows by more than 2^15 (fp16 P) or 2^30
//               (bf16 P), which is exact because they always share one
//               reference max.  P overwrites S: in fp16, or in bf16 as
//               P_hi + P_lo (the remainder), both fed to the P V product, so
//               that O is accurate to fp32 accumulation and not to bf16's 8
//               bits; one fp32 sum of P divides O and gives LSE.
//   warp 3      arrives on P_j's barrier once V_j has landed, so that barrier
//               covers every input of P_j V_j and the MMA warp waits once per
//               block for it.
// TMEM columns: [0,128) S0/P0, [128,256) S1/P1, [256,256+D) O, [384,384+D/2) Q (packed
// 16-bit pairs: the S products take Q from TMEM and only K from shared memory, which
// keeps their operand traffic, with the K and V tile loads, under shared memory's rate).
#include "internal.h"

namespace sda {

namespace {

struct FwdArgs {
  Geom g;
  int Hh, k, b, kb_begin, kb_end;
  int all_full;  // every tile lies inside the grid (no clipped edge tiles)
  long long N;
  float scale_log2;  // softmax scale * log2(e)
  const int32_t* idx;
  const uint8_t* qb_active;
  float* LSE;
  unsigned* status;
};

constexpr int kThreads = 384;  // warps 0, 2 TMA, warp 1 MMA, warp 3 V arrivals, warps 4-11 softmax
constexpr int kSBufs = 2;      // S / P buffers in TMEM: S runs up to two blocks ahead of P V
constexpr int kTQ = 384;       // TMEM column of Q (the S products' A operand, d / 2 packed columns)
// P_j barrier: the 256 softmax threads and warp 3 (V_j landed).
constexpr int kPfullCount = 256 + 1;
// Lazy rescale: O_hf and its sum are rescaled only when the half-row max grows by more
// than this many powers of two (P then stays below 2^threshold).  fp16 holds P up to
// 2^15 (65504 max); bf16 up to about 2^127, and the fp32 accumulators far more, so bf16
// takes 2^30.  Fewer rescales means fewer waits for the previous P V product.
template <bool kF16>
__device__ __forceinline__ float rescale_threshold() {
  return kF16 ? 15.0f : 30.0f;
}
constexpr int kSeenWords = 8192 / 32;       // one bit per key block (n_b <= 8192)

template <int D>
struct FwdCfg {
  static constexpr int CH = D / 64;                  // 128-byte chunks of the head dim
  static constexpr int TILE = 128 * D * 2;           // bytes of one 128-row 16-bit tile
  static constexpr int KST = D == 128 ? 3 : 5;       // K ring depth (K is consumed first)
  static constexpr int VST = D == 128 ? 2 : 4;       // V ring depth
  static constexpr int SMEM_TILES = TILE * (1 + KST + VST);
};

__device__ __forceinline__ bool wait_plain(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > SDA_WAIT_LIMIT_NS) return false;
  return true;
}

// P = 2^(s scale_log2 - m) for one thread's 64 keys (two 32-column chunks of S in u0,
// u1), written over S and added to l.  kF16: P in fp16, in the first 16 TMEM columns of
// each chunk.  Otherwise P = P_hi + P_lo, two bf16 values (P_lo the rounding remainder
// of P_hi), in the first and the second 16 columns of each chunk: the P V product takes
// both, so P enters it with about 16 bits instead of bf16's 8.  kMask: keys whose bit in
// vm0 / vm1 is clear (outside the grid) get P = 0.
template <bool kMask, bool kF16>
__device__ __forceinline__ void softmax_p(const uint32_t (&u0)[32], const uint32_t (&u1)[32], uint32_t vm0,
                                          uint32_t vm1, float m, float scale_log2, uint32_t tS, float& l) {
  // pairs of columns through the packed fp32x2 FMA: the same roundings as two scalar FMAs
  float2 sab = make_float2(0.f, 0.f);
  const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-m, -m);
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const uint32_t(&u)[32] = cc ? u1 : u0;
    const uint32_t vm = cc ? vm1 : vm0;
    uint32_t ph[16], pl[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float2 s2 = ffma2(make_float2(__uint_as_float(u[2 * e]), __uint_as_float(u[2 * e + 1])), sc2, nm2);
      float s0 = s2.x, s1 = s2.y;
      if (kMask) {
        if (!((vm >> (2 * e)) & 1u)) s0 = -INFINITY;
        if (!((vm >> (2 * e + 1)) & 1u)) s1 = -INFINITY;
      }
      const float p0 = ex2(s0), p1 = ex2(s1);
      sab = fadd2(sab, make_float2(p0, p1));
      if (kF16) {
        ph[e] = pack_f16(p0, p1);
      } else {
        ph[e] = pack_bf16(p0, p1);
        pl[e] = pack_bf16(p0 - __uint_as_float(ph[e] << 16), p1 - __uint_as_float(ph[e] & 0xFFFF0000u));
      }
    }
    tmem_st16(tS + cc * 32, ph);
    if (!kF16) tmem_st16(tS + cc * 32 + 16, pl);
  }
  l += sab.x + sab.y;
}

// kF16: operands and P in fp16 (training), otherwise bf16.  kO16: O is written in bf16
// through tmO; kO32: O is written in fp32 through tmO32 (the training forward writes
// both; an fp32 partition state only the second).
template <int D, bool kF16, bool kO16, bool kO32>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const __grid_constant__ CUtensorMap tmO32, FwdArgs a) {
  using C = FwdCfg<D>;
  constexpr int KST = C::KST, VST = C::VST;
  const int I = blockIdx.x, h = blockIdx.y;
  if (a.qb_active && !a.qb_active[I]) return;  // cached state stays untouched

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::TILE;
  uint8_t* sV = sK + KST * C::TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::SMEM_TILES);
  uint64_t* qfull = bars;
  uint64_t* kfull = bars + 1;      // KST
  uint64_t* kempty = kfull + KST;  // KST
  uint64_t* vfull = kempty + KST;  // VST
  uint64_t* vempty = vfull + VST;  // VST
  uint64_t* sfull = vempty + VST;  // kSBufs
  uint64_t* pfull = sfull + kSBufs;  // kSBufs
  uint64_t* odone = pfull + kSBufs;  // 2: P V of blocks of each parity done
  uint64_t* qtmem = odone + 2;       // 1: Q is in TMEM (the 256 softmax threads)
  uint64_t* drain = qtmem + 1;       // 1
  uint64_t* pairbar = drain + 1;     // 4: the two softmax warps of a lane quarter meet here at the end
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pairbar + 4);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* n_sel_s = abort_flag + 1;
  int* warp_cnt = n_sel_s + 1;  // 16
  float* half_max = reinterpret_cast<float*>(warp_cnt + 16);  // [2 block parities][2 halves][128 rows]
  float* half_l = half_max + 512;                              // [2 halves][128 rows]
  unsigned* seen = reinterpret_cast<unsigned*>(half_l + 256);  // kSeenWords: blocks met in this row
  int* sel = reinterpret_cast<int*>(seen + kSeenWords);        // k

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(kfull + s, 1);
      mbar_init(kempty + s, 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(vfull + s, 1);
      mbar_init(vempty + s, 1);
    }
    for (int s = 0; s < kSBufs; ++s) {
      mbar_init(sfull + s, 1);
      mbar_init(pfull + s, kPfullCount);
    }
    mbar_init(odone, 1);
    mbar_init(odone + 1, 1);
    mbar_init(qtmem, 256);
    mbar_init(drain, 1);
    for (int q = 0; q < 4; ++q) mbar_init(pairbar + q, 2);
    *abort_flag = 0;
    *n_sel_s = 0;
    fence_mbar_init();
  }
  for (int e = tid; e < kSeenWords; e += kThreads) seen[e] = 0u;
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  // Kept blocks of this query block that fall in the key range, in list order.  An
  // entry outside [0, n_b), or one met before in the row, is skipped and latched.
  const int32_t* row = a.idx + (((long long)a.b * a.Hh + h) * a.g.nb + I) * a.k;
  __syncthreads();
  for (int base = 0; base < a.k; base += kThreads) {
    const int j = base + tid;
    int J = j < a.k ? row[j] : -1;
    const bool valid = j < a.k && J >= 0 && J < a.g.nb;
    bool repeated = false;
    if (valid) repeated = (atomicOr(seen + (J >> 5), 1u << (J & 31)) >> (J & 31)) & 1u;
    if (j < a.k && (!valid || repeated)) atomicOr(a.status, kStatusBadIndex);
    bool keep = valid && !repeated && J >= a.kb_begin && J < a.kb_end;
    unsigned m = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) warp_cnt[warp] = __popc(m);
    __syncthreads();
    int pos = *n_sel_s + __popc(m & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) pos += warp_cnt[w];
    if (keep) sel[pos] = J;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < kThreads / 32; ++w) tot += warp_cnt[w];
      *n_sel_s += tot;
    }
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_sel = *n_sel_s;
  int t0, h0, w0;
  block_origin(a.g, I, t0, h0, w0);

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------- producers
    // warp 0: Q once, then the K tiles of the kept blocks (a KST-deep ring, a slot freed
    // once its S is computed); warp 2: the V tiles (a VST-deep ring, freed after P V).
    const bool is_k = warp == 0;
    if (lane == 0 && n_sel > 0) {
      const int RS = is_k ? KST : VST;
      uint8_t* ring = is_k ? sK : sV;
      uint64_t* full = is_k ? kfull : vfull;
      uint64_t* empty = is_k ? kempty : vempty;
      const CUtensorMap* map = is_k ? &tmK : &tmV;
      prefetch_tmap(map);
      if (is_k) {
        prefetch_tmap(&tmQ);
        mbar_expect_tx(qfull, C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) tma_load_5d(sQ + c * 16384, &tmQ, qfull, c * 64, h, w0, h0, t0);
      }
      int issued = 0;
      for (; issued < n_sel; ++issued) {
        const int i = issued, s = i % RS;
        if (i >= RS && !mbar_wait(empty + s, ((i / RS) - 1) & 1, a.status, abort_flag)) break;
        int jt0, jh0, jw0;
        block_origin(a.g, sel[i], jt0, jh0, jw0);
        mbar_expect_tx(full + s, C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_load_5d(ring + s * C::TILE + c * 16384, map, full + s, c * 64, h, jw0, jh0, jt0);
      }
      if (*abort_flag) {  // let copies in flight land before the CTA exits
        if (is_k) wait_plain(qfull, 0);
        for (int j = issued - RS < 0 ? 0 : issued - RS; j < issued; ++j) wait_plain(full + j % RS, (j / RS) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------- V arrivals
    // Arrive on pfull_j once V_j has landed, so the MMA warp's pfull_j wait covers it.
    if (lane == 0) {
      for (int j = 0; j < n_sel; ++j) {
        if (!mbar_wait(vfull + j % VST, (j / VST) & 1, a.status, abort_flag)) break;
        // phase j - kSBufs of the same barrier completes before this arrival for phase j
        if (j >= kSBufs && !mbar_wait(pfull + j % kSBufs, ((j / kSBufs) - 1) & 1, a.status, abort_flag)) break;
        mbar_arrive(pfull + j % kSBufs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    // Whole warp, one elected lane issues; descriptors advance by adding to the
    // start-address field (16-byte units).  S runs kSBufs blocks ahead: S_0 and S_1 as
    // their K tiles land (and Q is in TMEM), then per block j: wait for pfull_j (softmax of
    // block j done, V_j landed), P_j V_j, then S_{j+2} into the buffer P_j leaves (the
    // tensor pipe runs its products in order, so P_j is read before S_{j+2} overwrites it)
    // once K_{j+2} has landed.
    if (n_sel > 0) {
      const uint32_t leader = elect_leader();
      constexpr uint32_t idS = kF16 ? idesc_f16(128, 128, 0, 0) : idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idO = kF16 ? idesc_f16(128, D, 0, 1) : idesc_bf16(128, D, 0, 1);
      const uint64_t dK = smem_desc(smem_u32(sK), 16, 1024, 2);
      const uint64_t dV = smem_desc(smem_u32(sV), 16384, 1024, 2);
      const uint32_t tO = tmem + kSBufs * 128;
      auto issue_S = [&](int t) {
        const int s = t % KST;
        const uint32_t tS = tmem + (t % kSBufs) * 128;
        const uint64_t dKs = dK + (uint64_t)((s * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          constexpr int kChunk = 16384 >> 4;
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 2;  // 64-column chunk, 16-column step
          mma_ts_by(leader, tS, tmem + kTQ + kk * 8, dKs + off, idS, kk > 0);
        }
        mma_commit_by(leader, sfull + t % kSBufs);
        mma_commit_by(leader, kempty + s);  // K_t is no longer needed once S_t is done
      };
      bool ok = warp_wait(qtmem, 0, a.status, abort_flag);
      for (int t = 0; ok && t < kSBufs && t < n_sel; ++t) {
        if (!(ok = warp_wait(kfull + t % KST, (t / KST) & 1, a.status, abort_flag))) break;
        tc_fence_after();
        issue_S(t);
      }
      for (int j = 0; ok && j < n_sel; ++j) {
        if (!(ok = warp_wait(pfull + j % kSBufs, (j / kSBufs) & 1, a.status, abort_flag))) break;
        tc_fence_after();
        const int s = j % VST;
        const uint32_t tP = tmem + (j % kSBufs) * 128;
        const uint64_t dVs = dV + (uint64_t)((s * C::TILE) >> 4);
        // keys 16 kk .. 16 kk + 15; in bf16 each step takes P_hi, then P_lo (16 columns further)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t tA = tP + (kk >> 1) * 32 + (kk & 1) * 8;
          const uint64_t bV = dVs + (uint64_t)(kk * (2048 >> 4));
          mma_ts_by(leader, tO, tA, bV, idO, (j > 0 || kk > 0));
          if (!kF16) mma_ts_by(leader, tO, tA + 16, bV, idO, 1u);
        }
        mma_commit_by(leader, vempty + s);
        mma_commit_by(leader, odone + (j & 1));
        const int t = j + kSBufs;
        if (t < n_sel) {
          if (!(ok = warp_wait(kfull + t % KST, (t / KST) & 1, a.status, abort_flag))) break;
          tc_fence_after();
          issue_S(t);
        }
      }
      mma_commit_by(leader, drain);
      wait_plain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------- softmax + epilogue
    // Two warps per TMEM lane quarter: warp half hf owns S columns [64 hf, 64 hf + 64) and
    // O columns [hf D/2, (hf + 1) D/2) of the quarter's 32 rows.  The pair swaps its
    // half-row maxima through shared memory (double-buffered by block parity) at a named
    // barrier, so both warps hold the same row maxima and take the same rescale
    // decisions; a bounded wait's failure is ANDed into the same barrier, so both warps
    // stop at the same point.
    const int quarter = warp & 3, hf = (warp - 4) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t tO = tmem + kSBufs * 128 + lane_base;
    auto pair_sync = [&](uint32_t phase) -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(pairbar + quarter);
      return mbar_wait(pairbar + quarter, phase & 1, a.status, abort_flag);
    };
    float m = -INFINITY;  // row max, log2 units (scaled), the same in both warps of the pair
    float l = 0.f;        // this warp's sum of P (fp32) over its keys
    bool ok = true;
    // Q into TMEM, the A operand of every S product (so S reads only K from shared
    // memory): this thread's row, elements [hf d/2, (hf + 1) d/2), 16-byte vectors of the
    // swizzled tile, 8 values = 4 packed columns each.
    if (n_sel > 0 && warp_wait(qfull, 0, a.status, abort_flag)) {
      constexpr int kV = D / 16;  // vectors of this half row
      uint32_t u[kV * 4];
#pragma unroll
      for (int v = 0; v < kV; ++v) {
        const int qq = hf * kV + v;  // 16-byte vector of the row
        const uint4 x = *reinterpret_cast<const uint4*>(sQ + (qq >> 3) * 16384 + sw128_offset(r, qq & 7));
        u[4 * v] = x.x;
        u[4 * v + 1] = x.y;
        u[4 * v + 2] = x.z;
        u[4 * v + 3] = x.w;
      }
      if constexpr (D == 128)
        tmem_st32(tmem + kTQ + lane_base + hf * 32, u);
      else
        tmem_st16(tmem + kTQ + lane_base + hf * 16, u);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(qtmem);
    }
    for (int j = 0; j < n_sel; ++j) {
      const bool okw = warp_wait(sfull + j % kSBufs, (j / kSBufs) & 1, a.status, abort_flag);
      const uint32_t tS = tmem + (j % kSBufs) * 128 + lane_base + hf * 64;
      uint32_t u0[32], u1[32];
      uint32_t vm0 = ~0u, vm1 = ~0u;  // key rows of J inside the grid
      float mx = -INFINITY;
      bool fullj = true;
      if (okw) {
        tc_fence_after();
        const int J = sel[j];
        fullj = a.all_full || block_is_full(a.g, J);
        if (!fullj) {
          vm0 = block_rows_mask32(a.g, J, hf * 64);
          vm1 = block_rows_mask32(a.g, J, hf * 64 + 32);
        }
        float c0, c1;
        tmem_ld32_max(tS, u0, c0);  // values and, from the same load, their maximum
        tmem_ld32_max(tS + 32, u1, c1);
        tmem_wait_ld();
        if (fullj) {
          mx = fmaxf(c0, c1);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if ((vm0 >> e) & 1u) mx = fmaxf(mx, __uint_as_float(u0[e]));
            if ((vm1 >> e) & 1u) mx = fmaxf(mx, __uint_as_float(u1[e]));
          }
        }
        half_max[((j & 1) * 2 + hf) * 128 + r] = mx;
      }
      if (!named_bar_and(2 + quarter, 64, okw)) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, half_max[((j & 1) * 2 + (hf ^ 1)) * 128 + r]) * a.scale_log2;  // same in both warps
      const float m_new = fmaxf(m, mx);
      if (j == 0) {
        m = m_new;
      } else {
        const bool need = m_new > m + rescale_threshold<kF16>();
        if (__any_sync(0xffffffffu, need)) {  // both warps of the pair take this branch together
          // O holds sum_{<j} P V relative to m: wait for P_{j-1} V_{j-1} (odone of block
          // j - 1; S_j being done implies the products of block j - 3 and before are), then
          // rescale this warp's half of O.
          const int jp = j - 1;
          if (!named_bar_and(2 + quarter, 64, mbar_wait(odone + (jp & 1), (jp >> 1) & 1, a.status, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = need ? ex2(m - m_new) : 1.f;
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t u[32];
            const uint32_t tc = tO + hf * (D / 2) + cc * 32;
            tmem_ld32(tc, u);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            tmem_st32(tc, u);
          }
          tmem_wait_st();
          l *= alpha;
          if (need) m = m_new;
        }
      }
      // P over S (fp16, or bf16 hi + lo).  Full tiles skip the per-key mask.
      if (fullj)
        softmax_p<false, kF16>(u0, u1, vm0, vm1, m, a.scale_log2, tS, l);
      else
        softmax_p<true, kF16>(u0, u1, vm0, vm1, m, a.scale_log2, tS, l);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(pfull + j % kSBufs);
    }
    // Epilogue: O / (l_0 + l_1) -> bf16 (and fp32) -> swizzled staging tiles (the Q tile,
    // and the K ring for fp32) -> TMA stores.  `drain` completes once every MMA of the
    // CTA has finished (the MMA warp commits it last).
    if (n_sel > 0) ok = mbar_wait(drain, 0, a.status, abort_flag) && ok;
    tc_fence_after();
    half_l[hf * 128 + r] = l;
    ok = pair_sync(0) && ok;
    const float L = l + half_l[(hf ^ 1) * 128 + r];
    const float inv = (n_sel > 0 && L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
    for (int cc = 0; cc < D / 64; ++cc) {
      const int col = hf * (D / 2) + cc * 32;  // first O column of this 32-column chunk
      float f[32];
      if (n_sel > 0) {
        uint32_t u[32];
        tmem_ld32(tO + col, u);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(u[e]) * inv;
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = 0.f;
      }
      if (kO16) {
        uint8_t* dst = sQ + (col >> 6) * 16384;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 v;
          v.x = pack_bf16(f[q4 * 8 + 0], f[q4 * 8 + 1]);
          v.y = pack_bf16(f[q4 * 8 + 2], f[q4 * 8 + 3]);
          v.z = pack_bf16(f[q4 * 8 + 4], f[q4 * 8 + 5]);
          v.w = pack_bf16(f[q4 * 8 + 6], f[q4 * 8 + 7]);
          *reinterpret_cast<uint4*>(dst + sw128_offset(r, ((col & 63) >> 3) + q4)) = v;
        }
      }
      if (kO32) {  // fp32 boxes of 32 columns
        uint8_t* box = sK + (col >> 5) * 16384;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(box + sw128_offset(r, q)) =
              make_uint4(__float_as_uint(f[4 * q]), __float_as_uint(f[4 * q + 1]), __float_as_uint(f[4 * q + 2]),
                         __float_as_uint(f[4 * q + 3]));
      }
    }
    const int n = block_row_token(a.g, I, r);
    if (hf == 0 && n >= 0)
      a.LSE[((long long)a.b * a.Hh + h) * a.N + n] =
          (n_sel > 0 && L > 0.f) ? (m + __log2f(L)) * 0.69314718055994531f : -INFINITY;
    fence_async_smem();
    named_bar(1, 256);
    if (warp == 4 && lane == 0) {
      if (kO16) {
#pragma unroll
        for (int c = 0; c < C::CH; ++c) tma_store_5d(&tmO, sQ + c * 16384, c * 64, h, w0, h0, t0);
      }
      if (kO32) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tma_store_5d(&tmO32, sK + c * 16384, c * 32, h, w0, h0, t0);
      }
      bulk_commit();
      bulk_wait_all();
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kF16, bool kO16, bool kO32>
cudaError_t launch_fwd(const Prob& p, const void* Q, const void* K, const void* V, const int32_t* idx, int kb_begin,
                       int kb_end, const uint8_t* qb_active, void* O, float* LSE, float* O32, cudaStream_t st) {
  using C = FwdCfg<D>;
  const size_t smem = 1024 + C::SMEM_TILES + 8 * (2 * (C::KST + C::VST) + 2 * kSBufs + 9) + 4 * (3 + 16) +
                      4 * 768 + 4 * kSeenWords + 4 * (size_t)p.k + 64;
  auto kern = fwd_tc_kernel<D, kF16, kO16, kO32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  const size_t per_batch = (size_t)p.N * p.Hh * p.d * 2;
  const TokType in_t = kF16 ? kTokF16 : kTokBF16;
  for (int b = 0; b < p.B; ++b) {
    CUtensorMap mQ, mK, mV, mO, mO32;
    const char* q = static_cast<const char*>(Q) + b * per_batch;
    const char* k = static_cast<const char*>(K) + b * per_batch;
    const char* v = static_cast<const char*>(V) + b * per_batch;
    const Geom& g = p.g;
    if (!make_token_map(&mQ, q, in_t, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw) ||
        !make_token_map(&mK, k, in_t, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw) ||
        !make_token_map(&mV, v, in_t, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw))
      return cudaErrorInvalidValue;
    if (kO16 && !make_token_map(&mO, static_cast<char*>(O) + b * per_batch, kTokBF16, g.T, g.H, g.W, p.Hh, p.d, g.bt,
                                g.bh, g.bw))
      return cudaErrorInvalidValue;
    if (kO32 && !make_token_map(&mO32, O32 + (size_t)b * p.N * p.Hh * p.d, kTokF32, g.T, g.H, g.W, p.Hh, p.d, g.bt,
                                g.bh, g.bw))
      return cudaErrorInvalidValue;
    if (!kO16) mO = mQ;   // not read
    if (!kO32) mO32 = mQ;  // not read
    FwdArgs a;
    a.g = g;
    a.Hh = p.Hh;
    a.k = p.k;
    a.b = b;
    a.kb_begin = kb_begin;
    a.kb_end = kb_end;
    a.all_full = (g.T % g.bt == 0 && g.H % g.bh == 0 && g.W % g.bw == 0) ? 1 : 0;
    a.N = p.N;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.idx = idx;
    a.qb_active = qb_active;
    a.LSE = LSE;
    a.status = status;
    dim3 grid(g.nb, p.Hh);
    kern<<<grid, kThreads, smem, st>>>(mQ, mK, mV, mO, mO32, a);
    note_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t fwd_tc(const Prob& p, const void* Q, const void* K, const void* V, const int32_t* idx, int kb_begin,
                   int kb_end, const uint8_t* qb_active, void* O, bool out_f32, float* LSE, cudaStream_t st) {
  float* O32 = static_cast<float*>(O);
  if (p.d == 64)
    return out_f32 ? launch_fwd<64, false, false, true>(p, Q, K, V, idx, kb_begin, kb_end, qb_active, nullptr, LSE, O32,
                                                        st)
                   : launch_fwd<64, false, true, false>(p, Q, K, V, idx, kb_begin, kb_end, qb_active, O, LSE, nullptr,
                                                        st);
  return out_f32 ? launch_fwd<128, false, false, true>(p, Q, K, V, idx, kb_begin, kb_end, qb_active, nullptr, LSE, O32,
                                                       st)
                 : launch_fwd<128, false, true, false>(p, Q, K, V, idx, kb_begin, kb_end, qb_active, O, LSE, nullptr,
                                                       st);
}

cudaError_t fwd_tc_f16(const Prob& p, const void* Q16, const void* K16, const void* V16, const int32_t* idx, void* O,
                       float* LSE, float* O32, cudaStream_t st) {
  if (p.d == 64) return launch_fwd<64, true, true, true>(p, Q16, K16, V16, idx, 0, p.g.nb, nullptr, O, LSE, O32, st);
  return launch_fwd<128, true, true, true>(p, Q16, K16, V16, idx, 0, p.g.nb, nullptr, O, LSE, O32, st);
}

}  // namespace sda
