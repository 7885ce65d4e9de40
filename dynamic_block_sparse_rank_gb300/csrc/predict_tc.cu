// Low-rank block predictor with top-k on the 5th-generation tensor cores.
//
// "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT
// Training", section 3a ("low-rank predictor": a cheap estimate picks the ~10%
// of attention worth computing) and 3b ("query grouping": neighbouring tokens
// share the decision).  Form: q~ = Q Wq, k~ = K Wk (rank r, per head);
// s(I, J) = max over i in I, j in J of q~_i . k~_j; keep the k highest J per I,
// ties to the lower J, reported ascending.
//
// Two kernels:
//   proj_kernel   q~ (and k~) per (tile, head): fp32 FMA over d, rounded to
//                 bf16 and written straight into the tensor-core operand layout
//                 (no-swizzle K-major core matrices, tile after tile), so the
//                 score kernel fetches each tile with one bulk copy.  Rows
//                 outside the grid are written as zeros.
//   score_kernel  per (two query blocks, head): streams every k~ tile through
//                 an 8-deep ring; for each key block J two MMAs (one per query
//                 block, M=128, N=128, K=r) land in a double-buffered TMEM
//                 accumulator; 16 epilogue warps (one per TMEM lane quarter,
//                 query block and column half) reduce each 128x128 tile to its
//                 max: the reducing TMEM load gives each thread the max of its
//                 columns, then one redux.sync over order-preserving keys and a
//                 shared-memory atomic max per warp.  When the row of n_b scores is complete, the 8
//                 warps of each query block select its top k (radix select).
#include "internal.h"
#include "topk.cuh"

namespace sda {

namespace {

// ------------------------------------------------------------------ projection
// Byte offset of element (row, col) of a 128 x r bf16 tile in the operand layout:
// 8x8 core matrices (8 rows x 16 bytes, rows contiguous), K-adjacent core
// matrices 128 bytes apart (LBO), 8-row groups r*16 bytes apart (SBO).
__device__ __forceinline__ uint32_t op_offset(int row, int col, int r) {
  return (uint32_t)((row >> 3) * (r >> 3) * 128 + (col >> 3) * 128 + (row & 7) * 16 + (col & 7) * 2);
}

template <int R>
__global__ void __launch_bounds__(256) proj_kernel(Geom g, int Hh, int d, long long N, const __nv_bfloat16* __restrict__ X,
                                                   const __nv_bfloat16* __restrict__ Wt, uint8_t* __restrict__ out, int b) {
  extern __shared__ float psm[];
  float* ws = psm;               // d x R
  float* xs = ws + d * R;        // 128 x (d + 1)
  const int I = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int ld = d + 1;
  for (int e = tid; e < d * R; e += 256) ws[e] = __bfloat162float(Wt[(long long)h * d * R + e]);
  const int vpr = d / 8;  // 16-byte vectors per row
  for (int e = tid; e < 128 * vpr; e += 256) {
    const int row = e / vpr, v = e % vpr;
    const int n = block_row_token(g, I, row);
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (n >= 0) raw = *reinterpret_cast<const uint4*>(X + (((long long)b * N + n) * Hh + h) * d + v * 8);
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      xs[row * ld + v * 8 + 2 * q] = __uint_as_float(w4[q] << 16);
      xs[row * ld + v * 8 + 2 * q + 1] = __uint_as_float(w4[q] & 0xFFFF0000u);
    }
  }
  __syncthreads();
  constexpr int PER = R / 2;  // outputs per thread: 128 rows x R cols over 256 threads
  const int row = tid >> 1, c0 = (tid & 1) * PER;
  float acc[PER];
#pragma unroll
  for (int a = 0; a < PER; ++a) acc[a] = 0.f;
  for (int c = 0; c < d; ++c) {
    const float x = xs[row * ld + c];
#pragma unroll
    for (int a = 0; a < PER; ++a) acc[a] = fmaf(x, ws[c * R + c0 + a], acc[a]);
  }
  uint8_t* tile = out + (((long long)b * Hh + h) * g.nb + I) * (128LL * R * 2);
#pragma unroll
  for (int a = 0; a < PER; a += 8) {
    uint4 v;
    v.x = pack_bf16(acc[a + 0], acc[a + 1]);
    v.y = pack_bf16(acc[a + 2], acc[a + 3]);
    v.z = pack_bf16(acc[a + 4], acc[a + 5]);
    v.w = pack_bf16(acc[a + 6], acc[a + 7]);
    *reinterpret_cast<uint4*>(tile + op_offset(row, c0 + a, R)) = v;
  }
}

// ------------------------------------------------------------------ scores + top-k
template <int R>
struct ScoreCfg {
  static constexpr int ST = R <= 32 ? 8 : 4;  // k~ ring depth
};
// warp 0 producer, warp 1 MMA, warps 2..17 epilogue: 4 warps per TMEM lane
// quarter, one for each (query block, column half) pair.
constexpr int kEpiWarps = 16;
constexpr int kScoreThreads = (2 + kEpiWarps) * 32;

struct ScoreArgs {
  Geom g;
  int Hh, k, b;
  const uint8_t* qt;
  const uint8_t* kt;
  int32_t* idx;
  float* score;
  unsigned* status;
};

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ unsigned warp_max_u32(unsigned v) {
  unsigned r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ bool wait_plain(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > SDA_WAIT_LIMIT_NS) return false;
  return true;
}

template <int R>
__global__ void __launch_bounds__(kScoreThreads, 1) score_kernel(ScoreArgs a) {
  constexpr int TB = 128 * R * 2;  // bytes of one operand tile
  constexpr int kStages = ScoreCfg<R>::ST;
  const int nb = a.g.nb;
  const int h = blockIdx.y;
  const int I0 = 2 * blockIdx.x;
  const int I1 = I0 + 1 < nb ? I0 + 1 : I0;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                      // 2 query tiles
  uint8_t* sB = sA + 2 * TB;               // kStages key tiles
  unsigned* keys = reinterpret_cast<unsigned*>(sB + kStages * TB);  // 2 x nb
  TopkScratch* tks = reinterpret_cast<TopkScratch*>(keys + 2 * nb);  // 2
  uint64_t* bars = reinterpret_cast<uint64_t*>(tks + 2);
  uint64_t* afull_q = bars;                // query tiles loaded
  uint64_t* kfull = bars + 1;              // kStages
  uint64_t* kempty = kfull + kStages;      // kStages
  uint64_t* accf = kempty + kStages;       // 2: accumulator buffer ready
  uint64_t* acce = accf + 2;               // 2: accumulator buffer drained
  uint64_t* drain = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  uint8_t* full = reinterpret_cast<uint8_t*>(abort_flag + 1);  // nb: key block J lies inside the grid

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(afull_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kfull + s, 1);
      mbar_init(kempty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(accf + s, 1);
      mbar_init(acce + s, kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int e = tid; e < 2 * nb; e += kScoreThreads) keys[e] = 0u;  // below every real key
  for (int J = tid; J < nb; J += kScoreThreads) full[J] = block_is_full(a.g, J) ? 1 : 0;
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long head_tiles = ((long long)a.b * a.Hh + h) * nb;

  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(afull_q, 2 * TB);
      bulk_load(sA, a.qt + (head_tiles + I0) * TB, TB, afull_q);
      bulk_load(sA + TB, a.qt + (head_tiles + I1) * TB, TB, afull_q);
      int issued = 0;
      for (int J = 0; J < nb; ++J) {
        const int s = J % kStages;
        if (J >= kStages && !mbar_wait(kempty + s, ((J / kStages) - 1) & 1, a.status, abort_flag)) break;
        mbar_expect_tx(kfull + s, TB);
        bulk_load(sB + s * TB, a.kt + (head_tiles + J) * TB, TB, kfull + s);
        issued = J + 1;
      }
      if (*abort_flag) {
        wait_plain(afull_q, 0);
        for (int J = issued - kStages < 0 ? 0 : issued - kStages; J < issued; ++J)
          wait_plain(kfull + J % kStages, (J / kStages) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t SBO = (R / 8) * 128;
      const uint32_t aA = smem_u32(sA), aB = smem_u32(sB);
      bool ok = mbar_wait(afull_q, 0, a.status, abort_flag);
      for (int J = 0; ok && J < nb; ++J) {
        const int s = J % kStages, buf = J & 1;
        if (!mbar_wait(kfull + s, (J / kStages) & 1, a.status, abort_flag)) break;
        if (J >= 2 && !mbar_wait(acce + buf, ((J >> 1) - 1) & 1, a.status, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
#pragma unroll
          for (int kk = 0; kk < R / 16; ++kk) {
            const uint64_t da = smem_desc(aA + q * TB + kk * 256, 128, SBO, 0);
            const uint64_t db = smem_desc(aB + s * TB + kk * 256, 128, SBO, 0);
            mma_ss(tmem + buf * 256 + q * 128, da, db, id, kk > 0);
          }
        }
        mma_commit(accf + buf);
        mma_commit(kempty + s);
      }
      mma_commit(drain);
      wait_plain(drain, 0);
    }
    __syncwarp();
  } else {
    // epilogue warp e: TMEM lane quarter = warp % 4, (query block, column half) = e / 4
    const int e = warp - 2;
    const int quarter = warp & 3;
    const int grp = (e >> 2) >> 1, half = (e >> 2) & 1;
    const int I = grp ? I1 : I0;
    const int row = quarter * 32 + lane;
    const bool row_ok = block_row_token(a.g, I, row) >= 0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    unsigned* mykeys = keys + grp * nb;
    for (int J = 0; J < nb; ++J) {
      const int buf = J & 1;
      if (!mbar_wait(accf + buf, (J >> 1) & 1, a.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + buf * 256 + grp * 128 + half * 64 + lane_base;
      uint32_t u0[32], u1[32];
      float mx0, mx1;
      tmem_ld32_max(taddr, u0, mx0);  // the load also reduces each thread's 32 values to their max
      tmem_ld32_max(taddr + 32, u1, mx1);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce + buf);  // values are in registers: the buffer may be refilled
      float m;
      if (full[J]) {
        m = fmaxf(mx0, mx1);
      } else {
        m = -INFINITY;
        const uint32_t v0 = block_rows_mask32(a.g, J, half * 64), v1 = block_rows_mask32(a.g, J, half * 64 + 32);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if ((v0 >> c) & 1u) m = fmaxf(m, __uint_as_float(u0[c]));
          if ((v1 >> c) & 1u) m = fmaxf(m, __uint_as_float(u1[c]));
        }
      }
      // order-preserving key; 0 (below every real key) for rows/columns outside the grid
      const unsigned key = (row_ok && m > -INFINITY) ? order_key(m) : 0u;
      const unsigned wmax = warp_max_u32(key);
      if (lane == 0 && wmax != 0u) atomicMax(mykeys + J, wmax);
    }
    named_bar(1, kEpiWarps * 32);
    // keys -> scores (inverse of order_key), in place; then top-k per query block by its 8 warps
    const int tg = (e & 7) * 32 + lane;  // thread index inside this query block's 8 warps
    float* srow = reinterpret_cast<float*>(mykeys);
    for (int J = tg; J < nb; J += 256) {
      const unsigned kq = mykeys[J];
      const unsigned u = (kq & 0x80000000u) ? (kq & 0x7FFFFFFFu) : ~kq;
      srow[J] = kq == 0u ? -INFINITY : __uint_as_float(u);
    }
    named_bar(2 + grp, 256);
    const bool write = grp == 0 || I1 != I0;
    if (write) {
      if (a.score)
        for (int J = tg; J < nb; J += 256) a.score[(head_tiles + I) * nb + J] = srow[J];
      topk_select(srow, nb, a.k, a.idx + (head_tiles + I) * a.k, tg, 256, 2 + grp, tks + grp);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int R>
cudaError_t launch_predict(const Prob& p, const void* Q, const void* K, const void* Wq, const void* Wk, int32_t* idx,
                           float* score, void* ws, cudaStream_t st) {
  const size_t tiles = (size_t)p.B * p.Hh * p.g.nb;
  uint8_t* qt = static_cast<uint8_t*>(ws);
  uint8_t* kt = qt + align_up(tiles * 128 * R * 2, 256);
  const size_t psmem = ((size_t)p.d * R + 128 * (p.d + 1)) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(proj_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
  if (e != cudaSuccess) return e;
  dim3 pg(p.g.nb, p.Hh);
  for (int b = 0; b < p.B; ++b) {
    proj_kernel<R><<<pg, 256, psmem, st>>>(p.g, p.Hh, p.d, p.N, static_cast<const __nv_bfloat16*>(Q),
                                           static_cast<const __nv_bfloat16*>(Wq), qt, b);
    proj_kernel<R><<<pg, 256, psmem, st>>>(p.g, p.Hh, p.d, p.N, static_cast<const __nv_bfloat16*>(K),
                                           static_cast<const __nv_bfloat16*>(Wk), kt, b);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  constexpr int kStages = ScoreCfg<R>::ST;
  const size_t ssmem_raw = 1024 + (size_t)(2 + kStages) * 128 * R * 2 + 2 * (size_t)p.g.nb * 4 + 2 * sizeof(TopkScratch) +
                       8 * (1 + 2 * kStages + 5) + 16 + (size_t)p.g.nb + 64;
  // Keep one CTA per SM: each CTA owns all 512 TMEM columns.
  const size_t ssmem = ssmem_raw > 120 * 1024 ? ssmem_raw : 120 * 1024;
  if ((e = cudaFuncSetAttribute(score_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssmem)) !=
      cudaSuccess)
    return e;
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  ScoreArgs a;
  a.g = p.g;
  a.Hh = p.Hh;
  a.k = p.k;
  a.qt = qt;
  a.kt = kt;
  a.idx = idx;
  a.score = score;
  a.status = status;
  dim3 sg((p.g.nb + 1) / 2, p.Hh);
  for (int b = 0; b < p.B; ++b) {
    a.b = b;
    score_kernel<R><<<sg, kScoreThreads, ssmem, st>>>(a);
  }
  note_launches(3 * p.B);
  return cudaGetLastError();
}

}  // namespace

size_t predict_ws_tc(const Prob& p) {
  return 2 * align_up((size_t)p.B * p.Hh * p.g.nb * 128 * p.r * 2, 256);
}

cudaError_t predict_tc(const Prob& p, const void* Q, const void* K, const void* Wq, const void* Wk, int32_t* idx,
                       float* score, void* ws, cudaStream_t st) {
  switch (p.r) {
    case 16:
      return launch_predict<16>(p, Q, K, Wq, Wk, idx, score, ws, st);
    case 32:
      return launch_predict<32>(p, Q, K, Wq, Wk, idx, score, ws, st);
    case 48:
      return launch_predict<48>(p, Q, K, Wq, Wk, idx, score, ws, st);
    case 64:
      return launch_predict<64>(p, Q, K, Wq, Wk, idx, score, ws, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sda
