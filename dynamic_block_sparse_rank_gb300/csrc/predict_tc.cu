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
//   proj_kernel   q~ (and k~) per (tile, head): d/16 tensor-core MMAs of the
//                 TMA-loaded tile with W^T (fp32 accumulation), rounded to bf16
//                 and written straight into the tensor-core operand layout
//                 (no-swizzle K-major core matrices, tile after tile), so the
//                 score kernel fetches each tile with one bulk copy.  Rows
//                 outside the grid are zeros.
//   score_kernel  per (QB query blocks, head), QB = 4 when its score rows fit in
//                 shared memory (else 2 or 1): streams every k~ tile through a
//                 ring; each (key block, query block) pair is one M=128, N=128,
//                 K=r accumulation in one of four 128-column TMEM buffers, issued
//                 by one of two warp-converged MMA warps (even and odd pairs).
//                 Four epilogue groups of four warps (one per TMEM lane
//                 quarter) each drain one buffer: the
//                 reducing TMEM load gives each thread the max of its columns,
//                 then one redux.sync over order-preserving keys and a shared-
//                 memory atomic max per warp.  Four buffers let the MMA run
//                 three pairs ahead of the slowest group.  When the rows of n_b
//                 scores are complete, each query block's team of warps selects
//                 its top k (radix select).
#include "internal.h"
#include "topk.cuh"

namespace sda {

namespace {

// ------------------------------------------------------------------ projection
__device__ __forceinline__ uint32_t op_offset(int row, int col, int r) { return coremat_offset(row, col, r); }

// One CTA per (128-token tile, head): the tile arrives by TMA (the 5-D box of one
// space-time tile, 128-byte swizzled, zero outside the grid), W^T is written to shared
// memory in the operand layout, and d/16 MMAs (M=128, N=R) accumulate q~ (or k~) in
// TMEM; each thread then rounds its row to bf16 and writes it in the score kernel's
// operand layout.  fp32 accumulation of exact bf16 products, as the product of the
// projection needs.
template <int R, int D>
__global__ void __launch_bounds__(128) proj_kernel(const __grid_constant__ CUtensorMap tmX, Geom g, int Hh,
                                                   const __nv_bfloat16* __restrict__ W, uint8_t* __restrict__ out,
                                                   int b, unsigned* status) {
  constexpr int CH = D / 64;
  constexpr uint32_t kCols = R <= 32 ? 32 : 64;  // TMEM allocation (a power of two)
  const int I = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sX = smem;                 // 128 x D bf16, CH chunks of 16 KB
  uint8_t* sW = sX + CH * 16384;      // W^T: R x D bf16, no-swizzle K-major core matrices
  uint64_t* bars = reinterpret_cast<uint64_t*>(sW + R * D * 2);
  uint64_t* xfull = bars;
  uint64_t* done = bars + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int t0, h0, w0;
  block_origin(g, I, t0, h0, w0);
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(xfull, 1);
    mbar_init(done, 1);
    fence_mbar_init();
    prefetch_tmap(&tmX);
    mbar_expect_tx(xfull, CH * 16384);
#pragma unroll
    for (int c = 0; c < CH; ++c) tma_load_5d(sX + c * 16384, &tmX, xfull, c * 64, h, w0, h0, t0);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  // W[h] is [D, R] row-major; element (k, n) goes to row n, column k of W^T.
  const __nv_bfloat16* Wh = W + (long long)h * D * R;
  for (int e = tid; e < D * R; e += 128) {
    const int k = e / R, n = e % R;
    *reinterpret_cast<__nv_bfloat16*>(sW + op_offset(n, k, D)) = Wh[e];
  }
  fence_async_smem();  // W^T (generic stores) is read by the MMA (async proxy)
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  if (warp == 0) {
    const uint32_t leader = elect_leader();
    ok = warp_wait(xfull, 0, status, abort_flag);
    if (ok) {
      tc_fence_after();
      constexpr uint32_t id = idesc_bf16(128, R, 0, 0);
      const uint64_t dX = smem_desc(smem_u32(sX), 16, 1024, 2);
      const uint64_t dW = smem_desc(smem_u32(sW), 128, (D / 8) * 128, 0);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_by(leader, tmem, dX + (uint64_t)((kk >> 2) * (16384 >> 4) + (kk & 3) * 2),
                  dW + (uint64_t)(kk * (256 >> 4)), id, kk > 0);
      mma_commit_by(leader, done);
    }
  }
  // every thread: row = TMEM lane = tid
  ok = mbar_wait(done, 0, status, abort_flag) && ok;
  tc_fence_after();
  if (__all_sync(0xffffffffu, ok)) {
    uint8_t* tile = out + (((long long)b * Hh + h) * g.nb + I) * (128LL * R * 2);
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
    for (int c = 0; c < R; c += 16) {
      uint32_t u[16];
      tmem_ld16(taddr + c, u);
      tmem_wait_ld();
#pragma unroll
      for (int a = 0; a < 16; a += 8) {
        uint4 v;
        v.x = pack_bf16(__uint_as_float(u[a + 0]), __uint_as_float(u[a + 1]));
        v.y = pack_bf16(__uint_as_float(u[a + 2]), __uint_as_float(u[a + 3]));
        v.z = pack_bf16(__uint_as_float(u[a + 4]), __uint_as_float(u[a + 5]));
        v.w = pack_bf16(__uint_as_float(u[a + 6]), __uint_as_float(u[a + 7]));
        *reinterpret_cast<uint4*>(tile + op_offset(tid, c + a, R)) = v;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------------ scores + top-k
template <int R>
struct ScoreCfg {
  static constexpr int TB = 128 * R * 2;      // bytes of one operand tile
  static constexpr int ST = R <= 32 ? 8 : 4;  // k~ ring depth
};
// warp 0 producer, warps 1 and 18 the MMA issuers (even and odd pairs), warps 2..17
// epilogue in 4 groups of 4 (one warp per TMEM lane quarter); group g drains
// accumulator buffer g.
constexpr int kEpiWarps = 16;
// warp 0 copies, warps 1 and 2 + kEpiWarps issue the MMAs (even and odd pairs), warps 2 .. 1 + kEpiWarps drain
constexpr int kScoreThreads = (3 + kEpiWarps) * 32;
constexpr int kAccBufs = 4;  // TMEM accumulators of 128 columns: one (query block, key block) pair each

struct ScoreArgs {
  Geom g;
  int Hh, k, b;
  const uint8_t* qt;
  const uint8_t* kt;
  int32_t* idx;
  float* score;
  unsigned* status;
};

// Shared memory of one CTA: QB query tiles, the k~ ring, QB rows of nb keys,
// top-k scratch, barriers, flags.  The first 1024 bytes absorb the alignment.
__host__ __device__ inline size_t score_smem_bytes(int R, int ST, int QB, int nb) {
  const size_t TB = (size_t)128 * R * 2;
  size_t off = 1024 + (QB + ST) * TB + (size_t)QB * nb * 4 + QB * sizeof(TopkScratch);
  off = (off + 7) & ~size_t(7);
  off += 8 * (1 + 2 * ST + 2 * kAccBufs + 1) + 8 + nb;
  return off + 64;
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

// One CTA per (QB consecutive query blocks, head).  For every key block J and
// query block q the pair P = J QB + q is accumulated (M=128 query rows, N=128
// key rows, K=r) in TMEM buffer P mod 4 and reduced to its max by group P mod 4.
template <int R, int QB>
__global__ void __launch_bounds__(kScoreThreads, 1) score_kernel(ScoreArgs a) {
  constexpr int TB = ScoreCfg<R>::TB;
  constexpr int kStages = ScoreCfg<R>::ST;
  const int nb = a.g.nb;
  const int h = blockIdx.y;
  const int I0 = QB * blockIdx.x;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                                                // QB query tiles
  uint8_t* sB = sA + QB * TB;                                        // kStages key tiles
  unsigned* keys = reinterpret_cast<unsigned*>(sB + kStages * TB);  // QB x nb
  TopkScratch* tks = reinterpret_cast<TopkScratch*>(keys + QB * nb);
  uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(tks + QB) + 7) & ~uintptr_t(7));
  uint64_t* afull_q = bars;            // query tiles loaded
  uint64_t* kfull = bars + 1;          // kStages
  uint64_t* kempty = kfull + kStages;  // kStages
  uint64_t* accf = kempty + kStages;   // kAccBufs: accumulator holds a finished pair
  // kAccBufs counters (in the space of as many barriers): warps that have read buffer b
  // out, 4 per use.  The MMA warp usually finds the count reached, and one shared load
  // costs far less than a wait on an already completed mbarrier.
  unsigned* drained = reinterpret_cast<unsigned*>(accf + kAccBufs);
  uint64_t* drain = accf + 2 * kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  uint8_t* full = reinterpret_cast<uint8_t*>(abort_flag + 1);  // nb: key block J lies inside the grid

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(afull_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kfull + s, 1);
      mbar_init(kempty + s, 2);  // both MMA issuers
    }
    for (int s = 0; s < kAccBufs; ++s) {
      mbar_init(accf + s, 1);
      drained[s] = 0u;
    }
    mbar_init(drain, 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int e = tid; e < QB * nb; e += kScoreThreads) keys[e] = 0u;  // below every real key
  for (int J = tid; J < nb; J += kScoreThreads) full[J] = block_is_full(a.g, J) ? 1 : 0;
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long head_tiles = ((long long)a.b * a.Hh + h) * nb;
  const int n_pairs = nb * QB;

  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(afull_q, QB * TB);
      for (int q = 0; q < QB; ++q) {
        const int I = I0 + q < nb ? I0 + q : nb - 1;
        bulk_load(sA + q * TB, a.qt + (head_tiles + I) * TB, TB, afull_q);
      }
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
  } else if (warp == 1 || warp == 2 + kEpiWarps) {
    // Two issuers, each a whole warp with one elected lane issuing: warp 1 the even pairs,
    // warp 2 + kEpiWarps the odd ones, so that one issuer's hand-offs (its counter poll, the
    // fence, the commit) overlap the other's MMAs.  Both wait for every key stage and both
    // release it, so neither can run a stage ahead.  Descriptors advance by adding to the
    // start-address field (16-byte units).
    const int w = warp == 1 ? 0 : 1;
    const uint32_t leader = elect_leader();
    constexpr uint32_t id = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t SBO = (R / 8) * 128;
    const uint64_t dA = smem_desc(smem_u32(sA), 128, SBO, 0), dB = smem_desc(smem_u32(sB), 128, SBO, 0);
    bool ok = warp_wait(afull_q, 0, a.status, abort_flag);
    for (int J = 0; ok && J < nb; ++J) {
      const int s = J % kStages;
      if (!(ok = warp_wait(kfull + s, (J / kStages) & 1, a.status, abort_flag))) break;
#pragma unroll
      for (int q = 0; q < QB; ++q) {
        const int P = J * QB + q, buf = P & (kAccBufs - 1);
        if ((P & 1) != w) continue;
        // buffer `buf` was read out for its previous (P >> 2) uses: 4 warps each
        if (P >= kAccBufs && !(ok = warp_wait_count(drained + buf, 4u * (unsigned)(P >> 2), a.status, abort_flag)))
          break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < R / 16; ++kk)
          mma_ss_by(leader, tmem + buf * 128, dA + (uint64_t)((q * TB + kk * 256) >> 4),
                    dB + (uint64_t)((s * TB + kk * 256) >> 4), id, kk > 0);
        mma_commit_by(leader, accf + buf);
      }
      mma_commit_by(leader, kempty + s);
    }
    mma_commit_by(leader, drain);
    wait_plain(drain, 0);
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    const int e = warp - 2;
    const int grp = e >> 2;         // accumulator buffer this warp drains
    const int quarter = warp & 3;   // TMEM lanes 32 quarter .. 32 quarter + 31 (query rows)
    const int row = quarter * 32 + lane;
    unsigned rowok = 0;
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      const int I = I0 + q < nb ? I0 + q : nb - 1;
      rowok |= (block_row_token(a.g, I, row) >= 0 ? 1u : 0u) << q;
    }
    const uint32_t taddr = tmem + grp * 128 + ((uint32_t)(quarter * 32) << 16);
    for (int P = grp; P < n_pairs; P += kAccBufs) {
      const int J = P / QB, q = P % QB;
      if (!mbar_wait(accf + grp, (P >> 2) & 1, a.status, abort_flag)) break;
      tc_fence_after();
      const bool fj = full[J] != 0;
      uint32_t v0 = ~0u, v1 = ~0u, v2 = ~0u, v3 = ~0u;  // key rows of J inside the grid, per 32 columns
      if (!fj) {
        v0 = block_rows_mask32(a.g, J, 0);
        v1 = block_rows_mask32(a.g, J, 32);
        v2 = block_rows_mask32(a.g, J, 64);
        v3 = block_rows_mask32(a.g, J, 96);
      }
      uint32_t u0[32], u1[32];
      float m0, m1;
      tmem_ld32_max(taddr, u0, m0);  // the load also reduces each thread's 32 values to their max
      tmem_ld32_max(taddr + 32, u1, m1);
      tmem_wait_ld();
      float m = fj ? fmaxf(m0, m1) : masked_max64(v0, v1, u0, u1);
      tmem_ld32_max(taddr + 64, u0, m0);
      tmem_ld32_max(taddr + 96, u1, m1);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) count_release_add(drained + grp, 1u);  // values are in registers: the buffer may be refilled
      m = fmaxf(m, fj ? fmaxf(m0, m1) : masked_max64(v2, v3, u0, u1));
      // order-preserving key; 0 (below every real key) for rows/columns outside the grid
      const unsigned key = (((rowok >> q) & 1u) && m > -INFINITY) ? order_key(m) : 0u;
      const unsigned wmax = warp_max_u32(key);
      if (lane == 0 && wmax != 0u) atomicMax(keys + q * nb + J, wmax);
    }
    named_bar(1, kEpiWarps * 32);
    // keys -> scores (inverse of order_key), in place; then top-k per query block
    // by its team of kEpiWarps / QB warps
    constexpr int kTeam = (kEpiWarps / QB) * 32;
    const int q = e % QB;
    const int tg = (e / QB) * 32 + lane;
    unsigned* mykeys = keys + q * nb;
    float* srow = reinterpret_cast<float*>(mykeys);
    for (int J = tg; J < nb; J += kTeam) {
      const unsigned kq = mykeys[J];
      const unsigned u = (kq & 0x80000000u) ? (kq & 0x7FFFFFFFu) : ~kq;
      srow[J] = kq == 0u ? -INFINITY : __uint_as_float(u);
    }
    named_bar(2 + q, kTeam);
    const int I = I0 + q;
    if (I < nb) {
      if (a.score)
        for (int J = tg; J < nb; J += kTeam) a.score[(head_tiles + I) * nb + J] = srow[J];
      topk_select(srow, nb, a.k, a.idx + (head_tiles + I) * a.k, tg, kTeam, 2 + q, tks + q);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int R, int QB>
cudaError_t launch_score(const Prob& p, ScoreArgs& a, cudaStream_t st) {
  constexpr int kStages = ScoreCfg<R>::ST;
  const size_t raw = score_smem_bytes(R, kStages, QB, p.g.nb);
  // Keep one CTA per SM: each CTA owns all 512 TMEM columns.
  const size_t smem = raw > 120 * 1024 ? raw : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(score_kernel<R, QB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 sg((p.g.nb + QB - 1) / QB, p.Hh);
  for (int b = 0; b < p.B; ++b) {
    a.b = b;
    score_kernel<R, QB><<<sg, kScoreThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

template <int R, int D>
cudaError_t launch_proj(const Prob& p, const void* Q, const void* K, const void* Wq, const void* Wk, uint8_t* qt,
                        uint8_t* kt, unsigned* status, cudaStream_t st) {
  const size_t smem = 1024 + (size_t)(D / 64) * 16384 + (size_t)R * D * 2 + 8 * 2 + 8;
  cudaError_t e = cudaFuncSetAttribute(proj_kernel<R, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const size_t per_batch = (size_t)p.N * p.Hh * p.d * 2;
  const Geom& g = p.g;
  dim3 grid(g.nb, p.Hh);
  for (int b = 0; b < p.B; ++b) {
    CUtensorMap mQ, mK;
    if (!make_token_map(&mQ, static_cast<const char*>(Q) + b * per_batch, kTokBF16, g.T, g.H, g.W, p.Hh, p.d, g.bt,
                        g.bh, g.bw) ||
        !make_token_map(&mK, static_cast<const char*>(K) + b * per_batch, kTokBF16, g.T, g.H, g.W, p.Hh, p.d, g.bt,
                        g.bh, g.bw))
      return cudaErrorInvalidValue;
    proj_kernel<R, D><<<grid, 128, smem, st>>>(mQ, g, p.Hh, static_cast<const __nv_bfloat16*>(Wq), qt, b, status);
    proj_kernel<R, D><<<grid, 128, smem, st>>>(mK, g, p.Hh, static_cast<const __nv_bfloat16*>(Wk), kt, b, status);
  }
  return cudaGetLastError();
}

constexpr size_t kMaxScoreSmem = 227 * 1024;

template <int R>
cudaError_t launch_predict(const Prob& p, const void* Q, const void* K, const void* Wq, const void* Wk, int32_t* idx,
                           float* score, void* ws, cudaStream_t st) {
  const size_t tiles = (size_t)p.B * p.Hh * p.g.nb;
  uint8_t* qt = static_cast<uint8_t*>(ws);
  uint8_t* kt = qt + align_up(tiles * 128 * R * 2, 256);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  cudaError_t e = p.d == 64 ? launch_proj<R, 64>(p, Q, K, Wq, Wk, qt, kt, status, st)
                            : launch_proj<R, 128>(p, Q, K, Wq, Wk, qt, kt, status, st);
  if (e != cudaSuccess) return e;
  ScoreArgs a;
  a.g = p.g;
  a.Hh = p.Hh;
  a.k = p.k;
  a.qt = qt;
  a.kt = kt;
  a.idx = idx;
  a.score = score;
  a.status = status;
  constexpr int kStages = ScoreCfg<R>::ST;
  // As many query blocks per CTA as their score rows allow in shared memory.
  if (score_smem_bytes(R, kStages, 4, p.g.nb) <= kMaxScoreSmem)
    e = launch_score<R, 4>(p, a, st);
  else if (score_smem_bytes(R, kStages, 2, p.g.nb) <= kMaxScoreSmem)
    e = launch_score<R, 2>(p, a, st);
  else
    e = launch_score<R, 1>(p, a, st);
  note_launches(3 * p.B);
  return e;
}

}  // namespace

cudaError_t project_tc(const Prob& p, const void* Q, const void* K, const void* Wq, const void* Wk, void* ws,
                       cudaStream_t st) {
  const size_t tiles = (size_t)p.B * p.Hh * p.g.nb;
  uint8_t* qt = static_cast<uint8_t*>(ws);
  uint8_t* kt = qt + align_up(tiles * 128 * p.r * 2, 256);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  cudaError_t e = cudaErrorInvalidValue;
#define SDA_PROJ(R)                                                                     \
  case R:                                                                               \
    e = p.d == 64 ? launch_proj<R, 64>(p, Q, K, Wq, Wk, qt, kt, status, st)            \
                  : launch_proj<R, 128>(p, Q, K, Wq, Wk, qt, kt, status, st);          \
    break;
  switch (p.r) { SDA_PROJ(16) SDA_PROJ(32) SDA_PROJ(48) SDA_PROJ(64) }
#undef SDA_PROJ
  note_launches(2 * p.B);
  return e;
}

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
