// Training signal of the low-rank predictor: the gradient of a distillation loss
// with respect to Wq and Wk.
//
// "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT Training",
// section 4 ("two-stage training": in the first stage the predictor learns while
// attention runs dense).  The page gives no loss.  Read: the low-rank block score
// s(I, J) = max over i in I, j in J of q~_i . k~_j estimates the full-rank block-max
// logit t(I, J) = max of q_i . k_j over the same pairs, and
// L = 1/2 sum over (b, h, I, J) of (s - t)^2.  The max passes its gradient to its
// maximising pair (i*, j*), the first in the tiles' (row, column) order on ties; the
// bf16 rounding of q~ and k~ passes it unchanged; t, computed from the attention's own
// Q and K, is a target.  With e = s - t:
//   dL/dWq[h] = sum e Q_i*^T k~_j*,   dL/dWk[h] = sum e K_j*^T q~_i*.
//
// Steps (after the projections of the predictor, which fill the q~ / k~ tiles):
//   tile_norm_kernel  the largest row norm of every q~ / k~ tile, which bounds the
//                     fp32 rounding of any low-rank score of a tile pair;
//   distill_kernel    per (2 query blocks, head): for every key block J and query
//                     block q, S = Q_I K_J^T (K = d) and S~ = q~_I k~_J^T (K = r) on
//                     the tensor cores (one MMA issuer warp per query block) into the
//                     block's TMEM buffer pair; an epilogue group of four warps takes
//                     t = max S, hands the S half back, finds the fp32 maximum of S~
//                     and marks the entries within twice its rounding bound as
//                     candidates, hands the S~ half back and passes the candidates to
//                     a scorer warp (two per group, alternate pairs), which re-scores
//                     them from the bf16 operands with the whole warp (a compensated
//                     fp32 sum of exact products good to about 2^-44; equal operands
//                     tie exactly and go to the first row, then column), then adds
//                     e k~_j* to the query token's r-vector G_q[i*] and
//                     e q~_i* to the key token's G_k[j*] (fp32 atomics) and e^2 / 2
//                     to the loss;
//   dw_kernel         dWq[h] = sum_n Q_n^T G_q[n] and dWk[h] = sum_n K_n^T G_k[n].
#include "internal.h"

namespace sda {

namespace {

constexpr int kDistQB = 2;                     // query blocks per CTA (one per epilogue group)
// warp 0 TMA, warps 1-2 one MMA issuer per group, warps 3-10 two epilogue groups, warps 11-14
// two scorers per group (one per slot: alternate pairs)
constexpr int kDistMma = 1, kDistEpi = kDistMma + kDistQB, kDistScore = kDistEpi + 4 * kDistQB;
constexpr int kDistThreads = (kDistScore + 2 * kDistQB) * 32;
constexpr int kCandWords = 2 * kDistQB * 4 * 4 * 32;  // candidate masks: [slot][group][quarter][chunk][lane]
constexpr float kUnitF = 5.9604644775390625e-8f;  // 2^-24, fp32's unit roundoff

template <int R, int D>
struct DistCfg {
  static constexpr int TB = 128 * R * 2;   // q~ / k~ tile bytes (unswizzled operand layout)
  static constexpr int TILE = 128 * D * 2;  // Q / K tile bytes (128B-swizzled, D / 64 chunks of 16 KB)
  static constexpr int CH = D / 64;
  static constexpr int JS = (R <= 32 || D == 64) ? 3 : 2;  // key-block ring stages
  static constexpr int TILES_BYTES = kDistQB * (TILE + TB) + JS * (TILE + TB);
};

struct DistArgs {
  Geom g;
  int Hh, b;
  long long N;
  const uint8_t* qt;    // [B, Hh, nb] tiles of 128 x r bf16
  const uint8_t* kt;
  const float* qnorm;   // [B, Hh, nb]: largest row 2-norm of each q~ tile
  const float* knorm;
  float* Gq;            // [B, Hh, N, r]
  float* Gk;
  double* loss;
  float* s_out;         // [B, Hh, nb, nb] or null
  float* t_out;
  unsigned* status;
};

__device__ __forceinline__ bool wait_plain(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > SDA_WAIT_LIMIT_NS) return false;
  return true;
}

__device__ __forceinline__ float bf16_at(const uint8_t* tile, int row, int col, int ncols) {
  const uint16_t v = *reinterpret_cast<const uint16_t*>(tile + coremat_offset(row, col, ncols));
  return __uint_as_float((uint32_t)v << 16);
}

// One warp per tile: max over its 128 rows of the row's 2-norm (rows outside the grid
// are zeros).
template <int R>
__global__ void tile_norm_kernel(const uint8_t* __restrict__ tiles, long long n_tiles, float* __restrict__ out) {
  const long long t = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= n_tiles) return;  // whole warps
  const uint8_t* tile = tiles + t * (128LL * R * 2);
  float best = 0.f;
  for (int row = lane; row < 128; row += 32) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < R; ++c) {
      const float v = bf16_at(tile, row, c, R);
      s = fmaf(v, v, s);
    }
    best = fmaxf(best, sqrtf(s));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
  if (lane == 0) out[t] = best;
}

// A candidate's low-rank score as an unevaluated sum hi + lo of two fp32 numbers,
// normalised so that hi = fl(hi + lo).  FP64 issues at a small fraction of the FP32 rate
// on this part, so the re-scoring of candidates stays in fp32.
struct Score2 {
  float hi, lo;
};

// The lexicographic order of candidate maxima: larger score, then lower row, then lower
// column.  On normalised pairs, (hi, lo) order is the order of hi + lo.
__device__ __forceinline__ bool better(Score2 v, int i, int j, Score2 bv, int bi, int bj) {
  if (v.hi != bv.hi) return v.hi > bv.hi;
  if (v.lo != bv.lo) return v.lo > bv.lo;
  return i < bi || (i == bi && j < bj);
}

// q~_row . k~_j from the bf16 tiles, formed by a whole warp: every bf16 x bf16 product is
// exact in fp32, and each addition's rounding error is recovered exactly (two-sum) and
// summed in lo, so hi + lo is the exact sum up to about r^2 2^-48 of sum |q~_c k~_c|.
// Lane c takes the products of columns c, c + 32, ... (two-sum within the lane), then five
// butterfly steps add the partners' (hi, lo) with the exact error of each hi addition
// (two-sum is error-free in either operand order, so both partners hold identical values
// after every step and all lanes end with the same result; equal operands give equal
// results).  About 200 cycles for one candidate, against ~1,200 for one lane walking the
// r terms.  A row of a tile is r / 8 runs of 16 bytes, 128 bytes apart (the core-matrix
// layout).
template <int R>
__device__ __forceinline__ Score2 exact_score_warp(const uint8_t* qtile, int row, const uint8_t* ktile, int j,
                                                   int lane) {
  float hi = 0.f, lo = 0.f;
#pragma unroll
  for (int u = 0; u < (R + 31) / 32; ++u) {
    const int c = lane + 32 * u;
    const float p = c < R ? bf16_at(qtile, row, c, R) * bf16_at(ktile, j, c, R) : 0.f;
    const float t = hi + p, bb = t - hi;
    lo += (hi - (t - bb)) + (p - bb);
    hi = t;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, hi, o), ol = __shfl_xor_sync(0xffffffffu, lo, o);
    const float t = hi + oh, bb = t - hi;
    const float err = (hi - (t - bb)) + (oh - bb);
    lo = (lo + ol) + err;
    hi = t;
  }
  const float u = hi + lo;  // |lo| <= |hi| here: fast two-sum
  return {u, lo - (u - hi)};
}

template <int R, int D>
__global__ void __launch_bounds__(kDistThreads, 1)
    distill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK, DistArgs a) {
  using C = DistCfg<R, D>;
  constexpr int JS = C::JS;
  // twice the rounding bound of one low-rank score per unit of ||q~|| ||k~||: (4 r + 4) u
  constexpr float kBoundCoef = (4.0f * R + 4.0f) * kUnitF;
  const int nb = a.g.nb;
  const int h = blockIdx.y;
  const int I0 = kDistQB * blockIdx.x;
  // Key blocks are visited from a per-CTA offset within a window of 64: CTAs running side by
  // side add their G_k terms to different key tokens (the same few rows of one key block
  // would otherwise take every CTA's atomics at once) while their key tiles stay close in L2.
  const int rot = (int)(blockIdx.x % 64u) % nb;
  auto key_block = [&](int it) {
    const int J = it + rot;
    return J >= nb ? J - nb : J;
  };

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                        // kDistQB x TILE
  uint8_t* sK = sQ + kDistQB * C::TILE;      // JS x TILE
  uint8_t* sqt = sK + JS * C::TILE;          // kDistQB x TB
  uint8_t* skt = sqt + kDistQB * C::TB;      // JS x TB
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::TILES_BYTES);
  uint64_t* qfull = bars;
  uint64_t* kfull = qfull + 1;        // JS
  uint64_t* kempty = kfull + JS;      // JS: the MMAs and both epilogue groups are done with the stage
  uint64_t* accf = kempty + JS;       // 2: a buffer pair holds a finished (S~, S)
  uint64_t* accempty = accf + 2;      // 2: its four warps have read the S~ half out
  uint64_t* sempty = accempty + 2;    // 2: its four warps have read the S half out
  uint64_t* drain = sempty + 2;
  // per [slot][group]: lready — the group's four warps published a pair's maxima and candidate
  // masks in the slot; lfree — the group's scorer has read them (the slot may be rewritten)
  uint64_t* lready = drain + 1;            // 2 * kDistQB
  uint64_t* lfree = lready + 2 * kDistQB;  // 2 * kDistQB
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lfree + 2 * kDistQB);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  // 16-byte aligned from here (the barriers end on an 8-byte boundary; the slot and flag fill it):
  // the scorer reads a group's four chunk flags as one uint4
  uint32_t* cflag = reinterpret_cast<uint32_t*>(
      (reinterpret_cast<uintptr_t>(abort_flag + 1) + 15) & ~uintptr_t(15));  // [slot][group][quarter]: chunks
  float* gmax = reinterpret_cast<float*>(cflag + 2 * kDistQB * 4);         // [slot][group][quarter] max of S~
  float* gtmax = gmax + 2 * kDistQB * 4;                                     // [slot][group][quarter] max of S
  uint32_t* cmask = reinterpret_cast<uint32_t*>(gtmax + 2 * kDistQB * 4);   // kCandWords
  uint8_t* fullb = reinterpret_cast<uint8_t*>(cmask + kCandWords);  // nb: key block J lies inside the grid

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < JS; ++s) {
      mbar_init(kfull + s, 1);
      mbar_init(kempty + s, 2 * kDistQB);  // each group's MMA issuer and scorer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf + b, 1);
      mbar_init(accempty + b, 4);
      mbar_init(sempty + b, 4);
    }
    mbar_init(drain, kDistQB);
    for (int b = 0; b < 2 * kDistQB; ++b) {
      mbar_init(lready + b, 4);
      mbar_init(lfree + b, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int J = tid; J < nb; J += kDistThreads) fullb[J] = block_is_full(a.g, J) ? 1 : 0;
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long head_tiles = ((long long)a.b * a.Hh + h) * nb;
  const int n_pairs = nb * kDistQB;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      mbar_expect_tx(qfull, kDistQB * (C::TILE + C::TB));
      for (int q = 0; q < kDistQB; ++q) {
        const int I = I0 + q < nb ? I0 + q : nb - 1;
        int t0, h0, w0;
        block_origin(a.g, I, t0, h0, w0);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_load_5d(sQ + q * C::TILE + c * 16384, &tmQ, qfull, c * 64, h, w0, h0, t0);
        bulk_load(sqt + q * C::TB, a.qt + (head_tiles + I) * C::TB, C::TB, qfull);
      }
      int issued = 0;
      for (int it = 0; it < nb; ++it) {
        const int s = it % JS, J = key_block(it);
        if (it >= JS && !mbar_wait(kempty + s, ((it / JS) - 1) & 1, a.status, abort_flag)) break;
        int t0, h0, w0;
        block_origin(a.g, J, t0, h0, w0);
        mbar_expect_tx(kfull + s, C::TILE + C::TB);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_load_5d(sK + s * C::TILE + c * 16384, &tmK, kfull + s, c * 64, h, w0, h0, t0);
        bulk_load(skt + s * C::TB, a.kt + (head_tiles + J) * C::TB, C::TB, kfull + s);
        issued = it + 1;
      }
      if (*abort_flag) {  // let copies in flight land before the CTA exits
        wait_plain(qfull, 0);
        for (int it = issued - JS < 0 ? 0 : issued - JS; it < issued; ++it) wait_plain(kfull + it % JS, (it / JS) & 1);
      }
    }
    __syncwarp();
  } else if (warp < kDistEpi) {
    // MMA issuer of group q (whole warp, one elected lane issues): for every key block it
    // issues S = Q_I K_J^T (K = d) into columns [256 q + 128, 256 q + 256) as soon as the
    // group has read the previous S out, then S~ = q~_I k~_J^T (K = r) into [256 q, 256 q +
    // 128) once the previous S~ is read out, and commits the pair.  One issuer per group:
    // a commit covers only its own group's products.
    const int q = warp - kDistMma;
    const uint32_t leader = elect_leader();
    constexpr uint32_t id = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t SBO = (R / 8) * 128;
    const uint64_t dA = smem_desc(smem_u32(sqt), 128, SBO, 0), dB = smem_desc(smem_u32(skt), 128, SBO, 0);
    const uint64_t dQd = smem_desc(smem_u32(sQ), 16, 1024, 2), dKd = smem_desc(smem_u32(sK), 16, 1024, 2);
    const uint32_t tL = tmem + q * 256, tF = tL + 128;
    bool ok = warp_wait(qfull, 0, a.status, abort_flag);
    for (int it = 0; ok && it < nb; ++it) {
      const int s = it % JS;
      if (!(ok = warp_wait(kfull + s, (it / JS) & 1, a.status, abort_flag))) break;
      if (it >= 1 && !(ok = warp_wait(sempty + q, (it - 1) & 1, a.status, abort_flag))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * (16384 >> 4) + (kk & 3) * 2;  // 64-column chunk, 16-column step
        mma_ss_by(leader, tF, dQd + (uint64_t)((q * C::TILE) >> 4) + off, dKd + (uint64_t)((s * C::TILE) >> 4) + off,
                  id, kk > 0);
      }
      if (it >= 1 && !(ok = warp_wait(accempty + q, (it - 1) & 1, a.status, abort_flag))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < R / 16; ++kk)
        mma_ss_by(leader, tL, dA + (uint64_t)((q * C::TB + kk * 256) >> 4), dB + (uint64_t)((s * C::TB + kk * 256) >> 4),
                  id, kk > 0);
      mma_commit_by(leader, accf + q);
      mma_commit_by(leader, kempty + s);
    }
    mma_commit_by(leader, drain);
    wait_plain(drain, 0);
    __syncwarp();
  } else if (warp < kDistScore) {
    // Epilogue group grp (warps kDistEpi + 4 grp .. + 3, one per TMEM lane quarter) handles
    // query block I0 + grp against every key block.  Thread = query row.  Per pair it reads
    // S~ and S out of TMEM, finds the maxima and marks the candidates for the exact maximum,
    // publishes them in slot u & 1 to the group's scorer warp and releases the TMEM pair.
    const int grp = (warp - kDistEpi) >> 2;
    const int quarter = warp & 3;  // a warp reaches TMEM lanes 32 (warp % 4) .. + 31
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t tL = tmem + grp * 256 + lane_base, tF = tL + 128;
    const int I = I0 + grp;
    const bool active = I < nb;
    const bool row_ok = active && block_row_token(a.g, I, row) >= 0;
    const float qn = active ? a.qnorm[head_tiles + I] : 0.f;
    for (int P = grp; P < n_pairs; P += 2) {
      const int u = P >> 1, slot = u & 1, J = key_block(u);
      const int sg = slot * kDistQB + grp;  // this pair's slot of the group
      const float kn = a.knorm[head_tiles + J];  // issued before the waits: its latency overlaps them
      // a failed wait stops all four warps of the group at the same barrier below
      bool okw = warp_wait(accf + grp, u & 1, a.status, abort_flag);
      // the slot's previous pair (u - 2) has been read by the scorer before any of it is rewritten
      if (okw && u >= 2) okw = warp_wait(lfree + sg, ((u >> 1) - 1) & 1, a.status, abort_flag);
      const bool fj = fullb[J] != 0;
      // The row maxima of S~ (mi) and S (ti), over the key rows inside the grid; the
      // reducing TMEM load gives them for full key blocks.
      float mi = -INFINITY, ti = -INFINITY;
      float cmx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // per 32 columns of S~
      if (okw) {
        tc_fence_after();
        // S first: its half of the buffer goes back to the MMA issuer, whose next S product
        // (the long one, K = d) then overlaps the rest of this epilogue
#pragma unroll 1
        for (int cc = 0; cc < 4; cc += 2) {
          uint32_t w0[32], w1[32];
          float x0, x1;
          tmem_ld32_max(tF + cc * 32, w0, x0);
          tmem_ld32_max(tF + cc * 32 + 32, w1, x1);
          tmem_wait_ld();
          if (fj) {
            ti = fmaxf(ti, fmaxf(x0, x1));
          } else {
            ti = fmaxf(ti, masked_max64(block_rows_mask32(a.g, J, cc * 32), block_rows_mask32(a.g, J, cc * 32 + 32),
                                        w0, w1));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sempty + grp);
#pragma unroll
        for (int cc = 0; cc < 4; cc += 2) {
          uint32_t w0[32], w1[32];
          float x0, x1;
          tmem_ld32_max(tL + cc * 32, w0, x0);
          tmem_ld32_max(tL + cc * 32 + 32, w1, x1);
          tmem_wait_ld();
          if (!fj) {
            x0 = masked_max64(block_rows_mask32(a.g, J, cc * 32), 0u, w0, w1);
            x1 = masked_max64(0u, block_rows_mask32(a.g, J, cc * 32 + 32), w0, w1);
          }
          cmx[cc] = x0;
          cmx[cc + 1] = x1;
        }
        mi = fmaxf(fmaxf(cmx[0], cmx[1]), fmaxf(cmx[2], cmx[3]));
      }
      if (!row_ok) {
        mi = -INFINITY;
        ti = -INFINITY;
      }
      float wm = mi, wt = ti;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
        wt = fmaxf(wt, __shfl_xor_sync(0xffffffffu, wt, o));
      }
      if (lane == 0) {
        gmax[sg * 4 + quarter] = wm;
        gtmax[sg * 4 + quarter] = wt;
      }
      if (!named_bar_and(2 + grp, 128, okw)) break;
      const float M = fmaxf(fmaxf(gmax[sg * 4], gmax[sg * 4 + 1]), fmaxf(gmax[sg * 4 + 2], gmax[sg * 4 + 3]));
      // Every fp32 score within twice the rounding bound of the fp32 maximum M is a
      // candidate for the exact maximum.  An r-term dot product accumulated in fp32, with
      // each of at most r additions rounded to nearest or truncated, is off by at most
      // 2 r u ||q~|| ||k~|| (1 + O(u)), u = 2^-24; delta_f rounds (4 r + 4) u ||q~|| ||k~||
      // up and floor_f rounds M - delta_f down, so the entries >= floor_f of the candidate
      // rows (mi >= floor_f) hold every entry that can be the exact maximum.  The tests
      // stay in fp32 (FP64 is slow on this part); only candidates are re-scored.
      const float delta_f = __fmul_ru(__fmul_ru(kBoundCoef, qn), kn);
      const float floor_f = __fsub_rd(M, delta_f);
      const bool cand = row_ok && mi >= floor_f;
      uint32_t chunks = 0;  // the 32-column chunks in which some row of this warp has a candidate
      if (__any_sync(0xffffffffu, cand)) {  // usually one warp of the four: its candidate row's columns, again from TMEM
        uint32_t needm = 0;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) needm |= (cand && cmx[cc] >= floor_f ? 1u : 0u) << cc;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          const bool need = (needm >> cc) & 1u;
          if (!__any_sync(0xffffffffu, need)) continue;
          uint32_t w[32];
          tmem_ld32(tL + cc * 32, w);
          tmem_wait_ld();
          uint32_t cm = 0;
          if (need) {
            uint32_t m4[4] = {0u, 0u, 0u, 0u};  // four independent chains of compares
#pragma unroll
            for (int e = 0; e < 32; ++e) m4[e & 3] |= (__uint_as_float(w[e]) >= floor_f ? 1u : 0u) << e;
            cm = ((m4[0] | m4[1]) | (m4[2] | m4[3])) & (fj ? 0xffffffffu : block_rows_mask32(a.g, J, cc * 32));
          }
          cmask[((sg * 4 + quarter) * 4 + cc) * 32 + lane] = cm;
          if (__any_sync(0xffffffffu, cm != 0u)) chunks |= 1u << cc;
        }
      }
      if (lane == 0) cflag[sg * 4 + quarter] = chunks;
      // the S~ half is read out: the MMA issuer may refill it; the slot goes to the scorer
      tc_fence_before();
      __threadfence_block();  // this lane's masks before the arrive that publishes them
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(accempty + grp);
        mbar_arrive(lready + sg);
      }
    }
  } else {
    // Scorer warps of group grp, one per slot (the group's even or odd pairs): per pair the
    // candidates marked in the slot are re-scored exactly (each by the whole warp), the first
    // exact maximum (i*, j*) gives e = s~(i*, j*) - t, and e k~_j* and e q~_i* are added to
    // G_q[i*] and G_k[j*] and e^2 / 2 to the loss.  The key stage is released after the
    // operands are read.
    const int grp = (warp - kDistScore) >> 1, which = (warp - kDistScore) & 1;
    const int I = I0 + grp;
    const bool active = I < nb;
    const uint8_t* qtile = sqt + grp * C::TB;
    float loss_acc = 0.f, loss_comp = 0.f;  // compensated sum of this scorer's e^2 / 2 (lane 0)
    for (int P = grp + 2 * which; P < n_pairs; P += 4) {
      const int u = P >> 1, slot = u & 1, s = u % JS, J = key_block(u);  // slot == which
      const int sg = slot * kDistQB + grp;
      if (!warp_wait(lready + sg, (u >> 1) & 1, a.status, abort_flag)) break;
      const float T = fmaxf(fmaxf(gtmax[sg * 4], gtmax[sg * 4 + 1]), fmaxf(gtmax[sg * 4 + 2], gtmax[sg * 4 + 3]));
      const uint8_t* ktile = skt + s * C::TB;
      Score2 bv = {-INFINITY, 0.f};  // the same in every lane: exact_score_warp returns one value to all
      int bi = 0x7fffffff, bj = 0x7fffffff;
      // the (quarter, chunk) pairs holding candidates, as one 16-bit set: usually one bit
      const uint4 f4 = *reinterpret_cast<const uint4*>(cflag + sg * 4);
      uint32_t todo = f4.x | (f4.y << 4) | (f4.z << 8) | (f4.w << 12);
      while (todo != 0u) {
        const int qc = __ffs(todo) - 1, qd = qc >> 2, cc = qc & 3;
        todo &= todo - 1u;
        uint32_t cm = cmask[((sg * 4 + qd) * 4 + cc) * 32 + lane];
        for (;;) {  // every candidate of the chunk: lowest lane (row), then lowest column
          const unsigned who = __ballot_sync(0xffffffffu, cm != 0u);
          if (who == 0u) break;
          const int src = __ffs(who) - 1;
          const int e = __ffs(__shfl_sync(0xffffffffu, cm, src)) - 1;
          if (lane == src) cm &= cm - 1u;
          const int crow = qd * 32 + src, j = cc * 32 + e;
          const Score2 v = exact_score_warp<R>(qtile, crow, ktile, j, lane);
          if (better(v, crow, j, bv, bi, bj)) {
            bv = v;
            bi = crow;
            bj = j;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(lfree + sg);  // the slot's maxima and masks are read
      if (active && bi < 128 && bj < 128) {
        const float e = (bv.hi - T) + bv.lo;
        const long long pair = (head_tiles + I) * nb + J;
        if (lane == 0) {
          const float y = 0.5f * e * e - loss_comp;
          const float t1 = loss_acc + y;
          loss_comp = (t1 - loss_acc) - y;
          loss_acc = t1;
          if (a.s_out) a.s_out[pair] = bv.hi;
          if (a.t_out) a.t_out[pair] = T;
        }
        // the operand values leave the stage before it is released; the atomics follow
        // the release (an arrive orders the thread's earlier memory operations before it,
        // and would otherwise wait for these atomics to reach L2)
        float kv[(R + 31) / 32], qv[(R + 31) / 32];
#pragma unroll
        for (int uu = 0; uu < (R + 31) / 32; ++uu) {
          const int c = lane + 32 * uu;
          kv[uu] = c < R ? bf16_at(ktile, bj, c, R) : 0.f;
          qv[uu] = c < R ? bf16_at(qtile, bi, c, R) : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(kempty + s);  // this group no longer reads stage s
        const long long hrow = ((long long)a.b * a.Hh + h) * a.N;
        float* gq = a.Gq + (hrow + block_row_token(a.g, I, bi)) * R;
        float* gk = a.Gk + (hrow + block_row_token(a.g, J, bj)) * R;
#pragma unroll
        for (int uu = 0; uu < (R + 31) / 32; ++uu) {
          const int c = lane + 32 * uu;
          if (c < R) {
            atomicAdd(gq + c, e * kv[uu]);
            atomicAdd(gk + c, e * qv[uu]);
          }
        }
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(kempty + s);
      }
    }
    if (lane == 0 && loss_acc != 0.f) atomicAdd(a.loss, (double)loss_acc - (double)loss_comp);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dW_z[h] = sum over tokens of X_z[token, h, :]^T G_z[h, token, :] with X_0 = Q, G_0 = G_q
// (dWq) and X_1 = K, G_1 = G_k (dWk), over every batch entry.  A CTA sums a run of
// tokens for one (head, z) in registers (each thread owns D R / 256 of the d x r
// outputs) and adds its partial with fp32 atomics.
template <int D, int R>
__global__ void __launch_bounds__(256) dw_kernel(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
                                                 const float* __restrict__ Gq, const float* __restrict__ Gk, int Hh,
                                                 long long N, long long total, int per_cta, float* __restrict__ dWq,
                                                 float* __restrict__ dWk) {
  constexpr int OUT = D * R / 256;
  constexpr int TT = 16;  // tokens staged per step
  __shared__ float xs[TT][D];
  __shared__ float gs[TT][R];
  const int h = blockIdx.y, z = blockIdx.z;
  const __nv_bfloat16* X = z == 0 ? Q : K;
  const float* G = z == 0 ? Gq : Gk;
  float* out = z == 0 ? dWq : dWk;
  float acc[OUT];
#pragma unroll
  for (int u = 0; u < OUT; ++u) acc[u] = 0.f;
  const long long n0 = blockIdx.x * (long long)per_cta;
  const long long n1 = n0 + per_cta < total ? n0 + per_cta : total;
  for (long long base = n0; base < n1; base += TT) {
    __syncthreads();
    for (int e = threadIdx.x; e < TT * D; e += 256) {
      const int t = e / D, c = e % D;
      const long long bn = base + t;  // b * N + n
      xs[t][c] = bn < n1 ? __bfloat162float(X[(bn * Hh + h) * D + c]) : 0.f;
    }
    for (int e = threadIdx.x; e < TT * R; e += 256) {
      const int t = e / R, c = e % R;
      const long long bn = base + t;
      const long long b = bn / N, n = bn % N;
      gs[t][c] = bn < n1 ? G[((b * Hh + h) * N + n) * R + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int t = 0; t < TT; ++t) {
#pragma unroll
      for (int u = 0; u < OUT; ++u) {
        const int o = threadIdx.x + 256 * u;
        acc[u] = fmaf(xs[t][o / R], gs[t][o % R], acc[u]);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < OUT; ++u) {
    const int o = threadIdx.x + 256 * u;
    atomicAdd(out + (long long)h * D * R + o, acc[u]);
  }
}

struct DistWs {
  uint8_t* qt;
  uint8_t* kt;
  float* qnorm;
  float* knorm;
  float* Gq;
  float* Gk;
  size_t bytes;
};

DistWs dist_layout(const Prob& p, void* base) {
  DistWs w;
  const size_t tiles = (size_t)p.B * p.Hh * p.g.nb;
  const size_t tile_bytes = align_up(tiles * 128 * p.r * 2, 256);
  const size_t g_bytes = align_up((size_t)p.B * p.Hh * p.N * p.r * 4, 256);
  char* c = static_cast<char*>(base);
  w.qt = reinterpret_cast<uint8_t*>(c);
  w.kt = reinterpret_cast<uint8_t*>(c + tile_bytes);
  size_t off = 2 * tile_bytes;
  w.qnorm = reinterpret_cast<float*>(c + off);
  off += align_up(tiles * 4, 256);
  w.knorm = reinterpret_cast<float*>(c + off);
  off += align_up(tiles * 4, 256);
  w.Gq = reinterpret_cast<float*>(c + off);
  off += g_bytes;
  w.Gk = reinterpret_cast<float*>(c + off);
  off += g_bytes;
  w.bytes = off;
  return w;
}

template <int R, int D>
cudaError_t launch_distill(const Prob& p, const void* Q, const void* K, float* dWq, float* dWk, double* loss,
                           float* s_out, float* t_out, const DistWs& w, unsigned* status, cudaStream_t st) {
  using C = DistCfg<R, D>;
  const size_t tiles = (size_t)p.B * p.Hh * p.g.nb;
  const int nt_blocks = (int)((tiles * 32 + 255) / 256);
  tile_norm_kernel<R><<<nt_blocks, 256, 0, st>>>(w.qt, (long long)tiles, w.qnorm);
  tile_norm_kernel<R><<<nt_blocks, 256, 0, st>>>(w.kt, (long long)tiles, w.knorm);
  note_launches(2);
  // tiles, the barriers (qfull, 2 JS ring, 2 accf, 2 accempty, 2 sempty, drain, 4 kDistQB slot barriers),
  // the TMEM slot and abort flag (with the padding to 16 bytes), the chunk flags and maxima
  // (3 x [2][kDistQB][4] words), the candidate masks, fullb
  const size_t smem = 1024 + C::TILES_BYTES + 8 * (1 + 2 * C::JS + 7 + 4 * kDistQB) + 16 + 3 * 2 * kDistQB * 4 * 4 +
                      (size_t)kCandWords * 4 + (size_t)p.g.nb + 64;
  cudaError_t e = cudaFuncSetAttribute(distill_kernel<R, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const size_t per_batch = (size_t)p.N * p.Hh * p.d * 2;
  const Geom& g = p.g;
  for (int b = 0; b < p.B; ++b) {
    CUtensorMap mQ, mK;
    if (!make_token_map(&mQ, static_cast<const char*>(Q) + b * per_batch, kTokBF16, g.T, g.H, g.W, p.Hh, p.d, g.bt,
                        g.bh, g.bw) ||
        !make_token_map(&mK, static_cast<const char*>(K) + b * per_batch, kTokBF16, g.T, g.H, g.W, p.Hh, p.d, g.bt,
                        g.bh, g.bw))
      return cudaErrorInvalidValue;
    DistArgs a;
    a.g = g;
    a.Hh = p.Hh;
    a.b = b;
    a.N = p.N;
    a.qt = w.qt;
    a.kt = w.kt;
    a.qnorm = w.qnorm;
    a.knorm = w.knorm;
    a.Gq = w.Gq;
    a.Gk = w.Gk;
    a.loss = loss;
    a.s_out = s_out;
    a.t_out = t_out;
    a.status = status;
    distill_kernel<R, D><<<dim3((g.nb + kDistQB - 1) / kDistQB, p.Hh), kDistThreads, smem, st>>>(mQ, mK, a);
    note_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const long long total = (long long)p.B * p.N;
  const int per_cta = 2048;
  dw_kernel<D, R><<<dim3((unsigned)((total + per_cta - 1) / per_cta), p.Hh, 2), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K), w.Gq, w.Gk, p.Hh, p.N, total, per_cta,
      dWq, dWk);
  note_launches(1);
  return cudaGetLastError();
}

template <int R>
cudaError_t dispatch_d(const Prob& p, const void* Q, const void* K, float* dWq, float* dWk, double* loss,
                       float* s_out, float* t_out, const DistWs& w, unsigned* status, cudaStream_t st) {
  return p.d == 64 ? launch_distill<R, 64>(p, Q, K, dWq, dWk, loss, s_out, t_out, w, status, st)
                   : launch_distill<R, 128>(p, Q, K, dWq, dWk, loss, s_out, t_out, w, status, st);
}

}  // namespace

size_t distill_ws_tc(const Prob& p) { return dist_layout(p, nullptr).bytes; }

cudaError_t distill_tc(const Prob& p, const void* Q, const void* K, const void* Wq, const void* Wk, float* dWq,
                       float* dWk, double* loss, float* s_out, float* t_out, void* ws, cudaStream_t st) {
  const DistWs w = dist_layout(p, ws);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  cudaError_t e = project_tc(p, Q, K, Wq, Wk, ws, st);  // q~, k~ tiles at the start of ws
  if (e != cudaSuccess) return e;
  const size_t g_bytes = (size_t)p.B * p.Hh * p.N * p.r * 4;
  const size_t w_bytes = (size_t)p.Hh * p.d * p.r * 4;
  if ((e = cudaMemsetAsync(w.Gq, 0, g_bytes, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(w.Gk, 0, g_bytes, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dWq, 0, w_bytes, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dWk, 0, w_bytes, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(loss, 0, sizeof(double), st)) != cudaSuccess) return e;
  switch (p.r) {
    case 16:
      return dispatch_d<16>(p, Q, K, dWq, dWk, loss, s_out, t_out, w, status, st);
    case 32:
      return dispatch_d<32>(p, Q, K, dWq, dWk, loss, s_out, t_out, w, status, st);
    case 48:
      return dispatch_d<48>(p, Q, K, dWq, dWk, loss, s_out, t_out, w, status, st);
    case 64:
      return dispatch_d<64>(p, Q, K, dWq, dWk, loss, s_out, t_out, w, status, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sda
