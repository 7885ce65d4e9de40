// Block-sparse flash-attention backward on the 5th-generation tensor cores.
//
// Gradients of the forward of "DSV: Exploiting Dynamic Sparsity to Accelerate
// Large-Scale Video DiT Training" (section 4, stage 2: compute only on the kept
// blocks) with the block map held fixed: with P = exp(scale Q K^T - LSE) on the
// kept blocks and D_i = dO_i . O_i,
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Deterministic, no atomics on gradient values.  Every MMA of the backward
// takes fp16 operands: prepare writes fp16 copies of Q, K, V and dO (exact for
// bf16 values inside fp16's normal range), so that P and dS can be rounded to
// fp16 (8x finer than bf16) for the products that consume them — one MMA
// needs A and B of the same type.  Phases, in stream order:
//   prepare   block-map transpose (for every key block, the query blocks that
//             kept it, ascending; key blocks visited longest list first),
//             D~_i = dO_i . O_i from the stored O and LSE_i * log2(e), both in
//             tile order (+inf LSE for rows outside the grid, so their P is 0),
//             and the fp16 copies.
//   dq        per query block: S = Q K_J^T and dP = dO V_J^T (M=128, N=128,
//             K=d), then dQ with the exact-D correction (see dq_kernel); it also
//             writes the exact D_i for the next phase.
//   dkdv      per key block: S^T = K Q_I^T and dP^T = V dO_I^T, P^T and dS^T in
//             TMEM, dV += P^T dO_I, dK += dS^T Q_I.  For d = 128 the four
//             128-column accumulators fill all 512 TMEM columns.
// The dq kernel repeats the S and dP products of the dK/dV kernel in exchange
// for no fp32 dQ reduction buffer.
#include "internal.h"

namespace sda {

namespace {

constexpr int kThreads = 384;  // warp 0 TMA, warp 1 MMA, warp 2 arrival helper, warps 4-11 compute
constexpr float kLog2e = 1.4426950408889634f;

struct BwdArgs {
  Geom g;
  int Hh, k, b;
  int all_full;  // every tile lies inside the grid (no clipped edge tiles)
  long long N;
  float scale_log2;  // softmax scale * log2(e)
  float scale;
  const int32_t* idx;     // [B, Hh, nb, k]
  float* Dv;              // [B, Hh, nb, 128]: D~ after prepare, exact D after dq
  const float* L2v;       // [B, Hh, nb, 128]
  const int32_t* offsets; // [B, Hh, nb + 1]
  const int32_t* lists;   // [B, Hh, nb * k]
  const int32_t* order;   // [B, Hh, nb]
  // A partition state's backward: each query block's kept blocks inside the key range
  // (none for an inactive block), compacted, and dL/dLSE in tile order; null otherwise.
  const int32_t* qlist;   // [B, Hh, nb, k]
  const int32_t* qcount;  // [B, Hh, nb]
  const float* G;         // [B, Hh, nb, 128]
  unsigned* status;
  // dK/dV half tiles: query rows [0,64) and [64,128) of a tile are the two halves of
  // its slowest even extent (0: tt, 1: hh, 2: ww); the second half starts hoff further.
  int hdim, hoff;
};

__device__ __forceinline__ bool wait_plain(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > SDA_WAIT_LIMIT_NS) return false;
  return true;
}

// ------------------------------------------------------------------ preprocess
// D~_i = dO_i . O_i - dLSE_i (dLSE of a partition state's backward, else 0) and
// LSE_i log2(e) in tile order; G receives dLSE_i in tile order when given.  O is the
// stored bf16 output, or (kO32) the training forward's fp32 copy of it.
template <int D, bool kO32>
__global__ void __launch_bounds__(128) pre_kernel(Geom g, int Hh, long long N, int b, const void* __restrict__ O,
                                                  const __nv_bfloat16* __restrict__ dO, const float* __restrict__ LSE,
                                                  const float* __restrict__ dLSE, float* __restrict__ Dv,
                                                  float* __restrict__ L2v, float* __restrict__ G) {
  const int I = blockIdx.x, h = blockIdx.y, r = threadIdx.x;
  const int n = block_row_token(g, I, r);
  float dsum = 0.f, l2 = INFINITY, gl = 0.f;
  if (n >= 0) {
    const long long row = ((long long)b * N + n) * Hh + h;
    const uint4* go = reinterpret_cast<const uint4*>(dO + row * D);
#pragma unroll 4
    for (int v = 0; v < D / 8; ++v) {
      const uint4 c = go[v];
      const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
      float ov[8];
      if (kO32) {
        const float4* o = reinterpret_cast<const float4*>(static_cast<const float*>(O) + row * D) + 2 * v;
        const float4 a0 = o[0], a1 = o[1];
        ov[0] = a0.x, ov[1] = a0.y, ov[2] = a0.z, ov[3] = a0.w, ov[4] = a1.x, ov[5] = a1.y, ov[6] = a1.z,
        ov[7] = a1.w;
      } else {
        const uint4 a = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(O) + row * D)[v];
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          ov[2 * q] = __uint_as_float(aw[q] << 16);
          ov[2 * q + 1] = __uint_as_float(aw[q] & 0xFFFF0000u);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dsum = fmaf(ov[2 * q], __uint_as_float(cw[q] << 16), dsum);
        dsum = fmaf(ov[2 * q + 1], __uint_as_float(cw[q] & 0xFFFF0000u), dsum);
      }
    }
    const float lse = LSE[((long long)b * Hh + h) * N + n];
    l2 = lse == -INFINITY ? INFINITY : lse * kLog2e;
    if (dLSE) gl = dLSE[((long long)b * Hh + h) * N + n];
  }
  const long long o = (((long long)b * Hh + h) * g.nb + I) * 128 + r;
  Dv[o] = dsum - gl;
  L2v[o] = l2;
  if (G) G[o] = gl;
}

// bf16 -> fp16, 8 elements per thread-iteration.  A value outside fp16's finite
// range becomes inf (or stays NaN); the thread then latches kStatusRange once.
__global__ void half_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n8,
                            unsigned* __restrict__ status) {
  uint32_t bad = 0;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      o[q] = pack_f16(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xFFFF0000u));
      // an all-ones fp16 exponent field: inf or NaN
      bad |= ((o[q] & 0x7C00u) == 0x7C00u) | ((o[q] & 0x7C000000u) == 0x7C000000u);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (bad) atomicOr(status, kStatusRange);
}

// ------------------------------------------------------------------ block-map transpose
// bitmap[bh, I, J] = query block I kept key block J (for a partition state: J in
// [kb_begin, kb_end) and I active).
__global__ void csr_bitmap_kernel(const int32_t* __restrict__ idx, long long entries, int nb, int k, int words,
                                  int kb_begin, int kb_end, const uint8_t* __restrict__ qb_active,
                                  unsigned* __restrict__ bitmap, unsigned* __restrict__ status) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < entries;
       e += (long long)gridDim.x * blockDim.x) {
    const long long row = e / k;  // (bh, I)
    const int J = idx[e];
    if (J < 0 || J >= nb) {
      atomicOr(status, kStatusBadIndex);
      continue;
    }
    if (J < kb_begin || J >= kb_end || (qb_active && !qb_active[row % nb])) continue;
    if (atomicOr(bitmap + row * words + (J >> 5), 1u << (J & 31)) & (1u << (J & 31)))
      atomicOr(status, kStatusBadIndex);  // the same block twice in one row
  }
}

// A partition state's dQ rows: each query block's kept blocks inside [kb_begin,
// kb_end), in list order, and their count (0 for an inactive block).
__global__ void rowlist_kernel(const int32_t* __restrict__ idx, long long rows, int nb, int k, int kb_begin,
                               int kb_end, const uint8_t* __restrict__ qb_active, int32_t* __restrict__ qlist,
                               int32_t* __restrict__ qcount) {
  for (long long row = blockIdx.x * (long long)blockDim.x + threadIdx.x; row < rows;
       row += (long long)gridDim.x * blockDim.x) {
    int c = 0;
    if (!qb_active || qb_active[row % nb])
      for (int s = 0; s < k; ++s) {
        const int J = idx[row * k + s];
        if (J >= kb_begin && J < kb_end) qlist[row * k + c++] = J;
      }
    qcount[row] = c;
  }
}

// counts[bh, J] = number of query blocks that kept J.  One warp per (bh, J): lane i
// reads row I0 + i of the bitmap column, the warp counts with a ballot.
__global__ void csr_count_kernel(const unsigned* __restrict__ bitmap, int nb, int words, long long total,
                                 int32_t* __restrict__ counts) {
  const long long t = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= total) return;  // whole warps: t is the same on every lane
  const long long bh = t / nb;
  const int J = (int)(t % nb);
  const unsigned* col = bitmap + bh * nb * words + (J >> 5);
  const unsigned bit = 1u << (J & 31);
  int c = 0;
  for (int I0 = 0; I0 < nb; I0 += 32) {
    const int I = I0 + lane;
    c += __popc(__ballot_sync(0xffffffffu, I < nb && (col[(long long)I * words] & bit)));
  }
  if (lane == 0) counts[t] = c;
}

// Per (batch, head): exclusive scan of counts -> offsets.
__global__ void __launch_bounds__(1024) csr_scan_kernel(const int32_t* __restrict__ counts, int nb,
                                                        int32_t* __restrict__ offsets) {
  extern __shared__ int32_t cs[];  // nb
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  const long long bh = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int J = tid; J < nb; J += blockDim.x) cs[J] = counts[bh * nb + J];
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < nb; base += blockDim.x) {
    const int J = base + tid;
    int v = J < nb ? cs[J] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int before = carry;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    if (J < nb) offsets[bh * (nb + 1) + J] = before + x - v;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += warp_tot[w];
      carry += tot;
    }
    __syncthreads();
  }
  if (tid == 0) offsets[bh * (nb + 1) + nb] = carry;
}

// The visiting order of key blocks: descending count, ties by ascending J (the rank
// of J counts the blocks before it).  Grid (chunks of 256 key blocks, B * heads).
__global__ void __launch_bounds__(256) csr_order_kernel(const int32_t* __restrict__ counts, int nb,
                                                        int32_t* __restrict__ order) {
  extern __shared__ int32_t cs[];  // nb
  const long long bh = blockIdx.y;
  for (int J = threadIdx.x; J < nb; J += blockDim.x) cs[J] = counts[bh * nb + J];
  __syncthreads();
  const int J = blockIdx.x * blockDim.x + threadIdx.x;
  if (J >= nb) return;
  const int c = cs[J];
  int rank = 0;
  for (int J2 = 0; J2 < nb; ++J2) {
    const int c2 = cs[J2];
    rank += (c2 > c) || (c2 == c && J2 < J);
  }
  order[bh * nb + rank] = J;
}

// lists: for each key block J, the query blocks that kept it, ascending.  One warp
// per (bh, J); each 32-row step's hits are written contiguously.
__global__ void csr_fill_kernel(const unsigned* __restrict__ bitmap, const int32_t* __restrict__ offsets, int nb,
                                int k, int words, long long total, int32_t* __restrict__ lists) {
  const long long t = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= total) return;  // whole warps
  const long long bh = t / nb;
  const int J = (int)(t % nb);
  const unsigned* col = bitmap + bh * nb * words + (J >> 5);
  const unsigned bit = 1u << (J & 31);
  int pos = offsets[bh * (nb + 1) + J];
  int32_t* out = lists + bh * nb * k;
  for (int I0 = 0; I0 < nb; I0 += 32) {
    const int I = I0 + lane;
    const bool hit = I < nb && (col[(long long)I * words] & bit);
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (hit) out[pos + __popc(m & ((1u << lane) - 1u))] = I;
    pos += __popc(m);
  }
}

// ------------------------------------------------------------------ shared pieces
// The two compute warpgroups each own 64 of the 128 columns of an S / dP tile
// and write their packed bf16 results (P, dS) into the first half of their own
// column range, never into columns the other group may still be reading.
// TMEM column of the K-step `kk` (16 elements = 8 packed columns) of such an operand:
__device__ __forceinline__ uint32_t packed_col(int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); }

template <int D>
struct Cfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE = 128 * D * 2;
  static constexpr int ST = D == 128 ? 2 : 4;   // dK/dV: Q + dO stages
  static constexpr int KST = D == 128 ? 3 : 4;  // dQ: K ring (K is read until the block's dQ MMAs)
  static constexpr int VST = D == 128 ? 2 : 4;  // dQ: V ring (V is read by dP only)
};

// Store this thread's row of a 128 x D accumulator, columns [c_lo, c_lo + ncols),
// as mul * (a + coef * b) (b only when tb != 0) into a 128B-swizzled staging
// area laid out as TMA boxes of 128 bytes of the row (bf16: 64 columns per
// box, fp32: 32 columns per box).  zero writes zeros.
template <bool F32>
__device__ __forceinline__ void stage_row(uint8_t* stage, uint32_t ta, uint32_t tb, float coef, int row, int c_lo,
                                          int ncols, float mul, bool zero) {
  for (int c0 = c_lo; c0 < c_lo + ncols; c0 += 32) {
    float f[32];
    if (!zero) {
      uint32_t u[32];
      tmem_ld32(ta + c0, u);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(u[e]);
      if (tb) {
        tmem_ld32(tb + c0, u);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = fmaf(coef, __uint_as_float(u[e]), f[e]);
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) f[e] *= mul;
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) f[e] = 0.f;
    }
    if (F32) {
      uint8_t* box = stage + (c0 >> 5) * 16384;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(box + sw128_offset(row, q)) =
            make_uint4(__float_as_uint(f[4 * q]), __float_as_uint(f[4 * q + 1]), __float_as_uint(f[4 * q + 2]),
                       __float_as_uint(f[4 * q + 3]));
    } else {
      uint8_t* box = stage + (c0 >> 6) * 16384;
      const int cbase = ((c0 & 63) >> 3);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(box + sw128_offset(row, cbase + q)) =
            make_uint4(pack_bf16(f[8 * q], f[8 * q + 1]), pack_bf16(f[8 * q + 2], f[8 * q + 3]),
                       pack_bf16(f[8 * q + 4], f[8 * q + 5]), pack_bf16(f[8 * q + 6], f[8 * q + 7]));
    }
  }
}

// ------------------------------------------------------------------ dQ
// D_i has to be known before dS can be formed, but the D~_i that prepare
// derives from the stored bf16 O carries that output's rounding.  This kernel
// therefore uses D~ for dS~ = P o (dP - D~), accumulates the exact
// D_i = sum_j P_ij dP_ij in fp32 over the same pass, and corrects at the end:
//   dQ_i = scale * ( sum_j dS~_ij k_j + (D~_i - D_i) sum_j P_ij k_j ),
// which equals scale * sum_j P_ij (dP_ij - D_i) k_j.  The exact D is written
// back for the dK/dV kernel.  TMEM: S [0,128), dP [128,256), dQ~ [256,256+D),
// P K [256+D, 256+2D).
template <int D, bool F32OUT>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const __grid_constant__ CUtensorMap tmdQ, BwdArgs a) {
  using C = Cfg<D>;
  constexpr int KST = C::KST, VST = C::VST;
  const int I = blockIdx.x, h = blockIdx.y;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + C::TILE;
  uint8_t* sK = sdO + C::TILE;        // KST tiles
  uint8_t* sV = sK + KST * C::TILE;   // VST tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + VST * C::TILE);
  uint64_t* qfull = bars;
  uint64_t* kvfull = qfull + 1;       // KST: K_j and V_j of block j landed (index j mod KST)
  uint64_t* kempty = kvfull + KST;    // KST
  uint64_t* vempty = kempty + KST;    // VST
  uint64_t* sdpfull = vempty + VST;   // 2: S/dP columns of half h are ready
  uint64_t* dsfull = sdpfull + 2;     // 2: packed dS~ / P of half h are written
  uint64_t* drain = dsfull + 2;       // 1
  float* dpart = reinterpret_cast<float*>(drain + 1);  // 2 x 128 partial row sums of P dP
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dpart + 256);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long qrow = ((long long)a.b * a.Hh + h) * a.g.nb + I;
  const int32_t* sel = (a.qlist ? a.qlist : a.idx) + qrow * a.k;
  const int n = a.qcount ? a.qcount[qrow] : a.k;  // 0 only for a partition state's empty rows
  if (tid == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(kvfull + s, 1);
      mbar_init(kempty + s, 1);
    }
    for (int s = 0; s < VST; ++s) mbar_init(vempty + s, 1);
    for (int hh = 0; hh < 2; ++hh) {
      mbar_init(sdpfull + hh, 1);
      mbar_init(dsfull + hh, hh == 0 ? 128 + 1 : 128);  // + warp 2: K/V of the next block landed
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256, tPK = tmem + 256 + D;
  int t0, h0, w0;
  block_origin(a.g, I, t0, h0, w0);

  if (warp == 0) {
    if (lane == 0 && n > 0) {  // with no block nothing is loaded: the epilogue reuses sQ at once
      mbar_expect_tx(qfull, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_5d(sQ + c * 16384, &tmQ, qfull, c * 64, h, w0, h0, t0);
        tma_load_5d(sdO + c * 16384, &tmdO, qfull, c * 64, h, w0, h0, t0);
      }
      int issued = 0;
      int Jn = sel[0];  // block index read one iteration ahead of its use
      for (int j = 0; j < n; ++j) {
        const int sk = j % KST, sv = j % VST;
        const int Jc = Jn;
        if (j + 1 < n) Jn = sel[j + 1];
        if (j >= KST && !mbar_wait(kempty + sk, ((j / KST) - 1) & 1, a.status, abort_flag)) break;
        if (j >= VST && !mbar_wait(vempty + sv, ((j / VST) - 1) & 1, a.status, abort_flag)) break;
        int jt0, jh0, jw0;
        block_origin(a.g, Jc, jt0, jh0, jw0);
        mbar_expect_tx(kvfull + sk, 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_5d(sK + sk * C::TILE + c * 16384, &tmK, kvfull + sk, c * 64, h, jw0, jh0, jt0);
          tma_load_5d(sV + sv * C::TILE + c * 16384, &tmV, kvfull + sk, c * 64, h, jw0, jh0, jt0);
        }
        issued = j + 1;
      }
      if (*abort_flag) {
        wait_plain(qfull, 0);
        for (int j = issued - KST < 0 ? 0 : issued - KST; j < issued; ++j) wait_plain(kvfull + j % KST, (j / KST) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // Arrive on dsfull[0] of block j once K/V of block j + 1 have landed, so the MMA
    // warp's wait for block j's first dS half also covers the next block's tiles.
    if (lane == 0) {
      for (int j = 0; j < n; ++j) {
        const int t = j + 1;
        if (t < n && !mbar_wait(kvfull + t % KST, (t / KST) & 1, a.status, abort_flag)) break;
        // phase j - 1 completes before this arrival for phase j
        if (j >= 1 && !mbar_wait(dsfull, (j - 1) & 1, a.status, abort_flag)) break;
        mbar_arrive(dsfull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // Half-tile ping-pong: S/dP are produced and consumed in two column halves
    // (keys [0,64) and [64,128) of the block), one per compute warpgroup, so the
    // tensor pipe works on one half while a warpgroup works on the other.  Whole
    // warp, one elected lane issues; descriptors advance by adding to the
    // start-address field (16-byte units).
    const uint32_t leader = elect_leader();
    constexpr uint32_t idS = idesc_f16(128, 64, 0, 0);  // Q K^T and dO V^T, one 64-key half
    constexpr uint32_t idQ = idesc_f16(128, D, 0, 1);   // dS~ K and P K
    const uint64_t dQk = smem_desc(smem_u32(sQ), 16, 1024, 2), ddOk = smem_desc(smem_u32(sdO), 16, 1024, 2);
    const uint64_t dKk = smem_desc(smem_u32(sK), 16, 1024, 2), dVk = smem_desc(smem_u32(sV), 16, 1024, 2);
    const uint64_t dKm = smem_desc(smem_u32(sK), 16384, 1024, 2);  // K as the MN-major B of dS~ K
    auto issue_sdp = [&](int j, int hh) {
      const uint32_t sko = (uint32_t)(((j % KST) * C::TILE + hh * 8192) >> 4);
      const uint32_t svo = (uint32_t)(((j % VST) * C::TILE + hh * 8192) >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * (16384 >> 4) + (kk & 3) * 2;
        mma_ss_by(leader, tS + hh * 64, dQk + off, dKk + sko + off, idS, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * (16384 >> 4) + (kk & 3) * 2;
        mma_ss_by(leader, tdP + hh * 64, ddOk + off, dVk + svo + off, idS, kk > 0);
      }
      mma_commit_by(leader, sdpfull + hh);
      if (hh == 1) mma_commit_by(leader, vempty + j % VST);  // V_j is read by dP only
    };
    auto issue_dq = [&](int j, int hh) {
      const uint64_t bK0 = dKm + (uint64_t)(((j % KST) * C::TILE) >> 4);
      // four MMAs into one accumulator, then four into the other (alternating
      // accumulators issues measurably slower than a run into one)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = hh * 4 + q;
        mma_ts_by(leader, tdQ, tS + packed_col(kk), bK0 + (uint64_t)(kk * (2048 >> 4)), idQ, (j > 0 || kk > 0));
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = hh * 4 + q;
        mma_ts_by(leader, tPK, tdP + packed_col(kk), bK0 + (uint64_t)(kk * (2048 >> 4)), idQ, (j > 0 || kk > 0));
      }
    };
    bool ok = n > 0 && warp_wait(qfull, 0, a.status, abort_flag) && warp_wait(kvfull, 0, a.status, abort_flag);
    if (ok) {
      tc_fence_after();
      issue_sdp(0, 0);
      issue_sdp(0, 1);
    }
    for (int j = 0; ok && j < n; ++j) {
      const bool more = j + 1 < n;
      if (!(ok = warp_wait(dsfull, j & 1, a.status, abort_flag))) break;
      tc_fence_after();
      issue_dq(j, 0);
      // dsfull[0] of block j also means K/V_{j+1} landed (warp 2 arrives on it)
      if (more) issue_sdp(j + 1, 0);
      if (!(ok = warp_wait(dsfull + 1, j & 1, a.status, abort_flag))) break;
      tc_fence_after();
      issue_dq(j, 1);
      mma_commit_by(leader, kempty + j % KST);  // K_j: last read by this block's dQ MMAs
      if (more) issue_sdp(j + 1, 1);
    }
    if (n > 0) {  // no MMA was issued for an empty row: nothing to drain
      mma_commit_by(leader, drain);
      wait_plain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int grp = (warp - 4) >> 2;                 // key columns [64 grp, 64 grp + 64)
    const int row = (warp & 3) * 32 + lane;          // query row = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const long long tile_row = (((long long)a.b * a.Hh + h) * a.g.nb + I) * 128 + row;
    const float l2 = a.L2v[tile_row];
    const float Dt = a.Dv[tile_row];  // D~ from the stored O
    float dsum0 = 0.f, dsum1 = 0.f;   // this group's share of D = sum_j P_ij dP_ij
    for (int j = 0; j < n; ++j) {
      if (!warp_wait(sdpfull + grp, j & 1, a.status, abort_flag)) break;
      tc_fence_after();
      const int J = a.all_full ? 0 : sel[j];
      const bool full = a.all_full || block_is_full(a.g, J);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = grp * 64 + cc * 32;
        uint32_t us[32], up[32];
        tmem_ld32(tS + lane_base + col0, us);
        tmem_ld32(tdP + lane_base + col0, up);
        tmem_wait_ld();
        uint32_t pds[16], pp[16];
        const uint32_t vm = full ? 0xffffffffu : block_rows_mask32(a.g, J, col0);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float p0 = ex2(fmaf(__uint_as_float(us[2 * e]), a.scale_log2, -l2));
          float p1 = ex2(fmaf(__uint_as_float(us[2 * e + 1]), a.scale_log2, -l2));
          if (!((vm >> (2 * e)) & 1u)) p0 = 0.f;
          if (!((vm >> (2 * e + 1)) & 1u)) p1 = 0.f;
          const float dp0 = __uint_as_float(up[2 * e]), dp1 = __uint_as_float(up[2 * e + 1]);
          dsum0 = fmaf(p0, dp0, dsum0);
          dsum1 = fmaf(p1, dp1, dsum1);
          pds[e] = pack_f16(p0 * (dp0 - Dt), p1 * (dp1 - Dt));
          pp[e] = pack_f16(p0, p1);
        }
        tmem_st16(tS + lane_base + grp * 64 + cc * 16, pds);
        tmem_st16(tdP + lane_base + grp * 64 + cc * 16, pp);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(dsfull + grp);
    }
    dpart[grp * 128 + row] = dsum0 + dsum1;
    if (n > 0) mbar_wait(drain, 0, a.status, abort_flag);
    tc_fence_after();
    named_bar(1, 256);
    // exact D; a partition state's LSE gradient enters it as D - dLSE, as in D~
    const float Dx = dpart[row] + dpart[128 + row] - (a.G ? a.G[tile_row] : 0.f);
    if (grp == 0) a.Dv[tile_row] = Dx;  // exact D for the dK/dV kernel
    // dQ = scale * (dQ~ + (D~ - D) P K) -> staging (Q and dO tiles are free once all MMAs are done)
    stage_row<F32OUT>(sQ, tdQ + lane_base, tPK + lane_base, Dt - Dx, row, grp * (D / 2), D / 2, a.scale, n == 0);
    fence_async_smem();
    named_bar(1, 256);
    if (tid == 128) {
      constexpr int boxes = F32OUT ? D / 32 : D / 64;
      constexpr int per = F32OUT ? 32 : 64;
#pragma unroll
      for (int c = 0; c < boxes; ++c) tma_store_5d(&tmdQ, sQ + c * 16384, c * per, h, w0, h0, t0);
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

// ------------------------------------------------------------------ dQ with the exact D (training pair)
// After the training forward, which kept O in fp32 with P rounded to fp16, D_i = dO_i . O_i
// (prepare) is exact to well within the tolerance, so dS = P o (dP - D) needs no correction
// and each block takes three products (S, dP, dQ) instead of four.  Q and dO are copied into
// TMEM once and serve as the A operand of S = Q K^T and dP = dO V^T: those 64-key half
// products then read only their B tile from shared memory and run at the tensor pipe's
// full rate.  TMEM: S [0,128), dP [128,256), dQ [256,256+D), Q [256+D,256+3D/2),
// dO [256+3D/2,256+2D) (A-operand layout: row = lane, elements 2c and 2c+1 in column c).
// dS = P (dP - D) for 32 key columns of one query row, P = exp2(S scale log2(e) - LSE log2(e)),
// packed to fp16 pairs; with kMask the keys outside the grid (clear bits of vm) get P = 0.
template <bool kMask>
__device__ __forceinline__ void ds_pairs(const uint32_t (&us)[32], const uint32_t (&up)[32], uint32_t vm, float2 sc2,
                                         float2 nl2, float2 nD2, uint32_t (&pds)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float2 x2 = ffma2(make_float2(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])), sc2, nl2);
    float p0 = ex2(x2.x), p1 = ex2(x2.y);
    if (kMask) {
      if (!((vm >> (2 * e)) & 1u)) p0 = 0.f;
      if (!((vm >> (2 * e + 1)) & 1u)) p1 = 0.f;
    }
    const float2 d2 = fadd2(make_float2(__uint_as_float(up[2 * e]), __uint_as_float(up[2 * e + 1])), nD2);
    const float2 r2 = fmul2(make_float2(p0, p1), d2);
    pds[e] = pack_f16(r2.x, r2.y);
  }
}

template <int D, bool F32OUT>
__global__ void __launch_bounds__(kThreads, 1)
    dqx_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
               const __grid_constant__ CUtensorMap tmdQ, BwdArgs a) {
  using C = Cfg<D>;
  constexpr int KST = C::KST, VST = C::VST;
  const int I = blockIdx.x, h = blockIdx.y;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + C::TILE;
  uint8_t* sK = sdO + C::TILE;        // KST tiles
  uint8_t* sV = sK + KST * C::TILE;   // VST tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + VST * C::TILE);
  uint64_t* qfull = bars;
  uint64_t* kvfull = qfull + 1;       // KST: K_j and V_j of block j landed (index j mod KST)
  uint64_t* kempty = kvfull + KST;    // KST
  uint64_t* vempty = kempty + KST;    // VST
  uint64_t* sdpfull = vempty + VST;   // 2: S/dP columns of half h are ready
  uint64_t* dsfull = sdpfull + 2;     // 2: packed dS of half h is written
  uint64_t* qtmem = dsfull + 2;       // 1: Q and dO are in TMEM
  uint64_t* drain = qtmem + 1;        // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long qrow = ((long long)a.b * a.Hh + h) * a.g.nb + I;
  const int32_t* sel = a.idx + qrow * a.k;
  const int n = a.k;
  if (tid == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(kvfull + s, 1);
      mbar_init(kempty + s, 1);
    }
    for (int s = 0; s < VST; ++s) mbar_init(vempty + s, 1);
    for (int hh = 0; hh < 2; ++hh) {
      mbar_init(sdpfull + hh, 1);
      mbar_init(dsfull + hh, hh == 0 ? 128 + 1 : 128);  // + warp 2: K/V of the next block landed
    }
    mbar_init(qtmem, 256);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256, tQt = tmem + 256 + D, tdOt = tQt + D / 2;
  int t0, h0, w0;
  block_origin(a.g, I, t0, h0, w0);

  if (warp == 0) {
    if (lane == 0 && n > 0) {
      mbar_expect_tx(qfull, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_5d(sQ + c * 16384, &tmQ, qfull, c * 64, h, w0, h0, t0);
        tma_load_5d(sdO + c * 16384, &tmdO, qfull, c * 64, h, w0, h0, t0);
      }
      int issued = 0;
      int Jn = sel[0];  // block index read one iteration ahead of its use
      for (int j = 0; j < n; ++j) {
        const int sk = j % KST, sv = j % VST;
        const int Jc = Jn;
        if (j + 1 < n) Jn = sel[j + 1];
        if (j >= KST && !mbar_wait(kempty + sk, ((j / KST) - 1) & 1, a.status, abort_flag)) break;
        if (j >= VST && !mbar_wait(vempty + sv, ((j / VST) - 1) & 1, a.status, abort_flag)) break;
        int jt0, jh0, jw0;
        block_origin(a.g, Jc, jt0, jh0, jw0);
        mbar_expect_tx(kvfull + sk, 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_5d(sK + sk * C::TILE + c * 16384, &tmK, kvfull + sk, c * 64, h, jw0, jh0, jt0);
          tma_load_5d(sV + sv * C::TILE + c * 16384, &tmV, kvfull + sk, c * 64, h, jw0, jh0, jt0);
        }
        issued = j + 1;
      }
      if (*abort_flag) {
        wait_plain(qfull, 0);
        for (int j = issued - KST < 0 ? 0 : issued - KST; j < issued; ++j) wait_plain(kvfull + j % KST, (j / KST) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // Arrive on dsfull[0] of block j once K/V of block j + 1 have landed, so the MMA
    // warp's wait for block j's first dS half also covers the next block's tiles.
    if (lane == 0) {
      for (int j = 0; j < n; ++j) {
        const int t = j + 1;
        if (t < n && !mbar_wait(kvfull + t % KST, (t / KST) & 1, a.status, abort_flag)) break;
        if (j >= 1 && !mbar_wait(dsfull, (j - 1) & 1, a.status, abort_flag)) break;
        mbar_arrive(dsfull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // Half-tile ping-pong as in dq_kernel; S and dP take A from TMEM.
    const uint32_t leader = elect_leader();
    constexpr uint32_t idS = idesc_f16(128, 64, 0, 0);  // Q K^T and dO V^T, one 64-key half
    constexpr uint32_t idQ = idesc_f16(128, D, 0, 1);   // dS K
    const uint64_t dKk = smem_desc(smem_u32(sK), 16, 1024, 2), dVk = smem_desc(smem_u32(sV), 16, 1024, 2);
    const uint64_t dKm = smem_desc(smem_u32(sK), 16384, 1024, 2);  // K as the MN-major B of dS K
    auto issue_sdp = [&](int j, int hh) {
      const uint32_t sko = (uint32_t)(((j % KST) * C::TILE + hh * 8192) >> 4);
      const uint32_t svo = (uint32_t)(((j % VST) * C::TILE + hh * 8192) >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * (16384 >> 4) + (kk & 3) * 2;
        mma_ts_by(leader, tS + hh * 64, tQt + kk * 8, dKk + sko + off, idS, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * (16384 >> 4) + (kk & 3) * 2;
        mma_ts_by(leader, tdP + hh * 64, tdOt + kk * 8, dVk + svo + off, idS, kk > 0);
      }
      mma_commit_by(leader, sdpfull + hh);
      if (hh == 1) mma_commit_by(leader, vempty + j % VST);  // V_j is read by dP only
    };
    auto issue_dq = [&](int j, int hh) {
      const uint64_t bK0 = dKm + (uint64_t)(((j % KST) * C::TILE) >> 4);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = hh * 4 + q;
        mma_ts_by(leader, tdQ, tS + packed_col(kk), bK0 + (uint64_t)(kk * (2048 >> 4)), idQ, (j > 0 || kk > 0));
      }
    };
    bool ok = n > 0 && warp_wait(qtmem, 0, a.status, abort_flag) && warp_wait(kvfull, 0, a.status, abort_flag);
    if (ok) {
      tc_fence_after();
      issue_sdp(0, 0);
      issue_sdp(0, 1);
    }
    for (int j = 0; ok && j < n; ++j) {
      const bool more = j + 1 < n;
      if (!(ok = warp_wait(dsfull, j & 1, a.status, abort_flag))) break;
      tc_fence_after();
      issue_dq(j, 0);
      // dsfull[0] of block j also means K/V_{j+1} landed (warp 2 arrives on it)
      if (more) issue_sdp(j + 1, 0);
      if (!(ok = warp_wait(dsfull + 1, j & 1, a.status, abort_flag))) break;
      tc_fence_after();
      issue_dq(j, 1);
      mma_commit_by(leader, kempty + j % KST);  // K_j: last read by this block's dQ MMAs
      if (more) issue_sdp(j + 1, 1);
    }
    if (n > 0) {
      mma_commit_by(leader, drain);
      wait_plain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int grp = (warp - 4) >> 2;                 // key columns [64 grp, 64 grp + 64)
    const int row = (warp & 3) * 32 + lane;          // query row = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // Q (group 0) or dO (group 1) into TMEM: this thread's row, 16-byte vectors of the
    // swizzled tile, 8 fp16 = 4 packed columns each.
    if (n > 0 && warp_wait(qfull, 0, a.status, abort_flag)) {
      const uint8_t* src = grp == 0 ? sQ : sdO;
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t u[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int qq = c0 / 4 + q;  // 16-byte vector of the row
          const uint4 v = *reinterpret_cast<const uint4*>(src + (qq >> 3) * 16384 + sw128_offset(row, qq & 7));
          u[4 * q] = v.x;
          u[4 * q + 1] = v.y;
          u[4 * q + 2] = v.z;
          u[4 * q + 3] = v.w;
        }
        tmem_st32(tQt + grp * (D / 2) + lane_base + c0, u);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(qtmem);
    }
    const long long tile_row = qrow * 128 + row;
    const float l2 = a.L2v[tile_row];
    const float Dx = a.Dv[tile_row];  // exact D (from the fp32 O)
    for (int j = 0; j < n; ++j) {
      if (!warp_wait(sdpfull + grp, j & 1, a.status, abort_flag)) break;
      tc_fence_after();
      const int J = a.all_full ? 0 : sel[j];
      const bool full = a.all_full || block_is_full(a.g, J);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = grp * 64 + cc * 32;
        uint32_t us[32], up[32];
        tmem_ld32(tS + lane_base + col0, us);
        tmem_ld32(tdP + lane_base + col0, up);
        tmem_wait_ld();
        uint32_t pds[16];
        // column pairs through the packed fp32x2 forms: the same roundings as the scalar ones;
        // full key blocks (all but the grid's edge tiles) skip the per-key mask
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nl2 = make_float2(-l2, -l2);
        const float2 nD2 = make_float2(-Dx, -Dx);
        if (full)
          ds_pairs<false>(us, up, 0xffffffffu, sc2, nl2, nD2, pds);
        else
          ds_pairs<true>(us, up, block_rows_mask32(a.g, J, col0), sc2, nl2, nD2, pds);
        tmem_st16(tS + lane_base + grp * 64 + cc * 16, pds);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(dsfull + grp);
    }
    if (n > 0) mbar_wait(drain, 0, a.status, abort_flag);
    tc_fence_after();
    // dQ = scale * dQ~ -> staging (the Q and dO tiles are free: they were copied to TMEM)
    stage_row<F32OUT>(sQ, tdQ + lane_base, 0u, 0.f, row, grp * (D / 2), D / 2, a.scale, n == 0);
    fence_async_smem();
    named_bar(1, 256);
    if (tid == 128) {
      constexpr int boxes = F32OUT ? D / 32 : D / 64;
      constexpr int per = F32OUT ? 32 : 64;
#pragma unroll
      for (int c = 0; c < boxes; ++c) tma_store_5d(&tmdQ, sQ + c * 16384, c * per, h, w0, h0, t0);
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

// ------------------------------------------------------------------ dK, dV
template <int D, bool F32OUT>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV, BwdArgs a) {
  using C = Cfg<D>;
  // The ring holds half stages: for one query block that kept this key block, query
  // rows [64 hh, 64 hh + 64) of Q and dO and of the LSE and D rows.  Half hh is read
  // only by the products of column half hh (S^T, dP^T halves and their dV, dK terms),
  // so it is released as soon as those are done.
  constexpr int HST = 2 * C::ST;        // half-stage slots
  constexpr int HTILE = C::TILE;        // Q half + dO half (64 rows each)
  constexpr int HCHUNK = 64 * 128;      // one 64-column chunk of a 64-row half tile
  const int h = blockIdx.y;
  const long long bh = (long long)a.b * a.Hh + h;
  const int J = a.order[bh * a.g.nb + blockIdx.x];
  const int off0 = a.offsets[bh * (a.g.nb + 1) + J];
  const int n = a.offsets[bh * (a.g.nb + 1) + J + 1] - off0;
  const int32_t* users = a.lists + bh * (long long)a.g.nb * a.k + off0;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::TILE;
  uint8_t* ring = sV + C::TILE;           // HST half tiles (Q half, then dO half)
  uint8_t* rows = ring + HST * HTILE;     // HST x (64 LSE*log2e, 64 D)
  uint64_t* bars = reinterpret_cast<uint64_t*>(rows + HST * 512);
  uint64_t* kvfull = bars;
  uint64_t* qfull = kvfull + 1;      // HST
  uint64_t* qempty = qfull + HST;    // HST
  uint64_t* sdpfull = qempty + HST;  // 2: S^T/dP^T columns of half h are ready
  uint64_t* pdsfull = sdpfull + 2;  // 2: packed P^T / dS^T of half h are written
  uint64_t* drain = pdsfull + 2;    // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(kvfull, 1);
    for (int s = 0; s < HST; ++s) {
      mbar_init(qfull + s, 1);
      mbar_init(qempty + s, 1);
    }
    for (int hh = 0; hh < 2; ++hh) {
      mbar_init(sdpfull + hh, 1);
      mbar_init(pdsfull + hh, 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
  int t0, h0, w0;
  block_origin(a.g, J, t0, h0, w0);

  if (warp == 0) {
    if (lane == 0 && n > 0) {
      mbar_expect_tx(kvfull, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_5d(sK + c * 16384, &tmK, kvfull, c * 64, h, w0, h0, t0);
        tma_load_5d(sV + c * 16384, &tmV, kvfull, c * 64, h, w0, h0, t0);
      }
      int issued = 0;
      for (int i = 0; i < 2 * n; ++i) {  // half stage i: query block users[i / 2], half i % 2
        const int s = i % HST, hh = i & 1;
        if (i >= HST && !mbar_wait(qempty + s, ((i / HST) - 1) & 1, a.status, abort_flag)) break;
        const int I = users[i >> 1];
        int it0, ih0, iw0;
        block_origin(a.g, I, it0, ih0, iw0);
        const int ho = hh * a.hoff;
        it0 += a.hdim == 0 ? ho : 0;
        ih0 += a.hdim == 1 ? ho : 0;
        iw0 += a.hdim == 2 ? ho : 0;
        uint8_t* st = ring + s * HTILE;
        mbar_expect_tx(qfull + s, HTILE + 512);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_5d(st + c * HCHUNK, &tmQ, qfull + s, c * 64, h, iw0, ih0, it0);
          tma_load_5d(st + HTILE / 2 + c * HCHUNK, &tmdO, qfull + s, c * 64, h, iw0, ih0, it0);
        }
        const long long trow = (bh * a.g.nb + I) * 128 + hh * 64;
        bulk_load(rows + s * 512, a.L2v + trow, 256, qfull + s);
        bulk_load(rows + s * 512 + 256, a.Dv + trow, 256, qfull + s);
        issued = i + 1;
      }
      if (*abort_flag) {
        wait_plain(kvfull, 0);
        for (int i = issued - HST < 0 ? 0 : issued - HST; i < issued; ++i) wait_plain(qfull + i % HST, (i / HST) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // Half-tile ping-pong over the query columns [0,64) / [64,128) of S^T and dP^T
    // (one per compute warpgroup), as in dq_kernel; converged-warp issue.
    if (n > 0) {
      const uint32_t leader = elect_leader();
      constexpr uint32_t idS = idesc_f16(128, 64, 0, 0);  // K Q^T and V dO^T, one 64-query half
      constexpr uint32_t idG = idesc_f16(128, D, 0, 1);   // P^T dO and dS^T Q
      const uint64_t dKk = smem_desc(smem_u32(sK), 16, 1024, 2), dVk = smem_desc(smem_u32(sV), 16, 1024, 2);
      const uint64_t dRk = smem_desc(smem_u32(ring), 16, 1024, 2);      // half tiles, K-major
      const uint64_t dRm = smem_desc(smem_u32(ring), HCHUNK, 1024, 2);  // the same as MN-major B
      auto issue_sdp = [&](int u, int hh) {
        const uint32_t sq = (uint32_t)((((2 * u + hh) % HST) * HTILE) >> 4), sd = sq + (uint32_t)((HTILE / 2) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offA = (kk >> 2) * (16384 >> 4) + (kk & 3) * 2;   // K, V: 128-row tiles
          const uint32_t offB = (kk >> 2) * (HCHUNK >> 4) + (kk & 3) * 2;  // 64-row half tiles
          mma_ss_by(leader, tS + hh * 64, dKk + offA, dRk + sq + offB, idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offA = (kk >> 2) * (16384 >> 4) + (kk & 3) * 2;
          const uint32_t offB = (kk >> 2) * (HCHUNK >> 4) + (kk & 3) * 2;
          mma_ss_by(leader, tdP + hh * 64, dVk + offA, dRk + sd + offB, idS, kk > 0);
        }
        mma_commit_by(leader, sdpfull + hh);
      };
      auto issue_grad = [&](int u, int hh) {
        const int s = (2 * u + hh) % HST;
        const uint32_t sq = (uint32_t)((s * HTILE) >> 4), sd = sq + (uint32_t)((HTILE / 2) >> 4);
        // a run into dV, then a run into dK; K-step q covers query rows 64 hh + 16 q ..
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int kk = hh * 4 + q;
          mma_ts_by(leader, tdV, tS + packed_col(kk), dRm + sd + (uint32_t)(q * (2048 >> 4)), idG, (u > 0 || kk > 0));
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int kk = hh * 4 + q;
          mma_ts_by(leader, tdK, tdP + packed_col(kk), dRm + sq + (uint32_t)(q * (2048 >> 4)), idG, (u > 0 || kk > 0));
        }
        mma_commit_by(leader, qempty + s);  // this half stage is no longer read
      };
      auto wait_half = [&](int u, int hh) -> bool {
        const int i = 2 * u + hh;
        return warp_wait(qfull + i % HST, (i / HST) & 1, a.status, abort_flag);
      };
      bool ok = warp_wait(kvfull, 0, a.status, abort_flag) && wait_half(0, 0) && wait_half(0, 1);
      if (ok) {
        tc_fence_after();
        issue_sdp(0, 0);
        issue_sdp(0, 1);
      }
      for (int u = 0; ok && u < n; ++u) {
        const bool more = u + 1 < n;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (!(ok = warp_wait(pdsfull + hh, u & 1, a.status, abort_flag))) break;
          tc_fence_after();
          issue_grad(u, hh);
          if (more) {
            if (!(ok = wait_half(u + 1, hh))) break;
            tc_fence_after();
            issue_sdp(u + 1, hh);
          }
        }
      }
      mma_commit_by(leader, drain);
      wait_plain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int grp = (warp - 4) >> 2;         // query columns [64 grp, 64 grp + 64)
    const int row = (warp & 3) * 32 + lane;  // key row = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool row_ok = block_row_token(a.g, J, row) >= 0;
    for (int u = 0; u < n; ++u) {
      if (!warp_wait(sdpfull + grp, u & 1, a.status, abort_flag)) break;
      tc_fence_after();
      // LSE*log2e and D of this group's 64 query rows, indexed by the column c as l2[c]
      const float* l2 = reinterpret_cast<const float*>(rows + ((2 * u + grp) % HST) * 512) - grp * 64;
      const float* dv = l2 + 64;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = grp * 64 + cc * 32;
        uint32_t us[32], up[32];
        tmem_ld32(tS + lane_base + col0, us);
        tmem_ld32(tdP + lane_base + col0, up);
        tmem_wait_ld();
        uint32_t pp[16], pd[16];
        // column pairs through the packed fp32x2 forms: the same roundings as the scalar ones
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = col0 + 2 * e;
          const float2 x2 = ffma2(make_float2(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])), sc2,
                                  make_float2(-l2[c], -l2[c + 1]));
          float p0 = ex2(x2.x), p1 = ex2(x2.y);
          if (!row_ok) p0 = p1 = 0.f;
          pp[e] = pack_f16(p0, p1);
          const float2 d2 = fadd2(make_float2(__uint_as_float(up[2 * e]), __uint_as_float(up[2 * e + 1])),
                                  make_float2(-dv[c], -dv[c + 1]));
          const float2 r2 = fmul2(make_float2(p0, p1), d2);
          pd[e] = pack_f16(r2.x, r2.y);
        }
        tmem_st16(tS + lane_base + grp * 64 + cc * 16, pp);
        tmem_st16(tdP + lane_base + grp * 64 + cc * 16, pd);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(pdsfull + grp);
    }
    if (n > 0) mbar_wait(drain, 0, a.status, abort_flag);
    tc_fence_after();
    // staging: dK boxes then dV boxes, starting at sK (K, V and the ring are free now)
    constexpr int GB = F32OUT ? 128 * D * 4 : 128 * D * 2;  // bytes of one staged gradient tile
    stage_row<F32OUT>(sK, tdK + lane_base, 0u, 0.f, row, grp * (D / 2), D / 2, a.scale, n == 0);
    stage_row<F32OUT>(sK + GB, tdV + lane_base, 0u, 0.f, row, grp * (D / 2), D / 2, 1.f, n == 0);
    fence_async_smem();
    named_bar(1, 256);
    if (tid == 128) {
      constexpr int boxes = F32OUT ? D / 32 : D / 64;
      constexpr int per = F32OUT ? 32 : 64;
#pragma unroll
      for (int c = 0; c < boxes; ++c) {
        tma_store_5d(&tmdK, sK + c * 16384, c * per, h, w0, h0, t0);
        tma_store_5d(&tmdV, sK + GB + c * 16384, c * per, h, w0, h0, t0);
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

struct WsLayout {
  float* Dv;
  float* L2v;
  int32_t* counts;
  int32_t* offsets;
  int32_t* lists;
  int32_t* order;
  unsigned* bitmap;
  int32_t* qlist;   // partition states only
  int32_t* qcount;
  float* G;
  char* Q16;
  char* K16;
  char* V16;
  char* dO16;
  float* O32;  // the training forward's fp32 O (training workspace only)
  size_t bytes;
};

// train: also the fp32 O of the training forward, placed last so that every other
// region sits at the same offset in both workspaces.
WsLayout ws_layout(const Prob& p, void* base, bool train = false) {
  WsLayout w;
  const size_t bh = (size_t)p.B * p.Hh;
  const size_t nb = p.g.nb;
  const size_t words = (nb + 31) / 32;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align_up(bytes, 256);
    return static_cast<char*>(base) + o;
  };
  w.Dv = reinterpret_cast<float*>(take(bh * nb * 128 * 4));
  w.L2v = reinterpret_cast<float*>(take(bh * nb * 128 * 4));
  w.counts = reinterpret_cast<int32_t*>(take(bh * nb * 4));
  w.offsets = reinterpret_cast<int32_t*>(take(bh * (nb + 1) * 4));
  w.lists = reinterpret_cast<int32_t*>(take(bh * nb * p.k * 4));
  w.order = reinterpret_cast<int32_t*>(take(bh * nb * 4));
  w.bitmap = reinterpret_cast<unsigned*>(take(bh * nb * words * 4));
  w.qlist = reinterpret_cast<int32_t*>(take(bh * nb * p.k * 4));
  w.qcount = reinterpret_cast<int32_t*>(take(bh * nb * 4));
  w.G = reinterpret_cast<float*>(take(bh * nb * 128 * 4));
  w.Q16 = take((size_t)p.B * p.N * p.Hh * p.d * 2);
  w.K16 = take((size_t)p.B * p.N * p.Hh * p.d * 2);
  w.V16 = take((size_t)p.B * p.N * p.Hh * p.d * 2);
  w.dO16 = take((size_t)p.B * p.N * p.Hh * p.d * 2);
  w.O32 = train ? reinterpret_cast<float*>(take((size_t)p.B * p.N * p.Hh * p.d * 4)) : nullptr;
  w.bytes = off;
  return w;
}

BwdArgs make_args(const Prob& p, const WsLayout& w, const int32_t* idx, unsigned* status, int b,
                  const Part* part = nullptr) {
  BwdArgs a;
  a.g = p.g;
  a.Hh = p.Hh;
  a.k = p.k;
  a.b = b;
  a.N = p.N;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  a.all_full = (p.g.T % p.g.bt == 0 && p.g.H % p.g.bh == 0 && p.g.W % p.g.bw == 0) ? 1 : 0;
  a.idx = idx;
  a.Dv = w.Dv;
  a.L2v = w.L2v;
  a.offsets = w.offsets;
  a.lists = w.lists;
  a.order = w.order;
  a.qlist = part ? w.qlist : nullptr;
  a.qcount = part ? w.qcount : nullptr;
  a.G = part && part->dLSE ? w.G : nullptr;
  a.status = status;
  const Geom& g = p.g;
  a.hdim = g.bt % 2 == 0 ? 0 : (g.bh % 2 == 0 ? 1 : 2);
  a.hoff = a.hdim == 0 ? g.bt / 2 : (a.hdim == 1 ? g.bh / 2 : g.bw / 2);
  return a;
}

bool token_map(CUtensorMap* m, const Prob& p, const void* base, int b, TokType t) {
  const size_t es = t == kTokF32 ? 4 : 2;
  const char* x = static_cast<const char*>(base) + (size_t)b * p.N * p.Hh * p.d * es;
  const Geom& g = p.g;
  return make_token_map(m, x, t, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw);
}

template <int D, bool F32OUT>
cudaError_t launch_dq(const Prob& p, const void* V, const void* dO, const int32_t* idx, void* dQ, void* ws,
                      cudaStream_t st, const Part* part) {
  using C = Cfg<D>;
  WsLayout w = ws_layout(p, ws);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  const size_t smem = 1024 + (size_t)C::TILE * (2 + C::KST + C::VST) + 8 * (6 + 2 * C::KST + C::VST) + 1024 + 8 + 64;
  cudaError_t e = cudaFuncSetAttribute(dq_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const TokType gt = F32OUT ? kTokF32 : kTokBF16;
  for (int b = 0; b < p.B; ++b) {
    CUtensorMap mQ, mK, mV, mdO, mdQ;
    if (!token_map(&mQ, p, w.Q16, b, kTokF16) || !token_map(&mK, p, w.K16, b, kTokF16) ||
        !token_map(&mV, p, w.V16, b, kTokF16) || !token_map(&mdO, p, w.dO16, b, kTokF16) ||
        !token_map(&mdQ, p, dQ, b, gt))
      return cudaErrorInvalidValue;
    dq_kernel<D, F32OUT><<<dim3(p.g.nb, p.Hh), kThreads, smem, st>>>(mQ, mK, mV, mdO, mdQ,
                                                                     make_args(p, w, idx, status, b, part));
    note_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D, bool F32OUT>
cudaError_t launch_dqx(const Prob& p, const int32_t* idx, void* dQ, void* ws, cudaStream_t st) {
  using C = Cfg<D>;
  WsLayout w = ws_layout(p, ws);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  const size_t smem = 1024 + (size_t)C::TILE * (2 + C::KST + C::VST) + 8 * (7 + 2 * C::KST + C::VST) + 8 + 64;
  cudaError_t e = cudaFuncSetAttribute(dqx_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const TokType gt = F32OUT ? kTokF32 : kTokBF16;
  for (int b = 0; b < p.B; ++b) {
    CUtensorMap mQ, mK, mV, mdO, mdQ;
    if (!token_map(&mQ, p, w.Q16, b, kTokF16) || !token_map(&mK, p, w.K16, b, kTokF16) ||
        !token_map(&mV, p, w.V16, b, kTokF16) || !token_map(&mdO, p, w.dO16, b, kTokF16) ||
        !token_map(&mdQ, p, dQ, b, gt))
      return cudaErrorInvalidValue;
    dqx_kernel<D, F32OUT><<<dim3(p.g.nb, p.Hh), kThreads, smem, st>>>(mQ, mK, mV, mdO, mdQ,
                                                                      make_args(p, w, idx, status, b));
    note_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D, bool F32OUT>
cudaError_t launch_dkdv(const Prob& p, const void* V, const void* dO, void* dK, void* dV, void* ws, cudaStream_t st) {
  using C = Cfg<D>;
  WsLayout w = ws_layout(p, ws);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  // K, V tiles; 2 ST half-stage tiles; their LSE/D rows; barriers; TMEM slot and abort flag
  const size_t smem = 1024 + (size_t)C::TILE * 2 + (size_t)C::ST * (2 * C::TILE + 1024) + 8 * (6 + 4 * C::ST) + 8 + 64;
  cudaError_t e =
      cudaFuncSetAttribute(dkdv_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const TokType gt = F32OUT ? kTokF32 : kTokBF16;
  const Geom& g = p.g;
  const BwdArgs a0 = make_args(p, w, nullptr, status, 0);
  const int hbt = a0.hdim == 0 ? g.bt / 2 : g.bt, hbh = a0.hdim == 1 ? g.bh / 2 : g.bh,
            hbw = a0.hdim == 2 ? g.bw / 2 : g.bw;
  auto half_map = [&](CUtensorMap* m, const void* base, int b) {
    const char* x = static_cast<const char*>(base) + (size_t)b * p.N * p.Hh * p.d * 2;
    return make_token_map(m, x, kTokF16, g.T, g.H, g.W, p.Hh, p.d, hbt, hbh, hbw);
  };
  for (int b = 0; b < p.B; ++b) {
    CUtensorMap mQ, mK, mV, mdO, mdK, mdV;  // Q and dO maps load 64-row half tiles
    if (!half_map(&mQ, w.Q16, b) || !token_map(&mK, p, w.K16, b, kTokF16) ||
        !token_map(&mV, p, w.V16, b, kTokF16) || !half_map(&mdO, w.dO16, b) ||
        !token_map(&mdK, p, dK, b, gt) || !token_map(&mdV, p, dV, b, gt))
      return cudaErrorInvalidValue;
    dkdv_kernel<D, F32OUT><<<dim3(p.g.nb, p.Hh), kThreads, smem, st>>>(mQ, mK, mV, mdO, mdK, mdV,
                                                                       make_args(p, w, nullptr, status, b));
    note_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

size_t bwd_ws_tc(const Prob& p) { return ws_layout(p, nullptr).bytes; }
size_t train_ws_tc(const Prob& p) { return ws_layout(p, nullptr, true).bytes; }

namespace {
// The block-map transpose (all batches and heads at once): for every key block the query
// blocks that kept it, ascending, their counts and offsets, and the visiting order.
cudaError_t build_csr(const Prob& p, const WsLayout& w, const int32_t* idx, const Part* part, unsigned* status,
                      cudaStream_t st) {
  const Geom& g = p.g;
  cudaError_t e;
  const int words = (g.nb + 31) / 32;
  const long long bhn = (long long)p.B * p.Hh * g.nb;
  if ((e = cudaMemsetAsync(w.bitmap, 0, (size_t)bhn * words * 4, st)) != cudaSuccess) return e;
  const long long entries = bhn * p.k;
  const int kb0 = part ? part->kb_begin : 0, kb1 = part ? part->kb_end : g.nb;
  const uint8_t* act = part ? part->qb_active : nullptr;
  csr_bitmap_kernel<<<(int)std::min<long long>((entries + 255) / 256, 1 << 20), 256, 0, st>>>(
      idx, entries, g.nb, p.k, words, kb0, kb1, act, w.bitmap, status);
  if (part) {
    rowlist_kernel<<<(int)std::min<long long>((bhn + 255) / 256, 152LL * 16), 256, 0, st>>>(idx, bhn, g.nb, p.k, kb0,
                                                                                           kb1, act, w.qlist, w.qcount);
    note_launches(1);
  }
  csr_count_kernel<<<(int)((bhn * 32 + 255) / 256), 256, 0, st>>>(w.bitmap, g.nb, words, bhn, w.counts);
  csr_scan_kernel<<<p.B * p.Hh, 1024, g.nb * sizeof(int32_t), st>>>(w.counts, g.nb, w.offsets);
  csr_order_kernel<<<dim3((g.nb + 255) / 256, p.B * p.Hh), 256, g.nb * sizeof(int32_t), st>>>(w.counts, g.nb,
                                                                                               w.order);
  csr_fill_kernel<<<(int)((bhn * 32 + 255) / 256), 256, 0, st>>>(w.bitmap, w.offsets, g.nb, p.k, words, bhn, w.lists);
  note_launches(5);
  return cudaGetLastError();
}

// bf16 -> fp16 copy of one [B, N, heads, d] tensor (range latched into status).
void half_copy(const Prob& p, const void* src, char* dst, unsigned* status, cudaStream_t st) {
  const long long n8 = (long long)p.B * p.N * p.Hh * p.d / 8;
  const int cb = (int)std::min<long long>((n8 + 255) / 256, 152LL * 16);
  half_kernel<<<cb, 256, 0, st>>>(static_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), n8, status);
  note_launches(1);
}

// D and the LSE rows in tile order, one launch per batch entry.
void row_terms(const Prob& p, const WsLayout& w, const void* O, bool o32, const float* LSE, const void* dO,
               const float* dLSE, cudaStream_t st) {
  const Geom& g = p.g;
  float* G = dLSE ? w.G : nullptr;
  const __nv_bfloat16* gO = static_cast<const __nv_bfloat16*>(dO);
  for (int b = 0; b < p.B; ++b) {
    const dim3 grid(g.nb, p.Hh);
    if (p.d == 64 && o32)
      pre_kernel<64, true><<<grid, 128, 0, st>>>(g, p.Hh, p.N, b, O, gO, LSE, dLSE, w.Dv, w.L2v, G);
    else if (p.d == 64)
      pre_kernel<64, false><<<grid, 128, 0, st>>>(g, p.Hh, p.N, b, O, gO, LSE, dLSE, w.Dv, w.L2v, G);
    else if (o32)
      pre_kernel<128, true><<<grid, 128, 0, st>>>(g, p.Hh, p.N, b, O, gO, LSE, dLSE, w.Dv, w.L2v, G);
    else
      pre_kernel<128, false><<<grid, 128, 0, st>>>(g, p.Hh, p.N, b, O, gO, LSE, dLSE, w.Dv, w.L2v, G);
  }
  note_launches(p.B);
}
}  // namespace

cudaError_t bwd_prepare_tc(const Prob& p, const void* Q, const void* K, const void* V, const void* O,
                           const float* LSE, const void* dO, const int32_t* idx, void* ws, cudaStream_t st,
                           const Part* part) {
  WsLayout w = ws_layout(p, ws);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  cudaError_t e = build_csr(p, w, idx, part, status, st);
  if (e != cudaSuccess) return e;
  half_copy(p, Q, w.Q16, status, st);
  half_copy(p, K, w.K16, status, st);
  half_copy(p, V, w.V16, status, st);
  half_copy(p, dO, w.dO16, status, st);
  row_terms(p, w, O, false, LSE, dO, part ? part->dLSE : nullptr, st);
  return cudaGetLastError();
}

cudaError_t fwd_train_tc(const Prob& p, const void* Q, const void* K, const void* V, const int32_t* idx, void* O,
                         float* LSE, void* ws, cudaStream_t st) {
  WsLayout w = ws_layout(p, ws, true);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  half_copy(p, Q, w.Q16, status, st);
  half_copy(p, K, w.K16, status, st);
  half_copy(p, V, w.V16, status, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return fwd_tc_f16(p, w.Q16, w.K16, w.V16, idx, O, LSE, w.O32, st);
}

cudaError_t bwd_train_tc(const Prob& p, const float* LSE, const void* dO, const int32_t* idx, void* dQ, void* dK,
                         void* dV, int grad_dtype, void* ws, int phases, cudaStream_t st) {
  WsLayout w = ws_layout(p, ws, true);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  cudaError_t e;
  const bool f32 = grad_dtype == SDA_F32;
  if (phases & 1) {
    if ((e = build_csr(p, w, idx, nullptr, status, st)) != cudaSuccess) return e;
    half_copy(p, dO, w.dO16, status, st);
    row_terms(p, w, w.O32, true, LSE, dO, nullptr, st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (phases & 2) {
    if (p.d == 64)
      e = f32 ? launch_dqx<64, true>(p, idx, dQ, ws, st) : launch_dqx<64, false>(p, idx, dQ, ws, st);
    else
      e = f32 ? launch_dqx<128, true>(p, idx, dQ, ws, st) : launch_dqx<128, false>(p, idx, dQ, ws, st);
    if (e != cudaSuccess) return e;
  }
  if (phases & 4) {
    if (p.d == 64)
      e = f32 ? launch_dkdv<64, true>(p, nullptr, nullptr, dK, dV, ws, st)
              : launch_dkdv<64, false>(p, nullptr, nullptr, dK, dV, ws, st);
    else
      e = f32 ? launch_dkdv<128, true>(p, nullptr, nullptr, dK, dV, ws, st)
              : launch_dkdv<128, false>(p, nullptr, nullptr, dK, dV, ws, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t bwd_dq_tc(const Prob& p, const void* V, const void* dO, const int32_t* idx, void* dQ, int grad_dtype,
                      void* ws, cudaStream_t st, const Part* part) {
  const bool f32 = grad_dtype == SDA_F32;
  if (p.d == 64)
    return f32 ? launch_dq<64, true>(p, V, dO, idx, dQ, ws, st, part)
               : launch_dq<64, false>(p, V, dO, idx, dQ, ws, st, part);
  return f32 ? launch_dq<128, true>(p, V, dO, idx, dQ, ws, st, part)
             : launch_dq<128, false>(p, V, dO, idx, dQ, ws, st, part);
}

cudaError_t bwd_dkdv_tc(const Prob& p, const void* V, const void* dO, void* dK, void* dV, int grad_dtype, void* ws,
                        cudaStream_t st) {
  const bool f32 = grad_dtype == SDA_F32;
  if (p.d == 64)
    return f32 ? launch_dkdv<64, true>(p, V, dO, dK, dV, ws, st) : launch_dkdv<64, false>(p, V, dO, dK, dV, ws, st);
  return f32 ? launch_dkdv<128, true>(p, V, dO, dK, dV, ws, st) : launch_dkdv<128, false>(p, V, dO, dK, dV, ws, st);
}

}  // namespace sda
