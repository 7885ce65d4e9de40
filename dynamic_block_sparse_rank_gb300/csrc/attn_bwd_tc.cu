// Block-sparse flash-attention backward on the 5th-generation tensor cores.
//
// Gradients of the forward of "DSV: Exploiting Dynamic Sparsity to Accelerate
// Large-Scale Video DiT Training" (section 4, stage 2: compute only on the kept
// blocks) with the block map held fixed: with P = exp(scale Q K^T - LSE) on the
// kept blocks and D_i = dO_i . O_i,
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Deterministic, no atomics on gradient values.  Kernels, in stream order:
//   pre_kernel      D_i and LSE_i * log2(e) per row, tile-ordered (+inf for
//                   rows outside the grid so that their P is exactly zero).
//   csr kernels     transpose the block map: for every key block J the query
//                   blocks that kept it, ascending; key blocks are then visited
//                   longest list first (LPT) to balance the dK/dV CTAs.
//   dq_kernel       per query block: S = Q K_J^T and dP = dO V_J^T (M=128,
//                   N=128, K=d), dS in TMEM, dQ += dS K_J; 8 compute warps.
//   dkdv_kernel     per key block: S^T = K Q_I^T and dP^T = V dO_I^T, P^T and
//                   dS^T in TMEM, dV += P^T dO_I, dK += dS^T Q_I.  For d = 128
//                   the four 128-column accumulators fill all 512 TMEM columns.
// The dq kernel repeats the S and dP products of the dK/dV kernel (7 GEMMs per
// block pair instead of 5) in exchange for no fp32 dQ reduction buffer.
#include "internal.h"

namespace sda {

namespace {

constexpr int kThreads = 384;  // warp 0 TMA, warp 1 MMA, warps 4-11 compute
constexpr float kLog2e = 1.4426950408889634f;

struct BwdArgs {
  Geom g;
  int Hh, k, b;
  long long N;
  float scale_log2;  // softmax scale * log2(e)
  float scale;
  const int32_t* idx;     // [B, Hh, nb, k]
  const float* Dv;        // [B, Hh, nb, 128]
  const float* L2v;       // [B, Hh, nb, 128]
  const int32_t* offsets; // [B, Hh, nb + 1]
  const int32_t* lists;   // [B, Hh, nb * k]
  const int32_t* order;   // [B, Hh, nb]
  unsigned* status;
};

__device__ __forceinline__ bool wait_plain(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > SDA_WAIT_LIMIT_NS) return false;
  return true;
}

// ------------------------------------------------------------------ preprocess
template <int D>
__global__ void __launch_bounds__(128) pre_kernel(Geom g, int Hh, long long N, int b, const __nv_bfloat16* __restrict__ O,
                                                  const __nv_bfloat16* __restrict__ dO, const float* __restrict__ LSE,
                                                  float* __restrict__ Dv, float* __restrict__ L2v) {
  const int I = blockIdx.x, h = blockIdx.y, r = threadIdx.x;
  const int n = block_row_token(g, I, r);
  float dsum = 0.f, l2 = INFINITY;
  if (n >= 0) {
    const uint4* o = reinterpret_cast<const uint4*>(O + (((long long)b * N + n) * Hh + h) * D);
    const uint4* go = reinterpret_cast<const uint4*>(dO + (((long long)b * N + n) * Hh + h) * D);
#pragma unroll 4
    for (int v = 0; v < D / 8; ++v) {
      const uint4 a = o[v], c = go[v];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dsum = fmaf(__uint_as_float(aw[q] << 16), __uint_as_float(cw[q] << 16), dsum);
        dsum = fmaf(__uint_as_float(aw[q] & 0xFFFF0000u), __uint_as_float(cw[q] & 0xFFFF0000u), dsum);
      }
    }
    const float lse = LSE[((long long)b * Hh + h) * N + n];
    l2 = lse == -INFINITY ? INFINITY : lse * kLog2e;
  }
  const long long o = (((long long)b * Hh + h) * g.nb + I) * 128 + r;
  Dv[o] = dsum;
  L2v[o] = l2;
}

// ------------------------------------------------------------------ block-map transpose
__global__ void csr_bitmap_kernel(const int32_t* __restrict__ idx, long long entries, int nb, int k, int words,
                                  unsigned* __restrict__ bitmap, unsigned* __restrict__ status) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < entries;
       e += (long long)gridDim.x * blockDim.x) {
    const long long row = e / k;  // (bh, I)
    const int J = idx[e];
    if (J < 0 || J >= nb) {
      atomicOr(status, kStatusBadIndex);
      continue;
    }
    atomicOr(bitmap + row * words + (J >> 5), 1u << (J & 31));
  }
}

// counts[bh, J] = number of query blocks that kept J.
__global__ void csr_count_kernel(const unsigned* __restrict__ bitmap, int nb, int words, long long total,
                                 int32_t* __restrict__ counts) {
  const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (t >= total) return;
  const long long bh = t / nb;
  const int J = (int)(t % nb);
  const unsigned* col = bitmap + bh * nb * words + (J >> 5);
  const unsigned bit = 1u << (J & 31);
  int c = 0;
  for (int I = 0; I < nb; ++I) c += (col[(long long)I * words] & bit) ? 1 : 0;
  counts[t] = c;
}

// Per (batch, head): exclusive scan of counts -> offsets, and the visiting order
// of key blocks by descending count (ties by ascending J).
__global__ void __launch_bounds__(1024) csr_scan_kernel(const int32_t* __restrict__ counts, int nb,
                                                        int32_t* __restrict__ offsets, int32_t* __restrict__ order) {
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
  for (int J = tid; J < nb; J += blockDim.x) {
    const int c = cs[J];
    int rank = 0;
    for (int J2 = 0; J2 < nb; ++J2) {
      const int c2 = cs[J2];
      rank += (c2 > c) || (c2 == c && J2 < J);
    }
    order[bh * nb + rank] = J;
  }
}

__global__ void csr_fill_kernel(const unsigned* __restrict__ bitmap, const int32_t* __restrict__ offsets, int nb,
                                int k, int words, long long total, int32_t* __restrict__ lists) {
  const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (t >= total) return;
  const long long bh = t / nb;
  const int J = (int)(t % nb);
  const unsigned* col = bitmap + bh * nb * words + (J >> 5);
  const unsigned bit = 1u << (J & 31);
  int pos = offsets[bh * (nb + 1) + J];
  int32_t* out = lists + bh * nb * k;
  for (int I = 0; I < nb; ++I)
    if (col[(long long)I * words] & bit) out[pos++] = I;
}

// ------------------------------------------------------------------ shared pieces
template <int D>
struct Cfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE = 128 * D * 2;
  static constexpr int ST = D == 128 ? 2 : 4;
};

// Store a 128 x D accumulator slice (this thread's row, columns [c_lo, c_lo + ncols))
// scaled by `mul` into a 128B-swizzled staging area laid out as TMA boxes of 128
// bytes of the row (bf16: 64 columns per box, fp32: 32 columns per box).
template <bool F32>
__device__ __forceinline__ void stage_row(uint8_t* stage, uint32_t taddr, int row, int c_lo, int ncols, float mul,
                                          bool zero) {
  for (int c0 = c_lo; c0 < c_lo + ncols; c0 += 32) {
    uint32_t u[32];
    if (!zero) {
      tmem_ld32(taddr + c0, u);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) u[e] = 0u;
    }
    if (F32) {
      uint8_t* box = stage + (c0 >> 5) * 16384;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint4 v = make_uint4(__float_as_uint(__uint_as_float(u[4 * q]) * mul),
                             __float_as_uint(__uint_as_float(u[4 * q + 1]) * mul),
                             __float_as_uint(__uint_as_float(u[4 * q + 2]) * mul),
                             __float_as_uint(__uint_as_float(u[4 * q + 3]) * mul));
        *reinterpret_cast<uint4*>(box + sw128_offset(row, q)) = v;
      }
    } else {
      uint8_t* box = stage + (c0 >> 6) * 16384;
      const int cbase = ((c0 & 63) >> 3);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 v;
        v.x = pack_bf16(__uint_as_float(u[8 * q + 0]) * mul, __uint_as_float(u[8 * q + 1]) * mul);
        v.y = pack_bf16(__uint_as_float(u[8 * q + 2]) * mul, __uint_as_float(u[8 * q + 3]) * mul);
        v.z = pack_bf16(__uint_as_float(u[8 * q + 4]) * mul, __uint_as_float(u[8 * q + 5]) * mul);
        v.w = pack_bf16(__uint_as_float(u[8 * q + 6]) * mul, __uint_as_float(u[8 * q + 7]) * mul);
        *reinterpret_cast<uint4*>(box + sw128_offset(row, cbase + q)) = v;
      }
    }
  }
}

// ------------------------------------------------------------------ dQ
template <int D, bool F32OUT>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const __grid_constant__ CUtensorMap tmdQ, BwdArgs a) {
  using C = Cfg<D>;
  constexpr int ST = C::ST;
  const int I = blockIdx.x, h = blockIdx.y;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + C::TILE;
  uint8_t* sK = sdO + C::TILE;        // ST tiles
  uint8_t* sV = sK + ST * C::TILE;    // ST tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + ST * C::TILE);
  uint64_t* qfull = bars;
  uint64_t* kvfull = qfull + 1;       // ST
  uint64_t* kvempty = kvfull + ST;    // ST
  uint64_t* sdpfull = kvempty + ST;   // 1
  uint64_t* dsfull = sdpfull + 1;     // 1
  uint64_t* drain = dsfull + 1;       // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t* sel = a.idx + (((long long)a.b * a.Hh + h) * a.g.nb + I) * a.k;
  const int n = a.k;
  if (tid == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(kvfull + s, 1);
      mbar_init(kvempty + s, 1);
    }
    mbar_init(sdpfull, 1);
    mbar_init(dsfull, 256);
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
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256;
  int t0, h0, w0;
  block_origin(a.g, I, t0, h0, w0);

  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(qfull, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_load_5d(sQ + c * 16384, &tmQ, qfull, c * 64, h, w0, h0, t0);
        tma_load_5d(sdO + c * 16384, &tmdO, qfull, c * 64, h, w0, h0, t0);
      }
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int s = j % ST;
        if (j >= ST && !mbar_wait(kvempty + s, ((j / ST) - 1) & 1, a.status, abort_flag)) break;
        int jt0, jh0, jw0;
        block_origin(a.g, sel[j], jt0, jh0, jw0);
        mbar_expect_tx(kvfull + s, 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_5d(sK + s * C::TILE + c * 16384, &tmK, kvfull + s, c * 64, h, jw0, jh0, jt0);
          tma_load_5d(sV + s * C::TILE + c * 16384, &tmV, kvfull + s, c * 64, h, jw0, jh0, jt0);
        }
        issued = j + 1;
      }
      if (*abort_flag) {
        wait_plain(qfull, 0);
        for (int j = issued - ST < 0 ? 0 : issued - ST; j < issued; ++j) wait_plain(kvfull + j % ST, (j / ST) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idQ = idesc_bf16(128, D, 0, 1);
      const uint32_t aQ = smem_u32(sQ), adO = smem_u32(sdO), aK = smem_u32(sK), aV = smem_u32(sV);
      bool ok = mbar_wait(qfull, 0, a.status, abort_flag);
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % ST;
        if (!mbar_wait(kvfull + s, (j / ST) & 1, a.status, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tS, smem_desc(aQ + off, 16, 1024, 2), smem_desc(aK + s * C::TILE + off, 16, 1024, 2), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tdP, smem_desc(adO + off, 16, 1024, 2), smem_desc(aV + s * C::TILE + off, 16, 1024, 2), idS,
                 kk > 0);
        }
        mma_commit(sdpfull);
        if (!mbar_wait(dsfull, j & 1, a.status, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tdQ, tS + kk * 8, smem_desc(aK + s * C::TILE + kk * 2048, 16384, 1024, 2), idQ, (j > 0 || kk > 0));
        mma_commit(kvempty + s);
      }
      mma_commit(drain);
      wait_plain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int grp = (warp - 4) >> 2;                 // key columns [64 grp, 64 grp + 64)
    const int row = (warp & 3) * 32 + lane;          // query row = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const long long tile_row = (((long long)a.b * a.Hh + h) * a.g.nb + I) * 128 + row;
    const float l2 = a.L2v[tile_row];
    const float Di = a.Dv[tile_row];
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait(sdpfull, j & 1, a.status, abort_flag)) break;
      tc_fence_after();
      const int J = sel[j];
      const bool full = block_is_full(a.g, J);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = grp * 64 + cc * 32;
        uint32_t us[32], up[32];
        tmem_ld32(tS + lane_base + col0, us);
        tmem_ld32(tdP + lane_base + col0, up);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float p0 = ex2(fmaf(__uint_as_float(us[2 * e]), a.scale_log2, -l2));
          float p1 = ex2(fmaf(__uint_as_float(us[2 * e + 1]), a.scale_log2, -l2));
          if (!full) {
            if (block_row_token(a.g, J, col0 + 2 * e) < 0) p0 = 0.f;
            if (block_row_token(a.g, J, col0 + 2 * e + 1) < 0) p1 = 0.f;
          }
          pk[e] = pack_bf16(p0 * (__uint_as_float(up[2 * e]) - Di), p1 * (__uint_as_float(up[2 * e + 1]) - Di));
        }
        tmem_st16(tS + lane_base + col0 / 2, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(dsfull);
    }
    // epilogue: dQ = scale * (dS K) -> staging (Q and dO tiles are free once all MMAs are done)
    mbar_wait(drain, 0, a.status, abort_flag);
    tc_fence_after();
    stage_row<F32OUT>(sQ, tdQ + lane_base, row, grp * (D / 2), D / 2, a.scale, n == 0);
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
  constexpr int ST = C::ST;
  constexpr int STAGE = 2 * C::TILE + 2 * 512;  // Q, dO, L2 row, D row
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
  uint8_t* ring = sV + C::TILE;  // ST stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + ST * STAGE);
  uint64_t* kvfull = bars;
  uint64_t* qfull = kvfull + 1;     // ST
  uint64_t* qempty = qfull + ST;    // ST
  uint64_t* sdpfull = qempty + ST;  // 1
  uint64_t* pdsfull = sdpfull + 1;  // 1
  uint64_t* drain = pdsfull + 1;    // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(kvfull, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(qfull + s, 1);
      mbar_init(qempty + s, 1);
    }
    mbar_init(sdpfull, 1);
    mbar_init(pdsfull, 256);
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
      for (int u = 0; u < n; ++u) {
        const int s = u % ST;
        if (u >= ST && !mbar_wait(qempty + s, ((u / ST) - 1) & 1, a.status, abort_flag)) break;
        const int I = users[u];
        int it0, ih0, iw0;
        block_origin(a.g, I, it0, ih0, iw0);
        uint8_t* st = ring + s * STAGE;
        mbar_expect_tx(qfull + s, STAGE);
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_5d(st + c * 16384, &tmQ, qfull + s, c * 64, h, iw0, ih0, it0);
          tma_load_5d(st + C::TILE + c * 16384, &tmdO, qfull + s, c * 64, h, iw0, ih0, it0);
        }
        const long long trow = (bh * a.g.nb + I) * 128;
        bulk_load(st + 2 * C::TILE, a.L2v + trow, 512, qfull + s);
        bulk_load(st + 2 * C::TILE + 512, a.Dv + trow, 512, qfull + s);
        issued = u + 1;
      }
      if (*abort_flag) {
        wait_plain(kvfull, 0);
        for (int u = issued - ST < 0 ? 0 : issued - ST; u < issued; ++u) wait_plain(qfull + u % ST, (u / ST) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idG = idesc_bf16(128, D, 0, 1);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aR = smem_u32(ring);
      bool ok = mbar_wait(kvfull, 0, a.status, abort_flag);
      for (int u = 0; ok && u < n; ++u) {
        const int s = u % ST;
        const uint32_t aQ = aR + s * STAGE, adO = aQ + C::TILE;
        if (!mbar_wait(qfull + s, (u / ST) & 1, a.status, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tS, smem_desc(aK + off, 16, 1024, 2), smem_desc(aQ + off, 16, 1024, 2), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tdP, smem_desc(aV + off, 16, 1024, 2), smem_desc(adO + off, 16, 1024, 2), idS, kk > 0);
        }
        mma_commit(sdpfull);
        if (!mbar_wait(pdsfull, u & 1, a.status, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_ts(tdV, tS + kk * 8, smem_desc(adO + kk * 2048, 16384, 1024, 2), idG, (u > 0 || kk > 0));
          mma_ts(tdK, tdP + kk * 8, smem_desc(aQ + kk * 2048, 16384, 1024, 2), idG, (u > 0 || kk > 0));
        }
        mma_commit(qempty + s);
      }
      mma_commit(drain);
      wait_plain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int grp = (warp - 4) >> 2;         // query columns [64 grp, 64 grp + 64)
    const int row = (warp & 3) * 32 + lane;  // key row = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool row_ok = block_row_token(a.g, J, row) >= 0;
    for (int u = 0; u < n; ++u) {
      if (!mbar_wait(sdpfull, u & 1, a.status, abort_flag)) break;
      tc_fence_after();
      const uint8_t* st = ring + (u % ST) * STAGE;
      const float* l2 = reinterpret_cast<const float*>(st + 2 * C::TILE);
      const float* dv = l2 + 128;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = grp * 64 + cc * 32;
        uint32_t us[32], up[32];
        tmem_ld32(tS + lane_base + col0, us);
        tmem_ld32(tdP + lane_base + col0, up);
        tmem_wait_ld();
        uint32_t pp[16], pd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = col0 + 2 * e;
          float p0 = ex2(fmaf(__uint_as_float(us[2 * e]), a.scale_log2, -l2[c]));
          float p1 = ex2(fmaf(__uint_as_float(us[2 * e + 1]), a.scale_log2, -l2[c + 1]));
          if (!row_ok) p0 = p1 = 0.f;
          pp[e] = pack_bf16(p0, p1);
          pd[e] = pack_bf16(p0 * (__uint_as_float(up[2 * e]) - dv[c]), p1 * (__uint_as_float(up[2 * e + 1]) - dv[c + 1]));
        }
        tmem_st16(tS + lane_base + col0 / 2, pp);
        tmem_st16(tdP + lane_base + col0 / 2, pd);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(pdsfull);
    }
    if (n > 0) mbar_wait(drain, 0, a.status, abort_flag);
    tc_fence_after();
    // staging: dK boxes then dV boxes, starting at sK (K, V and the ring are free now)
    constexpr int GB = F32OUT ? 128 * D * 4 : 128 * D * 2;  // bytes of one staged gradient tile
    stage_row<F32OUT>(sK, tdK + lane_base, row, grp * (D / 2), D / 2, a.scale, n == 0);
    stage_row<F32OUT>(sK + GB, tdV + lane_base, row, grp * (D / 2), D / 2, 1.f, n == 0);
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
  size_t bytes;
};

WsLayout ws_layout(const Prob& p, void* base) {
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
  w.bytes = off;
  return w;
}

template <int D, bool F32OUT>
cudaError_t launch_bwd(const Prob& p, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                       const void* dO, const int32_t* idx, void* dQ, void* dK, void* dV, void* ws, cudaStream_t st) {
  using C = Cfg<D>;
  const Geom& g = p.g;
  WsLayout w = ws_layout(p, ws);
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  cudaError_t e;
  // block-map transpose (all batches and heads at once)
  const int words = (g.nb + 31) / 32;
  const long long bhn = (long long)p.B * p.Hh * g.nb;
  if ((e = cudaMemsetAsync(w.bitmap, 0, (size_t)bhn * words * 4, st)) != cudaSuccess) return e;
  const long long entries = bhn * p.k;
  csr_bitmap_kernel<<<(int)std::min<long long>((entries + 255) / 256, 1 << 20), 256, 0, st>>>(idx, entries, g.nb, p.k,
                                                                                              words, w.bitmap, status);
  csr_count_kernel<<<(int)((bhn + 255) / 256), 256, 0, st>>>(w.bitmap, g.nb, words, bhn, w.counts);
  csr_scan_kernel<<<p.B * p.Hh, 1024, g.nb * sizeof(int32_t), st>>>(w.counts, g.nb, w.offsets, w.order);
  csr_fill_kernel<<<(int)((bhn + 255) / 256), 256, 0, st>>>(w.bitmap, w.offsets, g.nb, p.k, words, bhn, w.lists);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const size_t smem_dq = 1024 + (size_t)C::TILE * (2 + 2 * C::ST) + 8 * (4 + 2 * C::ST) + 64;
  const size_t smem_dkdv = 1024 + (size_t)C::TILE * 2 + (size_t)C::ST * (2 * C::TILE + 1024) + 8 * (4 + 2 * C::ST) + 64;
  if ((e = cudaFuncSetAttribute(dq_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dq)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(dkdv_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_dkdv)) != cudaSuccess)
    return e;
  const size_t per_batch = (size_t)p.N * p.Hh * p.d * 2;
  const size_t per_batch_g = (size_t)p.N * p.Hh * p.d * (F32OUT ? 4 : 2);
  const int ges = F32OUT ? 4 : 2;
  for (int b = 0; b < p.B; ++b) {
    auto at = [&](const void* x, size_t pb) { return static_cast<const char*>(x) + b * pb; };
    pre_kernel<D><<<dim3(g.nb, p.Hh), 128, 0, st>>>(
        g, p.Hh, p.N, b, static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), LSE, w.Dv, w.L2v);
    CUtensorMap mQ, mK, mV, mdO, mdQ, mdK, mdV;
    if (!make_token_map(&mQ, at(Q, per_batch), 2, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw) ||
        !make_token_map(&mK, at(K, per_batch), 2, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw) ||
        !make_token_map(&mV, at(V, per_batch), 2, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw) ||
        !make_token_map(&mdO, at(dO, per_batch), 2, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw) ||
        !make_token_map(&mdQ, at(dQ, per_batch_g), ges, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw) ||
        !make_token_map(&mdK, at(dK, per_batch_g), ges, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw) ||
        !make_token_map(&mdV, at(dV, per_batch_g), ges, g.T, g.H, g.W, p.Hh, p.d, g.bt, g.bh, g.bw))
      return cudaErrorInvalidValue;
    BwdArgs a;
    a.g = g;
    a.Hh = p.Hh;
    a.k = p.k;
    a.b = b;
    a.N = p.N;
    a.scale = p.scale;
    a.scale_log2 = p.scale * kLog2e;
    a.idx = idx;
    a.Dv = w.Dv;
    a.L2v = w.L2v;
    a.offsets = w.offsets;
    a.lists = w.lists;
    a.order = w.order;
    a.status = status;
    dim3 grid(g.nb, p.Hh);
    dq_kernel<D, F32OUT><<<grid, kThreads, smem_dq, st>>>(mQ, mK, mV, mdO, mdQ, a);
    dkdv_kernel<D, F32OUT><<<grid, kThreads, smem_dkdv, st>>>(mQ, mK, mV, mdO, mdK, mdV, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

size_t bwd_ws_tc(const Prob& p) { return ws_layout(p, nullptr).bytes; }

cudaError_t bwd_tc(const Prob& p, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                   const void* dO, const int32_t* idx, void* dQ, void* dK, void* dV, int grad_dtype, void* ws,
                   cudaStream_t st) {
  const bool f32 = grad_dtype == SDA_F32;
  if (p.d == 64)
    return f32 ? launch_bwd<64, true>(p, Q, K, V, O, LSE, dO, idx, dQ, dK, dV, ws, st)
               : launch_bwd<64, false>(p, Q, K, V, O, LSE, dO, idx, dQ, dK, dV, ws, st);
  return f32 ? launch_bwd<128, true>(p, Q, K, V, O, LSE, dO, idx, dQ, dK, dV, ws, st)
             : launch_bwd<128, false>(p, Q, K, V, O, LSE, dO, idx, dQ, dK, dV, ws, st);
}

}  // namespace sda
