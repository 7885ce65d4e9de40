// fp32 problems: CUDA-core kernels for the predictor, the block-sparse forward
// and the backward.  They follow the same definitions as the tensor-core path
// (see the header of include/sda.h) in full fp32 arithmetic, one thread per
// token row.  Sizes they cover: tiles up to 1024 tokens, d <= 128, r <= 64.
#include "internal.h"
#include "topk.cuh"

namespace sda {

namespace {

constexpr int kChunk = 32;  // key/query rows staged in shared memory at a time

__device__ __forceinline__ int valid_token(const Geom& g, int I, int r) { return block_row_token(g, I, r); }

// q~ = X Wt (per head), stored tile-ordered [B, Hh, nb*bs, r]; rows outside the grid are zero.
__global__ void proj_f32_kernel(Geom g, int B, int Hh, int d, int r, const float* __restrict__ X,
                                const float* __restrict__ Wt, float* __restrict__ out) {
  const long long rows = (long long)g.nb * g.bs;
  const long long total = (long long)B * Hh * rows * r;
  const long long N = (long long)g.T * g.H * g.W;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    int a = (int)(i % r);
    long long row = (i / r) % rows;
    long long bh = i / (r * rows);
    int b = (int)(bh / Hh), h = (int)(bh % Hh);
    int I = (int)(row / g.bs), rr = (int)(row % g.bs);
    int n = valid_token(g, I, rr);
    float acc = 0.f;
    if (n >= 0) {
      const float* x = X + (((long long)b * N + n) * Hh + h) * d;
      const float* w = Wt + (long long)h * d * r + a;
      for (int c = 0; c < d; ++c) acc = fmaf(x[c], w[(long long)c * r], acc);
    }
    out[i] = acc;
  }
}

// Block max of q~_i . k~_j over i in I, j in J for every J, then top-k.
__global__ void __launch_bounds__(256) scores_topk_f32_kernel(Geom g, int Hh, int r, int k,
                                                              const float* __restrict__ qt,
                                                              const float* __restrict__ kt,
                                                              int32_t* __restrict__ idx, float* __restrict__ score) {
  extern __shared__ float smem[];
  const int I = blockIdx.x, bh = blockIdx.y;
  const int tid = threadIdx.x;
  float* qs = smem;                      // bs * r
  float* srow = qs + g.bs * r;           // nb
  float* red = srow + g.nb;              // 32
  TopkScratch* ts = reinterpret_cast<TopkScratch*>(red + 32);
  const long long rows = (long long)g.nb * g.bs;
  const float* qbase = qt + ((long long)bh * rows + (long long)I * g.bs) * r;
  for (int i = tid; i < g.bs * r; i += blockDim.x) qs[i] = qbase[i];
  __syncthreads();
  for (int J = 0; J < g.nb; ++J) {
    const float* kbase = kt + ((long long)bh * rows + (long long)J * g.bs) * r;
    float best = -INFINITY;
    for (int p = tid; p < g.bs * g.bs; p += blockDim.x) {
      int i = p / g.bs, j = p % g.bs;
      if (valid_token(g, I, i) < 0 || valid_token(g, J, j) < 0) continue;
      float acc = 0.f;
      for (int a = 0; a < r; ++a) acc = fmaf(qs[i * r + a], kbase[(long long)j * r + a], acc);
      best = fmaxf(best, acc);
    }
    for (int o = 16; o > 0; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
    if ((tid & 31) == 0) red[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
      float m = red[0];
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
      srow[J] = m;
    }
    __syncthreads();
  }
  if (score)
    for (int J = tid; J < g.nb; J += blockDim.x) score[((long long)bh * g.nb + I) * g.nb + J] = srow[J];
  topk_select(srow, g.nb, k, idx + ((long long)bh * g.nb + I) * k, tid, blockDim.x, 1, ts);
}

// Compact the kept blocks of row I that fall in [kb_begin, kb_end) into sel (ascending input order kept).
// With a status word, an entry outside [0, nb) latches kStatusBadIndex (it is skipped either way, as
// 0 <= kb_begin <= kb_end <= nb).
__device__ int filter_sel(const int32_t* row, int k, int kb_begin, int kb_end, int* sel, int nb = 0,
                          unsigned* status = nullptr) {
  __shared__ int n_sel;
  if (threadIdx.x == 0) {
    int n = 0;
    for (int s = 0; s < k; ++s) {
      int J = row[s];
      if (status && (J < 0 || J >= nb)) atomicOr(status, kStatusBadIndex);
      if (J >= kb_begin && J < kb_end) sel[n++] = J;
    }
    n_sel = n;
  }
  __syncthreads();
  return n_sel;
}

template <int DM>
__global__ void fwd_f32_kernel(Geom g, int Hh, int d, int k, float scale, const float* __restrict__ Q,
                               const float* __restrict__ K, const float* __restrict__ V,
                               const int32_t* __restrict__ idx, int kb_begin, int kb_end,
                               const uint8_t* __restrict__ qb_active, float* __restrict__ O,
                               float* __restrict__ LSE, int b, unsigned* __restrict__ status) {
  extern __shared__ float smem[];
  const int I = blockIdx.x, h = blockIdx.y;
  if (qb_active && !qb_active[I]) return;
  float* ks = smem;                 // kChunk * d
  float* vs = ks + kChunk * d;      // kChunk * d
  int* kv_ok = reinterpret_cast<int*>(vs + kChunk * d);  // kChunk
  int* sel = kv_ok + kChunk;        // k
  const long long N = (long long)g.T * g.H * g.W;
  const int n_sel =
      filter_sel(idx + (((long long)b * Hh + h) * g.nb + I) * k, k, kb_begin, kb_end, sel, g.nb, status);
  const int row = threadIdx.x;
  const int n = row < g.bs ? valid_token(g, I, row) : -1;
  float q[DM], o[DM];
#pragma unroll
  for (int c = 0; c < DM; ++c) {
    q[c] = (n >= 0 && c < d) ? Q[(((long long)b * N + n) * Hh + h) * d + c] : 0.f;
    o[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int s = 0; s < n_sel; ++s) {
    const int J = sel[s];
    for (int c0 = 0; c0 < g.bs; c0 += kChunk) {
      __syncthreads();
      for (int e = threadIdx.x; e < kChunk * d; e += blockDim.x) {
        int j = e / d, c = e % d;
        int tok = (c0 + j < g.bs) ? valid_token(g, J, c0 + j) : -1;
        long long off = (((long long)b * N + (tok < 0 ? 0 : tok)) * Hh + h) * d + c;
        ks[e] = tok >= 0 ? K[off] : 0.f;
        vs[e] = tok >= 0 ? V[off] : 0.f;
        if (c == 0) kv_ok[j] = tok >= 0;
      }
      __syncthreads();
      if (n < 0) continue;
      for (int j = 0; j < kChunk; ++j) {
        if (!kv_ok[j]) continue;
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < DM; ++c)
          if (c < d) acc = fmaf(q[c], ks[j * d + c], acc);
        const float sc = acc * scale;
        const float m_new = fmaxf(m, sc);
        const float corr = expf(m - m_new);
        const float p = expf(sc - m_new);
        l = l * corr + p;
#pragma unroll
        for (int c = 0; c < DM; ++c)
          if (c < d) o[c] = fmaf(p, vs[j * d + c], o[c] * corr);
        m = m_new;
      }
    }
  }
  if (n < 0) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* orow = O + (((long long)b * N + n) * Hh + h) * d;
#pragma unroll
  for (int c = 0; c < DM; ++c)
    if (c < d) orow[c] = o[c] * inv;
  LSE[((long long)b * Hh + h) * N + n] = l > 0.f ? m + logf(l) : -INFINITY;
}

// D_i = dO_i . O_i - dLSE_i for every token row, into Dbuf [B, Hh, N] (the LSE
// gradient of a partition state enters dS = P (dP - D + dLSE) with D's sign).
__global__ void bwd_pre_f32_kernel(long long rows, int Hh, long long N, int d, const float* __restrict__ O,
                                   const float* __restrict__ dO, const float* __restrict__ dLSE,
                                   float* __restrict__ Dbuf) {
  for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows; r += (long long)gridDim.x * blockDim.x) {
    // r enumerates (b, n, h) in memory order
    const int h = (int)(r % Hh);
    const long long bn = r / Hh;
    const long long b = bn / N, n = bn % N;
    float acc = 0.f;
    for (int c = 0; c < d; ++c) acc = fmaf(dO[r * d + c], O[r * d + c], acc);
    const long long t = (b * Hh + h) * N + n;
    Dbuf[t] = dLSE ? acc - dLSE[t] : acc;
  }
}

// dQ for each query row.
template <int DM>
__global__ void bwd_dq_f32_kernel(Geom g, int Hh, int d, int k, float scale, const float* __restrict__ Q,
                                  const float* __restrict__ K, const float* __restrict__ V,
                                  const float* __restrict__ LSE, const float* __restrict__ dO,
                                  const int32_t* __restrict__ idx, float* __restrict__ dQ,
                                  const float* __restrict__ Dbuf, int b, int kb_begin, int kb_end,
                                  const uint8_t* __restrict__ qb_active) {
  extern __shared__ float smem[];
  const int I = blockIdx.x, h = blockIdx.y;
  float* ks = smem;
  float* vs = ks + kChunk * d;
  int* kv_ok = reinterpret_cast<int*>(vs + kChunk * d);
  int* sel = kv_ok + kChunk;
  const long long N = (long long)g.T * g.H * g.W;
  int n_sel = filter_sel(idx + (((long long)b * Hh + h) * g.nb + I) * k, k, kb_begin, kb_end, sel);
  if (qb_active && !qb_active[I]) n_sel = 0;  // an inactive query block contributes nothing
  const int row = threadIdx.x;
  const int n = row < g.bs ? valid_token(g, I, row) : -1;
  float q[DM], go[DM], dq[DM];
  float Di = 0.f, lse = 0.f;
  if (n >= 0) {
    const long long off = (((long long)b * N + n) * Hh + h) * d;
#pragma unroll
    for (int c = 0; c < DM; ++c) {
      q[c] = c < d ? Q[off + c] : 0.f;
      go[c] = c < d ? dO[off + c] : 0.f;
      dq[c] = 0.f;
    }
    lse = LSE[((long long)b * Hh + h) * N + n];
    Di = Dbuf[((long long)b * Hh + h) * N + n];
  }
  for (int s = 0; s < n_sel; ++s) {
    const int J = sel[s];
    for (int c0 = 0; c0 < g.bs; c0 += kChunk) {
      __syncthreads();
      for (int e = threadIdx.x; e < kChunk * d; e += blockDim.x) {
        int j = e / d, c = e % d;
        int tok = (c0 + j < g.bs) ? valid_token(g, J, c0 + j) : -1;
        long long off = (((long long)b * N + (tok < 0 ? 0 : tok)) * Hh + h) * d + c;
        ks[e] = tok >= 0 ? K[off] : 0.f;
        vs[e] = tok >= 0 ? V[off] : 0.f;
        if (c == 0) kv_ok[j] = tok >= 0;
      }
      __syncthreads();
      if (n < 0) continue;
      for (int j = 0; j < kChunk; ++j) {
        if (!kv_ok[j]) continue;
        float sc = 0.f, dp = 0.f;
#pragma unroll
        for (int c = 0; c < DM; ++c)
          if (c < d) {
            sc = fmaf(q[c], ks[j * d + c], sc);
            dp = fmaf(go[c], vs[j * d + c], dp);
          }
        const float p = expf(sc * scale - lse);
        const float ds = p * (dp - Di);
#pragma unroll
        for (int c = 0; c < DM; ++c)
          if (c < d) dq[c] = fmaf(ds, ks[j * d + c], dq[c]);
      }
    }
  }
  if (n < 0) return;
  float* out = dQ + (((long long)b * N + n) * Hh + h) * d;
#pragma unroll
  for (int c = 0; c < DM; ++c)
    if (c < d) out[c] = dq[c] * scale;
}

// dK, dV for each key row of block J, summing over the query blocks that kept J (ascending I).
template <int DM>
__global__ void bwd_dkdv_f32_kernel(Geom g, int Hh, int d, int k, float scale, const float* __restrict__ Q,
                                    const float* __restrict__ K, const float* __restrict__ V,
                                    const float* __restrict__ LSE, const float* __restrict__ dO,
                                    const int32_t* __restrict__ idx, const float* __restrict__ Dbuf,
                                    float* __restrict__ dK, float* __restrict__ dV, int b, int kb_begin, int kb_end,
                                    const uint8_t* __restrict__ qb_active) {
  extern __shared__ float smem[];
  const int J = blockIdx.x, h = blockIdx.y;
  float* qs = smem;                   // kChunk * d
  float* gs = qs + kChunk * d;        // kChunk * d
  float* ls = gs + kChunk * d;        // kChunk
  float* ds_ = ls + kChunk;           // kChunk
  int* qok = reinterpret_cast<int*>(ds_ + kChunk);  // kChunk
  int* users = qok + kChunk;          // nb
  __shared__ int n_users;
  const long long N = (long long)g.T * g.H * g.W;
  const int32_t* rows = idx + ((long long)b * Hh + h) * g.nb * k;
  if (threadIdx.x == 0) {
    int cnt = 0;
    if (J >= kb_begin && J < kb_end)  // outside the key range: no user, zero gradient
      for (int I = 0; I < g.nb; ++I) {
        if (qb_active && !qb_active[I]) continue;
        for (int s = 0; s < k; ++s)
          if (rows[(long long)I * k + s] == J) {
            users[cnt++] = I;
            break;
          }
      }
    n_users = cnt;
  }
  __syncthreads();
  const int row = threadIdx.x;
  const int n = row < g.bs ? valid_token(g, J, row) : -1;
  float kr[DM], vr[DM], dk[DM], dv[DM];
  if (n >= 0) {
    const long long off = (((long long)b * N + n) * Hh + h) * d;
#pragma unroll
    for (int c = 0; c < DM; ++c) {
      kr[c] = c < d ? K[off + c] : 0.f;
      vr[c] = c < d ? V[off + c] : 0.f;
      dk[c] = 0.f;
      dv[c] = 0.f;
    }
  }
  for (int u = 0; u < n_users; ++u) {
    const int I = users[u];
    for (int c0 = 0; c0 < g.bs; c0 += kChunk) {
      __syncthreads();
      for (int e = threadIdx.x; e < kChunk * d; e += blockDim.x) {
        int i = e / d, c = e % d;
        int tok = (c0 + i < g.bs) ? valid_token(g, I, c0 + i) : -1;
        long long off = (((long long)b * N + (tok < 0 ? 0 : tok)) * Hh + h) * d + c;
        qs[e] = tok >= 0 ? Q[off] : 0.f;
        gs[e] = tok >= 0 ? dO[off] : 0.f;
        if (c == 0) {
          qok[i] = tok >= 0;
          ls[i] = tok >= 0 ? LSE[((long long)b * Hh + h) * N + tok] : 0.f;
          ds_[i] = tok >= 0 ? Dbuf[((long long)b * Hh + h) * N + tok] : 0.f;
        }
      }
      __syncthreads();
      if (n < 0) continue;
      for (int i = 0; i < kChunk; ++i) {
        if (!qok[i]) continue;
        float sc = 0.f, dp = 0.f;
#pragma unroll
        for (int c = 0; c < DM; ++c)
          if (c < d) {
            sc = fmaf(qs[i * d + c], kr[c], sc);
            dp = fmaf(gs[i * d + c], vr[c], dp);
          }
        const float p = expf(sc * scale - ls[i]);
        const float dsv = p * (dp - ds_[i]);
#pragma unroll
        for (int c = 0; c < DM; ++c)
          if (c < d) {
            dv[c] = fmaf(p, gs[i * d + c], dv[c]);
            dk[c] = fmaf(dsv, qs[i * d + c], dk[c]);
          }
      }
    }
  }
  if (n < 0) return;
  const long long off = (((long long)b * N + n) * Hh + h) * d;
#pragma unroll
  for (int c = 0; c < DM; ++c)
    if (c < d) {
      dK[off + c] = dk[c] * scale;
      dV[off + c] = dv[c];
    }
}

inline int threads_for(int bs) { return (bs + 31) / 32 * 32; }

}  // namespace

size_t predict_ws_f32(const Prob& p) {
  return 2 * align_up((size_t)p.B * p.Hh * p.g.nb * p.g.bs * p.r * sizeof(float), 256);
}

cudaError_t predict_f32(const Prob& p, const float* Q, const float* K, const float* Wq, const float* Wk,
                        int32_t* idx, float* score, void* ws, cudaStream_t st) {
  const size_t one = align_up((size_t)p.B * p.Hh * p.g.nb * p.g.bs * p.r * sizeof(float), 256);
  float* qt = static_cast<float*>(ws);
  float* kt = reinterpret_cast<float*>(static_cast<char*>(ws) + one);
  const long long total = (long long)p.B * p.Hh * p.g.nb * p.g.bs * p.r;
  const int blocks = (int)std::min<long long>((total + 255) / 256, 65535LL * 16);
  proj_f32_kernel<<<blocks, 256, 0, st>>>(p.g, p.B, p.Hh, p.d, p.r, Q, Wq, qt);
  proj_f32_kernel<<<blocks, 256, 0, st>>>(p.g, p.B, p.Hh, p.d, p.r, K, Wk, kt);
  size_t smem = (size_t)(p.g.bs * p.r + p.g.nb + 32) * sizeof(float) + sizeof(TopkScratch) + 16;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(scores_topk_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(p.g.nb, p.B * p.Hh);
  scores_topk_f32_kernel<<<grid, 256, smem, st>>>(p.g, p.Hh, p.r, p.k, qt, kt, idx, score);
  note_launches(3);
  return cudaGetLastError();
}

template <int DM>
static cudaError_t fwd_f32_t(const Prob& p, const float* Q, const float* K, const float* V, const int32_t* idx,
                             int kb_begin, int kb_end, const uint8_t* qb_active, float* O, float* LSE,
                             cudaStream_t st) {
  size_t smem = (size_t)2 * kChunk * p.d * sizeof(float) + (kChunk + p.k) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(fwd_f32_kernel<DM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  unsigned* status = status_ptr();
  if (!status) return cudaErrorUnknown;
  dim3 grid(p.g.nb, p.Hh);
  for (int b = 0; b < p.B; ++b)
    fwd_f32_kernel<DM><<<grid, threads_for(p.g.bs), smem, st>>>(p.g, p.Hh, p.d, p.k, p.scale, Q, K, V, idx,
                                                                kb_begin, kb_end, qb_active, O, LSE, b, status);
  note_launches(p.B);
  return cudaGetLastError();
}

cudaError_t fwd_f32(const Prob& p, const float* Q, const float* K, const float* V, const int32_t* idx,
                    int kb_begin, int kb_end, const uint8_t* qb_active, float* O, float* LSE, cudaStream_t st) {
  if (p.d <= 64) return fwd_f32_t<64>(p, Q, K, V, idx, kb_begin, kb_end, qb_active, O, LSE, st);
  return fwd_f32_t<128>(p, Q, K, V, idx, kb_begin, kb_end, qb_active, O, LSE, st);
}

size_t bwd_ws_f32(const Prob& p) { return align_up((size_t)p.B * p.Hh * p.N * sizeof(float), 256); }

cudaError_t bwd_prepare_f32(const Prob& p, const float* O, const float* dO, void* ws, cudaStream_t st,
                            const float* dLSE) {
  const long long rows = (long long)p.B * p.N * p.Hh;
  const int blocks = (int)std::min<long long>((rows + 255) / 256, 152LL * 32);
  bwd_pre_f32_kernel<<<blocks, 256, 0, st>>>(rows, p.Hh, p.N, p.d, O, dO, dLSE, static_cast<float*>(ws));
  note_launches(1);
  return cudaGetLastError();
}

template <int DM>
static cudaError_t dq_f32_t(const Prob& p, const float* Q, const float* K, const float* V, const float* LSE,
                            const float* dO, const int32_t* idx, float* dQ, void* ws, cudaStream_t st,
                            const Part* part) {
  size_t smem = (size_t)2 * kChunk * p.d * sizeof(float) + (kChunk + p.k) * sizeof(int);
  cudaError_t e;
  if (smem > 48 * 1024 &&
      (e = cudaFuncSetAttribute(bwd_dq_f32_kernel<DM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
          cudaSuccess)
    return e;
  for (int b = 0; b < p.B; ++b)
    bwd_dq_f32_kernel<DM><<<dim3(p.g.nb, p.Hh), threads_for(p.g.bs), smem, st>>>(
        p.g, p.Hh, p.d, p.k, p.scale, Q, K, V, LSE, dO, idx, dQ, static_cast<const float*>(ws), b,
        part ? part->kb_begin : 0, part ? part->kb_end : p.g.nb, part ? part->qb_active : nullptr);
  note_launches(p.B);
  return cudaGetLastError();
}

template <int DM>
static cudaError_t dkdv_f32_t(const Prob& p, const float* Q, const float* K, const float* V, const float* LSE,
                              const float* dO, const int32_t* idx, float* dK, float* dV, void* ws, cudaStream_t st,
                              const Part* part) {
  size_t smem = (size_t)2 * kChunk * p.d * sizeof(float) + 3 * kChunk * sizeof(float) + p.g.nb * sizeof(int);
  cudaError_t e;
  if (smem > 48 * 1024 &&
      (e = cudaFuncSetAttribute(bwd_dkdv_f32_kernel<DM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
          cudaSuccess)
    return e;
  for (int b = 0; b < p.B; ++b)
    bwd_dkdv_f32_kernel<DM><<<dim3(p.g.nb, p.Hh), threads_for(p.g.bs), smem, st>>>(
        p.g, p.Hh, p.d, p.k, p.scale, Q, K, V, LSE, dO, idx, static_cast<const float*>(ws), dK, dV, b,
        part ? part->kb_begin : 0, part ? part->kb_end : p.g.nb, part ? part->qb_active : nullptr);
  note_launches(p.B);
  return cudaGetLastError();
}

cudaError_t bwd_dq_f32(const Prob& p, const float* Q, const float* K, const float* V, const float* LSE,
                       const float* dO, const int32_t* idx, float* dQ, void* ws, cudaStream_t st, const Part* part) {
  if (p.d <= 64) return dq_f32_t<64>(p, Q, K, V, LSE, dO, idx, dQ, ws, st, part);
  return dq_f32_t<128>(p, Q, K, V, LSE, dO, idx, dQ, ws, st, part);
}

cudaError_t bwd_dkdv_f32(const Prob& p, const float* Q, const float* K, const float* V, const float* LSE,
                         const float* dO, const int32_t* idx, float* dK, float* dV, void* ws, cudaStream_t st,
                         const Part* part) {
  if (p.d <= 64) return dkdv_f32_t<64>(p, Q, K, V, LSE, dO, idx, dK, dV, ws, st, part);
  return dkdv_f32_t<128>(p, Q, K, V, LSE, dO, idx, dK, dV, ws, st, part);
}

}  // namespace sda
