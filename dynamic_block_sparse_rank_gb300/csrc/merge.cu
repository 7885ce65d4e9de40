// LSE merge of partial attention states — the state-reuse primitive of
// "DiTango: Cost-Effective Parallel Diffusion Generation with Selective
// Attention State Reuse": per row, LSE = log sum_s exp(LSE_s) and
// O = sum_s exp(LSE_s - LSE) O_s; rows with every LSE_s = -inf give (0, -inf).
//
// Its gradient (training through the merge, the fresh states carrying the
// gradient): with w_s = exp(LSE_s - LSE), dO_s = w_s dO and
// dLSE_s = w_s (dO . (O_s - O) + dLSE).
//
// HBM-bound: every byte of every state is read once and the result written
// once.  A CTA covers 64 consecutive tokens of one (batch, head): the LSE
// reads are 256-byte runs and each O row is a contiguous d-element run read
// with 16-byte vector loads by a group of lanes (LPR lanes per row).
#include "internal.h"

namespace sda {

namespace {

constexpr int kRowsPerCta = 64;
constexpr int kThreads = 256;

template <typename T>
struct Vec;  // 16 bytes of T
template <>
struct Vec<float> {
  static constexpr int n = 4;
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int n = 8;
};

__device__ __forceinline__ void unpack(const uint4& v, float* f, const float*) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4& v, float* f, const __nv_bfloat16*) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint4 pack(const float* f, const float*) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}
__device__ __forceinline__ uint4 pack(const float* f, const __nv_bfloat16*) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}

template <typename T, int NS>
__global__ void __launch_bounds__(kThreads) merge_kernel(MergeArgs a, int lpr) {
  constexpr int VN = Vec<T>::n;
  const int h = blockIdx.y, b = blockIdx.z;
  const int n0 = blockIdx.x * kRowsPerCta;
  const int rows_per_pass = kThreads / lpr;
  const int sub = threadIdx.x / lpr, lane = threadIdx.x % lpr;
  const int nvec = a.d / VN;  // vectors per row
  for (int rr = sub; rr < kRowsPerCta; rr += rows_per_pass) {
    const int n = n0 + rr;
    if (n >= a.N) break;
    const size_t lrow = ((size_t)b * a.Hh + h) * a.N + n;
    const size_t orow = (((size_t)b * a.N + n) * a.Hh + h) * (size_t)a.d;
    float ls[NS];
    float m = -INFINITY;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      ls[s] = a.L[s][lrow];
      m = fmaxf(m, ls[s]);
    }
    float lse, w[NS];
    if (m == -INFINITY) {
      lse = -INFINITY;
#pragma unroll
      for (int s = 0; s < NS; ++s) w[s] = 0.f;
    } else {
      float sum = 0.f;
#pragma unroll
      for (int s = 0; s < NS; ++s) sum += __expf(ls[s] - m);
      lse = m + __logf(sum);
#pragma unroll
      for (int s = 0; s < NS; ++s) w[s] = __expf(ls[s] - lse);
    }
    for (int v = lane; v < nvec; v += lpr) {
      uint4 raw[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s)
        raw[s] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const T*>(a.O[s]) + orow) + v);
      float acc[VN];
#pragma unroll
      for (int e = 0; e < VN; ++e) acc[e] = 0.f;
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        float f[VN];
        unpack(raw[s], f, static_cast<const T*>(nullptr));
#pragma unroll
        for (int e = 0; e < VN; ++e) acc[e] = fmaf(w[s], f[e], acc[e]);
      }
      reinterpret_cast<uint4*>(static_cast<T*>(a.O_out) + orow)[v] = pack(acc, static_cast<const T*>(nullptr));
    }
    if (lane == 0) a.L_out[lrow] = lse;
  }
}

// Gradient of the merge for one row per group of lpr consecutive lanes: the row's
// weights as in merge_kernel; per 16-byte vector, O = sum_s w_s O_s, the partial
// dot products dO . (O_s - O) and the stores of w_s dO; the dot products are summed
// over the row's lanes by shuffles within the lane group.  Parts with w_s = 0 (an
// empty part, or an empty row) are skipped and get zero gradients.  The weights use
// the accurate expf / logf: dLSE_s scales with |dO| |O_s - O| d, so their error shows.
template <typename T, int NS>
__global__ void __launch_bounds__(kThreads) merge_bwd_kernel(MergeBwdArgs a, int lpr) {
  constexpr int VN = Vec<T>::n;
  const int h = blockIdx.y, b = blockIdx.z;
  const int n0 = blockIdx.x * kRowsPerCta;
  const int rows_per_pass = kThreads / lpr;
  const int sub = threadIdx.x / lpr, lane = threadIdx.x % lpr;
  const int wl = threadIdx.x & 31;
  const unsigned grp = lpr == 32 ? 0xffffffffu : (((1u << lpr) - 1u) << (wl & ~(lpr - 1)));
  const int nvec = a.d / VN;
  for (int rr = sub; rr < kRowsPerCta; rr += rows_per_pass) {
    const int n = n0 + rr;
    if (n >= a.N) break;  // the whole lane group leaves together
    const size_t lrow = ((size_t)b * a.Hh + h) * a.N + n;
    const size_t orow = (((size_t)b * a.N + n) * a.Hh + h) * (size_t)a.d;
    float ls[NS];
    float m = -INFINITY;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      ls[s] = a.L[s][lrow];
      m = fmaxf(m, ls[s]);
    }
    float w[NS];
    if (m == -INFINITY) {
#pragma unroll
      for (int s = 0; s < NS; ++s) w[s] = 0.f;
    } else {
      float sum = 0.f;
#pragma unroll
      for (int s = 0; s < NS; ++s) sum += expf(ls[s] - m);
      const float lse = m + logf(sum);
#pragma unroll
      for (int s = 0; s < NS; ++s) w[s] = expf(ls[s] - lse);
    }
    float dot[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) dot[s] = 0.f;
    for (int v = lane; v < nvec; v += lpr) {
      uint4 raw[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s)
        raw[s] = w[s] != 0.f ? __ldcs(reinterpret_cast<const uint4*>(static_cast<const T*>(a.O[s]) + orow) + v)
                             : make_uint4(0u, 0u, 0u, 0u);
      float g[VN], o[VN];
      unpack(__ldcs(reinterpret_cast<const uint4*>(static_cast<const T*>(a.dO) + orow) + v), g,
             static_cast<const T*>(nullptr));
#pragma unroll
      for (int e = 0; e < VN; ++e) o[e] = 0.f;
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        float f[VN];
        unpack(raw[s], f, static_cast<const T*>(nullptr));
#pragma unroll
        for (int e = 0; e < VN; ++e) o[e] = fmaf(w[s], f[e], o[e]);
      }
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        float f[VN], out[VN];
        unpack(raw[s], f, static_cast<const T*>(nullptr));
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < VN; ++e) {
          acc = fmaf(g[e], f[e] - o[e], acc);
          out[e] = w[s] * g[e];
        }
        if (w[s] != 0.f) dot[s] += acc;
        __stcs(reinterpret_cast<uint4*>(static_cast<T*>(a.dO_out[s]) + orow) + v, pack(out, static_cast<const T*>(nullptr)));
      }
    }
#pragma unroll
    for (int s = 0; s < NS; ++s)
      for (int off = lpr >> 1; off > 0; off >>= 1) dot[s] += __shfl_xor_sync(grp, dot[s], off);
    if (lane == 0) {
      const float gl = a.dL ? a.dL[lrow] : 0.f;
#pragma unroll
      for (int s = 0; s < NS; ++s) a.dL_out[s][lrow] = w[s] != 0.f ? w[s] * (dot[s] + gl) : 0.f;
    }
  }
}

template <typename T, int NS>
cudaError_t launch_bwd_ns(const MergeBwdArgs& a, cudaStream_t st) {
  constexpr int VN = Vec<T>::n;
  int nvec = a.d / VN;
  int lpr = 1;
  while (lpr < nvec && lpr < 32) lpr <<= 1;
  dim3 grid((a.N + kRowsPerCta - 1) / kRowsPerCta, a.Hh, a.B);
  merge_bwd_kernel<T, NS><<<grid, kThreads, 0, st>>>(a, lpr);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_t(const MergeBwdArgs& a, cudaStream_t st) {
  switch (a.n_states) {
#define SDA_CASE(n) \
  case n:           \
    return launch_bwd_ns<T, n>(a, st);
    SDA_CASE(1) SDA_CASE(2) SDA_CASE(3) SDA_CASE(4) SDA_CASE(5) SDA_CASE(6) SDA_CASE(7) SDA_CASE(8)
    SDA_CASE(9) SDA_CASE(10) SDA_CASE(11) SDA_CASE(12) SDA_CASE(13) SDA_CASE(14) SDA_CASE(15) SDA_CASE(16)
#undef SDA_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

template <typename T, int NS>
cudaError_t launch_ns(const MergeArgs& a, cudaStream_t st) {
  constexpr int VN = Vec<T>::n;
  int nvec = a.d / VN;
  int lpr = 1;
  while (lpr < nvec && lpr < 32) lpr <<= 1;
  dim3 grid((a.N + kRowsPerCta - 1) / kRowsPerCta, a.Hh, a.B);
  merge_kernel<T, NS><<<grid, kThreads, 0, st>>>(a, lpr);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const MergeArgs& a, cudaStream_t st) {
  switch (a.n_states) {
#define SDA_CASE(n) \
  case n:           \
    return launch_ns<T, n>(a, st);
    SDA_CASE(1) SDA_CASE(2) SDA_CASE(3) SDA_CASE(4) SDA_CASE(5) SDA_CASE(6) SDA_CASE(7) SDA_CASE(8)
    SDA_CASE(9) SDA_CASE(10) SDA_CASE(11) SDA_CASE(12) SDA_CASE(13) SDA_CASE(14) SDA_CASE(15) SDA_CASE(16)
#undef SDA_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, int dtype, cudaStream_t st) {
  return dtype == SDA_BF16 ? launch_t<__nv_bfloat16>(a, st) : launch_t<float>(a, st);
}

cudaError_t launch_merge_bwd(const MergeBwdArgs& a, int dtype, cudaStream_t st) {
  return dtype == SDA_BF16 ? launch_bwd_t<__nv_bfloat16>(a, st) : launch_bwd_t<float>(a, st);
}

}  // namespace sda
