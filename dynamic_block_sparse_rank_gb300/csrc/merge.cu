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
// once.  Rows of at most one 16-byte vector per lane go through the staged kernels
// (merge_async_kernel, merge_bwd_async_kernel: each thread's loads run two passes
// ahead through shared memory); wider rows through the register kernels below.  A CTA covers 64 consecutive tokens of one (batch, head): the LSE
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
// weights as in merge_kernel; per 16-byte vector, the partial dot products dO . O_s
// and the stores of w_s dO; the dot products are summed over the row's lanes by
// shuffles within the lane group, and dO . (O_s - O) = dO . O_s - sum_t w_t dO . O_t
// is formed from the sums (O itself is never built: fewer instructions per byte).  Every state's vector is
// loaded whatever its weight, so the loads of a row go out together with its LSE
// loads instead of after them.  Parts with w_s = 0 (an
// empty part, or an empty row) are skipped and get zero gradients.  The weights use
// the accurate expf / logf: dLSE_s scales with |dO| |O_s - O| d, so their error shows.
template <typename T, int NS>
__global__ void __launch_bounds__(kThreads, NS <= 4 ? 4 : 1) merge_bwd_kernel(MergeBwdArgs a, int lpr) {
  constexpr int VN = Vec<T>::n;
  const long long rows = (long long)a.B * a.N * a.Hh;
  const long long r0 = (long long)blockIdx.x * kRowsPerCta;  // rows in memory order: (b, n, h)
  const int rows_per_pass = kThreads / lpr;
  const int sub = threadIdx.x / lpr, lane = threadIdx.x % lpr;
  const int wl = threadIdx.x & 31;
  const unsigned grp = lpr == 32 ? 0xffffffffu : (((1u << lpr) - 1u) << (wl & ~(lpr - 1)));
  const int nvec = a.d / VN;
  for (int rr = sub; rr < kRowsPerCta; rr += rows_per_pass) {
    const long long r = r0 + rr;
    if (r >= rows) break;  // the whole lane group leaves together
    const int h = (int)(r % a.Hh);
    const long long bn = r / a.Hh;
    const long long n = bn % a.N, b = bn / a.N;
    const size_t lrow = ((size_t)b * a.Hh + h) * a.N + n;
    const size_t orow = (size_t)r * a.d;
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
      // loaded whatever the weight, so the loads need not wait for the LSE rows
      uint4 raw[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s) raw[s] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const T*>(a.O[s]) + orow) + v);
      float g[VN];
      unpack(__ldcs(reinterpret_cast<const uint4*>(static_cast<const T*>(a.dO) + orow) + v), g,
             static_cast<const T*>(nullptr));
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        float f[VN], out[VN];
        unpack(raw[s], f, static_cast<const T*>(nullptr));
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < VN; ++e) {
          acc = fmaf(g[e], f[e], acc);
          out[e] = w[s] * g[e];
        }
        if (w[s] != 0.f) dot[s] += acc;  // an empty part's stored values never enter
        reinterpret_cast<uint4*>(static_cast<T*>(a.dO_out[s]) + orow)[v] = pack(out, static_cast<const T*>(nullptr));
      }
    }
#pragma unroll
    for (int s = 0; s < NS; ++s)
      for (int off = lpr >> 1; off > 0; off >>= 1) dot[s] += __shfl_xor_sync(grp, dot[s], off);
    if (lane == 0) {
      const float gl = a.dL ? a.dL[lrow] : 0.f;
      float go = 0.f;  // dO . O = sum_s w_s dO . O_s
#pragma unroll
      for (int s = 0; s < NS; ++s) go = fmaf(w[s], dot[s], go);
#pragma unroll
      for (int s = 0; s < NS; ++s) a.dL_out[s][lrow] = w[s] != 0.f ? w[s] * (dot[s] - go + gl) : 0.f;
    }
  }
}

// The same gradient with the row data staged through shared memory by cp.async, for
// rows of at most one 16-byte vector per lane (d * size(T) <= 512).  Each thread
// copies its own vector of every state and of dO for the pass kAhead passes ahead and
// later reads back only what it copied, so it waits on its own copy groups and no
// CTA barrier is needed; the LSE rows of the next pass are loaded a pass early.
// Keeps (kAhead + 1) passes of loads in flight instead of one.
constexpr int kPasses = 16;  // passes of kThreads / lpr rows per CTA
constexpr int kAhead = 2;   // stage slots

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T, int NS>
__global__ void __launch_bounds__(kThreads, NS <= 4 ? 4 : 1) merge_bwd_async_kernel(MergeBwdArgs a, int lpr) {
  constexpr int VN = Vec<T>::n;
  extern __shared__ uint4 stage[];  // [kAhead][NS + 1][kThreads]
  const long long rows = (long long)a.B * a.N * a.Hh;
  const int rpp = kThreads / lpr;  // rows per pass
  const long long r0 = (long long)blockIdx.x * kPasses * rpp;
  const int tid = threadIdx.x, sub = tid / lpr, lane = tid % lpr;
  const int wl = tid & 31;
  const unsigned grp = lpr == 32 ? 0xffffffffu : (((1u << lpr) - 1u) << (wl & ~(lpr - 1)));
  const bool has_vec = lane < a.d / VN;
  auto row_of = [&](int pass) { return r0 + (long long)pass * rpp + sub; };
  // (b, n, h) of this lane group's row, divided out once and then advanced by rpp rows
  // per pass with carries (memory order (b, n, h)): the LSE index needs no division
  // per pass.
  int hh, bb;
  long long nn;
  {
    const long long r = row_of(0);
    hh = (int)(r % a.Hh);
    const long long bn = r / a.Hh;
    nn = bn % a.N;
    bb = (int)(bn / a.N);
  }
  auto advance = [&]() {
    hh += rpp;
    if (hh >= a.Hh) {
      const int q = hh / a.Hh;
      hh -= q * a.Hh;
      nn += q;
      if (nn >= a.N) {
        bb += (int)(nn / a.N);
        nn %= a.N;
      }
    }
  };
  auto lse_index = [&]() { return ((long long)bb * a.Hh + hh) * a.N + nn; };
  auto issue = [&](int pass) {  // always commits a group, so group counting stays uniform
    const long long r = row_of(pass);
    if (pass < kPasses && r < rows && has_vec) {
      uint4* slot = stage + (size_t)(pass % kAhead) * (NS + 1) * kThreads;
#pragma unroll
      for (int s = 0; s < NS; ++s)
        cp_async16(slot + s * kThreads + tid, static_cast<const T*>(a.O[s]) + (size_t)r * a.d + lane * VN);
      cp_async16(slot + NS * kThreads + tid, static_cast<const T*>(a.dO) + (size_t)r * a.d + lane * VN);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int q = 0; q < kAhead; ++q) issue(q);
  float ls_next[NS], gl_next = 0.f;
  long long lr_next;  // LSE index of the row the next pass handles
  {
    const long long r = row_of(0);
    lr_next = r < rows ? lse_index() : 0;
#pragma unroll
    for (int s = 0; s < NS; ++s) ls_next[s] = r < rows ? a.L[s][lr_next] : -INFINITY;
    if (a.dL && r < rows) gl_next = a.dL[lr_next];
  }
  for (int pass = 0; pass < kPasses; ++pass) {
    const long long r = row_of(pass);
    const bool valid = r < rows;  // the same on the lane group's lanes
    float ls[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) ls[s] = ls_next[s];
    const float gl = gl_next;
    const long long lr = lr_next;
    {  // the next pass's LSE rows, a pass early
      const long long r2 = row_of(pass + 1);
      const bool v2 = pass + 1 < kPasses && r2 < rows;
      advance();
      lr_next = v2 ? lse_index() : 0;
#pragma unroll
      for (int s = 0; s < NS; ++s) ls_next[s] = v2 ? a.L[s][lr_next] : -INFINITY;
      gl_next = (a.dL && v2) ? a.dL[lr_next] : 0.f;
    }
    float m = -INFINITY;
#pragma unroll
    for (int s = 0; s < NS; ++s) m = fmaxf(m, ls[s]);
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
    cp_async_wait<kAhead - 1>();  // this pass's group (and every older one) has landed
    float dot[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) dot[s] = 0.f;
    if (valid && has_vec) {
      // dot[s] = this lane's share of dO . O_s; dO . O = sum_s w_s dO . O_s is formed
      // after the row reduction, so O itself is never built
      const uint4* slot = stage + (size_t)(pass % kAhead) * (NS + 1) * kThreads;
      float g[VN];
      unpack(slot[NS * kThreads + tid], g, static_cast<const T*>(nullptr));
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        float f[VN], out[VN];
        unpack(slot[s * kThreads + tid], f, static_cast<const T*>(nullptr));
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < VN; ++e) {
          acc = fmaf(g[e], f[e], acc);
          out[e] = w[s] * g[e];
        }
        if (w[s] != 0.f) dot[s] = acc;  // an empty part's stored values never enter
        reinterpret_cast<uint4*>(static_cast<T*>(a.dO_out[s]) + (size_t)r * a.d)[lane] =
            pack(out, static_cast<const T*>(nullptr));
      }
    }
    issue(pass + kAhead);  // the slot just read takes the pass kAhead ahead
    if (valid) {
#pragma unroll
      for (int s = 0; s < NS; ++s)
        for (int off = lpr >> 1; off > 0; off >>= 1) dot[s] += __shfl_xor_sync(grp, dot[s], off);
      if (lane == 0) {
        float go = 0.f;  // dO . O
#pragma unroll
        for (int s = 0; s < NS; ++s) go = fmaf(w[s], dot[s], go);
#pragma unroll
        for (int s = 0; s < NS; ++s) a.dL_out[s][lr] = w[s] != 0.f ? w[s] * (dot[s] - go + gl) : 0.f;
      }
    }
  }
  cp_async_wait<0>();
}

// The merge itself, staged the same way (rows of at most one 16-byte vector per lane).
// In place is safe: a row's data is staged before that row is written, and no write
// touches a row still to be staged.
template <typename T, int NS>
__global__ void __launch_bounds__(kThreads, NS <= 4 ? 4 : 1) merge_async_kernel(MergeArgs a, int lpr) {
  constexpr int VN = Vec<T>::n;
  extern __shared__ uint4 stage[];  // [kAhead][NS][kThreads]
  const long long rows = (long long)a.B * a.N * a.Hh;
  const int rpp = kThreads / lpr;
  const long long r0 = (long long)blockIdx.x * kPasses * rpp;
  const int tid = threadIdx.x, sub = tid / lpr, lane = tid % lpr;
  const bool has_vec = lane < a.d / VN;
  auto row_of = [&](int pass) { return r0 + (long long)pass * rpp + sub; };
  int hh, bb;
  long long nn;
  {
    const long long r = row_of(0);
    hh = (int)(r % a.Hh);
    const long long bn = r / a.Hh;
    nn = bn % a.N;
    bb = (int)(bn / a.N);
  }
  auto advance = [&]() {
    hh += rpp;
    if (hh >= a.Hh) {
      const int q = hh / a.Hh;
      hh -= q * a.Hh;
      nn += q;
      if (nn >= a.N) {
        bb += (int)(nn / a.N);
        nn %= a.N;
      }
    }
  };
  auto lse_index = [&]() { return ((long long)bb * a.Hh + hh) * a.N + nn; };
  auto issue = [&](int pass) {
    const long long r = row_of(pass);
    if (pass < kPasses && r < rows && has_vec) {
      uint4* slot = stage + (size_t)(pass % kAhead) * NS * kThreads;
#pragma unroll
      for (int s = 0; s < NS; ++s)
        cp_async16(slot + s * kThreads + tid, static_cast<const T*>(a.O[s]) + (size_t)r * a.d + lane * VN);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int q = 0; q < kAhead; ++q) issue(q);
  float ls_next[NS];
  long long lr_next;
  {
    const long long r = row_of(0);
    lr_next = r < rows ? lse_index() : 0;
#pragma unroll
    for (int s = 0; s < NS; ++s) ls_next[s] = r < rows ? a.L[s][lr_next] : -INFINITY;
  }
  for (int pass = 0; pass < kPasses; ++pass) {
    const long long r = row_of(pass);
    const bool valid = r < rows;
    float ls[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) ls[s] = ls_next[s];
    const long long lr = lr_next;
    {
      const long long r2 = row_of(pass + 1);
      const bool v2 = pass + 1 < kPasses && r2 < rows;
      advance();
      lr_next = v2 ? lse_index() : 0;
#pragma unroll
      for (int s = 0; s < NS; ++s) ls_next[s] = v2 ? a.L[s][lr_next] : -INFINITY;
    }
    float m = -INFINITY;
#pragma unroll
    for (int s = 0; s < NS; ++s) m = fmaxf(m, ls[s]);
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
    cp_async_wait<kAhead - 1>();
    if (valid && has_vec) {
      const uint4* slot = stage + (size_t)(pass % kAhead) * NS * kThreads;
      float acc[VN];
#pragma unroll
      for (int e = 0; e < VN; ++e) acc[e] = 0.f;
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        float f[VN];
        unpack(slot[s * kThreads + tid], f, static_cast<const T*>(nullptr));
#pragma unroll
        for (int e = 0; e < VN; ++e) acc[e] = fmaf(w[s], f[e], acc[e]);
      }
      reinterpret_cast<uint4*>(static_cast<T*>(a.O_out) + (size_t)r * a.d)[lane] = pack(acc, static_cast<const T*>(nullptr));
    }
    issue(pass + kAhead);
    if (valid && lane == 0) a.L_out[lr] = lse;
  }
  cp_async_wait<0>();
}

template <typename T, int NS>
cudaError_t launch_bwd_ns(const MergeBwdArgs& a, cudaStream_t st) {
  constexpr int VN = Vec<T>::n;
  int nvec = a.d / VN;
  int lpr = 1;
  while (lpr < nvec && lpr < 32) lpr <<= 1;
  const long long rows = (long long)a.B * a.N * a.Hh;
  if (nvec <= lpr) {  // one vector per lane: the staged kernel
    const size_t smem = (size_t)kAhead * (NS + 1) * kThreads * sizeof(uint4);
    cudaError_t e = cudaFuncSetAttribute(merge_bwd_async_kernel<T, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const long long per_cta = (long long)kPasses * (kThreads / lpr);
    merge_bwd_async_kernel<T, NS><<<(unsigned)((rows + per_cta - 1) / per_cta), kThreads, smem, st>>>(a, lpr);
  } else {
    merge_bwd_kernel<T, NS><<<(unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta), kThreads, 0, st>>>(a, lpr);
  }
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
  if (nvec <= lpr) {  // one vector per lane: the staged kernel
    const size_t smem = (size_t)kAhead * NS * kThreads * sizeof(uint4);
    cudaError_t e =
        cudaFuncSetAttribute(merge_async_kernel<T, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long rows = (long long)a.B * a.N * a.Hh;
    const long long per_cta = (long long)kPasses * (kThreads / lpr);
    merge_async_kernel<T, NS><<<(unsigned)((rows + per_cta - 1) / per_cta), kThreads, smem, st>>>(a, lpr);
  } else {
    dim3 grid((a.N + kRowsPerCta - 1) / kRowsPerCta, a.Hh, a.B);
    merge_kernel<T, NS><<<grid, kThreads, 0, st>>>(a, lpr);
  }
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
