// C-ABI entry points: argument validation, workspace sizing and dispatch to
// the fp32 (CUDA-core) or bf16 (tensor-core) kernels.  No entry point
// allocates memory; none synchronises except sda_get_device_status.
#include <math.h>

#include "internal.h"

using namespace sda;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validate a problem and derive sizes.  Returns SDA_OK or the error to report.
sda_status make_prob(const sda_problem* pp, Prob* out) {
  if (!pp || !out) return SDA_ERR_INVALID_ARG;
  const sda_problem& p = *pp;
  if (p.B < 1 || p.heads < 1 || p.T < 1 || p.H < 1 || p.W < 1 || p.head_dim < 1) return SDA_ERR_INVALID_ARG;
  if (p.bt < 1 || p.bh < 1 || p.bw < 1 || p.rank < 1) return SDA_ERR_INVALID_ARG;
  if (!(p.keep_ratio > 0.0) || !isfinite(p.keep_ratio)) return SDA_ERR_INVALID_ARG;
  if (p.dtype != SDA_F32 && p.dtype != SDA_BF16) return SDA_ERR_INVALID_ARG;
  if (!(p.softmax_scale >= 0.f) || !isfinite(p.softmax_scale)) return SDA_ERR_INVALID_ARG;
  Prob q;
  q.g.T = p.T;
  q.g.H = p.H;
  q.g.W = p.W;
  q.g.bt = p.bt;
  q.g.bh = p.bh;
  q.g.bw = p.bw;
  q.g.nT = (p.T + p.bt - 1) / p.bt;
  q.g.nH = (p.H + p.bh - 1) / p.bh;
  q.g.nW = (p.W + p.bw - 1) / p.bw;
  long long nb = (long long)q.g.nT * q.g.nH * q.g.nW;
  long long bs = (long long)p.bt * p.bh * p.bw;
  q.N = (long long)p.T * p.H * p.W;
  if (nb > (1 << 20) || bs > (1 << 20) || q.N > (1LL << 31) - 1) return SDA_ERR_UNSUPPORTED;
  q.g.nb = (int)nb;
  q.g.bs = (int)bs;
  q.B = p.B;
  q.Hh = p.heads;
  q.d = p.head_dim;
  q.r = p.rank;
  q.dtype = p.dtype;
  q.scale = p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)p.head_dim);
  // Two roundings, as plain double arithmetic does them: the product is stored
  // through a volatile so that no compiler fuses it with the sum into an FMA
  // (aarch64 compilers contract by default), which could move k by one.
  volatile double kprod = p.keep_ratio * (double)nb;
  const double kval = floor(kprod + 1e-9);
  long long k = kval > (double)nb ? nb : (long long)kval;
  if (k < 1) k = 1;
  if (k > nb) k = nb;
  q.k = (int)k;
  *out = q;
  return SDA_OK;
}

// Which kernels cover the problem.
sda_status check_supported(const Prob& q) {
  if (q.g.nb > 8192) return SDA_ERR_UNSUPPORTED;  // score row of a query block lives in shared memory
  if (q.dtype == SDA_BF16) {
    if (q.g.bs != 128) return SDA_ERR_UNSUPPORTED;
    if (q.d != 64 && q.d != 128) return SDA_ERR_UNSUPPORTED;
    if (q.r % 16 != 0 || q.r > 64) return SDA_ERR_UNSUPPORTED;
    if (q.k > 4096) return SDA_ERR_UNSUPPORTED;
  } else {
    if (q.g.bs > 1024 || q.d > 128 || q.r > 64) return SDA_ERR_UNSUPPORTED;
    if ((size_t)(q.g.bs * q.r + q.g.nb) * 4 > 160 * 1024) return SDA_ERR_UNSUPPORTED;
  }
  return SDA_OK;
}

sda_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SDA_OK : SDA_ERR_CUDA; }

}  // namespace

extern "C" {

const char* sda_status_string(sda_status s) {
  switch (s) {
    case SDA_OK:
      return "ok";
    case SDA_ERR_INVALID_ARG:
      return "invalid argument";
    case SDA_ERR_UNSUPPORTED:
      return "unsupported problem";
    case SDA_ERR_WORKSPACE:
      return "workspace too small";
    case SDA_ERR_CUDA:
      return "CUDA error";
    case SDA_ERR_DEVICE_TIMEOUT:
      return "device wait timed out";
    case SDA_ERR_DEVICE_BAD_INDEX:
      return "block index out of range or repeated";
    case SDA_ERR_DEVICE_RANGE:
      return "input value outside fp16 range";
  }
  return "unknown status";
}

sda_status sda_num_blocks(const sda_problem* p, int* n_blocks, int* k) {
  Prob q;
  sda_status s = make_prob(p, &q);
  if (s != SDA_OK) return s;
  if (n_blocks) *n_blocks = q.g.nb;
  if (k) *k = q.k;
  return SDA_OK;
}

sda_status sda_workspace_size(const sda_problem* p, int op, size_t* bytes) {
  Prob q;
  sda_status s = make_prob(p, &q);
  if (s != SDA_OK) return s;
  if (!bytes) return SDA_ERR_INVALID_ARG;
  if ((s = check_supported(q)) != SDA_OK) return s;
  if (op == SDA_OP_PREDICT)
    *bytes = q.dtype == SDA_BF16 ? predict_ws_tc(q) : predict_ws_f32(q);
  else if (op == SDA_OP_BWD)
    *bytes = q.dtype == SDA_BF16 ? bwd_ws_tc(q) : bwd_ws_f32(q);
  else if (op == SDA_OP_TRAIN) {
    if (q.dtype != SDA_BF16) return SDA_ERR_UNSUPPORTED;
    *bytes = train_ws_tc(q);
  } else if (op == SDA_OP_PREDICTOR_GRAD) {
    if (q.dtype != SDA_BF16) return SDA_ERR_UNSUPPORTED;
    *bytes = distill_ws_tc(q);
  } else
    return SDA_ERR_INVALID_ARG;
  return SDA_OK;
}

sda_status sda_predict_blocks(const sda_problem* p, const void* Q, const void* K, const void* Wq, const void* Wk,
                              int32_t* block_idx, float* block_score, void* ws, size_t ws_bytes, void* stream) {
  Prob q;
  sda_status s = make_prob(p, &q);
  if (s != SDA_OK) return s;
  if (!Q || !K || !Wq || !Wk || !block_idx || !ws) return SDA_ERR_INVALID_ARG;
  if ((s = check_supported(q)) != SDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q.dtype == SDA_BF16) {
    if (!aligned16(Q) || !aligned16(K) || !aligned16(Wq) || !aligned16(Wk) || !aligned16(ws))
      return SDA_ERR_INVALID_ARG;
    if (ws_bytes < predict_ws_tc(q)) return SDA_ERR_WORKSPACE;
    return from_cuda(predict_tc(q, Q, K, Wq, Wk, block_idx, block_score, ws, st));
  }
  if (ws_bytes < predict_ws_f32(q)) return SDA_ERR_WORKSPACE;
  return from_cuda(predict_f32(q, static_cast<const float*>(Q), static_cast<const float*>(K),
                               static_cast<const float*>(Wq), static_cast<const float*>(Wk), block_idx, block_score,
                               ws, st));
}

sda_status sda_predictor_grad(const sda_problem* p, const void* Q, const void* K, const void* Wq, const void* Wk,
                              float* dWq, float* dWk, double* loss, float* s_out, float* t_out, void* ws,
                              size_t ws_bytes, void* stream) {
  Prob q;
  sda_status s = make_prob(p, &q);
  if (s != SDA_OK) return s;
  if (!Q || !K || !Wq || !Wk || !dWq || !dWk || !loss || !ws) return SDA_ERR_INVALID_ARG;
  if ((s = check_supported(q)) != SDA_OK) return s;
  if (q.dtype != SDA_BF16) return SDA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(Wq) || !aligned16(Wk) || !aligned16(ws)) return SDA_ERR_INVALID_ARG;
  if (ws_bytes < distill_ws_tc(q)) return SDA_ERR_WORKSPACE;
  return from_cuda(distill_tc(q, Q, K, Wq, Wk, dWq, dWk, loss, s_out, t_out, ws, static_cast<cudaStream_t>(stream)));
}

sda_status sda_attn_fwd(const sda_problem* p, const void* Q, const void* K, const void* V, const int32_t* block_idx,
                        int kb_begin, int kb_end, const uint8_t* qb_active, void* O, float* LSE, int out_dtype,
                        void* stream) {
  Prob q;
  sda_status s = make_prob(p, &q);
  if (s != SDA_OK) return s;
  if (!Q || !K || !V || !block_idx || !O || !LSE) return SDA_ERR_INVALID_ARG;
  if (kb_begin < 0 || kb_end < kb_begin || kb_end > q.g.nb) return SDA_ERR_INVALID_ARG;
  if (out_dtype != SDA_F32 && out_dtype != q.dtype) return SDA_ERR_INVALID_ARG;
  if ((s = check_supported(q)) != SDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q.dtype == SDA_BF16) {
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SDA_ERR_INVALID_ARG;
    return from_cuda(fwd_tc(q, Q, K, V, block_idx, kb_begin, kb_end, qb_active, O, out_dtype == SDA_F32, LSE, st));
  }
  return from_cuda(fwd_f32(q, static_cast<const float*>(Q), static_cast<const float*>(K),
                           static_cast<const float*>(V), block_idx, kb_begin, kb_end, qb_active,
                           static_cast<float*>(O), LSE, st));
}

namespace {
// Shared argument checks of the backward entry points.
// ptrs[0 .. n_tensors) are token tensors (16-byte alignment on the tensor-core
// path); the rest (LSE, block_idx) only need to be non-null.
sda_status bwd_common(const sda_problem* p, Prob* q, const void* const* ptrs, int nptrs, int n_tensors, int grad_dtype,
                      void* ws, size_t ws_bytes) {
  sda_status s = make_prob(p, q);
  if (s != SDA_OK) return s;
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i]) return SDA_ERR_INVALID_ARG;
  if (!ws) return SDA_ERR_INVALID_ARG;
  if (grad_dtype != SDA_F32 && grad_dtype != q->dtype) return SDA_ERR_INVALID_ARG;
  if ((s = check_supported(*q)) != SDA_OK) return s;
  if (q->dtype == SDA_BF16) {
    for (int i = 0; i < n_tensors; ++i)
      if (!aligned16(ptrs[i])) return SDA_ERR_INVALID_ARG;
    if (!aligned16(ws)) return SDA_ERR_INVALID_ARG;
    if (ws_bytes < bwd_ws_tc(*q)) return SDA_ERR_WORKSPACE;
  } else if (ws_bytes < bwd_ws_f32(*q)) {
    return SDA_ERR_WORKSPACE;
  }
  return SDA_OK;
}
}  // namespace

sda_status sda_attn_bwd_prepare(const sda_problem* p, const void* Q, const void* K, const void* V, const void* O,
                                const float* LSE, const void* dO, const int32_t* block_idx, void* ws,
                                size_t ws_bytes, void* stream) {
  Prob q;
  const void* ptrs[] = {Q, K, V, O, dO, LSE, block_idx};
  sda_status s = bwd_common(p, &q, ptrs, 7, 5, p ? p->dtype : SDA_F32, ws, ws_bytes);
  if (s != SDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q.dtype == SDA_BF16) return from_cuda(bwd_prepare_tc(q, Q, K, V, O, LSE, dO, block_idx, ws, st));
  return from_cuda(bwd_prepare_f32(q, static_cast<const float*>(O), static_cast<const float*>(dO), ws, st));
}

sda_status sda_attn_bwd_dq(const sda_problem* p, const void* Q, const void* K, const void* V, const float* LSE,
                           const void* dO, const int32_t* block_idx, void* dQ, int grad_dtype, void* ws,
                           size_t ws_bytes, void* stream) {
  Prob q;
  const void* ptrs[] = {Q, K, V, dO, dQ, LSE, block_idx};
  sda_status s = bwd_common(p, &q, ptrs, 7, 5, grad_dtype, ws, ws_bytes);
  if (s != SDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q.dtype == SDA_BF16) return from_cuda(bwd_dq_tc(q, V, dO, block_idx, dQ, grad_dtype, ws, st));
  return from_cuda(bwd_dq_f32(q, static_cast<const float*>(Q), static_cast<const float*>(K),
                              static_cast<const float*>(V), LSE, static_cast<const float*>(dO), block_idx,
                              static_cast<float*>(dQ), ws, st));
}

sda_status sda_attn_bwd_dkdv(const sda_problem* p, const void* Q, const void* K, const void* V, const float* LSE,
                             const void* dO, const int32_t* block_idx, void* dK, void* dV, int grad_dtype, void* ws,
                             size_t ws_bytes, void* stream) {
  Prob q;
  const void* ptrs[] = {Q, K, V, dO, dK, dV, LSE, block_idx};
  sda_status s = bwd_common(p, &q, ptrs, 8, 6, grad_dtype, ws, ws_bytes);
  if (s != SDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q.dtype == SDA_BF16) return from_cuda(bwd_dkdv_tc(q, V, dO, dK, dV, grad_dtype, ws, st));
  return from_cuda(bwd_dkdv_f32(q, static_cast<const float*>(Q), static_cast<const float*>(K),
                                static_cast<const float*>(V), LSE, static_cast<const float*>(dO), block_idx,
                                static_cast<float*>(dK), static_cast<float*>(dV), ws, st));
}

sda_status sda_attn_bwd(const sda_problem* p, const void* Q, const void* K, const void* V, const void* O,
                        const float* LSE, const void* dO, const int32_t* block_idx, void* dQ, void* dK, void* dV,
                        int grad_dtype, void* ws, size_t ws_bytes, void* stream) {
  Prob q;
  const void* ptrs[] = {Q, K, V, O, dO, dQ, dK, dV, LSE, block_idx};
  sda_status s = bwd_common(p, &q, ptrs, 10, 8, grad_dtype, ws, ws_bytes);
  if (s != SDA_OK) return s;
  if ((s = sda_attn_bwd_prepare(p, Q, K, V, O, LSE, dO, block_idx, ws, ws_bytes, stream)) != SDA_OK) return s;
  if ((s = sda_attn_bwd_dq(p, Q, K, V, LSE, dO, block_idx, dQ, grad_dtype, ws, ws_bytes, stream)) != SDA_OK)
    return s;
  return sda_attn_bwd_dkdv(p, Q, K, V, LSE, dO, block_idx, dK, dV, grad_dtype, ws, ws_bytes, stream);
}

sda_status sda_attn_fwd_train(const sda_problem* p, const void* Q, const void* K, const void* V,
                              const int32_t* block_idx, void* O, float* LSE, void* ws, size_t ws_bytes,
                              void* stream) {
  Prob q;
  sda_status s = make_prob(p, &q);
  if (s != SDA_OK) return s;
  if (!Q || !K || !V || !block_idx || !O || !LSE || !ws) return SDA_ERR_INVALID_ARG;
  if ((s = check_supported(q)) != SDA_OK) return s;
  if (q.dtype != SDA_BF16) return SDA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(ws)) return SDA_ERR_INVALID_ARG;
  if (ws_bytes < train_ws_tc(q)) return SDA_ERR_WORKSPACE;
  return from_cuda(fwd_train_tc(q, Q, K, V, block_idx, O, LSE, ws, static_cast<cudaStream_t>(stream)));
}

sda_status sda_attn_bwd_train(const sda_problem* p, const float* LSE, const void* dO, const int32_t* block_idx,
                              void* dQ, void* dK, void* dV, int grad_dtype, int phases, void* ws, size_t ws_bytes,
                              void* stream) {
  Prob q;
  sda_status s = make_prob(p, &q);
  if (s != SDA_OK) return s;
  if (!LSE || !dO || !block_idx || !ws) return SDA_ERR_INVALID_ARG;
  if (phases < 1 || phases > 7) return SDA_ERR_INVALID_ARG;
  if (((phases & 2) && !dQ) || ((phases & 4) && (!dK || !dV))) return SDA_ERR_INVALID_ARG;
  if ((s = check_supported(q)) != SDA_OK) return s;
  if (q.dtype != SDA_BF16) return SDA_ERR_UNSUPPORTED;
  if (grad_dtype != SDA_F32 && grad_dtype != q.dtype) return SDA_ERR_INVALID_ARG;
  if (!aligned16(dO) || !aligned16(ws) || (dQ && !aligned16(dQ)) || (dK && !aligned16(dK)) || (dV && !aligned16(dV)))
    return SDA_ERR_INVALID_ARG;
  if (ws_bytes < train_ws_tc(q)) return SDA_ERR_WORKSPACE;
  return from_cuda(bwd_train_tc(q, LSE, dO, block_idx, dQ, dK, dV, grad_dtype, ws, phases,
                                static_cast<cudaStream_t>(stream)));
}

sda_status sda_attn_bwd_partition(const sda_problem* p, const void* Q, const void* K, const void* V, const void* O,
                                  const float* LSE, const void* dO, const float* dLSE, const int32_t* block_idx,
                                  int kb_begin, int kb_end, const uint8_t* qb_active, void* dQ, void* dK, void* dV,
                                  int grad_dtype, void* ws, size_t ws_bytes, void* stream) {
  Prob q;
  const void* ptrs[] = {Q, K, V, O, dO, dQ, dK, dV, LSE, block_idx};
  sda_status s = bwd_common(p, &q, ptrs, 10, 8, grad_dtype, ws, ws_bytes);
  if (s != SDA_OK) return s;
  if (kb_begin < 0 || kb_end < kb_begin || kb_end > q.g.nb) return SDA_ERR_INVALID_ARG;
  const Part part{kb_begin, kb_end, qb_active, dLSE};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (q.dtype == SDA_BF16) {
    if ((e = bwd_prepare_tc(q, Q, K, V, O, LSE, dO, block_idx, ws, st, &part)) != cudaSuccess) return from_cuda(e);
    if ((e = bwd_dq_tc(q, V, dO, block_idx, dQ, grad_dtype, ws, st, &part)) != cudaSuccess) return from_cuda(e);
    return from_cuda(bwd_dkdv_tc(q, V, dO, dK, dV, grad_dtype, ws, st));
  }
  const float *Qf = static_cast<const float*>(Q), *Kf = static_cast<const float*>(K),
              *Vf = static_cast<const float*>(V), *dOf = static_cast<const float*>(dO);
  if ((e = bwd_prepare_f32(q, static_cast<const float*>(O), dOf, ws, st, dLSE)) != cudaSuccess) return from_cuda(e);
  if ((e = bwd_dq_f32(q, Qf, Kf, Vf, LSE, dOf, block_idx, static_cast<float*>(dQ), ws, st, &part)) != cudaSuccess)
    return from_cuda(e);
  return from_cuda(bwd_dkdv_f32(q, Qf, Kf, Vf, LSE, dOf, block_idx, static_cast<float*>(dK), static_cast<float*>(dV),
                                ws, st, &part));
}

sda_status sda_merge_states(int n_states, const void* const* O_parts, const float* const* LSE_parts, int B, int N,
                            int heads, int head_dim, int dtype, void* O_out, float* LSE_out, void* stream) {
  if (n_states < 1 || n_states > kMaxStates || !O_parts || !LSE_parts || !O_out || !LSE_out)
    return SDA_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || heads < 1 || head_dim < 1) return SDA_ERR_INVALID_ARG;
  if (dtype != SDA_F32 && dtype != SDA_BF16) return SDA_ERR_INVALID_ARG;
  const int es = dtype == SDA_BF16 ? 2 : 4;
  if ((head_dim * es) % 16 != 0 || head_dim * es > 16 * 32 * 8) return SDA_ERR_UNSUPPORTED;
  MergeArgs a;
  for (int s = 0; s < n_states; ++s) {
    if (!O_parts[s] || !LSE_parts[s] || !aligned16(O_parts[s])) return SDA_ERR_INVALID_ARG;
    a.O[s] = O_parts[s];
    a.L[s] = LSE_parts[s];
  }
  if (!aligned16(O_out)) return SDA_ERR_INVALID_ARG;
  a.n_states = n_states;
  a.B = B;
  a.N = N;
  a.Hh = heads;
  a.d = head_dim;
  a.O_out = O_out;
  a.L_out = LSE_out;
  return from_cuda(launch_merge(a, dtype, static_cast<cudaStream_t>(stream)));
}

sda_status sda_merge_states_bwd(int n_states, const void* const* O_parts, const float* const* LSE_parts,
                                const void* dO, const float* dLSE, int B, int N, int heads, int head_dim,
                                int dtype, void* const* dO_parts, float* const* dLSE_parts, void* stream) {
  if (n_states < 1 || n_states > kMaxStates || !O_parts || !LSE_parts || !dO || !dO_parts || !dLSE_parts)
    return SDA_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || heads < 1 || head_dim < 1) return SDA_ERR_INVALID_ARG;
  if (dtype != SDA_F32 && dtype != SDA_BF16) return SDA_ERR_INVALID_ARG;
  const int es = dtype == SDA_BF16 ? 2 : 4;
  if ((head_dim * es) % 16 != 0 || head_dim * es > 16 * 32 * 8) return SDA_ERR_UNSUPPORTED;
  if (!aligned16(dO)) return SDA_ERR_INVALID_ARG;
  MergeBwdArgs a;
  for (int s = 0; s < n_states; ++s) {
    if (!O_parts[s] || !LSE_parts[s] || !dO_parts[s] || !dLSE_parts[s]) return SDA_ERR_INVALID_ARG;
    if (!aligned16(O_parts[s]) || !aligned16(dO_parts[s])) return SDA_ERR_INVALID_ARG;
    a.O[s] = O_parts[s];
    a.L[s] = LSE_parts[s];
    a.dO_out[s] = dO_parts[s];
    a.dL_out[s] = dLSE_parts[s];
  }
  a.dO = dO;
  a.dL = dLSE;
  a.n_states = n_states;
  a.B = B;
  a.N = N;
  a.Hh = heads;
  a.d = head_dim;
  return from_cuda(launch_merge_bwd(a, dtype, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ------------------------------------------------------------ 3D deformable sliding attention
static sda_status dsa3d_args(const sda_dsa3d_problem* p, sda::Dsa3dArgs& a) {
  if (!p) return SDA_ERR_INVALID_ARG;
  if (p->B < 1 || p->T < 1 || p->H < 1 || p->W < 1 || p->heads < 1 || p->d < 1) return SDA_ERR_INVALID_ARG;
  if (p->kt < 1 || p->kh < 1 || p->kw < 1 || p->kt % 2 == 0 || p->kh % 2 == 0 || p->kw % 2 == 0)
    return SDA_ERR_INVALID_ARG;
  const long long N = (long long)p->T * p->H * p->W;
  if (N > 0x7fffffffLL || N * p->heads * (long long)p->d * p->B > (1LL << 40)) return SDA_ERR_INVALID_ARG;
  const long long S = (long long)p->kt * p->kh * p->kw;
  if (p->d != 64 && p->d != 128) return SDA_ERR_UNSUPPORTED;
  if (S > 125) return SDA_ERR_UNSUPPORTED;
  if (p->heads > 65535 || p->B > 65535) return SDA_ERR_UNSUPPORTED;
  a.B = p->B;
  a.T = p->T;
  a.H = p->H;
  a.W = p->W;
  a.heads = p->heads;
  a.d = p->d;
  a.kt = p->kt;
  a.kh = p->kh;
  a.kw = p->kw;
  a.S = (int)S;
  a.scale = p->scale > 0.f ? p->scale : (float)(1.0 / sqrt((double)p->d));
  return SDA_OK;
}

sda_status sda_dsa3d_offsets(const sda_dsa3d_problem* p, const void* Q, const float* Wc, const float* bc,
                             const float* Wl, const float* bl, float* offsets, void* stream) {
  sda::Dsa3dArgs a;
  const sda_status st = dsa3d_args(p, a);
  if (st != SDA_OK) return st;
  if (!Q || !Wc || !bc || !Wl || !bl || !offsets || !aligned16(Q)) return SDA_ERR_INVALID_ARG;
  return from_cuda(sda::dsa3d_offsets(a, Q, Wc, bc, Wl, bl, offsets, static_cast<cudaStream_t>(stream)));
}

sda_status sda_dsa3d_fwd(const sda_dsa3d_problem* p, const void* Q, const void* K, const void* V,
                         const float* offsets, void* O, float* LSE, void* stream) {
  sda::Dsa3dArgs a;
  const sda_status st = dsa3d_args(p, a);
  if (st != SDA_OK) return st;
  if (!Q || !K || !V || !offsets || !O || !LSE) return SDA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SDA_ERR_INVALID_ARG;
  return from_cuda(sda::dsa3d_fwd(a, Q, K, V, offsets, O, LSE, static_cast<cudaStream_t>(stream)));
}

// The window attention's backward buckets its samples with 32-bit indices.
static sda_status dsa3d_bwd_args(const sda_dsa3d_problem* p, sda::Dsa3dArgs& a) {
  const sda_status st = dsa3d_args(p, a);
  if (st != SDA_OK) return st;
  const long long N = (long long)a.T * a.H * a.W;
  if (N * a.S > 0x7fffffffLL || (long long)(a.T + 1) * (a.H + 1) * (a.W + 1) >= 0x7fffffffLL)
    return SDA_ERR_UNSUPPORTED;
  return SDA_OK;
}

sda_status sda_dsa3d_bwd_workspace_size(const sda_dsa3d_problem* p, size_t* bytes) {
  sda::Dsa3dArgs a;
  const sda_status st = dsa3d_bwd_args(p, a);
  if (st != SDA_OK) return st;
  if (!bytes) return SDA_ERR_INVALID_ARG;
  *bytes = sda::dsa3d_bwd_ws_bytes(a);
  return SDA_OK;
}

sda_status sda_dsa3d_bwd(const sda_dsa3d_problem* p, const void* Q, const void* K, const void* V,
                         const float* offsets, const float* LSE, const void* dO, float* dQ, float* dK, float* dV,
                         float* d_offsets, void* ws, size_t ws_bytes, void* stream) {
  sda::Dsa3dArgs a;
  const sda_status st = dsa3d_bwd_args(p, a);
  if (st != SDA_OK) return st;
  if (!Q || !K || !V || !offsets || !LSE || !dO || !dQ || !dK || !dV || !d_offsets || !ws)
    return SDA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dO) || !aligned16(dQ) || !aligned16(dK) ||
      !aligned16(dV) || !aligned16(ws))
    return SDA_ERR_INVALID_ARG;
  if (ws_bytes < sda::dsa3d_bwd_ws_bytes(a)) return SDA_ERR_WORKSPACE;
  return from_cuda(sda::dsa3d_bwd(a, Q, K, V, offsets, LSE, dO, dQ, dK, dV, d_offsets, ws,
                                  static_cast<cudaStream_t>(stream)));
}

sda_status sda_dsa3d_offsets_bwd_workspace_size(const sda_dsa3d_problem* p, size_t* bytes) {
  sda::Dsa3dArgs a;
  const sda_status st = dsa3d_args(p, a);
  if (st != SDA_OK) return st;
  if (!bytes) return SDA_ERR_INVALID_ARG;
  *bytes = sda::dsa3d_offsets_bwd_ws_bytes(a);
  return SDA_OK;
}

sda_status sda_dsa3d_offsets_bwd(const sda_dsa3d_problem* p, const void* Q, const float* Wc, const float* bc,
                                 const float* Wl, const float* d_offsets, float* dQ, float* dWc, float* dbc,
                                 float* dWl, float* dbl, void* ws, size_t ws_bytes, void* stream) {
  sda::Dsa3dArgs a;
  const sda_status st = dsa3d_args(p, a);
  if (st != SDA_OK) return st;
  if (!Q || !Wc || !bc || !Wl || !d_offsets || !dQ || !dWc || !dbc || !dWl || !dbl || !ws)
    return SDA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(ws)) return SDA_ERR_INVALID_ARG;
  if (ws_bytes < sda::dsa3d_offsets_bwd_ws_bytes(a)) return SDA_ERR_WORKSPACE;
  return from_cuda(sda::dsa3d_offsets_bwd(a, Q, Wc, bc, Wl, d_offsets, dQ, dWc, dbc, dWl, dbl, ws,
                                          static_cast<cudaStream_t>(stream)));
}
