// Internal host-side interfaces between the C-ABI layer (api.cu) and the
// kernel translation units.  Nothing here is exported.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sda.h"
#include "common.cuh"

namespace sda {

// Validated problem with derived sizes.
struct Prob {
  Geom g;
  int B, Hh, d, r, k, dtype;
  float scale;  // softmax scale
  long long N;  // tokens per batch entry
};

constexpr int kMaxStates = 16;

struct MergeArgs {
  const void* O[kMaxStates];
  const float* L[kMaxStates];
  int n_states;
  int B, N, Hh, d;
  void* O_out;
  float* L_out;
};

// Device status word of the current device (see status.cu).
unsigned* status_ptr();
// Count kernels launched by the library (reported by sda_kernel_launch_count).
void note_launches(int n);

// ---- merge.cu
cudaError_t launch_merge(const MergeArgs& a, int dtype, cudaStream_t st);

struct MergeBwdArgs {
  const void* O[kMaxStates];
  const float* L[kMaxStates];
  const void* dO;
  const float* dL;  // may be null (zero LSE gradient)
  void* dO_out[kMaxStates];
  float* dL_out[kMaxStates];
  int n_states;
  int B, N, Hh, d;
};
cudaError_t launch_merge_bwd(const MergeBwdArgs& a, int dtype, cudaStream_t st);

// The backward of one partition state (DiTango reuse, training): the state that
// sda_attn_fwd computes with key range [kb_begin, kb_end) and the active query
// blocks, given dL/dO of that state and dL/dLSE (dLSE, may be null).  A null Part
// is the whole map with no LSE gradient.
struct Part {
  int kb_begin, kb_end;
  const uint8_t* qb_active;
  const float* dLSE;
};

// ---- simt.cu (fp32 problems)
size_t predict_ws_f32(const Prob& p);
cudaError_t predict_f32(const Prob& p, const float* Q, const float* K, const float* Wq, const float* Wk,
                        int32_t* idx, float* score, void* ws, cudaStream_t st);
cudaError_t fwd_f32(const Prob& p, const float* Q, const float* K, const float* V, const int32_t* idx,
                    int kb_begin, int kb_end, const uint8_t* qb_active, float* O, float* LSE, cudaStream_t st);
size_t bwd_ws_f32(const Prob& p);
cudaError_t bwd_prepare_f32(const Prob& p, const float* O, const float* dO, void* ws, cudaStream_t st,
                            const float* dLSE = nullptr);
cudaError_t bwd_dq_f32(const Prob& p, const float* Q, const float* K, const float* V, const float* LSE,
                       const float* dO, const int32_t* idx, float* dQ, void* ws, cudaStream_t st,
                       const Part* part = nullptr);
cudaError_t bwd_dkdv_f32(const Prob& p, const float* Q, const float* K, const float* V, const float* LSE,
                         const float* dO, const int32_t* idx, float* dK, float* dV, void* ws, cudaStream_t st,
                         const Part* part = nullptr);

// ---- tensor maps (tmap.cu)
// 5-D map over a [T, H, W, heads, d] tensor of one batch entry; box = 128
// bytes of d x 1 head x bw x bh x bt tokens, 128B swizzle.
enum TokType { kTokBF16 = 0, kTokF16 = 1, kTokF32 = 2 };
bool make_token_map(CUtensorMap* m, const void* base, TokType t, int T, int H, int W, int Hh, int d, int bt, int bh,
                    int bw);

// ---- predict_tc.cu (bf16 problems)
// 3D deformable sliding attention (dsa3d.cu)
struct Dsa3dArgs {
  int B, T, H, W, heads, d, kt, kh, kw, S;
  float scale;
};
cudaError_t dsa3d_offsets(const Dsa3dArgs& a, const void* Q, const float* Wc, const float* bc, const float* Wl,
                          const float* bl, float* off, cudaStream_t st);
cudaError_t dsa3d_fwd(const Dsa3dArgs& a, const void* Q, const void* K, const void* V, const float* off, void* O,
                      float* LSE, cudaStream_t st);
cudaError_t dsa3d_bwd(const Dsa3dArgs& a, const void* Q, const void* K, const void* V, const float* off,
                      const float* LSE, const void* dO, float* dQ, float* dK, float* dV, float* doff, void* ws,
                      cudaStream_t st);
size_t dsa3d_bwd_ws_bytes(const Dsa3dArgs& a);
cudaError_t dsa3d_offsets_bwd(const Dsa3dArgs& a, const void* Q, const float* Wc, const float* bc, const float* Wl,
                              const float* doff, float* dQ, float* dWc, float* dbc, float* dWl, float* dbl,
                              void* ws, cudaStream_t st);
size_t dsa3d_offsets_bwd_ws_bytes(const Dsa3dArgs& a);

size_t predict_ws_tc(const Prob& p);
cudaError_t predict_tc(const Prob& p, const void* Q, const void* K, const void* Wq, const void* Wk, int32_t* idx,
                       float* score, void* ws, cudaStream_t st);

// The projections alone (q~, k~ tiles into the predictor workspace, as predict_tc lays them out).
cudaError_t project_tc(const Prob& p, const void* Q, const void* K, const void* Wq, const void* Wk, void* ws,
                       cudaStream_t st);

// ---- distill_tc.cu (the predictor's training signal)
size_t distill_ws_tc(const Prob& p);
cudaError_t distill_tc(const Prob& p, const void* Q, const void* K, const void* Wq, const void* Wk, float* dWq,
                       float* dWk, double* loss, float* s_out, float* t_out, void* ws, cudaStream_t st);

// ---- attn_fwd_tc.cu
// O in bf16, or (out_f32) in fp32.
cudaError_t fwd_tc(const Prob& p, const void* Q, const void* K, const void* V, const int32_t* idx, int kb_begin,
                   int kb_end, const uint8_t* qb_active, void* O, bool out_f32, float* LSE, cudaStream_t st);
// The training forward's kernel: fp16 copies of Q, K, V, P in fp16, O also written in fp32.
cudaError_t fwd_tc_f16(const Prob& p, const void* Q16, const void* K16, const void* V16, const int32_t* idx, void* O,
                       float* LSE, float* O32, cudaStream_t st);

// ---- attn_bwd_tc.cu
// Backward in three phases sharing the workspace, in this order: prepare
// (block-map transpose, D and LSE rows, fp16 copies of Q, K, V, dO), dQ (also
// writes the exact D rows), dK/dV.
size_t bwd_ws_tc(const Prob& p);
cudaError_t bwd_prepare_tc(const Prob& p, const void* Q, const void* K, const void* V, const void* O,
                           const float* LSE, const void* dO, const int32_t* idx, void* ws, cudaStream_t st,
                           const Part* part = nullptr);
cudaError_t bwd_dq_tc(const Prob& p, const void* V, const void* dO, const int32_t* idx, void* dQ, int grad_dtype,
                      void* ws, cudaStream_t st, const Part* part = nullptr);
cudaError_t bwd_dkdv_tc(const Prob& p, const void* V, const void* dO, void* dK, void* dV, int grad_dtype, void* ws,
                        cudaStream_t st);
// The training pair: the forward writes fp16 copies of Q, K, V and an fp32 O into the
// training workspace; the backward (phases: 1 prepare, 2 dQ, 4 dK/dV) reads them.
size_t train_ws_tc(const Prob& p);
cudaError_t fwd_train_tc(const Prob& p, const void* Q, const void* K, const void* V, const int32_t* idx, void* O,
                         float* LSE, void* ws, cudaStream_t st);
cudaError_t bwd_train_tc(const Prob& p, const float* LSE, const void* dO, const int32_t* idx, void* dQ, void* dK,
                         void* dV, int grad_dtype, void* ws, int phases, cudaStream_t st);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace sda
