/*
 * sda.h — C ABI of the dynamic block-sparse attention library (sm_103a).
 *
 * The library computes the three steps of learned block-sparse attention for
 * video diffusion transformers:
 *
 *   1. sda_predict_blocks — a low-rank predictor picks, for every query block,
 *      the key blocks worth attending to.  "DSV: Exploiting Dynamic Sparsity to
 *      Accelerate Large-Scale Video DiT Training", section 3a ("low-rank
 *      predictor": a cheap estimate guesses which ~10% matters before the
 *      expensive attention runs) and section 3b ("query grouping": neighbouring
 *      tokens share the decision).  Form used: q~ = Q Wq, k~ = K Wk (rank r);
 *      s(I, J) = max over i in I, j in J of q~_i . k~_j; keep the k highest J
 *      per I, ties to the lower J, k = clamp(floor(keep_ratio * n_b + 1e-9), 1, n_b).
 *   2. sda_attn_fwd / sda_attn_bwd — flash attention restricted to the kept
 *      blocks (DSV section 4, stage 2: compute only on the predicted parts),
 *      emitting O and the natural-log log-sum-exp, and the gradients dQ, dK, dV
 *      with the block map held fixed.
 *   3. sda_merge_states — the log-sum-exp merge of partial attention states
 *      computed over separate key partitions: the state-reuse primitive of
 *      "DiTango: Cost-Effective Parallel Diffusion Generation with Selective
 *      Attention State Reuse" (near partitions recomputed, far ones reused),
 *      and sda_merge_states_bwd, its gradient for training through the reuse.
 *
 * A second sparse-attention family, 3D deformable sliding attention
 * ("MegaSlide-DiT"), has its own calls (sda_dsa3d_*) and problem struct below.
 *
 * Conventions shared by every call
 *   - Tokens of a T x H x W latent grid are in raster order n = (t*H + h)*W + w.
 *     Q, K, V, O, dO, dQ, dK, dV are contiguous row-major [B, N, heads, d].
 *     LSE is [B, heads, N] (fp32, natural log).
 *   - Blocks are compact bt x bh x bw space-time tiles numbered t-major,
 *     I = (it*nH + ih)*nW + iw with nT = ceil(T/bt) etc.; edge tiles of a
 *     non-divisible grid are clipped (they hold only real tokens).
 *   - All device pointers are owned by the caller; the library allocates no
 *     device or host memory.  Scratch comes from the caller's workspace (ws).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Argument errors are reported synchronously and nothing is
 *     launched.  A device-side bounded wait that runs out sets a latched status
 *     word that sda_get_device_status reports.
 *   - dtype SDA_F32 runs fp32 CUDA-core kernels (any d <= 128, any tile up to
 *     1024 tokens); SDA_BF16 runs the tensor-core path, which requires
 *     bt*bh*bw == 128, d in {64, 128} and rank in {16, 32, 48, 64}.
 *     Unsupported shapes return SDA_ERR_UNSUPPORTED.
 *   - Pointers used by the tensor-core path must be 16-byte aligned.
 *   - The library keeps per-device addresses of its own device objects (the
 *     status word) for the life of the process; a cudaDeviceReset makes them
 *     stale, so a process that resets a device must not call the library on
 *     that device afterwards.
 */
#ifndef SDA_H_
#define SDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDA_OK = 0,
  SDA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad range */
  SDA_ERR_UNSUPPORTED = 2,   /* valid problem the kernels do not cover */
  SDA_ERR_WORKSPACE = 3,     /* ws_bytes smaller than sda_workspace_size */
  SDA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  SDA_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait ran out (see sda_get_device_status) */
  SDA_ERR_DEVICE_BAD_INDEX = 6, /* a kernel met a block_idx entry outside [0, n_b) or a repeated
                                   entry in one row (see sda_get_device_status) */
  SDA_ERR_DEVICE_RANGE = 7    /* the tensor-core backward met an input value outside fp16's
                                 finite range (|x| > 65504, inf or NaN) */
} sda_status;

typedef enum { SDA_F32 = 0, SDA_BF16 = 1 } sda_dtype;

/* Problem description (DSV problem statement: a T x H x W latent grid with
 * heads and head dim, query/key block sizes, predictor rank, keep ratio). */
typedef struct {
  int B, heads, T, H, W, head_dim;
  int bt, bh, bw;      /* block (tile) extent along t, h, w */
  int rank;            /* predictor rank r */
  double keep_ratio;   /* fraction of key blocks kept per query block; k is
                          floor(keep_ratio * n_b + 1e-9) in IEEE double with
                          the product and the sum each rounded once, so a
                          caller's decimal keep ratio (a double) gives the
                          same k in any language that does that arithmetic */
  int dtype;           /* sda_dtype of Q, K, V, O, dO, Wq, Wk */
  float softmax_scale; /* 0 selects 1/sqrt(head_dim) */
} sda_problem;

/* Workspace queries (op argument of sda_workspace_size). */
enum { SDA_OP_PREDICT = 0, SDA_OP_BWD = 1, SDA_OP_TRAIN = 2, SDA_OP_PREDICTOR_GRAD = 3 };

/* Host only.  n_blocks = nT*nH*nW and k = kept key blocks per query block. */
sda_status sda_num_blocks(const sda_problem* p, int* n_blocks, int* k);

/* Host only.  Bytes of device workspace that `op` needs for problem p. */
sda_status sda_workspace_size(const sda_problem* p, int op, size_t* bytes);

/* Step 1: predictor + top-k.
 *   Q, K        [B, N, heads, d] (dtype)
 *   Wq, Wk      [heads, d, r]    (dtype)
 *   block_idx   out [B, heads, n_b, k] int32, each row ascending
 *   block_score optional out [B, heads, n_b, n_b] fp32 block scores s(I, J)
 *               (pass NULL to skip; it is for inspection, O(n_b^2) bytes)
 *   ws          device workspace of at least sda_workspace_size(SDA_OP_PREDICT).
 * For bf16 problems q~ and k~ are stored in bf16 (round to nearest even)
 * before the score products, which accumulate in fp32. */
sda_status sda_predict_blocks(const sda_problem* p, const void* Q, const void* K, const void* Wq,
                              const void* Wk, int32_t* block_idx, float* block_score, void* ws,
                              size_t ws_bytes, void* stream);

/* The predictor's training signal (DSV section 4, "two-stage training": the
 * predictor learns in a stage of its own; the page gives no loss).  For every
 * (b, head, query block I, key block J): the low-rank block score
 * s = max over i in I, j in J of q~_i . k~_j (as sda_predict_blocks computes it)
 * at its maximising pair (i*, j*) — the first in (row, column) order of the two
 * tiles on ties; fp32 candidates within twice their rounding bound are
 * re-scored to about 2^-44, so equal scores tie exactly — and the full-rank
 * target t = max of q_i . k_j
 * over the same pairs.  With e = s - t and L = 1/2 sum e^2:
 *   dWq[h] = dL/dWq[h] = sum e Q_i*^T k~_j*,   dWk[h] = sum e K_j*^T q~_i*
 * (the bf16 rounding of q~, k~ passes the gradient unchanged; t is a target).
 *   Q, K, Wq, Wk  as sda_predict_blocks (tensor-core path only: SDA_BF16)
 *   dWq, dWk      out [heads, d, r] fp32, summed over the batch
 *   loss          out, one fp64 value: L over the whole batch
 *   s_out, t_out  optional out [B, heads, n_b, n_b] fp32 (NULL to skip)
 *   ws            at least sda_workspace_size(SDA_OP_PREDICTOR_GRAD) bytes.
 * Its cost is one low-rank and one full-rank (K = d) product per block pair, 1 + d/r
 * times the predictor's.  The gradient sums use fp32 atomics: results agree
 * from run to run to fp32 rounding, not bit for bit. */
sda_status sda_predictor_grad(const sda_problem* p, const void* Q, const void* K, const void* Wq,
                              const void* Wk, float* dWq, float* dWk, double* loss, float* s_out,
                              float* t_out, void* ws, size_t ws_bytes, void* stream);

/* Step 2a: block-sparse attention forward over the kept blocks J of each query
 * block I that satisfy kb_begin <= J < kb_end (0, n_b = all keys).
 *   block_idx  [B, heads, n_b, k] int32 (as written by sda_predict_blocks;
 *              entries must be distinct and in [0, n_b); order is free).  An
 *              entry outside that range is skipped, and so is (on the bf16
 *              path) a repeat of an entry earlier in its row; either latches
 *              SDA_ERR_DEVICE_BAD_INDEX for sda_get_device_status.
 *   qb_active  optional [n_b] uint8; query blocks with 0 are not written at all
 *              (their O and LSE rows keep the caller's previous contents — the
 *              cached state of DiTango's reuse).  NULL = all active.
 *   O          out [B, N, heads, d] in out_dtype: p->dtype, or SDA_F32 (for
 *              a bf16 problem: O before any rounding to bf16 — the form to
 *              keep partition states in when they will be merged, so that
 *              the merged result is rounded once, not twice);
 *   LSE        out [B, heads, N] fp32.
 * A row whose block has no kept key in the range gets O = 0, LSE = -inf.  On
 * the bf16 path P enters the P V product as two bf16 terms (the value and its
 * rounding remainder), so O is exact to fp32 accumulation. */
sda_status sda_attn_fwd(const sda_problem* p, const void* Q, const void* K, const void* V,
                        const int32_t* block_idx, int kb_begin, int kb_end, const uint8_t* qb_active,
                        void* O, float* LSE, int out_dtype, void* stream);

/* Step 2b: gradients of sda_attn_fwd (full key range) with the map fixed.
 *   O, LSE      the forward outputs;  dO [B, N, heads, d] (dtype)
 *   dQ, dK, dV  out [B, N, heads, d] in grad_dtype (SDA_F32, or p->dtype)
 *   ws          device workspace of at least sda_workspace_size(SDA_OP_BWD).
 * Deterministic: no atomics on gradient values. */
sda_status sda_attn_bwd(const sda_problem* p, const void* Q, const void* K, const void* V,
                        const void* O, const float* LSE, const void* dO, const int32_t* block_idx,
                        void* dQ, void* dK, void* dV, int grad_dtype, void* ws, size_t ws_bytes,
                        void* stream);

/* Step 2b in phases.  sda_attn_bwd is exactly these three calls, in this
 * order, on one workspace; they are exposed so that a caller can time them or
 * interleave other work between them.  All three take the same problem,
 * inputs and workspace.
 *   prepare: transposes the block map (for every key block, the query blocks
 *            that kept it, ascending), computes D~_i = dO_i . O_i from the
 *            stored O and the LSE rows in tile order, and (tensor-core path)
 *            fp16 copies of Q, K, V and dO.
 *   dq:      dQ = scale * sum_j dS_ij k_j over each query block's kept blocks;
 *            it forms D_i = sum_j P_ij dP_ij exactly in the same pass (the
 *            stored bf16 O would carry its rounding into D~) and writes it
 *            back for the next phase.
 *   dkdv:    dK = scale * sum_i dS_ij q_i and dV = sum_i P_ij dO_i over the
 *            query blocks that kept each key block.
 * On the tensor-core path every product runs on fp16 operands (P and dS are
 * rounded to fp16), so Q, K, V, dO and dP - D must stay inside fp16's range
 * (|x| < 65504). */
sda_status sda_attn_bwd_prepare(const sda_problem* p, const void* Q, const void* K, const void* V, const void* O,
                                const float* LSE, const void* dO, const int32_t* block_idx, void* ws,
                                size_t ws_bytes, void* stream);
sda_status sda_attn_bwd_dq(const sda_problem* p, const void* Q, const void* K, const void* V, const float* LSE,
                           const void* dO, const int32_t* block_idx, void* dQ, int grad_dtype, void* ws,
                           size_t ws_bytes, void* stream);
sda_status sda_attn_bwd_dkdv(const sda_problem* p, const void* Q, const void* K, const void* V, const float* LSE,
                             const void* dO, const int32_t* block_idx, void* dK, void* dV, int grad_dtype, void* ws,
                             size_t ws_bytes, void* stream);

/* The training pair: a forward that keeps what its backward needs, and that
 * backward.  Same attention as sda_attn_fwd over the whole key range and
 * sda_attn_bwd, computed with finer intermediates and fewer products
 * (tensor-core path only: dtype SDA_BF16).
 *
 * sda_attn_fwd_train writes fp16 copies of Q, K and V into ws (exact for bf16
 * values inside fp16's range; a value outside it latches SDA_ERR_DEVICE_RANGE),
 * runs the forward on them with P rounded to fp16 (eight times finer than the
 * bf16 P of sda_attn_fwd), writes O (dtype) and LSE like sda_attn_fwd and also
 * keeps O in fp32 in ws.
 *
 * sda_attn_bwd_train then computes dQ, dK, dV (grad_dtype: SDA_F32 or dtype)
 * for the same problem, block_idx and ws: D_i = dO_i . O_i is taken from the
 * fp32 O, which is exact enough that dS = P (dP - D) needs no correction, so
 * the dQ pass runs three products per kept block instead of the four of
 * sda_attn_bwd.  Deterministic, no atomics on gradient values.  `phases`
 * selects its steps, in this order (pass 7 for all): 1 prepares (block-map
 * transpose, fp16 copy of dO, D and the LSE rows), 2 computes dQ, 4 computes dK
 * and dV; a call with a subset is for timing the steps.
 *   ws   at least sda_workspace_size(SDA_OP_TRAIN) bytes, 16-byte aligned;
 *        between the two calls the caller keeps it (and block_idx, LSE) intact.
 * Errors and alignment as sda_attn_fwd / sda_attn_bwd; SDA_ERR_UNSUPPORTED for
 * SDA_F32 problems. */
sda_status sda_attn_fwd_train(const sda_problem* p, const void* Q, const void* K, const void* V,
                              const int32_t* block_idx, void* O, float* LSE, void* ws, size_t ws_bytes,
                              void* stream);
sda_status sda_attn_bwd_train(const sda_problem* p, const float* LSE, const void* dO, const int32_t* block_idx,
                              void* dQ, void* dK, void* dV, int grad_dtype, int phases, void* ws, size_t ws_bytes,
                              void* stream);

/* Backward of one partition state, for training through DiTango's state reuse:
 * the gradient with respect to Q, K, V of the state (O_p, LSE_p) that
 * sda_attn_fwd computes with the same block_idx, kb_begin, kb_end and
 * qb_active, given
 *   dO    [B, N, heads, d] (dtype): dL/dO_p (from sda_merge_states_bwd)
 *   dLSE  [B, heads, N] fp32: dL/dLSE_p, or NULL for zero
 *   O, LSE the state itself (rows of inactive query blocks are not read for
 *          anything that reaches an output)
 * Since d LSE_i / d S_ij = P_ij, dS_ij = P_ij (dP_ij - D_i + dLSE_i) over the
 * kept keys in [kb_begin, kb_end).  dQ is written for every row (zero for
 * inactive query blocks and rows with no key in the range), dK and dV for every
 * key row (zero outside the range); the gradient of a step sums these over its
 * fresh partitions.  Workspace, grad_dtype, alignment and errors as
 * sda_attn_bwd; 0 <= kb_begin <= kb_end <= n_b.  With the whole range, no
 * qb_active and no dLSE it computes what sda_attn_bwd computes. */
sda_status sda_attn_bwd_partition(const sda_problem* p, const void* Q, const void* K, const void* V, const void* O,
                                  const float* LSE, const void* dO, const float* dLSE, const int32_t* block_idx,
                                  int kb_begin, int kb_end, const uint8_t* qb_active, void* dQ, void* dK, void* dV,
                                  int grad_dtype, void* ws, size_t ws_bytes, void* stream);

/* Step 3: LSE merge of n_states partial states (DiTango state reuse).
 *   O_parts[s]   device pointer, [B, N, heads, d] (dtype)
 *   LSE_parts[s] device pointer, [B, heads, N] fp32
 *   (the two pointer arrays themselves are host memory; 1 <= n_states <= 16)
 *   O_out, LSE_out  same layouts.  LSE = log sum_s exp(LSE_s),
 *   O = sum_s exp(LSE_s - LSE) O_s; rows with every LSE_s = -inf give (0, -inf).
 * O_out may alias O_parts[0] and LSE_out may alias LSE_parts[0]. */
sda_status sda_merge_states(int n_states, const void* const* O_parts, const float* const* LSE_parts,
                            int B, int N, int heads, int head_dim, int dtype, void* O_out,
                            float* LSE_out, void* stream);

/* Gradient of sda_merge_states, for training through DiTango's state reuse:
 * the fresh partition states carry the gradient (reused states are constants
 * of the step and need none).  Same states and layouts as sda_merge_states:
 *   O_parts[s], LSE_parts[s]  the merged states (1 <= n_states <= 16)
 *   dO         [B, N, heads, d] (dtype): gradient of the merged O
 *   dLSE       [B, heads, N] fp32, or NULL for a zero gradient of the merged LSE
 *   dO_parts[s]   [B, N, heads, d] (dtype): w_s dO
 *   dLSE_parts[s] [B, heads, N] fp32:       w_s (dO . (O_s - O) + dLSE)
 * with w_s = exp(LSE_s - LSE), LSE and O recomputed from the states in fp32 as
 * the merge computes them.  Parts with LSE_s = -inf, and rows where every
 * LSE_s is -inf, get zero gradients.  Each dO_parts[s] / dLSE_parts[s] pair is
 * then the (dO, dLSE) input of that partition's backward.  Outputs must not
 * overlap any input or each other; the pointer arrays are host memory; O, dO
 * and dO_parts 16-byte aligned. */
sda_status sda_merge_states_bwd(int n_states, const void* const* O_parts, const float* const* LSE_parts,
                                const void* dO, const float* dLSE, int B, int N, int heads, int head_dim,
                                int dtype, void* const* dO_parts, float* const* dLSE_parts, void* stream);

/* Synchronises `stream`, then reads and clears the current device's status
 * latch, which kernels of this library set since the last call:
 *   SDA_ERR_DEVICE_TIMEOUT    a bounded wait ran out (the kernel stopped early,
 *                             its outputs are incomplete);
 *   SDA_ERR_DEVICE_BAD_INDEX  a block_idx entry was outside [0, n_b) or repeated
 *                             within its row (the forward skips such entries;
 *                             other results computed from that map are undefined);
 *   SDA_ERR_DEVICE_RANGE      the tensor-core backward converted a Q, K, V or dO
 *                             value outside fp16's finite range (the gradients
 *                             hold inf or NaN).
 * When several were latched the first in this order is returned.  SDA_ERR_CUDA
 * on a CUDA error, else SDA_OK.  None of these leaves the context unusable. */
sda_status sda_get_device_status(void* stream);

/* Static description of a status code. */
const char* sda_status_string(sda_status s);

/* sda_predict_blocks for callers that cannot allocate device memory.  The
 * paper has no counterpart: this is a deployment convenience.
 *
 * Hosts that own all device memory themselves (a server that reserves one
 * arena at start-up, a plugin whose framework forbids device allocation, a
 * latency-critical loop that cannot afford cudaMalloc's implicit device
 * synchronisation) may have no buffer to pass as workspace.  This call runs
 * the same kernels as sda_predict_blocks but takes the q~ / k~ scratch from a
 * fixed array of SDA_NOALLOC_SCRATCH_BYTES compiled into the library, which
 * every GPU that loads the library keeps until process exit.  The caller still
 * passes inputs and outputs (same meaning as sda_predict_blocks); it allocates
 * nothing itself.
 *   - Problems whose predictor workspace (sda_workspace_size, SDA_OP_PREDICT)
 *     exceeds SDA_NOALLOC_SCRATCH_BYTES return SDA_ERR_WORKSPACE, launching
 *     nothing.
 *   - The first call on a device looks up the array's device address for that
 *     device (cudaGetSymbolAddress, with the device current); make that first
 *     call before any stream capture.  The address is kept for the life of the
 *     process: after a cudaDeviceReset of that device (which destroys the
 *     array with the context) the kept address is stale, so do not call this
 *     entry point again in a process that has reset the device.
 *   - All calls share the one array on a device: calls that overlap on the GPU
 *     (other streams, other threads) race on it.  Calls ordered on one stream
 *     are safe; nothing in the array needs clearing between calls. */
#define SDA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
sda_status sda_predict_blocks_noalloc(const sda_problem* p, const void* Q, const void* K, const void* Wq,
                                      const void* Wk, int32_t* block_idx, float* block_score, void* stream);

/* Diagnostic: launches one small kernel whose mbarrier wait can never complete
 * and lets the bounded wait that every kernel of this library uses run out
 * after limit_us microseconds (1 .. 1e6).  The kernel writes 0 to the device
 * int *completed (1 would mean the wait completed) and latches the timeout
 * bit, so a following sda_get_device_status returns SDA_ERR_DEVICE_TIMEOUT
 * (and clears it).  Nothing faults or hangs; the context stays usable. */
sda_status sda_selftest_wait_timeout(unsigned limit_us, int* completed, void* stream);

/* ---------------------------------------------------------------------------
 * 3D deformable sliding attention ("MegaSlide-DiT", gist.science explainer,
 * section 2 "3D deformable sliding attention (3D-DSA)"): every token attends
 * to S = kt*kh*kw keys and values sampled by trilinear interpolation around
 * it, at window points moved by offsets that a depthwise 3x3x3 convolution and
 * a linear layer predict from the token's query.  Cost linear in N.
 *
 * Tokens of one batch entry are the T x H x W raster (n = (t*H + h)*W + w).
 * Window point s = (a*kh + b)*kw + c of token (t, h, w) sits at
 * (t + a - (kt-1)/2, h + b - (kh-1)/2, w + c - (kw-1)/2) plus its offset
 * (dt, dh, dw) in token units.  K and V there are the trilinear interpolation
 * of the grid's rows, grid points outside the raster counting as zero rows (a
 * sample wholly outside gives k = v = 0 and logit 0; so does a non-finite
 * offset).  Logits scale * q.k, softmax over the S samples, O the weighted sum
 * of the sampled v, LSE the natural-log log-sum-exp of the logits.
 *
 * Layouts (row-major, device pointers, caller-owned, no aliasing between
 * inputs and outputs):
 *   Q, K, V, O  bf16 [B, N, heads, d], d in {64, 128}, 16-byte aligned
 *   offsets     fp32 [B, N, heads, S, 3]  (dt, dh, dw) per window point
 *   LSE         fp32 [B, heads, N]
 *   Wc          fp32 [heads, d, 3, 3, 3]  depthwise kernel, taps (dt, dh, dw)
 *                                         with the centre at [1, 1, 1]
 *   bc          fp32 [heads, d]
 *   Wl          fp32 [heads, d, 3*S]      output j = 3*s + axis
 *   bl          fp32 [heads, 3*S]
 * Both calls are asynchronous on `stream` (a cudaStream_t, or NULL), allocate
 * nothing and keep no state.  SDA_ERR_INVALID_ARG for a null pointer,
 * non-positive sizes, even window sizes or a misaligned tensor;
 * SDA_ERR_UNSUPPORTED for d outside {64, 128} or S > 125.
 * ------------------------------------------------------------------------- */
typedef struct {
  int B, T, H, W; /* batch entries and the token grid, N = T*H*W */
  int heads, d;   /* heads, head dimension */
  int kt, kh, kw; /* odd window sizes, S = kt*kh*kw */
  float scale;    /* softmax scale; <= 0 selects 1/sqrt(d) */
} sda_dsa3d_problem;

/* Offsets of every window point: Y = depthwise conv3d(Q of the head, Wc) + bc
 * (zero padding), offsets = Y Wl[h] + bl[h], all in fp32 from the bf16 Q. */
sda_status sda_dsa3d_offsets(const sda_dsa3d_problem* p, const void* Q, const float* Wc, const float* bc,
                             const float* Wl, const float* bl, float* offsets, void* stream);

/* Attention over the sampled window points (O bf16, LSE fp32), fp32 inside. */
sda_status sda_dsa3d_fwd(const sda_dsa3d_problem* p, const void* Q, const void* K, const void* V,
                         const float* offsets, void* O, float* LSE, void* stream);

/* Host only.  Bytes of device workspace that sda_dsa3d_bwd needs: 32 per
 * sample (B*N*heads*S of them: its two coefficients, in token order and again
 * in cell order, and a 16-byte record), plus two 4-byte counters per cell of
 * the (T+1) x (H+1) x (W+1) grid of floor positions and one more, per batch
 * entry and head.  SDA_ERR_UNSUPPORTED when N*S or the cell count reaches
 * 2^31. */
sda_status sda_dsa3d_bwd_workspace_size(const sda_dsa3d_problem* p, size_t* bytes);

/* Gradients of sda_dsa3d_fwd for a loss that reaches it through O (no LSE
 * gradient): with P the window softmax, dP_s = dO.v~_s and
 * da_s = P_s (dP_s - sum_u P_u dP_u),
 *   dQ        = scale sum_s da_s k~_s (the attention's part: the offset
 *               network's contribution to dQ is not included),
 *   dK, dV    at every trilinear corner row m of every sample: w_m scale da_s q
 *               and w_m P_s dO, summed over all tokens and samples,
 *   d_offsets = the derivative through the interpolation weights (one-sided
 *               from above on the integer grid, as floor() sees it).
 * Inputs as sda_dsa3d_fwd plus LSE (the forward's, fp32 [B, heads, N]) and dO
 * (bf16 [B, N, heads, d]); outputs fp32: dQ, dK, dV [B, N, heads, d] (16-byte
 * aligned), d_offsets [B, N, heads, S, 3]; all are written (not added to).
 * dK and dV rows are gathered: the samples are bucketed by the cell of their
 * floor position and each row sums the samples of the 8 cells it is a corner
 * of, in an order that the bucketing's atomics set (their last bits can vary
 * between runs).
 *   ws  device workspace of at least sda_dsa3d_bwd_workspace_size bytes,
 *       16-byte aligned.
 * Errors as sda_dsa3d_fwd, plus SDA_ERR_WORKSPACE for a smaller workspace and
 * the limits of sda_dsa3d_bwd_workspace_size. */
sda_status sda_dsa3d_bwd(const sda_dsa3d_problem* p, const void* Q, const void* K, const void* V,
                         const float* offsets, const float* LSE, const void* dO, float* dQ, float* dK, float* dV,
                         float* d_offsets, void* ws, size_t ws_bytes, void* stream);

/* Host only.  Bytes of device workspace that sda_dsa3d_offsets_bwd needs:
 * B*N*heads*d*4 (the fp32 gradient of the convolution output Y). */
sda_status sda_dsa3d_offsets_bwd_workspace_size(const sda_dsa3d_problem* p, size_t* bytes);

/* Gradients of sda_dsa3d_offsets (the offset network) for the offsets'
 * gradient d_offsets (fp32 [B, N, heads, S, 3], e.g. from sda_dsa3d_bwd).
 * With Y the convolution output and G = d_offsets of a head:
 *   dY  = G Wl[h]^T,   dWl[h] = Y^T G,   dbl[h] = sum over tokens of G,
 *   dWc[h][c][tap] = sum_n dY[n][c] Q[n + tap][c] (zero outside the raster),
 *   dbc[h][c] = sum_n dY[n][c],
 *   dQ += the transposed convolution of dY with Wc[h] (zero padding).
 * dQ (fp32 [B, N, heads, d]) is ADDED to, so that a caller passes the dQ of
 * sda_dsa3d_bwd and receives the total; dWc, dbc, dWl, dbl (fp32, shaped as
 * Wc, bc, Wl, bl) are cleared by the call and then accumulated with atomics
 * (their last bits depend on the order of the additions).  bl does not enter.
 *   ws  device workspace of at least
 *       sda_dsa3d_offsets_bwd_workspace_size bytes, 16-byte aligned.
 * Asynchronous on `stream`; allocates nothing.  Errors as sda_dsa3d_fwd, plus
 * SDA_ERR_WORKSPACE for a workspace smaller than that size. */
sda_status sda_dsa3d_offsets_bwd(const sda_dsa3d_problem* p, const void* Q, const float* Wc, const float* bc,
                                 const float* Wl, const float* d_offsets, float* dQ, float* dWc, float* dbc,
                                 float* dWl, float* dbl, void* ws, size_t ws_bytes, void* stream);

/* Host only.  Number of CUDA kernels the library has launched in this process
 * (all devices, all calls); a caller can difference it around a region. */
unsigned long long sda_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SDA_H_ */
