// TMA tensor maps over token tensors laid out [T, H, W, heads, d] (one batch
// entry).  A box is one space-time tile of one head: 128 bytes of the head
// dimension x 1 head x bw x bh x bt tokens, 128-byte swizzled, so that the
// tile lands in shared memory as bw*bh*bt rows of 128 bytes in (tt, hh, ww)
// order — the canonical K-major SWIZZLE_128B layout the tensor cores read.
// Reads outside the grid (clipped edge tiles) are filled with zeros and
// stores outside it are dropped.
#include "internal.h"

namespace sda {

namespace {
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  }
  return fn;
}
}  // namespace

bool make_token_map(CUtensorMap* m, const void* base, TokType t, int T, int H, int W, int Hh, int d, int bt, int bh,
                    int bw) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  const int es = t == kTokF32 ? 4 : 2;
  const CUtensorMapDataType dt = t == kTokF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : t == kTokF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[5] = {(cuuint64_t)d, (cuuint64_t)Hh, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[4] = {(cuuint64_t)d * es, (cuuint64_t)Hh * d * es, (cuuint64_t)W * Hh * d * es,
                           (cuuint64_t)H * W * Hh * d * es};
  cuuint32_t box[5] = {(cuuint32_t)(128 / es), 1, (cuuint32_t)bw, (cuuint32_t)bh, (cuuint32_t)bt};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(m, dt, 5,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace sda
