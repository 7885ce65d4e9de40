// sda_predict_blocks_noalloc: the predictor for callers that cannot allocate
// device memory.
//
// Some hosts own every byte of device memory themselves (a serving process
// that carves one arena at start-up, a plugin whose framework forbids device
// allocations, a latency-critical loop where cudaMalloc's implicit device
// synchronisation is not acceptable) and have no spare buffer to hand over as
// workspace.  For them this entry point runs the same predictor kernels as
// sda_predict_blocks, with the q~ / k~ scratch taken from a fixed array that
// is part of the library image instead of from a caller's workspace.
//
// The array is a file-scope __device__ object of SDA_NOALLOC_SCRATCH_BYTES:
// every GPU that loads the library holds it until the process exits.  In host
// code its name only stands for the object; its device address is looked up
// with cudaGetSymbolAddress once per device (on the first call made with that
// device current) and cached.  Nothing here calls cudaMalloc, cudaFree or an
// allocating library routine.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = SDA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" sda_status sda_predict_blocks_noalloc(const sda_problem* p, const void* Q, const void* K, const void* Wq,
                                                 const void* Wk, int32_t* block_idx, float* block_score,
                                                 void* stream) {
  size_t need = 0;
  sda_status s = sda_workspace_size(p, SDA_OP_PREDICT, &need);
  if (s != SDA_OK) return s;
  if (need > kScratchBytes) return SDA_ERR_WORKSPACE;  // problem larger than the built-in scratch
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SDA_ERR_CUDA;
  // The projection kernels overwrite every q~ / k~ byte the score kernel reads
  // (rows outside the grid are written as zeros), so the previous call's
  // contents never need clearing.
  return sda_predict_blocks(p, Q, K, Wq, Wk, block_idx, block_score, scratch, kScratchBytes, stream);
}
