// Device status latch: one word per device that kernels of this library set
// (atomicOr) when a bounded wait runs out.  sda_get_device_status reads and
// clears it.
#include <atomic>

#include "internal.h"

namespace sda {

static std::atomic<unsigned long long> g_launches{0};

void note_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

__device__ unsigned g_status_word;

unsigned* status_ptr() {
  static unsigned* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<unsigned*>(p);
  }
  return cached[dev];
}

}  // namespace sda

extern "C" sda_status sda_get_device_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SDA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, sda::g_status_word, sizeof(v)) != cudaSuccess) return SDA_ERR_CUDA;
  if (v != 0) {
    unsigned zero = 0;
    if (cudaMemcpyToSymbol(sda::g_status_word, &zero, sizeof(zero)) != cudaSuccess) return SDA_ERR_CUDA;
    return SDA_ERR_DEVICE_TIMEOUT;
  }
  return SDA_OK;
}

extern "C" unsigned long long sda_kernel_launch_count(void) { return sda::g_launches.load(std::memory_order_relaxed); }
