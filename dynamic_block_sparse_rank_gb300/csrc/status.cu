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
    if (v & sda::kStatusWaitTimeout) return SDA_ERR_DEVICE_TIMEOUT;
    if (v & sda::kStatusBadIndex) return SDA_ERR_DEVICE_BAD_INDEX;
    return SDA_ERR_DEVICE_RANGE;
  }
  return SDA_OK;
}

extern "C" unsigned long long sda_kernel_launch_count(void) { return sda::g_launches.load(std::memory_order_relaxed); }

namespace sda {
namespace {
// A wait that nothing completes: the mbarrier expects one arrival that never
// comes, so the bounded wait (the same code every kernel here uses) must run
// out, latch the timeout bit and return.
__global__ void wait_selftest_kernel(unsigned* status, unsigned long long limit_ns, int* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) *result = mbar_wait(&bar, 0, status, &abort_flag, limit_ns) ? 1 : 0;
}
}  // namespace
}  // namespace sda

extern "C" sda_status sda_selftest_wait_timeout(unsigned limit_us, int* completed, void* stream) {
  if (limit_us == 0 || limit_us > 1000000u || !completed) return SDA_ERR_INVALID_ARG;
  unsigned* status = sda::status_ptr();
  if (!status) return SDA_ERR_CUDA;
  sda::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      status, 1000ull * limit_us, completed);
  sda::note_launches(1);
  return cudaGetLastError() == cudaSuccess ? SDA_OK : SDA_ERR_CUDA;
}
