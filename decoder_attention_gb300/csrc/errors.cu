// The device error word that kernels set (kErrIndex, kErrTimeout) and da_check_device_error reads.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace da {

__device__ int g_error_word = 0;

// Device address of g_error_word on the current device, looked up once per device.
int* error_word_ptr() {
  static std::mutex mu;
  static int* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

// Reads and clears the error word (stream-ordered), after waiting for `stream`.
int read_and_clear_error_word(cudaStream_t stream, int* flags) {
  *flags = 0;
  int* p = error_word_ptr();
  if (!p) return DA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DA_ERR_CUDA;
  int host = 0;
  if (cudaMemcpy(&host, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DA_ERR_CUDA;
  const int zero = 0;
  if (host && cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return DA_ERR_CUDA;
  *flags = host;
  return DA_OK;
}

}  // namespace da
