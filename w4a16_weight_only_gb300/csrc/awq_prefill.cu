// Prefill path of awq_gemm (large M): tcgen05/TMEM tensor-core kernel.  Placeholder
// until the kernel lands: prefill_supported() reports the path unavailable, and the
// device status word used by bounded waits lives here.
#include "awq_internal.cuh"

namespace awq {

__device__ unsigned int g_status_word = 0u;

bool prefill_supported(const GemmProblem&, const char** why) {
  if (why) *why = "prefill kernel not built";
  return false;
}

cudaError_t launch_prefill(const GemmProblem&) { return cudaErrorNotSupported; }

cudaError_t status_word_ptr(unsigned int** ptr) {
  static unsigned int* cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev]) {
    *ptr = cache[dev];
    return cudaSuccess;
  }
  void* a = nullptr;
  e = cudaGetSymbolAddress(&a, g_status_word);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev] = static_cast<unsigned int*>(a);
  *ptr = static_cast<unsigned int*>(a);
  return cudaSuccess;
}

cudaError_t read_and_clear_status(cudaStream_t stream, unsigned int* value) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  unsigned int v = 0u;
  e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v != 0u) {
    const unsigned int zero = 0u;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *value = v;
  return cudaSuccess;
}

}  // namespace awq
