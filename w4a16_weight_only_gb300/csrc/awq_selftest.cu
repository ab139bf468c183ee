// Failure-detection self test: one thread waits, bounded in wall time, on an mbarrier that
// nothing completes.  The wait gives up exactly as a stalled pipeline stage in the GEMM
// kernels would (status word set, kernel returns), without any fault or hang.
#include "awq_internal.cuh"
#include "awq_ptx.cuh"

namespace awq {
namespace {

constexpr unsigned int kStatusSelfTest = 0x80u;

__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  ptx::mbar_init(&bar, 1);  // one arrival expected; none ever comes
  ptx::fence_mbar_init();
  ptx::mbar_wait_bounded(&bar, 0u, status, kStatusSelfTest, limit_ns);
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream) {
  unsigned int* status = nullptr;
  cudaError_t e = status_word_ptr(&status);
  if (e != cudaSuccess) return e;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace awq
