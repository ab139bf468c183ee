// Internal declarations shared by the translation units of libawq_gb300.so.
// Nothing here is part of the public C ABI (include/awq.h).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace awq {

// One AWQ GEMM-layout linear plus activations (tensref.org/formats/awq, "Reader").
struct GemmProblem {
  const __half* x;        // [M, K]
  const uint32_t* qw;     // [K, N/8]
  const uint32_t* qz;     // [K/G, N/8]
  const __half* sc;       // [K/G, N]
  const __half* bias;     // [N] or nullptr
  __half* y;              // [M, N]
  int M, K, N, G;         // G already resolved (K when group_size == -1)
  cudaStream_t stream;
};

// Kernel families; values equal awq_path_t.
enum Path { kAuto = 0, kDecode = 1, kPrefill = 2, kGeneric = 3 };

// Dequant (awq_dequant).  out_f32 selects fp32 vs fp16 output.
cudaError_t launch_dequant(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int N,
                           int G, void* out, bool out_f32, cudaStream_t stream);

// Any valid shape / alignment.
cudaError_t launch_generic(const GemmProblem& p);

// Split-K tensor-core streaming kernel.  decode_supported() is a pure host check.
bool decode_supported(const GemmProblem& p, const char** why);
cudaError_t launch_decode(const GemmProblem& p);

// tcgen05/TMEM kernel for large M.
bool prefill_supported(const GemmProblem& p, const char** why);
cudaError_t launch_prefill(const GemmProblem& p);

// Loads the module (used by awq_runtime_available to prove the sm_103a image runs here).
cudaError_t probe_kernel_image(cudaFuncAttributes* attr);

// Device status word (bounded waits that gave up set it).
cudaError_t read_and_clear_status(cudaStream_t stream, unsigned int* value);

// Column of a nibble: nibble i of a packed word holds column ORDER[i] of its eight,
// ORDER = {0,2,4,6,1,3,5,7} (tensref.org/formats/awq, "Reader").
__host__ __device__ constexpr int nibble_column(int i) { return ((i & 3) << 1) | (i >> 2); }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace awq
