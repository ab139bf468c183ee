// Internal declarations shared by the translation units of libawq_gb300.so.
// Nothing here is part of the public C ABI (include/awq.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
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
  bool bf16 = false;      // x, scales, bias and y hold bf16 (same 16-bit storage)
  // Grouped (mixture-of-experts) problems: E experts' weights stacked ([E, K, N/8],
  // [E, K/G, N/8], [E, K/G, N], bias [E, N]); rows offsets[e]..offsets[e+1]-1 of x / y
  // belong to expert e (device array of E + 1 ints).  E == 0: a plain linear.
  const int* offsets = nullptr;
  int E = 0;
  // Code width: 4 (ORDER-interleaved nibbles, N/8 words a row) or 8 (little-endian bytes,
  // N/4 words a row; GPTQModel wiki "AWQ", "Saved formats and packing").
  int bits = 4;
  // The caller declares qweight, qzeros, scales and bias complete before the kernel launched
  // just before this one on the stream (AWQ_GEMM_STATIC_WEIGHTS): the small-M kernel may then
  // stream them before its programmatic-launch wait.
  bool static_weights = false;
};

// Kernel families; values equal awq_path_t.
enum Path { kAuto = 0, kDecode = 1, kPrefill = 2, kGeneric = 3 };

// Dequant (awq_dequant).  out_f32 selects fp32 vs fp16 output.
cudaError_t launch_dequant(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int N,
                           int G, void* out, bool out_f32, cudaStream_t stream, bool bf16 = false);
// 8-bit codes (awq_dequant_w8): qweight [K, N/4], qzeros [K/G, N/4], fp16 scales.
cudaError_t launch_dequant8(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int N,
                            int G, void* out, bool out_f32, cudaStream_t stream);

// Round-to-nearest group quantization (awq_quantize_rtn): w fp16 [N, K] -> qweight
// [K, N/8], qzeros [K/G, N/8], scales [K/G, N].
cudaError_t launch_quantize_rtn(const __half* w, int N, int K, int G, bool sym, uint32_t* qw,
                                uint32_t* qz, __half* sc, cudaStream_t stream);

// Any valid shape / alignment.
cudaError_t launch_generic(const GemmProblem& p);

// Split-K tensor-core streaming kernels for small M.  decode_supported() is a pure host
// check; launch_decode() uses the TMA-fed kernel when it takes the shape, else the
// register-streaming one.
bool decode_supported(const GemmProblem& p, const char** why);
cudaError_t launch_decode(const GemmProblem& p);
bool decode_ldg_supported(const GemmProblem& p, const char** why);
cudaError_t launch_decode_ldg(const GemmProblem& p);
bool decode_tma_supported(const GemmProblem& p, const char** why);
cudaError_t launch_decode_tma(const GemmProblem& p);

// Grouped decode (awq_gemm_grouped): the TMA decode kernel over stacked experts.
bool decode_grouped_supported(const GemmProblem& p, const char** why);
cudaError_t launch_decode_grouped(const GemmProblem& p);

// Row-major 3D tensor map: dim0 contiguous elements, dim1 rows, dim2 planes (box depth 1).
bool make_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes,
                  const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2, uint32_t box0,
                  uint32_t box1, CUtensorMapSwizzle swizzle, const char** why);

// Row-major 2D tensor map: dim0 contiguous elements per row, dim1 rows.
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes,
                  const void* base, uint64_t dim0, uint64_t dim1, uint32_t box0, uint32_t box1,
                  CUtensorMapSwizzle swizzle, const char** why);

// Device address of the status word on the current device (bounded waits that give up
// OR a code into it).
cudaError_t status_word_ptr(unsigned int** ptr);

// tcgen05/TMEM kernel for large M.
bool prefill_supported(const GemmProblem& p, const char** why);
// Estimated duration (us) of launch_prefill for p on a device with `sms` SMs.
double prefill_estimate_us(const GemmProblem& p, int sms);
cudaError_t launch_prefill(const GemmProblem& p);

// Tile-packed layout (awq_repack / awq_gemm_packed): shape rule, size in bytes, the
// one-off conversion, and the linear that reads it (x, bias, y, M, K, N, G, stream of p).
bool packed_supported(int64_t K, int64_t N, int64_t G, const char** why);
size_t packed_bytes(int64_t K, int64_t N);
cudaError_t launch_repack(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int N,
                          int G, void* out, cudaStream_t stream);
// The same for 8-bit codes (qweight [K, N/4]): shape rule, size, conversion.  launch_packed
// reads this layout when p.bits == 8 (fp16 only).
bool packed8_supported(int64_t K, int64_t N, int64_t G, const char** why);
size_t packed8_bytes(int64_t K, int64_t N);
cudaError_t launch_repack8(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int N,
                           int G, void* out, cudaStream_t stream);
// With a workspace of at least packed_workspace_bytes(SM count) bytes (flags zero), launches
// with M > 128 whose tiles fill the SMs poorly run the stream-K kernel.
size_t packed_workspace_bytes(int sms);
size_t packed_workspace_flag_bytes(int sms);  // the leading flag area of that workspace
// Grouped (mixture-of-experts) linear on E stacked 4-bit packed layouts, fp16 or bf16 (p.bf16): p.offsets
// (device, E + 1) and p.E (1 .. kPackedGroupedMaxE) as for launch_decode_grouped, p.M = R.
constexpr int kPackedGroupedMaxE = 256;
cudaError_t launch_packed_grouped(const GemmProblem& p, const void* packed);
// The library's fixed device scratch (awq_gemm_packed_noalloc): its size, and its address on
// the current device (looked up once per device).
size_t packed_static_scratch_bytes();
cudaError_t packed_static_scratch(void** ptr);
cudaError_t launch_packed(const GemmProblem& p, const void* packed, void* workspace = nullptr,
                          size_t workspace_bytes = 0);

// Failure-detection self test: a bounded wait that nothing completes (see awq.h).
cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream);

// Loads the module (used by awq_runtime_available to prove the sm_103a image runs here).
cudaError_t probe_kernel_image(cudaFuncAttributes* attr);

// Device status word (bounded waits that gave up set it).
cudaError_t read_and_clear_status(cudaStream_t stream, unsigned int* value);

// Column of a nibble: nibble i of a packed word holds column ORDER[i] of its eight,
// ORDER = {0,2,4,6,1,3,5,7} (tensref.org/formats/awq, "Reader").
__host__ __device__ constexpr int nibble_column(int i) { return ((i & 3) << 1) | (i >> 2); }

// 16-bit activation / scale elements: fp16, or bf16 when kBF (same storage).
template <bool kBF>
__device__ __forceinline__ float elem_to_float(uint16_t u) {
  if constexpr (kBF) return __uint_as_float(static_cast<uint32_t>(u) << 16);
  else return __half2float(__ushort_as_half(u));
}
// One rounding (to nearest even) of fp32 to the element type, as its 16-bit pattern.
template <bool kBF>
__device__ __forceinline__ uint16_t float_to_elem(float f) {
  if constexpr (kBF) return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  else return __half_as_ushort(__float2half_rn(f));
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace awq
