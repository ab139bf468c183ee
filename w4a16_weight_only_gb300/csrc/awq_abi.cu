// C ABI of libawq_gb300.so (declared in include/awq.h): host-side validation, error
// reporting and kernel-family dispatch.  All argument checks run on the host before any
// CUDA call, so an invalid call touches no device.
#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/awq.h"
#include "awq_internal.cuh"

namespace {

thread_local std::string g_err;

awq_status_t fail(awq_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

awq_status_t ok() {
  g_err.clear();
  return AWQ_OK;
}

awq_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(AWQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int64_t kDimLimit = (int64_t{1} << 31) - 1;
constexpr int64_t kProdLimit = int64_t{1} << 40;

// Shape rules shared by awq_dequant and awq_gemm.  Returns AWQ_OK and the resolved G.
awq_status_t check_weight_shape(int64_t K, int64_t N, int64_t group_size, int* G_out,
                                int per_word = 8) {
  if (K <= 0) return fail(AWQ_ERR_INVALID_ARGUMENT, "K must be positive (got %lld)", (long long)K);
  if (N < 0) return fail(AWQ_ERR_INVALID_ARGUMENT, "N must be >= 0 (got %lld)", (long long)N);
  if (group_size == 0 || group_size < -1)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "group_size must be -1 or positive (got %lld)",
                (long long)group_size);
  if (K > kDimLimit || N > kDimLimit)
    return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "K and N must be below 2^31");
  if (K * N >= kProdLimit) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "K*N must be below 2^40");
  if (N % per_word != 0)
    return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "N=%lld is not a multiple of %d (codes per int32 word)",
                (long long)N, per_word);
  const int64_t G = group_size == -1 ? K : group_size;
  if (K % G != 0)
    return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "K=%lld is not a multiple of group_size=%lld",
                (long long)K, (long long)G);
  *G_out = static_cast<int>(G);
  return AWQ_OK;
}

// Current device must be compute capability 10.3 (the only code this library carries).
awq_status_t check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(AWQ_ERR_UNSUPPORTED_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  int major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(AWQ_ERR_UNSUPPORTED_DEVICE,
                "device %d is compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                dev, major, minor);
  return AWQ_OK;
}

bool al(const void* p, uintptr_t a) { return awq::aligned(p, a); }

awq_status_t build_problem(const void* x, const int32_t* qweight, const int32_t* qzeros,
                           const void* scales, const void* bias, int64_t M, int64_t K, int64_t N,
                           int64_t group_size, void* y, awq_stream_t stream, awq::GemmProblem* p,
                           bool* empty, bool bf16 = false, int bits = 4) {
  if (M < 0) return fail(AWQ_ERR_INVALID_ARGUMENT, "M must be >= 0 (got %lld)", (long long)M);
  int G = 0;
  awq_status_t st = check_weight_shape(K, N, group_size, &G, bits == 8 ? 4 : 8);
  if (st != AWQ_OK) return st;
  if (M > kDimLimit) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "M must be below 2^31");
  if (M * N >= kProdLimit || M * K >= kProdLimit)
    return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "M*N and M*K must be below 2^40");
  *empty = (M == 0 || N == 0);
  if (*empty) return AWQ_OK;
  if (!x || !qweight || !qzeros || !scales || !y)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "null pointer among x, qweight, qzeros, scales, y");
  if (!al(x, 2) || !al(scales, 2) || !al(y, 2) || (bias && !al(bias, 2)))
    return fail(AWQ_ERR_MISALIGNED, "16-bit tensors must be 2-byte aligned");
  if (!al(qweight, 4) || !al(qzeros, 4))
    return fail(AWQ_ERR_MISALIGNED, "qweight and qzeros must be 4-byte aligned");
  p->x = static_cast<const __half*>(x);
  p->qw = reinterpret_cast<const uint32_t*>(qweight);
  p->qz = reinterpret_cast<const uint32_t*>(qzeros);
  p->sc = static_cast<const __half*>(scales);
  p->bias = static_cast<const __half*>(bias);
  p->y = static_cast<__half*>(y);
  p->M = static_cast<int>(M);
  p->K = static_cast<int>(K);
  p->N = static_cast<int>(N);
  p->G = G;
  p->stream = reinterpret_cast<cudaStream_t>(stream);
  p->bf16 = bf16;
  p->bits = bits;
  return AWQ_OK;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    (void)cudaGetLastError();
    return 152;
  }
  return sms;
}

// Above 32 rows both tensor-core families can run; estimates fitted to GB300 timings of
// both kernels on the 7B and 70B linears at M = 8 .. 512 pick the faster.  Decode: the
// first 32-row tile streams the weights (about 3 TB/s plus 8 us of launch chain), each
// further 32-row tile costs 0.25 ns per code (its unpack and MMAs; the weights come from
// L2).  Prefill: the estimate of the plan it would launch (awq_prefill.cu).
bool prefill_faster(const awq::GemmProblem& p) {
  const double kn = static_cast<double>(p.K) * static_cast<double>(p.N);
  const double weight_bytes = kn * p.bits / 8.0 + 3.0 * static_cast<double>(p.K / p.G) * p.N;
  const double row_tiles = static_cast<double>((p.M + 31) / 32);
  const double decode_us = weight_bytes / 3.0e6 + 8.0 + (row_tiles - 1.0) * kn * 2.5e-7;
  return awq::prefill_estimate_us(p, sm_count()) < decode_us;
}

awq::Path choose_path(const awq::GemmProblem& p) {
  const bool dec = awq::decode_supported(p, nullptr);
  if (p.M <= 32 && dec) return awq::kDecode;
  const bool pre = awq::prefill_supported(p, nullptr);
  if (pre && dec) return prefill_faster(p) ? awq::kPrefill : awq::kDecode;
  if (pre) return awq::kPrefill;
  if (dec) return awq::kDecode;
  return awq::kGeneric;
}

awq_status_t run(const awq::GemmProblem& p, awq::Path path) {
  const char* why = "";
  cudaError_t e = cudaSuccess;
  switch (path) {
    case awq::kDecode:
      if (!awq::decode_supported(p, &why)) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "decode path: %s", why);
      e = awq::launch_decode(p);
      break;
    case awq::kPrefill:
      if (!awq::prefill_supported(p, &why)) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "prefill path: %s", why);
      e = awq::launch_prefill(p);
      break;
    case awq::kGeneric:
      e = awq::launch_generic(p);
      break;
    default:
      return fail(AWQ_ERR_INVALID_ARGUMENT, "unknown path %d", static_cast<int>(path));
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return ok();
}

}  // namespace

extern "C" {

int awq_runtime_available(void) {
  if (check_device() != AWQ_OK) return 0;
  cudaFuncAttributes attr;
  const cudaError_t e = awq::probe_kernel_image(&attr);
  if (e != cudaSuccess) {
    cuda_fail(e, "loading sm_103a kernels");
    return 0;
  }
  ok();
  return 1;
}

const char* awq_last_error(void) { return g_err.c_str(); }

const char* awq_status_string(awq_status_t s) {
  switch (s) {
    case AWQ_OK: return "AWQ_OK";
    case AWQ_ERR_INVALID_ARGUMENT: return "AWQ_ERR_INVALID_ARGUMENT";
    case AWQ_ERR_UNSUPPORTED_SHAPE: return "AWQ_ERR_UNSUPPORTED_SHAPE";
    case AWQ_ERR_MISALIGNED: return "AWQ_ERR_MISALIGNED";
    case AWQ_ERR_UNSUPPORTED_DEVICE: return "AWQ_ERR_UNSUPPORTED_DEVICE";
    case AWQ_ERR_CUDA: return "AWQ_ERR_CUDA";
    case AWQ_ERR_TIMEOUT: return "AWQ_ERR_TIMEOUT";
  }
  return "AWQ_ERR_UNKNOWN";
}

awq_status_t awq_dequant(const int32_t* qweight, const int32_t* qzeros, const void* scales_f16,
                         int64_t K, int64_t N, int64_t group_size, void* w_out,
                         awq_dtype_t out_dtype, awq_stream_t stream) {
  int G = 0;
  awq_status_t st = check_weight_shape(K, N, group_size, &G);
  if (st != AWQ_OK) return st;
  if (out_dtype != AWQ_DTYPE_F16 && out_dtype != AWQ_DTYPE_F32)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "out_dtype must be AWQ_DTYPE_F16 or AWQ_DTYPE_F32");
  if (N == 0) return ok();
  if (!qweight || !qzeros || !scales_f16 || !w_out)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "null pointer among qweight, qzeros, scales, w_out");
  if (!al(qweight, 4) || !al(qzeros, 4)) return fail(AWQ_ERR_MISALIGNED, "qweight/qzeros must be 4-byte aligned");
  if (!al(scales_f16, 2)) return fail(AWQ_ERR_MISALIGNED, "scales must be 2-byte aligned");
  if (!al(w_out, out_dtype == AWQ_DTYPE_F32 ? 4 : 2)) return fail(AWQ_ERR_MISALIGNED, "w_out misaligned for its dtype");
  st = check_device();
  if (st != AWQ_OK) return st;
  const cudaError_t e = awq::launch_dequant(
      reinterpret_cast<const uint32_t*>(qweight), reinterpret_cast<const uint32_t*>(qzeros),
      static_cast<const __half*>(scales_f16), static_cast<int>(K), static_cast<int>(N), G, w_out,
      out_dtype == AWQ_DTYPE_F32, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "awq_dequant launch");
  return ok();
}

awq_status_t awq_quantize_rtn(const void* w_f16, int64_t N, int64_t K, int64_t group_size,
                              int sym, int32_t* qweight, int32_t* qzeros, void* scales_f16,
                              awq_stream_t stream) {
  int G = 0;
  awq_status_t st = check_weight_shape(K, N, group_size, &G);
  if (st != AWQ_OK) return st;
  if (sym != 0 && sym != 1) return fail(AWQ_ERR_INVALID_ARGUMENT, "sym must be 0 or 1 (got %d)", sym);
  if (G % 8 != 0)
    return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "group size %d is not a multiple of 8 (16-byte group rows)", G);
  if (K / G > 65535) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "K / group_size must be at most 65535");
  if (N == 0) return ok();
  if (!w_f16 || !qweight || !qzeros || !scales_f16)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "null pointer among w, qweight, qzeros, scales");
  if (!al(w_f16, 16)) return fail(AWQ_ERR_MISALIGNED, "w must be 16-byte aligned");
  if (!al(qweight, 4) || !al(qzeros, 4)) return fail(AWQ_ERR_MISALIGNED, "qweight/qzeros must be 4-byte aligned");
  if (!al(scales_f16, 2)) return fail(AWQ_ERR_MISALIGNED, "scales must be 2-byte aligned");
  st = check_device();
  if (st != AWQ_OK) return st;
  const cudaError_t e = awq::launch_quantize_rtn(
      static_cast<const __half*>(w_f16), static_cast<int>(N), static_cast<int>(K), G, sym == 1,
      reinterpret_cast<uint32_t*>(qweight), reinterpret_cast<uint32_t*>(qzeros),
      static_cast<__half*>(scales_f16), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "awq_quantize_rtn launch");
  return ok();
}

static awq_status_t gemm_any(const void* x, const int32_t* qweight, const int32_t* qzeros,
                      const void* scales, const void* bias, int64_t M, int64_t K, int64_t N,
                      int64_t group_size, void* y, awq_path_t path, awq_stream_t stream, bool bf16,
                      int bits = 4, uint32_t flags = 0u) {
  if (path < AWQ_PATH_AUTO || path > AWQ_PATH_GENERIC)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "unknown path %d", static_cast<int>(path));
  if ((flags & ~static_cast<uint32_t>(AWQ_GEMM_STATIC_WEIGHTS)) != 0u)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "unknown flag bits 0x%x", flags);
  awq::GemmProblem p{};
  bool empty = false;
  awq_status_t st = build_problem(x, qweight, qzeros, scales, bias, M, K, N, group_size, y,
                                  stream, &p, &empty, bf16, bits);
  if (st != AWQ_OK) return st;
  if (empty) return ok();
  p.static_weights = (flags & AWQ_GEMM_STATIC_WEIGHTS) != 0u;
  st = check_device();
  if (st != AWQ_OK) return st;
  const awq::Path use = path == AWQ_PATH_AUTO ? choose_path(p) : static_cast<awq::Path>(path);
  return run(p, use);
}

awq_status_t awq_gemm_any(const void* x, const int32_t* qweight, const int32_t* qzeros,
                          const void* scales, const void* bias, int64_t M, int64_t K, int64_t N,
                          int64_t group_size, void* y, awq_dtype_t dtype, int32_t bits,
                          awq_path_t path, uint32_t flags, awq_stream_t stream) {
  if (dtype != AWQ_DTYPE_F16 && dtype != AWQ_DTYPE_BF16)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "dtype must be AWQ_DTYPE_F16 or AWQ_DTYPE_BF16");
  if (bits != 4 && bits != 8) return fail(AWQ_ERR_INVALID_ARGUMENT, "bits must be 4 or 8 (got %d)", bits);
  if (bits == 8 && dtype != AWQ_DTYPE_F16)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "8-bit codes take fp16 activations and scales");
  return gemm_any(x, qweight, qzeros, scales, bias, M, K, N, group_size, y, path, stream,
                  dtype == AWQ_DTYPE_BF16, bits, flags);
}

awq_status_t awq_gemm_ex(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                         const void* scales_f16, const void* bias_f16, int64_t M, int64_t K,
                         int64_t N, int64_t group_size, void* y_f16, awq_path_t path,
                         awq_stream_t stream) {
  return gemm_any(x_f16, qweight, qzeros, scales_f16, bias_f16, M, K, N, group_size, y_f16, path,
                  stream, false);
}

awq_status_t awq_gemm_bf16_ex(const void* x_bf16, const int32_t* qweight, const int32_t* qzeros,
                              const void* scales_bf16, const void* bias_bf16, int64_t M, int64_t K,
                              int64_t N, int64_t group_size, void* y_bf16, awq_path_t path,
                              awq_stream_t stream) {
  return gemm_any(x_bf16, qweight, qzeros, scales_bf16, bias_bf16, M, K, N, group_size, y_bf16,
                  path, stream, true);
}

awq_status_t awq_gemm_grouped(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                              const void* scales_f16, const void* bias_f16,
                              const int32_t* expert_offsets, int64_t R, int64_t E, int64_t K,
                              int64_t N, int64_t group_size, void* y_f16, awq_stream_t stream) {
  if (E <= 0 || E > 4096) return fail(AWQ_ERR_INVALID_ARGUMENT, "E must be in 1..4096 (got %lld)", (long long)E);
  awq::GemmProblem p{};
  bool empty = false;
  awq_status_t st = build_problem(x_f16, qweight, qzeros, scales_f16, bias_f16, R, K, N, group_size,
                                  y_f16, stream, &p, &empty, false);
  if (st != AWQ_OK) return st;
  if (K * N * E >= kProdLimit) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "E*K*N must be below 2^40");
  if ((R + 7) / 8 + E > 65535) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "R/8 + E must be at most 65535");
  if (empty) return ok();
  if (!expert_offsets) return fail(AWQ_ERR_INVALID_ARGUMENT, "null expert_offsets");
  if (!al(expert_offsets, 4)) return fail(AWQ_ERR_MISALIGNED, "expert_offsets must be 4-byte aligned");
  p.offsets = expert_offsets;
  p.E = static_cast<int>(E);
  const char* why = "";
  if (!awq::decode_grouped_supported(p, &why)) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "grouped: %s", why);
  st = check_device();
  if (st != AWQ_OK) return st;
  const cudaError_t e = awq::launch_decode_grouped(p);
  if (e != cudaSuccess) return cuda_fail(e, "awq_gemm_grouped launch");
  return ok();
}

awq_status_t awq_gemm_w8_ex(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                            const void* scales_f16, const void* bias_f16, int64_t M, int64_t K,
                            int64_t N, int64_t group_size, void* y_f16, awq_path_t path,
                            awq_stream_t stream) {
  return gemm_any(x_f16, qweight, qzeros, scales_f16, bias_f16, M, K, N, group_size, y_f16, path,
                  stream, false, 8);
}

awq_status_t awq_gemm_w8(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                         const void* scales_f16, const void* bias_f16, int64_t M, int64_t K,
                         int64_t N, int64_t group_size, void* y_f16, awq_stream_t stream) {
  return gemm_any(x_f16, qweight, qzeros, scales_f16, bias_f16, M, K, N, group_size, y_f16,
                  AWQ_PATH_AUTO, stream, false, 8);
}

awq_status_t awq_dequant_w8(const int32_t* qweight, const int32_t* qzeros, const void* scales_f16,
                            int64_t K, int64_t N, int64_t group_size, void* w_out,
                            awq_dtype_t out_dtype, awq_stream_t stream) {
  int G = 0;
  awq_status_t st = check_weight_shape(K, N, group_size, &G, 4);
  if (st != AWQ_OK) return st;
  if (out_dtype != AWQ_DTYPE_F16 && out_dtype != AWQ_DTYPE_F32)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "out_dtype must be AWQ_DTYPE_F16 or AWQ_DTYPE_F32");
  if (N == 0) return ok();
  if (!qweight || !qzeros || !scales_f16 || !w_out)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "null pointer among qweight, qzeros, scales, w_out");
  if (!al(qweight, 4) || !al(qzeros, 4)) return fail(AWQ_ERR_MISALIGNED, "qweight/qzeros must be 4-byte aligned");
  if (!al(scales_f16, 2)) return fail(AWQ_ERR_MISALIGNED, "scales must be 2-byte aligned");
  if (!al(w_out, out_dtype == AWQ_DTYPE_F32 ? 4 : 2)) return fail(AWQ_ERR_MISALIGNED, "w_out misaligned for its dtype");
  st = check_device();
  if (st != AWQ_OK) return st;
  const cudaError_t e = awq::launch_dequant8(
      reinterpret_cast<const uint32_t*>(qweight), reinterpret_cast<const uint32_t*>(qzeros),
      static_cast<const __half*>(scales_f16), static_cast<int>(K), static_cast<int>(N), G, w_out,
      out_dtype == AWQ_DTYPE_F32, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "awq_dequant_w8 launch");
  return ok();
}

awq_status_t awq_gemm_bf16(const void* x_bf16, const int32_t* qweight, const int32_t* qzeros,
                           const void* scales_bf16, const void* bias_bf16, int64_t M, int64_t K,
                           int64_t N, int64_t group_size, void* y_bf16, awq_stream_t stream) {
  return gemm_any(x_bf16, qweight, qzeros, scales_bf16, bias_bf16, M, K, N, group_size, y_bf16,
                  AWQ_PATH_AUTO, stream, true);
}

awq_status_t awq_dequant_bf16(const int32_t* qweight, const int32_t* qzeros, const void* scales_bf16,
                              int64_t K, int64_t N, int64_t group_size, void* w_out,
                              awq_dtype_t out_dtype, awq_stream_t stream) {
  int G = 0;
  awq_status_t st = check_weight_shape(K, N, group_size, &G);
  if (st != AWQ_OK) return st;
  if (out_dtype != AWQ_DTYPE_BF16 && out_dtype != AWQ_DTYPE_F32)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "out_dtype must be AWQ_DTYPE_BF16 or AWQ_DTYPE_F32");
  if (N == 0) return ok();
  if (!qweight || !qzeros || !scales_bf16 || !w_out)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "null pointer among qweight, qzeros, scales, w_out");
  if (!al(qweight, 4) || !al(qzeros, 4)) return fail(AWQ_ERR_MISALIGNED, "qweight/qzeros must be 4-byte aligned");
  if (!al(scales_bf16, 2)) return fail(AWQ_ERR_MISALIGNED, "scales must be 2-byte aligned");
  if (!al(w_out, out_dtype == AWQ_DTYPE_F32 ? 4 : 2)) return fail(AWQ_ERR_MISALIGNED, "w_out misaligned for its dtype");
  st = check_device();
  if (st != AWQ_OK) return st;
  const cudaError_t e = awq::launch_dequant(
      reinterpret_cast<const uint32_t*>(qweight), reinterpret_cast<const uint32_t*>(qzeros),
      static_cast<const __half*>(scales_bf16), static_cast<int>(K), static_cast<int>(N), G, w_out,
      out_dtype == AWQ_DTYPE_F32, reinterpret_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return cuda_fail(e, "awq_dequant_bf16 launch");
  return ok();
}

awq_status_t awq_gemm(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                      const void* scales_f16, const void* bias_f16, int64_t M, int64_t K,
                      int64_t N, int64_t group_size, void* y_f16, awq_stream_t stream) {
  return awq_gemm_ex(x_f16, qweight, qzeros, scales_f16, bias_f16, M, K, N, group_size, y_f16,
                     AWQ_PATH_AUTO, stream);
}

awq_path_t awq_gemm_select_path(int64_t M, int64_t K, int64_t N, int64_t group_size,
                                const void* x_f16, const int32_t* qweight,
                                const int32_t* qzeros, const void* scales_f16,
                                const void* bias_f16, const void* y_f16) {
  awq::GemmProblem p{};
  bool empty = false;
  if (build_problem(x_f16, qweight, qzeros, scales_f16, bias_f16, M, K, N, group_size,
                    const_cast<void*>(y_f16), nullptr, &p, &empty) != AWQ_OK || empty)
    return AWQ_PATH_AUTO;
  ok();
  return static_cast<awq_path_t>(choose_path(p));
}

awq_path_t awq_gemm_select_path_ex(int64_t M, int64_t K, int64_t N, int64_t group_size,
                                   const void* x, const int32_t* qweight, const int32_t* qzeros,
                                   const void* scales, const void* bias, const void* y,
                                   awq_dtype_t dtype, int32_t bits) {
  if ((dtype != AWQ_DTYPE_F16 && dtype != AWQ_DTYPE_BF16) || (bits != 4 && bits != 8) ||
      (bits == 8 && dtype != AWQ_DTYPE_F16))
    return AWQ_PATH_AUTO;
  awq::GemmProblem p{};
  bool empty = false;
  if (build_problem(x, qweight, qzeros, scales, bias, M, K, N, group_size, const_cast<void*>(y),
                    nullptr, &p, &empty, dtype == AWQ_DTYPE_BF16, bits) != AWQ_OK || empty)
    return AWQ_PATH_AUTO;
  ok();
  return static_cast<awq_path_t>(choose_path(p));
}

// Tile-packed layout of 4- or 8-bit codes: size and the one-off conversion.
static awq_status_t repack_size_bits(int64_t K, int64_t N, int64_t group_size, size_t* bytes, int bits) {
  int G = 0;
  awq_status_t st = check_weight_shape(K, N, group_size, &G, bits == 8 ? 4 : 8);
  if (st != AWQ_OK) return st;
  if (!bytes) return fail(AWQ_ERR_INVALID_ARGUMENT, "null bytes pointer");
  const char* why = "";
  if (!(bits == 8 ? awq::packed8_supported(K, N, G, &why) : awq::packed_supported(K, N, G, &why)))
    return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "%s", why);
  *bytes = bits == 8 ? awq::packed8_bytes(K, N) : awq::packed_bytes(K, N);
  return ok();
}

static awq_status_t repack_bits(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                                int64_t K, int64_t N, int64_t group_size, void* packed_out,
                                awq_stream_t stream, int bits) {
  int G = 0;
  awq_status_t st = check_weight_shape(K, N, group_size, &G, bits == 8 ? 4 : 8);
  if (st != AWQ_OK) return st;
  const char* why = "";
  if (!(bits == 8 ? awq::packed8_supported(K, N, G, &why) : awq::packed_supported(K, N, G, &why)))
    return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "%s", why);
  if (N == 0) return ok();
  if (!qweight || !qzeros || !scales || !packed_out)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "null pointer among qweight, qzeros, scales, packed_out");
  if (!al(qweight, 4) || !al(qzeros, 4)) return fail(AWQ_ERR_MISALIGNED, "qweight/qzeros must be 4-byte aligned");
  if (!al(scales, 2)) return fail(AWQ_ERR_MISALIGNED, "scales must be 2-byte aligned");
  if (!al(packed_out, 16)) return fail(AWQ_ERR_MISALIGNED, "packed_out must be 16-byte aligned");
  if (K / 64 > 65535) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "K / 64 must be at most 65535");
  st = check_device();
  if (st != AWQ_OK) return st;
  const auto* qw = reinterpret_cast<const uint32_t*>(qweight);
  const auto* qz = reinterpret_cast<const uint32_t*>(qzeros);
  const auto* sc = static_cast<const __half*>(scales);
  const auto strm = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      bits == 8 ? awq::launch_repack8(qw, qz, sc, static_cast<int>(K), static_cast<int>(N), G, packed_out, strm)
                : awq::launch_repack(qw, qz, sc, static_cast<int>(K), static_cast<int>(N), G, packed_out, strm);
  if (e != cudaSuccess) return cuda_fail(e, "awq_repack launch");
  return ok();
}

awq_status_t awq_repack_size(int64_t K, int64_t N, int64_t group_size, size_t* bytes) {
  return repack_size_bits(K, N, group_size, bytes, 4);
}
awq_status_t awq_repack(const int32_t* qweight, const int32_t* qzeros, const void* scales_f16,
                        int64_t K, int64_t N, int64_t group_size, void* packed_out,
                        awq_stream_t stream) {
  return repack_bits(qweight, qzeros, scales_f16, K, N, group_size, packed_out, stream, 4);
}
awq_status_t awq_repack_w8_size(int64_t K, int64_t N, int64_t group_size, size_t* bytes) {
  return repack_size_bits(K, N, group_size, bytes, 8);
}
awq_status_t awq_repack_w8(const int32_t* qweight, const int32_t* qzeros, const void* scales_f16,
                           int64_t K, int64_t N, int64_t group_size, void* packed_out,
                           awq_stream_t stream) {
  return repack_bits(qweight, qzeros, scales_f16, K, N, group_size, packed_out, stream, 8);
}

// Checks of the packed linear's arguments; fills *p, and *launch = false when there is nothing
// to compute (M == 0 or N == 0).
static awq_status_t packed_problem(const void* x_f16, const void* packed, const void* bias_f16, int64_t M,
                                   int64_t K, int64_t N, int64_t group_size, void* y_f16,
                                   awq_stream_t stream, awq::GemmProblem* p, bool* launch, bool bf16 = false,
                                   int bits = 4) {
  *launch = false;
  if (M < 0) return fail(AWQ_ERR_INVALID_ARGUMENT, "M must be >= 0 (got %lld)", (long long)M);
  int G = 0;
  awq_status_t st = check_weight_shape(K, N, group_size, &G, bits == 8 ? 4 : 8);
  if (st != AWQ_OK) return st;
  const char* why = "";
  if (!(bits == 8 ? awq::packed8_supported(K, N, G, &why) : awq::packed_supported(K, N, G, &why)))
    return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "%s", why);
  if (M > kDimLimit) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "M must be below 2^31");
  if (M * N >= kProdLimit || M * K >= kProdLimit)
    return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "M*N and M*K must be below 2^40");
  if (M == 0 || N == 0) return ok();
  if (!x_f16 || !packed || !y_f16) return fail(AWQ_ERR_INVALID_ARGUMENT, "null pointer among x, packed, y");
  if (!al(x_f16, 16)) return fail(AWQ_ERR_MISALIGNED, "x must be 16-byte aligned");
  if (!al(packed, 16)) return fail(AWQ_ERR_MISALIGNED, "packed must be 16-byte aligned");
  if (!al(y_f16, 2) || (bias_f16 && !al(bias_f16, 2)))
    return fail(AWQ_ERR_MISALIGNED, "y and bias must be 2-byte aligned");
  st = check_device();
  if (st != AWQ_OK) return st;
  p->x = static_cast<const __half*>(x_f16);
  p->bias = static_cast<const __half*>(bias_f16);
  p->y = static_cast<__half*>(y_f16);
  p->M = static_cast<int>(M);
  p->K = static_cast<int>(K);
  p->N = static_cast<int>(N);
  p->G = G;
  p->stream = reinterpret_cast<cudaStream_t>(stream);
  p->bf16 = bf16;
  p->bits = bits;
  *launch = true;
  return ok();
}

static awq_status_t gemm_packed(const void* x_f16, const void* packed, const void* bias_f16, int64_t M,
                                int64_t K, int64_t N, int64_t group_size, void* y_f16, void* workspace,
                                size_t workspace_bytes, awq_stream_t stream) {
  awq::GemmProblem p{};
  bool launch = false;
  const awq_status_t st = packed_problem(x_f16, packed, bias_f16, M, K, N, group_size, y_f16, stream, &p, &launch);
  if (st != AWQ_OK || !launch) return st;
  const cudaError_t e = awq::launch_packed(p, packed, workspace, workspace_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "awq_gemm_packed launch");
  return ok();
}

awq_status_t awq_gemm_packed(const void* x_f16, const void* packed, const void* bias_f16, int64_t M,
                             int64_t K, int64_t N, int64_t group_size, void* y_f16,
                             awq_stream_t stream) {
  return gemm_packed(x_f16, packed, bias_f16, M, K, N, group_size, y_f16, nullptr, 0, stream);
}

awq_status_t awq_gemm_packed_workspace_size(size_t* bytes) {
  if (!bytes) return fail(AWQ_ERR_INVALID_ARGUMENT, "null bytes pointer");
  awq_status_t st = check_device();
  if (st != AWQ_OK) return st;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "reading the SM count");
  *bytes = awq::packed_workspace_bytes(sms);
  return ok();
}

awq_status_t awq_gemm_packed_noalloc(const void* x_f16, const void* packed, const void* bias_f16, int64_t M,
                                     int64_t K, int64_t N, int64_t group_size, void* y_f16,
                                     awq_stream_t stream) {
  awq::GemmProblem p{};
  bool launch = false;
  awq_status_t st = packed_problem(x_f16, packed, bias_f16, M, K, N, group_size, y_f16, stream, &p, &launch);
  if (st != AWQ_OK || !launch) return st;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "reading the SM count");
  const size_t need = awq::packed_workspace_bytes(sms);
  if (need > awq::packed_static_scratch_bytes())
    return fail(AWQ_ERR_UNSUPPORTED_DEVICE,
                "this device's %d SMs need %zu bytes of scratch, more than the %zu-byte static array", sms,
                need, awq::packed_static_scratch_bytes());
  void* scratch = nullptr;
  e = awq::packed_static_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "locating the static scratch");
  // the ready flags start every call lowered (a call that gave up a wait may leave some raised)
  e = cudaMemsetAsync(scratch, 0, awq::packed_workspace_flag_bytes(sms), p.stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the scratch flags");
  e = awq::launch_packed(p, packed, scratch, need);
  if (e != cudaSuccess) return cuda_fail(e, "awq_gemm_packed_noalloc launch");
  return ok();
}

awq_status_t awq_gemm_packed_ex(const void* x, const void* packed, const void* bias, int64_t M, int64_t K,
                                int64_t N, int64_t group_size, void* y, awq_dtype_t dtype, void* workspace,
                                size_t workspace_bytes, awq_stream_t stream) {
  if (dtype != AWQ_DTYPE_F16 && dtype != AWQ_DTYPE_BF16)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "dtype must be AWQ_DTYPE_F16 or AWQ_DTYPE_BF16");
  if (workspace && !al(workspace, 256)) return fail(AWQ_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  awq::GemmProblem p{};
  bool launch = false;
  const awq_status_t st = packed_problem(x, packed, bias, M, K, N, group_size, y, stream, &p, &launch,
                                         dtype == AWQ_DTYPE_BF16);
  if (st != AWQ_OK || !launch) return st;
  const cudaError_t e = awq::launch_packed(p, packed, workspace, workspace_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "awq_gemm_packed_ex launch");
  return ok();
}

awq_status_t awq_gemm_packed_w8(const void* x_f16, const void* packed, const void* bias_f16, int64_t M,
                                int64_t K, int64_t N, int64_t group_size, void* y_f16, void* workspace,
                                size_t workspace_bytes, awq_stream_t stream) {
  if (workspace && !al(workspace, 256)) return fail(AWQ_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  awq::GemmProblem p{};
  bool launch = false;
  const awq_status_t st = packed_problem(x_f16, packed, bias_f16, M, K, N, group_size, y_f16, stream, &p,
                                         &launch, false, 8);
  if (st != AWQ_OK || !launch) return st;
  const cudaError_t e = awq::launch_packed(p, packed, workspace, workspace_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "awq_gemm_packed_w8 launch");
  return ok();
}

awq_status_t awq_gemm_packed_grouped(const void* x, const void* packed, const void* bias,
                                     const int32_t* expert_offsets, int64_t R, int64_t E, int64_t K,
                                     int64_t N, int64_t group_size, void* y, awq_dtype_t dtype,
                                     awq_stream_t stream) {
  if (dtype != AWQ_DTYPE_F16 && dtype != AWQ_DTYPE_BF16)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "dtype must be AWQ_DTYPE_F16 or AWQ_DTYPE_BF16");
  if (E <= 0 || E > awq::kPackedGroupedMaxE)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "E must be in 1..%d (got %lld)", awq::kPackedGroupedMaxE, (long long)E);
  awq::GemmProblem p{};
  bool launch = false;
  awq_status_t st = packed_problem(x, packed, bias, R, K, N, group_size, y, stream, &p, &launch,
                                   dtype == AWQ_DTYPE_BF16);
  if (st != AWQ_OK || !launch) return st;
  if (K * N * E >= kProdLimit) return fail(AWQ_ERR_UNSUPPORTED_SHAPE, "E*K*N must be below 2^40");
  if (!expert_offsets) return fail(AWQ_ERR_INVALID_ARGUMENT, "null expert_offsets");
  if (!al(expert_offsets, 4)) return fail(AWQ_ERR_MISALIGNED, "expert_offsets must be 4-byte aligned");
  p.offsets = expert_offsets;
  p.E = static_cast<int>(E);
  const cudaError_t e = awq::launch_packed_grouped(p, packed);
  if (e != cudaSuccess) return cuda_fail(e, "awq_gemm_packed_grouped launch");
  return ok();
}

awq_status_t awq_gemm_packed_ws(const void* x_f16, const void* packed, const void* bias_f16, int64_t M,
                                int64_t K, int64_t N, int64_t group_size, void* y_f16, void* workspace,
                                size_t workspace_bytes, awq_stream_t stream) {
  if (workspace && !al(workspace, 256)) return fail(AWQ_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  return gemm_packed(x_f16, packed, bias_f16, M, K, N, group_size, y_f16, workspace, workspace_bytes, stream);
}

awq_status_t awq_device_status(awq_stream_t stream) {
  awq_status_t st = check_device();
  if (st != AWQ_OK) return st;
  unsigned int v = 0u;
  const cudaError_t e = awq::read_and_clear_status(reinterpret_cast<cudaStream_t>(stream), &v);
  if (e != cudaSuccess) return cuda_fail(e, "reading device status");
  if (v != 0u) return fail(AWQ_ERR_TIMEOUT, "a kernel gave up a bounded wait (code 0x%x)", v);
  return ok();
}

awq_status_t awq_selftest_wait_timeout(uint64_t limit_ns, awq_stream_t stream) {
  if (limit_ns < 1000ull || limit_ns > 1000000000ull)
    return fail(AWQ_ERR_INVALID_ARGUMENT, "limit_ns must be within [1e3, 1e9]");
  awq_status_t st = check_device();
  if (st != AWQ_OK) return st;
  const cudaError_t e = awq::launch_selftest_wait(static_cast<unsigned long long>(limit_ns),
                                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the wait self test");
  return ok();
}

}  // extern "C"
