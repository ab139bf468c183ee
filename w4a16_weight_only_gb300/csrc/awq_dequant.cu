// awq_dequant: full unpack + dequant of an AWQ GEMM-layout weight to a dense [K, N]
// matrix, and the generic (any-shape) fused GEMM used for ragged shapes.
//
// Unpack and dequant follow tensref.org/formats/awq, "Reader": nibble i of packed word c
// holds column 8c + ORDER[i]; w = (code - zero) * scale with the scale/zero row k / G and
// no +1 on the zero (reject rule AWQ-005 on the same page).
#include "awq_internal.cuh"

namespace awq {
namespace {

// Each thread handles one packed word (8 output columns of one row) per iteration.
// The fp32 value (code - zero) * scale is exact (a 5-bit integer times an 11-bit
// significand); the fp16 output is that value rounded once to nearest even.
template <bool kF32, bool kVec, bool kBF>
__global__ void __launch_bounds__(256) dequant_kernel(const uint32_t* __restrict__ qw,
                                                      const uint32_t* __restrict__ qz,
                                                      const __half* __restrict__ sc, int K, int C,
                                                      int G, void* __restrict__ out) {
  const long long total = (long long)K * C;
  const long long N = 8LL * C;
  for (long long w = blockIdx.x * (long long)blockDim.x + threadIdx.x; w < total;
       w += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(w / C);
    const int cw = (int)(w - (long long)k * C);
    const int g = k / G;
    const uint32_t q = __ldcs(qw + w);
    const uint32_t z = __ldg(qz + (long long)g * C + cw);
    const __half* srow = sc + (long long)g * N + 8LL * cw;
    __half s[8];
    if (kVec) {
      *reinterpret_cast<uint4*>(s) = __ldg(reinterpret_cast<const uint4*>(srow));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) s[j] = srow[j];
    }
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int code = (int)((q >> (4 * i)) & 0xFu);
      const int zero = (int)((z >> (4 * i)) & 0xFu);
      v[nibble_column(i)] = __fmul_rn((float)(code - zero), elem_to_float<kBF>(__half_as_ushort(s[nibble_column(i)])));
    }
    const long long o = (long long)k * N + 8LL * cw;
    if (kF32) {
      float* dst = static_cast<float*>(out) + o;
      if (kVec) {
        __stcs(reinterpret_cast<float4*>(dst), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4*>(dst) + 1, make_float4(v[4], v[5], v[6], v[7]));
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = v[j];
      }
    } else {
      uint16_t* dst = static_cast<uint16_t*>(out) + o;
      uint16_t h[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) h[j] = float_to_elem<kBF>(v[j]);
      if (kVec) {
        __stcs(reinterpret_cast<uint4*>(dst), *reinterpret_cast<uint4*>(h));
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = h[j];
      }
    }
  }
}

// 8-bit codes: one thread per packed word (4 output columns, byte i = column 4c + i); the
// fp32 value (code - zero) * scale is exact (a 9-bit integer times an 11-bit significand).
template <bool kF32>
__global__ void __launch_bounds__(256) dequant8_kernel(const uint32_t* __restrict__ qw,
                                                       const uint32_t* __restrict__ qz,
                                                       const __half* __restrict__ sc, int K, int C,
                                                       int G, void* __restrict__ out) {
  const long long total = (long long)K * C;
  const long long N = 4LL * C;
  for (long long w = blockIdx.x * (long long)blockDim.x + threadIdx.x; w < total;
       w += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(w / C);
    const int cw = (int)(w - (long long)k * C);
    const int g = k / G;
    const uint32_t q = __ldcs(qw + w);
    const uint32_t z = __ldg(qz + (long long)g * C + cw);
    const __half* srow = sc + (long long)g * N + 4LL * cw;
    const long long o = (long long)k * N + 4LL * cw;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int code = (int)((q >> (8 * i)) & 0xFFu);
      const int zero = (int)((z >> (8 * i)) & 0xFFu);
      const float v = __fmul_rn((float)(code - zero), __half2float(srow[i]));
      if (kF32) static_cast<float*>(out)[o + i] = v;
      else static_cast<__half*>(out)[o + i] = __float2half_rn(v);
    }
  }
}

// Generic fused GEMM: one thread per output column, kMT activation rows per block row,
// activations staged through shared memory in kKT-wide slices.  fp32 accumulation in
// increasing k order.  Used for shapes the fast kernels do not take (K or G not a
// multiple of 16, N not a multiple of the decode tile, unaligned pointers).
constexpr int kMT = 8;
constexpr int kKT = 64;

template <bool kBF, int kBits>
__global__ void __launch_bounds__(128) generic_gemm_kernel(GemmProblem p) {
  const uint16_t* x16 = reinterpret_cast<const uint16_t*>(p.x);
  const uint16_t* sc16 = reinterpret_cast<const uint16_t*>(p.sc);
  __shared__ float xs[kMT][kKT];
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int C = kBits == 4 ? p.N >> 3 : p.N >> 2;
  const bool active = n < p.N;
  const int cw = kBits == 4 ? n >> 3 : n >> 2;
  const int j = n & 7;
  // bit offset of column n in its word: nibble holding column j (inverse of ORDER), or byte n % 4
  const int shift = kBits == 4 ? 4 * (((j & 1) << 2) | (j >> 1)) : 8 * (n & 3);
  const uint32_t mask = kBits == 4 ? 0xFu : 0xFFu;
  for (int m0 = blockIdx.y * kMT; m0 < p.M; m0 += gridDim.y * kMT) {
  float acc[kMT];
#pragma unroll
  for (int m = 0; m < kMT; ++m) acc[m] = 0.f;
  for (int k0 = 0; k0 < p.K; k0 += kKT) {
    __syncthreads();
    for (int e = threadIdx.x; e < kMT * kKT; e += blockDim.x) {
      const int m = e / kKT, kk = e % kKT;
      const int gm = m0 + m, gk = k0 + kk;
      xs[m][kk] = (gm < p.M && gk < p.K) ? elem_to_float<kBF>(x16[(long long)gm * p.K + gk]) : 0.f;
    }
    __syncthreads();
    if (active) {
      const int kend = min(kKT, p.K - k0);
      for (int kk = 0; kk < kend; ++kk) {
        const int k = k0 + kk;
        const int g = k / p.G;
        const uint32_t q = p.qw[(long long)k * C + cw];
        const uint32_t z = p.qz[(long long)g * C + cw];
        const int code = (int)((q >> shift) & mask);
        const int zero = (int)((z >> shift) & mask);
        const float w = __fmul_rn((float)(code - zero), elem_to_float<kBF>(sc16[(long long)g * p.N + n]));
#pragma unroll
        for (int m = 0; m < kMT; ++m) acc[m] = __fmaf_rn(xs[m][kk], w, acc[m]);
      }
    }
  }
  if (active) {
    const float b = p.bias ? elem_to_float<kBF>(reinterpret_cast<const uint16_t*>(p.bias)[n]) : 0.f;
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
      const int gm = m0 + m;
      if (gm < p.M) reinterpret_cast<uint16_t*>(p.y)[(long long)gm * p.N + n] = float_to_elem<kBF>(acc[m] + b);
    }
  }
  }  // m0
}

template <bool kBF>
void launch_dequant_t(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int C, int G,
                      void* out, bool out_f32, bool vec, int blocks, cudaStream_t stream) {
  if (out_f32) {
    if (vec) dequant_kernel<true, true, kBF><<<blocks, 256, 0, stream>>>(qw, qz, sc, K, C, G, out);
    else dequant_kernel<true, false, kBF><<<blocks, 256, 0, stream>>>(qw, qz, sc, K, C, G, out);
  } else {
    if (vec) dequant_kernel<false, true, kBF><<<blocks, 256, 0, stream>>>(qw, qz, sc, K, C, G, out);
    else dequant_kernel<false, false, kBF><<<blocks, 256, 0, stream>>>(qw, qz, sc, K, C, G, out);
  }
}

}  // namespace

cudaError_t launch_dequant(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int N,
                           int G, void* out, bool out_f32, cudaStream_t stream, bool bf16) {
  const int C = N / 8;
  const long long total = (long long)K * C;
  if (total == 0) return cudaSuccess;
  const bool vec = aligned(sc, 16) && aligned(out, out_f32 ? 16 : 16);
  int blocks = (int)((total + 255) / 256);
  const int cap = 152 * 16;
  if (blocks > cap) blocks = cap;
  if (bf16) launch_dequant_t<true>(qw, qz, sc, K, C, G, out, out_f32, vec, blocks, stream);
  else launch_dequant_t<false>(qw, qz, sc, K, C, G, out, out_f32, vec, blocks, stream);
  return cudaGetLastError();
}

cudaError_t launch_dequant8(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int N,
                            int G, void* out, bool out_f32, cudaStream_t stream) {
  const int C = N / 4;
  const long long total = (long long)K * C;
  if (total == 0) return cudaSuccess;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (out_f32) dequant8_kernel<true><<<blocks, 256, 0, stream>>>(qw, qz, sc, K, C, G, out);
  else dequant8_kernel<false><<<blocks, 256, 0, stream>>>(qw, qz, sc, K, C, G, out);
  return cudaGetLastError();
}

cudaError_t probe_kernel_image(cudaFuncAttributes* attr) {
  return cudaFuncGetAttributes(attr, dequant_kernel<false, true, false>);
}

cudaError_t launch_generic(const GemmProblem& p) {
  const int mtiles = (p.M + kMT - 1) / kMT;
  dim3 grid((p.N + 127) / 128, mtiles < 65535 ? mtiles : 65535);
  if (p.bits == 8) generic_gemm_kernel<false, 8><<<grid, 128, 0, p.stream>>>(p);
  else if (p.bf16) generic_gemm_kernel<true, 4><<<grid, 128, 0, p.stream>>>(p);
  else generic_gemm_kernel<false, 4><<<grid, 128, 0, p.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace awq
