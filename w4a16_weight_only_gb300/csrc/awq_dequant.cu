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

// Generic fused GEMM, for the shapes the tensor-core kernels do not take (any K, any group
// size dividing K, any N the packing allows, 4-byte aligned words and 2-byte aligned
// elements).  A CTA of kGW warps owns TW consecutive packed words of every row (the
// TW * 32 / kBits columns they hold) and MT activation rows; K is cut into kGW contiguous
// chunks, one per warp.  Inside a warp lane (kr, w) takes word w of rows kr, kr + LK,
// kr + 2 LK, ... of the chunk (LK = 32 / TW), so one load instruction reads LK whole row
// segments of the tile.  Per group a lane accumulates sum x * code for each of its
// columns and sum x (fp32), and folds them once at the group's end:
// acc += scale * (sum x code - zero * sum x).  The LK lanes of a word are then added by
// butterfly shuffles, the warps in warp order through shared memory, the bias last, and
// y is rounded once.  Every order is fixed: repeated calls give the same bits.
constexpr int kGW = 16;

template <bool kBF, int kBits, int TW, int MT>
__global__ void __launch_bounds__(kGW * 32, 1) generic_gemm_kernel(GemmProblem p) {
  constexpr int CPW = 32 / kBits;  // columns per packed word
  constexpr int LK = 32 / TW;      // rows of K a warp step covers
  constexpr int NC = TW * CPW;     // columns of the tile
  constexpr uint32_t kMask = kBits == 4 ? 0xFu : 0xFFu;
  __shared__ float part[kGW][MT][NC];
  const uint16_t* x16 = reinterpret_cast<const uint16_t*>(p.x);
  const uint16_t* sc16 = reinterpret_cast<const uint16_t*>(p.sc);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int kr = lane / TW, wi = lane % TW;
  const int C = p.N / CPW;
  const int cw = blockIdx.x * TW + wi;
  const bool col_ok = cw < C;
  const int chunk = ((p.K + kGW - 1) / kGW + LK - 1) / LK * LK;
  const int klo = min(p.K, warp * chunk), khi = min(p.K, klo + chunk);
  // bit offset of column j of a word: the nibble holding it (inverse of ORDER), or byte j
  auto shift_of = [](int j) { return kBits == 4 ? 4 * (((j & 1) << 2) | (j >> 1)) : 8 * j; };
  for (int m0 = blockIdx.y * MT; m0 < p.M; m0 += gridDim.y * MT) {
    float acc[MT][CPW];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int j = 0; j < CPW; ++j) acc[m][j] = 0.f;
    int k = klo + kr;
    if (col_ok && k < khi) {
      float a[MT][CPW], sx[MT], zf[CPW], sf[CPW];
      int g = k / p.G, gend = (g + 1) * p.G;
      auto open_group = [&]() {
        const uint32_t z = p.qz[(long long)g * C + cw];
#pragma unroll
        for (int j = 0; j < CPW; ++j) {
          zf[j] = static_cast<float>((z >> shift_of(j)) & kMask);
          sf[j] = elem_to_float<kBF>(sc16[(long long)g * p.N + CPW * cw + j]);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          sx[m] = 0.f;
#pragma unroll
          for (int j = 0; j < CPW; ++j) a[m][j] = 0.f;
        }
      };
      auto fold = [&]() {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int j = 0; j < CPW; ++j)
            acc[m][j] = __fmaf_rn(sf[j], __fmaf_rn(-zf[j], sx[m], a[m][j]), acc[m][j]);
      };
      open_group();
      for (; k < khi; k += LK) {
        if (k >= gend) {
          fold();
          g = k / p.G;
          gend = (g + 1) * p.G;
          open_group();
        }
        const uint32_t q = p.qw[(long long)k * C + cw];
        float xv[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m)
          xv[m] = (m0 + m < p.M) ? elem_to_float<kBF>(x16[(long long)(m0 + m) * p.K + k]) : 0.f;
#pragma unroll
        for (int j = 0; j < CPW; ++j) {
          const float c = static_cast<float>((q >> shift_of(j)) & kMask);
#pragma unroll
          for (int m = 0; m < MT; ++m) a[m][j] = __fmaf_rn(xv[m], c, a[m][j]);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) sx[m] += xv[m];
      }
      fold();
    }
#pragma unroll
    for (int off = TW; off < 32; off <<= 1)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < CPW; ++j) acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], off);
    if (kr == 0)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < CPW; ++j) part[warp][m][wi * CPW + j] = acc[m][j];
    __syncthreads();
    for (int e = threadIdx.x; e < MT * NC; e += blockDim.x) {
      const int m = e / NC, c = e - m * NC;
      const int n = blockIdx.x * NC + c, gm = m0 + m;
      if (gm >= p.M || n >= p.N) continue;
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kGW; ++w) sum += part[w][m][c];
      if (p.bias) sum += elem_to_float<kBF>(reinterpret_cast<const uint16_t*>(p.bias)[n]);
      reinterpret_cast<uint16_t*>(p.y)[(long long)gm * p.N + n] = float_to_elem<kBF>(sum);
    }
    __syncthreads();
  }
}

template <bool kBF, int kBits, int TW>
void launch_generic_t(const GemmProblem& p, int C) {
  const int tiles = (C + TW - 1) / TW;
  const int mt = p.M == 1 ? 1 : 4;
  const int mtiles = (p.M + mt - 1) / mt;
  dim3 grid(tiles, mtiles < 65535 ? mtiles : 65535);
  if (mt == 1) generic_gemm_kernel<kBF, kBits, TW, 1><<<grid, kGW * 32, 0, p.stream>>>(p);
  else generic_gemm_kernel<kBF, kBits, TW, 4><<<grid, kGW * 32, 0, p.stream>>>(p);
}

template <bool kBF, int kBits>
void launch_generic_b(const GemmProblem& p) {
  const int C = p.N / (32 / kBits);
  const int mtiles = p.M == 1 ? 1 : (p.M + 3) / 4;
  // 8-word tiles (32-byte row segments) when they give at least two CTAs per SM, else 4
  if ((long long)((C + 7) / 8) * mtiles >= 2 * 152) launch_generic_t<kBF, kBits, 8>(p, C);
  else launch_generic_t<kBF, kBits, 4>(p, C);
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
  if (p.bits == 8) launch_generic_b<false, 8>(p);
  else if (p.bf16) launch_generic_b<true, 4>(p);
  else launch_generic_b<false, 4>(p);
  return cudaGetLastError();
}

}  // namespace awq
