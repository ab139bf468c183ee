// awq_quantize_rtn: round-to-nearest group quantization of an fp16 linear weight into the
// AWQ GEMM layout (GPTQModel wiki "AWQ", "Group quantization and zero points", the table
// of the asymmetric and symmetric modes; packing with ORDER as in tensref.org/formats/awq,
// "Reader").
//
//   per output channel n and group g of G input features:
//     asymmetric  scale = max(max - min, 1e-5) / 15,  zero = clamp(-round(min / scale), 0, 15)
//                 code  = clamp(round(w / scale) + zero, 0, 15)
//     symmetric   scale = max(max |w|, 1e-5) / 7,     zero = 8
//                 code  = clamp(round(w / scale), -8, 7) + 8
//
// Arithmetic: fp32 on the fp16 weights, every operation correctly rounded (__fsub_rn,
// __fdiv_rn, rintf = round half to even); the scale is rounded to fp16 as stored and the
// codes are taken against that stored value.
//
// One CTA (8 warps) per 128 output channels x one group.  Pass 1: a warp per channel reads
// the group with 16-byte loads and reduces min / max; lane 0 derives scale and zero.
// Pass 2, 64 input features at a time: codes into a shared byte tile (rows padded to 68
// bytes so the packing reads spread over the banks), then 16 packed words per input row
// (nibble i of word c holds channel 8c + ORDER[i]), 64 contiguous bytes per row.
#include "awq_internal.cuh"

namespace awq {
namespace {

constexpr int kRows = 128;     // output channels per CTA
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kKC = 64;        // input features per code tile
constexpr int kPitch = kKC + 4;  // bytes per code-tile row

template <bool kSym>
__global__ void __launch_bounds__(kThreads) quantize_rtn_kernel(const __half* __restrict__ w, int N,
                                                              int K, int G,
                                                              uint32_t* __restrict__ qw,
                                                              uint32_t* __restrict__ qz,
                                                              __half* __restrict__ sc) {
  __shared__ float s_scale[kRows];
  __shared__ int s_zero[kRows];
  __shared__ __align__(16) unsigned char s_code[kRows * kPitch];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kRows;
  const int g = blockIdx.y;
  const int rows = min(kRows, N - n0);  // a multiple of 8
  const int C = N / 8;
  const long long kbase = static_cast<long long>(g) * G;

  // ---- pass 1: scale and zero of every channel of the tile
  for (int r = warp; r < rows; r += kWarps) {
    const __half* row = w + static_cast<long long>(n0 + r) * K + kbase;
    float mx = -INFINITY, mn = INFINITY;
    for (int c = lane; c < G / 8; c += 32) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + c);
      const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(h[j]);
        mx = fmaxf(mx, fmaxf(f.x, f.y));
        mn = fminf(mn, fminf(f.x, f.y));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
      float s;
      int z;
      if (kSym) {
        const float amax = fmaxf(fmaxf(fabsf(mx), fabsf(mn)), 1e-5f);
        const __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
        s = __half2float(s16);
        z = 8;
        sc[static_cast<long long>(g) * N + n0 + r] = s16;
      } else {
        const float range = fmaxf(__fsub_rn(mx, mn), 1e-5f);
        const __half s16 = __float2half_rn(__fdiv_rn(range, 15.0f));
        s = __half2float(s16);
        const float zf = -rintf(__fdiv_rn(mn, s));
        z = static_cast<int>(fminf(fmaxf(zf, 0.0f), 15.0f));
        sc[static_cast<long long>(g) * N + n0 + r] = s16;
      }
      s_scale[r] = s;
      s_zero[r] = z;
    }
  }
  __syncthreads();

  // packed zeros of this group: word c holds channels 8c + ORDER[i] in nibble i
  if (threadIdx.x < rows / 8) {
    const int c = threadIdx.x;
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= static_cast<uint32_t>(s_zero[8 * c + nibble_column(i)]) << (4 * i);
    qz[static_cast<long long>(g) * C + n0 / 8 + c] = word;
  }

  // ---- pass 2: codes, 64 input features at a time
  for (int kc = 0; kc < G; kc += kKC) {
    const int klen = min(kKC, G - kc);  // a multiple of 8
    // lane -> (channel 4j + lane / 8 of the warp's slice, 8 features lane % 8)
    for (int r0 = warp * 4; r0 < rows; r0 += kWarps * 4) {
      const int r = r0 + (lane >> 3);
      const int c8 = lane & 7;
      if (r < rows && 8 * c8 < klen) {
        const __half* src = w + static_cast<long long>(n0 + r) * K + kbase + kc + 8 * c8;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
        const __half2* h = reinterpret_cast<const __half2*>(&v);
        const float s = s_scale[r];
        const int z = s_zero[r];
        uint32_t b[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(h[j]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float q = rintf(__fdiv_rn(e ? f.y : f.x, s));
            int code;
            if (kSym) code = static_cast<int>(fminf(fmaxf(q, -8.0f), 7.0f)) + 8;
            else code = static_cast<int>(fminf(fmaxf(q + static_cast<float>(z), 0.0f), 15.0f));
            const int idx = 2 * j + e;
            b[idx >> 2] |= static_cast<uint32_t>(code) << (8 * (idx & 3));
          }
        }
        *reinterpret_cast<uint32_t*>(&s_code[r * kPitch + 8 * c8]) = b[0];
        *reinterpret_cast<uint32_t*>(&s_code[r * kPitch + 8 * c8 + 4]) = b[1];
      }
    }
    __syncthreads();
    // pack: 16 words per input row of the tile, word c = channels 8c + ORDER[i]
    const int words = rows / 8;
    for (int idx = threadIdx.x; idx < klen * words; idx += kThreads) {
      const int kl = idx / words;
      const int c = idx - kl * words;
      uint32_t word = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        word |= static_cast<uint32_t>(s_code[(8 * c + nibble_column(i)) * kPitch + kl]) << (4 * i);
      qw[(kbase + kc + kl) * C + n0 / 8 + c] = word;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_quantize_rtn(const __half* w, int N, int K, int G, bool sym, uint32_t* qw,
                                uint32_t* qz, __half* sc, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((N + kRows - 1) / kRows), static_cast<unsigned>(K / G));
  if (sym) quantize_rtn_kernel<true><<<grid, kThreads, 0, stream>>>(w, N, K, G, qw, qz, sc);
  else quantize_rtn_kernel<false><<<grid, kThreads, 0, stream>>>(w, N, K, G, qw, qz, sc);
  return cudaGetLastError();
}

}  // namespace awq
