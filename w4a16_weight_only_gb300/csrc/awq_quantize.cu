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
// One CTA (8 warps) per 128 output channels x one group (the weight is read once).
// Phase A: the tile's 16-byte chunks in row-major order, consecutive threads on
// consecutive chunks (coalesced), four loads in flight a thread; the lanes holding one
// channel's chunks combine their min / max with shuffles and one of them updates the
// channel's shared slot (integer atomics on an order-preserving key); for groups of up to
// 128 features the chunks are also kept in shared memory (rows padded by 16 bytes).  Then
// one thread per channel derives scale and zero.  Phase B, kKT features at a time: one
// thread per (channel, 8 features), consecutive threads on consecutive channels, writes
// its codes into a feature-major byte tile; each packed word is then one 8-byte read
// (channels 8c..8c+7 of one feature) and a byte permute into ORDER, kRows / 8 words per
// input row, contiguous in qweight.
//
// The quotient w / scale is screened with a reciprocal multiply: when the approximate
// quotient lies further than 2^-20 |q| from every half-integer, the correctly rounded
// quotient rounds to the same integer (the two differ by less than 2^-21 |q|); otherwise
// the exact __fdiv_rn quotient is used.  Codes are therefore those of the correctly
// rounded division.
#include "awq_internal.cuh"

namespace awq {
namespace {

constexpr int kRows = 128;       // output channels per CTA
constexpr int kThreads = 256;
constexpr int kKT = 128;         // features per code tile; groups up to this stay in smem
constexpr int kUnroll = 4;       // chunk loads in flight per thread
constexpr int kWPad = 8;         // halves of padding per kept row
constexpr int kCPitch = kRows + 8;  // bytes per feature row of the code tile (8-byte reads)
constexpr size_t kSmemW = static_cast<size_t>(kRows) * (kKT + kWPad) * 2;  // kept fp16 tile
constexpr size_t kSmemCode = static_cast<size_t>(kKT) * kCPitch;           // code tile
constexpr size_t kSmem = kSmemW + kSmemCode;

// Order-preserving map float -> int (finite values; -0 and +0 land next to each other).
__device__ __forceinline__ int fkey(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float funkey(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

// round(x * rs) with rs = fl(1 / s); *near is set when the product lies within 2^-20 |q|
// of a half-integer (then round(fl(x / s)) must come from the exact quotient).
__device__ __forceinline__ float round_screened(float x, float rs, bool* near) {
  const float qa = x * rs;
  const float k = rintf(qa);
  *near = fabsf(fabsf(qa - k) - 0.5f) <= fabsf(qa) * 0x1p-20f;
  return k;
}

// The code as a byte: the clamped integer-valued float plus 2^23 holds the integer in its
// low mantissa bits (exact for 0..15).
template <bool kSym>
__device__ __forceinline__ uint32_t code_byte(float q, float zf) {
  const float c = kSym ? fminf(fmaxf(q, -8.0f), 7.0f) + 8.0f : fminf(fmaxf(q + zf, 0.0f), 15.0f);
  return __float_as_uint(c + 8388608.0f) & 0xFFu;
}

template <bool kSym>
__global__ void __launch_bounds__(kThreads) quantize_rtn_kernel(const __half* __restrict__ w, int N,
                                                              int K, int G,
                                                              uint32_t* __restrict__ qw,
                                                              uint32_t* __restrict__ qz,
                                                              __half* __restrict__ sc) {
  extern __shared__ __align__(16) unsigned char smem[];
  __half* s_w = reinterpret_cast<__half*>(smem);          // [kRows][G + kWPad] when G <= kKT
  unsigned char* s_code = smem + kSmemW;                    // [kKT][kCPitch], feature-major
  __shared__ int s_max[kRows], s_min[kRows];
  __shared__ float s_scale[kRows], s_rcp[kRows];
  __shared__ int s_zero[kRows];
  __shared__ float s_zf[kRows];

  const int tid = threadIdx.x;
  const int n0 = blockIdx.x * kRows;
  const int g = blockIdx.y;
  const int rows = min(kRows, N - n0);  // a multiple of 8
  const int C = N / 8;
  const int cpr = G / 8;                // 16-byte chunks per channel row
  const bool keep = G <= kKT;
  const int gp = G + kWPad;             // kept row pitch (halves)
  // lanes of one warp holding the same channel (cpr a power of two up to 32) pre-reduce
  const bool pow2 = (cpr & (cpr - 1)) == 0;
  const int seg = (cpr <= 32 && pow2) ? cpr : 1;
  const int cshift = pow2 ? __ffs(cpr) - 1 : -1;  // row of chunk idx = idx >> cshift
  const long long kbase = static_cast<long long>(g) * G;
  const __half* tile = w + static_cast<long long>(n0) * K + kbase;

  for (int r = tid; r < kRows; r += kThreads) {
    s_max[r] = fkey(-INFINITY);
    s_min[r] = fkey(INFINITY);
  }
  __syncthreads();

  // ---- phase A: min / max of every channel (and the kept tile)
  const int total = rows * cpr;
  // whole warps iterate together (the shuffles need every lane); chunks past the tile
  // contribute nothing
  const int total_w = (total + 31) & ~31;
  for (int base = tid; base < total_w; base += kThreads * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int idx = base + u * kThreads;
      if (idx < total) {
        const int r = cshift >= 0 ? idx >> cshift : idx / cpr, c = idx - r * cpr;
        v[u] = __ldcs(reinterpret_cast<const uint4*>(tile + static_cast<long long>(r) * K) + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int idx = base + u * kThreads;
      if (idx >= total_w) continue;  // warp-uniform
      // {max, -min} of the chunk as one half2 (fp16 comparisons and negation are exact),
      // combined across the channel's lanes with one max per shuffle round
      __half2 mm = __halves2half2(__ushort_as_half(0xFC00u), __ushort_as_half(0xFC00u));  // -inf
      int r = 0;
      if (idx < total) {
        r = cshift >= 0 ? idx >> cshift : idx / cpr;
        const int c = idx - r * cpr;
        const __half2* h = reinterpret_cast<const __half2*>(&v[u]);
        const __half2 hx = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
        const __half2 hn = __hmin2(__hmin2(h[0], h[1]), __hmin2(h[2], h[3]));
        // lo: max of (hx.lo, hx.hi); hi: -min of (hn.lo, hn.hi)
        const __half2 a = __lows2half2(hx, __hneg2(hn));   // {hx.lo, -hn.lo}
        const __half2 b = __highs2half2(hx, __hneg2(hn));  // {hx.hi, -hn.hi}
        mm = __hmax2(a, b);
        if (keep) *reinterpret_cast<uint4*>(s_w + r * gp + 8 * c) = v[u];
      }
      for (int o = 1; o < seg; o <<= 1) {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<uint32_t*>(&mm), o);
        mm = __hmax2(mm, *reinterpret_cast<const __half2*>(&other));
      }
      if (idx < total && (idx & (seg - 1)) == 0) {
        atomicMax(&s_max[r], fkey(__low2float(mm)));
        atomicMin(&s_min[r], fkey(-__high2float(mm)));
      }
    }
  }
  __syncthreads();

  // ---- scale and zero, one thread per channel
  if (tid < rows) {
    const float mx = funkey(s_max[tid]), mn = funkey(s_min[tid]);
    float s;
    int z;
    __half s16;
    if (kSym) {
      const float amax = fmaxf(fmaxf(fabsf(mx), fabsf(mn)), 1e-5f);
      s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
      s = __half2float(s16);
      z = 8;
    } else {
      const float range = fmaxf(__fsub_rn(mx, mn), 1e-5f);
      s16 = __float2half_rn(__fdiv_rn(range, 15.0f));
      s = __half2float(s16);
      z = static_cast<int>(fminf(fmaxf(-rintf(__fdiv_rn(mn, s)), 0.0f), 15.0f));
    }
    sc[static_cast<long long>(g) * N + n0 + tid] = s16;
    s_scale[tid] = s;
    s_rcp[tid] = __frcp_rn(s);
    s_zero[tid] = z;
    s_zf[tid] = static_cast<float>(z);
  }
  __syncthreads();

  // packed zeros of this group: word c holds channels 8c + ORDER[i] in nibble i
  if (tid < rows / 8) {
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= static_cast<uint32_t>(s_zero[8 * tid + nibble_column(i)]) << (4 * i);
    qz[static_cast<long long>(g) * C + n0 / 8 + tid] = word;
  }

  // ---- phase B: codes and packed words, kKT features at a time
  const int words = rows / 8;
  for (int kc = 0; kc < G; kc += kKT) {
    const int kt = min(kKT, G - kc);  // a multiple of 8
    const int cpt = kt / 8;
    // thread -> (channel tid % 128, features 8c..8c+7 for c = tid / 128, + 2, ...);
    // consecutive threads on consecutive channels
    const int r = tid & (kRows - 1);
    if (r < rows) {
      const float s = s_scale[r], rs = s_rcp[r], zf = s_zf[r];
      for (int c = tid >> 7; c < cpt; c += kThreads / kRows) {
        uint4 v;
        if (keep) v = *reinterpret_cast<const uint4*>(s_w + r * gp + 8 * c);
        else v = __ldg(reinterpret_cast<const uint4*>(tile + static_cast<long long>(r) * K + kc) + c);
        const __half2* h = reinterpret_cast<const __half2*>(&v);
        float x[8], q[8];
        uint32_t near = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(h[j]);
          x[2 * j] = f.x;
          x[2 * j + 1] = f.y;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          bool nr;
          q[e] = round_screened(x[e], rs, &nr);
          near |= static_cast<uint32_t>(nr) << e;
        }
        // rare: some lane has a quotient next to a half-integer; take the exact division
        if (__any_sync(__activemask(), near != 0u)) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if ((near >> e) & 1u) q[e] = rintf(__fdiv_rn(x[e], s));
        }
        unsigned char* dst = s_code + (8 * c) * kCPitch + r;
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e * kCPitch] = static_cast<unsigned char>(code_byte<kSym>(q[e], zf));
      }
    }
    __syncthreads();
    // word (feature kl, column-word c): bytes b0..b7 = channels 8c..8c+7; nibble i takes
    // channel ORDER[i]: b0 | b2 << 4 | b4 << 8 | b6 << 12 | b1 << 16 | b3 << 20 | ...
    // thread -> (column-word tid % 16, features tid / 16, + 16, ...)
    const int cw = tid & 15;
    if (cw < words) {
      for (int kl = tid >> 4; kl < kt; kl += kThreads / 16) {
        const uint2 b = *reinterpret_cast<const uint2*>(s_code + kl * kCPitch + 8 * cw);
        const uint32_t t = b.x | (b.x >> 12);  // byte 0: b0 | b2 << 4, byte 1: b1 | b3 << 4
        const uint32_t u = b.y | (b.y >> 12);  // byte 0: b4 | b6 << 4, byte 1: b5 | b7 << 4
        uint32_t word;
        asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(word) : "r"(t), "r"(u));
        __stcs(qw + (kbase + kc + kl) * C + n0 / 8 + cw, word);
      }
    }
    __syncthreads();
  }
}

template <bool kSym>
cudaError_t set_smem_once() {
  static cudaError_t err = cudaFuncSetAttribute(quantize_rtn_kernel<kSym>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                static_cast<int>(kSmem));
  return err;
}

}  // namespace

cudaError_t launch_quantize_rtn(const __half* w, int N, int K, int G, bool sym, uint32_t* qw,
                                uint32_t* qz, __half* sc, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((N + kRows - 1) / kRows), static_cast<unsigned>(K / G));
  cudaError_t e = sym ? set_smem_once<true>() : set_smem_once<false>();
  if (e != cudaSuccess) return e;
  if (sym) quantize_rtn_kernel<true><<<grid, kThreads, kSmem, stream>>>(w, N, K, G, qw, qz, sc);
  else quantize_rtn_kernel<false><<<grid, kThreads, kSmem, stream>>>(w, N, K, G, qw, qz, sc);
  return cudaGetLastError();
}

}  // namespace awq
