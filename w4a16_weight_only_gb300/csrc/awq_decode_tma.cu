// Decode path of awq_gemm, TMA-fed (small M, HBM-bound):
//
//   y[m][n] = sum_k x[m][k] * (code[k][n] - zero[k/G][n]) * scale[k/G][n]  (+ bias[n])
//
// (tensref.org/formats/awq, "Reader"; GPTQModel wiki "AWQ", "Native GEMM": fused
// dequant-GEMM, fp32 accumulation, split over K.)
//
// GB300 design.  Every warp owns a contiguous run of 64-row stages of one column tile and
// streams it through its own two-slot shared-memory ring: lane 0 issues the bulk tensor
// copies (packed weights, activations, the stage's zero and scale rows) on an mbarrier,
// the warp waits with a bounded try-wait, computes, and refills the slot.  The activation
// tile lands 128-byte swizzled; the weight tile is unswizzled and the row order of the
// fragment reads (row parity swapped on odd lanes of a quad) spreads each read over all
// 32 banks, so both need the minimum number of shared-memory wavefronts.  No register or instruction is spent on address streams for the weights, and a
// CTA keeps 16 stages (64 KB of packed weights) in flight.
//
// Unpack without shifts: two rows (k, k+1) of one packed column are byte-permuted (prmt)
// so each 16-bit half holds one row's four low (or high) nibbles; then one LOP3 with the
// fp16 exponent pattern 0x6400 per nibble pair yields (1024 + c) (even nibbles, bits
// 0-3) or (1024 + 16c) (odd nibbles, bits 4-7) for both rows, and one HSUB2 with the same
// construction applied to the zero word gives exactly (c - z) or 16 (c - z).  Those half2
// pairs are the A operand of m16n8k16 tensor-core MMAs (weights on the 16-row side,
// activations on the 8-wide side).  With kFactor the MMA accumulates x * (c - z) over a
// stage (one quantization group) and the scale (divided by 16 for odd nibbles, exact) is
// applied once per output element per stage; without it the exact fp16 weight
// (c - z) * scale is formed with HMUL2 first.
//
// Split-K: warps of a CTA and CTAs of a thread-block cluster take consecutive K ranges;
// partial sums are reduced in a fixed order through shared memory and distributed shared
// memory (no global workspace, no atomics), so repeated calls are bitwise identical.
#include <mutex>

#include "awq_internal.cuh"
#include "awq_ptx.cuh"

namespace awq {
namespace {

using namespace ptx;

constexpr int kNW = 8;        // warps per CTA
constexpr int kSlots = 2;     // ring slots per warp
constexpr int kRS = 64;       // rows of K per stage
constexpr uint32_t kMagic = 0x64006400u;
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 200 ms per wait
constexpr unsigned int kStatusDecodeTimeout = 0x1u;

struct __align__(64) TmaDecodeParams {
  CUtensorMap tm_w;  // qweight [K][C] u32, box {CW_W, 64}, unswizzled
  CUtensorMap tm_x;  // x [M][K] f16, box {64, 8*TB}, 128B swizzle
  CUtensorMap tm_z;  // qzeros [K/G][C] u32, box {CW_W, 1}
  CUtensorMap tm_s;  // scales [K/G][N] f16, box {8*CW_W, 1}
  const __half* bias;
  __half* y;
  unsigned int* status;
  int M, K, N, C, G;
};

template <int TB, int CWL>
struct Geo {
  static constexpr int CW_W = 8 * CWL;              // packed column-words per warp / CTA
  static constexpr int W_BYTES = kRS * CW_W * 4;    // packed weight tile per stage
  static constexpr int X_BYTES = 8 * TB * kRS * 2;  // activation tile per stage
  static constexpr int Z_BYTES = CW_W * 4;
  static constexpr int S_BYTES = 8 * CW_W * 2;
  static constexpr int X_OFF = W_BYTES;             // both multiples of 1024
  static constexpr int Z_OFF = W_BYTES + X_BYTES;
  static constexpr int S_OFF = Z_OFF + 128;
  static constexpr int SLOT = ((S_OFF + S_BYTES + 1023) / 1024) * 1024;
  static constexpr uint32_t TX = W_BYTES + X_BYTES + Z_BYTES + S_BYTES;
  static constexpr int NMMA = 4 * CWL;
  static constexpr int E = NMMA * TB * 4 * 32;      // partial sums per warp
  static constexpr size_t SMEM = 1024 + (size_t)kNW * kSlots * SLOT + kNW * kSlots * 8;
  static_assert((size_t)kNW * E * 4 <= (size_t)kNW * kSlots * SLOT, "reduction buffer");
};

template <int CWL>
__device__ __forceinline__ constexpr int mma_cw(int mi, int rs) {
  return CWL == 1 ? 0 : 2 * (mi >> 3) + rs;
}
template <int CWL>
__device__ __forceinline__ constexpr int mma_nib(int mi, int rs) {
  return CWL == 1 ? mi + 4 * rs : (mi & 7);
}

template <int TB, int CWL, bool kFactor>
__global__ void __launch_bounds__(kNW * 32, 2)
    decode_tma_kernel(const __grid_constant__ TmaDecodeParams p) {
  using GE = Geo<TB, CWL>;
  constexpr int NMMA = GE::NMMA;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kNW * kSlots * GE::SLOT);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g8 = lane >> 2;
  const int q = lane & 3;
  const uint32_t rank = cluster_ctarank();
  const uint32_t cs = cluster_nctarank();
  const int cw0 = static_cast<int>(blockIdx.x / cs) * GE::CW_W;
  const int m0 = blockIdx.y * 8 * TB;

  const int TS = p.K / kRS;
  const int P = static_cast<int>(cs) * kNW;
  const int wid = static_cast<int>(rank) * kNW + warp;
  const int j0 = static_cast<int>((long long)TS * wid / P);
  const int j1 = static_cast<int>((long long)TS * (wid + 1) / P);

  unsigned char* my_slots = smem + (size_t)warp * kSlots * GE::SLOT;
  uint64_t* my_bars = bars + warp * kSlots;

  if (lane == 0) {
    prefetch_tmap(&p.tm_w);
    prefetch_tmap(&p.tm_x);
    for (int s = 0; s < kSlots; ++s) mbar_init(&my_bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int slot, int j) {
    unsigned char* b = my_slots + slot * GE::SLOT;
    uint64_t* bar = &my_bars[slot];
    mbar_arrive_expect_tx(bar, GE::TX);
    const int grp = (j * kRS) / p.G;
    tma_load_2d(b, &p.tm_w, bar, cw0, j * kRS);
    tma_load_2d(b + GE::X_OFF, &p.tm_x, bar, j * kRS, m0);
    tma_load_2d(b + GE::Z_OFF, &p.tm_z, bar, cw0, grp);
    tma_load_2d(b + GE::S_OFF, &p.tm_s, bar, 8 * cw0, grp);
  };

  if (lane == 0) {
    for (int s = 0; s < kSlots && j0 + s < j1; ++s) issue(s, j0 + s);
  }

  float acc[NMMA][TB][4];
#pragma unroll
  for (int i = 0; i < NMMA; ++i)
#pragma unroll
    for (int b = 0; b < TB; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][b][e] = 0.f;

  int done = j0;  // first stage not yet waited for
  bool failed = false;
  for (int j = j0; j < j1; ++j) {
    const int slot = (j - j0) % kSlots;
    const uint32_t parity = static_cast<uint32_t>(((j - j0) / kSlots) & 1);
    if (!mbar_wait_bounded(&my_bars[slot], parity, p.status, kStatusDecodeTimeout, kWaitLimitNs)) {
      failed = true;
      break;
    }
    done = j + 1;
    const unsigned char* b = my_slots + slot * GE::SLOT;
#ifdef AWQ_DECODE_DEBUG_DUMP
    AWQ_DECODE_DEBUG_DUMP(b, GE::SLOT);
#endif
    const uint32_t* Z = reinterpret_cast<const uint32_t*>(b + GE::Z_OFF);
    const uint4* S = reinterpret_cast<const uint4*>(b + GE::S_OFF);

    // Zero pairs for this stage's group: (1024 + z) for even nibbles, (1024 + 16 z) for odd.
    uint32_t zp[CWL][8];
    uint32_t sv[CWL][4];
#pragma unroll
    for (int c = 0; c < CWL; ++c) {
      const uint32_t zw = Z[g8 * CWL + c];
      const uint32_t lo = prmt(zw, zw, 0x5410u), hi = prmt(zw, zw, 0x7632u);
      const uint32_t lo8 = lo >> 8, hi8 = hi >> 8;
      if (kFactor) {
        zp[c][0] = and_or(lo, 0x000F000Fu, kMagic);
        zp[c][1] = and_or(lo, 0x00F000F0u, kMagic);
        zp[c][2] = and_or(lo8, 0x000F000Fu, kMagic);
        zp[c][3] = and_or(lo8, 0x00F000F0u, kMagic);
        zp[c][4] = and_or(hi, 0x000F000Fu, kMagic);
        zp[c][5] = and_or(hi, 0x00F000F0u, kMagic);
        zp[c][6] = and_or(hi8, 0x000F000Fu, kMagic);
        zp[c][7] = and_or(hi8, 0x00F000F0u, kMagic);
      } else {
        zp[c][0] = and_or(lo, 0x000F000Fu, kMagic);
        zp[c][1] = and_or(lo >> 4, 0x000F000Fu, kMagic);
        zp[c][2] = and_or(lo8, 0x000F000Fu, kMagic);
        zp[c][3] = and_or(lo8 >> 4, 0x000F000Fu, kMagic);
        zp[c][4] = and_or(hi, 0x000F000Fu, kMagic);
        zp[c][5] = and_or(hi >> 4, 0x000F000Fu, kMagic);
        zp[c][6] = and_or(hi8, 0x000F000Fu, kMagic);
        zp[c][7] = and_or(hi8 >> 4, 0x000F000Fu, kMagic);
      }
      const uint4 s4 = S[g8 * CWL + c];
      sv[c][0] = s4.x; sv[c][1] = s4.y; sv[c][2] = s4.z; sv[c][3] = s4.w;
    }

    float accg[kFactor ? NMMA : 1][TB][4];
    // prmt selectors: low (high) 16 bits of row 2q in the low half, of row 2q+1 in the high.
    const uint32_t sel_lo = (q & 1) ? 0x1054u : 0x5410u;
    const uint32_t sel_hi = (q & 1) ? 0x3276u : 0x7632u;
#pragma unroll
    for (int ks = 0; ks < kRS / 16; ++ks) {
      // Packed words of lane (g8, q), column-words g8*CWL .. +CWL-1, rows
      //   r = 0, 1 -> 16ks + 2q + {0, 1},   r = 2, 3 -> 16ks + 2q + 8 + {0, 1},
      // the row parity swapped for odd q so that, with 64-byte rows, the four q-lanes of a
      // read cover both halves of the bank space (the prmt selectors undo the swap).
      uint32_t w[4][CWL];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = 16 * ks + 2 * q + ((r ^ q) & 1) + 8 * (r >> 1);
        if constexpr (CWL == 2) {
          const uint32_t off = static_cast<uint32_t>(row * 64 + g8 * 8);
          const uint2 v = *reinterpret_cast<const uint2*>(b + off);
          w[r][0] = v.x;
          w[r][1] = v.y;
        } else {
          const uint32_t off = static_cast<uint32_t>(row * 32 + g8 * 4);
          w[r][0] = *reinterpret_cast<const uint32_t*>(b + off);
        }
      }
      // Activations: token 8tb + g8, k = 16ks + 2q + {0,1} and 16ks + 2q + 8 + {0,1}.
      uint32_t bx[TB][2];
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) {
        const uint32_t base = static_cast<uint32_t>((8 * tb + g8) * (kRS * 2) + (16 * ks + 2 * q) * 2);
        bx[tb][0] = *reinterpret_cast<const uint32_t*>(b + GE::X_OFF + swz128(base));
        bx[tb][1] = *reinterpret_cast<const uint32_t*>(b + GE::X_OFF + swz128(base + 16));
      }
      // Half2 operands v[c][rp][i]: rows (2q + 8rp, 2q + 8rp + 1), nibble i of word c.
      uint32_t v[CWL][2][8];
#pragma unroll
      for (int c = 0; c < CWL; ++c)
#pragma unroll
        for (int rp = 0; rp < 2; ++rp) {
          const uint32_t plo = prmt(w[2 * rp][c], w[2 * rp + 1][c], sel_lo);
          const uint32_t phi = prmt(w[2 * rp][c], w[2 * rp + 1][c], sel_hi);
          const uint32_t plo8 = plo >> 8, phi8 = phi >> 8;
          uint32_t h[8];
          if (kFactor) {
            h[0] = and_or(plo, 0x000F000Fu, kMagic);
            h[1] = and_or(plo, 0x00F000F0u, kMagic);
            h[2] = and_or(plo8, 0x000F000Fu, kMagic);
            h[3] = and_or(plo8, 0x00F000F0u, kMagic);
            h[4] = and_or(phi, 0x000F000Fu, kMagic);
            h[5] = and_or(phi, 0x00F000F0u, kMagic);
            h[6] = and_or(phi8, 0x000F000Fu, kMagic);
            h[7] = and_or(phi8, 0x00F000F0u, kMagic);
          } else {
            h[0] = and_or(plo, 0x000F000Fu, kMagic);
            h[1] = and_or(plo >> 4, 0x000F000Fu, kMagic);
            h[2] = and_or(plo8, 0x000F000Fu, kMagic);
            h[3] = and_or(plo8 >> 4, 0x000F000Fu, kMagic);
            h[4] = and_or(phi, 0x000F000Fu, kMagic);
            h[5] = and_or(phi >> 4, 0x000F000Fu, kMagic);
            h[6] = and_or(phi8, 0x000F000Fu, kMagic);
            h[7] = and_or(phi8 >> 4, 0x000F000Fu, kMagic);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t d = hsub2(h[i], zp[c][i]);
            if (!kFactor) {
              const int col = nibble_column(i);
              d = hmul2(d, prmt(sv[c][col >> 1], 0u, (col & 1) ? 0x3232u : 0x1010u));
            }
            v[c][rp][i] = d;
          }
        }
#ifdef AWQ_DECODE_DEBUG_OPS
      AWQ_DECODE_DEBUG_OPS(ks, bx, v, w);
#endif
#pragma unroll
      for (int mi = 0; mi < NMMA; ++mi) {
        const int ca = mma_cw<CWL>(mi, 0), ia = mma_nib<CWL>(mi, 0);
        const int cb = mma_cw<CWL>(mi, 1), ib = mma_nib<CWL>(mi, 1);
#pragma unroll
        for (int tb = 0; tb < TB; ++tb) {
          if (kFactor) {
            if (ks == 0)
              mma16816_zero(accg[mi][tb], v[ca][0][ia], v[cb][0][ib], v[ca][1][ia], v[cb][1][ib],
                            bx[tb][0], bx[tb][1]);
            else
              mma16816(accg[mi][tb], v[ca][0][ia], v[cb][0][ib], v[ca][1][ia], v[cb][1][ib],
                       bx[tb][0], bx[tb][1]);
          } else {
            mma16816(acc[mi][tb], v[ca][0][ia], v[cb][0][ib], v[ca][1][ia], v[cb][1][ib],
                     bx[tb][0], bx[tb][1]);
          }
        }
      }
    }
    if (kFactor) {
      // acc += scale * accg; odd nibbles carry a factor 16, removed exactly.
#pragma unroll
      for (int mi = 0; mi < NMMA; ++mi)
#pragma unroll
        for (int rs = 0; rs < 2; ++rs) {
          const int c = mma_cw<CWL>(mi, rs);
          const int nib = mma_nib<CWL>(mi, rs);
          const int col = nibble_column(nib);
          const uint32_t pr = sv[c][col >> 1];
          float s = __half2float(__ushort_as_half(
              static_cast<unsigned short>((col & 1) ? (pr >> 16) : (pr & 0xFFFFu))));
          if (nib & 1) s *= 0.0625f;
#pragma unroll
          for (int tb = 0; tb < TB; ++tb) {
            acc[mi][tb][2 * rs] = __fmaf_rn(s, accg[mi][tb][2 * rs], acc[mi][tb][2 * rs]);
            acc[mi][tb][2 * rs + 1] = __fmaf_rn(s, accg[mi][tb][2 * rs + 1], acc[mi][tb][2 * rs + 1]);
          }
        }
    }
#ifdef AWQ_DECODE_DEBUG_ACC
    AWQ_DECODE_DEBUG_ACC(acc);
#endif
    __syncwarp();
    if (lane == 0 && j + kSlots < j1) issue(slot, j + kSlots);
  }
  if (failed) {
    // Let copies already issued land (bounded) before the slots are reused below.
    const int issued_end = min(j1, done + kSlots);
    for (int j = done; j < issued_end; ++j) {
      const int slot = (j - j0) % kSlots;
      const uint32_t parity = static_cast<uint32_t>(((j - j0) / kSlots) & 1);
      mbar_wait_bounded(&my_bars[slot], parity, p.status, kStatusDecodeTimeout, kWaitLimitNs);
    }
  }

  // Reduce: warps of the CTA (fixed order), then CTAs of the cluster (fixed order).
  __syncthreads();  // the ring is reused as the reduction buffer
  float* red = reinterpret_cast<float*>(smem);
  float* mine = red + warp * GE::E;
#pragma unroll
  for (int mi = 0; mi < NMMA; ++mi)
#pragma unroll
    for (int tb = 0; tb < TB; ++tb)
#pragma unroll
      for (int e = 0; e < 4; ++e) mine[((mi * TB + tb) * 4 + e) * 32 + lane] = acc[mi][tb][e];
  __syncthreads();
  for (int e = threadIdx.x; e < GE::E; e += kNW * 32) {
    float s = red[e];
#pragma unroll
    for (int w = 1; w < kNW; ++w) s += red[w * GE::E + e];
    red[e] = s;
  }
  cluster_sync_all();
  const int e_lo = static_cast<int>((long long)GE::E * rank / cs);
  const int e_hi = static_cast<int>((long long)GE::E * (rank + 1) / cs);
  for (int e = e_lo + threadIdx.x; e < e_hi; e += kNW * 32) {
    const int ln = e & 31;
    const int j = (e >> 5) & 3;
    const int tb = (e >> 7) % TB;
    const int mi = (e >> 7) / TB;
    const int rs = j >> 1;
    const int tok = m0 + 8 * tb + 2 * (ln & 3) + (j & 1);
    const int cw = cw0 + (ln >> 2) * CWL + mma_cw<CWL>(mi, rs);
    if (tok < p.M && cw < p.C) {
      float s = 0.f;
      for (uint32_t r = 0; r < cs; ++r) s += ld_dsmem_f32(red + e, r);
      const int n = 8 * cw + nibble_column(mma_nib<CWL>(mi, rs));
      if (p.bias) s += __half2float(p.bias[n]);
      p.y[(long long)tok * p.N + n] = __float2half_rn(s);
    }
  }
  cluster_sync_all();
}

struct Variant {
  int TB, CWL;
  bool factor;
};

Variant pick(const GemmProblem& p) {
  if (p.M <= 8) return Variant{1, 2, true};
  if (p.M <= 16) return Variant{2, 1, true};
  return Variant{4, 1, false};
}

template <int TB, int CWL, bool F>
cudaError_t launch_v(const GemmProblem& p, const Variant&) {
  using GE = Geo<TB, CWL>;
  auto kern = decode_tma_kernel<TB, CWL, F>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(GE::SMEM));
  });
  if (attr_err != cudaSuccess) return attr_err;

  TmaDecodeParams dp;
  const char* why = nullptr;
  const int C = p.N / 8;
  const int ngrp = p.K / p.G;
  if (!make_tmap_2d(&dp.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.qw, C, p.K, GE::CW_W, kRS,
                    CU_TENSOR_MAP_SWIZZLE_NONE, &why) ||
      !make_tmap_2d(&dp.tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.x, p.K, p.M, kRS, 8 * TB,
                    CU_TENSOR_MAP_SWIZZLE_128B, &why) ||
      !make_tmap_2d(&dp.tm_z, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.qz, C, ngrp, GE::CW_W, 1,
                    CU_TENSOR_MAP_SWIZZLE_NONE, &why) ||
      !make_tmap_2d(&dp.tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.sc, p.N, ngrp, 8 * GE::CW_W, 1,
                    CU_TENSOR_MAP_SWIZZLE_NONE, &why))
    return cudaErrorInvalidValue;
  dp.bias = p.bias;
  dp.y = p.y;
  cudaError_t e = status_word_ptr(&dp.status);
  if (e != cudaSuccess) return e;
  dp.M = p.M; dp.K = p.K; dp.N = p.N; dp.C = C; dp.G = p.G;

  const int nt = (C + GE::CW_W - 1) / GE::CW_W;
  const int mz = (p.M + 8 * TB - 1) / (8 * TB);
  const int ts = p.K / kRS;
  int cs = 1;
  while (cs < 8 && (long long)nt * mz * cs * 2 <= 2 * 152 && ts >= 2 * cs * kNW) cs *= 2;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nt * cs), static_cast<unsigned>(mz), 1);
  cfg.blockDim = dim3(kNW * 32, 1, 1);
  cfg.dynamicSmemBytes = GE::SMEM;
  cfg.stream = p.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, dp);
}

}  // namespace

bool decode_tma_supported(const GemmProblem& p, const char** why) {
  static const char* dummy;
  if (!why) why = &dummy;
  if (p.K % kRS != 0) { *why = "TMA decode needs K % 64 == 0"; return false; }
  if (p.G % kRS != 0) { *why = "TMA decode needs group_size % 64 == 0"; return false; }
  if (p.N % 32 != 0) { *why = "TMA decode needs N % 32 == 0"; return false; }
  if (!aligned(p.x, 16) || !aligned(p.qw, 16) || !aligned(p.qz, 16) || !aligned(p.sc, 16)) {
    *why = "TMA decode needs 16-byte aligned x, qweight, qzeros, scales";
    return false;
  }
  if ((p.M + 31) / 32 > 65535) { *why = "M too large for the decode grid"; return false; }
  return true;
}

cudaError_t launch_decode_tma(const GemmProblem& p) {
  const Variant v = pick(p);
  if (v.TB == 1) return launch_v<1, 2, true>(p, v);
  if (v.TB == 2) return launch_v<2, 1, true>(p, v);
  return launch_v<4, 1, false>(p, v);
}

}  // namespace awq
