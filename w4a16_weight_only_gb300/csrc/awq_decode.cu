// Decode path of awq_gemm: small M (a few activation rows), HBM-bound.
//
// y[m][n] = sum_k x[m][k] * (code[k][n] - zero[k/G][n]) * scale[k/G][n]  (+ bias[n])
// (tensref.org/formats/awq, "Reader"; GPTQModel wiki "AWQ", "Native GEMM": fused
// dequant-GEMM with fp32 accumulation and a split over K).
//
// Design (GB300): the packed weight is streamed exactly once from HBM with wide
// non-allocating loads, several k-steps in flight per warp.  Each lane unpacks its words
// in registers: two rows of the same packed column are byte-permuted (prmt) so that one
// mask-and-or per nibble yields a half2 holding (1024 + code) for two consecutive k, the
// zero pair is subtracted exactly (HSUB2), and the pair feeds an m16n8k16 tensor-core
// MMA directly as its A operand (weights as the 16-row side, activations as the 8-wide
// side, fp32 accumulators).  K is split over the warps of a CTA and over the CTAs of a
// thread-block cluster; partial sums are reduced in a fixed order through shared memory
// and then distributed shared memory, so results are bitwise reproducible and no global
// workspace or atomics are used.  One launch per call.
//
// Accumulation: with kFactor the MMA accumulates x*(code - zero) (exact small integers in
// fp16) per quantization group and the group's scale is applied once per output element
// when the group ends; without it the A operand is the exact fp16 dequantized weight
// (code - zero) * scale.  Both are fp32 accumulations of the same products.
#include <mutex>

#include "awq_internal.cuh"

namespace awq {
namespace {

constexpr int kNW = 8;  // warps per CTA
constexpr int kD = 4;   // k16-steps of packed weights in flight per warp

struct DecodeParams {
  const __half* x;
  const uint32_t* qw;
  const uint32_t* qz;
  const __half* sc;
  const __half* bias;
  __half* y;
  int M, K, N, C, G;
  int grp_cap;  // meta rows staged per CTA (upper bound over cluster ranks)
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// (a & m) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(m), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int CWL>
__device__ __forceinline__ void ldg_stream(uint32_t (&w)[CWL], const uint32_t* p) {
  if constexpr (CWL == 1) {
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(w[0]) : "l"(p));
  } else if constexpr (CWL == 2) {
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(w[0]), "=r"(w[1])
                 : "l"(p));
  } else {
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "l"(p));
  }
}

__device__ __forceinline__ uint2 ldg_x(const __half* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ float ld_dsmem(const float* local, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// Which packed column-word (0..CWL-1 within the lane's run) and which nibble feed A row
// `g` (rowsel 0) or `g + 8` (rowsel 1) of MMA `mi`.
template <int CWL>
__device__ __forceinline__ constexpr int mma_cw(int mi, int rowsel) {
  return CWL == 1 ? 0 : 2 * (mi >> 3) + rowsel;
}
template <int CWL>
__device__ __forceinline__ constexpr int mma_nib(int mi, int rowsel) {
  return CWL == 1 ? mi + 4 * rowsel : (mi & 7);
}

// TB: 8-token blocks per CTA (M tile = 8*TB).  CWL: packed column-words per lane (one
// vector load of CWL words per row).  A warp covers 8*CWL column-words = 64*CWL columns.
template <int TB, int CWL, bool kFactor>
__global__ void __launch_bounds__(kNW * 32) decode_kernel(const DecodeParams p) {
  constexpr int NMMA = 4 * CWL;
  constexpr int CW_CTA = 8 * CWL;
  constexpr int E = NMMA * TB * 4 * 32;  // partial sums per warp
  extern __shared__ __align__(16) unsigned char smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g8 = lane >> 2;
  const int q = lane & 3;
  const uint32_t rank = cluster_rank();
  int cs;
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(cs));
  const int nb = blockIdx.x / cs;
  const int cwb = nb * CW_CTA;
  const int m0 = blockIdx.y * 8 * TB;
  const int T = p.K >> 4;

  const int cta_t0 = static_cast<int>((long long)T * rank / cs);
  const int cta_t1 = static_cast<int>((long long)T * (rank + 1) / cs);
  const int nt = cta_t1 - cta_t0;
  const int t_begin = cta_t0 + static_cast<int>((long long)nt * warp / kNW);
  const int t_end = cta_t0 + static_cast<int>((long long)nt * (warp + 1) / kNW);

  uint32_t* zs = reinterpret_cast<uint32_t*>(smem);                       // [grp_cap][CW_CTA]
  uint4* ss = reinterpret_cast<uint4*>(smem + p.grp_cap * CW_CTA * 4);     // [grp_cap][CW_CTA]
  float* red = reinterpret_cast<float*>(smem + p.grp_cap * CW_CTA * 20);   // [kNW][E]

  const int cwl = cwb + g8 * CWL;
  const bool cw_ok = cwl < p.C;

  // 1. Put the first kD k-steps of packed weights in flight.
  uint32_t wb[kD][4][CWL];
  const uint32_t* qbase = p.qw + (long long)(4 * q) * p.C + cwl;
#pragma unroll
  for (int d = 0; d < kD; ++d) {
    const int t = t_begin + d;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (cw_ok && t < t_end) {
        ldg_stream<CWL>(wb[d][r], qbase + (long long)(16 * t + r) * p.C);
      } else {
#pragma unroll
        for (int c = 0; c < CWL; ++c) wb[d][r][c] = 0u;
      }
    }
  }

  // 2. Stage this CTA's zero/scale rows (its k-range, its column-words) in shared memory.
  const int grp0 = (cta_t0 * 16) / p.G;
  const int ngrp = nt > 0 ? ((cta_t1 * 16 - 1) / p.G - grp0 + 1) : 0;
  for (int e = threadIdx.x; e < ngrp * CW_CTA; e += kNW * 32) {
    const int gr = e / CW_CTA, c = e % CW_CTA;
    const int cw = cwb + c;
    uint32_t z = 0u;
    uint4 s = make_uint4(0u, 0u, 0u, 0u);
    if (cw < p.C) {
      z = __ldg(p.qz + (long long)(grp0 + gr) * p.C + cw);
      s = __ldg(reinterpret_cast<const uint4*>(p.sc + (long long)(grp0 + gr) * p.N + 8LL * cw));
    }
    zs[gr * CW_CTA + c] = z;
    ss[gr * CW_CTA + c] = s;
  }
  __syncthreads();

  float acc[NMMA][TB][4];
  float accg[kFactor ? NMMA : 1][TB][4];
#pragma unroll
  for (int i = 0; i < NMMA; ++i)
#pragma unroll
    for (int b = 0; b < TB; ++b)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[i][b][j] = 0.f;
        if (kFactor) accg[i][b][j] = 0.f;
      }

  uint32_t zp[CWL][8];                 // (1024+zero) in both halves, per column-word/nibble
  uint32_t sv[CWL][4];                 // the column-word's 8 fp16 scales, packed
  int cur = -1;

  auto fold = [&]() {
    // acc += scale * accg for the group just finished; accg = 0.
#pragma unroll
    for (int mi = 0; mi < NMMA; ++mi) {
#pragma unroll
      for (int rs = 0; rs < 2; ++rs) {
        const int c = mma_cw<CWL>(mi, rs);
        const int col = nibble_column(mma_nib<CWL>(mi, rs));
        const uint32_t pr = sv[c][col >> 1];
        const float s = __half2float(__ushort_as_half(
            static_cast<unsigned short>((col & 1) ? (pr >> 16) : (pr & 0xFFFFu))));
#pragma unroll
        for (int b = 0; b < TB; ++b) {
          acc[mi][b][2 * rs + 0] = __fmaf_rn(s, accg[mi][b][2 * rs + 0], acc[mi][b][2 * rs + 0]);
          acc[mi][b][2 * rs + 1] = __fmaf_rn(s, accg[mi][b][2 * rs + 1], acc[mi][b][2 * rs + 1]);
          accg[mi][b][2 * rs + 0] = 0.f;
          accg[mi][b][2 * rs + 1] = 0.f;
        }
      }
    }
  };

  // 3. Main loop over this warp's k16-steps.
  for (int t0 = t_begin; t0 < t_end; t0 += kD) {
#pragma unroll
    for (int d = 0; d < kD; ++d) {
      const int t = t0 + d;
      if (t < t_end) {
        const int grp = (16 * t) / p.G;
        if (grp != cur) {
          if (kFactor && cur >= 0) fold();
          cur = grp;
          const int lg = grp - grp0;
#pragma unroll
          for (int c = 0; c < CWL; ++c) {
            const uint32_t zw = zs[lg * CW_CTA + g8 * CWL + c];
            const uint4 s4 = ss[lg * CW_CTA + g8 * CWL + c];
            sv[c][0] = s4.x; sv[c][1] = s4.y; sv[c][2] = s4.z; sv[c][3] = s4.w;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t z = (zw >> (4 * i)) & 0xFu;
              zp[c][i] = (z | (z << 16)) | 0x64006400u;
            }
          }
        }

        // Activation fragments: token 8b+g8, k = 16t + 4q .. 16t + 4q + 3.
        uint32_t bx[TB][2];
#pragma unroll
        for (int b = 0; b < TB; ++b) {
          const int tok = m0 + 8 * b + g8;
          if (tok < p.M) {
            const uint2 v = ldg_x(p.x + (long long)tok * p.K + 16 * t + 4 * q);
            bx[b][0] = v.x;
            bx[b][1] = v.y;
          } else {
            bx[b][0] = 0u;
            bx[b][1] = 0u;
          }
        }

        // Row pairs (4q, 4q+1) and (4q+2, 4q+3): nibbles 0-3 and 4-7 of both rows.
        uint32_t pp[CWL][2][2];
#pragma unroll
        for (int c = 0; c < CWL; ++c)
#pragma unroll
          for (int rp = 0; rp < 2; ++rp) {
            pp[c][rp][0] = prmt(wb[d][2 * rp][c], wb[d][2 * rp + 1][c], 0x5410u);
            pp[c][rp][1] = prmt(wb[d][2 * rp][c], wb[d][2 * rp + 1][c], 0x7632u);
          }

        auto pair = [&](int c, int rp, int i) -> uint32_t {
          const uint32_t src = pp[c][rp][i >> 2] >> (4 * (i & 3));
          uint32_t v = hsub2_u(and_or(src, 0x000F000Fu, 0x64006400u), zp[c][i]);
          if (!kFactor) {
            const int col = nibble_column(i);
            const uint32_t spair = prmt(sv[c][col >> 1], 0u, (col & 1) ? 0x3232u : 0x1010u);
            v = hmul2_u(v, spair);
          }
          return v;
        };

#pragma unroll
        for (int mi = 0; mi < NMMA; ++mi) {
          const int ca = mma_cw<CWL>(mi, 0), ia = mma_nib<CWL>(mi, 0);
          const int cb = mma_cw<CWL>(mi, 1), ib = mma_nib<CWL>(mi, 1);
          const uint32_t a0 = pair(ca, 0, ia);
          const uint32_t a1 = pair(cb, 0, ib);
          const uint32_t a2 = pair(ca, 1, ia);
          const uint32_t a3 = pair(cb, 1, ib);
#pragma unroll
          for (int b = 0; b < TB; ++b) {
            if (kFactor) mma16816(accg[mi][b], a0, a1, a2, a3, bx[b][0], bx[b][1]);
            else mma16816(acc[mi][b], a0, a1, a2, a3, bx[b][0], bx[b][1]);
          }
        }

        // Refill this slot with the k-step kD ahead.
        const int tn = t + kD;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (cw_ok && tn < t_end) ldg_stream<CWL>(wb[d][r], qbase + (long long)(16 * tn + r) * p.C);
        }
      }
    }
  }
  if (kFactor && cur >= 0) fold();

  // 4. Reduce: warps of the CTA (fixed order), then CTAs of the cluster (fixed order).
  float* mine = red + warp * E;
#pragma unroll
  for (int mi = 0; mi < NMMA; ++mi)
#pragma unroll
    for (int b = 0; b < TB; ++b)
#pragma unroll
      for (int j = 0; j < 4; ++j) mine[((mi * TB + b) * 4 + j) * 32 + lane] = acc[mi][b][j];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kNW * 32) {
    float s = red[e];
#pragma unroll
    for (int w = 1; w < kNW; ++w) s += red[w * E + e];
    red[e] = s;
  }
  cluster_sync_all();

  const int e_lo = static_cast<int>((long long)E * rank / cs);
  const int e_hi = static_cast<int>((long long)E * (rank + 1) / cs);
  for (int e = e_lo + threadIdx.x; e < e_hi; e += kNW * 32) {
    float s = 0.f;
    for (int r = 0; r < cs; ++r) s += ld_dsmem(red + e, static_cast<uint32_t>(r));
    const int ln = e & 31;
    const int j = (e >> 5) & 3;
    const int b = (e >> 7) % TB;
    const int mi = (e >> 7) / TB;
    const int rs = j >> 1;
    const int tok = m0 + 8 * b + 2 * (ln & 3) + (j & 1);
    const int cw = cwb + (ln >> 2) * CWL + mma_cw<CWL>(mi, rs);
    const int n = 8 * cw + nibble_column(mma_nib<CWL>(mi, rs));
    if (tok < p.M && cw < p.C) {
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

template <int TB, int CWL, bool F>
cudaError_t launch_variant(const DecodeParams& dp, dim3 grid, int cs, size_t smem, cudaStream_t st) {
  auto kern = decode_kernel<TB, CWL, F>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kNW * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, dp);
}

Variant pick_variant(const GemmProblem& p) {
  const int C = p.N / 8;
  if (p.M <= 8) return (C % 2 == 0) ? Variant{1, 2, true} : Variant{1, 1, true};
  if (p.M <= 16) return Variant{2, 1, true};
  return Variant{4, 1, false};
}

struct Plan {
  Variant v;
  int cs;
  int grp_cap;
  size_t smem;
  dim3 grid;
};

bool make_plan(const GemmProblem& p, Plan* plan, const char** why) {
  const int C = p.N / 8;
  const int T = p.K / 16;
  const Variant v = pick_variant(p);
  const int cw_cta = 8 * v.CWL;
  const long long nbl = (C + cw_cta - 1) / cw_cta;
  const long long mz = (p.M + 8 * v.TB - 1) / (8 * v.TB);
  if (mz > 65535) { *why = "M too large for the decode grid"; return false; }
  // Cluster split of K: grow until the grid has about two CTAs per SM, keeping at least
  // one k16-step per warp.
  int cs = 1;
  while (cs < 8 && nbl * mz * cs < 2 * 152 && T >= 2 * cs * kNW) cs *= 2;
  const size_t red_bytes = (size_t)kNW * (4 * v.CWL) * v.TB * 4 * 32 * sizeof(float);
  for (;;) {
    const int rows = (T + cs - 1) / cs * 16;            // max k-rows per CTA
    const int grp_cap = rows / p.G + 2;
    const size_t meta = (size_t)grp_cap * cw_cta * 20;
    if (meta + red_bytes <= 200 * 1024) {
      plan->v = v;
      plan->cs = cs;
      plan->grp_cap = grp_cap;
      plan->smem = meta + red_bytes;
      if (nbl * cs > 0x7fffffffLL) { *why = "N too large for the decode grid"; return false; }
      plan->grid = dim3(static_cast<unsigned>(nbl * cs), static_cast<unsigned>(mz), 1);
      return true;
    }
    if (cs >= 8) break;
    cs *= 2;
  }
  *why = "zero/scale rows per CTA exceed shared memory";
  return false;
}

}  // namespace

bool decode_ldg_supported(const GemmProblem& p, const char** why) {
  static const char* dummy;
  if (!why) why = &dummy;
  if (p.bits != 4) { *why = "4-bit codes only"; return false; }
  if (p.K % 16 != 0) { *why = "decode needs K % 16 == 0"; return false; }
  if (p.G % 16 != 0) { *why = "decode needs group_size % 16 == 0"; return false; }
  const Variant v = pick_variant(p);
  if (!aligned(p.x, 8)) { *why = "decode needs x 8-byte aligned"; return false; }
  if (!aligned(p.qw, 4 * v.CWL)) { *why = "decode needs qweight aligned to its vector width"; return false; }
  if (!aligned(p.sc, 16)) { *why = "decode needs scales 16-byte aligned"; return false; }
  Plan plan;
  return make_plan(p, &plan, why);
}

cudaError_t launch_decode_ldg(const GemmProblem& p) {
  Plan plan;
  const char* why = nullptr;
  if (!make_plan(p, &plan, &why)) return cudaErrorInvalidValue;
  DecodeParams dp;
  dp.x = p.x; dp.qw = p.qw; dp.qz = p.qz; dp.sc = p.sc; dp.bias = p.bias; dp.y = p.y;
  dp.M = p.M; dp.K = p.K; dp.N = p.N; dp.C = p.N / 8; dp.G = p.G;
  dp.grp_cap = plan.grp_cap;
  const Variant v = plan.v;
  if (v.TB == 1 && v.CWL == 2) return launch_variant<1, 2, true>(dp, plan.grid, plan.cs, plan.smem, p.stream);
  if (v.TB == 1 && v.CWL == 1) return launch_variant<1, 1, true>(dp, plan.grid, plan.cs, plan.smem, p.stream);
  if (v.TB == 2) return launch_variant<2, 1, true>(dp, plan.grid, plan.cs, plan.smem, p.stream);
  return launch_variant<4, 1, false>(dp, plan.grid, plan.cs, plan.smem, p.stream);
}

bool decode_supported(const GemmProblem& p, const char** why) {
  if (p.bf16) return decode_tma_supported(p, why);  // the register-streaming kernel is fp16-only
  if (decode_tma_supported(p, nullptr)) return true;
  return decode_ldg_supported(p, why);
}

cudaError_t launch_decode(const GemmProblem& p) {
  if (decode_tma_supported(p, nullptr)) return launch_decode_tma(p);
  return launch_decode_ldg(p);
}

}  // namespace awq
