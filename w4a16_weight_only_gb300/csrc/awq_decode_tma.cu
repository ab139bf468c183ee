// Decode path of awq_gemm, TMA-fed (small M, HBM-bound):
//
//   y[m][n] = sum_k x[m][k] * (code[k][n] - zero[k/G][n]) * scale[k/G][n]  (+ bias[n])
//
// (tensref.org/formats/awq, "Reader"; GPTQModel wiki "AWQ", "Native GEMM": fused
// dequant-GEMM, fp32 accumulation, split over K.)
//
// Streaming.  Every warp owns a contiguous run of 64-row stages of one column tile (16
// packed words, 64-byte rows) and streams it through its own ring of S slots (S set at
// launch from the shared memory each CTA gets): lane 0 issues the bulk tensor copies
// (packed weights, the group's zero and scale rows when a stage opens a group, the
// activations) on the slot's mbarrier, the warp waits with a bounded try-wait, computes,
// and refills the slot.  The weight copies are issued before the kernel waits on the
// preceding grid (programmatic dependent launch): only the activation copies and the
// output stores are ordered after it, so the weight stream of one linear overlaps the
// tail of the previous kernel.
//
// Unpack (kSub mode, up to 16 activation rows).  Two rows (k, k+1) of one packed column
// are byte-permuted (prmt) so each 16-bit half holds one row's nibbles; one AND per
// nibble pair leaves the code in the low mantissa bits of an fp16, i.e. the exact
// subnormal value c * 2^-24 (even nibbles, bits 0-3) or c * 2^-20 (odd nibbles, bits
// 4-7), for both rows at once.  Those half2 pairs are the A operand of m16n8k16
// tensor-core MMAs (weights on the 16-row side, activations on the 8-wide side) that
// accumulate sum_k x * c per quantization group in fp32 (tensor cores take fp16
// subnormals exactly).  One more MMA with an all-ones A operand accumulates sum_k x.
// When the group ends, each output element gets
//     acc += scale * (2^24 (or 2^20) * sum x c  -  zero * sum x)
// which is sum x (c - zero) * scale with no per-weight zero subtraction or scaling.
// (kExact mode, 17..32 rows: the A operand is the exact fp16 weight (c - zero) * scale,
// formed with the 0x6400 exponent trick, HSUB2 and HMUL2; accumulators go straight to
// the output sums.)
//
// Split-K: the warps of a CTA and the CTAs of a thread-block cluster take consecutive K
// ranges.  Each CTA sums its warps' partials in a fixed order in shared memory and pushes
// the result (st.async into distributed shared memory, counted on an mbarrier) to the
// cluster's rank-0 CTA, which adds the partials in rank order, adds the bias and stores
// y; the other CTAs exit right after their push.  No global workspace, no atomics:
// repeated calls are bitwise identical.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "awq_internal.cuh"
#include "awq_ptx.cuh"

namespace awq {
namespace {

using namespace ptx;

#ifndef AWQ_DECODE_WARPS
#define AWQ_DECODE_WARPS 4
#endif
constexpr int kNW = AWQ_DECODE_WARPS;  // warps per CTA (the one-token variant may take 8)
#ifndef AWQ_DECODE_L2_PREFETCH
#define AWQ_DECODE_L2_PREFETCH 0  // L2 prefetch of the stages past the ring, before the wait
#endif
constexpr int kRS = 64;      // rows of K per stage
constexpr int kMaxCluster = 16;
constexpr uint32_t kMagic = 0x64006400u;     // fp16 1024 in both halves
constexpr uint32_t kOnes = 0x3C003C00u;      // fp16 1.0 in both halves
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 200 ms per wait
// One-token variant: quantization groups a warp may span (one MMA token column each).
constexpr int kOneGroups = 8;
constexpr unsigned int kStatusDecodeTimeout = 0x1u;

struct __align__(64) TmaDecodeParams {
  CUtensorMap tm_w;  // qweight [K][C] u32, box {CW_W, 64}, unswizzled
  CUtensorMap tm_x;  // x [M][K] f16, box {64, x_rows}, 128B swizzle
  CUtensorMap tm_z;  // qzeros [K/G][C] u32, box {CW_W, 1}
  CUtensorMap tm_s;  // scales [K/G][N] f16, box {8*CW_W, 1}
  const __half* bias;
  __half* y;
  unsigned int* status;
  int M, K, N, C, G;
  int x_rows;   // rows of the activation box: min(M, 8*TB)
  int slots;    // ring slots per warp
  int meta_n;   // meta entries per warp: ring slots, or (one token) groups of the warp
  int x_pitch;  // bytes per activation slot: 128 (one row, unswizzled) or 1024*TB
  // Byte offsets inside the 1024-aligned dynamic shared memory (activation rings at 0).
  int w_off, m_off, zl_off, bias_off, bar_off, recv_off;
  int owners;  // CTAs of the cluster that finish a slice of the output tile (1 or cs)
  const int* offsets;  // grouped: expert row offsets (device, E + 1), else null
  int E;               // grouped: experts
  int slice;   // floats of the packed partial each owner finishes (multiple of 4)
  int early;   // 1: the caller declared the weights static; stream them before the grid wait
};

template <int TB, int CWL, int NW, int BITS = 4>
struct Geo {
  static_assert(BITS == 4 || BITS == 8, "4- or 8-bit codes");
  static constexpr int CPW = 32 / BITS;             // columns per packed word
  static constexpr int CW_W = 8 * CWL;              // packed column-words per warp / CTA
  static constexpr int NCOL = CPW * CW_W;           // output columns per CTA
  static constexpr int W_BYTES = kRS * CW_W * 4;    // packed weight tile per stage
  static constexpr int Z_BYTES = CW_W * 4;
  static constexpr int S_BYTES = NCOL * 2;
  static constexpr int META_SLOT = ((128 + S_BYTES + 127) / 128) * 128;  // zeros at 0, scales at 128
  static constexpr uint32_t META_TX = Z_BYTES + S_BYTES;
  static constexpr int NMMA = (CPW / 2) * CWL;      // 16-column MMAs per k16-step
  static constexpr int E = NMMA * TB * 4 * 32;      // partial sums per warp
  static constexpr int PACK = 8 * TB * NCOL;        // packed partial: tokens x columns
  static constexpr int EP = E + E / 128;            // partials per warp, padded
  static constexpr int RED_BYTES = (NW * EP + PACK) * 4;  // reuses the activation+weight rings
};

__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

#ifndef AWQ_DECODE_MIN_BLOCKS_M8
#define AWQ_DECODE_MIN_BLOCKS_M8 3
#endif
// CTAs per SM the register budget must allow (3: up to 168 registers a thread; tighter
// budgets measured slower, the extra registers buy instruction-level parallelism).
#ifndef AWQ_DECODE_MIN_BLOCKS_WIDE
#define AWQ_DECODE_MIN_BLOCKS_WIDE 3
#endif
// 8-warp CTAs: two per SM (up to 128 registers a thread).
template <int TB, int NW>
constexpr int kMinBlocks = NW == 8 ? 2 : (TB == 1 ? AWQ_DECODE_MIN_BLOCKS_M8 : AWQ_DECODE_MIN_BLOCKS_WIDE);

// kOne: exactly one activation row (M = 1).  The MMA's 8 token columns would hold 7
// zero columns, so they hold the warp's quantization groups instead: the activations of a
// stage of group slot gs (groups counted from the warp's first one, at most kOneGroups)
// go into token column 2 (gs % 4) + gs / 4, the other columns read zeros.  Each column
// then accumulates sum x c (and, in the ones-MMA, sum x) of one group on its own, so no
// accumulator is folded or cleared inside the loop; after it every lane folds the groups
// of its own columns once (zero and scale rows kept in a per-warp stash indexed by group
// slot) and the reduction also sums over the four lanes of each quad.
// kBF: bf16 activations, scales, bias and output.  A code c then enters the MMA as the
// exact bf16 value 128 + c (0x4300 | c: the subnormal trick has no room for a 4-bit code
// above bf16's 7-bit significand without leaving fp32's normal range in the products), so
// the fold is acc += scale * (sum x (128 + c) - (128 + zero) * sum x).
// kGrp: grouped (mixture-of-experts) launch.  Weights, zeros, scales (and bias) are stacked
// over E experts and read through 3D tensor maps; blockIdx.y counts 8-row tiles over the
// experts in order, each CTA finding its expert and rows in the device offsets after the
// grid-dependency wait (the offsets come from the routing); tiles past the last expert's
// exit at once (whole clusters share blockIdx.y).  Rows of a tile that belong to the next
// expert are computed and discarded.
// BITS = 8: four 8-bit codes per word, byte i of word c is column 4c + i (no interleave).
// A lane's half-word then holds two columns of one K row; the codes enter the MMA as the
// exact fp16 subnormals c * 2^-24 (both bytes: an 8-bit code fits the 10-bit subnormal
// significand), or as 1024 + c in the exact-operand variant.  Same tiles, ring, cluster
// reduction and launch plan as 4 bits, half the output columns per CTA.  fp16 only
// (128 + c leaves bf16's 8 significant bits for c > 127).
template <int TB, int CWL, bool kSub, bool kOne, int NW, bool kBF, bool kGrp = false, int BITS = 4>
__global__ void __launch_bounds__(NW * 32, kMinBlocks<TB, NW>)
    decode_tma_kernel(const __grid_constant__ TmaDecodeParams p) {
  static_assert(!kGrp || (TB == 1 && !kOne), "grouped launches use 8-row tiles");
  static_assert(BITS == 4 || (!kBF && !kGrp), "8-bit codes: fp16, plain launches");
  static_assert(NW == 4 || NW == 8, "4 or 8 warps per CTA");
  constexpr uint32_t kOne2 = kBF ? 0x3F803F80u : kOnes;     // 1.0 in both halves
  constexpr uint32_t kMag = kBF ? 0x43004300u : kMagic;     // 128 (bf16) / 1024 (fp16)
  constexpr uint32_t kMag64 = 0x54005400u;                   // fp16 64 in both halves
  constexpr float kBias = kBF ? 128.f : 0.f;                 // offset the operand carries
  using GE = Geo<TB, CWL, NW, BITS>;
  constexpr int NMMA = GE::NMMA;
  constexpr int CPW = GE::CPW, NCOL = GE::NCOL;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.slots;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g8 = lane >> 2;
  const int q = lane & 3;
  const uint32_t rank = cluster_ctarank();
  const uint32_t cs = cluster_nctarank();
  const int cw0 = static_cast<int>(blockIdx.x / cs) * GE::CW_W;
  int m0 = blockIdx.y * 8 * TB;
  int m_lim = p.M;  // rows of this tile are m0 .. min(m0 + 8 TB, m_lim) - 1
  int ex = 0;       // expert (grouped)
  if constexpr (kGrp) {
    grid_dependency_wait();
    int t = static_cast<int>(blockIdx.y);
    bool found = false;
    for (int e = 0; e < p.E && !found; ++e) {
      const int a = p.offsets[e], b = p.offsets[e + 1];
      const int n = b > a ? (b - a + 8 * TB - 1) / (8 * TB) : 0;
      if (t < n) {
        m0 = a + 8 * TB * t;
        m_lim = min(b, p.M);
        ex = e;
        found = true;
      } else {
        t -= n;
      }
    }
    if (!found) return;
  }

  // 32-bit arithmetic throughout: TS * P < 2^31 (checked on the host).
  const uint32_t TS = static_cast<uint32_t>(p.K / kRS);
  const uint32_t P = cs * NW;
  const uint32_t wid = rank * NW + static_cast<uint32_t>(warp);
  const int j0 = static_cast<int>(TS * wid / P);
  const int j1 = static_cast<int>(TS * (wid + 1) / P);

  unsigned char* x_ring = smem + (size_t)warp * S * p.x_pitch;
  unsigned char* w_ring = smem + p.w_off + (size_t)warp * S * GE::W_BYTES;
  // Meta rows: a ring of S slots, or (kOne) a stash with one entry per group of the warp.
  unsigned char* m_ring = smem + p.m_off + (size_t)warp * p.meta_n * GE::META_SLOT;
  uint64_t* my_bars = bars + warp * S;
  const uint32_t x_ring_u32 = smem_u32(x_ring);
  const uint32_t w_ring_u32 = smem_u32(w_ring);
  const uint32_t m_ring_u32 = smem_u32(m_ring);

#ifdef AWQ_DECODE_DEBUG_TIME
  AWQ_DECODE_DEBUG_TIME(0);
#endif
  // Reduction mbarrier (after all ring barriers): in the cluster's rank-0 CTA it counts
  // the bytes of the partial sums every CTA of the cluster pushes (its own included).
  uint64_t* red_bar = bars + NW * S;
  const int pack_n = p.x_rows * NCOL;  // floats of one packed partial
  if (lane == 0) {
    prefetch_tmap(&p.tm_w);
    prefetch_tmap(&p.tm_x);
    for (int s = 0; s < S; ++s) mbar_init(&my_bars[s], 1);
    if (warp == 0) {
      mbar_init(red_bar, 1);
      const int my_len = min(p.slice, max(0, pack_n - static_cast<int>(rank) * p.slice));
      if (static_cast<int>(rank) < p.owners)
        mbar_arrive_expect_tx(red_bar, cs * static_cast<uint32_t>(my_len) * 4u);
    }
    fence_mbar_init();
  }
  __syncwarp();
  // Publish the barrier initialisation to the cluster; the matching wait comes right
  // before the first push, long after every CTA has arrived here.
  cluster_arrive_relaxed();

  // Stage j of this warp: packed weights always, the group's zero and scale rows only when
  // stage j opens a group (or is the warp's first stage), activations separately.
  // Weights and their metadata are streamed once: evict them from L2 first; the activations
  // (read by every column tile, and the next call's input may be this call's output) last.
  const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
  const int spg = p.G / kRS;  // stages per quantization group
  const uint32_t x_tx = static_cast<uint32_t>(p.x_rows) * kRS * 2;
  // Issue-side stage/group counters (advanced by lane 0 only; no division per stage).
  const int g_first = j0 / spg;  // the warp's first group
  int iss_grp = g_first;
  int iss_left = spg - (j0 - iss_grp * spg);  // stages left in iss_grp, counting the next
  auto issue_weights = [&](int slot, int j) {
    uint64_t* bar = &my_bars[slot];
    const bool meta = (j == j0) || (iss_left == spg);
    mbar_arrive_expect_tx(bar, GE::W_BYTES + x_tx + (meta ? GE::META_TX : 0u));
    if constexpr (kGrp) tma_load_3d(w_ring + slot * GE::W_BYTES, &p.tm_w, bar, cw0, j * kRS, ex);
    else tma_load_2d_hint(w_ring + slot * GE::W_BYTES, &p.tm_w, bar, cw0, j * kRS, pol_w);
    if (meta) {
      unsigned char* md = m_ring + (kOne ? iss_grp - g_first : slot) * GE::META_SLOT;
      if constexpr (kGrp) {
        tma_load_3d(md, &p.tm_z, bar, cw0, iss_grp, ex);
        tma_load_3d(md + 128, &p.tm_s, bar, CPW * cw0, iss_grp, ex);
      } else {
        tma_load_2d_hint(md, &p.tm_z, bar, cw0, iss_grp, pol_w);
        tma_load_2d_hint(md + 128, &p.tm_s, bar, CPW * cw0, iss_grp, pol_w);
      }
    }
    if (--iss_left == 0) {
      ++iss_grp;
      iss_left = spg;
    }
  };
  auto issue_x = [&](int slot, int j) {
    tma_load_2d_hint(x_ring + slot * p.x_pitch, &p.tm_x, &my_bars[slot], j * kRS, m0, pol_x);
  };

  // Static weights (declared by the caller: complete before the preceding kernel launch)
  // do not depend on the preceding grid: stream them first, under its tail.  By default
  // every read waits for the preceding grid.  Activations and the output stores are always
  // ordered after it.
  if (lane == 0 && p.early)
    for (int s = 0; s < S && j0 + s < j1; ++s) issue_weights(s, j0 + s);
#if AWQ_DECODE_L2_PREFETCH
  // Stages past the ring: pull their packed weights (and any group rows they open) into
  // L2 now, so the refills after the wait hit L2.  Whole tiles only (no partial boxes).
  if (lane == 0 && cw0 + GE::CW_W <= p.C)
    for (int j = j0 + S; j < j1; ++j) {
      tma_prefetch_l2_2d(&p.tm_w, cw0, j * kRS);
      if (j % spg == 0) {
        tma_prefetch_l2_2d(&p.tm_z, cw0, j / spg);
        tma_prefetch_l2_2d(&p.tm_s, CPW * cw0, j / spg);
      }
    }
#endif
  grid_dependency_wait();
#ifdef AWQ_DECODE_DEBUG_TIME
  AWQ_DECODE_DEBUG_TIME(5);
#endif
  if (lane == 0) {
    if (!p.early)
      for (int s = 0; s < S && j0 + s < j1; ++s) issue_weights(s, j0 + s);
    for (int s = 0; s < S && j0 + s < j1; ++s) issue_x(s, j0 + s);
  }
#if !AWQ_DECODE_LATE_TRIGGER
  launch_dependents();
#endif

  // Weight fragments: ldmatrix.trans on the 16-bit view of the packed tile.  An 8x8
  // matrix of half-words (8 rows of K x 8 half-words), transposed, hands lane (g8, q) the
  // register (row 2q, row 2q+1) of half-word g8: four nibbles (columns) of two
  // consecutive K rows, paired as the MMA A operand wants.  Per k16-step the warp's tile
  // is row blocks rb (rows 0-7, 8-15) x half-word blocks hb (8 half-words = 4 words);
  // the lane holds half-word 8hb + g8 of every block: word 4hb + g8/2, half g8 % 2.
  // Rows are 64 bytes (TMA 64-byte swizzle) or 32 bytes (32-byte swizzle); the swizzle
  // puts the 8 row reads of every matrix in distinct banks.
  constexpr int HB = GE::CW_W / 4;  // half-word blocks per row
  uint32_t w_lds[2];
  {
    const int rr = lane & 7, jm = lane >> 3;
    if constexpr (CWL == 2) {  // ldmatrix rb: matrices (rb, hb = jm)
#pragma unroll
      for (int rb = 0; rb < 2; ++rb)
        w_lds[rb] = static_cast<uint32_t>((8 * rb + rr) * 64 + 16 * (jm ^ ((rr >> 1) & 3)));
    } else {  // one ldmatrix: matrix jm = (rb, hb) = (jm / 2, jm % 2)
      w_lds[0] = static_cast<uint32_t>((8 * (jm >> 1) + rr) * 32 + 16 * ((jm & 1) ^ ((rr >> 2) & 1)));
      w_lds[1] = w_lds[0];
    }
  }
  const int hh = g8 & 1;  // half of its word each of the lane's half-words is
  const int wq = g8 >> 1;  // word of the lane inside every 4-word block
  const uint32_t sc_sel = hh ? 0x7632u : 0x5410u;  // scales of columns 2n + hh
  // ldmatrix row addresses for the activation tile (128-byte rows, 128B swizzle): lane l
  // addresses row (l & 7) of 16-byte chunk 4*pair + (l >> 3).  Rows past the activation
  // box (fewer than 8 tokens) read this warp's zero line instead.
  const uint32_t zero_line = smem_u32(smem + p.zl_off + warp * 128);
  if (lane < 32) reinterpret_cast<uint32_t*>(smem + p.zl_off + warp * 128)[lane] = 0u;
  __syncwarp();
  // Bias of this CTA's columns, read now (off the critical path) for the epilogue.
  {
    float* bias_s = reinterpret_cast<float*>(smem + p.bias_off);
    for (int i = threadIdx.x; i < NCOL; i += NW * 32) {
      const int n = CPW * cw0 + i;
      bias_s[i] = (p.bias != nullptr && n < p.N)
                      ? elem_to_float<kBF>(reinterpret_cast<const uint16_t*>(p.bias)[(long long)ex * p.N + n])
                      : 0.f;
    }
  }
  uint32_t x_off[TB][2];
  bool x_real[TB];
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) {
    const int rr = lane & 7;
    x_real[tb] = (8 * tb + rr) < p.x_rows;
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const int chunk = 4 * pr + (lane >> 3);
      x_off[tb][pr] = x_real[tb]
                          ? static_cast<uint32_t>((8 * tb + rr) * 128 + ((chunk ^ rr) << 4))
                          : static_cast<uint32_t>(chunk << 4);
    }
  }

  float acc[NMMA][TB][4];
#pragma unroll
  for (int i = 0; i < NMMA; ++i)
#pragma unroll
    for (int b = 0; b < TB; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][b][e] = 0.f;
  float accg[kSub ? NMMA : 1][TB][4];
  float xs[TB][4];
  if constexpr (kOne) {  // accumulated over the whole range, cleared once
#pragma unroll
    for (int i = 0; i < NMMA; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) accg[i][0][e] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) xs[0][e] = 0.f;
  }
  uint32_t zh[HB];         // the lane's zero half-word (4 nibbles) of every block
  uint32_t sv[HB][2];      // its scales: nibbles (0, 1) and (2, 3) as half2
  uint32_t zp[kSub ? 1 : HB][4];  // kExact: 1024 + zero, per nibble, both halves
  uint32_t sp[kSub ? 1 : HB][4];  // kExact: scale, per nibble, both halves
  auto load_meta = [&](uint32_t mb) {
#pragma unroll
    for (int hb = 0; hb < HB; ++hb) {
      const uint32_t wofs = 4u * static_cast<uint32_t>(4 * hb + wq);  // word offset, bytes
      zh[hb] = lds32(mb + wofs) >> (16 * hh);
      if constexpr (BITS == 8) {  // the half-word's two columns 4w + 2hh, +1: adjacent scales
        sv[hb][0] = lds32(mb + 128 + 2 * wofs + 4 * hh);
        sv[hb][1] = 0u;
      } else {
        const uint4 v = lds128(mb + 128 + 4 * wofs);  // the word's 8 scales, column order
        sv[hb][0] = prmt(v.x, v.y, sc_sel);
        sv[hb][1] = prmt(v.z, v.w, sc_sel);
      }
    }
  };
  // Fold terms of code u (nibble 0-3 / byte 0-1) of the lane's half-word in block hb:
  // its MMA mi (rows g8 + 8 (hb % 2)), the factor on sum x c, and -scale * (zero + offset).
  auto fold8 = [&](int hb, int u, float& sa, float& sz) {
    const float2 s2 = pair_to_float2<false>(sv[hb][0]);
    const float sc = u ? s2.y : s2.x;
    const float z = __uint_as_float(((zh[hb] >> (8 * u)) & 0xFFu) | 0x4B000000u) - 8388608.f;
    sa = sc * 16777216.f;
    sz = -sc * z;
  };
  int cur = -1;
  bool x_on = x_real[0];  // kOne: this lane's ldmatrix row is the current group's column
  // Group of stage j is j / spg; tracked incrementally (one division per warp).
  int grp_of = j0 / spg;
  int grp_left = spg - (j0 - grp_of * spg);  // stages left in grp_of, counting j0

  auto fold = [&]() {
    // acc += scale * (2^24 or 2^20 * sum x c - zero * sum x) for the group just finished.
    // Nibble nib of block hb is MMA mi = 4 (hb / 2) + nib, A rows g8 + 8 (hb % 2); byte u
    // (8 bits) is MMA 2 (hb / 2) + u.
    if constexpr (BITS == 8) {
#pragma unroll
      for (int hb = 0; hb < HB; ++hb)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float sa, sz;
          fold8(hb, u, sa, sz);
          const int mi = 2 * (hb >> 1) + u, rs = hb & 1;
#pragma unroll
          for (int tb = 0; tb < TB; ++tb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float a = __fmaf_rn(sz, xs[tb][e], acc[mi][tb][2 * rs + e]);
              acc[mi][tb][2 * rs + e] = __fmaf_rn(sa, accg[mi][tb][2 * rs + e], a);
            }
        }
    } else {
#pragma unroll
      for (int hb = 0; hb < HB; ++hb)
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const float2 s2 = pair_to_float2<kBF>(sv[hb][pp]);
#pragma unroll
          for (int n2 = 0; n2 < 2; ++n2) {
            const int nib = 2 * pp + n2;
            const float sc = n2 ? s2.y : s2.x;
            // zero nibble as a float: 2^23 + z read as an fp32 bit pattern, minus 2^23
            const float z = __uint_as_float(((zh[hb] >> (4 * nib)) & 0xFu) | 0x4B000000u) - 8388608.f;
            const float sa = kBF ? sc : sc * ((nib & 1) ? 1048576.f : 16777216.f);
            const float sz = -sc * (z + kBias);
            const int mi = 4 * (hb >> 1) + nib, rs = hb & 1;
#pragma unroll
            for (int tb = 0; tb < TB; ++tb)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float a = __fmaf_rn(sz, xs[tb][e], acc[mi][tb][2 * rs + e]);
                acc[mi][tb][2 * rs + e] = __fmaf_rn(sa, accg[mi][tb][2 * rs + e], a);
              }
          }
        }
    }
  };

  int done = j0;  // first stage not yet waited for
  bool failed = false;
  int slot = 0;
  uint32_t parity = 0u;
  for (int j = j0; j < j1; ++j) {
    if (!mbar_wait_bounded(&my_bars[slot], parity, p.status, kStatusDecodeTimeout, kWaitLimitNs)) {
      failed = true;
      break;
    }
    done = j + 1;
#ifdef AWQ_DECODE_DEBUG_TIME
    if (j == j0) AWQ_DECODE_DEBUG_TIME(1);
    if (j == j1 - 1) AWQ_DECODE_DEBUG_TIME(4);
#endif
    const uint32_t xb = x_ring_u32 + slot * p.x_pitch;
    const uint32_t wb = w_ring_u32 + slot * GE::W_BYTES;
    const uint32_t mb = m_ring_u32 + slot * GE::META_SLOT;
    if (grp_left == 0) {
      ++grp_of;
      grp_left = spg;
    }
    --grp_left;
    const int grp = grp_of;
    if (kOne && grp != cur) {
      cur = grp;
      const int gs = grp - g_first;
      x_on = (lane & 7) == 2 * (gs & 3) + (gs >> 2);
    } else if (!kOne && grp != cur) {
      if (kSub && cur >= 0) fold();
      cur = grp;
      load_meta(mb);
      if (kSub) {
#pragma unroll
        for (int i = 0; i < NMMA; ++i)
#pragma unroll
          for (int b = 0; b < TB; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) accg[i][b][e] = 0.f;
#pragma unroll
        for (int b = 0; b < TB; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e) xs[b][e] = 0.f;
      } else {
#pragma unroll
        for (int hb = 0; hb < HB; ++hb) {
          const uint32_t zd = prmt(zh[hb], zh[hb], 0x1010u);  // zero half-word in both halves
          if constexpr (BITS == 8) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              zp[kSub ? 0 : hb][u] = and_or(zd >> (8 * u), 0x00FF00FFu, kMag);
              sp[kSub ? 0 : hb][u] = prmt(sv[hb][0], 0u, u ? 0x3232u : 0x1010u);
            }
          } else {
#pragma unroll
            for (int nib = 0; nib < 4; ++nib) {
              // fp16: odd nibbles stay in bits 4-7 under the exponent of 64 (the operand below)
              zp[kSub ? 0 : hb][nib] = (kBF || !(nib & 1))
                                           ? and_or(zd >> (4 * nib), 0x000F000Fu, kMag)
                                           : and_or(zd >> (4 * nib - 4), 0x00F000F0u, kMag64);
              sp[kSub ? 0 : hb][nib] = prmt(sv[hb][nib >> 1], 0u, (nib & 1) ? 0x3232u : 0x1010u);
            }
          }
        }
      }
    }

#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      // Activation fragments for k16-steps 2pr and 2pr+1: xr[tb][2kk + h] holds token
      // 8tb + g8, k = 16(2pr+kk) + 2q + 8h .. +1.
      uint32_t xr[TB][4];
#pragma unroll
      for (int tb = 0; tb < TB; ++tb)
        ldmatrix_x4(xr[tb], ((kOne ? x_on : x_real[tb]) ? xb : zero_line) + x_off[tb][pr]);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int ks = 2 * pr + kk;
        // wr[rb][hb]: rows (2q + 8rb, +1) of the lane's half-word in block hb
        uint32_t wr[2][HB];
        if constexpr (CWL == 2) {
          uint32_t t0[4], t1[4];
          ldmatrix_x4_trans(t0, wb + w_lds[0] + ks * 16 * 64);
          ldmatrix_x4_trans(t1, wb + w_lds[1] + ks * 16 * 64);
#pragma unroll
          for (int hb = 0; hb < HB; ++hb) {
            wr[0][hb] = t0[hb];
            wr[1][hb] = t1[hb];
          }
        } else {
          uint32_t t0[4];
          ldmatrix_x4_trans(t0, wb + w_lds[0] + ks * 16 * 32);
          wr[0][0] = t0[0]; wr[0][1] = t0[1]; wr[1][0] = t0[2]; wr[1][1] = t0[3];
        }
        auto operand = [&](int rb, int hb, int nib) -> uint32_t {
          const uint32_t s = wr[rb][hb];
          if constexpr (BITS == 8 && kSub) {
            // byte nib of both half-words as the exact fp16 subnormal c * 2^-24
            return (nib ? (s >> 8) : s) & 0x00FF00FFu;
          } else if constexpr (BITS == 8) {
            const uint32_t h = and_or(s >> (8 * nib), 0x00FF00FFu, kMag);  // 1024 + c
            return hmul2(hsub2(h, zp[kSub ? 0 : hb][nib]), sp[kSub ? 0 : hb][nib]);
          } else if constexpr (kSub && kBF) {
            return and_or(s >> (4 * nib), 0x000F000Fu, kMag);  // exact bf16 128 + c
          } else if constexpr (kSub) {
            // exact fp16 subnormals c * 2^-24 (even nibble) or c * 2^-20 (odd nibble)
            return ((nib & 2) ? (s >> 8) : s) & ((nib & 1) ? 0x00F000F0u : 0x000F000Fu);
          } else if constexpr (kBF) {
            const uint32_t h = and_or(s >> (4 * nib), 0x000F000Fu, kMag);
            return hmul2_bf16(hsub2_bf16(h, zp[kSub ? 0 : hb][nib]), sp[kSub ? 0 : hb][nib]);
          } else {
            // fp16 1024 + c (even nibble, bits 0-3) or 64 + c (odd nibble left in bits 4-7:
            // the mantissa step of 64 is 1/16), exact either way; one shift serves nibbles 2, 3
            const uint32_t h = (nib & 1) ? and_or((nib & 2) ? (s >> 8) : s, 0x00F000F0u, kMag64)
                                         : and_or((nib & 2) ? (s >> 8) : s, 0x000F000Fu, kMag);
            return hmul2(hsub2(h, zp[kSub ? 0 : hb][nib]), sp[kSub ? 0 : hb][nib]);
          }
        };
#pragma unroll
        for (int mi = 0; mi < NMMA; ++mi) {
          // 4 bits: MMA mi = nibble mi % 4 of blocks 2 (mi / 4), +1; 8 bits: byte mi % 2 of
          // blocks 2 (mi / 2), +1
          const int hb0 = BITS == 8 ? 2 * (mi >> 1) : 2 * (mi >> 2), nib = BITS == 8 ? (mi & 1) : (mi & 3);
          const uint32_t a0 = operand(0, hb0, nib), a1 = operand(0, hb0 + 1, nib);
          const uint32_t a2 = operand(1, hb0, nib), a3 = operand(1, hb0 + 1, nib);
#pragma unroll
          for (int tb = 0; tb < TB; ++tb) {
            if constexpr (kSub && kBF)
              mma16816_bf16(accg[mi][tb], a0, a1, a2, a3, xr[tb][2 * kk], xr[tb][2 * kk + 1]);
            else if constexpr (kSub)
              mma16816(accg[mi][tb], a0, a1, a2, a3, xr[tb][2 * kk], xr[tb][2 * kk + 1]);
            else if constexpr (kBF)
              mma16816_bf16(acc[mi][tb], a0, a1, a2, a3, xr[tb][2 * kk], xr[tb][2 * kk + 1]);
            else
              mma16816(acc[mi][tb], a0, a1, a2, a3, xr[tb][2 * kk], xr[tb][2 * kk + 1]);
          }
        }
        if (kSub) {
#pragma unroll
          for (int tb = 0; tb < TB; ++tb)
            if constexpr (kBF) mma16816_bf16(xs[tb], kOne2, kOne2, kOne2, kOne2, xr[tb][2 * kk], xr[tb][2 * kk + 1]);
            else mma16816(xs[tb], kOne2, kOne2, kOne2, kOne2, xr[tb][2 * kk], xr[tb][2 * kk + 1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && j + S < j1) {
      issue_weights(slot, j + S);
      issue_x(slot, j + S);
    }
    if (++slot == S) {
      slot = 0;
      parity ^= 1u;
    }
  }
  // kOne: the fold of every group, once; lane (g8, q) owns group slots q and q + 4
  // (token columns 2q and 2q + 1).  out[mi][rs]: rows g8 + 8 rs of MMA mi.
  float out[kOne ? NMMA : 1][2];
  if constexpr (kOne) {
#pragma unroll
    for (int mi = 0; mi < NMMA; ++mi) out[mi][0] = out[mi][1] = 0.f;
    const int ng = j1 > j0 ? (j1 - 1) / spg - g_first + 1 : 0;  // groups of this warp
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int gs = q + 4 * e;
      if (e == 1 && ng <= 4) continue;  // warp-uniform
      if (failed || gs >= ng) continue;
      load_meta(m_ring_u32 + gs * GE::META_SLOT);
      if constexpr (BITS == 8) {
#pragma unroll
        for (int hb = 0; hb < HB; ++hb)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            float sa, sz;
            fold8(hb, u, sa, sz);
            const int mi = 2 * (hb >> 1) + u, rs = hb & 1;
            const float a = __fmaf_rn(sz, xs[0][e], out[mi][rs]);
            out[mi][rs] = __fmaf_rn(sa, accg[mi][0][2 * rs + e], a);
          }
      } else {
#pragma unroll
        for (int hb = 0; hb < HB; ++hb)
#pragma unroll
          for (int pp = 0; pp < 2; ++pp) {
            const float2 s2 = pair_to_float2<kBF>(sv[hb][pp]);
#pragma unroll
            for (int n2 = 0; n2 < 2; ++n2) {
              const int nib = 2 * pp + n2;
              const float sc = n2 ? s2.y : s2.x;
              const float z = __uint_as_float(((zh[hb] >> (4 * nib)) & 0xFu) | 0x4B000000u) - 8388608.f;
              const float sa = kBF ? sc : sc * ((nib & 1) ? 1048576.f : 16777216.f);
              const float sz = -sc * (z + kBias);
              const int mi = 4 * (hb >> 1) + nib, rs = hb & 1;
              const float a = __fmaf_rn(sz, xs[0][e], out[mi][rs]);
              out[mi][rs] = __fmaf_rn(sa, accg[mi][0][2 * rs + e], a);
            }
          }
      }
    }
  }
  if (kSub && !kOne && cur >= 0 && !failed) fold();
  if (failed) {
    // Let copies already issued land (bounded) before the slots are reused below.
    const int issued_end = min(j1, done + S);
    for (int j = done; j < issued_end; ++j) {
      const int slot = (j - j0) % S;
      const uint32_t parity = static_cast<uint32_t>(((j - j0) / S) & 1);
      mbar_wait_bounded(&my_bars[slot], parity, p.status, kStatusDecodeTimeout, kWaitLimitNs);
    }
  }

#ifdef AWQ_DECODE_DEBUG_TIME
  AWQ_DECODE_DEBUG_TIME(2);
#endif
#if AWQ_DECODE_LATE_TRIGGER
  launch_dependents();
#endif
  // Reduce: the warps of the CTA in a fixed order into a packed partial [token][column];
  // slice o of it is pushed (st.async, counted on the owner's mbarrier) into owner CTA o,
  // which adds the cluster's partials of its slice in rank order, adds the bias and stores
  // y.  One owner (rank 0) for small partials, every CTA a slice for large ones; CTAs that
  // own nothing exit right after their push.
  __syncthreads();  // the ring is reused as the reduction buffer
  // Per-warp partials in fragment order (row X = (mi*TB + tb)*4 + e, 32 lanes), one float
  // of padding per 4 rows so the packed-order reads below spread over the banks.
  float* red = reinterpret_cast<float*>(smem);
  float* mine = red + warp * GE::EP;
#pragma unroll
  for (int mi = 0; mi < NMMA; ++mi)
#pragma unroll
    for (int tb = 0; tb < TB; ++tb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (kOne && (e & 1)) continue;  // the token-0 slots carry the lane's fold
        const int X = (mi * TB + tb) * 4 + e;
        mine[X * 32 + lane + (X >> 2)] = kOne ? out[mi][e >> 1] : acc[mi][tb][e];
      }
  __syncthreads();
  // Packed partial: element (token t, column col) of the tile, summed over the warps.
  // Column col = 32 hb + 8 (g8 / 2) + 2 nib + g8 % 2 comes from lane group g8, nibble nib
  // of block hb, i.e. MMA mi = 4 (hb / 2) + nib, rows g8 + 8 (hb % 2); g8 varies fastest
  // across threads, the token slowest.
  float* pack = red + NW * GE::EP;
  // 8 bits: column col = 16 hb + 4 (g8 / 2) + 2 (g8 % 2) + u from byte u of block hb, MMA
  // mi = 2 (hb / 2) + u.
  for (int i = threadIdx.x; i < pack_n; i += NW * 32) {
    const int g8i = i & 7, r = i >> 3;
    constexpr int U = CPW / 2, LU = BITS == 8 ? 1 : 2;  // codes per half-word, log2
    const int nib = r & (U - 1), hb = (r >> LU) % HB, t = (r >> LU) / HB;
    const int col = BITS == 8 ? 16 * hb + 4 * (g8i >> 1) + 2 * (g8i & 1) + nib
                              : 32 * hb + 8 * (g8i >> 1) + 2 * nib + (g8i & 1);
    const int mi = U * (hb >> 1) + nib, rs = hb & 1;
    const int X = (mi * TB + (t >> 3)) * 4 + 2 * rs + (t & 1);
    const int e = X * 32 + g8i * 4 + ((t & 7) >> 1) + (X >> 2);
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      if constexpr (kOne) {  // the quad's four lanes hold different groups
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) v += red[w * GE::EP + e + qq];
      } else {
        v += red[w * GE::EP + e];
      }
    }
    pack[t * NCOL + col] = v;
  }
  __syncthreads();
#ifdef AWQ_DECODE_DEBUG_TIME
  AWQ_DECODE_DEBUG_TIME(6);
#endif
  float* recv = reinterpret_cast<float*>(smem + p.recv_off);
  cluster_wait_acquire();  // rank 0's receive barrier is initialised
#ifdef AWQ_DECODE_DEBUG_TIME
  AWQ_DECODE_DEBUG_TIME(7);
#endif
  for (int v = threadIdx.x; v < pack_n / 4; v += NW * 32) {
    const int owner = (4 * v) / p.slice;
    st_async_dsmem_v4(recv + rank * p.slice + (4 * v - owner * p.slice), red_bar,
                      static_cast<uint32_t>(owner), *reinterpret_cast<const float4*>(pack + 4 * v));
  }
  if (static_cast<int>(rank) >= p.owners) {
#ifdef AWQ_DECODE_DEBUG_TIME
    AWQ_DECODE_DEBUG_TIME(3);
#endif
    return;
  }
  const bool got = mbar_wait_bounded(red_bar, 0u, p.status, kStatusDecodeTimeout, kWaitLimitNs);
#ifdef AWQ_DECODE_DEBUG_TIME
  AWQ_DECODE_DEBUG_TIME(8);
#endif
  const float* bias_s = reinterpret_cast<const float*>(smem + p.bias_off);
  const int lo = static_cast<int>(rank) * p.slice;
  const int hi = min(pack_n, lo + p.slice);
  for (int i = lo + threadIdx.x; got && i < hi; i += NW * 32) {
    const int t = i / NCOL, col = i - t * NCOL;
    if (m0 + t >= m_lim || m0 + t < 0 || CPW * cw0 + col >= p.N) continue;
    float sum = 0.f;
    for (uint32_t r = 0; r < cs; ++r) sum += recv[r * p.slice + (i - lo)];
    reinterpret_cast<uint16_t*>(p.y)[(long long)(m0 + t) * p.N + CPW * cw0 + col] =
        float_to_elem<kBF>(sum + bias_s[col]);
  }
#ifdef AWQ_DECODE_DEBUG_TIME
  AWQ_DECODE_DEBUG_TIME(3);
#endif
}

struct Variant {
  int TB, CWL;
  bool sub;
};

#ifndef AWQ_DECODE_TB1_MAX_M
#define AWQ_DECODE_TB1_MAX_M 8
#endif
Variant pick(const GemmProblem& p) {
  if (p.M <= AWQ_DECODE_TB1_MAX_M) return Variant{1, 2, true};
  // 9..16 rows: two 8-row tiles of the wide variant beat one 16-row tile of the narrow one
  // where N is at most 4096 (4096 x 4096, 11008 x 4096: 6-8 % faster), not above
  if (p.M <= 16 && p.N <= 4096) return Variant{1, 2, true};
  if (p.M <= 16) return Variant{2, 1, true};
  return Variant{4, 1, false};
}

constexpr int kRecvCap = 64 * 1024;  // bytes of a CTA's receive region
// One owner sums cs partials of pack_n floats; from this many values on (and clusters of
// at least 4) every CTA of the cluster finishes a slice instead.
constexpr int kMultiOwnerMin = 4096;
// Launch-plan limits (compile-time; overridable for tuning builds).
#ifndef AWQ_DECODE_LATE_TRIGGER
#define AWQ_DECODE_LATE_TRIGGER 0
#endif
#ifndef AWQ_DECODE_WIDE_X
#define AWQ_DECODE_WIDE_X 0
#endif
#ifndef AWQ_DECODE_WIDE_STAGES
#define AWQ_DECODE_WIDE_STAGES 5  // one-token variant: stages per warp that call for 8 warps
#endif
constexpr int kWideStages = AWQ_DECODE_WIDE_STAGES;
#ifndef AWQ_DECODE_WIDE_SLOTS
#define AWQ_DECODE_WIDE_SLOTS 2  // ring slots per warp of 8-warp CTAs
#endif
#ifndef AWQ_DECODE_MAX_SLOTS
#define AWQ_DECODE_MAX_SLOTS 4
#endif
#ifndef AWQ_DECODE_WAVE_FILL_PCT
#define AWQ_DECODE_WAVE_FILL_PCT 90
#endif
#ifndef AWQ_DECODE_MAX_CTAS_PER_SM
#define AWQ_DECODE_MAX_CTAS_PER_SM 4
#endif
constexpr int kMaxSlots = AWQ_DECODE_MAX_SLOTS;             // ring slots per warp
constexpr int kWaveFillPct = AWQ_DECODE_WAVE_FILL_PCT;      // share of the slots one wave may fill
constexpr int kMaxCtasPerSm = AWQ_DECODE_MAX_CTAS_PER_SM;   // CTAs of one launch per SM

// Cluster size, ring depth and shared memory layout of one launch.
struct Plan {
  int cs = 0, slots = 0, x_pitch = 0, meta_n = 0;
  int w_off = 0, m_off = 0, zl_off = 0, bias_off = 0, bar_off = 0, recv_off = 0, smem = 0;
  int owners = 1, slice = 0;
};

template <int TB, int CWL, bool O, int NW, int BITS = 4>
Plan layout(int cs, int slots, int x_rows, int groups) {
  using GE = Geo<TB, CWL, NW, BITS>;
  const int meta_entries = O ? groups : slots;  // stash per group, or ring per slot
  Plan pl;
  pl.cs = cs;
  pl.slots = slots;
  pl.meta_n = meta_entries;
  pl.x_pitch = (x_rows == 1 && !AWQ_DECODE_WIDE_X) ? 128 : 1024 * TB;
  pl.w_off = NW * slots * pl.x_pitch;
  pl.m_off = pl.w_off + NW * slots * GE::W_BYTES;
  pl.zl_off = pl.m_off + NW * meta_entries * GE::META_SLOT;
  pl.bias_off = pl.zl_off + NW * 128;
  pl.bar_off = pl.bias_off + GE::NCOL * 4;
  pl.recv_off = ((pl.bar_off + (NW * slots + 1) * 8 + 15) / 16) * 16;
  const int pack_n = x_rows * GE::NCOL;
  pl.owners = (pack_n * cs >= kMultiOwnerMin && cs >= 4) ? cs : 1;
  pl.slice = pl.owners == 1 ? pack_n : ((pack_n + 4 * cs - 1) / (4 * cs)) * 4;
  pl.smem = 1024 + pl.recv_off + cs * pl.slice * 4;
  return pl;
}

struct DevLimits {
  int sms = 0, smem_per_sm = 0, smem_optin = 0, reserved = 0;
};

cudaError_t dev_limits(DevLimits* out) {
  static std::mutex mu;
  static DevLimits cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  DevLimits& d = cache[dev];
  if (d.sms == 0) {
    DevLimits t;
    e = cudaDeviceGetAttribute(&t.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&t.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&t.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&t.reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    d = t;
  }
  *out = d;
  return cudaSuccess;
}

// Most quantization groups one warp's stage range touches: warp w of the P warps of a
// column tile takes stages [TS w / P, TS (w + 1) / P), spg stages per group.
int max_warp_groups(int TS, int P, int spg) {
  int worst = 0;
  for (int w = 0; w < P; ++w) {
    const int j0 = static_cast<int>(static_cast<long long>(TS) * w / P);
    const int j1 = static_cast<int>(static_cast<long long>(TS) * (w + 1) / P);
    if (j1 > j0 && (j1 - 1) / spg - j0 / spg + 1 > worst) worst = (j1 - 1) / spg - j0 / spg + 1;
  }
  return worst;
}

// Co-resident clusters of size cs at `smem` bytes per CTA (occupancy API).
template <int TB, int CWL, bool S, bool O, int NW, bool B, bool GR = false, int BITS = 4>
int max_clusters(int cs, int smem) {
  auto kern = decode_tma_kernel<TB, CWL, S, O, NW, B, GR, BITS>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, 1, 1);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  return n;
}

// Plan: the cluster size giving the largest grid that is resident in one wave while
// leaving some slots free (the next kernel's clusters can start while this one drains),
// each warp keeping at least one 64-row stage; ties go to the smaller cluster.  Ring
// depth: as many slots as the shared memory left per CTA allows, up to the warp's stage
// count.  Cached per shape.
template <int TB, int CWL, bool S, bool O, int NW, bool B, bool GR = false, int BITS = 4>
cudaError_t plan_for(const GemmProblem& p, Plan* out) {
  using GE = Geo<TB, CWL, NW, BITS>;
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, Plan> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int x_rows = p.M < 8 * TB ? p.M : 8 * TB;
  const int C = p.N / GE::CPW;
  const int nt = (C + GE::CW_W - 1) / GE::CW_W;
  // grouped: the 8-row tiles that will hold rows, estimated (the offsets live on the device):
  // R rows over E experts fill about max(R / 8, min(R, E)) tiles; the grid itself covers the
  // upper bound R / 8 + E and the empty tiles exit at once
  const long long mz = GR ? std::min<long long>((p.M + 7) / 8 + p.E,
                                                std::max<long long>((p.M + 7) / 8, std::min(p.M, p.E)))
                          : (p.M + 8 * TB - 1) / (8 * TB);
  const auto key = std::make_tuple(dev, p.K, nt * (int)mz, x_rows);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  DevLimits dl;
  e = dev_limits(&dl);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    auto kern = decode_tma_kernel<TB, CWL, S, O, NW, B, GR, BITS>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dl.smem_optin);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long tiles = (long long)nt * mz;
  const int TS = p.K / kRS;
  const int x_pitch = (x_rows == 1 && !AWQ_DECODE_WIDE_X) ? 128 : 1024 * TB;
  const int red_slots = (GE::RED_BYTES + NW * (x_pitch + GE::W_BYTES) - 1) / (NW * (x_pitch + GE::W_BYTES));
  Plan best;
  long long best_grid = -1;
  for (int cs = 1; cs <= kMaxCluster; ++cs) {
    if (cs > 1 && cs * NW > TS) break;
    // Power-of-two clusters only: they still pack into SMs left partly free by the
    // previous launch (programmatic dependent launch overlap); 3-, 5-, 6-CTA clusters
    // were measured to split into a second wave there.
    if ((cs & (cs - 1)) != 0) continue;
    // one-token variant, 4 warps: kOneGroups stash entries per warp whatever the warp's
    // group span (sizing the stash to the span gave one shape a deeper ring, which measured
    // slower); 8 warps: as many entries as the warp's groups.
    const int groups = !O ? 0
                       : NW == 4 ? kOneGroups
                                 : std::min(kOneGroups, max_warp_groups(TS, cs * NW, p.G / kRS));
    if (layout<TB, CWL, O, NW, BITS>(cs, 1, x_rows, groups).smem - layout<TB, CWL, O, NW, BITS>(cs, 1, x_rows, groups).recv_off - 1024 > kRecvCap) break;
    const long long grid = tiles * cs;
    long long per_sm = (grid + dl.sms - 1) / dl.sms;
    if (per_sm < 1) per_sm = 1;
    if (per_sm > kMaxCtasPerSm && cs > 1) continue;
    const int budget = static_cast<int>(dl.smem_per_sm / per_sm) - dl.reserved - 256;
    const int spw = (TS + cs * NW - 1) / (cs * NW);  // stages of the busiest warp
    const int max_slots = NW == 8 ? AWQ_DECODE_WIDE_SLOTS : kMaxSlots;
    int slots = spw < max_slots ? spw : max_slots;
    while (slots > 1 && layout<TB, CWL, O, NW, BITS>(cs, slots, x_rows, groups).smem > budget) --slots;
    if (slots < red_slots) slots = red_slots;
    Plan pl = layout<TB, CWL, O, NW, BITS>(cs, slots, x_rows, groups);
    if (pl.smem > dl.smem_optin) continue;
    // single wave with slack, checked against the occupancy API at this size
    bool fits = false;
    while (true) {
      long long cap = (long long)max_clusters<TB, CWL, S, O, NW, B, GR, BITS>(cs, pl.smem) * cs;
      if (cap > (long long)kMaxCtasPerSm * dl.sms) cap = (long long)kMaxCtasPerSm * dl.sms;
      if (grid * 100 <= cap * kWaveFillPct) { fits = true; break; }
      if (pl.slots <= red_slots || pl.slots <= 1) break;
      pl = layout<TB, CWL, O, NW, BITS>(cs, pl.slots - 1, x_rows, groups);
    }
    if (!fits && cs > 1) continue;
    const long long score = fits ? grid : 0;
    if (score > best_grid) {
      best_grid = score;
      best = pl;
    }
  }
  if (best.cs == 0) return cudaErrorInvalidConfiguration;
  cache[key] = best;
  *out = best;
  return cudaSuccess;
}

template <int TB, int CWL, bool S, bool O, int NW, bool B, bool GR = false, int BITS = 4>
cudaError_t launch_v(const GemmProblem& p) {
  using GE = Geo<TB, CWL, NW, BITS>;
  Plan pl;
  cudaError_t e = plan_for<TB, CWL, S, O, NW, B, GR, BITS>(p, &pl);
  if (e != cudaSuccess) return e;
  const int x_rows = p.M < 8 * TB ? p.M : 8 * TB;

  TmaDecodeParams dp;
  const char* why = nullptr;
  const int C = p.N / GE::CPW;
  const int ngrp = p.K / p.G;
  const CUtensorMapSwizzle wsw = CWL == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  const CUtensorMapDataType et = B ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  bool maps_ok = make_tmap_2d(&dp.tm_x, et, 2, p.x, p.K, p.M, kRS, x_rows,
                              (x_rows == 1 && !AWQ_DECODE_WIDE_X) ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, &why);
  if (GR) {  // stacked experts: [E][K][C], [E][K/G][C], [E][K/G][N]
    maps_ok = maps_ok &&
              make_tmap_3d(&dp.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.qw, C, p.K, p.E, GE::CW_W, kRS, wsw, &why) &&
              make_tmap_3d(&dp.tm_z, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.qz, C, ngrp, p.E, GE::CW_W, 1,
                           CU_TENSOR_MAP_SWIZZLE_NONE, &why) &&
              make_tmap_3d(&dp.tm_s, et, 2, p.sc, p.N, ngrp, p.E, GE::NCOL, 1, CU_TENSOR_MAP_SWIZZLE_NONE, &why);
  } else {
    maps_ok = maps_ok &&
              make_tmap_2d(&dp.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.qw, C, p.K, GE::CW_W, kRS, wsw, &why) &&
              make_tmap_2d(&dp.tm_z, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.qz, C, ngrp, GE::CW_W, 1,
                           CU_TENSOR_MAP_SWIZZLE_NONE, &why) &&
              make_tmap_2d(&dp.tm_s, et, 2, p.sc, p.N, ngrp, GE::NCOL, 1, CU_TENSOR_MAP_SWIZZLE_NONE, &why);
  }
  if (!maps_ok)
    return cudaErrorInvalidValue;
  dp.bias = p.bias;
  dp.y = p.y;
  e = status_word_ptr(&dp.status);
  if (e != cudaSuccess) return e;
  dp.M = p.M; dp.K = p.K; dp.N = p.N; dp.C = C; dp.G = p.G;
  dp.x_rows = x_rows;
  dp.slots = pl.slots;
  dp.meta_n = pl.meta_n;
  dp.x_pitch = pl.x_pitch;
  dp.w_off = pl.w_off; dp.m_off = pl.m_off; dp.zl_off = pl.zl_off;
  dp.bias_off = pl.bias_off; dp.bar_off = pl.bar_off; dp.recv_off = pl.recv_off;
  dp.owners = pl.owners; dp.slice = pl.slice;
  dp.offsets = p.offsets;
  dp.E = p.E;
  dp.early = (p.static_weights && !GR) ? 1 : 0;

  const int nt = (C + GE::CW_W - 1) / GE::CW_W;
  const int mz = GR ? (p.M + 7) / 8 + p.E : (p.M + 8 * TB - 1) / (8 * TB);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nt * pl.cs), static_cast<unsigned>(mz), 1);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(pl.smem);
  cfg.stream = p.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_tma_kernel<TB, CWL, S, O, NW, B, GR, BITS>, dp);
}

}  // namespace

bool decode_tma_supported(const GemmProblem& p, const char** why) {
  static const char* dummy;
  if (!why) why = &dummy;
  if (p.bits != 4 && p.bits != 8) { *why = "4- or 8-bit codes only"; return false; }
  if (p.bits == 8 && (p.bf16 || p.offsets != nullptr)) { *why = "8-bit codes: fp16 plain launches only"; return false; }
  if (p.K % kRS != 0) { *why = "TMA decode needs K % 64 == 0"; return false; }
  if (p.G % kRS != 0) { *why = "TMA decode needs group_size % 64 == 0"; return false; }
  // packed rows a multiple of 16 bytes (tensor-map strides): N % 32 (4 bits), N % 16 (8)
  if (p.N % (p.bits == 8 ? 16 : 32) != 0) { *why = "TMA decode needs N % 32 == 0 (N % 16 for 8 bits)"; return false; }
  if (!aligned(p.x, 16) || !aligned(p.qw, 16) || !aligned(p.qz, 16) || !aligned(p.sc, 16)) {
    *why = "TMA decode needs 16-byte aligned x, qweight, qzeros, scales";
    return false;
  }
  if ((p.M + 31) / 32 > 65535) { *why = "M too large for the decode grid"; return false; }
  if ((long long)(p.K / kRS) * kMaxCluster * 8 >= (1LL << 31)) { *why = "K too large for the decode kernel"; return false; }
  return true;
}

template <bool B, int BITS = 4>
cudaError_t launch_decode_tma_t(const GemmProblem& p) {
  const Variant v = pick(p);
  if (v.TB == 1) {
    if (p.M == 1) {
      // One token: at most kOneGroups groups per warp.  8-warp CTAs where 4-warp ones
      // would leave a warp kWideStages or more stages (long K: more warps share the work).
      const int TS = p.K / kRS, spg = p.G / kRS;
      Plan p4;
      cudaError_t e = plan_for<1, 2, true, true, 4, B, false, BITS>(p, &p4);
      if (e != cudaSuccess) return e;
      if ((TS + 4 * p4.cs - 1) / (4 * p4.cs) >= kWideStages) {
        Plan p8;
        e = plan_for<1, 2, true, true, 8, B, false, BITS>(p, &p8);
        if (e != cudaSuccess) return e;
        if (max_warp_groups(TS, 8 * p8.cs, spg) <= kOneGroups) return launch_v<1, 2, true, true, 8, B, false, BITS>(p);
      }
      if (max_warp_groups(TS, 4 * p4.cs, spg) <= kOneGroups) return launch_v<1, 2, true, true, 4, B, false, BITS>(p);
    }
    return launch_v<1, 2, true, false, kNW, B, false, BITS>(p);
  }
  if (v.TB == 2) return launch_v<2, 1, true, false, kNW, B, false, BITS>(p);
  return launch_v<4, 1, false, false, kNW, B, false, BITS>(p);
}

bool decode_grouped_supported(const GemmProblem& p, const char** why) {
  static const char* dummy;
  if (!why) why = &dummy;
  if (p.bf16) { *why = "grouped launches take fp16"; return false; }
  if (p.bits != 4) { *why = "grouped launches take 4-bit codes"; return false; }
  if (p.E <= 0 || p.offsets == nullptr) { *why = "grouped launch without experts"; return false; }
  return decode_tma_supported(p, why);
}

cudaError_t launch_decode_grouped(const GemmProblem& p) {
  return launch_v<1, 2, true, false, kNW, false, true>(p);
}

cudaError_t launch_decode_tma(const GemmProblem& p) {
  if (p.bits == 8) return launch_decode_tma_t<false, 8>(p);
  return p.bf16 ? launch_decode_tma_t<true>(p) : launch_decode_tma_t<false>(p);
}

}  // namespace awq
