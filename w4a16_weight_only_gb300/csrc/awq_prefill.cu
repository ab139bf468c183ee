// Prefill path of awq_gemm (large M): persistent tcgen05 / TMEM tensor-core kernel.
//
//   y[m][n] = sum_k x[m][k] * (code[k][n] - zero[k/G][n]) * scale[k/G][n]  (+ bias[n])
//
// (tensref.org/formats/awq, "Reader"; GPTQModel wiki "AWQ", "Native GEMM": fused
// dequant-GEMM with fp32 accumulation.)
//
// Tiling (operands swapped so the dequantized side is the small one): one UMMA tile is
// 128 output columns (the MMA's M side, A operand = dequantized W^T) by 256 activation
// rows (the MMA's N side, B operand = x), K = 64 per pipeline stage, four
// tcgen05.mma.kind::f16 (K = 16) per stage, fp32 accumulators in TMEM.  Each dequantized
// 128 x 64 weight tile therefore feeds 256 activation rows.
//
// Warp roles (448 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: activation tile (256 x 64 fp16, 128B swizzle), packed weight
//               tile (64 rows x 16 words), the stage's zero and scale rows -> 4-deep ring
//   warp 1      TMEM allocation (512 columns = two 128 x 256 fp32 accumulators) and the
//               single MMA-issuing thread
//   warps 2-9   dequantize the packed tile into the MN-major, 128B-swizzled fp16 A tile
//               (one packed word = one 16-byte chunk of 8 adjacent columns, no transpose):
//               w = (c - z) * s exactly (fp16 exponent trick, HSUB2, HMUL2) -> 4-deep ring
//   warps 10-13 epilogue: tcgen05.ld (32 lanes x 32 columns), + bias, fp16, store; the
//               second accumulator lets the next tile's MMAs run meanwhile
// Every wait is an mbarrier try-wait bounded in wall time; on give-up the kernel sets the
// device status word, all roles leave their loops, in-flight copies and MMAs are drained
// (bounded) and TMEM is freed before exit.
//
// Pair variant (kPair, compile-time option): a cluster of two CTAs shares a 256 x 256
// tile through tcgen05.mma.cta_group::2 (M = 256: each CTA dequantizes its own 128
// columns; N = 256: each CTA loads its own 128 activation rows, no TMA multicast); the
// even CTA issues the MMAs and commits to both CTAs' barriers, the odd CTA's dequant warps
// signal readiness with a counted st.async into the even CTA's barrier.
//
// 8-bit variant (kBits = 8, fp16, one CTA per tile): the same 128-column tile is 32 packed
// words a row (byte i of word c = column 4c + i), so the stage's packed tile is 64 rows x
// 32 words and its zero row 32 words; a dequant thread reads four words of each of its
// rows, and one byte permute per column pair puts two codes under the 0x6400 exponent
// (1024 + c, exact) before the same HSUB2 / HMUL2 and the same A-tile chunks.
#include <algorithm>
#include <mutex>

#include "awq_internal.cuh"
#include "awq_ptx.cuh"

namespace awq {

__device__ unsigned int g_status_word = 0u;

namespace {

using namespace ptx;

constexpr int kBN = 128;   // output columns per tile (UMMA M)
#ifndef AWQ_PREFILL_BT
#define AWQ_PREFILL_BT 256
#endif
#ifndef AWQ_PREFILL_ST
#define AWQ_PREFILL_ST 4
#endif
#ifndef AWQ_PREFILL_SA
#define AWQ_PREFILL_SA 4
#endif
constexpr int kBT = AWQ_PREFILL_BT;   // activation rows per tile (UMMA N)
constexpr int kBK = 64;    // K per stage
constexpr int kST = AWQ_PREFILL_ST;  // TMA ring depth
constexpr int kSA = AWQ_PREFILL_SA;  // dequantized-A ring depth
#ifndef AWQ_PREFILL_SMALL_ST
#define AWQ_PREFILL_SMALL_ST 8
#endif
constexpr int kSTsmall = AWQ_PREFILL_SMALL_ST;  // TMA ring depth of the narrow token tiles
#ifndef AWQ_PREFILL_SMALL_SA
#define AWQ_PREFILL_SMALL_SA 8
#endif
constexpr int kSAsmall = AWQ_PREFILL_SMALL_SA;  // dequantized-A ring depth of the narrow tiles
constexpr int kDQ = 8;                        // dequant warps
constexpr int kThreads = (2 + kDQ + 4) * 32;  // producer, MMA, dequant, epilogue
#ifndef AWQ_PREFILL_ACC_BUFS
#define AWQ_PREFILL_ACC_BUFS 2
#endif
constexpr int kAccBufs = AWQ_PREFILL_ACC_BUFS;      // TMEM accumulators (tile overlap)
// TMEM columns allocated (a power of two): the accumulators take kAccBufs * kBT of them.
constexpr int kTmemCols = kAccBufs * kBT <= 256 ? 256 : 512;
static_assert(kAccBufs * kBT <= 512 && kBT % 32 == 0 && kBT <= 256, "accumulators");
constexpr uint32_t kMagic = 0x64006400u;
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;
constexpr unsigned int kStatusPrefillTimeout = 0x2u;

// Shared memory layout (offsets from a 1024-aligned base).  Pair mode loads half the
// activation rows per CTA, and its stages wait on a cross-SM round trip (remote barrier
// arrivals, multicast commits), so it spends the room on deeper rings.
#ifndef AWQ_PREFILL_PAIR_ST
#define AWQ_PREFILL_PAIR_ST 7
#endif
#ifndef AWQ_PREFILL_PAIR_SA
#define AWQ_PREFILL_PAIR_SA 5
#endif
constexpr int A_BYTES = kBN * kBK * 2;       // 16 KB
// Narrow token tiles (BT < 256) keep one dequantized-A slot fewer, so that two CTAs fit on
// an SM; split-K launches (SPLIT > 1) add the receive area of the cluster's partial sums.
template <bool kPair, int kBits = 4, int BT = kBT, int SPLIT = 1>
struct Layout {
  static constexpr int W_BYTES = kBK * (kBN * kBits / 32) * 4;  // packed tile: 4 or 8 KB
  static constexpr int X_BYTES = (kPair ? BT / 2 : BT) * kBK * 2;  // 4 .. 32 KB
  // narrow tiles: the receive area first, then as deep a dequantized-A ring as fits beside
  // a 4-stage TMA ring (at most kSAsmall), then as deep a TMA ring as fits (at most kSTsmall)
  static constexpr int kBudget = 227 * 1024 - 2048 - (SPLIT - 1) * kBN * (BT + 4) * 4;
  static constexpr int SA_FIT = (kBudget - 4 * (X_BYTES + W_BYTES + 384)) / (kBN * kBK * 2);
  static constexpr int SA = kPair ? AWQ_PREFILL_PAIR_SA
                                  : (BT < kBT ? (SA_FIT < kSAsmall ? SA_FIT : kSAsmall) : kSA);  // dequantized-A ring depth
  static_assert(SA >= 2, "dequantized-A ring");
  static constexpr int ST_FIT = (kBudget - SA * kBN * kBK * 2) / (X_BYTES + W_BYTES + 384);
  static constexpr int ST = kPair ? AWQ_PREFILL_PAIR_ST
                                  : (BT < kBT ? (ST_FIT < kSTsmall ? ST_FIT : kSTsmall) : kST);  // TMA ring depth
  static_assert(ST >= 2, "TMA ring");
  static constexpr int X_OFF = 0;
  static constexpr int A_OFF = X_OFF + ST * X_BYTES;
  static constexpr int W_OFF = A_OFF + SA * A_BYTES;
  static constexpr int Z_OFF = W_OFF + ST * W_BYTES;  // 128 B per stage (16 or 32 words)
  static constexpr int S_OFF = Z_OFF + ST * 128;      // 256 B per stage
  static constexpr int BAR_OFF = S_OFF + ST * 256;
  // barriers: full_t[ST], empty_t[ST], full_a[SA], empty_a[SA], tfull[2], tempty[2], drain, recv
  static constexpr int NBARS = 2 * ST + 2 * SA + 4 + 2;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base (u32), abort flag (u32)
  static constexpr int SIG_OFF = MISC_OFF + 16;         // pair: targets of the peer's signals
  // split-K: rank 0 receives ranks 1 .. SPLIT-1's fp32 partials, [rank - 1][column][token],
  // rows padded by 4 floats (odd multiples of 16 bytes: conflict-free 128-bit reads)
  static constexpr int RECV_PITCH = BT + 4;
  static constexpr int RECV_OFF = ((SIG_OFF + 64 + 15) / 16) * 16;
  static constexpr int RECV_BYTES = (SPLIT - 1) * kBN * RECV_PITCH * 4;
  static constexpr size_t SMEM = 1024 + RECV_OFF + RECV_BYTES;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  // TMEM: whatever the register count, shared memory alone keeps at most two CTAs of this
  // kernel on an SM, and each allocates at most 256 columns below 256-row tiles (512 at
  // 256 rows, where one CTA fills the SM): tcgen05.alloc never waits for another CTA.
  static_assert(BT == kBT || SMEM > 228 * 1024 / 3, "at most two narrow-tile CTAs per SM");
};

// Bytes one CTA's stage copies land: its activation rows, packed tile, zero and scale rows.
template <bool kPair, int kBits = 4, int BT = kBT>
__host__ __device__ constexpr uint32_t stage_tx() {
  return (kPair ? BT / 2 : BT) * kBK * 2 + Layout<kPair, kBits>::W_BYTES + (kBN * kBits / 32) * 4 + 128 * 2;
}

struct __align__(64) PrefillParams {
  CUtensorMap tm_x;  // x [M][K] f16, box {64, 256}, 128B swizzle
  CUtensorMap tm_w;  // qweight [K][C] u32, box {16, 64} (8 bits: {32, 64})
  CUtensorMap tm_z;  // qzeros [K/G][C] u32, box {16, 1} (8 bits: {32, 1})
  CUtensorMap tm_s;  // scales [K/G][N] f16, box {128, 1}
  const __half* bias;
  __half* y;
  unsigned int* status;
  int M, K, N, C, G;
  int tiles_t, tiles;  // activation-row tiles, total tiles
};

// tcgen05 shared-memory matrix descriptor with 128-byte swizzle.
//   K-major operand (B = activations): rows of 128 B (64 fp16 along K), 8-row groups
//     1024 B apart (stride byte offset); the leading byte offset is unused.
//   MN-major operand (A = dequantized weights): 1024-byte atoms of 8 K-rows x 64 columns;
//     leading byte offset = distance between atoms along MN, stride byte offset =
//     distance between atoms along K.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);       // start address / 16
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;   // leading byte offset / 16
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;   // stride byte offset / 16
  d |= static_cast<uint64_t>(1u) << 46;                     // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                     // layout: 128-byte swizzle
  return d;
}

// A tile (MN-major): atom (column half ma, K group kg) at (ma * 8 + kg) * 1024.
constexpr uint32_t kA_LBO = 8 * 1024;  // between the two 64-column halves
constexpr uint32_t kA_SBO = 1024;      // between 8-row K groups

// Instruction descriptor, kind::f16: fp32 accumulate, fp16 A and B, A MN-major, B K-major,
// N = 256, M = 128.
template <int BT>
__host__ __device__ constexpr uint32_t idesc_n() {
  return (1u << 4) | (0u << 7) | (0u << 10) | (1u << 15) | (0u << 16) |
         (static_cast<uint32_t>(BT >> 3) << 17) | (static_cast<uint32_t>(kBN >> 4) << 24);
}
constexpr uint32_t kIdesc = idesc_n<kBT>();

// Pair mode (cta_group::2): the MMA spans the two CTAs of a cluster, M = 256 (128 A rows
// from each CTA's shared memory), N = 256 (128 B rows from each); every CTA's TMEM holds
// the accumulator rows of its own A half.
constexpr uint32_t kIdescPair = (kIdesc & ~(0x1Fu << 24)) | (static_cast<uint32_t>((2 * kBN) >> 4) << 24);

// kind::f16 with bf16 A and B: formats 1 in the A and B format fields (bits 7-9, 10-12).
constexpr uint32_t kIdescBF16 = (1u << 7) | (1u << 10);

template <bool kPair, bool kBF = false, int BT = kBT>
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t accumulate) {
  if constexpr (kPair) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kIdescPair | (kBF ? kIdescBF16 : 0u)), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc_n<BT>() | (kBF ? kIdescBF16 : 0u)), "r"(accumulate)
        : "memory");
  }
}

// Arrive on `bar` once the MMAs issued so far complete: in pair mode on the barrier at the
// same offset in both CTAs of the cluster.
template <bool kPair>
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  if constexpr (kPair) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(static_cast<unsigned short>(0x3))
        : "memory");
  } else {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
  }
}

// Bounded wait on phase `parity` of a local mbarrier with cluster-scope acquire (the
// phase was completed by arrivals released from the other CTA of the pair).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          unsigned int* status, unsigned int code,
                                                          uint64_t limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(status, code);
      return false;
    }
  }
  return true;
}

// Arrive (release, cluster scope) on the mbarrier at `local`'s offset in CTA `rank`.
__device__ __forceinline__ void mbar_arrive_rank(uint64_t* local, uint32_t rank) {
  uint32_t ra;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}

// Cluster-window address of `local`'s offset in CTA `rank`, and an asynchronous 16-byte
// store to such an address whose bytes complete on the (cluster-window) mbarrier `rbar`.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t ra;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  return ra;
}
__device__ __forceinline__ void st_async_v4_at(uint32_t raddr, uint32_t rbar, uint32_t a, uint32_t b,
                                               uint32_t c, uint32_t d) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(raddr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(rbar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ uint32_t lds32p(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64p(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128p(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

// kBF: bf16 activations, scales, bias and output; the dequantized A tile is bf16
// ((c - z) * s rounded once), the MMA kind::f16 with bf16 operands.
// BT: activation rows per tile (UMMA N = BT).  SPLIT > 1: a cluster of SPLIT CTAs shares
// one tile, CTA r taking K stages [r KB / SPLIT, (r + 1) KB / SPLIT); ranks 1 .. SPLIT-1
// push their fp32 accumulators into rank 0's receive area (st.async, counted on rank 0's
// recv barrier), and rank 0 adds them in rank order, adds the bias and stores y.  Split
// launches give every cluster exactly one tile.
template <bool kPair, bool kBF = false, int kBits = 4, int BT = kBT, int SPLIT = 1>
__global__ void __launch_bounds__(kThreads, BT < kBT ? 2 : 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  static_assert(kBits == 4 || (kBits == 8 && !kBF && !kPair), "8-bit codes: fp16, one CTA per tile");
  static_assert(SPLIT == 1 || !kPair, "split-K launches use one CTA per tile share");
  static_assert(BT % 32 == 0 && BT >= 32 && BT <= 256 && (kPair ? BT == kBT : true), "token tile");
  // TMEM columns allocated (a power of two, at least 32): kAccBufs accumulators of BT
  constexpr int kCols = kAccBufs * BT <= 32 ? 32 : kAccBufs * BT <= 64 ? 64 : kAccBufs * BT <= 128 ? 128
                                            : kAccBufs * BT <= 256 ? 256 : 512;
  constexpr uint32_t kMag = kBF ? 0x43004300u : kMagic;  // 128 (bf16) / 1024 (fp16), both halves
  constexpr int CPW = 32 / kBits;                        // columns per packed word
  using L = Layout<kPair, kBits, BT, SPLIT>;
  constexpr int W_BYTES = L::W_BYTES;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* full_t = bars;
  uint64_t* empty_t = bars + L::ST;
  uint64_t* full_a = bars + 2 * L::ST;
  uint64_t* empty_a = bars + 2 * L::ST + L::SA;
  uint64_t* tfull = bars + 2 * L::ST + 2 * L::SA;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* recv_bar = drain + 1;  // split-K: rank 0's partials received
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::MISC_OFF);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = p.K / kBK;  // stages per tile
  // Pair mode: the cluster's two CTAs share each tile; rank 0 (the leader) issues the MMAs.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0u;
  // Split-K: this CTA's share of the tile's K stages.
  const uint32_t krank = SPLIT > 1 ? cluster_ctarank() : 0u;
  const int kb0 = static_cast<int>(static_cast<long long>(KB) * krank / SPLIT);
  const int kb1 = static_cast<int>(static_cast<long long>(KB) * (krank + 1) / SPLIT);
  const int tile0 = kPair ? static_cast<int>(blockIdx.x >> 1)
                          : static_cast<int>(blockIdx.x) / SPLIT;
  const int tstep = kPair ? static_cast<int>(gridDim.x >> 1)
                          : static_cast<int>(gridDim.x) / SPLIT;
  constexpr int kTileWords = (kPair ? 2 * kBN : kBN) / CPW;  // packed words per tile
  constexpr int kXR = kPair ? BT / 2 : BT;                   // activation rows this CTA loads
#ifdef AWQ_PREFILL_DEBUG_DECL
  AWQ_PREFILL_DEBUG_DECL
#endif

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::ST; ++s) {
      mbar_init(&full_t[s], 1);
      mbar_init(&empty_t[s], kDQ + 1);  // dequant warps + one MMA commit
    }
    for (int s = 0; s < L::SA; ++s) {
      // own dequant warps (pair leader: one of them also expects the peer's signal bytes)
      mbar_init(&full_a[s], kDQ);
      mbar_init(&empty_a[s], 1);                     // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);                       // MMA commit
      mbar_init(&tempty[b], kPair ? 8 : 4);          // epilogue warps (of both CTAs)
    }
    mbar_init(drain, 1);
    mbar_init(recv_bar, 1);
    if (SPLIT > 1 && krank == 0u)  // the partials of ranks 1 .. SPLIT-1, one phase
      mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((SPLIT - 1) * kBN * BT * 4));
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {  // one warp of each CTA of the pair, collectively
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(const_cast<uint32_t*>(tmem_slot))), "n"(kCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(const_cast<uint32_t*>(tmem_slot))), "n"(kCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  __syncthreads();
  if constexpr (kPair || SPLIT > 1) cluster_sync_all();  // the cluster's barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Bounded waits; a phase already complete returns at once (the abort flag, set by a role
  // that gave up, is read only before a wait that would block).
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, p.status, kStatusPrefillTimeout, kWaitLimitNs)) return true;
    *abort_flag = 1u;
    return false;
  };
  auto wait_cl = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait_cluster_bounded(bar, parity, p.status, kStatusPrefillTimeout, kWaitLimitNs)) return true;
    *abort_flag = 1u;
    return false;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_x);
      prefetch_tmap(&p.tm_w);
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < p.tiles; tile += tstep) {
        const int m0 = (tile % p.tiles_t) * BT + static_cast<int>(rank) * kXR;
        const int cw0 = (tile / p.tiles_t) * kTileWords + static_cast<int>(rank) * (kBN / CPW);
        for (int kb = kb0; kb < kb1; ++kb) {
#ifdef AWQ_PREFILL_DEBUG_ROLE
          AWQ_PREFILL_DEBUG_ROLE(0, 0);
#endif
          if (!wait(&empty_t[s], ph ^ 1u)) { ok = false; break; }
#ifdef AWQ_PREFILL_DEBUG_ROLE
          AWQ_PREFILL_DEBUG_ROLE(0, 1);
#endif
          const int k0 = kb * kBK;
          const int grp = k0 / p.G;
          mbar_arrive_expect_tx(&full_t[s], stage_tx<kPair, kBits, BT>());
          tma_load_2d(smem + L::X_OFF + s * L::X_BYTES, &p.tm_x, &full_t[s], k0, m0);
          tma_load_2d(smem + L::W_OFF + s * W_BYTES, &p.tm_w, &full_t[s], cw0, k0);
          tma_load_2d(smem + L::Z_OFF + s * 128, &p.tm_z, &full_t[s], cw0, grp);
          tma_load_2d(smem + L::S_OFF + s * 256, &p.tm_s, &full_t[s], CPW * cw0, grp);
          ++issued;
          if (++s == L::ST) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        // drain: every issued stage's copies must land before the CTA can exit
        for (int i = 0; i < L::ST && i < issued; ++i) {
          if (--s < 0) { s = L::ST - 1; ph ^= 1u; }
          mbar_wait_bounded(&full_t[s], ph, p.status, kStatusPrefillTimeout, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && kPair && !leader) {
      // the leader's MMAs write this CTA's TMEM and read its shared memory: wait for the
      // last of them before the CTA may free TMEM
      if (tile0 < p.tiles) mbar_wait_bounded(drain, 0u, p.status, kStatusPrefillTimeout, kWaitLimitNs);
    } else if (lane == 0) {
#ifdef AWQ_PREFILL_DEBUG_WAIT
      unsigned long long dbg_t0 = 0;
#endif
      int s = 0, sa = 0;
      uint32_t ph = 0, pha = 0;
      int li = 0;
      bool ok = true;
      bool any = false;
      for (int tile = tile0; ok && tile < p.tiles; tile += tstep, ++li) {
        const int b = li % kAccBufs;
#ifdef AWQ_PREFILL_DEBUG_WAIT
        AWQ_PREFILL_DEBUG_WAIT(0);
#endif
        if (!wait(&tempty[b], static_cast<uint32_t>(((li / kAccBufs) & 1) ^ 1))) { ok = false; break; }
#ifdef AWQ_PREFILL_DEBUG_WAIT
        AWQ_PREFILL_DEBUG_WAIT(1);
#endif
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(b * BT);
        // full_a completes only after every dequant warp has seen full_t[s], so the
        // activation tile of stage s is in place as well.  One wait per stage: waiting once
        // per stage pair (every dequant warp arrives in stage order) was measured slower
        // here, the shared-memory A ring being only four stages deep.
        constexpr int kGroup = 1;
        for (int kb = kb0; kb < kb1; kb += kGroup) {
          const int ng = kb1 - kb < kGroup ? kb1 - kb : kGroup;
          const int sl = sa + ng - 1 < L::SA ? sa + ng - 1 : sa + ng - 1 - L::SA;
          const uint32_t phl = sa + ng - 1 < L::SA ? pha : pha ^ 1u;
          if (!(kPair ? wait_cl(&full_a[sl], phl) : wait(&full_a[sl], phl))) { ok = false; break; }
          tc_fence_after();
          for (int i = 0; i < ng; ++i) {
            const uint64_t adesc = sw128_desc(sbase + L::A_OFF + sa * A_BYTES, kA_LBO, kA_SBO);
            const uint64_t bdesc = sw128_desc(sbase + L::X_OFF + s * L::X_BYTES, 16u, 1024u);
#pragma unroll
            for (int ks = 0; ks < kBK / 16; ++ks)  // K += 16: A two atoms (2048 B), B 32 B
              mma_f16<kPair, kBF, BT>(d, adesc + (2u * kA_SBO >> 4) * ks, bdesc + 2 * ks,
                                      (kb + i > kb0 || ks > 0) ? 1u : 0u);
            mma_commit<kPair>(&empty_t[s]);
            mma_commit<kPair>(&empty_a[sa]);
            if (++s == L::ST) { s = 0; ph ^= 1u; }
            if (++sa == L::SA) { sa = 0; pha ^= 1u; }
          }
          any = true;
        }
        if (!ok) break;
        mma_commit<kPair>(&tfull[b]);
      }
      if (any) {
        // all MMAs issued by this thread complete before TMEM is released
        mma_commit<kPair>(drain);
        mbar_wait_bounded(drain, 0u, p.status, kStatusPrefillTimeout, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp < 2 + kDQ) {
    // ---------------------------------------------------------------- dequant
    // thread -> rows rp, rp + 32 x column-words 2cg, 2cg+1 of the stage.  Each packed word
    // becomes one 16-byte chunk (its 8 columns in order) of the MN-major A tile.  A warp
    // reads four consecutive 64-byte rows (each half-warp two whole rows: no bank
    // conflict) and, per store, lanes cg >= 4 take their odd word first so the eight
    // 16-byte chunks of one store phase land in eight different bank groups.
    const int dq = threadIdx.x - 64;
    const int rp = dq >> 3;
    const int cg = dq & 7;
    const int csel = (cg >> 2) & 1;
    int s = 0, sa = 0;
    uint32_t ph = 0, pha = 0;
    bool ok = true;
    for (int tile = tile0; ok && tile < p.tiles; tile += tstep) {
      for (int kb = kb0; kb < kb1; ++kb) {
#ifdef AWQ_PREFILL_DEBUG_ROLE
        AWQ_PREFILL_DEBUG_ROLE(1, 0);
#endif
        if (!wait(&full_t[s], ph)) { ok = false; break; }
#ifdef AWQ_PREFILL_DEBUG_ROLE
        AWQ_PREFILL_DEBUG_ROLE(1, 1);
#endif
        if (!wait(&empty_a[sa], pha ^ 1u)) { ok = false; break; }
#ifdef AWQ_PREFILL_DEBUG_ROLE
        AWQ_PREFILL_DEBUG_ROLE(1, 2);
#endif
        const uint32_t wb = sbase + L::W_OFF + s * W_BYTES;
        const uint32_t ab = sbase + L::A_OFF + sa * A_BYTES;
        if constexpr (kBits == 8) {
          // words 4cg .. 4cg+3 of rows rp, rp + 32 (128-byte rows: a quarter-warp reads one
          // whole row), the matching zero words; chunk cw = 2cg + cc is words 2cc, 2cc + 1
          const uint4 r0 = lds128p(wb + rp * 128 + cg * 16);
          const uint4 r1 = lds128p(wb + (rp + 32) * 128 + cg * 16);
          const uint4 z4 = lds128p(sbase + L::Z_OFF + s * 128 + cg * 16);
          const uint32_t w8[2][4] = {{r0.x, r0.y, r0.z, r0.w}, {r1.x, r1.y, r1.z, r1.w}};
          const uint32_t zw8[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int cc = c ^ csel;
            const int cw = 2 * cg + cc;
            const uint4 s4 = lds128p(sbase + L::S_OFF + s * 256 + cw * 16);
            const uint32_t sp[4] = {s4.x, s4.y, s4.z, s4.w};  // (s[2j], s[2j+1])
            // column pair j = bytes (2 (j % 2), +1) of word 2cc + j / 2, as 1024 + code
            const uint32_t za = cc ? zw8[2] : zw8[0], zb = cc ? zw8[3] : zw8[1];
            uint32_t zp[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) zp[j] = prmt(j < 2 ? za : zb, kMag, (j & 1) ? 0x7352u : 0x7150u);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const uint32_t wa = cc ? w8[e][2] : w8[e][0], wb2 = cc ? w8[e][3] : w8[e][1];
              uint32_t v[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t h = prmt(j < 2 ? wa : wb2, kMag, (j & 1) ? 0x7352u : 0x7150u);
                v[j] = hmul2(hsub2(h, zp[j]), sp[j]);
              }
              const int k = rp + 32 * e;
              const int off = ((cw >> 3) * 8 + (k >> 3)) * 1024 + (k & 7) * 128 +
                              (((cw & 7) ^ (k & 7)) << 4);
              sts128(ab + off, v[0], v[1], v[2], v[3]);
            }
          }
        } else {
        const uint2 r0 = lds64p(wb + rp * 64 + cg * 8);
        const uint2 r1 = lds64p(wb + (rp + 32) * 64 + cg * 8);
        const uint2 z2 = lds64p(sbase + L::Z_OFF + s * 128 + cg * 8);
        const uint32_t w[2][2] = {{r0.x, r0.y}, {r1.x, r1.y}};
        const uint32_t zw[2] = {z2.x, z2.y};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int cc = c ^ csel;
          const int cw = 2 * cg + cc;
          const uint4 s4 = lds128p(sbase + L::S_OFF + s * 256 + cw * 16);
          const uint32_t sp[4] = {s4.x, s4.y, s4.z, s4.w};  // (s[2j], s[2j+1])
          uint32_t zp[4];                                    // (1024+z[2j], 1024+z[2j+1])
          const uint32_t zc = cc ? zw[1] : zw[0];
          // fp16: odd pairs are read in bits 4-7 under the exponent of 64 (mantissa step 1/16):
          // 64 + c and 64 + z, exact as 1024 + c is; one shift serves pairs 2 and 3
          constexpr uint32_t kMag64 = 0x54005400u;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            zp[j] = (kBF || !(j & 1)) ? and_or(zc >> (4 * j), 0x000F000Fu, kMag)
                                      : and_or(zc >> (4 * j - 4), 0x00F000F0u, kMag64);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint32_t v[4];
            const uint32_t wc = cc ? w[e][1] : w[e][0];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t h = (kBF || !(j & 1)) ? and_or(wc >> (4 * j), 0x000F000Fu, kMag)
                                                   : and_or(wc >> (4 * j - 4), 0x00F000F0u, kMag64);
              v[j] = kBF ? hmul2_bf16(hsub2_bf16(h, zp[j]), sp[j]) : hmul2(hsub2(h, zp[j]), sp[j]);
            }
            const int k = rp + 32 * e;
            const int off = ((cw >> 3) * 8 + (k >> 3)) * 1024 + (k & 7) * 128 +
                            (((cw & 7) ^ (k & 7)) << 4);
            sts128(ab + off, v[0], v[1], v[2], v[3]);
          }
        }
        }  // kBits
        fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair) {
            if (leader) {
              // warp 2 also arms the bytes the peer's eight dequant warps will signal
              if (warp == 2) mbar_arrive_expect_tx(&full_a[sa], kDQ * 4u);
              else mbar_arrive(&full_a[sa]);
            } else {
              // A half in place (ordered before this async-proxy store by the fence above):
              // signal the leader with a 4-byte store counted on its full_a[sa]
              st_async_dsmem_f32(reinterpret_cast<float*>(smem + L::SIG_OFF + 4 * (warp - 2)),
                                 &full_a[sa], 0u, 0.f);
            }
          } else {
            mbar_arrive(&full_a[sa]);
          }
          mbar_arrive(&empty_t[s]);
        }
#ifdef AWQ_PREFILL_DEBUG_ROLE
        AWQ_PREFILL_DEBUG_ROLE(1, 3);
#endif
        if (++s == L::ST) { s = 0; ph ^= 1u; }
        if (++sa == L::SA) { sa = 0; pha ^= 1u; }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;           // TMEM lanes 32*quad .. +31
    const int nl = quad * 32 + lane;     // output column inside the tile
    int li = 0;
    for (int tile = tile0; tile < p.tiles; tile += tstep, ++li) {
      const int b = li % kAccBufs;
      const int m0 = (tile % p.tiles_t) * BT;
      const int n = (tile / p.tiles_t) * (CPW * kTileWords) + static_cast<int>(rank) * kBN + nl;
      const float bias = (p.bias != nullptr && n < p.N)
                             ? elem_to_float<kBF>(reinterpret_cast<const uint16_t*>(p.bias)[n])
                             : 0.f;
      if (!wait(&tfull[b], static_cast<uint32_t>((li / kAccBufs) & 1))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(b * BT);
      if constexpr (SPLIT > 1) {
        float* recv = reinterpret_cast<float*>(smem + L::RECV_OFF);
        if (krank != 0u) {
          // this share's partial sums of column nl, all BT tokens, into rank 0
          const uint32_t rbar = cluster_addr(recv_bar, 0u);
          const uint32_t rdst = cluster_addr(recv + (static_cast<int>(krank - 1) * kBN + nl) * L::RECV_PITCH, 0u);
#pragma unroll 1
          for (int c = 0; c < BT / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(taddr + c * 32, v);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              st_async_v4_at(rdst + static_cast<uint32_t>((c * 32 + j) * 4), rbar, v[j], v[j + 1], v[j + 2], v[j + 3]);
          }
        } else {
          if (!wait_cl(recv_bar, 0u)) break;
#pragma unroll 1
          for (int c = 0; c < BT / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(taddr + c * 32, v);
#pragma unroll
            for (int r = 1; r < SPLIT; ++r) {  // rank order, summed in place
              const float* src = recv + ((r - 1) * kBN + nl) * L::RECV_PITCH + c * 32;
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                const float4 q4 = *reinterpret_cast<const float4*>(src + j);
                v[j] = __float_as_uint(__uint_as_float(v[j]) + q4.x);
                v[j + 1] = __float_as_uint(__uint_as_float(v[j + 1]) + q4.y);
                v[j + 2] = __float_as_uint(__uint_as_float(v[j + 2]) + q4.z);
                v[j + 3] = __float_as_uint(__uint_as_float(v[j + 3]) + q4.w);
              }
            }
            const int t0 = m0 + c * 32;
            if (n < p.N) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (t0 + j < p.M)
                  reinterpret_cast<uint16_t*>(p.y)[(long long)(t0 + j) * p.N + n] =
                      float_to_elem<kBF>(__uint_as_float(v[j]) + bias);
              }
            }
          }
        }
      } else {
#pragma unroll 1
      for (int c = 0; c < BT / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(taddr + c * 32, v);
        const int t0 = m0 + c * 32;
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (t0 + j < p.M)
              reinterpret_cast<uint16_t*>(p.y)[(long long)(t0 + j) * p.N + n] =
                  float_to_elem<kBF>(__uint_as_float(v[j]) + bias);
          }
        }
      }
      }  // SPLIT
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair) mbar_arrive_rank(&tempty[b], 0u);  // the leader's barrier
        else mbar_arrive(&tempty[b]);
      }
    }
  }

  // Split-K: rank 0 leaves only once the other ranks' pushes have landed (bounded: after a
  // give-up elsewhere they may never come).
  if (SPLIT > 1 && krank == 0u && threadIdx.x == 0)
    (void)mbar_wait_cluster_bounded(recv_bar, 0u, p.status, kStatusPrefillTimeout, kWaitLimitNs);
  __syncthreads();
  // Pair mode: neither CTA leaves while the other may still arrive on its barriers; split
  // mode: nor while its pushes into rank 0 may be in flight.
  if constexpr (kPair || SPLIT > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "n"(kCols) : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "n"(kCols) : "memory");
  }
}

template <bool kPair, bool kBF = false, int kBits = 4, int BT = kBT, int SPLIT = 1>
cudaError_t set_smem_attr() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(prefill_kernel<kPair, kBF, kBits, BT, SPLIT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(Layout<kPair, kBits, BT, SPLIT>::SMEM));
    if (err == cudaSuccess && SPLIT > 1)
      err = cudaFuncSetAttribute(prefill_kernel<kPair, kBF, kBits, BT, SPLIT>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  return err;
}

// Clusters of two that fit at once (one CTA per SM), from the occupancy API; cached.
int pair_capacity() {
  static std::once_flag once;
  static int cap = 0;
  std::call_once(once, [] {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Layout<true>::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&cap, prefill_kernel<true>, &cfg) != cudaSuccess) cap = 0;
    (void)cudaGetLastError();
  });
  return cap;
}

}  // namespace

bool prefill_supported(const GemmProblem& p, const char** why) {
  static const char* dummy;
  if (!why) why = &dummy;
  if (p.bits != 4 && p.bits != 8) { *why = "4- or 8-bit codes only"; return false; }
  if (p.bits == 8 && p.bf16) { *why = "8-bit codes: fp16 only"; return false; }
  if (p.K % kBK != 0) { *why = "prefill needs K % 64 == 0"; return false; }
  if (p.G % kBK != 0) { *why = "prefill needs group_size % 64 == 0"; return false; }
  // packed rows a multiple of 16 bytes (tensor-map strides): N % 32 (4 bits), N % 16 (8)
  if (p.N % (p.bits == 8 ? 16 : 32) != 0) { *why = "prefill needs N % 32 == 0 (N % 16 for 8 bits)"; return false; }
  if (!aligned(p.x, 16) || !aligned(p.qw, 16) || !aligned(p.qz, 16) || !aligned(p.sc, 16)) {
    *why = "prefill needs 16-byte aligned x, qweight, qzeros, scales";
    return false;
  }
  return true;
}

// Pair mode (cta_group::2) is exact but measured slower than one CTA per tile on GB300
// (1079 vs 1143 TFLOP/s at M = 2048, K = 4096, N = 11008): each stage's activation copy in
// the peer waits on a commit from the other SM and the peer's readiness signal crosses
// back, and the rings that fit in shared memory do not cover that loop.  Off by default.
#ifndef AWQ_PREFILL_PAIR
#define AWQ_PREFILL_PAIR 0
#endif

namespace {

// CTAs of a narrow-tile launch that are resident on the device at once (occupancy API;
// whole clusters for split launches); cached.  At most two CTAs of this kernel share an SM
// (shared memory, checked in Layout), so the TMEM they allocate (at most 256 columns each
// for BT <= 128) never exceeds the SM's 512 columns and tcgen05.alloc never waits.
template <bool BF, int BITS, int BT, int SPLIT>
int small_capacity() {
  static std::once_flag once;
  static int cap = 0;
  std::call_once(once, [] {
    if (set_smem_attr<false, BF, BITS, BT, SPLIT>() != cudaSuccess) { (void)cudaGetLastError(); return; }
    auto kern = prefill_kernel<false, BF, BITS, BT, SPLIT>;
    const size_t smem = Layout<false, BITS, BT, SPLIT>::SMEM;
    if (SPLIT == 1) {
      int dev = 0, sms = 0, per_sm = 0;
      if (cudaGetDevice(&dev) == cudaSuccess &&
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) == cudaSuccess)
        cap = per_sm * sms;
    } else {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(SPLIT, 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = SPLIT;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess) cap = clusters * SPLIT;
    }
    (void)cudaGetLastError();
  });
  return cap;
}

template <bool BF, int BITS, int BT, int SPLIT>
cudaError_t launch_small_t(const GemmProblem& p, PrefillParams& pp) {
  cudaError_t e = set_smem_attr<false, BF, BITS, BT, SPLIT>();
  if (e != cudaSuccess) return e;
  pp.tiles_t = (p.M + BT - 1) / BT;
  const long long tiles = (long long)pp.tiles_t * ((p.N + kBN - 1) / kBN);
  if (tiles * SPLIT > 0x7fffffffLL) return cudaErrorInvalidValue;
  pp.tiles = static_cast<int>(tiles);
  auto kern = prefill_kernel<false, BF, BITS, BT, SPLIT>;
  const size_t smem = Layout<false, BITS, BT, SPLIT>::SMEM;
  if (SPLIT == 1) {  // persistent over the tiles
    const int cap = small_capacity<BF, BITS, BT, 1>();
    const int grid = pp.tiles < cap ? pp.tiles : (cap > 0 ? cap : 1);
    kern<<<grid, kThreads, smem, p.stream>>>(pp);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pp.tiles * SPLIT), 1, 1);  // one tile per cluster
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = p.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = SPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, pp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Narrow-tile variant for M <= 128 (fp16 or bf16, 4- or 8-bit codes): the narrowest token
// tile holding M rows, and K split over a cluster of 2 or 4 CTAs when that keeps more CTAs
// busy in one wave (at least four stages each).  bt = 0: the 256-row kernel.
struct SmallPlan {
  int bt = 0, split = 1;
};
long long small_cap(const GemmProblem& p, int bt, int split);
SmallPlan plan_small(const GemmProblem& p) {
  SmallPlan sp;
#ifdef AWQ_PREFILL_NO_SMALL
  return sp;
#endif
  if (p.M > 128) return sp;
  sp.bt = p.M <= 32 ? 32 : p.M <= 64 ? 64 : 128;
  const long long tiles = (long long)((p.N + kBN - 1) / kBN) * ((p.M + sp.bt - 1) / sp.bt);
  const int KB = p.K / kBK;
  auto cap = [&](int split) -> long long { return small_cap(p, sp.bt, split); };
  long long best = std::min(tiles, cap(1));
  for (int split : {2, 4}) {
    if (KB < 4 * split) continue;
    const long long c = cap(split);
    if (tiles * split <= c && tiles * split > best) {
      best = tiles * split;
      sp.split = split;
    }
  }
  return sp;
}

template <bool BF, int BITS>
long long small_cap_t(int bt, int split) {
  if (bt == 32)
    return split == 1 ? small_capacity<BF, BITS, 32, 1>() : split == 2 ? small_capacity<BF, BITS, 32, 2>()
                                                                       : small_capacity<BF, BITS, 32, 4>();
  if (bt == 64)
    return split == 1 ? small_capacity<BF, BITS, 64, 1>() : split == 2 ? small_capacity<BF, BITS, 64, 2>()
                                                                       : small_capacity<BF, BITS, 64, 4>();
  return split == 1 ? small_capacity<BF, BITS, 128, 1>() : split == 2 ? small_capacity<BF, BITS, 128, 2>() : 0;
}
long long small_cap(const GemmProblem& p, int bt, int split) {
  if (p.bits == 8) return small_cap_t<false, 8>(bt, split);
  return p.bf16 ? small_cap_t<true, 4>(bt, split) : small_cap_t<false, 4>(bt, split);
}

template <bool BF, int BITS>
cudaError_t launch_small_b(const GemmProblem& p, PrefillParams& pp, const SmallPlan& sp) {
  if (sp.bt == 32)
    return sp.split == 4 ? launch_small_t<BF, BITS, 32, 4>(p, pp)
                         : sp.split == 2 ? launch_small_t<BF, BITS, 32, 2>(p, pp) : launch_small_t<BF, BITS, 32, 1>(p, pp);
  if (sp.bt == 64)
    return sp.split == 4 ? launch_small_t<BF, BITS, 64, 4>(p, pp)
                         : sp.split == 2 ? launch_small_t<BF, BITS, 64, 2>(p, pp) : launch_small_t<BF, BITS, 64, 1>(p, pp);
  return sp.split == 2 ? launch_small_t<BF, BITS, 128, 2>(p, pp) : launch_small_t<BF, BITS, 128, 1>(p, pp);
}
cudaError_t launch_small(const GemmProblem& p, PrefillParams& pp, const SmallPlan& sp) {
  if (p.bits == 8) return launch_small_b<false, 8>(p, pp, sp);
  return p.bf16 ? launch_small_b<true, 4>(p, pp, sp) : launch_small_b<false, 4>(p, pp, sp);
}

}  // namespace

// Estimated duration of launch_prefill for p, in microseconds, from the plan it would take
// (fitted to GB300 timings of the 7B and 70B linears at M = 8 .. 512, within about 10 %):
// waves of CTAs over what is resident at once, each CTA about 0.45-0.5 us per 64-deep K
// stage of its share plus a fixed part (split launches: the partial-sum exchange, growing
// with the token tile).
double prefill_estimate_us(const GemmProblem& p, int sms) {
  const SmallPlan sp = plan_small(p);
  if (sp.bt) {
    const long long tiles = (long long)((p.N + kBN - 1) / kBN) * ((p.M + sp.bt - 1) / sp.bt);
    long long cap = small_cap(p, sp.bt, sp.split);
    if (cap <= 0) cap = sms;
    const double waves = static_cast<double>((tiles * sp.split + cap - 1) / cap);
    return waves * ((p.K / kBK) / static_cast<double>(sp.split) * 0.45 + 2.0 + 0.04 * sp.bt * (sp.split - 1));
  }
  const long long tiles = (long long)((p.N + kBN - 1) / kBN) * ((p.M + kBT - 1) / kBT);
  return static_cast<double>((tiles + sms - 1) / sms) * (p.K / kBK) * 0.5 + 2.0;
}

cudaError_t launch_prefill(const GemmProblem& p) {
  const bool w8 = p.bits == 8;
  const SmallPlan sp = plan_small(p);
  cudaError_t e = w8 ? set_smem_attr<false, false, 8>() : p.bf16 ? set_smem_attr<false, true>() : set_smem_attr<false>();
  if (e == cudaSuccess && !p.bf16 && !w8 && AWQ_PREFILL_PAIR) e = set_smem_attr<true>();
  if (e != cudaSuccess) return e;
  // Pair mode (two CTAs per 256 x 256 tile) when enabled and pairs of SMs can be co-scheduled.
  const int pairs = (AWQ_PREFILL_PAIR && !p.bf16 && !w8) ? pair_capacity() : 0;  // pair mode: fp16, 4 bits
  const bool pair = pairs > 0;
  PrefillParams pp;
  const char* why = nullptr;
  const int C = p.N / (w8 ? 4 : 8);
  const int box_w = kBN / (w8 ? 4 : 8);  // packed words of a tile row
  const int ngrp = p.K / p.G;
  const int x_rows = sp.bt ? sp.bt : (pair ? kBT / 2 : kBT);
  const CUtensorMapDataType et = p.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!make_tmap_2d(&pp.tm_x, et, 2, p.x, p.K, p.M, kBK, x_rows,
                    CU_TENSOR_MAP_SWIZZLE_128B, &why) ||
      !make_tmap_2d(&pp.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.qw, C, p.K, box_w, kBK,
                    CU_TENSOR_MAP_SWIZZLE_NONE, &why) ||
      !make_tmap_2d(&pp.tm_z, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.qz, C, ngrp, box_w, 1,
                    CU_TENSOR_MAP_SWIZZLE_NONE, &why) ||
      !make_tmap_2d(&pp.tm_s, et, 2, p.sc, p.N, ngrp, 128, 1,
                    CU_TENSOR_MAP_SWIZZLE_NONE, &why))
    return cudaErrorInvalidValue;
  pp.bias = p.bias;
  pp.y = p.y;
  e = status_word_ptr(&pp.status);
  if (e != cudaSuccess) return e;
  pp.M = p.M; pp.K = p.K; pp.N = p.N; pp.C = C; pp.G = p.G;
  if (sp.bt) return launch_small(p, pp, sp);
  pp.tiles_t = (p.M + kBT - 1) / kBT;
  const int tile_n = pair ? 2 * kBN : kBN;
  const long long tiles = (long long)pp.tiles_t * ((p.N + tile_n - 1) / tile_n);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  pp.tiles = static_cast<int>(tiles);
  if (pair) {
    const int clusters = pp.tiles < pairs ? pp.tiles : pairs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Layout<true>::SMEM;
    cfg.stream = p.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prefill_kernel<true>, pp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = pp.tiles < sms ? pp.tiles : sms;
  if (w8) prefill_kernel<false, false, 8><<<grid, kThreads, Layout<false, 8>::SMEM, p.stream>>>(pp);
  else if (p.bf16) prefill_kernel<false, true><<<grid, kThreads, Layout<false>::SMEM, p.stream>>>(pp);
  else prefill_kernel<false><<<grid, kThreads, Layout<false>::SMEM, p.stream>>>(pp);
  return cudaGetLastError();
}

// Looked up on every call (no cache): the address belongs to the current context, which a
// device reset or a new context replaces.
cudaError_t status_word_ptr(unsigned int** ptr) {
  void* a = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&a, g_status_word);
  if (e != cudaSuccess) return e;
  *ptr = static_cast<unsigned int*>(a);
  return cudaSuccess;
}

cudaError_t read_and_clear_status(cudaStream_t stream, unsigned int* value) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  unsigned int v = 0u;
  e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v != 0u) {
    const unsigned int zero = 0u;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *value = v;
  return cudaSuccess;
}

}  // namespace awq
