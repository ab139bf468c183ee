// Tile-packed layout: the one-off repack (awq_repack, awq_repack_w8) and the tensor-core
// linear that reads it (awq_gemm_packed and its workspace, bf16, 8-bit, no-allocation and
// grouped forms).
//
// Layout (this library's kernel-native order; repacking the AWQ order away for a kernel is
// the prior art of the vLLM article, section 5.1, and of the GPTQModel wiki, "Marlin and
// Machete").  For output-column tile t (128 columns) and K stage s (64 rows) one block of
// 1152 words sits at word (t * K/64 + s) * 1152:
//   words 512 h + 4 c + j (h < 2, c < 128, j < 4): the 4-bit codes of column 128 t + c for
//     rows 64 s + 32 h + 8 j + 0..7, row offset ORDER[p] in nibble p (ORDER = {0,2,4,6,1,3,
//     5,7}: the checkpoint's column interleave applied along K, so (word >> 4 i) & 0x000F000F
//     holds rows (2 i, 2 i + 1) of the run in its two halves);
//   words 1024 + c: scale bits (fp16) | zero << 16 of column 128 t + c, for the group of
//     row 64 s (every stage of a group carries a copy);
//   columns past N: all zero.
// A CTA's K loop over one column tile reads consecutive blocks: one bulk copy per stage.
//
// The linear (y = x W + bias, w = (code - zero) * scale; tensref.org/formats/awq,
// "Reader"; GPTQModel wiki "AWQ", "Native GEMM": fused dequant-GEMM, fp32 accumulation):
// persistent tcgen05 kernel, one CTA per SM, tiles of 128 output columns (the MMA's M side)
// by BT activation rows (its N side).  The dequantized weights never touch shared memory:
// each dequant thread owns one output column (one TMEM lane), turns the 32 codes of its
// half-stage into 16 fp16 pairs ((c - z) * s exactly: 0x6400 exponent trick, HSUB2,
// HMUL2) and stores them with tcgen05.st into a TMEM ring that the MMA reads as its A
// operand.  Shared memory carries only the activation tiles (TMA, 128-byte swizzle) and the
// packed blocks, which keeps its traffic per stage well below the checkpoint-layout kernel's
// (no A tile written and read back).
//
// Warp roles (448 threads): warp 0 producer (one TMA copy of the activation tile and one
// bulk copy of the packed block per stage), warp 1 TMEM allocation and the MMA-issuing
// thread, warps 2-9 dequant (warp w: TMEM lanes 32 (w % 4) .., K half (w - 2) / 4), warps
// 10-13 epilogue (tcgen05.ld, + bias, rounding, stores).  Every wait is bounded in wall time;
// on give-up the kernel sets the device status word, every role leaves its loop, issued
// copies and MMAs are drained (bounded) and TMEM is freed.
//
// Variants, all of the same kernel body: token tiles of 32 / 64 / 128 rows with a K split over
// a cluster (few rows), 256-row tiles (one accumulator; y staged through shared memory as
// 16-byte stores), stream-K over one CTA per SM with a caller workspace (tiles that fill the
// SMs poorly), a two-CTA cta_group::2 kernel (long K), bf16 activations and scales, 8-bit codes
// (their own block layout, below), and a grouped mode over stacked experts' layouts.  4-bit
// launches of at most 32 rows take a kernel of their own (packed_small_kernel: four
// independent pipelines per CTA, below).
//
// 8-bit codes: the same tiles and meta words (8-bit zeros), 2176-word blocks: word
// 1024 h + 512 k + 4 c + j holds column c's codes for rows 32 h + 16 k + 4 j + 0..3, one
// byte each, so a dequant thread's 32 rows are two 16-byte loads.
#include <mutex>

#include "awq_internal.cuh"
#include "awq_ptx.cuh"

namespace awq {
namespace {

using namespace ptx;

constexpr int kTN = 128;                    // output columns per tile / block
constexpr int kTK = 64;                     // K rows per stage / block
constexpr int kBlockWords = 1024 + kTN;     // codes + meta (4-bit codes)
constexpr int kBlockBytes = 4 * kBlockWords;  // 4608
// Block of one (column tile, K stage) for BITS-bit codes: code words, then kTN meta words at
// word META.  8-bit codes: word (h, k, c, j) at 1024 h + 512 k + 4 c + j holds column c's
// codes for rows 32 h + 16 k + 4 j + 0..3 (row offset b in byte b).
template <int BITS>
struct Blk {
  static constexpr int META = BITS == 8 ? 2048 : 1024;
  static constexpr int WORDS = META + kTN;
  static constexpr int BYTES = 4 * WORDS;  // 4608 / 8704
};
constexpr int kDQ = 8;                      // dequant warps
constexpr int kThreads = (2 + kDQ + 4) * 32;
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;
constexpr unsigned int kStatusPackedTimeout = 0x4u;
constexpr uint32_t kMagic = 0x64006400u;    // fp16 1024 in both halves
constexpr uint32_t kMagicBF = 0x43004300u;  // bf16 128 in both halves
constexpr uint32_t kIdescBF = (1u << 7) | (1u << 10);  // instruction descriptor: A and B bf16
constexpr int kSmemCap = 227 * 1024;
constexpr int kSmemMin = 120 * 1024;        // one CTA per SM: it allocates all 512 TMEM columns
constexpr int kPairMinK = 8192;             // K from which M > 128 runs the two-CTA kernel

// ------------------------------------------------------------------- repack ----

// One CTA per block (column tile t = blockIdx.y, stage s = blockIdx.x).  Thread (h, j, cw):
// rows 64 s + 32 h + 8 j + 0..7 of checkpoint word 16 t + cw hold 8 columns x 8 rows of
// codes; it writes the 8 columns' code words.  Thread c also writes meta word c.  The
// block is assembled in shared memory and stored with 16-byte writes.
__global__ void __launch_bounds__(128) repack_kernel(const uint32_t* __restrict__ qw,
                                                     const uint32_t* __restrict__ qz,
                                                     const uint16_t* __restrict__ sc,
                                                     uint32_t* __restrict__ out, int K, int N, int G) {
  __shared__ __align__(16) uint32_t blk[kBlockWords];
  const int s = blockIdx.x, t = blockIdx.y, KS = K / kTK;
  const int C = N / 8;
  const int tid = threadIdx.x;
  {
    const int h = tid >> 6, j = (tid >> 4) & 3, cw = tid & 15;
    const int word = 16 * t + cw;
    const int r0 = kTK * s + 32 * h + 8 * j;
    uint32_t in[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) in[r] = word < C ? __ldg(qw + static_cast<size_t>(r0 + r) * C + word) : 0u;
#pragma unroll
    for (int q = 0; q < 8; ++q) {  // column 8 cw + q: nibble of position q in ORDER
      int nib = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) nib = nibble_column(i) == q ? i : nib;
      uint32_t v = 0u;
#pragma unroll
      for (int p = 0; p < 8; ++p) v |= ((in[nibble_column(p)] >> (4 * nib)) & 0xFu) << (4 * p);
      blk[512 * h + 4 * (8 * cw + q) + j] = v;
    }
  }
  {
    const int n = kTN * t + tid;
    const int g = (kTK * s) / G;
    uint32_t m = 0u;
    if (n < N) {
      int nib = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) nib = nibble_column(i) == (n & 7) ? i : nib;
      const uint32_t z = (__ldg(qz + static_cast<size_t>(g) * C + n / 8) >> (4 * nib)) & 0xFu;
      m = static_cast<uint32_t>(__ldg(sc + static_cast<size_t>(g) * N + n)) | (z << 16);
    }
    blk[1024 + tid] = m;
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(t * KS + s) * kBlockWords);
  const uint4* src = reinterpret_cast<const uint4*>(blk);
  for (int i = tid; i < kBlockWords / 4; i += 128) dst[i] = src[i];
}

// 8-bit codes: one CTA per block; task (q, cw) (q: rows 4 q .. 4 q + 3 of the stage, cw: one of
// the tile's 32 checkpoint words of 4 columns) transposes a 4 x 4 byte square into the four
// columns' code words.  Thread c also writes meta word c.
__global__ void __launch_bounds__(128) repack8_kernel(const uint32_t* __restrict__ qw,
                                                      const uint32_t* __restrict__ qz,
                                                      const uint16_t* __restrict__ sc,
                                                      uint32_t* __restrict__ out, int K, int N, int G) {
  constexpr int W8 = Blk<8>::WORDS;
  __shared__ __align__(16) uint32_t blk[W8];
  const int s = blockIdx.x, t = blockIdx.y, KS = K / kTK;
  const int C = N / 4;
  const int tid = threadIdx.x;
  for (int task = tid; task < 16 * 32; task += 128) {
    const int cw = task & 31, q = task >> 5;
    const int word = 32 * t + cw;
    const int r0 = kTK * s + 4 * q;
    uint32_t in[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) in[r] = word < C ? __ldg(qw + static_cast<size_t>(r0 + r) * C + word) : 0u;
    const int h = q >> 3, k = (q >> 2) & 1, j = q & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // column 4 cw + i: byte i of rows r0 .. r0 + 3
      const uint32_t sel = static_cast<uint32_t>((4 + i) << 4 | i);
      blk[1024 * h + 512 * k + 4 * (4 * cw + i) + j] = prmt(prmt(in[0], in[1], sel), prmt(in[2], in[3], sel), 0x5410u);
    }
  }
  {
    const int n = kTN * t + tid;
    const int g = (kTK * s) / G;
    uint32_t m = 0u;
    if (n < N) {
      const uint32_t z = (__ldg(qz + static_cast<size_t>(g) * C + n / 4) >> (8 * (n & 3))) & 0xFFu;
      m = static_cast<uint32_t>(__ldg(sc + static_cast<size_t>(g) * N + n)) | (z << 16);
    }
    blk[Blk<8>::META + tid] = m;
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(t * KS + s) * W8);
  const uint4* src = reinterpret_cast<const uint4*>(blk);
  for (int i = tid; i < W8 / 4; i += 128) dst[i] = src[i];
}

// ------------------------------------------------------------ packed linear ----

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// D (TMEM) += A (TMEM, 128 lanes x 16 fp16) * B (shared memory descriptor).
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// tcgen05.ld of 32 columns without the wait (tmem_wait_ld completes every load issued
// before it).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
// Waits for every tcgen05.ld issued before it; the 32 registers pass through the asm so
// that no use of them can be scheduled above the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                 "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                 "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]),
                 "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]),
                 "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// tcgen05.ld of 16 TMEM lanes x 32 columns without the wait, in the MMA-fragment layout:
// thread t gets, for each 8-column group k, registers 4k .. 4k + 3 = (lane t/4, column
// 2(t%4)), (lane t/4, 2(t%4) + 1), (lane t/4 + 8, 2(t%4)), (lane t/4 + 8, 2(t%4) + 1).
__device__ __forceinline__ void tmem_ld16x256_nowait(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
// Four 8x8 b16 matrices into shared memory, transposed: register m of every thread holds its
// fragment of matrix m (thread t: row t/4, elements 2(t%4), +1); lanes 8m .. 8m + 7 give the
// addresses of the rows of the stored (transposed) matrix m.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t saddr, const uint32_t (&m)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr),
               "r"(m[0]), "r"(m[1]), "r"(m[2]), "r"(m[3])
               : "memory");
}
__device__ __forceinline__ uint4 lds128_u(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
// Two values rounded once to the element type (fp16, or bf16 when kBF), lo in the low half.
template <bool kBF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kBF) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}
template <bool kBF>
__device__ __forceinline__ float load_bias(const __half* bias, int n) {
  return elem_to_float<kBF>(reinterpret_cast<const uint16_t*>(bias)[n]);
}
// (c - z) * s on element pairs: the subtraction is exact, the product rounds once.
template <bool kBF>
__device__ __forceinline__ uint32_t dq_sub(uint32_t a, uint32_t b) {
  if constexpr (kBF) return hsub2_bf16(a, b);
  else return hsub2(a, b);
}
template <bool kBF>
__device__ __forceinline__ uint32_t dq_mul(uint32_t a, uint32_t b) {
  if constexpr (kBF) return hmul2_bf16(a, b);
  else return hmul2(a, b);
}

// Pair mode (tcgen05 cta_group::2): the MMA spans the two CTAs of a cluster.
__device__ __forceinline__ void mma_ts_pair(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive, once the MMAs issued so far complete, on the barrier at `bar`'s offset in both CTAs.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<unsigned short>(0x3))
      : "memory");
}
// Arrive (release, cluster scope) on the barrier at `local`'s offset in CTA `rank`.
__device__ __forceinline__ void mbar_arrive_at(uint64_t* local, uint32_t rank) {
  uint32_t ra;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}
// Cluster-window address of `local`'s offset in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t ra;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  return ra;
}
// Asynchronous 16-byte store to a cluster-window address, counted on the (cluster-window)
// barrier `rbar`.
__device__ __forceinline__ void st_async_v4_at(uint32_t raddr, uint32_t rbar, uint32_t a, uint32_t b,
                                               uint32_t c, uint32_t d) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(raddr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(rbar)
               : "memory");
}

// Asynchronous 4-byte store into CTA `rank`'s shared memory at `local`'s offset, counted (4
// bytes) on that CTA's barrier at `bar`'s offset.  It does not block the issuing thread; the
// barrier's completion releases the thread's earlier operations at cluster scope.
__device__ __forceinline__ void st_async_signal(const void* local, uint64_t* bar, uint32_t rank) {
  uint32_t ra, rb;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra),
               "r"(0u), "r"(rb)
               : "memory");
}
// try_wait with cluster-scope acquire (the phase completes through arrivals from the peer CTA).
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
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

// Shared-memory descriptor of a K-major operand with 128-byte swizzle: rows of 128 B (64
// fp16 along K), 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;            // leading byte offset (unused), 16 B
  d |= static_cast<uint64_t>(1024u >> 4) << 32;    // stride byte offset: 8-row groups
  d |= static_cast<uint64_t>(1u) << 46;            // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;            // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, fp16 A and B, both K-major (A comes
// from TMEM), N = BT, M = 128.
template <int BT>
constexpr uint32_t idesc_ts() {
  return (1u << 4) | (static_cast<uint32_t>(BT >> 3) << 17) | (static_cast<uint32_t>(kTN >> 4) << 24);
}

// Resources of a (token tile BT, K split SPLIT) configuration.  TMEM holds NACC accumulators
// of BT columns and one A slot of 32 columns (64 K rows of fp16 pairs) per pipeline slot;
// shared memory holds, per slot, the activation tile and the packed block (one ring: slot s
// carries stage j's activations, packed block and A operand, j = s mod ST), plus, in rank 0 of
// a split, the other ranks' partial sums.  Narrow tiles (BT <= 64) allocate 256 TMEM columns
// and at most half an SM's shared memory, so two CTAs share an SM (per-CTA %smid and
// globaltimer stamps show two resident at once; the occupancy calculator reports one).
template <int BT, int SPLIT, int BITS = 4>
struct Cfg {
  static constexpr int NACC = BT >= 256 ? 1 : 2;
  static constexpr bool kNarrow = BT <= 64;
  static constexpr int COLS = kNarrow ? 256 : 512;           // TMEM columns allocated
  static constexpr int SA_FIT = (COLS - NACC * BT) / 32;
  static constexpr int X_BYTES = BT * kTK * 2;
  static constexpr int BLK = Blk<BITS>::BYTES;
  static constexpr int STAGE = X_BYTES + BLK;
  static constexpr int RECV_PITCH = BT + 4;                  // floats per received column
  static constexpr int RECV_BYTES = (SPLIT - 1) * kTN * RECV_PITCH * 4;
  static constexpr int CAP = kNarrow ? 112 * 1024 : kSmemCap;
  // one accumulator (the MMA waits for the epilogue): y leaves through a 1 KB staging tile
  // per epilogue warp (16 rows x 32 columns) as 16-byte stores
  static constexpr int YST_BYTES = NACC == 1 ? 4 * 1024 : 0;
  static constexpr int ST_FIT = (CAP - 2048 - RECV_BYTES - YST_BYTES) / STAGE;
  static constexpr int ST0 = ST_FIT < SA_FIT ? ST_FIT : SA_FIT;
  static constexpr int ST = ST0 < 8 ? ST0 : 8;
  static constexpr int X_OFF = 0;
  static constexpr int B_OFF = ST * X_BYTES;
  static constexpr int BAR_OFF = B_OFF + ST * BLK;
  // full_t[ST], empty[ST], full_a[ST], acc_full[2], acc_empty[2], drain, recv
  static constexpr int NBARS = 3 * ST + 6;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr int RECV_OFF = ((MISC_OFF + 16 + 15) / 16) * 16;
  static constexpr int YST_OFF = RECV_OFF + RECV_BYTES;
  static constexpr int USED = 1024 + YST_OFF + YST_BYTES;
  // at most one CTA per SM with 512 columns, at most two with 256: tcgen05.alloc never waits
  static constexpr int SMEM_MIN = kNarrow ? 80 * 1024 : kSmemMin;
  static constexpr int SMEM = USED < SMEM_MIN ? SMEM_MIN : USED;
  static constexpr uint32_t A_COL0 = NACC * BT;
  // narrow tiles: two stages per dequant iteration (the dequant latency bounds them)
  static constexpr bool kDqPairs = kNarrow;
  static_assert(ST >= 3 && SMEM <= CAP, "resources");
  static_assert(NACC * BT + ST * 32 <= COLS, "TMEM columns");
};

struct __align__(128) PackedParams {
  CUtensorMap tm_x;          // x [M][K] f16, box {64, BT}, 128B swizzle
  const uint32_t* packed;    // tile-packed weights
  const __half* bias;
  __half* y;
  unsigned int* status;
  int M, K, N;
  int tiles_t, tiles;        // activation-row tiles, total tiles
  int y_vec;                 // y 16-byte aligned and N % 8 == 0: 16-byte stores of y allowed
  // grouped (experts) only: device row offsets [E + 1], column tiles per expert, words per
  // expert's packed layout
  const int* offsets;
  int E, grp_nt;
  size_t expert_words;
  // stream-K only: work units (tiles x stages), ready flags and partial-sum slots
  long long units;
  unsigned int* flags;       // [grid], zero between calls
  float* partial;            // [grid][kSkRows][kTN] fp32
};

// Grouped (mixture-of-experts) launches: rows offsets[e] .. offsets[e + 1] - 1 of x and y belong
// to expert e, whose packed layout is the e-th of E stacked ones.  Tiles run over (expert,
// 256-row tile of its rows, column tile), row tiles fastest; the CTAs find the tile starts
// of the experts in a table built at the start (E <= kGrpMaxE).  Offsets are clamped into
// [0, R] and made non-decreasing, so bad offsets give wrong rows, never a bad access.
constexpr int kGrpMaxE = kPackedGroupedMaxE;
constexpr int kGrpBytes = 4 * (kGrpMaxE + 4);
__device__ __forceinline__ void grp_rows(const PackedParams& p, int e, int& a, int& b) {
  a = min(max(__ldg(p.offsets + e), 0), p.M);
  b = min(max(__ldg(p.offsets + e + 1), a), p.M);
}
__device__ __forceinline__ int grp_count(const PackedParams& p, int e) {
  int a, b;
  grp_rows(p, e, a, b);
  return (b - a + 255) / 256 * p.grp_nt;
}
// One warp: ts[e] = tiles of experts 0 .. e - 1, ts[E] = all tiles.
__device__ __forceinline__ void grp_build_table(const PackedParams& p, int* ts, int lane) {
  const int per = (p.E + 31) / 32;
  const int e0 = min(p.E, lane * per), e1 = min(p.E, e0 + per);
  int mine = 0;
  for (int e = e0; e < e1; ++e) mine += grp_count(p, e);
  int incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += v;
  }
  int run = incl - mine;
  for (int e = e0; e < e1; ++e) {
    ts[e] = run;
    run += grp_count(p, e);
  }
  if (lane == 31) ts[p.E] = incl;
}
struct GrpTile {
  int e, row0, rowb, nt;
};
// Tile -> its expert (the last e with ts[e] <= tile: the tile lies in e's non-empty range),
// first row, end of the expert's rows, column tile.
__device__ __forceinline__ GrpTile grp_tile(const PackedParams& p, const int* ts, int tile) {
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ts[mid] <= tile) lo = mid;
    else hi = mid;
  }
  int a, b;
  grp_rows(p, lo, a, b);
  const int mt = (b - a + 255) / 256;
  const int local = tile - ts[lo];
  GrpTile g;
  g.e = lo;
  g.row0 = a + 256 * (local % mt);
  g.rowb = b;
  g.nt = local / mt;
  return g;
}

// A dequant thread's share of one stage's block (thread = output column c, K half h): its codes
// (4-bit: one 16-byte load; 8-bit: two) and its column's meta word.
template <int BITS>
struct StageCodes {
  uint4 a, b;
  uint32_t meta;
};
template <int BITS>
__device__ __forceinline__ void load_codes(const unsigned char* blk, int h, int c, StageCodes<BITS>& r) {
  if constexpr (BITS == 8) {
    r.a = *reinterpret_cast<const uint4*>(blk + 4096 * h + 16 * c);
    r.b = *reinterpret_cast<const uint4*>(blk + 4096 * h + 2048 + 16 * c);
  } else {
    r.a = *reinterpret_cast<const uint4*>(blk + 16 * (128 * h + c));
  }
  r.meta = *reinterpret_cast<const uint32_t*>(blk + 4 * (Blk<BITS>::META + c));
}
// The 16 element pairs (rows 32 h + 2 i, + 1) of the A operand: (c - z) * s, exact subtraction
// and one rounding.  4-bit: (word >> 4 i') & 0x000F000F holds rows (2 i', 2 i' + 1) of the
// word's eight (ORDER interleave along K), or'ed into 1024 + c (bf16: 128 + c).  8-bit: word q
// holds rows 4 q .. 4 q + 3 one byte each; a byte permute places two of them as 1024 + c.
template <int BITS, bool kBF>
__device__ __forceinline__ void convert_codes(const StageCodes<BITS>& cd, uint32_t (&v)[16]) {
  constexpr uint32_t kMag = kBF ? kMagicBF : kMagic;
  const uint32_t zz = kMag | ((cd.meta >> 16) * 0x00010001u);  // (1024 + z), bf16: (128 + z)
  const uint32_t ss = prmt(cd.meta, 0u, 0x1010u);                // scale in both halves
  if constexpr (BITS == 8) {
    const uint32_t w[8] = {cd.a.x, cd.a.y, cd.a.z, cd.a.w, cd.b.x, cd.b.y, cd.b.z, cd.b.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {  // bytes (0, 1) and (2, 3) under kMag's exponent bytes
      v[2 * q] = dq_mul<kBF>(dq_sub<kBF>(prmt(w[q], kMag, 0x7150u), zz), ss);
      v[2 * q + 1] = dq_mul<kBF>(dq_sub<kBF>(prmt(w[q], kMag, 0x7352u), zz), ss);
    }
  } else if constexpr (kBF) {
    const uint32_t w[4] = {cd.a.x, cd.a.y, cd.a.z, cd.a.w};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
        v[4 * jj + ii] = dq_mul<kBF>(dq_sub<kBF>(and_or(w[jj] >> (4 * ii), 0x000F000Fu, kMag), zz), ss);
  } else {
    // fp16: a nibble in bits 4-7 of a half lies inside the mantissa, so or'ed under the
    // exponent of 64 (mantissa step 1/16) it reads exactly 64 + c; pairs 1 and 3 then need
    // no shift of their own (one shift by 8 serves pairs 2 and 3), and subtracting 64 + z
    // leaves the same exact c - z
    constexpr uint32_t kMag64 = 0x54005400u;                            // fp16 64 in both halves
    const uint32_t zz64 = kMag64 | (((cd.meta >> 16) * 0x00010001u) << 4);  // (64 + z)
    const uint32_t w[4] = {cd.a.x, cd.a.y, cd.a.z, cd.a.w};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t hi = w[jj] >> 8;
      v[4 * jj + 0] = dq_mul<false>(dq_sub<false>(and_or(w[jj], 0x000F000Fu, kMag), zz), ss);
      v[4 * jj + 1] = dq_mul<false>(dq_sub<false>(and_or(w[jj], 0x00F000F0u, kMag64), zz64), ss);
      v[4 * jj + 2] = dq_mul<false>(dq_sub<false>(and_or(hi, 0x000F000Fu, kMag), zz), ss);
      v[4 * jj + 3] = dq_mul<false>(dq_sub<false>(and_or(hi, 0x00F000F0u, kMag64), zz64), ss);
    }
  }
}

// The tiles a CTA takes (tile0, tile0 + tstep, ...) and its K stages [kb0, kb1): without a
// split, tiles blockIdx.x + k gridDim.x and all stages; with one, the cluster's tile and rank
// r's share of the stages.  Each role of the kernel builds its own copy where it loops: one
// copy built before the roles diverge made the 256-row kernel 11% slower.
template <int SPLIT>
struct Span {
  int tile0, tstep, kb0, kb1;
  __device__ __forceinline__ Span(int tiles, int KS, uint32_t krank)
      : tile0(SPLIT > 1 ? static_cast<int>(blockIdx.x) / SPLIT : static_cast<int>(blockIdx.x)),
        tstep(SPLIT > 1 ? tiles : static_cast<int>(gridDim.x)),
        kb0(SPLIT > 1 ? static_cast<int>(static_cast<long long>(KS) * krank / SPLIT) : 0),
        kb1(SPLIT > 1 ? static_cast<int>(static_cast<long long>(KS) * (krank + 1) / SPLIT) : KS) {}
};

// Rows t0 .. t0 + 31 of the warp's 32 output columns c0 + lane (lane's values in v), plus the
// bias, rounded once to fp16.  With a staging tile (16 rows x 32 columns of the warp's own
// shared memory) the rows leave as 16-byte stores, 16 at a time; without, one 2-byte store
// per value.
template <bool kBF>
__device__ __forceinline__ void store_y32(const PackedParams& p, __half* stage, const uint32_t (&v)[32],
                                          float bias, int t0, int c0, int lane, int mlim) {
  if (stage != nullptr) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      __syncwarp();  // the previous round's reads of the tile are done
#pragma unroll
      for (int i = 0; i < 16; ++i)
        stage[i * 32 + lane] = __ushort_as_half(float_to_elem<kBF>(__uint_as_float(v[16 * k + i]) + bias));
      __syncwarp();
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int piece = lane + 32 * r;  // 16 rows x 4 pieces of 8 columns
        const int row = piece >> 2, col = (piece & 3) * 8;
        const int t = t0 + 16 * k + row;
        if (t < mlim && c0 + col < p.N)  // N % 8 == 0: a piece is wholly inside or outside
          *reinterpret_cast<uint4*>(p.y + static_cast<size_t>(t) * p.N + c0 + col) =
              *reinterpret_cast<const uint4*>(stage + row * 32 + col);
      }
    }
    return;
  }
  const int n = c0 + lane;
  if (n < p.N) {
    __half* yp = p.y + static_cast<size_t>(t0) * p.N + n;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (t0 + j < mlim) yp[static_cast<size_t>(j) * p.N] = __ushort_as_half(float_to_elem<kBF>(__uint_as_float(v[j]) + bias));
  }
}

// Rows t_base .. t_base + 31 of the warp's 32 output columns c0 .. c0 + 31 from two 16x256b
// fragment loads (f[0..15]: the quadrant's lanes 0-15, f[16..31]: lanes 16-31), plus the bias
// (ba[h]: column c0 + 16 h + t/4, bb[h]: that + 8), rounded once to fp16.  Sixteen rows at a
// time go into the warp's staging tile (16 rows x 64 bytes) transposed by stmatrix, each
// 16-byte chunk of a row XOR-swizzled by (row / 2) % 4 so the eight rows of a matrix fall in
// distinct banks, and leave as 16-byte stores.
template <bool kBF>
__device__ __forceinline__ void store_y32_frag(const PackedParams& p, __half* stage, const uint32_t (&f)[32],
                                               const float (&ba)[2], const float (&bb)[2], int t_base,
                                               int c0, int lane, int mlim) {
  const uint32_t sbase = smem_u32(stage);
#pragma unroll
  for (int r = 0; r < 2; ++r) {  // tokens 16 r .. 16 r + 15: 8-token groups 2 r, 2 r + 1
    __syncwarp();                // the previous round's reads of the tile are done
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t m[4];
#pragma unroll
      for (int gg = 0; gg < 2; ++gg) {
        const int g = 2 * r + gg;
        m[2 * gg] = pack2<kBF>(__uint_as_float(f[16 * h + 4 * g]) + ba[h], __uint_as_float(f[16 * h + 4 * g + 1]) + ba[h]);
        m[2 * gg + 1] = pack2<kBF>(__uint_as_float(f[16 * h + 4 * g + 2]) + bb[h], __uint_as_float(f[16 * h + 4 * g + 3]) + bb[h]);
      }
      // matrix mm = (token group gg = mm / 2, column block mm % 2); lane 8 mm + i: its row i
      const int mm = lane >> 3, i = lane & 7;
      const int row = 8 * (mm >> 1) + i;
      const int chunk = 2 * h + (mm & 1);  // columns 8 chunk .. 8 chunk + 7 of the warp's 32
      stmatrix_x4_trans(sbase + static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) * 16)), m);
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int piece = lane + 32 * k;  // 16 rows x 4 chunks
      const int row = piece >> 2, chunk = piece & 3;
      const int t = t_base + 16 * r + row;
      const int col = c0 + 8 * chunk;
      if (t < mlim && col < p.N)  // N % 8 == 0: a chunk is wholly inside or outside
        *reinterpret_cast<uint4*>(p.y + static_cast<size_t>(t) * p.N + col) =
            lds128_u(sbase + static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) * 16)));
    }
  }
}

// Stream-K (256-row tiles, one CTA per SM): the tiles' K stages form one sequence of units
// (unit u: stage u % KS of tile u / KS) and CTA i takes units [U i / G, U (i + 1) / G) of the U
// units, so every CTA does the same work whatever the tile count.  A tile cut between CTAs is
// finished by the CTA holding its first stage, which reaches that piece last (it ends its
// range); the CTAs holding later stages of it start their ranges there, write their fp32
// partial sums to their own slot of a global workspace and raise their flag.  Only a range's
// first piece can start inside a tile, so a CTA writes at most one partial.  The finisher adds
// the partials in CTA order (bitwise repeatable), adds the bias, stores y and lowers the flags.
constexpr int kSkRows = 256;                  // token rows of a stream-K tile
constexpr size_t kSkSlotBytes = static_cast<size_t>(kSkRows) * kTN * 4;
constexpr int kSkMinUnits = 8;                // stages per CTA below which stream-K is not used
constexpr int kSkMaxStaged = 3;               // contributors whose rows fit the idle ring twice
__device__ __forceinline__ long long sk_bound(long long units, long long i, long long grid) {
  return units * i / grid;
}
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* ptr) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_release_gpu(unsigned int* ptr, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// SPLIT > 1: a cluster of SPLIT CTAs shares one tile, CTA r taking K stages
// [r KS / SPLIT, (r + 1) KS / SPLIT); ranks 1 .. SPLIT-1 push their fp32 accumulators into
// rank 0's shared memory (st.async, counted on rank 0's recv barrier), and rank 0 adds them
// in rank order, adds the bias and stores y.  Split launches give every cluster one tile.
template <int BT, int SPLIT, bool SK = false, bool kBF = false, int BITS = 4, bool GRP = false>
__global__ void __launch_bounds__(kThreads, Cfg<BT, SPLIT, BITS>::kNarrow ? 2 : 1)
    packed_kernel(const __grid_constant__ PackedParams p) {
  using CF = Cfg<BT, SPLIT, BITS>;
  using BK = Blk<BITS>;
  static_assert(BITS == 4 || (BITS == 8 && !kBF), "8-bit codes: fp16 only");
  static_assert(!GRP || (BT == 256 && SPLIT == 1 && !SK), "grouped: the persistent 256-row kernel");
  static_assert(!SK || (BT == kSkRows && SPLIT == 1), "stream-K: 256-row tiles, no cluster split");
  constexpr int ST = CF::ST, NACC = CF::NACC;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CF::BAR_OFF);
  uint64_t* full_t = bars;            // activation tile + packed block of the slot landed
  uint64_t* empty = bars + ST;        // slot free: block read by the dequant warps, MMAs done
  uint64_t* full_a = bars + 2 * ST;   // dequantized A operand of the slot in TMEM
  uint64_t* acc_full = bars + 3 * ST;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* recv_bar = drain + 1;     // split rank 0: the other ranks' partials landed
  uint64_t* epi_sync = drain + 1;     // stream-K: the four epilogue warps meet (same slot)
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + CF::MISC_OFF);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + CF::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KS = p.K / kTK;
  const uint32_t krank = SPLIT > 1 ? cluster_ctarank() : 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full_t[s], 1);
      mbar_init(&empty[s], kDQ + 1);  // dequant warps (block read) + the MMA commit
      mbar_init(&full_a[s], kDQ);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain, 1);
    mbar_init(recv_bar, SK ? 4 : 1);
    if (SPLIT > 1 && krank == 0u)  // the partials of ranks 1 .. SPLIT-1, one phase
      mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((SPLIT - 1) * kTN * BT * 4));
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(const_cast<uint32_t*>(tmem_slot))), "n"(CF::COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // grouped: the experts' tile starts, after the ring (the host adds kGrpBytes to the launch)
  int* grp_ts = reinterpret_cast<int*>(smem + CF::YST_OFF + CF::YST_BYTES);
  if constexpr (GRP) {
    if (warp == 2 + kDQ) grp_build_table(p, grp_ts, lane);
  }
  __syncthreads();
  if constexpr (SPLIT > 1) cluster_sync_all();  // rank 0's recv barrier exists before any push
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = GRP ? grp_ts[p.E] : p.tiles;

  // Bounded wait; on give-up every role learns it through the abort flag (read only then,
  // and before each blocking wait of the roles that poll it).
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, p.status, kStatusPackedTimeout, kWaitLimitNs)) return true;
    *abort_flag = 1u;
    return false;
  };
  // the same with cluster-scope acquire (phases completed by other CTAs' pushes)
  auto wait_cluster = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if (*abort_flag) return false;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_cl(bar, parity)) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(p.status, kStatusPackedTimeout);
        *abort_flag = 1u;
        return false;
      }
    }
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const Span<SPLIT> sp(p.tiles, KS, krank);
    const int tile0 = sp.tile0, tstep = sp.tstep, kb0 = sp.kb0, kb1 = sp.kb1;
    if (lane == 0) {
      prefetch_tmap(&p.tm_x);
      // packed blocks are read by the token tiles of one column tile, close together in time:
      // evict them first; activation tiles are re-read by every column tile: evict them last
      const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      if constexpr (SK) {
        const long long u0 = sk_bound(p.units, blockIdx.x, gridDim.x);
        const long long u1 = sk_bound(p.units, blockIdx.x + 1, gridDim.x);
        int tile = static_cast<int>(u0 / KS), kb = static_cast<int>(u0 - static_cast<long long>(tile) * KS);
        for (long long u = u0; u < u1; ++u) {
          const int m0 = (tile % p.tiles_t) * BT;
          const uint32_t* src = p.packed + static_cast<size_t>(tile / p.tiles_t) * KS * BK::WORDS;
          if (!wait(&empty[s], ph ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(&full_t[s], static_cast<uint32_t>(CF::X_BYTES + BK::BYTES));
          tma_load_2d_hint(smem + CF::X_OFF + s * CF::X_BYTES, &p.tm_x, &full_t[s], kb * kTK, m0, pol_x);
          bulk_load(smem + CF::B_OFF + s * BK::BYTES, src + static_cast<size_t>(kb) * BK::WORDS,
                    BK::BYTES, &full_t[s], pol_w);
          ++issued;
          if (++s == ST) { s = 0; ph ^= 1u; }
          if (++kb == KS) { kb = 0; ++tile; }
        }
      } else
      for (int tile = tile0; ok && tile < ntiles; tile += tstep) {
        int m0, t;
        const uint32_t* src = p.packed;
        if constexpr (GRP) {
          const GrpTile g = grp_tile(p, grp_ts, tile);
          m0 = g.row0;
          t = g.nt;
          src += static_cast<size_t>(g.e) * p.expert_words;
        } else {
          m0 = (tile % p.tiles_t) * BT;
          t = tile / p.tiles_t;
        }
        src += static_cast<size_t>(t) * KS * BK::WORDS;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait(&empty[s], ph ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(&full_t[s], static_cast<uint32_t>(CF::X_BYTES + BK::BYTES));
          tma_load_2d_hint(smem + CF::X_OFF + s * CF::X_BYTES, &p.tm_x, &full_t[s], kb * kTK, m0, pol_x);
          bulk_load(smem + CF::B_OFF + s * BK::BYTES, src + static_cast<size_t>(kb) * BK::WORDS,
                    BK::BYTES, &full_t[s], pol_w);
          ++issued;
          if (++s == ST) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {  // every issued stage's copies land before the CTA may exit
        for (int i = 0; i < ST && i < issued; ++i) {
          if (--s < 0) { s = ST - 1; ph ^= 1u; }
          mbar_wait_bounded(&full_t[s], ph, p.status, kStatusPackedTimeout, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    const Span<SPLIT> sp(p.tiles, KS, krank);
    const int tile0 = sp.tile0, tstep = sp.tstep, kb0 = sp.kb0, kb1 = sp.kb1;
    // Stages go in pairs: one wait on the later stage's full_a covers both (every dequant
    // warp arrives on its slots in stage order, and each arrival releases the warp's TMEM
    // stores of all earlier stages); the activation tiles are in place once full_a is (the
    // dequant warps waited for them).  One commit per stage frees its slot.
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_ts<BT>() | (kBF ? kIdescBF : 0u);
      int s = 0, li = 0;
      uint32_t ph = 0;
      bool ok = true, any = false;
      if constexpr (SK) {  // one accumulator round per piece of a tile in the CTA's range
        const long long u0 = sk_bound(p.units, blockIdx.x, gridDim.x);
        const long long u1 = sk_bound(p.units, blockIdx.x + 1, gridDim.x);
        for (long long u = u0; ok && u < u1; ++li) {
          const int tile = static_cast<int>(u / KS);
          const int kb0 = static_cast<int>(u - static_cast<long long>(tile) * KS);
          const int kb1 = u1 - u < KS - kb0 ? kb0 + static_cast<int>(u1 - u) : KS;
          u += kb1 - kb0;
          const int b = li % NACC;
          if (!wait(&acc_empty[b], static_cast<uint32_t>(((li / NACC) & 1) ^ 1))) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(b * BT);
          for (int kb = kb0; kb < kb1; kb += 2) {
            const int n2 = kb1 - kb < 2 ? kb1 - kb : 2;
            const int sl = s + n2 - 1 < ST ? s + n2 - 1 : s + n2 - 1 - ST;
            const uint32_t phl = s + n2 - 1 < ST ? ph : ph ^ 1u;
            if (!wait(&full_a[sl], phl)) { ok = false; break; }
            tc_fence_after();
            for (int i = 0; i < n2; ++i) {
              const uint32_t a = tmem_base + CF::A_COL0 + static_cast<uint32_t>(s * 32);
              const uint64_t bdesc = sw128_kmajor_desc(sbase + CF::X_OFF + s * CF::X_BYTES);
#pragma unroll
              for (int ks = 0; ks < kTK / 16; ++ks)  // K += 16: A 8 TMEM columns, B 32 bytes
                mma_ts(d, a + 8u * ks, bdesc + 2u * ks, idesc, (kb + i > kb0 || ks > 0) ? 1u : 0u);
              mma_commit(&empty[s]);
              if (++s == ST) { s = 0; ph ^= 1u; }
            }
            any = true;
          }
          if (!ok) break;
          mma_commit(&acc_full[b]);
        }
      } else
      for (int tile = tile0; ok && tile < ntiles; tile += tstep, ++li) {
        const int b = li % NACC;
        if (!wait(&acc_empty[b], static_cast<uint32_t>(((li / NACC) & 1) ^ 1))) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(b * BT);
        for (int kb = kb0; kb < kb1; kb += 2) {
          const int n2 = kb1 - kb < 2 ? kb1 - kb : 2;
          const int sl = s + n2 - 1 < ST ? s + n2 - 1 : s + n2 - 1 - ST;
          const uint32_t phl = s + n2 - 1 < ST ? ph : ph ^ 1u;
          if (!wait(&full_a[sl], phl)) { ok = false; break; }
          tc_fence_after();
          for (int i = 0; i < n2; ++i) {
            const uint32_t a = tmem_base + CF::A_COL0 + static_cast<uint32_t>(s * 32);
            const uint64_t bdesc = sw128_kmajor_desc(sbase + CF::X_OFF + s * CF::X_BYTES);
#pragma unroll
            for (int ks = 0; ks < kTK / 16; ++ks)  // K += 16: A 8 TMEM columns, B 32 bytes
              mma_ts(d, a + 8u * ks, bdesc + 2u * ks, idesc, (kb + i > kb0 || ks > 0) ? 1u : 0u);
            mma_commit(&empty[s]);
            if (++s == ST) { s = 0; ph ^= 1u; }
          }
          any = true;
        }
        if (!ok) break;
        mma_commit(&acc_full[b]);
      }
      if (any) {  // every MMA completes before TMEM is released
        mma_commit(drain);
        mbar_wait_bounded(drain, 0u, p.status, kStatusPackedTimeout, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp < 2 + kDQ) {
    // ------------------------------------------------------------------ dequant
    const Span<SPLIT> sp(p.tiles, KS, krank);
    const int tile0 = sp.tile0, tstep = sp.tstep, kb0 = sp.kb0, kb1 = sp.kb1;
    // Thread = output column c of the tile (TMEM lane), K half h of every stage: the four
    // code words of its half-run (one 16-byte load, lanes contiguous) and its meta word;
    // pair i of the result holds rows 32 h + 2 i, +1 (nibbles i % 4 and i % 4 + 4 of word
    // i / 4), stored to TMEM columns 16 h + i of the slot's A operand.  The slot's A operand
    // is free once its activations have landed: the producer refilled the slot only after
    // the previous round's MMAs completed.  Narrow tiles take two consecutive stages per
    // iteration (the CTA's stages of all its tiles form one sequence), overlapping the
    // pair's waits, loads and TMEM stores.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int c = 32 * q + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const int my_tiles = tile0 < ntiles ? (ntiles - 1 - tile0) / tstep + 1 : 0;
    const long long total =  // the CTA's stages
        SK ? sk_bound(p.units, blockIdx.x + 1, gridDim.x) - sk_bound(p.units, blockIdx.x, gridDim.x)
           : static_cast<long long>(my_tiles) * (kb1 - kb0);
    constexpr int kStep = CF::kDqPairs ? 2 : 1;
    int s = 0;
    uint32_t ph = 0;
    for (long long g = 0; g < total; g += kStep) {
      const bool two = kStep == 2 && g + 1 < total;
      const int s1 = s + 1 == ST ? 0 : s + 1;
      const uint32_t ph1 = s + 1 == ST ? ph ^ 1u : ph;
      if (!wait(&full_t[s], ph)) break;
      StageCodes<BITS> c0, c1;
      load_codes<BITS>(smem + CF::B_OFF + s * BK::BYTES, h, c, c0);
      if (two) {
        if (!wait(&full_t[s1], ph1)) break;
        load_codes<BITS>(smem + CF::B_OFF + s1 * BK::BYTES, h, c, c1);
      }
      tc_fence_after();  // the TMEM stores below come after the previous round's MMAs
      uint32_t v[16];
      convert_codes<BITS, kBF>(c0, v);
      tmem_st16(tmem_base + lane_addr + CF::A_COL0 + static_cast<uint32_t>(s * 32 + 16 * h), v);
      if (two) {
        convert_codes<BITS, kBF>(c1, v);
        tmem_st16(tmem_base + lane_addr + CF::A_COL0 + static_cast<uint32_t>(s1 * 32 + 16 * h), v);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&full_a[s]);
        mbar_arrive(&empty[s]);
        if (two) {
          mbar_arrive(&full_a[s1]);
          mbar_arrive(&empty[s1]);
        }
      }
      if (two) {
        s = s1 + 1 == ST ? 0 : s1 + 1;
        ph = s1 + 1 == ST ? ph1 ^ 1u : ph1;
      } else {
        s = s1;
        ph = ph1;
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const Span<SPLIT> sp(p.tiles, KS, krank);
    const int tile0 = sp.tile0, tstep = sp.tstep;
    // The next 32-column chunk is loaded from TMEM while the current one is stored.
    const int q = warp & 3;              // TMEM lanes 32 q .. 32 q + 31
    const int nl = 32 * q + lane;        // output column inside the tile
    float* recv = reinterpret_cast<float*>(smem + CF::RECV_OFF);
    __half* ystage = (CF::YST_BYTES > 0 && p.y_vec != 0)
                         ? reinterpret_cast<__half*>(smem + CF::YST_OFF) + q * 512 : nullptr;
    int li = 0;
    if constexpr (SK) {
      const int bid = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
      const long long u0 = sk_bound(p.units, bid, G), u1 = sk_bound(p.units, bid + 1, G);
      volatile uint32_t* sk_ok = reinterpret_cast<volatile uint32_t*>(smem + CF::MISC_OFF + 8);
      const bool leader = warp == 2 + kDQ && lane == 0;
      uint32_t mph = 0;
      // the four epilogue warps meet (bounded; arrival releases each warp's earlier stores)
      auto meet = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_sync);
        const bool met = wait(epi_sync, mph);
        mph ^= 1u;
        return met;
      };
      for (long long u = u0; u < u1; ++li) {
        const int tile = static_cast<int>(u / KS);
        const int kb0 = static_cast<int>(u - static_cast<long long>(tile) * KS);
        const int kb1 = u1 - u < KS - kb0 ? kb0 + static_cast<int>(u1 - u) : KS;
        u += kb1 - kb0;
        const int b = li % NACC;
        const int m0 = (tile % p.tiles_t) * BT;
        const int n = (tile / p.tiles_t) * kTN + nl;
        const int mlim = p.M;
        if (!wait(&acc_full[b], static_cast<uint32_t>((li / NACC) & 1))) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * BT);
        if (kb0 != 0) {
          // a later piece of the tile (the range's first): partial sums to this CTA's slot,
          // [row][column] so that each warp store covers 128 contiguous bytes, then the flag
          float* slot = p.partial + static_cast<size_t>(bid) * (kSkRows * kTN);
#pragma unroll 1
          for (int cc = 0; cc < BT / 32; ++cc) {
            uint32_t v[32];
            tmem_ld32_nowait(taddr + 32 * cc, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int j = 0; j < 32; ++j) __stcg(slot + static_cast<size_t>(32 * cc + j) * kTN + nl, __uint_as_float(v[j]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[b]);
          const bool met = meet();
          if (met && leader) {
            __threadfence();
            st_release_gpu(p.flags + bid, 1u);
          }
          if (!met) break;
          continue;
        }
        // the tile's first piece: add the partials of the CTAs whose ranges start inside it
        const long long tile_end = static_cast<long long>(tile + 1) * KS;
        int c1 = bid + 1;
        while (c1 < G && sk_bound(p.units, c1, G) < tile_end) ++c1;
        if (leader) {
          uint32_t ok = 1u;
          for (int c = bid + 1; ok != 0u && c < c1; ++c) {
            if (ld_acquire_gpu(p.flags + c) != 0u) continue;
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(p.flags + c) == 0u) {
              if (*abort_flag != 0u || globaltimer_ns() - t0 > kWaitLimitNs) {
                atomicOr(p.status, kStatusPackedTimeout);
                *abort_flag = 1u;
                ok = 0u;
                break;
              }
            }
          }
          *sk_ok = ok;
        }
        if (!meet()) break;
        const bool have = *sk_ok != 0u;
        const int nc = c1 - bid - 1;  // contributors
        // This piece ends the CTA's range: its MMAs are complete, so the ring's shared memory
        // is idle.  The contributors' rows of each 32-row chunk (nc x 16 KB, [row][column])
        // come in there by cp.async, double-buffered a chunk ahead, and are added from
        // shared memory, so no y store waits behind a global load.
        const bool staged = have && nc <= kSkMaxStaged;
        const int et = threadIdx.x - (2 + kDQ) * 32;  // 0 .. 127
        auto fetch = [&](int cc) {
          float* buf = reinterpret_cast<float*>(smem) + (cc & 1) * (kSkMaxStaged * 32 * kTN);
          for (int c = 0; c < nc; ++c) {
            const float* src = p.partial + static_cast<size_t>(bid + 1 + c) * (kSkRows * kTN) +
                               static_cast<size_t>(32 * cc) * kTN;
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // 16 KB: 1024 pieces of 16 bytes over 128 threads
              const int i = et + 128 * k;
              cp_async16(buf + c * (32 * kTN) + 4 * i, src + 4 * i);
            }
          }
          cp_async_commit();
        };
        if (staged) fetch(0);
        const float bias = (p.bias != nullptr && n < p.N) ? load_bias<kBF>(p.bias, n) : 0.f;
        uint32_t va[32], vb[32];
        tmem_ld32_nowait(taddr, va);
        tmem_wait_ld(va);
        bool chunks_met = true;
#pragma unroll
        for (int cc = 0; cc < BT / 32; ++cc) {
          uint32_t (&cur)[32] = (cc & 1) ? vb : va;
          uint32_t (&nxt)[32] = (cc & 1) ? va : vb;
          if (cc + 1 < BT / 32) tmem_ld32_nowait(taddr + 32 * (cc + 1), nxt);
          if (staged) {
            cp_async_wait_all();        // this thread's pieces of chunk cc landed
            if (chunks_met) chunks_met = meet();  // all pieces of chunk cc landed; chunk cc - 1 read
            if (cc + 1 < BT / 32) fetch(cc + 1);
            const float* buf = reinterpret_cast<const float*>(smem) + (cc & 1) * (kSkMaxStaged * 32 * kTN);
#pragma unroll 1
            for (int c = 0; c < nc; ++c) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                cur[j] = __float_as_uint(__uint_as_float(cur[j]) + buf[c * (32 * kTN) + j * kTN + nl]);
            }
          } else if (have) {
#pragma unroll 1
            for (int c = bid + 1; c < c1; ++c) {
              const float* slot = p.partial + static_cast<size_t>(c) * (kSkRows * kTN);
#pragma unroll
              for (int j = 0; j < 32; ++j)
                cur[j] = __float_as_uint(__uint_as_float(cur[j]) +
                                         __ldcg(slot + static_cast<size_t>(32 * cc + j) * kTN + nl));
            }
          }
          store_y32<kBF>(p, ystage, cur, bias, m0 + 32 * cc, n - lane, lane, mlim);
          if (cc + 1 < BT / 32) tmem_wait_ld(nxt);
        }
        if (!chunks_met) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[b]);
        const bool met = meet();  // every epilogue thread has read the partials: lower the flags
        if (met && have && leader)
          for (int c = bid + 1; c < c1; ++c) p.flags[c] = 0u;
        if (!met) break;
      }
    } else
    for (int tile = tile0; tile < ntiles; tile += tstep, ++li) {
      const int b = li % NACC;
      int m0, n, mlim = p.M;
      const __half* bias_row = p.bias;
      if constexpr (GRP) {
        const GrpTile g = grp_tile(p, grp_ts, tile);
        m0 = g.row0;
        n = g.nt * kTN + nl;
        mlim = g.rowb;  // the next expert's rows are computed and discarded
        if (bias_row != nullptr) bias_row += static_cast<size_t>(g.e) * p.N;
      } else {
        m0 = (tile % p.tiles_t) * BT;
        n = (tile / p.tiles_t) * kTN + nl;
      }
      const float bias = (bias_row != nullptr && n < p.N) ? load_bias<kBF>(bias_row, n) : 0.f;
      if (!wait(&acc_full[b], static_cast<uint32_t>((li / NACC) & 1))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * BT);
      if (SPLIT > 1 && krank != 0u) {
        // this rank's partial sums of column nl, all BT rows, into rank 0
        const uint32_t rbar = cluster_addr(recv_bar, 0u);
        const uint32_t rdst = cluster_addr(recv + (static_cast<int>(krank - 1) * kTN + nl) * CF::RECV_PITCH, 0u);
#pragma unroll 1
        for (int cc = 0; cc < BT / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32_nowait(taddr + 32 * cc, v);
          tmem_wait_ld(v);
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            st_async_v4_at(rdst + static_cast<uint32_t>((32 * cc + j) * 4), rbar, v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      } else {
        if (SPLIT > 1 && !wait_cluster(recv_bar, 0u)) break;
        // chunk cc of the accumulator (in cur), plus the other ranks' partials in rank order,
        // plus the bias, rounded once and stored
        auto finish = [&](int cc, uint32_t (&cur)[32]) {
#pragma unroll
          for (int r = 1; r < SPLIT; ++r) {
            const float* src = recv + ((r - 1) * kTN + nl) * CF::RECV_PITCH + 32 * cc;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 q4 = *reinterpret_cast<const float4*>(src + j);
              cur[j] = __float_as_uint(__uint_as_float(cur[j]) + q4.x);
              cur[j + 1] = __float_as_uint(__uint_as_float(cur[j + 1]) + q4.y);
              cur[j + 2] = __float_as_uint(__uint_as_float(cur[j + 2]) + q4.z);
              cur[j + 3] = __float_as_uint(__uint_as_float(cur[j + 3]) + q4.w);
            }
          }
          store_y32<kBF>(p, ystage, cur, bias, m0 + 32 * cc, n - lane, lane, mlim);
        };
        if constexpr (CF::kNarrow) {  // one or two chunks: no prefetch (register budget)
#pragma unroll 1
          for (int cc = 0; cc < BT / 32; ++cc) {
            uint32_t v[32];
            tmem_ld32_nowait(taddr + 32 * cc, v);
            tmem_wait_ld(v);
            finish(cc, v);
          }
        } else if (SPLIT == 1 && ystage != nullptr) {
          // one accumulator: MMA-fragment loads, stmatrix into the staging tile, 16-byte stores
          const int c0 = n - lane;
          float ba[2], bb[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int na = c0 + 16 * h + (lane >> 2), nb = na + 8;
            ba[h] = (bias_row != nullptr && na < p.N) ? load_bias<kBF>(bias_row, na) : 0.f;
            bb[h] = (bias_row != nullptr && nb < p.N) ? load_bias<kBF>(bias_row, nb) : 0.f;
          }
          const uint32_t fbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * BT);
          uint32_t va[32], vb[32];
          tmem_ld16x256_nowait(fbase, va);
          tmem_ld16x256_nowait(fbase + (16u << 16), va + 16);
          tmem_wait_ld(va);
#pragma unroll
          for (int cc = 0; cc < BT / 32; ++cc) {
            uint32_t (&cur)[32] = (cc & 1) ? vb : va;
            uint32_t (&nxt)[32] = (cc & 1) ? va : vb;
            if (cc + 1 < BT / 32) {
              tmem_ld16x256_nowait(fbase + 32 * (cc + 1), nxt);
              tmem_ld16x256_nowait(fbase + (16u << 16) + 32 * (cc + 1), nxt + 16);
            }
            store_y32_frag<kBF>(p, ystage, cur, ba, bb, m0 + 32 * cc, c0, lane, mlim);
            if (cc + 1 < BT / 32) tmem_wait_ld(nxt);
          }
        } else {
          uint32_t va[32], vb[32];
          tmem_ld32_nowait(taddr, va);
          tmem_wait_ld(va);
#pragma unroll
          for (int cc = 0; cc < BT / 32; ++cc) {
            uint32_t (&cur)[32] = (cc & 1) ? vb : va;
            uint32_t (&nxt)[32] = (cc & 1) ? va : vb;
            if (cc + 1 < BT / 32) tmem_ld32_nowait(taddr + 32 * (cc + 1), nxt);
            finish(cc, cur);
            if (cc + 1 < BT / 32) tmem_wait_ld(nxt);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }

  // split: rank 0 leaves only once the other ranks' pushes have landed (bounded: after a
  // give-up elsewhere some may never come), and no rank leaves before the others are done
  if (SPLIT > 1 && krank == 0u && threadIdx.x == 0) (void)wait_cluster(recv_bar, 0u);
  __syncthreads();
  if constexpr (SPLIT > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "n"(CF::COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------ small batches ----
// Token tiles of 16 or 32 rows (M <= 32; 4-bit codes, or 8-bit ones in their own blocks).  A 32-row tile gives the tensor core
// about 32 cycles of work a stage, far less than the issue cost of the stage's own async
// instructions on one thread (each tcgen05.mma, commit, bulk copy or barrier wait takes
// some 60-100 cycles to issue, measured with clock stamps), so one pipeline per SM leaves
// the SM idle.  A CTA here runs P independent pipelines side by side (P = 4: one CTA per SM,
// all 512 TMEM columns and nearly all shared memory; P = 2: two CTAs per SM, half of each,
// which lets more CTAs split a tile count that fills the SMs poorly), each with its own producer
// thread (one TMA copy and one bulk copy per stage), MMA-issuing thread, four dequant warps
// (one per TMEM lane quadrant), ring of ST shared-memory stages, SA A slots and accumulator
// in its own 128 TMEM columns.  Pipeline j takes the j-th quarter of the CTA's K stages; the
// dequant warps of pipeline 0 add the P accumulators in order.  The K loop of one 128-column
// tile is further split over a cluster of CS CTAs (1 .. 16, set at launch so the grid is
// resident in one wave); rank r finishes output columns [128 r / CS, 128 (r + 1) / CS): the
// other ranks push their fp32 sums of those columns into its shared memory (st.async,
// counted on one barrier) and it adds all CS partials in rank order (bitwise repeatable),
// adds the bias and stores y.
constexpr int kSmallMaxCS = 16;
template <int BT, int NP, int BITS = 4>
struct SmallCfg {
  static_assert(BT == 16 || BT == 32, "token tiles of 16 or 32 rows");
  static_assert(NP == 2 || NP == 4, "two or four pipelines");
  static constexpr int BLK = Blk<BITS>::BYTES;        // packed block of a stage
  static constexpr int P = NP;
  static constexpr int THREADS = P * 6 * 32;
  static constexpr int PER_SM = 4 / P;                // CTAs per SM
  static constexpr int COLS = 128 * P;                // 128 per pipeline
  static constexpr int SA = 3;                        // A slots per pipeline, after its accumulator
  static constexpr int X_BYTES = BT * kTK * 2;        // 1024-byte multiple (SW128 atoms)
  static constexpr int RECV_PITCH = BT + 4;           // floats per received column
  static constexpr int RECV_BYTES = (kTN + kSmallMaxCS) * RECV_PITCH * 4;
  // an SM's shared memory over its CTAs, less the per-CTA reservation
  static constexpr int CAP = P == 4 ? kSmemCap : 228 * 1024 / PER_SM - 1024;
  static constexpr int ST0 = (CAP - 2048 - RECV_BYTES) / (P * (X_BYTES + BLK));
  // the ring must be deeper than the A slots (8-bit codes with 32-row tiles leave two
  // pipelines too little shared memory: that variant does not exist)
  static constexpr bool FITS = ST0 > SA;
  static constexpr int ST = !FITS ? SA + 1 : ST0 < 8 ? ST0 : 8;  // ring stages per pipeline
  static constexpr int X_OFF = 0;                     // x ring of pipeline j, stage s: (j ST + s) X_BYTES
  static constexpr int B_OFF = P * ST * X_BYTES;
  static constexpr int BAR_OFF = B_OFF + P * ST * BLK;
  // per pipeline: full_t[ST], empty_t[ST], full_a[SA], acc_full; then recv
  static constexpr int ACC = 2 * ST + SA;             // acc_full's index in a pipeline's barriers
  static constexpr int NB = ACC + 1;
  static constexpr int MISC_OFF = BAR_OFF + (P * NB + 1) * 8;
  static constexpr int RECV_OFF = ((MISC_OFF + 8 + 15) / 16) * 16;
  static constexpr int SMEM = 1024 + RECV_OFF + RECV_BYTES;
  static_assert(!FITS || SMEM <= CAP, "resources");
  static_assert(32 + SA * 32 <= COLS / P, "TMEM columns");
};

template <int BT, int NP, bool kBF, int BITS>
__global__ void __launch_bounds__(SmallCfg<BT, NP, BITS>::THREADS, SmallCfg<BT, NP, BITS>::PER_SM)
    packed_small_kernel(const __grid_constant__ PackedParams p) {
  using CF = SmallCfg<BT, NP, BITS>;
  using BK = Blk<BITS>;
  static_assert(CF::FITS, "ring deeper than the A slots");
  static_assert(BITS == 4 || !kBF, "8-bit codes: fp16 only");
  constexpr int ST = CF::ST, SA = CF::SA, P = CF::P, NB = CF::NB;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + CF::BAR_OFF);
  uint64_t* recv_bar = bars_all + P * NB;  // the other ranks' sums of this rank's columns landed
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + CF::MISC_OFF);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + CF::MISC_OFF + 4);
  float* recv = reinterpret_cast<float*>(smem + CF::RECV_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pipe = warp / 6, role = warp % 6;  // role 0 producer, 1 MMA issuer, 2-5 dequant
  const int KS = p.K / kTK;
  const int cs = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int tile = static_cast<int>(blockIdx.x) / cs;  // token tiles fastest
  const int m0 = (tile % p.tiles_t) * BT;
  const int nt = tile / p.tiles_t;
  const int kr0 = KS * rank / cs, kr = KS * (rank + 1) / cs - kr0;  // this rank's stages; KS * 16 < 2^31
  const int kb0 = kr0 + kr * pipe / P, nst = kr0 + kr * (pipe + 1) / P - kb0;  // this pipeline's
  const int own_lo = kTN * rank / cs, own_hi = kTN * (rank + 1) / cs;
  // this pipeline's barriers, ring and TMEM columns
  uint64_t* bars = bars_all + pipe * NB;
  uint64_t* full_t = bars;             // activation tile + packed block of the slot landed
  uint64_t* empty_t = bars + ST;       // slot free: block read by the dequant warps, MMAs done
  uint64_t* full_a = bars + 2 * ST;    // A slot dequantized
  uint64_t* acc_full = bars + CF::ACC;  // every MMA of the pipeline done
  unsigned char* xring = smem + CF::X_OFF + pipe * ST * CF::X_BYTES;
  unsigned char* bring = smem + CF::B_OFF + pipe * ST * BK::BYTES;

  if (threadIdx.x == 0) {
    for (int j = 0; j < P; ++j) {
      uint64_t* b = bars_all + j * NB;
      for (int s = 0; s < ST; ++s) {
        mbar_init(&b[s], 1);
        mbar_init(&b[ST + s], 4 + 1);  // four dequant warps (block read) + the MMA commit
      }
      for (int a = 0; a < SA; ++a) mbar_init(&b[2 * ST + a], 4);
      mbar_init(&b[CF::ACC], 1);
    }
    mbar_init(recv_bar, 1);
    if (cs > 1)  // the other ranks' sums of this rank's columns, one phase
      mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((cs - 1) * (own_hi - own_lo) * BT * 4));
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(const_cast<uint32_t*>(tmem_slot))), "n"(CF::COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  __syncthreads();
  if (cs > 1) cluster_sync_all();  // every rank's recv barrier exists before any push
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tcol = tmem_base + static_cast<uint32_t>(pipe * (CF::COLS / P));  // accumulator

  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, p.status, kStatusPackedTimeout, kWaitLimitNs)) return true;
    *abort_flag = 1u;
    return false;
  };

  if (role == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_x);
      const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
      const uint32_t* src = p.packed + (static_cast<size_t>(nt) * KS + kb0) * BK::WORDS;
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < nst; ++i) {
        const int s = i % ST;
        if (!wait(&empty_t[s], static_cast<uint32_t>((i / ST) & 1) ^ 1u)) { ok = false; break; }
        mbar_arrive_expect_tx(&full_t[s], static_cast<uint32_t>(CF::X_BYTES + BK::BYTES));
        tma_load_2d_hint(xring + s * CF::X_BYTES, &p.tm_x, &full_t[s], (kb0 + i) * kTK, m0, pol_x);
        bulk_load(bring + s * BK::BYTES, src + static_cast<size_t>(i) * BK::WORDS, BK::BYTES, &full_t[s], pol_w);
        ++issued;
      }
      if (!ok)  // every issued stage's copies land before the CTA may exit
        for (int i = issued - 1; i >= 0 && i >= issued - ST; --i)
          mbar_wait_bounded(&full_t[i % ST], static_cast<uint32_t>((i / ST) & 1), p.status, kStatusPackedTimeout,
                            kWaitLimitNs);
    }
  } else if (role == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_ts<BT>() | (kBF ? kIdescBF : 0u);
      const uint32_t xbase = sbase + static_cast<uint32_t>(xring - smem);
      // Stages in pairs: one wait on the later stage's full_a covers both (every dequant warp
      // arrives in stage order, and each arrival releases its TMEM stores of earlier stages).
      // One commit per stage frees its ring slot; the dequant warps take that as the signal
      // that the A slot of the same stage is free too.
      for (int i = 0; i < nst; i += 2) {
        const int n2 = nst - i < 2 ? nst - i : 2, il = i + n2 - 1;
        if (!wait(&full_a[il % SA], static_cast<uint32_t>((il / SA) & 1))) break;
        tc_fence_after();
        for (int h = 0; h < n2; ++h) {
          const int s = (i + h) % ST, a = (i + h) % SA;
          const uint32_t aaddr = tcol + 32u + static_cast<uint32_t>(32 * a);
          const uint64_t bdesc = sw128_kmajor_desc(xbase + s * CF::X_BYTES);
#pragma unroll
          for (int ks = 0; ks < kTK / 16; ++ks)  // K += 16: A 8 TMEM columns, B 32 bytes
            mma_ts(tcol, aaddr + 8u * ks, bdesc + 2u * ks, idesc, (i + h > 0 || ks > 0) ? 1u : 0u);
          mma_commit(&empty_t[s]);
        }
      }
      // completes once every MMA issued above is done (after a give-up too: TMEM is freed
      // only after this wait)
      mma_commit(acc_full);
      mbar_wait_bounded(acc_full, 0u, p.status, kStatusPackedTimeout, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ dequant, finish
    // Thread = output column c of the tile (TMEM lane): per stage its codes of both K halves
    // (two 16-byte loads) and its meta word, 32 element pairs stored to the stage's A slot.
    const int q = warp & 3;  // TMEM lanes 32 q .. 32 q + 31
    const int c = 32 * q + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    bool ok = true;
    for (int i = 0; i < nst; ++i) {
      const int s = i % ST, a = i % SA;
      if (!wait(&full_t[s], static_cast<uint32_t>((i / ST) & 1))) { ok = false; break; }
      StageCodes<BITS> c0, c1;
      const unsigned char* blk = bring + s * BK::BYTES;
      load_codes<BITS>(blk, 0, c, c0);
      if constexpr (BITS == 8) {
        load_codes<8>(blk, 1, c, c1);
      } else {
        c1.a = *reinterpret_cast<const uint4*>(blk + 16 * (128 + c));
        c1.meta = c0.meta;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_t[s]);  // the block is read; the MMAs commit the rest
      // A slot a was last read by stage i - SA, whose MMAs complete the phase of its ring slot
      // (that slot cannot move on before this warp's arrival for stage i - SA + ST > i)
      if (i >= SA && !wait(&empty_t[(i - SA) % ST], static_cast<uint32_t>(((i - SA) / ST) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();  // the TMEM stores below come after the slot's previous MMAs
      uint32_t v[16];
      convert_codes<BITS, kBF>(c0, v);
      tmem_st16(tcol + lane_addr + 32u + static_cast<uint32_t>(32 * a), v);
      convert_codes<BITS, kBF>(c1, v);
      tmem_st16(tcol + lane_addr + 48u + static_cast<uint32_t>(32 * a), v);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_a[a]);
    }
    if (pipe == 0) {
      // Finish: column c's BT sums over the pipelines (in order), pushed to the rank that
      // finishes column c, or added there.
      float acc[BT];
#pragma unroll
      for (int j = 0; j < BT; ++j) acc[j] = 0.f;
      for (int j = 0; j < P; ++j) {
        if (ok) ok = wait(bars_all + j * NB + CF::ACC, 0u);
        tc_fence_after();
        const int nj = kr0 + kr * (j + 1) / P - (kr0 + kr * j / P);  // pipeline j's stages
        uint32_t v[32];
        const uint32_t ta = tmem_base + static_cast<uint32_t>(j * (CF::COLS / P)) + lane_addr;
        if constexpr (BT == 32) {
          tmem_ld32_nowait(ta, v);
        } else {
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
              : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
              : "r"(ta)
              : "memory");
#pragma unroll
          for (int jj = 16; jj < 32; ++jj) v[jj] = 0u;
        }
        tmem_wait_ld(v);
        if (ok && nj > 0) {
#pragma unroll
          for (int jj = 0; jj < BT; ++jj) acc[jj] += __uint_as_float(v[jj]);
        }
      }
      const int wmax = (kTN + cs - 1) / cs;
      const bool mine = c >= own_lo && c < own_hi;
      if (!mine) {
        int r = c * cs / kTN;  // the rank whose columns hold c
        while (kTN * (r + 1) / cs <= c) ++r;
        while (kTN * r / cs > c) --r;
        const uint32_t rbar = cluster_addr(recv_bar, static_cast<uint32_t>(r));
        const uint32_t rdst = cluster_addr(recv + (rank * wmax + (c - kTN * r / cs)) * CF::RECV_PITCH,
                                           static_cast<uint32_t>(r));
#pragma unroll
        for (int j = 0; j < BT; j += 4)
          st_async_v4_at(rdst + static_cast<uint32_t>(4 * j), rbar, __float_as_uint(acc[j]),
                         __float_as_uint(acc[j + 1]), __float_as_uint(acc[j + 2]), __float_as_uint(acc[j + 3]));
      } else {
        bool have = true;
        if (cs > 1) {
          have = mbar_try_wait_cl(recv_bar, 0u);
          if (!have && *abort_flag == 0u) {
            const uint64_t t0 = globaltimer_ns();
            while (!(have = mbar_try_wait_cl(recv_bar, 0u))) {
              if (globaltimer_ns() - t0 > kWaitLimitNs) {
                atomicOr(p.status, kStatusPackedTimeout);
                *abort_flag = 1u;
                break;
              }
            }
          }
        }
        const int n = nt * kTN + c;
        if (have && n < p.N) {
          float sum[BT];
#pragma unroll
          for (int j = 0; j < BT; ++j) sum[j] = 0.f;
          for (int r = 0; r < cs; ++r) {  // rank order
            if (r == rank) {
#pragma unroll
              for (int j = 0; j < BT; ++j) sum[j] += acc[j];
            } else {
              const float* src = recv + (r * wmax + (c - own_lo)) * CF::RECV_PITCH;
#pragma unroll
              for (int j = 0; j < BT; j += 4) {
                const float4 q4 = *reinterpret_cast<const float4*>(src + j);
                sum[j] += q4.x;
                sum[j + 1] += q4.y;
                sum[j + 2] += q4.z;
                sum[j + 3] += q4.w;
              }
            }
          }
          const float bias = p.bias != nullptr ? load_bias<kBF>(p.bias, n) : 0.f;
          uint16_t* yp = reinterpret_cast<uint16_t*>(p.y) + static_cast<size_t>(m0) * p.N + n;
#pragma unroll
          for (int j = 0; j < BT; ++j)
            if (m0 + j < p.M) yp[static_cast<size_t>(j) * p.N] = float_to_elem<kBF>(sum[j] + bias);
        }
      }
    }
  }

  // no rank leaves while another may still push into its shared memory (its owners waited,
  // bounded, for every push), and TMEM is freed after every MMA completed
  __syncthreads();
  if (cs > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "n"(CF::COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ pair mode ----
// Large M: a cluster of two CTAs shares one tile of 256 output columns (M = 256 of
// tcgen05.mma.cta_group::2: each CTA dequantizes its own 128 columns, its own column tile of
// the packed layout, into its own TMEM) by 256 activation rows (N = 256: each CTA loads its
// own 128 rows, so each SM's shared memory carries half the activations per MMA of the
// single-CTA kernel).  CTA 0 issues the MMAs and commits to the barriers of both CTAs; the
// dequant and epilogue warps of CTA 1 arrive on CTA 0's barriers.  Each CTA's TMEM holds the
// accumulator rows of its own columns.
template <int BITS = 4>
struct PairCfg {
  static constexpr int BT = 256;
  static constexpr int XH_BYTES = (BT / 2) * kTK * 2;  // this CTA's half of the activation tile
  static constexpr int BLK = Blk<BITS>::BYTES;
  static constexpr int STAGE = XH_BYTES + BLK;
  static constexpr int SA_FIT = (512 - BT) / 32;
  static constexpr int ST_FIT = (kSmemCap - 2048) / STAGE;
  static constexpr int ST0 = ST_FIT < SA_FIT ? ST_FIT : SA_FIT;
  static constexpr int ST = ST0 < 8 ? ST0 : 8;
  static constexpr int X_OFF = 0;
  static constexpr int B_OFF = ST * XH_BYTES;
  static constexpr int BAR_OFF = B_OFF + ST * BLK;
  // full_t[ST], empty[ST], full_a[ST], acc_full, acc_empty, drain
  static constexpr int NBARS = 3 * ST + 3;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr int SIG_OFF = MISC_OFF + 16;         // CTA 0: targets of CTA 1's signals
  static constexpr int YST_OFF = ((SIG_OFF + 4 * kDQ + 15) / 16) * 16;  // y staging, 1 KB a warp
  static constexpr int USED = 1024 + YST_OFF + 4 * 1024;
  static constexpr int SMEM = USED < kSmemMin ? kSmemMin : USED;
  static constexpr uint32_t A_COL0 = BT;
  static_assert(ST >= 3 && SMEM <= kSmemCap, "resources");
  static_assert(BT + ST * 32 <= 512, "TMEM columns");
};
// kind::f16, fp32 accumulate, fp16 A (TMEM) and B (K-major), N = 256, M = 256.
constexpr uint32_t kIdescPair = (1u << 4) | (static_cast<uint32_t>(256 >> 3) << 17) |
                                (static_cast<uint32_t>(256 >> 4) << 24);

template <bool kBF, int BITS = 4>
__global__ void __launch_bounds__(kThreads, 1) packed_pair_kernel(const __grid_constant__ PackedParams p) {
  using CF = PairCfg<BITS>;
  using BK = Blk<BITS>;
  static_assert(BITS == 4 || (BITS == 8 && !kBF), "8-bit codes: fp16 only");
  constexpr int ST = CF::ST, BT = CF::BT;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CF::BAR_OFF);
  uint64_t* full_t = bars;            // this CTA's activation half + packed block landed
  uint64_t* empty = bars + ST;        // slot free: block read here, the pair's MMAs done
  uint64_t* full_a = bars + 2 * ST;   // CTA 0 only: both CTAs' A operands of the slot in TMEM
  uint64_t* acc_full = bars + 3 * ST;
  uint64_t* acc_empty = acc_full + 1; // CTA 0 only: both CTAs' epilogues read the accumulator
  uint64_t* drain = acc_empty + 1;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + CF::MISC_OFF);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + CF::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KS = p.K / kTK;
  const uint32_t rank = cluster_ctarank();
  const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full_t[s], 1);
      mbar_init(&empty[s], kDQ + 1);   // this CTA's dequant warps + CTA 0's commit
      // CTA 0's dequant warps (one of them also expects the 4-byte signals of CTA 1's eight)
      mbar_init(&full_a[s], kDQ);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 8);           // the epilogue warps of both CTAs
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {  // one warp of each CTA of the pair, collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(const_cast<uint32_t*>(tmem_slot)))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, p.status, kStatusPackedTimeout, kWaitLimitNs)) return true;
    *abort_flag = 1u;
    return false;
  };
  auto wait_cl = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if (*abort_flag) return false;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_cl(bar, parity)) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(p.status, kStatusPackedTimeout);
        *abort_flag = 1u;
        return false;
      }
    }
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_x);
      const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < p.tiles; tile += npairs) {
        const int m0 = (tile % p.tiles_t) * BT + static_cast<int>(rank) * (BT / 2);
        const int t = (tile / p.tiles_t) * 2 + static_cast<int>(rank);
        const uint32_t* src = p.packed + static_cast<size_t>(t) * KS * BK::WORDS;
        for (int kb = 0; kb < KS; ++kb) {
          if (!wait(&empty[s], ph ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(&full_t[s], static_cast<uint32_t>(CF::XH_BYTES + BK::BYTES));
          tma_load_2d_hint(smem + CF::X_OFF + s * CF::XH_BYTES, &p.tm_x, &full_t[s], kb * kTK, m0, pol_x);
          bulk_load(smem + CF::B_OFF + s * BK::BYTES, src + static_cast<size_t>(kb) * BK::WORDS,
                    BK::BYTES, &full_t[s], pol_w);
          ++issued;
          if (++s == ST) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {
        for (int i = 0; i < ST && i < issued; ++i) {
          if (--s < 0) { s = ST - 1; ph ^= 1u; }
          mbar_wait_bounded(&full_t[s], ph, p.status, kStatusPackedTimeout, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (CTA 0)
    if (lane == 0 && rank == 0) {
      int s = 0, li = 0;
      uint32_t ph = 0;
      bool ok = true, any = false;
      for (int tile = pair; ok && tile < p.tiles; tile += npairs, ++li) {
        if (!wait_cl(acc_empty, static_cast<uint32_t>((li & 1) ^ 1))) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < KS; kb += 2) {
          // Both CTAs' A operands of a pair of stages (their dequant warps waited for their
          // activation halves first): one wait on the later stage's full_a covers both (the
          // warps of CTA 0 arrive in stage order, CTA 1 signals once per pair, after its
          // stores of both stages).
          const int n2 = KS - kb < 2 ? KS - kb : 2;
          const int sl = s + n2 - 1 < ST ? s + n2 - 1 : s + n2 - 1 - ST;
          const uint32_t phl = s + n2 - 1 < ST ? ph : ph ^ 1u;
          if (!wait_cl(&full_a[sl], phl)) { ok = false; break; }
          tc_fence_after();
          for (int i = 0; i < n2; ++i) {
            const uint32_t a = tmem_base + CF::A_COL0 + static_cast<uint32_t>(s * 32);
            const uint64_t bdesc = sw128_kmajor_desc(sbase + CF::X_OFF + s * CF::XH_BYTES);
#pragma unroll
            for (int ks = 0; ks < kTK / 16; ++ks)
              mma_ts_pair(tmem_base, a + 8u * ks, bdesc + 2u * ks, kIdescPair | (kBF ? kIdescBF : 0u),
                          (kb + i > 0 || ks > 0) ? 1u : 0u);
            mma_commit_pair(&empty[s]);
            if (++s == ST) { s = 0; ph ^= 1u; }
          }
          any = true;
        }
        if (!ok) break;
        mma_commit_pair(acc_full);
      }
      if (any) {  // every MMA completes (in both CTAs) before TMEM is released
        mma_commit_pair(drain);
        mbar_wait_bounded(drain, 0u, p.status, kStatusPackedTimeout, kWaitLimitNs);
      }
    } else if (lane == 0 && pair < p.tiles) {
      // CTA 1: CTA 0's MMAs read this CTA's shared memory and TMEM until the last commit
      mbar_wait_bounded(drain, 0u, p.status, kStatusPackedTimeout, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp < 2 + kDQ) {
    // ------------------------------------------------------------------ dequant
    // As in the single-CTA kernel (thread = output column of this CTA's tile, K half h).
    // Readiness goes to CTA 0's full_a: an arrival from CTA 0's warps, a counted asynchronous
    // store from CTA 1's (a remote arrive would stall the warp for over a thousand cycles).
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int c = 32 * q + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = pair; ok && tile < p.tiles; tile += npairs) {
      for (int kb = 0; kb < KS; ++kb) {
        if (!wait(&full_t[s], ph)) { ok = false; break; }
        tc_fence_after();
        StageCodes<BITS> cd;
        load_codes<BITS>(smem + CF::B_OFF + s * BK::BYTES, h, c, cd);
        uint32_t v[16];
        convert_codes<BITS, kBF>(cd, v);
        tmem_st16(tmem_base + lane_addr + CF::A_COL0 + static_cast<uint32_t>(s * 32 + 16 * h), v);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // the MMA waits on the second stage of each pair (or a tile's last, unpaired stage)
          const bool sig = (kb & 1) || kb + 1 == KS;
          if (rank == 0) {
            if (warp == 2 && sig) mbar_arrive_expect_tx(&full_a[s], 4u * kDQ);
            else mbar_arrive(&full_a[s]);
          } else if (sig) {
            st_async_signal(smem + CF::SIG_OFF + 4 * (warp - 2), &full_a[s], 0u);
          }
          mbar_arrive(&empty[s]);
        }
        if (++s == ST) { s = 0; ph ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int nl = 32 * q + lane;
    __half* ystage = p.y_vec != 0 ? reinterpret_cast<__half*>(smem + CF::YST_OFF) + q * 512 : nullptr;
    int li = 0;
    for (int tile = pair; tile < p.tiles; tile += npairs, ++li) {
      const int m0 = (tile % p.tiles_t) * BT;
      const int n = ((tile / p.tiles_t) * 2 + static_cast<int>(rank)) * kTN + nl;
      const int mlim = p.M;
      const float bias = (p.bias != nullptr && n < p.N) ? load_bias<kBF>(p.bias, n) : 0.f;
      if (!wait(acc_full, static_cast<uint32_t>(li & 1))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
      uint32_t va[32], vb[32];
      if (ystage != nullptr) {  // MMA-fragment loads, stmatrix into the staging tile, 16-byte stores
        const int c0 = n - lane;
        float ba[2], bb[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int na = c0 + 16 * h + (lane >> 2), nb = na + 8;
          ba[h] = (p.bias != nullptr && na < p.N) ? load_bias<kBF>(p.bias, na) : 0.f;
          bb[h] = (p.bias != nullptr && nb < p.N) ? load_bias<kBF>(p.bias, nb) : 0.f;
        }
        tmem_ld16x256_nowait(taddr, va);
        tmem_ld16x256_nowait(taddr + (16u << 16), va + 16);
        tmem_wait_ld(va);
#pragma unroll
        for (int cc = 0; cc < BT / 32; ++cc) {
          uint32_t (&cur)[32] = (cc & 1) ? vb : va;
          uint32_t (&nxt)[32] = (cc & 1) ? va : vb;
          if (cc + 1 < BT / 32) {
            tmem_ld16x256_nowait(taddr + 32 * (cc + 1), nxt);
            tmem_ld16x256_nowait(taddr + (16u << 16) + 32 * (cc + 1), nxt + 16);
          }
          store_y32_frag<kBF>(p, ystage, cur, ba, bb, m0 + 32 * cc, c0, lane, mlim);
          if (cc + 1 < BT / 32) tmem_wait_ld(nxt);
        }
      } else {
        tmem_ld32_nowait(taddr, va);
        tmem_wait_ld(va);
#pragma unroll
        for (int cc = 0; cc < BT / 32; ++cc) {
          uint32_t (&cur)[32] = (cc & 1) ? vb : va;
          uint32_t (&nxt)[32] = (cc & 1) ? va : vb;
          if (cc + 1 < BT / 32) tmem_ld32_nowait(taddr + 32 * (cc + 1), nxt);
          store_y32<kBF>(p, nullptr, cur, bias, m0 + 32 * cc, n - lane, lane, mlim);
          if (cc + 1 < BT / 32) tmem_wait_ld(nxt);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_at(acc_empty, 0u);
    }
  }

  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still arrive on its barriers
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(tmem_base) : "memory");
  }
}

template <bool kBF, int BITS>
cudaError_t launch_pair(const PackedParams& base, const GemmProblem& p) {
  using CF = PairCfg<BITS>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int cap = 0;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(packed_pair_kernel<kBF, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
    if (attr_err != cudaSuccess) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = CF::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&cap, packed_pair_kernel<kBF, BITS>, &cfg) != cudaSuccess) cap = 0;
    (void)cudaGetLastError();
  });
  if (attr_err != cudaSuccess) return attr_err;
  if (cap <= 0) return cudaErrorInvalidConfiguration;
  PackedParams pp = base;
  const char* why = nullptr;
  if (!make_tmap_2d(&pp.tm_x, kBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.x, p.K, p.M, kTK, CF::BT / 2,
                    CU_TENSOR_MAP_SWIZZLE_128B, &why))
    return cudaErrorInvalidValue;
  pp.tiles_t = (p.M + CF::BT - 1) / CF::BT;
  const long long tiles = static_cast<long long>(pp.tiles_t) * ((p.N + 2 * kTN - 1) / (2 * kTN));
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  pp.tiles = static_cast<int>(tiles);
  const int clusters = pp.tiles < cap ? pp.tiles : cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = CF::SMEM;
  cfg.stream = p.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, packed_pair_kernel<kBF, BITS>, pp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BT, int SPLIT, bool kBF, int BITS>
cudaError_t launch_bt(const PackedParams& base, const GemmProblem& p) {
  using CF = Cfg<BT, SPLIT, BITS>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(packed_kernel<BT, SPLIT, false, kBF, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  PackedParams pp = base;
  const char* why = nullptr;
  if (!make_tmap_2d(&pp.tm_x, kBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.x, p.K, p.M, kTK, BT,
                    CU_TENSOR_MAP_SWIZZLE_128B, &why))
    return cudaErrorInvalidValue;
  pp.tiles_t = (p.M + BT - 1) / BT;
  const long long tiles = static_cast<long long>(pp.tiles_t) * ((p.N + kTN - 1) / kTN);
  if (tiles * SPLIT > 0x7fffffffLL) return cudaErrorInvalidValue;
  pp.tiles = static_cast<int>(tiles);
  if (SPLIT == 1) {  // persistent over the tiles, as many CTAs as are resident at once
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int cap = (CF::kNarrow ? 2 : 1) * sms;
    const int grid = pp.tiles < cap ? pp.tiles : cap;
    packed_kernel<BT, SPLIT, false, kBF, BITS><<<grid, kThreads, CF::SMEM, p.stream>>>(pp);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pp.tiles * SPLIT), 1, 1);  // one tile per cluster
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = CF::SMEM;
  cfg.stream = p.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = SPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, packed_kernel<BT, SPLIT, false, kBF, BITS>, pp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Small-batch launch (M <= 32, 4-bit).  Clusters of c CTAs placeable at one CTA per SM come
// from the occupancy API on the four-pipeline kernel (whose resources allow one per SM; the
// API reports one per SM for every kernel that allocates tensor memory, so the two-pipeline
// kernel counts twice that, as measured).  Per variant the cluster size is the largest
// (at most kSmallMaxCS and the stage count) whose grid of tiles x c CTAs is resident in one
// wave; the variant is the one whose busiest SM has the least work: four pipelines each take
// about 800 cycles a stage when four share an SM, two alone about 650.
struct SmallPlan {
  int np = 4, cs = 1;
};
template <int BT, int NP, bool kBF, int BITS>
cudaError_t small_attrs(int dev) {
  using CF = SmallCfg<BT, NP, BITS>;
  static std::mutex mu;
  static bool set[64];
  std::lock_guard<std::mutex> lock(mu);
  if (set[dev]) return cudaSuccess;
  auto kern = packed_small_kernel<BT, NP, kBF, BITS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) set[dev] = true;
  return e;
}
template <int BT, bool kBF, int BITS>
cudaError_t small_plan(int dev, long long tiles, int KS, int sms, SmallPlan* out) {
  using C4 = SmallCfg<BT, 4, BITS>;
  constexpr bool kTwo = SmallCfg<BT, 2, BITS>::FITS;
  static std::mutex mu;
  static int fits[64][kSmallMaxCS + 1];  // clusters of c CTAs x c at one CTA per SM (0: not asked)
  cudaError_t e = small_attrs<BT, 4, kBF, BITS>(dev);
  if constexpr (kTwo)
    if (e == cudaSuccess) e = small_attrs<BT, 2, kBF, BITS>(dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int c = 1; c <= kSmallMaxCS && c <= KS; ++c) {
    if (fits[dev][c] != 0) continue;
    if (c == 1) { fits[dev][c] = sms; continue; }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c), 1, 1);
    cfg.blockDim = dim3(C4::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C4::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(c);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, packed_small_kernel<BT, 4, kBF, BITS>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    fits[dev][c] = n > 0 ? n * c : -1;
  }
  double best = 0.0;
  for (int np : {4, 2}) {
    if (np == 2 && !kTwo) continue;
    const int per_sm = 4 / np;
    int cs = 1;
    for (int c = 2; c <= kSmallMaxCS && c <= KS; ++c)
      if (fits[dev][c] > 0 && tiles * c <= static_cast<long long>(per_sm) * fits[dev][c]) cs = c;
    const long long ctas = tiles * cs;
    const double waves = static_cast<double>((ctas + static_cast<long long>(per_sm) * sms - 1) / (static_cast<long long>(per_sm) * sms));
    const double stages = static_cast<double>((KS + cs - 1) / cs);
    // cycles on the busiest SM: four pipelines at ~800 a stage; two alone at ~650
    const bool shared = np == 4 || ctas > sms;
    const double cost = waves * stages * (np == 4 ? 200.0 : (shared ? 400.0 : 325.0));
    if (np == 4 || cost < best) {
      best = cost;
      out->np = np;
      out->cs = cs;
    }
  }
  return cudaSuccess;
}

template <int BT, int NP, bool kBF, int BITS>
cudaError_t launch_small_np(const PackedParams& pp, const GemmProblem& p, int cs) {
  using CF = SmallCfg<BT, NP, BITS>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(pp.tiles) * cs), 1, 1);
  cfg.blockDim = dim3(CF::THREADS, 1, 1);
  cfg.dynamicSmemBytes = CF::SMEM;
  cfg.stream = p.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, packed_small_kernel<BT, NP, kBF, BITS>, pp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BT, bool kBF, int BITS>
cudaError_t launch_small(const PackedParams& base, const GemmProblem& p) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  PackedParams pp = base;
  const char* why = nullptr;
  if (!make_tmap_2d(&pp.tm_x, kBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.x, p.K, p.M, kTK, BT,
                    CU_TENSOR_MAP_SWIZZLE_128B, &why))
    return cudaErrorInvalidValue;
  pp.tiles_t = (p.M + BT - 1) / BT;
  const long long tiles = static_cast<long long>(pp.tiles_t) * ((p.N + kTN - 1) / kTN);
  if (tiles * kSmallMaxCS > 0x7fffffffLL) return cudaErrorInvalidValue;
  pp.tiles = static_cast<int>(tiles);
  SmallPlan pl;
  e = small_plan<BT, kBF, BITS>(dev, tiles, p.K / kTK, sms, &pl);
  if (e != cudaSuccess) return e;
  if constexpr (SmallCfg<BT, 2, BITS>::FITS)
    if (pl.np == 2) return launch_small_np<BT, 2, kBF, BITS>(pp, p, pl.cs);
  return launch_small_np<BT, 4, kBF, BITS>(pp, p, pl.cs);
}

// Stream-K launch (256-row tiles): one CTA per SM, at least kSkMinUnits stages each.
size_t sk_flag_bytes(int sms) { return (static_cast<size_t>(sms) * 4 + 255) / 256 * 256; }

template <bool kBF, int BITS>
cudaError_t launch_sk(const PackedParams& base, const GemmProblem& p, void* workspace, int sms) {
  using CF = Cfg<kSkRows, 1, BITS>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(packed_kernel<kSkRows, 1, true, kBF, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    CF::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  PackedParams pp = base;
  const char* why = nullptr;
  if (!make_tmap_2d(&pp.tm_x, kBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.x, p.K, p.M, kTK, kSkRows,
                    CU_TENSOR_MAP_SWIZZLE_128B, &why))
    return cudaErrorInvalidValue;
  pp.tiles_t = (p.M + kSkRows - 1) / kSkRows;
  const long long tiles = static_cast<long long>(pp.tiles_t) * ((p.N + kTN - 1) / kTN);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  pp.tiles = static_cast<int>(tiles);
  pp.units = tiles * (p.K / kTK);
  long long grid = pp.units / kSkMinUnits;
  if (grid > sms) grid = sms;
  if (grid < 1) grid = 1;
  pp.flags = static_cast<unsigned int*>(workspace);
  pp.partial = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + sk_flag_bytes(sms));
  packed_kernel<kSkRows, 1, true, kBF, BITS><<<static_cast<unsigned>(grid), kThreads, CF::SMEM, p.stream>>>(pp);
  return cudaGetLastError();
}

// Whether a launch with M > 128 rows takes the stream-K kernel, by estimated time in stage
// periods: the persistent launch needs rounds x K/64 of them (x 0.85 for the pair kernel, its
// measured time per stage against the single-CTA kernel's on the 7B linears at M = 2048);
// stream-K needs ceil(units / SMs) plus kSkOverheadStages (partial sums, the finishers' tails:
// about 16 us, 37 stage periods, on GB300 at 512 x 4096 x 11008, where it ran 47.7 against
// 50.2 us; 45.5 against 64.0 at 512 x 11008 x 4096; slower at M = 2048 on both 7B shapes).
constexpr int kSkOverheadStages = 40;
bool use_stream_k(int M, int K, int N, int sms, bool pair) {
  const long long KS = K / kTK;
  const long long NT = (N + kTN - 1) / kTN;
  const long long tiles = static_cast<long long>((M + kSkRows - 1) / kSkRows) * NT;
  const long long units = tiles * KS;
  if (units < static_cast<long long>(sms) * kSkMinUnits) return false;
  const long long work = pair ? tiles / 2 : tiles;   // pair tiles span two column tiles
  const long long slots = pair ? sms / 2 : sms;
  const double persistent = static_cast<double>((work + slots - 1) / slots * KS) * (pair ? 0.85 : 1.0);
  const double stream_k = static_cast<double>((units + sms - 1) / sms + kSkOverheadStages);
  return stream_k < persistent;
}

// Token tile and K split of a launch with M <= 128 rows: the narrowest tile holding M rows
// (32, 64 or 128), and the largest split (2 or 4 for 32 rows, 2 for 64 and 128) that keeps
// every CTA resident in one wave (two CTAs per SM below 128-row tiles) with at least four
// stages each.  (Launches of at most 32 rows take the small-batch kernel instead.)
struct PackedPlan {
  int bt = 256, split = 1;
};
PackedPlan packed_plan(int M, int K, int N, int sms) {
  PackedPlan pl;
  if (M > 128) return pl;
  pl.bt = M <= 32 ? 32 : M <= 64 ? 64 : 128;
  const long long tiles = static_cast<long long>((M + pl.bt - 1) / pl.bt) * ((N + kTN - 1) / kTN);
  const long long cap = static_cast<long long>(pl.bt <= 64 ? 2 : 1) * sms;
  const int KS = K / kTK;
  for (int split : {2, 4}) {
    if (split == 4 && pl.bt != 32) continue;
    if (KS / split < 4 || tiles * split > cap) continue;
    pl.split = split;
  }
  return pl;
}

// The plan of one launch (token tile, K split, stream-K or the pair kernel) and the launch.
template <bool kBF, int BITS>
cudaError_t launch_planned(const PackedParams& pp, const GemmProblem& p, void* workspace, size_t workspace_bytes,
                           int sms) {
  const PackedPlan pl = packed_plan(p.M, p.K, p.N, sms);
  if (p.M <= 32) return p.M <= 16 ? launch_small<16, kBF, BITS>(pp, p) : launch_small<32, kBF, BITS>(pp, p);
  if (pl.bt == 32)
    return pl.split == 4 ? launch_bt<32, 4, kBF, BITS>(pp, p) : pl.split == 2 ? launch_bt<32, 2, kBF, BITS>(pp, p) : launch_bt<32, 1, kBF, BITS>(pp, p);
  if (pl.bt == 64) return pl.split == 2 ? launch_bt<64, 2, kBF, BITS>(pp, p) : launch_bt<64, 1, kBF, BITS>(pp, p);
  if (pl.bt == 128) return pl.split == 2 ? launch_bt<128, 2, kBF, BITS>(pp, p) : launch_bt<128, 1, kBF, BITS>(pp, p);
  // Pairs of column tiles (the packed layout holds ceil(N / 128) of them) for long K: sustained
  // under the power cap the pair kernel ran 1508 against 1460 TFLOP/s on the 70B linears at
  // M = 4096 (it moves half the activations per SM, so it clocks higher at the same power);
  // at K = 4096 the single-CTA kernel was ahead (1374 against 1343 on the 7B linears).
  const bool pair = p.K >= kPairMinK && ((p.N + kTN - 1) / kTN) % 2 == 0;
  if (workspace != nullptr && workspace_bytes >= packed_workspace_bytes(sms) &&
      use_stream_k(p.M, p.K, p.N, sms, pair))
    return launch_sk<kBF, BITS>(pp, p, workspace, sms);
  if (pair) return launch_pair<kBF, BITS>(pp, p);
  return launch_bt<256, 1, kBF, BITS>(pp, p);
}

}  // namespace

bool packed8_supported(int64_t K, int64_t N, int64_t G, const char** why) {
  static const char* dummy;
  if (!why) why = &dummy;
  if (K % kTK != 0) { *why = "the tile-packed layout needs K % 64 == 0"; return false; }
  if (G % kTK != 0) { *why = "the tile-packed layout needs group_size % 64 == 0 (or -1)"; return false; }
  if (N % 4 != 0) { *why = "N must be a multiple of 4"; return false; }
  return true;
}

size_t packed8_bytes(int64_t K, int64_t N) {
  return static_cast<size_t>((N + kTN - 1) / kTN) * static_cast<size_t>(K / kTK) * Blk<8>::BYTES;
}

cudaError_t launch_repack8(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int N, int G,
                           void* out, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(K / kTK), static_cast<unsigned>((N + kTN - 1) / kTN));
  repack8_kernel<<<grid, 128, 0, stream>>>(qw, qz, reinterpret_cast<const uint16_t*>(sc),
                                           static_cast<uint32_t*>(out), K, N, G);
  return cudaGetLastError();
}

bool packed_supported(int64_t K, int64_t N, int64_t G, const char** why) {
  static const char* dummy;
  if (!why) why = &dummy;
  if (K % kTK != 0) { *why = "the tile-packed layout needs K % 64 == 0"; return false; }
  if (G % kTK != 0) { *why = "the tile-packed layout needs group_size % 64 == 0 (or -1)"; return false; }
  if (N % 8 != 0) { *why = "N must be a multiple of 8"; return false; }
  return true;
}

size_t packed_bytes(int64_t K, int64_t N) {
  return static_cast<size_t>((N + kTN - 1) / kTN) * static_cast<size_t>(K / kTK) * kBlockBytes;
}

cudaError_t launch_repack(const uint32_t* qw, const uint32_t* qz, const __half* sc, int K, int N,
                          int G, void* out, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(K / kTK), static_cast<unsigned>((N + kTN - 1) / kTN));
  repack_kernel<<<grid, 128, 0, stream>>>(qw, qz, reinterpret_cast<const uint16_t*>(sc),
                                          static_cast<uint32_t*>(out), K, N, G);
  return cudaGetLastError();
}

size_t packed_workspace_flag_bytes(int sms) { return sk_flag_bytes(sms); }

namespace {
template <bool kBF>
cudaError_t launch_grouped_t(const GemmProblem& p, const void* packed) {
  using CF = Cfg<256, 1, 4>;
  static_assert(CF::USED + kGrpBytes <= kSmemCap, "grouped: tile-start table after the ring");
  constexpr int kSmem = CF::SMEM + kGrpBytes;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(packed_kernel<256, 1, false, kBF, 4, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  PackedParams pp{};
  pp.packed = static_cast<const uint32_t*>(packed);
  pp.bias = p.bias;
  pp.y = p.y;
  cudaError_t e = status_word_ptr(&pp.status);
  if (e != cudaSuccess) return e;
  pp.M = p.M; pp.K = p.K; pp.N = p.N;
  pp.y_vec = (aligned(p.y, 16) && p.N % 8 == 0) ? 1 : 0;
  const char* why = nullptr;
  if (!make_tmap_2d(&pp.tm_x, kBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    p.x, p.K, p.M, kTK, 256, CU_TENSOR_MAP_SWIZZLE_128B, &why))
    return cudaErrorInvalidValue;
  const int NT = (p.N + kTN - 1) / kTN, KS = p.K / kTK;
  pp.offsets = p.offsets;
  pp.E = p.E;
  pp.grp_nt = NT;
  pp.expert_words = static_cast<size_t>(NT) * KS * Blk<4>::WORDS;
  const long long tmax = (static_cast<long long>(p.M + 255) / 256 + p.E) * NT;  // tiles at most
  if (tmax > 0x7fffffffLL) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long grid = tmax < sms ? tmax : sms;
  packed_kernel<256, 1, false, kBF, 4, true><<<static_cast<unsigned>(grid), kThreads, kSmem, p.stream>>>(pp);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_packed_grouped(const GemmProblem& p, const void* packed) {
  return p.bf16 ? launch_grouped_t<true>(p, packed) : launch_grouped_t<false>(p, packed);
}

size_t packed_workspace_bytes(int sms) {
  return sk_flag_bytes(sms) + static_cast<size_t>(sms) * kSkSlotBytes;
}

// Fixed device scratch for awq_gemm_packed_noalloc: the stream-K workspace of a device with up
// to 159 SMs (768 bytes of flags + 159 x 128 KB), reserved with the module, so that entry point
// needs no allocation.  One array per device context, shared by every call on that device.
namespace {
constexpr size_t kStaticScratchBytes = 20u << 20;
static __device__ __align__(256) unsigned char g_packed_scratch[kStaticScratchBytes];
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];
}  // namespace

size_t packed_static_scratch_bytes() { return kStaticScratchBytes; }

cudaError_t packed_static_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // the symbol's address on this device, looked up once with the device current
  std::call_once(g_scratch_once[dev], [dev] {
    g_scratch_err[dev] = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_packed_scratch);
  });
  if (g_scratch_err[dev] != cudaSuccess) return g_scratch_err[dev];
  *ptr = g_scratch_ptr[dev];
  return cudaSuccess;
}

cudaError_t launch_packed(const GemmProblem& p, const void* packed, void* workspace, size_t workspace_bytes) {
  PackedParams pp{};
  pp.packed = static_cast<const uint32_t*>(packed);
  pp.bias = p.bias;
  pp.y = p.y;
  cudaError_t e = status_word_ptr(&pp.status);
  if (e != cudaSuccess) return e;
  pp.M = p.M; pp.K = p.K; pp.N = p.N;
  // 16-byte stores of y need a 16-byte aligned base and rows of whole 16-byte pieces (N % 8
  // == 0: always for 4-bit codes; 8-bit codes allow N % 4 == 0, whose y takes 2-byte stores)
  pp.y_vec = (aligned(p.y, 16) && p.N % 8 == 0) ? 1 : 0;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (p.bits == 8) return launch_planned<false, 8>(pp, p, workspace, workspace_bytes, sms);
  return p.bf16 ? launch_planned<true, 4>(pp, p, workspace, workspace_bytes, sms)
                : launch_planned<false, 4>(pp, p, workspace, workspace_bytes, sms);
}

}  // namespace awq
