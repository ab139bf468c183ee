/*
 * awq.h -- C ABI of libawq_gb300.so: AWQ W4A16 weight-only linear on GB300 (sm_103a).
 *
 * The weight layout is the AWQ "GEMM" checkpoint pack (tensref.org/formats/awq,
 * "Reader" pseudo-code; GPTQModel wiki "AWQ", "Saved formats and packing"):
 *
 *   qweight int32 [K, N/8]    row-major; nibble i (bits 4i..4i+3) of word c in row k
 *                             holds the 4-bit code of output column 8c + ORDER[i],
 *                             ORDER = {0,2,4,6,1,3,5,7}
 *   qzeros  int32 [K/G, N/8]  zero points, packed exactly like qweight
 *   scales  fp16  [K/G, N]    row-major
 *   bias    fp16  [N]         optional
 *
 * with K = in_features, N = out_features, G = group_size (G = K when group_size is -1:
 * one group across the row, GPTQModel wiki "AWQ", "Group quantization and zero points").
 * Every weight is  w[k][n] = (code[k][n] - zero[k/G][n]) * scale[k/G][n]  with the zero
 * used as stored (no +1; format page, reject rule AWQ-005).
 *
 * Conventions shared by every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller, dense and row-major.  The
 *    library never frees or retains them and allocates no device memory per call.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream) and never
 *    synchronize.  Argument errors are found on the host BEFORE any launch and returned
 *    synchronously; nothing is launched then.
 *  - On failure the call returns a non-zero awq_status_t and awq_last_error() holds a
 *    message for the calling thread.  On success awq_last_error() returns "".
 *  - Launch failures (cudaGetLastError after the launch) return AWQ_ERR_CUDA with the CUDA
 *    error string.
 *  - The library is built for compute capability 10.3 only; on another device every
 *    compute entry point returns AWQ_ERR_UNSUPPORTED_DEVICE.
 *  - Sizes are int64; each of M, K, N must be below 2^31, and M*N, K*N below 2^40.
 */
#ifndef AWQ_GB300_H
#define AWQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* awq_stream_t;

typedef enum awq_status {
  AWQ_OK = 0,
  AWQ_ERR_INVALID_ARGUMENT = 1,  /* null pointer, negative size, bad group_size, bad enum */
  AWQ_ERR_UNSUPPORTED_SHAPE = 2, /* N not a multiple of 8, K not a multiple of G, size limits */
  AWQ_ERR_MISALIGNED = 3,        /* a pointer below its element alignment */
  AWQ_ERR_UNSUPPORTED_DEVICE = 4,/* current device is not compute capability 10.3 */
  AWQ_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed */
  AWQ_ERR_TIMEOUT = 6            /* a bounded device-side wait gave up (see awq_device_status) */
} awq_status_t;

typedef enum awq_dtype { AWQ_DTYPE_F16 = 0, AWQ_DTYPE_F32 = 1, AWQ_DTYPE_BF16 = 2 } awq_dtype_t;

/* Kernel family used by awq_gemm_ex.  AUTO picks by M, K, N, G and alignment: decode for
 * M <= 32; above that, when both tensor-core families take the shape, whichever a cost
 * model fitted to GB300 timings predicts faster (decode's 32-row tiles win up to M = 64 ..
 * 192 depending on N and K); else the family whose contract holds, else generic. */
typedef enum awq_path {
  AWQ_PATH_AUTO = 0,
  AWQ_PATH_DECODE = 1,   /* split-K streaming kernel for small M (tensor-core m16n8k16) */
  AWQ_PATH_PREFILL = 2,  /* tcgen05/TMEM tensor-core kernel with TMA-fed tiles, large M */
  AWQ_PATH_GENERIC = 3   /* any valid shape and alignment; slow, used for ragged shapes */
} awq_path_t;

/* 1 when the current CUDA device is compute capability 10.3 and this library's kernels
 * load on it, else 0 (the reason is then in awq_last_error()).  Mirrors the wiki's
 * awq_runtime_available() / awq_runtime_error() pair (GPTQModel wiki "AWQ",
 * "Native AWQ runtime helpers"). */
int awq_runtime_available(void);

/* Thread-local message of the last failing call on this thread; "" after a success. */
const char* awq_last_error(void);

/* Static name of a status code ("AWQ_OK", ...). */
const char* awq_status_string(awq_status_t status);

/*
 * awq_dequant -- unpack and dequantize the whole weight (format page, "Reader"; the
 * wiki's awq_dequantize_weights in "Native AWQ runtime helpers").
 *
 *   w_out[k][n] = (code[k][n] - zero[k/G][n]) * scale[k/G][n]     row-major [K, N]
 *
 * out_dtype AWQ_DTYPE_F32: the exact fp32 value (it is always representable).
 * out_dtype AWQ_DTYPE_F16: that value rounded once, to nearest even.
 * Note the orientation: [K, N] (what x @ W needs); the format page's pseudo-code returns
 * the transpose [N, K].
 * Requirements: K > 0, N >= 0, N % 8 == 0, group_size == -1 or (> 0 and K % group_size
 * == 0); qweight/qzeros 4-byte aligned, scales 2-byte aligned, w_out aligned to its
 * element size.  N == 0 returns AWQ_OK without a launch.  One kernel launch otherwise.
 */
awq_status_t awq_dequant(const int32_t* qweight, const int32_t* qzeros, const void* scales_f16,
                         int64_t K, int64_t N, int64_t group_size,
                         void* w_out, awq_dtype_t out_dtype, awq_stream_t stream);

/*
 * bf16 activations and scales on the same weight layout (the native GEMM kernel's declared
 * contract lists FP16/BF16: GPTQModel wiki "AWQ", "Selection and compatibility", its
 * kernel table; vLLM accepts half and bfloat16: the vLLM article, section 4).  Same contract as awq_gemm_ex / awq_gemm / awq_dequant with
 * bf16 in place of fp16 for x, scales, bias and y (and for w_out when out_dtype is
 * AWQ_DTYPE_BF16):
 *
 *   y[m][n] = bf16_rne( sum_k x[m][k] * w[k][n]  (+ bias[n]) ),  w = (code - zero) * scale
 *
 * fp32 accumulation always.  The decode kernel carries each code into the MMA as the exact
 * bf16 value 128 + c and folds (128 + zero) * sum x out per group; the prefill kernel rounds
 * (c - zero) * scale once to bf16 for its tensor-core operand.  Paths: DECODE needs the
 * TMA decode kernel's contract (K % 64, G % 64, N % 32, 16-byte aligned x, qweight,
 * qzeros, scales); PREFILL as for fp16; GENERIC any valid shape.  AUTO chooses among them.
 * awq_dequant_bf16 writes the exact fp32 value (AWQ_DTYPE_F32) or that value rounded once
 * to bf16 (AWQ_DTYPE_BF16).
 */
awq_status_t awq_gemm_bf16_ex(const void* x_bf16, const int32_t* qweight, const int32_t* qzeros,
                              const void* scales_bf16, const void* bias_bf16, int64_t M, int64_t K,
                              int64_t N, int64_t group_size, void* y_bf16, awq_path_t path,
                              awq_stream_t stream);
awq_status_t awq_gemm_bf16(const void* x_bf16, const int32_t* qweight, const int32_t* qzeros,
                           const void* scales_bf16, const void* bias_bf16, int64_t M, int64_t K,
                           int64_t N, int64_t group_size, void* y_bf16, awq_stream_t stream);
awq_status_t awq_dequant_bf16(const int32_t* qweight, const int32_t* qzeros, const void* scales_bf16,
                              int64_t K, int64_t N, int64_t group_size, void* w_out,
                              awq_dtype_t out_dtype, awq_stream_t stream);

/*
 * 8-bit weights in the GEMM layout (GPTQModel wiki "AWQ", "Saved formats and packing":
 * widths other than 4 pack as a continuous little-endian bit stream, without the INT4
 * order; Marlin-class kernels take 8 bits, "Selection and compatibility").  Column 4c + i of
 * a row is byte i of word c:
 *
 *   qweight int32 [K, N/4], qzeros int32 [K/G, N/4], scales fp16 [K/G, N]
 *   w[k][n] = (code[k][n] - zero[k/G][n]) * scale[k/G][n],  codes 0..255
 *
 * awq_gemm_w8 / awq_gemm_w8_ex: the awq_gemm contract with 8-bit weights (N % 4 == 0).
 * The tensor-core families take 8-bit codes when K % 64 == 0, group_size % 64 == 0,
 * N % 16 == 0 and x, qweight, qzeros, scales are 16-byte aligned (AWQ_PATH_DECODE and
 * AWQ_PATH_PREFILL for any M, chosen as for 4-bit codes); everything else runs
 * AWQ_PATH_GENERIC.  Forcing a family whose contract the shape breaks returns
 * AWQ_ERR_UNSUPPORTED_SHAPE.  (awq_gemm_select_path_ex describes 8-bit calls.)
 * awq_dequant_w8: the awq_dequant contract (exact fp32, or one rounding to fp16).
 */
awq_status_t awq_gemm_w8_ex(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                            const void* scales_f16, const void* bias_f16, int64_t M, int64_t K,
                            int64_t N, int64_t group_size, void* y_f16, awq_path_t path,
                            awq_stream_t stream);
awq_status_t awq_gemm_w8(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                         const void* scales_f16, const void* bias_f16, int64_t M, int64_t K,
                         int64_t N, int64_t group_size, void* y_f16, awq_stream_t stream);
awq_status_t awq_dequant_w8(const int32_t* qweight, const int32_t* qzeros, const void* scales_f16,
                            int64_t K, int64_t N, int64_t group_size, void* w_out,
                            awq_dtype_t out_dtype, awq_stream_t stream);

/*
 * awq_gemm_grouped -- grouped (mixture-of-experts) W4A16 linear in one launch (routed expert
 * layers with 4-bit AWQ weights: the vLLM article, section 5.4).  E experts' weights are
 * stacked; the routed rows of x are sorted by expert:
 *
 *   y[r][n] = fp16_rne( sum_k x[r][k] * w_e[k][n] (+ bias[e][n]) )  for offsets[e] <= r < offsets[e+1]
 *
 *   x_f16           fp16 [R, K]            routed rows, sorted by expert
 *   qweight         int32 [E, K, N/8], qzeros int32 [E, K/G, N/8], scales_f16 fp16 [E, K/G, N]
 *   bias_f16        fp16 [E, N] or NULL
 *   expert_offsets  DEVICE int32 [E + 1]: 0 = offsets[0] <= ... <= offsets[E] = R (may come
 *                   from a routing kernel on the same stream; it is read on the device only,
 *                   after the preceding kernel completes)
 *   y_f16           fp16 [R, N]
 *
 * Requirements: those of the decode path's TMA kernel (K % 64 == 0, group size % 64 == 0,
 * N % 32 == 0, x / qweight / qzeros / scales 16-byte aligned), 1 <= E <= 4096,
 * R / 8 + E <= 65535, E*K*N < 2^40.  Offsets outside [0, R] or not rising give unspecified
 * values in y but never an access outside x, y or the stacked weights.  R == 0 returns
 * AWQ_OK without a launch.  One kernel launch; asynchronous on `stream`.
 */
awq_status_t awq_gemm_grouped(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                              const void* scales_f16, const void* bias_f16,
                              const int32_t* expert_offsets, int64_t R, int64_t E, int64_t K,
                              int64_t N, int64_t group_size, void* y_f16, awq_stream_t stream);

/*
 * awq_quantize_rtn -- round-to-nearest 4-bit group quantization of a linear layer's fp16
 * weight into this layout (GPTQModel wiki "AWQ", "Group quantization and zero points":
 * the asymmetric and symmetric modes of its table; packing with ORDER as the format
 * page's "Reader" unpacks it).  Per output channel n and group g of G input features:
 *
 *   sym == 0:  scale = max(max - min, 1e-5) / 15
 *              zero  = clamp(-round(min / scale), 0, 15)
 *              code  = clamp(round(w / scale) + zero, 0, 15)
 *   sym == 1:  scale = max(max |w|, 1e-5) / 7,  zero = 8
 *              code  = clamp(round(w / scale), -8, 7) + 8
 *
 * Arithmetic is fp32 on the fp16 weights with every operation correctly rounded; the
 * scale is rounded to fp16 (as stored) and the codes are taken against the stored scale;
 * round is half to even.  Weights must be finite.
 *
 *   w_f16        fp16 [N, K] row-major: out_features x in_features (an nn.Linear weight)
 *   qweight      int32 [K, N/8] out, qzeros int32 [K/G, N/8] out, scales_f16 fp16 [K/G, N] out
 *
 * Requirements: K > 0, N >= 0, N % 8 == 0, group_size == -1 or (> 0 and K % group_size
 * == 0), the group size a multiple of 8 and K / group_size <= 65535; w 16-byte aligned,
 * qweight/qzeros 4-byte aligned, scales 2-byte aligned; outputs must not overlap w.
 * N == 0 returns AWQ_OK without a launch.  Argument errors are returned before any device
 * access.  One kernel launch otherwise; asynchronous on `stream`.
 */
awq_status_t awq_quantize_rtn(const void* w_f16, int64_t N, int64_t K, int64_t group_size,
                              int sym, int32_t* qweight, int32_t* qzeros, void* scales_f16,
                              awq_stream_t stream);

/*
 * awq_gemm -- fused W4A16 linear (the wiki's awq_gemm_forward in "Native GEMM" /
 * "Native AWQ runtime helpers"; fp32 accumulation always, as with its default
 * GPTQMODEL_FP32_ACCUM):
 *
 *   y[m][n] = fp16_rne( sum_k x[m][k] * w[k][n]  (+ bias[n]) )
 *
 *   x_f16     fp16 [M, K] activations
 *   qweight   int32 [K, N/8], qzeros int32 [K/G, N/8], scales_f16 fp16 [K/G, N]
 *   bias_f16  fp16 [N] or NULL
 *   y_f16     fp16 [M, N] output; must not overlap any input
 *
 * Argument order is x, qweight, qzeros, scales, bias: qzeros BEFORE scales.  (The wiki's
 * Python wrappers pass scales before qzeros; bindings must not copy that order here.)
 * The dense weight is never written to memory.  The dequantized values never leave
 * registers or shared memory.  Accumulation is fp32 with a fixed summation order for a
 * given (M, K, N, G): repeated calls give bitwise-identical y.
 * Requirements: as awq_dequant, plus x/y/bias 2-byte aligned.  M == 0 or N == 0 returns
 * AWQ_OK without a launch (the wiki's "Empty input returns an appropriately shaped output
 * without launching").  Exactly one kernel launch otherwise.
 * Accuracy: |y - y_exact| <= 1e-2 * max(1, |y_exact|) elementwise, y_exact being the
 * same sum in exact arithmetic.
 * Stream ordering: plain stream order.  The small-M kernel is a programmatic dependent
 * launch (its set-up overlaps the tail of the preceding kernel on `stream`), but it reads
 * no input and writes no output before that kernel's results are visible, so a kernel
 * that writes x or the weights (awq_quantize_rtn, a copy kernel, ...) may come directly
 * before it.  awq_gemm_any with AWQ_GEMM_STATIC_WEIGHTS relaxes this for the weights.
 */
awq_status_t awq_gemm(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                      const void* scales_f16, const void* bias_f16,
                      int64_t M, int64_t K, int64_t N, int64_t group_size,
                      void* y_f16, awq_stream_t stream);

/* awq_gemm with an explicit kernel family (tests and benchmarks).  A family that cannot
 * take the shape or alignment returns AWQ_ERR_UNSUPPORTED_SHAPE / AWQ_ERR_MISALIGNED. */
awq_status_t awq_gemm_ex(const void* x_f16, const int32_t* qweight, const int32_t* qzeros,
                         const void* scales_f16, const void* bias_f16,
                         int64_t M, int64_t K, int64_t N, int64_t group_size,
                         void* y_f16, awq_path_t path, awq_stream_t stream);

/* Flags of awq_gemm_any. */
typedef enum awq_gemm_flags {
  AWQ_GEMM_DEFAULT = 0,
  /* The caller promises that qweight, qzeros, scales and bias are complete before the kernel
   * launched immediately before this call on `stream` is launched (weights loaded once, as
   * at model load): the small-M kernel then starts streaming them before that kernel has
   * finished, under its tail.  x is still read, and y written, only after that kernel's
   * results are visible.  Breaking the promise (e.g. the preceding kernel writes the
   * weights) gives unspecified y. */
  AWQ_GEMM_STATIC_WEIGHTS = 1
} awq_gemm_flags_t;

/*
 * awq_gemm_any -- one entry point for every activation type and code width, with flags:
 * dtype AWQ_DTYPE_F16 (the awq_gemm_ex contract) or AWQ_DTYPE_BF16 (awq_gemm_bf16_ex),
 * bits 4 (qweight [K, N/8]) or 8 (awq_gemm_w8_ex: qweight [K, N/4], fp16 only); flags a
 * combination of awq_gemm_flags_t (unknown bits: AWQ_ERR_INVALID_ARGUMENT).  With
 * AWQ_GEMM_DEFAULT it behaves exactly as the matching entry point above.
 */
awq_status_t awq_gemm_any(const void* x, const int32_t* qweight, const int32_t* qzeros,
                          const void* scales, const void* bias, int64_t M, int64_t K, int64_t N,
                          int64_t group_size, void* y, awq_dtype_t dtype, int32_t bits,
                          awq_path_t path, uint32_t flags, awq_stream_t stream);

/* The family awq_gemm would pick for this shape and these pointers (no launch; above
 * 32 rows it reads the current device's SM count, 152 if there is none).  Returns
 * AWQ_PATH_AUTO (0) on an invalid shape. */
awq_path_t awq_gemm_select_path(int64_t M, int64_t K, int64_t N, int64_t group_size,
                                const void* x_f16, const int32_t* qweight,
                                const int32_t* qzeros, const void* scales_f16,
                                const void* bias_f16, const void* y_f16);

/* The same for any entry point: dtype AWQ_DTYPE_F16 or AWQ_DTYPE_BF16 (activations, scales,
 * bias, output), bits 4 (qweight [K, N/8]) or 8 (qweight [K, N/4], fp16 only).  Returns
 * AWQ_PATH_AUTO (0) on an invalid shape or combination. */
awq_path_t awq_gemm_select_path_ex(int64_t M, int64_t K, int64_t N, int64_t group_size,
                                   const void* x, const int32_t* qweight, const int32_t* qzeros,
                                   const void* scales, const void* bias, const void* y,
                                   awq_dtype_t dtype, int32_t bits);

/*
 * Tile-packed layout: an optional one-off conversion of the checkpoint layout into this
 * library's kernel-native order, and the linear that reads it.  (No page prints such a
 * layout; converting the AWQ order away for a kernel is the prior art of the vLLM article,
 * section 5.1, and of the GPTQModel wiki, "Marlin and Machete".)  Lossless on codes, zeros
 * and scales.  For output-column tile t (128 columns) and K stage s (64 rows) one block of
 * 1152 uint32 words at word (t * K/64 + s) * 1152:
 *   word 512 h + 4 c + j (h < 2, c < 128, j < 4): 4-bit codes of column 128 t + c for rows
 *     64 s + 32 h + 8 j + 0..7, row offset ORDER[p] in nibble p (ORDER = {0,2,4,6,1,3,5,7});
 *   word 1024 + c: scale bits (fp16 or bf16) | zero << 16 of column 128 t + c, group of row 64 s;
 *   columns past N: zero.
 * Requirements: those of awq_dequant plus K % 64 == 0 and group size % 64 == 0 (or -1).
 *
 * awq_repack_size: bytes of the packed weights, ceil(N / 128) * (K / 64) * 4608 (host only,
 *   no device access).
 * awq_repack: writes them to packed_out (DEVICE, caller-owned, 16-byte aligned,
 *   awq_repack_size bytes); reads qweight/qzeros/scales as awq_dequant does; K / 64 <=
 *   65535.  The scale words are copied bit for bit, so bf16 scales give the packed weights
 *   of awq_gemm_packed_ex with AWQ_DTYPE_BF16.  One kernel launch, asynchronous on `stream`.
 *   N == 0: AWQ_OK, no launch.
 * awq_gemm_packed: y = fp16_rne(x W (+ bias)) as awq_gemm, W read from the packed layout
 *   (x fp16 [M, K] 16-byte aligned, packed 16-byte aligned, bias fp16 [N] or NULL, y fp16
 *   [M, N]; fp32 accumulation, a fixed summation order: repeated calls are bitwise
 *   identical; |y - y_exact| <= 1e-2 * max(1, |y_exact|)).  A tcgen05 kernel whose
 *   dequantized weights stay in tensor memory; built for prefill-sized M (any M >= 1 runs;
 *   below 128 rows awq_gemm on the checkpoint layout is mostly faster, except near 32 rows
 *   on wide linears).  M == 0 or N == 0:
 *   AWQ_OK, no launch.  One kernel launch otherwise, asynchronous on `stream`, plain stream
 *   order.
 */
awq_status_t awq_repack_size(int64_t K, int64_t N, int64_t group_size, size_t* bytes);
awq_status_t awq_repack(const int32_t* qweight, const int32_t* qzeros, const void* scales_f16,
                        int64_t K, int64_t N, int64_t group_size, void* packed_out,
                        awq_stream_t stream);
awq_status_t awq_gemm_packed(const void* x_f16, const void* packed, const void* bias_f16,
                             int64_t M, int64_t K, int64_t N, int64_t group_size, void* y_f16,
                             awq_stream_t stream);

/*
 * The packed linear with a workspace, for prefill shapes whose 256-row x 128-column tiles
 * leave SMs idle in the last round (e.g. 512 x 4096 x 11008: 172 tiles on 152 SMs).  Such
 * calls run a stream-K kernel: the tiles' 64-row K stages form one sequence split evenly over
 * one CTA per SM; a tile cut between CTAs is finished by the CTA holding its first stages,
 * which adds the other CTAs' fp32 partial sums (written to the workspace) in CTA order.  Other
 * shapes run exactly as awq_gemm_packed.  (No page prints a work split; stream-K is the
 * published decomposition of Osama et al., "Stream-K", PPoPP 2023.)
 *
 * awq_gemm_packed_workspace_size: bytes the current device needs (256-byte flag area sized by
 *   the SM count, then 128 KB per SM).
 * awq_gemm_packed_ws: arguments as awq_gemm_packed, plus workspace (DEVICE, caller-owned,
 *   256-byte aligned, workspace_bytes >= awq_gemm_packed_workspace_size, its first
 *   256-byte-rounded 4 * SM-count bytes ZERO before the first call; each call leaves them
 *   zero).  A workspace smaller than required (or NULL) gives awq_gemm_packed's plan.
 *   Results: awq_gemm_packed's criterion, and bitwise repeatable for a given shape and
 *   device; they may differ from awq_gemm_packed's in the last bits (another summation
 *   order).  Calls that share a workspace must not overlap in time (order them on one
 *   stream).  After awq_device_status reports a timeout, zero the flag area again.
 */
awq_status_t awq_gemm_packed_workspace_size(size_t* bytes);
awq_status_t awq_gemm_packed_ws(const void* x_f16, const void* packed, const void* bias_f16,
                                int64_t M, int64_t K, int64_t N, int64_t group_size, void* y_f16,
                                void* workspace, size_t workspace_bytes, awq_stream_t stream);

/*
 * awq_gemm_packed_noalloc: awq_gemm_packed_ws without a caller workspace.  No page has a
 * counterpart: it is a convenience of this library.  It works in scratch memory the library
 * reserves on each device when it is loaded, one fixed 20 MiB array (the workspace of a device
 * with up to 159 SMs; GB300 has 152).  On a device that would need more it returns
 * AWQ_ERR_UNSUPPORTED_DEVICE and launches nothing.
 *
 * It is meant for callers that cannot give the library device memory at the call site: a
 * host application whose device memory is all handed to its own pool before the first call,
 * or code behind an interface that passes only the layer's tensors, so that neither an
 * allocation inside the library nor an extra buffer argument is possible.
 *
 * It allocates nothing.  The first call on a device looks up the array's address (once per
 * device, with that device current, kept for the life of the process: do not use this entry
 * point after resetting the device); make that first call before any stream capture that is
 * to contain it.  Every call then clears the array's flag area with one asynchronous memset
 * on `stream` and launches what awq_gemm_packed_ws would launch with a workspace of its own,
 * with the same results.  All calls on one device share the array: calls that overlap in time
 * (on different streams, or from host threads without ordering between them) race on it and
 * may produce wrong results; order them on one stream.  Arguments, requirements and errors
 * otherwise as awq_gemm_packed.
 */
awq_status_t awq_gemm_packed_noalloc(const void* x_f16, const void* packed, const void* bias_f16,
                                     int64_t M, int64_t K, int64_t N, int64_t group_size,
                                     void* y_f16, awq_stream_t stream);

/*
 * awq_gemm_packed_ex: the packed linear for either activation type.  dtype AWQ_DTYPE_F16 (x,
 * bias, y fp16; the packed weights written from fp16 scales) or AWQ_DTYPE_BF16 (x, bias, y
 * bf16; the packed weights written by awq_repack from bf16 scales: it copies the 16-bit scale
 * words as they are).  bf16 dequantizes exactly as awq_dequant_bf16 does (c - z exact, one
 * rounding of (c - z) * s to bf16; GPTQModel wiki "AWQ", "Selection and compatibility": FP16
 * and BF16 activations) and accumulates in fp32; y is rounded once to bf16.  workspace /
 * workspace_bytes as awq_gemm_packed_ws (NULL / 0: awq_gemm_packed's plan).  Other arguments,
 * requirements, results and errors as awq_gemm_packed_ws; AWQ_ERR_INVALID_ARGUMENT for
 * another dtype.
 */
awq_status_t awq_gemm_packed_ex(const void* x, const void* packed, const void* bias, int64_t M,
                                int64_t K, int64_t N, int64_t group_size, void* y,
                                awq_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                awq_stream_t stream);

/*
 * Tile-packed layout of 8-bit codes (GPTQModel wiki "AWQ", "Saved formats and packing": the
 * 8-bit GEMM layout, byte i of word c = column 4c + i; qweight [K, N/4], qzeros [K/G, N/4],
 * fp16 scales).  Same tiles and meta words as the 4-bit layout; for tile t, stage s one block
 * of 2176 uint32 words at word (t * K/64 + s) * 2176:
 *   word 1024 h + 512 k + 4 c + j (h, k < 2, c < 128, j < 4): the 8-bit codes of column
 *     128 t + c for rows 64 s + 32 h + 16 k + 4 j + 0..3, row offset b in byte b;
 *   word 2048 + c: fp16 scale bits | zero << 16 (8-bit zero) of column 128 t + c;
 *   columns past N: zero.
 * Requirements: those of awq_dequant_w8 plus K % 64 == 0 and group size % 64 == 0 (or -1).
 * awq_repack_w8_size: ceil(N / 128) * (K / 64) * 8704 bytes (host only).
 * awq_repack_w8: as awq_repack, from 8-bit checkpoint tensors.
 * awq_gemm_packed_w8: y = fp16_rne(x W (+ bias)) from the 8-bit packed layout (fp16 x, bias,
 *   y; (c - z) * s formed exactly and rounded once to fp16, fp32 accumulation), with an
 *   optional workspace as awq_gemm_packed_ws (NULL / 0: no stream-K).  Arguments, results and
 *   errors otherwise as awq_gemm_packed_ws.
 */
/*
 * awq_gemm_packed_grouped: the grouped (mixture-of-experts) linear of awq_gemm_grouped on
 * tile-packed weights, for routed batches of prefill size (vLLM article, section 5.4: routed
 * expert layers).  packed holds E tile-packed layouts of 4-bit experts back to back, expert
 * e's at byte e * awq_repack_size(K, N, group_size) (awq_repack of qweight[e], qzeros[e],
 * scales[e] into that slice); x [R, K] routed rows sorted by expert, expert_offsets DEVICE
 * int32 [E + 1] as for awq_gemm_grouped (read on the device only), bias [E, N] or NULL,
 * y [R, N]; x, bias, y (and the scales the layouts were written from) fp16 (dtype
 * AWQ_DTYPE_F16) or bf16 (AWQ_DTYPE_BF16, as awq_gemm_packed_ex).  One persistent launch over (expert, 256-row tile,
 * column tile); a tile's rows of the next expert are computed and discarded.  Requirements:
 * those of awq_gemm_packed, 1 <= E <= 256, E*K*N < 2^40.  Offsets outside [0, R] or not
 * rising give unspecified values in y but never an access outside x, y, bias or packed.
 * R == 0 or N == 0: AWQ_OK, no launch.
 */
awq_status_t awq_gemm_packed_grouped(const void* x, const void* packed, const void* bias,
                                     const int32_t* expert_offsets, int64_t R, int64_t E,
                                     int64_t K, int64_t N, int64_t group_size, void* y,
                                     awq_dtype_t dtype, awq_stream_t stream);

awq_status_t awq_repack_w8_size(int64_t K, int64_t N, int64_t group_size, size_t* bytes);
awq_status_t awq_repack_w8(const int32_t* qweight, const int32_t* qzeros, const void* scales_f16,
                           int64_t K, int64_t N, int64_t group_size, void* packed_out,
                           awq_stream_t stream);
awq_status_t awq_gemm_packed_w8(const void* x_f16, const void* packed, const void* bias_f16,
                                int64_t M, int64_t K, int64_t N, int64_t group_size, void* y_f16,
                                void* workspace, size_t workspace_bytes, awq_stream_t stream);

/* Synchronizes `stream`, then reads and clears the library's device status word on the
 * current device.  Returns AWQ_ERR_TIMEOUT if a kernel gave up a bounded wait since the
 * last check (its output is then unspecified), AWQ_OK otherwise. */
awq_status_t awq_device_status(awq_stream_t stream);

/* Failure-detection self test.  Launches one thread that waits on an mbarrier nothing
 * ever completes, bounded by limit_ns of wall time (1e3 .. 1e9, else
 * AWQ_ERR_INVALID_ARGUMENT): the wait gives up the same way a stalled stage of the GEMM
 * kernels would -- it sets the device status word and the kernel returns, with no fault,
 * trap or hang -- so a following awq_device_status returns AWQ_ERR_TIMEOUT (and clears
 * the word).  Asynchronous on `stream`; one launch.  No counterpart on the pages. */
awq_status_t awq_selftest_wait_timeout(uint64_t limit_ns, awq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_GB300_H */
