"""Plain CPU oracle for the AWQ W4A16 GEMM-layout linear.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference leg may import this module.  The
product path (the CUDA library and its binding) never imports, links or
calls it, and this module imports nothing from the product path.

What it computes, and where each step comes from:

* Unpack (tensref.org/formats/awq, "Reader", function ``unpack_awq_gemm``):
  nibble ``i`` of int32 word ``c`` in a row holds output column
  ``8*c + ORDER[i]`` with ``ORDER = [0, 2, 4, 6, 1, 3, 5, 7]``; the code is
  ``(word >> 4*i) & 0xF``.  Zeros are unpacked the same way.  Words are read
  as their unsigned 32-bit pattern; with the ``& 0xF`` mask an arithmetic
  right shift of the signed word would give the same nibbles.
* Dequantize (same function): for input row ``k`` the scale/zero row is
  ``g = k // G``; ``w = (code - zero) * scale`` evaluated in fp32.  Zeros
  are used as stored, with no +1 (same page, reject rule AWQ-005; GPTQModel
  wiki "AWQ", "Group quantization and zero points").  ``group_size == -1``
  means one group spanning all of K (GPTQModel wiki "AWQ", same section).
  The page returns the transpose ``[out_features, in_features]``;
  :func:`dequant_page_layout` reproduces that, :func:`dequant_f32` gives the
  ``[K, N]`` orientation used by ``x @ W``.
* fp16 dequant output: one round-to-nearest-even conversion of the exact
  fp32 value (the fp32 value is exact: |code - zero| <= 15 times an fp16
  scale fits in 24 bits).
* GEMM: ``y = x @ W (+ bias)`` in fp64, ``x`` fp16 [M, K] widened exactly,
  ``W`` the fp32 dequant widened exactly; bias broadcast over rows as in a
  linear layer (format page, "bias ... optional, shape [out_features]").

* Round-to-nearest quantization (:func:`quantize_rtn`; GPTQModel wiki "AWQ",
  "Group quantization and zero points", the table of the asymmetric and
  symmetric modes): per output channel and group of ``G`` input features,
  asymmetric ``scale = max(max - min, 1e-5) / 15``, ``zero = clamp(-round(min /
  scale), 0, 15)``, ``code = clamp(round(w / scale) + zero, 0, 15)``;
  symmetric ``scale = max(max|w|, 1e-5) / 7``, ``code = clamp(round(w /
  scale), -8, 7) + 8`` with zero 8 (the page: packing shifts signed codes to
  unsigned and supplies zero 2^(bits-1)).  Readings where the page is silent:
  fp32 arithmetic on the fp16 weights (each operation correctly rounded), the
  scale rounded to fp16 as a checkpoint stores it and the codes taken against
  that stored scale, round half to even.

* bf16 (the native GEMM's declared FP16/BF16 contract; GPTQModel wiki "AWQ",
  "Selection and compatibility"): activations, scales and bias hold bf16
  values; the GEMM definition is unchanged (fp64 of the exact values);
  :func:`dequant_bf16` is the exact fp32 dequant rounded once to bf16
  (:func:`round_to_bf16`, nearest even: bf16 is the upper half of an fp32).

* Grouped (mixture-of-experts) linear (:func:`gemm_grouped`; vLLM article,
  section 5.4: routed expert layers with 4-bit AWQ weights): rows
  ``offsets[e] .. offsets[e+1]-1`` of ``x`` (routed rows sorted by expert) go
  through expert ``e``'s AWQ linear, each as :func:`gemm` defines it.

* 8-bit weights (GPTQModel wiki "AWQ", "Saved formats and packing": widths
  other than 4 pack as a continuous little-endian bit stream, and the INT4
  order is not applied): column ``4*c + i`` of a row is byte ``i`` of word
  ``c`` (:func:`unpack_codes8`); qweight ``[K, N/4]``, qzeros ``[K/G, N/4]``,
  scales ``[K/G, N]``; ``w = (code - zero) * scale`` as for 4 bits
  (:func:`dequant8_f32`, :func:`gemm8`).

* Tile-packed layout (:func:`repack`, :func:`unpack_repacked`): the optional one-off
  conversion into a kernel-native layout (no page prints one; repacking the AWQ order
  away for a kernel is the prior art of the vLLM article, section 5.1, and of the
  GPTQModel wiki, "Marlin and Machete").  It is lossless on codes, zeros and scales and
  needs K % 64 == 0 and G % 64 == 0.  For output-column tile t (columns 128t .. 128t+127)
  and K stage s (rows 64s .. 64s+63) one block of 4608 bytes sits at byte (t*K/64 + s) *
  4608: two halves h (rows 64s + 32h ..), each 128 columns x 4 words, word (h, c, j) at
  index 512h + 4c + j holding the codes of column 128t + c for rows 64s + 32h + 8j + 0..7,
  row offset ORDER[p] in nibble p (the checkpoint's column interleave, applied along K);
  then 128 meta words, word c = scale bits (fp16) | zero << 16 of column 128t + c for the
  group of row 64s.  Columns past N hold code 0, zero 0, scale 0.
* Tile-packed layout of 8-bit codes (:func:`repack8`, :func:`unpack_repacked8`): the same
  tiles and stages, one block of 8704 bytes each: two halves h, two 16-row quarters k of
  each, 128 columns x 4 words, word (h, k, c, j) at index 1024h + 512k + 4c + j holding the
  codes of column 128t + c for rows 64s + 32h + 16k + 4j + 0..3, row offset b in byte b;
  then the 128 meta words as above (8-bit zeros fit the upper half).  Needs N % 4 == 0.

Pins (tests/test_oracle.py, run without a GPU): ORDER and its inverse from
the wiki's "Saved formats and packing" section, a hand-packed word, AWQ-004
(sequential-nibble decode differs), AWQ-005 (zero equal to code gives an
exact 0), group_size -1 equals group_size K, symmetric zero 8, exact
rational dequant values, a pure-Python brute-force GEMM written separately,
and an exact-arithmetic GEMM case; for the quantizer a hand-worked group
(tests/golden/rtn_worked_example.txt), exact round trips of weights that lie on
a grid spanning the whole code range, the half-step error bound, the clamped
degenerate groups and group_size -1 equal to group_size K.  Every function
here has at least one pin (bf16 rounding: hand-worked ties and torch's own
bf16 conversion on random and edge values).
"""
from __future__ import annotations

import numpy as np

# Nibble i of a packed word holds column 8*c + ORDER[i]
# (tensref.org/formats/awq, "Reader"; GPTQModel wiki "AWQ", "Saved formats
# and packing").
ORDER = (0, 2, 4, 6, 1, 3, 5, 7)
# Inverse permutation, as printed in the wiki's "Saved formats and packing".
REVERSE_ORDER = (0, 4, 1, 5, 2, 6, 3, 7)


def resolve_group_size(K: int, group_size: int) -> int:
    """G = K for group_size -1, else group_size; K must split into whole groups.

    GPTQModel wiki "AWQ", "Group quantization and zero points": positive
    values need compatible dimensions, -1 is one group across the row.
    """
    G = K if group_size == -1 else int(group_size)
    if G <= 0 or K % G != 0:
        raise ValueError(f"group_size {group_size} incompatible with K={K}")
    return G


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """[R, C] int32 words -> [R, 8C] int64 codes in 0..15 (format page, "Reader")."""
    packed = np.ascontiguousarray(packed)
    assert packed.dtype == np.int32 and packed.ndim == 2
    u = packed.view(np.uint32).astype(np.uint64)
    R, C = packed.shape
    out = np.empty((R, 8 * C), dtype=np.int64)
    for i in range(8):
        # every word c of the row: column 8*c + ORDER[i] <- (word >> 4i) & 0xF
        out[:, ORDER[i]::8] = ((u >> np.uint64(4 * i)) & np.uint64(0xF)).astype(np.int64)
    return out


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Inverse of :func:`unpack_codes`: [R, 8C] codes 0..15 -> [R, C] int32.

    The wiki's ``pack_awq`` (section "Saved formats and packing") rejects
    INT4 widths that are not a multiple of eight; so does this.
    """
    codes = np.asarray(codes)
    R, N = codes.shape
    if N % 8 != 0:
        raise ValueError("INT4 AWQ packing needs a width divisible by 8")
    if codes.min(initial=0) < 0 or codes.max(initial=0) > 15:
        raise ValueError("codes must lie in 0..15")
    c = codes.astype(np.uint64)
    word = np.zeros((R, N // 8), dtype=np.uint64)
    for i in range(8):
        word |= c[:, ORDER[i]::8] << np.uint64(4 * i)
    return word.astype(np.uint32).view(np.int32)


def dequant_f32(qweight, qzeros, scales, group_size) -> np.ndarray:
    """W[k, n] = (code[k, n] - zero[k // G, n]) * scale[k // G, n], fp32, [K, N]."""
    K = qweight.shape[0]
    G = resolve_group_size(K, group_size)
    codes = unpack_codes(qweight).astype(np.float32)
    zeros = unpack_codes(qzeros).astype(np.float32)
    sc = np.asarray(scales).astype(np.float32)
    n_groups = K // G
    assert zeros.shape[0] == n_groups and sc.shape[0] == n_groups
    assert zeros.shape[1] == codes.shape[1] == sc.shape[1]
    g_of_k = np.arange(K) // G
    return ((codes - zeros[g_of_k]) * sc[g_of_k]).astype(np.float32)


def dequant_f16(qweight, qzeros, scales, group_size) -> np.ndarray:
    """fp16 [K, N]: round-to-nearest-even of :func:`dequant_f32`."""
    return dequant_f32(qweight, qzeros, scales, group_size).astype(np.float16)


def round_to_bf16(values) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even), returned as fp32 arrays
    holding the bf16 values.  bf16 keeps the upper 16 bits of an fp32 pattern, so
    rounding adds 0x7FFF plus the kept part's lowest bit and clears the low half."""
    u = np.ascontiguousarray(values, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32)


def dequant_bf16(qweight, qzeros, scales, group_size) -> np.ndarray:
    """bf16 dequant output: the exact fp32 value rounded once to bf16 (as fp32 values).
    ``scales`` holds bf16 values (any float dtype that represents them exactly)."""
    return round_to_bf16(dequant_f32(qweight, qzeros, scales, group_size))


def dequant_page_layout(qweight, qzeros, scales, group_size) -> np.ndarray:
    """fp32 [N, K] ([out_features, in_features]) exactly as the format page
    returns it: column k of the output is filled from input row k."""
    K = qweight.shape[0]
    G = resolve_group_size(K, group_size)
    w = unpack_codes(qweight)
    z = unpack_codes(qzeros)
    sc = np.asarray(scales)
    out = np.empty((w.shape[1], K), dtype=np.float32)
    for k in range(K):
        g = k // G
        out[:, k] = (w[k].astype(np.float32) - z[g].astype(np.float32)) * sc[g].astype(np.float32)
    return out


def gemm(x, qweight, qzeros, scales, bias, group_size) -> np.ndarray:
    """y[m, n] = sum_k x[m, k] * W[k, n] (+ bias[n]) in fp64, [M, N]."""
    W = dequant_f32(qweight, qzeros, scales, group_size).astype(np.float64)
    y = np.asarray(x).astype(np.float64) @ W
    if bias is not None:
        y = y + np.asarray(bias).astype(np.float64)[None, :]
    return y


def dequant_columns_f32(qweight, qzeros, scales, group_size, cols) -> np.ndarray:
    """fp32 [K, len(cols)]: :func:`dequant_f32` restricted to output columns
    ``cols`` (column n sits in word n // 8, nibble REVERSE_ORDER[n % 8])."""
    K = qweight.shape[0]
    G = resolve_group_size(K, group_size)
    cols = np.asarray(cols, dtype=np.int64)
    words = np.ascontiguousarray(qweight).view(np.uint32)[:, cols // 8].astype(np.uint64)
    zwords = np.ascontiguousarray(qzeros).view(np.uint32)[:, cols // 8].astype(np.uint64)
    shift = (4 * np.asarray(REVERSE_ORDER, dtype=np.int64)[cols % 8]).astype(np.uint64)
    codes = ((words >> shift[None, :]) & np.uint64(0xF)).astype(np.float32)
    zeros = ((zwords >> shift[None, :]) & np.uint64(0xF)).astype(np.float32)
    sc = np.asarray(scales)[:, cols].astype(np.float32)
    g_of_k = np.arange(K) // G
    return ((codes - zeros[g_of_k]) * sc[g_of_k]).astype(np.float32)


def gemm_sampled(x, qweight, qzeros, scales, bias, group_size, rows, cols) -> np.ndarray:
    """fp64 y[rows[i], cols[i]] for each sampled pair i (same definition as
    :func:`gemm`, evaluated only where asked)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    ucols, inv = np.unique(cols, return_inverse=True)
    Wc = dequant_columns_f32(qweight, qzeros, scales, group_size, ucols).astype(np.float64)
    xr = np.asarray(x)[rows].astype(np.float64)           # [S, K]
    y = np.einsum("sk,sk->s", xr, Wc[:, inv].T)
    if bias is not None:
        y = y + np.asarray(bias).astype(np.float64)[cols]
    return y


def gemm_rows(x, qweight, qzeros, scales, bias, group_size, rows) -> np.ndarray:
    """fp64 y[rows, :] for a subset of activation rows (full N)."""
    W = dequant_f32(qweight, qzeros, scales, group_size).astype(np.float64)
    y = np.asarray(x)[np.asarray(rows)].astype(np.float64) @ W
    if bias is not None:
        y = y + np.asarray(bias).astype(np.float64)[None, :]
    return y


def within_tolerance(y, y_ref, rel: float = 1e-2):
    """Elementwise |y - y_ref| <= rel * max(1, |y_ref|); returns (ok, worst ratio)."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    bound = rel * np.maximum(1.0, np.abs(y_ref))
    err = np.abs(y - y_ref)
    finite = bool(np.all(np.isfinite(y)))
    ratio = err / bound
    worst = float(np.max(ratio)) if (ratio.size and finite) else (0.0 if finite else float("inf"))
    ok = bool(finite and np.all(err <= bound))
    return ok, worst


def quantize_rtn(w, group_size, sym=False):
    """Round-to-nearest group quantization of a linear layer's fp16 weight into
    the AWQ GEMM layout (GPTQModel wiki "AWQ", "Group quantization and zero
    points").

    ``w``: fp16 ``[N, K]`` (out_features x in_features: one row per output
    channel; groups of ``G`` consecutive input features along each row).
    Returns ``(qweight int32 [K, N/8], qzeros int32 [K/G, N/8], scales fp16
    [K/G, N])``, packed with ORDER like a checkpoint.
    """
    w = np.asarray(w)
    if w.dtype != np.float16:
        raise ValueError("w must be fp16")
    N, K = w.shape
    G = resolve_group_size(K, group_size)
    if N % 8 != 0:
        raise ValueError("out_features must be a multiple of 8")
    wf = w.astype(np.float32).reshape(N, K // G, G)  # exact widening
    if not sym:
        wmax = wf.max(axis=2)
        wmin = wf.min(axis=2)
        rng = np.maximum(wmax - wmin, np.float32(1e-5))           # fp32 subtraction
        scale16 = (rng / np.float32(15)).astype(np.float16)        # fp32 division, RNE to fp16
        s = scale16.astype(np.float32)
        zero = np.clip(-np.rint(wmin / s), 0, 15)
        code = np.clip(np.rint(wf / s[:, :, None]) + zero[:, :, None], 0, 15)
    else:
        amax = np.maximum(np.abs(wf).max(axis=2), np.float32(1e-5))
        scale16 = (amax / np.float32(7)).astype(np.float16)
        s = scale16.astype(np.float32)
        zero = np.full(scale16.shape, 8.0, dtype=np.float32)
        code = np.clip(np.rint(wf / s[:, :, None]), -8, 7) + 8
    codes_kn = code.reshape(N, K).T.astype(np.int64)     # [K, N]
    zeros_gn = zero.T.astype(np.int64)                   # [K/G, N]
    return pack_codes(codes_kn), pack_codes(zeros_gn), np.ascontiguousarray(scale16.T)


def gemm_grouped(x, qweight, qzeros, scales, bias, group_size, offsets) -> np.ndarray:
    """y [R, N]: rows offsets[e]..offsets[e+1]-1 of x [R, K] times expert e's weight
    (qweight [E, K, N/8], qzeros [E, K/G, N/8], scales [E, K/G, N], bias [E, N] or
    None), each block as :func:`gemm` (fp64)."""
    offsets = np.asarray(offsets, dtype=np.int64)
    E = len(offsets) - 1
    R = np.asarray(x).shape[0]
    N = np.asarray(qweight).shape[2] * 8
    if offsets[0] != 0 or offsets[-1] != R or (np.diff(offsets) < 0).any():
        raise ValueError("offsets must rise from 0 to the number of rows")
    y = np.zeros((R, N), dtype=np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b] = gemm(np.asarray(x)[a:b], qweight[e], qzeros[e], scales[e],
                          None if bias is None else bias[e], group_size)
    return y


def unpack_codes8(packed: np.ndarray) -> np.ndarray:
    """[R, C] int32 words -> [R, 4C] 8-bit codes: column 4c + i is byte i of word c
    (little-endian bit stream of 8-bit codes)."""
    u = np.ascontiguousarray(packed).view(np.uint32).astype(np.uint64)
    R, C = u.shape
    out = np.empty((R, 4 * C), dtype=np.int64)
    for i in range(4):
        out[:, i::4] = ((u >> np.uint64(8 * i)) & np.uint64(0xFF)).astype(np.int64)
    return out


def pack_codes8(codes: np.ndarray) -> np.ndarray:
    """Inverse of :func:`unpack_codes8`: [R, 4C] codes 0..255 -> [R, C] int32."""
    codes = np.asarray(codes)
    R, N = codes.shape
    if N % 4 != 0:
        raise ValueError("8-bit packing needs a width divisible by 4")
    if codes.min(initial=0) < 0 or codes.max(initial=0) > 255:
        raise ValueError("codes must lie in 0..255")
    c = codes.astype(np.uint64)
    word = np.zeros((R, N // 4), dtype=np.uint64)
    for i in range(4):
        word |= c[:, i::4] << np.uint64(8 * i)
    return word.astype(np.uint32).view(np.int32)


def dequant8_f32(qweight, qzeros, scales, group_size) -> np.ndarray:
    """8-bit W[k, n] = (code[k, n] - zero[k // G, n]) * scale[k // G, n], fp32, [K, N]
    (exact: a 9-bit integer times an 11-bit significand)."""
    K = np.asarray(qweight).shape[0]
    G = resolve_group_size(K, group_size)
    codes = unpack_codes8(qweight).astype(np.float32)
    zeros = unpack_codes8(qzeros).astype(np.float32)
    sc = np.asarray(scales).astype(np.float32)
    g_of_k = np.arange(K) // G
    return ((codes - zeros[g_of_k]) * sc[g_of_k]).astype(np.float32)


def gemm8(x, qweight, qzeros, scales, bias, group_size) -> np.ndarray:
    """y = x @ W8 (+ bias) in fp64 with the 8-bit dequant."""
    W = dequant8_f32(qweight, qzeros, scales, group_size).astype(np.float64)
    y = np.asarray(x).astype(np.float64) @ W
    if bias is not None:
        y = y + np.asarray(bias).astype(np.float64)[None, :]
    return y



# ------------------------------------------------------------ tile-packed layout ----
# The optional one-off repack into this library's kernel-native layout (see the module
# docstring): blocks of PACK_TN columns x PACK_TK K rows.
PACK_TN = 128
PACK_TK = 64
PACK_BLOCK_WORDS = PACK_TN * PACK_TK // 8 + PACK_TN  # 1024 code words + 128 meta words
PACK_BLOCK_BYTES = 4 * PACK_BLOCK_WORDS              # 4608


def repack_size(K: int, N: int, group_size: int) -> int:
    """Bytes of the tile-packed layout: one block per (column tile, K stage)."""
    G = resolve_group_size(K, group_size)
    if K % PACK_TK != 0 or G % PACK_TK != 0 or N % 8 != 0:
        raise ValueError("the tile-packed layout needs K % 64 == 0, G % 64 == 0, N % 8 == 0")
    return -(-N // PACK_TN) * (K // PACK_TK) * PACK_BLOCK_BYTES


def repack(qweight, qzeros, scales, group_size) -> np.ndarray:
    """Checkpoint layout -> tile-packed layout, as uint32 words (see the module docstring).
    Steps: unpack codes and zeros with the page's reader, pad the columns to whole tiles,
    then write every block word by word.  scales: fp16 values, or their 16-bit words as a
    uint16 array (bf16 scales: the layout carries the scale word unchanged, whatever its
    format)."""
    K, C = qweight.shape
    N = 8 * C
    G = resolve_group_size(K, group_size)
    nbytes = repack_size(K, N, group_size)
    codes = unpack_codes(qweight)                  # [K, N]
    zeros = unpack_codes(qzeros)                   # [K/G, N]
    sc = np.asarray(scales)
    sbits = (sc if sc.dtype == np.uint16 else np.ascontiguousarray(sc, dtype=np.float16).view(np.uint16))
    sbits = sbits.astype(np.uint64)
    NT, KS = -(-N // PACK_TN), K // PACK_TK
    Np = NT * PACK_TN
    cp = np.zeros((K, Np), dtype=np.uint64)
    cp[:, :N] = codes
    zp = np.zeros((K // G, Np), dtype=np.uint64)
    zp[:, :N] = zeros
    sp = np.zeros((K // G, Np), dtype=np.uint64)
    sp[:, :N] = sbits
    out = np.zeros(nbytes // 4, dtype=np.uint64)
    for t in range(NT):
        cols = slice(PACK_TN * t, PACK_TN * (t + 1))
        for s in range(KS):
            base = (t * KS + s) * PACK_BLOCK_WORDS
            blk = cp[PACK_TK * s:PACK_TK * (s + 1), cols]     # [64 rows, 128 columns]
            for h in range(2):
                for j in range(4):
                    word = np.zeros(PACK_TN, dtype=np.uint64)
                    for p in range(8):
                        row = 32 * h + 8 * j + ORDER[p]
                        word |= blk[row] << np.uint64(4 * p)
                    out[base + 512 * h + 4 * np.arange(PACK_TN) + j] = word
            g = (PACK_TK * s) // G
            out[base + 1024:base + 1024 + PACK_TN] = sp[g, cols] | (zp[g, cols] << np.uint64(16))
    return out.astype(np.uint32)


def unpack_repacked(packed, K: int, N: int, group_size: int):
    """Tile-packed words -> (codes [K, N], zeros [K/G, N], scales fp16 [K/G, N]), reading
    every block back; the zero and scale of a group are taken from its first stage."""
    G = resolve_group_size(K, group_size)
    words = np.asarray(packed, dtype=np.uint32).astype(np.uint64)
    assert words.size * 4 == repack_size(K, N, group_size)
    NT, KS = -(-N // PACK_TN), K // PACK_TK
    codes = np.zeros((K, NT * PACK_TN), dtype=np.int64)
    zeros = np.zeros((K // G, NT * PACK_TN), dtype=np.int64)
    sbits = np.zeros((K // G, NT * PACK_TN), dtype=np.uint16)
    for t in range(NT):
        for s in range(KS):
            base = (t * KS + s) * PACK_BLOCK_WORDS
            for h in range(2):
                for j in range(4):
                    word = words[base + 512 * h + 4 * np.arange(PACK_TN) + j]
                    for p in range(8):
                        row = PACK_TK * s + 32 * h + 8 * j + ORDER[p]
                        codes[row, PACK_TN * t:PACK_TN * (t + 1)] = (word >> np.uint64(4 * p)) & np.uint64(0xF)
            if (PACK_TK * s) % G == 0:
                meta = words[base + 1024:base + 1024 + PACK_TN]
                g = (PACK_TK * s) // G
                sbits[g, PACK_TN * t:PACK_TN * (t + 1)] = (meta & np.uint64(0xFFFF)).astype(np.uint16)
                zeros[g, PACK_TN * t:PACK_TN * (t + 1)] = (meta >> np.uint64(16)) & np.uint64(0xF)
    return codes[:, :N], zeros[:, :N], sbits[:, :N].view(np.float16)


def gemm_packed(x, packed, bias, K: int, N: int, group_size: int) -> np.ndarray:
    """y = x @ W (+ bias) in fp64 with W read back from the tile-packed layout:
    W[k, n] = (code[k, n] - zero[k // G, n]) * scale[k // G, n] in fp32, as :func:`gemm`."""
    G = resolve_group_size(K, group_size)
    codes, zeros, sc = unpack_repacked(packed, K, N, group_size)
    g_of_k = np.arange(K) // G
    W = ((codes.astype(np.float32) - zeros[g_of_k].astype(np.float32))
         * sc[g_of_k].astype(np.float32)).astype(np.float64)
    y = np.asarray(x).astype(np.float64) @ W
    if bias is not None:
        y = y + np.asarray(bias).astype(np.float64)[None, :]
    return y


PACK8_BLOCK_WORDS = PACK_TN * PACK_TK // 4 + PACK_TN  # 2048 code words + 128 meta words
PACK8_BLOCK_BYTES = 4 * PACK8_BLOCK_WORDS              # 8704


def repack8_size(K: int, N: int, group_size: int) -> int:
    """Bytes of the 8-bit tile-packed layout: one block per (column tile, K stage)."""
    G = resolve_group_size(K, group_size)
    if K % PACK_TK != 0 or G % PACK_TK != 0 or N % 4 != 0:
        raise ValueError("the 8-bit tile-packed layout needs K % 64 == 0, G % 64 == 0, N % 4 == 0")
    return -(-N // PACK_TN) * (K // PACK_TK) * PACK8_BLOCK_BYTES


def repack8(qweight, qzeros, scales, group_size) -> np.ndarray:
    """8-bit checkpoint layout -> 8-bit tile-packed layout, as uint32 words (module docstring).
    Steps: unpack codes and zeros with the 8-bit reader, pad the columns to whole tiles, then
    write every block word by word."""
    K, C = qweight.shape
    N = 4 * C
    G = resolve_group_size(K, group_size)
    nbytes = repack8_size(K, N, group_size)
    codes = unpack_codes8(qweight)
    zeros = unpack_codes8(qzeros)
    sbits = np.ascontiguousarray(scales, dtype=np.float16).view(np.uint16).astype(np.uint64)
    NT, KS = -(-N // PACK_TN), K // PACK_TK
    Np = NT * PACK_TN
    cp = np.zeros((K, Np), dtype=np.uint64)
    cp[:, :N] = codes
    zp = np.zeros((K // G, Np), dtype=np.uint64)
    zp[:, :N] = zeros
    sp = np.zeros((K // G, Np), dtype=np.uint64)
    sp[:, :N] = sbits
    out = np.zeros(nbytes // 4, dtype=np.uint64)
    for t in range(NT):
        cols = slice(PACK_TN * t, PACK_TN * (t + 1))
        for s in range(KS):
            base = (t * KS + s) * PACK8_BLOCK_WORDS
            for h in range(2):
                for k in range(2):
                    for j in range(4):
                        word = np.zeros(PACK_TN, dtype=np.uint64)
                        for b in range(4):
                            row = PACK_TK * s + 32 * h + 16 * k + 4 * j + b
                            word |= cp[row, cols] << np.uint64(8 * b)
                        out[base + 1024 * h + 512 * k + 4 * np.arange(PACK_TN) + j] = word
            g = (PACK_TK * s) // G
            out[base + 2048:base + 2048 + PACK_TN] = sp[g, cols] | (zp[g, cols] << np.uint64(16))
    return out.astype(np.uint32)


def unpack_repacked8(packed, K: int, N: int, group_size: int):
    """8-bit tile-packed words -> (codes [K, N], zeros [K/G, N], scales fp16 [K/G, N]), reading
    every block back; the zero and scale of a group are taken from its first stage."""
    G = resolve_group_size(K, group_size)
    words = np.asarray(packed, dtype=np.uint32).astype(np.uint64)
    assert words.size * 4 == repack8_size(K, N, group_size)
    NT, KS = -(-N // PACK_TN), K // PACK_TK
    codes = np.zeros((K, NT * PACK_TN), dtype=np.int64)
    zeros = np.zeros((K // G, NT * PACK_TN), dtype=np.int64)
    sbits = np.zeros((K // G, NT * PACK_TN), dtype=np.uint16)
    for t in range(NT):
        for s in range(KS):
            base = (t * KS + s) * PACK8_BLOCK_WORDS
            for h in range(2):
                for k in range(2):
                    for j in range(4):
                        word = words[base + 1024 * h + 512 * k + 4 * np.arange(PACK_TN) + j]
                        for b in range(4):
                            row = PACK_TK * s + 32 * h + 16 * k + 4 * j + b
                            codes[row, PACK_TN * t:PACK_TN * (t + 1)] = (word >> np.uint64(8 * b)) & np.uint64(0xFF)
            if (PACK_TK * s) % G == 0:
                meta = words[base + 2048:base + 2048 + PACK_TN]
                g = (PACK_TK * s) // G
                sbits[g, PACK_TN * t:PACK_TN * (t + 1)] = (meta & np.uint64(0xFFFF)).astype(np.uint16)
                zeros[g, PACK_TN * t:PACK_TN * (t + 1)] = (meta >> np.uint64(16)) & np.uint64(0xFF)
    return codes[:, :N], zeros[:, :N], sbits[:, :N].view(np.float16)


def gemm_packed8(x, packed, bias, K: int, N: int, group_size: int) -> np.ndarray:
    """y = x @ W (+ bias) in fp64 with W read back from the 8-bit tile-packed layout:
    W[k, n] = (code[k, n] - zero[k // G, n]) * scale[k // G, n] in fp32, as :func:`gemm8`."""
    G = resolve_group_size(K, group_size)
    codes, zeros, sc = unpack_repacked8(packed, K, N, group_size)
    g_of_k = np.arange(K) // G
    W = ((codes.astype(np.float32) - zeros[g_of_k].astype(np.float32))
         * sc[g_of_k].astype(np.float32)).astype(np.float64)
    y = np.asarray(x).astype(np.float64) @ W
    if bias is not None:
        y = y + np.asarray(bias).astype(np.float64)
    return y