"""Pins for the CPU oracle: each check rests on something other than the oracle
itself -- values worked by hand from the pages, closed forms, exact rational
arithmetic, or a pure-Python brute force written separately below."""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from synth import awq_linear, SYM_ZERO_WORD

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "awq_word_layout.txt")

# Restated literally from the format page (tensref.org/formats/awq, "Reader")
# and from GPTQModel wiki "AWQ", "Saved formats and packing".
PAGE_ORDER = [0, 2, 4, 6, 1, 3, 5, 7]
PAGE_REVERSE_ORDER = [0, 4, 1, 5, 2, 6, 3, 7]


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, word, cols, seq = line.split()
            rows.append((name, int(word, 16), [int(v) for v in cols.split(",")],
                         [int(v) for v in seq.split(",")]))
    return rows


def _word(u32):
    return np.array([[np.uint32(u32)]], dtype=np.uint32).view(np.int32)


# ---------------------------------------------------------------- ORDER ----

def test_order_tables_match_pages_and_are_inverse():
    assert list(oracle.ORDER) == PAGE_ORDER
    assert list(oracle.REVERSE_ORDER) == PAGE_REVERSE_ORDER
    for i in range(8):
        assert oracle.REVERSE_ORDER[oracle.ORDER[i]] == i
        assert oracle.ORDER[oracle.REVERSE_ORDER[i]] == i


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_golden_words_unpack(row):
    name, word, cols, _ = row
    assert oracle.unpack_codes(_word(word))[0].tolist() == cols


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_golden_words_pack(row):
    name, word, cols, _ = row
    packed = oracle.pack_codes(np.array([cols]))
    assert int(packed.view(np.uint32)[0, 0]) == word


def test_awq004_sequential_decode_differs():
    """AWQ-004: sequential nibbles are not the AWQ order."""
    for name, word, cols, seq in _golden_rows():
        sequential = [(word >> (4 * j)) & 0xF for j in range(8)]
        assert sequential == seq
        if len(set(cols)) > 1 and name != "sign_nibble":
            assert sequential != cols
    # and the oracle does not decode sequentially
    assert oracle.unpack_codes(_word(0x75316420))[0].tolist() != [0, 2, 4, 6, 1, 3, 5, 7]


def test_pack_unpack_round_trip_random_words():
    rng = np.random.default_rng(7)
    q = rng.integers(0, 1 << 32, size=(37, 19), dtype=np.uint64).astype(np.uint32).view(np.int32)
    codes = oracle.unpack_codes(q)
    assert codes.shape == (37, 152) and codes.min() >= 0 and codes.max() <= 15
    assert np.array_equal(oracle.pack_codes(codes), q)


def test_pack_rejects_width_not_multiple_of_8():
    with pytest.raises(ValueError):
        oracle.pack_codes(np.zeros((2, 12), dtype=np.int64))


def test_half2_pair_property():
    """(q >> 4j) & 0x000F000F holds columns 2j (low half) and 2j+1 (high half):
    a property of ORDER that the CUDA kernels rely on; checked here against the
    oracle's unpack on random words."""
    rng = np.random.default_rng(3)
    words = rng.integers(0, 1 << 32, size=4096, dtype=np.uint64).astype(np.uint32)
    codes = oracle.unpack_codes(words.view(np.int32).reshape(-1, 1))
    for j in range(4):
        pair = (words >> np.uint32(4 * j)) & np.uint32(0x000F000F)
        assert np.array_equal(pair & 0xF, codes[:, 2 * j])
        assert np.array_equal(pair >> 16, codes[:, 2 * j + 1])


# ------------------------------------------------------------- dequant ----

def test_awq005_no_plus_one_on_zeros():
    """AWQ-005: code == zero gives exactly 0; zero 0 and code 1 gives the scale."""
    K, N = 4, 8
    codes = np.full((K, N), 3)
    codes[1] = 1
    zeros = np.full((1, N), 3)
    zeros_row1 = np.zeros((1, N), dtype=np.int64)
    scales = np.full((1, N), 0.25, dtype=np.float16)
    W = oracle.dequant_f32(oracle.pack_codes(codes), oracle.pack_codes(zeros), scales, -1)
    assert np.all(W[0] == 0.0) and np.all(W[2:] == 0.0)
    assert np.all(W[1] == np.float32(-0.5))            # (1 - 3) * 0.25
    W2 = oracle.dequant_f32(oracle.pack_codes(codes), oracle.pack_codes(zeros_row1), scales, -1)
    assert np.all(W2[1] == np.float32(0.25))            # (1 - 0) * 0.25, no +1


def test_group_index_is_k_div_G():
    """Rows 0..G-1 use scale row 0, rows G..2G-1 scale row 1 (k // G)."""
    K, N, G = 8, 8, 4
    codes = np.full((K, N), 5)
    zeros = np.stack([np.full(N, 1), np.full(N, 2)])
    scales = np.stack([np.full(N, 1.0), np.full(N, 2.0)]).astype(np.float16)
    W = oracle.dequant_f32(oracle.pack_codes(codes), oracle.pack_codes(zeros), scales, G)
    assert np.all(W[:4] == 4.0) and np.all(W[4:] == 6.0)   # (5-1)*1, (5-2)*2


def test_group_minus_one_equals_group_K():
    d = awq_linear(11, 2, 64, 32, group_size=-1, bias=True)
    a = oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], -1)
    b = oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], 64)
    assert np.array_equal(a, b)
    assert d["scales"].shape == (1, 32) and d["qzeros"].shape == (1, 4)


def test_symmetric_zero_eight():
    d = awq_linear(12, 1, 32, 16, group_size=16, sym=True)
    assert np.all(d["qzeros"] == SYM_ZERO_WORD)
    codes = oracle.unpack_codes(d["qweight"]).astype(np.float32)
    W = oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], 16)
    s = d["scales"].astype(np.float32)[np.arange(32) // 16]
    assert np.array_equal(W, (codes - 8.0) * s)


def test_dequant_exact_rational_and_fp16_rne():
    d = awq_linear(13, 1, 256, 64, group_size=32)
    W32 = oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], 32)
    W16 = oracle.dequant_f16(d["qweight"], d["qzeros"], d["scales"], 32)
    rng = np.random.default_rng(0)
    for _ in range(400):
        k, n = int(rng.integers(256)), int(rng.integers(64))
        word = int(d["qweight"].view(np.uint32)[k, n // 8])
        zword = int(d["qzeros"].view(np.uint32)[k // 32, n // 8])
        nib = PAGE_ORDER.index(n % 8)
        c, z = (word >> 4 * nib) & 15, (zword >> 4 * nib) & 15
        exact = Fraction(c - z) * Fraction(float(d["scales"][k // 32, n]))
        assert Fraction(float(W32[k, n])) == exact
        # one round-to-nearest-even to fp16 (Python's half packing rounds half-even)
        assert struct.pack("<e", float(exact)) == W16[k, n].tobytes()


def test_page_layout_is_transpose():
    d = awq_linear(14, 1, 64, 24, group_size=16)
    P = oracle.dequant_page_layout(d["qweight"], d["qzeros"], d["scales"], 16)
    assert P.shape == (24, 64)
    assert np.array_equal(P, oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], 16).T)


def test_dequant_columns_matches_full():
    d = awq_linear(15, 1, 128, 80, group_size=32)
    W = oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], 32)
    cols = np.array([0, 1, 7, 8, 13, 42, 79, 79, 3])
    assert np.array_equal(oracle.dequant_columns_f32(d["qweight"], d["qzeros"], d["scales"], 32, cols),
                          W[:, cols])


def test_bad_group_size_rejected():
    with pytest.raises(ValueError):
        oracle.resolve_group_size(100, 48)
    with pytest.raises(ValueError):
        oracle.resolve_group_size(64, 0)


# ---------------------------------------------------------------- GEMM ----

def _brute_force_gemm(d):
    """Pure-Python restatement: for every (m, n) find the nibble holding column
    n by searching the page's ORDER list, decode code and zero with explicit
    shifts, and sum x * ((code - zero) * scale) with math.fsum."""
    x, qw, qz, sc, b = d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"]
    M, K = x.shape
    N = qw.shape[1] * 8
    G = K if d["group_size"] == -1 else d["group_size"]
    y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            nib = [i for i in range(8) if PAGE_ORDER[i] == n % 8][0]
            terms = []
            for k in range(K):
                word = int(qw[k, n // 8]) & 0xFFFFFFFF
                zword = int(qz[k // G, n // 8]) & 0xFFFFFFFF
                code = (word >> (4 * nib)) & 0xF
                zero = (zword >> (4 * nib)) & 0xF
                terms.append(float(x[m, k]) * ((code - zero) * float(sc[k // G, n])))
            if b is not None:
                terms.append(float(b[n]))
            y[m, n] = math.fsum(terms)
    return y


@pytest.mark.parametrize("M,K,N,G,bias", [(3, 32, 16, 8, True), (2, 48, 24, -1, False),
                                          (1, 64, 8, 16, True), (4, 16, 32, 16, False)])
def test_gemm_brute_force(M, K, N, G, bias):
    d = awq_linear(100 + M + K + N, M, K, N, group_size=G, bias=bias)
    y = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    yb = _brute_force_gemm(d)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12)


def test_gemm_exact_dyadic_case():
    """x small integers, scales powers of two, dyadic bias: every product and
    sum is exact, so the fp64 oracle equals exact rational arithmetic."""
    d = awq_linear(21, 3, 64, 16, group_size=16, bias=True, x_kind="smallint",
                   scale_kind="pow2", bias_kind="dyadic")
    y = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 16)
    codes = oracle.unpack_codes(d["qweight"])
    zeros = oracle.unpack_codes(d["qzeros"])
    for m in range(3):
        for n in range(16):
            acc = Fraction(float(d["bias"][n]))
            for k in range(64):
                acc += Fraction(int(d["x"][m, k])) * (codes[k, n] - zeros[k // 16, n]) * \
                    Fraction(float(d["scales"][k // 16, n]))
            assert Fraction(float(y[m, n])) == acc


def test_gemm_sampled_and_rows_match_full():
    d = awq_linear(22, 5, 96, 40, group_size=32, bias=True)
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 32)
    y = oracle.gemm(*args)
    rows = np.array([0, 4, 2, 2, 1])
    cols = np.array([0, 39, 17, 18, 8])
    np.testing.assert_allclose(oracle.gemm_sampled(*args, rows, cols), y[rows, cols], rtol=1e-13)
    np.testing.assert_allclose(oracle.gemm_rows(*args, [1, 3]), y[[1, 3]], rtol=1e-13)


def test_within_tolerance_definition():
    ok, worst = oracle.within_tolerance([1.0, 200.0], [1.009, 201.0])
    assert ok and worst < 1.0
    ok, _ = oracle.within_tolerance([0.0], [0.011])
    assert not ok
    ok, _ = oracle.within_tolerance([np.nan], [0.0])
    assert not ok


def test_synth_is_seeded_and_shaped():
    a = awq_linear(5, 2, 256, 64, group_size=128, bias=True)
    b = awq_linear(5, 2, 256, 64, group_size=128, bias=True)
    for key in ("x", "qweight", "qzeros", "scales", "bias"):
        assert np.array_equal(a[key], b[key])
    assert a["qweight"].shape == (256, 8) and a["qzeros"].shape == (2, 8)
    assert a["scales"].shape == (2, 64) and a["scales"].dtype == np.float16
    s = a["scales"].astype(np.float32)
    assert s.min() >= 9.99e-4 and s.max() <= 1.0001e-2
    codes = oracle.unpack_codes(awq_linear(6, 1, 512, 512)["qweight"])
    counts = np.bincount(codes.ravel(), minlength=16)
    assert counts.min() > 0.9 * codes.size / 16   # uniform codes 0..15


# ------------------------------------------------ round-to-nearest quantizer ----
# GPTQModel wiki "AWQ", "Group quantization and zero points": the asymmetric and symmetric
# 4-bit modes.  The pins below rest on a group worked by hand, on exact round trips of
# weights lying on a grid that spans the whole code range (the formulas then recover the
# grid exactly), and on the half-step error bound of rounding.

RTN_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rtn_worked_example.txt")


def _rtn_golden_rows():
    rows = []
    with open(RTN_GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            mode, w, scale_hex, zero, codes = line.split()
            rows.append((mode, [float(v) for v in w.split(",")], int(scale_hex, 16), int(zero),
                         [int(v) for v in codes.split(",")]))
    return rows


def _rtn_unpacked(w, G, sym):
    qw, qz, sc = oracle.quantize_rtn(w, G, sym)
    return oracle.unpack_codes(qw), oracle.unpack_codes(qz), sc


@pytest.mark.parametrize("row", _rtn_golden_rows(), ids=lambda r: f"{r[0]}:{r[1]}")
def test_rtn_worked_example(row):
    mode, vals, scale_bits, zero, codes = row
    # every output channel (row of the [N, K] weight) holds the worked group
    w = np.tile(np.array(vals, dtype=np.float16), (8, 1))
    c, z, sc = _rtn_unpacked(w, 4, mode == "sym")
    assert c.shape == (4, 8) and z.shape == (1, 8) and sc.shape == (1, 8)
    assert (c == np.array(codes)[:, None]).all()
    assert (z == zero).all()
    assert (sc.view(np.uint16) == scale_bits).all()


def _grid_weight(rng, N, K, G, sym):
    """W[n, k] = (code - zero) * s with s a power of two, every group spanning the full
    code range (asymmetric: codes 0 and 15 present; symmetric: -7 or 7 as the largest
    magnitude), so the page's formulas must give back codes, zeros and scales exactly."""
    ng = K // G
    p = rng.integers(4, 12, size=(N, ng))
    s = np.ldexp(1.0, -p)                                     # exact in fp16
    if sym:
        code = rng.integers(-7, 8, size=(N, ng, G))
        code[:, :, 0] = np.where(rng.random((N, ng)) < 0.5, -7, 7)
        zero = np.full((N, ng), 8)
        w = code * s[:, :, None]
        code = code + 8
    else:
        code = rng.integers(0, 16, size=(N, ng, G))
        code[:, :, 0] = 0
        code[:, :, 1] = 15
        zero = rng.integers(0, 16, size=(N, ng))
        w = (code - zero[:, :, None]) * s[:, :, None]
    w16 = w.reshape(N, K).astype(np.float16)
    assert np.array_equal(w16.astype(np.float64), w.reshape(N, K))  # on the grid exactly
    return w16, code.reshape(N, K), zero, s


@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("N,K,G", [(8, 32, 16), (16, 64, 64), (24, 96, 32)])
def test_rtn_recovers_grid_exactly(sym, N, K, G):
    rng = np.random.default_rng(N * K + G + sym)
    w16, code, zero, s = _grid_weight(rng, N, K, G, sym)
    c, z, sc = _rtn_unpacked(w16, G, sym)
    assert np.array_equal(c, code.T)
    assert np.array_equal(z, zero.T)
    assert np.array_equal(sc.astype(np.float64), s.T)


def test_rtn_error_is_at_most_half_a_step():
    rng = np.random.default_rng(7)
    N, K, G = 32, 256, 64
    w16 = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    c, z, sc = _rtn_unpacked(w16, G, False)
    s = sc.astype(np.float64)[np.arange(K) // G]             # [K, N]
    rec = (c - z[np.arange(K) // G]) * s
    err = np.abs(rec - w16.astype(np.float64).T)
    # the range holds 15 steps, so no code or zero clamps for these groups
    assert (err <= 0.5 * s * (1 + 1e-3)).all()


def test_rtn_symmetric_zero_is_eight_and_zero_maps_to_eight():
    rng = np.random.default_rng(8)
    w16 = (rng.standard_normal((16, 128)) * 0.1).astype(np.float16)
    w16[:, 5] = 0
    c, z, _ = _rtn_unpacked(w16, 32, True)
    assert (z == 8).all()
    assert (c[5] == 8).all()


def test_rtn_group_minus_one_equals_group_k():
    rng = np.random.default_rng(9)
    w16 = rng.standard_normal((8, 96)).astype(np.float16)
    for sym in (False, True):
        a = oracle.quantize_rtn(w16, -1, sym)
        b = oracle.quantize_rtn(w16, 96, sym)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_rtn_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.quantize_rtn(np.zeros((12, 64), np.float16), 32)
    with pytest.raises(ValueError):
        oracle.quantize_rtn(np.zeros((8, 64), np.float16), 24)
    with pytest.raises(ValueError):
        oracle.quantize_rtn(np.zeros((8, 64), np.float32), 32)


# ------------------------------------------------------------------ bf16 ----
# bf16 = the upper 16 bits of an fp32 (7 stored significand bits); rounding to nearest, ties
# to even.  Worked by hand around 1.0 (ulp 2^-7) and checked against torch's own conversion.

def test_bf16_rounding_hand_worked():
    one = 1.0
    cases = [
        (one + 2.0 ** -8, one),                         # exactly half an ulp: tie, to even (1.0)
        (one + 3 * 2.0 ** -8, one + 2.0 ** -6),         # 1.5 ulp: tie between m=1 and m=2, to even
        (one + 2.0 ** -8 + 2.0 ** -20, one + 2.0 ** -7),  # just above half: up
        (one + 2.0 ** -8 - 2.0 ** -20, one),            # just below half: down
        (-(one + 3 * 2.0 ** -8), -(one + 2.0 ** -6)),   # sign symmetric
        (0.0, 0.0),
        (3.0, 3.0),                                     # exact values unchanged
    ]
    got = oracle.round_to_bf16(np.array([c[0] for c in cases], dtype=np.float32))
    assert np.array_equal(got, np.array([c[1] for c in cases], dtype=np.float32))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    v = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 20000),
                        np.array([1e-40, -3e-39, 65504.0, 3.3e38, 1.0 + 2 ** -8], dtype=np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    assert np.array_equal(oracle.round_to_bf16(v).view(np.uint32), ref.view(np.uint32))


def test_dequant_bf16_is_one_rounding_of_the_exact_value():
    d = awq_linear(41, 1, 64, 16, group_size=32, dtype="bf16")
    exact = oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], 32)
    got = oracle.dequant_bf16(d["qweight"], d["qzeros"], d["scales"], 32)
    assert np.array_equal(got, oracle.round_to_bf16(exact))
    # the bf16 value is within half a bf16 ulp of the exact one
    assert (np.abs(got - exact) <= np.abs(exact) * 2.0 ** -8 + 1e-30).all()


# ------------------------------------------------------- grouped (MoE) ----
# vLLM article, section 5.4: routed expert layers with 4-bit AWQ weights.  The grouped oracle
# must reduce to the pinned single-linear GEMM: identical experts give one GEMM over all
# rows; empty experts own no rows; relabelling experts (and moving their row blocks) only
# moves rows.

def test_grouped_identical_experts_equal_one_gemm():
    from synth import moe_inputs
    d = moe_inputs(51, 12, 2, 4, 64, 16, group_size=32, bias=True)
    qw = np.stack([d["qweight"][0]] * 4)
    qz = np.stack([d["qzeros"][0]] * 4)
    sc = np.stack([d["scales"][0]] * 4)
    b = np.stack([d["bias"][0]] * 4)
    y = oracle.gemm_grouped(d["x"], qw, qz, sc, b, 32, d["offsets"])
    assert np.array_equal(y, oracle.gemm(d["x"], qw[0], qz[0], sc[0], b[0], 32))


def test_grouped_blocks_and_empty_experts():
    from synth import moe_inputs
    d = moe_inputs(52, 5, 1, 8, 64, 16, group_size=-1)   # 5 rows over 8 experts: some empty
    offs = d["offsets"]
    assert (np.diff(offs) == 0).any()
    y = oracle.gemm_grouped(d["x"], d["qweight"], d["qzeros"], d["scales"], None, -1, offs)
    for e in range(8):
        a, b = offs[e], offs[e + 1]
        ref = oracle.gemm(d["x"][a:b], d["qweight"][e], d["qzeros"][e], d["scales"][e], None, -1)
        assert np.array_equal(y[a:b], ref)


def test_grouped_relabelling_moves_rows():
    from synth import moe_inputs
    d = moe_inputs(53, 9, 2, 3, 64, 16, group_size=32)
    offs = d["offsets"]
    y = oracle.gemm_grouped(d["x"], d["qweight"], d["qzeros"], d["scales"], None, 32, offs)
    perm = [2, 0, 1]  # new expert i is old expert perm[i]
    blocks = [np.arange(offs[p], offs[p + 1]) for p in perm]
    rows = np.concatenate(blocks)
    new_offs = np.concatenate([[0], np.cumsum([len(b) for b in blocks])])
    y2 = oracle.gemm_grouped(d["x"][rows], d["qweight"][perm], d["qzeros"][perm], d["scales"][perm],
                             None, 32, new_offs)
    assert np.array_equal(y2, y[rows])


def test_grouped_rejects_bad_offsets():
    from synth import moe_inputs
    d = moe_inputs(54, 4, 1, 2, 64, 16, group_size=32)
    with pytest.raises(ValueError):
        oracle.gemm_grouped(d["x"], d["qweight"], d["qzeros"], d["scales"], None, 32, [0, 3, 2])


# ---------------------------------------------------------------- 8-bit ----
# GPTQModel wiki "AWQ", "Saved formats and packing": widths other than 4 pack as a continuous
# little-endian bit stream (no INT4 order).  Worked by hand: columns 0..3 holding codes
# 0x01, 0x02, 0x03, 0x04 make the word 0x04030201; column 3 = 0xFF makes the sign byte.

def test_w8_hand_packed_words():
    w = np.array([[0x04030201, 0xFF000000]], dtype=np.uint32).view(np.int32)
    assert oracle.unpack_codes8(w).tolist() == [[1, 2, 3, 4, 0, 0, 0, 255]]
    assert np.array_equal(oracle.pack_codes8(np.array([[1, 2, 3, 4, 0, 0, 0, 255]])), w)


def test_w8_round_trip_and_rejects():
    rng = np.random.default_rng(61)
    words = rng.integers(0, 1 << 32, size=(5, 6), dtype=np.uint64).astype(np.uint32).view(np.int32)
    assert np.array_equal(oracle.pack_codes8(oracle.unpack_codes8(words)), words)
    with pytest.raises(ValueError):
        oracle.pack_codes8(np.zeros((1, 6), np.int64))
    with pytest.raises(ValueError):
        oracle.pack_codes8(np.full((1, 4), 256))


def test_w8_dequant_exact_values_and_zero_point():
    # code == zero gives exactly 0 (no +1, as for 4 bits); code 255 - zero 0 times scale
    codes = np.array([[7, 255, 0, 128]] * 4)
    zeros = np.array([[7, 0, 0, 200]])
    scales = np.array([[0.5, 2.0 ** -10, 3.0, 0.25]], dtype=np.float16)
    W = oracle.dequant8_f32(oracle.pack_codes8(codes), oracle.pack_codes8(zeros), scales, 4)
    assert W[0].tolist() == [0.0, 255 * 2.0 ** -10, 0.0, (128 - 200) * 0.25]


def test_w8_gemm_brute_force():
    d = synth.awq8_linear(62, 3, 32, 8, group_size=16, bias=True)
    y = oracle.gemm8(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 16)
    K, N = 32, 8
    for m in range(3):
        for n in range(N):
            terms = []
            for k in range(K):
                word = int(d["qweight"][k, n // 4]) & 0xFFFFFFFF
                zword = int(d["qzeros"][k // 16, n // 4]) & 0xFFFFFFFF
                code = (word >> (8 * (n % 4))) & 0xFF
                zero = (zword >> (8 * (n % 4))) & 0xFF
                terms.append(float(d["x"][m, k]) * ((code - zero) * float(d["scales"][k // 16, n])))
            terms.append(float(d["bias"][n]))
            assert abs(y[m, n] - math.fsum(terms)) <= 1e-12 * max(1.0, abs(y[m, n]))


# ------------------------------------------------------------ tile-packed layout ----

def _packed_case(name):
    """The two hand-worked inputs of tests/golden/packed_layout.txt."""
    if name == "A":
        K, N, G = 64, 8, 64
    else:
        K, N, G = 128, 136, 64
    k = np.arange(K)[:, None]
    n = np.arange(N)[None, :]
    codes = (k + n) % 16
    g = np.arange(K // G)[:, None]
    if name == "A":
        zeros = np.broadcast_to(n % 16, (1, N))
        scales = (1.0 + n / 8.0).astype(np.float16)
    else:
        zeros = (n + 3 * g) % 16
        scales = np.broadcast_to(2.0 ** -(g + 1.0), (K // G, N)).astype(np.float16)
    return (oracle.pack_codes(codes), oracle.pack_codes(np.ascontiguousarray(zeros)),
            np.ascontiguousarray(scales), K, N, G)


def _golden_packed():
    path = os.path.join(os.path.dirname(__file__), "golden", "packed_layout.txt")
    sizes, words = {}, []
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "size":
            sizes[f[1]] = int(f[2])
        else:
            words.append((f[0], int(f[1]), int(f[2], 16)))
    return sizes, words


def test_packed_layout_golden_words():
    sizes, words = _golden_packed()
    packed = {}
    for name in ("A", "B"):
        qw, qz, sc, K, N, G = _packed_case(name)
        packed[name] = oracle.repack(qw, qz, sc, G)
        assert packed[name].size == sizes[name]
        assert oracle.repack_size(K, N, G) == 4 * sizes[name]
    for name, idx, want in words:
        assert int(packed[name][idx]) == want, (name, idx, hex(int(packed[name][idx])))


@pytest.mark.parametrize("K,N,G", [(64, 8, 64), (128, 136, 64), (256, 384, 128), (512, 264, -1),
                                   (192, 1032, 64), (1024, 128, 256)])
def test_packed_round_trip_is_lossless(K, N, G):
    # repack -> read back == the checkpoint reader's codes, zeros and scales (pinned to the
    # pages above); the layout is only a permutation plus padding
    d = awq_linear(300 + K + N, 1, K, N, group_size=G)
    pk = oracle.repack(d["qweight"], d["qzeros"], d["scales"], G)
    codes, zeros, sc = oracle.unpack_repacked(pk, K, N, G)
    assert np.array_equal(codes, oracle.unpack_codes(d["qweight"]))
    assert np.array_equal(zeros, oracle.unpack_codes(d["qzeros"]))
    assert np.array_equal(sc.view(np.uint16), d["scales"].view(np.uint16))


def test_packed_scale_words_pass_through():
    # the layout stores each scale's 16-bit word unchanged: fp16 words give the fp16 layout, and
    # bf16 words (bf16 scales) read back bit for bit
    K, N, G = 256, 264, 64
    d = awq_linear(305, 1, K, N, group_size=G)
    pk = oracle.repack(d["qweight"], d["qzeros"], d["scales"], G)
    assert np.array_equal(oracle.repack(d["qweight"], d["qzeros"], d["scales"].view(np.uint16), G), pk)
    db = awq_linear(306, 1, K, N, group_size=G, dtype="bf16")
    words = (np.ascontiguousarray(db["scales"], dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((words.astype(np.uint32) << 16).view(np.float32), db["scales"].astype(np.float32))
    pkb = oracle.repack(db["qweight"], db["qzeros"], words, G)
    codes, zeros, sc = oracle.unpack_repacked(pkb, K, N, G)
    assert np.array_equal(sc.view(np.uint16), words)
    assert np.array_equal(codes, oracle.unpack_codes(db["qweight"]))
    assert np.array_equal(zeros, oracle.unpack_codes(db["qzeros"]))


def oracle_w8_case(seed, K, N, G, M=1, bias=False):
    return synth.awq8_linear(seed, M, K, N, group_size=G, bias=bias)


def test_packed8_hand_derived_words():
    # K = 64, N = 4 (one 8-bit word per row), code[k][n] = k + 64 n, zero 0x2A in column 1,
    # scale 1.0 (0x3C00): words written out by hand from the layout's definition
    K, N, G = 64, 4, 64
    codes = np.array([[k + 64 * n for n in range(N)] for k in range(K)])
    zeros = np.zeros((1, N), dtype=np.int64)
    zeros[0, 1] = 0x2A
    qw, qz = oracle.pack_codes8(codes), oracle.pack_codes8(zeros)
    sc = np.full((1, N), 1.0, dtype=np.float16)
    pk = oracle.repack8(qw, qz, sc, G)
    assert pk.size * 4 == oracle.repack8_size(K, N, G) == 8704
    assert int(pk[0]) == 0x03020100                 # h 0, k 0, column 0, j 0: rows 0..3
    assert int(pk[1]) == 0x07060504                 # j 1: rows 4..7
    assert int(pk[4]) == 0x43424140                 # column 1 (codes 64 + row): rows 0..3
    assert int(pk[512 + 4 * 2 + 3]) == 0x9F9E9D9C   # k 1, column 2, j 3: rows 28..31 -> 156..159
    assert int(pk[1024 + 512 + 4 * 3 + 3]) == 0xFFFEFDFC  # h 1, k 1, column 3, j 3: rows 60..63
    assert int(pk[2048 + 1]) == (0x2A << 16) | 0x3C00     # meta of column 1
    assert int(pk[2048 + 0]) == 0x3C00
    assert not pk[4 * 4:512].any() and not pk[2048 + 4:].any()   # columns 4..127: padding


@pytest.mark.parametrize("K,N,G", [(64, 4, 64), (128, 136, 64), (256, 384, 128), (512, 260, -1)])
def test_packed8_round_trip_is_lossless(K, N, G):
    d = oracle_w8_case(330 + K + N, K, N, G)
    pk = oracle.repack8(d["qweight"], d["qzeros"], d["scales"], G)
    codes, zeros, sc = oracle.unpack_repacked8(pk, K, N, G)
    assert np.array_equal(codes, oracle.unpack_codes8(d["qweight"]))
    assert np.array_equal(zeros, oracle.unpack_codes8(d["qzeros"]))
    assert np.array_equal(sc.view(np.uint16), d["scales"].view(np.uint16))


def test_packed8_gemm_equals_checkpoint_gemm():
    d = oracle_w8_case(340, 256, 264, 64, M=3, bias=True)
    pk = oracle.repack8(d["qweight"], d["qzeros"], d["scales"], 64)
    y = oracle.gemm_packed8(d["x"], pk, d["bias"], 256, 264, 64)
    assert np.array_equal(y, oracle.gemm8(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 64))


def test_packed8_rejects_unsupported_shapes():
    for K, N, G in [(96, 64, 32), (128, 64, 32), (64, 6, 64)]:
        with pytest.raises(ValueError):
            oracle.repack8_size(K, N, G)


def test_packed_padding_and_group_copies():
    # columns past N are all-zero words; every stage of a group carries the same meta row
    K, N, G = 256, 136, 128
    d = awq_linear(310, 1, K, N, group_size=G)
    pk = oracle.repack(d["qweight"], d["qzeros"], d["scales"], G).reshape(2, K // 64, 1152)
    assert not pk[1, :, 8 * 4:512].any() and not pk[1, :, 512 + 8 * 4:1024].any()
    assert not pk[1, :, 1024 + 8:].any()
    assert np.array_equal(pk[:, 0, 1024:], pk[:, 1, 1024:])
    assert np.array_equal(pk[:, 2, 1024:], pk[:, 3, 1024:])
    assert not np.array_equal(pk[:, 1, 1024:], pk[:, 2, 1024:])


def test_packed_gemm_equals_checkpoint_gemm():
    d = awq_linear(320, 3, 256, 264, group_size=64, bias=True)
    pk = oracle.repack(d["qweight"], d["qzeros"], d["scales"], 64)
    y = oracle.gemm_packed(d["x"], pk, d["bias"], 256, 264, 64)
    assert np.array_equal(y, oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 64))


def test_packed_rejects_unsupported_shapes():
    for K, N, G in [(96, 64, 32), (128, 64, 32), (64, 12, 64)]:
        with pytest.raises(ValueError):
            oracle.repack_size(K, N, G)
