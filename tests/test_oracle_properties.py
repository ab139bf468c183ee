"""Property tests of the oracle (no GPU): exact algebraic relations of the dequant and the
linear that any slip in the oracle (a dropped term, a wrong sign, a transposed operand, a
wrong group index) would break, on random shapes and values.  The relations follow from
the definition on the format page ("Reader": w = (code - zero) * scale with the group row
k // G; y = x W + bias) and hold exactly in fp64 for the integer-valued inputs used."""
import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies
given, settings = hypothesis.given, hypothesis.settings


def _linear(rng, M, K, N, G, bits=4, int_x=True):
    per = 32 // bits
    hi = (1 << bits)
    codes = rng.integers(0, hi, size=(K, N))
    zeros = rng.integers(0, hi, size=(K // G, N))
    pack = oracle.pack_codes if bits == 4 else oracle.pack_codes8
    qw, qz = pack(codes), pack(zeros)
    p = rng.integers(6, 12, size=(K // G, N))
    sc = np.ldexp(np.ones((K // G, N)), -p).astype(np.float16)  # powers of two: exact products
    x = (rng.integers(-3, 4, size=(M, K)) if int_x else rng.standard_normal((M, K))).astype(np.float16)
    return x, qw, qz, sc, codes, zeros


dims = st.tuples(st.integers(1, 5), st.sampled_from([8, 16, 32, 64]), st.integers(1, 4), st.integers(1, 4))


@settings(max_examples=40, deadline=None)
@given(dims, st.integers(0, 2**31 - 1))
def test_dequant_is_code_minus_zero_times_scale(d, seed):
    M, G, ng, nw = d
    K, N = G * ng, 8 * nw
    rng = np.random.default_rng(seed)
    x, qw, qz, sc, codes, zeros = _linear(rng, M, K, N, G)
    w = oracle.dequant_f32(qw, qz, sc, G)
    g = np.arange(K) // G
    assert np.array_equal(w, ((codes - zeros[g]) * sc.astype(np.float64)[g]).astype(np.float32))
    # the unpacked codes are the packed ones, whatever the word bits
    assert np.array_equal(oracle.unpack_codes(qw), codes)


@settings(max_examples=40, deadline=None)
@given(dims, st.integers(0, 2**31 - 1), st.integers(-3, 3))
def test_linear_in_x_and_additive_in_bias(d, seed, e):
    M, G, ng, nw = d
    K, N = G * ng, 8 * nw
    rng = np.random.default_rng(seed)
    x, qw, qz, sc, _, _ = _linear(rng, M, K, N, G)
    b = np.ldexp(rng.integers(-64, 65, size=N), -6).astype(np.float16)
    y0 = oracle.gemm(x, qw, qz, sc, None, G)
    # scaling x by a power of two scales y exactly; a bias adds exactly
    xs = (x.astype(np.float64) * 2.0 ** e).astype(np.float16)
    assert np.array_equal(oracle.gemm(xs, qw, qz, sc, None, G), y0 * 2.0 ** e)
    assert np.array_equal(oracle.gemm(x, qw, qz, sc, b, G), y0 + b.astype(np.float64)[None, :])
    # rows are independent: a row permutation of x permutes y
    perm = rng.permutation(M)
    assert np.array_equal(oracle.gemm(x[perm], qw, qz, sc, None, G), y0[perm])


@settings(max_examples=30, deadline=None)
@given(dims, st.integers(0, 2**31 - 1))
def test_zero_shift_is_minus_scale_times_row_sum(d, seed):
    # raising every zero of group g by 1 changes y by -x_g . scale_g (exactly, small ints)
    M, G, ng, nw = d
    K, N = G * ng, 8 * nw
    rng = np.random.default_rng(seed)
    x, qw, qz, sc, codes, zeros = _linear(rng, M, K, N, G)
    zeros = np.minimum(zeros, 14)
    qz = oracle.pack_codes(zeros)
    y0 = oracle.gemm(x, qw, qz, sc, None, G)
    y1 = oracle.gemm(x, qw, oracle.pack_codes(zeros + 1), sc, None, G)
    xs = x.astype(np.float64).reshape(M, ng, G).sum(axis=2)   # [M, groups]
    assert np.array_equal(y1 - y0, -(xs @ sc.astype(np.float64)))


@settings(max_examples=30, deadline=None)
@given(dims, st.integers(0, 2**31 - 1))
def test_columns_are_independent(d, seed):
    # column n of y depends only on column n of the weights: splitting N at word
    # boundaries and concatenating gives the same y (the column-parallel shard)
    M, G, ng, nw = d
    K, N = G * ng, 8 * nw
    rng = np.random.default_rng(seed)
    x, qw, qz, sc, _, _ = _linear(rng, M, K, N, G)
    y = oracle.gemm(x, qw, qz, sc, None, G)
    c = nw // 2 if nw > 1 else 1
    if c >= nw:
        return
    ya = oracle.gemm(x, qw[:, :c], qz[:, :c], sc[:, :8 * c], None, G)
    yb = oracle.gemm(x, qw[:, c:], qz[:, c:], sc[:, 8 * c:], None, G)
    assert np.array_equal(np.concatenate([ya, yb], axis=1), y)


@settings(max_examples=30, deadline=None)
@given(st.tuples(st.integers(1, 4), st.sampled_from([8, 16, 32]), st.integers(1, 3), st.integers(1, 4)),
       st.integers(0, 2**31 - 1))
def test_8bit_dequant_and_linear(d, seed):
    M, G, ng, nw = d
    K, N = G * ng, 4 * nw
    rng = np.random.default_rng(seed)
    x, qw, qz, sc, codes, zeros = _linear(rng, M, K, N, G, bits=8)
    w = oracle.dequant8_f32(qw, qz, sc, G)
    g = np.arange(K) // G
    assert np.array_equal(w, ((codes - zeros[g]) * sc.astype(np.float64)[g]).astype(np.float32))
    y = oracle.gemm8(x, qw, qz, sc, None, G)
    assert np.array_equal(y, x.astype(np.float64) @ w.astype(np.float64))
