"""Two-oracle agreement (no GPU): the C oracle (oracle/awq_oracle_c.c) and the numpy oracle
are written separately from the same definitions (format page "Reader"; GPTQModel wiki
"AWQ", "Saved formats and packing" for 8-bit codes), so a slip in either one shows here.
Dequant must agree bit for bit; the fp64 GEMMs (sequential k in C, BLAS order in numpy)
within 1e-12 relative; on exact-arithmetic inputs both must give the same bits."""
import os

import numpy as np
import pytest

import oracle
import synth
from oracle import c_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "awq_word_layout.txt")


def test_binary16_decoding_matches_numpy_for_every_pattern():
    # the C oracle widens fp16 by decoding the IEEE fields itself; numpy's conversion is
    # the library routine it must reproduce, on all 65536 bit patterns
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    mine = c_oracle.widen_f16(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_hand_packed_word():
    # codes 0..7 for columns 0..7 pack to 0x75316420 (format page ORDER); zero 0, scale 1
    word = np.array([[0x75316420]], dtype=np.uint32).view(np.int32)
    w = c_oracle.dequant_f32(word, np.zeros((1, 1), np.int32), np.ones((1, 8), np.float16), -1)
    assert w.tolist() == [[0, 1, 2, 3, 4, 5, 6, 7]]
    assert "0x75316420" in open(GOLDEN).read()


def test_sign_word_and_no_plus_one():
    # 0xF0000000: column 7 = 15 (the word is negative as int32); zero = code gives exactly 0
    word = np.array([[0xF0000000]], dtype=np.uint32).view(np.int32)
    w = c_oracle.dequant_f32(word, np.zeros((1, 1), np.int32), np.ones((1, 8), np.float16), -1)
    assert w.tolist() == [[0, 0, 0, 0, 0, 0, 0, 15]]
    w = c_oracle.dequant_f32(word, word, np.full((1, 8), 0.5, np.float16), -1)
    assert not w.any()


@pytest.mark.parametrize("K,N,G", [(256, 256, 128), (48, 24, 16), (64, 32, -1), (1000, 8, 8),
                                   (512, 1024, 64)])
def test_dequant_agrees_bitwise(K, N, G):
    d = synth.awq_linear(3100 + K + N, 1, K, N, group_size=G)
    a = c_oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], G)
    b = oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], G)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("M,K,N,G,bias", [(1, 256, 256, 128, False), (5, 512, 192, 64, True),
                                          (33, 1024, 64, -1, True), (3, 200, 64, 8, False)])
def test_gemm_agrees(M, K, N, G, bias):
    d = synth.awq_linear(3200 + M + K, M, K, N, group_size=G, bias=bias)
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    a, b = c_oracle.gemm(*args), oracle.gemm(*args)
    assert np.all(np.abs(a - b) <= 1e-12 * np.maximum(1.0, np.abs(b)))


def test_gemm_exact_case_agrees_bitwise():
    # small-integer x, power-of-two scales, dyadic bias: every sum is exact in fp64 on any
    # order, so the two oracles must agree to the bit
    d = synth.awq_linear(3300, 7, 1024, 256, group_size=128, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic")
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128)
    assert np.array_equal(c_oracle.gemm(*args), oracle.gemm(*args))


@pytest.mark.parametrize("K,N,G", [(256, 256, 128), (48, 12, 16), (64, 4, -1)])
def test_8bit_agrees(K, N, G):
    d = synth.awq8_linear(3400 + K + N, 3, K, N, group_size=G, bias=True)
    a = c_oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], G, bits=8)
    b = oracle.dequant8_f32(d["qweight"], d["qzeros"], d["scales"], G)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    ya, yb = c_oracle.gemm(*args, bits=8), oracle.gemm8(*args)
    assert np.all(np.abs(ya - yb) <= 1e-12 * np.maximum(1.0, np.abs(yb)))


def test_invalid_shapes_are_refused():
    qw = np.zeros((96, 4), np.int32)
    with pytest.raises(ValueError):
        c_oracle.dequant_f32(qw, np.zeros((1, 4), np.int32), np.zeros((1, 32), np.float16), 64)
