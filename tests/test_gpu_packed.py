"""GPU parity of the tile-packed layout (awq_repack, awq_gemm_packed) against the CPU oracle
on the same seeded inputs: the repacked words must equal the oracle's bit for bit (the
layout is a lossless permutation plus padding); the linear on the packed weights must
satisfy |y - y_ref| <= 1e-2 * max(1, |y_ref|) elementwise (fp16 output, fp32
accumulation, y_ref fp64) and be bit-exact where every partial sum is exact."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def awq():
    from w4a16_weight_only_gb300 import build
    build.build()
    import w4a16_weight_only_gb300 as awq
    assert awq.runtime_available(), awq.last_error()
    return awq


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def packed_of(awq, d):
    return awq.awq_repack(dev(d["qweight"]), dev(d["qzeros"]), dev(d["scales"]), d["group_size"])


def run(awq, d, pk=None):
    pk = packed_of(awq, d) if pk is None else pk
    b = None if d["bias"] is None else dev(d["bias"])
    y = awq.awq_gemm_packed(dev(d["x"]), pk, b, d["K"], d["N"], d["group_size"])
    torch.cuda.synchronize()
    return y.cpu().numpy()


def assert_close(y, y_ref, what):
    ok, worst = oracle.within_tolerance(y.astype(np.float64), y_ref, 1e-2)
    assert ok, f"{what}: worst |err|/(1e-2*max(1,|ref|)) = {worst:.3f}"


@pytest.mark.parametrize("K,N,G", [(64, 8, 64), (128, 136, 64), (256, 384, 128), (512, 264, -1),
                                   (4096, 4096, 128), (11008, 4096, 128), (4096, 11008, -1),
                                   (1024, 1032, 256)])
def test_repack_bit_exact(awq, K, N, G):
    d = synth.awq_linear(21000 + K + N, 1, K, N, group_size=G)
    got = packed_of(awq, d)
    torch.cuda.synchronize()
    assert got.numel() * 4 == awq.awq_repack_size(K, N, G) == oracle.repack_size(K, N, G)
    want = oracle.repack(d["qweight"], d["qzeros"], d["scales"], G)
    assert np.array_equal(got.cpu().numpy().view(np.uint32), want)


# token tiles of 64 (M <= 64), 128 (M <= 128) and 256 rows, ragged rows and column tiles,
# one group per K (G = -1), several tiles per CTA
SMALL = [(1, 256, 256, 128, False), (17, 512, 136, 64, True), (64, 1024, 264, 128, True),
         (65, 256, 128, -1, False), (128, 2048, 512, 256, True), (129, 512, 392, 64, True),
         (256, 1024, 256, 128, False), (300, 768, 1032, 64, True), (600, 512, 520, 128, True),
         (1000, 256, 128, 64, False)]


@pytest.mark.parametrize("M,K,N,G,bias", SMALL)
def test_gemm_packed_vs_oracle(awq, M, K, N, G, bias):
    d = synth.awq_linear(22000 + M + K + N, M, K, N, group_size=G, bias=bias)
    y = run(awq, d)
    y_ref = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    assert_close(y, y_ref, f"packed M={M} K={K} N={N} G={G}")


@pytest.mark.parametrize("M", [1, 40, 100, 256, 300])
def test_gemm_packed_exact_case_bitwise(awq, M):
    # small-integer x, power-of-two scales, dyadic bias: every product and partial sum is
    # exact in fp32, so y is the oracle's value rounded once to fp16
    d = synth.awq_linear(23000 + M, M, 2048, 392, group_size=128, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic")
    y = run(awq, d)
    want = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("M,K,N", [(300, 8192, 512), (256, 8192, 256), (512, 8192, 384), (260, 4096, 512)])
def test_gemm_packed_long_k_pairs(awq, M, K, N):
    # K >= 8192 with an even number of 128-column tiles runs the two-CTA (cta_group::2) kernel,
    # an odd number (N = 384) and K = 4096 the single-CTA one; exact-arithmetic inputs make
    # both bitwise checkable, random ones check the tolerance
    d = synth.awq_linear(23200 + M + N, M, K, N, group_size=128, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic")
    y = run(awq, d)
    want = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), want.view(np.uint16))
    d = synth.awq_linear(23300 + M + N, M, K, N, group_size=128, bias=True)
    assert_close(run(awq, d), oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128),
                 f"packed M={M} K={K} N={N}")


# narrow token tiles (32 / 64 / 128 rows) with K split over clusters of 2 or 4 CTAs, chosen by
# tile count: 8 tiles of 32 rows (4-way), 4 of 64 (2-way), 8 of 128 (2-way), an uneven split
# (K = 4160: 65 stages), a persistent unsplit launch (N = 28672: 224 tiles)
NARROW = [(16, 4096, 1024), (32, 4096, 1024), (48, 2048, 512), (100, 4096, 1024), (9, 4160, 512),
          (1, 4096, 4096), (24, 8192, 28672), (128, 11008, 4096)]


@pytest.mark.parametrize("M,K,N", NARROW)
def test_gemm_packed_narrow_split(awq, M, K, N):
    d = synth.awq_linear(23400 + M + K, M, K, N, group_size=64, bias=True)
    y = run(awq, d)
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 64)
    if K * N <= 64 * 1024 * 1024:
        assert_close(y, oracle.gemm(*args), f"packed narrow M={M} K={K} N={N}")
    else:
        rng = np.random.default_rng(6)
        rows = np.concatenate([rng.integers(0, M, 2048), [0, M - 1]])
        cols = np.concatenate([rng.integers(0, N, 2048), [0, N - 1]])
        assert_close(y[rows, cols], oracle.gemm_sampled(*args, rows, cols), f"packed narrow M={M} K={K} N={N}")
    assert np.array_equal(run(awq, d).view(np.uint16), y.view(np.uint16))  # fixed reduction order


@pytest.mark.parametrize("M", [8, 32, 64, 128])
def test_gemm_packed_narrow_split_exact_bitwise(awq, M):
    # exact-arithmetic inputs: the split partial sums are exact in fp32, so y is the oracle's
    # value rounded once to fp16 whatever the split
    d = synth.awq_linear(23600 + M, M, 4096, 1024, group_size=128, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic")
    y = run(awq, d)
    want = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), want.view(np.uint16))


# Small batches (M <= 32: 16- or 32-row token tiles, several CTAs per SM, K split over a
# cluster of 1 .. 16 CTAs, each rank finishing a slice of the columns): one stage in all (no
# split), two, five (a 5-CTA cluster), a 16-CTA cluster (few column tiles), ragged column
# tiles, G = 64 / 128 / -1, the 7B shapes
SMALLB = [(1, 64, 128, 64, True), (2, 128, 136, 64, False), (5, 320, 264, 64, True), (16, 4096, 512, 128, True),
          (17, 1024, 1032, -1, True), (31, 2048, 384, 128, False), (32, 4096, 11008, 128, True),
          (16, 11008, 4096, 128, False), (8, 4096, 4096, 128, True)]


@pytest.mark.parametrize("M,K,N,G,bias", SMALLB)
def test_gemm_packed_small_batch(awq, M, K, N, G, bias):
    d = synth.awq_linear(24000 + M + K + N, M, K, N, group_size=G, bias=bias)
    y = run(awq, d)
    assert_close(y, oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G),
                 f"packed small M={M} K={K} N={N} G={G}")
    assert np.array_equal(run(awq, d).view(np.uint16), y.view(np.uint16))  # fixed reduction order


@pytest.mark.parametrize("M,K,N", [(1, 4096, 520), (16, 4096, 520), (17, 1024, 4096), (32, 4096, 520), (32, 320, 136)])
def test_gemm_packed_small_batch_exact_bitwise(awq, M, K, N):
    # exact-arithmetic inputs: every rank's partial sums are exact in fp32, so y is the
    # oracle's value rounded once to fp16 whatever the cluster size
    d = synth.awq_linear(24500 + M + K, M, K, N, group_size=64, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic")
    y = run(awq, d)
    want = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 64).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), want.view(np.uint16))


# Stream-K (awq_gemm_packed_ws): shapes whose 256-row tiles fill the SMs poorly, with K
# stages cut between CTAs (a tile spread over several CTAs at 257 x 4096 x 2048), ragged rows
# and columns, G = 64 / 128 / -1, and a long-K shape the pair kernel would otherwise take
# (up to three contributors per finished tile at 512 x 11008 x 4096)
SK = [(257, 4096, 2048, 128, True), (384, 4096, 2048, -1, True), (700, 8192, 1032, 64, True),
      (512, 4096, 11008, 128, False), (512, 11008, 4096, 128, True)]


def sk_flag_bytes():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return (sms * 4 + 255) // 256 * 256


def run_ws(awq, d, ws, pk=None):
    pk = packed_of(awq, d) if pk is None else pk
    b = None if d["bias"] is None else dev(d["bias"])
    y = awq.awq_gemm_packed(dev(d["x"]), pk, b, d["K"], d["N"], d["group_size"], workspace=ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("M,K,N,G,bias", SK)
def test_gemm_packed_stream_k(awq, M, K, N, G, bias):
    d = synth.awq_linear(24000 + M + K, M, K, N, group_size=G, bias=bias)
    ws = torch.zeros(awq.awq_gemm_packed_workspace_size(), dtype=torch.uint8, device="cuda")
    pk = packed_of(awq, d)
    y = run_ws(awq, d, ws, pk)
    fb = sk_flag_bytes()
    assert not ws[:fb].any().item()      # every flag lowered again
    assert ws[fb:].any().item()          # partial sums were written: the stream-K kernel ran
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    if K * N <= 64 * 1024 * 1024:
        assert_close(y, oracle.gemm(*args), f"stream-K M={M} K={K} N={N} G={G}")
    else:
        rng = np.random.default_rng(8)
        rows = np.concatenate([rng.integers(0, M, 4096), [0, M - 1]])
        cols = np.concatenate([rng.integers(0, N, 4096), [0, N - 1]])
        assert_close(y[rows, cols], oracle.gemm_sampled(*args, rows, cols), f"stream-K M={M} K={K} N={N}")
    assert np.array_equal(run_ws(awq, d, ws, pk).view(np.uint16), y.view(np.uint16))  # fixed order


def test_gemm_packed_stream_k_exact_bitwise(awq):
    # exact-arithmetic inputs: every partial sum is exact in fp32, so the CTA-cut tiles give the
    # oracle's value rounded once to fp16
    d = synth.awq_linear(24500, 257, 4096, 2048, group_size=128, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic")
    ws = torch.zeros(awq.awq_gemm_packed_workspace_size(), dtype=torch.uint8, device="cuda")
    y = run_ws(awq, d, ws)
    assert ws[sk_flag_bytes():].any().item()
    want = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), want.view(np.uint16))


def test_gemm_packed_stream_k_workspace_reuse(awq):
    # one workspace across stream-K shapes of different grids and a shape that does not take
    # stream-K, in rotation: each result bit for bit its first value
    cases = [synth.awq_linear(24600 + i, M, K, N, group_size=128, bias=True)
             for i, (M, K, N) in enumerate([(257, 4096, 2048), (1000, 512, 256), (384, 4096, 2048)])]
    ws = torch.zeros(awq.awq_gemm_packed_workspace_size(), dtype=torch.uint8, device="cuda")
    pks = [packed_of(awq, d) for d in cases]
    first = [run_ws(awq, d, ws, pk) for d, pk in zip(cases, pks)]
    for _ in range(3):
        for d, pk, y0 in zip(cases, pks, first):
            assert np.array_equal(run_ws(awq, d, ws, pk).view(np.uint16), y0.view(np.uint16))
    assert not ws[:sk_flag_bytes()].any().item()


def test_gemm_packed_ws_small_workspace_is_the_plain_plan(awq):
    # a workspace below the required size gives awq_gemm_packed's own launch, bit for bit
    d = synth.awq_linear(24700, 257, 4096, 2048, group_size=128, bias=True)
    pk = packed_of(awq, d)
    small = torch.zeros(awq.awq_gemm_packed_workspace_size() - 256, dtype=torch.uint8, device="cuda")
    y = run_ws(awq, d, small, pk)
    assert not small.any().item()
    assert np.array_equal(y.view(np.uint16), run(awq, d, pk).view(np.uint16))


def test_gemm_packed_deterministic(awq):
    d = synth.awq_linear(23500, 700, 4096, 1024, group_size=128, bias=True)
    pk = packed_of(awq, d)
    a, b = run(awq, d, pk), run(awq, d, pk)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


@pytest.mark.parametrize("name", ["7b_prefill_m512_4096x11008", "7b_prefill_m2048_11008x4096",
                                  "70b_m4096_8192x28672", "70b_m16_8192x8192", "7b_decode_m1_4096x4096_bias"])
def test_gemm_packed_workloads(awq, name):
    d = synth.workload_inputs(name)
    M, K, N, G = d["M"], d["K"], d["N"], d["group_size"]
    y = run(awq, d)
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    if M * K * N <= 32 * 4096 * 11008 and K * N <= 64 * 1024 * 1024:
        assert_close(y, oracle.gemm(*args), name)
    else:
        rng = np.random.default_rng(5)
        rows = np.concatenate([rng.integers(0, M, 2048), np.zeros(256, np.int64), np.full(256, M - 1)])
        cols = np.concatenate([rng.integers(0, N, 2048), rng.integers(0, N, 512)])
        assert_close(y[rows, cols], oracle.gemm_sampled(*args, rows, cols), name)
    assert np.all(np.isfinite(y.astype(np.float32)))


def test_gemm_packed_empty_and_errors(awq):
    d = synth.awq_linear(23900, 0, 256, 128, group_size=128)
    pk = packed_of(awq, d)
    y = awq.awq_gemm_packed(dev(d["x"]), pk, None, 256, 128, 128)
    assert tuple(y.shape) == (0, 128)
    with pytest.raises(awq.AwqError):  # K % 64
        awq.awq_repack_size(96, 64, 32)
    with pytest.raises(awq.AwqError):  # group size % 64
        awq.awq_repack_size(256, 64, 32)
