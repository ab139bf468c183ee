"""GPU parity of the 8-bit entry points (awq_dequant_w8, awq_gemm_w8; AutoAWQ's
"w_bit" knob on the format page: 8-bit codes packed four to an int32 word) against the
CPU oracle on the same seeded inputs.  Dequant must be bit-exact (fp32: the exact
product; fp16: that product rounded once to nearest-even).  The GEMM is held to the fp16
path's bar, |y - y_ref| <= 1e-2 * max(1, |y_ref|), and must be bit-exact where every
product and partial sum is exact."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

REL_TOL = 1e-2


@pytest.fixture(scope="module")
def awq():
    from w4a16_weight_only_gb300 import build
    build.build()
    import w4a16_weight_only_gb300 as awq
    assert awq.runtime_available(), awq.last_error()
    return awq


def to_dev(d):
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda()
         for k in ("x", "qweight", "qzeros", "scales")}
    t["bias"] = None if d["bias"] is None else torch.from_numpy(d["bias"]).cuda()
    return t


def run(awq, d, path="auto"):
    t = to_dev(d)
    y = awq.awq_gemm_w8(t["x"], t["qweight"], t["qzeros"], t["scales"], t["bias"],
                        group_size=d["group_size"], path=path)
    torch.cuda.synchronize()
    assert y.dtype == torch.float16
    return y.cpu().numpy()


def assert_close(y, y_ref, what):
    err = np.abs(y.astype(np.float64) - y_ref)
    tol = REL_TOL * np.maximum(1.0, np.abs(y_ref))
    assert np.isfinite(y).all(), what
    worst = float((err / tol).max()) if err.size else 0.0
    assert worst <= 1.0, f"{what}: worst |err|/(1e-2*max(1,|ref|)) = {worst:.3f}"


@pytest.mark.parametrize("K,N,G", [(256, 256, 128), (48, 12, 16), (4096, 4096, 128), (64, 4, -1),
                                   (1000, 36, 8)])
def test_dequant_w8_bit_exact(awq, K, N, G):
    d = synth.awq8_linear(12000 + K + N, 1, K, N, group_size=G)
    t = to_dev(d)
    w16 = awq.awq_dequant_w8(t["qweight"], t["qzeros"], t["scales"], group_size=G)
    w32 = awq.awq_dequant_w8(t["qweight"], t["qzeros"], t["scales"], group_size=G,
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.dequant8_f32(d["qweight"], d["qzeros"], d["scales"], G)
    assert np.array_equal(w32.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(w16.cpu().numpy().view(np.uint16), ref.astype(np.float16).view(np.uint16))


SMALL = [(1, 256, 256, 128, False), (3, 512, 192, 64, True), (8, 1024, 512, 128, True),
         (17, 2048, 1024, 256, True), (32, 4096, 128, -1, False), (33, 256, 60, 16, True),
         (100, 512, 132, 64, False), (300, 1024, 256, 128, True), (1, 64, 4, -1, False),
         (12, 1024, 1024, 128, True)]


def decode_ok(K, N, G):
    G = K if G == -1 else G
    return K % 64 == 0 and G % 64 == 0 and N % 16 == 0


@pytest.mark.parametrize("M,K,N,G,bias", SMALL)
@pytest.mark.parametrize("path", ["auto", "decode", "prefill", "generic"])
def test_gemm_w8_small_vs_oracle(awq, M, K, N, G, bias, path):
    if path in ("decode", "prefill") and not decode_ok(K, N, G):
        pytest.skip("shape outside the tensor-core kernel's contract")
    d = synth.awq8_linear(13000 + M + K + N, M, K, N, group_size=G, bias=bias)
    y = run(awq, d, path)
    y_ref = oracle.gemm8(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    assert_close(y, y_ref, f"w8 {path} M={M} K={K} N={N} G={G}")


@pytest.mark.parametrize("M", [1, 5, 16, 32, 300])
@pytest.mark.parametrize("path", ["decode", "prefill", "generic"])
def test_gemm_w8_exact_case_bitwise(awq, M, path):
    # x small integers, power-of-two scales, K = 256: |partial sums| <= 256 * 4 * 255 * 2^-8
    # on a 2^-13 grid (23 bits), so fp32 accumulation is exact on any order and y must be
    # the oracle's value rounded once to fp16
    d = synth.awq8_linear(13500 + M, M, 256, 384, group_size=64, x_kind="smallint",
                          scale_kind="pow2")
    y = run(awq, d, path)
    y_ref = oracle.gemm8(d["x"], d["qweight"], d["qzeros"], d["scales"], None, 64)
    assert np.array_equal(y.view(np.uint16), y_ref.astype(np.float16).view(np.uint16))


# the decode kernel's variants at 8 bits: one token with 4- and 8-warp CTAs (long K), one
# group per row (G = K), 8-row tiles, 16-row tiles, the exact-operand 32-row tiles, a
# ragged column tile (N = 48: 12 of a tile's 16 words), M past 32 (several row tiles)
WORK = [(1, 4096, 4096, 128), (1, 11008, 4096, 128), (1, 28672, 1024, 128), (1, 4096, 1024, -1),
        (16, 4096, 4096, 128),
        (4, 4096, 11008, 128), (16, 4096, 11008, 128), (24, 4096, 4096, 128), (32, 11008, 4096, 128),
        (7, 1024, 48, 64), (1, 1024, 16, 128), (64, 11008, 4096, 128)]


@pytest.mark.parametrize("M,K,N,G", WORK)
def test_gemm_w8_workload_shapes(awq, M, K, N, G):
    d = synth.awq8_linear(13700 + M + K + N, M, K, N, group_size=G, bias=True)
    y = run(awq, d)
    assert_close(y, oracle.gemm8(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G),
                 f"w8 M={M} K={K} N={N} G={G}")


@pytest.mark.parametrize("M,K,N", [(300, 4096, 1024), (512, 4096, 11008), (2048, 11008, 4096),
                                   (257, 1024, 4112), (64, 4096, 1024), (32, 4096, 4096),
                                   (100, 11008, 4096)])
def test_gemm_w8_prefill_shapes(awq, M, K, N):
    # the tcgen05 kernel: several row and column tiles, a ragged row tile (M = 257), a ragged
    # column tile (N = 4112: 16 of the last tile's 128 columns); the oracle on sampled rows
    d = synth.awq8_linear(14100 + M + K, M, K, N, group_size=128, bias=True)
    y = run(awq, d, "prefill")
    rows = np.unique(np.concatenate([np.random.default_rng(M).integers(0, M, 24), [0, M - 1]]))
    ref = oracle.gemm8(d["x"][rows], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128)
    assert_close(y[rows], ref, f"w8 prefill M={M} K={K} N={N}")


@pytest.mark.parametrize("M", [1, 24, 600])
def test_gemm_w8_deterministic(awq, M):
    d = synth.awq8_linear(13900 + M, M, 4096, 1024, group_size=128, bias=True)
    a, b = run(awq, d), run(awq, d)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_gemm_w8_selected_families(awq):
    for (M, want) in ((1, "decode"), (16, "decode"), (2048, "prefill")):
        d = synth.awq8_linear(13970 + M, M, 4096, 1024, group_size=128)
        t = to_dev(d)
        assert awq.select_path(t["x"], t["qweight"], t["qzeros"], t["scales"], bits=8) == want


def test_gemm_w8_auto_matches_decode(awq):
    # small M takes the decode kernel: same bits as forcing it
    d = synth.awq8_linear(13960, 3, 4096, 4096, group_size=128, bias=True)
    assert np.array_equal(run(awq, d).view(np.uint16), run(awq, d, "decode").view(np.uint16))


def test_gemm_w8_tensor_core_contract(awq):
    # both tensor-core kernels refuse N % 16 != 0 at 8 bits (packed rows must be whole
    # 16-byte units for the tensor maps); the automatic path then takes the generic kernel
    d = synth.awq8_linear(13951, 40, 256, 40, group_size=128)
    for path in ("decode", "prefill"):
        with pytest.raises(Exception):
            run(awq, d, path)
    y = run(awq, d)
    assert_close(y, oracle.gemm8(d["x"], d["qweight"], d["qzeros"], d["scales"], None, 128), "w8 N=40")


# Tile-packed layout of 8-bit codes (awq_repack_w8, awq_gemm_packed_w8): the repack is a
# byte permutation plus padding (bit-exact against the oracle); the linear forms (c - z) * s
# exactly and rounds it once to fp16, like the fp16 4-bit packed path.  Shapes: narrow split
# tiles, the 256-row kernel with ragged rows and columns (N % 128 != 0), stream-K (through a
# workspace), the pair kernel (K = 8192, even column-tile count).
@pytest.mark.parametrize("K,N,G", [(64, 4, 64), (256, 260, 64), (4096, 11008, 128), (512, 1028, -1)])
def test_repack_w8_bit_exact(awq, K, N, G):
    d = synth.awq8_linear(12500 + K + N, 1, K, N, group_size=G)
    t = to_dev(d)
    pk = awq.awq_repack(t["qweight"], t["qzeros"], t["scales"], G, bits=8)
    torch.cuda.synchronize()
    assert pk.numel() * 4 == awq.awq_repack_size(K, N, G, bits=8) == oracle.repack8_size(K, N, G)
    want = oracle.repack8(d["qweight"], d["qzeros"], d["scales"], G)
    assert np.array_equal(pk.cpu().numpy().view(np.uint32), want)


# M <= 32 runs the small-batch kernel (16- or 32-row tiles, several pipelines per CTA):
# ragged N (N % 8 != 0: 2-byte y stores), G = -1, a 5-stage K split, the 7B shape
PACKED8 = [(1, 1024, 260, 128, True, None), (16, 4096, 512, 64, True, None), (17, 320, 516, -1, False, None),
           (32, 4096, 11008, 128, True, None),
           (40, 1024, 512, 128, True, None), (300, 1024, 260, 64, True, None),
           (257, 4096, 2048, 128, True, "ws"), (300, 8192, 512, 128, False, None),
           (700, 512, 1028, -1, True, None)]


@pytest.mark.parametrize("M,K,N,G,bias,ws", PACKED8)
def test_gemm_packed_w8_vs_oracle(awq, M, K, N, G, bias, ws):
    d = synth.awq8_linear(12600 + M + K, M, K, N, group_size=G, bias=bias)
    t = to_dev(d)
    pk = awq.awq_repack(t["qweight"], t["qzeros"], t["scales"], G, bits=8)
    w = None
    if ws:
        w = torch.zeros((awq.awq_gemm_packed_workspace_size(),), dtype=torch.uint8, device="cuda")
    y = awq.awq_gemm_packed(t["x"], pk, t["bias"], K, N, G, workspace=w, bits=8)
    torch.cuda.synchronize()
    if ws:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert w[(sms * 4 + 255) // 256 * 256:].any().item()  # the stream-K kernel ran
    y_ref = oracle.gemm8(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    assert_close(y.cpu().numpy(), y_ref, f"packed w8 M={M} K={K} N={N} G={G}")
    y2 = awq.awq_gemm_packed(t["x"], pk, t["bias"], K, N, G, workspace=w, bits=8)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


@pytest.mark.parametrize("M,K,N,ws", [(300, 2048, 384, None), (257, 4096, 2048, "ws"), (64, 2048, 384, None),
                                      (1, 2048, 384, None), (16, 4096, 260, None), (32, 1024, 516, None)])
def test_gemm_packed_w8_exact_case_bitwise(awq, M, K, N, ws):
    # small-integer activations, power-of-two scales: every product and partial sum is exact,
    # so y is the oracle's value rounded once to fp16 whatever the summation order
    d = synth.awq8_linear(12700 + M + K, M, K, N, group_size=128, x_kind="smallint", scale_kind="pow2")
    t = to_dev(d)
    pk = awq.awq_repack(t["qweight"], t["qzeros"], t["scales"], 128, bits=8)
    w = None if not ws else torch.zeros((awq.awq_gemm_packed_workspace_size(),), dtype=torch.uint8, device="cuda")
    y = awq.awq_gemm_packed(t["x"], pk, None, K, N, 128, workspace=w, bits=8).cpu().numpy()
    want = oracle.gemm8(d["x"], d["qweight"], d["qzeros"], d["scales"], None, 128).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), want.view(np.uint16))


def test_linear_packed_w8(awq):
    M, K, N, G = 300, 4096, 2048, 128
    d = synth.awq8_linear(12800, M, K, N, group_size=G, bias=True)
    t = to_dev(d)
    lin = awq.AwqLinear(t["qweight"], t["qzeros"], t["scales"], t["bias"], group_size=G, bits=8, packed=True)
    y = lin(t["x"])
    pk = awq.awq_repack(t["qweight"], t["qzeros"], t["scales"], G, bits=8)
    y_ref = awq.awq_gemm_packed(t["x"], pk, t["bias"], K, N, G, workspace="auto", bits=8)
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)
    assert_close(y.cpu().numpy(), oracle.gemm8(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G),
                 "AwqLinear packed w8")
