"""GPU parity of the bf16 entry points (awq_gemm_bf16, awq_dequant_bf16; the native GEMM's
declared FP16/BF16 contract, GPTQModel wiki "AWQ", "Selection and compatibility") against
the CPU oracle on the same seeded inputs (synth draws rounded to bf16).  Dequant must be
bit-exact.  The GEMM is held to the fp16 path's criterion, |y - y_ref| <= 1e-2 *
max(1, |y_ref|) elementwise, against the reference its arithmetic defines:

* kernels that carry exact weights into an fp32 accumulation (the decode kernel up to 16
  rows: codes as the exact bf16 values 128 + c with zero and scale folded per group; the
  generic kernel) against the oracle's fp64 GEMM of the exact weights;
* kernels that round each dequantized weight once to bf16 for the tensor core (prefill,
  and decode's 17..32-row tiles) against the fp64 GEMM of the oracle's bf16-rounded
  dequant (``oracle.dequant_bf16``): weight rounding alone (2^-9 relative, random signs)
  moves y by about 2^-9 sqrt(K) rms(x w), which reaches the 1e-2 criterion at K >= 2048.

and the GEMM must be bit-exact (after the oracle's own bf16 rounding) where every product
and partial sum is exact."""
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


def bf(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def to_dev(d):
    return {"x": bf(d["x"]), "qweight": torch.from_numpy(d["qweight"]).cuda(),
            "qzeros": torch.from_numpy(d["qzeros"]).cuda(), "scales": bf(d["scales"]),
            "bias": None if d["bias"] is None else bf(d["bias"])}


def run(awq, d, path="auto"):
    """y (as fp32) and the kernel family that ran."""
    t = to_dev(d)
    used = path if path != "auto" else awq.select_path(t["x"], t["qweight"], t["qzeros"],
                                                        t["scales"], t["bias"], d["group_size"])
    y = awq.awq_gemm(t["x"], t["qweight"], t["qzeros"], t["scales"], t["bias"],
                     group_size=d["group_size"], path=path)
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16
    return y.float().cpu().numpy(), used


def rounds_weights(used, M):
    """The kernel rounds each dequantized weight once to bf16 (its tensor-core operand)."""
    return used == "prefill" or (used == "decode" and M > 16)


def reference(d, rounded, rows=None, cols=None):
    """fp64 y of the exact weights (the oracle's GEMM), or of the weights rounded once to
    bf16 (the oracle's dequant_bf16); all (m, n), or the sampled pairs."""
    G = d["group_size"]
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    if not rounded:
        return oracle.gemm(*args) if rows is None else oracle.gemm_sampled(*args, rows, cols)
    b = 0.0 if d["bias"] is None else d["bias"].astype(np.float64)
    if rows is None:
        W = oracle.dequant_bf16(d["qweight"], d["qzeros"], d["scales"], G).astype(np.float64)
        return d["x"].astype(np.float64) @ W + b
    ucols, inv = np.unique(cols, return_inverse=True)
    Wc = oracle.round_to_bf16(oracle.dequant_columns_f32(d["qweight"], d["qzeros"], d["scales"],
                                                        G, ucols)).astype(np.float64)
    out = np.einsum("sk,sk->s", d["x"][rows].astype(np.float64), Wc[:, inv].T)
    return out + (0.0 if d["bias"] is None else d["bias"][cols].astype(np.float64))


def assert_close(y, y_ref, what):
    assert np.isfinite(y).all(), what
    ok, worst = oracle.within_tolerance(y.astype(np.float64), y_ref, 1e-2)
    assert ok, f"{what}: worst |err|/(1e-2*max(1,|ref|)) = {worst:.3f}"


def decode_ok(K, N, G):
    G = K if G == -1 else G
    return K % 64 == 0 and G % 64 == 0 and N % 32 == 0


@pytest.mark.parametrize("K,N,G", [(256, 256, 128), (48, 24, 16), (4096, 4096, 128), (64, 32, -1)])
def test_dequant_bf16_bit_exact(awq, K, N, G):
    d = synth.awq_linear(7500 + K + N, 1, K, N, group_size=G, dtype="bf16")
    t = to_dev(d)
    w = awq.awq_dequant(t["qweight"], t["qzeros"], t["scales"], group_size=G)
    w32 = awq.awq_dequant(t["qweight"], t["qzeros"], t["scales"], group_size=G, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert w.dtype == torch.bfloat16
    ref = oracle.dequant_bf16(d["qweight"], d["qzeros"], d["scales"], G)
    assert np.array_equal(w.float().cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(w32.cpu().numpy(), oracle.dequant_f32(d["qweight"], d["qzeros"], d["scales"], G))


SMALL = [(1, 256, 256, 128, False), (3, 512, 192, 64, True), (8, 1024, 512, 128, True),
         (13, 768, 256, 128, False), (17, 2048, 1024, 256, True), (32, 4096, 128, -1, False),
         (33, 256, 64, 16, True), (100, 512, 136, 64, False), (64, 1024, 2048, 128, True),
         (1, 64, 32, -1, False), (300, 1024, 256, 128, True)]


@pytest.mark.parametrize("M,K,N,G,bias", SMALL)
@pytest.mark.parametrize("path", ["auto", "decode", "prefill", "generic"])
def test_gemm_bf16_small_vs_oracle(awq, M, K, N, G, bias, path):
    if path in ("decode", "prefill") and not decode_ok(K, N, G):
        pytest.skip("shape outside the tensor-core kernels' contract")
    d = synth.awq_linear(8800 + M + K + N, M, K, N, group_size=G, bias=bias, dtype="bf16")
    y, used = run(awq, d, path)
    assert_close(y, reference(d, rounds_weights(used, M)), f"bf16 {path}->{used} M={M} K={K} N={N} G={G}")


@pytest.mark.parametrize("M", [1, 5, 8, 16, 32, 300])
@pytest.mark.parametrize("path", ["decode", "prefill", "generic"])
def test_gemm_bf16_exact_case_bitwise(awq, M, path):
    # x small integers, power-of-two scales, dyadic bias: every product and partial sum is
    # exact in fp32 on every path, so y must be the oracle's value rounded once to bf16
    d = synth.awq_linear(9700 + M, M, 2048, 384, group_size=128, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic", dtype="bf16")
    y, _ = run(awq, d, path)
    y_ref = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128)
    want = oracle.round_to_bf16(y_ref.astype(np.float32))
    assert np.array_equal(y.view(np.uint32), want.view(np.uint32))


# decode M=1 (one token: 4- and 8-warp CTAs), M=8, M=16 (16-token tiles), M=32 (exact-A
# variant), prefill
WORK = [(1, 4096, 11008, 128), (1, 11008, 4096, 128), (8, 4096, 4096, 128), (16, 4096, 4096, 128),
        (32, 4096, 4096, 128), (512, 4096, 11008, 128), (1, 28672, 8192, 128)]


@pytest.mark.parametrize("M,K,N,G", WORK)
def test_gemm_bf16_workload_shapes(awq, M, K, N, G):
    d = synth.awq_linear(9900 + M + K, M, K, N, group_size=G, bias=True, dtype="bf16")
    y, used = run(awq, d)
    rounded = rounds_weights(used, M)
    if M * K * N <= 32 * 4096 * 11008 and K * N <= 64 * 1024 * 1024:
        assert_close(y, reference(d, rounded), f"bf16 {used} M={M} K={K} N={N}")
    else:
        rng = np.random.default_rng(3)
        rows = np.concatenate([rng.integers(0, M, 2048), [0, M - 1]])
        cols = np.concatenate([rng.integers(0, N, 2048), [0, N - 1]])
        assert_close(y[rows, cols], reference(d, rounded, rows, cols), f"bf16 {used} M={M} K={K} N={N}")


@pytest.mark.parametrize("M", [1, 16, 600])
def test_gemm_bf16_deterministic(awq, M):
    d = synth.awq_linear(9950 + M, M, 4096, 1024, group_size=128, bias=True, dtype="bf16")
    a, b = run(awq, d)[0], run(awq, d)[0]
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_bf16_rejects_mixed_dtypes(awq):
    d = synth.awq_linear(9990, 2, 256, 64, group_size=128, dtype="bf16")
    t = to_dev(d)
    with pytest.raises(TypeError):
        awq.awq_gemm(t["x"], t["qweight"], t["qzeros"], t["scales"].half(), None, group_size=128)


# Tile-packed layout with bf16 (awq_repack copies the bf16 scale words; awq_gemm_packed_ex with
# AWQ_DTYPE_BF16): the kernels round each dequantized weight once to bf16, so the reference is
# the fp64 GEMM of the oracle's bf16-rounded dequant.  Shapes: narrow split tiles, the 256-row
# kernel with ragged rows and columns, stream-K (through a workspace), the pair kernel (K = 8192).
PACKED_BF = [(1, 1024, 520, 128, True, None), (16, 2048, 264, 64, True, None), (32, 4096, 1032, -1, False, None),
             (40, 1024, 512, 128, True, None), (300, 1024, 264, 64, True, None),
             (257, 4096, 2048, 128, True, "ws"), (300, 8192, 512, 128, False, None),
             (700, 512, 1032, -1, True, None)]


def bf_words(a):
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def packed_bf(awq, t, G):
    return awq.awq_repack(t["qweight"], t["qzeros"], t["scales"], G)


@pytest.mark.parametrize("K,N,G", [(256, 264, 64), (4096, 11008, 128), (512, 1032, -1)])
def test_repack_bf16_scale_words(awq, K, N, G):
    d = synth.awq_linear(9800 + K + N, 1, K, N, group_size=G, dtype="bf16")
    pk = packed_bf(awq, to_dev(d), G)
    torch.cuda.synchronize()
    want = oracle.repack(d["qweight"], d["qzeros"], bf_words(d["scales"]), G)
    assert np.array_equal(pk.cpu().numpy().view(np.uint32), want)


@pytest.mark.parametrize("M,K,N,G,bias,ws", PACKED_BF)
def test_gemm_packed_bf16_vs_oracle(awq, M, K, N, G, bias, ws):
    d = synth.awq_linear(9850 + M + K, M, K, N, group_size=G, bias=bias, dtype="bf16")
    t = to_dev(d)
    pk = packed_bf(awq, t, G)
    w = None
    if ws:
        w = torch.zeros((awq.awq_gemm_packed_workspace_size(),), dtype=torch.uint8, device="cuda")
    y = awq.awq_gemm_packed(t["x"], pk, t["bias"], K, N, G, workspace=w)
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16
    if ws:
        assert w[(torch.cuda.get_device_properties(0).multi_processor_count * 4 + 255) // 256 * 256:].any().item()
    assert_close(y.float().cpu().numpy(), reference(d, True), f"packed bf16 M={M} K={K} N={N} G={G}")
    y2 = awq.awq_gemm_packed(t["x"], pk, t["bias"], K, N, G, workspace=w)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


@pytest.mark.parametrize("M,K,N,ws", [(300, 2048, 384, None), (257, 4096, 2048, "ws"), (64, 2048, 384, None),
                                      (32, 4096, 520, None), (5, 2048, 384, None)])
def test_gemm_packed_bf16_exact_case_bitwise(awq, M, K, N, ws):
    # exact-arithmetic inputs: every weight (c - z) * 2^k and every partial sum is exact, so y
    # is the oracle's value rounded once to bf16 whatever the kernel's summation order
    d = synth.awq_linear(9900 + M + K, M, K, N, group_size=128, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic", dtype="bf16")
    t = to_dev(d)
    pk = packed_bf(awq, t, 128)
    w = None if not ws else torch.zeros((awq.awq_gemm_packed_workspace_size(),), dtype=torch.uint8, device="cuda")
    y = awq.awq_gemm_packed(t["x"], pk, t["bias"], K, N, 128, workspace=w).float().cpu().numpy()
    want = oracle.round_to_bf16(oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128).astype(np.float32))
    assert np.array_equal(y.view(np.uint32), want.view(np.uint32))


def test_linear_packed_bf16(awq):
    # AwqLinear(packed=True) with bf16 scales: calls of >= 128 rows on the packed copy, bit for
    # bit the functional call with the stream's workspace
    M, K, N, G = 257, 4096, 2048, 128
    d = synth.awq_linear(9960, M, K, N, group_size=G, bias=True, dtype="bf16")
    t = to_dev(d)
    lin = awq.AwqLinear(t["qweight"], t["qzeros"], t["scales"], t["bias"], group_size=G, packed=True)
    y = lin(t["x"])
    y_ref = awq.awq_gemm_packed(t["x"], packed_bf(awq, t, G), t["bias"], K, N, G, workspace="auto")
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)
    assert_close(y.float().cpu().numpy(), reference(d, True), "AwqLinear packed bf16")
