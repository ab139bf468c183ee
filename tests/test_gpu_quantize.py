"""GPU parity of awq_quantize_rtn (round-to-nearest 4-bit group quantization into the AWQ
GEMM layout; GPTQModel wiki "AWQ", "Group quantization and zero points") against the CPU
oracle: qweight, qzeros and scales must be bit-exact, since both sides take every
rounding decision with the same correctly rounded fp32 operations."""
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


def _weights(seed, N, K, kind="normal"):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        w = rng.standard_normal((N, K)) * 0.02
    elif kind == "wide":  # outliers and sign-skewed rows
        w = rng.standard_normal((N, K)) * 0.02
        w[::3, ::17] *= 40.0
        w[1::5] = np.abs(w[1::5])
        w[2::7] = -np.abs(w[2::7])
    elif kind == "degenerate":  # constant, zero and single-spike rows
        w = rng.standard_normal((N, K)) * 0.02
        w[0::4] = 0.25
        w[1::4] = 0.0
        w[2::4] = -0.125
        w[3::8, 5] = 3.0
    else:
        raise ValueError(kind)
    return w.astype(np.float16)


def _check(awq, w, G, sym):
    qw, qz, sc = awq.awq_quantize_rtn(torch.from_numpy(w).cuda(), group_size=G, sym=sym)
    torch.cuda.synchronize()
    rqw, rqz, rsc = oracle.quantize_rtn(w, G, sym)
    assert np.array_equal(qz.cpu().numpy(), rqz), "qzeros"
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), rsc.view(np.uint16)), "scales"
    got = qw.cpu().numpy()
    if not np.array_equal(got, rqw):
        bad = np.argwhere(got != rqw)
        raise AssertionError(f"qweight differs at {len(bad)} words, first {bad[:4].tolist()}")


# (N, K, G): ragged 128-channel tiles (N = 8, 136, 11008), groups of 8 / 40 / 64 / 128 /
# K (partial 64-wide code tiles: G = 40, K = 4104 with G = K), many groups (K / G = 512)
SHAPES = [(8, 64, 32), (136, 256, 64), (16, 64, 8), (24, 200, 40), (128, 4096, 128),
          (4096, 4096, 128), (11008, 4096, 128), (4096, 11008, 128), (8, 2048, -1),
          (256, 4104, -1), (64, 4096, 8)]


@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("N,K,G", SHAPES)
def test_quantize_bit_exact(awq, N, K, G, sym):
    _check(awq, _weights(N + K + (G if G > 0 else 7), N, K), G, sym)


@pytest.mark.parametrize("kind", ["wide", "degenerate"])
@pytest.mark.parametrize("sym", [False, True])
def test_quantize_edge_distributions(awq, kind, sym):
    _check(awq, _weights(11, 264, 512, kind), 64, sym)


def test_quantize_recovers_grid_weights(awq):
    # weights on a grid spanning the whole code range come back exactly
    rng = np.random.default_rng(12)
    N, K, G = 256, 1024, 128
    ng = K // G
    code = rng.integers(0, 16, size=(N, ng, G))
    code[:, :, 0] = 0
    code[:, :, 1] = 15
    zero = rng.integers(0, 16, size=(N, ng))
    s = np.ldexp(1.0, -rng.integers(4, 12, size=(N, ng)))
    w = ((code - zero[:, :, None]) * s[:, :, None]).reshape(N, K).astype(np.float16)
    qw, qz, sc = awq.awq_quantize_rtn(torch.from_numpy(w).cuda(), group_size=G)
    assert np.array_equal(oracle.unpack_codes(qw.cpu().numpy()), code.reshape(N, K).T)
    assert np.array_equal(oracle.unpack_codes(qz.cpu().numpy()), zero.T)
    assert np.array_equal(sc.cpu().numpy().astype(np.float64), s.T)


def test_quantize_then_gemm(awq):
    # the quantizer's output feeds awq_gemm like any checkpoint
    N, K, G, M = 1024, 2048, 128, 4
    w = _weights(13, N, K)
    qw, qz, sc = awq.awq_quantize_rtn(torch.from_numpy(w).cuda(), group_size=G)
    x = synth.awq_linear(14, M, K, 8, group_size=G)["x"]
    y = awq.awq_gemm(torch.from_numpy(x).cuda(), qw, qz, sc, None, group_size=G).cpu().numpy()
    rqw, rqz, rsc = oracle.quantize_rtn(w, G)
    y_ref = oracle.gemm(x, rqw, rqz, rsc, None, G)
    ok, worst = oracle.within_tolerance(y.astype(np.float64), y_ref, 1e-2)
    assert ok, worst


@pytest.mark.parametrize("M", [1, 4, 16])
def test_quantize_then_gemm_back_to_back(awq, M):
    # the quantizer rewrites the weight buffers and awq_gemm runs directly after it on the
    # same stream, no copy or synchronize between: the GEMM must see the new weights (its
    # programmatic launch may overlap the quantizer's tail, its reads may not)
    N, K, G = 11008, 4096, 128
    wa, wb = _weights(31, N, K), _weights(32, N, K)
    x = synth.awq_linear(33 + M, M, K, 8, group_size=G)["x"]
    xd = torch.from_numpy(x).cuda()
    wad, wbd = torch.from_numpy(wa).cuda(), torch.from_numpy(wb).cuda()
    out = (torch.empty((K, N // 8), dtype=torch.int32, device="cuda"),
           torch.empty((K // G, N // 8), dtype=torch.int32, device="cuda"),
           torch.empty((K // G, N), dtype=torch.float16, device="cuda"))
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    awq.awq_quantize_rtn(wad, group_size=G, out=out)
    awq.awq_gemm(xd, *out, None, group_size=G, out=y)
    awq.awq_quantize_rtn(wbd, group_size=G, out=out)
    awq.awq_gemm(xd, *out, None, group_size=G, out=y)
    got = y.cpu().numpy()
    rqw, rqz, rsc = oracle.quantize_rtn(wb, G)
    y_ref = oracle.gemm(x, rqw, rqz, rsc, None, G)
    ok, worst = oracle.within_tolerance(got.astype(np.float64), y_ref, 1e-2)
    assert ok, worst


def test_quantize_empty_and_errors(awq):
    w = torch.zeros((0, 64), dtype=torch.float16, device="cuda")
    qw, qz, sc = awq.awq_quantize_rtn(w, group_size=32)
    assert qw.shape == (64, 0) and qz.shape == (2, 0) and sc.shape == (2, 0)
    with pytest.raises(awq.AwqError):
        awq.awq_quantize_rtn(torch.zeros((8, 48), dtype=torch.float16, device="cuda"), group_size=12)
