"""GPU checks of AwqLinear, the prepared-layer binding (weights validated once, x and out
checked per call): it must produce exactly the functional entry points' bits for every
dtype and code width, honour the requested kernel family, and refuse bad activations."""
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


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.float().to(dtype)


def same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M,K,N,G", [(1, 4096, 4096, 128), (5, 1024, 512, 64), (300, 512, 256, 128),
                                     (3, 200, 64, 8)])
@pytest.mark.parametrize("path", ["auto", "generic"])
def test_linear_fp16_matches_awq_gemm(awq, M, K, N, G, path):
    d = synth.awq_linear(20000 + M + K, M, K, N, group_size=G, bias=True)
    x, qw, qz, sc, b = (dev(d[k]) for k in ("x", "qweight", "qzeros", "scales", "bias"))
    lin = awq.AwqLinear(qw, qz, sc, b, group_size=G, path=path)
    y = lin(x)
    y_ref = awq.awq_gemm(x, qw, qz, sc, b, group_size=G, path=path)
    torch.cuda.synchronize()
    assert same(y, y_ref)
    ref = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert (err <= 1e-2 * np.maximum(1.0, np.abs(ref))).all()


def test_linear_bf16_and_leading_dims(awq):
    d = synth.awq_linear(20100, 6, 1024, 512, group_size=128, bias=True, dtype="bf16")
    x = dev(d["x"], torch.bfloat16).reshape(2, 3, 1024)
    qw, qz = dev(d["qweight"]), dev(d["qzeros"])
    sc, b = dev(d["scales"], torch.bfloat16), dev(d["bias"], torch.bfloat16)
    lin = awq.AwqLinear(qw, qz, sc, b, group_size=128)
    y = lin(x)
    assert y.shape == (2, 3, 512) and y.dtype == torch.bfloat16
    out = torch.empty((6, 512), dtype=torch.bfloat16, device="cuda")
    lin(x, out=out)
    y_ref = awq.awq_gemm(x.reshape(6, 1024), qw, qz, sc, b, group_size=128)
    torch.cuda.synchronize()
    assert same(y.reshape(6, 512), y_ref) and same(out, y_ref)


def test_linear_w8_matches_awq_gemm_w8(awq):
    d = synth.awq8_linear(20200, 4, 4096, 1024, group_size=128, bias=True)
    x, qw, qz, sc, b = (dev(d[k]) for k in ("x", "qweight", "qzeros", "scales", "bias"))
    lin = awq.AwqLinear(qw, qz, sc, b, group_size=128, bits=8)
    assert lin.N == 1024
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = lin(x, stream=s)
    s.synchronize()
    y_ref = awq.awq_gemm_w8(x, qw, qz, sc, b, group_size=128)
    torch.cuda.synchronize()
    assert same(y, y_ref)


def test_linear_refuses_bad_activations(awq):
    d = synth.awq_linear(20300, 2, 256, 128, group_size=128)
    x, qw, qz, sc = (dev(d[k]) for k in ("x", "qweight", "qzeros", "scales"))
    lin = awq.AwqLinear(qw, qz, sc, None, group_size=128)
    with pytest.raises(TypeError):
        lin(x.float())
    with pytest.raises(ValueError):
        lin(x[:, :128].contiguous())                        # wrong K
    with pytest.raises(ValueError):
        lin(torch.cat([x, x], 1)[:, ::2])                   # not contiguous
    with pytest.raises(ValueError):
        lin(x.cpu())                                        # host tensor
    with pytest.raises(ValueError):
        lin(x, out=torch.empty((3, 128), dtype=torch.float16, device="cuda"))
    with pytest.raises(TypeError):
        awq.AwqLinear(qw, qz, sc.float(), None, group_size=128)
    with pytest.raises(ValueError):
        awq.AwqLinear(qw, qz[:1, :8], sc, None, group_size=64)


@pytest.mark.parametrize("M", [1, 40, 127, 128, 700])
def test_linear_packed_switches_layout_by_rows(awq, M):
    # packed=True keeps a tile-packed copy: calls of >= packed_min_rows rows run
    # awq_gemm_packed_ws on it (bit for bit the functional call with the stream's workspace),
    # smaller ones the checkpoint layout (bit for bit awq_gemm); both within the oracle's
    # tolerance
    K, N, G = 1024, 392, 128
    d = synth.awq_linear(20400 + M, M, K, N, group_size=G, bias=True)
    x, qw, qz, sc, b = (dev(d[k]) for k in ("x", "qweight", "qzeros", "scales", "bias"))
    lin = awq.AwqLinear(qw, qz, sc, b, group_size=G, packed=True)
    y = lin(x)
    if M >= lin.packed_min_rows:
        y_ref = awq.awq_gemm_packed(x, awq.awq_repack(qw, qz, sc, G), b, K, N, G, workspace="auto")
    else:
        y_ref = awq.awq_gemm(x, qw, qz, sc, b, group_size=G)
    torch.cuda.synchronize()
    assert same(y, y_ref)
    ref = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert (err <= 1e-2 * np.maximum(1.0, np.abs(ref))).all()


def test_linear_packed_stream_k_shape(awq):
    # 2 x 16 tiles of 256 x 128 on one CTA per SM: the layer's call runs the stream-K kernel
    # through the stream's workspace, bit for bit the functional call with that workspace
    M, K, N, G = 257, 4096, 2048, 128
    d = synth.awq_linear(20450, M, K, N, group_size=G, bias=True)
    x, qw, qz, sc, b = (dev(d[k]) for k in ("x", "qweight", "qzeros", "scales", "bias"))
    lin = awq.AwqLinear(qw, qz, sc, b, group_size=G, packed=True)
    y = lin(x)
    y_ref = awq.awq_gemm_packed(x, awq.awq_repack(qw, qz, sc, G), b, K, N, G, workspace="auto")
    torch.cuda.synchronize()
    assert same(y, y_ref)
    ref = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert (err <= 1e-2 * np.maximum(1.0, np.abs(ref))).all()


def test_linear_packed_refuses_other_formats(awq):
    # shapes outside the layout have no tile-packed form (bf16 scales and 8-bit codes do: see
    # tests/test_gpu_bf16.py and tests/test_gpu_w8.py); 8-bit codes with bf16 scales are refused
    d8 = synth.awq8_linear(20501, 2, 256, 128, group_size=128)
    with pytest.raises(TypeError):
        awq.AwqLinear(dev(d8["qweight"]), dev(d8["qzeros"]), dev(d8["scales"]).to(torch.bfloat16), None,
                      group_size=128, bits=8, packed=True)
    d2 = synth.awq_linear(20502, 2, 96, 64, group_size=32)
    with pytest.raises(awq.AwqError):  # K % 64: no tile-packed layout
        awq.AwqLinear(dev(d2["qweight"]), dev(d2["qzeros"]), dev(d2["scales"]), None, group_size=32,
                      packed=True)
