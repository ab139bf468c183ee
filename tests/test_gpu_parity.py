"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same
seeded inputs.  awq_dequant must be bit-exact; awq_gemm must satisfy
|y - y_ref| <= 1e-2 * max(1, |y_ref|) elementwise (y fp16 with fp32 accumulation,
y_ref fp64), and bit-exact on inputs where every partial sum is exact."""
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


def run_gemm(awq, d, path="auto", t=None):
    t = t or to_dev(d)
    y = awq.awq_gemm(t["x"], t["qweight"], t["qzeros"], t["scales"], t["bias"],
                     group_size=d["group_size"], path=path)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def assert_close(y, y_ref, what):
    ok, worst = oracle.within_tolerance(y.astype(np.float64), y_ref, REL_TOL)
    assert ok, f"{what}: worst |err|/(1e-2*max(1,|ref|)) = {worst:.3f}"


def decode_ok(K, G):
    G = K if G == -1 else G
    return K % 16 == 0 and G % 16 == 0


def prefill_ok(K, N, G):
    G = K if G == -1 else G
    return K % 64 == 0 and G % 64 == 0 and N % 32 == 0


# ------------------------------------------------------------------ dequant ----

@pytest.mark.parametrize("K,N,G", [(256, 256, 128), (48, 24, 16), (96, 40, 32), (4096, 4096, 128),
                                   (11008, 4096, -1), (64, 8, 8), (136, 1032, 8)])
@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
def test_dequant_bit_exact(awq, K, N, G, dtype):
    d = synth.awq_linear(7000 + K + N, 1, K, N, group_size=G)
    t = to_dev(d)
    w = awq.awq_dequant(t["qweight"], t["qzeros"], t["scales"], group_size=G, out_dtype=dtype)
    torch.cuda.synchronize()
    ref = (oracle.dequant_f16 if dtype == torch.float16 else oracle.dequant_f32)(
        d["qweight"], d["qzeros"], d["scales"], G)
    got = w.cpu().numpy()
    assert got.shape == (K, N)
    assert np.array_equal(got.view(np.uint16 if dtype == torch.float16 else np.uint32),
                          ref.view(np.uint16 if dtype == torch.float16 else np.uint32))


def test_dequant_unaligned_output_uses_scalar_path(awq):
    d = synth.awq_linear(7100, 1, 64, 32, group_size=32)
    t = to_dev(d)
    buf = torch.empty(64 * 32 + 1, dtype=torch.float16, device="cuda")
    out = buf[1:].view(64, 32)      # 2-byte aligned, not 16-byte aligned
    awq.awq_dequant(t["qweight"], t["qzeros"], t["scales"], group_size=32, out=out)
    torch.cuda.synchronize()
    ref = oracle.dequant_f16(d["qweight"], d["qzeros"], d["scales"], 32)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), ref.view(np.uint16))


# ---------------------------------------------------- GEMM, small and ragged ----

SMALL = [(1, 256, 256, 128, False), (3, 512, 192, 64, True), (8, 1024, 520, 32, True),
         (13, 768, 264, 128, False), (17, 2048, 1032, 256, True), (32, 4096, 128, -1, False),
         (33, 256, 64, 16, True), (100, 512, 136, 64, False), (5, 200, 64, 8, True),
         (2, 48, 8, 16, False), (64, 1024, 2048, 128, True),
         # TMA decode: ragged column tile, 16- and 32-token tiles, two 32-token tiles, K = 64
         (9, 1024, 160, 128, True), (24, 2048, 96, 64, False), (40, 4096, 4096, 128, True),
         (1, 64, 32, -1, False), (7, 192, 32, 64, True), (16, 8192, 544, 256, True)]


@pytest.mark.parametrize("M,K,N,G,bias", SMALL)
@pytest.mark.parametrize("path", ["auto", "decode", "prefill", "generic"])
def test_gemm_small_vs_oracle(awq, M, K, N, G, bias, path):
    if path == "decode" and not decode_ok(K, G):
        pytest.skip("shape outside the decode kernel's contract")
    if path == "prefill" and not prefill_ok(K, N, G):
        pytest.skip("shape outside the prefill kernel's contract")
    d = synth.awq_linear(8000 + M + K + N, M, K, N, group_size=G, bias=bias)
    y = run_gemm(awq, d, path)
    y_ref = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    assert_close(y, y_ref, f"{path} M={M} K={K} N={N} G={G}")


# One token: the decode kernel gives each quantization group a warp spans its own MMA
# token column (up to 8 groups per warp; beyond that the general small-batch variant runs),
# with 8-warp CTAs where 4-warp ones would leave a warp 5 or more 64-row stages.  With 224
# column tiles (N = 28672) the launch plan takes clusters of one CTA, so with G = 64 a warp
# of an 8-warp CTA spans K / 512 groups: 3, 4 (first token column of each lane only), 4-5
# (K = 2112: second column used by some warps), 8, and 16 for K = 8192 (general variant).
# K = 4096, N = 11008 stays on 4-warp CTAs (4 stages a warp).
ONE_TOKEN = [(1536, 28672, 64, True), (2048, 28672, 64, False), (2112, 28672, 64, True),
             (4096, 28672, 64, False), (8192, 28672, 64, True), (4096, 4096, -1, True),
             (11008, 4096, 64, False), (4096, 11008, 64, True), (28672, 8192, 128, False)]


@pytest.mark.parametrize("K,N,G,bias", ONE_TOKEN)
def test_one_token_group_spans(awq, K, N, G, bias):
    d = synth.awq_linear(8500 + K + N + G, 1, K, N, group_size=G, bias=bias)
    y = run_gemm(awq, d, "decode")
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    if K * N <= 32 * 1024 * 1024:
        assert_close(y, oracle.gemm(*args), f"one token K={K} N={N} G={G}")
    else:  # every column of a tile sees all of the tile's warps: sample columns
        cols = np.concatenate([np.arange(512), np.arange(N - 512, N),
                               np.random.default_rng(2).integers(0, N, 3072)])
        rows = np.zeros_like(cols)
        assert_close(y[rows, cols], oracle.gemm_sampled(*args, rows, cols), f"one token K={K} N={N} G={G}")


@pytest.mark.parametrize("M", [1, 5, 8, 12, 16, 30, 32, 40, 300])
@pytest.mark.parametrize("path", ["decode", "prefill", "generic"])
def test_gemm_exact_case_bitwise(awq, M, path):
    """Small-integer x, power-of-two scales, dyadic bias: every product and partial sum
    is exact in fp32, so y must equal the fp16 rounding of the exact result bit for bit
    whatever the summation order."""
    d = synth.awq_linear(9000 + M, M, 2048, 384, group_size=128, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic")
    y = run_gemm(awq, d, path)
    y_ref = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128)
    assert np.array_equal(y.view(np.uint16), y_ref.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("M", [1, 16, 32, 96, 600])
def test_gemm_deterministic(awq, M):
    d = synth.awq_linear(9100 + M, M, 4096, 1024, group_size=128, bias=True)
    t = to_dev(d)
    a = run_gemm(awq, d, t=t)
    b = run_gemm(awq, d, t=t)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_gemm_symmetric_checkpoint(awq):
    d = synth.awq_linear(9200, 4, 1024, 512, group_size=64, sym=True)
    y = run_gemm(awq, d)
    assert_close(y, oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], None, 64), "sym")


def test_gemm_empty_batch(awq):
    d = synth.awq_linear(9300, 0, 256, 64, group_size=128)
    t = to_dev(d)
    y = awq.awq_gemm(t["x"], t["qweight"], t["qzeros"], t["scales"], None, group_size=128)
    assert tuple(y.shape) == (0, 64)


def test_gemm_leading_dims_flattened(awq):
    d = synth.awq_linear(9400, 6, 256, 64, group_size=128)
    t = to_dev(d)
    y = awq.awq_gemm(t["x"].view(2, 3, 256), t["qweight"], t["qzeros"], t["scales"], None,
                     group_size=128)
    torch.cuda.synchronize()
    assert tuple(y.shape) == (2, 3, 64)
    assert_close(y.cpu().numpy().reshape(6, 64),
                 oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], None, 128), "3d")


def test_binding_rejects_wrong_dtype_and_layout(awq):
    d = synth.awq_linear(9500, 2, 256, 64, group_size=128)
    t = to_dev(d)
    with pytest.raises(TypeError):
        awq.awq_gemm(t["x"].float(), t["qweight"], t["qzeros"], t["scales"], None, group_size=128)
    with pytest.raises(ValueError):
        awq.awq_gemm(t["x"], t["qweight"], t["qzeros"], t["scales"][:, :32], None, group_size=128)
    with pytest.raises(ValueError):
        xt = torch.empty(256, 2, dtype=torch.float16, device="cuda").t()
        awq.awq_gemm(xt, t["qweight"], t["qzeros"], t["scales"], None, group_size=128)


def test_device_status_clean(awq):
    awq.device_status()


def test_bounded_wait_gives_up_and_reports(awq):
    """A wait that nothing completes gives up after its limit, sets the status word and
    returns (no fault, no hang); the context stays usable afterwards."""
    awq.device_status()
    awq.selftest_wait_timeout(2_000_000)
    with pytest.raises(awq.AwqError, match="bounded wait"):
        awq.device_status()
    awq.device_status()  # cleared by the read
    d = synth.awq_linear(9600, 1, 256, 64, group_size=128)
    assert_close(run_gemm(awq, d), oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], None, 128),
                 "after timeout")


# --------------------------------------------- every workload at full size ----

def _sample(M, N, rng, n=2048):
    rows = np.concatenate([rng.integers(0, M, n), np.zeros(256, np.int64), np.full(256, M - 1)])
    cols = np.concatenate([rng.integers(0, N, n), rng.integers(0, N, 512)])
    return rows, cols


@pytest.mark.parametrize("name", [w[2] for w in synth.WORKLOADS])
def test_workload_parity(awq, name):
    d = synth.workload_inputs(name)
    M, K, N, G = d["M"], d["K"], d["N"], d["group_size"]
    y = run_gemm(awq, d)
    args = (d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
    if M * K * N <= 32 * 4096 * 11008 and K * N <= 64 * 1024 * 1024:
        assert_close(y, oracle.gemm(*args), name)
    else:
        rng = np.random.default_rng(1)
        rows, cols = _sample(M, N, rng)
        assert_close(y[rows, cols], oracle.gemm_sampled(*args, rows, cols), name)
    assert np.all(np.isfinite(y.astype(np.float32)))


def test_workload_70b_prefill_full_matrix(awq):
    # every element of one 70B prefill linear (M = 4096, 8192 x 8192, bias) against the plain
    # C oracle (fp64, OpenMP over rows on the host cores), not a sample
    from oracle import c_oracle
    d = synth.workload_inputs("70b_m4096_8192x8192")
    y = run_gemm(awq, d)
    y_ref = c_oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], d["group_size"])
    assert y.shape == y_ref.shape == (4096, 8192)
    assert_close(y, y_ref, "70b_m4096_8192x8192 (full matrix)")


@pytest.mark.parametrize("M", [33, 64, 100, 192, 256])
@pytest.mark.parametrize("path", ["auto", "decode", "prefill"])
def test_medium_batch_both_families(awq, M, path):
    # 33..256 rows: both tensor-core kernels take the shape (decode in several 32-row tiles,
    # prefill in one row tile); the automatic choice between them is a cost model
    d = synth.awq_linear(15000 + M, M, 4096, 1024, group_size=128, bias=True)
    y = run_gemm(awq, d, path)
    assert_close(y, oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128),
                 f"M={M} {path}")


@pytest.mark.parametrize("M,K,N,want", [(64, 4096, 4096, "decode"), (192, 4096, 4096, "decode"),
                                        (512, 4096, 4096, "prefill"), (64, 4096, 11008, "decode"),
                                        (128, 4096, 11008, "prefill"), (192, 11008, 4096, "decode"),
                                        (512, 11008, 4096, "prefill"), (2048, 4096, 11008, "prefill")])
def test_automatic_family_choice(awq, M, K, N, want):
    # the measured crossovers the cost model was fitted to (152 SMs)
    x = torch.empty((M, K), dtype=torch.float16, device="cuda")
    qw = torch.empty((K, N // 8), dtype=torch.int32, device="cuda")
    qz = torch.empty((K // 128, N // 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((K // 128, N), dtype=torch.float16, device="cuda")
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert awq.select_path(x, qw, qz, sc, None, 128, y) == want


# narrow-tile prefill (32/64/128-row token tiles; K split over clusters of 4, 2 or 1 CTAs by
# tile count): 4096 x 4096 at 32 and 64 rows (4-way split), 11008 x 4096 at 128 rows (2-way),
# K = 4160 (65 stages: an uneven 4-way split), 4096 x 11008 (no split), one row
@pytest.mark.parametrize("M,K,N", [(32, 4096, 4096), (64, 4096, 4096), (128, 11008, 4096),
                                   (17, 4160, 1024), (100, 4096, 11008), (1, 1024, 512)])
def test_prefill_narrow_tiles(awq, M, K, N):
    d = synth.awq_linear(16000 + M + K, M, K, N, group_size=64, bias=True)
    y = run_gemm(awq, d, "prefill")
    assert_close(y, oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 64),
                 f"narrow prefill M={M} K={K} N={N}")
    assert np.array_equal(run_gemm(awq, d, "prefill").view(np.uint16), y.view(np.uint16))


@pytest.mark.parametrize("M", [32, 64, 128])
def test_prefill_narrow_tiles_exact_bitwise(awq, M):
    # exact-arithmetic inputs: the split partial sums are exact in fp32, so y is the oracle's
    # value rounded once to fp16 whatever the split
    d = synth.awq_linear(16500 + M, M, 4096, 1024, group_size=128, bias=True, x_kind="smallint",
                         scale_kind="pow2", bias_kind="dyadic")
    y = run_gemm(awq, d, "prefill")
    want = oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], 128).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), want.view(np.uint16))
