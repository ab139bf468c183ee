"""GPU parity of awq_gemm_grouped (mixture-of-experts W4A16 linear in one launch; routed expert
layers with 4-bit AWQ weights, the vLLM article, section 5.4) against the grouped oracle on
the same seeded experts and routing: |y - y_ref| <= 1e-2 * max(1, |y_ref|) elementwise,
bit-exact run to run."""
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


def run(awq, d):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    y = awq.awq_gemm_grouped(dev(d["x"]), dev(d["qweight"]), dev(d["qzeros"]), dev(d["scales"]),
                             dev(d["offsets"]), None if d["bias"] is None else dev(d["bias"]),
                             group_size=d["group_size"])
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check(y, d):
    y_ref = oracle.gemm_grouped(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"],
                                d["group_size"], d["offsets"])
    ok, worst = oracle.within_tolerance(y.astype(np.float64), y_ref, 1e-2)
    assert ok, f"worst |err|/(1e-2*max(1,|ref|)) = {worst:.3f}"


# (T tokens, top-k, E experts, K, N, G, bias): few rows per expert, empty experts (5 rows
# over 8), more than one 8-row tile per expert (64 x 2 over 4), a one-row layer, 7B-sized
CASES = [(12, 2, 4, 256, 128, 64, True), (5, 1, 8, 512, 256, 128, False),
         (64, 2, 4, 1024, 512, 128, True), (1, 1, 4, 256, 64, -1, False),
         (16, 2, 8, 4096, 1024, 128, True), (3, 2, 16, 2048, 512, 64, False)]


@pytest.mark.parametrize("T,topk,E,K,N,G,bias", CASES)
def test_grouped_vs_oracle(awq, T, topk, E, K, N, G, bias):
    d = synth.moe_inputs(600 + T + E + K, T, topk, E, K, N, group_size=G, bias=bias)
    check(run(awq, d), d)


def test_grouped_deterministic(awq):
    d = synth.moe_inputs(700, 32, 2, 8, 2048, 512, group_size=128, bias=True)
    a, b = run(awq, d), run(awq, d)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_grouped_rejects_outside_contract(awq):
    d = synth.moe_inputs(701, 4, 1, 2, 96, 64, group_size=32)  # K % 64 != 0
    with pytest.raises(awq.AwqError):
        run(awq, d)


# Grouped linear on stacked tile-packed experts (awq_repack_experts, awq_gemm_packed_grouped):
# prefill-sized routed batches.  Cases: uneven experts with some empty, one expert holding all
# rows, expert boundaries inside and at the edges of 256-row tiles, ragged column tiles.
def run_packed(awq, d):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    pk = awq.awq_repack_experts(dev(d["qweight"]), dev(d["qzeros"]), dev(d["scales"]), d["group_size"])
    y = awq.awq_gemm_packed_grouped(dev(d["x"]), pk, dev(d["offsets"]), d["K"], d["N"],
                                    None if d["bias"] is None else dev(d["bias"]), group_size=d["group_size"])
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("T,topk,E,K,N,G,bias", [(600, 2, 8, 1024, 520, 128, True), (300, 1, 1, 512, 256, 64, False),
                                                 (700, 2, 16, 512, 384, -1, True), (2048, 2, 8, 2048, 1024, 128, True)])
def test_grouped_packed_vs_oracle(awq, T, topk, E, K, N, G, bias):
    d = synth.moe_inputs(31000 + T + E, T, topk, E, K, N, group_size=G, bias=bias)
    y = run_packed(awq, d)
    check(y, d)
    assert np.array_equal(run_packed(awq, d).view(np.uint16), y.view(np.uint16))


def test_grouped_packed_tile_edges(awq):
    # hand-set offsets: empty first expert, an expert of exactly 256 rows, one of 257, one of 1,
    # an empty one in the middle, the rest in the last
    d = synth.moe_inputs(31500, 800, 1, 6, 512, 264, group_size=128, bias=True)
    d["offsets"] = np.array([0, 0, 256, 513, 514, 514, 800], dtype=np.int32)
    y = run_packed(awq, d)
    check(y, d)


def test_grouped_packed_exact_case_bitwise(awq):
    # small-integer activations, power-of-two scales: every product and sum is exact, so y is
    # the oracle's value rounded once to fp16
    E, K, N, G, R = 4, 1024, 384, 128, 700
    ex = [synth.awq_linear(31600 + e, 1, K, N, group_size=G, x_kind="smallint", scale_kind="pow2")
          for e in range(E)]
    x = synth.awq_linear(31650, R, K, N, group_size=G, x_kind="smallint", scale_kind="pow2")["x"]
    d = {"x": x, "qweight": np.stack([a["qweight"] for a in ex]), "qzeros": np.stack([a["qzeros"] for a in ex]),
         "scales": np.stack([a["scales"] for a in ex]), "bias": None, "group_size": G, "K": K, "N": N,
         "offsets": np.array([0, 100, 400, 401, R], dtype=np.int32)}
    y = run_packed(awq, d)
    want = oracle.gemm_grouped(d["x"], d["qweight"], d["qzeros"], d["scales"], None, G, d["offsets"])
    assert np.array_equal(y.view(np.uint16), want.astype(np.float16).view(np.uint16))


# bf16 (experts repacked from bf16 scales; x, bias, y bf16).  The packed kernel rounds each
# dequantized weight once to bf16 for the tensor core, so the reference is the fp64 GEMM of
# the oracle's bf16-rounded dequant, expert by expert, under the same 1e-2 criterion.
def run_packed_bf16(awq, d):
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    pk = awq.awq_repack_experts(dev(d["qweight"]), dev(d["qzeros"]), bf(d["scales"]), d["group_size"])
    y = awq.awq_gemm_packed_grouped(bf(d["x"]), pk, dev(d["offsets"]), d["K"], d["N"],
                                    None if d["bias"] is None else bf(d["bias"]), group_size=d["group_size"])
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16
    return y.float().cpu().numpy()


def reference_bf16_rounded(d):
    off, G = d["offsets"], d["group_size"]
    y = np.zeros((d["x"].shape[0], d["N"]))
    for e in range(len(off) - 1):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        W = oracle.dequant_bf16(d["qweight"][e], d["qzeros"][e], d["scales"][e], G).astype(np.float64)
        y[r0:r1] = d["x"][r0:r1].astype(np.float64) @ W
        if d["bias"] is not None:
            y[r0:r1] += d["bias"][e].astype(np.float64)
    return y


@pytest.mark.parametrize("T,topk,E,K,N,G,bias", [(600, 2, 8, 1024, 520, 128, True), (700, 2, 16, 512, 384, -1, False)])
def test_grouped_packed_bf16_vs_oracle(awq, T, topk, E, K, N, G, bias):
    d = synth.moe_inputs(32000 + T + E, T, topk, E, K, N, group_size=G, bias=bias, dtype="bf16")
    y = run_packed_bf16(awq, d)
    assert np.isfinite(y).all()
    ok, worst = oracle.within_tolerance(y.astype(np.float64), reference_bf16_rounded(d), 1e-2)
    assert ok, f"worst |err|/(1e-2*max(1,|ref|)) = {worst:.3f}"
    assert np.array_equal(run_packed_bf16(awq, d).view(np.uint32), y.view(np.uint32))


def test_grouped_packed_bf16_exact_case_bitwise(awq):
    # exact-arithmetic inputs as in the fp16 case: y is the oracle's value rounded once to bf16
    E, K, N, G, R = 4, 1024, 384, 128, 700
    ex = [synth.awq_linear(32600 + e, 1, K, N, group_size=G, bias=True, x_kind="smallint", scale_kind="pow2",
                           bias_kind="dyadic", dtype="bf16") for e in range(E)]
    x = synth.awq_linear(32650, R, K, N, group_size=G, x_kind="smallint", scale_kind="pow2", dtype="bf16")["x"]
    d = {"x": x, "qweight": np.stack([a["qweight"] for a in ex]), "qzeros": np.stack([a["qzeros"] for a in ex]),
         "scales": np.stack([a["scales"] for a in ex]), "bias": np.stack([a["bias"] for a in ex]), "group_size": G,
         "K": K, "N": N, "offsets": np.array([0, 0, 300, 557, R], dtype=np.int32)}
    y = run_packed_bf16(awq, d)
    want = oracle.round_to_bf16(oracle.gemm_grouped(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G,
                                                     d["offsets"]).astype(np.float32))
    assert np.array_equal(y.view(np.uint32), want.view(np.uint32))
