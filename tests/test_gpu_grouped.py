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
