"""GPU check of awq_gemm_packed_noalloc, the packed linear on the library's fixed device
scratch, against the workspace entry point (awq_gemm_packed_ws with a caller workspace) on the
same seeded inputs: two calls in a row, each within |y - y_ws| <= 1e-2 * max(1, |y_ws|)
elementwise.  Shapes: two that take the stream-K kernel (the scratch holds its flags and
partial sums) and one that does not.  This file is collected last, so the check also runs
after every other test has used the library on the device."""
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


@pytest.mark.parametrize("M,K,N,G", [(257, 4096, 2048, 128), (512, 4096, 11008, 128), (300, 768, 1032, 64)])
def test_noalloc_matches_workspace_entry_point(awq, M, K, N, G):
    d = synth.awq_linear(26000 + M + K, M, K, N, group_size=G, bias=True)
    x, b = dev(d["x"]), dev(d["bias"])
    pk = awq.awq_repack(dev(d["qweight"]), dev(d["qzeros"]), dev(d["scales"]), G)
    ws = torch.zeros((awq.awq_gemm_packed_workspace_size(),), dtype=torch.uint8, device="cuda")
    y_ws = awq.awq_gemm_packed(x, pk, b, K, N, G, workspace=ws)
    y1 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    y2 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    awq.awq_gemm_packed_noalloc(x, pk, b, K, N, G, out=y1)
    awq.awq_gemm_packed_noalloc(x, pk, b, K, N, G, out=y2)
    torch.cuda.synchronize()
    awq.device_status()
    ref = y_ws.cpu().numpy().astype(np.float64)
    for y in (y1, y2):
        ok, worst = oracle.within_tolerance(y.cpu().numpy().astype(np.float64), ref, 1e-2)
        assert ok, f"noalloc M={M} K={K} N={N}: worst |err|/(1e-2*max(1,|ref|)) = {worst:.3f}"
