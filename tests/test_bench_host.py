"""Host-side bench logic without a GPU: the multi-rank path (replicas only, gloo, world
size 2), whole-job aggregation, the reference arm's rank rule, algorithmic bytes, and the
traffic figure's source check."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import torch.distributed as dist
    r, w, local = bench.dist_setup(None)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    elapsed = 1.0 + rank  # the slower rank decides the job time
    m = bench.reduce_max(elapsed, w)
    out[rank] = (m, bench.job_gbs(1_000_000, 10, w, m))
    # the reference arm runs on rank 0 only: the other ranks return without work
    if rank != 0:
        out[world + rank] = bench.run_reference(None, rank, w) is None
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_ranks_gloo_max_and_aggregate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        m, gbs = res[r]
        assert m == 2.0
        assert gbs == pytest.approx(2 * 1_000_000 * 10 / 2.0 / 1e9)
    assert res[world + 1] is True  # rank 1 skipped the reference arm


def test_single_rank_helpers_are_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.job_gbs(55_681_536, 100, 1, 1e-3) == pytest.approx(5568.1536)


def test_algorithmic_bytes_by_hand():
    # 7B MLP up-projection, M = 1, G = 128, bias: weights + zeros + scales + x + y + bias
    K, N, G = 4096, 11008, 128
    expect = K * N // 2 + (K // G) * N // 2 + 2 * (K // G) * N + 2 * K + 2 * N + 2 * N
    assert bench.algorithmic_bytes(1, K, N, G, True) == expect == 23_477_248
    assert bench.algorithmic_bytes(8, K, N, -1, False) == K * N // 2 + N // 2 + 2 * N + 16 * K + 16 * N


def test_traffic_reported_only_for_measured_source(monkeypatch):
    assert bench.measured_traffic() in (None, bench.TRAFFIC_BYTES_PER_LAUNCH)
    bad = {k: "0" * 64 for k in bench.TRAFFIC_SOURCES}
    monkeypatch.setattr(bench, "TRAFFIC_SOURCES", bad)
    assert bench.measured_traffic() is None


def test_cpu_oracle_mode_prints_one_line_per_shape():
    # the C oracle timed on the tiny config (no GPU involved), one JSON line per workload
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-oracle", "--configs", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert [d["workload"] for d in lines] == ["tiny_m1_256x256"]
    d = lines[0]
    assert d["kind"] == "C oracle" and d["threads"] == 2 and d["linear_s"] > 0 and d["dequant_s"] > 0
    assert d["GB_s"] > 0 and d["M"] == 1 and d["K"] == 256 and d["N"] == 256
