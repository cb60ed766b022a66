"""Host-side logic without a GPU: the multi-rank helpers of bench.py on two
gloo ranks, the oracle arm's JSON line, and the forced environment-failure
path of the C ABI (which returns before any device work)."""
import ctypes
import json
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, ws, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    try:
        got_ws, got_rank, _ = bench.dist_env()
        bench.init_dist(got_ws, backend="gloo")
        bench.barrier(got_ws)
        m = bench.max_over_ranks(1.5 + got_rank, got_ws)
        bench.barrier(got_ws)
        q.put((got_rank, got_ws, m))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    # every rank sees the maximum over ranks (rank 1's 2.5), and its own rank
    assert res == [(0, 2, 2.5), (1, 2, 2.5)]


def test_reference_arm_other_ranks_exit_silently(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    import bench

    # stand-in rates: the line's arithmetic and keys, not the oracle's speed
    rates = {name: 1e7 for name, _, _ in bench.ROWS_SPEC}
    samples = {name: "1 x 10 elements" for name, _, _ in bench.ROWS_SPEC}
    monkeypatch.setattr(bench, "oracle_rates", lambda seconds: (rates, samples))
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference"
    assert line["unit"] == "GElements/s" and line["higher_is_better"] is True
    assert line["value"] == pytest.approx(0.01, rel=1e-6)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]
    assert line["metric"] == bench.METRIC and line["config"]["workload"] == bench.WORKLOAD


def test_forced_environment_failure(monkeypatch):
    """REPRO_FORCE_ENV_FAIL=1 makes validation fail before any device call,
    so every compute entry point reports REPRO_ERR_ENV on a machine without a
    GPU, after its argument checks."""
    from compensated_bit_reproducible_gb300 import api

    lib = api.lib()
    ENV = 4
    monkeypatch.setenv("REPRO_FORCE_ENV_FAIL", "1")
    lib.repro_validate_environment.restype = ctypes.c_int
    assert lib.repro_validate_environment(None) == ENV
    x = np.ones(64, dtype=np.float32)
    r = ctypes.c_float(7.0)
    p = ctypes.c_void_p(x.ctypes.data)
    assert lib.repro_sum_f32(p, ctypes.c_size_t(64), 3, None, ctypes.byref(r)) == ENV
    assert r.value == 7.0          # result untouched
    # argument errors still come first
    assert lib.repro_sum_f32(p, ctypes.c_size_t(64), 1, None, ctypes.byref(r)) == 1
    out = np.zeros(64, dtype=np.float32)
    q = ctypes.c_void_p(out.ctypes.data)
    assert lib.repro_cumsum_f32(p, q, ctypes.c_size_t(64), 3, None) == ENV
    assert lib.stable_var_f32(p, ctypes.c_int64(8), ctypes.c_int64(8), 1, 0, q, None, None) == ENV
    assert lib.repro_segsum_f32(p, ctypes.c_int64(8), ctypes.c_int64(8), 1, 3, q, None) == ENV
    assert lib.repro_sum_kahan_f32(p, ctypes.c_size_t(64), q, None) == ENV
    assert not out.any()
    monkeypatch.delenv("REPRO_FORCE_ENV_FAIL")


@pytest.mark.parametrize("n,nch", [(100_000_000, 8), (100_000_000, 1), (40_000_000, 12), (1000, 8), (100, 8),
                                   (64, 3), (1, 4)])
def test_end_to_end_chunk_bounds(n, nch):
    """The end-to-end leg's chunks tile [0, n) in order, start on 64-element
    boundaries (256-byte aligned for both element types) and number at most
    nch."""
    import bench
    b = bench.chunk_bounds(n, nch)
    assert 1 <= len(b) <= nch
    assert b[0][0] == 0 and b[-1][1] == n
    assert all(x[1] == y[0] for x, y in zip(b, b[1:]))
    assert all(e > s and s % 64 == 0 for s, e in b)
