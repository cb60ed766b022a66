"""The multi-rank exchange step (binned states gathered, merged in rank
order): two gloo ranks on the CPU with a host stand-in for the device state
calls, and two ranks on one GPU with the real kernels."""
import socket

import pytest

from tests import dist_ranks


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _run(target, ws=2, timeout=300):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(ws):
            r, res = q.get(timeout=timeout)
            out[r] = res
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    return out


def test_two_gloo_ranks_exchange_protocol():
    out = _run(dist_ranks.cpu_protocol_rank)
    for r in range(2):
        assert isinstance(out[r], dict), out[r]
        for k, (s_ok, c_ok) in out[r].items():
            assert s_ok and c_ok, (r, k)


@pytest.mark.gpu
def test_two_ranks_on_one_gpu_match_the_whole_input():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = _run(dist_ranks.gpu_rank, timeout=600)
    for r in range(2):
        assert isinstance(out[r], dict), out[r]
        for k, (s_ok, c_ok) in out[r].items():
            assert s_ok and c_ok, (r, k)
