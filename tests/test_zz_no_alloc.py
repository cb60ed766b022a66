"""The allocation-free binned float sum (repro_sum_f32_noalloc).

It is meant for callers that cannot allocate device memory: another
allocator holds the GPU's memory, or the call sits where an allocation could
synchronize or fail.  Its workspace is a fixed device array inside the
library.  This file is collected last; it must pass alone in a fresh process
and after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from compensated_bit_reproducible_gb300 import api, inputs
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _reference(x: torch.Tensor, K: int) -> np.ndarray:
    out = torch.empty(1, dtype=torch.float32, device=x.device)
    api.repro_sum_async(x, out, K)
    return out.cpu().numpy()


def _noalloc(x: torch.Tensor, K: int) -> np.ndarray:
    out = torch.full((1,), 7.0, dtype=torch.float32, device=x.device)
    L = api.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.repro_sum_f32_noalloc(ctypes.c_void_p(x.data_ptr()) if x.numel() else None, x.numel(), K, s,
                                 ctypes.c_void_p(out.data_ptr()))
    assert rc == 0, api.lib().repro_strerror(rc)
    return out.cpu().numpy()


def test_matches_the_allocating_sum_on_consecutive_calls():
    """Same bits as repro_sum_f32_async (the tests' tolerance for binned sums
    is zero), over two calls in a row on different data: the shared workspace
    carries nothing from one call to the next."""
    d = _dev()
    cases = [
        (inputs.normal_f32(1_000_003, seed=21, spikes=True), 3),
        (inputs.wide_f64(2_000_001, seed=22).astype(np.float32), 3),
        (inputs.inject_specials(inputs.normal_f32(70_001, seed=23), "nan"), 3),
        (inputs.normal_f32(5, seed=24), 21),
        (inputs.normal_f32(123_457, seed=25), 2),
    ]
    for x, K in cases:
        t = torch.from_numpy(x).to(d)
        want = _reference(t, K)
        first = _noalloc(t, K)
        second = _noalloc(t, K)
        assert first.tobytes() == want.tobytes()
        assert second.tobytes() == want.tobytes()
        # and the oracle's binned sum of the same input
        assert first.tobytes() == np.array([orc.adn_sum(x, K)], np.float32).tobytes()


def test_forced_environment_failure(monkeypatch):
    """REPRO_FORCE_ENV_FAIL=1 makes the environment check fail here as in
    every other entry point, before anything is launched."""
    d = _dev()
    x = torch.ones(1000, dtype=torch.float32, device=d)
    out = torch.full((1,), 7.0, dtype=torch.float32, device=d)
    L = api.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    monkeypatch.setenv("REPRO_FORCE_ENV_FAIL", "1")
    assert L.repro_sum_f32_noalloc(ctypes.c_void_p(x.data_ptr()), 1000, 3, s, ctypes.c_void_p(out.data_ptr())) == 4
    monkeypatch.delenv("REPRO_FORCE_ENV_FAIL")
    assert L.repro_sum_f32_noalloc(ctypes.c_void_p(x.data_ptr()), 1000, 3, s, ctypes.c_void_p(out.data_ptr())) == 0
    assert out.item() == 1000.0


def test_empty_input_and_rejected_arguments():
    d = _dev()
    assert _noalloc(torch.empty(0, dtype=torch.float32, device=d), 3).tobytes() == np.float32(0).tobytes()
    L = api.lib()
    out = torch.empty(1, dtype=torch.float32, device=d)
    p = ctypes.c_void_p(out.data_ptr())
    assert L.repro_sum_f32_noalloc(p, 1, 22, None, p) == 1          # K above 21
    assert L.repro_sum_f32_noalloc(None, 4294966785, 3, None, p) == 2   # above the float capacity
