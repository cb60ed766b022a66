"""Helpers shared by the GPU parity tests."""
import numpy as np
import pytest
import torch


def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def to_dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev())


def same_bits(a, b) -> bool:
    a = np.asarray(a)
    b = np.asarray(b)
    return a.dtype == b.dtype and a.shape == b.shape and a.tobytes() == b.tobytes()


def first_diff(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    ia = a.view(np.uint32 if a.dtype == np.float32 else np.uint64)
    ib = b.view(np.uint32 if b.dtype == np.float32 else np.uint64)
    idx = np.flatnonzero(ia != ib)
    if idx.size == 0:
        return None
    i = int(idx[0])
    return i, a.flat[i], b.flat[i], idx.size


def lib_sum(x: np.ndarray, K: int = 3, block: int = 0, grid: int = 0, offset: int = 0):
    """Binned sum through the C-ABI, stream-ordered variant, of x[offset:]."""
    from compensated_bit_reproducible_gb300 import api
    t = to_dev(x)
    if offset:
        t = t[offset:]
    out = torch.empty(1, dtype=t.dtype, device=t.device)
    api.repro_sum_async(t, out, K, block=block, grid=grid)
    return out.cpu().numpy()[0]
