"""Binned cumulative sum on the GPU against the CPU oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.gpu_util import dev, first_diff, same_bits, to_dev

pytestmark = pytest.mark.gpu
F32, F64 = np.float32, np.float64


def gpu_cumsum(x, K=3, inplace=False, block=0):
    t = to_dev(x)
    out = t if inplace else None
    r = api.repro_cumsum(t, out=out, K=K, block=block)
    return r.cpu().numpy()


@pytest.mark.parametrize("n", [1, 2, 17, 255, 4095, 4096, 4097, 8193, 12289, 50001])
@pytest.mark.parametrize("dt", [F32, F64])
def test_parity_k3(n, dt):
    dev()
    x = inputs.normal_f32(n, seed=n, spikes=True).astype(dt) if dt == F32 else inputs.wide_f64(n, seed=n)
    # a mid-sequence raise of the bin index
    x = x.copy()
    x[: n // 2] *= dt(1e-9)
    got = gpu_cumsum(x, 3)
    want = oracle.adn_cumsum(x, 3)
    assert same_bits(got, want), first_diff(got, want)


@pytest.mark.parametrize("dt,K", [(F32, 2), (F32, 4), (F32, 6), (F32, 11), (F32, 21),
                                  (F64, 2), (F64, 4), (F64, 6), (F64, 9), (F64, 52)])
def test_parity_other_k(dt, K):
    dev()
    x = inputs.wide_f64(9000, seed=K).astype(dt)
    got = gpu_cumsum(x, K)
    want = oracle.adn_cumsum(x, K)
    assert same_bits(got, want), first_diff(got, want)


@pytest.mark.parametrize("dt,K", [(F64, 2), (F64, 4), (F64, 6), (F32, 4), (F32, 8)])
def test_parity_other_k_many_tiles(dt, K):
    """More tiles than one scan segment (256 tiles of 4096): the tile scan
    runs in two levels; a ragged last segment and tile."""
    dev()
    x = inputs.wide_f64(1_300_003, seed=K + 100).astype(dt)
    got = gpu_cumsum(x, K)
    want = oracle.adn_cumsum(x, K)
    assert same_bits(got, want), first_diff(got, want)


def test_quickstart_last_prefix_equals_sum():
    dev()
    x = inputs.quickstart_f64()
    for seed in range(10):
        xp = inputs.permuted(x, seed)
        cs = gpu_cumsum(xp, 3)
        assert cs[-1] == 10000.0
        assert same_bits(cs, oracle.adn_cumsum(xp, 3))


@pytest.mark.parametrize("dt", [F32, F64])
def test_in_place(dt):
    dev()
    x = inputs.wide_f64(30011, seed=3).astype(dt)
    got = gpu_cumsum(x, 3, inplace=True)
    assert same_bits(got, oracle.adn_cumsum(x, 3))


@pytest.mark.parametrize("dt", [F32, F64])
def test_specials(dt):
    dev()
    base = inputs.wide_f64(20000, seed=8).astype(dt)
    for kind in ("nan", "pinf", "pninf"):
        y = inputs.inject_specials(base, kind, seed=1)
        got = gpu_cumsum(y, 3)
        want = oracle.adn_cumsum(y, 3)
        assert same_bits(got, want), (kind, first_diff(got, want))


@pytest.mark.parametrize("dt", [F32, F64])
def test_launch_shape_invariance(dt):
    dev()
    x = inputs.wide_f64(40000, seed=11).astype(dt)
    ref = gpu_cumsum(x, 3)
    for block in (128, 256, 512):
        assert same_bits(gpu_cumsum(x, 3, block=block), ref)
    assert same_bits(ref, oracle.adn_cumsum(x, 3))


def test_last_equals_sum():
    dev()
    for x in (inputs.normal_f32(123457, seed=2, spikes=True), inputs.wide_f64(123457, seed=2)):
        cs = gpu_cumsum(x, 3)
        t = to_dev(x)
        out = torch.empty(1, dtype=t.dtype, device=t.device)
        api.repro_sum_async(t, out, 3)
        assert same_bits(cs[-1], out.cpu().numpy()[0])


@pytest.mark.slow
@pytest.mark.parametrize("dt,K", [(F64, 3), (F64, 6), (F32, 3)])
def test_full_size_sampled(dt, K):
    """100M elements: every prefix computed on the GPU; sampled prefixes
    (including tile boundaries and the last) checked against the oracle."""
    dev()
    n = 100_000_000
    x = inputs.wide_f64(n, seed=2) if dt == F64 else inputs.normal_f32(n, seed=1)
    got = gpu_cumsum(x, K)
    rng = np.random.default_rng(5)
    pos = np.unique(np.concatenate([rng.integers(0, n, 400), [0, 4095, 4096, 4097, n // 2, n - 1]]))
    want = oracle.adn_cumsum_at(x, pos, K)
    assert same_bits(got[pos], want), first_diff(got[pos], want)


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("n", [1000, 200_003])
def test_host_pointers(dt, n):
    """Plain host memory in and/or out (copied by the library; the call
    waits), in place on the host, and pinned host memory used directly."""
    dev()
    x = inputs.normal_f32(n, seed=9, spikes=True).astype(dt) if dt == F32 else inputs.wide_f64(n, seed=9)
    want = oracle.adn_cumsum(x, 3)
    h = torch.from_numpy(x.copy())
    assert same_bits(api.repro_cumsum(h, K=3).numpy(), want)                      # host -> host
    o = torch.empty(n, dtype=h.dtype, device="cuda")
    assert same_bits(api.repro_cumsum(h, out=o, K=3).cpu().numpy(), want)         # host -> device
    ho = torch.empty(n, dtype=h.dtype)
    assert same_bits(api.repro_cumsum(to_dev(x), out=ho, K=3).numpy(), want)      # device -> host
    api.repro_cumsum(h, out=h, K=3)                                               # in place on the host
    assert same_bits(h.numpy(), want)
    p = torch.from_numpy(x.copy()).pin_memory()
    po = torch.empty(n, dtype=p.dtype).pin_memory()
    api.repro_cumsum(p, out=po, K=3)                                              # pinned: stream-ordered
    torch.cuda.synchronize()
    assert same_bits(po.numpy(), want)
