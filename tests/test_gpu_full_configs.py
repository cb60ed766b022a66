"""The benchmark's input configurations at their full sizes (100M elements),
against the oracle run on the same inputs.

- 100M float32 N(0,1), seed 1, and its 1%-spike variant, K = 3: ten seeded
  permutations, each summed with blocks of 128, 256 and 512 threads, all
  with the oracle's bits (order and launch shape do not matter).
- 100M float64 wide-range values, seed 2, with NaN, +Inf or both infinities
  injected, K = 3 and 6: the sum, and the cumulative sum at sampled prefixes
  on both sides of the first special value.
The oracle values use its sequential form, which its pins tie to the closed
form.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.gpu_util import dev, first_diff, same_bits, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
N = 100_000_000


@functools.lru_cache(maxsize=1)
def _wide():
    return inputs.wide_f64(N, seed=2)


def _perm(t, seed):
    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    return t[torch.randperm(t.numel(), generator=g, device=t.device)]


def _sum(t, K, block=0):
    out = torch.empty(1, dtype=t.dtype, device=t.device)
    api.repro_sum_async(t, out, K, block=block)
    return out.cpu().numpy()[0]


@pytest.mark.parametrize("spikes", [False, True])
def test_f32_ten_permutations_three_block_sizes(spikes):
    dev()
    x = inputs.normal_f32(N, seed=1, spikes=spikes)
    want = oracle.adn_sum(x, 3, "fp")
    t = to_dev(x)
    for seed in range(10):
        tp = _perm(t, seed)
        for block in (128, 256, 512):
            assert same_bits(_sum(tp, 3, block), want), (seed, block)
        del tp


def test_f64_permutations_and_block_sizes():
    dev()
    x = _wide()
    t = to_dev(x)
    for K in (3, 6):
        want = oracle.adn_sum(x, K, "fp")
        for seed in range(3):
            tp = _perm(t, 100 + seed)
            for block in (128, 256, 512):
                assert same_bits(_sum(tp, K, block), want), (K, seed, block)
            del tp


@pytest.mark.parametrize("K", [3, 6])
@pytest.mark.parametrize("kind", ["nan", "pinf", "pninf"])
def test_f64_specials_sum_and_cumsum(K, kind):
    dev()
    y = inputs.inject_specials(_wide(), kind, seed=K)
    first = int(np.flatnonzero(~np.isfinite(y))[0])
    t = to_dev(y)
    assert same_bits(_sum(t, K), oracle.adn_sum(y, K, "fp"))
    got = api.repro_cumsum(t, K=K)
    rng = np.random.default_rng(K)
    pos = np.unique(np.concatenate([rng.integers(0, N, 300), [0, 4095, 4096, first - 1, first, first + 1,
                                                               N // 2, N - 1]]))
    pos = pos[(pos >= 0) & (pos < N)]
    g = got[torch.from_numpy(pos).to(got.device)].cpu().numpy()
    want = oracle.adn_cumsum_at(y, pos, K)
    assert same_bits(g, want), first_diff(g, want)
    assert np.all(np.isfinite(g[pos < first])) and not np.any(np.isfinite(g[pos >= first]))


def test_general_cumsum_segment_scan_walks_several_segments():
    """The per-fold cumulative sum scans 4096-element tiles in segments of 256
    and then the segment totals in one block of 1024 threads; above 2^30
    elements (1024 segments) each thread of that block walks more than one
    segment.  1.1e9 floats, K = 4 (the per-fold path for float), prefixes
    sampled around segment boundaries on both sides of the 1024th."""
    dev()
    n = 1_100_000_000
    rng = np.random.default_rng(77)
    x = rng.standard_normal(n, dtype=np.float32)
    x[rng.integers(0, n, 1000)] *= np.float32(1e6)
    t = to_dev(x)
    got = api.repro_cumsum(t, K=4)
    del t
    seg = 256 * 4096
    pos = [0, n - 1]
    for k in (1, 2, 1022, 1023, 1024, 1025, 1026, 1048):
        for d in (-2, -1, 0, 1, 4097):
            pos.append(k * seg + d)
    pos = np.unique(np.array([p for p in pos if 0 <= p < n] + rng.integers(0, n, 200).tolist()))
    g = got[torch.from_numpy(pos).to(got.device)].cpu().numpy()
    want = oracle.adn_cumsum_at(x, pos, 4)
    assert same_bits(g, want), first_diff(g, want)
