"""Binned states: deposits of any split of the input, merged in any order
and finalized, equal the oracle's sum of the whole input bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.gpu_util import dev, same_bits, to_dev

pytestmark = pytest.mark.gpu
F32, F64 = np.float32, np.float64
TD = {F32: torch.float32, F64: torch.float64}


def data(dt, n, seed):
    return inputs.normal_f32(n, seed=seed, spikes=True) if dt == F32 else inputs.wide_f64(n, seed=seed)


def split_points(n, rng, big):
    """Random cut points: tiny chunks, empty ones, and (if big) chunks above
    the one-block size, so both deposit paths run."""
    cuts = set(rng.integers(0, n, 12).tolist()) | {0, n}
    if big:
        cuts |= {min(n, 20000), min(n, 60000)}
    cuts |= {c + 1 for c in list(cuts) if c + 1 < n}   # one-element chunks
    return sorted(cuts)


def deposit_all(x, K, cuts, state=None):
    t = to_dev(x)
    st = state if state is not None else api.state_new(t.dtype, K)
    for a, b in zip(cuts[:-1], cuts[1:]):
        api.state_deposit(st, t[a:b], K)
    api.state_deposit(st, t[:0], K)   # empty deposit: no effect
    return st


def final(st, dt, K):
    return api.state_finalize(st, TD[dt], K).cpu().numpy()[0]


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("K", [2, 3, 6, 9])
def test_random_splits_equal_the_whole(dt, K):
    dev()
    rng = np.random.default_rng(K)
    x = data(dt, 100_003, 50 + K)
    want = oracle.adn_sum(x, K, "fp")
    for rep in range(3):
        st = deposit_all(x, K, split_points(x.size, rng, big=True))
        assert same_bits(final(st, dt, K), want), rep


@pytest.mark.parametrize("dt", [F32, F64])
def test_shards_merged_in_any_order(dt):
    """Four 'ranks' each deposit a contiguous shard; merging the four states
    in different tree shapes and orders gives the whole input's sum."""
    dev()
    rng = np.random.default_rng(3)
    x = data(dt, 80_000, 61)
    want = oracle.adn_sum(x, 3, "fp")
    q = np.array_split(np.arange(x.size), 4)
    for order in ([0, 1, 2, 3], [3, 2, 1, 0], [2, 0, 3, 1]):
        sts = [deposit_all(x[idx], 3, [0, idx.size]) for idx in q]
        api.state_merge(sts[order[0]], sts[order[1]], TD[dt], 3)
        api.state_merge(sts[order[2]], sts[order[3]], TD[dt], 3)
        api.state_merge(sts[order[2]], sts[order[0]], TD[dt], 3)
        assert same_bits(final(sts[order[2]], dt, 3), want), order
    # a copy of a state (bytes moved elsewhere) merges like the original
    s = deposit_all(x, 3, [0, x.size])
    c = s.clone()
    api.state_merge(c, s, TD[dt], 3)
    assert same_bits(final(c, dt, 3), oracle.adn_sum(np.concatenate([x, x]), 3, "fp"))


@pytest.mark.parametrize("dt", [F32, F64])
def test_index_raise_between_deposits(dt):
    dev()
    small = data(dt, 30_000, 70) * (dt(1e-9) if dt == F32 else 1e-30)
    large = data(dt, 30_000, 71)
    for first, second in ((small, large), (large, small)):
        x = np.concatenate([first, second])
        st = deposit_all(first, 3, [0, first.size])
        deposit_all(second, 3, [0, 9, second.size], state=st)
        assert same_bits(final(st, dt, 3), oracle.adn_sum(x, 3, "fp"))


@pytest.mark.parametrize("dt", [F32, F64])
def test_specials_across_deposits(dt):
    dev()
    b = data(dt, 9000, 72)
    pinf, ninf, nan = b.copy(), b.copy(), b.copy()
    pinf[5] = np.inf
    ninf[7] = -np.inf
    nan[11] = np.nan
    for parts, expect in (([b, pinf, b], "pinf"), ([ninf, b], "ninf"), ([pinf, b, ninf], "nan"), ([b, nan], "nan")):
        st = api.state_new(TD[dt], 3)
        for p in parts:
            api.state_deposit(st, to_dev(p), 3)
        got = final(st, dt, 3)
        want = oracle.adn_sum(np.concatenate(parts), 3, "fp")
        assert same_bits(got, want), expect


@pytest.mark.parametrize("dt", [F32, F64])
def test_empty_and_zero_states(dt):
    dev()
    st = api.state_new(TD[dt], 3)
    got = final(st, dt, 3)
    assert got == 0 and not np.signbit(got)
    api.state_deposit(st, to_dev(-np.zeros(1000, dt)), 3)
    got = final(st, dt, 3)
    assert got == 0 and not np.signbit(got)


def test_mismatched_k_or_type_finalizes_to_nan():
    dev()
    x = to_dev(data(F64, 1000, 73))
    st = api.state_new(torch.float64, 3)
    api.state_deposit(st, x, 4)          # K differs from the init
    assert np.isnan(final(st, F64, 3))
    a = api.state_new(torch.float32, 3)
    b = api.state_new(torch.float64, 3)
    api.state_merge(a, b, torch.float32, 3)   # a double state merged as float
    assert np.isnan(final(a, F32, 3))
    c = api.state_new(torch.float64, 3)
    assert np.isnan(final(c, F64, 2))   # finalized with another K


@pytest.mark.parametrize("dt", [F32, F64])
def test_state_bytes_through_host_memory(dt):
    """A state copied to host memory and back (as it would travel to another
    GPU) merges like the original: the layout holds no pointers."""
    dev()
    x = data(dt, 50_000, 80)
    a = deposit_all(x[:20_000], 3, [0, 20_000])
    b = deposit_all(x[20_000:], 3, [0, 30_000])
    host = b.cpu().numpy().copy()
    assert host.size == api.state_bytes(3)
    b2 = torch.from_numpy(host).to(a.device)
    api.state_merge(a, b2, TD[dt], 3)
    assert same_bits(final(a, dt, 3), oracle.adn_sum(x, 3, "fp"))


# ------------------------------------------- cumulative sums from a state
@pytest.mark.parametrize("dt,K", [(F32, 3), (F64, 3), (F32, 2), (F64, 4), (F64, 6), (F32, 6), (F64, 9)])
def test_cumsum_from_state_continues_the_whole_scan(dt, K):
    """A state holding x[:p] and the cumulative sum of x[p:] started from it
    give the whole input's cumulative sum at positions p.. (prefix indices,
    raises on either side of the cut, one- and multi-tile shards)."""
    dev()
    rng = np.random.default_rng(50 + K)
    n = 30_011
    x = data(dt, n, 60 + K).copy()
    x[:7000] *= dt(1e-12) if dt == F32 else 1e-40   # the index rises after the cut for some p
    want = oracle.adn_cumsum(x, K)
    for p in (0, 1, 4096, 6999, 7001, 12_345, n - 1):
        t = to_dev(x)
        st = api.state_new(t.dtype, K)
        if p:
            api.state_deposit(st, t[:p], K)
        got = api.repro_cumsum_from_state(t[p:].contiguous(), st, K).cpu().numpy()
        assert same_bits(got, want[p:]), (p, np.flatnonzero(got.view(np.uint8) != want[p:].view(np.uint8))[:3])
    # chained over shards: each shard starts from the merged states before it
    cuts = [0, 3000, 3001, 17_000, n]
    t = to_dev(x)
    carry = api.state_new(t.dtype, K)
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        parts.append(api.repro_cumsum_from_state(t[a:b].contiguous(), carry, K).cpu().numpy())
        api.state_deposit(carry, t[a:b], K)
    assert same_bits(np.concatenate(parts), want)


@pytest.mark.parametrize("dt", [F32, F64])
def test_chunked_pipeline_equals_one_call(dt):
    """The chunked form of a long input (as the benchmark's end-to-end leg
    streams it over the host link): chunk 0 by the plain cumulative sum
    (fixed-index path), chunk j from the state of chunks 0..j-1, each chunk
    then deposited; the outputs and the state's value are the oracle's
    cumulative sum and sum of the whole input."""
    dev()
    n = 2_000_003
    x = data(dt, n, 71)
    want = oracle.adn_cumsum(x, 3)
    t = to_dev(x)
    out = torch.empty_like(t)
    st = api.state_new(t.dtype, 3)
    step = -(-n // 8)
    step = -(-step // 64) * 64
    for j, a in enumerate(range(0, n, step)):
        b = min(n, a + step)
        if j == 0:
            api.repro_cumsum(t[a:b], out=out[a:b], K=3)
        else:
            api.repro_cumsum_from_state(t[a:b], st, 3, out=out[a:b])
        api.state_deposit(st, t[a:b], 3)
    got = out.cpu().numpy()
    assert same_bits(got, want), np.flatnonzero(got.view(np.uint8) != want.view(np.uint8))[:3]
    assert same_bits(final(st, dt, 3), np.array([oracle.adn_sum(x, 3, "fp")], dt)[0])


@pytest.mark.parametrize("dt", [F32, F64])
def test_cumsum_from_state_specials_and_mismatch(dt):
    dev()
    x = data(dt, 5000, 71)
    t = to_dev(x)
    nan_bits = np.array([np.nan], dt).view(np.uint32 if dt == F32 else np.uint64)[0]
    # a state holding a NaN makes every output the canonical NaN
    bad = x[:10].copy()
    bad[3] = np.nan
    st = api.state_new(t.dtype, 3)
    api.state_deposit(st, to_dev(bad), 3)
    got = api.repro_cumsum_from_state(t, st, 3).cpu().numpy()
    want = oracle.adn_cumsum(np.concatenate([bad, x]), 3)[10:]
    assert same_bits(got, want) and np.all(np.isnan(got))
    # a state of another K gives the canonical NaN, and no fold of it is read
    st6 = api.state_new(t.dtype, 6)
    got = api.repro_cumsum_from_state(t, st6, 3).cpu().numpy()
    canon = 0x7fc00000 if dt == F32 else 0x7ff8000000000000
    assert np.all(got.view(np.uint32 if dt == F32 else np.uint64) == canon)
    # in place
    st = api.state_new(t.dtype, 3)
    api.state_deposit(st, t[:100], 3)
    y = t[100:].clone()
    api.repro_cumsum_from_state(y, st, 3, out=y)
    assert same_bits(y.cpu().numpy(), oracle.adn_cumsum(x, 3)[100:])
