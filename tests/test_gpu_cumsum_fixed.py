"""Cumulative sums for n >= 2^17 on the fixed-index fast paths (K = 3 for
both types; K = 4..6 for double), with the first tile recomputed per fold
when the prefix index is still settling there, and the general kernels as
their fallback.  Every prefix must equal the oracle's."""
import numpy as np
import pytest

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.gpu_util import dev, first_diff, same_bits, to_dev

pytestmark = pytest.mark.gpu
F32, F64 = np.float32, np.float64
N = 200_003   # above the fast-path threshold; odd, so the last tile is partial


# (type, K): both K = 3 paths and the K = 4..6 double path
CASES = [(F32, 3), (F64, 3), (F64, 4), (F64, 6)]
CASE_IDS = ["f32-K3", "f64-K3", "f64-K4", "f64-K6"]


def cumsum(x, inplace=False, offset=0, K=3):
    t = to_dev(x)
    if offset:
        t = t[offset:]
    r = api.repro_cumsum(t, out=t if inplace else None, K=K)
    return r.cpu().numpy()


def check(x, K=3, **kw):
    off = kw.get("offset", 0)
    got = cumsum(x, K=K, **kw)
    want = oracle.adn_cumsum(x[off:], K)
    assert same_bits(got, want), first_diff(got, want)


def base(dt, seed):
    return inputs.wide_f64(N, seed=seed) if dt == F64 else inputs.normal_f32(N, seed=seed, spikes=True)


@pytest.mark.parametrize("dt,K", CASES, ids=CASE_IDS)
def test_typical_and_ties(dt, K):
    dev()
    check(base(dt, 21), K)
    from tests.test_oracle import tie_heavy
    check(tie_heavy(dt, N, 22, K=K), K)


@pytest.mark.parametrize("dt,K", CASES, ids=CASE_IDS)
@pytest.mark.parametrize("first", [0, 1, 4000, 4095, 4096, 9000, N // 2])
def test_where_the_index_settles(dt, K, first):
    """Everything before `first` is scaled far down, so the prefix index
    settles there: in the first tile (per-fold replay of that tile), at
    position 0 (all fast), or later (the general path)."""
    dev()
    x = base(dt, 23).copy()
    x[:first] *= dt(1e-9) if dt == F32 else 1e-30
    big = np.argmax(np.abs(x))
    x[first], x[big] = x[big], x[first]   # the maximum sits at `first`
    check(x, K)


@pytest.mark.parametrize("dt,K", CASES, ids=CASE_IDS)
@pytest.mark.parametrize("pos", [3, 5000, N - 1])
def test_outlier_outside_the_guessed_bin(dt, K, pos):
    dev()
    x = base(dt, 24).copy()
    x[pos] = dt(3e30) if dt == F32 else 3e200
    check(x, K)


@pytest.mark.parametrize("dt,K", CASES, ids=CASE_IDS)
def test_specials_zeros_subnormals(dt, K):
    dev()
    b = base(dt, 25)
    for kind in ("nan", "pinf", "pninf"):
        check(inputs.inject_specials(b, kind, seed=2), K)
    check(np.zeros(N, dt), K)
    m = b.copy()
    m[::3] = 0
    m[1::7] = dt(1e-45) if dt == F32 else 5e-324
    check(m, K)


@pytest.mark.parametrize("dt,K", CASES, ids=CASE_IDS)
def test_in_place_and_misaligned(dt, K):
    dev()
    x = base(dt, 26)
    check(x, K, inplace=True)
    for off in (1, 3):
        check(x, K, offset=off)


@pytest.mark.parametrize("n", [(1 << 17) - 1, 1 << 17, (1 << 17) + 1, 4096 * 40])
@pytest.mark.parametrize("dt,K", CASES, ids=CASE_IDS)
def test_threshold_sizes(n, dt, K):
    dev()
    x = inputs.wide_f64(n, seed=n).astype(dt)
    check(x, K)


@pytest.mark.parametrize("K", [3, 4, 6])
def test_cancellation_f64(K):
    """Every prefix of the second half cancels toward zero: lanes whose
    window cannot hold their prefixes take the exact conversion."""
    dev()
    a = inputs.wide_f64(N // 2, seed=27)
    check(np.concatenate([a, -a[::-1], [1.0]]), K)


@pytest.mark.parametrize("dt,K", CASES, ids=CASE_IDS)
def test_many_chunks_in_and_out_of_place_repeatable(dt, K):
    """About 2000 chunks (two levels of the chunk scan): out of place equal
    to the oracle, in place equal to it, and repeats bit for bit."""
    dev()
    n = 1_000_003
    x = inputs.wide_f64(n, seed=31).astype(dt) if dt == F64 else inputs.normal_f32(n, seed=31, spikes=True)
    want = oracle.adn_cumsum(x, K)
    got = cumsum(x, K=K)
    assert same_bits(got, want), first_diff(got, want)
    assert same_bits(cumsum(x, inplace=True, K=K), want)
    for _ in range(3):
        assert same_bits(cumsum(x, K=K), got)


def test_float_totals_beyond_64_bits():
    """Float: identical values just below the top of their bin (each rounded
    value about 2^38 grid units) push the running total past 2^62 units after
    2^24 elements, so later lanes take the 96-bit path instead of 64 bits.
    Sampled prefixes on both sides of the switch equal the oracle's."""
    dev()
    n = (1 << 24) + 300_000
    x = np.full(n, np.float32(4095.9), np.float32)
    x[::7] = np.float32(4095.5)
    got = cumsum(x)
    pos = np.array([0, 1, 4095, 4096, 1 << 20, (1 << 24) - 1, 1 << 24, (1 << 24) + 1,
                    (1 << 24) + 4096, (1 << 24) + 150_001, n - 1])
    want = oracle.adn_cumsum_at(x, pos, 3)
    assert same_bits(got[pos], want), first_diff(got[pos], want)


def test_double_totals_beyond_128_bits():
    """Double: runs of +v and -v with v just below the top of its bin (each
    rounded value about 2^119 grid units) move the running total back and
    forth across 2^126 units, so lanes take both the 128-bit and the 192-bit
    path.  Every prefix equals the oracle's."""
    dev()
    n = 200_003
    v = 0.999 * 2.0 ** 25
    i = np.arange(n)
    x = np.where((i // 1000) % 2 == 0, v, -v)
    x[::13] *= 0.75
    check(x)


@pytest.mark.parametrize("K", [4, 5, 6])
def test_wide_folds_magnitudes(K):
    """K = 4..6: values spread over the whole width of the folds (rounded
    values up to 2^(10 + 40 (K - 1)) grid units, down to ties on the finest
    grid), with runs that push the running total up and back."""
    dev()
    from tests.test_oracle import tie_heavy
    x = tie_heavy(F64, N, 40 + K, K=K)
    rng = np.random.default_rng(K)
    x[rng.integers(0, N, 500)] *= 2.0 ** 40
    check(x, K)
    runs = np.repeat(np.where(np.arange(N // 997 + 1) % 2 == 0, 1.0, -1.0), 997)[:N]
    check(base(F64, 41) * runs * 1e10, K)
