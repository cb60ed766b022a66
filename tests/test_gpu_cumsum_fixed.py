"""K = 3 cumulative sum for n >= 2^17: the fixed-index fast path (first tile
replayed per fold when the prefix index is still settling there), and the
general kernels as its fallback.  Every prefix must equal the oracle's."""
import numpy as np
import pytest

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.gpu_util import dev, first_diff, same_bits, to_dev

pytestmark = pytest.mark.gpu
F32, F64 = np.float32, np.float64
N = 200_003   # above the fast-path threshold; odd, so the last tile is partial


def cumsum(x, inplace=False, offset=0):
    t = to_dev(x)
    if offset:
        t = t[offset:]
    r = api.repro_cumsum(t, out=t if inplace else None, K=3)
    return r.cpu().numpy()


def check(x, **kw):
    off = kw.get("offset", 0)
    got = cumsum(x, **kw)
    want = oracle.adn_cumsum(x[off:], 3)
    assert same_bits(got, want), first_diff(got, want)


def base(dt, seed):
    return inputs.wide_f64(N, seed=seed) if dt == F64 else inputs.normal_f32(N, seed=seed, spikes=True)


@pytest.mark.parametrize("dt", [F32, F64])
def test_typical_and_ties(dt):
    dev()
    check(base(dt, 21))
    from tests.test_oracle import tie_heavy
    check(tie_heavy(dt, N, 22))


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("first", [0, 1, 4000, 4095, 4096, 9000, N // 2])
def test_where_the_index_settles(dt, first):
    """Everything before `first` is scaled far down, so the prefix index
    settles there: in the first tile (per-fold replay of that tile), at
    position 0 (all fast), or later (the general path)."""
    dev()
    x = base(dt, 23).copy()
    x[:first] *= dt(1e-9) if dt == F32 else 1e-30
    big = np.argmax(np.abs(x))
    x[first], x[big] = x[big], x[first]   # the maximum sits at `first`
    check(x)


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("pos", [3, 5000, N - 1])
def test_outlier_outside_the_guessed_bin(dt, pos):
    dev()
    x = base(dt, 24).copy()
    x[pos] = dt(3e30) if dt == F32 else 3e200
    check(x)


@pytest.mark.parametrize("dt", [F32, F64])
def test_specials_zeros_subnormals(dt):
    dev()
    b = base(dt, 25)
    for kind in ("nan", "pinf", "pninf"):
        check(inputs.inject_specials(b, kind, seed=2))
    check(np.zeros(N, dt))
    m = b.copy()
    m[::3] = 0
    m[1::7] = dt(1e-45) if dt == F32 else 5e-324
    check(m)


@pytest.mark.parametrize("dt", [F32, F64])
def test_in_place_and_misaligned(dt):
    dev()
    x = base(dt, 26)
    check(x, inplace=True)
    for off in (1, 3):
        check(x, offset=off)


@pytest.mark.parametrize("n", [(1 << 17) - 1, 1 << 17, (1 << 17) + 1, 4096 * 40])
@pytest.mark.parametrize("dt", [F32, F64])
def test_threshold_sizes(n, dt):
    dev()
    x = inputs.wide_f64(n, seed=n).astype(dt)
    check(x)


def test_cancellation_f64():
    dev()
    a = inputs.wide_f64(N // 2, seed=27)
    check(np.concatenate([a, -a[::-1], [1.0]]))


@pytest.mark.parametrize("dt", [F32, F64])
def test_many_chunks_in_and_out_of_place_repeatable(dt):
    """About 2000 chunks (two levels of the chunk scan): out of place equal
    to the oracle, in place equal to it, and repeats bit for bit."""
    dev()
    n = 1_000_003
    x = inputs.wide_f64(n, seed=31).astype(dt) if dt == F64 else inputs.normal_f32(n, seed=31, spikes=True)
    want = oracle.adn_cumsum(x, 3)
    got = cumsum(x)
    assert same_bits(got, want), first_diff(got, want)
    assert same_bits(cumsum(x, inplace=True), want)
    for _ in range(3):
        assert same_bits(cumsum(x), got)


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
