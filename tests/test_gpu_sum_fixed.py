"""Double binned sum for n >= 65536 and K = 2..6: the sampled fixed-index
kernel, with the general kernel as its fallback.  Every case must equal the
oracle bit for bit, whichever path produced it."""
import numpy as np
import pytest

import oracle
from compensated_bit_reproducible_gb300 import inputs
from tests.gpu_util import dev, lib_sum, same_bits

pytestmark = pytest.mark.gpu
F64 = np.float64
N = 200_003   # above the fixed-path threshold, odd (ragged tail)


def check(x, K=3, **kw):
    want = oracle.adn_sum(x, K, "fp")
    got = lib_sum(x, K, **kw)
    assert same_bits(got, want), (K, kw, got, want)


@pytest.mark.parametrize("K", [2, 3, 4, 5, 6])
def test_wide_and_ties(K):
    dev()
    from tests.test_oracle import tie_heavy
    check(inputs.wide_f64(N, seed=11), K)
    check(tie_heavy(F64, N, 12, K=K), K)


@pytest.mark.parametrize("K", [4, 5, 6])
def test_deep_folds(K):
    """A dynamic range of about 300 bits: elements on every fold's grid,
    below the finest grid, and ties there (K up to 6 keeps ten word
    positions and a 320-bit block total)."""
    dev()
    rng = np.random.default_rng(K)
    e = rng.integers(-250, 50, N)
    x = (rng.choice([-1.0, 1.0], N) * rng.uniform(1, 2, N) * np.exp2(e.astype(F64))).astype(F64)
    check(x, K)
    x[::11] = np.exp2(e[::11] - 60)                                  # far below the finest grid
    x[5::13] = np.exp2(-205.0) * (2 * rng.integers(0, 1000, x[5::13].size) + 1)
    check(x, K)
    check(np.concatenate([x, -x[:-1]]), K)                            # near-total cancellation


@pytest.mark.parametrize("pos", [1, 2, 777, 123457, N - 2, N - 1])
def test_outlier_outside_the_guessed_bin(pos):
    """One element far above the rest: wherever it sits, the result is the
    one at the true index (through the fallback if the sample missed it)."""
    dev()
    x = inputs.wide_f64(N, seed=13)
    x[pos] = 3.0e200
    check(x)
    check(x, 6)
    x[pos] = -3.0e200
    check(x, 2)
    check(x, 5)


def test_specials_at_size():
    dev()
    base = inputs.wide_f64(N, seed=14)
    for seed in range(3):
        y = inputs.inject_specials(base, "nan", seed=seed)
        assert np.array([lib_sum(y, 3)], F64).view(np.uint64)[0] == 0x7ff8000000000000
        y = inputs.inject_specials(base, "pninf", seed=seed)
        assert np.array([lib_sum(y, 3)], F64).view(np.uint64)[0] == 0x7ff8000000000000
        y = inputs.inject_specials(base, "pinf", seed=seed)
        assert lib_sum(y, 3) == np.inf and lib_sum(-y, 3) == -np.inf


@pytest.mark.parametrize("K", [3, 6])
def test_zeros_subnormals_and_extremes(K):
    dev()
    rng = np.random.default_rng(15)
    check(np.zeros(N, F64), K)
    check(-np.zeros(N, F64), K)
    check((rng.integers(-50, 50, N) * 5e-324).astype(F64), K)        # index too fine: fallback
    mixed = inputs.wide_f64(N, seed=16)
    mixed[::3] = 0.0
    mixed[1::7] = rng.integers(-9, 9, mixed[1::7].size) * 5e-324     # below the grid
    check(mixed, K)
    top = rng.uniform(-1, 1, N) * 1.7e308                             # index 0
    top[::5] = rng.standard_normal(top[::5].size)
    check(top, K)
    check(rng.integers(-2 ** 52, 2 ** 52, N).astype(F64), K)         # integers: low words zero
    check(np.full(N, 2.0 ** -30), K)                                   # identical values


@pytest.mark.parametrize("K", [3, 6])
def test_cancellation_and_permutation(K):
    dev()
    a = inputs.wide_f64(N // 2, seed=17)
    x = np.concatenate([a, -a, [1e-300]])
    check(x, K)
    ref = oracle.adn_sum(x, K, "fp")
    for seed in range(3):
        assert same_bits(lib_sum(inputs.permuted(x, seed), K), ref)


@pytest.mark.parametrize("K", [3, 6])
@pytest.mark.parametrize("block", [32, 96, 128, 256, 512, 1024])
def test_block_sizes_grids_offsets(block, K):
    dev()
    x = inputs.wide_f64(N, seed=18)
    ref = oracle.adn_sum(x, K, "fp")
    assert same_bits(lib_sum(x, K, block=block), ref)
    for grid in (1, 3, 2000):
        assert same_bits(lib_sum(x, K, block=block, grid=grid), ref), grid
    for off in (1, 3):
        assert same_bits(lib_sum(x, K, block=block, offset=off), oracle.adn_sum(x[off:], K, "fp")), off


@pytest.mark.parametrize("n", [65535, 65536, 65537, 131073])
def test_threshold_sizes(n):
    dev()
    x = inputs.wide_f64(n, seed=n)
    check(x, 3)
    check(x, 2)
    check(x, 6)


def test_paths_in_sequence():
    """Calls on one stream that take the first pass, the second pass (an
    element above the guessed bin) and the general kernel (specials, an
    index too fine) in turn: each leaves the stream's control words as it
    found them, so every result is the oracle's."""
    dev()
    base = inputs.wide_f64(N, seed=19)
    out = base.copy()
    out[4321] = -2.0e250
    top = base.copy()
    top[N // 3] = 1.7e308                                             # second pass at index 0
    tiny = (np.arange(N) % 17 - 8).astype(F64) * 5e-324
    nan = inputs.inject_specials(base, "nan", seed=5)
    for K in (3, 6, 3):
        for x in (base, out, base, top, tiny, out, base):
            check(x, K)
        assert np.isnan(lib_sum(nan, K))
        check(out, K)
        check(base, K)
