"""Binned sum on the GPU against the CPU oracle: bit for bit, for every
launch shape and input order."""
import numpy as np
import pytest
import torch

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.golden import load_kv
from tests.gpu_util import dev, first_diff, lib_sum, same_bits, to_dev

pytestmark = pytest.mark.gpu
F32, F64 = np.float32, np.float64


def tie_data(dt, n, seed):
    from tests.test_oracle import tie_heavy
    return tie_heavy(dt, n, seed)


def datasets():
    rng = np.random.default_rng(42)
    out = []
    for n in (1, 2, 3, 5, 7, 31, 100, 1000, 4097, 100003):
        out.append(("normal32_%d" % n, inputs.normal_f32(n, seed=n, spikes=True)))
        out.append(("wide64_%d" % n, inputs.wide_f64(n, seed=n)))
    out.append(("ties32", tie_data(F32, 5000, 1)))
    out.append(("ties64", tie_data(F64, 5000, 2)))
    out.append(("sub32", (rng.integers(-50, 50, 3000) * np.float32(1.4e-45)).astype(F32)))
    out.append(("sub64", (rng.integers(-50, 50, 3000) * 5e-324).astype(F64)))
    out.append(("top32", np.concatenate([rng.uniform(-1, 1, 500) * 3.4e38, rng.standard_normal(500)]).astype(F32)))
    out.append(("top64", np.concatenate([rng.uniform(-1, 1, 500) * 1.7e308, rng.standard_normal(500)]).astype(F64)))
    out.append(("zeros32", np.zeros(777, F32)))
    out.append(("negzero64", -np.zeros(777, F64)))
    out.append(("ints64", rng.integers(-2 ** 40, 2 ** 40, 20000).astype(F64)))
    out.append(("rising64", np.sort(np.abs(inputs.wide_f64(20000, seed=3)))))
    out.append(("rising32", np.sort(np.abs(inputs.normal_f32(20000, seed=3, spikes=True)))))
    out.append(("cancel64", np.concatenate([inputs.wide_f64(5000, seed=4), -inputs.wide_f64(5000, seed=4)])))
    return out


@pytest.mark.parametrize("name,x", datasets(), ids=lambda v: v if isinstance(v, str) else "")
def test_parity_k3(name, x):
    dev()
    want = oracle.adn_sum(x, 3, "fp")
    got = lib_sum(x, 3)
    assert same_bits(got, want), (name, got, want)


@pytest.mark.parametrize("K", [2, 4, 5, 6, 7, 8, 9, 13, 21])
def test_parity_other_k_f32(K):
    dev()
    for x in (inputs.normal_f32(30011, seed=K, spikes=True), tie_data(F32, 3000, K)):
        assert same_bits(lib_sum(x, K), oracle.adn_sum(x, K, "fp")), K


@pytest.mark.parametrize("K", [2, 4, 5, 6, 7, 8, 9, 20, 52])
def test_parity_other_k_f64(K):
    dev()
    for x in (inputs.wide_f64(30011, seed=K), tie_data(F64, 3000, K)):
        assert same_bits(lib_sum(x, K), oracle.adn_sum(x, K, "fp")), K


@pytest.mark.parametrize("dt", [F32, F64])
def test_misaligned_starts_and_ragged_tails(dt):
    dev()
    x = inputs.wide_f64(10007, seed=5).astype(dt)
    for off in (1, 2, 3, 5):
        got = lib_sum(x, 3, offset=off)
        assert same_bits(got, oracle.adn_sum(x[off:], 3)), off


def test_quickstart_permutations_and_block_sizes():
    dev()
    g = load_kv("quickstart.txt")
    x = inputs.quickstart_f64()
    want = np.float64(float(g["expect_sum"]))
    for seed in range(10):
        xp = inputs.permuted(x, seed)
        for block in (128, 256, 512):
            assert same_bits(lib_sum(xp, 3, block=block), want)
    # synchronous API with a host pointer: the library copies it to the device
    assert api.repro_sum(torch.from_numpy(x), 3) == 10000.0


def test_kahan_example():
    dev()
    g = load_kv("kahan_thousandth.txt")
    x = inputs.thousandth_f32(int(g["n"]))
    got = lib_sum(x, 3)
    assert "%.5f" % got == g["kahan"]
    assert same_bits(got, oracle.exact_sum(x))


@pytest.mark.parametrize("dt", [F32, F64])
def test_invariance_permutations_blocks_grids(dt):
    dev()
    x = inputs.normal_f32(1_000_003, seed=6, spikes=True) if dt == F32 else inputs.wide_f64(1_000_003, seed=6)
    ref = oracle.adn_sum(x, 3, "fp")
    for seed in range(10):
        xp = inputs.permuted(x, seed)
        for block in (128, 256, 512):
            assert same_bits(lib_sum(xp, 3, block=block), ref), (seed, block)
    for grid in (1, 7, 152, 1000, 5000):
        assert same_bits(lib_sum(x, 3, grid=grid), ref), grid


@pytest.mark.parametrize("dt", [F32, F64])
def test_specials(dt):
    dev()
    base = inputs.wide_f64(50001, seed=7).astype(dt)
    nan_bits = 0x7fc00000 if dt == F32 else 0x7ff8000000000000
    ui = np.uint32 if dt == F32 else np.uint64
    for seed in range(4):
        for kind in ("nan", "pninf"):
            y = inputs.inject_specials(base, kind, seed=seed)
            got = lib_sum(y, 3)
            assert np.array([got], dt).view(ui)[0] == nan_bits
        y = inputs.inject_specials(base, "pinf", seed=seed)
        assert lib_sum(y, 3) == np.inf and lib_sum(-y, 3) == -np.inf


def test_empty_and_zero():
    d = dev()
    for dt, tdt in ((F32, torch.float32), (F64, torch.float64)):
        out = torch.full((1,), 7.0, dtype=tdt, device=d)
        api.repro_sum_async(torch.empty(0, dtype=tdt, device=d), out, 3)
        assert same_bits(out.cpu().numpy()[0], dt(0.0))
        assert same_bits(lib_sum(np.array([-0.0, -0.0], dt), 3), dt(0.0))


@pytest.mark.parametrize("dt", [F32, F64])
def test_error_bound_against_exact(dt):
    dev()
    from fractions import Fraction
    W = 13 if dt == F32 else 40
    for seed in range(3):
        x = inputs.wide_f64(20000, seed=seed).astype(dt)
        ex = oracle.exact_sum_fraction(x)
        mx = Fraction(float(np.max(np.abs(x))))
        for K in (2, 3):
            r = lib_sum(x, K)
            ulp = Fraction(float(np.spacing(np.abs(r)))) if r != 0 else Fraction(0)
            assert abs(Fraction(float(r)) - ex) <= x.size * mx * Fraction(2) ** (-W * (K - 1)) + ulp / 2


@pytest.mark.slow
def test_full_size_f32_config():
    """100M N(0,1) float32 (and the 1%-spike variant), K=3: bit-exact with the
    oracle, and order-independent under a permutation."""
    dev()
    for spikes in (False, True):
        x = inputs.normal_f32(100_000_000, seed=1, spikes=spikes)
        want = oracle.adn_sum(x, 3, "fp")
        assert same_bits(lib_sum(x, 3), want)
        if spikes:
            assert same_bits(lib_sum(x[::-1].copy(), 3, block=512), want)


@pytest.mark.slow
def test_full_size_f64_config():
    """100M wide-range float64 with 10% cancelling pairs, K=3 and K=6."""
    dev()
    x = inputs.wide_f64(100_000_000, seed=2)
    for K in (3, 6):
        assert same_bits(lib_sum(x, K), oracle.adn_sum(x, K, "fp")), K


def test_segmented_rows_and_cols():
    dev()
    for rows, cols in ((1, 1), (3, 5), (17, 4096), (64, 1000), (5, 4099)):
        x = inputs.offset_rows(rows, cols, seed=rows)
        for axis in (1, 0):
            got = api.repro_segsum(to_dev(x), axis=axis, K=3).cpu().numpy()
            want = oracle.segsum(x, axis=axis, K=3)
            assert same_bits(got, want), (rows, cols, axis, first_diff(got, want))
    x = inputs.offset_rows(64, 333, seed=9, heavy=True)
    for K in (2, 5):
        got = api.repro_segsum(to_dev(x), axis=1, K=K).cpu().numpy()
        assert same_bits(got, oracle.segsum(x, axis=1, K=K))


def test_segmented_warp_and_block_rows_and_specials():
    """Rows up to 65536 columns take one warp per row, longer rows one block:
    both equal the oracle, also with Inf/NaN and tiny or huge rows."""
    dev()
    for rows, cols in ((3, 65536), (2, 65537), (2, 70001)):
        x = inputs.offset_rows(rows, cols, seed=cols)
        got = api.repro_segsum(to_dev(x), axis=1, K=3).cpu().numpy()
        assert same_bits(got, oracle.segsum(x, axis=1, K=3)), (rows, cols)
    x = inputs.offset_rows(8, 1000, seed=4)
    x[1, 5] = np.nan
    x[2, 7] = np.inf
    x[3, 9] = np.inf
    x[3, 10] = -np.inf
    x[4, :] = 0.0
    x[5, :] = np.float32(1e-45)
    x[6, ::2] = np.float32(3e38)
    for K in (2, 3):
        got = api.repro_segsum(to_dev(x), axis=1, K=K).cpu().numpy()
        assert same_bits(got, oracle.segsum(x, axis=1, K=K)), K


@pytest.mark.slow
def test_segmented_full_size_sampled_rows():
    """[4096, 4096] rows (offset + noise and the heavy-tailed variant): all
    rows computed on the GPU, 512 sampled rows checked against the oracle."""
    dev()
    rng = np.random.default_rng(0)
    for heavy in (False, True):
        x = inputs.offset_rows(4096, 4096, seed=3, heavy=heavy)
        got = api.repro_segsum(to_dev(x), axis=1, K=3).cpu().numpy()
        rows = np.sort(rng.choice(4096, 512, replace=False))
        want = oracle.segsum(x[rows], axis=1, K=3)
        assert same_bits(got[rows], want)
