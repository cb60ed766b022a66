"""Pins of the CPU oracle to what the pages print and to mathematics.

No GPU: these run on the CPU only.  Every value compared against comes from a
golden fixture (tests/golden/, each citing its page), a closed form, an
invariant, or a brute-force exact computation on tiny inputs.
"""
import itertools
import math
import struct
from fractions import Fraction

import numpy as np
import pytest

from compensated_bit_reproducible_gb300 import inputs
from tests.golden import load_kv, load_rows

F32, F64 = np.float32, np.float64
GEO = {F64: dict(W=40, nb=52, b0=986, prec=53, qmin=-1074, emax=1024),
       F32: dict(W=13, nb=21, b0=117, prec=24, qmin=-149, emax=128)}


def bits(v):
    if isinstance(v, np.float32):
        return struct.unpack("<I", struct.pack("<f", float(v)))[0]
    return struct.unpack("<Q", struct.pack("<d", float(v)))[0]


def same_bits(a, b):
    return bits(a) == bits(b)


# ---------------------------------------------------------------- brute force
def round_frac(fr: Fraction, prec, qmin, emax):
    """Round-to-nearest-even of an exact rational (brute force)."""
    if fr == 0:
        return 0.0
    s = -1 if fr < 0 else 1
    a = abs(fr)
    E = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** E > a:
        E -= 1
    while Fraction(2) ** (E + 1) <= a:
        E += 1
    q = max(E - prec + 1, qmin)
    sc = a / Fraction(2) ** q
    m = math.floor(sc)
    rem = sc - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    if m == 2 ** prec:
        m //= 2
        q += 1
    if m.bit_length() - 1 + q >= emax:
        return s * math.inf
    return s * math.ldexp(m, q)


def rna(v: Fraction) -> int:
    q = math.floor(v)
    rem = v - q
    if rem > Fraction(1, 2):
        return q + 1
    if rem == Fraction(1, 2):
        return q + 1 if v > 0 else q
    return q


def brute_adn(xs, K, dt):
    """Definition of the closed form with exact rationals: index from max|x|,
    chained round-half-away pieces, exact fold sums, one rounding."""
    g = GEO[dt]
    vals = [float(x) for x in xs if math.isfinite(float(x)) and float(x) != 0.0]
    I = g["nb"] - K
    for x in vals:
        E = math.frexp(abs(x))[1] - 1
        I = min(I, max(0, min(g["nb"] - 1, (g["b0"] + g["W"] - 2 - E) // g["W"])))
    F = [0] * K
    for x in vals:
        r = Fraction(x)
        for k in range(K):
            gu = Fraction(2) ** (g["b0"] - g["W"] * (I + k))
            a = rna(r / gu)
            F[k] += a
            r -= a * gu
    tot = sum(F[k] * Fraction(2) ** (g["b0"] - g["W"] * (I + k)) for k in range(K))
    return dt(round_frac(tot, g["prec"], g["qmin"], g["emax"])), I, F


def tie_heavy(dt, n, seed, K=3):
    """Values whose low bits sit exactly on half a fold grid (rounding ties),
    plus one large value that fixes the index."""
    g = GEO[dt]
    rng = np.random.default_rng(seed)
    top = 60 if dt == F64 else 20
    big = dt(2.0 ** top * 1.5)
    E = top
    I = (g["b0"] + g["W"] - 2 - E) // g["W"]
    out = [big]
    for _ in range(n - 1):
        k = int(rng.integers(0, K))
        half = 2.0 ** (g["b0"] - g["W"] * (I + k) - 1)
        odd = int(rng.integers(0, 1 << (g["prec"] - 2))) * 2 + 1
        v = odd * half * (1 if rng.random() < 0.5 else -1)
        if abs(v) >= 2.0 ** (top + 1):
            v = math.copysign(half, v)
        out.append(dt(v))
    return np.array(out, dtype=dt)


# --------------------------------------------------------------------- pins
def test_quickstart_example(orc):
    """SyclReproSum, Quick Start: 1e16 pairs + 10000 ones."""
    g = load_kv("quickstart.txt")
    x = inputs.quickstart_f64()
    assert x.size == 2 * int(g["pairs"]) + int(g["ones"])
    want = float(g["expect_sum"])
    K = int(g["K"])
    for seed in range(10):
        xp = inputs.permuted(x, seed)
        for form in ("closed", "fp"):
            assert orc.adn_sum(xp, K, form) == want
        cs = orc.adn_cumsum(xp, K)
        assert cs[-1] == want
    # the closed form's fold sums hold the pairs and ones exactly
    I, F, fl = orc.adn_state(x, K)
    assert fl == 0 and I == 24


def test_kahan_page_example(orc):
    """Kahan's Summation Formula: printed naive / Kahan / theoretical values."""
    g = load_kv("kahan_thousandth.txt")
    x = inputs.thousandth_f32(int(g["n"]))
    assert x[0] == np.float32(float(g["element"]))
    assert "%.5f" % orc.sum_mode(x, "naive") == g["naive"]
    assert "%.5f" % orc.sum_mode(x, "kahan") == g["kahan"]
    ex = orc.exact_sum(x)
    assert "%.5f" % ex == g["theoretical"]
    # 0.001f is a multiple of the finest float grid at K=3 (2^-39 here), so the
    # binned sum is the correctly rounded exact sum.
    for form in ("closed", "fp"):
        assert same_bits(orc.adn_sum(x, 3, form), ex)


def test_capacity_constants(orc):
    g = load_kv("capacity.txt")
    assert orc.max_count(F32) == int(g["float"])
    assert orc.max_count(F64) == int(g["double"])


def test_geometry_constants(orc):
    g = load_kv("geometry.txt")
    for dt, nm in ((F32, "float"), (F64, "double")):
        assert orc.bin_width(dt) == int(g[nm + ".W"])
        assert orc.max_k(dt) == int(g[nm + ".max_k"])


@pytest.mark.parametrize("dt,nm", [(F32, "float"), (F64, "double")])
def test_absorption_threshold(orc, dt, nm):
    """Values below ~2^-1055 / ~2^-144 round away (How It Works).  Reading:
    the threshold is half the finest grid; a tie rounds away from zero."""
    t = int(load_kv("geometry.txt")[nm + ".absorb_log2"])
    thr = dt(2.0 ** t)
    below = np.nextafter(thr, dt(0))
    for K in (3, 2, 5):
        for form in ("closed", "fp"):
            assert orc.adn_sum(np.array([below], dt), K, form) == 0
            assert orc.adn_sum(np.array([-below, below, -below], dt), K, form) == 0
            assert orc.adn_sum(np.array([thr], dt), K, form) == dt(2.0 ** (t + 1))
            assert orc.adn_sum(np.array([-thr], dt), K, form) == dt(-(2.0 ** (t + 1)))


@pytest.mark.parametrize("dt,nm", [(F32, "float"), (F64, "double")])
def test_canonical_nan_and_inf(orc, dt, nm):
    g = load_kv("geometry.txt")
    nan_bits = int(g[nm + ".nan_bits"], 16)
    base = inputs.normal_f32(257, seed=5).astype(dt)
    for seed in range(5):
        x = inputs.inject_specials(base, "nan", seed=seed)
        for form in ("closed", "fp"):
            assert bits(orc.adn_sum(x, 3, form)) == nan_bits
        y = inputs.inject_specials(base, "pninf", seed=seed)
        assert bits(orc.adn_sum(y, 3)) == nan_bits
        z = inputs.inject_specials(base, "pinf", seed=seed)
        assert orc.adn_sum(z, 3) == np.inf
        assert orc.adn_sum(-z, 3) == -np.inf
        cs = orc.adn_cumsum(x, 3)
        first = int(np.flatnonzero(np.isnan(x))[0])
        assert all(bits(v) == nan_bits for v in cs[first:])
        assert not np.isnan(cs[:first]).any()


def test_bin_index_boundaries(orc):
    """Finest bin j with |x| < 2^(b0 - W j + W - 1)."""
    assert orc.bin_index(np.float32(3.4e38)) == 0
    assert orc.bin_index(np.float32(2.0 ** 116)) == 0
    assert orc.bin_index(np.nextafter(np.float32(2.0 ** 116), np.float32(0))) == 1
    assert orc.bin_index(np.float32(1.4e-45)) == 20
    assert orc.bin_index(1.7976931348623157e308) == 0
    assert orc.bin_index(2.0 ** 985) == 0
    assert orc.bin_index(np.nextafter(2.0 ** 985, 0)) == 1
    assert orc.bin_index(5e-324) == 51
    assert orc.bin_index(1e16) == 24


# ------------------------------------------------------------- invariants
def _datasets():
    rng = np.random.default_rng(11)
    d = []
    d.append(("normal32", inputs.normal_f32(3000, seed=3), (2, 3, 4, 7, 21)))
    d.append(("spikes32", inputs.normal_f32(3000, seed=4, spikes=True), (2, 3, 6)))
    d.append(("wide64", inputs.wide_f64(3000, seed=5), (2, 3, 6, 11, 52)))
    up = np.sort(np.abs(inputs.wide_f64(800, seed=6))) * np.where(rng.random(800) < .5, -1, 1)
    d.append(("rising64", up, (2, 3, 6)))
    d.append(("rising32", np.sort(np.abs(inputs.normal_f32(800, seed=7, spikes=True))).astype(F32), (3, 5)))
    d.append(("ties64", tie_heavy(F64, 400, 1), (3,)))
    d.append(("ties32", tie_heavy(F32, 400, 2), (3,)))
    sub = np.concatenate([rng.integers(-50, 50, 300) * 5e-324, [1e-300, -2e-310]])
    d.append(("subnormal64", sub.astype(F64), (2, 3, 52)))
    subf = (rng.integers(-50, 50, 300) * np.float32(1.4e-45)).astype(F32)
    d.append(("subnormal32", subf, (2, 3, 21)))
    top64 = np.concatenate([rng.uniform(-1, 1, 200) * 1.7e308, rng.standard_normal(200)])
    d.append(("top64", top64.astype(F64), (2, 3, 4)))
    top32 = np.concatenate([rng.uniform(-1, 1, 200) * 3.4e38, rng.standard_normal(200)]).astype(F32)
    d.append(("top32", top32, (2, 3, 4)))
    # renormalisation: many deposits of near-maximal pieces on every fold
    g = GEO[F32]
    E = 20
    I = (g["b0"] + g["W"] - 2 - E) // g["W"]
    hi = np.nextafter(F32(2.0 ** (g["b0"] - g["W"] * I + g["W"] - 1)), F32(0))
    d.append(("drift32", np.full(5000, hi, F32), (3,)))
    d.append(("drift64", np.full(9000, np.nextafter(2.0 ** 65, 0)), (3,)))
    return d


@pytest.mark.parametrize("name,x,Ks", _datasets(), ids=lambda v: v if isinstance(v, str) else "")
def test_forms_agree(orc, name, x, Ks):
    """The page's floating-point primary form equals the closed form bit for bit."""
    for K in Ks:
        a = orc.adn_sum(x, K, "closed")
        b = orc.adn_sum(x, K, "fp")
        assert same_bits(a, b), (name, K, a, b)


@pytest.mark.parametrize("dt", [F32, F64])
def test_closed_form_brute_force(orc, dt):
    """The C closed form equals exact rational arithmetic on small inputs."""
    for seed in range(6):
        for K in (2, 3, 4, 5, 6):
            # ties on the half grid of every fold of this K
            for x in (tie_heavy(dt, 40, seed, K=K), inputs.wide_f64(40, seed=seed).astype(dt)):
                want, I, F = brute_adn(x, K, dt)
                got = orc.adn_sum(x, K)
                I2, F2, fl = orc.adn_state(x, K)
                assert (I, F) == (I2, F2)
                assert same_bits(got, want)


@pytest.mark.parametrize("dt", [F32, F64])
def test_permutation_brute_force(orc, dt):
    """Every order of a tie-heavy multiset gives the same bits (floating-point
    form, which is order dependent internally)."""
    for seed in range(3):
        x = tie_heavy(dt, 7, 100 + seed)
        ref = orc.adn_sum(x, 3, "closed")
        for p in itertools.permutations(range(x.size)):
            assert same_bits(orc.adn_sum(x[list(p)], 3, "fp"), ref)


@pytest.mark.parametrize("dt", [F32, F64])
def test_order_independence_large(orc, dt):
    x = (inputs.wide_f64(20000, seed=9) if dt == F64 else inputs.normal_f32(20000, seed=9, spikes=True))
    ref = orc.adn_sum(x, 3, "fp")
    for seed in range(4):
        assert same_bits(orc.adn_sum(inputs.permuted(x, seed), 3, "fp"), ref)
    for K in (2, 6):
        assert same_bits(orc.adn_sum(x[::-1].copy(), K, "fp"), orc.adn_sum(x, K, "closed"))


def test_grid_aligned_inputs_are_exact(orc):
    """When every input is a multiple of the finest grid, the binned sum is the
    correctly rounded exact sum (integers, powers of two, geometric and
    telescoping series)."""
    rng = np.random.default_rng(3)
    cases = [
        rng.integers(-2 ** 40, 2 ** 40, 5000).astype(F64),
        (np.where(rng.random(2000) < .5, -1, 1) * 2.0 ** rng.integers(-40, 60, 2000)).astype(F64),
        2.0 ** -np.arange(0, 60, dtype=F64),
        np.array([(k + 1) ** 2 - k ** 2 for k in range(3000)], dtype=F64),
        rng.integers(-2 ** 20, 2 ** 20, 5000).astype(F32),
        (2.0 ** -np.arange(0, 30)).astype(F32),
    ]
    for x in cases:
        ex = orc.exact_sum(x)
        for form in ("closed", "fp"):
            assert same_bits(orc.adn_sum(x, 3, form), ex)


@pytest.mark.parametrize("dt,nm", [(F32, "float"), (F64, "double")])
def test_error_bound(orc, dt, nm):
    """|ADN - exact| <= N * 2^(-W (K-1)) * max|x| + half an ulp of the result
    (Template Parameters: dominant binned error term; 2^-80 / 2^-26 at K=3)."""
    g = GEO[dt]
    assert -g["W"] * 2 == int(load_kv("geometry.txt")[nm + ".err_log2_k3"])
    for seed in range(4):
        x = inputs.wide_f64(4000, seed=seed).astype(dt)
        x = x[np.isfinite(x)]
        ex = orc.exact_sum_fraction(x)
        mx = Fraction(float(np.max(np.abs(x))))
        for K in (2, 3, 4, 6):
            r = orc.adn_sum(x, K)
            err = abs(Fraction(float(r)) - ex)
            ulp = Fraction(float(np.spacing(np.abs(r)))) if r != 0 else Fraction(0)
            bound = x.size * mx * Fraction(2) ** (-g["W"] * (K - 1)) + ulp / 2
            assert err <= bound


@pytest.mark.parametrize("dt", [F32, F64])
def test_single_value_and_index_rule(orc, dt):
    """At K=3 any single value comes back exactly (its bits fit in the three
    folds below the top of its bin); the top fold holds its leading bits.
    With K=2 a full-width value at the top of its bin does not fit."""
    g = GEO[dt]
    rng = np.random.default_rng(4)
    xs = (inputs.wide_f64(500, seed=1) * rng.uniform(0.5, 2, 500)).astype(dt)
    for v in xs:
        a = np.array([v], dt)
        assert same_bits(orc.adn_sum(a, 3), v)
        I, F, _ = orc.adn_state(a, 3)
        assert abs(F[0]) <= 2 ** (g["W"] - 1)
        assert F[0] == rna(Fraction(float(v)) / Fraction(2) ** (g["b0"] - g["W"] * I))
    # all-ones significand at the bottom of bin 10 (leading bit one below the
    # bin's grid unit): its p bits need K W >= W + p - 1 grid positions, so
    # K=3 holds it and K=2 does not.  A one-bin-coarser index would lose it at
    # K=3 as well.
    E = g["b0"] - g["W"] * 10 - 1
    v = dt((2.0 - 2.0 ** (1 - g["prec"])) * 2.0 ** E)
    assert orc.bin_index(v) == 10
    assert orc.adn_sum(np.array([v], dt), 3) == v
    assert orc.adn_sum(np.array([v], dt), 2) != v


def test_cumsum_prefixes(orc):
    """Each output is the binned sum of its own prefix (closed form per
    prefix), the last one the full sum; sampled evaluation agrees."""
    for dt, x in ((F64, inputs.wide_f64(300, seed=8)), (F32, inputs.normal_f32(300, seed=8, spikes=True))):
        x = np.concatenate([x[:150] * dt(1e-20), x[150:]]).astype(dt)   # index raises mid-way
        cs = orc.adn_cumsum(x, 3)
        for i in range(0, x.size, 7):
            assert same_bits(cs[i], orc.adn_sum(x[:i + 1], 3, "closed"))
        assert same_bits(cs[-1], orc.adn_sum(x, 3))
        pos = np.array([0, 5, 5, 77, x.size - 1])
        at = orc.adn_cumsum_at(x, pos, 3)
        assert all(same_bits(a, cs[p]) for a, p in zip(at, pos))


def test_empty_and_zero_inputs(orc):
    for dt in (F32, F64):
        assert same_bits(orc.adn_sum(np.array([], dt), 3), dt(0.0))
        assert same_bits(orc.adn_sum(np.array([-0.0, -0.0], dt), 3), dt(0.0))
        assert same_bits(orc.adn_sum(np.array([1.0, -1.0], dt), 3), dt(0.0))


def test_segmented_sums_are_per_slice_sums(orc):
    """A segmented sum is one ADN sum per slice of a row-major array: each
    row (axis 1) or column (axis 0) against the sequential primary form of
    that slice alone, a different route from the closed form the segmented
    oracle uses, and, on integer data, the exact sums."""
    rng = np.random.default_rng(21)
    a = (rng.standard_normal((37, 53)) * np.exp2(rng.integers(-30, 30, (37, 1)))).astype(F32)
    a[5, 7] = F32(3e30)                     # one slice with a far higher index
    for K in (2, 3, 5):
        rows = orc.segsum(a, 1, K)
        cols = orc.segsum(a, 0, K)
        assert rows.shape == (37,) and cols.shape == (53,)
        for r in range(37):
            assert same_bits(rows[r], F32(orc.adn_sum(np.ascontiguousarray(a[r]), K, "fp")))
        for c in range(53):
            assert same_bits(cols[c], F32(orc.adn_sum(np.ascontiguousarray(a[:, c]), K, "fp")))
    z = rng.integers(-1000, 1000, (19, 23)).astype(F32)
    assert np.array_equal(orc.segsum(z, 1, 3), z.astype(np.int64).sum(axis=1).astype(F32))
    assert np.array_equal(orc.segsum(z, 0, 3), z.astype(np.int64).sum(axis=0).astype(F32))


# ------------------------------------------------------ comparison modes
def test_comparison_modes(orc):
    # the controlled case the reductions page alludes to: Neumaier keeps the
    # two ones that plain Kahan loses
    x = np.array([1.0, 1e100, 1.0, -1e100])
    assert orc.sum_mode(x, "neumaier") == 2.0
    assert orc.sum_mode(x, "kahan") == 0.0
    assert orc.sum_mode(x, "naive") == 0.0
    # integer data: every mode exact
    r = np.random.default_rng(1).integers(-1000, 1000, 4097).astype(F64)
    for mode in ("naive", "pairwise", "kahan", "neumaier"):
        assert orc.sum_mode(r, mode) == r.sum()
    # pairwise over a power-of-two run splits into its halves' trees
    y = inputs.normal_f32(1024, seed=2)
    assert same_bits(orc.sum_mode(y, "pairwise"),
                     F32(orc.sum_mode(y[:512], "pairwise") + orc.sum_mode(y[512:], "pairwise")))
    # chunked forms reduce to the plain ones with one chunk
    assert same_bits(orc.sum_mode(y, "kahan", chunk=4096), orc.sum_mode(y, "kahan"))
    assert same_bits(orc.sum_mode(y, "neumaier", chunk=4096), orc.sum_mode(y, "neumaier"))


# -------------------------------------------------------------- variance
def test_identical_values_table(orc):
    """Variance note, section 3: identical values.  Kernel exactly 0; naive
    and reference formula as printed."""
    for row in load_rows("variance_identical.txt"):
        v = np.float32(float(row[0]))
        x = np.full((1, 3), v, np.float32)
        assert "%g" % orc.var_naive(x, 1)[0] == row[1]
        assert "%g" % orc.var_twoterm(x, 1)[0] == row[2]
        k, m = orc.var_kernel(x, 1)
        assert "%g" % k[0] == row[3] and k[0] == 0.0 and m[0] == v


def test_identical_rows_4096(orc):
    x = inputs.identical_rows(4096)
    v, m = orc.var_kernel(x, 1)
    assert np.all(v == 0.0) and np.array_equal(m, x[:, 0])
    ref = orc.var_twoterm(x, 1)
    assert np.isnan(ref[3]) and np.isnan(ref[7])     # 4096 * 1e38 overflows


def test_complex_check(orc):
    g = load_kv("variance_complex.txt")
    z = np.array([complex(t.replace("j", "j")) for t in g["values"].split()], dtype=np.complex64)
    assert orc.var_kernel_complex(z) == float(g["var"])


def test_variance_closed_forms(orc):
    x = np.array([[0, 1, 2, 3]], np.float32)
    assert orc.var_kernel(x, 1)[0][0] == 1.25
    assert orc.var_kernel(x, 1, ddof=1)[0][0] == np.float32(np.float32(1.25) * np.float32(4 / 3))
    assert orc.var_kernel(np.array([[1, 3]], np.float32), 1, ddof=1)[0][0] == 2.0
    v, m = orc.var_kernel(np.array([[5.0]], np.float32), 1)
    assert v[0] == 0.0 and m[0] == 5.0
    # axis 0 == axis 1 of the transpose
    r = inputs.offset_rows(37, 29, seed=1)
    a0 = orc.var_kernel(r, 0)
    a1 = orc.var_kernel(np.ascontiguousarray(r.T), 1)
    assert np.array_equal(a0[0], a1[0]) and np.array_equal(a0[1], a1[1])


def test_variance_accuracy(orc):
    """Relative error against the float64 two-pass value: <= 5e-7 and never
    worse than twice the formula of reference on the note's datasets."""
    for name, x, axis in inputs.var_datasets(0):
        ref64, _ = orc.var_f64(x, axis)
        k, _ = orc.var_kernel(x, axis)
        t = orc.var_twoterm(x, axis)
        ek = np.max(np.abs(k - ref64) / ref64)
        et = np.max(np.abs(t - ref64) / ref64)
        assert ek <= 5e-7, (name, ek)
        assert ek <= 2 * et, (name, ek, et)
    x = inputs.offset_rows(64, 4096, seed=3)
    ref64, _ = orc.var_f64(x, 1, ddof=1)
    k, _ = orc.var_kernel(x, 1, ddof=1)
    assert np.max(np.abs(k - ref64) / ref64) <= 5e-7


def test_shift_is_exact_within_factor_two(orc):
    """Sterbenz: y = x - x0 is exact when x lies in [x0/2, 2 x0]; then the
    mean output x0 + m reproduces the float64 mean to float32 rounding."""
    rng = np.random.default_rng(0)
    x = rng.normal(1e6, 1.0, (1000, 64)).astype(np.float32)
    y32 = (x - x[0:1, :]).astype(np.float32)
    y64 = x.astype(np.float64) - x[0:1, :].astype(np.float64)
    assert np.array_equal(y32.astype(np.float64), y64)
    v, m = orc.var_kernel(x, 0)
    _, m64 = orc.var_f64(x, 0)
    assert np.all(np.abs(m - m64) <= np.spacing(np.float32(1e6)))


# ------------------------------------------------- variance extras (oracle)
VARIANTS = (0, 1, 2, 3, 4, 5, 6)


def arr_same(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return a.dtype == b.dtype and a.shape == b.shape and a.tobytes() == b.tobytes()


def test_variants_closed_form(orc):
    """Data with an integer mean and small integer deviations: every
    rounding step of every variant is exact, so each gives the exact
    population variance 5.25 and mean 5 (section 4 changes steps, not the
    value)."""
    x = np.array([[3, 7, 1, 5, 9, 5, 4, 6]], np.float32)
    for v in VARIANTS:
        var, mean = orc.var_variant(x, v, 1)
        assert var[0] == 5.25 and mean[0] == 5.0, v
    # the same slice along axis 0
    var, mean = orc.var_variant(np.ascontiguousarray(x.T), 6, 0)
    assert var[0] == 5.25 and mean[0] == 5.0


def test_variants_identical_values(orc):
    """Section 4, [1e38]*3 column (GPU): 0 for every variant with the shift,
    NaN for the formula of reference and the variant without the shift.
    Section 3 rows: identical values give exactly 0 with the shift."""
    x = np.full((1, 3), np.float32(1e38))
    for v in (0, 2, 3, 5, 6):
        assert orc.var_variant(x, v, 1)[0][0] == 0.0, v
    for v in (1, 4):
        assert np.isnan(orc.var_variant(x, v, 1)[0][0]), v
    for val in (1e10, 7.5e10, 1e15):
        y = np.full((1, 3), np.float32(val))
        for v in (0, 2, 3, 5, 6):
            assert orc.var_variant(y, v, 1)[0][0] == 0.0, (val, v)


def test_variants_zero_and_one_are_the_kernel_and_the_reference(orc):
    for name, x, axis in inputs.var_datasets(0):
        for ddof in (0, 1):
            k, m = orc.var_kernel(x, axis, ddof)
            v0, m0 = orc.var_variant(x, 0, axis, ddof)
            assert arr_same(k, v0) and arr_same(m, m0), name
            v1, _ = orc.var_variant(x, 1, axis, ddof)
            assert arr_same(v1, orc.var_twoterm(x, axis, ddof)), name


def test_variants_accuracy(orc):
    """Every variant stays within 2e-6 relative of the float64 two-pass value
    on the note's datasets (the plain trees lose at most about log2(n) ulps);
    the two-term correction and the shift do not change it by more."""
    for name, x, axis in inputs.var_datasets(0):
        ref64, _ = orc.var_f64(x, axis)
        for v in VARIANTS:
            var, _ = orc.var_variant(x, v, axis)
            err = np.max(np.abs(var - ref64) / ref64)
            assert err <= 2e-6, (name, v, err)


def test_kahan_variant_uses_the_sequential_loop(orc):
    """Variant 6 differs from the kernel only in s2: recomputing s2 with the
    comparison-mode Kahan loop over the same d^2 reproduces it."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((1, 777)) * 3 + 1e4).astype(np.float32)
    var, mean = orc.var_variant(x, 6, 1)
    r = x[0]
    y = (r - r[0]).astype(np.float32)
    m = np.float32(orc.sum_mode(y, "pairwise") / np.float32(r.size))
    d = (y - m).astype(np.float32)
    s2 = orc.sum_mode((d * d).astype(np.float32), "kahan")
    s1 = orc.sum_mode(d, "pairwise")
    t = np.float32(s1 / np.float32(r.size))
    want = np.float32(np.float32(s2 / np.float32(r.size)) - np.float32(t * t))
    assert var[0] == max(want, np.float32(0)) and mean[0] == np.float32(r[0] + m)


def test_f64_kernel_closed_forms_and_exactness(orc):
    x = np.array([[3, 7, 1, 5, 9, 5, 4, 6]], np.float64)
    v, m = orc.var_kernel_f64(x, 1)
    assert v[0] == 5.25 and m[0] == 5.0
    for val in (1.0, 1e10, 1e300, 1e307):
        v, m = orc.var_kernel_f64(np.full((1, 3), val), 1)
        assert v[0] == 0.0 and m[0] == val
    from fractions import Fraction
    rng = np.random.default_rng(5)
    x = rng.normal(1e6, 1.0, (4, 1000))
    v, m = orc.var_kernel_f64(x, 1, ddof=1)
    for r in range(4):
        fr = [Fraction(float(t)) for t in x[r]]
        mu = sum(fr) / len(fr)
        exact = sum((t - mu) ** 2 for t in fr) / (len(fr) - 1)
        assert abs(Fraction(float(v[r])) - exact) / exact < Fraction(1, 10 ** 13), r
        assert abs(Fraction(float(m[r])) - mu) <= Fraction(1, 2 ** 31)


def test_complex_2d_matches_parts_and_the_page(orc):
    g = load_kv("variance_complex.txt")
    z = np.array([complex(t) for t in g["values"].split()], dtype=np.complex64)
    v, m = orc.var_kernel_c64_2d(z.reshape(1, -1), 1)
    assert v[0] == float(g["var"])
    v0, _ = orc.var_kernel_c64_2d(z.reshape(-1, 1).copy(), 0)
    assert v0[0] == float(g["var"])
    # [7.5e10+7.5e10j]*3 gives 0 (section 3 table)
    v, m = orc.var_kernel_c64_2d(np.full((1, 3), 7.5e10 + 7.5e10j, np.complex64), 1)
    assert v[0] == 0.0 and m[0] == np.complex64(7.5e10 + 7.5e10j)
    rng = np.random.default_rng(6)
    zz = (rng.standard_normal((5, 37)) + 1j * rng.standard_normal((5, 37)) * 3 + 100).astype(np.complex64)
    for axis in (0, 1):
        v, m = orc.var_kernel_c64_2d(zz, axis, 1)
        vr, mr = orc.var_kernel(np.ascontiguousarray(zz.real), axis, 1)
        vi, mi = orc.var_kernel(np.ascontiguousarray(zz.imag), axis, 1)
        assert arr_same(v, (vr + vi).astype(np.float32))
        assert arr_same(m.real.copy(), mr) and arr_same(m.imag.copy(), mi)


# ------------------------------------------- compensation and renormalisation
@pytest.mark.parametrize("dt", [F32, F64])
def test_two_sum_is_error_free(orc, dt):
    """Variance note, section 2, step 3: TwoSum returns the rounded sum and
    its exact rounding error, so s = RN(a + b) and s + e = a + b exactly,
    whatever the exponent spread of the two operands."""
    rng = np.random.default_rng(31)
    span = 30 if dt == F32 else 60
    nonzero_errors = 0
    for _ in range(3000):
        a = dt(rng.standard_normal() * 2.0 ** int(rng.integers(-span, span)))
        b = dt(rng.standard_normal() * 2.0 ** int(rng.integers(-span, span)))
        s, e = orc.two_sum(a, b)
        assert same_bits(s, dt(a + b))
        assert Fraction(float(s)) + Fraction(float(e)) == Fraction(float(a)) + Fraction(float(b))
        nonzero_errors += e != 0
    assert nonzero_errors > 1000      # the pairs do round


def _plain_tree(v, dt):
    """Adjacent-pair tree of plain rounded adds (only used to pick slices on
    which the plain tree and the compensated tree must differ)."""
    a = [dt(t) for t in v]
    while len(a) > 1:
        nxt = [dt(a[2 * i] + a[2 * i + 1]) for i in range(len(a) // 2)]
        if len(a) % 2:
            nxt.append(a[-1])
        a = nxt
    return a[0]


@pytest.mark.parametrize("dt", [F32, F64])
def test_twosum_tree_gives_the_rounded_exact_sum(orc, dt):
    """Variance note, section 2, step 3 (errors carried up a second array,
    final sum plus final carry).  On integer slices of a power-of-two length
    whose values sum to zero, the shift and centring are exact, so d = x,
    s1 = 0 and var = s2 / n exactly.  The TwoSum errors are small integers,
    so the carries add without rounding and s2 must be the correctly rounded
    exact sum of the leaves RN(d_i * d_i).  Deviations up to 1.2 * 2^(p/2)
    make some leaves round and most partial sums need more than p bits, so
    the plain tree (a dropped error term) gives another value on many of
    these slices."""
    g = GEO[dt]
    rng = np.random.default_rng(41)
    lim = int(1.2 * 2 ** (g["prec"] // 2))
    differ = 0
    for _ in range(300):
        n = int(rng.choice([4, 8, 16, 32]))
        half = rng.integers(1, lim, n // 2)
        d = np.concatenate([half, -half])
        rng.shuffle(d)
        x = d.astype(dt)[None, :]
        leaves = [dt(dt(v) * dt(v)) for v in d]
        want = round_frac(sum(Fraction(float(t)) for t in leaves), g["prec"], g["qmin"], g["emax"])
        if dt == F32:
            var, mean = orc.var_kernel(x, 1)
        else:
            var, mean = orc.var_kernel_f64(x, 1)
        assert float(var[0]) * n == want, (d.tolist(), float(var[0]) * n, want)
        assert mean[0] == 0
        differ += float(_plain_tree(leaves, dt)) != want
    assert differ >= 30, differ
    if dt == F32:
        # the plain-tree variant (section 4, row 3) is the dropped-error tree
        x = np.array([[4095, -4095, 1, -1, 4095, -4095, 3, -3]], F32)
        plain = float(orc.var_variant(x, 3, 1)[0][0]) * 8
        comp = float(orc.var_kernel(x, 1)[0][0]) * 8
        leaves = [F32(F32(v) * F32(v)) for v in x[0]]
        assert comp == round_frac(sum(Fraction(float(t)) for t in leaves), 24, -149, 128)
        assert plain == float(_plain_tree(leaves, F32))


def _odd_last_piece_values(dt, K):
    """(values, I) for the renormalisation pin: a leading value that fixes the
    index at I, then a value whose last-fold piece is 2^(W-1) - 1 grid units
    (odd, the largest a fold takes) and whose piece on the fold above it is
    4095 grid units."""
    g = GEO[dt]
    W = g["W"]
    I = 8 if dt == F32 else 24
    grid = [Fraction(2) ** (g["b0"] - W * (I + k)) for k in range(K)]
    lead = grid[0]                                   # pieces (1, 0, ...)
    v = 4095 * grid[K - 2] + (2 ** (W - 1) - 1) * grid[K - 1]
    if dt == F32:
        v = 2047 * grid[K - 2] + (2 ** (W - 1) - 1) * grid[K - 1]   # 24 bits
    out = [dt(float(lead)), dt(float(v))]
    assert [Fraction(float(t)) for t in out] == [lead, v]
    return out, I


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("K", [2, 3])
def test_renormalisation_period(orc, dt, K):
    """SyclReproSum, How It Works, step 2: every 2^(p-W-2) deposits the
    primaries give their drift to the carries.  A primary starts in
    [1.5, 1.75) of its binade and each deposit moves it by at most
    2^(W-1) grid units, so one period keeps it in its binade; a longer one
    lets it leave, its ulp doubles and odd pieces round.  In a fold above the
    last that only moves the rounding difference down to the next fold, and
    the total stays; the last fold drops it.  So the pin drifts the last fold
    with its largest odd piece, in runs of both signs, for several periods,
    and compares the sequential primary form with exact rationals."""
    g = GEO[dt]
    period = 2 ** (g["prec"] - g["W"] - 2)
    (lead, v), I = _odd_last_piece_values(dt, K)
    want1, I1, F1 = brute_adn([lead, v], K, dt)
    assert I1 == I and F1[K - 1] == 2 ** (g["W"] - 1) - 1 and F1[K - 2] != 0
    _, _, Fv = brute_adn([lead, v], K, dt)
    Fv = [Fv[k] - (1 if k == 0 else 0) for k in range(K)]      # v's own pieces
    # lead and -lead fix the index and cancel, so the result is small enough
    # for its last bits to show the last fold's grid unit
    for runs in ((4 * period, -4 * period + 1), (-4 * period, 4 * period - 1),
                 (3 * period, -5 * period, 2 * period + 5), (8 * period + 77, -8 * period)):
        xs = np.concatenate([[lead, -lead]] + [np.full(abs(r), v if r > 0 else -v, dt) for r in runs])
        xs = xs.astype(dt)
        m = sum(runs)
        tot = sum(m * Fv[k] * Fraction(2) ** (g["b0"] - g["W"] * (I + k)) for k in range(K))
        want = dt(round_frac(tot, g["prec"], g["qmin"], g["emax"]))
        assert same_bits(orc.adn_sum(xs, K, "fp"), want), (runs,)
        assert same_bits(orc.adn_sum(xs, K, "closed"), want), (runs,)
    # the fold sums themselves, by brute force on one run
    xs = np.concatenate([[lead], np.full(4 * period, v, dt)]).astype(dt)
    assert brute_adn(xs, K, dt)[2] == [(1 if k == 0 else 0) + 4 * period * Fv[k] for k in range(K)]
