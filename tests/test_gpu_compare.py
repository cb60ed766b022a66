"""Comparison summation modes on the GPU against the CPU oracle."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.golden import load_kv
from tests.gpu_util import dev, same_bits, to_dev

pytestmark = pytest.mark.gpu
F32, F64 = np.float32, np.float64


def run(x, mode):
    return api.compare_sum(to_dev(x), mode).cpu().numpy()[0]


@pytest.mark.parametrize("n", [0, 1, 2, 3, 1000, 4096, 4097, 100003, 1_000_001])
@pytest.mark.parametrize("dt", [F32, F64])
def test_deterministic_modes_bit_exact(n, dt):
    dev()
    x = inputs.wide_f64(n, seed=n + 1).astype(dt)
    chunk = api.compensated_chunk()
    assert same_bits(run(x, "pairwise"), oracle.sum_mode(x, "pairwise"))
    assert same_bits(run(x, "kahan"), oracle.sum_mode(x, "kahan", chunk=chunk))
    assert same_bits(run(x, "neumaier"), oracle.sum_mode(x, "neumaier", chunk=chunk))


@pytest.mark.parametrize("dt", [F32, F64])
def test_naive_error_bound(dt):
    dev()
    x = inputs.normal_f32(1_000_003, seed=4).astype(dt)
    r = run(x, "naive")
    ex = oracle.exact_sum_fraction(x)
    eps = Fraction(2) ** (-24 if dt == F32 else -53)
    bound = x.size * eps * Fraction(float(np.sum(np.abs(x.astype(F64)))))
    assert abs(Fraction(float(r)) - ex) <= bound


def test_kahan_page_example_chunked():
    """10^6 x 0.001f: the chunked Kahan sum stays within two float ulps of the
    exact sum (the printed sequential Kahan value is one ulp away), while the
    plain parallel sum also beats the printed sequential naive value."""
    dev()
    g = load_kv("kahan_thousandth.txt")
    x = inputs.thousandth_f32(int(g["n"]))
    ex = float(oracle.exact_sum_fraction(x))
    ulp = float(np.spacing(F32(1000.0)))
    assert abs(float(run(x, "kahan")) - ex) <= 2 * ulp
    assert abs(float(run(x, "neumaier")) - ex) <= 2 * ulp
    assert abs(float(run(x, "naive")) - ex) < abs(float(g["naive"]) - ex)
