"""Variance extras on the GPU against the oracle, bit for bit: the section 4
variants of the float32 kernel, the kernel on float64 input, and complex64
input (real and imaginary variances added)."""
import numpy as np
import pytest
import torch

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.golden import load_kv
from tests.gpu_util import dev, first_diff, same_bits, to_dev

pytestmark = pytest.mark.gpu
SHAPES = [(1, 1), (3, 5), (7, 33), (5, 256), (4, 257), (9, 1000), (3, 1024), (2, 4096), (3, 4097), (2, 20000),
          (1000, 64), (33, 7)]


def gpu(x, axis, ddof, variant=0):
    v, m = api.stable_var(to_dev(x), axis=axis, ddof=ddof, variant=variant)
    return v.cpu().numpy(), m.cpu().numpy()


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_variants_bit_exact(variant, rows, cols):
    dev()
    if variant == 6 and rows * cols > 100000:
        pytest.skip("sequential loop: covered on the smaller shapes")
    x = inputs.offset_rows(rows, cols, seed=rows * 11 + cols)
    for axis in (1, 0):
        n = cols if axis == 1 else rows
        for ddof in (0, 1):
            if ddof >= n:
                continue
            v, m = gpu(x, axis, ddof, variant)
            wv, wm = oracle.var_variant(x, variant, axis, ddof)
            assert same_bits(v, wv), (axis, ddof, first_diff(v, wv))
            assert same_bits(m, wm), (axis, ddof)


def test_variants_on_the_note_datasets_and_identical_values():
    dev()
    for name, x, axis in inputs.var_datasets(0):
        for variant in range(7):
            v, m = gpu(x, axis, 0, variant)
            wv, wm = oracle.var_variant(x, variant, axis, 0)
            assert same_bits(v, wv) and same_bits(m, wm), (name, variant)
    x = np.full((1, 3), np.float32(1e38))
    for variant in (0, 2, 3, 5, 6):
        assert gpu(x, 1, 0, variant)[0][0] == 0.0, variant
    for variant in (1, 4):
        assert np.isnan(gpu(x, 1, 0, variant)[0][0]), variant


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_f64_bit_exact(rows, cols):
    dev()
    x = inputs.offset_rows(rows, cols, seed=rows * 13 + cols).astype(np.float64) * 1.0000001
    for axis in (1, 0):
        n = cols if axis == 1 else rows
        for ddof in (0, 1):
            if ddof >= n:
                continue
            v, m = gpu(x, axis, ddof)
            wv, wm = oracle.var_kernel_f64(x, axis, ddof)
            assert v.dtype == np.float64 and same_bits(v, wv), (axis, ddof, first_diff(v, wv))
            assert same_bits(m, wm)


def test_f64_identical_values():
    dev()
    for val in (1.0, 1e10, 1e300, 1e307):
        v, m = gpu(np.full((2, 3), val), 1, 0)
        assert np.all(v == 0.0) and np.all(m == val)


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_complex_bit_exact(rows, cols):
    dev()
    rng = np.random.default_rng(rows * 17 + cols)
    z = (rng.standard_normal((rows, cols)) * 2 + 1e3
         + 1j * (rng.standard_normal((rows, cols)) - 50)).astype(np.complex64)
    for axis in (1, 0):
        n = cols if axis == 1 else rows
        for ddof in (0, 1):
            if ddof >= n:
                continue
            v, m = gpu(z, axis, ddof)
            wv, wm = oracle.var_kernel_c64_2d(z, axis, ddof)
            assert v.dtype == np.float32 and same_bits(v, wv), (axis, ddof, first_diff(v, wv))
            assert m.dtype == np.complex64 and same_bits(m, wm)


@pytest.mark.parametrize("rows,cols", [(1500, 2048), (600, 4096), (900, 3000)])
def test_complex_rows_one_pass_many_rows(rows, cols):
    """Rows of up to 4096 elements take both parts in one pass (pair
    nodes; 512 threads at 4096): more rows than resident blocks, full and
    ragged rows, a heavy-tailed imaginary part."""
    dev()
    rng = np.random.default_rng(rows + cols)
    z = (rng.standard_normal((rows, cols)) + 5e4
         + 1j * (1e-3 * rng.standard_t(3, (rows, cols)))).astype(np.complex64)
    v, m = gpu(z, 1, 1)
    wv, wm = oracle.var_kernel_c64_2d(z, 1, 1)
    assert same_bits(v, wv), first_diff(v, wv)
    assert same_bits(m, wm)


@pytest.mark.slow
def test_complex_rows_beyond_the_grid_cap():
    """The one-pass complex kernel with more rows than its grid: blocks walk
    several rows."""
    dev()
    rows = 65535 * 16 + 901
    rng = np.random.default_rng(7)
    z = (rng.standard_normal((rows, 3)) + 1e4 + 1j * rng.standard_normal((rows, 3))).astype(np.complex64)
    v, m = gpu(z, 1, 1)
    wv, wm = oracle.var_kernel_c64_2d(z, 1, 1)
    assert same_bits(v, wv), first_diff(v, wv)
    assert same_bits(m, wm)


def test_complex_page_values():
    dev()
    g = load_kv("variance_complex.txt")
    z = np.array([complex(t) for t in g["values"].split()], dtype=np.complex64)
    assert gpu(z.reshape(1, -1), 1, 0)[0][0] == float(g["var"])
    assert gpu(z.reshape(-1, 1).copy(), 0, 0)[0][0] == float(g["var"])
    v, m = gpu(np.full((1, 3), 7.5e10 + 7.5e10j, np.complex64), 1, 0)
    assert v[0] == 0.0 and m[0] == np.complex64(7.5e10 + 7.5e10j)


def test_variant_argument_checks():
    dev()
    x = to_dev(inputs.offset_rows(3, 10, seed=1))
    out = torch.empty(3, dtype=torch.float32, device=x.device)
    from compensated_bit_reproducible_gb300.api import ReproError
    for bad in (-1, 7):
        with pytest.raises(ReproError):
            api.stable_var(x, axis=1, out=out, variant=bad)
