"""Float32 variance kernel on the GPU against the CPU oracle (same tree
topology: bit for bit), plus the accuracy bounds against float64."""
import numpy as np
import pytest

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.golden import load_rows
from tests.gpu_util import dev, first_diff, same_bits, to_dev

pytestmark = pytest.mark.gpu


def gpu_var(x, axis, ddof):
    v, m = api.stable_var(to_dev(x), axis=axis, ddof=ddof)
    return v.cpu().numpy(), m.cpu().numpy()


def test_note_datasets_bit_exact_and_accurate():
    dev()
    for name, x, axis in inputs.var_datasets(0):
        v, m = gpu_var(x, axis, 0)
        wv, wm = oracle.var_kernel(x, axis, 0)
        assert same_bits(v, wv), (name, first_diff(v, wv))
        assert same_bits(m, wm), name
        ref64, _ = oracle.var_f64(x, axis, 0)
        tt = api.twoterm_var(to_dev(x), axis=axis).cpu().numpy()
        assert same_bits(tt, oracle.var_twoterm(x, axis, 0)), name
        ek = np.max(np.abs(v - ref64) / ref64)
        et = np.max(np.abs(tt - ref64) / ref64)
        assert ek <= 5e-7 and ek <= 2 * et, (name, ek, et)


def test_identical_values_exact_zero():
    dev()
    x = inputs.identical_rows(4096)
    v, m = gpu_var(x, 1, 0)
    assert np.all(v == 0.0) and same_bits(m, x[:, 0].copy())
    tt = api.twoterm_var(to_dev(x), axis=1).cpu().numpy()
    assert np.isnan(tt[3]) and np.isnan(tt[7])
    for row in load_rows("variance_identical.txt"):
        x3 = np.full((1, 3), np.float32(float(row[0])), np.float32)
        assert gpu_var(x3, 1, 0)[0][0] == 0.0
        assert "%g" % api.twoterm_var(to_dev(x3), axis=1).cpu().numpy()[0] == row[2]


@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 2), (3, 3), (5, 31), (7, 33), (4, 257), (9, 1000),
                                       (2, 4096), (3, 4097), (2, 70000), (1000, 64), (33, 7)])
@pytest.mark.parametrize("axis", [1, 0])
def test_ragged_shapes(rows, cols, axis):
    dev()
    x = inputs.offset_rows(rows, cols, seed=rows * 7 + cols)
    n = cols if axis == 1 else rows
    for ddof in (0, 1):
        if ddof >= n:
            continue
        v, m = gpu_var(x, axis, ddof)
        wv, wm = oracle.var_kernel(x, axis, ddof)
        assert same_bits(v, wv), (ddof, first_diff(v, wv))
        assert same_bits(m, wm)
        tt = api.twoterm_var(to_dev(x), axis=axis, ddof=ddof).cpu().numpy()
        assert same_bits(tt, oracle.var_twoterm(x, axis, ddof))


@pytest.mark.parametrize("rows,cols", [(3000, 37), (2600, 300), (1900, 1000), (1400, 2000), (1300, 4096),
                                       (1217, 4093), (1500, 256), (1300, 512), (1250, 1024), (1230, 2048)])
def test_more_rows_than_resident_blocks(rows, cols):
    """Row counts above one wave of resident blocks, for every per-thread
    leaf count C (1 to 16), rows that fill the block exactly (every thread
    holds C leaves) and rows with a ragged last thread."""
    dev()
    x = inputs.offset_rows(rows, cols, seed=rows + cols, heavy=(cols % 2 == 1))
    v, m = gpu_var(x, 1, 1)
    wv, wm = oracle.var_kernel(x, 1, 1)
    assert same_bits(v, wv), first_diff(v, wv)
    assert same_bits(m, wm)


@pytest.mark.slow
@pytest.mark.parametrize("cols", [4, 256])
def test_rows_beyond_the_grid_cap(cols):
    """More rows than the grid's 65535 * 16 blocks: blocks walk several rows
    (a ragged thread at 4 columns, rows that fill the block at 256)."""
    dev()
    rows = 65535 * 16 + 1237
    x = inputs.offset_rows(rows, cols, seed=cols)
    v, m = gpu_var(x, 1, 1)
    wv, wm = oracle.var_kernel(x, 1, 1)
    assert same_bits(v, wv), first_diff(v, wv)
    assert same_bits(m, wm)


def test_nonfinite_inputs():
    dev()
    x = inputs.offset_rows(6, 513, seed=1)
    x[1, 7] = np.nan
    x[2, 0] = np.inf
    x[3, 100] = -np.inf
    x[4, 5] = 3e38
    x[4, 6] = -3e38
    v, m = gpu_var(x, 1, 0)
    wv, wm = oracle.var_kernel(x, 1, 0)
    assert np.array_equal(np.isnan(v), np.isnan(wv))
    ok = ~np.isnan(wv)
    assert same_bits(v[ok], wv[ok])


@pytest.mark.slow
def test_full_size_config():
    """[4096, 4096] float32, axis 1, ddof 1 (offset + noise, and the
    heavy-tailed variant): bit-exact with the oracle; accuracy bound."""
    dev()
    for heavy in (False, True):
        x = inputs.offset_rows(4096, 4096, seed=3, heavy=heavy)
        v, m = gpu_var(x, 1, 1)
        wv, wm = oracle.var_kernel(x, 1, 1)
        assert same_bits(v, wv), first_diff(v, wv)
        assert same_bits(m, wm)
        ref64, _ = oracle.var_f64(x, 1, 1)
        assert np.max(np.abs(v - ref64) / ref64) <= 5e-7
