"""Small inputs: the one-block sum (n <= 16384) and the one-tile K = 3
cumulative sum (n <= 4096) against the oracle, across their thresholds, for
both the synchronous call (result in a pinned slot) and the stream-ordered
one."""
import threading

import numpy as np
import pytest
import torch

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.gpu_util import dev, first_diff, lib_sum, same_bits, to_dev

pytestmark = pytest.mark.gpu
F32, F64 = np.float32, np.float64
SUM_SIZES = [1, 2, 64, 1024, 2048, 2049, 16383, 16384, 16385]


def data(dt, n, seed):
    return inputs.normal_f32(n, seed=seed, spikes=True) if dt == F32 else inputs.wide_f64(n, seed=seed)


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("n", SUM_SIZES)
def test_sum_small_sizes(dt, n):
    dev()
    x = data(dt, n, n)
    for K in (2, 3, 6, 9):
        want = oracle.adn_sum(x, K, "fp")
        assert same_bits(lib_sum(x, K), want), (K, "async")
        got = api.repro_sum(to_dev(x), K)
        assert same_bits(np.array([got], dt)[0], want), (K, "sync")


@pytest.mark.parametrize("dt", [F32, F64])
def test_sum_one_block_shapes_and_grid_path_agree(dt):
    """The one-block kernel for every block size, and the grid path forced
    by an explicit grid, give the same bits."""
    dev()
    x = data(dt, 9001, 7)
    ref = oracle.adn_sum(x, 3, "fp")
    for block in (32, 96, 128, 256, 512, 1024):
        assert same_bits(lib_sum(x, 3, block=block), ref), block
    for grid in (1, 3, 40):
        assert same_bits(lib_sum(x, 3, grid=grid), ref), grid
    for off in (1, 3):
        assert same_bits(lib_sum(x, 3, offset=off), oracle.adn_sum(x[off:], 3, "fp")), off


@pytest.mark.parametrize("dt", [F32, F64])
def test_sum_small_specials_and_zero(dt):
    dev()
    b = data(dt, 1000, 3)
    for kind in ("nan", "pinf", "pninf"):
        y = inputs.inject_specials(b, kind, seed=1)
        assert same_bits(lib_sum(y, 3), oracle.adn_sum(y, 3, "fp")), kind
    z = -np.zeros(100, dt)
    got = api.repro_sum(to_dev(z), 3)
    assert np.array([got], dt).view(np.uint32 if dt == F32 else np.uint64)[0] == 0   # +0.0


def test_sync_sum_from_several_host_threads():
    """Each host thread has its own result slot: concurrent synchronous
    calls on separate streams return their own sums."""
    dev()
    xs = [data(F64, 5000 + 17 * i, 40 + i) for i in range(4)]
    want = [oracle.adn_sum(x, 3, "fp") for x in xs]
    tensors = [to_dev(x) for x in xs]
    got = [None] * len(xs)

    def work(i):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            vals = [api.repro_sum(tensors[i], 3, stream=s) for _ in range(50)]
        got[i] = vals

    th = [threading.Thread(target=work, args=(i,)) for i in range(len(xs))]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for i in range(len(xs)):
        assert all(v == want[i] for v in got[i]), i


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("n", [1, 2, 64, 1024, 2048, 2049, 4095, 4096, 4097])
def test_cumsum_one_tile(dt, n):
    dev()
    x = data(dt, n, n + 1).copy()
    x[: n // 2] *= dt(1e-9) if dt == F32 else 1e-30   # the index rises inside the tile
    want = oracle.adn_cumsum(x, 3)
    t = to_dev(x)
    got = api.repro_cumsum(t, K=3).cpu().numpy()
    assert same_bits(got, want), first_diff(got, want)
    api.repro_cumsum(t, out=t, K=3)   # in place
    assert same_bits(t.cpu().numpy(), want)


@pytest.mark.parametrize("dt", [F32, F64])
def test_cumsum_one_tile_specials(dt):
    dev()
    b = data(dt, 3000, 9)
    for kind in ("nan", "pinf", "pninf"):
        y = inputs.inject_specials(b, kind, seed=2)
        got = api.repro_cumsum(to_dev(y), K=3).cpu().numpy()
        assert same_bits(got, oracle.adn_cumsum(y, 3)), kind
