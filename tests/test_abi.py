"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments before touching pointers or the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "repro.h")


@pytest.fixture(scope="module")
def L():
    from compensated_bit_reproducible_gb300 import build, api
    build.build()
    return api.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    expected = {"repro_strerror", "repro_last_cuda_error", "repro_validate_environment",
                "repro_compensated_chunk", "stable_var_f32", "twoterm_var_f32", "repro_segsum_f32"}
    for t in ("f32", "f64"):
        expected |= {"repro_max_count_" + t, "repro_max_k_" + t, "repro_sum_" + t, "repro_sum_%s_async" % t,
                     "repro_cumsum_" + t, "repro_cumsum_%s_ex" % t}
        expected |= {"repro_sum_%s_%s" % (m, t) for m in ("naive", "pairwise", "kahan", "neumaier")}
    assert expected <= set(names), expected - set(names)
    for n in names:
        assert hasattr(L, n), n


def test_constants_match_the_pages(L):
    assert L.repro_max_count_f32() == 4294966784
    assert L.repro_max_count_f64() == 9223372036854773760
    assert L.repro_max_k_f32() == 21 and L.repro_max_k_f64() == 52
    assert L.repro_compensated_chunk() == 4096


def test_argument_errors_before_pointer_access(L):
    P = ctypes.c_void_p
    out = ctypes.c_float()
    outd = ctypes.c_double()
    bogus = P(0x10)   # never dereferenced: every case below fails its checks first
    # K out of range
    for K in (1, 22, 0, -3):
        assert L.repro_sum_f32(bogus, 10, K, None, ctypes.byref(out)) == 1
    assert L.repro_sum_f64(bogus, 10, 53, None, ctypes.byref(outd)) == 1
    # capacity, with a null pointer: the length check comes first
    assert L.repro_sum_f32(None, 4294966785, 3, None, ctypes.byref(out)) == 2
    assert L.repro_sum_f64(None, 9223372036854773761, 3, None, ctypes.byref(outd)) == 2
    assert L.repro_cumsum_f32(None, None, 4294966785, 3, None) == 2
    # null input with n > 0
    assert L.repro_sum_f32(None, 5, 3, None, ctypes.byref(out)) == 1
    # misaligned pointers
    assert L.repro_sum_f32(P(0x1002), 5, 3, None, ctypes.byref(out)) == 1
    assert L.repro_sum_f64(P(0x1004), 5, 3, None, ctypes.byref(outd)) == 1
    # overlapping (but not identical) cumsum ranges
    assert L.repro_cumsum_f32(P(0x100000), P(0x100004), 16, 3, None) == 3
    assert L.repro_cumsum_f64(P(0x100000), P(0x100040), 16, 3, None) == 3
    # n == 0 is a no-op / +0.0 without touching anything
    assert L.repro_cumsum_f32(None, None, 0, 3, None) == 0
    out.value = 7.0
    assert L.repro_sum_f32(None, 0, 3, None, ctypes.byref(out)) == 0 and out.value == 0.0
    # variance shape / ddof / axis checks
    assert L.stable_var_f32(bogus, 4, 4, 2, 0, bogus, None, None) == 1
    assert L.stable_var_f32(bogus, 4, 4, 1, 4, bogus, None, None) == 1
    assert L.stable_var_f32(bogus, 4, 4, 1, -1, bogus, None, None) == 1
    assert L.stable_var_f32(bogus, 0, 4, 1, 0, bogus, None, None) == 1
    assert L.repro_segsum_f32(bogus, 4, 4, 1, 22, bogus, None) == 1


def test_state_calls_check_arguments_first(L):
    P = ctypes.c_void_p
    assert L.repro_state_bytes(3) == 32 + 48
    assert L.repro_state_bytes(52) == 32 + 16 * 52
    assert L.repro_state_bytes(1) == 0 and L.repro_state_bytes(53) == 0
    good = P(0x100)   # aligned, never dereferenced: every case below fails first
    odd = P(0x108)    # not 16-byte aligned
    for t in ("f32", "f64"):
        init = getattr(L, "repro_state_init_" + t)
        dep = getattr(L, "repro_state_deposit_" + t)
        merge = getattr(L, "repro_state_merge_" + t)
        fin = getattr(L, "repro_state_finalize_" + t)
        assert init(good, 1, None) == 1
        assert init(None, 3, None) == 1
        assert init(odd, 3, None) == 1
        assert dep(good, None, 10, 3, None) == 1
        assert dep(odd, good, 10, 3, None) == 1
        assert dep(good, good, 10, 0, None) == 1
        cap = 4294966785 if t == "f32" else 9223372036854773761
        assert dep(good, None, cap, 3, None) == 2
        assert merge(good, None, 3, None) == 1
        assert merge(odd, good, 3, None) == 1
        assert fin(good, 3, None, None) == 1
        assert fin(odd, 3, good, None) == 1
    assert L.repro_state_init_f32(good, 22, None) == 1     # float folds: K <= 21
    assert L.repro_state_init_f64(good, 53, None) == 1
    # cumulative sums from a state: K, capacity, state, then the arrays
    for t, cap, esz in (("f32", 4294966785, 4), ("f64", 9223372036854773761, 8)):
        cs = getattr(L, "repro_cumsum_from_state_" + t)
        assert cs(good, good, 10, 1, good, None) == 1
        assert cs(None, None, cap, 3, good, None) == 2
        assert cs(good, good, 10, 3, None, None) == 1
        assert cs(good, good, 10, 3, odd, None) == 1
        assert cs(None, None, 0, 3, good, None) == 0          # empty: nothing is touched
        assert cs(None, good, 10, 3, good, None) == 1
        assert cs(P(0x1002), good, 10, 3, good, None) == 1   # misaligned input
        assert cs(P(0x100000), P(0x100000 + esz), 16, 3, good, None) == 3   # partial overlap


class Launch(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int), ("grid", ctypes.c_int)]


def test_launch_shapes_are_checked_first(L):
    """The *_ex and *_async calls reject a block size off [32, 1024] or not
    a multiple of 32, and a negative grid, before any pointer is touched."""
    P = ctypes.c_void_p
    good = P(0x100)
    bad = [Launch(16, 0), Launch(33, 0), Launch(2048, 0), Launch(256, -1)]
    for t in ("f32", "f64"):
        sa = getattr(L, "repro_sum_%s_async" % t)
        cx = getattr(L, "repro_cumsum_%s_ex" % t)
        for b in bad:
            assert sa(good, 1000, 3, None, good, ctypes.byref(b)) == 1, (t, b.block, b.grid)
            assert cx(good, good, 1000, 3, None, ctypes.byref(b)) == 1, (t, b.block, b.grid)
        assert sa(good, 1000, 3, None, None, None) == 1        # no result pointer
        assert sa(good, 1000, 3, None, P(0x101), None) == 1    # misaligned result pointer


def test_comparison_sums_check_arguments_first(L):
    P = ctypes.c_void_p
    good = P(0x100)
    for m in ("naive", "pairwise", "kahan", "neumaier"):
        for t, esz in (("f32", 4), ("f64", 8)):
            f = getattr(L, "repro_sum_%s_%s" % (m, t))
            assert f(None, 10, good, None) == 1                 # null input
            assert f(P(0x100 + esz // 2), 10, good, None) == 1  # misaligned input
            assert f(good, 10, None, None) == 1                 # null result
            assert f(good, 10, P(0x100 + esz // 2), None) == 1  # misaligned result
            assert f(good, (1 << 40) + 1, good, None) == 2      # above the supported length


def test_variance_and_noalloc_calls_check_arguments_first(L):
    P = ctypes.c_void_p
    good = P(0x100)
    i64 = ctypes.c_int64
    # float64 kernel: shape, ddof and alignment
    v64 = L.stable_var_f64
    assert v64(good, i64(4), i64(4), 2, 0, good, None, None) == 1
    assert v64(good, i64(4), i64(4), 1, 4, good, None, None) == 1
    assert v64(good, i64(0), i64(4), 1, 0, good, None, None) == 1
    assert v64(P(0x104), i64(4), i64(4), 1, 0, good, None, None) == 1
    assert v64(good, i64(4), i64(4), 1, 0, None, None, None) == 1
    assert v64(good, i64(4), i64(4), 1, 0, good, P(0x104), None) == 1
    # complex64: 8-byte pairs
    vc = L.stable_var_c64
    assert vc(P(0x104), i64(4), i64(4), 1, 0, good, None, None) == 1
    assert vc(good, i64(4), i64(4), 1, 0, good, P(0x104), None) == 1
    assert vc(good, i64(4), i64(4), 0, 4, good, None, None) == 1
    # variants 0..6 only
    vv = L.stable_var_f32_variant
    for variant in (-1, 7):
        assert vv(good, i64(4), i64(4), 1, 0, variant, good, None, None) == 1
    assert L.twoterm_var_f32(good, i64(4), i64(4), 3, 0, good, None) == 1
    # allocation-free sum: K, capacity, pointers
    na = L.repro_sum_f32_noalloc
    for K in (1, 22):
        assert na(good, 10, K, None, good) == 1
    assert na(None, 4294966785, 3, None, good) == 2
    assert na(None, 10, 3, None, good) == 1
    assert na(P(0x102), 10, 3, None, good) == 1
    assert na(good, 10, 3, None, None) == 1
    assert na(good, 10, 3, None, P(0x102)) == 1


def test_strerror(L):
    for s in range(7):
        assert L.repro_strerror(s)


def test_noalloc_cuda_error_reaches_last_cuda_error(L):
    """Without a usable GPU the allocation-free sum fails in its first CUDA
    call; the code must come back through repro_last_cuda_error() in the
    calling thread, like every other entry point's.  A fresh thread starts
    with an empty error slot, so a code kept anywhere else reads as 0."""
    import threading
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a usable GPU (the pointers here are not real)")
    P = ctypes.c_void_p
    got = {}

    def call():
        got["rc"] = L.repro_sum_f32_noalloc(P(0x1000), 16, 3, None, P(0x2000))
        got["cuda"] = L.repro_last_cuda_error()

    t = threading.Thread(target=call)
    t.start()
    t.join()
    assert got["rc"] == 5, got
    assert got["cuda"] != 0, got
