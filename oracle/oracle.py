"""ctypes binding of the C oracle (test infrastructure only).

`build()` compiles the oracle with gcc (strict IEEE: no contraction, no
fast-math) into oracle/_build/liboracle.so; every other function loads it on
first use and takes/returns numpy arrays and Python scalars.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from fractions import Fraction

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SOURCES = ["fixacc.c", "adn.c", "sums.c", "variance.c", "exact.c"]
_HEADERS = ["oracle.h", "fixacc.h"]
_lib = None

CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-frounding-math", "-fexcess-precision=standard", "-Wall"]


def _stale() -> bool:
    if not os.path.exists(_SO):
        return True
    t = os.path.getmtime(_SO)
    return any(os.path.getmtime(os.path.join(_HERE, f)) > t for f in _SOURCES + _HEADERS)


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent)."""
    if force or _stale():
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + ".tmp.%d" % os.getpid()
        cmd = ["gcc", *CFLAGS, "-o", tmp, *[os.path.join(_HERE, f) for f in _SOURCES], "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        sig = {
            "orc_exact_sum_f64": (ci, [P, i64, P]),
            "orc_exact_sum_f32": (ci, [P, i64, P]),
            "orc_exact_sum_limbs_f64": (ci, [P, i64, P, ci, P]),
            "orc_exact_sum_limbs_f32": (ci, [P, i64, P, ci, P]),
            "orc_max_count_f32": (ctypes.c_uint64, []),
            "orc_max_count_f64": (ctypes.c_uint64, []),
            "orc_max_k_f32": (ci, []),
            "orc_max_k_f64": (ci, []),
            "orc_bin_width_f32": (ci, []),
            "orc_bin_width_f64": (ci, []),
            "orc_bin_index_f64": (ci, [ctypes.c_double]),
            "orc_bin_index_f32": (ci, [ctypes.c_float]),
            "orc_adn_sum_closed_f64": (ctypes.c_double, [P, i64, ci]),
            "orc_adn_sum_closed_f32": (ctypes.c_float, [P, i64, ci]),
            "orc_adn_state_closed_f64": (None, [P, i64, ci, P, P, P, P]),
            "orc_adn_state_closed_f32": (None, [P, i64, ci, P, P, P, P]),
            "orc_adn_sum_fp_f64": (ctypes.c_double, [P, i64, ci]),
            "orc_adn_sum_fp_f32": (ctypes.c_float, [P, i64, ci]),
            "orc_adn_cumsum_f64": (None, [P, P, i64, ci]),
            "orc_adn_cumsum_f32": (None, [P, P, i64, ci]),
            "orc_adn_cumsum_at_f64": (None, [P, i64, ci, P, i64, P]),
            "orc_adn_cumsum_at_f32": (None, [P, i64, ci, P, i64, P]),
            "orc_sum_naive_f64": (ctypes.c_double, [P, i64]),
            "orc_sum_naive_f32": (ctypes.c_float, [P, i64]),
            "orc_sum_pairwise_f64": (ctypes.c_double, [P, i64]),
            "orc_sum_pairwise_f32": (ctypes.c_float, [P, i64]),
            "orc_sum_kahan_f64": (ctypes.c_double, [P, i64]),
            "orc_sum_kahan_f32": (ctypes.c_float, [P, i64]),
            "orc_sum_neumaier_f64": (ctypes.c_double, [P, i64]),
            "orc_sum_neumaier_f32": (ctypes.c_float, [P, i64]),
            "orc_sum_kahan_chunked_f64": (ctypes.c_double, [P, i64, i64]),
            "orc_sum_kahan_chunked_f32": (ctypes.c_float, [P, i64, i64]),
            "orc_sum_neumaier_chunked_f64": (ctypes.c_double, [P, i64, i64]),
            "orc_sum_neumaier_chunked_f32": (ctypes.c_float, [P, i64, i64]),
            "orc_var_kernel_f32": (None, [P, i64, i64, ci, ci, P, P]),
            "orc_var_twoterm_f32": (None, [P, i64, i64, ci, ci, P]),
            "orc_var_naive_f32": (None, [P, i64, i64, ci, ci, P]),
            "orc_var_f64": (None, [P, i64, i64, ci, ci, P, P]),
            "orc_segsum_f32": (None, [P, i64, i64, ci, ci, P]),
            "orc_var_kernel_c64": (None, [P, P, i64, ci, P]),
            "orc_var_kernel_c64_2d": (None, [P, i64, i64, ci, ci, P, P]),
            "orc_var_variant_f32": (None, [P, i64, i64, ci, ci, ci, P, P]),
            "orc_var_kernel_f64": (None, [P, i64, i64, ci, ci, P, P]),
            "orc_two_sum_f32": (None, [ctypes.c_float, ctypes.c_float, P, P]),
            "orc_two_sum_f64": (None, [ctypes.c_double, ctypes.c_double, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _arr(x, dtype):
    a = np.ascontiguousarray(x, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _sfx(x):
    a = np.asarray(x)
    if a.dtype == np.float32:
        return "f32", np.float32
    if a.dtype == np.float64:
        return "f64", np.float64
    raise TypeError("float32 or float64 input expected, got %s" % a.dtype)


# ---- constants -------------------------------------------------------------
def max_count(dtype) -> int:
    return int(_L().orc_max_count_f32() if np.dtype(dtype) == np.float32 else _L().orc_max_count_f64())


def max_k(dtype) -> int:
    return int(_L().orc_max_k_f32() if np.dtype(dtype) == np.float32 else _L().orc_max_k_f64())


def bin_width(dtype) -> int:
    return int(_L().orc_bin_width_f32() if np.dtype(dtype) == np.float32 else _L().orc_bin_width_f64())


def bin_index(x) -> int:
    if isinstance(x, np.float32):
        return int(_L().orc_bin_index_f32(float(x)))
    return int(_L().orc_bin_index_f64(float(x)))


# ---- exact sums --------------------------------------------------------------
def exact_sum(x):
    """Exact sum rounded once to the input type (None if Inf/NaN present)."""
    sfx, dt = _sfx(x)
    a, p = _arr(x, dt)
    out = np.zeros(1, dtype=dt)
    rc = getattr(_L(), "orc_exact_sum_" + sfx)(p, a.size, out.ctypes.data_as(ctypes.c_void_p))
    return None if rc else out[0]


def exact_sum_fraction(x) -> Fraction:
    """The exact sum as a Fraction (finite inputs only)."""
    sfx, dt = _sfx(x)
    a, p = _arr(x, dt)
    limbs = np.zeros(40, dtype=np.uint64)
    lsb = ctypes.c_int(0)
    n = getattr(_L(), "orc_exact_sum_limbs_" + sfx)(p, a.size, limbs.ctypes.data_as(ctypes.c_void_p),
                                                    40, ctypes.byref(lsb))
    if n == 0:
        raise ValueError("non-finite input")
    v = 0
    for i in range(n - 1, -1, -1):
        v = (v << 64) | int(limbs[i])
    if v >> (64 * n - 1):
        v -= 1 << (64 * n)
    e = lsb.value
    return Fraction(v) * (Fraction(2) ** e)


# ---- ADN -------------------------------------------------------------------
def adn_sum(x, K: int = 3, form: str = "closed"):
    sfx, dt = _sfx(x)
    a, p = _arr(x, dt)
    fn = getattr(_L(), "orc_adn_sum_%s_%s" % (form, sfx))
    return dt(fn(p, a.size, K))


def adn_state(x, K: int = 3):
    """(I, [F_k as Python ints], flags) of the closed form."""
    sfx, dt = _sfx(x)
    a, p = _arr(x, dt)
    I = ctypes.c_int(0)
    fl = ctypes.c_int(0)
    hi = np.zeros(max(K, 1), dtype=np.int64)
    lo = np.zeros(max(K, 1), dtype=np.uint64)
    getattr(_L(), "orc_adn_state_closed_" + sfx)(p, a.size, K, ctypes.byref(I),
                                                 hi.ctypes.data_as(ctypes.c_void_p),
                                                 lo.ctypes.data_as(ctypes.c_void_p), ctypes.byref(fl))
    F = [(int(hi[k]) << 64) | int(lo[k]) for k in range(K)]
    return I.value, F, fl.value


def adn_cumsum(x, K: int = 3):
    sfx, dt = _sfx(x)
    a, p = _arr(x, dt)
    out = np.empty_like(a)
    getattr(_L(), "orc_adn_cumsum_" + sfx)(p, out.ctypes.data_as(ctypes.c_void_p), a.size, K)
    return out


def adn_cumsum_at(x, pos, K: int = 3):
    """Prefix sums at sorted positions `pos` (int64), one pass over x."""
    sfx, dt = _sfx(x)
    a, p = _arr(x, dt)
    ps = np.ascontiguousarray(pos, dtype=np.int64)
    assert np.all(np.diff(ps) >= 0)
    out = np.empty(ps.size, dtype=dt)
    getattr(_L(), "orc_adn_cumsum_at_" + sfx)(p, a.size, K, ps.ctypes.data_as(ctypes.c_void_p), ps.size,
                                              out.ctypes.data_as(ctypes.c_void_p))
    return out


def segsum(x2d, axis: int = 1, K: int = 3):
    a, p = _arr(x2d, np.float32)
    rows, cols = a.shape
    out = np.empty(rows if axis == 1 else cols, dtype=np.float32)
    _L().orc_segsum_f32(p, rows, cols, axis, K, out.ctypes.data_as(ctypes.c_void_p))
    return out


# ---- comparison modes -------------------------------------------------------
def sum_mode(x, mode: str, chunk: int = 0):
    sfx, dt = _sfx(x)
    a, p = _arr(x, dt)
    if chunk:
        fn = getattr(_L(), "orc_sum_%s_chunked_%s" % (mode, sfx))
        return dt(fn(p, a.size, chunk))
    fn = getattr(_L(), "orc_sum_%s_%s" % (mode, sfx))
    return dt(fn(p, a.size))


# ---- variance ----------------------------------------------------------------
def var_kernel(x2d, axis: int = 1, ddof: int = 0):
    a, p = _arr(x2d, np.float32)
    rows, cols = a.shape
    ns = rows if axis == 1 else cols
    v = np.empty(ns, dtype=np.float32)
    m = np.empty(ns, dtype=np.float32)
    _L().orc_var_kernel_f32(p, rows, cols, axis, ddof, v.ctypes.data_as(ctypes.c_void_p),
                            m.ctypes.data_as(ctypes.c_void_p))
    return v, m


def var_twoterm(x2d, axis: int = 1, ddof: int = 0):
    a, p = _arr(x2d, np.float32)
    rows, cols = a.shape
    v = np.empty(rows if axis == 1 else cols, dtype=np.float32)
    _L().orc_var_twoterm_f32(p, rows, cols, axis, ddof, v.ctypes.data_as(ctypes.c_void_p))
    return v


def var_naive(x2d, axis: int = 1, ddof: int = 0):
    a, p = _arr(x2d, np.float32)
    rows, cols = a.shape
    v = np.empty(rows if axis == 1 else cols, dtype=np.float32)
    _L().orc_var_naive_f32(p, rows, cols, axis, ddof, v.ctypes.data_as(ctypes.c_void_p))
    return v


def var_f64(x2d, axis: int = 1, ddof: int = 0):
    a, p = _arr(x2d, np.float32)
    rows, cols = a.shape
    ns = rows if axis == 1 else cols
    v = np.empty(ns, dtype=np.float64)
    m = np.empty(ns, dtype=np.float64)
    _L().orc_var_f64(p, rows, cols, axis, ddof, v.ctypes.data_as(ctypes.c_void_p),
                     m.ctypes.data_as(ctypes.c_void_p))
    return v, m


def var_kernel_complex(z, ddof: int = 0):
    zz = np.asarray(z, dtype=np.complex64)
    re, pr = _arr(zz.real, np.float32)
    im, pi = _arr(zz.imag, np.float32)
    out = np.zeros(1, dtype=np.float32)
    _L().orc_var_kernel_c64(pr, pi, re.size, ddof, out.ctypes.data_as(ctypes.c_void_p))
    return out[0]


def var_variant(x2d, variant: int, axis: int = 1, ddof: int = 0):
    """Section 4 variants of the float32 kernel (see orc_var_variant_f32)."""
    a, p = _arr(x2d, np.float32)
    rows, cols = a.shape
    ns = rows if axis == 1 else cols
    v = np.empty(ns, dtype=np.float32)
    m = np.empty(ns, dtype=np.float32)
    _L().orc_var_variant_f32(p, rows, cols, axis, ddof, variant, v.ctypes.data_as(ctypes.c_void_p),
                             m.ctypes.data_as(ctypes.c_void_p))
    return v, m


def var_kernel_f64(x2d, axis: int = 1, ddof: int = 0):
    """The kernel on float64 input, every step in float64."""
    a, p = _arr(x2d, np.float64)
    rows, cols = a.shape
    ns = rows if axis == 1 else cols
    v = np.empty(ns, dtype=np.float64)
    m = np.empty(ns, dtype=np.float64)
    _L().orc_var_kernel_f64(p, rows, cols, axis, ddof, v.ctypes.data_as(ctypes.c_void_p),
                            m.ctypes.data_as(ctypes.c_void_p))
    return v, m


def var_kernel_c64_2d(z2d, axis: int = 1, ddof: int = 0):
    """Complex64 [rows, cols]: var(re) + var(im) per slice, and the complex mean."""
    zz = np.ascontiguousarray(np.asarray(z2d, dtype=np.complex64))
    rows, cols = zz.shape
    f = zz.view(np.float32)
    p = f.ctypes.data_as(ctypes.c_void_p)
    ns = rows if axis == 1 else cols
    v = np.empty(ns, dtype=np.float32)
    m = np.empty(ns, dtype=np.complex64)
    _L().orc_var_kernel_c64_2d(p, rows, cols, axis, ddof, v.ctypes.data_as(ctypes.c_void_p),
                               m.ctypes.data_as(ctypes.c_void_p))
    return v, m


def two_sum(a, b):
    """(s, e) of the variance tree's TwoSum, in the type of a (float32/float64)."""
    if isinstance(a, np.float32):
        s, e = ctypes.c_float(0), ctypes.c_float(0)
        _L().orc_two_sum_f32(float(a), float(b), ctypes.byref(s), ctypes.byref(e))
        return np.float32(s.value), np.float32(e.value)
    s, e = ctypes.c_double(0), ctypes.c_double(0)
    _L().orc_two_sum_f64(float(a), float(b), ctypes.byref(s), ctypes.byref(e))
    return np.float64(s.value), np.float64(e.value)
