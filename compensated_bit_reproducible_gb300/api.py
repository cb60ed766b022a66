"""ctypes binding of librepro_gb300.so (declared in include/repro.h).

Argument marshalling only: every function passes tensor data pointers, sizes
and the current CUDA stream to the C ABI, which does all the work on the GPU.
There is no CPU fallback: if the library is missing, loading raises.
PyTorch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librepro_gb300.so")
_lib = None

STATUS = {0: "ok", 1: "invalid argument", 2: "capacity", 3: "overlap", 4: "environment", 5: "cuda",
          6: "device timeout"}


class ReproError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = "%s: %s" % (where, lib().repro_strerror(status).decode())
        if status == 5:
            msg += " (cudaError %d)" % lib().repro_last_cuda_error()
        super().__init__(msg)


class Launch(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int), ("grid", ctypes.c_int)]


def lib():
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("librepro_gb300.so is missing: run __graft_entry__.build() "
                               "(or compensated_bit_reproducible_gb300/build.py) first")
        L = ctypes.CDLL(LIB_PATH)
        P, S, I, I64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64
        sig = {
            "repro_strerror": (ctypes.c_char_p, [I]),
            "repro_last_cuda_error": (I, []),
            "repro_max_count_f32": (ctypes.c_uint64, []),
            "repro_max_count_f64": (ctypes.c_uint64, []),
            "repro_max_k_f32": (I, []),
            "repro_max_k_f64": (I, []),
            "repro_validate_environment": (I, [P]),
            "repro_sum_f32": (I, [P, S, I, P, P]),
            "repro_sum_f64": (I, [P, S, I, P, P]),
            "repro_sum_f32_async": (I, [P, S, I, P, P, P]),
            "repro_sum_f64_async": (I, [P, S, I, P, P, P]),
            "repro_sum_f32_noalloc": (I, [P, S, I, P, P]),
            "repro_cumsum_f32": (I, [P, P, S, I, P]),
            "repro_cumsum_f64": (I, [P, P, S, I, P]),
            "repro_cumsum_f32_ex": (I, [P, P, S, I, P, P]),
            "repro_cumsum_f64_ex": (I, [P, P, S, I, P, P]),
            "repro_segsum_f32": (I, [P, I64, I64, I, I, P, P]),
            "stable_var_f32": (I, [P, I64, I64, I, I, P, P, P]),
            "twoterm_var_f32": (I, [P, I64, I64, I, I, P, P]),
            "stable_var_f64": (I, [P, I64, I64, I, I, P, P, P]),
            "stable_var_c64": (I, [P, I64, I64, I, I, P, P, P]),
            "stable_var_f32_variant": (I, [P, I64, I64, I, I, I, P, P, P]),
            "repro_compensated_chunk": (I, []),
            "repro_state_bytes": (S, [I]),
        }
        for t in ("f32", "f64"):
            sig["repro_state_init_" + t] = (I, [P, I, P])
            sig["repro_state_deposit_" + t] = (I, [P, P, S, I, P])
            sig["repro_state_merge_" + t] = (I, [P, P, I, P])
            sig["repro_state_finalize_" + t] = (I, [P, I, P, P])
            sig["repro_cumsum_from_state_" + t] = (I, [P, P, S, I, P, P])
        for mode in ("naive", "pairwise", "kahan", "neumaier"):
            for t in ("f32", "f64"):
                sig["repro_sum_%s_%s" % (mode, t)] = (I, [P, S, P, P])
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)


def _check(rc: int, where: str):
    if rc != 0:
        raise ReproError(rc, where)


def _sfx(t: torch.Tensor) -> str:
    if t.dtype == torch.float32:
        return "f32"
    if t.dtype == torch.float64:
        return "f64"
    raise TypeError("float32 or float64 tensor expected, got %s" % t.dtype)


def _launch(block: int = 0, grid: int = 0):
    if not block and not grid:
        return None
    return ctypes.byref(Launch(block, grid))


# ---------------------------------------------------------------- constants
def max_count(dtype) -> int:
    return int(lib().repro_max_count_f32() if dtype == torch.float32 else lib().repro_max_count_f64())


def max_k(dtype) -> int:
    return int(lib().repro_max_k_f32() if dtype == torch.float32 else lib().repro_max_k_f64())


def validate_environment(stream=None) -> None:
    _check(lib().repro_validate_environment(_stream(stream)), "repro_validate_environment")


# ---------------------------------------------------------------- binned sums
def repro_sum(x: torch.Tensor, K: int = 3, stream=None) -> float:
    """Synchronous binned sum of a contiguous 1-D tensor (device or host)."""
    sfx = _sfx(x)
    assert x.is_contiguous()
    out = (ctypes.c_float if sfx == "f32" else ctypes.c_double)()
    st = _stream(stream) if x.is_cuda or stream is not None else _stream()
    _check(getattr(lib(), "repro_sum_" + sfx)(_ptr(x), x.numel(), K, st, ctypes.byref(out)), "repro_sum_" + sfx)
    return out.value


def repro_sum_async(x: torch.Tensor, out: torch.Tensor, K: int = 3, block: int = 0, grid: int = 0,
                    stream=None) -> torch.Tensor:
    """Stream-ordered binned sum into the 1-element device tensor `out`."""
    sfx = _sfx(x)
    assert x.is_cuda and out.is_cuda and out.dtype == x.dtype and x.is_contiguous()
    _check(getattr(lib(), "repro_sum_%s_async" % sfx)(_ptr(x), x.numel(), K, _stream(stream), _ptr(out),
                                                      _launch(block, grid)), "repro_sum_%s_async" % sfx)
    return out


def repro_sum_noalloc(x: torch.Tensor, out: torch.Tensor, K: int = 3, stream=None) -> torch.Tensor:
    """Binned float sum whose workspace is a fixed device array inside the
    library: for callers that cannot allocate device memory (see
    include/repro.h).  Calls on one device must not overlap on the GPU."""
    assert x.is_cuda and out.is_cuda and x.dtype == torch.float32 and out.dtype == torch.float32
    assert x.is_contiguous()
    _check(lib().repro_sum_f32_noalloc(_ptr(x), x.numel(), K, _stream(stream), _ptr(out)), "repro_sum_f32_noalloc")
    return out


def repro_cumsum(x: torch.Tensor, out: torch.Tensor | None = None, K: int = 3, block: int = 0,
                 stream=None) -> torch.Tensor:
    """Binned cumulative sum; out may be x itself (in place).  x and out may
    be CUDA tensors or CPU tensors (plain host memory is copied by the
    library and the call then waits for the result)."""
    sfx = _sfx(x)
    assert x.is_contiguous()
    if out is None:
        out = torch.empty_like(x)
    assert out.dtype == x.dtype and out.is_contiguous() and out.numel() == x.numel()
    _check(getattr(lib(), "repro_cumsum_%s_ex" % sfx)(_ptr(x), _ptr(out), x.numel(), K, _stream(stream),
                                                      _launch(block, 0)), "repro_cumsum_" + sfx)
    return out


def repro_segsum(x: torch.Tensor, axis: int = 1, K: int = 3, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    assert x.is_cuda and x.dtype == torch.float32 and x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    if out is None:
        out = torch.empty(rows if axis == 1 else cols, dtype=torch.float32, device=x.device)
    _check(lib().repro_segsum_f32(_ptr(x), rows, cols, axis, K, _ptr(out), _stream(stream)), "repro_segsum_f32")
    return out


# ------------------------------------------------------------------ variance
def stable_var(x: torch.Tensor, axis: int = 1, ddof: int = 0, out=None, mean_out=None, with_mean: bool = True,
               stream=None, variant: int = 0):
    """Variance kernel: (var, mean) per slice along `axis` of a 2-D float32,
    float64 or complex64 tensor.  `variant` (float32 only) selects one of the
    section 4 step changes (0 = the kernel)."""
    assert x.is_cuda and x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    ns = rows if axis == 1 else cols
    vdt = {torch.float32: torch.float32, torch.float64: torch.float64, torch.complex64: torch.float32}[x.dtype]
    if out is None:
        out = torch.empty(ns, dtype=vdt, device=x.device)
    if with_mean and mean_out is None:
        mean_out = torch.empty(ns, dtype=x.dtype, device=x.device)
    mp = _ptr(mean_out) if with_mean else ctypes.c_void_p(0)
    st = _stream(stream)
    if x.dtype == torch.float32:
        if variant:
            rc = lib().stable_var_f32_variant(_ptr(x), rows, cols, axis, ddof, variant, _ptr(out), mp, st)
            _check(rc, "stable_var_f32_variant")
        else:
            _check(lib().stable_var_f32(_ptr(x), rows, cols, axis, ddof, _ptr(out), mp, st), "stable_var_f32")
    elif x.dtype == torch.float64:
        assert variant == 0
        _check(lib().stable_var_f64(_ptr(x), rows, cols, axis, ddof, _ptr(out), mp, st), "stable_var_f64")
    else:
        assert variant == 0
        _check(lib().stable_var_c64(_ptr(x), rows, cols, axis, ddof, _ptr(out), mp, st), "stable_var_c64")
    return out, mean_out


def twoterm_var(x: torch.Tensor, axis: int = 1, ddof: int = 0, out=None, stream=None) -> torch.Tensor:
    assert x.is_cuda and x.dtype == torch.float32 and x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    if out is None:
        out = torch.empty(rows if axis == 1 else cols, dtype=torch.float32, device=x.device)
    _check(lib().twoterm_var_f32(_ptr(x), rows, cols, axis, ddof, _ptr(out), _stream(stream)), "twoterm_var_f32")
    return out


# ---------------------------------------------------------- comparison sums
def compare_sum(x: torch.Tensor, mode: str, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """mode in naive / pairwise / kahan / neumaier; result in a 1-element device tensor."""
    sfx = _sfx(x)
    assert x.is_cuda and x.is_contiguous()
    if out is None:
        out = torch.empty(1, dtype=x.dtype, device=x.device)
    name = "repro_sum_%s_%s" % (mode, sfx)
    _check(getattr(lib(), name)(_ptr(x), x.numel(), _ptr(out), _stream(stream)), name)
    return out


def compensated_chunk() -> int:
    return int(lib().repro_compensated_chunk())


# ------------------------------------------------------------ binned states
def _tsfx(dtype) -> str:
    if dtype == torch.float32:
        return "f32"
    if dtype == torch.float64:
        return "f64"
    raise TypeError("float32 or float64 expected, got %s" % dtype)


def state_bytes(K: int = 3) -> int:
    return int(lib().repro_state_bytes(K))


def state_new(dtype, K: int = 3, device=None, stream=None) -> torch.Tensor:
    """A fresh (empty) binned state for `dtype` sums: a uint8 device tensor."""
    n = state_bytes(K)
    if n == 0:
        raise ReproError(1, "repro_state_bytes")
    st = torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda", torch.cuda.current_device()))
    state_init(st, dtype, K, stream)
    return st


def state_init(state: torch.Tensor, dtype, K: int = 3, stream=None) -> None:
    sfx = _tsfx(dtype)
    _check(getattr(lib(), "repro_state_init_" + sfx)(_ptr(state), K, _stream(stream)), "repro_state_init_" + sfx)


def state_deposit(state: torch.Tensor, x: torch.Tensor, K: int = 3, stream=None) -> None:
    sfx = _sfx(x)
    assert x.is_contiguous()
    _check(getattr(lib(), "repro_state_deposit_" + sfx)(_ptr(state), _ptr(x), x.numel(), K, _stream(stream)),
           "repro_state_deposit_" + sfx)


def state_merge(dst: torch.Tensor, src: torch.Tensor, dtype, K: int = 3, stream=None) -> None:
    sfx = _tsfx(dtype)
    _check(getattr(lib(), "repro_state_merge_" + sfx)(_ptr(dst), _ptr(src), K, _stream(stream)),
           "repro_state_merge_" + sfx)


def state_finalize(state: torch.Tensor, dtype, K: int = 3, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """Correctly rounded value of the state, as a one-element device tensor."""
    sfx = _tsfx(dtype)
    if out is None:
        out = torch.empty(1, dtype=dtype, device=state.device)
    _check(getattr(lib(), "repro_state_finalize_" + sfx)(_ptr(state), K, _ptr(out), _stream(stream)),
           "repro_state_finalize_" + sfx)
    return out


def repro_cumsum_from_state(x: torch.Tensor, state: torch.Tensor, K: int = 3, out: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """Binned cumulative sum of x that starts from a binned state: out[i]
    is the binned sum of the state's contents and x[0..i].  Device tensors
    only; out may be x itself."""
    sfx = _sfx(x)
    assert x.is_contiguous() and state.dtype == torch.uint8
    if out is None:
        out = torch.empty_like(x)
    assert out.dtype == x.dtype and out.is_contiguous() and out.numel() == x.numel()
    _check(getattr(lib(), "repro_cumsum_from_state_" + sfx)(_ptr(x), _ptr(out), x.numel(), K, _ptr(state),
                                                            _stream(stream)), "repro_cumsum_from_state_" + sfx)
    return out
