"""CPU oracle for the first-order linear-recurrence scan (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference leg may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it.

The arithmetic lives in ``linrec_oracle.c`` (plain sequential loops, see its
header for the definition followed and the passages cited).  This module only
compiles that file with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "linrec_oracle.c")
_LIB = os.path.join(_HERE, "liblinrec_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def build(force: bool = False) -> str:
    """Compile linrec_oracle.c into liblinrec_oracle.so (skipped when up to date)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def build_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used by the planted-mistake tests)."""
    src_path = out_path + ".c"
    with open(src_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *CFLAGS, src_path, "-o", out_path, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _bind(lib):
    i64, i32 = ctypes.c_int64, ctypes.c_int
    pf, pd = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    lib.linrec_oracle_f64.argtypes = [pf, pf, pd, i64, i64, i64, i32]
    lib.linrec_oracle_f64.restype = i32
    lib.linrec_oracle_f32seq.argtypes = [pf, pf, pf, i64, i64, i64, i32]
    lib.linrec_oracle_f32seq.restype = i32
    lib.linrec_oracle_f64_channel.argtypes = [pf, pf, pd, i64, i64, i64, i64, i64]
    lib.linrec_oracle_f64_channel.restype = i32
    lib.linrec_oracle_f64_carry.argtypes = [pf, pf, pd, pd, pd, i64, i64, i64]
    lib.linrec_oracle_f64_carry.restype = i32
    lib.linrec_oracle_f64_backward.argtypes = [pf, pf, pf, pd, pd, pd, pd, pd, i64, i64, i64]
    lib.linrec_oracle_f64_backward.restype = i32
    lib.linrec_oracle_f64_bdl.argtypes = [pf, pf, pd, pd, pd, i64, i64, i64]
    lib.linrec_oracle_f64_bdl.restype = i32
    pu16 = ctypes.POINTER(ctypes.c_uint16)
    lib.linrec_oracle_decode16.argtypes = [i32, pu16, pd, i64]
    lib.linrec_oracle_decode16.restype = i32
    lib.linrec_oracle_encode16.argtypes = [i32, pd, pu16, i64]
    lib.linrec_oracle_encode16.restype = i32
    lib.linrec_oracle_hardware_threads.argtypes = []
    lib.linrec_oracle_hardware_threads.restype = i32
    return lib


def load(path: str | None = None):
    """Load the oracle library (building it first if needed)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _as_f32(x) -> np.ndarray:
    if hasattr(x, "detach"):          # a CPU torch tensor
        x = x.detach().cpu().numpy()
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 3:
        raise ValueError("expected a (B, L, D) array")
    return x


def _ptr(x, ctype):
    return x.ctypes.data_as(ctypes.POINTER(ctype))


def _out(out, shape, dtype):
    """A caller's output array (reused across timed repetitions), or a new one."""
    if out is None:
        return np.empty(shape, dtype=dtype)
    if out.shape != shape or out.dtype != dtype or not out.flags.c_contiguous:
        raise ValueError(f"out must be a contiguous {np.dtype(dtype).name} array of shape {shape}")
    return out


def f64(a, b, nthreads: int = 0, lib=None, out=None):
    """h in float64 by the definition; returns (h, threads_used).  out: an array to write h into."""
    a, b = _as_f32(a), _as_f32(b)
    if a.shape != b.shape:
        raise ValueError("a and b differ in shape")
    lib = lib or load()
    h = _out(out, a.shape, np.float64)
    n = lib.linrec_oracle_f64(_ptr(a, ctypes.c_float), _ptr(b, ctypes.c_float),
                              _ptr(h, ctypes.c_double), *a.shape, nthreads)
    if n < 0:
        raise ValueError("oracle rejected its arguments")
    return h, n


def f32seq(a, b, nthreads: int = 0, lib=None, out=None):
    """h in fp32 with one rounded multiply and one rounded add per step; returns (h, threads_used)."""
    a, b = _as_f32(a), _as_f32(b)
    lib = lib or load()
    h = _out(out, a.shape, np.float32)
    n = lib.linrec_oracle_f32seq(_ptr(a, ctypes.c_float), _ptr(b, ctypes.c_float),
                                 _ptr(h, ctypes.c_float), *a.shape, nthreads)
    if n < 0:
        raise ValueError("oracle rejected its arguments")
    return h, n


def f64_channel(a, b, i: int, d: int, lib=None) -> np.ndarray:
    """One channel (i, d): h[i, :, d] in float64."""
    a, b = _as_f32(a), _as_f32(b)
    lib = lib or load()
    h = np.empty(a.shape[1], dtype=np.float64)
    rc = lib.linrec_oracle_f64_channel(_ptr(a, ctypes.c_float), _ptr(b, ctypes.c_float),
                                       _ptr(h, ctypes.c_double), *a.shape, i, d)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return h


def f64_carry(a, b, h0=None, lib=None):
    """The recurrence continued from h0 (a (B, D) array, or None for the plain
    definition); returns (h in float64, last state (B, D) in float64)."""
    a, b = _as_f32(a), _as_f32(b)
    lib = lib or load()
    B, L, D = a.shape
    h = np.empty(a.shape, dtype=np.float64)
    hlast = np.empty((B, D), dtype=np.float64)
    h0p = None
    if h0 is not None:
        h0 = np.ascontiguousarray(h0, dtype=np.float64).reshape(B, D)
        h0p = _ptr(h0, ctypes.c_double)
    rc = lib.linrec_oracle_f64_carry(_ptr(a, ctypes.c_float), _ptr(b, ctypes.c_float), h0p,
                                     _ptr(h, ctypes.c_double), _ptr(hlast, ctypes.c_double), B, L, D)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return h, hlast


def f64_backward(a, h, g, h0=None, dhlast=None, want_da=True, lib=None):
    """Gradient of the carried recurrence: returns (da or None, db, dh0), float64."""
    a, h, g = _as_f32(a), _as_f32(h), _as_f32(g)
    lib = lib or load()
    B, L, D = a.shape
    db = np.empty(a.shape, dtype=np.float64)
    da = np.empty(a.shape, dtype=np.float64) if want_da else None
    dh0 = np.empty((B, D), dtype=np.float64)

    def state(x):
        if x is None:
            return None, None
        x = np.ascontiguousarray(x, dtype=np.float64).reshape(B, D)
        return x, _ptr(x, ctypes.c_double)

    h0, h0p = state(h0)
    dhlast, dhp = state(dhlast)
    rc = lib.linrec_oracle_f64_backward(_ptr(a, ctypes.c_float), _ptr(h, ctypes.c_float), _ptr(g, ctypes.c_float),
                                        h0p, dhp, _ptr(da, ctypes.c_double) if want_da else None,
                                        _ptr(db, ctypes.c_double), _ptr(dh0, ctypes.c_double), B, L, D)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return da, db, dh0


def f64_bdl(a, b, h0=None, lib=None):
    """The definition for (B, D, L) tensors (time innermost), continued from h0
    ((B, D) or None); returns (h in float64, last state (B, D) in float64)."""
    a, b = _as_f32(a), _as_f32(b)
    if a.shape != b.shape:
        raise ValueError("a and b differ in shape")
    lib = lib or load()
    B, D, L = a.shape
    h = np.empty(a.shape, dtype=np.float64)
    hlast = np.empty((B, D), dtype=np.float64)
    h0p = None
    if h0 is not None:
        h0 = np.ascontiguousarray(h0, dtype=np.float64).reshape(B, D)
        h0p = _ptr(h0, ctypes.c_double)
    rc = lib.linrec_oracle_f64_bdl(_ptr(a, ctypes.c_float), _ptr(b, ctypes.c_float), h0p,
                                   _ptr(h, ctypes.c_double), _ptr(hlast, ctypes.c_double), B, D, L)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return h, hlast


KINDS16 = {"bf16": 0, "f16": 1}


def _bits16(w) -> np.ndarray:
    if hasattr(w, "detach"):          # a CPU torch tensor of 16-bit words (any 16-bit dtype)
        import torch
        w = w.detach().cpu().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(w).view(np.uint16)


def decode16(kind: str, w, lib=None) -> np.ndarray:
    """The exact value of every 16-bit word of format `kind` ("bf16" or "f16"), as float64."""
    w = _bits16(w)
    lib = lib or load()
    x = np.empty(w.shape, dtype=np.float64)
    if lib.linrec_oracle_decode16(KINDS16[kind], _ptr(w, ctypes.c_uint16), _ptr(x, ctypes.c_double), w.size):
        raise ValueError("oracle rejected its arguments")
    return x


def encode16(kind: str, x, lib=None) -> np.ndarray:
    """x (float64) rounded to the nearest word of format `kind`, ties to even; uint16 words."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    lib = lib or load()
    w = np.empty(x.shape, dtype=np.uint16)
    if lib.linrec_oracle_encode16(KINDS16[kind], _ptr(x, ctypes.c_double), _ptr(w, ctypes.c_uint16), x.size):
        raise ValueError("oracle rejected its arguments")
    return w


def f64_16(kind: str, a, b, h0=None, nthreads: int = 0, lib=None):
    """The scan of 16-bit inputs: each word decoded to its exact value, then the
    definition (continued from h0 if given) in float64.  Returns (h, last state).
    Without h0 the channel-threaded definition runs (same values as the carried
    loop with no state)."""
    lib = lib or load()
    xa, xb = decode16(kind, a, lib), decode16(kind, b, lib)
    # every bfloat16 and binary16 value is a float32 value: the narrowing is exact
    fa, fb = xa.astype(np.float32), xb.astype(np.float32)
    if not (np.array_equal(fa, xa, equal_nan=True) and np.array_equal(fb, xb, equal_nan=True)):
        raise AssertionError("a decoded 16-bit value is not a float32 value")
    if h0 is None:
        h, _ = f64(fa.reshape(fa.shape), fb, nthreads=nthreads, lib=lib)
        return h, np.ascontiguousarray(h[:, -1, :])
    return f64_carry(fa, fb, h0, lib=lib)


def hardware_threads() -> int:
    return int(load().linrec_oracle_hardware_threads())
