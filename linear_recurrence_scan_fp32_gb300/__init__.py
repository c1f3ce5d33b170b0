"""GB300-native first-order linear-recurrence scan: Python binding of liblinrec.

    h[i,0,d] = b[i,0,d];   h[i,t,d] = a[i,t,d] * h[i,t-1,d] + b[i,t,d]

for fp32 (B, L, D) tensors with D contiguous (POPCORNBENCH "Kimi-K2.6 l1_p9",
problem statement).  Every step runs in the CUDA kernels of ``liblinrec.so``
(built in-tree for sm_103a by ``_build.build()``); this module only checks
tensor properties and passes device pointers, sizes and the stream through the
C ABI declared in ``include/linrec.h``.  There is no CPU fallback: a missing
library raises ``LinrecError``.

Functions keep the C names:
    linrec_scan_f32(a, b, h=None, stream=None) -> h
    linrec_scan_f32_ex(a, b, h=None, stream=None, **options) -> h
    linrec_scan_f32_carry(a, b, h=None, h_init=None, h_last=None, stream=None) -> h
    linrec_scan_f32_backward(a, h, g, da=None, db=None, h_init=None, dh_last=None, dh_init=None) -> (da, db)
    linrec_scan_f32_host(a, b, h=None, stream=None) -> h   (host tensors; pipelined copies)
    linrec_scan_bf16(a, b, h=None, stream=None) -> h       (bfloat16 storage, fp32 arithmetic)
    linrec_scan_f16(a, b, h=None, stream=None) -> h        (binary16 storage, fp32 arithmetic)
    linrec_scan_bf16_ex / linrec_scan_f16_ex(a, b, h=None, stream=None, **options) -> h
    linrec_plan_f32(B, L, D, sm_count=152, align_bytes=16, resident_ctas=0, **options) -> dict
    linrec_plan_16(B, L, D, sm_count=152, align_bytes=16, resident_ctas=0, **options) -> dict
    linrec_scan_f32_bdl(a, b, h=None, stream=None) -> h    ((B, D, L) tensors: time innermost)
    linrec_scan_f32_bdl_ex / linrec_scan_bf16_bdl_ex / linrec_scan_f16_bdl_ex(a, b, h=None, stream=None, **options)
    linrec_plan_bdl(B, D, L, elem_bytes=4, sm_count=152, align_bytes=16, **options) -> dict
    linrec_stream_status(stream=None) -> int
    linrec_copy_f32(src, dst, stream=None)
    linrec_status_string(code) -> str
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# LINREC_LIBRARY names another build of the same library (the index-checked one, for instance)
LIB_PATH = os.environ.get("LINREC_LIBRARY") or os.path.join(_HERE, "liblinrec.so")

LINREC_OK = 0
LINREC_ERR_INVALID_VALUE = 1
LINREC_ERR_ALIAS = 2
LINREC_ERR_UNSUPPORTED_DEVICE = 3
LINREC_ERR_LAUNCH = 4
LINREC_ERR_WORKSPACE = 5
LINREC_ERR_LOOKBACK_TIMEOUT = 6
LINREC_ERR_TMA_TIMEOUT = 7

PATHS = {"auto": 0, "regcarry": 1, "chunked": 2, "rows": 3}
PATH_NAMES = {v: k for k, v in PATHS.items()}


class LinrecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


class Options(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int),
        ("vec", ctypes.c_int),
        ("prefetch", ctypes.c_int),
        ("tile_t", ctypes.c_int),
        ("tile_d", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("ctas_per_sm", ctypes.c_int),
        ("chunk_mode", ctypes.c_int),
        ("d_status", ctypes.c_void_p),
        ("h_init", ctypes.c_void_p),
        ("h_last", ctypes.c_void_p),
        ("spin_limit", ctypes.c_int64),
        ("test_silent_tile", ctypes.c_int64),
        ("rows_per_warp", ctypes.c_int),
        ("segments", ctypes.c_int),
        ("group", ctypes.c_int),
    ]


class Plan(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int),
        ("vec", ctypes.c_int),
        ("prefetch", ctypes.c_int),
        ("tile_t", ctypes.c_int),
        ("tile_d", ctypes.c_int),
        ("segments", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("lookback", ctypes.c_int),
        ("twopass", ctypes.c_int),
        ("threads", ctypes.c_int),
        ("grid", ctypes.c_int64),
        ("n_tiles", ctypes.c_int64),
        ("chunks", ctypes.c_int64),
        ("smem_bytes", ctypes.c_size_t),
        ("workspace_bytes", ctypes.c_size_t),
        ("blocks", ctypes.c_int),
        ("chain", ctypes.c_int),
        ("speculative", ctypes.c_int),
    ]


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded liblinrec.so (ctypes handle).  Raises LinrecError if it was not built."""
    global _lib
    if _lib is not None:                 # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise LinrecError(-1, f"liblinrec.so is missing at {LIB_PATH}: build it with "
                                  "__graft_entry__.build() (nvcc, sm_103a); there is no fallback")
        L = ctypes.CDLL(LIB_PATH)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        L.linrec_scan_f32.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        L.linrec_scan_f32.restype = i32
        L.linrec_scan_f32_ex.argtypes = [vp, vp, vp, i64, i64, i64, vp, ctypes.POINTER(Options)]
        L.linrec_scan_f32_ex.restype = i32
        L.linrec_plan_f32.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(Options), ctypes.POINTER(Plan)]
        L.linrec_plan_f32.restype = i32
        L.linrec_scan_f32_carry.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp]
        L.linrec_scan_f32_carry.restype = i32
        L.linrec_scan_f32_backward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp, vp, vp, vp]
        L.linrec_scan_f32_backward.restype = i32
        L.linrec_scan_f32_backward_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp, vp, vp, vp,
                                                  ctypes.POINTER(Options)]
        L.linrec_scan_f32_backward_ex.restype = i32
        L.linrec_plan_f32_backward.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(Options),
                                               ctypes.POINTER(Plan)]
        L.linrec_plan_f32_backward.restype = i32
        L.linrec_scan_f32_host.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        L.linrec_scan_f32_host.restype = i32
        for name in ("linrec_scan_bf16", "linrec_scan_f16"):
            getattr(L, name).argtypes = [vp, vp, vp, i64, i64, i64, vp]
            getattr(L, name).restype = i32
            getattr(L, name + "_ex").argtypes = [vp, vp, vp, i64, i64, i64, vp, ctypes.POINTER(Options)]
            getattr(L, name + "_ex").restype = i32
        L.linrec_plan_16.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(Options), ctypes.POINTER(Plan)]
        L.linrec_plan_16.restype = i32
        L.linrec_scan_f32_bdl.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        L.linrec_scan_f32_bdl.restype = i32
        for name in ("linrec_scan_f32_bdl_ex", "linrec_scan_bf16_bdl_ex", "linrec_scan_f16_bdl_ex"):
            getattr(L, name).argtypes = [vp, vp, vp, i64, i64, i64, vp, ctypes.POINTER(Options)]
            getattr(L, name).restype = i32
        L.linrec_plan_bdl.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(Options), ctypes.POINTER(Plan)]
        L.linrec_plan_bdl.restype = i32
        L.linrec_stream_status.argtypes = [vp]
        L.linrec_stream_status.restype = i32
        L.linrec_copy_f32.argtypes = [vp, vp, i64, vp]
        L.linrec_copy_f32.restype = i32
        L.linrec_status_string.argtypes = [i32]
        L.linrec_status_string.restype = ctypes.c_char_p
        L.linrec_version.argtypes = []
        L.linrec_version.restype = i32
        L.linrec_workspace_bytes.argtypes = [i64, i64, i64]
        L.linrec_workspace_bytes.restype = ctypes.c_size_t
        L.linrec_debug_checks.argtypes = []
        L.linrec_debug_checks.restype = i32
        L.linrec_debug_bad_accesses.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_int64), i64]
        L.linrec_debug_bad_accesses.restype = i32
        L.linrec_debug_range_covers.argtypes = [ctypes.c_size_t, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_size_t]
        L.linrec_debug_range_covers.restype = i32
        L.linrec_debug_set_epoch.argtypes = [vp, i32, ctypes.c_uint32]
        L.linrec_debug_set_epoch.restype = i32
        _lib = L
        return _lib


def linrec_status_string(code: int) -> str:
    return lib().linrec_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != LINREC_OK:
        raise LinrecError(code, f"{what}: {linrec_status_string(code)}")


CHUNK_MODES = {"auto": 0, "own": 1, "lookback": 2, "twopass": 3, "blocks": 4, "chain": 5, "speculative": 6}


def _addr(x):
    if x is None:
        return None
    return int(x.data_ptr() if hasattr(x, "data_ptr") else x)


_options_cache = {}


def make_options(path="auto", vec=0, prefetch=0, tile_t=0, tile_d=0, stages=0, ctas_per_sm=0,
                 chunk_mode="auto", d_status=None, h_init=None, h_last=None, spin_limit=0,
                 test_silent_tile=0, rows_per_warp=0, segments=0, group=0) -> Options:
    # The fields other than the three pointers are filled once per distinct combination and
    # copied from there (setting a ctypes field costs about 0.1 us; a repeated call with the
    # same options should not pay for 16 of them).
    key = (path, vec, prefetch, tile_t, tile_d, stages, ctas_per_sm, chunk_mode, spin_limit, test_silent_tile,
           rows_per_warp, segments, group)
    base = _options_cache.get(key)
    if base is None:
        base = Options()
        base.path = PATHS[path] if isinstance(path, str) else int(path)
        base.vec, base.prefetch, base.tile_t = int(vec), int(prefetch), int(tile_t)
        base.tile_d, base.stages = int(tile_d), int(stages)
        base.ctas_per_sm = int(ctas_per_sm)
        base.chunk_mode = CHUNK_MODES[chunk_mode] if isinstance(chunk_mode, str) else int(chunk_mode)
        base.spin_limit = int(spin_limit)
        base.test_silent_tile = int(test_silent_tile)
        base.rows_per_warp = int(rows_per_warp)
        base.segments = int(segments)
        base.group = int(group)
        if len(_options_cache) < 1024:
            _options_cache[key] = base
    o = Options.from_buffer_copy(base)
    if d_status is not None:
        o.d_status = _addr(d_status)
    if h_init is not None:
        o.h_init = _addr(h_init)
    if h_last is not None:
        o.h_last = _addr(h_last)
    return o


_torch = None
_raw_stream = None


def _torch_mod():
    global _torch, _raw_stream
    if _torch is None:
        import torch
        # the current stream's handle without building a Stream object (several us per call),
        # where this torch has the accessor; the public API otherwise
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _torch = torch
    return _torch


def _stream_handle(stream):
    """cudaStream_t of `stream`: a torch.cuda.Stream, a raw handle, or None for the current
    device's current stream."""
    if stream is None:
        torch = _torch_mod()
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _shape_of(a, b, h, dtype=None):
    """(B, L, D) of a, b (and h), after checking that they are contiguous 3-D CUDA tensors of
    `dtype` (float32 by default) of one shape.  One combined test on the per-call path; the
    detailed checks below only run to say what is wrong."""
    torch = _torch_mod()
    dtype = dtype or torch.float32
    try:
        ok = (a.dtype is dtype and b.dtype is dtype and a.is_cuda and b.is_cuda and a.dim() == 3 and
              a.is_contiguous() and b.is_contiguous() and a.shape == b.shape and
              (h is None or (h.dtype is dtype and h.is_cuda and h.is_contiguous() and h.shape == a.shape)))
    except AttributeError:
        ok = False
    if ok and isinstance(a, torch.Tensor) and isinstance(b, torch.Tensor) and (h is None or isinstance(h, torch.Tensor)):
        return tuple(a.shape)
    for name, t in (("a", a), ("b", b), ("h", h)):
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 3:
            raise ValueError(f"{name} must be 3-D (B, L, D)")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (B, L, D), D innermost")
    if a.shape != b.shape or (h is not None and h.shape != a.shape):
        raise ValueError("a, b and h must have the same shape")
    return tuple(a.shape)


def linrec_scan_f32_ex(a, b, h=None, stream=None, **options):
    """h = scan(a, b) with explicit options (path, vec, prefetch, tile_t, tile_d, stages, ...)."""
    import torch
    B, L, D = _shape_of(a, b, h)
    if h is None:
        h = torch.empty_like(a)
    opt = make_options(**options)
    code = lib().linrec_scan_f32_ex(a.data_ptr(), b.data_ptr(), h.data_ptr(), B, L, D,
                                    _stream_handle(stream), ctypes.byref(opt))
    _check(code, "linrec_scan_f32_ex")
    return h


def linrec_scan_f32(a, b, h=None, stream=None):
    """h = scan(a, b): fp32 CUDA tensors of shape (B, L, D), contiguous; h is allocated if None."""
    import torch
    B, L, D = _shape_of(a, b, h)
    if h is None:
        h = torch.empty_like(a)
    code = lib().linrec_scan_f32(a.data_ptr(), b.data_ptr(), h.data_ptr(), B, L, D, _stream_handle(stream))
    _check(code, "linrec_scan_f32")
    return h


def _scan16(fn, dtype, a, b, h, stream, options):
    import torch
    B, L, D = _shape_of(a, b, h, dtype)
    if h is None:
        h = torch.empty_like(a)
    if options is None:
        code = getattr(lib(), fn)(a.data_ptr(), b.data_ptr(), h.data_ptr(), B, L, D, _stream_handle(stream))
    else:
        _check_state(options.get("h_init"), "h_init", B, D)
        _check_state(options.get("h_last"), "h_last", B, D)
        opt = make_options(**options)
        code = getattr(lib(), fn)(a.data_ptr(), b.data_ptr(), h.data_ptr(), B, L, D, _stream_handle(stream),
                                  ctypes.byref(opt))
    _check(code, fn)
    return h


def linrec_scan_bf16(a, b, h=None, stream=None):
    """h = scan(a, b) on torch.bfloat16 CUDA tensors (B, L, D): fp32 arithmetic, h rounded once."""
    import torch
    return _scan16("linrec_scan_bf16", torch.bfloat16, a, b, h, stream, None)


def linrec_scan_f16(a, b, h=None, stream=None):
    """h = scan(a, b) on torch.float16 CUDA tensors (B, L, D): fp32 arithmetic, h rounded once."""
    import torch
    return _scan16("linrec_scan_f16", torch.float16, a, b, h, stream, None)


def linrec_scan_bf16_ex(a, b, h=None, stream=None, **options):
    """linrec_scan_bf16 with explicit options; h_init / h_last are float32 (B, D) tensors."""
    import torch
    return _scan16("linrec_scan_bf16_ex", torch.bfloat16, a, b, h, stream, options)


def linrec_scan_f16_ex(a, b, h=None, stream=None, **options):
    """linrec_scan_f16 with explicit options; h_init / h_last are float32 (B, D) tensors."""
    import torch
    return _scan16("linrec_scan_f16_ex", torch.float16, a, b, h, stream, options)


def _scan_bdl(fn, dtype, a, b, h, stream, options):
    import torch
    B, D, L = _shape_of(a, b, h, dtype)
    if h is None:
        h = torch.empty_like(a)
    if options is None:
        code = getattr(lib(), fn)(a.data_ptr(), b.data_ptr(), h.data_ptr(), B, D, L, _stream_handle(stream))
    else:
        _check_state(options.get("h_init"), "h_init", B, D)
        _check_state(options.get("h_last"), "h_last", B, D)
        opt = make_options(**options)
        code = getattr(lib(), fn)(a.data_ptr(), b.data_ptr(), h.data_ptr(), B, D, L, _stream_handle(stream),
                                  ctypes.byref(opt))
    _check(code, fn)
    return h


def linrec_scan_f32_bdl(a, b, h=None, stream=None):
    """h = scan(a, b) on float32 CUDA tensors laid out (B, D, L): time innermost, each channel a row."""
    import torch
    return _scan_bdl("linrec_scan_f32_bdl", torch.float32, a, b, h, stream, None)


def linrec_scan_f32_bdl_ex(a, b, h=None, stream=None, **options):
    """linrec_scan_f32_bdl with options (chunk_mode "own" = one pass, "twopass"; h_init / h_last (B, D))."""
    import torch
    return _scan_bdl("linrec_scan_f32_bdl_ex", torch.float32, a, b, h, stream, options)


def linrec_scan_bf16_bdl_ex(a, b, h=None, stream=None, **options):
    """The (B, D, L) scan on torch.bfloat16 tensors (fp32 arithmetic); h_init / h_last float32 (B, D)."""
    import torch
    return _scan_bdl("linrec_scan_bf16_bdl_ex", torch.bfloat16, a, b, h, stream, options)


def linrec_scan_f16_bdl_ex(a, b, h=None, stream=None, **options):
    """The (B, D, L) scan on torch.float16 tensors (fp32 arithmetic); h_init / h_last float32 (B, D)."""
    import torch
    return _scan_bdl("linrec_scan_f16_bdl_ex", torch.float16, a, b, h, stream, options)


def linrec_plan_bdl(B, D, L, elem_bytes=4, sm_count=152, align_bytes=16, **options) -> dict:
    """The (B, D, L) dispatcher's choice, without a GPU (elem_bytes 4: fp32, 2: 16-bit storage)."""
    opt = make_options(**options)
    plan = Plan()
    code = lib().linrec_plan_bdl(int(B), int(D), int(L), int(elem_bytes), int(sm_count), int(align_bytes),
                                 ctypes.byref(opt), ctypes.byref(plan))
    _check(code, "linrec_plan_bdl")
    out = {name: getattr(plan, name) for name, _ in Plan._fields_}
    out["path_name"] = PATH_NAMES.get(out["path"], "none")
    return out


def _check_state(x, name, B, D):
    import torch
    if x is None:
        return
    if not isinstance(x, torch.Tensor) or x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise TypeError(f"{name} must be a contiguous float32 CUDA tensor")
    if x.numel() != B * D:
        raise ValueError(f"{name} must hold B*D = {B * D} values (shape (B, D))")


def linrec_scan_f32_carry(a, b, h=None, h_init=None, h_last=None, stream=None):
    """The scan continued from h_init (B, D) (None: h_0 = b_0); the last state goes to h_last (B, D)
    if given.  Returns h."""
    import torch
    B, L, D = _shape_of(a, b, h)
    _check_state(h_init, "h_init", B, D)
    _check_state(h_last, "h_last", B, D)
    if h is None:
        h = torch.empty_like(a)
    code = lib().linrec_scan_f32_carry(a.data_ptr(), b.data_ptr(), h.data_ptr(), B, L, D, _addr(h_init),
                                       _addr(h_last), _stream_handle(stream))
    _check(code, "linrec_scan_f32_carry")
    return h


def linrec_scan_f32_backward(a, h, g, da=None, db=None, h_init=None, dh_last=None, dh_init=None, want_da=True,
                             stream=None, **options):
    """Gradient of the scan: returns (da, db).  With want_da=False, da is None and h is not read
    (h may then be None).  dh_init (B, D), if given, receives the gradient of the starting state."""
    import torch
    B, L, D = _shape_of(a, g, None)
    if want_da or da is not None:
        if h is None:
            raise ValueError("h (the forward output) is needed for da")
        _shape_of(a, h, None)
        if da is None:
            da = torch.empty_like(a)
        _shape_of(a, da, None)
    if db is None:
        db = torch.empty_like(a)
    _shape_of(a, db, None)
    for name, x in (("h_init", h_init), ("dh_last", dh_last), ("dh_init", dh_init)):
        _check_state(x, name, B, D)
    args = (a.data_ptr(), _addr(h) if da is not None else None, g.data_ptr(), _addr(da), db.data_ptr(), B, L, D,
            _addr(h_init), _addr(dh_last), _addr(dh_init), _stream_handle(stream))
    if options:
        opt = make_options(**options)
        code = lib().linrec_scan_f32_backward_ex(*args, ctypes.byref(opt))
    else:
        code = lib().linrec_scan_f32_backward(*args)
    _check(code, "linrec_scan_f32_backward")
    return da, db


def linrec_plan_f32_backward(B, L, D, sm_count=152, align_bytes=16, resident_ctas=0, **options) -> dict:
    """The dispatcher's choice for the gradient of a (B, L, D) scan, without a GPU."""
    opt = make_options(**options)
    plan = Plan()
    code = lib().linrec_plan_f32_backward(int(B), int(L), int(D), int(sm_count), int(align_bytes),
                                          int(resident_ctas), ctypes.byref(opt), ctypes.byref(plan))
    _check(code, "linrec_plan_f32_backward")
    out = {name: getattr(plan, name) for name, _ in Plan._fields_}
    out["path_name"] = PATH_NAMES.get(out["path"], "none")
    return out


def linrec_scan_f32_host(a, b, h=None, stream=None):
    """The scan on CPU tensors (pinned memory for full speed): the library pipelines the copies to the
    device, the kernels and the copies back.  Returns h (a CPU tensor, pinned if a is); it is complete
    once `stream` (default: the current CUDA stream) is synchronised."""
    import torch
    for name, t in (("a", a), ("b", b)) + ((("h", h),) if h is not None else ()):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.is_cuda or t.dim() != 3 \
                or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous float32 CPU tensor of shape (B, L, D)")
    if a.shape != b.shape or (h is not None and h.shape != a.shape):
        raise ValueError("a, b and h must have the same shape")
    if h is None:
        h = torch.empty(a.shape, dtype=torch.float32, pin_memory=a.is_pinned())
    B, L, D = a.shape
    code = lib().linrec_scan_f32_host(a.data_ptr(), b.data_ptr(), h.data_ptr(), B, L, D, _stream_handle(stream))
    _check(code, "linrec_scan_f32_host")
    return h


def linrec_plan_f32(B, L, D, sm_count=152, align_bytes=16, resident_ctas=0, **options) -> dict:
    """The dispatcher's choice for a (B, L, D) problem, without a GPU.

    resident_ctas: CTAs of the chunked kernel that fit on one SM (0 = estimate);
    options as for linrec_scan_f32_ex."""
    opt = make_options(**options)
    plan = Plan()
    code = lib().linrec_plan_f32(int(B), int(L), int(D), int(sm_count), int(align_bytes), int(resident_ctas),
                                 ctypes.byref(opt), ctypes.byref(plan))
    _check(code, "linrec_plan_f32")
    out = {name: getattr(plan, name) for name, _ in Plan._fields_}
    out["path_name"] = PATH_NAMES.get(out["path"], "none")
    return out


def linrec_plan_16(B, L, D, sm_count=152, align_bytes=16, resident_ctas=0, **options) -> dict:
    """The dispatcher's choice for 16-bit storage (bfloat16 and binary16 alike), without a GPU."""
    opt = make_options(**options)
    plan = Plan()
    code = lib().linrec_plan_16(int(B), int(L), int(D), int(sm_count), int(align_bytes), int(resident_ctas),
                                ctypes.byref(opt), ctypes.byref(plan))
    _check(code, "linrec_plan_16")
    out = {name: getattr(plan, name) for name, _ in Plan._fields_}
    out["path_name"] = PATH_NAMES.get(out["path"], "none")
    return out


def linrec_stream_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device-side status of the library's work on it."""
    return int(lib().linrec_stream_status(_stream_handle(stream)))


def linrec_copy_f32(src, dst, stream=None):
    """dst = src with the library's 16-byte copy kernel (copy-bandwidth ceiling)."""
    if src.numel() != dst.numel():
        raise ValueError("src and dst differ in size")
    code = lib().linrec_copy_f32(src.data_ptr(), dst.data_ptr(), src.numel(), _stream_handle(stream))
    _check(code, "linrec_copy_f32")
    return dst


def linrec_version() -> int:
    return int(lib().linrec_version())


def linrec_debug_checks() -> bool:
    """Whether the loaded library is the index-checked build."""
    return bool(lib().linrec_debug_checks())


def linrec_debug_bad_accesses(output_cap_bytes: int = 0):
    """(accesses skipped by the index checks since the last call, byte offset of the first or -1);
    sets the output cap for the calls that follow (0: none).  Synchronises the device."""
    count, first = ctypes.c_uint64(0), ctypes.c_int64(-1)
    _check(lib().linrec_debug_bad_accesses(ctypes.byref(count), ctypes.byref(first), int(output_cap_bytes)),
           "linrec_debug_bad_accesses")
    return int(count.value), int(first.value)


def linrec_debug_range_covers(range_start: int, range_size: int, p: int, nbytes: int) -> bool:
    """Whether [p, p + nbytes) lies inside [range_start, range_start + range_size) (the test the
    host entry point makes before it reads a page-locked buffer in place)."""
    return bool(lib().linrec_debug_range_covers(int(range_start), int(range_size), int(p), int(nbytes)))


def linrec_debug_set_epoch(epoch: int, stream=None, fixed_array: bool = False):
    """Tests only: write the epoch word of the stream's look-back workspace (or of the fixed array of
    linrec_scan_f32_noalloc) on the current device."""
    _check(lib().linrec_debug_set_epoch(_stream_handle(stream), 1 if fixed_array else 0, int(epoch) & 0xffffffff),
           "linrec_debug_set_epoch")


def linrec_workspace_bytes(B, L, D) -> int:
    """Device memory a default linrec_scan_f32 call on (B, L, D) holds on the current device (0 if none)."""
    return int(lib().linrec_workspace_bytes(int(B), int(L), int(D)))
