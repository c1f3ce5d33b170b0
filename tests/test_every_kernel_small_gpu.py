"""Every kernel and mode on small ragged shapes, against the oracle.

One compact sweep that reaches every device code path of the library: the
fp32 forward scan in each chunk mode and on the register path (each vector
width), 16-bit storage, the (B, D, L) layout in one and two passes, the
gradient, carried state, the host-buffer pipeline, the no-allocation entry
and the copy kernel.  The shapes are small, so the file also serves as the
workload of the index-checked build (test_checked_build_gpu.py runs it with
liblinrec_checked.so), whose last test requires that no access was skipped.
"""
import ctypes

import numpy as np
import pytest
import torch

import linear_recurrence_scan_fp32_gb300 as lr
import oracle
from linear_recurrence_scan_fp32_gb300 import inputs
from tests._util import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SHAPES = [(1, 1, 8), (2, 33, 40), (3, 300, 136), (1, 2500, 64), (2, 129, 6)]
UNIT = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)


def _draw(B, L, D, seed):
    return inputs.generate(B, L, D, seed=seed, a_dist="u[0.5,1)", b_dist="n(0,1)")


def _sync_ok(what):
    torch.cuda.synchronize()
    st = lr.linrec_stream_status()
    assert st == lr.LINREC_OK, f"{what}: {lr.linrec_status_string(st)}"


def _forward_options(L, D):
    opts = [{}, {"path": "regcarry", "vec": 1, "prefetch": 4}]
    if D % 2 == 0:
        opts.append({"path": "regcarry", "vec": 2, "prefetch": 8})
    if D % 4 == 0:
        opts.append({"path": "regcarry", "vec": 4, "prefetch": 16})
        for mode in ("own", "lookback", "twopass", "blocks", "chain"):
            opts.append({"path": "chunked", "chunk_mode": mode})
        opts.append({"path": "chunked", "chunk_mode": "blocks", "tile_d": 64, "group": 2})
        if L % 2 == 0 and L >= 2048:       # two segments at least 1024 steps long
            opts.append({"path": "chunked", "chunk_mode": "speculative"})
    return opts


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_forward_and_carry(shape):
    B, L, D = shape
    a, b = _draw(B, L, D, 200 + L)
    h0 = torch.randn((B, D), generator=torch.Generator().manual_seed(201))
    h64, _ = oracle.f64(a, b)
    hc64, last64 = oracle.f64_carry(a, b, h0.numpy().astype(np.float64))
    a_d, b_d, h0_d = a.to(DEV), b.to(DEV), h0.to(DEV)
    for opt in _forward_options(L, D):
        h = lr.linrec_scan_f32_ex(a_d, b_d, **opt) if opt else lr.linrec_scan_f32(a_d, b_d)
        _sync_ok(f"{shape} {opt}")
        assert_close(h.cpu().numpy(), h64, f"{shape} {opt}")
        last = torch.full((B, D), float("nan"), device=DEV)
        h = lr.linrec_scan_f32_ex(a_d, b_d, h_init=h0_d, h_last=last, **opt)
        _sync_ok(f"{shape} {opt} carry")
        assert_close(h.cpu().numpy(), hc64, f"{shape} {opt} carry")
        assert_close(last.cpu().numpy(), last64, f"{shape} {opt} h_last")


@pytest.mark.parametrize("kind", ("bf16", "f16"))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_16bit_storage(kind, shape):
    B, L, D = shape
    a, b = _draw(B, L, D, 210 + L)
    a16, b16 = inputs.to_storage16(a, kind), inputs.to_storage16(b, kind)
    h64, _ = oracle.f64_16(kind, a16, b16)
    a_d, b_d = a16.to(DEV), b16.to(DEV)
    scan = {"bf16": lr.linrec_scan_bf16_ex, "f16": lr.linrec_scan_f16_ex}[kind]
    opts = [{}, {"path": "regcarry", "vec": 1, "prefetch": 4}]
    if D % 8 == 0:
        opts += [{"path": "chunked", "chunk_mode": m} for m in ("own", "lookback", "twopass", "blocks", "chain")]
        opts.append({"path": "chunked", "chunk_mode": "own", "vec": 1})
    u = UNIT[kind]
    for opt in opts:
        h = scan(a_d, b_d, **opt)
        _sync_ok(f"{kind} {shape} {opt}")
        x = oracle.decode16(kind, h.cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
        bound = u * np.abs(h64) + (1 + u) * 1e-4 * (1 + np.abs(h64))
        assert (np.abs(x - h64) <= bound).all(), f"{kind} {shape} {opt}"


@pytest.mark.parametrize("shape", [(1, 8, 1), (2, 40, 33), (3, 136, 300), (1, 64, 2500), (2, 6, 129)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bdl_layout(shape):
    B, D, L = shape
    a, b = _draw(B, L, D, 220 + L)
    at, bt = a.transpose(1, 2).contiguous(), b.transpose(1, 2).contiguous()
    h64, _ = oracle.f64_bdl(at, bt)
    a_d, b_d = at.to(DEV), bt.to(DEV)
    opts = [{}, {"chunk_mode": "twopass"}] if L >= 64 else [{}]
    for opt in opts:
        try:
            h = lr.linrec_scan_f32_bdl_ex(a_d, b_d, **opt)
        except lr.LinrecError:
            assert opt, "the default must always run"
            continue                                   # two passes refused for rows this short
        _sync_ok(f"bdl {shape} {opt}")
        assert_close(h.cpu().numpy(), h64, f"bdl {shape} {opt}")


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gradient(shape):
    B, L, D = shape
    a, b = _draw(B, L, D, 230 + L)
    g = torch.randn((B, L, D), generator=torch.Generator().manual_seed(231))
    h = lr.linrec_scan_f32(a.to(DEV), b.to(DEV))
    torch.cuda.synchronize()
    da64, db64, _ = oracle.f64_backward(a, h.cpu(), g)
    a_d, g_d = a.to(DEV), g.to(DEV)
    opts = [{}, {"path": "regcarry"}]
    if D % 4 == 0:
        opts += [{"path": "chunked", "chunk_mode": m} for m in ("own", "lookback", "twopass")]
    for opt in opts:
        da, db = lr.linrec_scan_f32_backward(a_d, h, g_d, **opt)
        _sync_ok(f"gradient {shape} {opt}")
        assert_close(db.cpu().numpy(), db64, f"db {shape} {opt}")
        assert_close(da.cpu().numpy(), da64, f"da {shape} {opt}")


def test_host_buffers_noalloc_and_copy():
    B, L, D = 2, 700, 68
    a, b = _draw(B, L, D, 240)
    h64, _ = oracle.f64(a, b)
    # host buffers: pinned (the kernel reads them in place) and pageable (the copy pipeline)
    for pin in (True, False):
        ah, bh = (a.pin_memory(), b.pin_memory()) if pin else (a.clone(), b.clone())
        hh = torch.empty_like(ah).pin_memory() if pin else torch.empty_like(ah)
        lr.linrec_scan_f32_host(ah, bh, hh)
        _sync_ok(f"host pinned={pin}")
        assert_close(hh.numpy(), h64, f"host pinned={pin}")
    # the entry point that allocates nothing
    fn = lr.lib().linrec_scan_f32_noalloc
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 2
    fn.restype = ctypes.c_int
    a_d, b_d = a.to(DEV), b.to(DEV)
    h = torch.empty_like(a_d)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    code = fn(a_d.data_ptr(), b_d.data_ptr(), h.data_ptr(), B, L, D,
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), status.data_ptr())
    assert code == lr.LINREC_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(h.cpu().numpy(), h64, "noalloc")
    # the copy kernel, with a ragged tail
    src = torch.arange(1001, dtype=torch.float32, device=DEV)
    dst = torch.zeros_like(src)
    lr.linrec_copy_f32(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)


def test_no_access_skipped():
    """Run after the sweep above: in the index-checked build no access fell outside its array (in the
    normal build the count is always 0)."""
    count, first = lr.linrec_debug_bad_accesses()
    assert count == 0, f"{count} accesses outside their arrays, the first at byte offset {first}"
