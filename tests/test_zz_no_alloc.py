"""linrec_scan_f32_noalloc: the chunked scan with its look-back scratch in a
fixed array inside the library, for callers that must not allocate device
memory (graph capture, real-time loops, hosts that own every allocation).

Its results are checked against the ordinary entry point, linrec_scan_f32,
within the tolerance the other parity tests use, on two calls in a row (the
second call runs on the array as the first one left it), and every element
against the fp64 oracle.  This file is collected last so that a stop at the
first failure has run everything else.
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
SCRATCH_BYTES = 16 * 1024 * 1024


@pytest.fixture(scope="module")
def noalloc():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)
    fn = lr.lib().linrec_scan_f32_noalloc
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    fn.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape", [(32, 4096, 256), (1, 1 << 20, 64), (3, 1000, 260), (2, 77, 36)],
                         ids=lambda s: "x".join(map(str, s)))
def test_noalloc_matches_the_allocating_entry_point(noalloc, shape):
    B, L, D = shape
    a, b = inputs.generate(B, L, D, seed=31 + L, a_dist="u[0,1)", b_dist="n(0,1)")
    a_d, b_d = a.to(DEV), b.to(DEV)
    want = lr.linrec_scan_f32(a_d, b_d)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    h64, _ = oracle.f64(a, b)
    for call in range(2):
        h = torch.full_like(a_d, float("nan"))
        code = noalloc(a_d.data_ptr(), b_d.data_ptr(), h.data_ptr(), B, L, D, _stream(), status.data_ptr())
        assert code == lr.LINREC_OK, lr.linrec_status_string(code)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        got = h.cpu().numpy()
        assert_close(got, want.cpu().numpy().astype(np.float64), f"{shape} call {call}")
        assert_close(got, h64, f"{shape} call {call} against the oracle")


def test_noalloc_modes_alternating(noalloc):
    """Calls whose plans take slice-owner mode (many slices: only the control block is used) and
    look-back mode (few long slices: the look-back words) alternate on the one array; each output
    agrees with linrec_scan_f32 and with the oracle, and the array's own status word stays clear."""
    cases = []
    for (B, L, D, seed) in [(32, 4096, 256, 61), (1, 1 << 20, 64, 62), (3, 1000, 260, 63)]:
        a, b = inputs.generate(B, L, D, seed=seed, a_dist="u[0.9,1)", b_dist="n(0,1)")
        a_d, b_d = a.to(DEV), b.to(DEV)
        cases.append((B, L, D, a_d, b_d, lr.linrec_scan_f32(a_d, b_d), oracle.f64(a, b)[0]))
    for k in range(3):
        for (B, L, D, a_d, b_d, want, h64) in cases:
            h = torch.full_like(a_d, float("nan"))
            code = noalloc(a_d.data_ptr(), b_d.data_ptr(), h.data_ptr(), B, L, D, _stream(), None)
            assert code == lr.LINREC_OK, lr.linrec_status_string(code)
            torch.cuda.synchronize()
            assert_close(h.cpu().numpy(), want.cpu().numpy().astype(np.float64), f"{(B, L, D)} round {k}")
            assert_close(h.cpu().numpy(), h64, f"{(B, L, D)} round {k} against the oracle")
    # failures of calls made without a status word of their own would show here
    assert lr.linrec_stream_status() == lr.LINREC_OK


def test_noalloc_epoch_wraps_around(noalloc):
    """The array's epoch word set just below the point where it wraps: four look-back calls in a row
    each tag their words differently from the call before, so none takes the previous call's words
    for its own; every output agrees with linrec_scan_f32."""
    B, L, D = 1, 1 << 20, 64
    a, b = inputs.generate(B, L, D, seed=64, a_dist="u[0.9,1)", b_dist="n(0,1)")
    a_d, b_d = a.to(DEV), b.to(DEV)
    want = lr.linrec_scan_f32(a_d, b_d).cpu().numpy().astype(np.float64)
    h = torch.empty_like(a_d)
    assert noalloc(a_d.data_ptr(), b_d.data_ptr(), h.data_ptr(), B, L, D, _stream(), None) == lr.LINREC_OK
    lr.linrec_debug_set_epoch(0xFFFFFFFD, fixed_array=True)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for call in range(4):
        h.fill_(float("nan"))
        code = noalloc(a_d.data_ptr(), b_d.data_ptr(), h.data_ptr(), B, L, D, _stream(), status.data_ptr())
        assert code == lr.LINREC_OK, lr.linrec_status_string(code)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        assert_close(h.cpu().numpy(), want, f"call {call} across the epoch wrap")
    assert lr.linrec_stream_status() == lr.LINREC_OK


def test_noalloc_rejects_what_does_not_fit(noalloc):
    # (1, 2^24, 64): one slice in look-back mode, about 24*B*D*L/128 = 201 MB of look-back words:
    # refused, nothing launched
    B, L, D = 1, 1 << 24, 64
    # the entry point runs one launch on its fixed array: the look-back mode, never the two-pass mode
    plan = lr.linrec_plan_f32(B, L, D, path="chunked", chunk_mode="lookback",
                              sm_count=torch.cuda.get_device_properties(DEV).multi_processor_count)
    assert plan["lookback"] == 1
    assert plan["workspace_bytes"] > SCRATCH_BYTES
    base = 1 << 40                       # never dereferenced: the size check comes first
    n = B * L * D * 4
    code = noalloc(base, base + n, base + 2 * n, B, L, D, _stream(), None)
    assert code == lr.LINREC_ERR_WORKSPACE
    # misaligned or D % 4 != 0: refused
    x = torch.zeros(2 * 100 * 8 + 1, device=DEV)
    code = noalloc(x[1:].data_ptr(), x[1:].data_ptr(), x.data_ptr() + 4 * 1000, 1, 100, 8, _stream(), None)
    assert code in (lr.LINREC_ERR_INVALID_VALUE, lr.LINREC_ERR_ALIAS)
    code = noalloc(base, base + 4096, base + 8192, 1, 10, 6, _stream(), None)
    assert code == lr.LINREC_ERR_INVALID_VALUE
    assert noalloc(None, None, None, 0, 10, 8, _stream(), None) == lr.LINREC_OK
