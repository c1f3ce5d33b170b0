"""Problems past 2^31 elements per tensor: every offset beyond 32 bits.

(B, L, D) = (2, 2^20 + 5, 1024) holds 2,147,493,888 elements per tensor
(8.6 GB in fp32), a ragged last time chunk, and two batch indices whose second
starts past element 2^30.  The inputs are drawn on the device from a seeded
generator (the oracle could not hold them all); sampled channels, each a full
sequence of 2^20 + 5 steps, are copied back and checked against the fp64
oracle element by element within |h - h64| <= 1e-4 (1 + |h64|).
"""
import numpy as np
import pytest
import torch

import linear_recurrence_scan_fp32_gb300 as lr
import oracle
from tests._util import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
B, L, D = 2, (1 << 20) + 5, 1024
# (batch, channel): first and last channel, both ends of a 32-channel slice, the far end of the
# last batch index (its offsets are the largest)
SAMPLES = [(0, 0), (0, 1023), (1, 31), (1, 32), (1, 517), (1, 1023)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)


def _draw(seed, shape=(B, L, D)):
    g = torch.Generator(device=DEV).manual_seed(seed)
    a = 0.9 + 0.1 * torch.rand(shape, generator=g, device=DEV)
    b = torch.randn(shape, generator=g, device=DEV)
    return a, b


def _channel(x, i, d, bdl=False):
    """One channel's sequence, as a (1, L, 1) float32 array for the oracle."""
    col = x[i, d, :] if bdl else x[:, :, d][i]
    return col.float().contiguous().cpu().numpy().reshape(1, -1, 1)


def _check(h, a, b, what, bdl=False):
    torch.cuda.synchronize()
    for (i, d) in SAMPLES:
        h64, _ = oracle.f64(_channel(a, i, d, bdl), _channel(b, i, d, bdl))
        assert_close(_channel(h, i, d, bdl), h64, f"{what} channel ({i}, {d})")


def test_forward_every_path_past_2_31():
    assert B * L * D > 2 ** 31
    a, b = _draw(71)
    h = torch.empty_like(a)
    for opt in ({}, {"path": "chunked", "chunk_mode": "own"}, {"path": "chunked", "chunk_mode": "lookback"},
                {"path": "chunked", "chunk_mode": "twopass"}, {"path": "chunked", "chunk_mode": "blocks"},
                {"path": "regcarry"}):
        h.fill_(float("nan"))
        lr.linrec_scan_f32_ex(a, b, h, **opt) if opt else lr.linrec_scan_f32(a, b, h)
        _check(h, a, b, f"fp32 {opt or 'auto'}")
    assert lr.linrec_stream_status() == lr.LINREC_OK


def test_gradient_past_2_31():
    a, b = _draw(72)
    h = lr.linrec_scan_f32(a, b)
    del b
    g = torch.randn(a.shape, generator=torch.Generator(device=DEV).manual_seed(73), device=DEV)
    for opt in ({}, {"path": "chunked", "chunk_mode": "own"}):
        da, db = lr.linrec_scan_f32_backward(a, h, g, **opt)
        torch.cuda.synchronize()
        for (i, d) in SAMPLES:
            ac, hc, gc = (_channel(x, i, d) for x in (a, h, g))
            da64, db64, _ = oracle.f64_backward(ac, hc, gc)
            assert_close(_channel(db, i, d), db64, f"db {opt or 'auto'} channel ({i}, {d})")
            assert_close(_channel(da, i, d), da64, f"da {opt or 'auto'} channel ({i}, {d})")
        del da, db
    assert lr.linrec_stream_status() == lr.LINREC_OK


@pytest.mark.parametrize("kind", ["bf16", "f16"])
def test_16bit_past_2_31(kind):
    a32, b32 = _draw(74)
    dt = torch.bfloat16 if kind == "bf16" else torch.float16
    a, b = a32.to(dt), b32.to(dt)
    del a32, b32
    scan = lr.linrec_scan_bf16 if kind == "bf16" else lr.linrec_scan_f16
    h = scan(a, b)
    torch.cuda.synchronize()
    u = 2.0 ** -8 if kind == "bf16" else 2.0 ** -11
    for (i, d) in SAMPLES:
        # the stored words are the input; their float32 values are exact
        h64, _ = oracle.f64(_channel(a, i, d), _channel(b, i, d))
        got = _channel(h, i, d).astype(np.float64)
        bad = ~(np.abs(got - h64) <= u * np.abs(h64) + (1 + u) * 1e-4 * (1 + np.abs(h64)))
        assert not bad.any(), f"{kind} channel ({i}, {d}): {int(bad.sum())} elements out of bound"


def test_bdl_layout_past_2_31():
    a, b = _draw(75, (B, D, L))
    h = torch.empty_like(a)
    for opt in ({}, {"chunk_mode": "own"}, {"chunk_mode": "twopass"}):
        lr.linrec_scan_f32_bdl_ex(a, b, h, **opt) if opt else lr.linrec_scan_f32_bdl(a, b, h)
        _check(h, a, b, f"(B, D, L) {opt or 'auto'}", bdl=True)
