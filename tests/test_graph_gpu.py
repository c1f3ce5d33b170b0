"""The scan captured into a CUDA graph and replayed.

A call made while its stream is capturing allocates nothing: it uses the
workspace the library already holds for that stream (made by one call outside
capture), or returns LINREC_ERR_WORKSPACE and enqueues nothing.  Replays of
the captured kernels must give the same bits as the uncaptured call (the
kernels are deterministic), follow new data written into the captured
buffers, and leave the stream's status word clean.
"""
import numpy as np
import pytest
import torch

import linear_recurrence_scan_fp32_gb300 as lr
import oracle
from linear_recurrence_scan_fp32_gb300 import inputs
from tests._util import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)


MODES = [{}, {"path": "regcarry"}, {"path": "chunked", "chunk_mode": "own"},
         {"path": "chunked", "chunk_mode": "lookback"}, {"path": "chunked", "chunk_mode": "twopass"},
         {"path": "chunked", "chunk_mode": "blocks"}, {"path": "chunked", "chunk_mode": "chain"},
         {"path": "chunked", "chunk_mode": "speculative"}]


def _scan(a, b, h, opt, stream=None):
    if opt:
        lr.linrec_scan_f32_ex(a, b, h, stream=stream, **opt)
    else:
        lr.linrec_scan_f32(a, b, h, stream=stream)


@pytest.mark.parametrize("opt", MODES, ids=lambda o: o.get("chunk_mode", o.get("path", "auto")))
def test_captured_scan_replays(opt):
    B, L, D = 2, 20000, 96
    a, b = inputs.generate(B, L, D, seed=61, a_dist="u[0.9,1)", b_dist="n(0,1)")
    a_d, b_d = a.to(DEV), b.to(DEV)
    h = torch.empty_like(a_d)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _scan(a_d, b_d, h, opt, stream=s)          # outside capture: the stream's workspace
    s.synchronize()
    want = h.clone()
    assert_close(want.cpu().numpy(), oracle.f64(a, b)[0], f"uncaptured {opt}")

    g = torch.cuda.CUDAGraph()
    h.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        _scan(a_d, b_d, h, opt)                    # captured, not run
    torch.cuda.synchronize()
    assert torch.isnan(h).all(), "capture ran the kernels"
    for k in range(5):
        h.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(h, want), f"{opt} replay {k}: bits differ from the uncaptured call"
    # the graph reads whatever the captured buffers hold at replay time
    a2, b2 = inputs.generate(B, L, D, seed=62, a_dist="u[0.5,1)", b_dist="n(0,1)")
    a_d.copy_(a2)
    b_d.copy_(b2)
    g.replay()
    torch.cuda.synchronize()
    assert_close(h.cpu().numpy(), oracle.f64(a2, b2)[0], f"replay on new data {opt}")
    assert lr.linrec_stream_status(s) == lr.LINREC_OK


def test_capture_without_workspace_is_refused():
    """A fresh stream holds no workspace: the chunked call is refused and enqueues nothing, while
    the one-pass register path (a short sequence), which needs none, is captured; the capture
    itself stays valid."""
    B, L, D = 1, 4096, 64
    a, b = inputs.generate(B, L, D, seed=63, a_dist="u[0.5,1)", b_dist="n(0,1)")
    a_d, b_d = a.to(DEV), b.to(DEV)
    h = torch.full_like(a_d, float("nan"))
    a_s, b_s = a_d[:, :100].contiguous(), b_d[:, :100].contiguous()
    h_s = torch.full_like(a_s, float("nan"))
    assert lr.linrec_plan_f32(1, 100, D, path="regcarry")["twopass"] == 0
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        with pytest.raises(lr.LinrecError) as e:
            lr.linrec_scan_f32_ex(a_d, b_d, h, path="chunked", chunk_mode="lookback")
        assert e.value.code == lr.LINREC_ERR_WORKSPACE
        lr.linrec_scan_f32_ex(a_s, b_s, h_s, path="regcarry")
    g.replay()
    torch.cuda.synchronize()
    assert_close(h_s.cpu().numpy(), oracle.f64(a[:, :100], b[:, :100])[0], "captured register path")
    # outside capture the same stream allocates as usual
    with torch.cuda.stream(s):
        h2 = lr.linrec_scan_f32_ex(a_d, b_d, stream=s, path="chunked", chunk_mode="lookback")
    s.synchronize()
    assert_close(h2.cpu().numpy(), oracle.f64(a, b)[0], "after the capture")
    assert lr.linrec_stream_status(s) == lr.LINREC_OK


def test_captured_16bit_layout_and_gradient():
    """The other entry points under capture: 16-bit storage, the (B, D, L) layout (two-pass) and
    the gradient (two-pass), each warmed up once on the capturing stream."""
    s = torch.cuda.Stream()
    B, L, D = 1, 1 << 16, 64
    a, b = inputs.generate(B, L, D, seed=64, a_dist="u[0.9,1)", b_dist="n(0,1)")
    a_d, b_d = a.to(DEV), b.to(DEV)
    a16, b16 = a_d.to(torch.bfloat16), b_d.to(torch.bfloat16)
    h16 = torch.empty_like(a16)
    at, bt = a_d.transpose(1, 2).contiguous(), b_d.transpose(1, 2).contiguous()
    ht = torch.empty_like(at)
    h = lr.linrec_scan_f32(a_d, b_d)
    torch.cuda.synchronize()
    g_d = torch.randn_like(a_d)
    da, db = torch.empty_like(a_d), torch.empty_like(a_d)

    def calls():
        lr.linrec_scan_bf16_ex(a16, b16, h16, chunk_mode="twopass", path="chunked")
        lr.linrec_scan_f32_bdl_ex(at, bt, ht, chunk_mode="twopass")
        lr.linrec_scan_f32_backward(a_d, h, g_d, da=da, db=db, path="chunked", chunk_mode="twopass")

    with torch.cuda.stream(s):
        calls()
    s.synchronize()
    want = [x.clone() for x in (h16, ht, da, db)]
    g = torch.cuda.CUDAGraph()
    for x in (h16, ht, da, db):
        x.zero_()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        calls()
    for k in range(3):
        g.replay()
        torch.cuda.synchronize()
        for name, x, w in zip(("h16", "h (B, D, L)", "da", "db"), (h16, ht, da, db), want):
            assert torch.equal(x, w), f"{name} replay {k}: bits differ"
    assert lr.linrec_stream_status(s) == lr.LINREC_OK
