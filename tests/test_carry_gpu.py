"""linrec_scan_f32_carry: the scan continued from a state h_init, handing out h_last.

Checked against the oracle's carried recurrence (h_{-1} = h_init, a_0 used)
within |h - h64| <= 1e-4 (1 + |h64|), on every path and chunk mode.
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
PATHS = [{}, {"path": "regcarry"}, {"path": "regcarry", "vec": 1, "prefetch": 4},
         {"path": "chunked", "chunk_mode": "own"}, {"path": "chunked", "chunk_mode": "lookback"},
         {"path": "chunked", "chunk_mode": "lookback", "tile_d": 32, "tile_t": 64, "stages": 3},
         {"path": "chunked", "chunk_mode": "twopass"},
         {"path": "chunked", "chunk_mode": "twopass", "tile_d": 64, "tile_t": 64, "stages": 2},
         {"path": "chunked", "chunk_mode": "blocks"},
         {"path": "chunked", "chunk_mode": "blocks", "tile_d": 64, "group": 3},
         {"path": "chunked", "chunk_mode": "chain"}]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)


def _state(B, D, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((B, D), generator=g, dtype=torch.float32)


@pytest.mark.parametrize("shape", [(1, 1, 4), (2, 33, 36), (3, 1000, 260), (1, 20000, 64), (4, 129, 128),
                                   (2, 77, 6)], ids=lambda s: "x".join(map(str, s)))
def test_carry_parity(shape):
    B, L, D = shape
    a, b = inputs.generate(B, L, D, seed=40 + L, a_dist="u[0.5,1)", b_dist="n(0,1)")
    h0 = _state(B, D, 41)
    h64, hl64 = oracle.f64_carry(a, b, h0.numpy().astype(np.float64))
    a_d, b_d, h0_d = a.to(DEV), b.to(DEV), h0.to(DEV)
    for opt in PATHS:
        if D % 4 and opt.get("path") == "chunked":
            continue
        hl = torch.full((B, D), float("nan"), device=DEV)
        h = lr.linrec_scan_f32_ex(a_d, b_d, h_init=h0_d, h_last=hl, **opt)
        torch.cuda.synchronize()
        assert_close(h.cpu().numpy(), h64, f"{shape} {opt} h")
        assert_close(hl.cpu().numpy(), hl64, f"{shape} {opt} h_last")


def test_no_state_in_gives_the_plain_scan_and_its_last_state():
    B, L, D = 3, 777, 68
    a, b = inputs.generate(B, L, D, seed=42)
    a[:, 0, :] = float("inf")                      # a_0 unused without a state
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    for opt in PATHS:
        hl = torch.empty((B, D), device=DEV)
        h = lr.linrec_scan_f32_ex(a_d, b_d, h_last=hl, **opt)
        torch.cuda.synchronize()
        assert_close(h.cpu().numpy(), h64, f"{opt}")
        assert torch.equal(hl, h[:, -1, :]), f"{opt}: h_last is not h[:, L-1]"


def test_a0_is_used_with_a_state():
    B, L, D = 1, 8, 4
    a = torch.full((B, L, D), 2.0)
    b = torch.zeros((B, L, D))
    h0 = torch.ones((B, D))
    for opt in PATHS:
        h = lr.linrec_scan_f32_ex(a.to(DEV), b.to(DEV), h_init=h0.to(DEV), **opt)
        torch.cuda.synchronize()
        want = 2.0 ** (torch.arange(L, dtype=torch.float32) + 1)
        assert torch.equal(h[0, :, 0].cpu(), want), opt


@pytest.mark.parametrize("name", ["pages", "long"])
def test_segments_continue_exactly_where_the_last_stopped(name):
    """Scanning a workload in segments, each continued from the previous h_last, matches the oracle."""
    w = inputs.WORKLOADS[name]
    a, b = inputs.generate_workload(w)
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    del a, b
    h = torch.empty_like(a_d)
    state = torch.empty((w.B, w.D), device=DEV)
    cuts = [0, w.L // 7, w.L // 7 + 1, w.L // 2, w.L]
    for k, (lo, hi) in enumerate(zip(cuts[:-1], cuts[1:])):
        seg = lr.linrec_scan_f32_carry(a_d[:, lo:hi].contiguous(), b_d[:, lo:hi].contiguous(),
                                       h_init=None if k == 0 else state, h_last=state)
        h[:, lo:hi] = seg
    torch.cuda.synchronize()
    assert_close(h.cpu().numpy(), h64, f"{name} in segments")


def test_state_updated_in_place_and_overlaps_refused():
    B, L, D = 2, 300, 64
    a, b = inputs.generate(B, L, D, seed=43)
    h0 = _state(B, D, 44)
    h64, hl64 = oracle.f64_carry(a, b, h0.numpy().astype(np.float64))
    a_d, b_d = a.to(DEV), b.to(DEV)
    for opt in PATHS:
        st = h0.to(DEV).clone()
        h = lr.linrec_scan_f32_ex(a_d, b_d, h_init=st, h_last=st, **opt)   # same buffer: in place
        torch.cuda.synchronize()
        assert_close(h.cpu().numpy(), h64, f"in place {opt}")
        assert_close(st.cpu().numpy(), hl64, f"in place state {opt}")
    h = torch.empty_like(a_d)
    with pytest.raises(lr.LinrecError) as e:
        lr.linrec_scan_f32_carry(a_d, b_d, h, h_last=h.view(-1)[:B * D].view(B, D))
    assert e.value.code == lr.LINREC_ERR_ALIAS
    with pytest.raises(lr.LinrecError) as e:
        lr.linrec_scan_f32_carry(a_d, b_d, h, h_init=h.view(-1)[5:5 + B * D].view(B, D))
    assert e.value.code == lr.LINREC_ERR_ALIAS
