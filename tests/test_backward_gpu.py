"""linrec_scan_f32_backward: the gradient of the scan, against the oracle's
reverse loop (which is pinned by finite differences and the adjoint identity),
within |x - x64| <= 1e-4 (1 + |x64|) for da, db and dh_init."""
import numpy as np
import pytest
import torch

import linear_recurrence_scan_fp32_gb300 as lr
import oracle
from linear_recurrence_scan_fp32_gb300 import inputs
from tests._util import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
PATHS = [{}, {"path": "regcarry"}, {"path": "regcarry", "vec": 1},
         {"path": "chunked", "chunk_mode": "own"}, {"path": "chunked", "chunk_mode": "lookback"},
         {"path": "chunked", "chunk_mode": "own", "tile_d": 32, "tile_t": 64, "stages": 3},
         {"path": "chunked", "chunk_mode": "lookback", "tile_d": 64, "tile_t": 128, "stages": 2},
         {"path": "chunked", "chunk_mode": "twopass"},
         {"path": "chunked", "chunk_mode": "twopass", "tile_d": 64, "tile_t": 64, "stages": 2}]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32) * scale


def _legal(opt, D):
    return not (D % 4 and opt.get("path") == "chunked")


@pytest.mark.parametrize("shape", [(1, 1, 4), (2, 33, 36), (3, 1000, 260), (1, 20000, 64), (4, 129, 128),
                                   (2, 77, 6), (2, 64, 32)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("state", ["none", "both"])
def test_backward_parity(shape, state):
    B, L, D = shape
    a, b = inputs.generate(B, L, D, seed=50 + L, a_dist="u[0.5,1)", b_dist="n(0,1)")
    g = _rand((B, L, D), 51)
    h0 = _rand((B, D), 52) if state == "both" else None
    w = _rand((B, D), 53) if state == "both" else None
    h64, _ = oracle.f64_carry(a, b, None if h0 is None else h0.numpy().astype(np.float64))
    h32 = torch.from_numpy(h64.astype(np.float32))
    da64, db64, dx64 = oracle.f64_backward(a, h32, g, None if h0 is None else h0.numpy().astype(np.float64),
                                           None if w is None else w.numpy().astype(np.float64))
    a_d, h_d, g_d = a.to(DEV), h32.to(DEV), g.to(DEV)
    h0_d = None if h0 is None else h0.to(DEV)
    w_d = None if w is None else w.to(DEV)
    for opt in PATHS:
        if not _legal(opt, D):
            continue
        dx = torch.full((B, D), float("nan"), device=DEV)
        da, db = lr.linrec_scan_f32_backward(a_d, h_d, g_d, h_init=h0_d, dh_last=w_d, dh_init=dx, **opt)
        torch.cuda.synchronize()
        assert_close(db.cpu().numpy(), db64, f"{shape} {opt} db")
        assert_close(da.cpu().numpy(), da64, f"{shape} {opt} da")
        assert_close(dx.cpu().numpy(), dx64, f"{shape} {opt} dh_init")
        # db only: h is not read
        _, db2 = lr.linrec_scan_f32_backward(a_d, None, g_d, h_init=h0_d, dh_last=w_d, want_da=False, **opt)
        torch.cuda.synchronize()
        assert torch.equal(db2, db), f"{opt}: db changed without da"
    assert lr.linrec_stream_status() == lr.LINREC_OK


@pytest.mark.parametrize("name", ["pages", "gated", "long"])
def test_backward_full_size(name):
    w = inputs.WORKLOADS[name]
    a, b = inputs.generate_workload(w)
    a_d, b_d = a.to(DEV), b.to(DEV)
    h_d = lr.linrec_scan_f32(a_d, b_d)
    del b_d
    g = _rand(w.shape, 60)
    g_d = g.to(DEV)
    h = h_d.cpu()
    da64, db64, _ = oracle.f64_backward(a, h, g)
    del a, h, g
    for opt in [{}, {"path": "chunked", "chunk_mode": "own"}, {"path": "chunked", "chunk_mode": "lookback"},
                {"path": "chunked", "chunk_mode": "twopass"}]:
        da, db = lr.linrec_scan_f32_backward(a_d, h_d, g_d, **opt)
        torch.cuda.synchronize()
        assert_close(db.cpu().numpy(), db64, f"{name} {opt} db")
        assert_close(da.cpu().numpy(), da64, f"{name} {opt} da")
        del da, db


def test_backward_closed_forms_bit_exact():
    """a = 1 with integer g: db is the suffix sum of g, exact; a = 0: db = g."""
    B, L, D = 8, 4096, 64
    gen = torch.Generator().manual_seed(61)
    g = torch.randint(-8, 9, (B, L, D), generator=gen).float()
    want = torch.flip(torch.cumsum(torch.flip(g.double(), [1]), 1), [1]).float()
    g_d = g.to(DEV)
    ones = torch.ones_like(g_d)
    for opt in PATHS:
        _, db = lr.linrec_scan_f32_backward(ones, None, g_d, want_da=False, **opt)
        torch.cuda.synchronize()
        assert torch.equal(db.cpu(), want), f"a=1 {opt}"
        _, db = lr.linrec_scan_f32_backward(torch.zeros_like(g_d), None, g_d, want_da=False, **opt)
        torch.cuda.synchronize()
        assert torch.equal(db, g_d), f"a=0 {opt}"


@pytest.mark.parametrize("tile", [(32, 128, 2), (32, 64, 3), (32, 64, 4), (64, 64, 2), (64, 128, 2), (128, 64, 2),
                                  (256, 32, 2)],
                         ids=lambda t: f"d{t[0]}t{t[1]}s{t[2]}")
def test_backward_modes_agree_and_repeat(tile):
    td, tt, st = tile
    B, L, D = 2, 3000, 128
    a, b = inputs.generate(B, L, D, seed=62)
    g = _rand((B, L, D), 63)
    a_d, g_d = a.to(DEV), g.to(DEV)
    h_d = lr.linrec_scan_f32(a_d, b.to(DEV))
    opt = {"path": "chunked", "tile_d": td, "tile_t": tt, "stages": st}
    da1, db1 = lr.linrec_scan_f32_backward(a_d, h_d, g_d, chunk_mode="own", **opt)
    da2, db2 = lr.linrec_scan_f32_backward(a_d, h_d, g_d, chunk_mode="lookback", **opt)
    da3, db3 = lr.linrec_scan_f32_backward(a_d, h_d, g_d, chunk_mode="lookback", **opt)
    torch.cuda.synchronize()
    assert torch.equal(db1, db2) and torch.equal(da1, da2), "modes differ"
    assert torch.equal(db2, db3) and torch.equal(da2, da3), "not deterministic"
    da64, db64, _ = oracle.f64_backward(a, h_d.cpu(), g)
    assert_close(db1.cpu().numpy(), db64, f"db {tile}")
    assert_close(da1.cpu().numpy(), da64, f"da {tile}")


def test_backward_in_segments_chains_through_dh_init():
    """Gradient of a sequence scanned in segments: each segment's dh_init is the earlier one's dh_last."""
    B, L, D = 2, 5000, 64
    a, b = inputs.generate(B, L, D, seed=64, a_dist="u[0.9,1)")
    g = _rand((B, L, D), 65)
    h64, _ = oracle.f64(a, b)
    h32 = torch.from_numpy(h64.astype(np.float32))
    da64, db64, _ = oracle.f64_backward(a, h32, g)
    a_d, h_d, g_d = a.to(DEV), h32.to(DEV), g.to(DEV)
    cuts = [0, 1200, 1201, 3333, L]
    da = torch.empty_like(a_d)
    db = torch.empty_like(a_d)
    carry = None
    for k in range(len(cuts) - 2, -1, -1):            # last segment first
        lo, hi = cuts[k], cuts[k + 1]
        h_init = None if lo == 0 else h_d[:, lo - 1].contiguous()
        dx = torch.empty((B, D), device=DEV)
        sda, sdb = lr.linrec_scan_f32_backward(a_d[:, lo:hi].contiguous(), h_d[:, lo:hi].contiguous(),
                                               g_d[:, lo:hi].contiguous(), h_init=h_init, dh_last=carry,
                                               dh_init=dx)
        da[:, lo:hi] = sda
        db[:, lo:hi] = sdb
        carry = dx
    torch.cuda.synchronize()
    assert_close(db.cpu().numpy(), db64, "segments db")
    assert_close(da.cpu().numpy(), da64, "segments da")


def test_backward_in_place_and_overlaps():
    B, L, D = 2, 300, 64
    a, _ = inputs.generate(B, L, D, seed=66)
    g = _rand((B, L, D), 67)
    h = _rand((B, L, D), 68)
    da64, db64, _ = oracle.f64_backward(a, h, g)
    a_d, h_d = a.to(DEV), h.to(DEV)
    for opt in PATHS:
        gg = g.to(DEV)
        da, db = lr.linrec_scan_f32_backward(a_d, h_d, gg, db=gg, **opt)   # db written over g
        torch.cuda.synchronize()
        assert db.data_ptr() == gg.data_ptr()
        assert_close(db.cpu().numpy(), db64, f"in place {opt}")
        assert_close(da.cpu().numpy(), da64, f"in place da {opt}")
    gg = g.to(DEV)
    with pytest.raises(lr.LinrecError) as e:
        lr.linrec_scan_f32_backward(a_d, h_d, gg, da=gg)
    assert e.value.code == lr.LINREC_ERR_ALIAS
    with pytest.raises(lr.LinrecError) as e:
        lr.linrec_scan_f32_backward(a_d, h_d, gg, db=a_d)
    assert e.value.code == lr.LINREC_ERR_ALIAS
