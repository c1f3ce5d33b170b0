"""The (B, D, L) layout (time innermost, each channel a contiguous row) against the
oracle's linrec_oracle_f64_bdl, within |h - h64| <= 1e-4 (1 + |h64|) for fp32
storage and the 16-bit bound u |h64| + (1 + u) 1e-4 (1 + |h64|) for bfloat16
(u = 2^-8) and binary16 (u = 2^-11) storage.  The inputs are the five workloads'
draws, moved to (B, D, L)."""
import numpy as np
import pytest
import torch

import linear_recurrence_scan_fp32_gb300 as lr
import oracle
from linear_recurrence_scan_fp32_gb300 import inputs
from tests._util import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
MODES = [{}, {"chunk_mode": "own"}, {"chunk_mode": "twopass"}, {"chunk_mode": "own", "prefetch": 2},
         {"chunk_mode": "twopass", "prefetch": 2}, {"rows_per_warp": 5}]
UNIT = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}
SCAN16 = {"bf16": lr.linrec_scan_bf16_bdl_ex, "f16": lr.linrec_scan_f16_bdl_ex}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)


def run(a, b, **opt):
    h = lr.linrec_scan_f32_bdl_ex(a, b, **opt) if opt else lr.linrec_scan_f32_bdl(a, b)
    torch.cuda.synchronize()
    return h


def draw_bdl(B, D, L, seed, a_dist="u[0,1)", b_dist="n(0,1)"):
    a, b = inputs.generate(B, L, D, seed=seed, a_dist=a_dist, b_dist=b_dist)
    return inputs.to_bdl(a), inputs.to_bdl(b)


@pytest.mark.parametrize("name", inputs.CONFIG_ORDER)
def test_workload_full_size(name):
    w = inputs.WORKLOADS[name]
    a, b = inputs.generate_workload(w)
    a, b = inputs.to_bdl(a), inputs.to_bdl(b)
    h64, _ = oracle.f64_bdl(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    del a, b
    for opt in MODES:
        h = run(a_d, b_d, **opt)
        assert_close(h.cpu().numpy(), h64, f"{name} (B, D, L) {opt}")
        del h
    assert lr.linrec_stream_status() == lr.LINREC_OK


def test_geometric_long_rows():
    """Constant a = 0.99, b = 1 over 2^20 steps: h_t = (1 - 0.99^(t+1)) / 0.01, in both passes' modes."""
    B, D, L = 1, 64, 1 << 20
    a = torch.full((B, D, L), 0.99)
    b = torch.ones((B, D, L))
    t = np.arange(L, dtype=np.float64)
    want = np.broadcast_to((1 - 0.99 ** (t + 1)) / 0.01, (B, D, L))
    for opt in ({}, {"chunk_mode": "own"}, {"chunk_mode": "twopass"}):
        h = run(a.to(DEV), b.to(DEV), **opt)
        assert_close(h.cpu().numpy(), want, f"geometric {opt}")


@pytest.mark.parametrize("kind", ["ones", "zeros"])
def test_closed_forms_bit_exact(kind):
    B, D, L = 16, 256, 1000
    g = torch.Generator().manual_seed(90)
    b = torch.randint(-8, 9, (B, D, L), generator=g).float()
    a = torch.ones_like(b) if kind == "ones" else torch.zeros_like(b)
    want = torch.cumsum(b.double(), 2).float() if kind == "ones" else b
    for opt in MODES:
        h = run(a.to(DEV), b.to(DEV), **opt)
        assert torch.equal(h.cpu(), want), f"a = {kind} {opt}"


RAGGED = [(1, 1, 1), (1, 1, 4), (2, 3, 5), (1, 2, 31), (3, 1, 33), (1, 5, 127), (2, 2, 129), (1, 1, 4097),
          (2, 3, 1000), (1, 4, 5003), (1, 2, 70000), (1, 1, 262143)]


@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
def test_ragged_rows(shape):
    """Any L: vectors of 4, 2 or 1 elements per lane as L allows; partial last chunks; both modes."""
    B, D, L = shape
    a, b = draw_bdl(B, D, L, 91 + L, a_dist="u[0.5,1)")
    h64, _ = oracle.f64_bdl(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    extra = [{"vec": 8}, {"vec": 8, "chunk_mode": "twopass"}] if L % 8 == 0 else []   # 32-byte lanes
    for opt in MODES + [{"vec": 1}, {"vec": 1, "chunk_mode": "twopass"}] + extra:
        assert_close(run(a_d, b_d, **opt).cpu().numpy(), h64, f"{shape} {opt}")


def test_misaligned_pointers_narrow_the_vectors():
    B, D, L = 2, 8, 3000
    a, b = draw_bdl(B, D, L, 92)
    h64, _ = oracle.f64_bdl(a, b)
    n = B * D * L
    for shift in (1, 2):                              # 4 and 8 bytes off a 16-byte boundary
        bufs = [torch.empty(n + 4, device=DEV) for _ in range(3)]
        a_v, b_v, h_v = (x[shift:shift + n].view(B, D, L) for x in bufs)
        a_v.copy_(a.to(DEV))
        b_v.copy_(b.to(DEV))
        for opt in ({}, {"chunk_mode": "twopass"}):
            lr.linrec_scan_f32_bdl_ex(a_v, b_v, h=h_v, **opt)
            torch.cuda.synchronize()
            assert_close(h_v.cpu().numpy(), h64, f"shift {shift} {opt}")
        with pytest.raises(lr.LinrecError):
            lr.linrec_scan_f32_bdl_ex(a_v, b_v, h=h_v, vec=4)


@pytest.mark.parametrize("shape", [(2, 3, 40), (1, 64, 20000), (3, 5, 1001), (1, 2, 70000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_carry_state(shape):
    """h_init / h_last (B, D) as for linrec_scan_f32_carry, also updated in place."""
    B, D, L = shape
    a, b = draw_bdl(B, D, L, 93 + L, a_dist="u[0.5,1)")
    g = torch.Generator().manual_seed(94)
    h0 = torch.randn((B, D), generator=g)
    h64, last64 = oracle.f64_bdl(a, b, h0.double().numpy())
    a_d, b_d = a.to(DEV), b.to(DEV)
    for opt in MODES:
        last = torch.full((B, D), float("nan"), device=DEV)
        h = run(a_d, b_d, h_init=h0.to(DEV), h_last=last, **opt)
        assert_close(h.cpu().numpy(), h64, f"{shape} {opt} h")
        assert_close(last.cpu().numpy(), last64, f"{shape} {opt} h_last")
        st = h0.to(DEV).clone()
        h = run(a_d, b_d, h_init=st, h_last=st, **opt)        # same buffer: in place
        assert_close(h.cpu().numpy(), h64, f"{shape} {opt} in place")
        assert_close(st.cpu().numpy(), last64, f"{shape} {opt} in-place state")


@pytest.mark.parametrize("shape", [(2, 9, 5), (1, 40, 33), (3, 7, 128), (2, 11, 200), (1, 64, 1000), (4, 100, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_several_rows_per_warp(shape):
    """A warp streams consecutive rows through one chunk sequence: rows shorter than a chunk,
    rows straddling chunks, every vector width; the chain restarts at every row start."""
    B, D, L = shape
    a, b = draw_bdl(B, D, L, 98 + L + D, a_dist="u[0.5,1)")
    g = torch.Generator().manual_seed(99)
    h0 = torch.randn((B, D), generator=g)
    h64, _ = oracle.f64_bdl(a, b)
    hs64, last64 = oracle.f64_bdl(a, b, h0.double().numpy())
    a_d, b_d = a.to(DEV), b.to(DEV)
    for k in (1, 2, 3, 7, 64, B * D):
        for vec in (0, 1) + ((8,) if L % 8 == 0 else ()):
            opt = {"rows_per_warp": k, "vec": vec}
            assert_close(run(a_d, b_d, **opt).cpu().numpy(), h64, f"{shape} {opt}")
            last = torch.full((B, D), float("nan"), device=DEV)
            h = run(a_d, b_d, h_init=h0.to(DEV), h_last=last, **opt)
            assert_close(h.cpu().numpy(), hs64, f"{shape} {opt} with a state")
            assert_close(last.cpu().numpy(), last64, f"{shape} {opt} h_last")


def test_segments_chain_through_the_state():
    B, D, L = 1, 16, 50000
    a, b = draw_bdl(B, D, L, 95, a_dist="u[0.9,1)")
    h64, _ = oracle.f64_bdl(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    h = torch.empty_like(a_d)
    state = torch.empty((B, D), device=DEV)
    cuts = [0, 7, 4096, 4097, 30001, L]
    for k, (lo, hi) in enumerate(zip(cuts[:-1], cuts[1:])):
        seg = lr.linrec_scan_f32_bdl_ex(a_d[:, :, lo:hi].contiguous(), b_d[:, :, lo:hi].contiguous(),
                                        h_init=None if k == 0 else state, h_last=state)
        h[:, :, lo:hi] = seg
    torch.cuda.synchronize()
    assert_close(h.cpu().numpy(), h64, "segments")


def test_deterministic_and_errors():
    B, D, L = 4, 32, 9000
    a, b = draw_bdl(B, D, L, 96)
    a_d, b_d = a.to(DEV), b.to(DEV)
    for opt in ({"chunk_mode": "own"}, {"chunk_mode": "twopass"}):
        assert torch.equal(run(a_d, b_d, **opt), run(a_d, b_d, **opt)), opt
    h = torch.empty_like(a_d)
    with pytest.raises(lr.LinrecError) as e:
        lr.linrec_scan_f32_bdl(a_d, b_d, a_d)
    assert e.value.code == lr.LINREC_ERR_ALIAS
    with pytest.raises(lr.LinrecError):
        lr.linrec_scan_f32_bdl_ex(a_d, b_d, h, chunk_mode="lookback")
    with pytest.raises(lr.LinrecError):
        lr.linrec_scan_f32_bdl_ex(a_d, b_d, h, path="chunked")
    assert lr.linrec_stream_status() == lr.LINREC_OK


def _close16(kind, h, h64, what):
    x = oracle.decode16(kind, h.cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    u = UNIT[kind]
    bad = ~(np.abs(x - h64) <= u * np.abs(h64) + (1 + u) * 1e-4 * (1 + np.abs(h64)))
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of bound"


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(32, 256, 4096), (1, 64, 1 << 20), (2, 3, 1000), (1, 5, 4099), (1, 2, 70001)],
                         ids=lambda s: "x".join(map(str, s)))
def test_16bit_storage(kind, shape):
    B, D, L = shape
    a, b = draw_bdl(B, D, L, 97 + L)
    a16, b16 = inputs.to_storage16(a, kind), inputs.to_storage16(b, kind)
    h64, _ = oracle.f64_bdl(oracle.decode16(kind, a16).astype(np.float32),
                            oracle.decode16(kind, b16).astype(np.float32))
    a_d, b_d = a16.to(DEV), b16.to(DEV)
    # by default 32-byte lanes (16 elements) where L allows; 16-byte lanes on request
    extra = ({"vec": 8}, {"vec": 8, "chunk_mode": "twopass"}) if L % 8 == 0 else ()
    for opt in ({}, {"chunk_mode": "own"}, {"chunk_mode": "twopass"}) + extra:
        h = SCAN16[kind](a_d, b_d, **opt)
        torch.cuda.synchronize()
        _close16(kind, h, h64, f"{kind} {shape} {opt}")
