"""Parity of the CUDA kernels with the fp64 CPU oracle, through the C ABI.

Bound (per element): |h - h64| <= 1e-4 * (1 + |h64|).  The closed-form
variants with integer b (a = 1: prefix sums below 2^24; a = 0: h = b) must
match bit for bit on every path.
"""
import ctypes

import numpy as np
import pytest
import torch

import linear_recurrence_scan_fp32_gb300 as lr
import oracle
from linear_recurrence_scan_fp32_gb300 import inputs
from tests._util import assert_close, max_errors

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)


def run(a_d, b_d, **opt):
    h = lr.linrec_scan_f32_ex(a_d, b_d, **opt) if opt else lr.linrec_scan_f32(a_d, b_d)
    torch.cuda.synchronize()
    return h


def legal_paths(B, L, D, aligned=True):
    paths = [{"path": "regcarry"}]
    if aligned and D % 4 == 0:
        paths.append({"path": "chunked", "chunk_mode": "own"})
        paths.append({"path": "chunked", "chunk_mode": "lookback"})
        paths.append({"path": "chunked", "chunk_mode": "twopass"})
        paths.append({"path": "chunked", "chunk_mode": "blocks"})
        if B * -(-D // 32) <= 128:         # chain mode serves few slices only
            paths.append({"path": "chunked", "chunk_mode": "chain"})
    return paths


# ---------------------------------------------------------------------------
# the five workloads at full size, every path, against the full fp64 oracle
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", inputs.CONFIG_ORDER)
def test_workload_full_size(name):
    w = inputs.WORKLOADS[name]
    a, b = inputs.generate_workload(w)
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    del a, b
    for opt in [{}] + legal_paths(w.B, w.L, w.D):
        h = run(a_d, b_d, **opt).cpu().numpy()
        assert_close(h, h64, f"{name} {opt or 'auto'}")
        del h
    assert lr.linrec_stream_status() == lr.LINREC_OK


@pytest.mark.parametrize("name", ["short_ones_int", "short_zeros_int"])
def test_closed_forms_bit_exact(name):
    w = inputs.WORKLOADS[name]
    a, b = inputs.generate_workload(w)
    bn = b.numpy()
    if w.a_dist == "ones":
        want = np.cumsum(bn.astype(np.float64), axis=1).astype(np.float32)   # |sum| <= 1024: exact
    else:
        want = bn
    a_d, b_d = a.to(DEV), b.to(DEV)
    for opt in [{}] + legal_paths(w.B, w.L, w.D):
        h = run(a_d, b_d, **opt).cpu().numpy()
        assert np.array_equal(h, want), f"{name} {opt}: not bit-exact"


@pytest.mark.parametrize("name", ["short_ones", "short_zeros"])
def test_closed_forms_real_b(name):
    w = inputs.WORKLOADS[name]
    a, b = inputs.generate_workload(w)
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    for opt in [{}] + legal_paths(w.B, w.L, w.D):
        assert_close(run(a_d, b_d, **opt).cpu().numpy(), h64, f"{name} {opt}")
    if w.a_dist == "zeros":   # a = 0 copies b exactly even with real b
        for opt in [{}] + legal_paths(w.B, w.L, w.D):
            assert torch.equal(run(a_d, b_d, **opt), b_d)


def test_geometric_long_carry():
    """Long-sequence shape (1, 1048576, 64), a = 0.99, b = 1: h_t = (1 - 0.99^(t+1)) / 0.01."""
    B, L, D = 1, 1 << 20, 64
    a_d = torch.full((B, L, D), 0.99, device=DEV)
    b_d = torch.ones((B, L, D), device=DEV)
    t = np.arange(L, dtype=np.float64)
    want = (1.0 - np.float64(np.float32(0.99)) ** (t + 1)) / (1.0 - np.float64(np.float32(0.99)))
    for opt in [{}] + legal_paths(B, L, D):
        h = run(a_d, b_d, **opt).cpu().numpy()
        for d in (0, 17, 63):
            assert_close(h[0, :, d], want, f"geometric {opt} d={d}")


# ---------------------------------------------------------------------------
# ragged shapes, every path and every chunked variant
# ---------------------------------------------------------------------------

RAGGED = [(1, 1, 4), (1, 2, 8), (3, 31, 4), (2, 33, 36), (1, 65, 100), (3, 127, 132), (2, 129, 64),
          (1, 1000, 260), (2, 257, 68), (1, 5000, 32), (1, 4097, 8), (4, 300, 1),
          (1, 70, 3), (2, 33, 5), (3, 100, 33), (1, 2, 2), (2, 9, 6)]


@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
def test_ragged_shapes(shape):
    B, L, D = shape
    a, b = inputs.generate(B, L, D, seed=100 + L + D, a_dist="u[0.5,1)", b_dist="n(0,1)")
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    opts = [{}] + legal_paths(B, L, D)
    if D % 2 == 0:
        opts.append({"path": "regcarry", "vec": 2})
    opts.append({"path": "regcarry", "vec": 1, "prefetch": 4})
    for opt in opts:
        assert_close(run(a_d, b_d, **opt).cpu().numpy(), h64, f"{shape} {opt}")


VARIANTS = [(128, 64, 2), (128, 64, 3), (128, 32, 3), (256, 32, 2), (64, 128, 2), (64, 64, 2), (64, 64, 3),
            (32, 128, 2), (32, 128, 3), (32, 64, 3), (32, 64, 4), (32, 32, 6)]


def _variants():
    out = []
    for td, tt, st in VARIANTS:
        for mode in ("own", "lookback", "twopass"):
            out.append({"path": "chunked", "tile_d": td, "tile_t": tt, "stages": st, "chunk_mode": mode})
    return out


@pytest.mark.parametrize("opt", _variants(),
                         ids=lambda o: f"d{o['tile_d']}t{o['tile_t']}s{o['stages']}-{o['chunk_mode']}")
def test_every_chunked_variant(opt):
    for (B, L, D) in [(3, 1000, 260), (1, 20000, 64), (2, 777, 36)]:
        a, b = inputs.generate(B, L, D, seed=7 + L, a_dist="u[0.9,1)", b_dist="n(0,1)")
        h64, _ = oracle.f64(a, b)
        h = run(a.to(DEV), b.to(DEV), **opt).cpu().numpy()
        assert_close(h, h64, f"{(B, L, D)} {opt}")


@pytest.mark.parametrize("tile", VARIANTS, ids=lambda t: f"d{t[0]}t{t[1]}s{t[2]}")
def test_chunk_modes_agree_bit_for_bit(tile):
    """Both modes evaluate the carry as the same chain H_q = A_q*H_{q-1} + B_q: identical bits."""
    td, tt, st = tile
    for (B, L, D, seed) in [(2, 3000, 128, 1), (1, 50000, 64, 2)]:
        a, b = inputs.generate(B, L, D, seed=seed, a_dist="u[0,1)", b_dist="n(0,1)")
        a_d, b_d = a.to(DEV), b.to(DEV)
        opt = {"path": "chunked", "tile_d": td, "tile_t": tt, "stages": st}
        h_own = run(a_d, b_d, chunk_mode="own", **opt)
        h_lb = run(a_d, b_d, chunk_mode="lookback", **opt)
        assert torch.equal(h_own, h_lb), f"{tile} {(B, L, D)}"


@pytest.mark.parametrize("shape", [(2, 3000, 128), (1, 50000, 64), (3, 1000, 260), (1, 129, 32), (5, 4097, 36)],
                         ids=lambda s: "x".join(map(str, s)))
def test_chain_mode_same_bits_as_slice_owner(shape):
    """Chain mode folds every slice's tile maps in chunk order, H_q = A_q*H_{q-1} + B_q, the
    chain slice-owner mode carries in a register: the same tile gives identical bits, with
    and without a carried-in state."""
    B, L, D = shape
    a, b = inputs.generate(B, L, D, seed=7 + L, a_dist="u[0,1)", b_dist="n(0,1)")
    a_d, b_d = a.to(DEV), b.to(DEV)
    tile = {"path": "chunked", "tile_d": 32, "tile_t": 128}
    assert lr.linrec_plan_f32(B, L, D, chunk_mode="chain", **tile)["chain"] == 1
    assert torch.equal(run(a_d, b_d, chunk_mode="chain", **tile), run(a_d, b_d, chunk_mode="own", **tile))
    h0 = torch.randn(B, D, device=DEV)
    outs = []
    for mode in ("chain", "own"):
        last = torch.empty(B, D, device=DEV)
        outs.append((run(a_d, b_d, chunk_mode=mode, h_init=h0, h_last=last, **tile), last))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("shape", [(1, 40001, 36), (3, 33000, 64), (2, 65536, 100), (9, 32768, 32)],
                         ids=lambda s: "x".join(map(str, s)))
def test_chain_mode_long_tiles(shape):
    """Chain mode's 256-step tile (512 threads, 16 segments), taken from 32768 steps on: every
    element against the oracle, with and without a carried-in state, and the same bits on a
    second call."""
    B, L, D = shape
    a, b = inputs.generate(B, L, D, seed=9 + L, a_dist="u[0.9,1)", b_dist="n(0,1)")
    h0 = torch.randn(B, D)
    a_d, b_d = a.to(DEV), b.to(DEV)
    opt = {"path": "chunked", "chunk_mode": "chain"}
    assert lr.linrec_plan_f32(B, L, D, **opt)["tile_t"] == 256
    h = run(a_d, b_d, **opt)
    assert_close(h.cpu().numpy(), oracle.f64(a, b)[0], f"chain {shape}")
    assert torch.equal(run(a_d, b_d, **opt), h)
    last = torch.empty(B, D, device=DEV)
    h = run(a_d, b_d, h_init=h0.to(DEV), h_last=last, **opt)
    h64, last64 = oracle.f64_carry(a, b, h0.numpy().astype(np.float64))
    assert_close(h.cpu().numpy(), h64, f"chain {shape} with a state")
    assert_close(last.cpu().numpy(), last64, f"chain {shape} last state")


@pytest.mark.parametrize("vec,prefetch", [(v, p) for v in (1, 2, 4) for p in (4, 8, 16)])
def test_every_regcarry_variant(vec, prefetch):
    B, L, D = 2, 515, 132
    a, b = inputs.generate(B, L, D, seed=55, a_dist="u[0,1)", b_dist="n(0,1)")
    h64, _ = oracle.f64(a, b)
    h = run(a.to(DEV), b.to(DEV), path="regcarry", vec=vec, prefetch=prefetch).cpu().numpy()
    assert_close(h, h64, f"regcarry vec={vec} prefetch={prefetch}")


# ---------------------------------------------------------------------------
# memory safety, determinism, inputs untouched, misalignment
# ---------------------------------------------------------------------------

CANARY = 0x7fc0dead   # a NaN payload no kernel writes


def test_guard_bands_and_inputs_untouched():
    for (B, L, D) in [(3, 1000, 260), (1, 4097, 64), (2, 33, 5)]:
        a, b = inputs.generate(B, L, D, seed=3, a_dist="u[0.5,1)", b_dist="n(0,1)")
        h64, _ = oracle.f64(a, b)
        n = B * L * D
        guard = 4096
        for opt in [{}] + legal_paths(B, L, D):
            buf = torch.full((n + 2 * guard,), 0, dtype=torch.int32, device=DEV)
            buf.fill_(CANARY)
            hv = buf.view(torch.float32)[guard:guard + n].view(B, L, D)
            a_d, b_d = a.to(DEV), b.to(DEV)
            lr.linrec_scan_f32_ex(a_d, b_d, hv, **opt)
            torch.cuda.synchronize()
            assert (buf[:guard] == CANARY).all() and (buf[guard + n:] == CANARY).all(), f"guard band {opt}"
            assert torch.equal(a_d.cpu(), a) and torch.equal(b_d.cpu(), b), "inputs modified"
            assert_close(hv.cpu().numpy(), h64, f"guarded {opt}")


def test_deterministic_bits():
    for name in ("pages", "long"):
        w = inputs.WORKLOADS[name]
        a, b = inputs.generate_workload(w)
        a_d, b_d = a.to(DEV), b.to(DEV)
        for opt in [{}] + legal_paths(w.B, w.L, w.D):
            h1 = run(a_d, b_d, **opt).clone()
            for _ in range(3):
                assert torch.equal(run(a_d, b_d, **opt), h1), f"{name} {opt}: bits changed between calls"


@pytest.mark.parametrize("mode", ["lookback", "twopass", "blocks", "chain"])
def test_carry_modes_repeat_bit_identical(mode):
    """A race check on the cross-CTA carry: 50 calls of the look-back, two-pass, blocks or chain
    mode, whose tiles land on different CTAs in a different order every time, all return the same
    bits."""
    second = {"blocks": {"tile_d": 64, "group": 3}, "chain": {}}.get(mode, {"tile_d": 32, "tile_t": 64, "stages": 3})
    for (B, L, D, tile) in [(1, 1 << 18, 64, {}), (2, 50000, 128, second)]:
        a, b = inputs.generate(B, L, D, seed=19 + L, a_dist="u[0.9,1)", b_dist="n(0,1)")
        a_d, b_d = a.to(DEV), b.to(DEV)
        opt = dict(path="chunked", chunk_mode=mode, **tile)
        first = run(a_d, b_d, **opt).clone()
        h = torch.empty_like(first)
        for k in range(50):
            lr.linrec_scan_f32_ex(a_d, b_d, h, **opt)
            torch.cuda.synchronize()
            assert torch.equal(h, first), f"{mode} {(B, L, D)} call {k}: bits changed"
        h64, _ = oracle.f64(a, b)
        assert_close(first.cpu().numpy(), h64, f"{mode} {(B, L, D)}")
    assert lr.linrec_stream_status() == lr.LINREC_OK


@pytest.mark.parametrize("shape", [(7, 3000, 777), (1, 20000, 33), (3, 3001, 130), (4, 300, 1), (2, 5000, 6)],
                         ids=lambda s: "x".join(map(str, s)))
def test_segmented_register_path(shape):
    """Few channels the TMA path cannot take (D * 4 not a multiple of 16): the register path cuts the
    time axis into segments (a reduce launch, then an apply launch folding the earlier segments' maps),
    with and without a carried state; repeated calls give the same bits."""
    B, L, D = shape
    plan = lr.linrec_plan_f32(B, L, D, sm_count=torch.cuda.get_device_properties(DEV).multi_processor_count)
    assert plan["path_name"] == "regcarry" and plan["twopass"] == 1 and plan["segments"] > 1
    a, b = inputs.generate(B, L, D, seed=50 + L + D, a_dist="u[0.9,1)", b_dist="n(0,1)")
    a[:, 0, :] = float("nan")                 # a_0 is never used without a state
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    h = run(a_d, b_d)
    assert_close(h.cpu().numpy(), h64, f"segmented {shape}")
    assert torch.equal(run(a_d, b_d), h), f"segmented {shape}: bits changed"
    a[:, 0, :] = 0.5
    a_d = a.to(DEV)
    h0 = torch.randn((B, D), generator=torch.Generator().manual_seed(51))
    hc64, last64 = oracle.f64_carry(a, b, h0.numpy().astype(np.float64))
    last = torch.full((B, D), float("nan"), device=DEV)
    h = lr.linrec_scan_f32_carry(a_d, b_d, h_init=h0.to(DEV), h_last=last)
    torch.cuda.synchronize()
    assert_close(h.cpu().numpy(), hc64, f"segmented carry {shape}")
    assert_close(last.cpu().numpy(), last64, f"segmented h_last {shape}")
    assert lr.linrec_stream_status() == lr.LINREC_OK


def test_misaligned_pointers_take_the_scalar_path():
    B, L, D = 2, 300, 64
    a, b = inputs.generate(B, L, D, seed=9, a_dist="u[0.5,1)", b_dist="n(0,1)")
    h64, _ = oracle.f64(a, b)
    n = B * L * D
    ab = torch.empty(2 * n + 2, device=DEV)
    a_d = ab[1:1 + n]
    b_d = ab[n + 2:]
    a_d.copy_(a.reshape(-1).to(DEV))
    b_d.copy_(b.reshape(-1).to(DEV))
    hbuf = torch.empty(n + 1, device=DEV)
    h_d = hbuf[1:]
    L_ = lr.lib()
    code = L_.linrec_scan_f32(a_d.data_ptr(), b_d.data_ptr(), h_d.data_ptr(), B, L, D,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == lr.LINREC_OK
    torch.cuda.synchronize()
    assert_close(h_d.view(B, L, D).cpu().numpy(), h64, "misaligned auto")
    # forcing TMA on misaligned pointers is refused, not run
    opt = lr.make_options(path="chunked")
    code = L_.linrec_scan_f32_ex(a_d.data_ptr(), b_d.data_ptr(), h_d.data_ptr(), B, L, D,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(opt))
    assert code == lr.LINREC_ERR_INVALID_VALUE


def test_a0_is_ignored():
    a, b = inputs.generate(2, 500, 64, seed=11, a_dist="u[0.5,1)", b_dist="n(0,1)")
    h64, _ = oracle.f64(a, b)
    a[:, 0, :] = float("nan")
    a_d, b_d = a.to(DEV), b.to(DEV)
    for opt in [{}] + legal_paths(2, 500, 64):
        h = run(a_d, b_d, **opt).cpu().numpy()
        assert np.isfinite(h).all()
        assert_close(h, h64, f"a_0 = NaN {opt}")


def test_aliasing_rejected_on_device_pointers():
    a = torch.rand(1, 10, 8, device=DEV)
    b = torch.rand(1, 10, 8, device=DEV)
    with pytest.raises(lr.LinrecError) as e:
        lr.linrec_scan_f32(a, b, a)
    assert e.value.code == lr.LINREC_ERR_ALIAS
    h = lr.linrec_scan_f32(a, a)   # a and b may be the same buffer
    torch.cuda.synchronize()
    h64, _ = oracle.f64(a.cpu(), a.cpu())
    assert_close(h.cpu().numpy(), h64, "a is b")


def test_streams_run_independently():
    B, L, D = 1, 1 << 16, 64
    a, b = inputs.generate(B, L, D, seed=12, a_dist="u[0.9,1)", b_dist="n(0,1)")
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    streams = [torch.cuda.Stream() for _ in range(3)]
    outs = []
    for s in streams:
        with torch.cuda.stream(s):
            outs.append(lr.linrec_scan_f32_ex(a_d, b_d, stream=s, path="chunked", chunk_mode="lookback"))
    torch.cuda.synchronize()
    for h in outs:
        assert_close(h.cpu().numpy(), h64, "multi-stream")
    for s in streams:
        assert lr.linrec_stream_status(s) == lr.LINREC_OK


def test_concurrent_host_threads():
    """Calls from several host threads at once, each thread on its own stream and chunk mode: the
    library serialises its bookkeeping, each stream gets its own workspace, and every call returns
    the bits of the same call made alone."""
    import threading
    modes = ["own", "lookback", "twopass", "blocks", "regcarry", "chain", "speculative"]
    jobs = []
    for k, mode in enumerate(modes):
        a, b = inputs.generate(2, 20000, 96, seed=70 + k, a_dist="u[0.9,1)", b_dist="n(0,1)")
        opt = {"path": "regcarry"} if mode == "regcarry" else {"path": "chunked", "chunk_mode": mode}
        a_d, b_d = a.to(DEV), b.to(DEV)
        jobs.append((a_d, b_d, opt, run(a_d, b_d, **opt).clone()))
    errors = []

    def worker(k):
        try:
            a_d, b_d, opt, want = jobs[k]
            s = torch.cuda.Stream()
            h = torch.empty_like(a_d)
            for i in range(20):
                with torch.cuda.stream(s):
                    h.fill_(float("nan"))
                    lr.linrec_scan_f32_ex(a_d, b_d, h, stream=s, **opt)
                s.synchronize()
                if not torch.equal(h, want):
                    errors.append(f"thread {k} {opt} call {i}: bits differ")
                    return
            st = lr.linrec_stream_status(s)
            if st != lr.LINREC_OK:
                errors.append(f"thread {k}: status {lr.linrec_status_string(st)}")
        except Exception as e:          # reported below: a thread's exception would be lost
            errors.append(f"thread {k}: {e!r}")

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_modes_alternating_on_one_stream():
    """Two-pass, speculative and look-back calls take turns on one stream.  With a ~ U[0,1)
    the two-pass mode's tile products underflow to denormals whose bit patterns equal
    small look-back tags: the look-back must never see them.  The speculative and two-pass
    modes share the stream's array workspace."""
    a1, b1 = inputs.generate(1, 1 << 20, 64, seed=13, a_dist="u[0,1)", b_dist="n(0,1)")
    a2, b2 = inputs.generate(3, 1000, 260, seed=14, a_dist="u[0,1)", b_dist="n(0,1)")
    want1, _ = oracle.f64(a1, b1)
    want2, _ = oracle.f64(a2, b2)
    d1 = (a1.to(DEV), b1.to(DEV))
    d2 = (a2.to(DEV), b2.to(DEV))
    for k in range(3):
        h1 = run(*d1, path="chunked", chunk_mode="twopass")
        assert_close(h1.cpu().numpy(), want1, f"two-pass, call {k}")
        h1 = run(*d1, path="chunked", chunk_mode="speculative")
        assert_close(h1.cpu().numpy(), want1, f"speculative, call {k}")
        for mode in ("lookback", "twopass", "blocks", "chain", "lookback", "blocks", "chain"):
            h2 = run(*d2, path="chunked", chunk_mode=mode)
            assert_close(h2.cpu().numpy(), want2, f"{mode} after two-pass, call {k}")
    assert lr.linrec_stream_status() == lr.LINREC_OK


# ---------------------------------------------------------------------------
# speculative mode: G segments scanned from 0, then the unstored tiles from the true carry
# ---------------------------------------------------------------------------

SPEC = {"path": "chunked", "chunk_mode": "speculative"}


@pytest.mark.parametrize("case", [
    ((1, 131072, 64), "u[0.9,1)", 0),      # 1024-step segments: the product never reaches 0, all repaired
    ((3, 50000, 100), "u[0.5,1)", 25),     # ragged channel slice, 2000-step segments (a ragged last tile)
    ((2, 262144, 36), "u[0.9,1)", 256),    # 32 maps a lane in the repair's fold (two rounds); 1024 slices
    ((1, 65536, 32), "u[0,1)", 64),        # the product reaches 0 in the first tile
    ((1, 1 << 22, 32), "u[0.9,1)", 0),     # 256 segments of 16384 steps: a quarter of each repaired
], ids=lambda c: "x".join(map(str, c[0])) + f"-{c[1]}-G{c[2]}")
def test_speculative_mode(case):
    """Every element against the oracle, with and without a carried-in state, h_last, and the
    same bits on a second call (no atomics: the result is a fixed function of the input)."""
    (B, L, D), ad, G = case
    a, b = inputs.generate(B, L, D, seed=21 + L, a_dist=ad, b_dist="n(0,1)")
    h0 = torch.randn(B, D, generator=torch.Generator().manual_seed(22))
    opt = dict(SPEC, group=G) if G else SPEC
    p = lr.linrec_plan_f32(B, L, D, **opt)
    assert p["speculative"] == (G or p["speculative"]) and p["speculative"] >= 2 and L % p["speculative"] == 0
    a_d, b_d = a.to(DEV), b.to(DEV)
    h = run(a_d, b_d, **opt)
    assert_close(h.cpu().numpy(), oracle.f64(a, b)[0], f"speculative {case}")
    assert torch.equal(run(a_d, b_d, **opt), h)
    hc64, last64 = oracle.f64_carry(a, b, h0.numpy().astype(np.float64))
    last = torch.full((B, D), float("nan"), device=DEV)
    hc = run(a_d, b_d, h_init=h0.to(DEV), h_last=last, **opt)
    assert_close(hc.cpu().numpy(), hc64, f"speculative {case} carry")
    assert_close(last.cpu().numpy(), last64, f"speculative {case} h_last")
    assert lr.linrec_stream_status() == lr.LINREC_OK


def test_speculative_mode_closed_forms():
    """Closed forms the speculative mode must meet bit for bit.  a = 0: h = b, the product is
    0 after one step, so every later tile comes from the speculative launch.  a = 1 with
    integer b: h is the prefix sum, exact in fp32 below 2^24 in any order; the product never
    reaches 0, so every segment after the first is recomputed from the composed maps of the
    segments before it."""
    B, L, D = 2, 65536, 64
    b = torch.randint(-8, 9, (B, L, D), generator=torch.Generator().manual_seed(23)).float()
    b_d = b.to(DEV)
    for G in (0, 2, 64):
        opt = dict(SPEC, group=G) if G else SPEC
        h = run(torch.zeros_like(b_d), b_d, **opt)
        assert torch.equal(h, b_d), G
        h0 = torch.randint(-8, 9, (B, D), generator=torch.Generator().manual_seed(24)).float()
        last = torch.empty(B, D, device=DEV)
        h = run(torch.ones_like(b_d), b_d, h_init=h0.to(DEV), h_last=last, **opt)
        want = torch.cumsum(b.double(), dim=1) + h0.double()[:, None, :]
        assert torch.equal(h.cpu().double(), want), G
        assert torch.equal(last.cpu().double(), want[:, -1]), G
    assert lr.linrec_stream_status() == lr.LINREC_OK


def test_speculative_mode_propagates_nan():
    """a = 1/2: the slope product of a segment is 2^-128 after one tile and 0 after two, so the
    speculative launch stores the rest of each segment.  A NaN in a or b makes every later h of
    its channel NaN, in later segments too (0 * NaN is NaN), and a NaN slope turns a product that
    reached 0 into NaN.  Every element must be written: NaN exactly where the oracle has it, the
    rest within the bound."""
    B, L, D = 1, 4096, 32
    a = torch.full((B, L, D), 0.5)
    b = torch.randn(B, L, D, generator=torch.Generator().manual_seed(26))
    a[0, 1000, 5] = float("nan")      # first segment: carried into every later one
    b[0, 1500, 20] = float("nan")
    a[0, 3000, 9] = float("nan")      # after the second segment's product reached 0
    h64, _ = oracle.f64(a, b)
    assert np.isnan(h64[0, 1000:, 5]).all() and np.isnan(h64[0, 1500:, 20]).all()
    assert np.isnan(h64[0, 3000:, 9]).all() and np.isnan(h64).sum() == 3096 + 2596 + 1096
    a_d, b_d = a.to(DEV), b.to(DEV)
    for G in (2, 4):
        h = torch.full_like(a_d, 12345.0)
        lr.linrec_scan_f32_ex(a_d, b_d, h, group=G, **SPEC)
        torch.cuda.synchronize()
        got = h.cpu().numpy().astype(np.float64)
        assert not (got == 12345.0).any(), f"G = {G}: elements left unwritten"
        assert np.array_equal(np.isnan(got), np.isnan(h64)), f"G = {G}: NaN pattern differs"
        fin = ~np.isnan(h64)
        assert_close(got[fin], h64[fin], f"speculative, NaN inputs, G = {G}")
    assert lr.linrec_stream_status() == lr.LINREC_OK


def test_speculative_mode_is_the_default_for_long_chains():
    """The long workload (1, 1048576, 64) takes the speculative mode by default, and its result
    is the forced call's, bit for bit."""
    a, b = inputs.generate(1, 1 << 20, 64, seed=25, a_dist="u[0.9,1)", b_dist="n(0,1)")
    a_d, b_d = a.to(DEV), b.to(DEV)
    assert lr.linrec_plan_f32(1, 1 << 20, 64)["speculative"] == 128
    assert torch.equal(run(a_d, b_d), run(a_d, b_d, **SPEC))


# ---------------------------------------------------------------------------
# blocks mode: G consecutive tiles per block, one look-back per block
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("tile_d", [32, 64])
@pytest.mark.parametrize("group", [1, 2, 3, 8, 13])
def test_blocks_mode_every_group(tile_d, group):
    """Blocks of 1 to 13 tiles, with a last block of fewer tiles and a ragged last tile;
    repeated calls return the same bits (the block chain is evaluated in one fixed order)."""
    for (B, L, D) in [(2, 5000, 96), (1, 40001, 64), (3, 129, 260)]:
        a, b = inputs.generate(B, L, D, seed=23 + L + group, a_dist="u[0.9,1)", b_dist="n(0,1)")
        h64, _ = oracle.f64(a, b)
        a_d, b_d = a.to(DEV), b.to(DEV)
        opt = dict(path="chunked", chunk_mode="blocks", tile_d=tile_d, tile_t=128, group=group)
        plan = lr.linrec_plan_f32(B, L, D, **opt)
        assert plan["blocks"] == group and plan["lookback"] == 0 and plan["twopass"] == 0
        h = run(a_d, b_d, **opt)
        assert_close(h.cpu().numpy(), h64, f"blocks {(B, L, D)} {opt}")
        assert torch.equal(run(a_d, b_d, **opt), h), f"blocks {(B, L, D)} {opt}: bits changed"
    assert lr.linrec_stream_status() == lr.LINREC_OK


def test_blocks_timeout_reports_and_recovers():
    """Block 5 publishes nothing: block 6's look-back gives up after a bounded number of polls,
    the status word says so, and the next call on the stream is exact."""
    B, L, D = 1, 64 * 256, 64
    a, b = inputs.generate(B, L, D, seed=29, a_dist="u[0.5,1)", b_dist="n(0,1)")
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    opt = dict(path="chunked", chunk_mode="blocks", tile_d=64, tile_t=128, group=2)
    s = torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    with torch.cuda.stream(s):
        h = lr.linrec_scan_f32_ex(a_d, b_d, stream=s, spin_limit=2000, test_silent_tile=5 + 1, d_status=status,
                                  **opt)
    s.synchronize()
    assert int(status.item()) & (1 << lr.LINREC_ERR_LOOKBACK_TIMEOUT)
    hn = h.cpu().numpy()
    assert_close(hn[:, :6 * 256], h64[:, :6 * 256], "blocks before the timeout")
    assert np.isnan(hn[:, 6 * 256:]).any()
    assert lr.linrec_stream_status(s) == lr.LINREC_OK          # the failure went to d_status
    with torch.cuda.stream(s):
        h = lr.linrec_scan_f32_ex(a_d, b_d, stream=s, **opt)
    s.synchronize()
    assert_close(h.cpu().numpy(), h64, "blocks after recovery")
    assert lr.linrec_stream_status(s) == lr.LINREC_OK


# ---------------------------------------------------------------------------
# failure detection without a fault: a bounded look-back wait that runs out
# ---------------------------------------------------------------------------

def test_lookback_timeout_reports_and_recovers():
    B, L, D = 1, 64 * 64, 64
    a, b = inputs.generate(B, L, D, seed=13, a_dist="u[0.5,1)", b_dist="n(0,1)")
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    s = torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    with torch.cuda.stream(s):
        # tile 5 publishes nothing: tile 6 waits a bounded number of polls, then gives up
        h = lr.linrec_scan_f32_ex(a_d, b_d, stream=s, path="chunked", tile_d=64, tile_t=64, stages=2,
                                  chunk_mode="lookback", spin_limit=2000, test_silent_tile=5 + 1, d_status=status)
    s.synchronize()
    assert int(status.item()) & (1 << lr.LINREC_ERR_LOOKBACK_TIMEOUT)
    hn = h.cpu().numpy()
    # tiles before the silent one's successor are intact; the lost carry shows as NaN after it
    assert_close(hn[:, :6 * 64], h64[:, :6 * 64], "before the timeout")
    assert np.isnan(hn[:, 6 * 64:]).any()
    # the stream's own word: same failure through the plain status query
    with torch.cuda.stream(s):
        lr.linrec_scan_f32_ex(a_d, b_d, stream=s, path="chunked", tile_d=64, tile_t=64, stages=2,
                              chunk_mode="lookback", spin_limit=2000, test_silent_tile=5 + 1)
    assert lr.linrec_stream_status(s) == lr.LINREC_ERR_LOOKBACK_TIMEOUT
    assert lr.linrec_stream_status(s) == lr.LINREC_OK          # cleared
    # the context is healthy: the next call on the same stream is exact
    with torch.cuda.stream(s):
        h = lr.linrec_scan_f32_ex(a_d, b_d, stream=s, path="chunked", tile_d=64, tile_t=64, stages=2,
                                  chunk_mode="lookback")
    s.synchronize()
    assert_close(h.cpu().numpy(), h64, "after recovery")
    assert lr.linrec_stream_status(s) == lr.LINREC_OK


def test_chain_timeout_reports_and_recovers():
    """Chain mode: tile 5 publishes no map, so the resolver stops before it and the workers
    after it give up on their carries (bounded waits): the status word says so, the output
    before it is intact, NaN marks the lost carries, and the next call on the stream is exact."""
    B, L, D = 1, 64 * 128, 32
    a, b = inputs.generate(B, L, D, seed=17, a_dist="u[0.5,1)", b_dist="n(0,1)")
    h64, _ = oracle.f64(a, b)
    a_d, b_d = a.to(DEV), b.to(DEV)
    s = torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    opt = dict(path="chunked", chunk_mode="chain")
    with torch.cuda.stream(s):
        h = lr.linrec_scan_f32_ex(a_d, b_d, stream=s, spin_limit=2000, test_silent_tile=5 + 1, d_status=status,
                                  **opt)
    s.synchronize()
    assert int(status.item()) & (1 << lr.LINREC_ERR_LOOKBACK_TIMEOUT)
    hn = h.cpu().numpy()
    assert_close(hn[:, :6 * 128], h64[:, :6 * 128], "chain before the timeout")
    assert np.isnan(hn[:, 6 * 128:]).any()
    with torch.cuda.stream(s):
        lr.linrec_scan_f32_ex(a_d, b_d, stream=s, spin_limit=2000, test_silent_tile=5 + 1, **opt)
    assert lr.linrec_stream_status(s) == lr.LINREC_ERR_LOOKBACK_TIMEOUT
    with torch.cuda.stream(s):
        h = lr.linrec_scan_f32_ex(a_d, b_d, stream=s, **opt)
    s.synchronize()
    assert_close(h.cpu().numpy(), h64, "chain after recovery")
    assert lr.linrec_stream_status(s) == lr.LINREC_OK


@pytest.mark.parametrize("mode", ["lookback", "chain", "blocks"])
def test_epoch_wraps_around(mode):
    """The stream workspace's epoch word set just below the point where it wraps: consecutive
    launches still tag their words differently, so four calls in a row return slice-owner mode's
    bits (look-back, chain) or the same bits every time (blocks)."""
    B, L, D = 1, 1 << 19, 64
    a, b = inputs.generate(B, L, D, seed=65, a_dist="u[0.9,1)", b_dist="n(0,1)")
    a_d, b_d = a.to(DEV), b.to(DEV)
    s = torch.cuda.Stream()
    tile = {"tile_d": 32, "tile_t": 128} if mode != "blocks" else {}
    with torch.cuda.stream(s):
        first = lr.linrec_scan_f32_ex(a_d, b_d, stream=s, path="chunked", chunk_mode=mode, **tile)
        want = lr.linrec_scan_f32_ex(a_d, b_d, stream=s, path="chunked", chunk_mode="own", **tile) \
            if mode != "blocks" else first.clone()
    s.synchronize()
    lr.linrec_debug_set_epoch(0xFFFFFFFD, stream=s)
    h = torch.empty_like(a_d)
    for call in range(4):
        with torch.cuda.stream(s):
            h.fill_(float("nan"))
            lr.linrec_scan_f32_ex(a_d, b_d, h, stream=s, path="chunked", chunk_mode=mode, **tile)
        s.synchronize()
        assert torch.equal(h, want), f"{mode} call {call} across the epoch wrap"
    assert lr.linrec_stream_status(s) == lr.LINREC_OK


def test_workspace_bytes():
    """What a default call holds: the control block alone in slice-owner mode, plus three look-back
    words per tile and channel in look-back mode, plus the segments' maps in speculative mode, plus
    the tile maps and their scan's workspace in two-pass mode; nothing on the register path or for
    an empty shape."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert lr.linrec_workspace_bytes(32, 4096, 256) == 256
    assert lr.linrec_workspace_bytes(1, 64, 32) == 256               # one short slice: slice-owner mode
    assert lr.linrec_workspace_bytes(1, 4096, 32) == 256 + 3 * 32 * 32 * 8   # 32 chunks: look-back mode
    assert lr.linrec_workspace_bytes(256, 128, 4096) == 0
    assert lr.linrec_workspace_bytes(0, 64, 32) == 0
    assert lr.linrec_workspace_bytes(-1, 64, 32) == 0
    # speculative: the control block and the segments' maps
    p = lr.linrec_plan_f32(1, 1 << 20, 64, sm_count=sms)
    assert p["speculative"] == 128 and lr.linrec_workspace_bytes(1, 1 << 20, 64) == p["workspace_bytes"] == \
        256 + 2 * 256 * 32 * 4
    # two-pass, whose scan of the tile maps (1, 8192, 32) is two-pass too, and that scan's maps
    # (1, 64, 32) one short slice-owner call
    p = lr.linrec_plan_f32(1, 1 << 20, 32, sm_count=sms)
    inner = lr.linrec_plan_f32(1, p["chunks"], 32, sm_count=sms)
    inner2 = lr.linrec_plan_f32(1, inner["chunks"], 32, sm_count=sms)
    assert (p["twopass"], inner["twopass"], inner2["twopass"], inner2["lookback"]) == (1, 1, 0, 0)
    assert lr.linrec_workspace_bytes(1, 1 << 20, 32) == (p["workspace_bytes"] + inner["workspace_bytes"] +
                                                         inner2["workspace_bytes"])


def test_copy_kernel():
    x = torch.randn(1 << 20, device=DEV)
    y = torch.empty_like(x)
    lr.linrec_copy_f32(x, y)
    torch.cuda.synchronize()
    assert torch.equal(x, y)
    y2 = torch.empty(x.numel() + 1, device=DEV)[1:]
    lr.linrec_copy_f32(x[:-1], y2[:-1])
    torch.cuda.synchronize()
    assert torch.equal(x[:-1], y2[:-1])


def test_errors_reported():
    h64_err = max_errors(np.zeros(3), np.zeros(3))
    assert h64_err == (0.0, 0.0)
