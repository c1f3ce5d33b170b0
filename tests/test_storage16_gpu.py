"""16-bit storage (bfloat16 and binary16 words, fp32 arithmetic) against the oracle.

The oracle decodes the stored input words to their exact values, runs the
definition in fp64 and gives h64.  The kernels compute in fp32 (error e32 <=
1e-4 * (1 + |h64|), the bound the fp32 path meets) and round once to the
storage format, adding at most u * |h32| with u = 2^-8 (bfloat16) or 2^-11
(binary16).  So every element must satisfy

    |h16 - h64| <= u * |h64| + (1 + u) * 1e-4 * (1 + |h64|)

(u * |h32| <= u * (|h64| + e32)).  Where the fp32 value is exact (integer
closed forms) the stored word must equal the oracle's rounding of the exact
result, bit for bit.  And since the 16-bit kernels run the fp32 kernels'
arithmetic in the same order, their words must equal the fp32 path's result
on the decoded inputs, rounded once by the oracle, bit for bit.
"""
import numpy as np
import pytest
import torch

import linear_recurrence_scan_fp32_gb300 as lr
import oracle
from linear_recurrence_scan_fp32_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
KINDS = ("bf16", "f16")
UNIT = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}
SCAN = {"bf16": lr.linrec_scan_bf16_ex, "f16": lr.linrec_scan_f16_ex}
ONE = {"bf16": 0x3F80, "f16": 0x3C00}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)


def words(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close16(kind, h, h64, what):
    x = oracle.decode16(kind, words(h))
    u = UNIT[kind]
    bound = u * np.abs(h64) + (1 + u) * 1e-4 * (1 + np.abs(h64))
    bad = ~(np.abs(x - h64) <= bound)
    if bad.any():
        first = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of bound; first at {first}: "
                             f"got {x[first]}, want {h64[first]}")


def paths(D, aligned=True, B=1):
    out = [{"path": "regcarry"}]
    if aligned and D % 8 == 0:
        out += [{"path": "chunked", "chunk_mode": m} for m in ("own", "lookback", "twopass", "blocks")]
        if B * -(-D // 32) <= 64:          # chain mode serves few slices only
            out.append({"path": "chunked", "chunk_mode": "chain"})
    return out


def run(kind, a, b, **opt):
    h = SCAN[kind](a, b, **opt)
    torch.cuda.synchronize()
    return h


def draw16(kind, B, L, D, seed, a_dist="u[0,1)", b_dist="n(0,1)"):
    a, b = inputs.generate(B, L, D, seed=seed, a_dist=a_dist, b_dist=b_dist)
    return inputs.to_storage16(a, kind), inputs.to_storage16(b, kind)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("name", inputs.CONFIG_ORDER)
def test_workload_full_size(kind, name):
    w = inputs.WORKLOADS[name]
    a, b = inputs.generate_workload(w)
    a16, b16 = inputs.to_storage16(a, kind), inputs.to_storage16(b, kind)
    del a, b
    h64, _ = oracle.f64_16(kind, a16, b16)
    a_d, b_d = a16.to(DEV), b16.to(DEV)
    for opt in [{}] + paths(w.D, B=w.B):
        h = run(kind, a_d, b_d, **opt)
        assert_close16(kind, h, h64, f"{kind} {name} {opt}")
        del h
    assert lr.linrec_stream_status() == lr.LINREC_OK


@pytest.mark.parametrize("kind", KINDS)
def test_integer_closed_forms_bit_exact(kind):
    """a = 1 with integer b: prefix sums, exact in fp32, rounded once; a = 0: h = b."""
    B, L, D = 16, 128, 4096
    g = torch.Generator().manual_seed(80)
    bi = torch.randint(-8, 9, (B, L, D), generator=g).float()
    b16 = inputs.to_storage16(bi, kind)
    ones = torch.full((B, L, D), ONE[kind], dtype=torch.int16).view(inputs.STORAGE16[kind])
    want = oracle.encode16(kind, np.cumsum(bi.double().numpy(), axis=1))
    b_d, ones_d, zeros_d = b16.to(DEV), ones.to(DEV), torch.zeros_like(b16).to(DEV)
    for opt in [{}] + paths(D, B=B):
        assert np.array_equal(words(run(kind, ones_d, b_d, **opt)), want), f"a = 1 {opt}"
        assert torch.equal(run(kind, zeros_d, b_d, **opt), b_d), f"a = 0 {opt}"


@pytest.mark.parametrize("kind", KINDS)
def test_same_arithmetic_as_the_fp32_path(kind):
    """The 16-bit kernels' words are the fp32 path's results on the decoded inputs, rounded once."""
    B, L, D = 4, 5000, 128
    a16, b16 = draw16(kind, B, L, D, 81)
    a32 = torch.from_numpy(oracle.decode16(kind, words(a16)).astype(np.float32)).to(DEV)
    b32 = torch.from_numpy(oracle.decode16(kind, words(b16)).astype(np.float32)).to(DEV)
    a_d, b_d = a16.to(DEV), b16.to(DEV)
    # the same tile on both sides (the 16-bit default's 256 steps has no fp32 twin; the
    # ring depth does not change the arithmetic)
    # (blocks mode is compiled for the 256-step 16-bit tile only)
    same = {"tile_d": 32, "tile_t": 128, "stages": 3}
    # (chain mode's 16-bit variant has 256-step tiles only: no fp32 twin)
    opts = [dict(o, **same) if o.get("path") == "chunked" else o for o in paths(D, B=B)
            if o.get("chunk_mode") not in ("blocks", "chain")]
    for opt in opts + [{"path": "chunked", "tile_d": 64, "tile_t": 128, "stages": 2, "chunk_mode": "lookback"}]:
        h16 = run(kind, a_d, b_d, **opt)
        f32opt = dict(opt)
        if f32opt.get("path") == "regcarry":
            f32opt["vec"] = 4                       # the same per-channel fma chain at any width
        h32 = lr.linrec_scan_f32_ex(a32, b32, **f32opt)
        torch.cuda.synchronize()
        want = oracle.encode16(kind, h32.cpu().double().numpy())
        assert np.array_equal(words(h16), want), f"{kind} {opt}"


RAGGED = [(1, 1, 8), (1, 2, 8), (3, 31, 8), (2, 33, 40), (1, 65, 100), (3, 127, 136), (2, 129, 64),
          (1, 257, 8), (2, 1000, 264), (1, 4097, 16), (1, 5000, 72), (2, 77, 3), (2, 77, 6), (1, 300, 1)]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
def test_ragged_shapes(kind, shape):
    B, L, D = shape
    a16, b16 = draw16(kind, B, L, D, 82 + L + D, a_dist="u[0.5,1)")
    h64, _ = oracle.f64_16(kind, a16, b16)
    a_d, b_d = a16.to(DEV), b16.to(DEV)
    for opt in [{}] + paths(D, B=B):
        assert_close16(kind, run(kind, a_d, b_d, **opt), h64, f"{kind} {shape} {opt}")


@pytest.mark.parametrize("kind", KINDS)
def test_misaligned_pointers_take_the_register_path(kind):
    B, L, D = 2, 300, 64
    a16, b16 = draw16(kind, B, L, D, 83)
    h64, _ = oracle.f64_16(kind, a16, b16)
    n = B * L * D
    for shift in (1, 2, 4):                          # 2, 4 and 8 bytes off a 16-byte boundary
        buf_a = torch.empty(n + 8, dtype=a16.dtype, device=DEV)
        buf_b = torch.empty(n + 8, dtype=a16.dtype, device=DEV)
        buf_h = torch.empty(n + 8, dtype=a16.dtype, device=DEV)
        a_v = buf_a[shift:shift + n].view(B, L, D)
        b_v = buf_b[shift:shift + n].view(B, L, D)
        h_v = buf_h[shift:shift + n].view(B, L, D)
        a_v.copy_(a16.to(DEV))
        b_v.copy_(b16.to(DEV))
        run(kind, a_v, b_v, h=h_v)
        assert_close16(kind, h_v, h64, f"{kind} shifted by {shift}")
        with pytest.raises(lr.LinrecError):
            SCAN[kind](a_v, b_v, path="chunked")


# (tile_d, tile_t, stages, channels per thread, segments)
CHUNKED16 = [(32, 128, 3, 1, 8), (32, 128, 4, 1, 8), (32, 128, 6, 1, 8), (64, 128, 2, 1, 8), (64, 128, 3, 1, 8),
             (64, 64, 4, 1, 4), (32, 64, 6, 1, 4), (128, 64, 3, 1, 4), (32, 256, 2, 1, 8), (32, 256, 3, 1, 8),
             (32, 256, 2, 2, 16), (32, 256, 2, 2, 8), (32, 64, 6, 2, 8)]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("tile", CHUNKED16, ids=lambda t: f"d{t[0]}t{t[1]}s{t[2]}c{t[3]}g{t[4]}")
def test_every_chunked_variant_and_mode(kind, tile):
    td, tt, st, cpt, segs = tile
    B, L, D = 2, 3001, 200
    a16, b16 = draw16(kind, B, L, D, 84)
    h64, _ = oracle.f64_16(kind, a16, b16)
    a_d, b_d = a16.to(DEV), b16.to(DEV)
    var = dict(path="chunked", tile_d=td, tile_t=tt, stages=st, vec=cpt, segments=segs)
    assert lr.linrec_plan_16(B, L, D, **var)["threads"] == td // cpt * segs
    got = {}
    for mode in ("own", "lookback", "twopass"):
        h = run(kind, a_d, b_d, chunk_mode=mode, **var)
        assert_close16(kind, h, h64, f"{kind} {tile} {mode}")
        got[mode] = h
    assert torch.equal(got["own"], got["lookback"]), "slice-owner and look-back modes differ"
    again = run(kind, a_d, b_d, chunk_mode="lookback", **var)
    assert torch.equal(again, got["lookback"]), "not deterministic"
    assert lr.linrec_stream_status() == lr.LINREC_OK


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(2, 3001, 200), (1, 40000, 64), (1, 257, 8)], ids=lambda s: "x".join(map(str, s)))
def test_chain_mode_same_words_as_slice_owner(kind, shape):
    """Chain mode on 16-bit storage folds the tile maps in chunk order, as slice-owner mode does
    with the same tile (256 steps, two channels per thread, 8 segments): the same words."""
    B, L, D = shape
    a16, b16 = draw16(kind, B, L, D, 91 + L)
    h64, _ = oracle.f64_16(kind, a16, b16)
    a_d, b_d = a16.to(DEV), b16.to(DEV)
    tile = dict(path="chunked", tile_d=32, tile_t=256, vec=2, segments=8)
    h = run(kind, a_d, b_d, chunk_mode="chain", **tile)
    assert_close16(kind, h, h64, f"{kind} {shape} chain")
    assert torch.equal(h, run(kind, a_d, b_d, chunk_mode="own", stages=2, **tile))
    assert lr.linrec_stream_status() == lr.LINREC_OK


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(2, 3001, 200), (3, 1000, 264), (1, 257, 8)], ids=lambda s: "x".join(map(str, s)))
def test_two_channels_per_thread_same_bits(kind, shape):
    """One or two channels per thread, same tile and segments: the same fma sequence, the same words."""
    B, L, D = shape
    a16, b16 = draw16(kind, B, L, D, 87 + L, a_dist="u[0.5,1)")
    a_d, b_d = a16.to(DEV), b16.to(DEV)
    g = torch.Generator().manual_seed(88)
    h0 = torch.randn((B, D), generator=g).to(DEV)
    for mode in ("own", "lookback", "twopass"):
        outs = []
        for cpt in (1, 2):
            last = torch.full((B, D), float("nan"), device=DEV)
            h = run(kind, a_d, b_d, path="chunked", tile_d=32, tile_t=256, stages=2, segments=8, vec=cpt,
                    chunk_mode=mode, h_init=h0, h_last=last)
            outs.append((h, last))
        assert torch.equal(outs[0][0], outs[1][0]), f"{kind} {shape} {mode}: h differs"
        assert torch.equal(outs[0][1], outs[1][1]), f"{kind} {shape} {mode}: h_last differs"
    assert lr.linrec_stream_status() == lr.LINREC_OK


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(2, 33, 40), (3, 1000, 264), (1, 20000, 64), (2, 77, 6)],
                         ids=lambda s: "x".join(map(str, s)))
def test_carry_state_is_fp32(kind, shape):
    """h_init and h_last stay fp32 (B, D): h within the 16-bit bound, h_last within the fp32 one."""
    B, L, D = shape
    a16, b16 = draw16(kind, B, L, D, 85 + L, a_dist="u[0.5,1)")
    g = torch.Generator().manual_seed(86)
    h0 = torch.randn((B, D), generator=g)
    h64, last64 = oracle.f64_16(kind, a16, b16, h0.double().numpy())
    a_d, b_d, h0_d = a16.to(DEV), b16.to(DEV), h0.to(DEV)
    for opt in [{}] + paths(D, B=B):
        last = torch.full((B, D), float("nan"), device=DEV)
        h = run(kind, a_d, b_d, h_init=h0_d, h_last=last, **opt)
        assert_close16(kind, h, h64, f"{kind} {shape} {opt}")
        err = np.abs(last.cpu().double().numpy() - last64) - 1e-4 * (1 + np.abs(last64))
        assert (err <= 0).all(), f"{kind} {shape} {opt}: h_last off by {err.max()}"


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("group", [1, 3, 4, 7])
def test_blocks_mode_groups(kind, group):
    """Blocks of 1 to 7 tiles of 256 steps, a short last block, h_init / h_last in fp32;
    a second call gives the same words."""
    for (B, L, D) in [(1, 70001, 64), (2, 3001, 200)]:
        a16, b16 = draw16(kind, B, L, D, 89 + L + group, a_dist="u[0.9,1)")
        g = torch.Generator().manual_seed(90)
        h0 = torch.randn((B, D), generator=g)
        h64, last64 = oracle.f64_16(kind, a16, b16, h0.double().numpy())
        a_d, b_d, h0_d = a16.to(DEV), b16.to(DEV), h0.to(DEV)
        opt = dict(path="chunked", chunk_mode="blocks", group=group)
        assert lr.linrec_plan_16(B, L, D, **opt)["blocks"] == group
        last = torch.full((B, D), float("nan"), device=DEV)
        h = run(kind, a_d, b_d, h_init=h0_d, h_last=last, **opt)
        assert_close16(kind, h, h64, f"{kind} {(B, L, D)} {opt}")
        err = np.abs(last.cpu().double().numpy() - last64) - 1e-4 * (1 + np.abs(last64))
        assert (err <= 0).all(), f"{kind} {(B, L, D)} {opt}: h_last off by {err.max()}"
        assert torch.equal(run(kind, a_d, b_d, h_init=h0_d, **opt), h), f"{kind} {opt}: words changed"
    assert lr.linrec_stream_status() == lr.LINREC_OK
