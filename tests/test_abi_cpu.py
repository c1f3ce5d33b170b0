"""The C ABI without a GPU: the library loads, exports what include/linrec.h
declares, and its host logic (argument checks, dispatcher) behaves.  No call
here reaches a CUDA API: every one returns before touching a device."""
import ctypes
import glob
import os
import re

import pytest

import linear_recurrence_scan_fp32_gb300 as lr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    try:
        return lr.lib()
    except lr.LinrecError:
        from linear_recurrence_scan_fp32_gb300 import _build
        _build.build()
        return lr.lib()


def declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(linrec_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["linrec_scan_f32", "linrec_scan_f32_ex", "linrec_plan_f32", "linrec_stream_status",
              "linrec_copy_f32", "linrec_status_string", "linrec_version", "linrec_workspace_bytes"]:
        assert n in names


def test_normal_build_has_no_index_checks(L):
    # the index checks exist only in the -DLINREC_DEBUG build; here nothing is counted (no CUDA call)
    assert lr.linrec_debug_checks() is False
    assert lr.linrec_debug_bad_accesses() == (0, -1)
    with pytest.raises(lr.LinrecError):
        lr.linrec_debug_bad_accesses(output_cap_bytes=-1)


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_status_strings(L):
    for code in range(8):
        s = lr.linrec_status_string(code)
        assert s.startswith("LINREC_")
    assert "unknown" in lr.linrec_status_string(99)
    assert lr.linrec_version() >= 100


def _scan(L, a, b, h, B, Lx, D):
    return L.linrec_scan_f32(a, b, h, B, Lx, D, None)


def test_argument_checks_return_before_any_launch(L):
    # negative sizes
    assert _scan(L, 16, 4096, 8192, -1, 4, 4) == lr.LINREC_ERR_INVALID_VALUE
    assert _scan(L, 16, 4096, 8192, 1, -4, 4) == lr.LINREC_ERR_INVALID_VALUE
    # empty problems succeed with no launch, NULL pointers allowed
    assert _scan(L, None, None, None, 0, 5, 5) == lr.LINREC_OK
    assert _scan(L, None, None, None, 5, 0, 5) == lr.LINREC_OK
    assert _scan(L, None, None, None, 5, 5, 0) == lr.LINREC_OK
    # NULL with a non-zero size
    assert _scan(L, None, 4096, 1 << 30, 1, 4, 4) == lr.LINREC_ERR_INVALID_VALUE
    assert _scan(L, 4096, 4096, None, 1, 4, 4) == lr.LINREC_ERR_INVALID_VALUE
    # B*L*D*4 overflowing int64
    assert _scan(L, 16, 1 << 40, 1 << 41, 1 << 20, 1 << 20, 1 << 22) == lr.LINREC_ERR_INVALID_VALUE
    # h overlapping a or b (fake addresses: rejected before any device access)
    base = 1 << 32
    assert _scan(L, base, base + (1 << 20), base + 8, 1, 4, 4) == lr.LINREC_ERR_ALIAS
    assert _scan(L, base + (1 << 20), base, base + 60, 1, 4, 4) == lr.LINREC_ERR_ALIAS
    # a and b may be the same buffer; h right after them does not overlap
    n = 1 * 4 * 4
    assert L.linrec_copy_f32(base, base + 8, n, None) == lr.LINREC_ERR_ALIAS
    assert L.linrec_copy_f32(base, base + 8, -1, None) == lr.LINREC_ERR_INVALID_VALUE


def test_plan_paths():
    # very many channels (fp32 forward): the register path, 16 steps ahead for short L
    p = lr.linrec_plan_f32(256, 128, 4096, sm_count=152)
    assert p["path_name"] == "regcarry" and (p["vec"], p["prefetch"]) == (4, 16)
    p = lr.linrec_plan_f32(64, 1024, 4096, sm_count=152)
    assert p["path_name"] == "regcarry" and p["prefetch"] == 8
    # ... but not below 96 four-channel threads per SM, nor for the gradient
    p = lr.linrec_plan_f32(8, 4096, 4096, sm_count=152)
    assert p["path_name"] == "chunked" and p["lookback"] == 0
    assert lr.linrec_plan_f32_backward(256, 128, 4096, sm_count=152)["path_name"] == "chunked"
    # 16-bit storage: the register path only below 256 steps (eight channels per thread)
    p = lr.linrec_plan_16(256, 128, 4096, sm_count=152)
    assert p["path_name"] == "regcarry" and (p["vec"], p["prefetch"]) == (8, 16)
    assert lr.linrec_plan_16(64, 512, 4096, sm_count=152)["path_name"] == "chunked"
    assert lr.linrec_plan_16(8, 128, 4096, sm_count=152)["path_name"] == "chunked"
    # many channels, fewer of them: the chunked kernel, each CTA owning whole slices
    p = lr.linrec_plan_f32(32, 4096, 256, sm_count=152)
    assert p["path_name"] == "chunked" and p["lookback"] == 0
    # the register path when forced: 16-byte vectors, a grid covering every group
    p = lr.linrec_plan_f32(256, 128, 4096, path="regcarry")
    assert p["path_name"] == "regcarry" and p["vec"] == 4
    assert p["grid"] * p["threads"] >= 256 * 4096 // 4
    # few channel groups: narrower blocks so that every SM gets some
    p = lr.linrec_plan_f32(64, 2048, 1024, path="regcarry", sm_count=152)
    assert p["grid"] >= 2 * 152 or p["threads"] == 32
    # few channels, long sequence: the chunked speculative path (segments of 8192 steps, a map
    # per segment and channel) ...
    p = lr.linrec_plan_f32(1, 1 << 20, 64, sm_count=152)
    assert p["path_name"] == "chunked" and p["speculative"] == 128 and p["twopass"] == 0 and p["lookback"] == 0
    assert (p["tile_d"], p["tile_t"], p["stages"], p["chunks"], p["grid"]) == (32, 128, 2, 64, 256)
    assert p["n_tiles"] == 256 * 64 and p["workspace_bytes"] == 256 + 2 * 256 * 32 * 4
    # ... or, where its segments would be shorter, the two-pass path (per-tile A, B, H arrays)
    p = lr.linrec_plan_f32(1, 1 << 20, 32, sm_count=152)
    assert p["path_name"] == "chunked" and p["twopass"] == 1 and p["lookback"] == 0 and p["speculative"] == 0
    assert p["n_tiles"] == p["chunks"] * ((32 + p["tile_d"] - 1) // p["tile_d"])
    assert p["chunks"] == -(-(1 << 20) // p["tile_t"])
    assert p["workspace_bytes"] == 256 + 4 * (3 * p["n_tiles"] + 32 // p["tile_d"]) * p["tile_d"]
    # few channels, short sequence: look-back
    p = lr.linrec_plan_f32(1, 4096, 64)
    assert p["lookback"] == 1 and p["twopass"] == 0
    assert p["workspace_bytes"] >= 3 * 8 * p["n_tiles"] * p["tile_d"]
    # the pages' shape
    p = lr.linrec_plan_f32(32, 4096, 256)
    assert p["path_name"] in ("chunked", "regcarry")


def test_plan_alignment_and_odd_d():
    # D % 4 != 0 or pointers not 16-byte aligned: TMA is not allowed, scalar or pair loads instead
    assert lr.linrec_plan_f32(1, 1 << 20, 63)["path_name"] == "regcarry"
    assert lr.linrec_plan_f32(1, 1 << 20, 63)["vec"] == 1
    assert lr.linrec_plan_f32(1, 1 << 20, 62, align_bytes=8)["vec"] == 2
    assert lr.linrec_plan_f32(1, 1 << 20, 64, align_bytes=8)["path_name"] == "regcarry"
    assert lr.linrec_plan_f32(1, 1 << 20, 64, align_bytes=4)["vec"] == 1
    with pytest.raises(lr.LinrecError) as e:
        lr.linrec_plan_f32(1, 1000, 63, path="chunked")
    assert e.value.code == lr.LINREC_ERR_INVALID_VALUE
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(1, 1000, 64, align_bytes=4, path="chunked")
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(1, 1000, 64, path="regcarry", vec=4, align_bytes=8)


def test_plan_forced_options():
    p = lr.linrec_plan_f32(32, 4096, 256, path="chunked", tile_d=64, tile_t=64, stages=3)
    assert (p["tile_d"], p["tile_t"], p["stages"]) == (64, 64, 3)
    assert p["threads"] == p["tile_d"] * p["segments"]
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(32, 4096, 256, path="chunked", tile_d=48, tile_t=64)
    p = lr.linrec_plan_f32(32, 4096, 256, path="regcarry", vec=2, prefetch=4)
    assert (p["vec"], p["prefetch"]) == (2, 4)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(32, 4096, 256, path="regcarry", prefetch=5)


def _units(p, B, D):
    # slice-owner mode: one unit per channel slice; look-back and two-pass modes: one per tile;
    # speculative mode: one per channel slice of every segment
    if p["speculative"]:
        return B * p["speculative"] * -(-D // p["tile_d"])
    return p["n_tiles"] if (p["lookback"] or p["twopass"]) else B * -(-D // p["tile_d"])


def test_plan_grid_bounds():
    # grid never exceeds the work units nor SMs x resident CTAs
    for (B, L, D) in [(1, 64, 32), (1, 1 << 20, 64), (32, 4096, 256), (3, 5, 8), (256, 128, 4096)]:
        p = lr.linrec_plan_f32(B, L, D, path="chunked", sm_count=152, resident_ctas=2)
        assert 1 <= p["grid"] <= min(_units(p, B, D), 152 * 2)
    for mode in ("own", "lookback"):
        p = lr.linrec_plan_f32(32, 4096, 256, path="chunked", sm_count=152, resident_ctas=3, chunk_mode=mode)
        assert p["lookback"] == (mode == "lookback")
        assert p["grid"] == min(_units(p, 32, 256), 152 * 3)
        # the options' cap lowers the resident count
        p = lr.linrec_plan_f32(32, 4096, 256, path="chunked", sm_count=152, resident_ctas=3, ctas_per_sm=1,
                               chunk_mode=mode)
        assert p["grid"] == min(_units(p, 32, 256), 152)


def test_plan_wide_slices():
    # fp32, L >= 256: the widest of 256 or 128 channels whose slices split evenly over at
    # least 84 % of the SMs takes slice-owner mode ahead of the register path
    cases = [((64, 2048, 1024), (256, 32, 128)), ((128, 1024, 1024), (256, 32, 128)),
             ((8, 4096, 4096), (256, 32, 128)), ((64, 4096, 256), (128, 64, 128)),
             ((256, 1024, 256), (256, 32, 128)), ((19, 4096, 1024), (256, 32, 76))]
    for shape, (td, tt, grid) in cases:
        p = lr.linrec_plan_f32(*shape, sm_count=152, resident_ctas=1)
        slices = shape[0] * -(-shape[2] // td)
        if grid * 100 < 84 * 152:                      # no even split: not the wide tile
            assert p["tile_d"] != td or p["path_name"] != "chunked", shape
            continue
        assert (p["path_name"], p["tile_d"], p["tile_t"], p["lookback"], p["twopass"]) == ("chunked", td, tt, 0, 0)
        assert p["grid"] == grid and slices % grid == 0, shape
    p = lr.linrec_plan_f32(32, 512, 4096, sm_count=152, resident_ctas=1)              # 512 slices, 4 each
    assert (p["path_name"], p["tile_d"], p["grid"]) == ("chunked", 256, 128)
    # not without an even split, for 128 steps, 16-bit storage or a chosen tile or mode
    assert lr.linrec_plan_f32(64, 512, 4096, sm_count=152)["path_name"] == "regcarry"
    assert lr.linrec_plan_f32(32, 128, 4096, sm_count=152)["path_name"] == "regcarry"
    # 64-channel slices, forward only, from 4096 steps: the pages shape splits into 128 of them
    p = lr.linrec_plan_f32(32, 4096, 256, sm_count=152, resident_ctas=2)
    assert (p["tile_d"], p["tile_t"], p["threads"], p["grid"]) == (64, 128, 512, 128)
    assert lr.linrec_plan_f32(32, 2048, 256, sm_count=152, resident_ctas=2)["tile_d"] == 32
    assert lr.linrec_plan_f32_backward(32, 4096, 256, sm_count=152, resident_ctas=2)["tile_d"] == 32
    # never a tile wider than D (its boxes would be mostly padding)
    for shape in [(128, 1024, 64), (256, 1024, 100), (512, 512, 128)]:
        p = lr.linrec_plan_f32(*shape, sm_count=152, resident_ctas=2)
        assert p["path_name"] != "chunked" or p["tile_d"] <= shape[2], shape
    assert lr.linrec_plan_16(64, 2048, 1024, sm_count=152)["tile_d"] == 32
    p = lr.linrec_plan_f32_backward(128, 1024, 1024, sm_count=152, resident_ctas=1)    # the gradient too
    assert (p["tile_d"], p["tile_t"], p["grid"]) == (256, 32, 128)
    assert lr.linrec_plan_f32(64, 2048, 1024, sm_count=152, path="chunked", chunk_mode="own")["tile_d"] == 32
    assert lr.linrec_plan_f32(64, 2048, 1024, sm_count=152, path="regcarry")["path_name"] == "regcarry"


def test_plan_segmented_register_path():
    # few channel groups on the register path (odd D, misaligned pointers): the time axis in
    # segments of at least 64 steps, at most 256 of them; 2 floats per segment and channel
    p = lr.linrec_plan_f32(7, 3000, 777, sm_count=152)
    assert (p["path_name"], p["vec"], p["twopass"], p["segments"]) == ("regcarry", 1, 1, 22)
    assert p["workspace_bytes"] == 2 * 22 * 7 * 777 * 4
    assert p["grid"] == -(-7 * 777 * 22 // 256)
    assert lr.linrec_plan_f32(1, 1000000, 3, sm_count=152)["segments"] == 256
    assert lr.linrec_plan_f32(1, 100, 3, sm_count=152)["twopass"] == 0          # under 128 steps: one pass
    assert lr.linrec_plan_f32(256, 128, 4096, sm_count=152)["twopass"] == 0     # many channels: one pass
    assert lr.linrec_plan_f32_backward(7, 3000, 777, sm_count=152)["twopass"] == 0


def test_plan_slice_owner_thresholds():
    # fp32 forward: slice-owner mode from 84 % of the SM count in slices (128 on 152 SMs)
    p = lr.linrec_plan_f32(16, 4096, 256, sm_count=152, resident_ctas=2)
    assert (p["lookback"], p["twopass"], p["tile_d"], p["grid"]) == (0, 0, 32, 128)
    p = lr.linrec_plan_f32(15, 4096, 256, sm_count=152, resident_ctas=2)                 # 120 slices
    assert p["lookback"] or p["twopass"]
    # ... and at any slice count when every slice has at most 4 chunks of 128 steps
    for (B, L, D) in [(1, 64, 32), (1, 512, 32), (4, 128, 64), (127, 512, 32), (15, 300, 256)]:
        p = lr.linrec_plan_f32(B, L, D, sm_count=152)
        assert (p["path_name"], p["lookback"], p["twopass"], p["tile_d"], p["tile_t"]) == ("chunked", 0, 0, 32, 128), \
            (B, L, D)
        assert p["grid"] == B * -(-D // 32) and p["workspace_bytes"] == 256
    for (B, L, D) in [(1, 513, 32), (16, 1024, 32), (1, 4096, 64)]:              # 5 chunks and more
        assert lr.linrec_plan_f32(B, L, D, sm_count=152)["lookback"] == 1, (B, L, D)
    assert lr.linrec_plan_16(4, 512, 64, sm_count=152)["lookback"] == 1          # fp32 forward only
    assert lr.linrec_plan_f32_backward(4, 512, 64, sm_count=152)["lookback"] == 1
    # the 16-bit forms and the gradient keep one slice per SM as the threshold
    assert lr.linrec_plan_16(16, 4096, 256, sm_count=152)["lookback"] == 1
    assert lr.linrec_plan_f32_backward(16, 4096, 256, sm_count=152)["lookback"] == 1
    # slices just past one round of {32, 128} CTAs (304): 64-step tiles, 4-deep up to 1.2 rounds,
    # 3-deep up to 1.33; beyond that the {32, 128} tile again
    for (B, D, want) in [(40, 256, (64, 4)), (44, 256, (64, 4)), (48, 256, (64, 3)), (12, 1024, (64, 3)),
                         (56, 256, (128, 2))]:
        p = lr.linrec_plan_f32(B, 4096, D, sm_count=152)
        assert (p["tile_d"], p["tile_t"], p["stages"]) == (32,) + want, (B, D)
    # 128 to 152 slices of 64 channels: one 64-channel slice per CTA instead
    for (B, D) in [(32, 256), (36, 256), (38, 256)]:
        p = lr.linrec_plan_f32(B, 4096, D, sm_count=152)
        assert (p["tile_d"], p["tile_t"], p["grid"]) == (64, 128, B * D // 64), (B, D)
    assert lr.linrec_plan_f32(32, 2048, 256, sm_count=152)["tile_d"] == 32       # shorter: 32 channels
    p = lr.linrec_plan_f32(48, 4096, 256, sm_count=152, tile_d=32, tile_t=128)             # a chosen tile stays
    assert (p["tile_t"], p["stages"]) == (128, 2)


def test_plan_slices_spread_evenly():
    # fp32 slice-owner mode: the busiest CTA owns ceil(slices / resident) slices.  When fewer than
    # half the resident CTAs would own a slice in that last round, the grid is the fewest CTAs that
    # keep the same maximum (counts then differ by one at most); otherwise every resident CTA runs
    for (B, D, want) in [(8, 4096, 256), (64, 1024, 304), (32, 256, 256), (48, 256, 192), (40, 512, 214),
                         (19, 256, 152), (1000, 32, 250), (12, 1024, 192), (32, 2048, 304)]:
        p = lr.linrec_plan_f32(B, 2048, D, path="chunked", chunk_mode="own", sm_count=152, resident_ctas=2)
        slices = B * D // 32
        waves = -(-slices // 304)
        assert p["grid"] == want and -(-slices // p["grid"]) == waves, (B, D, p["grid"])
    # the gradient spreads the same way; 16-bit storage keeps every resident CTA
    assert lr.linrec_plan_f32_backward(48, 4096, 256, sm_count=152, resident_ctas=2)["grid"] == 192
    assert lr.linrec_plan_16(8, 4096, 4096, sm_count=152, resident_ctas=2)["grid"] == 304


def test_plan_chunk_modes():
    # many slices: each CTA owns whole slices, no look-back words needed
    p = lr.linrec_plan_f32(32, 4096, 256, path="chunked", sm_count=152)
    assert p["lookback"] == 0 and p["workspace_bytes"] == 256
    # one long slice: look-back mode with words for every tile when asked for it
    p = lr.linrec_plan_f32(1, 1 << 20, 64, path="chunked", sm_count=152, chunk_mode="lookback")
    assert p["lookback"] == 1 and p["workspace_bytes"] == 256 + 24 * p["n_tiles"] * p["tile_d"]
    # ... and the two-pass mode when asked for it
    p = lr.linrec_plan_f32(1, 1 << 20, 64, path="chunked", sm_count=152, chunk_mode="twopass")
    assert p["twopass"] == 1 and p["workspace_bytes"] == 256 + 4 * (3 * p["n_tiles"] + 64 // p["tile_d"]) * p["tile_d"]
    # the gradient takes the two-pass mode too, by default for few long slices
    p = lr.linrec_plan_f32_backward(1, 1 << 20, 64, sm_count=152)
    assert p["twopass"] == 1 and p["lookback"] == 0
    assert p["workspace_bytes"] == 256 + 4 * (3 * p["n_tiles"] + 64 // p["tile_d"]) * p["tile_d"]
    assert lr.linrec_plan_f32_backward(1, 1 << 20, 64, chunk_mode="lookback")["lookback"] == 1
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(1, 1000, 64, path="chunked", chunk_mode=7)
    # chain mode: one cooperative launch of every resident CTA (resolvers first, then workers),
    # its own tile, three look-back words per tile and channel; forward only
    p = lr.linrec_plan_f32(1, 1 << 20, 64, path="chunked", chunk_mode="chain", sm_count=152, resident_ctas=2)
    assert (p["chain"], p["lookback"], p["twopass"], p["blocks"]) == (1, 0, 0, 0)
    assert (p["tile_d"], p["tile_t"], p["stages"], p["grid"]) == (32, 256, 3, 304)     # 256 steps: long
    p = lr.linrec_plan_f32(1, 8192, 64, path="chunked", chunk_mode="chain", sm_count=152, resident_ctas=2)
    assert (p["tile_t"], p["threads"]) == (128, 256)                                      # 128 below 32768
    assert p["workspace_bytes"] == 256 + 24 * p["n_tiles"] * p["tile_d"]
    p = lr.linrec_plan_f32(1, 200, 32, path="chunked", chunk_mode="chain", sm_count=152, resident_ctas=2)
    assert p["n_tiles"] == 2 and 2 < p["grid"] <= 2 + 8      # no more workers than tiles
    q = lr.linrec_plan_16(1, 1 << 20, 64, path="chunked", chunk_mode="chain", sm_count=152, resident_ctas=2)
    assert (q["chain"], q["tile_t"], q["vec"], q["segments"]) == (1, 256, 2, 8)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32_backward(1, 1 << 20, 64, chunk_mode="chain")
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(1, 1 << 20, 64, chunk_mode="chain", tile_t=64)     # not compiled for chain mode
    # blocks mode: one launch, `group` tiles per block (1024 steps by default), three look-back
    # words per block and channel; forward only; group is taken by blocks mode alone
    p = lr.linrec_plan_f32(1, 1 << 20, 64, path="chunked", chunk_mode="blocks", sm_count=152, resident_ctas=2)
    assert (p["blocks"], p["lookback"], p["twopass"], p["tile_t"], p["grid"]) == (8, 0, 0, 128, 304)
    n_blocks = 2 * (8192 // 8)
    assert p["workspace_bytes"] == 256 + 3 * n_blocks * 32 * 8
    p = lr.linrec_plan_f32(1, 1000, 64, chunk_mode="blocks", group=3, tile_d=64)
    assert (p["blocks"], p["tile_d"], p["chunks"], p["grid"]) == (3, 64, 8, 3)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32_backward(1, 1 << 20, 64, chunk_mode="blocks")
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(1, 1 << 20, 64, chunk_mode="lookback", group=2)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(1, 1 << 20, 64, chunk_mode="blocks", group=-1)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(1, 1 << 20, 64, chunk_mode="blocks", tile_t=64)   # not compiled for blocks
    assert lr.linrec_plan_16(1, 1 << 20, 64, chunk_mode="blocks")["blocks"] == 4
    p = lr.linrec_plan_16(1, 64, 32, chunk_mode="blocks")            # short: still the 256-step tile
    assert (p["tile_t"], p["blocks"], p["grid"]) == (256, 4, 1)


def test_carry_state_overlap_checks(L):
    # fake, never-dereferenced addresses: every check runs before any device access
    B, Lx, D = 2, 100, 8
    n = B * Lx * D * 4
    a, b, h = 1 << 36, (1 << 36) + 2 * n, (1 << 36) + 4 * n
    s1 = h + n                                  # right after h: no overlap
    s2 = s1 + 1024
    vp = ctypes.c_void_p
    f = L.linrec_scan_f32_carry
    f.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vp, vp]
    f.restype = ctypes.c_int
    assert f(a, b, h, B, Lx, D, h + 4, None, None) == lr.LINREC_ERR_ALIAS        # h_init inside h
    assert f(a, b, h, B, Lx, D, None, a + n - 4, None) == lr.LINREC_ERR_ALIAS    # h_last ends a
    assert f(a, b, h, B, Lx, D, s1, s1 + 8, None) == lr.LINREC_ERR_ALIAS         # partial overlap
    assert f(a, b, h, -1, Lx, D, s1, s1, None) == lr.LINREC_ERR_INVALID_VALUE
    assert f(None, None, None, 0, Lx, D, s1, s2, None) == lr.LINREC_OK


def test_plan_16bit_storage():
    # 16-byte aligned with D % 8 == 0: the chunked kernel; 256-step tiles (the bytes of a
    # 128-step fp32 tile) with a 2-deep ring, 64-step tiles with a 6-deep ring below 256 steps
    p = lr.linrec_plan_16(32, 4096, 256, sm_count=152)
    assert p["path_name"] == "chunked" and p["lookback"] == 0
    assert (p["tile_d"], p["tile_t"], p["stages"]) == (32, 256, 2)
    # channels per thread and segments of the 256-step tile: two channels per thread; 8 segments
    # (128 threads) when the slices fill one wave of three CTAs per SM, and in two-pass mode
    assert (p["vec"], p["segments"], p["threads"]) == (2, 8, 128)                       # 256 slices
    p = lr.linrec_plan_16(19, 4096, 256, sm_count=152)                                   # 152 slices
    assert (p["lookback"], p["vec"], p["segments"], p["threads"]) == (0, 2, 16, 256)
    p = lr.linrec_plan_16(57, 4096, 256, sm_count=152)                                   # 456 slices
    assert (p["vec"], p["segments"]) == (2, 8)
    p = lr.linrec_plan_16(64, 2048, 1024, sm_count=152)                                  # 2048 slices
    assert (p["vec"], p["segments"], p["threads"]) == (2, 16, 256)
    p = lr.linrec_plan_16(1, 1 << 20, 64, sm_count=152)
    assert (p["twopass"], p["vec"], p["segments"]) == (1, 2, 8)
    p = lr.linrec_plan_16(4, 8192, 256, sm_count=152)                                    # look-back
    assert (p["lookback"], p["vec"], p["segments"]) == (1, 1, 8)
    # an explicit choice is kept, and other tiles keep their first variant
    p = lr.linrec_plan_16(32, 4096, 256, sm_count=152, vec=1)
    assert (p["vec"], p["segments"]) == (1, 8)
    p = lr.linrec_plan_16(32, 4096, 256, sm_count=152, segments=16)
    assert (p["vec"], p["segments"]) == (2, 16)
    p = lr.linrec_plan_16(32, 4096, 256, sm_count=152, tile_d=32, tile_t=256, stages=3)
    assert (p["vec"], p["segments"]) == (1, 8)
    p = lr.linrec_plan_16(256, 128, 4096, sm_count=152, path="chunked")
    assert (p["tile_d"], p["tile_t"], p["stages"], p["lookback"]) == (32, 64, 6, 0)
    # few long slices: two-pass, whose aggregates are fp32 whatever the storage
    p = lr.linrec_plan_16(1, 1 << 20, 64)
    assert p["twopass"] == 1
    assert p["workspace_bytes"] == 256 + 4 * (3 * p["n_tiles"] + 64 // p["tile_d"]) * p["tile_d"]
    # D % 8 != 0 or fewer than 16 bytes of alignment: the register path, widest vector allowed
    assert lr.linrec_plan_16(2, 77, 36)["path_name"] == "regcarry"
    assert lr.linrec_plan_16(2, 77, 36)["vec"] == 4
    assert lr.linrec_plan_16(2, 77, 40, align_bytes=16)["path_name"] == "chunked"
    assert lr.linrec_plan_16(2, 77, 40, align_bytes=8)["vec"] == 4
    assert lr.linrec_plan_16(2, 77, 40, align_bytes=4)["vec"] == 2
    assert lr.linrec_plan_16(2, 77, 40, align_bytes=2)["vec"] == 1
    assert lr.linrec_plan_16(2, 77, 7, align_bytes=16)["vec"] == 1
    assert lr.linrec_plan_16(256, 128, 4096, path="regcarry")["vec"] == 8
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_16(2, 77, 36, path="chunked")               # D * 2 bytes not a multiple of 16
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_16(2, 77, 40, path="regcarry", vec=8, align_bytes=8)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_16(32, 4096, 256, path="chunked", tile_d=32, tile_t=32)   # no such 16-bit variant
    # every variant the 16-bit table reports by default exists and is shaped like the fp32 ones
    for mode in ("own", "lookback", "twopass"):
        p = lr.linrec_plan_16(4, 5000, 128, path="chunked", chunk_mode=mode)
        assert p["threads"] == p["tile_d"] // p["vec"] * p["segments"] and p["tile_t"] % p["segments"] == 0


def test_plan_chunked_channels_per_thread():
    # vec on the chunked path: adjacent channels per thread; segments picks among variants of a tile
    p = lr.linrec_plan_16(32, 4096, 256, path="chunked", tile_d=32, tile_t=256, stages=2, vec=2, segments=8)
    assert (p["vec"], p["segments"], p["threads"]) == (2, 8, 128)
    p = lr.linrec_plan_16(32, 4096, 256, path="chunked", tile_d=32, tile_t=256, stages=2, vec=2, segments=16)
    assert (p["vec"], p["segments"], p["threads"]) == (2, 16, 256)
    p = lr.linrec_plan_16(32, 4096, 256, path="chunked", tile_d=32, tile_t=256, stages=2, vec=1)
    assert (p["vec"], p["segments"], p["threads"]) == (1, 8, 256)
    assert lr.linrec_plan_f32(32, 4096, 256, path="chunked")["vec"] == 1
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(32, 4096, 256, path="chunked", vec=2)          # fp32 keeps one channel per thread
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_16(32, 4096, 256, path="chunked", tile_d=32, tile_t=256, vec=2, segments=4)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32_backward(32, 4096, 256, path="chunked", vec=2)


def test_16bit_argument_checks_count_two_bytes(L):
    # fake, never-dereferenced addresses: the checks run before any device access
    B, Lx, D = 1, 4, 8
    n2 = B * Lx * D * 2
    base = 1 << 36
    for f in (L.linrec_scan_bf16, L.linrec_scan_f16):
        f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
        f.restype = ctypes.c_int
        assert f(base, base + 4 * n2, base + n2 - 2, B, Lx, D, None) == lr.LINREC_ERR_ALIAS   # h's first element in a
        assert f(base, base + 4 * n2, base + 5 * n2 - 2, B, Lx, D, None) == lr.LINREC_ERR_ALIAS
        assert f(None, base, base + 4 * n2, B, Lx, D, None) == lr.LINREC_ERR_INVALID_VALUE
        assert f(base, base, base, -1, Lx, D, None) == lr.LINREC_ERR_INVALID_VALUE
        assert f(None, None, None, 0, Lx, D, None) == lr.LINREC_OK


def test_plan_bdl_layout():
    # many rows: one pass, a warp per row, 16-byte vectors when L and the pointers allow
    p = lr.linrec_plan_bdl(32, 256, 4096, sm_count=152)
    assert (p["path_name"], p["vec"], p["twopass"], p["chunks"], p["n_tiles"]) == ("rows", 4, 0, 1, 32 * 256)
    assert p["grid"] * p["threads"] >= 32 * p["n_tiles"] and p["workspace_bytes"] == 0
    # few long rows: two passes over segments that are whole chunks, about 32 warps per SM
    p = lr.linrec_plan_bdl(1, 64, 1 << 20, sm_count=152)
    assert p["twopass"] == 1 and p["tile_t"] % (32 * p["vec"]) == 0
    assert p["chunks"] == -(-(1 << 20) // p["tile_t"]) and p["n_tiles"] == 64 * p["chunks"]
    assert 152 * 16 <= p["n_tiles"] <= 152 * 64
    assert p["workspace_bytes"] == 256 + 4 * (3 * p["n_tiles"] + 64)
    # short rows stay in one pass whatever their number
    assert lr.linrec_plan_bdl(1, 4, 1000)["twopass"] == 0
    # the vector width follows L and the alignment; 16-bit storage reaches 16 elements
    # (32 bytes, two 16-byte accesses: 16-byte alignment is enough)
    assert lr.linrec_plan_bdl(2, 3, 1001)["vec"] == 1
    assert lr.linrec_plan_bdl(2, 3, 1002)["vec"] == 2
    assert lr.linrec_plan_bdl(2, 3, 1000, align_bytes=8)["vec"] == 2
    assert lr.linrec_plan_bdl(2, 3, 1000, elem_bytes=2)["vec"] == 8
    assert lr.linrec_plan_bdl(2, 3, 1024, elem_bytes=2)["vec"] == 16
    assert lr.linrec_plan_bdl(2, 3, 1024, elem_bytes=2, align_bytes=8)["vec"] == 4
    assert lr.linrec_plan_bdl(2, 3, 1000, elem_bytes=2, align_bytes=2)["vec"] == 1
    assert lr.linrec_plan_bdl(2, 3, 1024, vec=8)["vec"] == 8          # fp32, 32-byte lanes on request
    # forced modes and invalid options
    assert lr.linrec_plan_bdl(32, 256, 4096, chunk_mode="twopass")["twopass"] == 1
    assert lr.linrec_plan_bdl(1, 64, 1 << 20, chunk_mode="own")["twopass"] == 0
    for bad in ({"chunk_mode": "lookback"}, {"path": "chunked"}, {"vec": 3}, {"vec": 16}, {"prefetch": 3}):
        with pytest.raises(lr.LinrecError):
            lr.linrec_plan_bdl(2, 3, 1000, **bad)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_bdl(2, 3, 1000, elem_bytes=8)


def test_bdl_argument_checks(L):
    base = 1 << 36
    B, D, Lx = 2, 3, 16
    n = B * D * Lx * 4
    f = L.linrec_scan_f32_bdl
    assert f(base, base + 2 * n, base + 2 * n - 4, B, D, Lx, None) == lr.LINREC_ERR_ALIAS
    assert f(None, base, base + 2 * n, B, D, Lx, None) == lr.LINREC_ERR_INVALID_VALUE
    assert f(base, base, base + n, B, -1, Lx, None) == lr.LINREC_ERR_INVALID_VALUE
    assert f(None, None, None, B, D, 0, None) == lr.LINREC_OK


def test_plan_invariants_over_a_grid():
    """Every plan the dispatcher returns over a grid of shapes, storages and options is consistent:
    the tile is a compiled one with threads = tile_d / vec * segments, the grid covers the work units
    without exceeding them, the tile count is slices x chunks, and the workspace matches the mode."""
    import itertools
    Bs, Ls, Ds = [1, 3, 16, 40, 128], [1, 100, 300, 2048, 1 << 16], [1, 6, 8, 33, 64, 256, 777, 1024, 4096]
    planners = [(lr.linrec_plan_f32, 4), (lr.linrec_plan_16, 2), (lr.linrec_plan_f32_backward, 4)]
    n_plans = n_chain = n_spec = 0
    for (B, L, D), (planner, eb), kw in itertools.product(
            itertools.product(Bs, Ls, Ds), planners,
            ({}, {"resident_ctas": 2}, {"align_bytes": 4}, {"path": "chunked"})):
        try:
            p = planner(B, L, D, sm_count=152, **kw)
        except lr.LinrecError:
            assert kw.get("path") == "chunked" or kw.get("align_bytes") == 4, (B, L, D, kw)
            continue
        n_plans += 1
        if p["path_name"] == "regcarry":
            assert D % p["vec"] == 0 and p["grid"] >= 1
            groups = B * (D // p["vec"])
            if p["twopass"]:                   # segmented: every (segment, group) a thread
                assert eb == 4 and 2 <= p["segments"] <= 256 and L // p["segments"] >= 64
                assert p["grid"] * p["threads"] >= groups * p["segments"]
                assert p["workspace_bytes"] == 2 * p["segments"] * B * D * 4
            else:
                assert p["grid"] * p["threads"] >= groups
            continue
        assert p["path_name"] == "chunked" and (D * eb) % 16 == 0
        assert p["threads"] == p["tile_d"] // p["vec"] * p["segments"] and p["tile_t"] % p["segments"] == 0
        slices = B * -(-D // p["tile_d"])
        if p["speculative"]:                   # fp32 forward, segments of 8192 steps at least
            G = p["speculative"]
            assert eb == 4 and planner is lr.linrec_plan_f32 and L % G == 0 and L // G >= 8192
            assert (p["tile_d"], p["tile_t"], p["stages"], p["twopass"], p["lookback"]) == (32, 128, 2, 0, 0)
            assert p["chunks"] == -(-(L // G) // 128) and p["n_tiles"] == slices * G * p["chunks"]
            assert 1 <= p["grid"] <= min(slices * G, 152 * 3)
            assert p["workspace_bytes"] == 256 + 2 * slices * G * 32 * 4
            n_spec += 1
            continue
        assert p["chunks"] == -(-L // p["tile_t"]) and p["n_tiles"] == slices * p["chunks"]
        if p["chain"]:                         # every resident CTA: resolvers, then one worker per tile at most
            assert eb == 4 and slices >= 8 and kw.get("path") != "regcarry"
            assert 1 < p["grid"] <= min(p["n_tiles"] + 16, 152 * 2)
            assert p["workspace_bytes"] == 256 + 24 * p["n_tiles"] * p["tile_d"]
            n_chain += 1
            continue
        units = slices if not (p["lookback"] or p["twopass"] or p["blocks"]) else p["n_tiles"]
        assert 1 <= p["grid"] <= units
        if p["lookback"]:
            assert p["workspace_bytes"] == 256 + 24 * p["n_tiles"] * p["tile_d"]
        elif not p["twopass"] and not p["blocks"]:
            assert p["workspace_bytes"] == 256
    assert n_plans > 1000 and n_chain > 0 and n_spec > 0


def test_plan_chain_mode_by_default():
    """fp32 forward scans that would take the two-pass mode and whose speculative segments
    would be short take chain mode from 8 slices of 32 channels on (256-step tiles from 32768
    steps on); fewer slices, 16-bit storage and the gradient keep the two-pass mode."""
    for (B, L, D, tt) in [(2, 16384, 256, 128), (16, 8192, 128, 128), (8, 65536, 64, 256), (3, 50000, 100, 256)]:
        p = lr.linrec_plan_f32(B, L, D, sm_count=152, resident_ctas=2)
        assert p["chain"] == 1 and p["twopass"] == 0 and p["speculative"] == 0 and p["tile_t"] == tt, (B, L, D)
    for (B, L, D) in [(1, 65536, 64), (1, 1 << 20, 32), (1, 131072, 64)]:
        p = lr.linrec_plan_f32(B, L, D, sm_count=152, resident_ctas=2)
        assert p["chain"] == 0 and p["twopass"] == 1 and p["speculative"] == 0, (B, L, D)
    assert lr.linrec_plan_16(4, 65536, 256, sm_count=152)["chain"] == 0
    assert lr.linrec_plan_f32_backward(4, 65536, 256, sm_count=152)["chain"] == 0
    # a forced tile keeps the mode it names or the two-pass mode
    p = lr.linrec_plan_f32(4, 65536, 256, sm_count=152, tile_d=32, tile_t=128, stages=2)
    assert p["chain"] == 0 and p["speculative"] == 0


def test_plan_speculative():
    """Speculative mode: by default where the two-pass or chain mode would be taken and the
    largest segment count G (a divisor of L, slices of the (B * G, L / G, D) view within one
    round of resident CTAs) leaves segments of 8192 steps at least; forced, segments of 1024
    steps at least; `group` names G; fp32 forward only."""
    for (B, L, D, G) in [(1, 1 << 20, 64, 128), (4, 65536, 256, 8), (4, 131072, 128, 16), (3, 32768, 1024, 2),
                         (2, 262144, 128, 32), (1, 524288, 128, 64), (1, 1 << 22, 32, 256)]:
        p = lr.linrec_plan_f32(B, L, D, sm_count=152, resident_ctas=2)
        assert (p["speculative"], p["chain"], p["twopass"], p["lookback"]) == (G, 0, 0, 0), (B, L, D)
        slices = B * G * -(-D // 32)
        assert p["grid"] == min(slices, 304) and p["n_tiles"] == slices * -(-(L // G) // 128)
    # one resident CTA per SM: at most 152 slices
    assert lr.linrec_plan_f32(1, 1 << 22, 32, sm_count=152, resident_ctas=1)["speculative"] == 128
    # G is chosen for at most two CTAs per SM (the repair copy's registers), so the plan made without
    # the occupancy query (three by shared memory) and the call's agree: 1638400 = 2^16 * 25 has the
    # divisor 200 within 3 * 152 / 2 slices per G but not within 2 * 152 / 2
    for res in (2, 3):
        assert lr.linrec_plan_f32(1, 1638400, 64, sm_count=152, resident_ctas=res)["speculative"] == 128
    sp = dict(path="chunked", chunk_mode="speculative", sm_count=152)
    assert lr.linrec_plan_f32(1, 131072, 64, **sp)["speculative"] == 128             # 1024-step segments
    assert lr.linrec_plan_f32(3, 50000, 100, **sp)["speculative"] == 25               # a divisor of L
    p = lr.linrec_plan_f32(1, 1 << 20, 64, group=64, **sp)
    assert (p["speculative"], p["chunks"], p["grid"]) == (64, 128, 128)
    p = lr.linrec_plan_f32(1, 1 << 20, 64, group=1024, **sp)                         # the most segments
    assert (p["speculative"], p["chunks"], p["grid"]) == (1024, 8, 456)              # more slices than CTAs
    for bad in (dict(group=3), dict(group=2048)):                                    # no divisor; 512 steps
        with pytest.raises(lr.LinrecError):
            lr.linrec_plan_f32(1, 1 << 20, 64, **sp, **bad)
    for bad in (dict(tile_d=64), dict(tile_t=64), dict(stages=3)):                   # its one compiled tile
        with pytest.raises(lr.LinrecError):
            lr.linrec_plan_f32(1, 1 << 20, 64, **sp, **bad)
    for shape in [(1, 2047, 64), (1, 1500, 32), (456, 4096, 32)]:                    # no 2 segments of 1024
        with pytest.raises(lr.LinrecError):
            lr.linrec_plan_f32(*shape, **sp)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_16(1, 1 << 20, 64, **sp)
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32_backward(1, 1 << 20, 64, chunk_mode="speculative")
    with pytest.raises(lr.LinrecError):
        lr.linrec_plan_f32(1, 1 << 20, 64, chunk_mode="own", group=8)


def test_gradient_host_and_noalloc_argument_checks(L):
    """The gradient, host-buffer and no-allocation entries reject bad sizes, null pointers, overlaps
    and (no-allocation entry) unaligned pointers before any CUDA call; fake addresses, never read."""
    vp = ctypes.c_void_p
    B, Lx, D = 2, 100, 8
    n = B * Lx * D * 4
    base = 1 << 36
    a, h, g, da, db = (base + k * n for k in range(5))
    st1, st2, st3 = base + 5 * n, base + 5 * n + 1024, base + 5 * n + 2048
    bw = L.linrec_scan_f32_backward_ex

    def grad(*args, **over):
        kw = dict(a=a, h=h, g=g, da=da, db=db, B=B, L=Lx, D=D, h_init=None, dh_last=None, dh_init=None)
        kw.update(over)
        return bw(kw["a"], kw["h"], kw["g"], kw["da"], kw["db"], kw["B"], kw["L"], kw["D"],
                  kw["h_init"], kw["dh_last"], kw["dh_init"], None, None)

    assert grad(B=-1) == lr.LINREC_ERR_INVALID_VALUE
    assert grad(a=None, h=None, g=None, da=None, db=None, L=0) == lr.LINREC_OK
    for missing in ("a", "g", "db"):
        assert grad(**{missing: None}) == lr.LINREC_ERR_INVALID_VALUE, missing
    assert grad(h=None) == lr.LINREC_ERR_INVALID_VALUE                      # da wanted without h
    assert grad(da=a + 4) == lr.LINREC_ERR_ALIAS                            # da inside a
    assert grad(db=h + n - 4) == lr.LINREC_ERR_ALIAS                        # db overlaps the end of h
    assert grad(db=da + 8) == lr.LINREC_ERR_ALIAS                           # the two outputs overlap
    assert grad(h_init=st1, dh_last=st2, dh_init=st2 + 4) == lr.LINREC_ERR_ALIAS
    assert grad(h_init=st1, dh_init=db + 16) == lr.LINREC_ERR_ALIAS         # dh_init inside db

    host = L.linrec_scan_f32_host
    b = h
    assert host(a, b, da, -1, Lx, D, None) == lr.LINREC_ERR_INVALID_VALUE
    assert host(None, None, None, B, Lx, 0, None) == lr.LINREC_OK
    assert host(a, None, da, B, Lx, D, None) == lr.LINREC_ERR_INVALID_VALUE
    assert host(a, b, a + 12, B, Lx, D, None) == lr.LINREC_ERR_ALIAS
    assert host(a, b, b - n + 4, B, Lx, D, None) == lr.LINREC_ERR_ALIAS
    assert host(16, 32, 64, 1 << 20, 1 << 20, 1 << 22, None) == lr.LINREC_ERR_INVALID_VALUE

    na = L.linrec_scan_f32_noalloc
    na.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vp]
    na.restype = ctypes.c_int
    assert na(a, b, da, B, -Lx, D, None, None) == lr.LINREC_ERR_INVALID_VALUE
    assert na(None, None, None, 0, Lx, D, None, None) == lr.LINREC_OK
    assert na(a, b, None, B, Lx, D, None, None) == lr.LINREC_ERR_INVALID_VALUE
    assert na(a, b, b + 16, B, Lx, D, None, None) == lr.LINREC_ERR_ALIAS
    assert na(a + 4, b, da, B, Lx, D, None, None) == lr.LINREC_ERR_INVALID_VALUE   # not 16-byte aligned
    assert na(a, b, da, B, Lx, 6, None, None) == lr.LINREC_ERR_INVALID_VALUE      # D not a multiple of 4
    assert na(16, 32, 64, 1 << 20, 1 << 20, 1 << 22, None, None) == lr.LINREC_ERR_INVALID_VALUE


def test_host_range_check():
    """linrec_scan_f32_host reads a page-locked buffer in place only when the registered range of
    its first byte holds every byte; a range that ends early (a registered prefix), starts late,
    or wraps around the address space sends the buffer through the copy pipeline."""
    covers = lr.linrec_debug_range_covers
    base, size = 1 << 40, 1 << 20
    assert covers(base, size, base, size)
    assert covers(base, size, base + 4096, size - 4096)
    assert covers(base, size, base + size - 4, 4)
    assert not covers(base, size, base, size + 1)                 # the last byte outside
    assert not covers(base, size, base + 4096, size)              # ends past the range
    assert not covers(base, size, base - 4, 8)                    # starts before it
    assert not covers(base, size, base + size, 4)                 # just past the end
    assert not covers(base, size, base, 0)                        # nothing to cover
    top = (1 << 64) - 4096
    assert covers(top, 4096, top, 4096)
    assert not covers(top, 4096, top + 8, (1 << 64) - 1)          # would wrap


def test_no_cpu_fallback():
    """CPU tensors are refused rather than scanned on the host, and a missing library is an error that
    names the build step, never a silent fallback (checked in a fresh interpreter)."""
    import subprocess
    import sys
    import torch
    a, b = torch.rand(1, 8, 4), torch.randn(1, 8, 4)
    for call in (lambda: lr.linrec_scan_f32(a, b), lambda: lr.linrec_scan_f32_ex(a, b, path="regcarry"),
                 lambda: lr.linrec_scan_f32_backward(a, a, b),
                 lambda: lr.linrec_scan_bf16_ex(a.bfloat16(), b.bfloat16()),
                 lambda: lr.linrec_scan_f32_bdl_ex(a, b)):
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
    code = ("import linear_recurrence_scan_fp32_gb300 as lr\n"
            "try:\n    lr.linrec_plan_f32(1, 64, 32)\nexcept lr.LinrecError as e:\n    print('refused:', e)\n")
    env = dict(os.environ, LINREC_LIBRARY=os.path.join(ROOT, "no_such_dir", "liblinrec.so"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "refused:" in r.stdout and "missing" in r.stdout and "no fallback" in r.stdout, r.stdout


@pytest.mark.parametrize("compiler", [["gcc", "-std=c99", "-pedantic"], ["g++", "-std=c++17", "-x", "c++"]],
                         ids=("c99", "c++17"))
def test_header_compiles_and_links_from_c(L, compiler, tmp_path):
    """A plain C (and C++) consumer of include/linrec.h, linked against liblinrec.so: the header is valid
    on its own and its declarations match what the library exports (tests/c/abi_check.c)."""
    import shutil
    import subprocess
    if shutil.which(compiler[0]) is None:
        pytest.skip(f"{compiler[0]} not installed")
    libdir = os.path.dirname(lr.LIB_PATH)
    exe = str(tmp_path / "abi_check")
    cmd = compiler + ["-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                      os.path.join(ROOT, "tests", "c", "abi_check.c"), "-L", libdir, "-llinrec",
                      f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "abi_check: ok" in r.stdout, r.stdout + r.stderr
