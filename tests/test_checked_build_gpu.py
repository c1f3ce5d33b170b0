"""The index-checked build (compiled with -DLINREC_DEBUG): every plain global load
and store of the scan kernels is tested against its array first, and one outside
is skipped and counted.  It stands in for an external memory checker.

Two runs, each in a fresh process that loads liblinrec_checked.so:
  1. the small sweep over every kernel and mode (test_every_kernel_small_gpu.py):
     parity with the oracle as in the normal build, and no access skipped;
  2. with the outputs capped 5 elements short of their end (a test hook, no real
     out-of-bounds access), each path skips exactly those stores, records the first
     skipped offset inside the cut-off part, leaves those elements untouched and
     writes the rest as the normal build does.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CAP_SCRIPT = r"""
import torch
import linear_recurrence_scan_fp32_gb300 as lr
assert lr.linrec_debug_checks(), "not the index-checked build"
torch.cuda.set_device(0)
g = torch.Generator(device="cuda").manual_seed(5)
B, L, D = 2, 300, 64
n = B * L * D
a = 0.5 + 0.5 * torch.rand((B, L, D), generator=g, device="cuda")
b = torch.randn((B, L, D), generator=g, device="cuda")
for opt in ({"path": "chunked", "chunk_mode": "own"}, {"path": "chunked", "chunk_mode": "lookback"},
            {"path": "chunked", "chunk_mode": "chain"},
            {"path": "regcarry", "vec": 1}, {"path": "regcarry", "vec": 4}):
    want = lr.linrec_scan_f32_ex(a, b, **opt)
    assert lr.linrec_debug_bad_accesses(output_cap_bytes=(n - 5) * 4) == (0, -1), "accesses skipped uncapped"
    h = torch.full_like(a, float("nan"))
    lr.linrec_scan_f32_ex(a, b, h, **opt)
    count, first = lr.linrec_debug_bad_accesses(output_cap_bytes=0)
    flat, ref = h.flatten(), want.flatten()
    stores = 2 if opt.get("vec") == 4 else 5          # a 16-byte store across the cut counts once
    assert count == stores, (opt, count)
    assert (n - 8) * 4 <= first < n * 4, (opt, first)
    assert torch.equal(flat[: n - 8], ref[: n - 8]), opt
    assert torch.isnan(flat[n - 5:]).all(), opt
    assert lr.linrec_stream_status() == lr.LINREC_OK
# speculative mode: two segments of 2048 steps, two launches; the slopes' product reaches 0
# within the second segment, so its last tile is stored by the speculative launch
B, L, D = 1, 4096, 64
n = B * L * D
a = 0.5 + 0.5 * torch.rand((B, L, D), generator=g, device="cuda")
b = torch.randn((B, L, D), generator=g, device="cuda")
opt = {"path": "chunked", "chunk_mode": "speculative", "group": 2}
assert lr.linrec_plan_f32(B, L, D, **opt)["speculative"] == 2
want = lr.linrec_scan_f32_ex(a, b, **opt)
assert lr.linrec_debug_bad_accesses(output_cap_bytes=(n - 5) * 4) == (0, -1), "accesses skipped uncapped"
h = torch.full_like(a, float("nan"))
lr.linrec_scan_f32_ex(a, b, h, **opt)
count, first = lr.linrec_debug_bad_accesses(output_cap_bytes=0)
flat, ref = h.flatten(), want.flatten()
assert count == 5, count
assert (n - 8) * 4 <= first < n * 4, first
assert torch.equal(flat[: n - 8], ref[: n - 8])
assert torch.isnan(flat[n - 5:]).all()
assert lr.linrec_stream_status() == lr.LINREC_OK
print("cap ok")
"""


def _checked_env():
    from linear_recurrence_scan_fp32_gb300 import _build
    path = _build.build(checked=True)
    return dict(os.environ, LINREC_LIBRARY=path)


def test_checked_build_runs_every_kernel_clean():
    env = _checked_env()
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join("tests", "test_every_kernel_small_gpu.py"),
                        "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


def test_checked_build_skips_and_records_capped_stores():
    env = _checked_env()
    r = subprocess.run([sys.executable, "-c", CAP_SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "cap ok" in r.stdout, r.stdout[-4000:] + r.stderr[-4000:]
