"""Comparison helpers shared by the tests (no recurrence arithmetic here)."""
import numpy as np

# Per-element bound |h - h64| <= ATOL + RTOL * |h64|; the fp32 convention
# atol = rtol = 1e-4 of the POPCORNBENCH harness ("Kimi-K2.6 l2_p1", the
# correctness check of the submitted kernel).
ATOL = 1e-4
RTOL = 1e-4


def excess(h, h64, atol=ATOL, rtol=RTOL):
    """max over elements of |h - h64| - (atol + rtol*|h64|); <= 0 means within bound."""
    h = np.asarray(h, dtype=np.float64)
    h64 = np.asarray(h64, dtype=np.float64)
    if h.shape != h64.shape:
        raise ValueError(f"shape mismatch {h.shape} vs {h64.shape}")
    if h.size == 0:
        return -np.inf
    err = np.abs(h - h64) - (atol + rtol * np.abs(h64))
    err = np.where(np.isnan(err), np.inf, err)
    return float(err.max())


def assert_close(h, h64, what="", atol=ATOL, rtol=RTOL):
    e = excess(h, h64, atol, rtol)
    if not e <= 0:
        h = np.asarray(h, dtype=np.float64)
        h64 = np.asarray(h64, dtype=np.float64)
        bad = np.argwhere(~(np.abs(h - h64) <= atol + rtol * np.abs(h64)))
        first = tuple(bad[0]) if len(bad) else None
        raise AssertionError(
            f"{what}: {len(bad)} elements out of bound; first at {first}: "
            f"got {h[first] if first else None}, want {h64[first] if first else None}")


def max_errors(h, h64):
    h = np.asarray(h, dtype=np.float64)
    h64 = np.asarray(h64, dtype=np.float64)
    d = np.abs(h - h64)
    return float(d.max()) if d.size else 0.0, float((d / (1 + np.abs(h64))).max()) if d.size else 0.0
