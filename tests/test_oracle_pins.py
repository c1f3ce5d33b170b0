"""Pins for the CPU oracle: what the pages and the mathematics fix, not the oracle itself.

Each pin is a function of an oracle library handle, so that the planted-mistake
test at the bottom can run every pin against edited copies of the oracle and
check that each planted mistake is caught by at least one of them.

Definition pinned (POPCORNBENCH trace "Kimi-K2.6 l1_p9", problem statement):
h_0 = b_0, h_t = a_t*h_{t-1} + b_t, per channel of (B, L, D) tensors, D contiguous.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from linear_recurrence_scan_fp32_gb300 import inputs
from tests._util import assert_close, excess

HERE = os.path.dirname(os.path.abspath(__file__))


def _rng(seed):
    return np.random.default_rng(seed)


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


# ---------------------------------------------------------------------------
# pins (each returns None or raises AssertionError)
# ---------------------------------------------------------------------------

def pin_walkthrough(lib):
    """The page's symbolic walk-through t = 0, 1, 2, on exact dyadic inputs."""
    vals = {}
    with open(os.path.join(HERE, "golden", "walkthrough_t012.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = [float(v) for v in rest.split()]
    B, L, D = (int(v) for v in vals["shape"])
    a = _f32(np.array(vals["a"]).reshape(B, L, D))
    b = _f32(np.array(vals["b"]).reshape(B, L, D))
    want = np.array(vals["h"]).reshape(B, L, D)
    h, _ = oracle.f64(a, b, lib=lib)
    assert np.array_equal(h, want), f"walk-through: got {h.ravel()} want {want.ravel()}"


def pin_prefix_sum(lib):
    """a = 1: h_t is the inclusive prefix sum of b (textbook scan), exact on integers."""
    rng = _rng(10)
    b_int = _f32(rng.integers(-8, 9, size=(3, 257, 5)))
    a = np.ones_like(b_int)
    h, _ = oracle.f64(a, b_int, lib=lib)
    assert np.array_equal(h, np.cumsum(b_int.astype(np.float64), axis=1)), "integer prefix sum"
    b = _f32(rng.standard_normal((2, 300, 7)))
    h, _ = oracle.f64(np.ones_like(b), b, lib=lib)
    ref = np.cumsum(b.astype(np.float64), axis=1)
    assert np.allclose(h, ref, rtol=0, atol=1e-12 * 300), "real prefix sum"


def pin_copy(lib):
    """a = 0: h = b exactly."""
    b = _f32(_rng(11).standard_normal((2, 77, 9)))
    h, _ = oracle.f64(np.zeros_like(b), b, lib=lib)
    assert np.array_equal(h, b.astype(np.float64)), "a=0 must copy b"


def pin_running_product(lib):
    """b = (1, 0, 0, ...): h_t = a_1 * a_2 * ... * a_t (a_0 unused)."""
    rng = _rng(12)
    a = _f32(rng.uniform(-1.5, 1.5, size=(2, 64, 6)))
    b = np.zeros_like(a)
    b[:, 0, :] = 1.0
    h, _ = oracle.f64(a, b, lib=lib)
    want = np.ones((2, 64, 6))
    want[:, 1:, :] = np.cumprod(a[:, 1:, :].astype(np.float64), axis=1)
    assert np.allclose(h, want, rtol=1e-13, atol=0), "running product"


def pin_geometric(lib):
    """Constant a = c, b = beta: h_t = beta*(1 - c^(t+1))/(1 - c)."""
    c, beta, L = 0.75, 1.25, 400
    a = np.full((1, L, 3), c, dtype=np.float32)
    b = np.full((1, L, 3), beta, dtype=np.float32)
    h, _ = oracle.f64(a, b, lib=lib)
    t = np.arange(L, dtype=np.float64)
    want = beta * (1.0 - c ** (t + 1)) / (1.0 - c)
    assert np.allclose(h[0, :, 1], want, rtol=1e-13, atol=0), "geometric series"
    # c = -0.5 makes the signs alternate; a dropped or flipped term shows at once
    c2 = -0.5
    h, _ = oracle.f64(np.full((1, 50, 1), c2, np.float32), np.full((1, 50, 1), beta, np.float32), lib=lib)
    t = np.arange(50, dtype=np.float64)
    assert np.allclose(h[0, :, 0], beta * (1 - c2 ** (t + 1)) / (1 - c2), rtol=1e-13, atol=1e-15)


def _expanded_exact(a, b):
    """h_t = sum_{s<=t} (prod_{s<r<=t} a_r) b_s in exact rational arithmetic."""
    B, L, D = a.shape
    out = np.empty((B, L, D), dtype=object)
    for i in range(B):
        for d in range(D):
            af = [Fraction(float(x)) for x in a[i, :, d]]
            bf = [Fraction(float(x)) for x in b[i, :, d]]
            for t in range(L):
                acc = Fraction(0)
                for s in range(t + 1):
                    p = Fraction(1)
                    for r in range(s + 1, t + 1):
                        p *= af[r]
                    acc += p * bf[s]
                out[i, t, d] = acc
    return out


def pin_bruteforce(lib):
    """Exact rational expansion of the recurrence on tiny random inputs (a_0 random too)."""
    rng = _rng(13)
    for L in (1, 2, 3, 5, 8):
        a = _f32(rng.uniform(-2, 2, size=(2, L, 3)))
        b = _f32(rng.standard_normal((2, L, 3)))
        exact = _expanded_exact(a, b)
        h, _ = oracle.f64(a, b, lib=lib)
        # bound: a few fp64 roundings of each partial product and sum
        for idx in np.ndindex(h.shape):
            e = exact[idx]
            err = abs(Fraction(float(h[idx])) - e)
            assert err <= Fraction(1, 10 ** 12) * (1 + abs(e)), f"L={L} at {idx}: {float(h[idx])} vs {float(e)}"


def pin_carry_closed_forms(lib):
    """Continued from h0 = x: a = c, b = 0 gives h_t = c^(t+1) x; a = 1 gives x + prefix sums of b."""
    B, L, D = 2, 60, 3
    x = np.array([[1.5, -2.0, 0.25], [4.0, 0.5, -1.0]])
    a = np.full((B, L, D), 0.5, np.float32)
    h, hl = oracle.f64_carry(a, np.zeros_like(a), x, lib=lib)
    want = x[:, None, :] * 0.5 ** (np.arange(L)[None, :, None] + 1.0)
    assert np.array_equal(h, want), "decay from the carried state"
    assert np.array_equal(hl, want[:, -1, :]), "last state"
    b = _f32(_rng(14).integers(-8, 9, size=(B, L, D)))
    h, hl = oracle.f64_carry(np.ones_like(b), b, x, lib=lib)
    want = x[:, None, :] + np.cumsum(b.astype(np.float64), axis=1)
    assert np.array_equal(h, want), "prefix sum continued from the carried state"
    assert np.array_equal(hl, want[:, -1, :])


def pin_carry_bruteforce(lib):
    """h_t = (a_0 ... a_t) x + sum_s (a_{s+1} ... a_t) b_s, exactly, a_0 used."""
    rng = _rng(15)
    for L in (1, 2, 5, 8):
        a = _f32(rng.uniform(-2, 2, size=(2, L, 2)))
        b = _f32(rng.standard_normal((2, L, 2)))
        x = rng.standard_normal((2, 2))
        h, hl = oracle.f64_carry(a, b, x, lib=lib)
        for i in range(2):
            for d in range(2):
                af = [Fraction(float(v)) for v in a[i, :, d]]
                bf = [Fraction(float(v)) for v in b[i, :, d]]
                for t in range(L):
                    p = Fraction(1)
                    for r in range(0, t + 1):
                        p *= af[r]
                    e = p * Fraction(float(x[i, d]))
                    for s_ in range(t + 1):
                        q = Fraction(1)
                        for r in range(s_ + 1, t + 1):
                            q *= af[r]
                        e += q * bf[s_]
                    assert abs(Fraction(float(h[i, t, d])) - e) <= Fraction(1, 10 ** 12) * (1 + abs(e)), (L, i, t, d)
                assert hl[i, d] == h[i, L - 1, d]


def pin_carry_segments(lib):
    """Scanning in segments, each continued from the last state of the one before, is the
    unsplit scan bit for bit; with no state the carry entry is the plain definition."""
    a, b = inputs.generate(3, 200, 7, seed=16)
    a, b = a.numpy(), b.numpy()
    full, _ = oracle.f64(a, b, lib=lib)
    h0, hl0 = oracle.f64_carry(a, b, None, lib=lib)
    assert np.array_equal(h0, full) and np.array_equal(hl0, full[:, -1, :])
    parts, state = [], None
    for lo, hi in [(0, 1), (1, 64), (64, 65), (65, 200)]:
        h, state = oracle.f64_carry(a[:, lo:hi], b[:, lo:hi], state, lib=lib)
        parts.append(h)
    assert np.array_equal(np.concatenate(parts, axis=1), full), "segments differ from the unsplit scan"


def _dyadic(rng, shape, lo, hi, bits=8):
    """Values on a 2^-bits grid, so that small power-of-two steps stay exact in fp32."""
    return _f32(np.round(rng.uniform(lo, hi, size=shape) * 2 ** bits) / 2 ** bits)


def pin_backward_finite_differences(lib):
    """Gradients of loss = sum(g*h) + sum(w*h_{L-1}) match central differences of the forward oracle."""
    rng = _rng(20)
    B, L, D = 2, 6, 3
    a = _dyadic(rng, (B, L, D), -1.25, 1.25)
    b = _dyadic(rng, (B, L, D), -1.0, 1.0)
    g = _dyadic(rng, (B, L, D), -1.0, 1.0)
    w = rng.standard_normal((B, D))
    x = rng.standard_normal((B, D))

    def loss(a_, b_, x_):
        h, hl = oracle.f64_carry(a_, b_, x_, lib=lib)
        return float((g.astype(np.float64) * h).sum() + (w * hl).sum())

    h, _ = oracle.f64_carry(a, b, x, lib=lib)
    da, db, dx = oracle.f64_backward(a, h.astype(np.float32), g, x, w, lib=lib)
    eps = 2.0 ** -12
    for idx in [(0, 0, 0), (0, 3, 1), (1, 5, 2), (1, 1, 0), (0, 5, 2)]:
        for arr, grad in ((a, da), (b, db)):
            p_, m_ = arr.copy(), arr.copy()
            p_[idx] += eps
            m_[idx] -= eps
            fd = (loss(p_ if arr is a else a, p_ if arr is b else b, x) -
                  loss(m_ if arr is a else a, m_ if arr is b else b, x)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-5 * (1 + abs(fd)), (idx, fd, grad[idx])
    for i, d in [(0, 0), (1, 2)]:
        xp, xm = x.copy(), x.copy()
        xp[i, d] += eps
        xm[i, d] -= eps
        fd = (loss(a, b, xp) - loss(a, b, xm)) / (2 * eps)
        assert abs(fd - dx[i, d]) <= 1e-7 * (1 + abs(fd)), ((i, d), fd, dx[i, d])


def pin_backward_adjoint(lib):
    """h is linear in b and in the start state: db = M^T g and dh0 = N^T g (dot-product test)."""
    rng = _rng(21)
    B, L, D = 2, 50, 4
    a = _f32(rng.uniform(-1.1, 1.1, (B, L, D)))
    g = _f32(rng.standard_normal((B, L, D)))
    v = _f32(rng.standard_normal((B, L, D)))
    w = rng.standard_normal((B, D))
    hv, _ = oracle.f64(a, v, lib=lib)
    _, db, _ = oracle.f64_backward(a, hv.astype(np.float32), g, None, None, want_da=False, lib=lib)
    lhs, rhs = (g.astype(np.float64) * hv).sum(), (db * v).sum()
    assert abs(lhs - rhs) <= 1e-10 * (1 + abs(lhs)), (lhs, rhs)
    hw, _ = oracle.f64_carry(a, np.zeros_like(a), w, lib=lib)
    _, _, dh0 = oracle.f64_backward(a, hw.astype(np.float32), g, w, None, lib=lib)
    lhs, rhs = (g.astype(np.float64) * hw).sum(), (dh0 * w).sum()
    assert abs(lhs - rhs) <= 1e-10 * (1 + abs(lhs)), (lhs, rhs)


def pin_backward_closed_forms(lib):
    """a = 1: db is the suffix sum of g (plus dh_last); a = 0: db = g; da_t = db_t * h_{t-1}."""
    rng = _rng(22)
    B, L, D = 2, 40, 3
    g = _f32(rng.integers(-8, 9, (B, L, D)))
    h = _f32(rng.integers(-8, 9, (B, L, D)))
    w = rng.integers(-8, 9, (B, D)).astype(np.float64)
    x = rng.integers(-8, 9, (B, D)).astype(np.float64)
    da, db, dx = oracle.f64_backward(np.ones_like(g), h, g, x, w, lib=lib)
    want = np.cumsum(g[:, ::-1].astype(np.float64), axis=1)[:, ::-1] + w[:, None, :]
    assert np.array_equal(db, want), "suffix sums"
    hprev = np.concatenate([x[:, None, :], h[:, :-1].astype(np.float64)], axis=1)
    assert np.array_equal(da, want * hprev), "da = c * h_{t-1}"
    assert np.array_equal(dx, want[:, 0, :]), "dh0 = a_0 c_0 with a_0 = 1"
    da, db, dx = oracle.f64_backward(np.zeros_like(g), h, g, None, w, lib=lib)
    want = g.astype(np.float64).copy()
    want[:, -1, :] += w
    assert np.array_equal(db, want), "a = 0: db = g"
    assert np.all(da[:, 0, :] == 0), "no start state: da_0 = 0"


def pin_backward_bruteforce(lib):
    """db_s = sum_{t>=s} g_t a_{s+1}..a_t + w a_{s+1}..a_{L-1}, exactly."""
    rng = _rng(23)
    for L in (1, 2, 4, 7):
        a = _f32(rng.uniform(-2, 2, (1, L, 2)))
        g = _f32(rng.standard_normal((1, L, 2)))
        w = rng.standard_normal((1, 2))
        _, db, _ = oracle.f64_backward(a, np.zeros_like(a), g, None, w, want_da=False, lib=lib)
        for d in range(2):
            af = [Fraction(float(v)) for v in a[0, :, d]]
            for s_ in range(L):
                e = Fraction(0)
                for t in range(s_, L):
                    p = Fraction(1)
                    for r in range(s_ + 1, t + 1):
                        p *= af[r]
                    e += p * Fraction(float(g[0, t, d]))
                p = Fraction(1)
                for r in range(s_ + 1, L):
                    p *= af[r]
                e += p * Fraction(float(w[0, d]))
                assert abs(Fraction(float(db[0, s_, d])) - e) <= Fraction(1, 10 ** 12) * (1 + abs(e)), (L, s_, d)


# ---- 16-bit storage: the formats' definitions and the libraries that implement them ----

_ALL16 = np.arange(1 << 16, dtype=np.uint16)
_TOP16 = {"bf16": 0x7F7F, "f16": 0x7BFF}     # largest finite word of each format
_INF16 = {"bf16": 0x7F80, "f16": 0x7C00}


def _same(x, y):
    return np.array_equal(np.asarray(x, dtype=np.float64), np.asarray(y, dtype=np.float64), equal_nan=True)


def pin_decode16_library(lib):
    """Every word's value against numpy's binary16 and torch's bfloat16 (and the
    bfloat16 definition as the top half of a binary32 word)."""
    import torch
    x = oracle.decode16("f16", _ALL16, lib)
    assert _same(x, _ALL16.view(np.float16).astype(np.float64)), "binary16 decode"
    x = oracle.decode16("bf16", _ALL16, lib)
    with np.errstate(invalid="ignore"):           # signalling NaN words widen to quiet NaNs
        ref = (_ALL16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert _same(x, ref), "bf16 decode"
    ref = torch.from_numpy(_ALL16.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert _same(x, ref), "bf16 decode vs torch"


def pin_encode16_neighbours(lib):
    """Round to nearest, ties to even, from the definition: every word encodes to
    itself; the midpoint of two adjacent words goes to the one with the even
    significand; a hair below or above it goes to the nearer word; the midpoint
    above the largest finite word overflows to infinity; the sign is separate."""
    for kind in ("bf16", "f16"):
        top = _TOP16[kind]
        w = _ALL16[: top + 1]                        # +0 .. largest finite
        v = oracle.decode16(kind, w, lib)
        assert np.array_equal(oracle.encode16(kind, v, lib), w), f"{kind}: a word is not its own encoding"
        ulp_top = v[top] - v[top - 1]
        upper = np.append(v[1:], v[top] + ulp_top)   # the next word up (infinity after the top)
        mid = (v + upper) / 2                        # exact: dyadic values of few bits
        nxt = np.append(w[1:], np.uint16(_INF16[kind]))
        want = np.where(w % 2 == 0, w, nxt)
        assert np.array_equal(oracle.encode16(kind, mid, lib), want), f"{kind}: ties"
        assert np.array_equal(oracle.encode16(kind, np.nextafter(mid, -np.inf), lib), w), f"{kind}: below a tie"
        assert np.array_equal(oracle.encode16(kind, np.nextafter(mid, np.inf), lib), nxt), f"{kind}: above a tie"
        assert np.array_equal(oracle.encode16(kind, -v, lib), w | np.uint16(0x8000)), f"{kind}: sign"
        assert oracle.encode16(kind, np.array([np.inf, 1e300]), lib).tolist() == [_INF16[kind]] * 2


def pin_encode16_library(lib):
    """Random doubles over each format's whole range against numpy's binary16
    conversion, and binary32 values against torch's bfloat16 conversion."""
    import torch
    rng = _rng(16)
    x = np.exp(rng.uniform(np.log(1e-9), np.log(7e4), 200_000)) * rng.choice([-1.0, 1.0], 200_000)
    with np.errstate(over="ignore"):              # above 65520 both give infinity
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.encode16("f16", x, lib), ref), "binary16"
    y = (np.exp(rng.uniform(np.log(1e-40), np.log(3e38), 200_000)) * rng.choice([-1.0, 1.0], 200_000)).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.encode16("bf16", y.astype(np.float64), lib), ref), "bf16"


def pin_scan16_closed_forms(lib):
    """The 16-bit scan: a = 1 with integer b gives the prefix sums exactly; a = 0 gives b."""
    rng = _rng(17)
    B, L, D = 2, 300, 8
    for kind, one in (("bf16", 0x3F80), ("f16", 0x3C00)):
        bi = rng.integers(-8, 9, (B, L, D)).astype(np.float64)
        bw = oracle.encode16(kind, bi, lib)
        ones = np.full((B, L, D), one, dtype=np.uint16)
        h, last = oracle.f64_16(kind, ones, bw, lib=lib)
        assert np.array_equal(h, np.cumsum(bi, axis=1)), f"{kind}: a = 1"
        assert np.array_equal(last, h[:, -1]), f"{kind}: last state"
        h, _ = oracle.f64_16(kind, np.zeros((B, L, D), np.uint16), bw, lib=lib)
        assert np.array_equal(h, bi), f"{kind}: a = 0"


# ---- (B, D, L) layout ---------------------------------------------------------

def pin_bdl_layout_invariance(lib):
    """Laying channels out as rows changes no value: the (B, D, L) oracle equals the
    transpose of the (B, L, D) oracle bit for bit, with and without a state, on
    shapes whose three sizes differ."""
    rng = _rng(30)
    for (B, D, L) in [(2, 3, 50), (1, 7, 5), (3, 2, 9), (2, 5, 1)]:
        a = rng.uniform(-1.2, 1.2, (B, D, L)).astype(np.float32)
        b = rng.normal(size=(B, D, L)).astype(np.float32)
        h0 = rng.normal(size=(B, D))
        at, bt = np.ascontiguousarray(a.transpose(0, 2, 1)), np.ascontiguousarray(b.transpose(0, 2, 1))
        h, last = oracle.f64_bdl(a, b, lib=lib)
        ht, _ = oracle.f64(at, bt, lib=lib)
        assert np.array_equal(h, ht.transpose(0, 2, 1)), (B, D, L)
        assert np.array_equal(last, h[:, :, -1]), (B, D, L)
        h, last = oracle.f64_bdl(a, b, h0, lib=lib)
        ht, lt = oracle.f64_carry(at, bt, h0, lib=lib)
        assert np.array_equal(h, ht.transpose(0, 2, 1)) and np.array_equal(last, lt), (B, D, L)


def pin_bdl_closed_forms(lib):
    """a = 1: prefix sums along the last axis (plus the state); a = 0: h = b."""
    rng = _rng(31)
    B, D, L = 3, 4, 200
    b = rng.integers(-8, 9, (B, D, L)).astype(np.float32)
    h0 = rng.integers(-5, 6, (B, D)).astype(np.float64)
    ones, zeros = np.ones_like(b), np.zeros_like(b)
    h, _ = oracle.f64_bdl(ones, b, lib=lib)
    assert np.array_equal(h, np.cumsum(b.astype(np.float64), axis=2))
    h, last = oracle.f64_bdl(ones, b, h0, lib=lib)
    assert np.array_equal(h, h0[:, :, None] + np.cumsum(b.astype(np.float64), axis=2))
    assert np.array_equal(last, h[:, :, -1])
    h, _ = oracle.f64_bdl(zeros, b, h0, lib=lib)
    assert np.array_equal(h, b.astype(np.float64))


PINS = [pin_walkthrough, pin_prefix_sum, pin_copy, pin_running_product, pin_geometric, pin_bruteforce,
        pin_carry_closed_forms, pin_carry_bruteforce, pin_carry_segments,
        pin_backward_finite_differences, pin_backward_adjoint, pin_backward_closed_forms,
        pin_backward_bruteforce, pin_decode16_library, pin_encode16_neighbours, pin_encode16_library,
        pin_scan16_closed_forms, pin_bdl_layout_invariance, pin_bdl_closed_forms]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


# ---------------------------------------------------------------------------
# properties of the oracle's own entry points
# ---------------------------------------------------------------------------

def test_a0_is_ignored(oracle_lib):
    """h_0 = b_0: non-finite a_0 leaves every output finite and unchanged."""
    a, b = inputs.generate(2, 40, 5, seed=21)
    a, b = a.numpy().copy(), b.numpy()
    h_ref, _ = oracle.f64(a, b)
    a[:, 0, :] = np.nan
    a[0, 0, 0] = np.inf
    h, _ = oracle.f64(a, b)
    assert np.array_equal(h, h_ref)
    h32, _ = oracle.f32seq(a, b)
    assert np.isfinite(h32).all()


def test_thread_count_does_not_change_bits(oracle_lib):
    a, b = inputs.generate(3, 500, 37, seed=22)
    h1, n1 = oracle.f64(a, b, nthreads=1)
    h7, n7 = oracle.f64(a, b, nthreads=7)
    assert n1 == 1 and n7 >= 1
    assert np.array_equal(h1, h7)
    g1, _ = oracle.f32seq(a, b, nthreads=1)
    g5, _ = oracle.f32seq(a, b, nthreads=5)
    assert np.array_equal(g1, g5)


def test_channel_entry_matches_full(oracle_lib):
    a, b = inputs.generate(2, 300, 9, seed=23)
    h, _ = oracle.f64(a, b)
    for (i, d) in [(0, 0), (1, 8), (1, 3)]:
        assert np.array_equal(oracle.f64_channel(a, b, i, d), h[i, :, d])


def test_empty_and_degenerate_shapes(oracle_lib):
    for shape in [(0, 5, 3), (2, 0, 3), (2, 5, 0)]:
        a = np.zeros(shape, np.float32)
        h, _ = oracle.f64(a, a)
        assert h.shape == shape
    a, b = inputs.generate(1, 1, 4, seed=24)   # L = 1: h = b
    h, _ = oracle.f64(a, b)
    assert np.array_equal(h, b.numpy().astype(np.float64))


def test_f32_loop_meets_bound_on_every_workload(oracle_lib):
    """The independent fp32 loop stays within 1e-4*(1+|h|) of fp64: the configs are well conditioned."""
    for name in inputs.CONFIG_ORDER:
        w = inputs.WORKLOADS[name]
        # the two 134M-element configs are checked on their first batches only
        B = w.B if w.numel <= 70_000_000 else max(1, w.B // 16)
        a, b = inputs.generate(B, w.L, w.D, w.seed, w.a_dist, w.b_dist)
        h64, _ = oracle.f64(a, b)
        h32, _ = oracle.f32seq(a, b)
        assert excess(h32, h64) <= 0, name
        del a, b, h64, h32


# ---------------------------------------------------------------------------
# planted mistakes: every edit of the oracle must fail at least one pin
# ---------------------------------------------------------------------------

_F64_STEP = "h[row + d] = (double)a[row + d] * h[prev + d] + (double)b[row + d];"
_F64_INIT = "h[base + d] = (double)b[base + d];                 /* h_0 = b_0 */"

_CARRY_START = "hv = h0[i * D + d];"
_CARRY_LAST = "if (hlast) hlast[i * D + d] = hv;"

MUTANTS = {
    "backward_slope_not_shifted": ("c = (double)g[k] + coef * c;", "c = (double)g[k] + (double)a[k] * c;"),
    "backward_h_not_shifted": ("if (t > 0) hprev = (double)h[k - D];", "if (t > 0) hprev = (double)h[k];"),
    "backward_dhlast_ignored": ("double c = dhlast ? dhlast[i * D + d] : 0.0;", "double c = 0.0;"),
    "backward_dh0_without_a0": ("if (dh0) dh0[i * D + d] = coef * c;", "if (dh0) dh0[i * D + d] = c;"),
    "carry_state_ignored": (_CARRY_START, "hv = 0.0;"),
    "carry_state_negated": (_CARRY_START, "hv = -h0[i * D + d];"),
    "carry_last_state_wrong": (_CARRY_LAST, "if (hlast) hlast[i * D + d] = hv * 0.5;"),
    "operands_transposed": (_F64_STEP, "h[row + d] = (double)b[row + d] * h[prev + d] + (double)a[row + d];"),
    "a_index_off_by_one": (_F64_STEP, "h[row + d] = (double)a[prev + d] * h[prev + d] + (double)b[row + d];"),
    "b_term_dropped": (_F64_STEP, "h[row + d] = (double)a[row + d] * h[prev + d];"),
    "b_sign_flipped": (_F64_STEP, "h[row + d] = (double)a[row + d] * h[prev + d] - (double)b[row + d];"),
    "carry_dropped": (_F64_STEP, "h[row + d] = (double)a[row + d] + (double)b[row + d];"),
    "a0_applied": (_F64_INIT, "h[base + d] = (double)a[base + d] * (double)b[base + d];"),
    "b_from_previous_step": (_F64_STEP, "h[row + d] = (double)a[row + d] * h[prev + d] + (double)b[prev + d];"),
    "f16_bias_off_by_one": ("{5, 10, 15}", "{5, 10, 16}"),
    "bf16_fraction_width": ("{{8, 7, 127}", "{{7, 8, 127}"),
    "subnormal_scale_wrong": ("ldexp((double)m, 1 - f.bias - f.fbits)", "ldexp((double)m, -f.bias - f.fbits)"),
    "encode_truncates": ("(long long)rint(ldexp(ax, f.fbits - e))", "(long long)floor(ldexp(ax, f.fbits - e))"),
    "encode_ties_away": ("(long long)rint(ldexp(ax, f.fbits - e))", "(long long)round(ldexp(ax, f.fbits - e))"),
    "encode_no_binade_carry": ("if (n == (1ll << (f.fbits + 1))) {", "if (0) {"),
    "encode_no_overflow": ("if (field >= emask) return (uint16_t)(sign | (emask << f.fbits));", ""),
    "bdl_wrong_row": ("const float *ar = a + row * L;", "const float *ar = a + (row % D) * L;"),
    "bdl_state_ignored": ("if (h0) hv = (double)ar[0] * h0[row] + (double)br[0];", ""),
    "bdl_b_from_previous_step": ("hv = (double)ar[t] * hv + (double)br[t];", "hv = (double)ar[t] * hv + (double)br[t - 1];"),
    "bdl_last_state_first_step": ("if (hlast) hlast[row] = hv;", "if (hlast) hlast[row] = hr[0];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, "the oracle source changed; update the planted edit"
    lib = oracle.load(oracle.build_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so")))
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"


# ---------------------------------------------------------------------------
# the composition order: a blocked scan is right with one order, wrong with the other
# ---------------------------------------------------------------------------

def _blocked_scan(a, b, block, combine):
    """Chunked inclusive scan of (a_t, b_t) pairs with a carried prefix, in fp64 (test helper)."""
    a = a.astype(np.float64).copy()
    b = b.astype(np.float64)
    a[:, 0, :] = 0.0   # h_{-1} = 0: the first map's slope never matters
    B, L, D = a.shape
    h = np.empty((B, L, D))
    carry = (np.ones((B, D)), np.zeros((B, D)))   # identity (1, 0)
    for t0 in range(0, L, block):
        acc = (np.ones((B, D)), np.zeros((B, D)))
        for t in range(t0, min(L, t0 + block)):
            acc = combine(acc, (a[:, t], b[:, t]))
            tot = combine(carry, acc)
            h[:, t] = tot[1]
        carry = combine(carry, acc)
    return h


def _combine_right(earlier, later):
    # apply the earlier map first: (a2, b2) o (a1, b1) = (a2*a1, a2*b1 + b2)
    # ("Kimi-K2.6 l1_p9", derivation of the associative operator)
    a1, b1 = earlier
    a2, b2 = later
    return (a2 * a1, a2 * b1 + b2)


def _combine_reversed(earlier, later):
    # the later map applied first, the ordering mistake of the "FW-GLM-5-1 l1_p9" kernel
    a1, b1 = earlier
    a2, b2 = later
    return (a1 * a2, a1 * b2 + b1)


def _combine_stale_a(earlier, later):
    # slope updated before it is used in the offset, the draft-kernel mistake of "Kimi-K2.6 l1_p9"
    a1, b1 = earlier
    a2, b2 = later
    a_new = a2 * a1
    return (a_new, a_new * b1 + b2)


def test_composition_order(oracle_lib):
    a, b = inputs.generate(2, 96, 8, seed=30)
    h64, _ = oracle.f64(a, b)
    a, b = a.numpy(), b.numpy()
    assert excess(_blocked_scan(a, b, 16, _combine_right), h64, 1e-12, 1e-12) <= 0
    assert excess(_blocked_scan(a, b, 16, _combine_reversed), h64) > 0
    assert excess(_blocked_scan(a, b, 16, _combine_stale_a), h64) > 0


# ---------------------------------------------------------------------------
# the comparison every parity test uses
# ---------------------------------------------------------------------------

def test_tolerance_helper_accepts_the_bound_and_nothing_past_it():
    want = np.array([0.0, 1.0, -3.0, 1e4, -2.5e-7])
    at_bound = want + (1e-4 + 1e-4 * np.abs(want)) * np.array([1, -1, 1, -1, 1]) * (1 - 1e-12)
    assert_close(at_bound, want, "on the bound")
    assert excess(want, want) < 0
    for k in range(want.size):                       # any single element just past the bound fails
        bad = at_bound.copy()
        bad[k] = want[k] + 1.01 * (1e-4 + 1e-4 * abs(want[k]))
        with pytest.raises(AssertionError):
            assert_close(bad, want, f"element {k} past the bound")
    for poison in (np.nan, np.inf, -np.inf):         # non-finite output never passes
        bad = want.copy()
        bad[2] = poison
        assert excess(bad, want) == np.inf
        with pytest.raises(AssertionError):
            assert_close(bad, want, "non-finite")
    with pytest.raises(ValueError):                  # a shape mismatch is an error, not a broadcast
        excess(want[:4], want)
    assert excess(np.empty((0, 3)), np.empty((0, 3))) == -np.inf
