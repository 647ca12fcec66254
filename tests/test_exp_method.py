"""The exact mode's exp method on the CPU (no GPU): a step-by-step fp32
emulation of the fast path of exp_cr2 (gated_softmax_kv_gb300/csrc/
csa_exp_cr.cuh: Tang's table-driven reduction with a two-float result and the
one-sided rounding test) over a seeded sample of arguments. Every result the
rounding test accepts must be the correctly rounded exp, and the test must
accept all but a small fraction of arguments.

The emulation rounds each fp32 operation as the device does; an FMA is an
exact product plus one rounding, computed in extended precision (the products
of two floats are exact there). Disagreements with fp64 exp rounded to fp32
are settled with mpmath, since that reference can itself be off by double
rounding."""
import numpy as np
import pytest

f32 = np.float32


def _bits(u):
    return np.array([u], np.uint32).view(np.float32)[0]


def _fma(a, b, c):
    return (a.astype(np.longdouble) * b.astype(np.longdouble) + c.astype(np.longdouble)).astype(
        np.float32)


def _table():
    v = np.exp2(np.arange(64) / 64.0)
    hi = v.astype(np.float32)
    return hi, (v - hi.astype(np.float64)).astype(np.float32)


def exp_fast_path(x):
    """(result, accepted) per argument, mirroring exp_cr2 operation by operation."""
    x = np.asarray(x, np.float32)
    full = lambda v: np.full_like(x, v)  # noqa: E731
    inv_c, c_hi, c2, c3 = _bits(0x42b8aa3b), _bits(0x3c318000), _bits(0xb65e8083), _bits(0x28e7bcd6)
    k6, k24, k120 = _bits(0x3e2aaaab), _bits(0x3d2aaaab), _bits(0x3c088889)
    shift = f32(12582912.0)
    t_hi, t_lo = _table()
    inr = np.abs(x) <= f32(86.0)
    t = _fma(x, full(inv_c), full(shift))
    nf = (t - shift).astype(np.float32)
    b = t.view(np.uint32).astype(np.int64)
    rh = _fma(nf, full(-c_hi), x)
    p = (nf * c2).astype(np.float32)
    pen = _fma(nf, full(-c2), p)
    s = (rh - p).astype(np.float32)
    sn = (p - rh).astype(np.float32)
    bb = (s - rh).astype(np.float32)
    se = ((rh - (s - bb).astype(np.float32)).astype(np.float32) - (p + bb).astype(np.float32))
    se = se.astype(np.float32)
    r = s
    rl = ((se + pen).astype(np.float32) - (nf * c3).astype(np.float32)).astype(np.float32)
    r2 = (r * r).astype(np.float32)
    r2en = _fma(sn, r, r2)
    h = (f32(0.5) * r2).astype(np.float32)
    v = _fma(r, _fma(r, full(k120), full(k24)), full(k6))
    cubic = ((r2 * r).astype(np.float32) * v).astype(np.float32)
    em = (r + h).astype(np.float32)
    emn = (sn - h).astype(np.float32)
    e3 = ((r - em).astype(np.float32) + h).astype(np.float32)
    rrl = (r * rl).astype(np.float32)
    eml = ((e3 + rl).astype(np.float32) + (_fma(full(f32(-0.5)), r2en, cubic) + rrl).astype(
        np.float32)).astype(np.float32)
    idx = b & 63
    th, tl = t_hi[idx], t_lo[idx]
    an = (th * emn).astype(np.float32)
    ae = _fma(th, em, an)
    bsum = (_fma(th, eml, _fma(tl, em, tl)) + ae).astype(np.float32)
    s2 = (th - an).astype(np.float32)
    e2 = ((th - s2).astype(np.float32) - an).astype(np.float32)
    tt = (e2 + bsum).astype(np.float32)
    y = (s2 + tt).astype(np.float32)
    er = (tt - (y - s2).astype(np.float32)).astype(np.float32)
    res = ((y.view(np.uint32).astype(np.int64) + ((b << 17) & 0xff800000)) & 0xffffffff).astype(
        np.uint32).view(np.float32)
    ok = inr & (_fma(er, full(_bits(0x3f800080)), y) == y)
    return res, ok


def test_fast_path_is_correctly_rounded():
    if np.finfo(np.longdouble).nmant < 60:
        pytest.skip("needs an extended-precision long double for the FMA emulation")
    mpmath = pytest.importorskip("mpmath")
    rng = np.random.default_rng(23)
    lo = np.float32(-86.0).view(np.uint32)
    xs = np.concatenate([
        rng.integers(0x80000000, lo, 600_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
        rng.uniform(-1.0, 0.0, 200_000).astype(np.float32),
        rng.uniform(-86.0, 86.0, 200_000).astype(np.float32),
        np.float32([0.0, -0.0, -86.0, 86.0, -1e-30, -1e-45]),
    ])
    got, ok = exp_fast_path(xs)
    assert ok.mean() > 0.9999, f"the rounding test accepts only {ok.mean():.6f}"
    want = np.exp(xs.astype(np.float64)).astype(np.float32)
    diff = np.nonzero(ok & (got.view(np.uint32) != want.view(np.uint32)))[0]
    mpmath.mp.prec = 200
    for i in diff:  # settle the fp64 reference's own double-rounding cases exactly
        exact = mpmath.exp(mpmath.mpf(float(xs[i])))
        f = np.float32(float(exact))
        cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
        nearest = min(cands, key=lambda c: abs(mpmath.mpf(float(c)) - exact))
        assert got[i] == nearest, (float(xs[i]), float(got[i]), float(nearest))
