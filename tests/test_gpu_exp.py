"""Accuracy of the kernels' softmax exp against the oracle's correctly rounded
fp32 exp, on the argument range the softmax produces (x = z - max <= 0)."""
import ctypes
import os

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _ulp_dist(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = a.view(np.int32).astype(np.int64)
    ib = b.view(np.int32).astype(np.int64)
    return np.abs(ia - ib)


def test_softmax_exp_within_two_ulp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_softmax_kv_gb300 import nvbuild
    nvbuild.build()
    lib = ctypes.CDLL(nvbuild.SELFTEST_LIB)
    lib.csa_selftest_softmax_exp.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                             ctypes.c_void_p]
    lib.csa_selftest_softmax_exp.restype = ctypes.c_int32
    # every 64th fp32 bit pattern in [-87, 0], plus dense samples near 0 and the specials
    lo, hi = np.float32(-87.0).view(np.uint32), np.uint32(0x80000000)
    xs = np.arange(hi, lo, 64, dtype=np.uint64).astype(np.uint32).view(np.float32)
    xs = np.concatenate([xs, np.linspace(-1.0, 0.0, 1 << 20, dtype=np.float32),
                         np.array([0.0, -0.0, -1e-30, -87.3, -88.0, -100.0, -1e4], np.float32)])
    x_d = torch.from_numpy(xs).cuda()
    y_d = torch.empty_like(x_d)
    assert lib.csa_selftest_softmax_exp(x_d.data_ptr(), y_d.data_ptr(), xs.size, None) == 0
    torch.cuda.synchronize()
    got = y_d.cpu().numpy()
    want = oracle.exp_f32_array(xs)
    normal = want >= np.float32(2.0 ** -126)
    ulp = _ulp_dist(got[normal], want[normal])
    print("max ulp", int(ulp.max()), "exact fraction", float(np.mean(ulp == 0)))
    assert int(ulp.max()) <= 2
    # results below the normal range are flushed to zero (or exact)
    assert np.all(got[~normal] <= np.float32(2.0 ** -126))
    # special inputs
    sp = torch.tensor([float("-inf"), float("nan")], device="cuda")
    out = torch.empty_like(sp)
    assert lib.csa_selftest_softmax_exp(sp.data_ptr(), out.data_ptr(), 2, None) == 0
    o = out.cpu().numpy()
    assert o[0] == 0.0 and np.isnan(o[1])


def test_division_from_reciprocal_is_correctly_rounded():
    """The kernels' a / b from one correctly rounded reciprocal per column
    (Markstein's correction step) against IEEE division, on the softmax range
    a = e in [0, 1], b = den in [1, 256], plus random normal operands. The
    correction needs an exact remainder, whose last bit ulp(b) * ulp(q) stays
    in range for quotients of at least 2^-103: that is the tested domain."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_softmax_kv_gb300 import nvbuild
    nvbuild.build()
    lib = ctypes.CDLL(nvbuild.SELFTEST_LIB)
    lib.csa_selftest_div.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_void_p]
    lib.csa_selftest_div.restype = ctypes.c_int32
    rng = np.random.default_rng(7)
    n = 1 << 24
    a = np.concatenate([rng.random(n, dtype=np.float32),
                        (2.0 ** rng.uniform(-99, 0, n)).astype(np.float32),
                        rng.uniform(-1e3, 1e3, n).astype(np.float32)])
    b = np.concatenate([rng.uniform(1.0, 256.0, n).astype(np.float32),
                        rng.uniform(1.0, 16.0, n).astype(np.float32),
                        (2.0 ** rng.uniform(-60, 60, n)).astype(np.float32)])
    keep = np.abs(a.astype(np.float64) / b) >= 2.0 ** -103
    a, b = np.ascontiguousarray(a[keep]), np.ascontiguousarray(b[keep])
    a_d, b_d = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    q_d = torch.empty_like(a_d)
    assert lib.csa_selftest_div(a_d.data_ptr(), b_d.data_ptr(), q_d.data_ptr(), a.size, None) == 0
    torch.cuda.synchronize()
    got = q_d.cpu().numpy()
    want = a / b  # numpy: IEEE fp32 division, correctly rounded
    normal = np.abs(want) >= np.float32(2.0 ** -126)
    bad = np.nonzero(normal & (got.view(np.uint32) != want.view(np.uint32)))[0]
    detail = [(float(a[i]), float(b[i]), float(got[i]), float(want[i])) for i in bad[:8]]
    assert bad.size == 0, f"{bad.size} quotients differ (a, b, got, want): {detail}"


def test_forward_fast_exp_error_bound():
    """The forward's single-rounding exp against the correctly rounded exp on
    [-87, 0]. Error budget: fp32(log2 e) is off by 1.34e-8 relative and the
    product x * fp32(log2 e) is rounded once (<= 2^-24 relative), which gives
    2^t a relative error of at most ln 2 * |x| log2 e * (1.34e-8 + 2^-24)
    = 1.23 |x| 2^-24; ex2.approx and the final rounding add a few units of
    2^-24. Bound used: (1.25 |x| + 8) * 2^-24."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_softmax_kv_gb300 import nvbuild
    nvbuild.build()
    lib = ctypes.CDLL(nvbuild.SELFTEST_LIB)
    lib.csa_selftest_softmax_exp_fast.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                  ctypes.c_void_p]
    lib.csa_selftest_softmax_exp_fast.restype = ctypes.c_int32
    lo, hi = np.float32(-87.0).view(np.uint32), np.uint32(0x80000000)
    xs = np.arange(hi, lo, 64, dtype=np.uint64).astype(np.uint32).view(np.float32)
    xs = np.concatenate([xs, np.linspace(-1.0, 0.0, 1 << 20, dtype=np.float32)])
    x_d = torch.from_numpy(xs).cuda()
    y_d = torch.empty_like(x_d)
    assert lib.csa_selftest_softmax_exp_fast(x_d.data_ptr(), y_d.data_ptr(), xs.size, None) == 0
    torch.cuda.synchronize()
    got = y_d.cpu().numpy().astype(np.float64)
    want = oracle.exp_f32_array(xs).astype(np.float64)
    normal = want >= 2.0 ** -126
    rel = np.abs(got[normal] - want[normal]) / want[normal]
    bound = (1.25 * np.abs(xs[normal].astype(np.float64)) + 8.0) * 2.0 ** -24
    print("max rel err", float(rel.max()), "max rel / bound", float((rel / bound).max()))
    assert np.all(rel <= bound)
    sp = torch.tensor([float("-inf"), float("nan")], device="cuda")
    out = torch.empty_like(sp)
    assert lib.csa_selftest_softmax_exp_fast(sp.data_ptr(), out.data_ptr(), 2, None) == 0
    o = out.cpu().numpy()
    assert o[0] == 0.0 and np.isnan(o[1])


def test_two_lane_fp32_ops_round_like_scalar():
    """The f32x2 helpers of the kernels (add/sub/mul/fma .rn.f32x2) against
    numpy's fp32 arithmetic, one rounding per operation: each alone, a product
    feeding a product, a difference feeding a product, a scalar product
    feeding a two-lane sum or difference, and the two-lane FMA against the
    scalar FMA. (A two-lane product feeding a two-lane add or subtract may be
    fused by the compiler; the kernels never chain them that way.) Random
    operands over wide exponent ranges plus signed zeros, infinities, NaN and
    subnormals."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_softmax_kv_gb300 import nvbuild
    nvbuild.build()
    lib = ctypes.CDLL(nvbuild.SELFTEST_LIB)
    lib.csa_selftest_pair_ops.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64, ctypes.c_void_p]
    lib.csa_selftest_pair_ops.restype = ctypes.c_int32
    rng = np.random.default_rng(7)
    n = 1 << 20
    def draw():
        m = rng.standard_normal(n).astype(np.float32)
        e = rng.integers(-20, 21, n).astype(np.float32)
        return (m * np.exp2(e)).astype(np.float32)
    a, b, c = draw(), draw(), draw()
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-40, -3e-39, 3.4e38], np.float32)
    a[:8], b[8:16], c[16:24] = special, special, special
    dev = [torch.from_numpy(x).cuda() for x in (a, b, c)]
    out = torch.empty(9 * n, dtype=torch.float32, device="cuda")
    assert lib.csa_selftest_pair_ops(*(t.data_ptr() for t in dev), out.data_ptr(), n // 2, None) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy().reshape(9, n)
    with np.errstate(all="ignore"):
        # numpy fp32: one rounding per step
        want = {0: a + b, 1: a - c, 2: b * c, 3: (a * b) * c, 4: (a - b) * c, 7: a + b * c,
                8: a * b - c}
    for row, w in want.items():
        same = (got[row].view(np.uint32) == w.view(np.uint32)) | (np.isnan(got[row]) & np.isnan(w))
        assert same.all(), f"pattern {row}: {int((~same).sum())} differ"
    same = (got[5].view(np.uint32) == got[6].view(np.uint32)) | (np.isnan(got[5]) & np.isnan(got[6]))
    assert same.all(), f"fma2: {int((~same).sum())} differ from the scalar FMA"


def test_correctly_rounded_exp_matches_the_oracle():
    """exp_cr2 (the exact mode's exp, two arguments per call) against the
    oracle's exp (fp64 exp rounded once to fp32), bit for bit: every 61st
    fp32 value in [-86, 0] (the table-driven path and its rounding test), a
    dense sweep of [-1, 0], [-104, -86] (the fp64 path, down through the
    subnormals to 0), the special values, and a shuffled copy of all of it so
    that pairs mix the two paths."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_softmax_kv_gb300 import nvbuild
    nvbuild.build()
    lib = ctypes.CDLL(nvbuild.SELFTEST_LIB)
    fn = lib.csa_selftest_exp_cr2
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    lo, hi = np.float32(-86.0).view(np.uint32), np.uint32(0x80000000)
    xs = np.concatenate([
        np.arange(hi, lo, 61, dtype=np.uint64).astype(np.uint32).view(np.float32),
        np.linspace(-1.0, 0.0, 1 << 22, dtype=np.float32),
        np.linspace(-104.0, -86.0, 1 << 20, dtype=np.float32),
        np.array([0.0, -0.0, -np.inf, np.nan, -86.0, -87.0, -103.97, -103.98, -104.0, -1e-30,
                  np.inf, 1.0], np.float32)])
    xs = np.concatenate([xs, np.random.default_rng(3).permutation(xs)])
    x_d = torch.from_numpy(xs).cuda()
    y_d = torch.empty_like(x_d)
    assert fn(x_d.data_ptr(), y_d.data_ptr(), xs.size // 2, None) == 0
    torch.cuda.synchronize()
    got = y_d.cpu().numpy()
    want = oracle.exp_f32_array(xs)
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    bad = np.nonzero(~same)[0]
    detail = [(float(xs[i]), float(got[i]), float(want[i])) for i in bad[:8]]
    assert bad.size == 0, f"{bad.size} of {xs.size} differ (x, got, want): {detail}"


def test_exact_mode_division_is_ieee():
    """div2_cr, the exact mode's e / den (one reciprocal per column, the
    correction step, IEEE division below 2^-102), against IEEE fp32 division
    on the softmax domain e in [0, 1], den in [1, 8], with e spread down to
    2^-149 and exact zeros, and with NaN denominators; every result, subnormal
    quotients included, must carry IEEE's bits."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_softmax_kv_gb300 import nvbuild
    nvbuild.build()
    lib = ctypes.CDLL(nvbuild.SELFTEST_LIB)
    fn = lib.csa_selftest_div2
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    rng = np.random.default_rng(11)
    n = 1 << 23
    a = np.concatenate([rng.random(n, dtype=np.float32),
                        (2.0 ** rng.uniform(-149, 0, n)).astype(np.float32),
                        np.zeros(64, np.float32), np.ones(64, np.float32)])
    b = np.concatenate([rng.uniform(1.0, 8.0, n).astype(np.float32),
                        rng.uniform(1.0, 8.0, n).astype(np.float32),
                        rng.uniform(1.0, 8.0, 64).astype(np.float32),
                        np.full(64, np.nan, np.float32)])
    a_d, b_d = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    q_d = torch.empty_like(a_d)
    assert fn(a_d.data_ptr(), b_d.data_ptr(), q_d.data_ptr(), a.size // 2, None) == 0
    torch.cuda.synchronize()
    got = q_d.cpu().numpy()
    want = a / b
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    bad = np.nonzero(~same)[0]
    detail = [(float(a[i]), float(b[i]), float(got[i]), float(want[i])) for i in bad[:8]]
    assert bad.size == 0, f"{bad.size} quotients differ (a, b, got, want): {detail}"


def test_fast_exp_envelope_on_every_argument():
    """The bitwise backward accepts the fast path's bits only inside an error
    enclosure built on softmax_exp_fast's envelope |fast(t) / CR(t) - 1| <=
    (C1 |t| + C0) 2^-24 for t in [-TMAX, 0] (constants from the library). Every
    fp32 t of that range (about 1.1e9 arguments) is checked on the device
    against exp in fp64 (within 2^-52 of the exact value): the measured
    excess over C1 |t| must stay below C0 - 1 - 2^-20 (the 1 covers the
    correct rounding of the reference, 2^-20 the fp64 reference's error)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_softmax_kv_gb300 import nvbuild
    nvbuild.build()
    lib = ctypes.CDLL(nvbuild.SELFTEST_LIB)
    c0, c1, tmax = ctypes.c_float(), ctypes.c_float(), ctypes.c_float()
    lib.csa_selftest_fast_exp_constants(ctypes.byref(c0), ctypes.byref(c1), ctypes.byref(tmax))
    lib.csa_selftest_fast_exp_envelope.argtypes = [ctypes.c_uint32, ctypes.c_uint32,
                                                   ctypes.c_void_p, ctypes.c_void_p]
    lib.csa_selftest_fast_exp_envelope.restype = ctypes.c_int32
    worst = torch.zeros(1, dtype=torch.int64, device="cuda")
    hi = int(np.float32(-tmax.value).view(np.uint32))
    assert lib.csa_selftest_fast_exp_envelope(0x80000000, hi, worst.data_ptr(), None) == 0
    torch.cuda.synchronize()
    w = float(worst.cpu().numpy().view(np.float64)[0])
    print(f"envelope: C0 {c0.value}, C1 {c1.value}, TMAX {tmax.value}; worst excess over "
          f"C1 |t| = {w:.4f} units of 2^-24")
    assert w <= c0.value - 1.0 - 2.0 ** -20
