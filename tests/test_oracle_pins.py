"""Pins of the CPU oracle to facts that do not come from the oracle itself:
hand-worked values, closed forms of special cases, invariances the page's
semantics imply, finite differences, IEEE/library routines and an independent
statement of the window geometry.

Subject: cuDNN-frontend "CSA Fused Compressor" (sections "Semantics",
"Numerics", "Support surface")."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from helpers import (bf16_to_f64, bf16_ulp, eager_windows, f64_to_bf16_bits, problem)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "handworked_r2_coff2.json")
F32_EPS = 2.0 ** -23


# ---------------------------------------------------------------- scalar pins


def test_exp_is_correctly_rounded(oracle_lib):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.uniform(-104.0, 88.7, 4000), rng.uniform(-20.0, 0.0, 4000),
                         np.array([0.0, -0.0, 1.0, -1.0, 88.72, -87.33, -103.9, 1e-30])])
    xs = xs.astype(np.float32)
    for x in xs:
        want = np.float32(float(mpmath.exp(mpmath.mpf(float(x)))))
        got = np.float32(oracle.exp_f32(float(x)))
        assert got == want, (float(x), float(got), float(want))
    assert oracle.exp_f32(float("-inf")) == 0.0
    assert math.isinf(oracle.exp_f32(float("inf")))
    assert math.isnan(oracle.exp_f32(float("nan")))


def test_bf16_rounding_matches_library(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    # ties, near-ties, subnormals, max finite, overflow to inf
    special = np.array([0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001, 0x00008000, 0x00018000,
                        0x00000001, 0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0xFF7FFFFF, 0x80000000,
                        0x7F800000, 0xFF800000], dtype=np.uint32)
    vals = np.concatenate([bits, special]).view(np.float32)
    vals = vals[~np.isnan(vals)]
    want = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)
    assert oracle.f32_to_bf16(float("nan")) == 0x7FC0


def test_products_and_sums_round_separately(oracle_lib):
    # (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24: the product rounds (tie to even) to
    # 1 + 2^-11, so with two roundings a*b - (1 + 2^-11) is exactly 0; a fused
    # multiply-add would return 2^-24.
    a = 1.0 + 2.0 ** -12
    c = -(1.0 + 2.0 ** -11)
    assert oracle.mul_add_f32(a, a, c) == 0.0


# ---------------------------------------------------------------- geometry


GEOMETRY_CASES = [
    ([37, 64, 19], 4, 2, 64, 4),
    ([5, 2, 1, 9, 3], 2, 2, 8, 3),
    ([5, 2, 1, 9, 3], 2, 1, 8, 2),
    ([300, 129, 127, 0, 256], 128, 1, 8, 2),
    ([300, 129, 256], 128, 2, 8, 1),
    ([7, 1, 4], 1, 1, 8, 2),
]


@pytest.mark.parametrize("lens,r,coff,d,pad", GEOMETRY_CASES)
def test_window_geometry_matches_eager_gather(oracle_lib, lens, r, coff, d, pad):
    case = workloads.make_case("geom", lens, r, coff, d, pad_rows=pad, fill=False)
    p = problem(case)
    table = eager_windows(lens, r, coff, case.capacity)
    assert len(table) == case.capacity
    for b, slots in enumerate(table):
        base, first, padding = oracle.row_map(p, b)
        assert padding == (b >= case.true_rows)
        for j in (0, d // 2, d - 1):
            for k, slot in enumerate(slots):
                tok, col, arow, valid = oracle.window_slot(p, base, first, j, k)
                if slot is None:
                    assert not valid
                else:
                    assert valid
                    want_tok, half, want_arow = slot
                    assert (tok, col, arow) == (want_tok, half * d + j, want_arow)


def test_validation_rejects_inconsistent_inputs(oracle_lib):
    case = workloads.make_case("v", [9, 4], 4, 2, 8, pad_rows=1, fill=False)
    p = problem(case)
    assert oracle.validate(p) == 0
    bad = [
        dict(cu_seqlens=np.array([1, 9, 13], np.int32)),               # does not start at 0
        dict(cu_seqlens=np.array([0, 9, 8], np.int32)),                # decreasing
        dict(cu_seqlens_comp=np.array([0, 2, 4], np.int32)),           # 4 // 4 = 1, not 2
        dict(capacity=2),                                              # fewer than the true rows
        dict(total_tokens=12),                                         # cu_seqlens[-1] > T
        dict(coff=3),
        dict(ratio=0),
    ]
    for change in bad:
        q = oracle.Problem(**{**p.__dict__, **change})
        assert oracle.validate(q) != 0, change
    tiny = oracle.Problem(np.array([0, 2], np.int32), np.array([0, 0], np.int32), 2, 1, 4, 2, 8)
    assert oracle.validate(tiny) != 0  # capacity > 0 needs total_tokens >= ratio


# ---------------------------------------------------------------- golden


def _golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    return g


def _num(s: str) -> float:
    ln3 = math.log(3.0)
    s = s.replace(" ", "")
    if "LN3" in s:
        return ln3 + float(s.replace("LN3", "") or 0.0)
    return float(Fraction(s))


def _arr(rows):
    return np.array([[_num(v) for v in row] for row in rows], dtype=np.float64)


def _golden_problem(g):
    pr = g["problem"]
    return oracle.Problem(np.array(pr["cu_seqlens"], np.int32), np.array(pr["cu_seqlens_comp"], np.int32),
                          pr["total_tokens"], pr["capacity"], pr["ratio"], pr["coff"], pr["head_dim"])


def test_golden_geometry(oracle_lib):
    g = _golden()
    p = _golden_problem(g)
    for b in range(p.capacity):
        base, first, _ = oracle.row_map(p, b)
        for k, slot in enumerate(g["problem"]["windows"][f"row{b}"]):
            tok, col, arow, valid = oracle.window_slot(p, base, first, 0, k)
            if slot is None:
                assert not valid
            else:
                assert valid and [tok, col, arow] == slot


def test_golden_weighted_fp64(oracle_lib):
    g = _golden()
    p = _golden_problem(g)
    c = g["cases"]["weighted_fp64"]
    kv, score, ape, go = _arr(c["kv"]), _arr(c["score"]), _arr(c["ape"]), _arr(c["grad_out"])
    out = oracle.fwd64(p, kv, score, ape)
    dkv, dscore, dape = oracle.bwd64(p, kv, score, ape, go)
    e = c["expected"]
    np.testing.assert_allclose(out, _arr(e["out"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dkv, _arr(e["dkv"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dscore, _arr(e["dscore"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dape, _arr(e["dape"]), rtol=0, atol=1e-13)


def test_golden_uniform_fp32_bitwise(oracle_lib):
    g = _golden()
    p = _golden_problem(g)
    c = g["cases"]["uniform_bf16"]
    kv = f64_to_bf16_bits(_arr(c["kv"]))
    score = f64_to_bf16_bits(_arr(c["score"]))
    ape = _arr(c["ape"]).astype(np.float32)
    go = f64_to_bf16_bits(_arr(c["grad_out"]))
    out = oracle.fwd32(p, kv, score, ape)
    dkv, dscore, dape = oracle.bwd32(p, kv, score, ape, go)
    e = c["expected"]
    assert np.array_equal(out, f64_to_bf16_bits(_arr(e["out"])))
    assert np.array_equal(dkv, f64_to_bf16_bits(_arr(e["dkv"])))
    assert np.array_equal(dscore, f64_to_bf16_bits(_arr(e["dscore"])))
    assert np.array_equal(dape, _arr(e["dape"]).astype(np.float32))


# ---------------------------------------------------------------- closed forms


def _window_gather(case, table, arr_bits, j):
    """Values of a [T, coff*d] bf16 tensor over each row's window for column j
    (masked slots -> NaN), via the independent eager table."""
    d = case.head_dim
    vals = np.full((case.capacity, case.coff * case.ratio), np.nan)
    for b, slots in enumerate(table):
        for k, s in enumerate(slots):
            if s is not None:
                tok, half, _ = s
                vals[b, k] = bf16_to_f64(arr_bits[tok, half * d + j])
    return vals


@pytest.mark.parametrize("name", ["tiny", "ragged_r2", "coff1_r4"])
def test_uniform_logits_give_the_window_mean(oracle_lib, name):
    lens, r, coff, d, pad = {"tiny": ([37, 64, 19], 4, 2, 64, 4),
                             "ragged_r2": ([5, 2, 1, 9, 3, 40], 2, 2, 16, 3),
                             "coff1_r4": ([37, 64, 19], 4, 1, 16, 2)}[name]
    case = workloads.make_case(name, lens, r, coff, d, pad_rows=pad, seed=3)
    case.score[:] = f64_to_bf16_bits(np.full(case.score.shape, 0.75))
    case.ape[:] = 0.0
    p = problem(case)
    out = oracle.fwd32(p, case.kv, case.score, case.ape)
    table = eager_windows(lens, r, coff, case.capacity)
    for j in range(d):
        vals = _window_gather(case, table, case.kv, j)
        mean = np.nanmean(vals, axis=1)
        got = bf16_to_f64(out[:, j])
        assert np.all(np.abs(got - mean) <= bf16_ulp(mean)), j


@pytest.mark.parametrize("coff", [1, 2])
def test_dominant_score_selects_one_token(oracle_lib, coff):
    lens, r, d = [37, 64, 19, 3], 4, 16
    case = workloads.make_case("dom", lens, r, coff, d, pad_rows=3, seed=4)
    p = problem(case)
    table = eager_windows(lens, r, coff, case.capacity)
    dom = {}
    for b, slots in enumerate(table):
        for j in range(d):
            # a valid slot; padding rows share row 0's window, so they pick row 0's slot
            k = (coff - 1) * r + (j + (b if b < case.true_rows else 0)) % r
            tok, half, _ = slots[k]
            case.score[tok, half * d + j] = f64_to_bf16_bits(np.array([60.0]))[0]
            dom[(b, j)] = (tok, half * d + j)
    out = oracle.fwd32(p, case.kv, case.score, case.ape)
    dkv, dscore, _ = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    for (b, j), (tok, col) in dom.items():
        assert out[b, j] == case.kv[tok, col]
        if b < case.true_rows:
            assert dkv[tok, col] == case.grad_out[b, j]
            assert bf16_to_f64(dscore[tok, col]) == 0.0


def test_ratio_one_own_block_is_identity(oracle_lib):
    lens = [7, 1, 4]
    case = workloads.make_case("id", lens, 1, 1, 24, pad_rows=2, seed=5)
    p = problem(case)
    out = oracle.fwd32(p, case.kv, case.score, case.ape)
    t = case.true_rows
    assert np.array_equal(out[:t], case.kv[:t])
    assert np.array_equal(out[t:], np.repeat(case.kv[:1], case.capacity - t, axis=0))
    dkv, dscore, dape = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    assert np.array_equal(dkv[:t], case.grad_out[:t])
    assert np.all(bf16_to_f64(dscore) == 0.0)
    assert np.all(dape == 0.0)


# ---------------------------------------------------------------- invariances


def test_first_block_mask_tails_and_segment_independence(oracle_lib):
    lens, r, coff, d = [37, 64, 19], 4, 2, 64
    case = workloads.make_case("tiny", lens, r, coff, d, pad_rows=4, seed=0)
    p = problem(case)
    out0 = oracle.fwd32(p, case.kv, case.score, case.ape)
    dkv0, ds0, dape0 = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    cu = case.cu_seqlens
    rng = np.random.default_rng(6)

    # segment 0's tokens do not reach segment 1's rows (first block masked)
    kv, sc = case.kv.copy(), case.score.copy()
    kv[cu[0]:cu[1]] = rng.integers(0, 0x7F00, kv[cu[0]:cu[1]].shape, dtype=np.uint16)
    sc[cu[0]:cu[1]] = rng.integers(0, 0x7F00, sc[cu[0]:cu[1]].shape, dtype=np.uint16)
    out1 = oracle.fwd32(p, kv, sc, case.ape)
    rows1 = slice(case.cu_seqlens_comp[1], case.cu_seqlens_comp[3])
    assert np.array_equal(out1[rows1], out0[rows1])

    # tail tokens (37 % 4 = 1, 19 % 4 = 3) are never read
    tails = [36, 117, 118, 119]
    kv, sc = case.kv.copy(), case.score.copy()
    kv[tails] = 0x7F00
    sc[tails] = 0x7F00
    assert np.array_equal(oracle.fwd32(p, kv, sc, case.ape), out0)
    for tok in tails:
        assert np.all(dkv0[tok] == 0) and np.all(ds0[tok] == 0)

    # a segment's last block: its first-half columns are never consumed
    for s in range(3):
        last = cu[s] + (lens[s] // r - 1) * r
        assert np.all(dkv0[last:last + r, :d] == 0) and np.all(ds0[last:last + r, :d] == 0)


def test_padding_rows(oracle_lib):
    case = workloads.make_case("pad", [37, 64, 19], 4, 2, 32, pad_rows=5, seed=7)
    p = problem(case)
    out = oracle.fwd32(p, case.kv, case.score, case.ape)
    t = case.true_rows
    # segment 0 has >= ratio tokens, so its first row reads the same window
    for b in range(t, case.capacity):
        assert np.array_equal(out[b], out[0])
    ref = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    for fill in (0x7FC0, 0x7149, 0xFF80):  # NaN, ~1e30, -inf
        go = case.grad_out.copy()
        go[t:] = fill
        got = oracle.bwd32(p, case.kv, case.score, case.ape, go)
        for a, b in zip(got, ref):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_extra_tokens_beyond_last_segment_get_zero_grads(oracle_lib):
    case = workloads.make_case("extra", [9, 6], 4, 2, 8, pad_rows=1, extra_tokens=5, seed=8)
    p = problem(case)
    dkv, ds, _ = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    end = case.cu_seqlens[-1]
    assert case.total_tokens == end + 5
    assert np.all(dkv[end:] == 0) and np.all(ds[end:] == 0)


# ---------------------------------------------------------------- scaling / non-finite


@pytest.mark.parametrize("r,coff,d", [(4, 2, 32), (2, 2, 16), (4, 1, 16)])
def test_power_of_two_scaling_is_exact(oracle_lib, r, coff, d):
    case = workloads.make_case("s", [37, 64, 19, 5], r, coff, d, pad_rows=2, seed=9)
    p = problem(case)

    def scale(bits, k):  # multiply bf16 values by 2^k exactly (exponent shift)
        return f64_to_bf16_bits(bf16_to_f64(bits) * 2.0 ** k)

    kv64, go64 = scale(case.kv, 6), scale(case.grad_out, 6)
    assert np.array_equal(bf16_to_f64(kv64), bf16_to_f64(case.kv) * 64)
    out = bf16_to_f64(oracle.fwd32(p, case.kv, case.score, case.ape))
    out_s = bf16_to_f64(oracle.fwd32(p, kv64, case.score, case.ape))
    assert np.array_equal(out_s, out * 64)
    dkv, ds, dape = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    dkv_s, ds_s, dape_s = oracle.bwd32(p, kv64, case.score, case.ape, go64)
    assert np.array_equal(bf16_to_f64(dkv_s), bf16_to_f64(dkv) * 64)
    assert np.array_equal(bf16_to_f64(ds_s), bf16_to_f64(ds) * 4096)
    assert np.array_equal(dape_s.astype(np.float64), dape.astype(np.float64) * 4096)


def test_overflowing_logits_poison_every_output(oracle_lib):
    case = workloads.make_case("ovf", [37, 64, 19], 4, 2, 16, pad_rows=2, seed=10)
    case.score[:] = 0x7F7F                      # bf16 max
    case.ape[:] = np.finfo(np.float32).max      # fp32 max: score + ape = +inf
    p = problem(case)
    out = bf16_to_f64(oracle.fwd32(p, case.kv, case.score, case.ape))
    assert np.all(np.isnan(out))
    dkv, ds, dape = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    consumed = np.zeros(dkv.shape, dtype=bool)
    for slots in eager_windows(case.seqlens, 4, 2, case.true_rows):
        for s in slots:
            if s is not None:
                consumed[s[0], s[1] * 16:(s[1] + 1) * 16] = True
    assert np.all(np.isnan(bf16_to_f64(dkv)[consumed]))
    assert np.all(np.isnan(bf16_to_f64(ds)[consumed]))
    assert np.all(dkv[~consumed] == 0) and np.all(ds[~consumed] == 0)
    assert np.all(np.isnan(dape))


# ---------------------------------------------------------------- fp64 twin


FD_CASES = [
    ([5, 3, 1, 6], 2, 2, 3, 2),   # r=2 overlapping, 1-token segment, padding
    ([5, 3, 4], 2, 1, 2, 1),      # own-block window
    ([9, 4, 2], 4, 2, 2, 1),      # r=4 overlapping, a segment shorter than r
]


@pytest.mark.parametrize("lens,r,coff,d,pad", FD_CASES)
def test_fp64_gradients_match_central_differences(oracle_lib, lens, r, coff, d, pad):
    case = workloads.make_case("fd", lens, r, coff, d, pad_rows=pad, extra_tokens=1, seed=11)
    p = problem(case)
    kv, sc = bf16_to_f64(case.kv), bf16_to_f64(case.score)
    ape = case.ape.astype(np.float64)
    go = bf16_to_f64(case.grad_out)
    rows = min(case.true_rows, case.capacity)
    go_loss = go.copy()
    go_loss[rows:] = 0.0   # padding rows carry no gradient

    def loss(kv_, sc_, ape_):
        return float(np.sum(go_loss * oracle.fwd64(p, kv_, sc_, ape_, nthreads=1)))

    dkv, dsc, dape = oracle.bwd64(p, kv, sc, ape, go, nthreads=1)
    for name, arr, an in (("kv", kv, dkv), ("score", sc, dsc), ("ape", ape, dape)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            h = 1e-6 * max(1.0, abs(arr[idx]))
            args = [kv, sc, ape]
            which = ("kv", "score", "ape").index(name)
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args[which] = plus
            lp = loss(*args)
            args[which] = minus
            lm = loss(*args)
            fd[idx] = (lp - lm) / (2 * h)
        scale = max(1e-12, np.max(np.abs(an)))
        assert np.max(np.abs(fd - an)) <= 1e-6 * scale, name


def test_softmax_gradient_sums_to_zero(oracle_lib):
    for coff in (1, 2):
        case = workloads.make_case("inv", [37, 64, 19, 200], 4, coff, 16, pad_rows=2, seed=12)
        p = problem(case)
        _, _, dape = oracle.bwd64(p, bf16_to_f64(case.kv), bf16_to_f64(case.score),
                                  case.ape.astype(np.float64), bf16_to_f64(case.grad_out))
        d = case.head_dim
        per_col = dape[:, :d].sum(axis=0) + (dape[:, d:].sum(axis=0) if coff == 2 else 0.0)
        assert np.max(np.abs(per_col)) <= 1e-12 * max(1.0, np.max(np.abs(dape)))


def test_fp32_twin_close_to_fp64_twin(oracle_lib):
    case = workloads.config("tiny")
    p = problem(case)
    out32, out32f = oracle.fwd32(p, case.kv, case.score, case.ape, want_f32=True)
    out64 = oracle.fwd64(p, bf16_to_f64(case.kv), bf16_to_f64(case.score), case.ape.astype(np.float64))
    assert np.max(np.abs(out32f.astype(np.float64) - out64)) <= 64 * F32_EPS
    assert np.array_equal(out32, f64_to_bf16_bits(out32f.astype(np.float64)))
    # after the bf16 rounding the fp32 twin is within half a bf16 step (+ the fp32 error)
    err = np.abs(bf16_to_f64(out32) - out64)
    assert np.all(err <= 0.5 * bf16_ulp(out64) + 64 * F32_EPS)
    dkv32, ds32, dape32 = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    dkv64, ds64, dape64 = oracle.bwd64(p, bf16_to_f64(case.kv), bf16_to_f64(case.score),
                                       case.ape.astype(np.float64), bf16_to_f64(case.grad_out))
    assert np.all(np.abs(bf16_to_f64(dkv32) - dkv64) <= 0.5 * bf16_ulp(dkv64) + 64 * F32_EPS)
    assert np.all(np.abs(bf16_to_f64(ds32) - ds64) <= 0.5 * bf16_ulp(ds64) + 64 * F32_EPS)
    assert np.max(np.abs(dape32 - dape64)) <= 1e-5 * np.max(np.abs(dape64))


def test_oracle_threading_does_not_change_results(oracle_lib):
    case = workloads.config("tiny")
    p = problem(case)
    a = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out, nthreads=1)
    b = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out, nthreads=4)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
