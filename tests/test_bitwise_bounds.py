"""The error bounds behind the exact mode's bitwise kernels, attacked on the CPU.

The kernels (gated_softmax_kv_gb300/csrc/csa_bitwise.cuh, csa_fwd_bitwise.cu,
csa_bwd_bitwise.cu) keep the fast arithmetic -- an exp within the envelope
(1.25 |t| + 3.25) 2^-24 of the correctly rounded one, p = RN(e RN(1/den)) --
and accept a result when an enclosure of the reference's fp32 value decides
its bf16 bits. These tests emulate that fast side in numpy fp32 with every
exp pushed to the edge of the envelope (random signs, adversarial ends), the
reference in the oracle's order with the correctly rounded exp, and check on
many random windows that

  * every weight satisfies p_ref / p - 1 in [-rho, rho], rho = rho_own + rho_com;
  * the pooled sum and S of the reference lie within
      sigma = (rho_own + 2^-23) A + rho_com |sum| + 2^-23 (sum of |partial sums|)
    of the fast ones,

with the constants of csa_bitwise.cuh restated here. A dropped or misweighted
term in that derivation lets the reference escape on some window."""
import numpy as np
import pytest

U = 2.0 ** -24
WIDE = 1.0009765625          # every term of rho widened by 2^-10
WIDEN = 1.0000152587890625   # sigma widened by 2^-16
C1, C0 = 1.25, 3.25          # the fast exp's envelope: (C1 |t| + C0) 2^-24


def rho_parts(tau, psd_over_den, W):
    own = (C1 * tau + C0 + 2.5) * U * WIDE
    com = (C0 + C1 * (W - 1) / np.e + 1.5) * U * WIDE + 2.0 * U * WIDE * psd_over_den
    return own, com


def seq_sum(terms):
    """Slot-order fp32 sum from +0; also the sum of |partial sums| after the first."""
    acc = np.zeros(terms.shape[0], np.float32)
    parts = np.zeros(terms.shape[0], np.float64)
    for k in range(terms.shape[1]):
        acc = (acc + terms[:, k]).astype(np.float32)
        if k > 0:
            parts += np.abs(acc.astype(np.float64))
    return acc, parts


def bf16(x):
    b = np.asarray(x, np.float32).view(np.uint32)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.view(np.float32)


def windows(n, W, spread, rng):
    """Exp arguments t = z - m <= 0 with one slot at 0 (the max), the rest
    spread over [-spread, 0]; tau = max |t|."""
    t = -rng.uniform(0.0, spread, (n, W))
    t[np.arange(n), rng.integers(0, W, n)] = 0.0
    t = t.astype(np.float32)
    return t, np.max(-t.astype(np.float64), axis=1)


def fast_and_ref(t, rng):
    """Reference exps (fp64 exp rounded once) and fast exps at the envelope's
    edge: e = RN(e_ref (1 + s b')) with b' one ulp inside the envelope so that
    the final rounding keeps |e / e_ref - 1| <= (C1 |t| + C0) 2^-24."""
    e_ref = np.exp(t.astype(np.float64)).astype(np.float32)
    b = (C1 * np.abs(t.astype(np.float64)) + C0 - 1.0) * U
    s = rng.choice([-1.0, 1.0], t.shape)
    e = (e_ref.astype(np.float64) * (1.0 + s * b)).astype(np.float32)
    ratio = e.astype(np.float64) / e_ref.astype(np.float64) - 1.0
    assert np.all(np.abs(ratio) <= (C1 * np.abs(t.astype(np.float64)) + C0) * U)
    return e_ref, e


def weights(e):
    den, parts = seq_sum(e)
    y = (np.float32(1.0) / den).astype(np.float32)
    p = (e * y[:, None]).astype(np.float32)
    return p, den, parts, y


def weights_ref(e_ref):
    den, _ = seq_sum(e_ref)
    return (e_ref / den[:, None]).astype(np.float32)


@pytest.mark.parametrize("W", [2, 4, 8])
@pytest.mark.parametrize("spread", [3.0, 12.0, 40.0])
def test_weights_within_rho(W, spread):
    rng = np.random.default_rng(100 * W + int(spread))
    t, tau = windows(200_000, W, spread, rng)
    e_ref, e = fast_and_ref(t, rng)
    p, den, psd, y = weights(e)
    p_ref = weights_ref(e_ref)
    own, com = rho_parts(tau, psd * y.astype(np.float64), W)
    rho = own + com
    rel = np.abs(p_ref.astype(np.float64) / p.astype(np.float64) - 1.0)
    ok = p > 0
    ratio = rel[ok] / rho[:, None].repeat(W, 1)[ok]
    assert np.all(ratio <= 1.0), float(np.max(ratio))
    # the attack is not idle: the worst weight reaches over half of rho
    # (0.53-0.90 measured over these W and spreads)
    assert np.max(ratio) > 0.45


def _check_sum(x, p, p_ref, tau, psd_over_den, W):
    """The reference's slot-order sum of RN(x p_ref) against the fast one of RN(x p)."""
    terms = (x * p).astype(np.float32)
    acc, pss = seq_sum(terms)
    acc_ref, _ = seq_sum((x * p_ref).astype(np.float32))
    aabs = np.sum(np.abs(terms.astype(np.float64)), axis=1)
    own, com = rho_parts(tau, psd_over_den, W)
    sigma = ((own + 2 * U * WIDE) * aabs + com * np.abs(acc.astype(np.float64)) + 2 * U * WIDE * pss) * WIDEN
    gap = np.abs(acc_ref.astype(np.float64) - acc.astype(np.float64))
    assert np.all(gap <= sigma), float(np.max(gap / np.maximum(sigma, 1e-300)))
    # the common part counts against |sum|: never wider than counting all of
    # rho against sum |terms| (|sum| exceeds sum |terms| by its roundings at
    # most), and much narrower when the terms cancel
    old = ((own + com + 2 * U * WIDE) * aabs + 2 * U * WIDE * pss) * WIDEN
    assert np.all(sigma <= old * (1 + 8 * U))
    assert np.any(sigma < 0.8 * old)
    return float(np.max(gap / np.maximum(sigma, 1e-300)))


@pytest.mark.parametrize("W", [2, 4, 8])
@pytest.mark.parametrize("spread", [3.0, 12.0])
def test_pooled_sum_and_S_within_sigma(W, spread):
    rng = np.random.default_rng(7 * W + int(spread))
    n = 200_000
    t, tau = windows(n, W, spread, rng)
    e_ref, e = fast_and_ref(t, rng)
    p, den, psd, y = weights(e)
    p_ref = weights_ref(e_ref)
    psd_over_den = psd * y.astype(np.float64)
    kv = bf16(rng.standard_normal((n, W)))
    # forward: the pooled sum of RN(p kv)
    worst_fwd = _check_sum(kv, p, p_ref, tau, psd_over_den, W)
    # backward: S = sum RN(dp p), dp = RN(g kv) exact for bf16 g and kv
    g = bf16(rng.standard_normal(n))
    dp = (g[:, None] * kv).astype(np.float32)
    worst_bwd = _check_sum(dp, p, p_ref, tau, psd_over_den, W)
    assert worst_fwd < 1.0 and worst_bwd < 1.0
    # the attack is not idle (0.30-0.56 of sigma measured over these W and spreads)
    assert max(worst_fwd, worst_bwd) > 0.2


def test_a_dropped_term_is_caught():
    """The attack bites: without the common part of rho the reference escapes."""
    rng = np.random.default_rng(5)
    W, n = 8, 200_000
    t, tau = windows(n, W, 3.0, rng)
    e_ref, e = fast_and_ref(t, rng)
    p, den, psd, y = weights(e)
    p_ref = weights_ref(e_ref)
    own, _ = rho_parts(tau, psd * y.astype(np.float64), W)
    rel = np.abs(p_ref.astype(np.float64) / p.astype(np.float64) - 1.0)
    assert np.any(rel > own[:, None])
