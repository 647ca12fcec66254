"""Test-side helpers: oracle problem construction, an independent statement of
the window geometry, bf16 comparisons and the tolerance gates."""
from __future__ import annotations

import numpy as np

import oracle
import workloads


def problem(case: workloads.Case) -> oracle.Problem:
    return oracle.Problem(case.cu_seqlens, case.cu_seqlens_comp, case.total_tokens,
                          case.capacity, case.ratio, case.coff, case.head_dim)


def eager_windows(seqlens, ratio: int, coff: int, capacity: int):
    """Window token lists built the slow way, as an eager gather pictures them
    (cuDNN-frontend "CSA Fused Compressor", section "Semantics"): walk the
    segments, cut each into blocks of `ratio` tokens, drop the tail, and give
    block i the token list [previous block | own block] (coff == 2; the
    previous block is absent on a segment's first block) or [own block]
    (coff == 1). Static-capacity rows repeat a first block from token 0.

    Returns a list (one entry per output row) of lists of window slots; a slot
    is (token, half, ape_row) with half 0 = first-half columns, 1 = second
    half, or None for a masked slot."""
    rows = []
    start = 0
    for seg_len in seqlens:
        n_blocks = int(seg_len) // ratio
        for i in range(n_blocks):
            own = [start + i * ratio + t for t in range(ratio)]
            if coff == 2:
                if i == 0:
                    prev = [None] * ratio
                else:
                    prev = [(start + (i - 1) * ratio + t, 0, t) for t in range(ratio)]
                rows.append(prev + [(tok, 1, t) for t, tok in enumerate(own)])
            else:
                rows.append([(tok, 0, t) for t, tok in enumerate(own)])
        start += int(seg_len)
    while len(rows) < capacity:
        own = [(t, 1 if coff == 2 else 0, t) for t in range(ratio)]
        rows.append(([None] * ratio + own) if coff == 2 else own)
    return rows[:capacity]


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return oracle.bf16_bits_to_f64(bits)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 -> bf16 nearest-even (finite inputs), for building inputs."""
    return workloads.f32_to_bf16_bits(np.asarray(x, dtype=np.float64).astype(np.float32))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def compare_bf16(got: np.ndarray, want: np.ndarray):
    """Differing count (bit patterns, +0 == -0, NaN == NaN), NaN-mask equality
    and max_abs over positions finite on both sides."""
    g = np.asarray(got, dtype=np.uint16)
    w = np.asarray(want, dtype=np.uint16)
    gf = bf16_to_f64(g)
    wf = bf16_to_f64(w)
    gnan, wnan = np.isnan(gf), np.isnan(wf)
    same = (g == w) | ((gf == 0) & (wf == 0)) | (gnan & wnan)
    differing = int(np.count_nonzero(~same))
    fin = np.isfinite(gf) & np.isfinite(wf)
    max_abs = float(np.max(np.abs(gf[fin] - wf[fin]))) if np.any(fin) else 0.0
    return {"differing": differing, "numel": int(g.size), "nan_mask_equal": bool(np.array_equal(gnan, wnan)),
            "max_abs": max_abs}


def gate_bf16(got, want, name: str, frac: float = 0.001, max_abs: float = 1.6e-2):
    """The headline tolerance gate: differing <= max(1, 0.1% of numel), equal NaN
    masks, max_abs <= 1.6e-2."""
    r = compare_bf16(got, want)
    allowed = max(1, int(np.floor(frac * r["numel"])))
    assert r["nan_mask_equal"], f"{name}: NaN masks differ"
    assert r["differing"] <= allowed, f"{name}: {r['differing']} differing > {allowed} ({r})"
    assert r["max_abs"] <= max_abs, f"{name}: max_abs {r['max_abs']} > {max_abs}"
    return r


def strict_differing(got, want) -> int:
    """Elements whose bf16 bits differ, NaN payloads aside (signed zeros count)."""
    g = np.asarray(got, dtype=np.uint16)
    w = np.asarray(want, dtype=np.uint16)
    both_nan = np.isnan(bf16_to_f64(g)) & np.isnan(bf16_to_f64(w))
    return int(np.count_nonzero((g != w) & ~both_nan))


def oracle_gate(case, out=None, dkv=None, dscore=None, dape=None, exact: bool = False,
                allowed: int = 0, label: str = ""):
    """Gate whichever outputs are given against the oracle on the same inputs:
    out / dkv / dscore against O32 (the bf16 gate; with `exact`, at most
    `allowed` elements whose bits differ), dape normwise against O64 (1e-5).
    Returns the comparison figures."""
    p = problem(case)
    res = {}
    if out is not None:
        o_out = oracle.fwd32(p, case.kv, case.score, case.ape)
        res["out"] = gate_bf16(out, o_out, f"{label} out")
        if exact:
            n = strict_differing(out, o_out)
            assert n <= allowed, f"{label} out: {n} elements differ from the oracle"
    if dkv is not None or dscore is not None:
        o_dkv, o_ds, _ = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
        for name, g, o in (("dkv", dkv, o_dkv), ("dscore", dscore, o_ds)):
            if g is None:
                continue
            res[name] = gate_bf16(g, o, f"{label} {name}")
            if exact:
                n = strict_differing(g, o)
                assert n <= allowed, f"{label} {name}: {n} elements differ from the oracle"
    if dape is not None:
        _, _, dape64 = oracle.bwd64(p, bf16_to_f64(case.kv), bf16_to_f64(case.score),
                                    case.ape.astype(np.float64), bf16_to_f64(case.grad_out))
        scale = max(float(np.max(np.abs(dape64))), 1e-30)
        rel = float(np.max(np.abs(np.asarray(dape, dtype=np.float64) - dape64))) / scale
        assert rel <= 1e-5, f"{label} dape: normwise rel err {rel}"
        res["dape_rel"] = rel
    return res
