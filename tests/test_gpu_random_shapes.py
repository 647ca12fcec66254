"""Seeded random shapes through the C ABI against the oracle.

The launch shapes depend on the problem: the long-window forward splits a
row's window over 1 to 8 warps by the problem's row count, the backward picks
its thread layout by window length and head_dim, and the dAPE reduce picks its
lane count from the number of partials. Each case draws a (ratio, coff), a
head_dim (a multiple of 8, on and off the compiled 128 / 512), ragged segment
lengths (empty, shorter than the ratio, with tails), padding rows and tokens
past the last segment, and must pass the parity gates of test_gpu_parity.py
with bitwise run-to-run determinism."""
import numpy as np
import pytest

import workloads

from test_gpu_parity import check_case

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

RATIOS = (2, 4, 8, 16, 32, 64, 128)
HEAD_DIMS = (8, 16, 24, 40, 64, 72, 128, 136, 256, 512)


def draw(seed: int):
    rng = np.random.default_rng(1000 + seed)
    ratio = int(rng.choice(RATIOS))
    coff = int(rng.integers(1, 3))
    d = int(rng.choice(HEAD_DIMS))
    nseg = int(rng.integers(1, 12))
    # keep the oracle's work (rows x window x head_dim) around a few million
    budget = max(ratio, 3_000_000 // (coff * ratio * d) * ratio)
    hi = max(2, min(budget // nseg, 64 * ratio))
    lens = rng.integers(0, hi, nseg)
    lens[rng.integers(0, nseg)] = max(int(lens.max()), ratio)  # at least one full block
    pad = int(rng.integers(0, 6))
    extra = int(rng.integers(0, 2 * ratio))
    return workloads.make_case(f"rand{seed}", lens.tolist(), ratio, coff, d, pad_rows=pad,
                               extra_tokens=extra, seed=seed)


@pytest.mark.parametrize("seed", range(24))
def test_random_shape(seed):
    case = draw(seed)
    res = check_case(case)
    print(seed, (case.ratio, case.coff, case.head_dim, len(case.seqlens), case.total_tokens,
                 case.capacity), {k: (v if not isinstance(v, dict) else (v["differing"], v["max_abs"]))
                                  for k, v in res.items()})


EXACT_SHAPES = ((2, 1), (4, 1), (8, 1), (2, 2), (4, 2))


@pytest.mark.parametrize("seed", range(12))
def test_random_shape_exact(seed):
    """The exact mode on seeded random shapes of its envelope (windows of at
    most 8 slots): out, dkv and dscore carry the oracle's bits."""
    from test_gpu_exact import check_exact
    rng = np.random.default_rng(5000 + seed)
    ratio, coff = EXACT_SHAPES[int(rng.integers(0, len(EXACT_SHAPES)))]
    d = int(rng.choice(HEAD_DIMS))
    nseg = int(rng.integers(1, 12))
    hi = max(2, min(3_000_000 // (coff * ratio * d) * ratio // nseg, 400 * ratio))
    lens = rng.integers(0, hi, nseg)
    lens[rng.integers(0, nseg)] = max(int(lens.max()), ratio)
    case = workloads.make_case(f"xrand{seed}", lens.tolist(), ratio, coff, d,
                               pad_rows=int(rng.integers(0, 6)),
                               extra_tokens=int(rng.integers(0, 2 * ratio)), seed=100 + seed)
    print(seed, (ratio, coff, d, len(lens), case.total_tokens), check_exact(case))
