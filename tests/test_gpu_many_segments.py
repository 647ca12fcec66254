"""Problems with many segments through the C ABI against the oracle.

Every kernel but the bitwise backward copies cu_seqlens and cu_seqlens_comp
into shared memory when each has at most 1024 entries (1023 segments) and
otherwise looks rows up in the global arrays. These cases sit on both sides of
that boundary, for the small- and long-window kernels of both directions (the
small backward's next-row prefetch at windows of up to 4 slots included) and
for the exact mode, with empty segments, segments shorter than the ratio,
tails, padding rows and tokens past the last segment."""
import numpy as np
import pytest

import workloads

from test_gpu_parity import check_case

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def many(nseg: int, ratio: int, coff: int, d: int, seed: int):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 3 * ratio, nseg)
    lens[rng.integers(0, nseg)] = max(int(lens.max()), ratio)  # at least one full block
    return workloads.make_case(f"many{nseg}-r{ratio}c{coff}d{d}", lens.tolist(), ratio, coff, d,
                               pad_rows=3, extra_tokens=ratio // 2 + 1, seed=seed)


@pytest.mark.parametrize("nseg", [1023, 1024, 2500])
@pytest.mark.parametrize("ratio,coff,d", [(2, 2, 64), (4, 2, 128), (8, 1, 64), (16, 2, 64),
                                          (128, 1, 64)])
def test_many_segments(nseg, ratio, coff, d):
    case = many(nseg, ratio, coff, d, seed=nseg + 7 * ratio + coff)
    assert len(case.seqlens) == nseg
    check_case(case)


@pytest.mark.parametrize("nseg", [1023, 1024])
@pytest.mark.parametrize("ratio,coff", [(2, 2), (4, 2), (8, 1)])
def test_many_segments_exact(nseg, ratio, coff):
    from test_gpu_exact import check_exact
    check_exact(many(nseg, ratio, coff, 64, seed=3 * nseg + ratio + coff))
