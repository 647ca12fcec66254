"""csa_check_segments: the device-side preconditions of the segment arrays,
each kind of violation on its own and all of them on valid seeded workloads."""
import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_softmax_kv_gb300 as g
    g.build()
    return g


def _check(gsk, cu, cuc, T, C, ratio):
    return gsk.csa_check_segments(torch.tensor(cu, dtype=torch.int32, device="cuda"),
                                  torch.tensor(cuc, dtype=torch.int32, device="cuda"), T, C, ratio)


@pytest.mark.parametrize("name", workloads.CONFIG_NAMES)
def test_valid_workloads_pass(gsk, name):
    c = workloads.config(name, fill=False)
    assert _check(gsk, c.cu_seqlens, c.cu_seqlens_comp, c.total_tokens, c.capacity, c.ratio) == 0


def test_each_violation(gsk):
    cu, cuc = [0, 9, 9, 20], [0, 2, 2, 4]      # ratio 4: lengths 9, 0, 11
    assert _check(gsk, cu, cuc, 20, 4, 4) == 0
    assert _check(gsk, [1, 9, 9, 20], cuc, 20, 4, 4) == 1      # does not start at 0
    assert _check(gsk, [0, 9, 8, 20], cuc, 20, 4, 4) & 2      # decreasing
    assert _check(gsk, cu, [0, 2, 3, 5], 20, 5, 4) == 4       # segment 1 has 0 rows, not 1
    assert _check(gsk, cu, cuc, 19, 4, 4) == 8                # past total_tokens
    assert _check(gsk, cu, cuc, 20, 3, 4) == 16               # more rows than capacity
    # cu_seqlens_comp starting at 1 also breaks segment 0's row count
    assert _check(gsk, [0, 9, 9, 20], [1, 2, 2, 4], 20, 4, 4) == 1 | 4
    assert set(gsk.SEG_VIOLATIONS) == {1, 2, 4, 8, 16}


def test_many_segments(gsk):
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 50, 100_000)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cuc = np.concatenate([[0], np.cumsum(lens // 4)]).astype(np.int32)
    assert _check(gsk, cu, cuc, int(cu[-1]), int(cuc[-1]), 4) == 0
    bad = cuc.copy()
    bad[77_777:] += 1                                          # one segment one row too many
    assert _check(gsk, cu, bad, int(cu[-1]), int(bad[-1]), 4) == 4
