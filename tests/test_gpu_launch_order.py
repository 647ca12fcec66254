"""Stream order across the library's own kernels.

Every kernel is launched with programmatic stream serialization: its launch
may overlap the previous kernel's tail, and griddepcontrol.wait at its start
holds it until that grid's writes are visible. These tests make one call
consume what the previous call just wrote on the same stream, with no host
synchronisation in between, and require the bits of the same calls separated
by a device-wide synchronize."""
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


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "r4d512", "r128c1"])
def test_backward_consumes_the_forward_output_in_stream_order(gsk, name):
    """grad_out of the backward is the forward's `out`, written by the kernel
    launched just before it; then a second forward overwrites `out` while
    nothing else has waited for the backward's reads of it."""
    case = workloads.config(name)
    kv, score = _bf16(case.kv), _bf16(case.score)
    ape = torch.from_numpy(case.ape).cuda()
    cu = torch.from_numpy(case.cu_seqlens).cuda()
    cuc = torch.from_numpy(case.cu_seqlens_comp).cuda()
    meta = (case.capacity, case.ratio, case.coff, case.head_dim)
    # a different kv for the second forward, so that its `out` differs
    kv2 = _bf16(workloads.config(name, seed=3).kv)

    def run(sync: bool):
        out = torch.full((case.capacity, case.head_dim), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        dkv = torch.full_like(kv, float("nan"))
        ds = torch.full_like(score, float("nan"))
        dape = torch.full_like(ape, float("nan"))
        torch.cuda.synchronize()
        gsk.csa_compress_fwd(kv, score, ape, cu, cuc, *meta, out=out)
        if sync:
            torch.cuda.synchronize()
        gsk.csa_compress_bwd(kv, score, ape, cu, cuc, *meta, out, dkv=dkv, dscore=ds, dape=dape)
        if sync:
            torch.cuda.synchronize()
        gsk.csa_compress_fwd(kv2, score, ape, cu, cuc, *meta, out=out)
        torch.cuda.synchronize()
        return [_bits(x) for x in (out, dkv, ds, dape)]

    ordered = run(sync=True)
    chained = run(sync=False)
    for a, b, what in zip(ordered, chained, ("second out", "dkv", "dscore", "dape")):
        assert np.array_equal(a, b), what
