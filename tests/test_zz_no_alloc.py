"""The allocation-free backward (csa_compress_bwd_noalloc), against the oracle
and against the regular backward (csa_compress_bwd).

csa_compress_bwd_noalloc serves callers that cannot allocate device memory
while the backward runs (for example a process whose device memory all
belongs to its own allocator from start-up, or a time-critical loop that
must stay out of the CUDA allocator). It keeps the backward's dape partials in
a fixed device buffer of the library instead of pool memory. Its results are
gated against the CPU oracle like every other backward (the bf16 gate for dkv
and dscore, 1e-5 normwise against the fp64 twin for dape) and must carry the
regular backward's bits, on two calls in a row (the second finds the first
call's partials in the buffer). This file runs last so that a failure here
comes after every other test has run; it builds and uploads everything it
needs, so it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import oracle_gate

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

SCRATCH_ERR = 6  # CSA_ERR_SCRATCH


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_softmax_kv_gb300 as gsk
    gsk.build()
    oracle.build()
    return gsk


def _upload(case):
    dev = torch.device("cuda")

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    return dict(kv=bf16(case.kv), score=bf16(case.score), go=bf16(case.grad_out),
                ape=torch.from_numpy(case.ape).to(dev),
                cu=torch.from_numpy(case.cu_seqlens).to(dev),
                cuc=torch.from_numpy(case.cu_seqlens_comp).to(dev))


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _noalloc(lib, case, t, dkv, ds, dape):
    """One call through the C ABI; returns its status (0 = CSA_OK)."""
    stream = torch.cuda.current_stream().cuda_stream
    return lib.load().csa_compress_bwd_noalloc(
        t["kv"].data_ptr(), t["score"].data_ptr(), t["ape"].data_ptr(), t["cu"].data_ptr(),
        t["cuc"].data_ptr(), case.num_seqs, case.total_tokens, case.capacity, case.ratio,
        case.coff, case.head_dim, t["go"].data_ptr(), dkv.data_ptr(), ds.data_ptr(),
        dape.data_ptr(), stream)


def _check_twice(lib, case):
    t = _upload(case)
    args = (case.capacity, case.ratio, case.coff, case.head_dim)
    ref_dkv, ref_ds, ref_dape = lib.csa_compress_bwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"],
                                                     *args, t["go"])
    torch.cuda.synchronize()
    ref_dkv, ref_ds, ref_dape = _bits(ref_dkv), _bits(ref_ds), ref_dape.cpu().numpy()
    gated = None
    for call in range(2):  # the second call finds the first call's partials in the buffer
        dkv = torch.full_like(t["kv"], float("nan"))
        ds = torch.full_like(t["score"], float("nan"))
        dape = torch.full_like(t["ape"], float("nan"))
        assert _noalloc(lib, case, t, dkv, ds, dape) == 0
        torch.cuda.synchronize()
        got_dkv, got_ds, got_dape = _bits(dkv), _bits(ds), dape.cpu().numpy()
        if gated is None:
            gated = oracle_gate(case, dkv=got_dkv, dscore=got_ds, dape=got_dape,
                                label=f"{case.name} no-alloc call {call}")
        # same kernels and launch shape as the regular backward: the same bits
        assert np.array_equal(got_dkv, ref_dkv) and np.array_equal(got_ds, ref_ds)
        assert np.array_equal(got_dape.view(np.uint32), ref_dape.view(np.uint32))
    return gated


@pytest.mark.parametrize("name", ["tiny", "r4d512", "r128c1", "headline"])
def test_noalloc_backward_matches_the_oracle_and_the_regular_backward_twice(lib, name):
    print(name, _check_twice(lib, workloads.config(name)))


def test_noalloc_scratch_limit_boundary(lib):
    """The buffer's edge on real buffers: the backward caps its row groups so
    that groups * ratio * coff * head_dim stays near 2.5 Mi floats at most,
    except when a single group alone is larger. Ratio 128, coff 2, one output
    row: head_dim 16384 needs exactly the 4 Mi floats of the buffer (accepted,
    checked against the oracle and the regular backward, twice), head_dim 16392
    needs 8192 floats more (refused with CSA_ERR_SCRATCH before anything is
    launched: the outputs keep their NaN prefill, and the regular backward
    takes the same problem from its pool)."""
    fits = workloads.make_case("noalloc-4mi", [128], 128, 2, 16384, seed=3)
    assert fits.capacity == 1 and 128 * 2 * 16384 == 4 * 1024 * 1024
    _check_twice(lib, fits)

    over = workloads.make_case("noalloc-4mi+", [128], 128, 2, 16392, seed=3)
    t = _upload(over)
    dkv = torch.full_like(t["kv"], float("nan"))
    ds = torch.full_like(t["score"], float("nan"))
    dape = torch.full_like(t["ape"], float("nan"))
    assert _noalloc(lib, over, t, dkv, ds, dape) == SCRATCH_ERR
    torch.cuda.synchronize()
    assert np.all(np.isnan(dkv.float().cpu().numpy())) and np.all(np.isnan(dape.cpu().numpy()))
    r_dkv, r_ds, r_dape = lib.csa_compress_bwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"],
                                               over.capacity, 128, 2, 16392, t["go"])
    torch.cuda.synchronize()
    oracle_gate(over, dkv=_bits(r_dkv), dscore=_bits(r_ds), dape=r_dape.cpu().numpy(),
                label="regular backward past the no-alloc limit")


def test_noalloc_rejects_problems_beyond_its_buffer(lib):
    # ratio 128, coff 2, head_dim 16392: one dape copy alone is
    # 128 * 2 * 16392 floats > 4 Mi; rejected before anything is launched
    # (the fake, aligned addresses are never dereferenced)
    fake = 0x10000
    with pytest.raises(lib.CsaError) as err:
        lib.csa_compress_bwd_noalloc_ptr(fake, fake, fake, fake, fake, 1, 256, 1, 128, 2, 16392,
                                         fake, fake, fake, fake, 0)
    assert err.value.status == SCRATCH_ERR
    # the same call straight through the C ABI (argument types declared by load())
    st = lib.load().csa_compress_bwd_noalloc(fake, fake, fake, fake, fake, 1, 256, 1, 128, 2, 16392,
                                             fake, fake, fake, fake, None)
    assert st == SCRATCH_ERR
