"""The allocation-free backward (csa_compress_bwd_noalloc) against the regular
one (csa_compress_bwd).

csa_compress_bwd_noalloc serves callers that cannot allocate device memory
while the backward runs (for example a process whose device memory all
belongs to its own allocator from start-up, or a time-critical loop that
must stay out of the CUDA allocator). It keeps the backward's dape partials in
a fixed device buffer of the library instead of pool memory. This file runs
last so that a failure here comes after every other test has run; it builds
and uploads everything it needs, so it also passes on its own in a fresh
process.
"""
import ctypes

import numpy as np
import pytest

import workloads
from helpers import gate_bf16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_softmax_kv_gb300 as gsk
    gsk.build()
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


@pytest.mark.parametrize("name", ["tiny", "r4d512", "r128c1"])
def test_noalloc_backward_matches_regular_backward_twice(lib, name):
    case = workloads.config(name)
    t = _upload(case)
    args = (case.capacity, case.ratio, case.coff, case.head_dim)
    ref_dkv, ref_ds, ref_dape = lib.csa_compress_bwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"],
                                                     *args, t["go"])
    torch.cuda.synchronize()
    ref_dkv, ref_ds, ref_dape = _bits(ref_dkv), _bits(ref_ds), ref_dape.cpu().numpy()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # the second call finds the first call's partials in the buffer
        dkv = torch.full_like(t["kv"], float("nan"))
        ds = torch.full_like(t["score"], float("nan"))
        dape = torch.full_like(t["ape"], float("nan"))
        lib.csa_compress_bwd_noalloc_ptr(
            t["kv"].data_ptr(), t["score"].data_ptr(), t["ape"].data_ptr(), t["cu"].data_ptr(),
            t["cuc"].data_ptr(), case.num_seqs, case.total_tokens, *args, t["go"].data_ptr(),
            dkv.data_ptr(), ds.data_ptr(), dape.data_ptr(), stream)
        torch.cuda.synchronize()
        got_dkv, got_ds, got_dape = _bits(dkv), _bits(ds), dape.cpu().numpy()
        gate_bf16(got_dkv, ref_dkv, f"dkv call {call}")
        gate_bf16(got_ds, ref_ds, f"dscore call {call}")
        rel = float(np.max(np.abs(got_dape.astype(np.float64) - ref_dape))) / \
            max(1e-30, float(np.max(np.abs(ref_dape))))
        assert rel <= 1e-5, f"dape call {call}: rel {rel}"
        # same kernels and launch shape: expected to agree bit for bit
        assert np.array_equal(got_dkv, ref_dkv) and np.array_equal(got_ds, ref_ds)
        assert np.array_equal(got_dape.view(np.uint32), ref_dape.view(np.uint32))


def test_noalloc_rejects_problems_beyond_its_buffer(lib):
    # ratio 128, coff 2, head_dim 16392: one dape copy alone is
    # 128 * 2 * 16392 floats > 4 Mi; rejected before anything is launched
    # (the fake, aligned addresses are never dereferenced)
    fake = 0x10000
    with pytest.raises(lib.CsaError) as err:
        lib.csa_compress_bwd_noalloc_ptr(fake, fake, fake, fake, fake, 1, 256, 1, 128, 2, 16392,
                                         fake, fake, fake, fake, 0)
    assert err.value.status == 6
    # the same call straight through the C ABI (argument types set by the wrapper above)
    st = lib.load().csa_compress_bwd_noalloc(fake, fake, fake, fake, fake, 1, 256, 1, 128, 2, 16392,
                                             fake, fake, fake, fake, None)
    assert st == 6
