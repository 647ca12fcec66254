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


def test_two_host_threads_on_two_streams(gsk):
    """Two host threads, each on its own stream, run forward + backward on
    different inputs at the same time, several times over: the library's
    shared state (the dape workspace pool, the occupancy and shared-memory
    caches) is behind locks and each call's workspace is stream-ordered, so
    every result equals the same calls made alone."""
    import threading
    cases = [workloads.config("r4d512"), workloads.config("r128c1")]

    def upload(case):
        return dict(kv=_bf16(case.kv), score=_bf16(case.score), go=_bf16(case.grad_out),
                    ape=torch.from_numpy(case.ape).cuda(), cu=torch.from_numpy(case.cu_seqlens).cuda(),
                    cuc=torch.from_numpy(case.cu_seqlens_comp).cuda())

    dev = [upload(c) for c in cases]
    torch.cuda.synchronize()  # the uploads ran on the default stream

    def run(i, stream):
        c, t = cases[i], dev[i]
        meta = (c.capacity, c.ratio, c.coff, c.head_dim)
        with torch.cuda.stream(stream):
            out = gsk.csa_compress_fwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"], *meta,
                                       stream=stream)
            dkv, ds, dape = gsk.csa_compress_bwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"],
                                                 *meta, t["go"], stream=stream)
        stream.synchronize()
        return [_bits(x) for x in (out, dkv, ds, dape)]

    alone = [run(i, torch.cuda.Stream()) for i in range(2)]
    results = {}

    def worker(i):
        s = torch.cuda.Stream()
        results[i] = [run(i, s) for _ in range(4)]

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    for i in range(2):
        for rep in results[i]:
            for a, b in zip(alone[i], rep):
                assert np.array_equal(a, b)


def test_two_host_threads_on_two_streams_exact_mode(gsk):
    """The same for the exact mode's kernels (its own launch shapes and
    workspace sizes): concurrent calls on two streams give the bits of the
    same calls made alone."""
    import threading
    cases = [workloads.config("r4d512"), workloads.config("r2d128rag")]
    dev = []
    for case in cases:
        dev.append(dict(kv=_bf16(case.kv), score=_bf16(case.score), go=_bf16(case.grad_out),
                        ape=torch.from_numpy(case.ape).cuda(),
                        cu=torch.from_numpy(case.cu_seqlens).cuda(),
                        cuc=torch.from_numpy(case.cu_seqlens_comp).cuda()))
    torch.cuda.synchronize()

    def run(i, stream):
        c, t = cases[i], dev[i]
        meta = (c.capacity, c.ratio, c.coff, c.head_dim)
        with torch.cuda.stream(stream):
            out = gsk.csa_compress_fwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"], *meta,
                                       stream=stream, exact=True)
            dkv, ds, dape = gsk.csa_compress_bwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"],
                                                 *meta, t["go"], stream=stream, exact=True)
        stream.synchronize()
        return [_bits(x) for x in (out, dkv, ds, dape)]

    alone = [run(i, torch.cuda.Stream()) for i in range(2)]
    results = {}

    def worker(i):
        s = torch.cuda.Stream()
        results[i] = [run(i, s) for _ in range(3)]

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    for i in range(2):
        for rep in results[i]:
            for a, b in zip(alone[i], rep):
                assert np.array_equal(a, b)
