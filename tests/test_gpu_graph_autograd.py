"""CUDA-graph capture/replay of both calls and the autograd wrapper.

Both calls launch on the caller's stream with no host synchronisation and no
compilation, so a captured forward + backward replays bit-identically to the
eager calls (cuDNN-frontend "CSA Fused Compressor", section "CUDA graphs"),
also after the inputs are overwritten in place. The autograd wrapper must give
exactly the C-ABI results (section "High-level wrappers"). Beyond those
self-consistency checks, every replayed and every autograd result is gated
against the CPU oracle on the same inputs: the bf16 gate for out / dkv /
dscore (no differing bits at all in the exact mode) and 1e-5 normwise against
the fp64 twin for dape."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import oracle_gate

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_softmax_kv_gb300 as g
    g.build()
    oracle.build()
    return g


def _up(case):
    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    return dict(kv=bf16(case.kv), score=bf16(case.score), go=bf16(case.grad_out),
                ape=torch.from_numpy(case.ape).cuda(), cu=torch.from_numpy(case.cu_seqlens).cuda(),
                cuc=torch.from_numpy(case.cu_seqlens_comp).cuda())


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


@pytest.mark.parametrize("name,exact", [("tiny", False), ("r128c1", False), ("r4d512", True)])
def test_graph_replay_matches_eager(gsk, name, exact):
    case = workloads.config(name)
    t = _up(case)
    args = (case.capacity, case.ratio, case.coff, case.head_dim)
    out = torch.empty((case.capacity, case.head_dim), dtype=torch.bfloat16, device="cuda")
    dkv, ds, dape = torch.empty_like(t["kv"]), torch.empty_like(t["score"]), torch.empty_like(t["ape"])

    def step():
        gsk.csa_compress_fwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"], *args, out=out,
                             exact=exact)
        gsk.csa_compress_bwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"], *args, t["go"],
                             dkv=dkv, dscore=ds, dape=dape, exact=exact)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside capture (first-call set-up)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [_bits(x) for x in (out, dkv, ds, dape)]

    graph = torch.cuda.CUDAGraph()
    for x in (out, dkv, ds, dape):
        x.fill_(float("nan"))
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    first = [_bits(x) for x in (out, dkv, ds, dape)]
    for a, b in zip(eager, first):
        assert np.array_equal(a, b)
    oracle_gate(case, out=first[0].view(np.uint16), dkv=first[1].view(np.uint16),
                dscore=first[2].view(np.uint16), dape=dape.cpu().numpy(),
                exact=exact, label=f"{name} replay seed 0")

    # new inputs in place: the replay follows them
    other = workloads.config(name, seed=7)
    t2 = _up(other)
    for k in ("kv", "score", "go", "ape"):
        t[k].copy_(t2[k])
    graph.replay()
    torch.cuda.synchronize()
    replayed = [_bits(x) for x in (out, dkv, ds, dape)]
    oracle_gate(other, out=replayed[0].view(np.uint16), dkv=replayed[1].view(np.uint16),
                dscore=replayed[2].view(np.uint16),
                dape=dape.cpu().numpy(), exact=exact, label=f"{name} replay seed 7")
    step()
    torch.cuda.synchronize()
    for a, b in zip(replayed, [_bits(x) for x in (out, dkv, ds, dape)]):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("exact", [False, True])
def test_autograd_wrapper_matches_the_c_abi(gsk, exact):
    from gated_softmax_kv_gb300.autograd import compressor
    case = workloads.config("tiny")
    t = _up(case)
    kv = t["kv"].clone().requires_grad_(True)
    score = t["score"].clone().requires_grad_(True)
    ape = t["ape"].clone().requires_grad_(True)
    out = compressor(kv, score, ape, t["cu"], t["cuc"], case.ratio, case.coff, case.head_dim,
                     capacity=case.capacity, exact=exact)
    out.backward(t["go"])
    ref_out = gsk.csa_compress_fwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"], case.capacity,
                                   case.ratio, case.coff, case.head_dim, exact=exact)
    r_dkv, r_ds, r_dape = gsk.csa_compress_bwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"],
                                               case.capacity, case.ratio, case.coff, case.head_dim,
                                               t["go"], exact=exact)
    torch.cuda.synchronize()
    oracle_gate(case, out=_bits(out.detach()).view(np.uint16), dkv=_bits(kv.grad).view(np.uint16),
                dscore=_bits(score.grad).view(np.uint16),
                dape=ape.grad.cpu().numpy(), exact=exact, label="autograd")
    assert np.array_equal(_bits(out.detach()), _bits(ref_out))
    assert np.array_equal(_bits(kv.grad), _bits(r_dkv))
    assert np.array_equal(_bits(score.grad), _bits(r_ds))
    assert np.array_equal(_bits(ape.grad), _bits(r_dape))
    # the default capacity reads cu_seqlens_comp[-1] (true rows, no padding rows)
    out2 = compressor(kv, score, ape, t["cu"], t["cuc"], case.ratio, case.coff, case.head_dim)
    assert out2.shape[0] == case.true_rows
