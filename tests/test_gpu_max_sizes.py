"""GPU parity at the largest sizes the ABI accepts (int32 flat offsets,
cuDNN-frontend "CSA Fused Compressor", section "Support surface").

Two problems:
  * total_tokens * coff * head_dim just below 2^31 (ratio 4, coff 2,
    head_dim 512: 2,097,151 tokens, 32 segments of up to 65536 tokens, a
    ragged last segment and tokens past the last segment);
  * capacity * head_dim just below 2^31 (ratio 2, coff 1, head_dim 8:
    268,435,455 output rows over a 120-token pack, almost all of them
    padding rows).

The first is too large to generate token by token in the time a test has,
so kv and score are a seeded block of an odd number of tokens (65537) from
the input generator, repeated along the tokens on the device: an offset that
wrapped or was truncated anywhere would read different values. Segments are
independent, so the oracle runs segment by segment over the whole problem and
every element is compared: out, dkv and dscore under the bf16 gate (default
mode) and bit for bit (exact mode); dape normwise against the sum of the
oracle's per-segment dape.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import compare_bf16, gate_bf16

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


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _strict(got, want):
    both_nan = np.isnan(oracle.bf16_bits_to_f64(got)) & np.isnan(oracle.bf16_bits_to_f64(want))
    return int(np.count_nonzero((got != want) & ~both_nan))


def _run(gsk, t, meta, exact):
    out = gsk.csa_compress_fwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"], *meta,
                               exact=exact)
    dkv, ds, dape = gsk.csa_compress_bwd(t["kv"], t["score"], t["ape"], t["cu"], t["cuc"], *meta,
                                         t["go"], exact=exact)
    torch.cuda.synchronize()
    return out, dkv, ds, dape


def test_token_offsets_at_the_int32_limit(gsk):
    ratio, coff, d = 4, 2, 512
    width = coff * d
    T = (1 << 31) // width - 1               # T * coff * d = 2^31 - 1024
    extra = 5                                # tokens past the last segment
    lens = [65536] * 31
    lens.append(T - extra - sum(lens))       # 65530: a 2-token tail
    R = sum(n // ratio for n in lens)
    C = R + 64                               # 64 padding rows
    assert T * width < (1 << 31) and C * d < (1 << 31)
    case = workloads.make_case("max-tokens", lens, ratio, coff, d, pad_rows=64,
                               extra_tokens=extra, seed=0, fill=False)
    assert case.total_tokens == T and case.capacity == C

    P, PG = 65537, 16383                     # periods (tokens, output rows), both odd
    base_kv = workloads.normal_bf16(11, workloads.STREAM_KV, P * width, 1.0).reshape(P, width)
    base_sc = workloads.normal_bf16(11, workloads.STREAM_SCORE, P * width, 1.5).reshape(P, width)
    base_go = workloads.normal_bf16(11, workloads.STREAM_GRAD, PG * d, 1.0).reshape(PG, d)
    ape = workloads.normal_f64(11, workloads.STREAM_APE, ratio * width, 0.25).astype(
        np.float32).reshape(ratio, width)

    reps = -(-T // P)
    t = dict(kv=_dev_bf16(base_kv).repeat(reps, 1)[:T], score=_dev_bf16(base_sc).repeat(reps, 1)[:T],
             go=_dev_bf16(base_go).repeat(-(-C // PG), 1)[:C], ape=torch.from_numpy(ape).cuda(),
             cu=torch.from_numpy(case.cu_seqlens).cuda(), cuc=torch.from_numpy(case.cu_seqlens_comp).cuda())
    meta = (C, ratio, coff, d)
    res = {}
    for exact in (False, True):
        out, dkv, ds, dape = _run(gsk, t, meta, exact)
        res[exact] = dict(out=out, dkv=dkv, ds=ds, dape=dape.cpu().numpy().astype(np.float64))
        # padding rows: first-block semantics from token 0, i.e. row 0 bit for bit
        pad = _host_bits(out[R:])
        assert np.all(pad == _host_bits(out[0:1])), "padding rows differ from row 0"
        # tokens past the last segment and the last segment's tail: exact +0
        tail0 = int(case.cu_seqlens[-2]) + (lens[-1] // ratio) * ratio
        for x in (dkv, ds):
            assert not torch.any(x[tail0:].view(torch.int16) != 0), "unread positions not +0"

    dape_sum = np.zeros((ratio, width), np.float64)
    cu, cuc = case.cu_seqlens.astype(np.int64), case.cu_seqlens_comp.astype(np.int64)
    worst = {}
    for s, n in enumerate(lens):
        t0, t1, r0, r1 = cu[s], cu[s + 1], cuc[s], cuc[s + 1]
        kv = base_kv[np.arange(t0, t1) % P]
        sc = base_sc[np.arange(t0, t1) % P]
        go = base_go[np.arange(r0, r1) % PG]
        sub = workloads.make_case("seg", [n], ratio, coff, d, fill=False)
        p = oracle.Problem(sub.cu_seqlens, sub.cu_seqlens_comp, n, r1 - r0, ratio, coff, d)
        o_out = oracle.fwd32(p, kv, sc, ape)
        o_dkv, o_ds, o_dape = oracle.bwd32(p, kv, sc, ape, go)
        dape_sum += o_dape.astype(np.float64)
        for exact in (False, True):
            r = res[exact]
            got = (_host_bits(r["out"][r0:r1]), _host_bits(r["dkv"][t0:t1]), _host_bits(r["ds"][t0:t1]))
            for name, g, o in zip(("out", "dkv", "dscore"), got, (o_out, o_dkv, o_ds)):
                if exact:
                    n_bad = _strict(g, o)
                    assert n_bad <= 2, f"exact {name}, segment {s}: {n_bad} elements differ"
                else:
                    gate_bf16(g, o, f"{name} segment {s}")
                    worst[name] = max(worst.get(name, 0), compare_bf16(g, o)["differing"])
    scale = max(float(np.max(np.abs(dape_sum))), 1e-30)
    for exact in (False, True):
        rel = float(np.max(np.abs(res[exact]["dape"] - dape_sum))) / scale
        assert rel <= 1e-5, f"dape (exact={exact}) normwise rel err {rel}"
    print("max tokens: worst differing per segment", worst)


def test_output_rows_at_the_int32_limit(gsk):
    ratio, coff, d = 2, 1, 8
    C = (1 << 31) // d - 1                   # capacity * head_dim = 2^31 - 8
    case = workloads.make_case("max-rows", [37, 64, 19], ratio, coff, d, pad_rows=0, seed=4)
    R = case.true_rows
    meta = (C, ratio, coff, d)
    go = torch.full((C, d), float("nan"), dtype=torch.bfloat16, device="cuda")  # padding: ignored
    go[:R] = _dev_bf16(case.grad_out[:R])
    t = dict(kv=_dev_bf16(case.kv), score=_dev_bf16(case.score), go=go,
             ape=torch.from_numpy(case.ape).cuda(), cu=torch.from_numpy(case.cu_seqlens).cuda(),
             cuc=torch.from_numpy(case.cu_seqlens_comp).cuda())
    # the oracle on the true rows plus one padding row
    p = oracle.Problem(case.cu_seqlens, case.cu_seqlens_comp, case.total_tokens, R + 1, ratio,
                       coff, d)
    o_out = oracle.fwd32(p, case.kv, case.score, case.ape)
    go_host = np.concatenate([case.grad_out[:R], np.zeros((1, d), np.uint16)])  # padding row: ignored
    o_dkv, o_ds, o_dape = oracle.bwd32(p, case.kv, case.score, case.ape, go_host)
    for exact in (False, True):
        out, dkv, ds, dape = _run(gsk, t, meta, exact)
        # every padding row equals the last one, which the oracle computes
        last = out[C - 1:C]
        assert not torch.any(out[R:].view(torch.int16) != last.view(torch.int16)), "padding rows differ"
        got = np.concatenate([_host_bits(out[:R]), _host_bits(last)])
        for name, g, o in (("out", got, o_out), ("dkv", _host_bits(dkv), o_dkv),
                           ("dscore", _host_bits(ds), o_ds)):
            if exact:
                assert _strict(g, o) == 0, f"exact {name} differs"
            else:
                gate_bf16(g, o, name)
        o64 = o_dape.astype(np.float64)
        rel = float(np.max(np.abs(dape.cpu().numpy() - o64))) / max(float(np.max(np.abs(o64))), 1e-30)
        assert rel <= 1e-5, f"dape (exact={exact}) normwise rel err {rel}"
        del out, dkv, ds, dape
        torch.cuda.empty_cache()
