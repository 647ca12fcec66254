"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs, element by element.

Gates (cuDNN-frontend "CSA Fused Compressor", section "Numerics"):
  * out / dkv / dscore: differing bf16 elements <= max(1, 0.1% of the tensor),
    identical NaN masks, max_abs <= 1.6e-2 against the fp32 eager-order oracle;
  * the fp64 parity rule err_gpu <= err_o32 * (1 + 1e-6) + 1e-4 (max_abs vs the
    fp64 twin over positions finite on both sides);
  * dape: max|gpu - o64| <= 1e-5 * max|o64| (normwise; entries near zero make
    an elementwise relative bound ill-posed);
  * bitwise run-to-run determinism with different NaN / canary prefills;
  * every dkv / dscore position written (NaN prefill never survives), nothing
    written outside the outputs (canary guard bands).
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import bf16_to_f64, compare_bf16, gate_bf16, problem

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_softmax_kv_gb300 as gsk
    gsk.build()
    gsk.load()
    oracle.build()


def _dev(case):
    from gpu_helpers import DeviceCase
    return DeviceCase(case)


def _fp64_parity(name, gpu_bits, o32_bits, o64):
    g, o = bf16_to_f64(gpu_bits), bf16_to_f64(o32_bits)
    fin = np.isfinite(g) & np.isfinite(o) & np.isfinite(o64)
    err_gpu = float(np.max(np.abs(g[fin] - o64[fin]))) if fin.any() else 0.0
    err_o32 = float(np.max(np.abs(o[fin] - o64[fin]))) if fin.any() else 0.0
    assert err_gpu <= err_o32 * (1 + 1e-6) + 1e-4, f"{name}: fp64 parity {err_gpu} vs {err_o32}"


def check_case(case, fp64=True, report=None):
    p = problem(case)
    dc = _dev(case)
    out = dc.fwd(prefill=0x7FC0)
    dkv, ds, dape = dc.bwd(prefill=0x7FC0)
    # determinism: a second run into differently prefilled buffers
    out2 = dc.fwd(prefill=0x1234)
    dkv2, ds2, dape2 = dc.bwd(prefill=0xFFFF)
    assert np.array_equal(out, out2), "forward not run-to-run deterministic"
    assert np.array_equal(dkv, dkv2) and np.array_equal(ds, ds2), "dkv/dscore not deterministic"
    assert np.array_equal(dape.view(np.uint32), dape2.view(np.uint32)), "dape not deterministic"

    o_out = oracle.fwd32(p, case.kv, case.score, case.ape)
    o_dkv, o_ds, o_dape = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    res = {"out": gate_bf16(out, o_out, "out"),
           "dkv": gate_bf16(dkv, o_dkv, "dkv"),
           "dscore": gate_bf16(ds, o_ds, "dscore")}
    if fp64:
        kv64, sc64 = bf16_to_f64(case.kv), bf16_to_f64(case.score)
        ape64, go64 = case.ape.astype(np.float64), bf16_to_f64(case.grad_out)
        out64 = oracle.fwd64(p, kv64, sc64, ape64)
        dkv64, ds64, dape64 = oracle.bwd64(p, kv64, sc64, ape64, go64)
        _fp64_parity("out", out, o_out, out64)
        _fp64_parity("dkv", dkv, o_dkv, dkv64)
        _fp64_parity("dscore", ds, o_ds, ds64)
        scale = max(float(np.max(np.abs(dape64))), 1e-30)
        rel = float(np.max(np.abs(dape.astype(np.float64) - dape64))) / scale
        assert rel <= 1e-5, f"dape normwise rel err {rel}"
        res["dape_rel"] = rel
    if report is not None:
        report.update(res)
    return res


@pytest.mark.parametrize("name", ["tiny", "r4d512", "r2d128rag", "r128c1"])
def test_parity_configs(name):
    case = workloads.config(name)
    res = check_case(case)
    print(name, {k: (v if not isinstance(v, dict) else (v["differing"], v["max_abs"]))
                 for k, v in res.items()})


def test_parity_headline_full_size():
    """The 256k-token headline workload at full size, through the same call the
    benchmark times; every element compared."""
    case = workloads.config("headline")
    res = check_case(case)
    print("headline", {k: (v if not isinstance(v, dict) else (v["differing"], v["max_abs"]))
                       for k, v in res.items()})


ENVELOPE = [(r, coff) for r in (2, 4, 8, 16, 32, 64, 128) for coff in (1, 2)]


@pytest.mark.parametrize("ratio,coff", ENVELOPE)
def test_parity_envelope_ragged(ratio, coff):
    """Every supported (ratio, coff): ragged segments (shorter than the ratio,
    empty, exact multiples, with tails), padding rows, tokens beyond the last
    segment, a head_dim that leaves a partial column tile."""
    rng = np.random.default_rng(ratio * 10 + coff)
    lens = [ratio - 1, 0, 3 * ratio + 1, ratio, 1, 5 * ratio + ratio // 2] + \
        list(rng.integers(1, 4 * ratio, 3))
    d = 72 if ratio <= 8 else 40
    case = workloads.make_case("env", lens, ratio, coff, d, pad_rows=3, extra_tokens=5,
                               seed=ratio + coff)
    check_case(case)


@pytest.mark.parametrize("d", [8, 64, 128, 520, 1024])
def test_parity_head_dims(d):
    case = workloads.make_case("hd", [37, 64, 19, 130], 4, 2, d, pad_rows=2, extra_tokens=3, seed=d)
    check_case(case)


def test_power_of_two_scaled_twin_is_exact():
    """x64 kv / grad_out: out and dkv scale by exactly 64, dscore and dape by
    exactly 4096, bitwise (section "Numerics", tolerance item 2)."""
    case = workloads.config("r2d128rag")
    dc = _dev(case)
    out, (dkv, ds, dape) = dc.fwd(), dc.bwd()
    scaled = workloads.config("r2d128rag")
    f = lambda bits: workloads.f32_to_bf16_bits((bf16_to_f64(bits) * 64).astype(np.float32))
    scaled.kv, scaled.grad_out = f(case.kv), f(case.grad_out)
    ds_ = _dev(scaled)
    out_s, (dkv_s, ds_s, dape_s) = ds_.fwd(), ds_.bwd()
    assert np.array_equal(bf16_to_f64(out_s), bf16_to_f64(out) * 64)
    assert np.array_equal(bf16_to_f64(dkv_s), bf16_to_f64(dkv) * 64)
    assert np.array_equal(bf16_to_f64(ds_s), bf16_to_f64(ds) * 4096)
    assert np.array_equal(dape_s.astype(np.float64), dape.astype(np.float64) * 4096)


@pytest.mark.parametrize("ratio,coff", [(128, 1), (4, 2), (128, 2)])
def test_overflowing_logits_match_oracle_nan_masks(ratio, coff):
    """score = bf16 max, ape = fp32 max: score + ape overflows to +inf, every
    output is NaN with the oracle's mask; never-read positions stay +0; the
    pattern replays bit-stable (section "Numerics", tolerance item 3)."""
    case = workloads.make_case("ovf", [8 * ratio, 3 * ratio + 1, ratio - 1], ratio, coff, 64,
                               pad_rows=2, extra_tokens=2, seed=5)
    case.score[:] = 0x7F7F
    case.ape[:] = np.finfo(np.float32).max
    p = problem(case)
    dc = _dev(case)
    out, (dkv, ds, dape) = dc.fwd(), dc.bwd()
    o_out = oracle.fwd32(p, case.kv, case.score, case.ape)
    o_dkv, o_ds, o_dape = oracle.bwd32(p, case.kv, case.score, case.ape, case.grad_out)
    for name, g, o in (("out", out, o_out), ("dkv", dkv, o_dkv), ("dscore", ds, o_ds)):
        r = compare_bf16(g, o)
        assert r["nan_mask_equal"] and r["differing"] == 0, (name, r)
    assert np.array_equal(np.isnan(dape), np.isnan(o_dape))
    out2, (dkv2, ds2, dape2) = dc.fwd(prefill=0), dc.bwd(prefill=0x3F80)
    assert np.array_equal(out, out2) and np.array_equal(dkv, dkv2) and np.array_equal(ds, ds2)
    assert np.array_equal(dape.view(np.uint32), dape2.view(np.uint32))


def test_padding_row_gradients_are_ignored():
    case = workloads.config("tiny")
    dc = _dev(case)
    ref = dc.bwd()
    go = case.grad_out.copy()
    go[case.true_rows:] = 0x7FC0  # NaN on every padding row
    from gpu_helpers import dev_bf16
    got = dc.bwd(grad_out=dev_bf16(go))
    for a, b in zip(got, ref):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_zero_capacity():
    """capacity == 0 (every segment shorter than the ratio): the forward launches
    nothing, the backward still writes exact zeros everywhere."""
    case = workloads.make_case("empty", [3, 1, 2], 4, 2, 64, seed=1)
    assert case.capacity == 0 and case.total_tokens == 6
    dc = _dev(case)
    dkv, ds, dape = dc.bwd(prefill=0x7FC0)
    assert np.all(dkv == 0) and np.all(ds == 0) and np.all(dape == 0)


@pytest.mark.parametrize("name", ["pack-r128c2d128-1x65536", "pack-r128c1d512-1x65536",
                                  "pack-r4c2d128-1x8192"])
def test_parity_page_packs(name):
    """Single-sequence packs at the sizes the page quotes kernel times for; with
    few output rows the long-window forward splits each window over several
    warps and merges the chunk states."""
    res = check_case(workloads.config(name))
    print(name, {k: (v if not isinstance(v, dict) else (v["differing"], v["max_abs"]))
                 for k, v in res.items()})


@pytest.mark.parametrize("ratio,coff,exact", [(4, 2, False), (128, 1, False), (4, 2, True)])
def test_rows_past_capacity(ratio, coff, exact):
    """cu_seqlens_comp[-1] > capacity: the forward writes the capacity rows,
    which equal the oracle's first rows; in the backward the rows without an
    output slot count as rows with zero gradient (the oracle's result with
    their grad_out zeroed), and every position is still written."""
    case = workloads.make_case("over", [8 * ratio + 1, 5 * ratio, 3 * ratio + 2], ratio, coff, 64,
                               extra_tokens=3, seed=13)
    R = case.true_rows
    C = R - 5
    full = problem(case)
    o_out = oracle.fwd32(full, case.kv, case.score, case.ape)
    go = case.grad_out.copy()
    go[C:] = 0
    o_dkv, o_ds, o_dape = oracle.bwd32(full, case.kv, case.score, case.ape, go)

    cut = workloads.make_case("over", list(case.seqlens), ratio, coff, 64, extra_tokens=3, seed=13,
                              fill=False)
    cut.kv, cut.score, cut.ape = case.kv, case.score, case.ape
    cut.capacity = C
    cut.grad_out = case.grad_out[:C].copy()
    dc = _dev(cut)
    out = dc.fwd(prefill=0x7FC0, exact=exact)
    dkv, ds, dape = dc.bwd(prefill=0x7FC0, exact=exact)
    for name, g, o in (("out", out, o_out[:C]), ("dkv", dkv, o_dkv), ("dscore", ds, o_ds)):
        r = gate_bf16(g, o, name)
        if exact:  # the oracle's bits (a zero-gradient row's dscore may be -0 there, +0 here)
            assert r["differing"] == 0, (name, r)
    scale = max(float(np.max(np.abs(o_dape))), 1e-30)
    assert float(np.max(np.abs(dape.astype(np.float64) - o_dape))) / scale <= 1e-5
