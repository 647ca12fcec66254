"""The ncu harness's parsing and summaries (no GPU): ncu's CSV layouts, unit
scaling, launch shares and the DRAM traffic record bench.py reads."""
import json

import pytest

import bench
from gated_softmax_kv_gb300 import ncu_harness as nh

LAUNCH_LOG = """==PROF== Connected to process 1 (python3)
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python3","h","void unnamed>::fwd_small_kernel<4, 2, 512>(FwdParams)","1","7","(64, 4, 1)","(1, 304, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","ns","180000"
"1","1","python3","h","void unnamed>::bwd_small_kernel<4, 2, 512>(BwdParams)","1","7","(128, 2, 1)","(1, 304, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","usecond","350"
"2","1","python3","h","unnamed>::dape_reduce_kernel(const float4 *, int, long, float4 *)","1","7","(8, 64, 1)","(128, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","ns","5000"
"3","1","python3","h","void unnamed>::fwd_small_kernel<4, 2, 512>(FwdParams)","1","7","(64, 4, 1)","(1, 304, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","ns","182000"
==PROF== Disconnected from process 1
"""

RAW = """"ID","Kernel Name","gpu__time_duration.sum","dram__bytes_read.sum","dram__bytes_write.sum","l1tex__t_sectors_pipe_lsu_mem_global_op_st.sum","launch__registers_per_thread"
"","","us","Mbyte","Kbyte","sector",""
"0","void unnamed>::fwd_small_kernel<4, 2, 512>(FwdParams)","54.0","268.0","11000.0","531250","124"
"1","void unnamed>::bwd_small_kernel<4, 2, 512>(BwdParams)","96.0","285.0","222000.0","8387500","128"
"2","unnamed>::dape_reduce_kernel(const float4 *, int, long, float4 *)","6.0","5.0","0","512","32"
"3","void unnamed>::fwd_small_kernel<4, 2, 512>(FwdParams)","55.0","999.0","0","0","124"
"""


def _only(raw, kernel):
    """The rows of one kernel, as a single-kernel capture holds them."""
    lines = raw.splitlines()
    return nh.parse_raw("\n".join(lines[:2] + [ln for ln in lines[2:] if kernel in ln]))


def test_short_names():
    assert nh.short_name("void unnamed>::fwd_small_kernel<4, 2, 512>(FwdParams)") == \
        "fwd_small_kernel<4, 2, 512>"
    assert nh.short_name("unnamed>::dape_reduce_kernel(const float4 *, int, long, float4 *)") == \
        "dape_reduce_kernel"


def test_launch_summary_and_shares():
    s = nh.parse_launches(LAUNCH_LOG)
    assert list(s) == ["fwd_small_kernel<4, 2, 512>", "bwd_small_kernel<4, 2, 512>",
                       "dape_reduce_kernel"]
    f = s["fwd_small_kernel<4, 2, 512>"]
    assert f["launches"] == 2 and f["total_us"] == pytest.approx(362.0)
    assert s["bwd_small_kernel<4, 2, 512>"]["total_us"] == pytest.approx(350.0)  # usecond
    table = nh.launches_table(s)
    # shares: 362 / 717, 350 / 717, 5 / 717, largest first
    lines = table.splitlines()[2:]
    assert lines[0].startswith("| `fwd_small_kernel") and "50.5%" in lines[0]
    assert "48.8%" in lines[1] and "0.7%" in lines[2]


def test_raw_units_scale_to_bytes():
    k = nh.parse_raw(RAW)
    assert [n for n, _ in k][:3] == ["fwd_small_kernel<4, 2, 512>", "bwd_small_kernel<4, 2, 512>",
                                     "dape_reduce_kernel"]
    assert nh.metric_value(k[0][1], "dram__bytes_read.sum") == pytest.approx(268e6)
    assert nh.metric_value(k[0][1], "dram__bytes_write.sum") == pytest.approx(11e6)  # Kbyte
    assert nh.metric_value(k[0][1], "gpu__time_duration.sum") == pytest.approx(54.0)
    assert nh.metric_value(k[0][1], "no_such_metric") is None
    assert "—" in nh.capture_table(k)  # metrics absent from the capture


def test_traffic_record_from_single_kernel_captures():
    reports = {"fwd": _only(RAW, "fwd_small"), "bwd": _only(RAW, "bwd_small"),
               "reduce": _only(RAW, "dape_reduce")}
    rec = nh.traffic_record(reports, 65536, "cmd")
    f, b = rec["csa_compress_fwd"], rec["csa_compress_bwd"]
    # forward: the first launch only; traffic = DRAM reads + bytes of global stores
    assert f["dram_read_bytes_per_unit"] == pytest.approx(268e6 / 65536)
    assert f["dram_write_bytes_per_unit"] == pytest.approx(11e6 / 65536)
    assert f["l2_write_bytes_per_unit"] == pytest.approx(531250 * 32 / 65536)
    assert f["dram_bytes_per_unit"] == pytest.approx((268e6 + 531250 * 32) / 65536)
    # backward call: its kernel plus the dape reduce
    assert b["dram_bytes_per_unit"] == pytest.approx((285e6 + 5e6 + (8387500 + 512) * 32) / 65536)
    assert b["kernel"] == "bwd_small_kernel<4, 2, 512> + dape_reduce_kernel"
    for key in ("csa_compress_fwd", "csa_compress_bwd"):
        assert rec[key]["source_hash"] == bench.source_hash(rec[key]["sources"])
    json.dumps(rec)


def test_traffic_record_refuses_multi_kernel_or_missing_captures():
    both = nh.parse_raw(RAW)  # three kernels in one capture
    with pytest.raises(ValueError):
        nh.traffic_record({"fwd": both, "bwd": _only(RAW, "bwd_small"),
                           "reduce": _only(RAW, "dape_reduce")}, 65536, "cmd")
    with pytest.raises(ValueError):
        nh.traffic_record({"fwd": _only(RAW, "fwd_small"), "bwd": _only(RAW, "bwd_small")},
                          65536, "cmd")


def test_capture_takes_one_kernel_name():
    assert nh.single_kernel_name("bwd_small_kernel") == "bwd_small_kernel"
    for bad in ("(fwd|bwd)_small", "fwd_small|dape_reduce", "", "bwd.*", "a b"):
        with pytest.raises(ValueError):
            nh.single_kernel_name(bad)
    with pytest.raises(SystemExit):  # --kernel is required
        nh.main(["capture"])


def test_committed_record_covers_the_bench_keys():
    with open(nh.TRAFFIC) as f:
        rec = json.load(f)
    for key, spec in nh.TRAFFIC_KERNELS.items():
        assert rec[key]["sources"] == spec["sources"]
        assert rec[key]["dram_bytes_per_unit"] > 4096  # at least kv + score of a token
