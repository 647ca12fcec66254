"""Host logic of bench.py without a GPU: the multi-rank bookkeeping (barrier
and max over ranks, as torchrun runs it with one process per GPU) on two
gloo ranks, the algorithmic byte counts and the reference arm's rank rule."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    sys.argv = ["bench.py"]
    import bench
    r = bench.Ranks(rank, world, backend="gloo")
    r.barrier()
    worst = r.max(1.5 * (rank + 1))   # each rank's elapsed time; the job's is the max
    r.barrier()
    r.close()
    q.put((rank, worst))


def test_two_gloo_ranks_take_the_max_elapsed_time():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 3.0), (1, 3.0)]


def test_single_process_ranks_are_noops():
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks(0, 1)
    r.barrier()
    assert r.max(2.5) == 2.5


def test_algorithmic_bytes_per_token_at_the_headline():
    import bench
    import workloads
    case = workloads.config("headline", fill=False)
    fwd, bwd = bench.algorithmic_bytes(case)
    # kv and score read once (4 B per token column), out written per capacity row
    assert fwd == 262144 * 1024 * 4 + case.capacity * 512 * 2 + 4 * 1024 * 4
    # plus dkv / dscore written in full, grad_out of the true rows, dape written
    assert bwd == 2 * 262144 * 1024 * 4 + case.true_rows * 512 * 2 + 2 * 4 * 1024 * 4
    assert abs(fwd / 262144 - 4352) / 4352 < 0.01
    assert abs(bwd / 262144 - 8448) / 8448 < 0.01


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench

    class A:
        steps, warmup, tokens, workload = 1, 0, 262144, "headline"

    assert bench.run_reference(A(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""


def test_cpu_baseline_reports_all_cores_and_one_thread():
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    case = workloads.make_case("tiny", [37, 64, 19, 200], 4, 2, 64, pad_rows=4, seed=0)
    rate, cores, desc, single = bench.oracle_rate(case, budget_s=0.05, min_tokens=64)
    assert rate > 0 and cores >= 1 and "O32 fwd + bwd" in desc
    assert single["value_1thread"] > 0
    assert "one thread" in single["sample_1thread"]


def test_reference_arm_line_carries_the_contract_keys(capsys):
    import json
    import bench

    class A:
        steps, warmup, tokens, workload = 1, 1, 4096, "headline"

    assert bench.run_reference(A(), rank=0, world=1) in (0, None)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_clock_sampler_summarises_the_timed_window(monkeypatch):
    """The NVML sampler (read-only queries from a host thread) reports the
    median SM clock and the union of active reasons over the samples taken
    between mark() and unmark(), with the sample counts."""
    import time

    import bench

    class FakeNvml:
        def __init__(self, *a):
            self.n = 0

        def sm_max_mhz(self):
            return 2070

        def sm_mhz(self):
            self.n += 1
            return 1500 if self.n < 1000 and self.phase == "warm" else 2070

        def reasons(self):
            return 0x4 if self.phase == "timed" else 0x8 * (self.phase == "after")

        def power_w(self):
            return 900.0

        def close(self):
            pass

    fake = FakeNvml()
    fake.phase = "warm"
    monkeypatch.setattr(bench, "_Nvml", lambda *a: fake)
    c = bench.ClockSampler(0, period_s=0.0005)
    c.start()
    time.sleep(0.02)
    fake.phase = "timed"
    c.mark()
    time.sleep(0.03)
    c.unmark()
    fake.phase = "after"
    time.sleep(0.02)
    r = c.stop()
    assert r["samples_timed"] >= 5 and r["samples"] > r["samples_timed"]
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]  # hw_slowdown came after the window
    assert r["power_w_max"] == 900.0
