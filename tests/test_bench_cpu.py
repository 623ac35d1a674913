"""bench.py without a GPU: the multi-rank timing path on two gloo ranks, the
whole-job throughput formula, and the reference arm's JSON line (CPU oracle on
a small problem; under torchrun only rank 0 prints)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.reduce_max(dist, 10.0 * (rank + 1), "cpu")
        value = bench.throughput_tops(3 * 2.0 * 8192 ** 3, 4, world, slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    expect = 3 * 2.0 * 8192 ** 3 * 4 * 2 / 20e-3 / 1e12
    for rank, slowest, value in got:
        assert slowest == 20.0
        assert value == pytest.approx(expect)


def test_throughput_formula_single_rank():
    assert bench.reduce_max(None, 3.5, "cpu") == 3.5
    # 2 N^3 ops in 1 ms at N = 1000 is 2 TOPS
    assert bench.throughput_tops(2e9, 1, 1, 1.0) == pytest.approx(2.0)


def _run_bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args,
                          capture_output=True, text=True, env=env, timeout=300)


def test_reference_arm_json_line():
    r = _run_bench(["--impl", "reference", "--n", "256", "--steps", "2", "--warmup", "1"], {})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TOPS" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--n", "256", "--steps", "2", "--warmup", "1"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_peak_fractions_denominators():
    per = {"fp16_tflops": 1500.0, "int8_tops": 1125.0, "int4_tops": 2250.0}
    mhz = {"fp16": 1500.0, "int8": 1800.0, "int4": 1800.0}
    f = bench.peak_fractions(per, 1500.0, mhz, 152)
    assert f["fp16"]["frac_nominal"] == pytest.approx(1500 / 2250)
    assert f["int8"]["frac_nominal"] == pytest.approx(1125 / 4500)
    assert f["fp16"]["frac_pipe_measured"] == pytest.approx(1.0)
    assert f["int8"]["pipe"] == "kind::f16" and f["int8"]["frac_pipe_measured"] == pytest.approx(0.75)
    assert f["int4"]["pipe"] == "kind::f8f6f4" and f["int4"]["pipe_peak_measured"] == pytest.approx(3000.0)
    # per-SM rate x SMs x the kernel's own clock: 8192 FLOP per clock for the
    # FP16 kind, 16384 for the E4M3 kind
    assert f["fp16"]["pipe_peak_clock_adjusted"] == pytest.approx(8192 * 152 * 1.5e9 / 1e12)
    assert f["int8"]["pipe_peak_clock_adjusted"] == pytest.approx(8192 * 152 * 1.8e9 / 1e12)
    assert f["int4"]["pipe_peak_clock_adjusted"] == pytest.approx(16384 * 152 * 1.8e9 / 1e12)
    assert f["int4"]["frac_pipe_clock_adjusted"] == pytest.approx(2250 / (16384 * 152 * 1.8e9 / 1e12))
    g = bench.peak_fractions(per, 1500.0, {"fp16": None, "int8": None, "int4": None}, 152)
    assert g["fp16"]["pipe_peak_clock_adjusted"] is None and g["fp16"]["frac_pipe_clock_adjusted"] is None


def test_traffic_record_is_tied_to_the_kernel_sources(tmp_path, monkeypatch):
    rec = tmp_path / "traffic.txt"
    rec.write_text(f"kernel: x\nsource_sha256_16: {bench.kernel_source_hash()}\n"
                   "dram_bytes_read: 1.0e9\ndram_bytes_write: 0.25e9\n")
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(rec))
    t, _ = bench.traffic_record()
    assert t == pytest.approx(1.25e9)
    rec.write_text("kernel: x\nsource_sha256_16: 0000000000000000\ndram_bytes_read: 1\ndram_bytes_write: 1\n")
    t, why = bench.traffic_record()
    assert t is None and "stale" in why
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(tmp_path / "absent.txt"))
    assert bench.traffic_record()[0] is None


def test_sweep_oracle_time_measured_and_extrapolated():
    import datagen
    A, B = datagen.s8_operands(64)
    full = bench._oracle_time("s8", A, B, 64, 2, budget_s=100.0)
    assert full["rows_timed"] == 64 and not full["extrapolated"] and full["seconds"] > 0
    part = bench._oracle_time("s8", A, B, 64, 2, budget_s=0.0)
    assert part["rows_timed"] == 2 and part["extrapolated"]
    assert part["tops"] == pytest.approx(2.0 * 64 ** 3 / part["seconds"] / 1e12)


def test_kernel_identity_ignores_comments_only():
    """The traffic record is tied to the kernel's code: comment and
    whitespace edits keep its hash, any code edit changes it."""
    import os
    base = {n: open(os.path.join(bench.ROOT, "precision_tensor_core_gb300", "csrc", n)).read()
            for n in bench.KERNEL_SOURCES}
    h0 = bench.kernel_source_hash(lambda n: base[n])
    assert h0 == bench.kernel_source_hash()
    commented = dict(base)
    commented["gemm_tc.cu"] = "// a new comment\n" + base["gemm_tc.cu"].replace("\n", "\n\n", 3) + "/* tail */\n"
    assert bench.kernel_source_hash(lambda n: commented[n]) == h0
    edited = dict(base)
    edited["ptx.cuh"] = base["ptx.cuh"] + "\nstatic int unused_symbol;\n"
    assert bench.kernel_source_hash(lambda n: edited[n]) != h0
