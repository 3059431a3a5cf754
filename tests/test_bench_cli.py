"""bench.py's reference arm (the float64 oracle on the host cores) prints
the contract's JSON line; runs on the CPU with the tiny workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         "tiny_mha_fp32", "--steps", "3", "--warmup", "1", "--reference-budget", "1"],
        capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 3 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["unit"] == line["unit"]
    assert line["config"]["workload"] == "tiny_mha_fp32"
    # the same configuration dict the library arm emits for this workload
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    assert line["config"] == bench.workload_config(workloads.make_workload("tiny_mha_fp32", seed=0))
    # ms_per_step is one whole step at the sampled rate
    kvb = line["config"]["kv_bytes_per_step"]
    assert abs(line["ms_per_step"] - kvb / (line["value"] * 1e9) * 1e3) <= 1e-3 * line["ms_per_step"] + 2e-3
    assert line["cpu_baseline"]["cpu_time_s"] >= 0 and "cpu_time_over_wall" in line["cpu_baseline"]


def test_reference_arm_declines_library_only_workloads():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         "swa_spec_page_table"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "unavailable" in line


def test_oracle_step_covers_fp8_and_alibi_workloads():
    """The CPU leg runs the oracle with the workload's cache format and
    slopes, and counts one byte per fp8 cache element."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    for name in ("ragged_v2_fp8", "mha_v1_alibi_fp16"):
        inp = workloads.make_workload(name, seed=0, num_seqs=3)
        spec = inp["spec"]
        kw = bench.oracle_variant_kwargs(inp)
        assert kw["kv_cache_dtype"] == spec.kv_cache_dtype
        assert (kw["alibi_slopes"] is not None) == spec.alibi
        splits = bench.oracle_metadata(inp, spec)
        nbytes, seconds, cpu_seconds = bench.oracle_step(inp, spec, [0, 2], splits)
        e = 1 if spec.kv_cache_dtype != "auto" else 2
        lens = inp["seq_lens_list"]
        assert nbytes == (lens[0] + lens[2]) * spec.num_kv_heads * 2 * spec.head_size * e
        assert seconds > 0 and cpu_seconds >= 0


def test_cpu_baseline_reports_threads_and_cpu_time():
    """The CPU leg states the threads it gave the oracle and measures how busy
    it kept them (process CPU time over wall time)."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    inp = workloads.make_workload("tiny_mha_fp32", seed=0)
    before = torch.get_num_threads()
    rec = bench.cpu_baseline(inp, inp["spec"], budget_s=0.2, threads=1)
    assert rec["cores"] == 1 and rec["kind"] == "oracle" and rec["value"] > 0
    assert rec["wall_s"] > 0 and rec["cpu_time_s"] >= 0
    assert abs(rec["cpu_time_over_wall"] - rec["cpu_time_s"] / rec["wall_s"]) <= 0.02 + 0.01 * rec["cpu_time_over_wall"]
    assert torch.get_num_threads() == before  # the thread count is restored


def test_step_statistics():
    sys.path.insert(0, ROOT)
    import bench
    ms = [0.5 + 0.01 * i for i in range(20)]
    st = bench.step_stats(list(reversed(ms)))
    assert st["p10"] <= st["median"] <= st["p90"]
    assert st["median"] == round(bench.percentile(sorted(ms), 0.5) * 1e3, 2)
    assert bench.percentile([1.0], 0.9) == 1.0


def test_reference_arm_applies_the_batch_overrides():
    """A cut or resized batch (--num-seqs, --seq-len, --partition-size) reaches
    the reference arm as it reaches the library arm: the same configuration
    dict, built from the same overrides."""
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         "long_v2_bf16", "--num-seqs", "2", "--seq-len", "700", "--partition-size", "256",
         "--steps", "2", "--warmup", "1", "--reference-budget", "1"],
        capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    over = bench.workload_overrides("long_v2_bf16", 2, 700, 256)
    assert over["seq_lens"] == [700, 700] and over["partition_size"] == 256
    inp = workloads.make_workload("long_v2_bf16", seed=0, **over)
    assert inp["spec"].partition_size == 256 and inp["seq_lens_list"] == [700, 700]
    assert line["config"] == bench.workload_config(inp)
    assert line["config"]["num_seqs"] == 2 and line["config"]["total_tokens"] == 1400
