"""bench.py's host-side bookkeeping (no GPU): the roofline's traffic figure is
used only while the kernel sources match the capture it came from, the clock
record flags throttling, and the metric arithmetic is what the line claims."""
import bench


def test_traffic_only_for_the_captured_source(monkeypatch):
    text = open(bench.os.path.join(bench.ROOT, "profiles",
                                   "attn_fwd_causal_b2h16n8192d128_traffic.txt")).read()
    fields = dict(line.split(":", 1) for line in text.splitlines() if ":" in line)
    sha = fields["kernel_source_sha"].strip()
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: sha)
    assert bench.recorded_traffic("causal_b2h16n8192d128") == float(fields["dram_bytes_per_launch"])
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic("causal_b2h16n8192d128") is None
    assert bench.recorded_traffic("no_such_workload") is None


def test_kernel_source_hash_is_stable():
    assert bench.kernel_source_hash() == bench.kernel_source_hash()
    assert len(bench.kernel_source_hash()) == 16


def test_source_hash_ignores_comments_only():
    code = "int f(int x) {\n    return x + 1;   // one more\n}\n"
    commented = "/* header\n   text */\nint f(int x) {\n\n    // a note\n    return x + 1;\n}\n"
    changed = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench.code_without_comments(code) == bench.code_without_comments(commented)
    assert bench.code_without_comments(code) != bench.code_without_comments(changed)
    assert bench.code_without_comments('asm("max.f32 %0, %1;");  // 2-input') == 'asm("max.f32 %0, %1;");'


def test_clock_summary_flags_throttling():
    # index, sm MHz, max MHz, power, active reasons, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    idle = ["0", "345", "2070", "100.0", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    busy = ["0", "2070", "2070", "450.5", "0x4", "Not Active", "Not Active", "Not Active", "Active"]
    slow = ["0", "1500", "2070", "300.0", "0x8", "Active", "Not Active", "Not Active", "Not Active"]
    s = bench.ClockSampler.summarise([idle, busy, busy, busy])
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 4 and s["power_w_max"] == 450.5
    s = bench.ClockSampler.summarise([busy, slow, slow])
    assert "hw_slowdown" in s["reasons"] and s["sm_mhz"] == 1500.0
    assert bench.ClockSampler.summarise([])["reasons"] == ["unsampled"]


def test_job_throughput_is_whole_job_flops_per_second():
    # 2 ranks x 10 steps x 1e12 FLOP in 4 s: 5 TFLOP/s for the job
    assert abs(bench.job_throughput(1e12, steps=10, world=2, seconds=4.0) - 5.0) < 1e-12


def test_reference_arm_prints_the_contract_line(capsys, monkeypatch):
    """bench.py --impl reference (the fp64 oracle on the host cores) prints one
    JSON line with the contract's keys, its own value repeated as the CPU
    baseline and as an e2e figure with no host-device copies."""
    import json

    from blocked_online_softmax_gb300.workloads import BY_NAME
    for var in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)

    class Args:
        steps, warmup = 1, 1

    w = BY_NAME["small_b1h2n256d64"]
    assert bench.run_reference(Args(), w) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"] == bench.workload_config(w)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
