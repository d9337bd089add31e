"""Host logic of bench.py that decides what the JSON line reports, on CPU.

The roofline's `traffic` comes from a committed ncu record only while the
record was taken on the current kernel sources and on the bench's workload;
otherwise it is null."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def _record(path, sha, workload, nbytes):
    with open(path, "w") as f:
        f.write(f"kernel: test\nworkload: {workload}\nsource_sha256: {sha}\n"
                f"dram_bytes_per_launch: {nbytes}\nderivation: test\n")


def test_traffic_reported_only_for_current_sources_and_workload(tmp_path):
    b = _bench()
    path = str(tmp_path / "traffic.txt")
    b.TRAFFIC_FILE = path
    assert b.recorded_traffic("dsv3_bf16_fwd") is None  # no record
    sha = b.source_hash()
    _record(path, sha, "dsv3_bf16_fwd", 16209799168)
    assert b.recorded_traffic("dsv3_bf16_fwd") == 16209799168.0
    assert b.recorded_traffic("dsv3_mxfp8_fwd") is None  # another workload
    _record(path, "0" * 16, "dsv3_bf16_fwd", 16209799168)
    assert b.recorded_traffic("dsv3_bf16_fwd") is None  # taken on other sources


def test_source_hash_covers_the_up_gate_kernel_sources():
    b = _bench()
    assert "gemm_pair.cu" in b.KERNEL_SOURCES and "pair.cuh" in b.KERNEL_SOURCES
    h = b.source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    assert b.source_hash() == h  # deterministic


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampled(b, tmp_path, lines):
    cs = b.ClockSampler(0)
    cs.proc = _DoneProc()
    cs.path = str(tmp_path / "clocks.csv")
    with open(cs.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return cs.stop()


def test_clock_samples_median_and_throttle_reasons(tmp_path):
    """The clocks key: median SM clock under load, the maximum, and every
    throttle reason seen active in any sample (nvidia-smi csv, no units)."""
    b = _bench()
    na = "Not Active"
    got = _sampled(b, tmp_path, [
        f"0, 2070, 2070, 900.5, 0x0000000000000000, {na}, {na}, {na}, {na}",
        f"0, 1500, 2070, 1400.2, 0x0000000000000004, {na}, {na}, {na}, Active",
        f"0, 1400, 2070, 1398.0, 0x0000000000000004, {na}, {na}, {na}, Active",
        f"0, [N/A], [N/A], [N/A], [N/A], {na}, {na}, {na}, {na}",
    ])
    assert got == {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0, "samples": 4, "reasons": ["sw_power_cap"]}
    got = _sampled(b, tmp_path, [f"0, 1200, 2070, 700.0, 0x0000000000000048, {na}, Active, {na}, {na}"])
    assert got["reasons"] == ["hw_thermal_slowdown"]  # a run the timing rules reject
    assert _sampled(b, tmp_path, ["garbage"]) is None


def _run_reference(env_extra):
    import json
    import subprocess
    import sys
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_line_on_host_cores():
    """bench.py --impl reference times the oracle on the host: one JSON line
    with the contract's keys, its own e2e (no copies) and cpu_baseline."""
    (line,) = _run_reference({"WORLD_SIZE": "1", "RANK": "0"})
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["steps"] == 3 and line["warmup"] == 3 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny"
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]


def test_reference_arm_other_ranks_exit_without_work():
    assert _run_reference({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"}) == []


PEAKS = dict(hbm_gbs=6781.1, bf16=1887.9, bf16_sustained=1649.2, source="measured")


def test_roofline_bound_per_workload():
    """The bench line's roofline compares the kernel with its own bound:
    the skewed layer's up/gate (about 1100 FLOP per algorithmic byte) against
    the tensor peak, the DSV3 up/gate (BF16 and MXFP8) and the backward call
    against HBM; every line names both figures."""
    from routing_grouped_expert_device_gb300 import workloads as W
    b = _bench()
    cases = {"skewed_bf16_fwd": (57, 1.9, "tensor"), "dsv3_bf16_fwd": (256, 2.5, "hbm"),
             "dsv3_mxfp8_fwd": (256, 1.5, "hbm"), "dsv3_bf16_fwdbwd": (256, 11.4, "hbm"),
             "dsv3_mxfp8_fwdbwd": (256, 9.4, "hbm")}
    for name, (nonempty, ms, bound) in cases.items():
        cfg = W.CONFIGS[name]
        r, tensor_peak, burst, bf16 = b.roofline_of(cfg, nonempty, ms, PEAKS, capped=False)
        assert r["bound"] == bound, name
        if bound == "tensor":
            assert r["unit"] == "TFLOP/s" and r["peak"] == tensor_peak and "gbs" in r
            assert r["intensity_flop_per_byte"] > r["ridge_flop_per_byte"]
        else:
            assert r["unit"] == "GB/s" and r["peak"] == PEAKS["hbm_gbs"] and "tflops" in r
            assert r["intensity_flop_per_byte"] <= r["ridge_flop_per_byte"]
        assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
        assert tensor_peak == PEAKS["bf16"] * (2.0 if cfg.dtype == "mxfp8" else 1.0)
    # under the power cap the sustained figure is the denominator
    _, tp, burst, bf16 = b.roofline_of(W.CONFIGS["skewed_bf16_fwd"], 57, 1.9, PEAKS, capped=True)
    assert tp == PEAKS["bf16_sustained"] and burst == PEAKS["bf16"]
    # the DSV3 up/gate's algorithmic bytes: weights of non-empty experts + xg + a
    r, *_ = b.roofline_of(W.CONFIGS["dsv3_bf16_fwd"], 256, 2.5, PEAKS, capped=False)
    assert r["algorithmic_bytes"] == 16089350144


def test_oracle_slice_every_kind_of_workload():
    """The cpu_baseline / reference-arm slice runs the oracle for BF16 and
    MXFP8, forward and forward+backward, and scales its work by FLOPs."""
    from routing_grouped_expert_device_gb300 import workloads as W
    b = _bench()
    base = W.MoEConfig("t", T=128, D=128, I=64, E=8, K=2, I_shared=64)
    for cfg in (base, base.replace(backward=True), base.replace(dtype="mxfp8"),
                base.replace(dtype="mxfp8", backward=True)):
        d = W.make_inputs(cfg, "cpu", with_dy=cfg.backward)
        sl = b.OracleSlice(cfg, d)
        ex = b.slice_experts(sl, 2)
        toks, dt = sl.run(ex)
        rows = sum(int(sl.counts[e]) for e in ex)
        n_sh = round(cfg.T * 2 / len(sl.nonempty))
        per = 3.0 if cfg.backward else 1.0
        want = cfg.T * per * (6.0 * rows * cfg.D * cfg.I + 6.0 * n_sh * cfg.D * cfg.I_shared) / (
            cfg.fwd_flops() + (cfg.bwd_flops() if cfg.backward else 0.0))
        assert abs(toks - want) < 1e-9 * want and dt > 0
        assert "scaled to layer tokens by FLOPs" in sl.describe(ex, dt)
