"""Host-side pieces of bench.py that need no GPU: the clock sampler that runs during the
timed region, driven here by a stand-in ``nvidia-smi`` on PATH that prints the same CSV
columns, and the rule that only samples taken after the timed region starts count."""
import os
import stat
import time

import bench

_FAKE_SMI = r"""#!/usr/bin/env python3
# Stand-in for nvidia-smi --query-gpu=... --format=csv,noheader,nounits -lms 200:
# one warm-up sample with a hardware slowdown, then, once the go-file exists, timed
# samples at 1965/2070 MHz with the power cap active.
import os, sys, time
go = os.environ["FAKE_SMI_GO"]
print("0, 1200, 2070, 900.0, 0x8, Active, Not Active, Not Active, Not Active", flush=True)
while not os.path.exists(go):
    time.sleep(0.02)
for mhz in (1965, 1950, 1980, 1965, 1965):
    print(f"0, {mhz}, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
          flush=True)
    time.sleep(0.02)
time.sleep(60)
"""


def _install_fake(tmp_path, monkeypatch):
    smi = tmp_path / "bin" / "nvidia-smi"
    smi.parent.mkdir()
    smi.write_text(_FAKE_SMI)
    smi.chmod(smi.stat().st_mode | stat.S_IXUSR)
    monkeypatch.setenv("PATH", str(smi.parent) + os.pathsep + os.environ["PATH"])
    go = tmp_path / "go"
    monkeypatch.setenv("FAKE_SMI_GO", str(go))
    return go


def test_clock_sampler_counts_only_the_timed_region(tmp_path, monkeypatch):
    go = _install_fake(tmp_path, monkeypatch)
    clk = bench.ClockSampler(0, str(tmp_path / "out" / "clocks_gpu{gpu}.csv"))
    clk.start()
    clk.mark()                       # the warm-up sample is before this point
    go.touch()
    deadline = time.time() + 20
    while time.time() < deadline:
        if sum(1 for _ in open(clk.path)) >= 6:
            break
        time.sleep(0.05)
    rec = clk.stop()
    assert clk.path.endswith(os.path.join("out", "clocks_gpu0.csv"))
    assert rec["samples"] == 5
    assert rec["sm_mhz"] == 1965.0
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"]      # the warm-up hw_slowdown is not counted


def test_clock_sampler_without_nvidia_smi_reports_unsampled(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))      # no nvidia-smi anywhere
    clk = bench.ClockSampler(3)
    assert os.path.basename(clk.path) == "mok_bench_clocks_gpu3.csv"
    clk.start()
    clk.mark()
    assert clk.stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}


def test_oracle_step_takes_experts_in_turn_up_to_the_row_bound():
    import moe_inputs as mi
    cfg = mi.CONFIGS["tiny"]                       # 8 experts, 512 routed rows
    step = bench.OracleStep(cfg)
    r = step.run(6, max_rows=100)
    assert r["rows"] >= 100 and r["experts"] >= 1
    assert r["experts"] < cfg.E
    assert r["next"] == (6 + r["experts"]) % cfg.E   # every tiny expert has rows; wraps at E
    whole = step.run(0)                            # no bound: every expert once
    assert whole["rows"] == cfg.T * cfg.k
    assert whole["experts"] == cfg.E and whole["next"] == 0
    assert whole["extrapolated"] >= whole["measured"] * 0.999


def test_reference_arm_line():
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "4", "--warmup", "3"], cwd=root, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 4 and d["warmup"] == 3
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    import moe_inputs as mi
    want = bench.workload_json(mi.CONFIGS["tiny"])
    assert {k: d["config"][k] for k in want} == want     # the GPU arm's workload keys


def test_method_roofline_bounds_the_layer_roofline():
    """The per-step path's own bound (every launch at its own roofline, one after another)
    is at least the layer's compulsory bound, and its grouped-GEMM part is the per-kernel
    algorithmic bytes (at the Kimi shape with fp32 results 146.57 GB: the weights four
    times, 22.5 + 11.3 + 11.3 + 22.5 GB, the fp32 weight gradients 67.6 GB, and the rows
    the GEMMs pass each other, U and V as bf16)."""
    import moe_inputs as mi
    pk = {"hbm_gbs": 6789.6, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1720.0}
    for name in ("kimi_8192", "kimi_2368", "dsv3_imbalanced", "ep64_slice", "mid", "tiny"):
        cfg = mi.CONFIGS[name]
        work = bench.method_work(cfg)
        f_fwd, f_bwd, b_fwd, b_bwd = bench.algorithmic(cfg)
        if not cfg.backward:
            f_bwd = b_bwd = 0.0
        m = bench.method_roofline(cfg, pk, 1.0)
        tc = pk["bf16_tflops"] * (2.0 if cfg.precision == "mxfp8" else 1.0)
        layer = max((f_fwd + f_bwd) / (tc * 1e12), (b_fwd + b_bwd) / (pk["hbm_gbs"] * 1e9))
        assert m["ms_per_step_bound"] >= layer * 1e3 * 0.999, name
        assert m["bytes_gb"] * 1e9 >= (b_fwd + b_bwd) * 0.999, name
        n_gemm = 6 if cfg.backward else 2
        assert sum(1 for n in work if n.startswith("gemm_")) == n_gemm, name
    kimi32 = mi.scaled(mi.CONFIGS["kimi_8192"], out="fp32")
    gemm_gb = sum(b for n, (f, b) in bench.method_work(kimi32).items()
                  if n.startswith("gemm_")) / 1e9
    assert abs(gemm_gb - 146.57) < 0.01
    # bf16 results: the weight gradients and O, dXg rows take half the bytes
    kimi = bench.method_work(mi.CONFIGS["kimi_8192"])
    gemm16 = sum(b for n, (f, b) in kimi.items() if n.startswith("gemm_")) / 1e9
    cfg = mi.CONFIGS["kimi_8192"]
    R, H, I, E = cfg.T * cfg.k, cfg.H, cfg.I, cfg.E
    assert abs((gemm_gb - gemm16) * 1e9 - 2.0 * (3 * H * I * E + 2 * R * H)) < 1e6


def test_compulsory_bytes_of_the_workloads():
    """The layer's compulsory bytes per step with bf16 results: the weights read in each
    pass, x, y, dY, dX, the bf16 weight gradients and the saved U, V read once as bf16:
    34.15 + 68.7 GB for the Kimi shape at T=8192 and 12.1 + 36.0 GB for the DeepSeek-V3
    shape in MXFP8 (weights 1 + 1/32 bytes, gradients bf16)."""
    import moe_inputs as mi
    f, b, bf, bb = bench.algorithmic(mi.CONFIGS["kimi_8192"])
    assert abs(bf / 1e9 - 34.15) < 0.05 and abs(bb / 1e9 - 68.7) < 0.1
    f, b, bf, bb = bench.algorithmic(mi.CONFIGS["dsv3_imbalanced"])
    assert abs(bf / 1e9 - 12.1) < 0.1 and abs(bb / 1e9 - 36.0) < 0.15
    f, b, bf32, bb32 = bench.algorithmic(mi.scaled(mi.CONFIGS["kimi_8192"], out="fp32"))
    assert bb32 - bb > 30e9            # fp32 weight gradients double their bytes


def test_data_movement_reads_the_profile_names():
    """The row-moving launches are found under the names the library's profile records
    use (BF16 and MXFP8), and their bandwidth is bytes over time per launch."""
    import moe_inputs as mi
    pk = {"hbm_gbs": 6789.6}
    cfg = mi.CONFIGS["kimi_8192"]
    prof = {"dispatch_gather": (10, 3.4), "combine": (10, 4.84), "gemm_fwd_down": (10, 24.3),
            "topk_rank": (10, 0.4)}
    got = bench.data_movement(cfg, prof, pk)
    assert set(got) == {"dispatch_gather", "combine"}
    R, H = cfg.T * cfg.k, cfg.H
    assert got["dispatch_gather"]["gb"] == round(4.0 * R * H / 1e9, 3)
    assert abs(got["dispatch_gather"]["gb_per_s"] - 4.0 * R * H / 0.34e-3 / 1e9) < 0.1
    mx = bench.data_movement(mi.CONFIGS["dsv3_imbalanced"],
                             {"dispatch_gather_mxfp8": (1, 0.45),
                              "replay_gather_rows_mxfp8": (1, 0.6),
                              "reverse_dispatch_gather_rows_mxfp8": (1, 0.6)}, pk)
    assert set(mx) == {"dispatch_gather_mxfp8", "replay_gather_rows_mxfp8",
                       "reverse_dispatch_gather_rows_mxfp8"}
