"""Benchmark: MoE SwiGLU layer forward + backward tokens/s on GB300 (one step = plan,
forward and backward of one batch), as one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Default workload: the Kimi-2.5-shaped layer (T=8192, H=7168, I=2048, E=384, top-8, one
BF16 shared expert with I=2048), BF16: bf16 operands in every GEMM (the weight gradients'
too), fp32 accumulation, bf16 results. Inputs are seeded synthetic tensors resident in HBM;
the expert weights alone are 34 GB, far larger than the 129 MB L2, so no flush is needed
between steps. Under torchrun each rank runs an independent replica on its own batch
(weak scaling, no collective on the data path).

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload on
the host cores (router for every token, a few experts and a slice of the shared expert,
extrapolated to the whole layer).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/sec fwd & bwd (BF16, MXFP8) on 1 GB300; grouped-GEMM % of TC peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="kimi_8192_plain")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--fwd-path", default="auto", choices=["auto", "megakernel", "launches"])
    ap.add_argument("--comm-sms", type=int, default=0,
                    help="gather/combine SMs of the forward megakernel (0: automatic)")
    ap.add_argument("--sm-limit", type=int, default=0,
                    help="most SMs any kernel uses (0: all)")
    ap.add_argument("--out", default="", choices=["", "bf16", "fp32"],
                    help="result type of y, dX and the weight gradients (default: the "
                         "workload's, bf16)")
    ap.add_argument("--row-pairs", default="auto", choices=["auto", "on", "off"],
                    help="row-tile pairs in the BF16 routed GEMMs")
    ap.add_argument("--sm-pairs", default="auto", choices=["auto", "on", "off"],
                    help="SM pairs (2-CTA clusters) in the BF16 weight-gradient GEMMs")
    ap.add_argument("--tile-order", default="static", choices=["static", "dynamic", "clc"],
                    help="tile order of the persistent grouped GEMMs")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the sub-records (fp32 results, forward megakernel, MXFP8)")
    ap.add_argument("--sub-steps", type=int, default=10,
                    help="timed steps of each sub-record")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="routed-expert time of the CPU oracle's one timed sample")
    ap.add_argument("--ref-rows-per-step", type=int, default=1024,
                    help="routed rows in each step of the reference arm (the oracle)")
    ap.add_argument("--clocks-csv", default="",
                    help="keep nvidia-smi's clock samples in this file (default: a temporary "
                         "file); {gpu} is replaced by the GPU index")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a kernel, from
# one ncu capture, scaled to the workload's launch as the profile summary of that kernel
# and workload states. A figure is valid only for the GEMM source revision it was taken on
# (gemm_source_rev) and the result type it was taken with.
NCU_TRAFFIC = {
    # the 24-expert profiling case (E=24, T=512) scaled by 16: 16 x (0.106 + 1.347) GB
    ("kimi_8192_plain", "gemm_bwd_dw_upgate", "bf16"): {"bytes": 23.25e9,
                                                       "rev": "3a358dec299f5f3f"},
}
GEMM_SOURCES = ("grouped_gemm_built_gb300/csrc/mok_gemm.cu",
                "grouped_gemm_built_gb300/csrc/mok_ptx.cuh",
                "grouped_gemm_built_gb300/csrc/mok_internal.h")


def gemm_source_rev():
    """First 16 hex digits of sha256 over the lines '<sha256>  <path>' of the GEMM sources
    (what `sha256sum <files> | sha256sum` prints)."""
    import hashlib
    text = ""
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            text += f"{hashlib.sha256(f.read()).hexdigest()}  {rel}\n"
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def ncu_traffic(workload, kernel, out="bf16"):
    rec = NCU_TRAFFIC.get((workload, kernel, out))
    if rec is None or rec["rev"] != gemm_source_rev():
        return None
    return rec["bytes"]


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, path=""):
        self.gpu = gpu_index
        self.proc = None
        self.path = (path.replace("{gpu}", str(gpu_index)) if path else
                     os.path.join(tempfile.gettempdir(), f"mok_bench_clocks_gpu{gpu_index}.csv"))

    def start(self):
        """Start sampling and wait for the first sample: nvidia-smi's start-up (NVML
        initialisation) can stall CUDA calls of this process for seconds, so it must be
        over before anything is timed."""
        try:
            os.makedirs(os.path.dirname(self.path) or ".", exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            if getattr(self, "f", None) is not None:
                self.f.close()
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 20:
            try:
                if os.path.getsize(self.path) > 0:
                    break
            except OSError:
                pass
            time.sleep(0.1)
        time.sleep(0.5)

    def mark(self):
        """Only samples taken after this point count (the timed region)."""
        if self.proc is None:
            return
        self.f.flush()
        try:
            self.skip = sum(1 for _ in open(self.path))
        except OSError:
            self.skip = 0

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for n_line, line in enumerate(open(self.path)):
            if n_line < getattr(self, "skip", 0):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w": round(statistics.median(power), 1) if power else None}


# ----------------------------------------------------------------------------- workload
def workload_config(name):
    import moe_inputs as mi
    return mi.CONFIGS[name]


def workload_json(cfg):
    """The workload keys of the JSON line, the same for both arms."""
    wb = 1.0 if cfg.precision == "mxfp8" else 2.0
    weights_gb = 3.0 * cfg.H * cfg.I * cfg.E * wb / 1e9
    return {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} k={cfg.k} "
                        f"shared_I={cfg.shared_I} {cfg.precision} "
                        + ("fwd+bwd" if cfg.backward else "fwd"),
            "step": "plan + forward" + (" + backward" if cfg.backward else ""),
            "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "k": cfg.k,
            "shared_I": cfg.shared_I, "precision": cfg.precision,
            "operands": {"bf16_plain": "bf16 in every GEMM, fp32 accumulation",
                         "bf16": "bf16, the weight-gradient GEMMs on bf16 hi + lo pairs",
                         "mxfp8": "E4M3 + UE8M0 per 32 (routed experts), bf16 shared expert",
                         }.get(cfg.precision, cfg.precision),
            "results": f"{cfg.out} (y, dX, weight gradients); dgates, dWr fp32",
            "l2": (f"inputs larger than L2 (expert weights {weights_gb:.3g} GB), no flush"
                   if weights_gb * 1e9 > 129e6 else "inputs smaller than L2, no flush")}


def result_bytes(cfg):
    """Bytes of one result element: y, dX, the weight gradients, and the expert output rows
    and routed dX rows the combines read (bf16 or fp32, as the layer was asked)."""
    return 2.0 if cfg.out == "bf16" else 4.0


def algorithmic(cfg):
    """Algorithmic FLOPs and compulsory HBM bytes of one step (plan + forward + backward).

    FLOPs: per routed row 6*H*I forward (up, gate, down), 12*H*I backward (dX, dW);
    shared expert the same per token; router 2*H*E per token forward, backward dWr and
    dX router path 4*H*k per token. Bytes, forward: the weights once (MXFP8: 1 + 1/32
    bytes per routed weight; the shared expert stays bf16), x in, y out, the router
    weights; backward: the weights once more, the weight gradients written once, x and dY
    in, dX out, the saved U, V read once as bf16 values, Wr in and dWr out. y, dX and the
    weight gradients count at the result type's size (bf16 by default)."""
    T, H, I, E, k, Is = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.shared_I
    R = T * k
    f_fwd = 6.0 * H * I * R + 6.0 * H * Is * T + 2.0 * H * E * T
    f_bwd = 12.0 * H * I * R + 12.0 * H * Is * T + 4.0 * H * k * T
    wb = 1.0 + 1.0 / 32 if cfg.precision == "mxfp8" else 2.0   # routed weight bytes read
    ob = result_bytes(cfg)
    w_read = wb * 3.0 * H * I * E + 2.0 * 3.0 * H * Is
    n_w = 3.0 * H * I * E + 3.0 * H * Is
    b_fwd = w_read + 2.0 * T * H + ob * T * H + 4.0 * H * E
    b_bwd = w_read + ob * n_w + 2.0 * 2 * T * H + ob * T * H + 2.0 * 2 * R * I \
        + 4.0 * H * E * 2
    return f_fwd, f_bwd, b_fwd, b_bwd


# per-kernel algorithmic work, for the roofline of the dominant kernel
def kernel_work(cfg, name, counts=None):
    T, H, I, E, k, Is = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.shared_I
    R = T * k
    rows = R
    mx = name.endswith("_mxfp8")
    name = name[:-len("_mxfp8")] if mx else name
    b = 1.0 + 1.0 / 32 if mx else 2.0     # bytes per operand element (MXFP8: + scales)
    uv = 2.0                              # bytes per saved U, V element (kept as bf16)
    ob = result_bytes(cfg)                # O / dXg rows and weight gradients written
    # (FLOPs, bytes): operands b bytes, U and V uv bytes, O / dXg rows and gradients ob
    tbl = {
        "gemm_fwd_upgate_swiglu": (4.0 * H * I * rows,
                                   b * (2 * H * I * E + rows * H + rows * I)
                                   + 2 * uv * rows * I),
        "gemm_fwd_down": (2.0 * H * I * rows, b * (H * I * E + rows * I) + ob * rows * H),
        "gemm_bwd_dh_swiglu": (2.0 * H * I * rows,
                               b * (H * I * E + rows * H + 3 * rows * I)
                               + 2 * uv * rows * I + 4.0 * rows),
        "gemm_bwd_dx": (4.0 * H * I * rows, b * (2 * H * I * E + 2 * rows * I) + ob * rows * H),
        "gemm_bwd_dw_down": (2.0 * H * I * rows, b * (rows * I + rows * H) + ob * H * I * E),
        "gemm_bwd_dw_upgate": (4.0 * H * I * rows,
                               b * (rows * H + 2 * rows * I) + ob * 2 * H * I * E),
        # the routed forward in one launch: weights once, x rows, U and V saved, y written
        "fwd_megakernel": (6.0 * H * I * rows,
                           b * 3 * H * I * E + 2.0 * rows * H + 2 * uv * rows * I + ob * T * H),
    }
    return tbl.get(name)


def method_work(cfg):
    """(FLOPs, bytes) of every launch of one step of the per-step path, keyed by the
    bench's kernel names: the grouped GEMMs as in ``kernel_work``; the shared expert's
    GEMMs with the same formulas (one expert, every token, BF16); the router's logits;
    dispatch and reverse dispatch (rows read as bf16, written in the GEMM operand format;
    MXFP8 gathers x and dY once more, quantised along the rows, for the dW GEMMs);
    combine and reverse combine (result-type rows read, result-type token rows written);
    the router's weight gradient. The launches with a few KB of traffic (top-k, scans,
    small transposes) are left out."""
    import dataclasses
    T, H, I, E, k, Is = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.shared_I
    R = T * k
    mx = cfg.precision == "mxfp8"
    sfx = "_mxfp8" if mx else ""
    b_op = 1.0 + 1.0 / 32 if mx else 2.0
    ob = result_bytes(cfg)
    fwd = ["gemm_fwd_upgate_swiglu", "gemm_fwd_down"]
    bwd = ["gemm_bwd_dh_swiglu", "gemm_bwd_dx", "gemm_bwd_dw_upgate", "gemm_bwd_dw_down"]
    names = fwd + (bwd if cfg.backward else [])
    out = {n + sfx: kernel_work(cfg, n + sfx) for n in names}
    if Is:
        sh = dataclasses.replace(cfg, k=1, E=1, I=Is, precision="bf16")
        for n in names:
            out["shared_" + n[len("gemm_"):]] = kernel_work(sh, n)
    if cfg.router:
        out["router_logits"] = (2.0 * T * H * E * 3, 2.0 * T * H + 3 * 2.0 * H * E + 4.0 * T * E)
    move = (0.0, 2.0 * R * H + b_op * R * H)          # bf16 rows in, operand rows out
    out["dispatch_gather" + sfx] = move
    comb = (0.0, ob * R * H + ob * T * H + (ob * T * H if Is else 0.0))
    out["combine"] = comb
    if cfg.backward:
        out["reverse_dispatch_gather" + sfx] = move
        if mx:   # the dW GEMMs' operands, quantised along the expert rows: x and dY again
            out["replay_gather_rows_mxfp8"] = move
            out["reverse_dispatch_gather_rows_mxfp8"] = move
        out["reverse_combine"] = comb
        if cfg.router:
            out["router_dwr"] = (2.0 * T * H * k, 2.0 * T * H + 4.0 * H * E + 4.0 * T * k)
    return out


def method_roofline(cfg, pk, ms_step):
    """The per-step path's own bound: every launch at its own roofline (its bytes at the
    measured copy bandwidth or its FLOPs at the measured tensor peak of its dtype,
    whichever is longer), launches one after another."""
    t = 0.0
    byts = flops = 0.0
    for name, (f, b) in method_work(cfg).items():
        tc = pk["bf16_tflops"] * (2.0 if name.endswith("_mxfp8") else 1.0)
        t += max(f / (tc * 1e12), b / (pk["hbm_gbs"] * 1e9))
        byts += b
        flops += f
    return {"ms_per_step_bound": round(t * 1e3, 3), "frac": round(t * 1e3 / ms_step, 4),
            "bytes_gb": round(byts / 1e9, 2), "tflop": round(flops / 1e12, 2)}


def data_movement(cfg, prof, pk):
    """Achieved bandwidth of the launches that move rows rather than multiply (router
    logits included): bytes from ``method_work`` over the launch's measured time, and its
    fraction of the measured copy bandwidth."""
    out = {}
    for name, (f, b) in method_work(cfg).items():
        if name.startswith(("gemm_", "shared_")) or name not in prof:
            continue
        c, t = prof[name]
        if c == 0 or t <= 0:
            continue
        gbs = b / (t / c / 1e3) / 1e9
        out[name] = {"gb": round(b / 1e9, 3), "ms": round(t / c, 4), "gb_per_s": round(gbs, 1),
                     "frac_of_copy": round(gbs / pk["hbm_gbs"], 4)}
    return out


# ----------------------------------------------------------------------------- replicas
def max_over_ranks(x, device):
    """x's maximum over the ranks of the default process group (x itself on one rank):
    the slowest replica's time is the job's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, tokens_per_rank, steps, ms):
    """Tokens per second of the whole job: each of ``world`` replicas processes
    ``tokens_per_rank`` tokens per step (weak scaling); ``ms`` is the slowest replica's
    time for ``steps`` steps."""
    return world * tokens_per_rank * steps / (ms / 1e3)


# ----------------------------------------------------------------------------- GPU arm
def make_layer_for(cfg, args, device="cuda", fwd_path=None):
    """The layer of one workload with its device inputs, weights, gradients and y."""
    import torch

    import moe_inputs as mi
    from grouped_gemm_built_gb300 import mok
    from grouped_gemm_built_gb300.layer import MoELayer
    rank = int(os.environ.get("RANK", "0"))
    inp = mi.make_inputs(cfg, seed=1000 + rank, device=device, with_dy=True)
    L = MoELayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, shared_I=cfg.shared_I, router=cfg.router,
                 macrobatches=cfg.macrobatches, ring_bytes=cfg.ring_bytes,
                 precision=cfg.precision, out=cfg.out)
    L.set_fwd_path(fwd_path or args.fwd_path)
    mok.mok_set_comm_sms(L.ctx, args.comm_sms)
    mok.mok_set_sm_limit(L.ctx, args.sm_limit)
    mok.mok_set_tile_order(L.ctx, {"static": mok.MOK_TILES_STATIC,
                                   "dynamic": mok.MOK_TILES_DYNAMIC,
                                   "clc": mok.MOK_TILES_CLC}[args.tile_order])
    mok.mok_set_row_pairs(L.ctx, {"auto": mok.MOK_PAIRS_AUTO, "on": mok.MOK_PAIRS_ON,
                                  "off": mok.MOK_PAIRS_OFF}[args.row_pairs])
    mok.mok_set_sm_pairs(L.ctx, {"auto": mok.MOK_SMPAIRS_AUTO, "on": mok.MOK_SMPAIRS_ON,
                                 "off": mok.MOK_SMPAIRS_OFF}[args.sm_pairs])
    mx = None
    if cfg.precision == "mxfp8":
        mx = L.quantize_weights(inp["W_up"], inp["W_gate"], inp["W_down"])
    w = L.weights(inp["W_up"], inp["W_gate"], inp["W_down"], inp["Ws_up"], inp["Ws_gate"],
                  inp["Ws_down"], mx=mx)
    grads = L.alloc_grads() if cfg.backward else None
    y = torch.empty((cfg.T, cfg.H), dtype=L.out_dtype, device=device)
    return L, inp, w, grads, y


def layer_step(cfg, L, inp, w, grads, y, x=None, dY=None, y_out=None, g_out=None):
    """One step: plan, forward and (where the workload has one) backward."""
    x = inp["x"] if x is None else x
    if cfg.router:
        L.plan(x=x, Wr=inp["Wr"], bias=inp["bias"])
    else:
        L.plan(topk_idx=inp["topk_idx"], gates=inp["gates"])
    L.forward(x, w, y if y_out is None else y_out)
    if cfg.backward:
        L.backward(x, inp["Wr"] if cfg.router else None, w, inp["dY"] if dY is None else dY,
                   grads if g_out is None else g_out)


def time_steps(cfg, L, step, steps, warmup, clk, world):
    """W untimed warm-up steps, then ``steps`` timed ones between barriers and device
    synchronisations, CUDA events on the launch stream, with the library's per-launch
    event records and the clock sampler's timed-region samples. Returns (ms of all timed
    steps, {kernel: (launches, ms)}, launches, megakernel phases, clocks)."""
    import torch
    import torch.distributed as dist

    from grouped_gemm_built_gb300 import mok

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(warmup, 0)):
        step()
    barrier()
    if L.status() != 0:
        raise RuntimeError(f"device status error during warm-up ({cfg.name})")
    stream = torch.cuda.current_stream()
    clk.mark()
    mok.mok_profile_enable(L.ctx, True)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    barrier()
    ms = e0.elapsed_time(e1)
    prof, launches = mok.mok_profile_report(L.ctx)
    # "fwd_megakernel:<phase>" lines are phases inside the megakernel, not launches
    phases = {n.split(":", 1)[1]: round(t / c, 4) for n, (c, t) in prof.items() if ":" in n and c}
    prof = {n: v for n, v in prof.items() if ":" not in n}
    mok.mok_profile_enable(L.ctx, False)
    clocks = clk.stop()
    if L.status() != 0:
        raise RuntimeError(f"device status error in the timed region ({cfg.name})")
    return ms, prof, launches, phases, clocks


def analyse(cfg, prof, ms_step, pk, workload):
    """Roofline of the dominant grouped GEMM, every GEMM's tensor throughput, the layer's
    compulsory bound, the per-step path's own bound and the row moves' bandwidth. Tensor
    fractions use the measured burst bf16 peak (x 2 for MXFP8, the nominal fp8/bf16 ratio):
    each GEMM launch runs for milliseconds inside a step, and the burst figure is the
    conservative denominator (the sustained one is lower)."""
    gemm = {n: v for n, v in prof.items() if kernel_work(cfg, n) is not None}
    top = max(gemm.items(), key=lambda kv: kv[1][1]) if gemm else None
    roofline = None
    per_kernel = {n: {"launches": c, "ms_per_launch": round(t / c, 5), "share": None}
                  for n, (c, t) in prof.items()}
    tot = sum(t for _, t in prof.values()) or 1.0
    for n, (c, t) in prof.items():
        per_kernel[n]["share"] = round(t / tot, 4)
    if top is not None:
        name, (cnt, tms) = top
        flops, byts = kernel_work(cfg, name)
        dur = tms / cnt / 1e3
        ai = flops / byts
        tpk = pk["bf16_tflops"] * (2.0 if name.endswith("_mxfp8") else 1.0)
        tsrc = pk["source"] + (" (burst bf16 x 2, MXFP8)" if name.endswith("_mxfp8")
                               else " (burst bf16)")
        ridge = tpk * 1e12 / (pk["hbm_gbs"] * 1e9)
        if ai < ridge:
            achieved = byts / dur / 1e9
            tr = ncu_traffic(workload, name, cfg.out)
            roofline = {"kernel": name, "bound": "hbm", "achieved": round(achieved, 1),
                        "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": round(achieved / pk["hbm_gbs"], 4),
                        "traffic": None if tr is None else round(tr / 1e9, 3),
                        "traffic_unit": "GB per launch",
                        "algorithmic": round(byts / 1e9, 3),
                        "peak_source": pk["source"] + " (copy bandwidth)"}
        else:
            achieved = flops / dur / 1e12
            roofline = {"kernel": name, "bound": "tensor", "achieved": round(achieved, 1),
                        "peak": round(tpk, 1), "unit": "TFLOP/s",
                        "frac": round(achieved / tpk, 4), "traffic": None,
                        "peak_source": tsrc}
    # every grouped GEMM's tensor throughput against its dtype's peak (the metric's
    # "grouped-GEMM % of TC peak"; meaningful where the GEMMs are compute-bound)
    gemm_tc = {}
    for n, (c, t) in prof.items():
        wk = kernel_work(cfg, n)
        if wk is None or c == 0 or t <= 0:
            continue
        tf = wk[0] / (t / c / 1e3) / 1e12
        peak_n = pk["bf16_tflops"] * (2.0 if n.endswith("_mxfp8") else 1.0)
        gemm_tc[n] = {"tflops": round(tf, 1), "frac_of_peak": round(tf / peak_n, 4),
                      "tb_per_s": round(wk[1] / (t / c / 1e3) / 1e12, 3)}
    f_fwd, f_bwd, b_fwd, b_bwd = algorithmic(cfg)
    if not cfg.backward:
        f_bwd = b_bwd = 0.0
    lpk = pk["bf16_tflops"] * (2.0 if cfg.precision == "mxfp8" else 1.0)
    t_roof = max((f_fwd + f_bwd) / (lpk * 1e12), (b_fwd + b_bwd) / (pk["hbm_gbs"] * 1e9))
    layer_roofline = {"ms_per_step_bound": round(t_roof * 1e3, 3),
                      "frac": round(t_roof * 1e3 / ms_step, 4),
                      "bytes_gb": round((b_fwd + b_bwd) / 1e9, 2),
                      "tflop": round((f_fwd + f_bwd) / 1e12, 2),
                      "bound": "hbm" if (b_fwd + b_bwd) / (pk["hbm_gbs"] * 1e9) >
                      (f_fwd + f_bwd) / (lpk * 1e12) else "tensor"}
    try:
        method = method_roofline(cfg, pk, ms_step)
        moves = data_movement(cfg, prof, pk)
    except Exception as exc:          # reporting only: never lose the line over it
        method = moves = {"error": repr(exc)}
    return {"roofline": roofline, "layer_roofline": layer_roofline, "method_roofline": method,
            "data_movement": moves, "kernels": per_kernel, "gemm_tc": gemm_tc}


def sub_record(name, cfg, args, pk, local, fwd_path=None, min_steps=3):
    """One more workload measured the same way in this process (one GPU): its own layer,
    warm-up, timed steps (at least ``min_steps``: short steps need more of them for the
    clock samples), clock samples and analysis; the buffers are freed afterwards."""
    import torch
    L, inp, w, grads, y = make_layer_for(cfg, args, fwd_path=fwd_path)
    clk = ClockSampler(local, args.clocks_csv.replace("{gpu}", f"{local}_{name}")
                       if args.clocks_csv else "")
    clk.start()
    steps = max(min_steps, args.sub_steps)
    ms, prof, launches, phases, clocks = time_steps(
        cfg, L, lambda: layer_step(cfg, L, inp, w, grads, y), steps, args.warmup, clk, 1)
    ms_step = ms / steps
    rec = {"workload": workload_json(cfg)["workload"], "out": cfg.out,
           "fwd_path": fwd_path or args.fwd_path,
           "value": round(cfg.T * steps / (ms / 1e3), 1), "unit": "tokens/s",
           "ms_per_step": round(ms_step, 4), "steps": steps, "warmup": args.warmup,
           "clocks": clocks, "gpu_launches": launches,
           "megakernel_phases_ms": phases or None}
    a = analyse(cfg, prof, ms_step, pk, cfg.name)
    a.pop("kernels")
    rec.update(a)
    del L, inp, w, grads, y
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_gpu(args):
    import dataclasses

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cfg = workload_config(args.workload)
    if args.out:
        cfg = dataclasses.replace(cfg, out=args.out)
    L, inp, w, grads, y = make_layer_for(cfg, args)
    stream = torch.cuda.current_stream()

    clk = ClockSampler(local, args.clocks_csv)
    clk.start()
    ms, prof, launches, phases, clocks = time_steps(
        cfg, L, lambda: layer_step(cfg, L, inp, w, grads, y), args.steps, args.warmup, clk,
        world)
    ms = max_over_ranks(ms, "cuda")
    ms_step = ms / args.steps
    value = whole_job_rate(world, cfg.T, args.steps, ms)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ------------------------------------------------------------ e2e (host buffers)
    e2e = None
    if not args.no_e2e:
        hx = torch.empty_like(inp["x"], device="cpu").pin_memory()
        hdy = torch.empty_like(inp["dY"], device="cpu").pin_memory()
        hx.copy_(inp["x"])
        hdy.copy_(inp["dY"])
        hy = torch.empty((cfg.T, cfg.H), dtype=L.out_dtype).pin_memory()
        hdx = torch.empty((cfg.T, cfg.H), dtype=L.out_dtype).pin_memory()
        # double-buffered device inputs and outputs: step i+1's host->device copies and
        # step i-1's device->host copies run on a copy stream while step i computes
        cs = torch.cuda.Stream()
        xin = [torch.empty_like(inp["x"]) for _ in range(2)]
        dyin = [torch.empty_like(inp["dY"]) for _ in range(2)]
        yb = [y, torch.empty_like(y)]
        gb = [grads, dict(grads, dX=torch.empty_like(grads["dX"]))] if cfg.backward else [None, None]
        ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer b on the device
        ev_done = [torch.cuda.Event() for _ in range(2)]  # step using buffer b computed
        ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of buffer b copied out
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)

        def h2d(j):
            b = j % 2
            with torch.cuda.stream(cs):
                if j >= 2:
                    cs.wait_event(ev_done[b])
                xin[b].copy_(hx, non_blocking=True)
                if cfg.backward:
                    dyin[b].copy_(hdy, non_blocking=True)
                ev_in[b].record(cs)

        def run_e2e(k, t0=None, t1=None):
            with torch.cuda.stream(cs):
                if t0 is not None:
                    t0.record(cs)
            h2d(0)
            for i in range(k):
                b = i % 2
                if i + 1 < k:
                    h2d(i + 1)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])
                layer_step(cfg, L, inp, w, grads, y, x=xin[b], dY=dyin[b], y_out=yb[b],
                           g_out=gb[b])
                ev_done[b].record(stream)
                with torch.cuda.stream(cs):
                    cs.wait_event(ev_done[b])
                    hy.copy_(yb[b], non_blocking=True)
                    if cfg.backward:
                        hdx.copy_(gb[b]["dX"], non_blocking=True)
                    ev_out[b].record(cs)
            with torch.cuda.stream(cs):
                if t1 is not None:
                    t1.record(cs)

        run_e2e(2)
        barrier()
        k_e2e = max(3, min(args.steps, 6))
        run_e2e(k_e2e, e0, e1)
        cs.synchronize()
        barrier()
        ms_e2e = max_over_ranks(e0.elapsed_time(e1), "cuda")
        e2e = {"value": whole_job_rate(world, cfg.T, k_e2e, ms_e2e), "unit": "tokens/s",
               "h2d_bytes_per_step": hx.numel() * 2 + (hdy.numel() * 2 if cfg.backward else 0),
               "d2h_bytes_per_step": hy.numel() * hy.element_size()
               + (hdx.numel() * hdx.element_size() if cfg.backward else 0),
               "steps": k_e2e,
               "pipeline": "inputs and results double-buffered; copies on a second stream "
                           "overlap the neighbouring steps' compute"}

    pk = peaks()
    a = analyse(cfg, prof, ms_step, pk, args.workload)
    mb = {"macrobatches": L.sizes.macrobatches, "ring_slots": L.sizes.ring_slots}
    del L, inp, w, grads, y
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # ------------------------------------------------------------ sub-records (one GPU)
    subs = None
    if world == 1 and not args.no_sub:
        subs = {}
        plans = []
        if cfg.out == "bf16":
            plans.append(("fp32_results", dataclasses.replace(cfg, out="fp32"), None))
        if args.workload.startswith("kimi_8192"):
            if cfg.precision == "bf16_plain":
                # the weight-gradient GEMMs on bf16 hi + lo operand pairs (MOK_BF16)
                plans.append(("bf16_hilo_wgrad", workload_config("kimi_8192"), None))
            plans.append(("megakernel_fwd", cfg, "megakernel"))
            plans.append(("mxfp8_dsv3_imbalanced", workload_config("dsv3_imbalanced"), None))
            # the pages' own megakernel setting: one EP=64 slice (6 experts, 2048 tokens of
            # 8 slots, MXFP8 forward), one launch per step and the megakernel
            ep = workload_config("ep64_slice")
            plans.append(("ep64_slice_launches", ep, "launches"))
            plans.append(("ep64_slice_megakernel", ep, "megakernel"))
        for name, c2, path in plans:
            try:
                subs[name] = sub_record(name, c2, args, pk, local, fwd_path=path,
                                        min_steps=200 if name.startswith("ep64") else 3)
            except Exception as exc:   # a sub-record never costs the headline line
                subs[name] = {"error": repr(exc)}
                torch.cuda.empty_cache()

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            try:
                cpu = cpu_baseline(cfg, args.cpu_seconds)
            except Exception as exc:   # a reported baseline only: keep the GPU line
                cpu = {"error": repr(exc), "kind": "oracle"}
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "mxfp8" if cfg.precision == "mxfp8" else "bf16", "data": "synthetic",
            "config": dict(workload_json(cfg), out=cfg.out, **mb,
                           fwd_path=args.fwd_path, tile_order=args.tile_order,
                           row_pairs=args.row_pairs, sm_pairs=args.sm_pairs,
                           parallelism=f"replicas x{world}"),
            "clocks": clocks, "gpu_launches": launches,
            "megakernel_phases_ms": phases or None,
            **a,
            "e2e": e2e, "cpu_baseline": cpu, "sub": subs,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- CPU oracle
class OracleStep:
    """The layer step (router, schedule, routed and shared experts: forward, and backward
    where the workload has one) run by the fp64 oracle on the host cores, on a bounded
    sample: the router and the schedule over all T tokens, some routed experts over the
    rows the router sends them, the shared expert over T/64 tokens. The time is extrapolated to the whole
    step by rows. Inputs are drawn once; every sampled expert uses the same drawn weights
    (the oracle's time does not depend on their values)."""

    def __init__(self, cfg, seed=0):
        import numpy as np
        self.np = np
        self.cfg = cfg
        rng = np.random.default_rng(seed)
        T, H, I, E, k, Is = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.shared_I
        self.x = rng.standard_normal((T, H), dtype=np.float32).astype(np.float64)
        self.dY = rng.standard_normal((T, H), dtype=np.float32).astype(np.float64)
        self.Wr = rng.normal(0, cfg.wr_std, (H, E)) if cfg.router else None
        self.bias = None
        if cfg.router and cfg.bias_experts:
            self.bias = np.zeros(E)
            self.bias[list(cfg.bias_experts)] = cfg.bias_value
        if not cfg.router:
            # caller-supplied routing with the workload's expert loads (Zipf counts)
            import moe_inputs as mi
            counts = (mi.zipf_counts(T * k, E, cfg.zipf_s) if cfg.zipf_s > 0
                      else [T * k // E] * E)
            labels = np.repeat(np.arange(E), counts)
            self.idx = rng.permutation(np.resize(labels, T * k)).reshape(T, k)
            u = rng.uniform(size=(T, k))
            self.gates = u / u.sum(axis=1, keepdims=True)
        self.precision = cfg.precision
        w = lambda *shape: rng.standard_normal(shape, dtype=np.float32).astype(np.float64) \
            * cfg.w_std
        self.W = (w(1, H, I), w(1, H, I), w(1, I, H))
        self.Ts = max(1, T // 64)
        self.shared = (w(H, Is), w(H, Is), w(Is, H)) if Is else None

    def run(self, first, max_rows=None, max_seconds=None):
        """Time one sample: routed experts first, first+1, ... (mod E), up to ``max_rows``
        rows or ``max_seconds`` of expert time, at least one non-empty expert and at most
        all E. Returns the measured and extrapolated seconds and where the next sample
        starts."""
        from oracle import moe
        np, cfg = self.np, self.cfg
        T, E, k = cfg.T, cfg.E, cfg.k
        t0 = time.perf_counter()
        if cfg.router:
            r = moe.route(self.x, self.Wr, k, self.bias)
            idx, gates = r.idx, r.gates
        else:
            idx, gates = self.idx, self.gates
        pl = moe.plan(idx, E)
        t_route = time.perf_counter() - t0
        t_exp, rows, n_exp, e = 0.0, 0, 0, first
        for step in range(E):
            if n_exp and ((max_rows is not None and rows >= max_rows) or
                          (max_seconds is not None and t_exp >= max_seconds)):
                break
            e = (first + step) % E
            r0, r1 = pl.offsets[e], pl.offsets[e + 1]
            n = int(r1 - r0)
            if n == 0:
                continue
            sel = pl.table[r0:r1]
            xs, dYs = self.x[sel[:, 0]], self.dY[sel[:, 0]]
            sub_idx = np.zeros((n, 1), np.int64)
            sub_g = gates[sel[:, 0], sel[:, 1]][:, None]
            t1 = time.perf_counter()
            _, saved = moe.forward(xs, sub_idx, sub_g, *self.W, precision=self.precision)
            if cfg.backward:
                moe.backward(xs, sub_idx, sub_g, *self.W, saved, dYs,
                             precision=self.precision)
            t_exp += time.perf_counter() - t1
            rows += n
            n_exp += 1
        t_shared = 0.0
        if self.shared is not None:
            xs, dYs = self.x[:self.Ts], self.dY[:self.Ts]
            t1 = time.perf_counter()
            _, ss = moe.shared_forward(xs, *self.shared, self.precision)
            if cfg.backward:
                moe.shared_backward(xs, *self.shared, ss, dYs, self.precision)
            t_shared = time.perf_counter() - t1
        total = t_route + (t_exp / max(rows, 1)) * T * k + t_shared * (T / self.Ts)
        return {"measured": t_route + t_exp + t_shared, "extrapolated": total,
                "experts": n_exp, "rows": rows, "next": (e + 1) % E}

    def describe(self, n_experts, rows):
        cfg = self.cfg
        passes = "fwd+bwd" if cfg.backward else "fwd"
        head = (f"router+schedule over all {cfg.T} tokens" if cfg.router else
                f"schedule over all {cfg.T} tokens (routing supplied)")
        shared = (f"; shared expert over {self.Ts} tokens scaled to {cfg.T}"
                  if self.shared is not None else "")
        return (f"{head}; {n_experts} of {cfg.E} routed experts {passes} ({rows} rows) "
                f"scaled to {cfg.T * cfg.k} rows{shared}; fp64 NumPy, "
                f"{self.precision} rounding model")


def cpu_baseline(cfg, seconds=10.0, seed=0):
    """The oracle on one bounded sample of the workload (routed experts in index order
    until about ``seconds`` of expert time), extrapolated to the whole step, in tokens per
    second."""
    step = OracleStep(cfg, seed)
    r = step.run(0, max_seconds=seconds)
    return {"value": round(cfg.T / r["extrapolated"], 3), "unit": "tokens/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": step.describe(r["experts"], r["rows"]),
            "seconds_measured": round(r["measured"], 2),
            "seconds_extrapolated": round(r["extrapolated"], 2)}


def run_reference(args):
    """The reference arm: the oracle, as it stands, on the host cores. W untimed warm-up
    steps, then K timed steps; every step is one bounded sample (the router and schedule
    over all tokens, routed experts taken in turn up to ``--ref-rows-per-step`` rows, the
    shared-expert slice), extrapolated to the whole step. Rank 0 alone runs it."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = workload_config(args.workload)
    step = OracleStep(cfg)
    nxt = 0

    def one():
        nonlocal nxt
        r = step.run(nxt, max_rows=args.ref_rows_per_step)
        nxt = r["next"]
        return r

    for _ in range(max(args.warmup, 0)):
        one()
    K = max(args.steps, 1)
    runs = [one() for _ in range(K)]
    ext = sum(r["extrapolated"] for r in runs)
    value = round(cfg.T * K / ext, 3)
    rows = sum(r["rows"] for r in runs)
    cpu = {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"each of {K} steps: " +
                     step.describe(round(sum(r["experts"] for r in runs) / K, 1), rows // K) +
                     " (experts taken in turn; mean per step)",
           "seconds_measured": round(sum(r["measured"] for r in runs), 2),
           "seconds_extrapolated": round(ext, 2)}
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(1e3 * ext / K, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_json(cfg), parallelism="replicas x1",
                       oracle="fp64 NumPy on the host cores, a bounded sample per step"),
        "cpu_baseline": cpu,
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
