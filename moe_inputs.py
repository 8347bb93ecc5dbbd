"""Seeded synthetic inputs for the MoE SwiGLU layer, shared by the CUDA path's tests,
the benchmark and the CPU oracle.

This module holds no arithmetic of the layer itself: it only draws random tensors with
the shapes and distributions of the workloads below and hands out the same bits to both
sides. The workloads are the ones the Mixture-of-Kittens articles discuss (a Kimi-2.5
shaped layer with H=7168, I=2048 from "Cursor abre código de megakernel MoE para GPUs
NVL72", section "Granularidade do overlap computação-comunicação"; a per-GPU EP=64 slice
with 2048 tokens per GPU from the same page, section "Resultados"; DeepSeek-V3 with
hundreds of experts from the sebask.de article, intro) plus a tiny and a mid case.

Draw order inside one seed: x, Wr, W_up, W_gate, W_down, shared (up, gate, down), dY.
Tensors are drawn with a seeded ``torch.Generator`` on the requested device; bf16
tensors are the fp32 draws rounded to bf16 by torch's own conversion.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens
    H: int            # hidden size
    I: int            # expert intermediate size
    E: int            # routed experts
    k: int            # experts per token
    shared_I: int = 0  # 0 = no shared expert
    router: bool = True          # False: routing (expert ids, gates) is an input
    zipf_s: float = 0.0          # >0: expert loads drawn with Zipf(s) counts (no router)
    bias_experts: tuple = ()     # experts that get a router-logit bias
    bias_value: float = 0.0
    x_std: float = 1.0
    w_std: float = 0.02
    wr_std: float = 0.02
    precision: str = "bf16"      # "bf16", "mxfp8" or "bf16_plain" (single bf16 dW operands)
    backward: bool = True
    macrobatches: int = 1
    ring_bytes: int = 0          # 0 = ring sized to hold every routed row
    out: str = "bf16"            # type of y, dX and the weight gradients: "bf16" or "fp32"
    minibatch_tokens: int = 0    # tokens per macrobatch (-1: the two-wave rule; 0: unused)

    @property
    def R(self) -> int:
        return self.T * self.k


CONFIGS = {
    "tiny": MoEConfig("tiny", T=256, H=256, I=128, E=8, k=2),
    "mid": MoEConfig("mid", T=4096, H=2048, I=1024, E=64, k=6),
    "kimi_2368": MoEConfig("kimi_2368", T=2368, H=7168, I=2048, E=384, k=8, shared_I=2048),
    "kimi_8192": MoEConfig("kimi_8192", T=8192, H=7168, I=2048, E=384, k=8, shared_I=2048),
    "kimi_8192_plain": MoEConfig("kimi_8192_plain", T=8192, H=7168, I=2048, E=384, k=8,
                                 shared_I=2048, precision="bf16_plain"),
    "ep64_slice": MoEConfig("ep64_slice", T=2048, H=7168, I=2048, E=6, k=8, router=False,
                            zipf_s=1.2, precision="mxfp8", backward=False, macrobatches=4,
                            ring_bytes=256 << 20),
    "dsv3_imbalanced": MoEConfig("dsv3_imbalanced", T=16384, H=7168, I=2048, E=256, k=8,
                                 bias_experts=(0, 1, 2, 3), bias_value=3.0,
                                 precision="mxfp8"),
    # Kimi-2.5 expert shape with 24 experts and the same ~171 rows per expert as T=8192:
    # a few GB on the device, for detailed kernel profiles.
    "kimi_e24_profile": MoEConfig("kimi_e24_profile", T=512, H=7168, I=2048, E=24, k=8),
    "kimi_e24_profile_plain": MoEConfig("kimi_e24_profile_plain", T=512, H=7168, I=2048,
                                        E=24, k=8, precision="bf16_plain"),
    # Kimi-2.5 hidden size, every token to all 8 experts (32768 routed rows, 0.47 GB of
    # gathered bf16 rows, more than L2): a few GB on the device, for the DRAM counters of
    # the row-moving kernels (dispatch, combine and their reverses) and the router's.
    "kimi_movement_profile": MoEConfig("kimi_movement_profile", T=4096, H=7168, I=2048, E=8,
                                       k=8, precision="bf16_plain"),
    # DeepSeek-V3 expert shape in MXFP8 with 16 experts and the same ~512 rows per expert
    # as T=16384 with 256 experts: a few GB on the device, for detailed kernel profiles.
    "dsv3_e16_profile": MoEConfig("dsv3_e16_profile", T=1024, H=7168, I=2048, E=16, k=8,
                                  precision="mxfp8"),
}


def scaled(cfg: MoEConfig, **over) -> MoEConfig:
    """A copy of ``cfg`` with some fields replaced (smaller cases of the same structure)."""
    return dataclasses.replace(cfg, **over)


def zipf_counts(total: int, n: int, s: float) -> list:
    """Deterministic per-expert row counts proportional to rank^-s, rounded by largest
    remainder so that they sum to ``total`` exactly (rank 1 first)."""
    w = [r ** (-s) for r in range(1, n + 1)]
    z = sum(w)
    raw = [total * wi / z for wi in w]
    base = [int(math.floor(v)) for v in raw]
    rest = total - sum(base)
    order = sorted(range(n), key=lambda i: (-(raw[i] - base[i]), i))
    for i in order[:rest]:
        base[i] += 1
    return base


def make_inputs(cfg: MoEConfig, seed: int = 0, device="cpu", with_dy: Optional[bool] = None):
    """Draw every input of one layer call. Returns a dict of torch tensors on ``device``:

    x [T,H] bf16; Wr [H,E] fp32 (router only); bias [E] fp32 (or None);
    W_up, W_gate [E,H,I] bf16; W_down [E,I,H] bf16;
    Ws_up, Ws_gate [H,Is] bf16, Ws_down [Is,H] bf16 (shared expert, or None);
    topk_idx [T,k] int32 and gates [T,k] fp32 when routing is an input;
    dY [T,H] bf16 when the config has a backward pass.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k

    def normal(shape, std, dtype=torch.bfloat16):
        t = torch.empty(shape, dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=g)
        return t.to(dtype)

    out = {}
    out["x"] = normal((T, H), cfg.x_std)
    if cfg.router:
        out["Wr"] = normal((H, E), cfg.wr_std, torch.float32)
        if cfg.bias_experts:
            b = torch.zeros(E, dtype=torch.float32)
            b[list(cfg.bias_experts)] = cfg.bias_value
            out["bias"] = b.to(device)
        else:
            out["bias"] = None
    else:
        out["Wr"] = None
        out["bias"] = None
    out["W_up"] = normal((E, H, I), cfg.w_std)
    out["W_gate"] = normal((E, H, I), cfg.w_std)
    out["W_down"] = normal((E, I, H), cfg.w_std)
    if cfg.shared_I:
        Is = cfg.shared_I
        out["Ws_up"] = normal((H, Is), cfg.w_std)
        out["Ws_gate"] = normal((H, Is), cfg.w_std)
        out["Ws_down"] = normal((Is, H), cfg.w_std)
    else:
        out["Ws_up"] = out["Ws_gate"] = out["Ws_down"] = None
    if not cfg.router:
        # Expert ids: Zipf(s) counts over the T*k slots, labels spread by a seeded
        # permutation (a token may hit the same expert twice); gates U(0,1) per slot,
        # renormalised over the token's k slots.
        counts = zipf_counts(T * k, E, cfg.zipf_s) if cfg.zipf_s > 0 else [T * k // E] * E
        labels = torch.cat([torch.full((c,), e, dtype=torch.int32) for e, c in enumerate(counts)])
        perm = torch.randperm(T * k, generator=torch.Generator().manual_seed(seed + 1))
        out["topk_idx"] = labels[perm].reshape(T, k).contiguous().to(device)
        u = torch.rand((T, k), generator=torch.Generator().manual_seed(seed + 2), dtype=torch.float32)
        out["gates"] = (u / u.sum(dim=1, keepdim=True)).contiguous().to(device)
    if with_dy is None:
        with_dy = cfg.backward
    out["dY"] = normal((T, H), 1.0) if with_dy else None
    return out


def to_f64(t):
    """torch tensor (any float dtype) -> numpy float64 array; None passes through."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float32).double().numpy()
