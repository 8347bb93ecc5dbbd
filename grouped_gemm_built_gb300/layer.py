"""Torch-facing convenience around the C ABI: owns the caller-side buffers (schedule,
aux, workspace, saved activations, gradients) as torch tensors and calls mok_plan,
mok_moe_fwd and mok_moe_bwd on the current CUDA stream. Memory and streams only; all
arithmetic happens inside libmok.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import mok


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _dev(t, name: str, dtype: torch.dtype, numel: int, optional: bool = False):
    """The device address of a tensor handed to the library, after checking that it can
    be one: a CUDA tensor (a host address would be dereferenced on the GPU), contiguous,
    of ``dtype`` and ``numel`` elements. ``None`` passes where ``optional``."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device, got {t.device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return t.data_ptr()


class MoELayer:
    """One MoE SwiGLU layer of fixed dims on one CUDA device."""

    def __init__(self, T, H, I, E, k, shared_I=0, router=True, macrobatches=0, ring_bytes=0,
                 precision="bf16", device="cuda", out="bf16", minibatch_tokens=0):
        self.device = torch.device(device)
        if self.device.type != "cuda":
            raise ValueError(f"the layer's buffers live on a CUDA device, got {self.device}")
        self.dims = mok.MokDims(T=T, H=H, I=I, E=E, k=k, shared_I=shared_I,
                                router=1 if router else 0, macrobatches=macrobatches,
                                ring_bytes=ring_bytes, minibatch_tokens=minibatch_tokens)
        self.T, self.H, self.I, self.E, self.k, self.Is = T, H, I, E, k, shared_I
        self.router = router
        self.ctx = mok.mok_create(self.dims)
        self.set_precision(precision)
        self.set_output_dtype(out)
        self.sizes = mok.mok_get_sizes(self.ctx)
        dev = self.device
        u8 = dict(dtype=torch.uint8, device=dev)
        self.topk_idx = torch.zeros((T, k), dtype=torch.int32, device=dev)
        self.gates = torch.zeros((T, k), dtype=torch.float32, device=dev)
        self.counts = torch.zeros(E, dtype=torch.int32, device=dev)
        self.offsets = torch.zeros(E + 1, dtype=torch.int32, device=dev)
        self.table = torch.zeros((T * k, 2), dtype=torch.int32, device=dev)
        self.inv = torch.zeros((T, k), dtype=torch.int32, device=dev)
        self.aux = torch.zeros(self.sizes.aux_bytes, **u8)
        self.workspace = torch.empty(self.sizes.workspace_bytes, **u8)
        self.saved = torch.empty(self.sizes.saved_bytes, **u8)
        self.sched = mok.MokSched(topk_idx=self.topk_idx.data_ptr(), gates=self.gates.data_ptr(),
                                  counts=self.counts.data_ptr(), offsets=self.offsets.data_ptr(),
                                  table=self.table.data_ptr(), inv=self.inv.data_ptr(),
                                  aux=self.aux.data_ptr())

    def __del__(self):
        try:
            mok.mok_destroy(self.ctx)
        except Exception:
            pass

    def set_fwd_path(self, path: str):
        """"auto" (default), "megakernel" or "launches"."""
        codes = {"megakernel": mok.MOK_FWD_MEGAKERNEL, "launches": mok.MOK_FWD_LAUNCHES,
                 "auto": mok.MOK_FWD_AUTO}
        if path not in codes:
            raise ValueError(f"forward path must be one of {sorted(codes)}, got {path!r}")
        mok.mok_set_fwd_path(self.ctx, codes[path])
        self.fwd_path = path

    def set_precision(self, precision: str):
        self.precision = precision
        codes = {"bf16": mok.MOK_BF16, "mxfp8": mok.MOK_MXFP8,
                 "bf16_plain": mok.MOK_BF16_WGRAD_PLAIN}
        if precision not in codes:
            raise ValueError(f"precision must be one of {sorted(codes)}, got {precision!r}")
        mok.mok_set_precision(self.ctx, codes[precision])

    def set_output_dtype(self, out: str):
        """"bf16" (default) or "fp32": the type of y, dX and the weight gradients."""
        codes = {"bf16": mok.MOK_OUT_BF16, "fp32": mok.MOK_OUT_F32}
        if out not in codes:
            raise ValueError(f"output type must be one of {sorted(codes)}, got {out!r}")
        mok.mok_set_output_dtype(self.ctx, codes[out])
        self.out = out
        self.out_dtype = torch.bfloat16 if out == "bf16" else torch.float32

    @staticmethod
    def _stream():
        return torch.cuda.current_stream().cuda_stream

    def _routed_weights(self, W_up, W_gate, W_down):
        bf, EHI = torch.bfloat16, self.E * self.H * self.I
        return (_dev(W_up, "W_up", bf, EHI), _dev(W_gate, "W_gate", bf, EHI),
                _dev(W_down, "W_down", bf, EHI))

    def weights(self, W_up, W_gate, W_down, Ws_up=None, Ws_gate=None, Ws_down=None, mx=None):
        """The weight pointers for forward and backward: W_up, W_gate [E,H,I] and W_down
        [E,I,H] bf16; the shared expert's Ws_up, Ws_gate [H,Is], Ws_down [Is,H] bf16 when
        the layer has one; ``mx`` from ``quantize_weights`` for MXFP8."""
        up, gate, down = self._routed_weights(W_up, W_gate, W_down)
        sh = self.H * self.Is
        opt = self.Is == 0
        self._w_keep = (W_up, W_gate, W_down, Ws_up, Ws_gate, Ws_down, mx)
        return mok.MokWeights(
            W_up=up, W_gate=gate, W_down=down,
            Ws_up=_dev(Ws_up, "Ws_up", torch.bfloat16, sh, opt),
            Ws_gate=_dev(Ws_gate, "Ws_gate", torch.bfloat16, sh, opt),
            Ws_down=_dev(Ws_down, "Ws_down", torch.bfloat16, sh, opt),
            mx=_dev(mx, "mx", torch.uint8, self.sizes.mx_weight_bytes, True))

    def quantize_weights(self, W_up, W_gate, W_down):
        """MXFP8 copies of the routed weights (library-private layout), as a uint8 tensor."""
        up, gate, down = self._routed_weights(W_up, W_gate, W_down)
        mx = torch.empty(self.sizes.mx_weight_bytes, dtype=torch.uint8, device=self.device)
        w = mok.MokWeights(W_up=up, W_gate=gate, W_down=down)
        mok.mok_quantize_weights_mxfp8(self.ctx, w, mx.data_ptr(), self._stream())
        return mx

    def plan(self, x=None, Wr=None, bias=None, topk_idx=None, gates=None):
        """Routing and schedule. With the router: x [T,H] bf16, Wr [H,E] fp32, optional
        bias [E] fp32. Without: the caller's topk_idx [T,k] and gates [T,k], copied into
        the schedule's buffers."""
        if not self.router:
            if x is not None or Wr is not None or bias is not None:
                raise ValueError("a layer without a router takes topk_idx and gates only")
            if topk_idx is None or gates is None:
                raise ValueError("a layer without a router needs topk_idx and gates")
            self.topk_idx.copy_(topk_idx)
            self.gates.copy_(gates)
            px = pw = pb = None
        else:
            px = _dev(x, "x", torch.bfloat16, self.T * self.H)
            pw = _dev(Wr, "Wr", torch.float32, self.H * self.E)
            pb = _dev(bias, "bias", torch.float32, self.E, optional=True)
        mok.mok_plan(self.ctx, px, pw, pb, self.sched, self.workspace.data_ptr(),
                     self._stream())

    def forward(self, x, w: "mok.MokWeights", y=None):
        """y [T,H] in the output type (allocated when not given) from x [T,H] bf16."""
        px = _dev(x, "x", torch.bfloat16, self.T * self.H)
        if y is None:
            y = torch.empty((self.T, self.H), dtype=self.out_dtype, device=self.device)
        py = _dev(y, "y", self.out_dtype, self.T * self.H)
        mok.mok_moe_fwd(self.ctx, self.sched, px, w, py, self.saved.data_ptr(),
                        self.workspace.data_ptr(), self._stream())
        return y

    def alloc_grads(self):
        """dX and the weight gradients in the output type; dgates and dWr fp32."""
        dev = self.device
        bf = dict(dtype=self.out_dtype, device=dev)
        g = {
            "dX": torch.empty((self.T, self.H), **bf),
            "dW_up": torch.empty((self.E, self.H, self.I), **bf),
            "dW_gate": torch.empty((self.E, self.H, self.I), **bf),
            "dW_down": torch.empty((self.E, self.I, self.H), **bf),
            "dgates": torch.empty((self.T, self.k), dtype=torch.float32, device=dev),
            "dWr": torch.empty((self.H, self.E), dtype=torch.float32, device=dev)
            if self.router else None,
        }
        if self.Is:
            g["dWs_up"] = torch.empty((self.H, self.Is), **bf)
            g["dWs_gate"] = torch.empty((self.H, self.Is), **bf)
            g["dWs_down"] = torch.empty((self.Is, self.H), **bf)
        else:
            g["dWs_up"] = g["dWs_gate"] = g["dWs_down"] = None
        return g

    def backward(self, x, Wr, w: "mok.MokWeights", dY, grads=None):
        """Gradients (the shapes and types of ``alloc_grads``, allocated when not given)
        from x and dY [T,H] bf16; Wr [H,E] fp32 when the layer runs its router, else None."""
        g = grads if grads is not None else self.alloc_grads()
        f32, od = torch.float32, self.out_dtype
        EHI, TH, sh = self.E * self.H * self.I, self.T * self.H, self.H * self.Is
        no_sh = self.Is == 0
        mg = mok.MokGrads(
            dW_up=_dev(g["dW_up"], "dW_up", od, EHI),
            dW_gate=_dev(g["dW_gate"], "dW_gate", od, EHI),
            dW_down=_dev(g["dW_down"], "dW_down", od, EHI),
            dgates=_dev(g["dgates"], "dgates", f32, self.T * self.k),
            dWr=_dev(g.get("dWr"), "dWr", f32, self.H * self.E, optional=True),
            dWs_up=_dev(g.get("dWs_up"), "dWs_up", od, sh, no_sh),
            dWs_gate=_dev(g.get("dWs_gate"), "dWs_gate", od, sh, no_sh),
            dWs_down=_dev(g.get("dWs_down"), "dWs_down", od, sh, no_sh))
        px = _dev(x, "x", torch.bfloat16, TH)
        pwr = _dev(Wr, "Wr", f32, self.H * self.E, optional=True)
        pdy = _dev(dY, "dY", torch.bfloat16, TH)
        pdx = _dev(g["dX"], "dX", od, TH)
        mok.mok_moe_bwd(self.ctx, self.sched, px, pwr, w, self.saved.data_ptr(), pdy, pdx, mg,
                        self.workspace.data_ptr(), self._stream())
        return g

    def status(self) -> int:
        return mok.mok_get_status(self.ctx, self.sched, self._stream())
