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


class MoELayer:
    """One MoE SwiGLU layer of fixed dims on one CUDA device."""

    def __init__(self, T, H, I, E, k, shared_I=0, router=True, macrobatches=0, ring_bytes=0,
                 precision="bf16", device="cuda"):
        self.device = torch.device(device)
        self.dims = mok.MokDims(T=T, H=H, I=I, E=E, k=k, shared_I=shared_I,
                                router=1 if router else 0, macrobatches=macrobatches,
                                ring_bytes=ring_bytes)
        self.T, self.H, self.I, self.E, self.k, self.Is = T, H, I, E, k, shared_I
        self.router = router
        self.ctx = mok.mok_create(self.dims)
        self.set_precision(precision)
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

    @staticmethod
    def _stream():
        return torch.cuda.current_stream().cuda_stream

    def weights(self, W_up, W_gate, W_down, Ws_up=None, Ws_gate=None, Ws_down=None, mx=None):
        self._w_keep = (W_up, W_gate, W_down, Ws_up, Ws_gate, Ws_down, mx)
        return mok.MokWeights(W_up=_ptr(W_up), W_gate=_ptr(W_gate), W_down=_ptr(W_down),
                              Ws_up=_ptr(Ws_up), Ws_gate=_ptr(Ws_gate), Ws_down=_ptr(Ws_down),
                              mx=_ptr(mx))

    def quantize_weights(self, W_up, W_gate, W_down):
        """MXFP8 copies of the routed weights (library-private layout), as a uint8 tensor."""
        mx = torch.empty(self.sizes.mx_weight_bytes, dtype=torch.uint8, device=self.device)
        w = mok.MokWeights(W_up=W_up.data_ptr(), W_gate=W_gate.data_ptr(),
                           W_down=W_down.data_ptr())
        mok.mok_quantize_weights_mxfp8(self.ctx, w, mx.data_ptr(), self._stream())
        return mx

    def plan(self, x=None, Wr=None, bias=None, topk_idx=None, gates=None):
        if not self.router:
            self.topk_idx.copy_(topk_idx)
            self.gates.copy_(gates)
        mok.mok_plan(self.ctx, _ptr(x), _ptr(Wr), _ptr(bias), self.sched,
                     self.workspace.data_ptr(), self._stream())

    def forward(self, x, w: "mok.MokWeights", y=None):
        if y is None:
            y = torch.empty((self.T, self.H), dtype=torch.float32, device=self.device)
        mok.mok_moe_fwd(self.ctx, self.sched, x.data_ptr(), w, y.data_ptr(),
                        self.saved.data_ptr(), self.workspace.data_ptr(), self._stream())
        return y

    def alloc_grads(self):
        dev = self.device
        bf = dict(dtype=torch.float32, device=dev)   # all gradients are fp32
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
        g = grads if grads is not None else self.alloc_grads()
        mg = mok.MokGrads(dW_up=_ptr(g["dW_up"]), dW_gate=_ptr(g["dW_gate"]),
                          dW_down=_ptr(g["dW_down"]), dgates=_ptr(g["dgates"]),
                          dWr=_ptr(g["dWr"]), dWs_up=_ptr(g["dWs_up"]),
                          dWs_gate=_ptr(g["dWs_gate"]), dWs_down=_ptr(g["dWs_down"]))
        mok.mok_moe_bwd(self.ctx, self.sched, x.data_ptr(), _ptr(Wr), w, self.saved.data_ptr(),
                        dY.data_ptr(), g["dX"].data_ptr(), mg, self.workspace.data_ptr(),
                        self._stream())
        return g

    def status(self) -> int:
        return mok.mok_get_status(self.ctx, self.sched, self._stream())
