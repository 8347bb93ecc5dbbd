"""The torch-facing layer hands raw addresses to the library, so it checks every tensor
first: a host tensor, a wrong dtype, a strided view or a wrong size never reaches a
kernel. These checks are plain Python and run here without a GPU; tensors that claim to
be on a CUDA device stand in for device tensors (their addresses are never used)."""
import pytest
import torch

from grouped_gemm_built_gb300 import layer as lay


class _OnDevice(torch.Tensor):
    """A host tensor that reports itself as a CUDA tensor, for the checks only."""

    @property
    def is_cuda(self):
        return True


def dev(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype).as_subclass(_OnDevice)


def test_dev_accepts_a_device_tensor_of_the_stated_kind():
    t = dev(4, 8)
    assert lay._dev(t, "x", torch.bfloat16, 32) == t.data_ptr()
    assert lay._dev(None, "bias", torch.float32, 8, optional=True) is None


@pytest.mark.parametrize("t,err,what", [
    (None, ValueError, "required"),
    (torch.zeros(4, 8, dtype=torch.bfloat16), ValueError, "CUDA device"),   # host memory
    (dev(4, 8, dtype=torch.float32), ValueError, "bfloat16"),
    (dev(8, 4).t(), ValueError, "contiguous"),
    (dev(4, 9), ValueError, "32 elements"),
    ([0.0] * 32, TypeError, "torch.Tensor"),
])
def test_dev_rejects(t, err, what):
    with pytest.raises(err, match=what):
        lay._dev(t, "x", torch.bfloat16, 32)


def test_layer_refuses_host_buffers():
    with pytest.raises(ValueError):
        lay.MoELayer(256, 256, 128, 8, 2, device="cpu")


def _bare_layer(router=True, shared_I=0, out_dtype=torch.float32):
    """The layer's dims without its device buffers or library context: enough for the
    argument checks, which all run before the library is called."""
    L = lay.MoELayer.__new__(lay.MoELayer)
    L.T, L.H, L.I, L.E, L.k, L.Is, L.router = 16, 128, 128, 4, 2, shared_I, router
    L.out_dtype = out_dtype
    L.ctx = None

    class _S:
        mx_weight_bytes = 1024

    L.sizes = _S()
    return L


def test_layer_calls_check_their_tensors_before_the_library():
    L = _bare_layer()
    x, Wr = dev(16, 128), dev(128, 4, dtype=torch.float32)
    W = [dev(4, 128, 128) for _ in range(3)]
    with pytest.raises(ValueError, match="CUDA"):
        L.plan(x=torch.zeros(16, 128, dtype=torch.bfloat16), Wr=Wr)
    with pytest.raises(ValueError, match="float32"):
        L.plan(x=x, Wr=dev(128, 4))
    with pytest.raises(ValueError, match="bias"):
        L.plan(x=x, Wr=Wr, bias=dev(5, dtype=torch.float32))
    with pytest.raises(ValueError, match="W_gate"):
        L.weights(W[0], dev(4, 128, 64), W[2])
    with pytest.raises(ValueError, match="mx"):
        L.weights(*W, mx=dev(1000, dtype=torch.uint8))
    with pytest.raises(ValueError, match="Ws_up"):
        L.weights(*W, Ws_up=dev(128, 128))                  # no shared expert here
    with pytest.raises(ValueError, match="y must be torch.float32"):
        L.forward(x, None, y=dev(16, 128))
    with pytest.raises(ValueError, match="x must be contiguous"):
        L.forward(x.t(), None)
    g = {"dX": dev(16, 128, dtype=torch.float32),
         "dW_up": dev(4, 128, 128, dtype=torch.float32),
         "dW_gate": dev(4, 128, 128, dtype=torch.float32),
         "dW_down": dev(4, 128, 128, dtype=torch.float32),
         "dgates": dev(16, 2, dtype=torch.float32), "dWr": dev(128, 4, dtype=torch.float32)}
    with pytest.raises(ValueError, match="dY"):
        L.backward(x, Wr, None, dev(16, 128, dtype=torch.float32), g)
    with pytest.raises(ValueError, match="dgates"):
        L.backward(x, Wr, None, dev(16, 128), dict(g, dgates=dev(16, 3, dtype=torch.float32)))
    with pytest.raises(ValueError, match="dX"):
        L.backward(x, Wr, None, dev(16, 128), dict(g, dX=torch.zeros(16, 128)))
    with pytest.raises(ValueError, match="Ws_up"):
        _bare_layer(shared_I=128).weights(*W)               # the shared expert's weights


def test_bf16_results_take_bf16_buffers():
    """With bf16 results, y, dX and the weight gradients must be bf16 tensors; dgates and
    dWr stay fp32."""
    L = _bare_layer(out_dtype=torch.bfloat16)
    x, Wr = dev(16, 128), dev(128, 4, dtype=torch.float32)
    with pytest.raises(ValueError, match="y must be torch.bfloat16"):
        L.forward(x, None, y=dev(16, 128, dtype=torch.float32))
    g = {"dX": dev(16, 128), "dW_up": dev(4, 128, 128), "dW_gate": dev(4, 128, 128),
         "dW_down": dev(4, 128, 128), "dgates": dev(16, 2, dtype=torch.float32),
         "dWr": dev(128, 4, dtype=torch.float32)}
    with pytest.raises(ValueError, match="dW_down must be torch.bfloat16"):
        L.backward(x, Wr, None, dev(16, 128),
                   dict(g, dW_down=dev(4, 128, 128, dtype=torch.float32)))
    with pytest.raises(ValueError, match="dgates must be torch.float32"):
        L.backward(x, Wr, None, dev(16, 128), dict(g, dgates=dev(16, 2)))
    with pytest.raises(ValueError, match="dX must be torch.bfloat16"):
        L.backward(x, Wr, None, dev(16, 128), dict(g, dX=dev(16, 128, dtype=torch.float32)))


def test_router_less_layer_takes_routing_only():
    L = _bare_layer(router=False)
    with pytest.raises(ValueError, match="topk_idx and gates only"):
        L.plan(x=dev(16, 128))
    with pytest.raises(ValueError, match="needs topk_idx and gates"):
        L.plan(topk_idx=dev(16, 2, dtype=torch.int32))


class _TorchOnDevice:
    """torch, except that the tensors the layer allocates come back as device stand-ins."""

    def __getattr__(self, name):
        return getattr(torch, name)

    @staticmethod
    def empty(*shape, **kw):
        kw.pop("device", None)
        return torch.empty(*shape, **kw).as_subclass(_OnDevice)


def _on_device(inp):
    return {k: (v.as_subclass(_OnDevice) if isinstance(v, torch.Tensor) else v)
            for k, v in inp.items()}


@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("name", ["tiny", "ragged_shared", "tiny_mx", "sparse", "router_less",
                                  "single_expert"])
def test_the_gpu_tests_call_pattern_passes_the_checks(monkeypatch, name, out):
    """The call sequence of the GPU tests and the bench (plan, quantize_weights for MXFP8,
    weights, forward, alloc_grads, backward), on the inputs ``moe_inputs`` makes for them,
    passes every tensor check; the library calls are stubbed out."""
    import moe_inputs as mi
    cases = {
        "tiny": mi.CONFIGS["tiny"],
        "ragged_shared": mi.MoEConfig("ragged_shared", T=300, H=256, I=256, E=12, k=3,
                                      shared_I=128),
        "tiny_mx": mi.scaled(mi.CONFIGS["tiny"], name="tiny_mx", precision="mxfp8"),
        "sparse": mi.MoEConfig("sparse", T=40, H=128, I=128, E=64, k=2),
        "router_less": mi.MoEConfig("rl", T=200, H=256, I=128, E=6, k=8, router=False,
                                    zipf_s=1.2),
        "single_expert": mi.MoEConfig("one", T=64, H=128, I=128, E=1, k=1, shared_I=128),
    }
    cfg = cases[name]
    calls = []
    for fn in ("mok_plan", "mok_moe_fwd", "mok_moe_bwd", "mok_quantize_weights_mxfp8"):
        monkeypatch.setattr(lay.mok, fn, lambda *a, fn=fn: calls.append(fn))
    monkeypatch.setattr(lay, "torch", _TorchOnDevice())
    L = lay.MoELayer.__new__(lay.MoELayer)
    L.T, L.H, L.I, L.E, L.k, L.Is, L.router = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, \
        cfg.shared_I, cfg.router
    L.device, L.ctx = torch.device("cpu"), None
    L.out_dtype = torch.bfloat16 if out == "bf16" else torch.float32

    class _S:
        mx_weight_bytes = 4096

    L.sizes = _S()
    L.topk_idx = torch.zeros((cfg.T, cfg.k), dtype=torch.int32)
    L.gates = torch.zeros((cfg.T, cfg.k))
    L.workspace = L.saved = torch.zeros(256, dtype=torch.uint8)
    L.sched = None
    L._stream = lambda: 0
    d = _on_device(mi.make_inputs(cfg, seed=0, device="cpu", with_dy=True))
    if cfg.router:
        L.plan(x=d["x"], Wr=d["Wr"], bias=d["bias"])
    else:
        L.plan(topk_idx=d["topk_idx"], gates=d["gates"])
    mx = L.quantize_weights(d["W_up"], d["W_gate"], d["W_down"]) \
        if cfg.precision == "mxfp8" else None
    w = L.weights(d["W_up"], d["W_gate"], d["W_down"], d["Ws_up"], d["Ws_gate"], d["Ws_down"],
                  mx=mx)
    y = L.forward(d["x"], w)
    L.forward(d["x"], w, torch.empty((cfg.T, cfg.H), dtype=L.out_dtype).as_subclass(_OnDevice))
    g = L.backward(d["x"], d["Wr"] if cfg.router else None, w, d["dY"])
    L.backward(d["x"], d["Wr"] if cfg.router else None, w, d["dY"], g)
    assert y.shape == (cfg.T, cfg.H) and y.dtype == L.out_dtype
    assert g["dW_up"].dtype == L.out_dtype and g["dgates"].dtype == torch.float32
    assert calls.count("mok_moe_bwd") == 2 and calls.count("mok_moe_fwd") == 2
