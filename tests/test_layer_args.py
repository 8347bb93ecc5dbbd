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


def _bare_layer(router=True, shared_I=0):
    """The layer's dims without its device buffers or library context: enough for the
    argument checks, which all run before the library is called."""
    L = lay.MoELayer.__new__(lay.MoELayer)
    L.T, L.H, L.I, L.E, L.k, L.Is, L.router = 16, 128, 128, 4, 2, shared_I, router
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


def test_router_less_layer_takes_routing_only():
    L = _bare_layer(router=False)
    with pytest.raises(ValueError, match="topk_idx and gates only"):
        L.plan(x=dev(16, 128))
    with pytest.raises(ValueError, match="needs topk_idx and gates"):
        L.plan(topk_idx=dev(16, 2, dtype=torch.int32))
