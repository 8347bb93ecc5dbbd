"""A mixed-precision training loop through the C ABI: fp32 master weights kept by the
caller, bf16 copies and their MXFP8 quantisation made each step, the routed experts in
MXFP8 and the shared expert in BF16 ("Outras características" on the stamatios.com page:
MXFP8 training with a BF16 shared expert), bf16 gradients applied to the fp32 masters.
The step's arithmetic outside the library (casts, the loss gradient, the update) is
plain torch; every layer operation runs in the library.

The loss is 0.5 |y - target|^2 / T. Each step moves the expert weights by -lr * grad with
lr fixed so that the first step's first-order decrease is 0.5% of the loss, and the router
weights by a step whose largest logit change is 0.005 (larger router steps move tokens
between experts, where the loss jumps). The measured decrease of the first step must
match its first-order prediction, lr * |grad|^2, which checks the gradients' direction and
scale against the forward, and the loss must fall at every step."""
import pytest
import torch

import moe_inputs as mi
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

EXPERT = (("W_up", "dW_up"), ("W_gate", "dW_gate"), ("W_down", "dW_down"),
          ("Ws_up", "dWs_up"), ("Ws_gate", "dWs_gate"), ("Ws_down", "dWs_down"))


def test_mixed_precision_steps_lower_the_loss():
    cfg = mi.MoEConfig("train_mx", T=512, H=256, I=256, E=8, k=2, shared_I=128,
                       precision="mxfp8")
    inp = gu.gpu_inputs(cfg, seed=21)
    d = gu.to_dev(inp)
    master = {n: d[n].float().clone() for n, _ in EXPERT}
    Wr = d["Wr"].clone()
    target = torch.randn((cfg.T, cfg.H), device="cuda", generator=torch.Generator(
        device="cuda").manual_seed(5))
    L = gu.make_layer(cfg)
    xf = d["x"].float()

    def evaluate():
        w16 = {n: v.to(torch.bfloat16).contiguous() for n, v in master.items()}
        mx = L.quantize_weights(w16["W_up"], w16["W_gate"], w16["W_down"])
        w = L.weights(w16["W_up"], w16["W_gate"], w16["W_down"], w16["Ws_up"], w16["Ws_gate"],
                      w16["Ws_down"], mx=mx)
        L.plan(x=d["x"], Wr=Wr, bias=None)
        y = L.forward(d["x"], w).float()
        diff = y - target
        loss = 0.5 * float((diff * diff).sum()) / cfg.T
        g = L.backward(d["x"], Wr, w, (diff / cfg.T).to(torch.bfloat16).contiguous())
        torch.cuda.synchronize()
        assert L.status() == 0
        return loss, g

    loss, g = evaluate()
    losses, predicted = [loss], []
    lr = None
    for _ in range(5):
        gsq = 0.0
        for n, gn in EXPERT:
            grad = g[gn].float()
            assert g[gn].dtype == torch.bfloat16 and torch.isfinite(grad).all(), gn
            gsq += float((grad * grad).sum())
        if lr is None:
            lr = 0.005 * losses[0] / gsq
        lr_r = 0.005 / float((xf @ g["dWr"]).abs().max())
        predicted.append(lr * gsq + lr_r * float((g["dWr"] ** 2).sum()))
        for n, gn in EXPERT:
            master[n] -= lr * g[gn].float()
        Wr -= lr_r * g["dWr"]
        loss, g = evaluate()
        losses.append(loss)
    drops = [a - b for a, b in zip(losses, losses[1:])]
    print("losses", losses, "first-order decreases", predicted)
    assert 0.7 < drops[0] / predicted[0] < 1.3, (drops[0], predicted[0])
    assert all(dr > 0 for dr in drops), losses
    assert losses[-1] < 0.985 * losses[0], losses
