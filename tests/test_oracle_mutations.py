"""The oracle's pins are strong enough: each test here plants one plausible mistake in the
oracle (on the CPU, for the duration of the test only) and checks that at least one of
the pins named for it then fails. A mistake is a source edit of one oracle function: a
dropped term, a wrong sign or index, a swapped operand, a rounding put in the wrong place.
The edited function replaces the original wherever the oracle or the pins hold it.
"""
import inspect
import sys
import textwrap

import numpy as np
import pytest

from oracle import moe, numerics, sampled
from tests import test_oracle_layer as tl
from tests import test_oracle_numerics as tn


def _rng():
    return np.random.default_rng(1234)


def _holders():
    return [m for name, m in list(sys.modules.items())
            if m is not None and (name == "oracle" or name.startswith("oracle.")
                                  or name.startswith("tests."))]


def plant(monkeypatch, owner, name, old, new):
    """Replace ``owner.name`` (a function of an oracle module, or a method of one of its
    classes) by a copy whose source has ``old`` replaced by ``new``."""
    orig = inspect.unwrap(getattr(owner, name))
    src = textwrap.dedent(inspect.getsource(orig))
    assert src.count(old) == 1, (name, old)
    glb = dict(orig.__globals__)
    exec(compile(src.replace(old, new), f"<planted mistake in {name}>", "exec"), glb)
    mutant = glb[name]
    if inspect.isclass(owner):
        monkeypatch.setattr(owner, name, mutant)
        return
    for m in _holders():
        for attr, v in list(vars(m).items()):
            if v is orig:
                monkeypatch.setattr(m, attr, mutant)


def _fails(pin):
    try:
        pin()
    except (AssertionError, ValueError, IndexError):
        return True
    return False


# The pins, as callables with their parameters.
P = {
    "route_brute": lambda: tl.test_route_matches_python_brute_force(_rng()),
    "route_ties": lambda: tl.test_route_ties_go_to_lower_expert(),
    "route_inv": lambda: tl.test_route_invariants(_rng()),
    "plan_loops": lambda: tl.test_plan_matches_loops_and_invariants(_rng(), 40, 6, 3),
    "fwd_brute": lambda: tl.test_forward_matches_per_token_brute_force(_rng()),
    "fwd_identity": lambda: tl.test_forward_identity_experts_return_input(_rng()),
    "fwd_dense": lambda: tl.test_forward_single_expert_is_dense_swiglu(_rng()),
    "fwd_gates": lambda: tl.test_forward_is_linear_in_gates(_rng()),
    "shared_fwd": lambda: tl.test_shared_expert_adds_dense_ffn(_rng()),
    "fd": lambda: tl.test_backward_matches_finite_differences(_rng(), False, False),
    "fd_shared": lambda: tl.test_backward_matches_finite_differences(_rng(), True, True),
    "fd_dgates": lambda: tl.test_dgates_match_finite_differences(_rng()),
    "router_inv": lambda: tl.test_router_backward_invariants(_rng()),
    "empty": lambda: tl.test_empty_experts_get_zero_gradients(_rng()),
    "sampled": lambda: tl.test_sampled_evaluators_match_the_dense_oracle(_rng(), "fp32"),
    "sampled_bf16": lambda: tl.test_sampled_evaluators_match_the_dense_oracle(_rng(), "bf16"),
    "mx_bwd_eval": lambda: tl.test_mx_backward_evaluators_match_the_dense_oracle(_rng(), "fp32"),
    "mx_bwd_eval_bf16": lambda: tl.test_mx_backward_evaluators_match_the_dense_oracle(
        _rng(), "bf16"),
    "out_fwd": lambda: tl.test_result_rounding_points_forward(_rng()),
    "out_bwd": lambda: tl.test_result_rounding_points_backward(_rng()),
    "saved_uv": lambda: tl.test_saved_uv_rounding_point(_rng()),
    "wgrad_plain": lambda: tl.test_weight_gradient_operand_rounding_point(_rng(), "bf16_plain"),
    "wgrad_hilo": lambda: tl.test_weight_gradient_operand_rounding_point(_rng(), "bf16"),
    "down_bf16": lambda: tl.test_down_gemm_operand_rounding_point(_rng(), "bf16"),
    "down_mx": lambda: tl.test_down_gemm_operand_rounding_point(_rng(), "mxfp8"),
    "dx_bf16": lambda: tl.test_dx_gemm_operand_rounding_point(_rng(), "bf16"),
    "dx_mx": lambda: tl.test_dx_gemm_operand_rounding_point(_rng(), "mxfp8"),
    "bf16_torch": lambda: tn.test_bf16_round_matches_torch(_rng()),
    "e4m3_torch": lambda: tn.test_e4m3_encode_matches_torch_in_range(_rng()),
    "e4m3_sat": lambda: tn.test_e4m3_saturates(),
    "mx_448": lambda: tn.test_mx_scale_for_amax_448_times_power_of_two(5, _rng()),
    "mx_pow2": lambda: tn.test_mx_powers_of_two_closed_form(),
    "mx_zero": lambda: tn.test_mx_zero_block_and_saturation(),
    "mx_axis": lambda: tn.test_mx_axis_and_error_bound(_rng()),
    "mx_rows": lambda: tn.test_mx_rows_padded_equals_explicit_zero_rows(_rng()),
    "silu": lambda: tn.test_silu_and_derivative(),
    "dw_lines_bf16": lambda: tl.test_dw_lines_and_mx_token_forward_match_the_dense_oracle(
        _rng(), "bf16", "fp32"),
    "dw_lines_plain": lambda: tl.test_dw_lines_and_mx_token_forward_match_the_dense_oracle(
        _rng(), "bf16_plain", "fp32"),
    "dw_lines_out": lambda: tl.test_dw_lines_and_mx_token_forward_match_the_dense_oracle(
        _rng(), "bf16", "bf16"),
    "shared_lines_plain": lambda: tl.test_shared_dw_lines_match_the_dense_oracle(
        _rng(), "bf16_plain", "fp32"),
    "shared_lines_mx": lambda: tl.test_shared_dw_lines_match_the_dense_oracle(
        _rng(), "mxfp8", "fp32"),
    "shared_lines_out": lambda: tl.test_shared_dw_lines_match_the_dense_oracle(
        _rng(), "bf16", "bf16"),
}

# (owner, function, original text, planted text, pins expected to catch it)
MISTAKES = {
    # routing
    "top-k picks the smallest logits": (
        moe, "select", "np.argsort(-logits,", "np.argsort(logits,", ["route_brute"]),
    "gates not renormalised over the chosen set": (
        moe, "select", "gates = pS / pS.sum(axis=1, keepdims=True)", "gates = pS",
        ["route_inv", "route_brute"]),
    "ties go to the higher expert": (
        moe, "select", 'order = np.argsort(-logits, axis=1, kind="stable")',
        'order = logits.shape[1] - 1 - np.argsort(-logits[:, ::-1], axis=1, kind="stable")',
        ["route_ties"]),
    # schedule
    "table holds (slot, token) instead of (token, slot)": (
        moe, "plan", "np.stack([order // k, order % k], axis=1)",
        "np.stack([order % k, order // k], axis=1)", ["plan_loops"]),
    "inverse is the table's order itself": (
        moe, "plan", "inv[order] = np.arange(T * k)", "inv[:] = order", ["plan_loops"]),
    "rows of an expert in descending slot order": (
        moe, "plan", 'order = np.argsort(flat, kind="stable")',
        'order = np.argsort(flat * (T * k) - np.arange(T * k), kind="stable")',
        ["plan_loops"]),
    # forward
    "combine drops the gate": (
        moe, "forward", "y += gates[:, j:j + 1] * O_rows[pl.inv[:, j]]",
        "y += O_rows[pl.inv[:, j]]", ["fwd_brute", "fwd_gates"]),
    "SwiGLU gates the wrong projection": (
        moe, "forward", "h = P.fwd_act(silu(V) * U, 1)", "h = P.fwd_act(silu(U) * V, 1)",
        ["fwd_brute", "fwd_dense"]),
    "another expert's up projection": (
        moe, "forward", "U = A @ P.op(W_up[e], 0)", "U = A @ P.op(W_up[(e + 1) % E], 0)",
        ["fwd_brute"]),
    "dispatch pulls by slot, not by token": (
        moe, "forward", "Xe = x[pl.table[r0:r1, 0]]", "Xe = x[pl.table[r0:r1, 1]]",
        ["fwd_brute", "fwd_identity"]),
    "shared expert left out of y": (
        moe, "forward", "y = y + Os", "y = y", ["shared_fwd"]),
    "h not rounded for the down GEMM": (
        moe.Precision, "fwd_act", "return mx_qdq(a, axis) if self.mx else bf16_round(a)",
        "return mx_qdq(a, axis) if self.mx else a", ["down_bf16", "dx_bf16"]),
    "h quantised along the wrong axis": (
        moe.Precision, "fwd_act", "return mx_qdq(a, axis) if self.mx else bf16_round(a)",
        "return mx_qdq(a, 0) if self.mx else bf16_round(a)", ["down_mx", "dx_mx"]),
    # backward
    "dv without the factor U": (
        moe, "backward", "dv = dh * Us * dsilu(Vs)", "dv = dh * dsilu(Vs)", ["fd"]),
    "du with V in place of silu(V)": (
        moe, "backward", "du = dh * silu(Vs)", "du = dh * Vs", ["fd"]),
    "router-weight gradient against U instead of h": (
        moe, "backward", "dgates[t, j] = (D * hv).sum(axis=1)",
        "dgates[t, j] = (D * Us).sum(axis=1)", ["fd_dgates"]),
    "dh without the gate": (
        moe, "backward", "dh = g * D", "dh = D", ["fd"]),
    "dW_down without the gate": (
        moe, "backward", "P.bwd_act_rows(g * hv).T", "P.bwd_act_rows(hv).T", ["fd"]),
    "dX GEMM reads dv where du belongs": (
        moe, "backward", "(P.dx_act(du, 1) @ P.op(W_up[e], 1).T",
        "(P.dx_act(dv, 1) @ P.op(W_up[e], 1).T", ["fd"]),
    "reverse combine applies the gate again": (
        moe, "backward", "dX += dXg[pl.inv[:, j]]",
        "dX += gates[:, j:j + 1] * dXg[pl.inv[:, j]]", ["fd"]),
    "router path of dX with the wrong sign": (
        moe, "backward", "res.dX = res.dX + dxr", "res.dX = res.dX - dxr", ["fd"]),
    "router backward with the wrong sign": (
        moe, "router_backward", "dlS = gates * (dgates - s)", "dlS = gates * (s - dgates)",
        ["fd", "router_inv"]),
    "router backward drops the softmax's own term": (
        moe, "router_backward", "dlS = gates * (dgates - s)", "dlS = gates * dgates",
        ["router_inv", "fd"]),
    "router backward skips the softmax Jacobian": (
        moe, "router_backward", "(np.arange(T), idx[:, j]), dlS[:, j])",
        "(np.arange(T), idx[:, j]), dgates[:, j])", ["router_inv", "fd"]),
    "shared expert's dv without U": (
        moe, "shared_backward", "dv = D * Us * dsilu(Vs)", "dv = D * dsilu(Vs)",
        ["fd_shared"]),
    "empty experts keep stale weight gradients": (
        moe, "backward", "dW_up = np.zeros(W_up.shape)", "dW_up = np.ones(W_up.shape)",
        ["empty"]),
    # rounding points
    "U, V kept unrounded for the backward": (
        moe.Precision, "saved_uv", 'return a if self.mode == "fp64" else bf16_round(a)',
        "return a", ["saved_uv"]),
    "U, V rounded in fp64 mode too": (
        moe.Precision, "saved_uv", 'return a if self.mode == "fp64" else bf16_round(a)',
        "return bf16_round(a)", ["saved_uv"]),
    "the shared expert keeps U, V unrounded": (
        moe, "shared_forward", 'return O, {"Us": P.saved_uv(U), "Vs": P.saved_uv(V)}',
        'return O, {"Us": U, "Vs": V}', ["saved_uv"]),
    "the sampled evaluator's backward reads unrounded U, V": (
        sampled, "_row_terms", "U, V = bf16_round(U), bf16_round(V)   # as kept for the backward",
        "U, V = U, V", ["sampled"]),
    "bf16_plain weight-gradient operands unrounded": (
        moe.Precision, "bwd_act_rows", "return bf16_round(a)", "return a", ["wgrad_plain"]),
    "hi/lo weight-gradient operands rounded to bf16": (
        moe.Precision, "bwd_act_rows", "\n    return a\n", "\n    return bf16_round(a)\n",
        ["wgrad_hilo"]),
    # number formats
    "bf16 rounding truncates": (
        numerics, "bf16_round", "r = np.round(scaled)", "r = np.trunc(scaled)",
        ["bf16_torch"]),
    "E4M3 ties round up, not to even": (
        numerics, "e4m3_encode", "((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))",
        "(d_hi == d_lo)", ["e4m3_torch"]),
    "E4M3 drops the sign": (
        numerics, "e4m3_encode", "code = np.where(np.signbit(v), code | 0x80, code)",
        "code = np.where(np.signbit(v), code, code)", ["e4m3_sat", "e4m3_torch"]),
    "MX scale exponent off by one": (
        numerics, "mx_quantize", "e[pos] = _floor_log2(amax[pos]) - E4M3_EMAX",
        "e[pos] = _floor_log2(amax[pos]) - E4M3_EMAX + 1", ["mx_448", "mx_pow2"]),
    "MX zero block gets the smallest exponent": (
        numerics, "mx_quantize", "e = np.zeros(amax.shape, dtype=np.int64)",
        "e = np.full(amax.shape, -127, dtype=np.int64)", ["mx_zero"]),
    "MX blocks taken along the wrong axis": (
        numerics, "mx_quantize", "a_m = np.moveaxis(a, axis, -1)",
        "a_m = np.moveaxis(a, axis - 1, -1)", ["mx_axis", "mx_448"]),
    "ragged MX rows padded at the front": (
        numerics, "mx_qdq_rows_padded",
        "a = np.concatenate([a, np.zeros((pad,) + a.shape[1:])], axis=0)",
        "a = np.concatenate([np.zeros((pad,) + a.shape[1:]), a], axis=0)", ["mx_rows"]),
    "silu' misses a term": (
        numerics, "dsilu", "return s * (1.0 + v * (1.0 - s))", "return s * (1.0 + v * s)",
        ["silu", "fd"]),
    "silu is the sigmoid": (
        numerics, "silu", "return np.asarray(v, dtype=np.float64) * sigmoid(v)",
        "return sigmoid(v)", ["silu"]),
    # full-size evaluators
    "sampled router-weight gradient against U": (
        sampled, "_row_terms", 'res["dg"] = float(D @ hv)', 'res["dg"] = float(D @ U)',
        ["sampled"]),
    "sampled forward leaves h unrounded": (
        sampled, "_row_terms", "h = bf16_round(silu(V) * U)", "h = silu(V) * U", ["sampled"]),
    "MXFP8 token backward reads U unrounded": (
        sampled, "token_backward_mx", "U = bf16_round(xq @ Wu)", "U = xq @ Wu",
        ["mx_bwd_eval"]),
    "MXFP8 token backward leaves dv unquantised": (
        sampled, "token_backward_mx", "dv = mx_qdq((g * D * U * dsilu(V))[None, :], 1)[0]",
        "dv = g * D * U * dsilu(V)", ["mx_bwd_eval"]),
    "MXFP8 dW lines quantise x along H, not the rows": (
        sampled, "dw_lines_mx", "XR = mx_qdq_rows_padded(X)", "XR = Xq", ["mx_bwd_eval"]),
    # the rest of the oracle's functions
    "router ignores the logit bias": (
        moe, "route", "logits = logits + np.asarray(bias, np.float64)[None, :]",
        "logits = logits", ["route_brute"]),
    "MXFP8 operands left unquantised": (
        moe.Precision, "op", "return mx_qdq(a, axis) if self.mx else a", "return a",
        ["saved_uv", "down_mx"]),
    "MXFP8 row operands left unquantised": (
        moe.Precision, "op_rows", "return mx_qdq_rows_padded(a) if self.mx else a",
        "return a", ["mx_bwd_eval"]),
    "shared expert's h not rounded": (
        moe, "shared_forward", "h = P.fwd_act(silu(V) * U, 1)", "h = silu(V) * U",
        ["sampled"]),
    "shared expert always in the routed experts' precision": (
        moe, "shared_forward", 'P = Precision("fp64" if mode == "fp64" else "bf16")',
        "P = Precision(mode)", ["shared_lines_mx"]),
    "MX dequantisation with the wrong exponent bias": (
        numerics, "mx_dequantize", "s.astype(np.int64) - 127", "s.astype(np.int64) - 126",
        ["mx_axis"]),
    "sampled router path with the wrong sign": (
        sampled, "token_outputs", "dl = gates[t] * (dg - s)", "dl = gates[t] * (s - dg)",
        ["sampled"]),
    "sampled dW elements: dv without U": (
        sampled, "dw_elements", "d = rnd(g * D * U * dsilu(V))", "d = rnd(g * D * dsilu(V))",
        ["sampled"]),
    "sampled dW lines: plain mode not rounded": (
        sampled, "dw_lines", "rnd = bf16_round if plain else (lambda v: v)",
        "rnd = (lambda v: v)", ["dw_lines_plain"]),
    "sampled dW lines: dW_down without the gate": (
        sampled, "dw_lines", "hg = rnd(g * silu(V) * U)", "hg = rnd(silu(V) * U)",
        ["dw_lines_bf16"]),
    "MXFP8 token forward: h unquantised": (
        sampled, "token_forward_mx", "hq = mx_qdq((silu(V) * U)[None, :], 1)[0]",
        "hq = silu(V) * U", ["dw_lines_bf16"]),
    "shared dW lines: plain mode not rounded": (
        sampled, "shared_dw_lines", "rnd = bf16_round if plain else (lambda v: v)",
        "rnd = (lambda v: v)", ["shared_lines_plain"]),
    "dX GEMM operands left unrounded": (
        moe.Precision, "dx_act", "return self.fwd_act(a, axis)", "return a", ["dx_bf16"]),
    "floor(log2) one too high": (
        numerics, "_floor_log2", "return e - 1", "return e", ["mx_448", "mx_pow2"]),
    "sigmoid of -v": (
        numerics, "sigmoid", "1.0 / (1.0 + np.exp(-v))", "1.0 / (1.0 + np.exp(v))",
        ["silu"]),
    "qdq dequantises along the last axis": (
        numerics, "mx_qdq", "return mx_dequantize(c, s, axis)",
        "return mx_dequantize(c, s, -1)", ["mx_axis"]),
    "E4M3 decode off by one code": (
        numerics, "e4m3_decode", "_E4M3[np.asarray(codes, dtype=np.uint8)]",
        "_E4M3[np.asarray(codes, dtype=np.uint8) ^ 1]", ["mx_axis"]),
    "expert rows lose their last row": (
        sampled, "expert_rows", "plan.table[plan.offsets[e]:plan.offsets[e + 1]]",
        "plan.table[plan.offsets[e]:plan.offsets[e + 1] - 1]", ["sampled", "dw_lines_bf16"]),
    "MXFP8 forward weights: W_down along H": (
        sampled, "mx_expert_weights", "mx_qdq(Wd, 0)", "mx_qdq(Wd, 1)", ["dw_lines_bf16"]),
    "MXFP8 backward weights: W_down along I": (
        sampled, "mx_expert_weights_bwd", "mx_qdq(Wd, 1)", "mx_qdq(Wd, 0)", ["mx_bwd_eval"]),
    # bf16 results
    "bf16 results left unrounded": (
        moe, "out_round", 'return bf16_round if out == "bf16" else (lambda v: v)',
        "return (lambda v: v)", ["out_fwd", "out_bwd"]),
    "expert output rows not rounded before the combine": (
        moe, "forward", "O_rows[r0:r1] = rnd(h @ P.op(W_down[e], 0))",
        "O_rows[r0:r1] = h @ P.op(W_down[e], 0)", ["out_fwd"]),
    "y not rounded after the combine": (
        moe, "forward", "return rnd(y), saved", "return y, saved", ["out_fwd"]),
    "shared expert output not rounded": (
        moe, "shared_forward", "O = out_round(out)(h @ Ws_down)", "O = h @ Ws_down",
        ["out_fwd"]),
    "routed dX rows not rounded before the reverse combine": (
        moe, "backward", "dXg[r0:r1] = rnd(P.dx_act(du, 1)",
        "dXg[r0:r1] = (P.dx_act(du, 1)", ["out_bwd"]),
    "gradients not rounded after their sums": (
        moe, "backward", "setattr(res, n, rnd(getattr(res, n)))",
        "setattr(res, n, getattr(res, n))", ["out_bwd"]),
    "shared expert dX row not rounded": (
        moe, "shared_backward", "dXs = out_round(out)(", "dXs = (", ["out_bwd"]),
    "sampled y not rounded": (
        sampled, "token_outputs", 'res = {"y": rnd(y), "y_unrounded": y}',
        'res = {"y": y, "y_unrounded": y}', ["sampled_bf16"]),
    "sampled expert output rows not rounded": (
        sampled, "_row_terms", "O = rnd(h @ Wd)", "O = h @ Wd", ["sampled_bf16"]),
    "sampled dW lines not rounded": (
        sampled, "dw_lines", 'return {"dW_down": ro(hg @ dYe)', 'return {"dW_down": (hg @ dYe)',
        ["dw_lines_out"]),
    "sampled MXFP8 y: expert rows not rounded": (
        sampled, "token_forward_mx", "y += float(gates[t, j]) * rnd(hq @ Wd)",
        "y += float(gates[t, j]) * (hq @ Wd)", ["dw_lines_out"]),
    "sampled MXFP8 dX rows not rounded": (
        sampled, "token_backward_mx", "part = rnd(Wu_rows @ du + Wg_rows @ dv)",
        "part = (Wu_rows @ du + Wg_rows @ dv)", ["mx_bwd_eval_bf16"]),
    "sampled MXFP8 dW lines not rounded": (
        sampled, "dw_lines_mx", 'res[i] = {"dW_down": ro(hg @ dYR)',
        'res[i] = {"dW_down": (hg @ dYR)', ["mx_bwd_eval_bf16"]),
    "sampled shared dW lines not rounded": (
        sampled, "shared_dw_lines", '"dWs_up": ro(x.T @ rnd(D * silu(V)))',
        '"dWs_up": (x.T @ rnd(D * silu(V)))', ["shared_lines_out"]),
    # the pins' own references
    "brute-force token forward drops the gate": (
        moe, "token_forward_bruteforce", "y += g * ((silu(v) * u) @ W_down[e])",
        "y += (silu(v) * u) @ W_down[e]", ["fwd_brute"]),
    "finite-difference loss without renormalised gates": (
        moe, "layer_loss", "gates = pS / pS.sum(axis=1, keepdims=True)", "gates = pS",
        ["fd"]),
    "loop-built schedule in descending token order": (
        moe, "plan_loops", "rows[idx[t][j]].append((t, j))",
        "rows[idx[t][j]].insert(0, (t, j))", ["plan_loops"]),
}


def test_every_oracle_function_has_a_planted_mistake():
    """No function of the oracle is left out of the planted mistakes (the E4M3 table is
    computed once at import and pinned by its known values and round trip)."""
    planted = {(getattr(owner, "__name__", ""), fn) for owner, fn, *_ in MISTAKES.values()}
    missing = []
    for mod in (moe, numerics, sampled):
        for name, obj in vars(mod).items():
            if inspect.isfunction(obj) and obj.__module__ == mod.__name__:
                if (mod.__name__, name) not in planted and name != "e4m3_decode_table":
                    missing.append(f"{mod.__name__}.{name}")
            if inspect.isclass(obj) and obj.__module__ == mod.__name__:
                for mname, m in vars(obj).items():
                    if inspect.isfunction(m) and not mname.startswith("__") and \
                            (obj.__name__, mname) not in planted:
                        missing.append(f"{obj.__name__}.{mname}")
    assert not missing, missing


def test_pins_pass_on_the_oracle_as_it_is():
    for name, pin in P.items():
        assert not _fails(pin), name


@pytest.mark.parametrize("mistake", sorted(MISTAKES))
def test_planted_mistake_is_caught(monkeypatch, mistake):
    owner, fn, old, new, pins = MISTAKES[mistake]
    plant(monkeypatch, owner, fn, old, new)
    caught = [p for p in pins if _fails(P[p])]
    assert caught, f"no pin catches: {mistake}"
