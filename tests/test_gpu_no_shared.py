"""Routed experts only (moe_config.no_shared_expert = 1), and the owner-side step
of expert parallelism built on it.

* A layer without the shared expert against the oracle with zero shared
  weights: the GPU is handed NaN shared weights, which it must not read, and
  shared main_grad buffers, which it must leave untouched. (The bf16-activation
  case has no clamp: its masks follow bf16-rounded SwiGLU inputs, and without
  the shared expert's share of dhidden the exact-definition bound compares the
  flipped masks with the routed part alone.)
* The expert-parallel owner step on one GPU: the experts are split over two
  owners; each owner runs its own experts, through moe_forward_topk and
  moe_backward on a top-1, no-shared-expert handle, on the token rows routed to
  them in (expert, token) order -- the rows an all-to-all would deliver (the
  exchange itself is tested on CPU ranks in test_expert_parallel.py). The token
  side adds the returned rows to the shared expert's output and gradient; out,
  dhidden, dprobs and every routed main_grad must match the single-GPU oracle.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_pack_gb300 as M
from oracle import moe_oracle as O
from tests.harness import (BF16_TOL, Case, assert_close, compare_layer, f64, make_inputs, oracle_full,
                           oracle_weights)

pytestmark = pytest.mark.gpu


def _nan_shared(inp):
    w = inp.weights
    return torch.full_like(w["shared_fc1"], float("nan")), torch.full_like(w["shared_fc2"], float("nan"))


@pytest.mark.parametrize("case", [
    Case(T=300, H=256, E=8, k=2, I=128, seed=91, drop="iid"),
    Case(T=260, H=256, E=8, k=2, I=128, seed=92, limit=0.5),
    Case(T=244, H=256, E=8, k=2, I=128, seed=97, act_bf16=True),
    Case(T=272, H=256, E=8, k=2, I=128, seed=93, mx=True),
])
def test_routed_only_layer_matches_oracle_without_shared_expert(case):
    from tests.harness import GpuResult, weight_views
    inp = make_inputs(case)
    c = inp.case
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, routed_wtype=M.binding.MOE_W_MXFP8 if c.mx else M.binding.MOE_W_BF16,
                       swiglu_limit=c.limit,
                       act_precision=M.binding.MOE_ACT_BF16 if c.act_bf16 else M.binding.MOE_ACT_FP32,
                       shared_expert=False)
    wv = weight_views(inp)
    nan1, nan2 = _nan_shared(inp)
    wv_nan = M.weights_from_combined(nan1, nan2, inp.weights["routed_fc1"], inp.weights["routed_fc2"])
    wv.shared_gate, wv.shared_up, wv.shared_down = wv_nan.shared_gate, wv_nan.shared_up, wv_nan.shared_down
    if c.mx:
        layer.prepare_weights(wv)
    out = layer.forward(inp.hidden, inp.probs, inp.routing_map.view(torch.uint8), wv)
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"])
    dh, dp = layer.backward(inp.grad_out, mgv)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    for n in ("shared_fc1", "shared_fc2"):                 # ignored buffers stay bitwise
        assert torch.equal(mg[n], inp.main_grads[n]), n
    res = GpuResult(out, dh, dp, mg, layer)
    # the oracle without a shared expert: zero shared weights (zero output, zero gradients)
    inp.weights["shared_fc1"] = torch.zeros_like(inp.weights["shared_fc1"])
    inp.weights["shared_fc2"] = torch.zeros_like(inp.weights["shared_fc2"])
    compare_layer(inp, res, mx_exact_bound=False)
    layer.close()


def test_rejects_an_output_gate_without_shared_expert():
    c = Case(T=64, H=128, E=4, k=2, I=64, seed=94, gated=True)
    inp = make_inputs(c)
    from tests.harness import weight_views
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, shared_expert=False)
    with pytest.raises(M.MoeError) as ei:
        layer.forward(inp.hidden, inp.probs, inp.routing_map.view(torch.uint8), weight_views(inp))
    assert ei.value.status == 1
    layer.close()


@pytest.mark.parametrize("case", [
    Case(T=320, H=256, E=8, k=2, I=128, seed=95),
    Case(T=288, H=256, E=7, k=3, I=128, seed=96, drop="iid"),
])
def test_expert_parallel_owner_step(case):
    inp = make_inputs(case)
    c = inp.case
    W = oracle_weights(inp)
    ref_out, ref_dx, ref_dp, ref_grads, _ = oracle_full(inp, "exact")
    ids, pp, over = O.route_pack(inp.map_np, inp.probs_np, c.k)
    assert not over.any()
    hidden, go = inp.hidden, inp.grad_out
    # the token side keeps the shared expert (here: the oracle's, in fp64)
    xs = f64(hidden)
    g_s, u_s, a_s, y_s = O.expert_forward(xs, *W.shared())
    dx_s = O.expert_backward(xs, f64(go), np.ones(c.T), g_s, u_s, a_s, *W.shared())[0]
    out = y_s.copy()
    dhidden = dx_s.copy()
    dprobs = np.zeros((c.T, c.E))
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    I = c.I
    first = [0, (c.E + 1) // 2, c.E]                       # owner r holds experts [first[r], first[r+1])
    for r in range(2):
        e0, e1 = first[r], first[r + 1]
        sel = [(e, t, s) for t in range(c.T) for s in range(c.k) if e0 <= ids[t, s] < e1
               for e in [int(ids[t, s])]]
        sel.sort()                                          # expert order, tokens ascending within an expert
        n = len(sel)
        if n == 0:
            continue
        tok = torch.tensor([t for _, t, _ in sel], device=hidden.device)
        rows = hidden[tok].contiguous()
        go_rows = go[tok].contiguous()
        lid = torch.tensor([[e - e0] for e, _, _ in sel], dtype=torch.int32, device=hidden.device)
        lp = torch.tensor([[pp[t, s]] for _, t, s in sel], dtype=torch.float32, device=hidden.device)
        owner = M.MoELayer(n, c.H, e1 - e0, 1, I, shared_expert=False)
        rf1, rf2 = inp.weights["routed_fc1"][e0:e1], inp.weights["routed_fc2"][e0:e1]
        wv = M.weights_from_combined(None, None, rf1, rf2)
        y_rows = owner.forward_topk(rows, lid, lp, wv)
        mgv = M.main_grads_from_combined(None, None, mg["routed_fc1"][e0:e1], mg["routed_fc2"][e0:e1])
        dx_rows, dp_rows = owner.backward(go_rows, mgv)
        torch.cuda.synchronize()
        assert owner.device_status() == 0
        assert dp_rows.shape == (n, 1)
        y_rows, dx_rows, dp_rows = f64(y_rows), f64(dx_rows), f64(dp_rows)
        for j, (e, t, s) in enumerate(sel):               # the token side adds the returned rows
            out[t] += y_rows[j]
            dhidden[t] += dx_rows[j]
            dprobs[t, e] = dp_rows[j, 0]
        owner.close()
    assert_close(out, ref_out, "out", **BF16_TOL)
    assert_close(dhidden, ref_dx, "dhidden", **BF16_TOL)
    assert_close(dprobs, ref_dp, "dprobs", **BF16_TOL)
    used = sorted(ref_grads["routed"])
    d1 = f64(mg["routed_fc1"]) - f64(inp.main_grads["routed_fc1"])
    d2 = f64(mg["routed_fc2"]) - f64(inp.main_grads["routed_fc2"])
    for j, (name, got) in enumerate((("gate", d1[:, :I]), ("up", d1[:, I:]), ("down", d2))):
        assert_close(np.stack([got[e] for e in used]), np.stack([ref_grads["routed"][e][j] for e in used]),
                     f"dW routed {name}", **BF16_TOL)
    for e in set(range(c.E)) - set(used):                 # experts without tokens: untouched
        assert torch.equal(mg["routed_fc1"][e], inp.main_grads["routed_fc1"][e])
