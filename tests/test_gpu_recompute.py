"""recompute_dispatch: a saved state keeps only the routing, and the backward
re-runs the row placement, the shared output gate and the gate/up GEMMs.

Results are bitwise those of the default mode, also with two microbatches in
flight on one handle (forward 1, forward 2, backward 2, backward 1), and the
saved state is a small fraction of the default one. The routed-only layer
(no shared expert, the owner step of expert parallelism) takes the same path."""
import pytest
import torch

import mixture_experts_layer_pack_gb300 as M
from tests.harness import Case, make_inputs, weight_views

pytestmark = pytest.mark.gpu

CASES = {   # (case, shared expert)
    "bf16_gated_clamp": (Case(T=300, H=256, E=8, k=2, I=128, seed=101, drop="iid", gated=True, limit=0.5), True),
    "mxfp8": (Case(T=260, H=256, E=6, k=2, I=128, seed=102, mx=True), True),
    "routed_only": (Case(T=280, H=256, E=8, k=2, I=128, seed=103, limit=0.5), False),
    "routed_only_mxfp8": (Case(T=250, H=256, E=6, k=2, I=128, seed=104, mx=True), False),
}


def _layer(c, recompute, shared=True):
    return M.MoELayer(c.T, c.H, c.E, c.k, c.I, routed_wtype=M.binding.MOE_W_MXFP8 if c.mx else M.binding.MOE_W_BF16,
                      swiglu_limit=c.limit, recompute_dispatch=recompute, shared_expert=shared)


def _grads(inp):
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    return mg, M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"],
                                          mg.get("shared_output_gate"))


@pytest.mark.parametrize("name", list(CASES))
def test_recompute_matches_saved_activations_bitwise(name):
    case, shared = CASES[name]
    inp = make_inputs(case)
    c = inp.case
    wv = weight_views(inp)
    rmap = inp.routing_map.view(torch.uint8)
    # two microbatches: the seeded batch and a rescaled, sign-flipped copy
    batches = [(inp.hidden, inp.grad_out), (inp.hidden * -1.5, inp.grad_out * 0.5)]

    ref = []                                   # default mode, one microbatch at a time
    A = _layer(c, False, shared)
    if c.mx:
        A.prepare_weights(wv)
    for hid, go in batches:
        mg, mgv = _grads(inp)
        out = A.forward(hid, inp.probs, rmap, wv)
        dh, dp = A.backward(go, mgv)
        ref.append((out.clone(), dh.clone(), dp.clone(), mg))
    torch.cuda.synchronize()
    assert A.device_status() == 0

    B = _layer(c, True, shared)                # recompute mode, both microbatches in flight
    if c.mx:
        B.prepare_weights(wv)
    assert M.moe_saved_size(B.cfg) * 4 < M.moe_saved_size(A.cfg)
    mem2 = torch.empty(M.moe_saved_size(B.cfg), dtype=torch.uint8, device=inp.hidden.device)
    saved = [B.saved, M.moe_saved_create(B.handle, mem2)]
    outs = [torch.empty_like(inp.hidden) for _ in batches]
    for i, (hid, _) in enumerate(batches):
        M.moe_forward(B.handle, c.T, hid, inp.probs, rmap, wv, outs[i], saved[i])
    got = [None, None]
    for i in (1, 0):
        mg, mgv = _grads(inp)
        dh = torch.empty_like(inp.hidden)
        dp = torch.empty((c.T, c.E), dtype=torch.float32, device=inp.hidden.device)
        M.moe_backward(B.handle, batches[i][1], saved[i], dh, dp, mgv)
        got[i] = (outs[i], dh, dp, mg)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    for i in range(2):
        for name_, x, y in zip(("out", "dhidden", "dprobs"), got[i][:3], ref[i][:3]):
            assert torch.equal(x, y), (i, name_)
        for n in ref[i][3]:
            assert torch.equal(got[i][3][n], ref[i][3][n]), (i, n)
    M.moe_saved_destroy(saved[1])
    A.close()
    B.close()


def test_recompute_with_other_token_counts_and_topk_input():
    """Microbatches of different sizes (the shared rows' region moves with T) and
    the top-k input, in recompute mode: bitwise the default mode."""
    from oracle import moe_oracle as O
    import numpy as np
    c = Case(T=300, H=256, E=8, k=3, I=128, seed=103, drop="iid", gated=True)
    inp = make_inputs(c)
    wv = weight_views(inp)
    ids, pp, _ = O.route_pack(inp.map_np, inp.probs_np, c.k)
    dev = inp.hidden.device
    ids_d = torch.from_numpy(ids.astype(np.int32)).to(dev)
    pp_d = torch.from_numpy(pp.astype(np.float32)).to(dev)
    sizes = [300, 130]                         # R0 = 384 and 256

    def run(layer, order):
        saved = [layer.saved]
        mems = []
        for _ in sizes[1:]:
            mems.append(torch.empty(M.moe_saved_size(layer.cfg), dtype=torch.uint8, device=dev))
            saved.append(M.moe_saved_create(layer.handle, mems[-1]))
        outs = [torch.empty_like(inp.hidden[:T]) for T in sizes]
        res = [None] * len(sizes)
        for i, T in enumerate(sizes):
            M.moe_forward_topk(layer.handle, T, inp.hidden[:T], ids_d[:T], pp_d[:T], wv, outs[i], saved[i])
            if order == "each":
                res[i] = _bwd(layer, saved[i], T, outs[i])
        if order == "reverse":
            for i in reversed(range(len(sizes))):
                res[i] = _bwd(layer, saved[i], sizes[i], outs[i])
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        for s_ in saved[1:]:
            M.moe_saved_destroy(s_)
        return res

    def _bwd(layer, sv, T, out):
        mg, mgv = _grads(inp)
        dh = torch.empty_like(inp.hidden[:T])
        dp = torch.empty((T, c.k), dtype=torch.float32, device=dev)
        M.moe_backward(layer.handle, inp.grad_out[:T], sv, dh, dp, mgv)
        return out, dh, dp, mg

    A = _layer(c, False)
    ref = run(A, "each")
    B = _layer(c, True)
    got = run(B, "reverse")
    for i in range(len(sizes)):
        for x, y in zip(got[i][:3], ref[i][:3]):
            assert torch.equal(x, y), i
        for n in ref[i][3]:
            assert torch.equal(got[i][3][n], ref[i][3][n]), (i, n)
    A.close()
    B.close()


def test_recompute_config2_full_size_bitwise():
    """Proxy-like layer (T=4096, H=2048, E=96, top-6, I=1024): recompute mode equals the
    default mode bit for bit, with a saved state a small fraction of the default one."""
    from tests.harness import config_case
    inp = make_inputs(config_case(2))
    c = inp.case
    wv = weight_views(inp)
    rmap = inp.routing_map.view(torch.uint8)
    res = []
    for recompute in (False, True):
        layer = _layer(c, recompute)
        mg, mgv = _grads(inp)
        out = layer.forward(inp.hidden, inp.probs, rmap, wv)
        dh, dp = layer.backward(inp.grad_out, mgv)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        res.append((out, dh, dp, mg, M.moe_saved_size(layer.cfg)))
        layer.close()
    (o0, h0, p0, m0, s0), (o1, h1, p1, m1, s1) = res
    assert s1 * 20 < s0
    assert torch.equal(o0, o1) and torch.equal(h0, h1) and torch.equal(p0, p1)
    for n in m0:
        assert torch.equal(m0[n], m1[n]), n


def test_default_mode_saved_states_interleave():
    """Default mode: two saved states of one handle, forward 1, forward 2, backward 2,
    backward 1, bitwise the sequential order (the workspace is scratch within a call)."""
    inp = make_inputs(Case(T=300, H=256, E=8, k=2, I=128, seed=104, drop="iid", gated=True))
    c = inp.case
    wv = weight_views(inp)
    rmap = inp.routing_map.view(torch.uint8)
    batches = [(inp.hidden, inp.grad_out), (inp.hidden * 0.75, inp.grad_out * -2.0)]
    A = _layer(c, False)
    ref = []
    for hid, go in batches:
        mg, mgv = _grads(inp)
        out = A.forward(hid, inp.probs, rmap, wv)
        dh, dp = A.backward(go, mgv)
        ref.append((out.clone(), dh.clone(), dp.clone(), mg))
    mem2 = torch.empty(M.moe_saved_size(A.cfg), dtype=torch.uint8, device=inp.hidden.device)
    saved = [A.saved, M.moe_saved_create(A.handle, mem2)]
    outs = [torch.empty_like(inp.hidden) for _ in batches]
    for i, (hid, _) in enumerate(batches):
        M.moe_forward(A.handle, c.T, hid, inp.probs, rmap, wv, outs[i], saved[i])
    for i in (1, 0):
        mg, mgv = _grads(inp)
        dh = torch.empty_like(inp.hidden)
        dp = torch.empty((c.T, c.E), dtype=torch.float32, device=inp.hidden.device)
        M.moe_backward(A.handle, batches[i][1], saved[i], dh, dp, mgv)
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref[i][0]) and torch.equal(dh, ref[i][1]) and torch.equal(dp, ref[i][2]), i
        for n in mg:
            assert torch.equal(mg[n], ref[i][3][n]), (i, n)
    assert A.device_status() == 0
    M.moe_saved_destroy(saved[1])
    A.close()
