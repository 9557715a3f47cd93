"""Per-expert descriptor tables (routed BF16 or MXFP8 weights and routed main_grads held
expert by expert in separate allocations, PR #6572 Design > MCore-owned
parameters and > Gradient accumulation: per-expert non-single storage), through
the C ABI.

The same kernels run with each expert's own TMA descriptor instead of one 3D
map, so every result must be bitwise identical to the strided single-tensor
run on the same values: out, dhidden, dprobs and every main_grad element.
Repeated calls reuse the uploaded descriptors; new pointers (the same values
copied elsewhere) re-encode them, again with identical results.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_pack_gb300 as M
from tests.harness import Case, config_case, make_inputs, weight_views

pytestmark = pytest.mark.gpu


def _run(inp, layer, wv, mgv):
    out = layer.forward(inp.hidden, inp.probs, inp.routing_map.view(torch.uint8), wv)
    dh, dp = layer.backward(inp.grad_out, mgv)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    return out.clone(), dh.clone(), dp.clone()


def _split_experts(t3, lo=None, hi=None):
    """Separate contiguous copies of t3[e, lo:hi] for every expert e."""
    return [t3[e, lo:hi].clone() for e in range(t3.shape[0])]


def _tables_match_strided(case, gate=True, up=True, down=True, mg_tables=True):
    inp = make_inputs(case)
    c = inp.case
    I = c.I
    w, mg = inp.weights, inp.main_grads
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, swiglu_limit=c.limit)

    # strided reference run
    mg_a = {n: t.clone() for n, t in mg.items()}
    ref = _run(inp, layer, weight_views(inp), M.main_grads_from_combined(
        mg_a["shared_fc1"], mg_a["shared_fc2"], mg_a["routed_fc1"], mg_a["routed_fc2"]))

    # per-expert storage holding the same values
    g_list, u_list = _split_experts(w["routed_fc1"], 0, I), _split_experts(w["routed_fc1"], I, 2 * I)
    d_list = _split_experts(w["routed_fc2"])
    mg_b = {n: t.clone() for n, t in mg.items()}
    mg_g, mg_u = _split_experts(mg_b["routed_fc1"], 0, I), _split_experts(mg_b["routed_fc1"], I, 2 * I)
    mg_d = _split_experts(mg_b["routed_fc2"])
    wv = weight_views(inp)
    M.set_expert_tables(wv, gate=g_list if gate else None, up=u_list if up else None,
                        down=d_list if down else None)
    mgv = M.main_grads_from_combined(mg_b["shared_fc1"], mg_b["shared_fc2"], mg_b["routed_fc1"], mg_b["routed_fc2"])
    if mg_tables:
        M.set_main_grad_tables(mgv, gate=mg_g, up=mg_u, down=mg_d)
    got = _run(inp, layer, wv, mgv)
    for a, b, n in zip(got, ref, ("out", "dhidden", "dprobs")):
        assert torch.equal(a, b), n
    if mg_tables:
        for e in range(c.E):
            assert torch.equal(mg_g[e], mg_a["routed_fc1"][e, :I]), e
            assert torch.equal(mg_u[e], mg_a["routed_fc1"][e, I:]), e
            assert torch.equal(mg_d[e], mg_a["routed_fc2"][e]), e
    else:
        assert torch.equal(mg_b["routed_fc1"], mg_a["routed_fc1"]) and torch.equal(mg_b["routed_fc2"], mg_a["routed_fc2"])
    for n in ("shared_fc1", "shared_fc2"):
        assert torch.equal(mg_b[n], mg_a[n]), n
    return inp, layer, wv, mgv, (g_list, u_list, d_list), ref


@pytest.mark.parametrize("name,case", [
    ("ragged", Case(T=300, H=256, E=8, k=2, I=128, seed=61, drop="iid")),
    ("bn64_skewed_clamped", Case(T=517, H=384, E=12, k=3, I=192, seed=62, routing="zipf", drop="multi", limit=0.3)),
])
def test_expert_tables_bitwise_equal_to_strided(name, case):
    _tables_match_strided(case)


def test_expert_tables_partial_and_weights_only():
    _tables_match_strided(Case(T=300, H=256, E=8, k=2, I=128, seed=63), gate=True, up=False, down=True,
                          mg_tables=False)


def test_expert_tables_reuse_and_refresh():
    case = Case(T=300, H=256, E=8, k=2, I=128, seed=64, drop="iid")
    inp, layer, wv, _, lists, ref = _tables_match_strided(case, mg_tables=False)
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"])
    again = _run(inp, layer, wv, mgv)                       # cached descriptors
    for a, b in zip(again, ref):
        assert torch.equal(a, b)
    moved = [[t.clone() for t in lst] for lst in lists]     # same values, new addresses
    wv2 = weight_views(inp)
    M.set_expert_tables(wv2, gate=moved[0], up=moved[1], down=moved[2])
    del lists
    torch.cuda.synchronize()
    third = _run(inp, layer, wv2, mgv)
    for a, b in zip(third, ref):
        assert torch.equal(a, b)


def test_expert_tables_config2_full():
    _tables_match_strided(config_case(2))


@pytest.mark.parametrize("name,case", [
    ("mx_ragged", Case(T=300, H=256, E=6, k=2, I=128, seed=65, drop="iid", mx=True)),
    ("mx_skewed_gated", Case(T=517, H=384, E=12, k=3, I=256, seed=66, routing="zipf", drop="multi", mx=True,
                             gated=True)),
])
def test_mxfp8_expert_tables_bitwise_equal_to_strided(name, case):
    """MXFP8 routed weights expert by expert (payloads, columnwise payloads and both
    scale arrays in separate allocations): the scale swizzle and the block-scaled
    GEMMs read them through per-expert pointers and descriptors, bit for bit the
    strided run."""
    inp = make_inputs(case)
    c = inp.case
    I = c.I
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, routed_wtype=M.binding.MOE_W_MXFP8)
    wv = weight_views(inp)
    layer.prepare_weights(wv)
    mg_a = {n: t.clone() for n, t in inp.main_grads.items()}
    ref = _run(inp, layer, wv, M.main_grads_from_combined(mg_a["shared_fc1"], mg_a["shared_fc2"],
                                                           mg_a["routed_fc1"], mg_a["routed_fc2"],
                                                           mg_a.get("shared_output_gate")))
    q1, s1, c1, cs1 = inp.mx["routed_fc1"]
    q2, s2, c2, cs2 = inp.mx["routed_fc2"]
    E = c.E
    gate = ([q1[e, :I].clone() for e in range(E)], [c1[e, :I].clone() for e in range(E)],
            [s1[e, :I].clone() for e in range(E)], [cs1[e, :I // 32].clone() for e in range(E)])
    up = ([q1[e, I:].clone() for e in range(E)], [c1[e, I:].clone() for e in range(E)],
          [s1[e, I:].clone() for e in range(E)], [cs1[e, I // 32:].clone() for e in range(E)])
    down = ([q2[e].clone() for e in range(E)], [c2[e].clone() for e in range(E)],
            [s2[e].clone() for e in range(E)], [cs2[e].clone() for e in range(E)])
    layer2 = M.MoELayer(c.T, c.H, c.E, c.k, c.I, routed_wtype=M.binding.MOE_W_MXFP8)
    wv2 = weight_views(inp)
    M.set_mx_expert_tables(wv2, gate=gate, up=up, down=down)
    layer2.prepare_weights(wv2)
    mg_b = {n: t.clone() for n, t in inp.main_grads.items()}
    got = _run(inp, layer2, wv2, M.main_grads_from_combined(mg_b["shared_fc1"], mg_b["shared_fc2"],
                                                            mg_b["routed_fc1"], mg_b["routed_fc2"],
                                                            mg_b.get("shared_output_gate")))
    for a, b, n in zip(got, ref, ("out", "dhidden", "dprobs")):
        assert torch.equal(a, b), n
    for n in mg_a:
        assert torch.equal(mg_b[n], mg_a[n]), n
