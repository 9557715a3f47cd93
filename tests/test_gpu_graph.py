"""The layer's forward and backward capture into one CUDA graph (no host
synchronisation, no allocation, device-side tile counts) and replay bitwise
identically to eager calls on the same inputs -- routing, outputs, dprobs and
main_grad accumulation -- including a replay after new input values are
copied into the captured buffers."""
import pytest
import torch

import mixture_experts_layer_pack_gb300 as M
from tests.harness import Case, make_inputs, weight_views

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    Case(T=300, H=256, E=8, k=2, I=128, seed=71, drop="iid"),
    Case(T=300, H=256, E=8, k=2, I=128, seed=72, mx=True, gated=True, limit=0.5),
])
def test_graph_replay_matches_eager(case):
    inp = make_inputs(case)
    c = inp.case
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, routed_wtype=M.binding.MOE_W_MXFP8 if c.mx else M.binding.MOE_W_BF16,
                       swiglu_limit=c.limit)
    wv = weight_views(inp)
    if c.mx:
        layer.prepare_weights(wv)
    rmap = inp.routing_map.view(torch.uint8)
    out = torch.empty_like(inp.hidden)
    dh = torch.empty_like(inp.hidden)
    dp = torch.empty((c.T, c.E), dtype=torch.float32, device=inp.hidden.device)

    def grads():
        mg = {n: t.clone() for n, t in inp.main_grads.items()}
        mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"],
                                         mg.get("shared_output_gate"))
        return mg, mgv

    def step(stream, mgv):
        M.moe_forward(layer.handle, c.T, inp.hidden, inp.probs, rmap, wv, out, layer.saved, stream)
        M.moe_backward(layer.handle, inp.grad_out, layer.saved, dh, dp, mgv, stream)

    # eager reference
    mg_e, mgv_e = grads()
    step(torch.cuda.current_stream(), mgv_e)
    torch.cuda.synchronize()
    ref = (out.clone(), dh.clone(), dp.clone(), {n: t.clone() for n, t in mg_e.items()})

    # capture, replay once from the same main_grad start
    mg_g, mgv_g = grads()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        step(cap, mgv_g)
    torch.cuda.synchronize()
    for n in mg_g:                                  # capture ran nothing: restart the accumulation
        mg_g[n].copy_(inp.main_grads[n])
    g.replay()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert torch.equal(out, ref[0]) and torch.equal(dh, ref[1]) and torch.equal(dp, ref[2])
    for n in mg_g:
        assert torch.equal(mg_g[n], ref[3][n]), n

    # new input values in the captured buffers: the replay follows them
    inp.hidden.mul_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    mg_e2, mgv_e2 = grads()
    for n in mg_e2:
        mg_e2[n].copy_(mg_g[n])
    assert not torch.equal(out, ref[0])
    out_g, dh_g, dp_g = out.clone(), dh.clone(), dp.clone()
    for n in mg_e2:                                 # eager on the same state as before the second replay
        mg_e2[n].copy_(ref[3][n])
    step(torch.cuda.current_stream(), mgv_e2)
    torch.cuda.synchronize()
    assert torch.equal(out, out_g) and torch.equal(dh, dh_g) and torch.equal(dp, dp_g)
    for n in mg_g:
        assert torch.equal(mg_g[n], mg_e2[n]), n
