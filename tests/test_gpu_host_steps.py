"""Pipelined steps from pinned host buffers (HostSteps) give, step by step, the
same outputs, dhidden, dprobs and main_grad accumulation as sequential
device-buffer calls on the same inputs -- bit for bit -- while the uploads and
downloads of neighbouring steps overlap the GPU work."""
import pytest
import torch

import mixture_experts_layer_pack_gb300 as M
from tests.harness import Case, make_inputs, weight_views

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    Case(T=300, H=256, E=8, k=2, I=128, seed=81, drop="iid"),
    Case(T=260, H=256, E=8, k=2, I=128, seed=82, gated=True, limit=0.5),
])
def test_host_steps_match_sequential_calls(case):
    inp = make_inputs(case)
    c = inp.case
    wv = weight_views(inp)
    steps = 4
    # per-step inputs: the seeded batch with sign flips and scales, so that no two steps agree
    hid = [inp.hidden * (1.0 if i % 2 == 0 else -1.0) * (1.0 + 0.25 * i) for i in range(steps)]
    gos = [inp.grad_out * (1.0 + 0.5 * i) for i in range(steps)]
    rmap = inp.routing_map.view(torch.uint8)

    def grads():
        mg = {n: t.clone() for n, t in inp.main_grads.items()}
        return mg, M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"],
                                              mg["routed_fc2"], mg.get("shared_output_gate"))

    # sequential calls on device buffers
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, swiglu_limit=c.limit)
    mg_s, mgv_s = grads()
    ref = []
    for i in range(steps):
        out = layer.forward(hid[i], inp.probs, rmap, wv)
        dh, dp = layer.backward(gos[i], mgv_s)
        ref.append((out.clone(), dh.clone(), dp.clone()))
    torch.cuda.synchronize()

    # the pipeline, from pinned host buffers
    layer2 = M.MoELayer(c.T, c.H, c.E, c.k, c.I, swiglu_limit=c.limit)
    mg_p, mgv_p = grads()
    pipe = layer2.host_steps(c.T)
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    h_in = [(pin(hid[i]), pin(inp.probs), pin(rmap), pin(gos[i])) for i in range(steps)]
    h_res = [tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in r) for r in ref]
    events = [pipe.step(*h_in[i][:3], h_in[i][3], wv, mgv_p, *h_res[i]) for i in range(steps)]
    events[-1].synchronize()
    pipe.synchronize()
    assert layer2.device_status() == 0
    for i in range(steps):
        for got, want, name in zip(h_res[i], ref[i], ("out", "dhidden", "dprobs")):
            assert torch.equal(got, want.cpu()), (i, name)
    for n in mg_s:
        assert torch.equal(mg_p[n], mg_s[n]), n
    layer.close()
    layer2.close()


def test_host_steps_reject_device_or_pageable_buffers():
    c = Case(T=64, H=128, E=4, k=2, I=64, seed=83)
    inp = make_inputs(c)
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I)
    pipe = layer.host_steps(c.T)
    wv = weight_views(inp)
    mgv = M.main_grads_from_combined(inp.main_grads["shared_fc1"], inp.main_grads["shared_fc2"],
                                     inp.main_grads["routed_fc1"], inp.main_grads["routed_fc2"])
    host = [inp.hidden.cpu(), inp.probs.cpu(), inp.routing_map.view(torch.uint8).cpu(), inp.grad_out.cpu()]
    res = [torch.empty((c.T, c.H), dtype=torch.bfloat16), torch.empty((c.T, c.H), dtype=torch.bfloat16),
           torch.empty((c.T, c.E), dtype=torch.float32)]
    with pytest.raises(ValueError):
        pipe.step(*host, wv, mgv, *res)                   # pageable
    with pytest.raises(ValueError):
        pipe.step(inp.hidden, *[t.pin_memory() for t in host[1:]], wv, mgv, *[t.pin_memory() for t in res])
    layer.close()
