"""Steps fed from host buffers through the C ABI's host pipeline
(moe_host_pipe_create / moe_host_step) give, step by step, the same outputs,
dhidden, dprobs and main_grad accumulation as sequential device-buffer calls on
the same inputs -- bit for bit -- while the uploads and downloads of
neighbouring steps overlap the GPU work; pageable host buffers give the same
results through the raw entry point; bad arguments are rejected."""
import ctypes

import pytest
import torch

import mixture_experts_layer_pack_gb300 as M
from mixture_experts_layer_pack_gb300 import binding as B
from tests.harness import Case, make_inputs, weight_views

pytestmark = pytest.mark.gpu


def _steps_inputs(inp, steps):
    # per-step inputs: the seeded batch with sign flips and scales, so that no two steps agree
    hid = [inp.hidden * (1.0 if i % 2 == 0 else -1.0) * (1.0 + 0.25 * i) for i in range(steps)]
    gos = [inp.grad_out * (1.0 + 0.5 * i) for i in range(steps)]
    return hid, gos


def _grads(inp):
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    return mg, M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"],
                                          mg["routed_fc2"], mg.get("shared_output_gate"))


def _sequential(inp, hid, gos, wv):
    c = inp.case
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, swiglu_limit=c.limit)
    mg, mgv = _grads(inp)
    rmap = inp.routing_map.view(torch.uint8)
    ref = []
    for i in range(len(hid)):
        out = layer.forward(hid[i], inp.probs, rmap, wv)
        dh, dp = layer.backward(gos[i], mgv)
        ref.append((out.clone(), dh.clone(), dp.clone()))
    torch.cuda.synchronize()
    layer.close()
    return ref, mg


@pytest.mark.parametrize("case", [
    Case(T=300, H=256, E=8, k=2, I=128, seed=81, drop="iid"),
    Case(T=260, H=256, E=8, k=2, I=128, seed=82, gated=True, limit=0.5),
])
def test_host_pipe_matches_sequential_calls(case):
    inp = make_inputs(case)
    c = inp.case
    wv = weight_views(inp)
    steps = 5
    hid, gos = _steps_inputs(inp, steps)
    ref, mg_s = _sequential(inp, hid, gos, wv)

    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, swiglu_limit=c.limit)
    mg_p, mgv_p = _grads(inp)
    pipe = layer.host_pipe(c.T)
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    rmap = inp.routing_map.view(torch.uint8)
    h_in = [(pin(hid[i]), pin(inp.probs), pin(rmap), pin(gos[i])) for i in range(steps)]
    h_res = [tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in r) for r in ref]
    for i in range(steps):
        pipe.step(*h_in[i], wv, mgv_p, *h_res[i])
    pipe.synchronize()
    assert layer.device_status() == 0
    for i in range(steps):
        for got, want, name in zip(h_res[i], ref[i], ("out", "dhidden", "dprobs")):
            assert torch.equal(got, want.cpu()), (i, name)
    torch.cuda.synchronize()
    for n in mg_s:
        assert torch.equal(mg_p[n], mg_s[n]), n
    pipe.close()
    layer.close()


def test_host_pipe_pageable_buffers_through_the_raw_entry():
    """Pageable host memory is legal in the C ABI (the call then waits for its
    step's downloads); results as with pinned memory."""
    case = Case(T=192, H=256, E=8, k=2, I=128, seed=84)
    inp = make_inputs(case)
    c = inp.case
    wv = weight_views(inp)
    hid, gos = _steps_inputs(inp, 2)
    ref, mg_s = _sequential(inp, hid, gos, wv)
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I)
    mg_p, mgv_p = _grads(inp)
    mem = torch.empty(M.moe_host_pipe_size(layer.cfg, c.T), dtype=torch.uint8, device="cuda")
    p = M.moe_host_pipe_create(layer.handle, c.T, mem)
    rmap = inp.routing_map.view(torch.uint8).cpu()
    probs = inp.probs.cpu()
    res = [tuple(torch.empty(t.shape, dtype=t.dtype) for t in r) for r in ref]
    stream = torch.cuda.Stream()
    for i in range(2):
        M.moe_host_step(p, hid[i].cpu(), probs, rmap, gos[i].cpu(), wv, mgv_p, *res[i], stream=stream)
    M.moe_host_pipe_sync(p)
    for i in range(2):
        for got, want, name in zip(res[i], ref[i], ("out", "dhidden", "dprobs")):
            assert torch.equal(got, want.cpu()), (i, name)
    torch.cuda.synchronize()
    for n in mg_s:
        assert torch.equal(mg_p[n], mg_s[n]), n
    M.moe_host_pipe_destroy(p)
    layer.close()


def test_host_pipe_rejects_bad_arguments():
    c = Case(T=64, H=128, E=4, k=2, I=64, seed=83)
    inp = make_inputs(c)
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I)
    L = M.load()
    need = M.moe_host_pipe_size(layer.cfg, c.T)
    mem = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p()
    # too little memory, misaligned memory, T out of range
    assert L.moe_host_pipe_create(layer.handle, c.T, mem.data_ptr(), need - 1, ctypes.byref(p)) == 1
    assert L.moe_host_pipe_create(layer.handle, c.T, mem.data_ptr() + 16, need, ctypes.byref(p)) == 1
    assert L.moe_host_pipe_create(layer.handle, c.T + 1, mem.data_ptr(), need + 512, ctypes.byref(p)) == 1
    cfg = M.moe_handle_config(layer.handle)
    assert (cfg.max_tokens, cfg.hidden, cfg.num_experts, cfg.topk, cfg.inter) == (c.T, c.H, c.E, c.k, c.I)
    pipe = layer.host_pipe(c.T)
    wv = weight_views(inp)
    mgv = M.main_grads_from_combined(inp.main_grads["shared_fc1"], inp.main_grads["shared_fc2"],
                                     inp.main_grads["routed_fc1"], inp.main_grads["routed_fc2"])
    host = [inp.hidden.cpu(), inp.probs.cpu(), inp.routing_map.view(torch.uint8).cpu(), inp.grad_out.cpu()]
    res = [torch.empty((c.T, c.H), dtype=torch.bfloat16), torch.empty((c.T, c.H), dtype=torch.bfloat16),
           torch.empty((c.T, c.E), dtype=torch.float32)]
    with pytest.raises(ValueError):
        pipe.step(*host, wv, mgv, *res)                   # pageable: the class wants pinned memory
    with pytest.raises(ValueError):
        pipe.step(inp.hidden, *[t.pin_memory() for t in host[1:]], wv, mgv, *[t.pin_memory() for t in res])
    with pytest.raises(B.MoeError):                       # a null host pointer
        M.moe_host_step(pipe.pipe, None, *host[1:], wv, mgv, *res)
    pipe.close()
    layer.close()


def test_host_pipe_usable_after_a_rejected_step():
    """A step whose backward is rejected (a null main_grad pointer) returns the
    error after its uploads and forward were enqueued; the pipeline drains it, and
    the next steps give the results of sequential calls."""
    case = Case(T=160, H=256, E=8, k=2, I=128, seed=85)
    inp = make_inputs(case)
    c = inp.case
    wv = weight_views(inp)
    hid, gos = _steps_inputs(inp, 2)
    ref, mg_s = _sequential(inp, hid, gos, wv)
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I)
    mg_p, mgv_p = _grads(inp)
    pipe = layer.host_pipe(c.T)
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    rmap = pin(inp.routing_map.view(torch.uint8))
    probs = pin(inp.probs)
    bad = M.main_grads_from_combined(mg_p["shared_fc1"], mg_p["shared_fc2"], mg_p["routed_fc1"], mg_p["routed_fc2"])
    bad.routed_down = None
    junk = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ref[0]]
    with pytest.raises(B.MoeError):
        pipe.step(pin(hid[0]), probs, rmap, pin(gos[0]), wv, bad, *junk)
    res = [tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in r) for r in ref]
    for i in range(2):
        pipe.step(pin(hid[i]), probs, rmap, pin(gos[i]), wv, mgv_p, *res[i])
    pipe.synchronize()
    assert layer.device_status() == 0
    for i in range(2):
        for got, want, name in zip(res[i], ref[i], ("out", "dhidden", "dprobs")):
            assert torch.equal(got, want.cpu()), (i, name)
    torch.cuda.synchronize()
    for n in mg_s:
        assert torch.equal(mg_p[n], mg_s[n]), n
    pipe.close()
    layer.close()
