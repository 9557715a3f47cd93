"""The forward fed by the router's top-k output (moe_forward_topk).

* Slots in ascending id order: bit for bit the dense-map path (outputs, dhidden,
  main_grad accumulation, routing), and dprobs per slot = the dense dprobs at
  the slot's expert.
* Slots in any order (empty slots anywhere): parity with the fp64 oracle on the
  equivalent dense map, dprobs per slot in the caller's order.
* Rows with an out-of-range or repeated id: reported as a routing error and
  dropped, like a map row with more than k routes.
"""
import dataclasses

import numpy as np
import pytest
import torch

import mixture_experts_layer_pack_gb300 as M
from moe_inputs import make_routing
from oracle import moe_oracle as O
from tests.harness import Case, GpuResult, make_inputs, run_gpu, weight_views
from tests.test_gpu_layer import _compare_full

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": Case(T=300, H=256, E=8, k=2, I=128, seed=91, drop="iid"),
    "skewed_gated": Case(T=517, H=384, E=12, k=3, I=192, seed=92, routing="zipf", drop="multi", gated=True),
    "mxfp8": Case(T=300, H=256, E=8, k=2, I=128, seed=95, drop="iid", mx=True),
}


def _run_topk(inp, ids, pp):
    c = inp.case
    dev = inp.hidden.device
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, device=dev, swiglu_limit=c.limit,
                       routed_wtype=M.binding.MOE_W_MXFP8 if c.mx else M.binding.MOE_W_BF16)
    wv = weight_views(inp)
    if c.mx:
        layer.prepare_weights(wv)
    out = layer.forward_topk(inp.hidden, torch.from_numpy(ids).to(dev), torch.from_numpy(pp).to(dev), wv)
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"],
                                     mg.get("shared_output_gate"))
    dh, dp = layer.backward(inp.grad_out, mgv)
    torch.cuda.synchronize()
    assert dp.shape == (c.T, c.k)
    return GpuResult(out, dh, dp, mg, layer)


def _dense_of_slots(dp_slots, ids, E):
    """dprobs per slot -> the dense [T,E] layout (0 off the routes)."""
    T, k = ids.shape
    d = np.zeros((T, E))
    for t in range(T):
        for s in range(k):
            if ids[t, s] >= 0:
                d[t, ids[t, s]] = dp_slots[t, s]
    return d


@pytest.mark.parametrize("name", list(CASES))
def test_topk_ascending_slots_match_the_dense_path_bitwise(name):
    inp = make_inputs(CASES[name])
    ids, pp, over = O.route_pack(inp.map_np, inp.probs_np, inp.case.k)
    assert not over.any()
    dense = run_gpu(inp)
    top = _run_topk(inp, ids.astype(np.int32), pp.astype(np.float32))
    assert top.layer.device_status() == 0
    assert torch.equal(top.out, dense.out)
    assert torch.equal(top.dhidden, dense.dhidden)
    for n in dense.main_grads:
        assert torch.equal(top.main_grads[n], dense.main_grads[n]), n
    dd = dense.dprobs.cpu().numpy()
    dt = top.dprobs.cpu().numpy()
    for t in range(inp.case.T):
        for s in range(inp.case.k):
            want = dd[t, ids[t, s]] if ids[t, s] >= 0 else 0.0
            assert dt[t, s] == want, (t, s)


@pytest.mark.parametrize("name", [n for n in CASES if not CASES[n].mx])
def test_topk_any_slot_order_matches_the_oracle(name):
    inp = make_inputs(CASES[name])
    c = inp.case
    ids, pp, _ = O.route_pack(inp.map_np, inp.probs_np, c.k)
    rng = np.random.default_rng(c.seed)
    for t in range(c.T):                       # each token's slots (empty ones included) shuffled
        p = rng.permutation(c.k)
        ids[t] = ids[t, p]
        pp[t] = pp[t, p]
    pp = np.where(ids >= 0, pp, rng.standard_normal(pp.shape))   # probs of empty slots are ignored
    top = _run_topk(inp, ids.astype(np.int32), pp.astype(np.float32))
    assert top.layer.device_status() == 0
    dense_dp = torch.from_numpy(_dense_of_slots(top.dprobs.cpu().numpy(), ids, c.E))
    _compare_full(inp, dataclasses.replace(top, dprobs=dense_dp))


def test_topk_rows_with_bad_ids_are_reported_and_dropped():
    c = Case(T=64, H=128, E=6, k=3, I=64, seed=93)
    r = make_routing(c.T, c.E, c.k, c.seed)
    ids, pp, _ = O.route_pack(r.routing_map, r.probs, c.k)
    ids = ids.astype(np.int32)
    ids[5, :2] = [2, 2]                        # the same expert twice
    ids[9, 0] = c.E                            # out of range
    ids[11, 1] = -3                            # below -1
    r.routing_map[[5, 9, 11]] = False          # the dense equivalent: those rows route nowhere
    inp = make_inputs(c, routing=r)
    dense = run_gpu(inp)
    assert dense.layer.device_status() == 0
    top = _run_topk(inp, ids, pp.astype(np.float32))
    assert top.layer.device_status() == 3      # MOE_ERR_ROUTING
    assert torch.equal(top.out, dense.out)
    assert torch.equal(top.dhidden, dense.dhidden)
    for n in dense.main_grads:
        assert torch.equal(top.main_grads[n], dense.main_grads[n]), n
    dt = top.dprobs.cpu().numpy()
    assert np.all(dt[[5, 9, 11]] == 0)


def test_topk_zero_tokens():
    c = Case(T=64, H=128, E=4, k=2, I=64, seed=94)
    inp = make_inputs(c)
    dev = inp.hidden.device
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, device=dev)
    wv = weight_views(inp)
    empty_ids = torch.empty((0, c.k), dtype=torch.int32, device=dev)
    empty_pp = torch.empty((0, c.k), dtype=torch.float32, device=dev)
    out = layer.forward_topk(inp.hidden[:0], empty_ids, empty_pp, wv)
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"])
    dh, dp = layer.backward(inp.grad_out[:0], mgv)
    torch.cuda.synchronize()
    assert out.shape == (0, c.H) and dh.shape == (0, c.H) and dp.shape == (0, c.k)
    for n in mg:                               # nothing accumulated
        assert torch.equal(mg[n], inp.main_grads[n]), n
    assert layer.device_status() == 0


def test_topk_config2_full_size_matches_the_dense_path_bitwise():
    """Proxy-like layer (T=4096, H=2048, E=96, top-6, I=1024) fed by its top-k ids and
    probs: every output, dhidden and main_grad element equal to the dense-map run."""
    from tests.harness import config_case
    inp = make_inputs(config_case(2))
    ids, pp, over = O.route_pack(inp.map_np, inp.probs_np, inp.case.k)
    assert not over.any()
    dense = run_gpu(inp)
    top = _run_topk(inp, ids.astype(np.int32), pp.astype(np.float32))
    assert top.layer.device_status() == 0
    assert torch.equal(top.out, dense.out)
    assert torch.equal(top.dhidden, dense.dhidden)
    for n in dense.main_grads:
        assert torch.equal(top.main_grads[n], dense.main_grads[n]), n
    dd = dense.dprobs.cpu().numpy()
    want = np.where(ids >= 0, np.take_along_axis(dd, np.maximum(ids, 0), axis=1), 0.0)
    assert np.array_equal(top.dprobs.cpu().numpy(), want)
