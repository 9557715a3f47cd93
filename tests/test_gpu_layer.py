"""Parity of the CUDA layer (through the C ABI) with the fp64 oracle.

Routing ids, probs, counts, offsets and permutation are compared bit-exactly.
Floating-point results of the default layer (fp32 activations) are compared,
element by element, with the exact definition (fp64, nothing rounded) within
|gpu - ref| <= 2e-2 |ref| + 1e-3 max|ref|, max over the whole compared tensor
(each routed main_grad buffer is one [E, I, H] or [E, H, I] tensor); no
envelope. Main-grad updates are compared as (main_grad_after -
main_grad_before) against dW. The layer with bf16 activations is compared with
the bf16-mode oracle plus its rounding envelope, and normwise with the exact
definition.
"""
import dataclasses

import numpy as np
import pytest
import torch

from moe_inputs import make_routing
from oracle import moe_oracle as O
from tests.harness import (BF16_TOL, Case, TorchWeights, assert_close, compare_layer, config_case, f64, make_inputs,
                           run_gpu)

pytestmark = pytest.mark.gpu

SMALL = {
    "cfg1": config_case(1),
    "tiles_ragged": Case(T=300, H=256, E=8, k=2, I=128, seed=21, drop="iid"),
    "bn64_skewed": Case(T=517, H=384, E=12, k=3, I=192, seed=22, routing="zipf", drop="multi"),
    "one_token": Case(T=1, H=128, E=4, k=2, I=64, seed=23),
    "odd_experts": Case(T=333, H=128, E=13, k=3, I=64, seed=24, drop="iid"),   # byte-wise map rows
    "max_experts_topk": Case(T=256, H=128, E=1024, k=32, I=64, seed=25),         # the largest E and k
    "single_expert": Case(T=200, H=128, E=1, k=1, I=64, seed=26),
    # ~512 rows per expert and more: the gate/up weight gradient's deep build (three stages,
    # one main_grad box buffer per warp)
    "long_k": Case(T=1100, H=256, E=4, k=2, I=128, seed=27, drop="iid"),
}


def _export_routing(res, inp):
    import mixture_experts_layer_pack_gb300 as M
    c = inp.case
    dev = inp.hidden.device
    ids = torch.empty((c.T, c.k), dtype=torch.int32, device=dev)
    pp = torch.empty((c.T, c.k), dtype=torch.float32, device=dev)
    counts = torch.empty(c.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(c.E + 1, dtype=torch.int32, device=dev)
    perm = torch.full((c.T * c.k,), -7, dtype=torch.int32, device=dev)
    row_of = torch.empty((c.T, c.k), dtype=torch.int32, device=dev)
    M.moe_export_routing(res.layer.handle, res.layer.saved, ids, pp, counts, offsets, perm, row_of)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (ids, pp, counts, offsets, perm, row_of)]


def _check_routing(res, inp):
    ids, pp, counts, offsets, perm, row_of = _export_routing(res, inp)
    rids, rpp, over = O.route_pack(inp.map_np, inp.probs_np, inp.case.k)
    assert not over.any()
    rc, ro, rsrc, rslot, rrow = O.dispatch_indices(rids, inp.case.E)
    R = int(rc.sum())
    assert np.array_equal(ids, rids)
    assert np.array_equal(pp.astype(np.float64), rpp)          # fp32 gather: bit-exact
    assert np.array_equal(counts, rc)
    assert np.array_equal(offsets, ro)
    assert np.array_equal(perm[:R], rsrc)
    assert np.all(perm[R:] == -7)
    assert np.array_equal(row_of, rrow)


@pytest.mark.parametrize("name", list(SMALL))
def test_routing_bit_exact(name):
    inp = make_inputs(SMALL[name])
    res = run_gpu(inp, backward=False)
    _check_routing(res, inp)
    assert res.layer.device_status() == 0


@pytest.mark.parametrize("cfg,variant", [(2, None), (2, "balanced"), (5, None)])
def test_routing_bit_exact_full_size(cfg, variant):
    c = config_case(cfg, variant=variant)
    inp = make_inputs(Case(c.T, 128, c.E, c.k, 64, c.seed, c.routing, c.drop))   # routing only depends on T, E, k
    res = run_gpu(inp, backward=False)
    _check_routing(res, inp)
    if variant == "balanced":
        _, _, counts, *_ = _export_routing(res, inp)
        assert np.all(counts == 256)


def _compare_full(inp, res):
    counts = {}
    errs = compare_layer(inp, res, exact_counts=counts)
    bad = {n: v for n, v in counts.items() if v[0]}
    assert inp.case.act_bf16 or inp.case.mx or not bad, bad
    return errs


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_parity_small(name):
    inp = make_inputs(SMALL[name])
    res = run_gpu(inp)
    _compare_full(inp, res)
    assert res.layer.device_status() == 0


def test_layer_parity_config2_full():
    """Proxy-like layer (T=4096, H=2048, E=96, top-6, I=1024): every output element."""
    inp = make_inputs(config_case(2))
    res = run_gpu(inp)
    counts = {}
    errs = compare_layer(inp, res, exact_counts=counts)
    print("config 2 max|err|/max|ref|:", {n: f"{v:.2e}" for n, v in errs.items()})
    print("config 2 worst err/bound:", {n: f"{v[1]:.3f}" for n, v in counts.items()})


@pytest.mark.parametrize("name", ["cfg1", "tiles_ragged", "bn64_skewed"])
def test_layer_parity_small_bf16_activations(name):
    """The layer with bf16 activations (MOE_ACT_BF16) against the bf16-mode oracle
    plus its rounding envelope, and normwise against the exact definition."""
    inp = make_inputs(dataclasses.replace(SMALL[name], act_bf16=True))
    res = run_gpu(inp)
    compare_layer(inp, res)
    assert res.layer.device_status() == 0


def test_layer_parity_config2_full_bf16_activations():
    inp = make_inputs(dataclasses.replace(config_case(2), act_bf16=True))
    res = run_gpu(inp)
    counts = {}
    errs = compare_layer(inp, res, exact_counts=counts)
    print("config 2 (bf16 activations) max|err|/max|exact|:", {n: f"{v:.2e}" for n, v in errs.items()})
    print("config 2 (bf16 activations) elements outside the BF16 tolerance of the exact definition:",
          {n: v[0] for n, v in counts.items()})


def test_layer_parity_config2_force_balanced():
    inp = make_inputs(config_case(2, variant="balanced"))
    res = run_gpu(inp)
    _compare_full(inp, res)


def test_wgrad_accumulates_once_bitwise():
    """main_grad += dW is one fp32 add per element: a pass from zero gives dW
    exactly, a pass from mg0 must equal fl32(mg0 + dW) bit for bit."""
    inp = make_inputs(SMALL["tiles_ragged"])
    zero = {n: torch.zeros_like(t) for n, t in inp.main_grads.items()}
    r0 = run_gpu(inp, main_grads=zero)
    r1 = run_gpu(inp, layer=r0.layer)
    for n in inp.main_grads:
        expect = inp.main_grads[n] + r0.main_grads[n]       # fp32 add on the device
        assert torch.equal(r1.main_grads[n], expect), n


def test_backward_twice_accumulates_twice():
    """Two backward passes over one forward (the skewed workload accumulates over
    two calls): the second adds the same dW again."""
    import mixture_experts_layer_pack_gb300 as M
    inp = make_inputs(SMALL["bn64_skewed"])
    zero = {n: torch.zeros_like(t) for n, t in inp.main_grads.items()}
    r0 = run_gpu(inp, main_grads=zero)
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"])
    r0.layer.backward(inp.grad_out, mgv)
    r0.layer.backward(inp.grad_out, mgv)
    torch.cuda.synchronize()
    for n in mg:
        expect = (inp.main_grads[n] + r0.main_grads[n]) + r0.main_grads[n]
        assert torch.equal(mg[n], expect), n


def test_determinism():
    inp = make_inputs(SMALL["bn64_skewed"])
    a = run_gpu(inp)
    b = run_gpu(inp)
    assert torch.equal(a.out, b.out) and torch.equal(a.dhidden, b.dhidden) and torch.equal(a.dprobs, b.dprobs)
    for n in a.main_grads:
        assert torch.equal(a.main_grads[n], b.main_grads[n]), n


@pytest.mark.parametrize("case", [
    Case(T=300, H=256, E=8, k=2, I=128, seed=35, drop="iid"),                 # fp32 activations
    Case(T=517, H=384, E=12, k=3, I=192, seed=36, routing="zipf", act_bf16=True),
    Case(T=290, H=256, E=6, k=2, I=128, seed=37, mx=True, limit=0.5),
])
def test_results_do_not_depend_on_workspace_contents(case):
    """The workspace and saved-state memory filled with NaN bytes (0xFF) or with zeros
    before the handle is created: bitwise the same results, two steps each. Padding rows
    past each expert's last 64-row block that holds a route are never written, so this
    also shows that nothing reads them into a result."""
    import mixture_experts_layer_pack_gb300 as M
    inp = make_inputs(case)
    c = inp.case
    res = []
    for fill in (0x00, 0xFF):
        layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, routed_wtype=M.binding.MOE_W_MXFP8 if c.mx else M.binding.MOE_W_BF16,
                           swiglu_limit=c.limit,
                           act_precision=M.binding.MOE_ACT_BF16 if c.act_bf16 else M.binding.MOE_ACT_FP32, fill=fill)
        steps = [run_gpu(inp, layer=layer) for _ in range(2)]
        assert layer.device_status() == 0
        res.append(steps)
        layer.close()
    for a, b in zip(*res):
        for name, x, y in (("out", a.out, b.out), ("dhidden", a.dhidden, b.dhidden), ("dprobs", a.dprobs, b.dprobs)):
            assert torch.equal(x, y), name
        for n in a.main_grads:
            assert torch.equal(a.main_grads[n], b.main_grads[n]), n
    assert torch.isfinite(res[1][0].out.float()).all()


def test_rows_without_routes_and_zero_token_experts():
    c = Case(T=200, H=128, E=6, k=2, I=64, seed=31)
    r = make_routing(c.T, c.E, c.k, c.seed)
    r.routing_map[:, 4] = False           # expert 4 gets no token
    r.probs[:, 4] = 0.0
    r.routing_map[::7] = False            # every 7th token has no route at all
    r.probs[::7] = 0.0
    inp = make_inputs(c, routing=r)
    res = run_gpu(inp)
    _compare_full(inp, res)
    assert torch.equal(res.main_grads["routed_fc1"][4], inp.main_grads["routed_fc1"][4])
    assert torch.equal(res.main_grads["routed_fc2"][4], inp.main_grads["routed_fc2"][4])
    assert torch.all(res.dprobs[::7] == 0)


def test_off_map_probs_ignored_and_prob_zero_routes():
    c = Case(T=150, H=128, E=5, k=2, I=64, seed=32)
    r = make_routing(c.T, c.E, c.k, c.seed)
    r.probs[~r.routing_map] = 123.0       # off-map probs: must be ignored
    on = np.argwhere(r.routing_map)[:10]
    r.probs[on[:, 0], on[:, 1]] = 0.0     # routed with prob 0: still computed
    inp = make_inputs(c, routing=r)
    res = run_gpu(inp)
    _compare_full(inp, res)
    assert torch.all(res.dprobs[~inp.routing_map] == 0)


def test_zero_tokens():
    import mixture_experts_layer_pack_gb300 as M
    c = Case(T=0, H=128, E=4, k=2, I=64, seed=33)
    inp = make_inputs(c)
    layer = M.MoELayer(16, c.H, c.E, c.k, c.I)
    w = inp.weights
    wv = M.weights_from_combined(w["shared_fc1"], w["shared_fc2"], w["routed_fc1"], w["routed_fc2"])
    layer.forward(inp.hidden, inp.probs, inp.routing_map.view(torch.uint8), wv)
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"])
    layer.backward(inp.grad_out, mgv)
    torch.cuda.synchronize()
    for n in mg:
        assert torch.equal(mg[n], inp.main_grads[n])
    assert layer.device_status() == 0


def test_row_with_too_many_routes_is_reported():
    c = Case(T=64, H=128, E=6, k=2, I=64, seed=34)
    r = make_routing(c.T, c.E, c.k, c.seed)
    r.routing_map[5, :3] = True           # three routes with k = 2
    inp = make_inputs(c, routing=r)
    res = run_gpu(inp, backward=False)
    assert res.layer.device_status() == 3     # MOE_ERR_ROUTING
    assert res.layer.device_status() == 0     # cleared by the read


def _routed_expert_grads(inp, W, e):
    """Exact oracle dW of expert e from the tokens routed to it (dW_e depends on
    nothing else)."""
    toks = np.flatnonzero(inp.map_np[:, e])
    m = np.zeros((toks.size, inp.case.E), bool)
    m[:, e] = True
    tt = torch.from_numpy(toks).to(inp.hidden.device)
    _, cache = O.forward(f64(inp.hidden[tt]), inp.probs_np[toks], m, W, inp.case.k, precision="exact")
    _, _, g = O.backward(f64(inp.grad_out[tt]), cache, W)
    return g["routed"][e]


@pytest.mark.slow
def test_layer_parity_config5_sampled():
    """Skewed layer (T=16384, H=4096, E=128, top-8, I=1536) at full size, against the
    exact definition: 96 sampled tokens for out/dhidden/dprobs, the hottest, a
    median and the least busy expert with tokens for routed main_grad (their
    gradients as one tensor), all tokens for the shared expert's main_grad. Then the accumulation over two
    consecutive backward calls: from mg0 the two calls give fl32(fl32(mg0 + dW) + dW)
    bit for bit, dW the update of a pass from zero."""
    import mixture_experts_layer_pack_gb300 as M
    inp = make_inputs(config_case(5))
    zero = {n: torch.zeros_like(t) for n, t in inp.main_grads.items()}
    res = run_gpu(inp, main_grads=zero)          # main_grad after = dW exactly
    c = inp.case
    W = TorchWeights(inp.weights)
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(c.T, 96, replace=False))
    tt = torch.from_numpy(toks).to(inp.hidden.device)
    out, cache = O.forward(f64(inp.hidden[tt]), inp.probs_np[toks], inp.map_np[toks], W, c.k, precision="exact")
    dx, dprobs, _ = O.backward(f64(inp.grad_out[tt]), cache, W)
    assert_close(f64(res.out[tt]), out, "out (sampled)", **BF16_TOL)
    assert_close(f64(res.dhidden[tt]), dx, "dhidden (sampled)", **BF16_TOL)
    assert_close(f64(res.dprobs[tt]), dprobs, "dprobs (sampled)", **BF16_TOL)
    assert torch.isfinite(res.out).all() and torch.isfinite(res.dhidden).all() and torch.isfinite(res.dprobs).all()

    counts = inp.map_np.sum(0)
    hot = int(np.argmax(counts))
    med = int(np.argsort(counts)[c.E // 2])
    cold = int(np.flatnonzero(counts == counts[counts > 0].min())[0])
    picked = (hot, med, cold)
    I = c.I
    ref = [_routed_expert_grads(inp, W, e) for e in picked]
    dW = {n: res.main_grads[n] for n in res.main_grads}
    for j, (kind, buf, rows) in enumerate((("gate", "routed_fc1", slice(0, I)), ("up", "routed_fc1", slice(I, 2 * I)),
                                           ("down", "routed_fc2", slice(None)))):
        got = np.stack([f64(dW[buf][e][rows]) for e in picked])
        assert_close(got, np.stack([r[j] for r in ref]), f"dW routed {kind} (hot, median, least busy)", **BF16_TOL)
    for e in np.flatnonzero(counts == 0):
        assert torch.equal(dW["routed_fc1"][e], zero["routed_fc1"][e])

    # shared expert over all tokens: a map with no routes leaves only the shared path
    m0 = np.zeros_like(inp.map_np)
    _, cache = O.forward(f64(inp.hidden), inp.probs_np, m0, W, c.k, precision="exact")
    _, _, g = O.backward(f64(inp.grad_out), cache, W)
    assert_close(f64(dW["shared_fc1"][:I]), g["shared_gate"], "dW shared gate", **BF16_TOL)
    assert_close(f64(dW["shared_fc1"][I:]), g["shared_up"], "dW shared up", **BF16_TOL)
    assert_close(f64(dW["shared_fc2"]), g["shared_down"], "dW shared down", **BF16_TOL)

    # two consecutive backward calls into main_grad = mg0
    mg = {n: t.clone() for n, t in inp.main_grads.items()}
    mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"])
    res.layer.backward(inp.grad_out, mgv)
    res.layer.backward(inp.grad_out, mgv)
    torch.cuda.synchronize()
    assert res.layer.device_status() == 0
    for n in mg:
        expect = (inp.main_grads[n] + dW[n]) + dW[n]      # fp32 adds on the device
        assert torch.equal(mg[n], expect), n


def test_bounded_wait_gives_up_and_the_handle_stays_usable():
    """The timeout path: a wait that nothing completes gives up after the library's limit
    (2 s), moe_device_status reports MOE_ERR_TIMEOUT once and clears it, and the same
    handle then runs a layer step that matches the one before."""
    import time
    import mixture_experts_layer_pack_gb300 as M
    inp = make_inputs(SMALL["tiles_ragged"])
    c = inp.case
    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I)
    before = run_gpu(inp, layer=layer)
    assert layer.device_status() == 0
    t0 = time.monotonic()
    M.moe_selftest_timeout(layer.handle)
    assert layer.device_status() == M.binding.MOE_ERR_TIMEOUT
    assert time.monotonic() - t0 >= 1.5
    assert layer.device_status() == 0
    after = run_gpu(inp, layer=layer)
    assert layer.device_status() == 0
    assert torch.equal(before.out, after.out) and torch.equal(before.dhidden, after.dhidden)
    for n in before.main_grads:
        assert torch.equal(before.main_grads[n], after.main_grads[n]), n
    layer.close()


def test_nan_in_one_token_stays_in_that_token():
    """A NaN in one token's hidden row: every other token's out, dhidden and dprobs row,
    and the main_grad of every routed expert the token is not routed to, are bitwise those
    of the clean run (each GEMM output row depends on its own input row only, each weight
    gradient's K range covers its expert's routes only, and padding rows are never read
    into a result); the token's own out row is NaN."""
    import dataclasses as dc
    inp = make_inputs(SMALL["tiles_ragged"])
    c = inp.case
    clean = run_gpu(inp)
    t0 = int(np.flatnonzero(inp.map_np.sum(1) > 0)[10])   # a token with routes
    hid = inp.hidden.clone()
    hid[t0, 5] = float("nan")
    bad = run_gpu(dc.replace(inp, hidden=hid))
    assert bad.layer.device_status() == 0
    keep = torch.ones(c.T, dtype=torch.bool, device=hid.device)
    keep[t0] = False
    assert torch.equal(bad.out[keep], clean.out[keep])
    assert torch.equal(bad.dhidden[keep], clean.dhidden[keep])
    assert torch.equal(bad.dprobs[keep], clean.dprobs[keep])
    assert torch.isnan(bad.out[t0].float()).any()
    routed_to = set(np.flatnonzero(inp.map_np[t0]).tolist())
    assert routed_to and len(routed_to) < c.E
    for e in range(c.E):
        if e in routed_to:
            continue
        for n in ("routed_fc1", "routed_fc2"):
            assert torch.equal(bad.main_grads[n][e], clean.main_grads[n][e]), (n, e)
