"""MXFP8 routed experts on the GPU, through the C ABI.

* quantisation (moe_quantize_mxfp8) is compared bit-exactly with the oracle
  codec on the same bf16 input, rowwise and columnwise;
* the layer with MXFP8 routed weights is compared, per element, with the oracle
  in mxfp8 mode -- the method: the same dequantised weights, the GEMM operands
  quantised on the fly at the same points -- within
  |gpu - ref| <= 6e-2 |ref| + 6e-3 max|ref| + env (env: the oracle's envelope of
  the other valid roundings of operands at a rounding midpoint within fp32
  evaluation precision) for every output and weight gradient;
* the distance from the exact oracle on the same dequantised weights with
  unquantised activations is reported (it measures MXFP8's own approximation
  error, e.g. dW_down averages the E4M3 error of a over only n_e tokens).
"""
import numpy as np
import pytest
import torch

from oracle import mxfp8 as MX
from tests.harness import Case, assert_close, config_case, f64, make_inputs, oracle_full, run_gpu

pytestmark = pytest.mark.gpu

MX_RTOL, MX_ATOL = 6e-2, 6e-3


def _bf16_matrix(rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 3)
    x[0, :32] = 0.0                                           # an all-zero block
    x[1, :32] = -0.0
    x[2, 5] = 1e-30                                           # far below its block's amax
    x[3, :32] = 448.0 * 2.0 ** torch.arange(-3, 29).float() / 2 ** 28   # spans the E4M3 range
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("axis", [1, 0])
def test_quantiser_bit_exact(axis):
    import mixture_experts_layer_pack_gb300 as M
    x = _bf16_matrix(256, 384, 7 + axis)
    dev = torch.device("cuda")
    xd = x.to(dev)
    q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    s = torch.empty((256, 384 // 32) if axis == 1 else (256 // 32, 384), dtype=torch.uint8, device=dev)
    M.moe_quantize_mxfp8(xd, axis, q, s)
    torch.cuda.synchronize()
    rq, rs = MX.quantize(x.double().numpy(), axis=axis)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def _compare(inp, res):
    c = inp.case
    I = c.I
    mg0 = {n: f64(t) for n, t in inp.main_grads.items()}
    mg1 = {n: f64(t) for n, t in res.main_grads.items()}
    d = {n: mg1[n] - mg0[n] for n in mg0}
    got = {"out": f64(res.out), "dhidden": f64(res.dhidden), "dprobs": f64(res.dprobs)}
    errs = {}
    for prec in ("mxfp8", "exact"):
        out, dx, dprobs, grads, cache = oracle_full(inp, prec)
        env = cache["envelope"]
        ref = {"out": out, "dhidden": dx, "dprobs": dprobs}
        ev = {}
        if env is not None:
            ev = {"out": env["out"], "dhidden": env["dhidden"], "dprobs": env["dprobs"],
                  "dW shared gate": env["shared_gate"], "dW shared up": env["shared_up"],
                  "dW shared down": env["shared_down"]}
        for e, (dWg, dWu, dWd) in grads["routed"].items():
            for j, (kind, r, gv) in enumerate((("gate", dWg, d["routed_fc1"][e, :I]),
                                               ("up", dWu, d["routed_fc1"][e, I:]),
                                               ("down", dWd, d["routed_fc2"][e]))):
                ref[f"dW routed {kind}[{e}]"] = r
                got[f"dW routed {kind}[{e}]"] = gv
                if env is not None:
                    ev[f"dW routed {kind}[{e}]"] = env["routed"][e][j]
        ref["dW shared gate"], got["dW shared gate"] = grads["shared_gate"], d["shared_fc1"][:I]
        ref["dW shared up"], got["dW shared up"] = grads["shared_up"], d["shared_fc1"][I:]
        ref["dW shared down"], got["dW shared down"] = grads["shared_down"], d["shared_fc2"]
        if "shared_output_gate" in grads:
            ref["dW shared output gate"] = grads["shared_output_gate"]
            got["dW shared output gate"] = d["shared_output_gate"]
            if env is not None:
                ev["dW shared output gate"] = env["shared_output_gate"]
        for n, r in ref.items():
            if prec == "mxfp8":
                errs[n] = assert_close(got[n], r, n, rtol=MX_RTOL, atol_frac=MX_ATOL, env=ev.get(n))
            else:
                errs["exact " + n] = float(np.max(np.abs(got[n] - r)) / max(np.max(np.abs(r)), 1e-300))
    return errs


MX_SMALL = {
    "tiles_ragged": Case(T=300, H=256, E=8, k=2, I=128, seed=41, drop="iid", mx=True),
    "skewed": Case(T=517, H=384, E=6, k=3, I=256, seed=42, routing="zipf", drop="multi", mx=True),
}


@pytest.mark.parametrize("name", list(MX_SMALL))
def test_mxfp8_layer_parity_small(name):
    inp = make_inputs(MX_SMALL[name])
    res = run_gpu(inp)
    errs = _compare(inp, res)
    assert res.layer.device_status() == 0
    print(name, "vs exact oracle:", {n: f"{v:.2e}" for n, v in errs.items() if n.startswith("exact") and "[" not in n})


def test_mxfp8_layer_parity_config3_full():
    """Proxy-like layer with MXFP8 routed weights (T=4096, H=2048, E=96, top-6, I=1024)."""
    inp = make_inputs(config_case(3))
    res = run_gpu(inp)
    errs = _compare(inp, res)
    print("config 3 max|err|/max|ref|:", {n: f"{v:.2e}" for n, v in errs.items() if "[" not in n})
    print("config 3 routed dW vs exact oracle, worst expert:",
          {k: f"{max(v for n, v in errs.items() if n.startswith('exact dW routed ' + k)):.2e}"
           for k in ("gate", "up", "down")})


@pytest.mark.slow
def test_mxfp8_layer_parity_config4_sampled():
    """DSv4-like layer (T=8192, H=7168, E=384, top-6, I=2048, MXFP8 routed, 2% of
    routes missing) at full size: sampled tokens for out/dhidden/dprobs, the
    busiest and a median expert for routed main_grad, all tokens for the shared
    expert's main_grad; the backward accumulates in place (main_grad is 68 GB)."""
    import mixture_experts_layer_pack_gb300 as M
    from oracle import moe_oracle as O
    from tests.harness import TorchMxWeights, weight_views
    inp = make_inputs(config_case(4))
    c = inp.case
    I = c.I
    W = TorchMxWeights(inp.weights, inp.mx)
    counts = inp.map_np.sum(0)
    hot = int(np.argmax(counts))
    med = int(np.argsort(counts)[c.E // 2])
    mg0 = {e: (inp.main_grads["routed_fc1"][e].cpu(), inp.main_grads["routed_fc2"][e].cpu()) for e in (hot, med)}
    mg0_shared = {n: inp.main_grads[n].cpu() for n in ("shared_fc1", "shared_fc2")}
    idle = np.flatnonzero(counts == 0)
    idle_before = {int(e): inp.main_grads["routed_fc1"][e].clone() for e in idle[:2]}

    layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, routed_wtype=M.binding.MOE_W_MXFP8)
    wv = weight_views(inp)
    layer.prepare_weights(wv)
    inp.weights["routed_fc1"] = inp.weights["routed_fc2"] = None        # the layer reads the MXFP8 copies
    torch.cuda.empty_cache()
    out = layer.forward(inp.hidden, inp.probs, inp.routing_map.view(torch.uint8), wv)
    mg = inp.main_grads
    mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"])
    dh, dp = layer.backward(inp.grad_out, mgv)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert torch.isfinite(out).all() and torch.isfinite(dh).all() and torch.isfinite(dp).all()

    rng = np.random.default_rng(4)
    toks = np.sort(rng.choice(c.T, 16, replace=False))
    tt = torch.from_numpy(toks).to(inp.hidden.device)
    ref, cache = O.forward(f64(inp.hidden[tt]), inp.probs_np[toks], inp.map_np[toks], W, c.k, precision="mxfp8")
    go = f64(inp.grad_out[tt])
    rdx, rdp, _ = O.backward(go, cache, W)
    env = O.envelope(go, cache, W)
    kw = dict(rtol=MX_RTOL, atol_frac=MX_ATOL)
    assert_close(f64(out[tt]), ref, "out (sampled)", env=env["out"], **kw)
    assert_close(f64(dh[tt]), rdx, "dhidden (sampled)", env=env["dhidden"], **kw)
    assert_close(f64(dp[tt]), rdp, "dprobs (sampled)", env=env["dprobs"], **kw)

    for e in (hot, med):
        rows = np.flatnonzero(inp.map_np[:, e])
        m = np.zeros((rows.size, c.E), bool)
        m[:, e] = True
        rt = torch.from_numpy(rows).to(inp.hidden.device)
        _, ce = O.forward(f64(inp.hidden[rt]), inp.probs_np[rows], m, W, c.k, precision="mxfp8")
        goe = f64(inp.grad_out[rt])
        _, _, ge = O.backward(goe, ce, W)
        ee = O.envelope(goe, ce, W)["routed"][e]
        d1 = f64(mg["routed_fc1"][e]) - mg0[e][0].double().numpy()
        d2 = f64(mg["routed_fc2"][e]) - mg0[e][1].double().numpy()
        assert_close(d1[:I], ge["routed"][e][0], f"dW routed gate[{e}]", env=ee[0], **kw)
        assert_close(d1[I:], ge["routed"][e][1], f"dW routed up[{e}]", env=ee[1], **kw)
        assert_close(d2, ge["routed"][e][2], f"dW routed down[{e}]", env=ee[2], **kw)
    for e, before in idle_before.items():
        assert torch.equal(mg["routed_fc1"][e], before)

    m0 = np.zeros_like(inp.map_np)
    _, cs = O.forward(f64(inp.hidden), inp.probs_np, m0, W, c.k, precision="mxfp8")
    gall = f64(inp.grad_out)
    _, _, gs = O.backward(gall, cs, W)
    es = O.envelope(gall, cs, W)
    d1 = f64(mg["shared_fc1"]) - mg0_shared["shared_fc1"].double().numpy()
    d2 = f64(mg["shared_fc2"]) - mg0_shared["shared_fc2"].double().numpy()
    assert_close(d1[:I], gs["shared_gate"], "dW shared gate", env=es["shared_gate"], **kw)
    assert_close(d1[I:], gs["shared_up"], "dW shared up", env=es["shared_up"], **kw)
    assert_close(d2, gs["shared_down"], "dW shared down", env=es["shared_down"], **kw)
