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
