"""BF16 main_grad accumulation on the GPU, through the C ABI.

The oracle accumulates its bf16-mode weight gradients with the BF16 rule
(main_grad = bf16(main_grad + bf16(dW))). The kernel's dW is its fp32
accumulator, within the layer's dW tolerance of the oracle's, so each new
main_grad element may differ from the oracle's by that tolerance plus one bf16
ulp of dW (the contribution's rounding) plus one ulp of the sum (its rounding).
Elsewhere the two agree bitwise. The rounding of a dW element differs wherever
the kernel's fp32 dW and the oracle's straddle a bf16 midpoint; the dg/du
operands that sit within the fp32 band of their own midpoint (about 1% of them
at H = 2048) each shift a dW row by a fraction of its ulp, which flips about
1.3% of the proxy-sized layer's main_grad roundings (0.1% on small layers).
The test requires 97% bitwise agreement. Experts without tokens keep their
main_grad bitwise.
"""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from tests.harness import Case, config_case, f64, make_inputs, oracle_full, run_gpu

pytestmark = pytest.mark.gpu


def _ulp(v):
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, e - 8)


def _split(mg, I):
    out = dict(shared_gate=mg["shared_fc1"][:I], shared_up=mg["shared_fc1"][I:], shared_down=mg["shared_fc2"],
               routed_gate=mg["routed_fc1"][:, :I], routed_up=mg["routed_fc1"][:, I:], routed_down=mg["routed_fc2"])
    if "shared_output_gate" in mg:
        out["shared_output_gate"] = mg["shared_output_gate"]
    return out


def _agree(got, want, d, ev, name):
    """got vs want within the dW tolerance plus one ulp of the contribution and
    one of the sum; returns the number of bitwise-equal elements."""
    bound = (2e-2 * np.abs(d) + 1e-3 * np.abs(d).max() + ev + _ulp(d) +
             _ulp(np.maximum(np.abs(want), np.abs(got))))
    err = np.abs(got - want)
    assert np.all(err <= bound), f"{name}: {int(np.sum(err > bound))} elements out of bound"
    return int(np.sum(got == want))


def _check(inp, res):
    c = inp.case
    _, _, _, grads, cache = oracle_full(inp, "bf16")
    env = cache["envelope"]
    mg0 = _split({n: f64(t) for n, t in inp.main_grads.items()}, c.I)
    mg1 = _split({n: f64(t) for n, t in res.main_grads.items()}, c.I)
    ref = O.accumulate_main_grads(mg0, grads, dtype="bf16")
    equal = total = 0
    for n in ("shared_gate", "shared_up", "shared_down", "shared_output_gate"):
        if n in grads:
            equal += _agree(mg1[n], ref[n], grads[n], env[n], n)
            total += ref[n].size
    for e in range(c.E):
        kinds = ("routed_gate", "routed_up", "routed_down")
        if e in grads["routed"]:
            for j, n in enumerate(kinds):
                equal += _agree(mg1[n][e], ref[n][e], grads["routed"][e][j], env["routed"][e][j], f"{n}[{e}]")
                total += ref[n][e].size
        else:
            for n in kinds:
                assert np.array_equal(mg1[n][e], mg0[n][e])
    assert equal >= 0.97 * total, f"only {equal / total:.4f} of the main_grad elements agree bitwise"
    return equal / total


CASES = {
    "ragged": Case(T=300, H=256, E=8, k=2, I=128, seed=51, drop="iid", mg_bf16=True),
    "bn64_skewed_gated": Case(T=517, H=384, E=12, k=3, I=192, seed=52, routing="zipf", drop="multi",
                              mg_bf16=True, gated=True, limit=0.3),
    "mxfp8": Case(T=300, H=256, E=8, k=2, I=128, seed=53, mx=True, mg_bf16=True),
}


@pytest.mark.parametrize("name", [n for n in CASES if not CASES[n].mx])
def test_bf16_main_grad_small(name):
    inp = make_inputs(CASES[name])
    res = run_gpu(inp)
    share = _check(inp, res)
    assert res.layer.device_status() == 0
    print(name, "bitwise-equal share:", share)


def test_bf16_main_grad_with_mxfp8_experts():
    """MXFP8 routed experts (weight gradients are bf16-operand GEMMs in that mode):
    against the mxfp8-mode oracle with the MXFP8 tolerance plus two bf16 ulps."""
    inp = make_inputs(CASES["mxfp8"])
    res = run_gpu(inp)
    assert res.layer.device_status() == 0
    _, _, _, grads, _ = oracle_full(inp, "mxfp8")
    mg0 = _split({n: f64(t) for n, t in inp.main_grads.items()}, inp.case.I)
    mg1 = _split({n: f64(t) for n, t in res.main_grads.items()}, inp.case.I)
    ref = O.accumulate_main_grads(mg0, grads, dtype="bf16")
    for n in ("shared_gate", "shared_up", "shared_down", "routed_gate", "routed_up", "routed_down"):
        d = ref[n] - mg0[n]
        bound = 6e-2 * np.abs(d) + 6e-3 * np.abs(d).max() + 2 * _ulp(np.abs(ref[n]) + 1e-30)
        assert np.all(np.abs(mg1[n] - ref[n]) <= bound), n


def test_bf16_main_grad_config2_full():
    inp = make_inputs(dataclasses.replace(config_case(2), mg_bf16=True))
    res = run_gpu(inp)
    share = _check(inp, res)
    print("config 2 bf16 main_grad bitwise-equal share:", share)
