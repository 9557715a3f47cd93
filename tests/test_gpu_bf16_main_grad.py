"""BF16 main_grad accumulation on the GPU, through the C ABI.

The oracle accumulates the exact weight gradients with the BF16 rule
(main_grad = bf16(main_grad + bf16(dW))). The kernel's dW is its fp32
accumulator, within the layer's dW tolerance of the exact one, so each new
main_grad element may differ from the oracle's by that tolerance plus one bf16
ulp of dW (the contribution's rounding) plus one ulp of the sum (its rounding).
Elsewhere the two agree bitwise: a rounding differs only where the kernel's dW
and the exact one straddle a bf16 midpoint. The test requires 97% bitwise
agreement. Experts without tokens keep their main_grad bitwise.
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


def _agree(got, want, d, ev, name, rtol, atol):
    """got vs want within the dW tolerance (atol relative to the whole buffer's
    max |dW|) plus one ulp of the contribution and one of the sum; returns the
    number of bitwise-equal elements."""
    bound = (rtol * np.abs(d) + atol * np.abs(d).max() + ev + _ulp(d) +
             _ulp(np.maximum(np.abs(want), np.abs(got))))
    err = np.abs(got - want)
    assert np.all(err <= bound), f"{name}: {int(np.sum(err > bound))} elements out of bound"
    return int(np.sum(got == want))


def _check(inp, res):
    c = inp.case
    rtol, atol = (6e-2, 6e-3) if c.mx else (2e-2, 1e-3)
    _, _, _, grads, cache = oracle_full(inp, "mxfp8" if c.mx else "exact")
    env = cache["jumps"]
    mg0 = _split({n: f64(t) for n, t in inp.main_grads.items()}, c.I)
    mg1 = _split({n: f64(t) for n, t in res.main_grads.items()}, c.I)
    ref = O.accumulate_main_grads(mg0, grads, dtype="bf16")
    equal = total = 0
    for n in ("shared_gate", "shared_up", "shared_down", "shared_output_gate"):
        if n in grads:
            equal += _agree(mg1[n], ref[n], grads[n], env[n], n, rtol, atol)
            total += ref[n].size
    experts = sorted(grads["routed"])
    for j, n in enumerate(("routed_gate", "routed_up", "routed_down")):
        st = lambda m: np.stack([m[e] for e in experts])  # noqa: E731
        d = np.stack([grads["routed"][e][j] for e in experts])
        ev = np.stack([env["routed"][e][j] for e in experts])
        equal += _agree(st(mg1[n]), st(ref[n]), d, ev, n, rtol, atol)
        total += d.size
        for e in range(c.E):
            if e not in grads["routed"]:
                assert np.array_equal(mg1[n][e], mg0[n][e])
    assert equal >= 0.97 * total, f"only {equal / total:.4f} of the main_grad elements agree bitwise"
    return equal / total


CASES = {
    "ragged": Case(T=300, H=256, E=8, k=2, I=128, seed=51, drop="iid", mg_bf16=True),
    "bn64_skewed_gated": Case(T=517, H=384, E=12, k=3, I=192, seed=52, routing="zipf", drop="multi",
                              mg_bf16=True, gated=True, limit=0.3),
    "mxfp8": Case(T=300, H=256, E=8, k=2, I=128, seed=53, mx=True, mg_bf16=True),
    "long_k": Case(T=1100, H=256, E=4, k=2, I=128, seed=54, mg_bf16=True),   # the deep weight-gradient build
}


@pytest.mark.parametrize("name", [n for n in CASES if not CASES[n].mx])
def test_bf16_main_grad_small(name):
    inp = make_inputs(CASES[name])
    res = run_gpu(inp)
    share = _check(inp, res)
    assert res.layer.device_status() == 0
    print(name, "bitwise-equal share:", share)


def test_bf16_main_grad_with_mxfp8_experts():
    """MXFP8 routed experts: against the mxfp8-mode oracle's weight gradients with
    the MXFP8 tolerance plus two bf16 ulps."""
    inp = make_inputs(CASES["mxfp8"])
    res = run_gpu(inp)
    assert res.layer.device_status() == 0
    share = _check(inp, res)
    print("mxfp8 bitwise-equal share:", share)


def test_bf16_main_grad_config2_full():
    inp = make_inputs(dataclasses.replace(config_case(2), mg_bf16=True))
    res = run_gpu(inp)
    share = _check(inp, res)
    print("config 2 bf16 main_grad bitwise-equal share:", share)
