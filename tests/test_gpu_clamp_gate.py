"""The swiglu_limit clamp and the shared expert's output gate on the GPU,
through the C ABI, against the oracle with the same clamp and gate.

Same bars as the plain layer: per element |gpu - ref| <= 2e-2 |ref| +
1e-3 max|ref| against the exact definition, plus, where a SwiGLU input's fp32
evaluation lies within its error band of a clamp bound, the other gradient
mask's effect (either side is a correct result); MXFP8 routed experts against
the mxfp8-mode oracle with 6e-2 / 6e-3 and normwise 6e-2 against the exact
definition. Every case checks that the clamp is active on a sizeable share of
the SwiGLU inputs, so a kernel that ignored it would fail.
"""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from tests.harness import Case, config_case, f64, make_inputs, oracle_weights, run_gpu
from tests.test_gpu_layer import _compare_full
from tests.test_gpu_mxfp8 import _compare as _compare_mx

pytestmark = pytest.mark.gpu

CASES = {
    "clamp_gate_ragged": Case(T=300, H=256, E=8, k=2, I=128, seed=31, drop="iid", limit=0.3, gated=True),
    "clamp_gate_bn64_skewed": Case(T=517, H=384, E=12, k=3, I=192, seed=32, routing="zipf", drop="multi",
                                   limit=0.3, gated=True),
    "gate_only": Case(T=300, H=256, E=8, k=2, I=128, seed=33, gated=True),
    "clamp_only": Case(T=300, H=256, E=8, k=2, I=128, seed=34, limit=0.3),
}


def _clamped_share(inp):
    """Share of the shared expert's gate and up inputs outside the clamp."""
    W = oracle_weights(inp)
    g, u, _, _ = O.expert_forward(f64(inp.hidden), *W.shared())
    L = inp.case.limit
    return float(np.mean(g > L)), float(np.mean(np.abs(u) > L))


@pytest.mark.parametrize("name", list(CASES))
def test_clamp_and_gate_parity_small(name):
    inp = make_inputs(CASES[name])
    if inp.case.limit:
        sg, su = _clamped_share(inp)
        assert sg > 0.05 and su > 0.1, (sg, su)
    res = run_gpu(inp)
    errs = _compare_full(inp, res)
    assert res.layer.device_status() == 0
    if inp.case.gated:
        assert "dW shared output gate" in errs


def test_clamp_and_gate_parity_config2_full():
    """Proxy-like layer (T=4096, H=2048, E=96, top-6, I=1024) with swiglu_limit 0.8
    and a gated shared expert: every output element and weight gradient."""
    inp = make_inputs(dataclasses.replace(config_case(2), limit=0.8, gated=True))
    sg, su = _clamped_share(inp)
    assert sg > 0.1 and su > 0.2, (sg, su)
    res = run_gpu(inp)
    errs = _compare_full(inp, res)
    print("config 2 + clamp + gate max|err|/max|ref|:", {n: f"{v:.2e}" for n, v in errs.items()})


def test_mxfp8_clamp_and_gate_parity_small():
    inp = make_inputs(Case(T=300, H=256, E=8, k=2, I=128, seed=35, drop="iid", mx=True, limit=0.3, gated=True))
    res = run_gpu(inp)
    _compare_mx(inp, res)
    assert res.layer.device_status() == 0
