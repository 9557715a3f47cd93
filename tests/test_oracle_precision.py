"""Pins for the oracle's bf16-operand precision mode.

* ``bf16_round`` against PyTorch's fp32 -> bfloat16 cast (round to nearest even),
  ties included;
* forward in bf16 mode equals a per-element textbook SwiGLU that rounds the
  activation a (the down projection's operand) to bf16;
* rigorous first-order bounds: every bf16-mode result differs from the exact
  one by no more than the rounding of its operands allows (unit roundoff
  2^-8 per rounded operand, propagated with absolute values).
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.test_oracle_forward import _rand_layer, _silu

U = 2.0 ** -8      # bf16 unit roundoff (8 significant bits)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-6, 6, 100000),
                        [0.0, -0.0, 1.0, -3.5, 65504.0, 1e-30]]).astype(np.float32)
    # exact ties: a bf16 value plus half its ulp (low 16 bits of the fp32 = 0x8000)
    hi = (rng.integers(100, 150, 5000, dtype=np.uint32) << 7) | rng.integers(0, 128, 5000, dtype=np.uint32)
    bits = (hi << 16) | np.uint32(0x8000)
    x = np.concatenate([x, bits.view(np.float32), -bits.view(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_round_idempotent_on_bf16_values():
    v = torch.randn(10000, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(v), v)


def _textbook_swiglu_bf16(x, Wg, Wu, Wd):
    I, H = Wg.shape
    a = []
    for i in range(I):
        g = sum(Wg[i, h] * x[h] for h in range(H))
        u = sum(Wu[i, h] * x[h] for h in range(H))
        a.append(float(torch.tensor(_silu(g) * u, dtype=torch.float32).to(torch.bfloat16).double())
                 if abs(_silu(g) * u) < 1e30 else _silu(g) * u)
    return np.array([sum(Wd[h, i] * a[i] for i in range(I)) for h in range(Wd.shape[0])])


def test_bf16_forward_rounds_the_activation_only():
    rng = np.random.default_rng(3)
    T, H, I, E, k = 4, 6, 5, 3, 2
    W = _rand_layer(rng, H, I, E)
    x = rng.standard_normal((T, H))
    m = np.zeros((T, E), bool)
    route = [1, 0, 2, 1]
    for t, e in enumerate(route):
        m[t, e] = True
    probs = rng.random((T, E))
    out, _ = O.forward(x, probs, m, W, k, precision="bf16")
    for t, e in enumerate(route):
        ref = probs[t, e] * _textbook_swiglu_bf16(x[t], *W.routed(e)) + _textbook_swiglu_bf16(x[t], *W.shared())
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-13)


def _case(seed, T=12, H=8, I=6, E=4, k=2):
    rng = np.random.default_rng(seed)
    W = _rand_layer(rng, H, I, E, scale=0.5)
    x = rng.standard_normal((T, H))
    go = rng.standard_normal((T, H))
    m = np.zeros((T, E), bool)
    for t in range(T):
        m[t, rng.choice(E, size=int(rng.integers(1, k + 1)), replace=False)] = True
    return W, x, go, m, rng.random((T, E)), k


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bf16_mode_within_rounding_bounds(seed):
    W, x, go, m, probs, k = _case(seed)
    out_e, ce = O.forward(x, probs, m, W, k, precision="exact")
    out_b, cb = O.forward(x, probs, m, W, k, precision="bf16")
    dx_e, dp_e, g_e = O.backward(go, ce, W)
    dx_b, dp_b, g_b = O.backward(go, cb, W)
    assert not np.array_equal(out_e, out_b)          # the mode does round something

    # forward: |delta y| <= sum_i U |a_i| |Wd_hi| per expert, combined with |p|
    gs, us, as_ = ce["shared"]
    Wsg, Wsu, Wsd = W.shared()
    bound = (U * np.abs(as_)) @ np.abs(Wsd).T
    ids, pp, row_of = ce["ids"], ce["pp"], ce["row_of"]
    routed_a = np.zeros((ce["perm_src"].size, as_.shape[1]))
    for e, (g, u, a) in ce["routed"].items():
        lo, hi = ce["offsets"][e], ce["offsets"][e + 1]
        routed_a[lo:hi] = a
    for s in range(k):
        v = ids[:, s] >= 0
        for t in np.flatnonzero(v):
            e = ids[t, s]
            bound[t] += abs(pp[t, s]) * (U * np.abs(routed_a[row_of[t, s]])) @ np.abs(W.routed(e)[2]).T
    assert np.all(np.abs(out_b - out_e) <= bound * (1 + 1e-9) + 1e-15)

    # dprobs = <go, y>: |delta| <= sum_h |go_h| |delta y_h|
    for t, s in zip(*np.nonzero(ids >= 0)):
        e = ids[t, s]
        dy = (U * np.abs(routed_a[row_of[t, s]])) @ np.abs(W.routed(e)[2]).T
        assert abs(dp_b[t, e] - dp_e[t, e]) <= np.abs(go[t]) @ dy * (1 + 1e-9) + 1e-15

    # shared backward: dg, du rounded once; p*a = a (p = 1) already bf16
    da = go @ Wsd
    dg = da * us * O.silu_grad(gs)
    du = da * O.silu(gs)
    ddg, ddu = U * np.abs(dg), U * np.abs(du)
    assert np.all(np.abs(g_b["shared_gate"] - g_e["shared_gate"]) <= ddg.T @ np.abs(x) * (1 + 1e-9) + 1e-15)
    assert np.all(np.abs(g_b["shared_up"] - g_e["shared_up"]) <= ddu.T @ np.abs(x) * (1 + 1e-9) + 1e-15)
    assert np.all(np.abs(g_b["shared_down"] - g_e["shared_down"]) <=
                  np.abs(go).T @ (U * np.abs(as_)) * (1 + 1e-9) + 1e-15)
    # routed down wgrad: p*a rounded after a was: |delta| <= U (|p a_b| + |p a|) per element
    for e, (dWg, dWu, dWd) in g_e["routed"].items():
        lo, hi = ce["offsets"][e], ce["offsets"][e + 1]
        src, slot = ce["perm_src"][lo:hi], ce["perm_slot"][lo:hi]
        p = pp[src, slot]
        a_e = ce["routed"][e][2]
        a_b = cb["routed"][e][2]
        bd = np.abs(go[src]).T @ (U * (np.abs(p[:, None] * a_b) + np.abs(p[:, None] * a_e)))
        assert np.all(np.abs(g_b["routed"][e][2] - dWd) <= bd * (1 + 1e-9) + 1e-15)
