"""Pins for the oracle's forward pass.

* a hand-derived worked example (tests/golden/tiny_layer_worked_example.json);
* the textbook dense SwiGLU, written as explicit per-element sums, for tokens
  routed to one expert, for E=1/k=1, and for rows with no route;
* an id of -1 contributes exactly zero (the dropped prob is ignored);
* the routed part is linear in the probs; tokens are independent.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sig(z):
    return 1.0 / (1.0 + math.exp(-z))


def _silu(z):
    return z * _sig(z)


def _dsilu(z):
    s = _sig(z)
    return s + z * s * (1.0 - s)


def eval_closed_form(expr):
    ns = {"silu": _silu, "sig": _sig, "dsilu": _dsilu, "__builtins__": {}}
    return np.vectorize(lambda s: float(eval(s, ns)), otypes=[float])(np.array(expr, dtype=object))


def load_worked_example():
    with open(os.path.join(GOLDEN, "tiny_layer_worked_example.json")) as f:
        ex = json.load(f)
    W = O.DenseWeights.from_combined(np.array(ex["shared_fc1"]), np.array(ex["shared_fc2"]),
                                     np.array(ex["routed_fc1"]), np.array(ex["routed_fc2"]))
    return ex, W


def test_worked_example_forward():
    ex, W = load_worked_example()
    out, cache = O.forward(np.array(ex["hidden"]), np.array(ex["probs"]),
                           np.array(ex["routing_map"], bool), W, ex["k"])
    exp = ex["expected"]
    assert cache["ids"].tolist() == exp["ids"]
    assert cache["counts"].tolist() == exp["counts"]
    assert cache["perm_src"].tolist() == exp["perm_src"]
    np.testing.assert_allclose(out, eval_closed_form(exp["out"]), rtol=1e-14, atol=1e-15)


def _textbook_swiglu(x, Wg, Wu, Wd):
    """Dense SwiGLU MLP of one token, as explicit sums (no matmul)."""
    I, H = Wg.shape
    a = []
    for i in range(I):
        g = sum(Wg[i, h] * x[h] for h in range(H))
        u = sum(Wu[i, h] * x[h] for h in range(H))
        a.append(_silu(g) * u)
    return np.array([sum(Wd[h, i] * a[i] for i in range(I)) for h in range(Wd.shape[0])])


def _rand_layer(rng, H, I, E, scale=0.3):
    return O.DenseWeights(rng.standard_normal((I, H)) * scale, rng.standard_normal((I, H)) * scale,
                          rng.standard_normal((H, I)) * scale, rng.standard_normal((E, I, H)) * scale,
                          rng.standard_normal((E, I, H)) * scale, rng.standard_normal((E, H, I)) * scale)


def test_single_route_token_is_dense_swiglu():
    rng = np.random.default_rng(7)
    T, H, I, E, k = 5, 6, 4, 3, 2           # H != I so a transposed operand cannot pass
    W = _rand_layer(rng, H, I, E)
    x = rng.standard_normal((T, H))
    m = np.zeros((T, E), bool)
    probs = rng.random((T, E))
    route = [2, 0, 1, 2, 0]
    for t, e in enumerate(route):
        m[t, e] = True
    out, _ = O.forward(x, probs, m, W, k)
    for t, e in enumerate(route):
        ref = probs[t, e] * _textbook_swiglu(x[t], *W.routed(e)) + _textbook_swiglu(x[t], *W.shared())
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-13)


def test_two_route_token_sums_in_prob_weights():
    rng = np.random.default_rng(8)
    T, H, I, E, k = 3, 5, 3, 4, 2
    W = _rand_layer(rng, H, I, E)
    x = rng.standard_normal((T, H))
    m = np.zeros((T, E), bool)
    m[0, [1, 3]] = True
    m[1, [0, 2]] = True
    m[2, [2, 3]] = True
    probs = rng.random((T, E))
    out, _ = O.forward(x, probs, m, W, k)
    for t in range(T):
        ref = _textbook_swiglu(x[t], *W.shared())
        for e in np.flatnonzero(m[t]):
            ref = ref + probs[t, e] * _textbook_swiglu(x[t], *W.routed(e))
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-13)


def test_one_expert_top1_is_two_dense_swiglus():
    rng = np.random.default_rng(9)
    T, H, I = 4, 7, 5
    W = _rand_layer(rng, H, I, 1)
    x = rng.standard_normal((T, H))
    out, _ = O.forward(x, np.ones((T, 1)), np.ones((T, 1), bool), W, 1)
    for t in range(T):
        ref = _textbook_swiglu(x[t], *W.routed(0)) + _textbook_swiglu(x[t], *W.shared())
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-13)


def test_missing_routes_contribute_exactly_zero():
    rng = np.random.default_rng(10)
    T, H, I, E, k = 8, 6, 4, 5, 3
    W = _rand_layer(rng, H, I, E)
    x = rng.standard_normal((T, H))
    m = rng.random((T, E)) < 0.35
    m[:, 3:] = False
    m[np.arange(T), rng.integers(0, 3, T)] = True
    probs = rng.random((T, E))
    out1, c1 = O.forward(x, probs, m, W, k)
    probs2 = probs.copy()
    probs2[~m] = rng.standard_normal(int((~m).sum())) * 100    # off-map probs: any value
    out2, _ = O.forward(x, probs2, m, W, k)
    assert np.array_equal(out1, out2)                            # bitwise
    # a row with no route at all is exactly the shared expert
    m[0] = False
    out3, _ = O.forward(x, probs, m, W, k)
    ys = O.expert_forward(x, *W.shared())[3]
    assert np.array_equal(out3[0], ys[0])
    np.testing.assert_allclose(out3[0], _textbook_swiglu(x[0], *W.shared()), rtol=1e-12, atol=1e-13)


def test_routed_part_linear_in_probs():
    rng = np.random.default_rng(11)
    T, H, I, E, k = 6, 4, 3, 4, 2
    W = _rand_layer(rng, H, I, E)
    x = rng.standard_normal((T, H))
    m = np.zeros((T, E), bool)
    for t in range(T):
        m[t, rng.choice(E, 2, replace=False)] = True
    probs = rng.random((T, E))
    ys = O.expert_forward(x, *W.shared())[3]
    out1, _ = O.forward(x, probs, m, W, k)
    out2, _ = O.forward(x, 3.5 * probs, m, W, k)
    np.testing.assert_allclose(out2 - ys, 3.5 * (out1 - ys), rtol=1e-12, atol=1e-13)


def test_tokens_are_independent():
    """The sampled full-size checks rest on this: forward on a subset of tokens
    gives exactly those rows of the full forward."""
    rng = np.random.default_rng(12)
    T, H, I, E, k = 16, 8, 4, 5, 2
    W = _rand_layer(rng, H, I, E)
    x = rng.standard_normal((T, H))
    m = np.zeros((T, E), bool)
    for t in range(T):
        m[t, rng.choice(E, int(rng.integers(0, 3)), replace=False)] = True
    probs = rng.random((T, E))
    out, _ = O.forward(x, probs, m, W, k)
    sub = np.array([3, 7, 8, 15])
    out_s, _ = O.forward(x[sub], probs[sub], m[sub], W, k)
    np.testing.assert_allclose(out_s, out[sub], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("z", [-30.0, -3.0, -0.5, 0.0, 0.7, 4.0, 30.0])
def test_silu_closed_form(z):
    assert O.silu(np.array(z)) == pytest.approx(_silu(z), rel=1e-15, abs=1e-300)
