"""Pins for the oracle's backward pass and main_grad accumulation.

* central finite differences of L = sum(grad_out * forward(...)) in fp64 for
  dhidden, every on-map dprob and all six weight gradients (the forward is
  pinned by test_oracle_forward, so this pins backward to it);
* dprobs is exactly 0 off the map; the hand-derived worked example;
* main_grad accumulation adds dW once; a zero-token expert's buffers are left
  bitwise unchanged.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O
from tests.test_oracle_forward import eval_closed_form, load_worked_example

H_FD = 1e-6


def _tiny_case(seed, T=6, H=5, I=3, E=4, k=2):
    rng = np.random.default_rng(seed)
    W = O.DenseWeights(rng.standard_normal((I, H)) * 0.5, rng.standard_normal((I, H)) * 0.5,
                       rng.standard_normal((H, I)) * 0.5, rng.standard_normal((E, I, H)) * 0.5,
                       rng.standard_normal((E, I, H)) * 0.5, rng.standard_normal((E, H, I)) * 0.5)
    x = rng.standard_normal((T, H))
    go = rng.standard_normal((T, H))
    m = np.zeros((T, E), bool)
    for t in range(T):
        m[t, rng.choice(E - 1, size=int(rng.integers(1, k + 1)), replace=False)] = True  # expert E-1 idle
    m[T - 1] = False                                                                      # a row with no route
    probs = rng.random((T, E))
    return W, x, go, m, probs, k


def _loss(W, x, go, m, probs, k):
    out, _ = O.forward(x, probs, m, W, k)
    return float(np.sum(go * out))


def _fd(f, arr, idx):
    old = arr[idx]
    arr[idx] = old + H_FD
    lp = f()
    arr[idx] = old - H_FD
    lm = f()
    arr[idx] = old
    return (lp - lm) / (2 * H_FD)


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_matches_finite_differences(seed):
    W, x, go, m, probs, k = _tiny_case(seed)
    _, cache = O.forward(x, probs, m, W, k)
    dx, dprobs, grads = O.backward(go, cache, W)

    f = lambda: _loss(W, x, go, m, probs, k)   # noqa: E731  (closes over the arrays it perturbs)
    fd_dx = np.array([[_fd(f, x, (t, h)) for h in range(x.shape[1])] for t in range(x.shape[0])])
    np.testing.assert_allclose(dx, fd_dx, rtol=1e-6, atol=1e-8)

    for t, e in zip(*np.nonzero(m)):
        assert dprobs[t, e] == pytest.approx(_fd(f, probs, (t, e)), rel=1e-6, abs=1e-8)
    assert np.all(dprobs[~m] == 0)
    for t, e in zip(*np.nonzero(~m)):           # off-map probs do not change the loss
        assert _fd(f, probs, (t, e)) == 0.0

    def check(arr, grad):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            fd[idx] = _fd(f, arr, idx)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)

    check(W.sg, grads["shared_gate"])
    check(W.su, grads["shared_up"])
    check(W.sd, grads["shared_down"])
    E = W.num_experts
    for e in range(E):
        if e in grads["routed"]:
            dWg, dWu, dWd = grads["routed"][e]
        else:
            dWg = np.zeros_like(W.rg[e]); dWu = np.zeros_like(W.ru[e]); dWd = np.zeros_like(W.rd[e])
        check(W.rg[e], dWg)
        check(W.ru[e], dWu)
        check(W.rd[e], dWd)


def test_worked_example_backward():
    ex, W = load_worked_example()
    _, cache = O.forward(np.array(ex["hidden"]), np.array(ex["probs"]),
                         np.array(ex["routing_map"], bool), W, ex["k"])
    dx, dprobs, g = O.backward(np.array(ex["grad_out"]), cache, W)
    e = ex["expected"]
    tol = dict(rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dx, eval_closed_form(e["dhidden"]), **tol)
    np.testing.assert_allclose(dprobs, eval_closed_form(e["dprobs"]), **tol)
    np.testing.assert_allclose(g["shared_down"], eval_closed_form(e["dW_shared_down"]), **tol)
    np.testing.assert_allclose(g["shared_gate"], eval_closed_form(e["dW_shared_gate"]), **tol)
    np.testing.assert_allclose(g["shared_up"], eval_closed_form(e["dW_shared_up"]), **tol)
    for ex_id in (0, 1):
        dWg, dWu, dWd = g["routed"][ex_id]
        np.testing.assert_allclose(dWg, eval_closed_form(e[f"dW_routed_gate_{ex_id}"]), **tol)
        np.testing.assert_allclose(dWu, eval_closed_form(e[f"dW_routed_up_{ex_id}"]), **tol)
        np.testing.assert_allclose(dWd, eval_closed_form(e[f"dW_routed_down_{ex_id}"]), **tol)


def test_main_grad_accumulation_and_idle_expert():
    W, x, go, m, probs, k = _tiny_case(3)
    _, cache = O.forward(x, probs, m, W, k)
    _, _, grads = O.backward(go, cache, W)
    rng = np.random.default_rng(5)
    E = W.num_experts
    mg = dict(shared_gate=rng.standard_normal(W.sg.shape), shared_up=rng.standard_normal(W.su.shape),
              shared_down=rng.standard_normal(W.sd.shape), routed_gate=rng.standard_normal(W.rg.shape),
              routed_up=rng.standard_normal(W.ru.shape), routed_down=rng.standard_normal(W.rd.shape))
    out = O.accumulate_main_grads(mg, grads)
    zero = {n: np.zeros_like(v) for n, v in mg.items()}
    dW = O.accumulate_main_grads(zero, grads)
    for n in mg:
        np.testing.assert_allclose(out[n], mg[n] + dW[n], rtol=1e-15, atol=1e-15)
    idle = E - 1
    assert idle not in grads["routed"]
    for n in ("routed_gate", "routed_up", "routed_down"):
        assert np.array_equal(out[n][idle], mg[n][idle])
    busy = next(iter(grads["routed"]))
    assert np.any(out["routed_gate"][busy] != mg["routed_gate"][busy])


def test_backward_tokens_are_independent():
    """dhidden and dprobs of a token depend only on that token (the sampled
    full-size checks rest on this)."""
    W, x, go, m, probs, k = _tiny_case(4, T=10)
    _, cache = O.forward(x, probs, m, W, k)
    dx, dp, _ = O.backward(go, cache, W)
    sub = np.array([1, 4, 9])
    _, cs = O.forward(x[sub], probs[sub], m[sub], W, k)
    dxs, dps, _ = O.backward(go[sub], cs, W)
    np.testing.assert_allclose(dxs, dx[sub], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dps, dp[sub], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- swiglu_limit clamp and shared output gate
def _gated_case(seed, limit):
    W, x, go, m, probs, k = _tiny_case(seed)
    rng = np.random.default_rng(100 + seed)
    W.shared_output_gate = rng.standard_normal(x.shape[1]) * 0.5
    # the clamp must be active somewhere and no input may sit within reach of
    # a finite-difference step of a clamp bound
    gs = []
    for Wg, Wu in [(W.sg, W.su)] + [(W.rg[e], W.ru[e]) for e in range(W.num_experts)]:
        gs.append((x @ Wg.T, x @ Wu.T))
    g_all = np.concatenate([g.ravel() for g, _ in gs])
    u_all = np.concatenate([u.ravel() for _, u in gs])
    assert np.any(g_all > limit) and np.any(np.abs(u_all) > limit) and np.any(g_all < limit)
    assert np.min(np.abs(g_all - limit)) > 1e-4 and np.min(np.abs(np.abs(u_all) - limit)) > 1e-4
    return W, x, go, m, probs, k


@pytest.mark.parametrize("seed", [0, 1])
def test_clamp_and_gate_match_finite_differences(seed):
    limit = 0.6
    W, x, go, m, probs, k = _gated_case(seed, limit)
    _, cache = O.forward(x, probs, m, W, k, swiglu_limit=limit)
    dx, dprobs, grads = O.backward(go, cache, W)

    def f():
        out, _ = O.forward(x, probs, m, W, k, swiglu_limit=limit)
        return float(np.sum(go * out))

    def check(arr, grad):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            fd[idx] = _fd(f, arr, idx)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)

    check(x, dx)
    for t, e in zip(*np.nonzero(m)):
        assert dprobs[t, e] == pytest.approx(_fd(f, probs, (t, e)), rel=1e-6, abs=1e-8)
    check(W.shared_output_gate, grads["shared_output_gate"])
    check(W.sg, grads["shared_gate"])
    check(W.su, grads["shared_up"])
    check(W.sd, grads["shared_down"])
    for e, (dWg, dWu, dWd) in grads["routed"].items():
        check(W.rg[e], dWg)
        check(W.ru[e], dWu)
        check(W.rd[e], dWd)


def test_clamp_single_unit_by_hand():
    """H = I = 1, one token, one expert: g = 3 > L = 1 and u = -6 < -L, so
    a = silu(1) * (-1), and neither clamped input passes a gradient."""
    W = O.DenseWeights(np.zeros((1, 1)), np.zeros((1, 1)), np.zeros((1, 1)),
                       np.array([[[1.5]]]), np.array([[[-3.0]]]), np.array([[[2.0]]]))
    x = np.array([[2.0]])
    m = np.array([[True]])
    p = np.array([[0.25]])
    out, cache = O.forward(x, p, m, W, 1, swiglu_limit=1.0)
    a = -1.0 / (1.0 + np.exp(-1.0))                 # silu(1) * (-1)
    assert out[0, 0] == pytest.approx(0.25 * 2.0 * a, rel=1e-15)
    dx, dp, g = O.backward(np.array([[4.0]]), cache, W)
    assert dx[0, 0] == 0.0
    dWg, dWu, dWd = g["routed"][0]
    assert dWg[0, 0] == 0.0 and dWu[0, 0] == 0.0
    assert dWd[0, 0] == pytest.approx(4.0 * 0.25 * a, rel=1e-15)
    assert dp[0, 0] == pytest.approx(4.0 * 2.0 * a, rel=1e-15)


def test_large_limit_changes_nothing():
    W, x, go, m, probs, k = _tiny_case(5)
    out0, c0 = O.forward(x, probs, m, W, k)
    out1, c1 = O.forward(x, probs, m, W, k, swiglu_limit=1e6)
    assert np.array_equal(out0, out1)
    d0 = O.backward(go, c0, W)
    d1 = O.backward(go, c1, W)
    assert np.array_equal(d0[0], d1[0]) and np.array_equal(d0[1], d1[1])


def test_zero_gate_weight_halves_the_shared_expert():
    """w = 0: gate = 1/2 for every token; the gate weight's gradient is
    x^T (1/4 <go, y_shared>), with y_shared the ungated shared expert."""
    W, x, go, m, probs, k = _tiny_case(6)
    out_u, _ = O.forward(x, probs, m, W, k)
    _, _, _, ys = O.expert_forward(x, *W.shared())
    W.shared_output_gate = np.zeros(x.shape[1])
    out_g, cache = O.forward(x, probs, m, W, k)
    np.testing.assert_allclose(out_g, out_u - 0.5 * ys, rtol=1e-13, atol=1e-13)
    _, _, grads = O.backward(go, cache, W)
    np.testing.assert_allclose(grads["shared_output_gate"], x.T @ (0.25 * np.sum(go * ys, axis=1)),
                               rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- BF16 main_grad accumulation
def test_bf16_main_grad_rounds_the_contribution_then_the_sum():
    """bf16(mg + bf16(dW)) by hand (bf16: 8 significant bits, ulp(1) = 2^-7):
    * dW = 2^-8 (exact in bf16): 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even, 1;
    * dW = 3 2^-8: 1 + 1.5 2^-7 is a tie -> even mantissa, 1 + 2^-6;
    * dW = 2^-8 + 2^-20 rounds to 2^-8 first, so the sum is the tie of the first
      case (1), where rounding the exact sum once would give 1 + 2^-7;
    * dW = -3 (exact): 1 - 3 = -2 exactly."""
    mg = {n: np.ones((1, 4)) for n in ("shared_gate", "shared_up", "shared_down")}
    mg.update({n: np.ones((1, 1, 4)) for n in ("routed_gate", "routed_up", "routed_down")})
    dW = np.array([[2.0 ** -8, 3 * 2.0 ** -8, 2.0 ** -8 + 2.0 ** -20, -3.0]])
    grads = dict(shared_gate=dW, shared_up=dW, shared_down=dW, routed={0: (dW, dW, dW)})
    out = O.accumulate_main_grads(mg, grads, dtype="bf16")
    want = np.array([[1.0, 1.0 + 2.0 ** -6, 1.0, -2.0]])
    for n in ("shared_gate", "shared_up", "shared_down"):
        np.testing.assert_array_equal(out[n], want)
    for n in ("routed_gate", "routed_up", "routed_down"):
        np.testing.assert_array_equal(out[n][0], want)
    single = O.bf16_round(1.0 + dW)                          # one rounding of the exact sum
    assert single[0, 2] == 1.0 + 2.0 ** -7 and out["shared_gate"][0, 2] == 1.0
    fp32 = O.accumulate_main_grads(mg, grads)                  # the fp32 path adds exactly
    np.testing.assert_array_equal(fp32["shared_gate"], 1.0 + dW)


def test_bf16_main_grad_matches_torch_bf16_arithmetic():
    import torch
    rng = np.random.default_rng(9)
    mg0 = torch.from_numpy(rng.standard_normal(4096).astype(np.float32) * 1e-3).to(torch.bfloat16)
    dW = rng.standard_normal(4096) * 10.0 ** rng.integers(-5, 1, 4096)
    dW32 = torch.from_numpy(dW.astype(np.float32))
    ref = (mg0.float() + dW32.to(torch.bfloat16).float()).to(torch.bfloat16).double().numpy()
    mg = {n: mg0.double().numpy().reshape(1, -1) for n in ("shared_gate", "shared_up", "shared_down")}
    mg.update({n: mg0.double().numpy().reshape(1, 1, -1) for n in ("routed_gate", "routed_up", "routed_down")})
    d = dW32.double().numpy().reshape(1, -1)
    out = O.accumulate_main_grads(mg, dict(shared_gate=d, shared_up=d, shared_down=d, routed={}), dtype="bf16")
    np.testing.assert_array_equal(out["shared_gate"][0], ref)
