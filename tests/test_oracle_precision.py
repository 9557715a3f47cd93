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


def _fp32_layer(x, go, m, probs, W, k, mx=False, limit=0.0):
    """An independent fp32 evaluation of the layer (numpy float32 matmuls and
    elementwise math, bf16 rounding of the GEMM operands -- MXFP8 for the routed
    forward/dgrad operands when mx -- fp64 afterwards): stands in for any kernel
    that evaluates the operands in fp32. ``limit`` clamps the SwiGLU inputs;
    W.shared_output_gate (if set) gates the shared expert with an fp32 sigmoid."""
    from oracle import mxfp8 as MXC
    f32 = np.float32
    rnd = O.bf16_round

    def mxr(v):
        q, sc = MXC.quantize(np.asarray(v, np.float64), axis=-1)
        return MXC.dequantize(q, sc, axis=-1)

    def sig(z):
        return f32(1) / (f32(1) + np.exp(-z))

    def expert(xr, gor, p, Wg, Wu, Wd, quant):
        xq = mxr(xr) if quant else xr
        goq = mxr(gor) if quant else gor
        xr32, Wg32, Wu32, Wd32, go32 = (a.astype(f32) for a in (xq, Wg, Wu, Wd, goq))
        g = xr32 @ Wg32.T
        u = xr32 @ Wu32.T
        mg = mu = f32(1)
        if limit:
            L = f32(limit)
            mg = (g <= L).astype(f32)
            mu = ((u >= -L) & (u <= L)).astype(f32)
            g = np.minimum(g, L)
            u = np.clip(u, -L, L)
        s = sig(g)
        a = (mxr if quant else rnd)((g * s * u).astype(np.float64))
        y = p[:, None] * (a @ Wd.T)
        da_u = go32 @ Wd32
        dprob = np.sum(a.astype(f32) * da_u, axis=1).astype(np.float64)
        da = p.astype(f32)[:, None] * da_u
        dg32 = da * u * (s * (f32(1) + g * (f32(1) - s))) * mg
        du32 = da * (g * s) * mu
        dg, du = rnd(dg32.astype(np.float64)), rnd(du32.astype(np.float64))
        if quant:
            qq = mxr(np.concatenate([dg32, du32], axis=1).astype(np.float64))
            dx = qq[:, :dg.shape[1]] @ Wg + qq[:, dg.shape[1]:] @ Wu
        else:
            dx = dg @ Wg + du @ Wu
        pa = rnd((p.astype(f32)[:, None] * a.astype(f32)).astype(np.float64))
        return y, dx, dg.T @ xr, du.T @ xr, gor.T @ pa, dprob

    T = x.shape[0]
    w_gate = getattr(W, "shared_output_gate", None)
    gate = np.ones(T) if w_gate is None else sig(x.astype(f32) @ w_gate.astype(f32)).astype(np.float64)
    ys, dxs, gsg, gsu, gsd, dgate = expert(x, go, gate, *W.shared(), False)
    grads = dict(shared_gate=gsg, shared_up=gsu, shared_down=gsd)
    if w_gate is not None:
        dz = (gate * (1 - gate)).astype(f32) * dgate.astype(f32)
        dxs = dxs + (dz[:, None] * w_gate.astype(f32)[None, :]).astype(np.float64)
        grads["shared_output_gate"] = (x.astype(f32).T @ dz).astype(np.float64)
    out, dh = ys.copy(), dxs.copy()
    ids, pp, _ = O.route_pack(m, probs, k)
    routed = {}
    for e in range(W.num_experts):
        rows, slots = np.nonzero(ids == e)
        if rows.size == 0:
            continue
        y, dx, g1, g2, g3, _ = expert(x[rows], go[rows], pp[rows, slots], *W.routed(e), mx)
        out[rows] += y
        dh[rows] += dx
        routed[e] = (g1, g2, g3)
    grads["routed"] = routed
    return out, dh, grads


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_envelope_covers_fp32_evaluation(seed):
    rng = np.random.default_rng(seed)
    T, H, I, E, k = 192, 256, 256, 3, 2
    W = O.DenseWeights(*(rng.standard_normal(s) * 0.06 for s in
                         ((I, H), (I, H), (H, I), (E, I, H), (E, I, H), (E, H, I))))
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    go = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    m = np.zeros((T, E), bool)
    for t in range(T):
        m[t, rng.choice(E, 2, replace=False)] = True
    probs = rng.random((T, E)).astype(np.float32).astype(np.float64)
    out_b, cache = O.forward(x, probs, m, W, k, precision="bf16")
    dh_b, _, g_b = O.backward(go, cache, W)
    env = O.envelope(go, cache, W)
    out_f, dh_f, g_f = _fp32_layer(x, go, m, probs, W, k)

    def check(a, b, ev, name):
        slack = 1e-5 * np.abs(b).max()          # fp32 differences that flip nothing
        d = np.abs(a - b)
        assert np.all(d <= ev + slack), f"{name}: {np.sum(d > ev + slack)} outside the envelope"
        return np.sum(d > slack)

    flipped = check(out_f, out_b, env["out"], "out")
    flipped += check(dh_f, dh_b, env["dhidden"], "dhidden")
    for n in ("shared_gate", "shared_up", "shared_down"):
        flipped += check(g_f[n], g_b[n], env[n], n)
    for e, gs in g_f["routed"].items():
        for j, n in enumerate(("gate", "up", "down")):
            flipped += check(gs[j], g_b["routed"][e][j], env["routed"][e][j], f"routed {n}[{e}]")
    assert flipped > 0, "the fp32 evaluation flipped no rounding: the test would prove nothing"
    # the envelope mostly stays far below the tolerance floor (1e-3 max|ref|) it is added to
    for n, ref in (("out", out_b), ("dhidden", dh_b), ("shared_gate", g_b["shared_gate"])):
        sc = np.abs(ref).max()
        assert np.median(env[n]) < 2.5e-4 * sc and np.percentile(env[n], 99) < 1e-3 * sc, n
        assert env[n].max() < 5e-3 * sc, n


@pytest.mark.parametrize("seed", [21, 22])
def test_mxfp8_envelope_covers_fp32_evaluation(seed):
    """mxfp8 mode: an fp32 evaluation that quantises the routed forward/dgrad
    operands with the codec stays within the oracle's result plus its envelope."""
    rng = np.random.default_rng(seed)
    T, H, I, E, k = 256, 256, 256, 3, 2
    W = O.DenseWeights(*(rng.standard_normal(s) * 0.06 for s in
                         ((I, H), (I, H), (H, I), (E, I, H), (E, I, H), (E, H, I))))
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    go = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    m = np.zeros((T, E), bool)
    for t in range(T):
        m[t, rng.choice(E, 2, replace=False)] = True
    probs = rng.random((T, E)).astype(np.float32).astype(np.float64)
    out_b, cache = O.forward(x, probs, m, W, k, precision="mxfp8")
    dh_b, _, g_b = O.backward(go, cache, W)
    env = O.envelope(go, cache, W)
    out_f, dh_f, g_f = _fp32_layer(x, go, m, probs, W, k, mx=True)
    for a, b, ev, name in ((out_f, out_b, env["out"], "out"), (dh_f, dh_b, env["dhidden"], "dhidden")):
        slack = 1e-5 * np.abs(b).max()
        assert np.all(np.abs(a - b) <= ev + slack), name
    for e, gs in g_f["routed"].items():
        for j in range(3):
            b = g_b["routed"][e][j]
            assert np.all(np.abs(gs[j] - b) <= env["routed"][e][j] + 1e-5 * np.abs(b).max()), (e, j)


@pytest.mark.parametrize("seed", [31, 32])
def test_envelope_covers_fp32_evaluation_with_clamp_and_gate(seed):
    """bf16 mode with the swiglu_limit clamp active on a fifth of the SwiGLU
    inputs and a gated shared expert: an fp32 evaluation stays within the
    oracle's result plus its envelope (clamp bounds and the fp32 gate included)."""
    rng = np.random.default_rng(seed)
    T, H, I, E, k = 192, 256, 256, 3, 2
    limit = 0.8
    W = O.DenseWeights(*(rng.standard_normal(s) * 0.06 for s in
                         ((I, H), (I, H), (H, I), (E, I, H), (E, I, H), (E, H, I))),
                       shared_output_gate=torch.from_numpy(rng.standard_normal(H) * 0.06).to(torch.bfloat16)
                       .double().numpy())
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    go = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    m = np.zeros((T, E), bool)
    for t in range(T):
        m[t, rng.choice(E, 2, replace=False)] = True
    probs = rng.random((T, E)).astype(np.float32).astype(np.float64)
    out_b, cache = O.forward(x, probs, m, W, k, precision="bf16", swiglu_limit=limit)
    g_s, u_s, _ = cache["shared"]
    assert 0.05 < np.mean(g_s > limit) < 0.5 and 0.05 < np.mean(np.abs(u_s) > limit) < 0.6
    dh_b, _, g_b = O.backward(go, cache, W)
    env = O.envelope(go, cache, W)
    out_f, dh_f, g_f = _fp32_layer(x, go, m, probs, W, k, limit=limit)
    for a, b, ev, name in ((out_f, out_b, env["out"], "out"), (dh_f, dh_b, env["dhidden"], "dhidden"),
                           (g_f["shared_output_gate"], g_b["shared_output_gate"], env["shared_output_gate"], "gate")):
        slack = 1e-5 * np.abs(b).max()
        d = np.abs(a - b)
        assert np.all(d <= ev + slack), f"{name}: {np.sum(d > ev + slack)} outside the envelope"
    for n in ("shared_gate", "shared_up", "shared_down"):
        assert np.all(np.abs(g_f[n] - g_b[n]) <= env[n] + 1e-5 * np.abs(g_b[n]).max()), n
    for e, gs in g_f["routed"].items():
        for j in range(3):
            b = g_b["routed"][e][j]
            assert np.all(np.abs(gs[j] - b) <= env["routed"][e][j] + 1e-5 * np.abs(b).max()), (e, j)
