"""Plain fp64 CPU oracle of the post-router MoE layer, forward and backward.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import or call anything under ``oracle/``. The
product path (the CUDA library and its Python binding) never does, and shares
no code, table or helper with it.

What the layer computes (sources, by page and section):

* "feat(moe): add a megakernel backend with MOK integration" (Megatron-LM PR
  #6572), Summary: the backend replaces the post-router path -- dispatch,
  routed and shared expert computation, combine.
* same page, Design > Authoritative routing maps: the dense routing map is
  turned into a fixed-width top-k representation, missing routes carry expert
  id -1, the matching probabilities are gathered; in backward the router-weight
  gradients go back into the dense probability tensor.
* same page, Design > Gradient accumulation, and "Add Mixture-of-Kittens MoE
  backend on main" (PR #8210), review thread on wgrad precision: expert weight
  gradients are accumulated into fp32 main_grad buffers (fused accumulation).
* same page #6572, Supported configurations > limitations: routed and shared
  experts share one intermediate size; shared expert BF16, no output gate.
* "core.transformer.moe.megakernel.mok.runtime", _gate_up_weight_arguments and
  _MoKWeightArguments: FC1 is a combined [2I, H] weight, rows [0,I) gate and
  [I,2I) up; argument order shared gate/up/down, routed gate/up/down.
* "core.transformer.moe.megakernel.mok.backend", MoKMegakernel.forward:
  out = layer(hidden[T,H], probs[T,E], routing_map[T,E]) with hidden's shape.

Two optional inputs the pages name without a formula, read as follows:

* ``swiglu_limit`` ("Add Mixture-of-Kittens MoE backend on main", review thread
  on the backend's swiglu_limit = the layer's activation clamp value): L > 0
  clamps the SwiGLU inputs of every expert, a = silu(min(g, L)) * clip(u, -L, L);
  the gradient passes where the clamp is inactive, bounds included.
* the shared expert's output gate ("core.transformer.moe.megakernel.mok.runtime",
  _MoKAutograd.forward: shared_output_gate_weight): a per-token scalar
  gate[t] = sigmoid(x_t . w) multiplies the shared expert's output.

Readings where the pages are silent (each also listed in the design notes):
the expert is a SwiGLU MLP, a = silu(x W_g^T) * (x W_u^T), y = a W_d^T with
silu(z) = z / (1 + e^-z); the prob weights the expert output after the down
projection; slots list a token's experts in ascending id order, -1 padding at
the tail; a row with more than k routes is an error, not truncated; a routed
(t, e) with prob 0 is still computed; probs off the map are ignored and get
gradient 0; within an expert, routes are ordered by token index.

Precision. The pages fix the weights (BF16, or MXFP8 routed experts: PR
#6572, Supported configurations), the FP32 GEMM accumulator and the FP32
main_grad accumulation (PR #8210, review thread on wgrad precision).
``precision="exact"`` is the plain definition in fp64, nothing rounded.
``precision="mxfp8"`` is the MXFP8 method on top of it: the routed experts'
forward and dgrad GEMM operands are quantised to MXFP8 on the fly, in blocks
of 32 along each GEMM's K -- x and a in forward, grad_out and [dg|du] in
dgrad -- with the weights given dequantised (rowwise for forward, columnwise
for dgrad through ``routed_dgrad``); nothing else is rounded (the dprob and
the weight gradients take the unquantised a, dg, du, as a backward through a
quantiser that passes gradients straight through does). ``precision="bf16"``
is a diagnostic mode for a layer that stores its activations in bf16: every
tensor a BF16 expert passes on is rounded to bf16 -- the gate/up projections
g and u (kept for backward), the activation a between the two projections,
the expert's output y (the prob, or the shared expert's gate, weights it in
the fp32 combine), the SwiGLU gradients dg and du, the prob-weighted
activation p*a that multiplies grad_out in the down projection's weight
gradient, and the expert's input gradient dx (summed in fp32 by the
un-permute); products accumulate in fp64. Inputs (hidden, grad_out, weights)
are bf16 already.

A bf16 rounding is a discrete decision taken on a value the kernel evaluates
in fp32 (FP32 accumulator), so near a rounding midpoint both neighbours are
correct results. ``envelope`` (bf16 mode) bounds, per output element, how far
the other valid roundings of every operand that lies within the fp32
evaluation band of a midpoint can move the result (propagated with absolute
values); elsewhere it is 0. The same holds for the swiglu_limit clamp's
gradient masks, which jump at the clamp bounds: ``clamp_jumps`` (any mode)
bounds the effect of the other mask value where g or |u| lies within its
fp32 evaluation band of the bound.

Everything here is fp64 numpy; ``@`` (a BLAS matmul) is the only library step.
"""
from __future__ import annotations

import numpy as np


class RoutingError(ValueError):
    """A token row of the routing map has more than k routes."""


# --------------------------------------------------------------------------
# weights: the six-argument order shared gate/up/down, routed gate/up/down
# --------------------------------------------------------------------------
class DenseWeights:
    """fp64 weights held in memory: Wg, Wu [I,H] (per expert [E,I,H]), Wd [H,I]."""

    def __init__(self, shared_gate, shared_up, shared_down, routed_gate, routed_up, routed_down,
                 shared_output_gate=None):
        self.sg, self.su, self.sd = (np.asarray(a, np.float64) for a in (shared_gate, shared_up, shared_down))
        self.rg, self.ru, self.rd = (np.asarray(a, np.float64) for a in (routed_gate, routed_up, routed_down))
        # optional [H] output gate of the shared expert (None: ungated)
        self.shared_output_gate = None if shared_output_gate is None else np.asarray(shared_output_gate, np.float64)

    @classmethod
    def from_combined(cls, shared_fc1, shared_fc2, routed_fc1, routed_fc2):
        """Split combined FC1 [.., 2I, H] into gate rows [0,I) and up rows [I,2I)
        ("core.transformer.moe.megakernel.mok.runtime", _gate_up_weight_arguments)."""
        inter = shared_fc1.shape[0] // 2
        return cls(shared_fc1[:inter], shared_fc1[inter:], shared_fc2,
                   routed_fc1[:, :inter], routed_fc1[:, inter:], routed_fc2)

    @property
    def num_experts(self):
        return self.rg.shape[0]

    def shared(self):
        return self.sg, self.su, self.sd

    def routed(self, e):
        return self.rg[e], self.ru[e], self.rd[e]

    def routed_dgrad(self, e):
        """Weights the dgrad GEMMs see (MXFP8: the columnwise-quantised copy)."""
        return self.routed(e)


# --------------------------------------------------------------------------
# routing: dense map -> fixed-width ids, then per-expert segments
# --------------------------------------------------------------------------
def route_pack(routing_map, probs, k):
    """Dense routing_map[T,E] -> ids[T,k] (ascending expert ids, -1 padding) and
    pp[T,k] (the probs at those ids, 0 for -1); ``over[t]`` marks rows with > k
    routes. PR #6572, Design > Authoritative routing maps."""
    routing_map = np.asarray(routing_map, bool)
    probs = np.asarray(probs, np.float64)
    T = routing_map.shape[0]
    ids = np.full((T, k), -1, np.int32)
    pp = np.zeros((T, k), np.float64)
    over = np.zeros(T, bool)
    for t in range(T):
        experts = np.flatnonzero(routing_map[t])
        if experts.size > k:
            over[t] = True
            continue
        ids[t, :experts.size] = experts
        pp[t, :experts.size] = probs[t, experts]
    return ids, pp, over


def dispatch_indices(ids, num_experts):
    """Dispatch on one GPU = a local permutation (PR #6572, Summary: dispatch).

    Valid routes (t, s) are ordered by (expert, token). Returns counts[E],
    offsets[E+1] (exclusive scan), perm_src[R] (token of each permuted row),
    perm_slot[R] (its slot) and row_of[T,k] (permuted row of each slot, -1 for
    missing routes)."""
    T, k = ids.shape
    tok, slot = np.nonzero(ids >= 0)
    exp = ids[tok, slot]
    order = np.lexsort((tok, exp))          # primary key expert, then token
    perm_src = tok[order].astype(np.int64)
    perm_slot = slot[order].astype(np.int64)
    counts = np.bincount(exp, minlength=num_experts).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    row_of = np.full((T, k), -1, np.int64)
    row_of[perm_src, perm_slot] = np.arange(perm_src.size)
    return counts, offsets, perm_src, perm_slot, row_of


# --------------------------------------------------------------------------
# operand precision
# --------------------------------------------------------------------------
def bf16_round(x):
    """Round to the nearest bf16 value (8 significant bits), ties to even."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)                     # x = m * 2^e, |m| in [0.5, 1)
    return np.ldexp(np.round(m * 256.0), e - 8)   # np.round: half to even


U32 = 2.0 ** -24        # fp32 unit roundoff


def bf16_alternative(x, band):
    """Distance from bf16_round(x) to the other neighbour of x where x lies
    within ``band`` of a rounding midpoint (both roundings are then valid
    results of an fp32 evaluation of x), else 0."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    ulp = np.ldexp(1.0, e - 8)
    scaled = np.abs(m) * 256.0
    dist = np.abs(scaled - np.floor(scaled) - 0.5) * ulp
    return np.where(dist <= band, ulp, 0.0)


def fp32_dot_band(terms_sq_sum, K):
    """Evaluation band of an fp32-accumulated dot product of length K whose
    terms t have sum(t^2) = terms_sq_sum: 8 U32 sqrt(K) ||t||_2.

    Derivation. A sum accumulated in fp32 in any order carries the error
    sum_j delta_j S_j, S_j the partial sums, |delta_j| <= U32. Under the
    probabilistic model of Higham and Mary ("A New Approach to Probabilistic
    Rounding Error Analysis", SIAM J. Sci. Comput. 41(5), 2019: rounding
    errors independent, mean zero) its variance is at most
    U32^2 sum_j E[S_j^2] / 3; for terms of random sign E[S_j^2] = j ||t||^2 / K,
    so the standard deviation is at most U32 sqrt(K) ||t||_2 / sqrt(6). The
    band is ~20 of those (a tail probability far below 1e-50 for the bounded,
    independent sum). An accumulator that adds 16-term partial products with
    truncation has a bias instead, at most U32 |S_j| per addition on partial
    sums |S_j| ~ sqrt(16 j) rms(t): summed over the K/16 additions at most about
    3 U32 (K/16)^(3/2) rms(t) = 3 U32 sqrt(K) ||t||_2 sqrt(K) / 64, which stays
    below the band for K up to 16384 (the layer's longest reductions)."""
    return 8.0 * U32 * np.sqrt(K) * np.sqrt(terms_sq_sum)


ELEMENTWISE_BAND = 2.0 ** -20   # relative band of fp32 elementwise evaluation (exp, products)


def _rounder(precision):
    if precision in ("exact", "mxfp8"):
        return lambda v: v
    if precision == "bf16":
        return bf16_round
    raise ValueError(precision)


def mxfp8_round(v):
    """Value of v after MXFP8 quantisation in blocks of 32 along the last axis."""
    from oracle import mxfp8
    q, sc = mxfp8.quantize(v, axis=-1)
    return mxfp8.dequantize(q, sc, axis=-1)


class Operands:
    """Where one expert's GEMM operands are rounded: nowhere (exact); bf16
    everywhere (bf16 mode); or, for routed experts in mxfp8 mode, MXFP8 along K
    for the forward and dgrad GEMMs' activation operands only; and, in bf16 mode,
    the bf16 tensors between the expert's GEMMs and the layer's sums (``inter``:
    g, u, y, dx)."""

    def __init__(self, precision, routed=True):
        self.rnd = _rounder(precision)
        self.mx = precision == "mxfp8" and routed

    def inter(self, v):                   # g, u, y, dx: GEMM results (bf16 mode: stored in bf16)
        return self.rnd(v)

    def x(self, x):                       # gate/up projection input, K = H
        return mxfp8_round(x) if self.mx else x

    def a(self, a):                       # down projection input, K = I
        return mxfp8_round(a) if self.mx else self.rnd(a)

    def go(self, go):                     # dgrad through the down projection, K = H
        return mxfp8_round(go) if self.mx else go

    def dgdu(self, dg, du):               # dgrad through gate/up, K = 2I
        if self.mx:
            q = mxfp8_round(np.concatenate([dg, du], axis=1))
            return q[:, :dg.shape[1]], q[:, dg.shape[1]:]
        return self.rnd(dg), self.rnd(du)

    def wgrad(self, v):                   # weight-gradient operands
        return self.rnd(v)

    def kept_a(self, a_val, a_op):        # the a that the backward's dprob and p*a take
        return a_op if self.rnd is bf16_round else a_val


# --------------------------------------------------------------------------
# the expert MLP (SwiGLU) and its derivative
# --------------------------------------------------------------------------
def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def silu_grad(z):
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def clamp_inputs(g, u, limit):
    """SwiGLU inputs after the swiglu_limit clamp (limit 0: unclamped) and the
    masks where the gradient passes: min(g, L), clip(u, -L, L), g <= L, |u| <= L."""
    if not limit:
        one = np.ones_like(g)
        return g, u, one, one
    return (np.minimum(g, limit), np.clip(u, -limit, limit), (g <= limit).astype(np.float64),
            ((u >= -limit) & (u <= limit)).astype(np.float64))


def expert_forward(x, Wg, Wu, Wd, ops=None, limit=0.0):
    """SwiGLU expert on rows x[n,H]: g = x Wg^T, u = x Wu^T, a = silu(g) u, y = a Wd^T
    (``ops`` holds the GEMM operands x and a at the GEMM precision; ``limit`` the
    swiglu_limit clamp of g and u). Returns the unclamped g, u."""
    ops = ops or Operands("exact")
    xq = ops.x(x)
    g = ops.inter(xq @ Wg.T)
    u = ops.inter(xq @ Wu.T)
    gc, uc, _, _ = clamp_inputs(g, u, limit)
    a_val = silu(gc) * uc
    a_op = ops.a(a_val)
    y = ops.inter(a_op @ Wd.T)
    return g, u, ops.kept_a(a_val, a_op), y


def expert_backward(x, go, p, g, u, a, Wg, Wu, Wd, ops=None, limit=0.0):
    """Gradients of sum(go * (p y)) for one expert, p[n] the rows' probs, with the
    dgrad weights Wg, Wu, Wd: returns dx, dWg, dWu, dWd and dprob[n] =
    sum_i a_i (go Wd)_i (= <go, y> in exact arithmetic). ``ops`` holds every
    GEMM operand (go, [dg|du], and the weight-gradient operands dg, du, p*a)
    at its GEMM's precision; g, u are the unclamped SwiGLU inputs."""
    ops = ops or Operands("exact")
    gc, uc, mg, mu = clamp_inputs(g, u, limit)
    da_u = ops.go(go) @ Wd
    da = p[:, None] * da_u
    dg = da * uc * silu_grad(gc) * mg
    du = da * silu(gc) * mu
    dgq, duq = ops.dgdu(dg, du)
    dx = ops.inter(dgq @ Wg + duq @ Wu)
    dgw, duw = ops.wgrad(dg), ops.wgrad(du)
    dprob = np.sum(a * da_u, axis=1)
    return dx, dgw.T @ x, duw.T @ x, go.T @ ops.wgrad(p[:, None] * a), dprob


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------
def forward(hidden, probs, routing_map, W, k, precision="exact", swiglu_limit=0.0):
    """out[T,H] = gate[t] SwiGLU_shared(x) + sum over valid slots s of pp[t,s] * SwiGLU_{ids[t,s]}(x),
    gate[t] = sigmoid(x_t . w) with the shared output gate w (1 without it).

    "core.transformer.moe.megakernel.mok.backend", MoKMegakernel.forward, and PR
    #6572 Summary (dispatch, routed and shared experts, combine). Returns
    (out, cache); the cache feeds ``backward``."""
    shared_ops, routed_ops = Operands(precision, routed=False), Operands(precision)
    x = np.asarray(hidden, np.float64)
    T, H = x.shape
    ids, pp, over = route_pack(routing_map, probs, k)
    if over.any():
        raise RoutingError(f"{int(over.sum())} token rows have more than k={k} routes")
    E = W.num_experts
    counts, offsets, perm_src, perm_slot, row_of = dispatch_indices(ids, E)

    gs, us, as_, ys = expert_forward(x, *W.shared(), ops=shared_ops, limit=swiglu_limit)
    w_gate = getattr(W, "shared_output_gate", None)
    gate = None
    if w_gate is not None:
        gate = sigmoid(x @ w_gate)
        ys = gate[:, None] * ys

    R = perm_src.size
    y = np.zeros((R, H))
    routed = {}
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        xe = x[perm_src[lo:hi]]
        g, u, a, ye = expert_forward(xe, *W.routed(e), ops=routed_ops, limit=swiglu_limit)
        y[lo:hi] = ye
        routed[e] = (g, u, a)

    out = ys.copy()
    for s in range(k):                        # combine, in slot order
        v = ids[:, s] >= 0
        out[v] += pp[v, s, None] * y[row_of[v, s]]

    cache = dict(x=x, ids=ids, pp=pp, counts=counts, offsets=offsets, perm_src=perm_src,
                 perm_slot=perm_slot, row_of=row_of, shared=(gs, us, as_), y=y, routed=routed, k=k,
                 precision=precision, limit=swiglu_limit, gate=gate)
    return out, cache


def backward(grad_out, cache, W):
    """Gradients of L = sum(grad_out * out).

    Returns dhidden[T,H], dprobs[T,E] (dense: <grad_out_t, y_{t,e}> on routed
    (t,e), 0 elsewhere -- PR #6572, Design > Authoritative routing maps, the
    backward adapter) and the six weight gradients {shared_gate, shared_up,
    shared_down} plus {e: (dWg, dWu, dWd)} for every expert with tokens.
    "core.transformer.moe.megakernel.mok.runtime", _MoKAutograd.backward."""
    shared_ops, routed_ops = Operands(cache["precision"], routed=False), Operands(cache["precision"])
    go = np.asarray(grad_out, np.float64)
    x, ids, pp, row_of = cache["x"], cache["ids"], cache["pp"], cache["row_of"]
    offsets, perm_src, perm_slot = cache["offsets"], cache["perm_src"], cache["perm_slot"]
    T, H = x.shape
    E = W.num_experts

    limit, gate = cache["limit"], cache["gate"]
    gs, us, as_ = cache["shared"]
    p_s = np.ones(T) if gate is None else gate
    dx_s, dWsg, dWsu, dWsd, dgate = expert_backward(x, go, p_s, gs, us, as_, *W.shared(), ops=shared_ops,
                                                    limit=limit)
    dW_gate = None
    if gate is not None:                      # d/dz of gate * y_s, z = x . w
        dz = gate * (1.0 - gate) * dgate
        dx_s = dx_s + dz[:, None] * W.shared_output_gate[None, :]
        dW_gate = x.T @ dz

    R = perm_src.size
    dx_perm = np.zeros((R, H))
    dprob_perm = np.zeros(R)
    routed_grads = {}
    pp_perm = pp[perm_src, perm_slot] if R else np.zeros(0)
    for e, (g, u, a) in cache["routed"].items():
        lo, hi = offsets[e], offsets[e + 1]
        go_e = go[perm_src[lo:hi]]
        dx, dWg, dWu, dWd, dprob_perm[lo:hi] = expert_backward(x[perm_src[lo:hi]], go_e, pp_perm[lo:hi], g, u, a,
                                                              *W.routed_dgrad(e), ops=routed_ops, limit=limit)
        dx_perm[lo:hi] = dx
        routed_grads[e] = (dWg, dWu, dWd)

    dhidden = dx_s.copy()
    dprobs = np.zeros((T, E))
    for s in range(cache["k"]):               # un-permute reduce, in slot order
        v = ids[:, s] >= 0
        dhidden[v] += dx_perm[row_of[v, s]]
        dprobs[np.flatnonzero(v), ids[v, s]] = dprob_perm[row_of[v, s]]

    grads = dict(shared_gate=dWsg, shared_up=dWsu, shared_down=dWsd, routed=routed_grads)
    if dW_gate is not None:
        grads["shared_output_gate"] = dW_gate
    return dhidden, dprobs, grads


def accumulate_main_grads(main_grads, grads, dtype="fp32"):
    """Fused accumulation (PR #6572, Design > Gradient accumulation). ``main_grads``
    holds shared_gate/up/down [I,H]/[I,H]/[H,I] and routed_gate/up/down [E,..]
    (and shared_output_gate [H] when present); experts with no tokens are left
    as they are.

    dtype "fp32": main_grad <- main_grad + dW, in fp64 (PR #8210 review: the
    fp32 accumulator stays fp32 through the reduction-store). dtype "bf16"
    (same review: with BF16 main_grad each contribution is rounded to BF16
    before the BF16 reduction-store): main_grad <- bf16(main_grad + bf16(dW)),
    both roundings to nearest even, the sum exact before its rounding."""
    if dtype not in ("fp32", "bf16"):
        raise ValueError(dtype)

    def add(m, d):
        return m + d if dtype == "fp32" else bf16_round(m + bf16_round(d))

    out = {name: np.array(v, np.float64, copy=True) for name, v in main_grads.items()}
    for n in ("shared_gate", "shared_up", "shared_down", "shared_output_gate"):
        if n in grads:
            out[n] = add(out[n], grads[n])
    for e, (dWg, dWu, dWd) in grads["routed"].items():
        out["routed_gate"][e] = add(out["routed_gate"][e], dWg)
        out["routed_up"][e] = add(out["routed_up"][e], dWu)
        out["routed_down"][e] = add(out["routed_down"][e], dWd)
    return out



def silu_grad2_bound():
    """max |d^2 silu / dz^2| over the reals (about 0.5)."""
    return 0.5


def _expert_envelope(x, go, p, g, u, Wf, Wb, limit=0.0, p_band=None):
    """bf16-mode envelopes of one expert's results for rows x[n,H] with probs
    p[n]. Wf are the forward weights (Wg, Wu, Wd), Wb the dgrad weights; g, u the
    mode's (bf16) gate/up values; ``limit`` the swiglu_limit clamp; ``p_band`` a
    bound on the kernel's error in p (the shared output gate, which the kernel
    evaluates in fp32; None: p is exact).

    Every bf16 tensor is a rounding of a value the kernel evaluates
    in fp32. Where that value lies within its evaluation band of a rounding
    midpoint, the other neighbour is also a correct result; the difference it
    makes is carried forward with absolute values (a change below a later
    rounding's distance to its midpoint is absorbed by it, a larger one may
    flip it in turn). Returns env_y [n,H] (the expert's output y), env_dx
    [n,H], env_dWg [I,H], env_dWu [I,H], env_dWd [H,I], env_dprob [n]."""
    ops = Operands("bf16")
    Wg, Wu, Wd = Wf
    Bg, Bu, Bd = Wb
    xq = x
    H = x.shape[1]
    I = g.shape[1]
    p_band = np.zeros_like(p) if p_band is None else p_band
    # g, u: fp32 GEMM results rounded to bf16
    g_raw, u_raw = xq @ Wg.T, xq @ Wu.T
    alt_g = bf16_alternative(g_raw, fp32_dot_band((xq * xq) @ (Wg * Wg).T, H))
    alt_u = bf16_alternative(u_raw, fp32_dot_band((xq * xq) @ (Wu * Wu).T, H))
    gc, uc, mg, mu = clamp_inputs(g, u, limit)
    s1 = silu_grad(gc)
    a_val = silu(gc) * uc
    # a: elementwise fp32 math on g, u, then rounded; a flipped g or u moves it by
    # the slopes (a is continuous across the clamp bounds)
    flip_a = np.abs(s1 * uc) * alt_g + np.abs(silu(gc)) * alt_u
    band_a = ELEMENTWISE_BAND * np.abs(a_val) + flip_a
    alt_a = bf16_alternative(a_val, band_a) + flip_a
    a_b = ops.a(a_val)
    # y = bf16(a_b Wd^T)
    ey_pre = alt_a @ np.abs(Wd).T
    band_y = fp32_dot_band((a_b * a_b) @ (Wd * Wd).T, I) + ey_pre
    env_y = ey_pre + bf16_alternative(a_b @ Wd.T, band_y)

    goq = go
    da_u = goq @ Bd
    env_dprob = np.sum(alt_a * np.abs(da_u), axis=1)
    da = p[:, None] * da_u
    dda = (np.abs(p)[:, None] * fp32_dot_band((goq * goq) @ (Bd * Bd), H) +
           p_band[:, None] * np.abs(da_u))
    dg_val = da * uc * s1 * mg
    du_val = da * silu(gc) * mu
    # changes of dg, du from a flipped g or u (not absorbed: comparable to their ulp)
    flip_dg = (np.abs(da * s1) * alt_u + np.abs(da * uc) * silu_grad2_bound() * alt_g) * mg
    flip_du = np.abs(da * s1) * alt_g * mu
    band_dg = (np.abs(uc * s1) * dda + ELEMENTWISE_BAND * np.abs(dg_val)) * mg + flip_dg
    band_du = (np.abs(silu(gc)) * dda + ELEMENTWISE_BAND * np.abs(du_val)) * mu + flip_du
    # the clamp's masks jump at its bounds: where g or |u| lies within one bf16
    # ulp of L, its rounding (either neighbour) may fall on either side of L,
    # and the whole unmasked value is an alternative -- between the kernel and
    # this mode, and between this mode and the unrounded definition
    jump_dg = jump_du = 0.0
    if limit:
        ulp = lambda v: np.ldexp(1.0, np.frexp(v)[1] - 8)  # noqa: E731
        near_g = np.abs(g_raw - limit) <= ulp(g_raw)
        near_u = np.abs(np.abs(u_raw) - limit) <= ulp(u_raw)
        jump_dg = np.where(near_g, np.abs(da * uc * s1), 0.0)
        jump_du = np.where(near_u, np.abs(da * silu(gc)), 0.0)
    alt_dg = bf16_alternative(dg_val, band_dg) + flip_dg + jump_dg   # dgrad and weight-gradient operands
    alt_du = bf16_alternative(du_val, band_du) + flip_du + jump_du
    edx_pre = alt_dg @ np.abs(Bg) + alt_du @ np.abs(Bu)
    # dx = bf16(dg Bg + du Bu)
    dgq, duq = ops.dgdu(dg_val, du_val)
    band_dx = fp32_dot_band((dgq * dgq) @ (Bg * Bg) + (duq * duq) @ (Bu * Bu), 2 * I) + edx_pre
    env_dx = edx_pre + bf16_alternative(dgq @ Bg + duq @ Bu, band_dx)
    env_dWg = alt_dg.T @ np.abs(x)
    env_dWu = alt_du.T @ np.abs(x)

    pa_val = p[:, None] * a_b
    alt_pa = bf16_alternative(pa_val, 2 * U32 * np.abs(pa_val) + p_band[:, None] * np.abs(a_b))
    alt_pa = alt_pa + np.where(alt_a > 0, np.abs(p)[:, None] * alt_a + np.ldexp(1.0, np.frexp(pa_val)[1] - 8), 0.0)
    env_dWd = np.abs(go).T @ alt_pa
    return env_y, env_dx, env_dWg, env_dWu, env_dWd, env_dprob


def envelope(grad_out, cache, W):
    """Per-element envelopes of out, dhidden, dprobs and the six weight
    gradients for a bf16-mode forward/backward (see the module notes)."""
    go = np.asarray(grad_out, np.float64)
    if cache["precision"] != "bf16":
        raise ValueError("the rounding envelope is defined for the bf16 mode")
    x, ids, pp, row_of = cache["x"], cache["ids"], cache["pp"], cache["row_of"]
    offsets, perm_src, perm_slot = cache["offsets"], cache["perm_src"], cache["perm_slot"]
    T, H = x.shape
    E = W.num_experts
    gs, us, _ = cache["shared"]
    limit, gate = cache["limit"], cache["gate"]
    if gate is None:
        p_s, p_band = np.ones(T), None
    else:                                  # the kernel's fp32 logit and sigmoid
        w_gate = W.shared_output_gate
        z_band = fp32_dot_band((x * x) @ (w_gate * w_gate), H)
        p_band = gate * (1.0 - gate) * z_band + ELEMENTWISE_BAND * gate
        p_s = gate
    ey_s, edx_s, eg_s, eu_s, ed_s, edg = _expert_envelope(x, go, p_s, gs, us, W.shared(), W.shared(),
                                                          limit=limit, p_band=p_band)
    env_gate = None
    if gate is not None:
        ey_s = gate[:, None] * ey_s
        env_dz = gate * (1.0 - gate) * edg
        edx_s = edx_s + env_dz[:, None] * np.abs(W.shared_output_gate)[None, :]
        env_gate = np.abs(x).T @ env_dz
    R = perm_src.size
    ey = np.zeros((R, H))
    edx = np.zeros((R, H))
    edp = np.zeros(R)
    pp_perm = pp[perm_src, perm_slot] if R else np.zeros(0)
    routed = {}
    for e, (g, u, _) in cache["routed"].items():
        lo, hi = offsets[e], offsets[e + 1]
        ey[lo:hi], edx[lo:hi], eg, eu, ed, edp[lo:hi] = _expert_envelope(
            x[perm_src[lo:hi]], go[perm_src[lo:hi]], pp_perm[lo:hi], g, u, W.routed(e), W.routed_dgrad(e),
            limit=limit)
        routed[e] = (eg, eu, ed)
    env_out = ey_s.copy()
    env_dh = edx_s.copy()
    env_dp = np.zeros((T, E))
    for s in range(cache["k"]):
        v = ids[:, s] >= 0
        r = row_of[v, s]
        env_out[v] += np.abs(pp[v, s, None]) * ey[r]
        env_dh[v] += edx[r]
        env_dp[np.flatnonzero(v), ids[v, s]] = edp[r]
    env = dict(out=env_out, dhidden=env_dh, dprobs=env_dp, shared_gate=eg_s, shared_up=eu_s,
               shared_down=ed_s, routed=routed)
    if env_gate is not None:
        env["shared_output_gate"] = env_gate
    return env


def _expert_clamp_jumps(x, go, p, Wf, Wb, ops, limit):
    """One expert's bounds on the effect of the clamp's other gradient mask where
    the fp32 evaluation of g = x Wg^T or u = x Wu^T lies within its band
    (``fp32_dot_band``) of the bound L (g) or of +-L (u): there either mask value
    is a correct result. Returns (env_dx [n,H], env_dWg [I,H], env_dWu [I,H])."""
    Wg, Wu, _ = Wf
    Bg, Bu, Bd = Wb
    H = x.shape[1]
    xq = ops.x(x)
    g, u = xq @ Wg.T, xq @ Wu.T
    near_g = np.abs(g - limit) <= fp32_dot_band((xq * xq) @ (Wg * Wg).T, H)
    near_u = np.abs(np.abs(u) - limit) <= fp32_dot_band((xq * xq) @ (Wu * Wu).T, H)
    gc, uc, _, _ = clamp_inputs(g, u, limit)
    da = p[:, None] * (ops.go(go) @ Bd)
    jump_dg = np.where(near_g, np.abs(da * uc * silu_grad(gc)), 0.0)
    jump_du = np.where(near_u, np.abs(da * silu(gc)), 0.0)
    return jump_dg @ np.abs(Bg) + jump_du @ np.abs(Bu), jump_dg.T @ np.abs(x), jump_du.T @ np.abs(x)


def clamp_jumps(grad_out, cache, W):
    """Per-element bounds (same keys as ``envelope``; zero for out, dprobs and the
    down projections' weight gradients, which the masks do not reach) on how far
    the swiglu_limit clamp's other gradient mask moves dhidden and the gate/up
    weight gradients, for the SwiGLU inputs whose fp32 evaluation cannot tell
    which side of a clamp bound they lie on. The clamp itself is continuous, so
    the forward is unaffected. All zero without a clamp."""
    go = np.asarray(grad_out, np.float64)
    x, ids, pp, row_of = cache["x"], cache["ids"], cache["pp"], cache["row_of"]
    offsets, perm_src, perm_slot = cache["offsets"], cache["perm_src"], cache["perm_slot"]
    T, H = x.shape
    E = W.num_experts
    limit, gate = cache["limit"], cache["gate"]
    z = lambda a: np.zeros_like(a)  # noqa: E731
    Ws = W.shared()
    env = dict(out=np.zeros((T, H)), dhidden=np.zeros((T, H)), dprobs=np.zeros((T, E)), shared_gate=z(Ws[0]),
               shared_up=z(Ws[1]), shared_down=z(Ws[2]), routed={})
    if gate is not None:
        env["shared_output_gate"] = np.zeros(H)
    for e in cache["routed"]:
        Wr = W.routed(e)
        env["routed"][e] = (z(Wr[0]), z(Wr[1]), z(Wr[2]))
    if not limit:
        return env
    p_s = np.ones(T) if gate is None else gate
    env["dhidden"], env["shared_gate"], env["shared_up"] = _expert_clamp_jumps(
        x, go, p_s, Ws, Ws, Operands(cache["precision"], routed=False), limit)
    R = perm_src.size
    edx = np.zeros((R, H))
    pp_perm = pp[perm_src, perm_slot] if R else np.zeros(0)
    for e in cache["routed"]:
        lo, hi = offsets[e], offsets[e + 1]
        edx[lo:hi], eg, eu = _expert_clamp_jumps(x[perm_src[lo:hi]], go[perm_src[lo:hi]], pp_perm[lo:hi],
                                                 W.routed(e), W.routed_dgrad(e), Operands(cache["precision"]), limit)
        env["routed"][e] = (eg, eu, env["routed"][e][2])
    for s in range(cache["k"]):
        v = ids[:, s] >= 0
        env["dhidden"][v] += edx[row_of[v, s]]
    return env
