"""Shared test plumbing: run the CUDA layer through the C ABI on seeded inputs and
run the fp64 oracle on the same inputs. No layer arithmetic lives here.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import moe_inputs as MI
from oracle import moe_oracle as O


@dataclasses.dataclass
class Case:
    T: int
    H: int
    E: int
    k: int
    I: int
    seed: int
    routing: str = "topk"
    drop: str = "none"
    mx: bool = False      # MXFP8 routed weights
    limit: float = 0.0    # swiglu_limit
    gated: bool = False   # shared expert with an output gate
    mg_bf16: bool = False  # bf16 main_grad buffers
    act_bf16: bool = False  # bf16 activations (MOE_ACT_BF16) instead of the default fp32 ones


def config_case(cfg_id: int, T: int | None = None, variant: str | None = None) -> Case:
    c = MI.CONFIGS[cfg_id]
    return Case(T or c["T"], c["H"], c["E"], c["k"], c["I"], MI.seed_of(cfg_id), variant or c["routing"], c["drop"],
                c["routed"] == "mxfp8")


@dataclasses.dataclass
class Inputs:
    case: Case
    hidden: torch.Tensor       # bf16 [T,H] on device
    grad_out: torch.Tensor     # bf16 [T,H]
    probs: torch.Tensor        # f32 [T,E]
    routing_map: torch.Tensor  # bool [T,E]
    weights: dict              # combined-layout bf16 tensors
    main_grads: dict           # fp32 combined-layout buffers (initial values)
    probs_np: np.ndarray
    map_np: np.ndarray
    mx: dict = None            # MXFP8 routed weights: name -> (payload, scale, col payload, col scale)
    gate_w: object = None      # bf16 [H] shared output gate (gated cases)


def make_inputs(case: Case, device="cuda", routing=None) -> Inputs:
    r = routing or MI.make_routing(case.T, case.E, case.k, case.seed, case.routing, case.drop)
    w = MI.make_weights(case.H, case.I, case.E, case.seed, device=device)
    hidden, grad_out = MI.make_activations(case.T, case.H, case.seed, device=device)
    mg = MI.make_main_grads(case.H, case.I, case.E, case.seed, device=device)
    probs = torch.from_numpy(r.probs).to(device)
    rmap = torch.from_numpy(r.routing_map).to(device)
    mx = MI.make_mxfp8_weights(w) if case.mx else None
    gate_w = None
    if case.gated:
        gate_w, mg["shared_output_gate"] = MI.make_shared_output_gate(case.H, case.seed, device=device)
    if case.mg_bf16:
        mg = {n: t.to(torch.bfloat16) for n, t in mg.items()}
    return Inputs(case, hidden, grad_out, probs, rmap, w, mg, r.probs, r.routing_map, mx, gate_w)


def weight_views(inp: Inputs):
    """moe_weights of the inputs: bf16 combined-FC1 views, or MXFP8 routed views."""
    import mixture_experts_layer_pack_gb300 as M
    w = inp.weights
    wv = M.weights_from_combined(w["shared_fc1"], w["shared_fc2"], w["routed_fc1"], w["routed_fc2"], inp.gate_w)
    if inp.mx:
        I = inp.case.I
        q1, s1, c1, cs1 = inp.mx["routed_fc1"]
        wv.routed_gate = M.mxfp8_view(q1[:, :I], s1[:, :I], c1[:, :I], cs1[:, :I // 32])
        wv.routed_up = M.mxfp8_view(q1[:, I:], s1[:, I:], c1[:, I:], cs1[:, I // 32:])
        wv.routed_down = M.mxfp8_view(*inp.mx["routed_fc2"])
    return wv


@dataclasses.dataclass
class GpuResult:
    out: torch.Tensor
    dhidden: torch.Tensor
    dprobs: torch.Tensor
    main_grads: dict
    layer: object


def run_gpu(inp: Inputs, backward=True, main_grads=None, layer=None) -> GpuResult:
    import mixture_experts_layer_pack_gb300 as M
    c = inp.case
    if layer is None:
        layer = M.MoELayer(c.T, c.H, c.E, c.k, c.I, device=inp.hidden.device,
                           routed_wtype=M.binding.MOE_W_MXFP8 if c.mx else M.binding.MOE_W_BF16,
                           swiglu_limit=c.limit,
                           act_precision=M.binding.MOE_ACT_BF16 if c.act_bf16 else M.binding.MOE_ACT_FP32)
    wv = weight_views(inp)
    if c.mx:
        layer.prepare_weights(wv)
    out = layer.forward(inp.hidden, inp.probs, inp.routing_map.view(torch.uint8), wv)
    dh = dp = None
    mg = None
    if backward:
        mg = {n: t.clone() for n, t in (main_grads or inp.main_grads).items()}
        mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"],
                                         mg.get("shared_output_gate"))
        dh, dp = layer.backward(inp.grad_out, mgv)
    torch.cuda.synchronize()
    return GpuResult(out, dh, dp, mg, layer)


class TorchWeights:
    """Oracle weight accessor over device bf16 tensors: fp64 copies per expert."""

    def __init__(self, w: dict, gate_w=None):
        self.w = w
        self.I = w["shared_fc1"].shape[0] // 2
        self._shared = None
        self.shared_output_gate = None if gate_w is None else self._f64(gate_w)

    @property
    def num_experts(self):
        return self.w["routed_fc1"].shape[0]

    @staticmethod
    def _f64(t):
        return t.detach().to("cpu", torch.float64).numpy()

    def shared(self):
        if self._shared is None:
            fc1 = self._f64(self.w["shared_fc1"])
            self._shared = (fc1[:self.I], fc1[self.I:], self._f64(self.w["shared_fc2"]))
        return self._shared

    def routed(self, e):
        fc1 = self._f64(self.w["routed_fc1"][e])
        return fc1[:self.I], fc1[self.I:], self._f64(self.w["routed_fc2"][e])

    def routed_dgrad(self, e):
        return self.routed(e)


class TorchMxWeights(TorchWeights):
    """Oracle weight accessor for MXFP8 routed weights: the oracle codec's exact
    dequantisation of the input payloads (rowwise for forward, columnwise for
    dgrad); shared weights bf16."""

    def __init__(self, w: dict, mx: dict, gate_w=None):
        super().__init__(w, gate_w)
        self.mx = mx

    @property
    def num_experts(self):
        return self.mx["routed_fc1"][0].shape[0]

    @staticmethod
    def _deq(q, s, axis):
        from oracle import mxfp8
        return mxfp8.dequantize(q.cpu().numpy(), s.cpu().numpy(), axis=axis)

    def routed(self, e):
        q1, s1, _, _ = self.mx["routed_fc1"]
        q2, s2, _, _ = self.mx["routed_fc2"]
        fc1 = self._deq(q1[e], s1[e], 1)
        return fc1[:self.I], fc1[self.I:], self._deq(q2[e], s2[e], 1)

    def routed_dgrad(self, e):
        _, _, c1, cs1 = self.mx["routed_fc1"]
        _, _, c2, cs2 = self.mx["routed_fc2"]
        fc1 = self._deq(c1[e], cs1[e], 0)
        return fc1[:self.I], fc1[self.I:], self._deq(c2[e], cs2[e], 0)


def oracle_weights(inp: Inputs):
    return TorchMxWeights(inp.weights, inp.mx, inp.gate_w) if inp.mx else TorchWeights(inp.weights, inp.gate_w)


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_full(inp: Inputs, precision="exact"):
    """Oracle forward + backward over all tokens. The cache also carries the bf16
    mode's rounding envelope ("envelope", bf16 mode only) and the clamp's
    gradient-mask alternatives ("jumps", the other modes; zero without a clamp)."""
    W = oracle_weights(inp)
    out, cache = O.forward(f64(inp.hidden), inp.probs_np, inp.map_np, W, inp.case.k, precision=precision,
                           swiglu_limit=inp.case.limit)
    go = f64(inp.grad_out)
    dx, dprobs, grads = O.backward(go, cache, W)
    cache["envelope"] = O.envelope(go, cache, W) if precision == "bf16" else None
    cache["jumps"] = O.clamp_jumps(go, cache, W) if precision != "bf16" else None
    return out, dx, dprobs, grads, cache


# The BF16 tolerance read per element (|gpu - ref| <= rtol |ref| + atol max|ref|,
# max over the whole compared tensor), and the MXFP8 one.
BF16_TOL = dict(rtol=2e-2, atol_frac=1e-3)
MX_TOL = dict(rtol=6e-2, atol_frac=6e-3)


def assert_close(gpu, ref, name, rtol=2e-2, atol_frac=1e-3, env=None, scale=None):
    """Per element |gpu - ref| <= rtol*|ref| + atol_frac*max|ref| (the BF16 tolerance),
    plus ``env`` where given: the other valid results of a discrete decision taken
    in fp32 (the bf16 mode's rounding envelope, or the clamp's gradient-mask
    alternatives). ``scale`` overrides max|ref| (a sample of a larger tensor)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values in the CUDA result"
    if scale is None:
        scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = np.abs(gpu - ref)
    bound = rtol * np.abs(ref) + atol_frac * scale
    if env is not None:
        bound = bound + np.asarray(env, np.float64)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())}/{bad.size} elements out of tolerance; worst at {i}: "
                             f"gpu={gpu[i]:.6g} ref={ref[i]:.6g}; max|err|/max|ref|={err.max() / max(scale, 1e-300):.3g}")
    return float(err.max() / max(scale, 1e-300)) if ref.size else 0.0


def count_outside(gpu, ref, rtol, atol_frac, env=None):
    """(elements outside rtol |ref| + atol_frac max|ref| (+ env), worst err / bound)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    if not ref.size:
        return 0, 0.0
    bound = rtol * np.abs(ref) + atol_frac * np.max(np.abs(ref))
    if env is not None:
        bound = bound + np.asarray(env, np.float64)
    err = np.abs(gpu - ref)
    return int(np.sum(err > bound)), float(np.max(err / np.maximum(bound, 1e-300)))


# Normwise bound of the bf16-activation layer against the exact (fp64, unrounded)
# definition. Each of its results passes through at most three bf16 operand
# roundings of relative rms error ~1.7e-3 (unit roundoff 2^-8); the largest of
# millions of Gaussian-like errors is ~5.5 sigma, the largest |ref| at least ~4 rms,
# so max|err|/max|ref| stays below ~4e-3; 1e-2 leaves headroom without hiding a
# real fault (the routed weight gradients are compared as whole tensors, so an
# expert with a handful of tokens, whose few rounding errors do not average out,
# is measured against the largest gradient of any expert).
EXACT_NORMWISE = 1e-2


def assert_normwise(gpu, ref, name, bound=EXACT_NORMWISE, env=None):
    """max|gpu - ref| / max|ref| <= bound, after taking off the envelope ``env``
    of the valid alternative decisions where one is given (the swiglu_limit
    clamp's gradient mask jumps at its bounds: within fp32 precision of a bound
    either side is a correct result, and one such element moves dhidden by
    percents of its maximum)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    if scale == 0.0:
        assert np.all(gpu == 0), name
        return 0.0
    err = np.abs(gpu - ref)
    if env is not None:
        err = np.maximum(err - np.asarray(env, np.float64), 0.0)
    r = float(np.max(err) / scale)
    assert r <= bound, f"{name}: max|gpu-exact|/max|exact| = {r:.3g} > {bound}"
    return r


def _named(out, dx, dprobs, grads, I, routed_experts):
    """The layer's results by name; routed weight gradients as the whole
    [E', I, H] / [E', H, I] tensors over ``routed_experts`` (one main_grad buffer each)."""
    r = {"out": out, "dhidden": dx, "dprobs": dprobs, "dW shared gate": grads["shared_gate"],
         "dW shared up": grads["shared_up"], "dW shared down": grads["shared_down"]}
    if "shared_output_gate" in grads:
        r["dW shared output gate"] = grads["shared_output_gate"]
    if routed_experts:
        for j, kind in enumerate(("gate", "up", "down")):
            r[f"dW routed {kind}"] = np.stack([grads["routed"][e][j] for e in routed_experts])
    return r


def gpu_named(inp: Inputs, res: GpuResult, routed_experts):
    """The CUDA results in the layout of ``_named`` (main_grad updates as after - before)."""
    I = inp.case.I
    d = {n: f64(res.main_grads[n]) - f64(inp.main_grads[n]) for n in inp.main_grads}
    grads = dict(shared_gate=d["shared_fc1"][:I], shared_up=d["shared_fc1"][I:], shared_down=d["shared_fc2"],
                 routed={e: (d["routed_fc1"][e, :I], d["routed_fc1"][e, I:], d["routed_fc2"][e])
                         for e in routed_experts})
    if "shared_output_gate" in d:
        grads["shared_output_gate"] = d["shared_output_gate"]
    return _named(f64(res.out), f64(res.dhidden), f64(res.dprobs), grads, I, routed_experts)


def _env_named(env, routed_experts):
    if env is None:
        return {}
    r = {"out": env["out"], "dhidden": env["dhidden"], "dprobs": env["dprobs"], "dW shared gate": env["shared_gate"],
         "dW shared up": env["shared_up"], "dW shared down": env["shared_down"]}
    if "shared_output_gate" in env:
        r["dW shared output gate"] = env["shared_output_gate"]
    if routed_experts:
        for j, kind in enumerate(("gate", "up", "down")):
            r[f"dW routed {kind}"] = np.stack([env["routed"][e][j] for e in routed_experts])
    return r


def _normwise(a, r):
    scale = float(np.max(np.abs(r))) if np.size(r) else 0.0
    return float(np.max(np.abs(np.asarray(a) - r)) / scale) if scale > 0 else 0.0


def compare_layer(inp: Inputs, res: GpuResult, exact_counts=None, mx_exact_bound=True):
    """Every output and weight gradient of the CUDA layer against the oracle on the
    same inputs, element by element. Experts without tokens must keep their
    main_grad bitwise. Returns {name: max|gpu - ref| / max|ref|} against the exact
    oracle.

    * fp32 activations (the default), BF16 routed weights: against the exact
      definition, |gpu - ref| <= 2e-2 |ref| + 1e-3 max|ref|, no envelope (with a
      swiglu_limit, plus the clamp's gradient-mask alternatives at its bounds).
    * fp32 activations, MXFP8 routed weights: against the MXFP8 method (the
      oracle's mxfp8 mode: same dequantised weights, the four GEMM activation
      operands quantised) within 6e-2 |ref| + 6e-3 max|ref|, and against the
      exact definition on the same dequantised weights within
      max|gpu - ref| <= 6e-2 max|ref| (``mx_exact_bound``, the workloads' sizes);
      otherwise no further from it than the MXFP8 method itself is (the
      mxfp8-mode oracle's own distance x 1.05 + 1e-3, or 6e-2 if that is larger).
    * bf16 activations: against the bf16-mode oracle plus its rounding envelope
      within the BF16 tolerance (BF16 weights), and against the exact definition
      normwise (1e-2 BF16, 6e-2 MXFP8).
    ``exact_counts`` (a dict) receives, per tensor, the elements outside the per
    element tolerance against the exact definition and the worst err/bound."""
    c = inp.case
    I = c.I
    counts = inp.map_np.sum(0)
    experts = [int(e) for e in np.flatnonzero(counts > 0)]
    for e in np.flatnonzero(counts == 0):    # an expert with no tokens keeps its main_grad bitwise
        assert torch.equal(res.main_grads["routed_fc1"][e], inp.main_grads["routed_fc1"][e]), e
        assert torch.equal(res.main_grads["routed_fc2"][e], inp.main_grads["routed_fc2"][e]), e
    got = gpu_named(inp, res, experts)
    tol = MX_TOL if c.mx else BF16_TOL
    ex = oracle_full(inp, "exact")
    ref_x = _named(*ex[:4], I, experts)
    jumps = _env_named(ex[4]["jumps"], experts) if c.limit else {}
    errs = {}
    if not c.act_bf16:
        if c.mx:
            mx = oracle_full(inp, "mxfp8")
            ref_m = _named(*mx[:4], I, experts)
            jm = _env_named(mx[4]["jumps"], experts) if c.limit else {}
            for n, r in ref_m.items():
                errs["mxfp8-mode " + n] = assert_close(got[n], r, "mxfp8-mode " + n, env=jm.get(n), **tol)
        for n, r in ref_x.items():
            if c.mx:
                if mx_exact_bound:
                    errs[n] = assert_normwise(got[n], r, n, bound=tol["rtol"], env=jumps.get(n))
                else:
                    # no further from the exact definition than the MXFP8 method itself is
                    # (its own error grows on experts with few tokens, and with a clamp,
                    # whose masks follow the quantised SwiGLU inputs)
                    own = _normwise(ref_m[n], r)
                    errs[n] = assert_normwise(got[n], r, n, bound=max(tol["rtol"], 1.05 * own + 1e-3))
                    errs["mxfp8 method vs exact " + n] = own
            else:
                errs[n] = assert_close(got[n], r, n, env=jumps.get(n), **tol)
    else:
        if not c.mx:
            bf = oracle_full(inp, "bf16")
            env = _env_named(bf[4]["envelope"], experts)
            for n, r in _named(*bf[:4], I, experts).items():
                assert_close(got[n], r, "bf16-mode " + n, env=env[n], **tol)
        for n, r in ref_x.items():
            errs[n] = assert_normwise(got[n], r, n, bound=tol["rtol"] if c.mx else EXACT_NORMWISE,
                                      env=jumps.get(n))
    if exact_counts is not None:
        for n, r in ref_x.items():
            exact_counts[n] = count_outside(got[n], r, tol["rtol"], tol["atol_frac"], env=jumps.get(n))
    return errs
