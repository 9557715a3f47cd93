#!/usr/bin/env python
"""MoE layer forward+backward throughput on GB300 (tokens/s, useful TFLOPS, roofline).

One step = one forward and one backward of the whole layer (route-pack,
dispatch, routed and shared SwiGLU experts, combine; dgrad, dense dprobs,
fused fp32 main_grad accumulation) over one batch of seeded synthetic input,
through the library's C ABI. Default workload: the Proxy-like layer, T=4096
tokens, H=2048, 96 routed experts top-6, one shared expert, I=1024, BF16.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N>1 runs one independent replica per GPU (launched by torch.distributed.run);
the layer has no exchange step on one GPU. `--impl reference` times the fp64
CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd tokens/s and TFLOPS, % of GB300 BF16/MXFP8 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--config", type=int, default=2)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--main-grad-dtype", choices=("fp32", "bf16"), default="fp32",
                   help="dtype of the main_grad buffers the backward accumulates into")
    p.add_argument("--act-precision", choices=("fp32", "bf16"), default="fp32",
                   help="activations between the expert GEMMs (include/moe.h, moe_act)")
    p.add_argument("--per-config", default="3,4,5",
                   help="further workloads measured after the headline one (comma list; empty: none)")
    p.add_argument("--per-config-steps", type=int, default=10)
    p.add_argument("--act-variant", type=int, default=1,
                   help="also time the headline workload with the other activation precision (0: skip)")
    p.add_argument("--ep-owner", type=int, default=16,
                   help="also time the expert-parallel owner step of the headline workload at this EP degree "
                        "(0: skip)")
    p.add_argument("--experts", type=int, default=0,
                   help="a reduced instance of the workload: this many routed experts (same H, I, top-k); "
                        "the token count scales with it unless --tokens is given (profiling captures)")
    p.add_argument("--tokens", type=int, default=0, help="with --experts: the token count of the reduced instance")
    return p.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- cross-rank helpers
def reduce_max(values, world, device):
    """Elementwise max over ranks (values: list of floats)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(units_per_rank, elapsed_s_max):
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    return sum(units_per_rank) / elapsed_s_max if elapsed_s_max > 0 else 0.0


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_id)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(dev_index):
    import torch
    try:
        u = torch.cuda.get_device_properties(dev_index).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return dev_index


# ----------------------------------------------------------------- algorithmic work
MX_ROUTED_GEMMS = ("gemm_fwd_gu_routed", "gemm_fwd_down_routed", "gemm_bwd_down_routed", "gemm_bwd_gu_routed")
# GEMM classes whose derived operand reaches the tensor cores as hi + lo bf16 terms
# with fp32 activations (the K range runs twice)
SPLIT_GEMMS = ("gemm_fwd_down", "gemm_bwd_gu", "gemm_wgrad_fc1", "gemm_wgrad_down")


def kernel_work(name, T, H, E, k, I, R, E_act, mx=False, mg_bytes=4, act32=True):
    """(algorithmic flops, algorithmic HBM bytes) of one launch of a kernel class.

    Bytes count each distinct operand element read once and each result written
    once (no padding rows, no re-reads: a hidden or grad_out row that k routes
    gather is read once); flops count a multiply-add as 2. Weights of experts
    without tokens are not read. mx: the routed forward/dgrad GEMMs read MXFP8
    operands (1 byte + 1/32 byte of scale per element) and the producers of
    those operands also write their MXFP8 copies. mg_bytes: main_grad element
    size (read and written once by the weight-gradient kernels). act32: g|u, y and
    dx are fp32 (4 bytes) and the derived GEMM operands a, [dg|du], p*a are two
    bf16 terms (4 bytes); else all of them bf16. With BF16 routed weights (not
    mx) the shared expert runs as group 0 of the routed launches: their classes
    carry the shared work too (their group 0 reads hidden / grad_out rows directly)."""
    b2, b4 = 2, 4
    bq = 1 + 1 / 32                          # MXFP8 element incl. its share of the scale
    f = 4 if act32 else 2                    # fp32 (or bf16) activation / two-term operand element
    wb = bq if mx else b2                    # routed weight element
    ab = bq if mx else b2                    # routed fprop/dgrad input-row operand element
    a_in = bq if mx else f                   # routed down / dgrad-gate-up derived operand element
    # routed gate/up epilogue's a besides its MXFP8 copy: none with fp32 activations (the dgrad-down
    # recomputes a from g, u), bf16 with bf16 ones; two terms when the down projection is BF16
    a_out = (0 if act32 else b2) if mx else f
    W_fc1, W_down = E_act * 2 * I * H * wb, E_act * H * I * wb
    q_a = R * I * bq if mx else 0
    q_dgdu = R * 2 * I * bq if mx else 0
    q_rows = R * H * bq if mx else 0
    gu_in = 2 * I * f if act32 else 3 * I * b2   # dgrad-down epilogue: fp32 g|u, or bf16 a and g|u
    table = {
        "route_pack": (0, T * E + T * k * (b4 * 3 + b4)),
        "route_scan": (0, T * E + T * k * b4 + E * b4),
        "route_place": (0, T * k * 12 + R * 12 + T * H * b2 + R * H * b2 + q_rows),
        "gather_rows": (0, T * H * b2 + R * H * b2 + q_rows),
        "gemm_fwd_gu_routed": (4 * R * H * I, R * H * ab + W_fc1 + R * I * a_out + R * 2 * I * f + q_a),
        "gemm_fwd_gu_shared": (4 * T * H * I, T * H * b2 + 2 * I * H * b2 + T * I * f + T * 2 * I * f),
        "gemm_fwd_down_routed": (2 * R * I * H, R * I * a_in + W_down + R * H * f),
        "gemm_fwd_down_shared": (2 * T * I * H, T * I * f + H * I * b2 + T * H * f),
        "combine": (0, T * H * f + R * H * f + T * k * 8 + T * H * b2),
        "gemm_bwd_down_routed": (2 * R * H * I, R * H * ab + W_down + R * gu_in + R * 2 * I * f + R * I * f
                                 + q_dgdu),
        "gemm_bwd_down_shared": (2 * T * H * I, T * H * b2 + H * I * b2 + T * gu_in + T * 2 * I * f + T * I * f),
        "gemm_bwd_gu_routed": (4 * R * I * H, R * 2 * I * a_in + W_fc1 + R * H * f),
        "gemm_bwd_gu_shared": (4 * T * I * H, T * 2 * I * f + 2 * I * H * b2 + T * H * f),
        "gemm_wgrad_fc1_routed": (4 * R * I * H, R * 2 * I * f + R * H * b2 + E_act * 2 * I * H * 2 * mg_bytes),
        "gemm_wgrad_down_routed": (2 * R * H * I, R * H * b2 + R * I * f + E_act * H * I * 2 * mg_bytes),
        "gemm_wgrad_fc1_shared": (4 * T * I * H, T * 2 * I * f + T * H * b2 + 2 * I * H * 2 * mg_bytes),
        "gemm_wgrad_down_shared": (2 * T * H * I, T * H * b2 + T * I * f + H * I * 2 * mg_bytes),
        "unpermute": (0, T * H * f + R * H * f + T * H * b2 + T * E * b4),
        "shared_gate_fwd": (2 * T * H, T * H * b2 + H * b2 + T * b4),
        "shared_gate_bwd": (2 * T * H, T * H * b2 + T * b4 * 3 + H * 2 * mg_bytes),
    }
    # the shared expert is group 0 of the routed launches: of all six GEMMs with BF16
    # routed weights, of the two weight gradients with MXFP8 ones
    for op in ("wgrad_fc1", "wgrad_down") if mx else ("fwd_gu", "fwd_down", "bwd_down", "bwd_gu", "wgrad_fc1",
                                                      "wgrad_down"):
        rf, rb = table[f"gemm_{op}_routed"]
        sf, sb = table[f"gemm_{op}_shared"]
        table[f"gemm_{op}_routed"] = (rf + sf, rb + sb)
    if not mx:
        f_, b_ = table["route_place"]
        table["route_place"] = (f_, b_ + T * 8)   # the shared rows' source and scale (the GEMMs read hidden)
    return table[name]


def mma_flops(name, flops, mx=False, act32=True):
    """Tensor-core work a GEMM launch executes: its algorithmic flops, twice over
    where a two-term operand runs the K range twice (fp32 activations; not the
    routed MXFP8 GEMMs, whose operands are quantised single terms)."""
    if not act32 or not name.startswith(SPLIT_GEMMS):
        return flops
    if mx and name in MX_ROUTED_GEMMS:
        return flops
    return 2 * flops


def roofline_of(name, ms_per_launch, work, peaks, peaks_kind, traffic=None, fp8=False):
    """Roofline of one kernel: tensor-bound if its intensity exceeds the ridge of
    the peak for its own dtype (fp8 = the measured bf16 peak x 2, the nominal
    dense ratio), else HBM-bound."""
    flops, nbytes = work
    tensor_peak = peaks["bf16_tflops_sustained"] * (2.0 if fp8 else 1.0)
    ridge = tensor_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if flops > 0 and flops / max(nbytes, 1) > ridge:
        achieved = flops / (ms_per_launch * 1e-3) / 1e12
        peak = tensor_peak
        r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    else:
        achieved = nbytes / (ms_per_launch * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        r = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    r.update({"frac": achieved / peak, "traffic": traffic, "kernel": name, "ms_per_launch": ms_per_launch,
              "algorithmic_flops": flops, "algorithmic_bytes": nbytes, "peak_source": f"of {peaks_kind}"})
    return r


def useful_flops(R, T, H, I):
    """18 (R + T) H I: forward, dgrad and wgrad are 6 (R+T) H I each."""
    return 18 * (R + T) * H * I


# ----------------------------------------------------------------- the oracle leg
def oracle_sample(cfg_id, T_sample, offset=0):
    """Inputs for the CPU oracle: a token sample of the workload, full weights (fp64)."""
    import numpy as np
    import torch

    import moe_inputs as MI
    from oracle import moe_oracle as O
    c = MI.CONFIGS[cfg_id]
    seed = MI.seed_of(cfg_id)
    r = MI.config_routing(cfg_id)
    w = MI.make_weights(c["H"], c["I"], c["E"], seed, device="cpu")
    hidden, grad_out = MI.make_activations(c["T"], c["H"], seed, device="cpu")
    W = O.DenseWeights.from_combined(*(w[n].to(torch.float64).numpy() for n in
                                       ("shared_fc1", "shared_fc2", "routed_fc1", "routed_fc2")))
    sl = slice(offset, offset + T_sample)
    return dict(W=W, x=hidden[sl].to(torch.float64).numpy(), go=grad_out[sl].to(torch.float64).numpy(),
                probs=r.probs[sl], map=np.ascontiguousarray(r.routing_map[sl]), k=c["k"])


def time_oracle(sample):
    from oracle import moe_oracle as O
    t0 = time.perf_counter()
    _, cache = O.forward(sample["x"], sample["probs"], sample["map"], sample["W"], sample["k"])
    O.backward(sample["go"], cache, sample["W"])
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_baseline(cfg_id, passes=3):
    """The oracle, as it stands, timed on the host cores: forward + backward of
    the workload's whole token batch (full weights), `passes` times."""
    import moe_inputs as MI
    T = MI.CONFIGS[cfg_id]["T"]
    s = oracle_sample(cfg_id, T)
    dt = sum(time_oracle(s) for _ in range(passes))
    return {"value": passes * T / dt, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"fp64 numpy oracle, forward+backward of the whole {T}-token batch of the workload "
                      f"(full weights), {passes} passes, {dt:.1f} s"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import moe_inputs as MI
    c = MI.CONFIGS[args.config]
    T_step = 128
    s = oracle_sample(args.config, T_step * 8)
    subs = []
    for j in range(8):
        sl = slice(j * T_step, (j + 1) * T_step)
        subs.append(dict(W=s["W"], x=s["x"][sl], go=s["go"][sl], probs=s["probs"][sl], map=s["map"][sl], k=s["k"]))
    for i in range(args.warmup):
        time_oracle(subs[i % 8])
    t = 0.0
    for i in range(args.steps):
        t += time_oracle(subs[i % 8])
    value = args.steps * T_step / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; the pages' training data are not available)",
            "config": {"workload": MI.WORKLOAD_NAMES[args.config], "T": c["T"], "H": c["H"], "E": c["E"],
                       "k": c["k"], "I": c["I"], "sample_tokens_per_step": T_step},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{T_step} tokens of the workload per step (full weights), fp64 numpy"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- our arm
def measure_config(cid, args, steps, warmup, full, dev, world, rank, local_rank):
    """One workload through the C ABI: K timed steps (forward + backward) after W
    warm-up steps, the per-kernel table from an untimed pass, the dominant
    kernel's roofline from its live duration inside the timed region. ``full``
    adds forward/backward timed apart, the CUDA-graph replay and the end-to-end
    host-buffer leg."""
    import torch

    import mixture_experts_layer_pack_gb300 as M
    import moe_inputs as MI

    c = dict(MI.CONFIGS[cid])
    reduced = ""
    if args.experts and cid == args.config:
        # a reduced instance: fewer experts, the same tokens per expert on average
        T0, E0 = c["T"], c["E"]
        c["E"] = args.experts
        c["T"] = args.tokens or max(128, (T0 * args.experts // E0 + 127) // 128 * 128)
        reduced = f"-reduced-E{c['E']}-T{c['T']}"
    mx = c["routed"] == "mxfp8"
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    seed = MI.seed_of(cid)
    r = MI.make_routing(T, E, k, seed, c["routing"], c["drop"])
    R = int(r.routing_map.sum())
    E_act = int((r.routing_map.sum(0) > 0).sum())
    act32 = args.act_precision == "fp32"
    w = MI.make_weights(H, I, E, seed, device=dev)
    hidden, grad_out = MI.make_activations(T, H, seed, device=dev)
    mg = MI.make_main_grads(H, I, E, seed, device=dev)
    mg_bf16 = args.main_grad_dtype == "bf16"
    mg_bytes = 2 if mg_bf16 else 4
    workload = (MI.WORKLOAD_NAMES[cid] + reduced + ("-bf16-main-grad" if mg_bf16 else "") +
                ("" if act32 else "-bf16-act"))
    if mg_bf16:
        mg = {n: t.to(torch.bfloat16) for n, t in mg.items()}
    probs = torch.from_numpy(r.probs).to(dev)
    rmap = torch.from_numpy(r.routing_map).to(dev).view(torch.uint8)

    layer = M.MoELayer(T, H, E, k, I, device=dev,
                       routed_wtype=M.binding.MOE_W_MXFP8 if mx else M.binding.MOE_W_BF16,
                       act_precision=M.binding.MOE_ACT_FP32 if act32 else M.binding.MOE_ACT_BF16)
    wv = M.weights_from_combined(w["shared_fc1"], w["shared_fc2"], w["routed_fc1"], w["routed_fc2"])
    if mx:   # MXFP8 routed weights (rowwise + columnwise), prepared outside the timed region
        wmx = MI.make_mxfp8_weights(w)
        w["routed_fc1"] = w["routed_fc2"] = None
        q1, s1, c1, cs1 = wmx["routed_fc1"]
        wv.routed_gate = M.mxfp8_view(q1[:, :I], s1[:, :I], c1[:, :I], cs1[:, :I // 32])
        wv.routed_up = M.mxfp8_view(q1[:, I:], s1[:, I:], c1[:, I:], cs1[:, I // 32:])
        wv.routed_down = M.mxfp8_view(*wmx["routed_fc2"])
        layer.prepare_weights(wv)
        torch.cuda.synchronize()
    mgv = M.main_grads_from_combined(mg["shared_fc1"], mg["shared_fc2"], mg["routed_fc1"], mg["routed_fc2"])
    out = torch.empty_like(hidden)
    dh = torch.empty_like(hidden)
    dp = torch.empty((T, E), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        M.moe_forward(layer.handle, T, hidden, probs, rmap, wv, out, layer.saved, stream)
        M.moe_backward(layer.handle, grad_out, layer.saved, dh, dp, mgv, stream)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise SystemExit("device status reported an error during warm-up")

    # ---- per-kernel pass (untimed): every kernel class bracketed by events, to
    # rank the kernels and find the dominant one
    M.moe_profile_read(layer.handle)                     # drop anything recorded before
    M.moe_profile_select(layer.handle, None)
    M.moe_profile_enable(layer.handle, True)
    n_profile = max(5, steps // 4) if full else 3
    for _ in range(n_profile):
        step()
    torch.cuda.synchronize()
    M.moe_profile_enable(layer.handle, False)
    kernels = M.moe_profile_read(layer.handle)
    top = max((n for n, (tot, cnt) in kernels.items() if cnt), key=lambda n: kernels[n][0])

    # ---- timed region: K steps, events only around the dominant kernel (live
    # duration for its roofline), clocks sampled
    sampler = ClockSampler(gpu_id_for(local_rank))
    sampler.start()
    M.moe_profile_select(layer.handle, [top])
    M.moe_profile_enable(layer.handle, True)
    launches0 = M.moe_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = M.moe_launch_count() - launches0
    M.moe_profile_enable(layer.handle, False)
    M.moe_profile_select(layer.handle, None)
    clocks = sampler.stop()
    top_ms, top_n = M.moe_profile_read(layer.handle)[top]
    top_ms_per_launch = top_ms / max(top_n, 1)
    ms = ev0.elapsed_time(ev1)
    ms_max = reduce_max([ms], world, dev)[0]
    value = aggregate([steps * T] * world, ms_max / 1e3)
    flops = useful_flops(R, T, H, I)
    tflops = flops * steps * world / (ms_max / 1e3) / 1e12
    peaks, peaks_kind = load_peaks()

    # ---- roofline of the dominant kernel (its duration from the timed region);
    # the per-kernel table comes from the untimed per-kernel pass
    per_kernel = {}
    for name, (tot, n) in kernels.items():
        if n:
            per_kernel[name] = {"ms_per_launch": tot / n, "launches": n, "share": 0.0}
    total_k = sum(v["ms_per_launch"] * v["launches"] for v in per_kernel.values())
    for v in per_kernel.values():
        v["share"] = v["ms_per_launch"] * v["launches"] / total_k if total_k else 0.0
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tr_path):
        try:
            traffic = json.load(open(tr_path)).get(workload, {}).get(top)
        except Exception:
            traffic = None
    work = lambda n: kernel_work(n, T, H, E, k, I, R, E_act, mx, mg_bytes, act32)  # noqa: E731
    roof = roofline_of(top, top_ms_per_launch, work(top), peaks, peaks_kind, traffic,
                       fp8=mx and top in MX_ROUTED_GEMMS)
    roof["timed_launches"] = top_n
    roof["mma_flops"] = mma_flops(top, work(top)[0], mx, act32)
    for name, v in per_kernel.items():
        f, b = work(name)
        ms_l = v["ms_per_launch"] * 1e-3
        v["tflops"] = f / ms_l / 1e12 if f else 0.0
        v["mma_tflops"] = mma_flops(name, f, mx, act32) / ms_l / 1e12 if f else 0.0
        v["gbs"] = b / ms_l / 1e9

    res = {"workload": workload, "T": T, "H": H, "E": E, "k": k, "I": I, "valid_routes": R, "mx": mx,
           "routing": c["routing"], "drop": c["drop"], "steps": steps, "warmup": warmup, "value": value,
           "ms_per_step": ms_max / steps, "tflops": tflops, "useful_flops_per_step": flops,
           "pct_bf16_peak": 100.0 * tflops / peaks["bf16_tflops"],
           "pct_fp8_peak": 100.0 * tflops / (2 * peaks["bf16_tflops"]) if mx else None,
           "roofline": roof, "kernels": per_kernel, "n_profile": n_profile, "top": top, "gpu_launches": launches,
           "clocks": clocks, "peaks": peaks, "peaks_kind": peaks_kind, "mg_bf16": mg_bf16, "act32": act32,
           "l2": "inputs larger than L2: routed weights %.2f GB + main_grad %.2f GB per step"
                 % (3 * E * I * H * (1.03 if mx else 2) / 1e9, 3 * (E + 1) * I * H * mg_bytes / 1e9)}
    if not full:
        layer.close()
        return res

    # ---- forward and backward timed apart, and the step replayed as one CUDA graph
    # (no per-kernel events; launch gaps are what the graph removes)
    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    n_split = max(5, steps // 4)
    res["fwd_ms"] = timed(lambda: M.moe_forward(layer.handle, T, hidden, probs, rmap, wv, out, layer.saved, stream),
                          n_split)
    res["bwd_ms"] = timed(lambda: M.moe_backward(layer.handle, grad_out, layer.saved, dh, dp, mgv, stream), n_split)
    graph = None
    try:
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            M.moe_forward(layer.handle, T, hidden, probs, rmap, wv, out, layer.saved, cap)
            M.moe_backward(layer.handle, grad_out, layer.saved, dh, dp, mgv, cap)
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        graph_ms = reduce_max([timed(g.replay, max(10, steps // 2))], world, dev)[0]
        graph = {"ms_per_step": graph_ms, "value": T * world / (graph_ms / 1e3), "unit": "tokens/s",
                 "kernels_per_step": launches // max(steps, 1)}
        del g
    except Exception as ex:                              # capture is reported, not required
        graph = {"unavailable": f"{type(ex).__name__}: {ex}"}
    res["cuda_graph"] = graph
    if layer.device_status() != 0:
        raise SystemExit("device status reported an error")

    # ---- end to end through the C ABI's host-buffer entry (moe_host_step): pinned
    # host inputs in, results out, every step
    h_hidden = hidden.cpu().pin_memory()
    h_grad = grad_out.cpu().pin_memory()
    h_probs = probs.cpu().pin_memory()
    h_map = rmap.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h_dh = torch.empty(dh.shape, dtype=dh.dtype, pin_memory=True)
    h_dp = torch.empty(dp.shape, dtype=dp.dtype, pin_memory=True)
    # two result sets, so that a step's results are not overwritten by the next
    # step's download while the host could still be reading them
    h_res = [(h_out, h_dh, h_dp)] + [tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                                           for t in (h_out, h_dh, h_dp))]
    pipe = layer.host_pipe(T)

    def e2e_step(i):
        pipe.step(h_hidden, h_probs, h_map, h_grad, wv, mgv, *h_res[i % 2])

    torch.cuda.synchronize()
    for i in range(3):
        e2e_step(i)
    pipe.synchronize()
    e2e_steps = max(10, steps // 4)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    pipe.synchronize()
    torch.cuda.synchronize()
    e2e_s = reduce_max([time.perf_counter() - t0], world, dev)[0]
    h2d = sum(t.numel() * t.element_size() for t in (h_hidden, h_grad, h_probs, h_map))
    d2h = sum(t.numel() * t.element_size() for t in (h_out, h_dh, h_dp))
    res["e2e"] = {"value": aggregate([e2e_steps * T] * world, e2e_s), "unit": "tokens/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "api": "moe_host_step"}
    pipe.close()
    layer.close()
    return res


def measure_ep_owner(cid, ep, steps, warmup, dev):
    """The owner-side step of expert parallelism at EP degree ``ep`` for workload
    ``cid``: the rank holding E/ep experts runs them (a routed-only handle, top-1)
    on the rows all ep ranks route to them -- T*k rows for ep ranks of T tokens
    each, split over the local experts in proportion to a seeded multinomial --
    forward + backward with main_grad accumulation. CUDA events over ``steps``
    steps after ``warmup``; useful FLOPs 18 n H I per step."""
    import numpy as np
    import torch
    import moe_inputs as MI
    import mixture_experts_layer_pack_gb300 as M
    c = MI.CONFIGS[cid]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    if E % ep or c["routed"] != "bf16":
        return {"unavailable": f"E={E} not divisible by EP{ep}, or MXFP8 routed weights (BF16 owner step only)"}
    el = E // ep
    n = T * k
    seed = MI.seed_of(cid) + 101
    rng = np.random.default_rng(seed)
    counts = rng.multinomial(n, np.full(el, 1.0 / el))
    ids = torch.from_numpy(np.repeat(np.arange(el, dtype=np.int32), counts)[:, None]).to(dev)
    probs = torch.from_numpy(rng.uniform(0.05, 0.5, size=(n, 1)).astype(np.float32)).to(dev)
    w = MI.make_weights(H, I, el, seed, device=dev)
    rows, go = MI.make_activations(n, H, seed, device=dev)
    mg = MI.make_main_grads(H, I, el, seed, device=dev)
    layer = M.MoELayer(n, H, el, 1, I, device=dev, shared_expert=False)
    wv = M.weights_from_combined(None, None, w["routed_fc1"], w["routed_fc2"])
    mgv = M.main_grads_from_combined(None, None, mg["routed_fc1"], mg["routed_fc2"])
    out = torch.empty_like(rows)
    dx = torch.empty_like(rows)
    dp = torch.empty((n, 1), dtype=torch.float32, device=dev)

    def step():
        layer.forward_topk(rows, ids, probs, wv, out=out)
        layer.backward(go, mgv, dhidden=dx, dprobs=dp)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        step()
    t1.record()
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise SystemExit("device status reported an error in the owner step")
    ms = t0.elapsed_time(t1) / steps
    flops = 18.0 * n * H * I
    layer.close()
    return {"workload": f"{MI.WORKLOAD_NAMES[cid]}-EP{ep}-owner", "experts": el, "rows": n,
            "rows_per_expert": [int(x) for x in counts], "steps": steps, "warmup": warmup, "ms_per_step": ms,
            "rows_per_s": n / (ms * 1e-3), "useful_tflops": flops / (ms * 1e-3) / 1e12,
            "note": "routed-only handle, top-1 over the received rows; the all-to-all exchange is not timed"}


def per_config_entry(res):
    """The compact record of one extra workload."""
    roof = res["roofline"]
    return {"workload": res["workload"], "steps": res["steps"], "warmup": res["warmup"],
            "ms_per_step": res["ms_per_step"], "tokens_per_s": res["value"], "useful_tflops": res["tflops"],
            "pct_bf16_peak": res["pct_bf16_peak"], "pct_fp8_peak": res["pct_fp8_peak"],
            "roofline": {kk: roof[kk] for kk in ("kernel", "bound", "achieved", "peak", "unit", "frac",
                                                 "ms_per_launch", "traffic", "peak_source")},
            "kernels": {n: {"ms_per_launch": v["ms_per_launch"], "share": v["share"], "gbs": v["gbs"],
                            "tflops": v["tflops"], "mma_tflops": v["mma_tflops"]} for n, v in res["kernels"].items()},
            "gpu_launches_per_step": res["gpu_launches"] // max(res["steps"], 1), "clocks": res["clocks"]}


def run_ours(args):
    import torch

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    res = measure_config(args.config, args, args.steps, args.warmup, True, dev, world, rank, local_rank)
    torch.cuda.empty_cache()
    cid = args.config
    per_config = {}
    extra = [int(x) for x in args.per_config.split(",") if x.strip()] if args.per_config else []
    for other in extra:
        if other == cid:
            continue
        try:
            r2 = measure_config(other, args, args.per_config_steps, 3, False, dev, world, rank, local_rank)
            per_config[str(other)] = per_config_entry(r2)
        except torch.cuda.OutOfMemoryError as ex:
            per_config[str(other)] = {"unavailable": f"out of device memory: {ex}"}
        torch.cuda.empty_cache()

    act_variant = None
    if args.act_variant:
        import copy
        a2 = copy.copy(args)
        a2.act_precision = "bf16" if args.act_precision == "fp32" else "fp32"
        r3 = measure_config(cid, a2, args.per_config_steps, 3, False, dev, world, rank, local_rank)
        act_variant = {"act_precision": a2.act_precision, **per_config_entry(r3),
                       "note": ("single bf16 activations between the expert GEMMs: faster; its parity is against "
                                "the bf16-rounding oracle, normwise 1e-2 of the exact definition")
                       if a2.act_precision == "bf16" else "fp32 activations, two-term operands"}
        torch.cuda.empty_cache()
    ep_owner = None
    if args.ep_owner > 1 and world == 1:
        ep_owner = measure_ep_owner(cid, args.ep_owner, max(10, args.per_config_steps), 3, dev)
        torch.cuda.empty_cache()

    peaks, peaks_kind = res["peaks"], res["peaks_kind"]
    mx = res["mx"]
    line = {"metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8 routed / bf16 shared" if mx else "bf16",
            "data": "synthetic (seeded routing, N(0,0.02) weights, N(0,1) activations; random init)",
            "config": {"workload": res["workload"], "T": res["T"], "H": res["H"], "E": res["E"], "k": res["k"],
                       "I": res["I"], "valid_routes": res["valid_routes"],
                       "routing": f"seeded router stand-in ({res['routing']}, drop={res['drop']})",
                       "main_grad": f"{args.main_grad_dtype}, accumulated in place every step",
                       "activations": ("fp32 between the expert GEMMs, derived GEMM operands as hi + lo bf16 terms"
                                       if res["act32"] else "bf16 between the expert GEMMs"),
                       "l2": res["l2"],
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "tflops": res["tflops"], "pct_bf16_peak": res["pct_bf16_peak"], "pct_fp8_peak": res["pct_fp8_peak"],
            "peaks": {**peaks, "source": peaks_kind},
            "useful_flops_per_step": res["useful_flops_per_step"],
            "roofline": res["roofline"], "kernels": res["kernels"],
            "kernels_note": f"per-kernel CUDA events over {res['n_profile']} untimed steps; the timed region "
                            f"brackets only {res['top']}",
            "gpu_launches": res["gpu_launches"], "clocks": res["clocks"], "e2e": res["e2e"],
            "fwd_ms": res["fwd_ms"], "bwd_ms": res["bwd_ms"], "cuda_graph": res["cuda_graph"]}
    if per_config:
        line["per_config"] = per_config
    if ep_owner is not None:
        line["ep_owner_step"] = ep_owner
    if act_variant is not None:
        line["act_precision_variant"] = act_variant
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cid)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
