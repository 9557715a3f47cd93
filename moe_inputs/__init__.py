"""Seeded synthetic inputs for the MoE layer (shared by the oracle tests, the GPU tests and the bench).

This module draws random numbers and lays them out; it holds none of the layer's
arithmetic. The router that produces ``probs``/``routing_map`` is the model's, not
the layer's, so a softmax + top-k stand-in for it lives here as input synthesis.

Recipe (the pages' training workloads, the Proxy model and DSv4-Pro, are not
available, so these layers stand in for them with the same E, top-k and
precision):

* routing: numpy PCG64 ``default_rng(seed)``; logits ~ N(0,1) [T,E] (plus an
  expert bias for the skewed case), softmax over E in fp64, top-k by prob, the
  kept softmax values stored as fp32 in a dense ``probs[T,E]`` (zeros elsewhere)
  and a bool ``routing_map[T,E]``; no renormalisation;
* dense tensors: a seeded ``torch.Generator`` on the target device; fp32 draws
  RNE-cast to bf16 (weights ~ N(0,0.02), hidden ~ N(0,1), grad_out ~ N(0,1));
  main_grad ~ N(0,1e-3) fp32;
* MXFP8 routed weights are input data too (the framework that owns the
  weights quantises them): made from the bf16 masters with PyTorch's
  float8_e4m3fn cast, rowwise and columnwise, OCP MX block rule.
"""
from __future__ import annotations

import dataclasses

import numpy as np

# Layer shapes of the five workloads (tokens T, hidden H, routed experts E,
# top-k, intermediate I shared by routed and shared experts).
CONFIGS = {
    1: dict(T=64, H=128, E=8, k=2, I=64, routed="bf16", routing="topk", drop="second"),
    2: dict(T=4096, H=2048, E=96, k=6, I=1024, routed="bf16", routing="topk", drop="none"),
    3: dict(T=4096, H=2048, E=96, k=6, I=1024, routed="mxfp8", routing="topk", drop="none"),
    4: dict(T=8192, H=7168, E=384, k=6, I=2048, routed="mxfp8", routing="topk", drop="iid"),
    5: dict(T=16384, H=4096, E=128, k=8, I=1536, routed="bf16", routing="zipf", drop="multi"),
}

WORKLOAD_NAMES = {
    1: "tiny-T64-H128-E8-top2-I64-bf16",
    2: "proxy-T4096-H2048-E96-top6-I1024-bf16",
    3: "proxy-T4096-H2048-E96-top6-I1024-mxfp8",
    4: "dsv4like-T8192-H7168-E384-top6-I2048-mxfp8",
    5: "skewed-T16384-H4096-E128-top8-I1536-bf16",
}


@dataclasses.dataclass
class Routing:
    probs: np.ndarray        # float32 [T, E]
    routing_map: np.ndarray  # bool [T, E]


def seed_of(config_id: int) -> int:
    return 1000 + config_id


def _softmax(logits: np.ndarray) -> np.ndarray:
    z = logits - logits.max(axis=1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=1, keepdims=True)


def make_routing(T: int, E: int, k: int, seed: int, routing: str = "topk",
                 drop: str = "none") -> Routing:
    """Router stand-in: dense probs/routing_map with the workload's missing-route pattern.

    routing: "topk" (softmax top-k), "balanced" (token t -> experts (k*t+j) mod E,
    probs = the softmax values there), "zipf" (logit bias -1.2*1.2*ln(rank_e) with
    ranks a seeded permutation of 1..E, so a few experts are hot and some get no
    tokens).
    drop: "none"; "second" (5% of tokens lose their second-highest route);
    "iid" (each route dropped independently with p=0.02); "multi" (10% of tokens
    lose 1-3 of their k routes, chosen uniformly). A dropped route has map=False
    and prob=0.
    """
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E))
    if routing == "zipf":
        ranks = rng.permutation(E) + 1
        logits = logits - 1.2 * 1.2 * np.log(ranks)[None, :]
    p_full = _softmax(logits)
    if routing == "balanced":
        sel = (k * np.arange(T)[:, None] + np.arange(k)[None, :]) % E
    else:
        sel = np.argsort(-p_full, axis=1, kind="stable")[:, :k]
    keep = np.ones((T, k), dtype=bool)
    if drop == "second" and k >= 2:
        n = int(round(0.05 * T))
        keep[rng.choice(T, size=n, replace=False), 1] = False
    elif drop == "iid":
        keep &= rng.random((T, k)) >= 0.02
    elif drop == "multi":
        n = int(round(0.10 * T))
        toks = rng.choice(T, size=n, replace=False)
        for t in toks:
            m = int(rng.integers(1, 4))
            keep[t, rng.choice(k, size=min(m, k), replace=False)] = False
    elif drop != "none":
        raise ValueError(drop)
    routing_map = np.zeros((T, E), dtype=bool)
    probs = np.zeros((T, E), dtype=np.float32)
    rows = np.repeat(np.arange(T), k).reshape(T, k)
    routing_map[rows[keep], sel[keep]] = True
    probs[rows[keep], sel[keep]] = p_full[rows[keep], sel[keep]].astype(np.float32)
    return Routing(probs=probs, routing_map=routing_map)


def config_routing(config_id: int, T: int | None = None, variant: str | None = None) -> Routing:
    c = CONFIGS[config_id]
    routing = variant or c["routing"]
    return make_routing(T or c["T"], c["E"], c["k"], seed_of(config_id), routing, c["drop"])


def _torch():
    import torch
    return torch


def _draw_bf16(gen, shape, std, device):
    torch = _torch()
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if len(shape) == 3:
        for e in range(shape[0]):
            out[e].copy_(torch.randn(shape[1:], generator=gen, device=device,
                                     dtype=torch.float32) * std)
    else:
        out.copy_(torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std)
    return out


def make_weights(H: int, I: int, E: int, seed: int, device="cpu", std: float = 0.02) -> dict:
    """BF16 weights in the combined-FC1 layout: fc1 rows [0,I) gate, [I,2I) up.

    shared_fc1 [2I,H], shared_fc2 [H,I], routed_fc1 [E,2I,H], routed_fc2 [E,H,I].
    """
    torch = _torch()
    g = torch.Generator(device=device).manual_seed(seed)
    return dict(
        shared_fc1=_draw_bf16(g, (2 * I, H), std, device),
        shared_fc2=_draw_bf16(g, (H, I), std, device),
        routed_fc1=_draw_bf16(g, (E, 2 * I, H), std, device),
        routed_fc2=_draw_bf16(g, (E, H, I), std, device),
    )


def make_activations(T: int, H: int, seed: int, device="cpu"):
    """hidden ~ N(0,1) and grad_out ~ N(0,1), both bf16 [T,H]."""
    torch = _torch()
    g = torch.Generator(device=device).manual_seed(seed + 7)
    hidden = _draw_bf16(g, (T, H), 1.0, device)
    grad_out = _draw_bf16(g, (T, H), 1.0, device)
    return hidden, grad_out


def make_main_grads(H: int, I: int, E: int, seed: int, device="cpu", std: float = 1e-3) -> dict:
    """fp32 main_grad buffers ~ N(0,1e-3) in the six-buffer order's logical shapes."""
    torch = _torch()
    g = torch.Generator(device=device).manual_seed(seed + 13)

    def draw(*shape):
        out = torch.empty(shape, dtype=torch.float32, device=device)
        if len(shape) == 3:
            for e in range(shape[0]):
                out[e].copy_(torch.randn(shape[1:], generator=g, device=device) * std)
        else:
            out.copy_(torch.randn(shape, generator=g, device=device) * std)
        return out

    return dict(
        shared_fc1=draw(2 * I, H), shared_fc2=draw(H, I),
        routed_fc1=draw(E, 2 * I, H), routed_fc2=draw(E, H, I),
    )


def make_shared_output_gate(H: int, seed: int, device="cpu", std: float = 0.05):
    """Shared-expert output gate weight, bf16 [H] ~ N(0, std), and its fp32 [H]
    main_grad ~ N(0, 1e-3). With hidden ~ N(0,1) the gate logit has std
    std * sqrt(H) (about 2.3 at H = 2048), so gates spread over (0, 1)."""
    torch = _torch()
    g = torch.Generator(device=device).manual_seed(seed + 19)
    w = _draw_bf16(g, (H,), std, device)
    mg = torch.randn((H,), generator=g, device=device, dtype=torch.float32) * 1e-3
    return w, mg


def mxfp8_quantize_torch(w, axis):
    """MXFP8 input weights from bf16 masters with PyTorch ops (float8_e4m3fn cast):
    blocks of 32 along ``axis`` (-1: along K, the row; -2: down the rows),
    E8M0 code = floor(log2 amax) - 8 + 127 clamped to [0, 254] (0 for an all-zero
    block), elements = x / 2^(code-127) clamped to +-448 and cast (round to nearest
    even). Returns (payload uint8 with w's shape, scale codes uint8)."""
    torch = _torch()
    x = w.float()
    if axis == -2:
        x = x.transpose(-1, -2)
    shp = x.shape
    blocks = x.reshape(*shp[:-1], shp[-1] // 32, 32)
    amax = blocks.abs().amax(dim=-1)
    _, ex = torch.frexp(amax)                                  # amax = m 2^ex, m in [0.5, 1)
    code = torch.clamp(ex - 1 - 8 + 127, 0, 254)
    code = torch.where(amax > 0, code, torch.zeros_like(code))
    scaled = blocks * torch.exp2(127.0 - code.float()).unsqueeze(-1)
    payload = torch.clamp(scaled, -448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).reshape(shp)
    code = code.to(torch.uint8)
    if axis == -2:
        payload = payload.transpose(-1, -2).contiguous()
        code = code.transpose(-1, -2).contiguous()
    return payload.contiguous(), code.contiguous()


def make_mxfp8_weights(w: dict) -> dict:
    """MXFP8 copies of the routed weights (combined FC1 [E,2I,H], FC2 [E,H,I]):
    rowwise payload + scales [E,N,K/32] for forward, columnwise payload +
    scales [E,N/32,K] for dgrad (quantised one expert at a time to bound the
    temporary memory)."""
    torch = _torch()
    out = {}
    for name in ("routed_fc1", "routed_fc2"):
        t = w[name]
        E, N, K = t.shape
        q = torch.empty((E, N, K), dtype=torch.uint8, device=t.device)
        s = torch.empty((E, N, K // 32), dtype=torch.uint8, device=t.device)
        qc = torch.empty((E, N, K), dtype=torch.uint8, device=t.device)
        sc = torch.empty((E, N // 32, K), dtype=torch.uint8, device=t.device)
        for e in range(E):
            q[e], s[e] = mxfp8_quantize_torch(t[e], -1)
            qc[e], sc[e] = mxfp8_quantize_torch(t[e], -2)
        out[name] = (q, s, qc, sc)
    return out
