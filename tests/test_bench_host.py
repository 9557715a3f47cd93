"""Host logic of bench.py's multi-replica mode on CPU ranks (gloo, world size 2):
max-over-ranks timing, whole-job throughput, and the reference arm's rank rule."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [1.5 + rank, 10.0 * (rank + 1)]                      # rank 1 is the slow one
        mx = bench.reduce_max(elapsed, world, torch.device("cpu"))
        bench.barrier(world)
        value = bench.aggregate([100] * world, mx[0])
        out[rank] = (mx, value)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    world = 2
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        mx, value = out[rank]
        assert mx == [2.5, 20.0]                       # every rank sees the slowest rank's time
        assert value == pytest.approx(200 / 2.5)       # units of all ranks / slowest time


def test_single_rank_helpers_need_no_process_group():
    assert bench.reduce_max([3.0, 4.0], 1, torch.device("cpu")) == [3.0, 4.0]
    assert bench.aggregate([50], 0.5) == 100.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args) == 0              # returns at once, prints nothing


def test_kernel_work_table_covers_every_kernel_class():
    import mixture_experts_layer_pack_gb300 as M
    names = [M.moe_kernel_name(i) for i in range(M.binding.MOE_K_COUNT)]
    assert None not in names and M.moe_kernel_name(M.binding.MOE_K_COUNT) is None
    for n in names:
        f, b = bench.kernel_work(n, 4096, 2048, 96, 6, 1024, 24576, 96)
        assert f >= 0 and b >= 0
    # the dominant wgrad kernel is HBM-bound at the proxy-like shape
    peaks = dict(hbm_gbs=6791.0, bf16_tflops=1902.3, bf16_tflops_sustained=1710.5)
    r = bench.roofline_of("gemm_wgrad_fc1_routed", 0.65, bench.kernel_work("gemm_wgrad_fc1_routed", 4096, 2048, 96,
                                                                           6, 1024, 24576, 96), peaks, "measured")
    assert r["bound"] == "hbm" and 0 < r["frac"] < 1.5


def test_kernel_work_counts_the_shared_expert_in_the_bf16_grouped_launches():
    """BF16 routed weights: the shared expert is group 0 of the routed launches, so their
    algorithmic work is the routed formula at R + T rows and E_act + 1 experts; with
    MXFP8 routed weights only the two weight gradients are grouped that way. fp32 activations: the
    two-term [dg|du] operand is 4 bytes an element; bf16 activations: 2."""
    T, H, E, k, I, R, Ea = 4096, 2048, 96, 6, 1024, 24576, 96
    for act32, f_ in ((True, 4), (False, 2)):
        f, b = bench.kernel_work("gemm_wgrad_fc1_routed", T, H, E, k, I, R, Ea, mx=False, mg_bytes=4, act32=act32)
        assert f == 4 * (R + T) * I * H
        assert b == (R + T) * 2 * I * f_ + (R + T) * H * 2 + (Ea + 1) * 2 * I * H * 2 * 4
        f, b = bench.kernel_work("gemm_fwd_gu_routed", T, H, E, k, I, R, Ea, mx=False, act32=act32)
        assert f == 4 * (R + T) * H * I
        assert b == (R + T) * H * 2 + (Ea + 1) * 2 * I * H * 2 + (R + T) * I * f_ + (R + T) * 2 * I * f_
    f, _ = bench.kernel_work("gemm_fwd_gu_routed", T, H, E, k, I, R, Ea, mx=True)
    assert f == 4 * R * I * H                         # MXFP8: the shared expert's forward runs apart
    f, _ = bench.kernel_work("gemm_wgrad_fc1_routed", T, H, E, k, I, R, Ea, mx=True)
    assert f == 4 * (R + T) * I * H                   # its weight gradients are group 0 of the routed ones
    # the useful flops of a step: forward, dgrad and wgrad over routed and shared rows
    assert bench.useful_flops(R, T, H, I) == sum(
        bench.kernel_work(n, T, H, E, k, I, R, Ea, mx=False)[0]
        for n in ("gemm_fwd_gu_routed", "gemm_fwd_down_routed", "gemm_bwd_down_routed", "gemm_bwd_gu_routed",
                  "gemm_wgrad_fc1_routed", "gemm_wgrad_down_routed"))
    # the tensor work executed: the four GEMMs with a two-term operand run K twice
    assert bench.mma_flops("gemm_fwd_down_routed", 10, mx=False, act32=True) == 20
    assert bench.mma_flops("gemm_fwd_gu_routed", 10, mx=False, act32=True) == 10
    assert bench.mma_flops("gemm_fwd_down_routed", 10, mx=True, act32=True) == 10
    assert bench.mma_flops("gemm_wgrad_fc1_routed", 10, mx=True, act32=True) == 20
    assert bench.mma_flops("gemm_bwd_gu_routed", 10, mx=False, act32=False) == 10


def test_gather_kernels_count_each_source_row_once():
    """A hidden (or grad_out) row that k routes gather is read from HBM once: the
    placement and the grad gather count T rows read and R rows written (the shared
    expert's GEMMs read hidden and grad_out themselves)."""
    T, H, E, k, I, R, Ea = 4096, 2048, 96, 6, 1024, 24576, 96
    _, b = bench.kernel_work("gather_rows", T, H, E, k, I, R, Ea, mx=False)
    assert b == T * H * 2 + R * H * 2
    _, b = bench.kernel_work("gather_rows", T, H, E, k, I, R, Ea, mx=True)
    assert b == pytest.approx(T * H * 2 + R * H * 2 + R * H * (1 + 1 / 32))


# Per-launch times (ms) of every kernel class at the proxy-like workload (T=4096,
# H=2048, E=96 top-6, I=1024, R=24576 routes, every expert with tokens), measured on
# one GB300 with `python bench.py` (CUDA events, fp32 and bf16 activations).
RECORDED_MS = {
    True: {"route_place": 0.0240, "gather_rows": 0.0222, "gemm_fwd_gu_routed": 0.2565,
           "gemm_fwd_down_routed": 0.1846, "combine": 0.0467, "gemm_bwd_down_routed": 0.2206,
           "gemm_bwd_gu_routed": 0.3326, "gemm_wgrad_fc1_routed": 0.5868, "gemm_wgrad_down_routed": 0.3078,
           "unpermute": 0.0550},
    False: {"route_place": 0.0240, "gather_rows": 0.0227, "gemm_fwd_gu_routed": 0.2269,
            "gemm_fwd_down_routed": 0.1188, "combine": 0.0314, "gemm_bwd_down_routed": 0.2505,
            "gemm_bwd_gu_routed": 0.2170, "gemm_wgrad_fc1_routed": 0.5361, "gemm_wgrad_down_routed": 0.2821,
            "unpermute": 0.0393},
}


@pytest.mark.parametrize("act32", [True, False])
def test_recorded_kernel_rates_stay_below_the_measured_peaks(act32):
    """The algorithmic bytes (and flops) of every kernel class over its measured time
    stay at or below the measured copy bandwidth (and bf16 tensor peak) x 1.05: the
    byte counts do not count a row that several routes read as read several times."""
    T, H, E, k, I, R, Ea = 4096, 2048, 96, 6, 1024, 24576, 96
    peaks = bench.load_peaks()[0]
    for name, ms in RECORDED_MS[act32].items():
        f, b = bench.kernel_work(name, T, H, E, k, I, R, Ea, mx=False, mg_bytes=4, act32=act32)
        assert b / (ms * 1e-3) / 1e9 <= 1.05 * peaks["hbm_gbs"], name
        mma = bench.mma_flops(name, f, mx=False, act32=act32)
        assert mma / (ms * 1e-3) / 1e12 <= 1.05 * peaks["bf16_tflops"], name


def test_recorded_traffic_matches_the_algorithmic_bytes():
    """profiles/traffic.json holds the ncu DRAM bytes (read + write) of the dominant launch
    of every workload the bench reports. Each lies within [0.9, 1.25] x the launch's
    algorithmic bytes at that workload's routing: far above would mean operand re-reads
    (or a stale capture), far below an accounting that counts bytes the launch never moves."""
    import json
    import os
    import moe_inputs as MI
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        traffic = json.load(f)
    for cid in (2, 3, 4, 5):
        assert MI.WORKLOAD_NAMES[cid] in traffic, cid
    for wl, entries in traffic.items():
        cid = next(c for c, n in MI.WORKLOAD_NAMES.items() if wl.startswith(n))
        c = MI.CONFIGS[cid]
        r = MI.config_routing(cid)
        R, Ea = int(r.routing_map.sum()), int((r.routing_map.sum(0) > 0).sum())
        for name, t in entries.items():
            _, b = bench.kernel_work(name, c["T"], c["H"], c["E"], c["k"], c["I"], R, Ea,
                                     mx=c["routed"] == "mxfp8", mg_bytes=4, act32=not wl.endswith("-bf16-act"))
            assert 0.9 <= t / b <= 1.25, (wl, name, t / b)
