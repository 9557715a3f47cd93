"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc at all -- a plugin inside a host framework
that owns every byte of device memory through its own pool, a serving loop that
forbids allocation after start-up. moe_route_noalloc gives them the layer's
routing (fixed-width ids, gathered probs, per-expert counts and offsets, the
dispatch permutation) with its scratch in a library-owned device array instead
of caller- or driver-allocated memory.

The test calls it through the C ABI twice in a row, on two different
workloads (the second smaller than the first, so stale scratch from the first
call would show), and checks every output against the regular entry points
(moe_forward + moe_export_routing) on the same inputs. Routing is integer
work, so the comparison is bit-exact -- the tolerance every routing test here
uses.
"""
import numpy as np
import pytest
import torch

from moe_inputs import make_routing
from tests.harness import Case, config_case, make_inputs, run_gpu

pytestmark = pytest.mark.gpu


def _regular(inp, status=0):
    import mixture_experts_layer_pack_gb300 as M
    res = run_gpu(inp, backward=False)
    c = inp.case
    dev = inp.hidden.device
    out = dict(ids=torch.empty((c.T, c.k), dtype=torch.int32, device=dev),
               pp=torch.empty((c.T, c.k), dtype=torch.float32, device=dev),
               counts=torch.empty(c.E, dtype=torch.int32, device=dev),
               offsets=torch.empty(c.E + 1, dtype=torch.int32, device=dev),
               perm_src=torch.full((c.T * c.k,), -7, dtype=torch.int32, device=dev),
               row_of=torch.empty((c.T, c.k), dtype=torch.int32, device=dev))
    M.moe_export_routing(res.layer.handle, res.layer.saved, **out)
    torch.cuda.synchronize()
    assert res.layer.device_status() == status
    return {n: t.cpu() for n, t in out.items()}


def _noalloc(inp, error=0):
    import mixture_experts_layer_pack_gb300 as M
    c = inp.case
    dev = inp.hidden.device
    out = dict(ids=torch.full((c.T, c.k), 99, dtype=torch.int32, device=dev),
               pp=torch.full((c.T, c.k), 9.0, dtype=torch.float32, device=dev),
               counts=torch.full((c.E,), 99, dtype=torch.int32, device=dev),
               offsets=torch.full((c.E + 1,), 99, dtype=torch.int32, device=dev),
               perm_src=torch.full((c.T * c.k,), -7, dtype=torch.int32, device=dev),
               row_of=torch.full((c.T, c.k), 99, dtype=torch.int32, device=dev))
    err = torch.full((1,), 5, dtype=torch.int32, device=dev)
    M.moe_route_noalloc(c.T, c.E, c.k, inp.routing_map.view(torch.uint8), inp.probs, out["ids"], out["pp"],
                        out["counts"], out["offsets"], out["perm_src"], out["row_of"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == error
    return {n: t.cpu() for n, t in out.items()}


def test_noalloc_routing_matches_regular_entry_points_twice():
    large = config_case(5)                                   # T*k = 131072: the scratch's full size
    large = Case(large.T, 128, large.E, large.k, 64, large.seed, large.routing, large.drop)
    small = Case(T=300, H=128, E=8, k=2, I=64, seed=21, drop="iid")
    for case in (large, small):
        inp = make_inputs(case)
        want = _regular(inp)
        got = _noalloc(inp)
        for name in want:
            assert torch.equal(got[name], want[name]), (case, name)
        R = int(want["offsets"][-1])
        assert R == int(inp.map_np.sum())
        assert np.all(got["perm_src"].numpy()[R:] == -7)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import mixture_experts_layer_pack_gb300 as M
    from mixture_experts_layer_pack_gb300.binding import MoeError
    dev = torch.device("cuda")
    T, E, k = 16385, 128, 8                                  # T*k = 131080 > 131072
    z = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(MoeError) as ei:
        M.moe_route_noalloc(T, E, k, z, z, z, z, z, z, z, z, z)
    assert ei.value.status == 2                              # MOE_ERR_UNSUPPORTED


def test_noalloc_drops_rows_with_too_many_routes_like_the_regular_path():
    """Rows of the map with k + 1 routes: routing_error is 1 and those rows are
    dropped (every slot -1), bitwise as the regular entry points drop them (which
    report MOE_ERR_ROUTING through the device status)."""
    c = Case(T=300, H=128, E=8, k=2, I=64, seed=61, drop="iid")
    r = make_routing(c.T, c.E, c.k, c.seed, c.routing, c.drop)
    bad = [3, 50, 299]
    for t in bad:
        r.routing_map[t, :] = False
        r.routing_map[t, [1, 4, 6]] = True                      # three routes with k = 2
        r.probs[t, [1, 4, 6]] = 0.25
    inp = make_inputs(c, routing=r)
    want = _regular(inp, status=3)                              # MOE_ERR_ROUTING
    got = _noalloc(inp, error=1)
    for name in want:
        assert torch.equal(got[name], want[name]), name
    assert np.all(got["ids"].numpy()[bad] == -1) and np.all(got["row_of"].numpy()[bad] == -1)
    R = int(want["offsets"][-1])
    assert R == int(inp.map_np.sum()) - 3 * len(bad)
