"""Expert-parallel dispatch and combine on CPU ranks (gloo, world sizes 2 and 3).

Each rank holds its share of the tokens and owns a contiguous range of the routed
experts (the first E mod W ranks one more). The exchange
(mixture_experts_layer_pack_gb300.expert_parallel) moves the token rows to the
owners and back; the experts, the shared expert and the sums on either side are
the fp64 oracle's. Against the single-rank oracle over all tokens:

* the dispatch is bit-exact: every owner receives, for each of its experts,
  exactly the rows (and probs) the single-rank permutation gives that expert,
  in the same order;
* out, dhidden, dprobs of every rank's tokens and every owner's routed weight
  gradients match to fp64 rounding; the shared expert's weight gradients summed
  over the ranks match too (that sum is the data-parallel gradient reduction,
  which the layer leaves to its caller).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixture_experts_layer_pack_gb300 import expert_parallel as EP

CASES = {
    "even": dict(T=96, H=64, E=6, k=2, I=32, seed=71),
    "odd_experts_missing_routes": dict(T=80, H=64, E=5, k=3, I=32, seed=72),
    "three_ranks": dict(T=91, H=64, E=7, k=2, I=32, seed=73, world=3),
}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(c):
    import moe_inputs as MI
    from oracle import moe_oracle as O
    r = MI.make_routing(c["T"], c["E"], c["k"], c["seed"], "topk", "iid" if c["E"] % 2 else "none")
    w = MI.make_weights(c["H"], c["I"], c["E"], c["seed"], device="cpu")
    hidden, grad_out = MI.make_activations(c["T"], c["H"], c["seed"], device="cpu")
    W = O.DenseWeights.from_combined(*(w[n].to(torch.float64).numpy() for n in
                                       ("shared_fc1", "shared_fc2", "routed_fc1", "routed_fc2")))
    if c["E"] % 2:                      # an expert without tokens on the second rank's range
        r.routing_map[:, c["E"] - 1] = False
        r.probs[:, c["E"] - 1] = 0.0
    return W, hidden.double().numpy(), grad_out.double().numpy(), r.probs.astype(np.float64), r.routing_map


def _worker(rank, world, port, name, q):
    from oracle import moe_oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c = CASES[name]
        W, x_all, go_all, probs_all, map_all = _inputs(c)
        T, k, E = c["T"], c["k"], c["E"]
        tl = slice(rank * T // world, (rank + 1) * T // world)
        x, go, probs, rmap = x_all[tl], go_all[tl], probs_all[tl], map_all[tl]
        part = EP.ExpertPartition(E, world)
        ids, pp, over = O.route_pack(rmap, probs, k)
        assert not over.any()
        dW = {}

        def experts_fwd(rows, local_counts, p_rows):
            rows = rows.numpy()
            y = np.zeros_like(rows)
            cache, lo = {}, 0
            for j, e in enumerate(part.local(rank)):
                n = int(local_counts[j])
                if n:
                    g, u, a, y[lo:lo + n] = O.expert_forward(rows[lo:lo + n], *W.routed(e))
                    cache[e] = (lo, n, g, u, a)
                lo += n
            return torch.from_numpy(y), cache

        def experts_bwd(x_rows, go_rows, p_rows, local_counts, cache):
            xr, gr, pr = x_rows.numpy(), go_rows.numpy(), p_rows.numpy()
            dx = np.zeros_like(xr)
            dprob = np.zeros(xr.shape[0])
            for e, (lo, n, g, u, a) in cache.items():
                sl = slice(lo, lo + n)
                dx[sl], dWg, dWu, dWd, dprob[sl] = O.expert_backward(xr[sl], gr[sl], pr[sl], g, u, a, *W.routed(e))
                dW[e] = (dWg, dWu, dWd)
            return torch.from_numpy(dx), torch.from_numpy(dprob)

        shared = {}

        def shared_fwd(h):
            g, u, a, y = O.expert_forward(h.numpy(), *W.shared())
            shared["gua"] = (g, u, a)
            return y

        def shared_bwd(g_out):
            dxs, dWg, dWu, dWd, _ = O.expert_backward(x, g_out.numpy(), np.ones(x.shape[0]), *shared["gua"],
                                                      *W.shared())
            shared["dW"] = (dWg, dWu, dWd)
            return dxs

        def combine(ys, y_back, row_of, pp_):
            out = ys.copy()
            yb, row_of, pp_ = y_back.numpy(), row_of.numpy(), pp_.numpy()
            for s in range(k):                          # slot order, as the layer sums
                v = row_of[:, s] >= 0
                out[v] += pp_[v, s, None] * yb[row_of[v, s]]
            return out

        def unpermute(dxs, dx_back, dprob_back, plan):
            dh = dxs.copy()
            dp = np.zeros((dxs.shape[0], E))
            db, pb = dx_back.numpy(), dprob_back.numpy()
            ro = plan.row_of.numpy()
            for s in range(k):
                v = ro[:, s] >= 0
                dh[v] += db[ro[v, s]]
                dp[np.flatnonzero(v), ids[v, s]] = pb[ro[v, s]]
            return dh, dp

        hidden_t = torch.from_numpy(x)
        out, state = EP.ep_forward(hidden_t, torch.from_numpy(ids), torch.from_numpy(pp), part, experts_fwd,
                                   shared_fwd, combine)
        dh, dp = EP.ep_backward(torch.from_numpy(go), state, experts_bwd, shared_bwd, unpermute)

        # the single-rank oracle over all tokens
        ref_out, cache = O.forward(x_all, probs_all, map_all, W, k)
        ref_dh, ref_dp, grads = O.backward(go_all, cache, W)
        np.testing.assert_allclose(out, ref_out[tl], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dh, ref_dh[tl], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dp, ref_dp[tl], rtol=1e-12, atol=1e-13)
        assert np.all(dp[~rmap] == 0)
        # dispatch bit-exact: the rows each owner holds for expert e are the single-rank
        # permutation's segment of e, in its order
        plan = state["plan"]
        x_rows = state["x_rows"].numpy()
        p_rows = state["p_rows"].numpy()
        pp_all = O.route_pack(map_all, probs_all, k)[1]
        lo = 0
        for j, e in enumerate(part.local(rank)):
            a, b = cache["offsets"][e], cache["offsets"][e + 1]
            n = int(plan.local_counts[j])
            assert n == b - a
            src, slot = cache["perm_src"][a:b], cache["perm_slot"][a:b]
            assert np.array_equal(x_rows[lo:lo + n], x_all[src])
            assert np.array_equal(p_rows[lo:lo + n], pp_all[src, slot])
            lo += n
        for e in part.local(rank):
            if e in grads["routed"]:
                for j in range(3):
                    np.testing.assert_allclose(dW[e][j], grads["routed"][e][j], rtol=1e-12, atol=1e-13)
            else:
                assert e not in dW
        sg = [torch.from_numpy(g.copy()) for g in shared["dW"]]
        for t in sg:
            dist.all_reduce(t)                          # the data-parallel reduction
        for t, key in zip(sg, ("shared_gate", "shared_up", "shared_down")):
            np.testing.assert_allclose(t.numpy(), grads[key], rtol=1e-10, atol=1e-12)
        q.put((rank, "ok"))
    except Exception as ex:                             # reported to the parent
        import traceback
        q.put((rank, traceback.format_exc()))
        raise
    finally:
        dist.destroy_process_group()


def test_partition_is_contiguous_and_covers_every_expert():
    p = EP.ExpertPartition(7, 3)
    assert [list(p.local(r)) for r in range(3)] == [[0, 1, 2], [3, 4], [5, 6]]
    assert [p.owner(e) for e in range(7)] == [0, 0, 0, 1, 1, 2, 2]
    assert p.owners().tolist() == [0, 0, 0, 1, 1, 2, 2]
    with pytest.raises(ValueError):
        EP.ExpertPartition(2, 3)


@pytest.mark.parametrize("name", list(CASES))
def test_expert_parallel_matches_single_rank_oracle(name):
    world = CASES[name].get("world", 2)
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, name, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    results = dict(q.get() for _ in range(world)) if all(p.exitcode == 0 for p in procs) else {}
    for p in procs:
        if p.is_alive():
            p.kill()
    assert results == {r: "ok" for r in range(world)}, (results, [p.exitcode for p in procs])
