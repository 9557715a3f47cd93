"""Pins for the oracle's routing steps (route-pack and the dispatch permutation).

Checked against brute force on tiny inputs and against closed forms: counts
sum to the number of valid routes, the permutation is a bijection onto the
valid routes, the force-balanced map has k*T/E tokens per expert.
"""
import itertools

import numpy as np
import pytest

from moe_inputs import config_routing, make_routing
from oracle import moe_oracle as O


def _brute_pack(routing_map, probs, k):
    T, E = routing_map.shape
    ids, pp, over = [], [], []
    for t in range(T):
        row = []
        for e in range(E):
            if routing_map[t][e]:
                row.append(e)
        over.append(len(row) > k)
        row = row[:k] if len(row) <= k else [-1] * k
        ids.append(row + [-1] * (k - len(row)))
        pp.append([float(probs[t][e]) if e >= 0 else 0.0 for e in ids[-1]])
    return np.array(ids), np.array(pp), np.array(over)


@pytest.mark.parametrize("seed", range(6))
def test_route_pack_brute_force(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 9, 5, 3
    m = rng.random((T, E)) < 0.45
    probs = rng.random((T, E)).astype(np.float32)
    ids, pp, over = O.route_pack(m, probs, k)
    bids, bpp, bover = _brute_pack(m, probs, k)
    assert np.array_equal(over, bover)
    ok = ~over
    assert np.array_equal(ids[ok], bids[ok])
    assert np.array_equal(pp[ok], bpp[ok])
    # a missing route gathers prob 0 whatever the dense tensor holds there
    assert np.all(pp[ids < 0] == 0)


def test_route_pack_flags_rows_over_k():
    m = np.array([[1, 1, 1, 0], [1, 0, 0, 0], [0, 0, 0, 0]], bool)
    ids, pp, over = O.route_pack(m, np.ones((3, 4), np.float32), 2)
    assert over.tolist() == [True, False, False]
    assert ids[1].tolist() == [0, -1] and ids[2].tolist() == [-1, -1]
    with pytest.raises(O.RoutingError):
        W = O.DenseWeights(np.zeros((1, 2)), np.zeros((1, 2)), np.zeros((2, 1)),
                           np.zeros((4, 1, 2)), np.zeros((4, 1, 2)), np.zeros((4, 2, 1)))
        O.forward(np.zeros((3, 2)), np.ones((3, 4)), m, W, 2)


def _brute_dispatch(ids, E):
    triples = sorted((int(ids[t, s]), t, s) for t, s in itertools.product(range(ids.shape[0]), range(ids.shape[1]))
                     if ids[t, s] >= 0)
    counts = [sum(1 for e, _, _ in triples if e == x) for x in range(E)]
    return counts, [t for _, t, _ in triples], [s for _, _, s in triples]


@pytest.mark.parametrize("seed", range(6))
def test_dispatch_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    T, E, k = 11, 6, 3
    m = np.zeros((T, E), bool)
    for t in range(T):
        m[t, rng.choice(E, size=int(rng.integers(0, k + 1)), replace=False)] = True
    ids, _, over = O.route_pack(m, np.ones((T, E)), k)
    assert not over.any()
    counts, offsets, perm_src, perm_slot, row_of = O.dispatch_indices(ids, E)
    bc, bsrc, bslot = _brute_dispatch(ids, E)
    assert counts.tolist() == bc
    assert perm_src.tolist() == bsrc and perm_slot.tolist() == bslot
    assert offsets[0] == 0 and offsets[-1] == perm_src.size
    assert np.array_equal(np.diff(offsets), counts)


@pytest.mark.parametrize("cfg", [1, 2, 4, 5])
def test_dispatch_invariants_on_workload_routing(cfg):
    from moe_inputs import CONFIGS
    c = CONFIGS[cfg]
    T = min(c["T"], 2048)
    r = config_routing(cfg, T=T)
    ids, pp, over = O.route_pack(r.routing_map, r.probs, c["k"])
    assert not over.any()
    counts, offsets, perm_src, perm_slot, row_of = O.dispatch_indices(ids, c["E"])
    R = int(r.routing_map.sum())
    assert counts.sum() == R == perm_src.size           # sum of counts = valid routes
    # row_of o perm = identity, and perm is a bijection onto the valid slots
    assert np.array_equal(row_of[perm_src, perm_slot], np.arange(R))
    assert np.array_equal(np.sort(row_of[row_of >= 0]), np.arange(R))
    assert np.all(row_of[ids < 0] == -1)
    # stable: (expert, token) non-decreasing along the permutation
    exp = ids[perm_src, perm_slot]
    key = exp.astype(np.int64) * T + perm_src
    assert np.all(np.diff(key) > 0)
    # each slot's id is on the map and its prob is the dense prob there
    v = ids >= 0
    tt = np.nonzero(v)[0]
    assert np.all(r.routing_map[tt, ids[v]])
    assert np.array_equal(pp[v], r.probs[tt, ids[v]].astype(np.float64))


def test_force_balanced_closed_form():
    # token t -> experts (6t + j) mod 96: every expert gets exactly 6*4096/96 = 256 tokens
    r = config_routing(2, variant="balanced")
    ids, _, _ = O.route_pack(r.routing_map, r.probs, 6)
    counts, *_ = O.dispatch_indices(ids, 96)
    assert np.all(counts == 256)


def test_missing_route_recipes():
    r1 = config_routing(1)
    assert (r1.routing_map.sum(1) == 1).sum() == round(0.05 * 64)
    r5 = make_routing(2048, 128, 8, 5, routing="zipf", drop="multi")
    per_tok = r5.routing_map.sum(1)
    assert per_tok.max() == 8 and per_tok.min() >= 5
    assert (per_tok < 8).sum() == round(0.10 * 2048)
