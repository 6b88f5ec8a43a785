"""Pins for the oracle planner (no GPU).

The planner restates the reverse walk of "Crossing the single-GPU memory
wall" §1.4.  It is pinned by things other than itself:
* the page's own einsum example (§3.1), worked by hand;
* the emergent property of §1.4 (every tensor sorted by remaining lifetime),
  written as an independent sort key;
* the GEMM shape it promises (operand A = [M || K], B = [N || K]);
* closed forms of the FLOP count (8 m n k for a single GEMM node) and an
  independent recount of C_t from plain mode-set products.
"""
import functools
import json
import os

import numpy as np
import pytest

from oracle import planner
from workloads import (gemm_network, greedy_tree, grid_circuit_network,
                       random_network, random_tiny_network, step_volume,
                       choose_slices, largest_intermediate)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _letters_net(spec, extents):
    ins, out = spec.split("->")
    a, b = ins.split(",")
    ids = {ch: i for i, ch in enumerate(sorted(set(a + b)))}
    ext = [extents[ch] for ch in sorted(ids, key=ids.get)]
    return [[ids[c] for c in a], [ids[c] for c in b]], ext, [ids[c] for c in out], ids


def test_einsum_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "einsum_example.json")))
    tensors, ext, open_modes, ids = _letters_net(g["einsum"], g["extents"])
    inv = {v: k for k, v in ids.items()}
    p = planner.plan(tensors, ext, open_modes, [(0, 1)])
    assert "".join(inv[x] for x in p.orders[0]) == g["expected_order_A"]
    assert "".join(inv[x] for x in p.orders[1]) == g["expected_order_B"]
    nd = p.nodes[0]
    assert (nd.m, nd.n, nd.k) == (g["expected_m"], g["expected_n"], g["expected_k"])
    assert p.C_t == g["expected_C_t"]
    assert p.C_s == g["expected_C_s"]


@functools.lru_cache(maxsize=1)
def _networks():
    out = []
    net, _ = grid_circuit_network(3, 3, 4, 0)
    out.append((net, greedy_tree(net, 0)))
    net, _ = grid_circuit_network(4, 4, 8, 5, n_open=3)
    out.append((net, greedy_tree(net, 1)))
    net = random_network(60, 1, with_data=False)
    out.append((net, greedy_tree(net, 0)))
    for s in range(30):
        tn = random_tiny_network(100 + s)
        out.append((tn, greedy_tree(tn, s)))
    return out


@pytest.mark.parametrize("idx", range(33))
def test_reverse_walk_equals_lifetime_sort(idx):
    net, tree = _networks()[idx]
    p = planner.plan(net.tensors, net.extents, net.open_modes, tree)
    cf = planner.closed_form_orders(net.tensors, net.open_modes, tree)
    for t, order in p.orders.items():
        assert order == cf[t], t


@pytest.mark.parametrize("idx", range(33))
def test_every_node_is_transpose_free_gemm(idx):
    net, tree = _networks()[idx]
    p = planner.plan(net.tensors, net.extents, net.open_modes, tree)
    n = net.n_tensors
    for nd in p.nodes:
        oa, ob, oc = p.orders[nd.a], p.orders[nd.b], p.orders[nd.out]
        assert oa == nd.M + nd.K
        assert ob == nd.N + nd.K
        assert sorted(oc) == sorted(nd.M + nd.N)
        # M and N keep the output's relative order
        assert [x for x in oc if x in set(nd.M)] == nd.M
        assert [x for x in oc if x in set(nd.N)] == nd.N
    # the root keeps the user's order
    root = n + len(tree) - 1
    assert p.orders[root] == list(net.open_modes)


@pytest.mark.parametrize("lm,ln,lk", [(8, 8, 8), (8, 12, 16), (16, 8, 12), (12, 12, 12), (16, 16, 16)])
def test_single_gemm_closed_form(lm, ln, lk):
    net = gemm_network(lm, ln, lk, 0, with_data=False)
    p = planner.plan(net.tensors, net.extents, net.open_modes, [(0, 1)])
    m, n, k = 1 << lm, 1 << ln, 1 << lk
    assert (p.nodes[0].m, p.nodes[0].n, p.nodes[0].k) == (m, n, k)
    assert p.C_t == 8 * m * n * k
    assert p.C_s == m * n
    # lifetime-ordered already: leaves need no permutation
    assert p.orders[0] == net.tensors[0]
    assert p.orders[1] == net.tensors[1]


@pytest.mark.parametrize("idx", range(33))
def test_flop_count_recount(idx):
    net, tree = _networks()[idx]
    p = planner.plan(net.tensors, net.extents, net.open_modes, tree)
    assert p.C_t == 8 * step_volume(net, tree)
    assert p.C_s == largest_intermediate(net, tree) or len(tree) == 0


def test_sliced_counts():
    net = random_network(60, 1, with_data=False)
    tree = greedy_tree(net, 0)
    full = planner.plan(net.tensors, net.extents, net.open_modes, tree)
    sl = choose_slices(net, tree, full.C_s // 16)
    p = planner.plan(net.tensors, net.extents, net.open_modes, tree, sl)
    nsl = int(np.prod([net.extents[x] for x in sl]))
    assert p.n_slices == nsl
    assert p.C_t == 8 * step_volume(net, tree, exclude=sl)
    assert p.C_t_total == nsl * p.C_t
    assert p.C_s <= full.C_s // 16
    assert p.C_t_total >= full.C_t
    # orders on the sliced network = unsliced orders with slice modes deleted
    for t, o in p.orders.items():
        assert o == [x for x in full.orders[t] if x not in set(sl)]


def _expect_error(tensors, extents, open_modes, pairs, slices=()):
    with pytest.raises(planner.PlanError):
        planner.plan(tensors, extents, open_modes, pairs, slices)


def test_rejects_malformed():
    good_t = [[0, 1], [1, 2]]
    planner.plan(good_t, [2, 2, 2], [0, 2], [(0, 1)])
    _expect_error([[0, 1], [1, 2], [1]], [2, 2, 2], [0, 2], [(0, 1), (2, 3)])  # hyperedge
    _expect_error([[0, 0], [1]], [2, 2], [1], [(0, 1)])                       # trace
    _expect_error(good_t, [2, 0, 2], [0, 2], [(0, 1)])                        # extent 0
    _expect_error(good_t, [2, 2, 2], [0, 2], [(0, 0)])                        # reuse
    _expect_error(good_t, [2, 2, 2], [0, 2], [])                              # missing step
    _expect_error(good_t, [2, 2, 2], [0, 2], [(0, 1)], [0])                   # sliced open
    _expect_error(good_t, [2, 2, 2], [0, 0, 2], [(0, 1)])                     # open twice
    _expect_error(good_t, [2, 2, 2], [0], [(0, 1)])                           # dangling mode
