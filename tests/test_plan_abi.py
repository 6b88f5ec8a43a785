"""C-ABI library on the host (no GPU): it loads, exports every declared
entry point, and its planner's integer output equals the oracle planner's
exactly (mode orders, m/n/k, C_t, C_s, slice count); malformed inputs are
rejected with TN_EINVAL."""
import ctypes
import functools
import os
import re

import numpy as np
import pytest

import exact_tensor_network_gb300 as tn
from exact_tensor_network_gb300 import build as tnbuild
from oracle import planner
from workloads import (choose_slices, gemm_network, greedy_tree, grid_circuit_network,
                       random_network, random_tiny_network, largest_intermediate)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    tnbuild.build()


def _declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"TN_API\s+[\w\s\*]*?\b(tn_\w+)\s*\(", src))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    names = _declared_symbols()
    assert "tn_plan" in names and "tn_execute" in names
    L = ctypes.CDLL(tn.LIB_PATH)
    for name in names:
        assert hasattr(L, name), name
    # the binding knows them all too
    assert set(names) <= set(tn.SIGNATURES)


@functools.lru_cache(maxsize=1)
def _cases():
    out = []
    net, _ = grid_circuit_network(3, 3, 4, 0)
    out.append((net, greedy_tree(net, 0), []))
    net, _ = grid_circuit_network(4, 4, 8, 5, n_open=3)
    out.append((net, greedy_tree(net, 1), []))
    net = random_network(60, 1, with_data=False)
    tree = greedy_tree(net, 0)
    out.append((net, tree, []))
    out.append((net, tree, choose_slices(net, tree, largest_intermediate(net, tree) // 64)))
    for s in range(24):
        t = random_tiny_network(300 + s)
        out.append((t, greedy_tree(t, s), []))
    out.append((gemm_network(12, 8, 16, 0, with_data=False), [(0, 1)], []))
    return out


@pytest.mark.parametrize("idx", range(29))
def test_planner_matches_oracle_exactly(idx):
    net, tree, sl = _cases()[idx]
    want = planner.plan(net.tensors, net.extents, net.open_modes, tree, sl)
    h = tn.tn_plan(net.tensors, net.extents, net.open_modes, tree, sl)
    try:
        assert tn.tn_plan_flops(h) == want.C_t_total
        assert tn.tn_plan_peak(h) == want.C_s
        assert tn.tn_plan_num_slices(h) == want.n_slices
        assert tn.tn_plan_num_steps(h) == len(tree)
        for tid, order in want.orders.items():
            assert tn.tn_plan_mode_order(h, tid) == order, tid
        for nd in want.nodes:
            assert tn.tn_plan_node_mnk(h, nd.step) == (nd.m, nd.n, nd.k)
        assert tn.tn_plan_workspace_bytes(h) >= 256
    finally:
        tn.tn_plan_destroy(h)


def _err(*args):
    with pytest.raises(tn.TNError) as e:
        tn.tn_plan(*args)
    return e.value.status


def test_rejects_malformed_inputs():
    good = ([[0, 1], [1, 2]], [2, 2, 2], [0, 2], [(0, 1)])
    h = tn.tn_plan(*good)
    tn.tn_plan_destroy(h)
    assert _err([[0, 1], [1, 2], [1]], [2, 2, 2], [0, 2], [(0, 1), (2, 3)]) == tn.TN_EINVAL
    assert _err([[0, 0], [1]], [2, 2], [1], [(0, 1)]) == tn.TN_EINVAL
    assert _err([[0, 1], [1, 2]], [2, 0, 2], [0, 2], [(0, 1)]) == tn.TN_EINVAL
    assert _err([[0, 1], [1, 2]], [2, 2, 2], [0, 2], [(0, 0)]) == tn.TN_EINVAL
    assert _err([[0, 1], [1, 2]], [2, 2, 2], [0, 2], []) == tn.TN_EINVAL
    assert _err([[0, 1], [1, 2]], [2, 2, 2], [0, 2], [(0, 1)], [0]) == tn.TN_EINVAL
    assert _err([[0, 1], [1, 2]], [2, 2, 2], [0, 0, 2], [(0, 1)]) == tn.TN_EINVAL
    assert _err([[0, 1], [1, 2]], [2, 2, 2], [0], [(0, 1)]) == tn.TN_EINVAL
    assert _err([[0, 1], [1, 2]], [2, 2, 2], [0, 2], [(0, 1)], (), 9) == tn.TN_EINVAL
    # 2^40 x 2^40 x 2^40 node: FLOP count overflows 64 bits
    big = [[0, 2], [1, 2]]
    assert _err(big, [1 << 40, 1 << 40, 1 << 40], [0, 1], [(0, 1)]) == tn.TN_EOVERFLOW
    assert "appears in" in tn.tn_last_error(None) or True


def test_workspace_errors_on_host():
    h = tn.tn_plan([[0, 1], [1, 2]], [3, 5, 7], [0, 2], [(0, 1)])
    try:
        need = tn.tn_plan_workspace_bytes(h)
        with pytest.raises(tn.TNError) as e:
            tn.tn_plan_set_workspace(h, 0, need)
        assert e.value.status == tn.TN_EINVAL
        with pytest.raises(tn.TNError) as e:
            tn.tn_plan_set_workspace(h, 4096, need - 1)
        assert e.value.status == tn.TN_ENOMEM
        with pytest.raises(tn.TNError) as e:
            tn.tn_execute(h, [1, 2], 3, 0)
        assert e.value.status == tn.TN_ENOMEM   # nothing bound
        with pytest.raises(tn.TNError) as e:
            tn.tn_execute(h, [0, 2], 3, 0)
        assert e.value.status == tn.TN_EINVAL
    finally:
        tn.tn_plan_destroy(h)


def test_single_leaf_and_scalar_plans():
    h = tn.tn_plan([[0, 1, 2]], [2, 3, 4], [2, 0, 1], [])
    assert tn.tn_plan_flops(h) == 0 and tn.tn_plan_peak(h) == 24
    assert tn.tn_plan_mode_order(h, 0) == [2, 0, 1]
    tn.tn_plan_destroy(h)
    h = tn.tn_plan([[], [0]], [3], [0], [(0, 1)])
    assert tn.tn_plan_node_mnk(h, 0) == (1, 3, 1)
    tn.tn_plan_destroy(h)


def test_hoisting_launch_counts():
    """Hoisting: the first slice runs every launch, each later slice the
    variant ones only; without slices the setting changes nothing."""
    net, _ = grid_circuit_network(4, 4, 8, 3)
    tree = greedy_tree(net, 0)
    sl = choose_slices(net, tree, max(1, largest_intermediate(net, tree) // 16))[:4]
    p = tn.Plan.from_network(net, tree, sl)
    p.set_fusion(False)   # fused leaf subtrees would hold every launch here
    ns = p.num_slices
    assert ns > 1
    on = p.launches
    p.set_hoisting(False)
    off = p.launches
    assert off % ns == 0
    per = off // ns
    assert on < off and (on - per) % (ns - 1) == 0 and (on - per) // (ns - 1) < per
    u = tn.Plan.from_network(net, tree)
    a = u.launches
    u.set_hoisting(False)
    assert u.launches == a


def test_precision_codes():
    """Split bf16 (3) plans like the other precisions; unknown codes fail."""
    net = gemm_network(8, 8, 8, 0)
    h = tn.tn_plan(net.tensors, net.extents, net.open_modes, [(0, 1)], (), tn.TN_PREC_BF16X3)
    assert tn.tn_plan_node_class(h, 0) == tn.TN_NODE_DENSE
    tn.tn_plan_destroy(h)
    with pytest.raises(RuntimeError):
        tn.tn_plan(net.tensors, net.extents, net.open_modes, [(0, 1)], (), 4)


def test_hoisting_workspace_and_replanning():
    """Pinned invariant buffers can only add to the arena; re-planning (a
    policy change) rebuilds both programs and keeps the hoisted count."""
    net, _ = grid_circuit_network(4, 4, 8, 3)
    tree = greedy_tree(net, 0)
    sl = choose_slices(net, tree, max(1, largest_intermediate(net, tree) // 16))[:4]
    p = tn.Plan.from_network(net, tree, sl)
    p.set_fusion(False)   # fused leaf subtrees would hold every launch here
    on_ws, on_l = p.workspace_bytes, p.launches
    p.set_hoisting(False)
    assert p.workspace_bytes <= on_ws and p.launches > on_l
    p.set_hoisting(True)
    assert (p.workspace_bytes, p.launches) == (on_ws, on_l)
    p.set_policy(tn.TN_POLICY_NO_TINY)
    p.set_policy(tn.TN_POLICY_AUTO)
    assert (p.workspace_bytes, p.launches) == (on_ws, on_l)


def test_binding_checks_buffer_sizes():
    """The binding refuses leaves or results whose entry count differs from
    the plan's (a short buffer would be read or written past its end)."""
    import torch
    net = random_tiny_network(404)
    plan = tn.Plan.from_network(net, greedy_tree(net, 0))
    leaves = [torch.from_numpy(np.ascontiguousarray(d)) for d in net.data]
    out = torch.zeros(plan.out_shape, dtype=torch.complex64)
    tn._check_buffers(plan, leaves, out, False, "host")
    big = max(range(len(leaves)), key=lambda i: leaves[i].numel())
    short = list(leaves)
    short[big] = leaves[big].reshape(-1)[:-1].clone()
    with pytest.raises(ValueError, match=f"leaf {big} has"):
        tn._check_buffers(plan, short, out, False, "host")
    with pytest.raises(ValueError, match="result has"):
        tn._check_buffers(plan, leaves, torch.zeros(plan.out_size + 1, dtype=torch.complex64),
                          False, "host")
    with pytest.raises(ValueError, match="leaves given"):
        tn._check_buffers(plan, leaves[:-1], out, False, "host")
    with pytest.raises(ValueError, match="complex64"):
        tn._check_buffers(plan, [x.to(torch.complex128) for x in leaves], out, False, "host")
    # device buffers are required where the call runs on the GPU
    with pytest.raises(ValueError, match="CUDA"):
        tn._check_buffers(plan, leaves, out, True, "execute")


def test_fused_leaf_subtrees_plan():
    """Fused leaf subtrees: the 3x3 circuit (every tensor small) becomes one
    group and one launch; the random network keeps its large steps on their
    kernels; other policies and fusion off leave no fused step."""
    net, _ = grid_circuit_network(3, 3, 4, 0)
    tree = greedy_tree(net, 0)
    p = tn.Plan.from_network(net, tree)
    assert all(p.node_class(s) == tn.TN_NODE_FUSED for s in range(len(tree)))
    assert p.launches == 1
    p.set_fusion(False)
    assert all(p.node_class(s) == tn.TN_NODE_TINY for s in range(len(tree)))
    assert p.launches > 10
    net = random_network(60, 1, with_data=False)
    tree = greedy_tree(net, 0)
    p = tn.Plan.from_network(net, tree)
    cls = [p.node_class(s) for s in range(len(tree))]
    assert tn.TN_NODE_FUSED in cls and tn.TN_NODE_DENSE in cls
    p.set_fusion(False)
    assert tn.TN_NODE_FUSED not in [p.node_class(s) for s in range(len(tree))]
    p.set_fusion(True)
    p.set_policy(tn.TN_POLICY_NO_TINY)
    assert tn.TN_NODE_FUSED not in [p.node_class(s) for s in range(len(tree))]
    # the leaves' and steps' integer plan data do not change with fusion
    p2 = tn.Plan.from_network(net, tree)
    p2.set_fusion(False)
    p3 = tn.Plan.from_network(net, tree)
    for s in range(len(tree)):
        assert p2.node_mnk(s) == p3.node_mnk(s)
    for t in range(net.n_tensors + len(tree)):
        assert p2.mode_order(t) == p3.mode_order(t)


def test_promotion_chunk_and_pairs_settings():
    """The promotion chunk accepts 0 (per plan) or multiples of 32 up to
    4096 and rejects the rest; CTA pairs and the chunk only re-plan."""
    net = random_network(60, 1, with_data=False)
    tree = greedy_tree(net, 0)
    p = tn.Plan.from_network(net, tree)
    ref = [p.node_mnk(s) for s in range(len(tree))]
    for c in (0, 32, 64, 256, 1024, 4096):
        p.set_promotion_chunk(c)
    for bad in (-1, 16, 48, 4128, 8192):
        with pytest.raises(tn.TNError) as e:
            p.set_promotion_chunk(bad)
        assert e.value.status == tn.TN_EINVAL
    p.set_cta_pairs(True)
    p.set_cta_pairs(False)
    assert [p.node_mnk(s) for s in range(len(tree))] == ref
