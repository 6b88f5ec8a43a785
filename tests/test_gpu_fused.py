"""Fused leaf subtrees ("leaf-gate absorption") against the fp64 oracle
(needs a GB300).

Small subtrees near the leaves run as one CTA each, reading their leaves
straight from the caller's buffers and keeping every intermediate in shared
memory.  Checked: whole networks with fusion on and off against the oracle
(circuits with open qubits, random networks of mixed extents, the random
60-tensor network), a network that is one single group whose root is the
tree's root (written, then accumulated over slices), slicing with and
without hoisting, leaves whose storage order differs from their lifetime
order, the launch records, and tn_execute_host / tn_execute_static on fused
plans.
"""
import numpy as np
import pytest

import exact_tensor_network_gb300 as tn
import oracle
from workloads import (choose_slices, configs, greedy_tree, grid_circuit_network,
                       largest_intermediate, random_network, random_tiny_network)

from helpers import TOL_C64, assert_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _ref(net, tree, slices=()):
    if slices:
        return oracle.contract_sliced(net.tensors, net.extents, net.open_modes, net.data, tree,
                                      slices)
    return oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)


def _run(net, tree, slices=(), fuse=True, hoist=True):
    import torch
    dev = torch.device("cuda:0")
    plan = tn.Plan.from_network(net, tree, slices)
    plan.set_fusion(fuse)
    plan.set_hoisting(hoist)
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    out = torch.full(plan.out_shape, complex(3.0, 1.0), dtype=torch.complex64, device=dev)
    plan.execute(leaves, out)
    plan.execute(leaves, out)      # the replayed graph
    torch.cuda.synchronize(dev)
    plan.check()
    fused = sum(plan.node_class(s) == tn.TN_NODE_FUSED for s in range(len(tree)))
    return out.cpu().numpy().astype(np.complex128), fused, plan


@pytest.mark.parametrize("case", ["3x3_d4", "3x3_open3", "4x4_d8_open2", "random_30", "random_60",
                                  "tiny_5", "tiny_17", "tiny_29"])
def test_fused_matches_oracle_and_unfused(case):
    if case == "3x3_d4":
        net, tree, _ = configs.circuit_3x3_d4()
    elif case == "3x3_open3":
        net, _ = grid_circuit_network(3, 3, 4, 0, n_open=3)
        tree = greedy_tree(net, 2)
    elif case == "4x4_d8_open2":
        net, _ = grid_circuit_network(4, 4, 8, 5, n_open=2)
        tree = greedy_tree(net, 1)
    elif case == "random_30":
        net = random_network(30, 4)
        tree = greedy_tree(net, 0)
    elif case == "random_60":
        net, tree, _ = configs.random_60()
    else:
        net = random_tiny_network(int(case.split("_")[1]))
        tree = greedy_tree(net, 3)
    got, fused, _ = _run(net, tree)
    assert fused > 0, "the case must contain a fused group"
    unf, nf, _ = _run(net, tree, fuse=False)
    assert nf == 0
    ref = _ref(net, tree)
    assert_close(got, ref, TOL_C64, f"{case} fused vs oracle")
    assert_close(unf, ref, TOL_C64, f"{case} unfused vs oracle")


def test_whole_network_one_group_sliced():
    """The 3x3 circuit is a single group rooted at the tree's root: it
    writes the output on the first slice and adds on the later ones."""
    net, tree, _ = configs.circuit_3x3_d4()
    sl = choose_slices(net, tree, max(1, largest_intermediate(net, tree) // 8))[:3]
    assert len(sl) >= 1
    for hoist in (True, False):
        got, fused, plan = _run(net, tree, sl, hoist=hoist)
        assert plan.num_slices > 1 and fused == len(tree) and plan.launches == plan.num_slices
        assert_close(got, _ref(net, tree, sl), TOL_C64, f"3x3 sliced hoist={hoist}")


@pytest.mark.parametrize("case", ["circuit_4x4", "random_40"])
def test_fused_with_slices_and_hoisting(case):
    if case == "circuit_4x4":
        net, _ = grid_circuit_network(4, 4, 8, 3)
        tree = greedy_tree(net, 0)
    else:
        net = random_network(40, 2)
        tree = greedy_tree(net, 0)
    sl = choose_slices(net, tree, max(1, largest_intermediate(net, tree) // 16))[:4]
    ref = _ref(net, tree, sl)
    for hoist in (True, False):
        got, fused, plan = _run(net, tree, sl, hoist=hoist)
        assert fused > 0 and plan.num_slices > 1
        assert_close(got, ref, TOL_C64, f"{case} sliced, hoist={hoist}")


def test_fused_leaves_in_caller_order():
    """Leaves stored in an order unlike their lifetime order (reversed
    axes): the group's load does the permutation."""
    net, _ = grid_circuit_network(3, 3, 4, 7, n_open=2)
    tensors, data = [], []
    for t, d in zip(net.tensors, net.data):
        tensors.append(list(reversed(t)))
        data.append(np.ascontiguousarray(np.transpose(d)))
    net.tensors, net.data = tensors, data
    tree = greedy_tree(net, 4)
    got, fused, _ = _run(net, tree)
    assert fused > 0
    assert_close(got, _ref(net, tree), TOL_C64, "reversed leaf axes")


def test_fused_launch_records():
    import torch
    net, tree, _ = configs.random_60()
    dev = torch.device("cuda:0")
    plan = tn.Plan.from_network(net, tree)
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    plan.set_profiling(True)
    plan.execute(leaves, out)
    torch.cuda.synchronize(dev)
    recs = plan.profile()
    assert len(recs) == plan.launches
    fused = [r for r in recs if r["kernel"] == "fused"]
    assert len(fused) == 1 and fused[0]["flops"] > 0 and fused[0]["ms"] > 0
    assert_close(out.cpu().numpy().astype(np.complex128), _ref(net, tree), TOL_C64, "profiled")


def test_fused_host_and_static_calls():
    import torch
    net, tree, _ = configs.circuit_3x3_d4(n_open=2)
    dev = torch.device("cuda:0")
    plan = tn.Plan.from_network(net, tree)
    assert all(plan.node_class(s) == tn.TN_NODE_FUSED for s in range(len(tree)))
    host = [torch.from_numpy(np.ascontiguousarray(d)).pin_memory() for d in net.data]
    hout = torch.empty(plan.out_shape, dtype=torch.complex64).pin_memory()
    dl = [torch.empty_like(h, device=dev) for h in host]
    dout = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    for _ in range(3):             # direct, recorded, replayed
        plan.execute_host(host, hout, dl, dout)
        assert_close(hout.numpy().astype(np.complex128), _ref(net, tree), TOL_C64, "host call")
    o = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    tn.tn_execute_static(plan.handle, [x.data_ptr() for x in dl], o.data_ptr(),
                         torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize(dev)
    plan.check()
    assert_close(o.cpu().numpy().astype(np.complex128), _ref(net, tree), TOL_C64, "static call")
