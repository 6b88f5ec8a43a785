"""tn_execute_static: the entry point for callers that cannot allocate
device memory (for instance code that may not allocate after start-up, or a
plugin inside a runtime that owns all device memory).  It runs the same
kernels as tn_execute but on the library's fixed 32 MiB device scratch
array.  Checked here through the C ABI on two calls in a row (the array keeps
the previous call's contents) against the fp64 oracle and against tn_execute,
then tn_execute again after the static calls (the tensor-core maps move back
to the bound workspace); device memory is unchanged by a static call; its
status word is read by tn_plan_check; oversized plans are refused.
This file sorts last so that a failure here never hides another test."""
import numpy as np
import pytest

import exact_tensor_network_gb300 as tn
import oracle
from workloads import configs, greedy_tree, random_network, random_tiny_network, choose_slices
from workloads import largest_intermediate

from helpers import TOL_C64, assert_close, node_network

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _dense_chain():
    """A[i, x] B[x, y] C[y, j]: two 256 x 256 x 256 steps, both on the
    tensor cores (the intermediate is a tensor-core operand)."""
    from workloads.network import Network
    rng = np.random.default_rng(91)

    def rnd(shape):
        return (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)
    net = Network([[0, 1], [1, 2], [2, 3]], [256, 256, 256, 256], [0, 3],
                  [rnd((256, 256)), rnd((256, 256)), rnd((256, 256))], "dense_chain_256")
    return net, [(0, 1), (3, 2)], []


def _cases():
    out = [configs.circuit_3x3_d4()]
    net = random_network(30, 4)
    tree = greedy_tree(net, 0)
    out.append((net, tree, choose_slices(net, tree, largest_intermediate(net, tree) // 4)[:2]))
    t = random_tiny_network(77)
    out.append((t, greedy_tree(t, 1), []))
    out.append(_dense_chain())
    out.append((node_network(384, 320, 512, 5), [(0, 1)], []))
    return out


def _oracle(net, tree, slices):
    if slices:
        return oracle.contract_sliced(net.tensors, net.extents, net.open_modes, net.data, tree,
                                      slices)
    return oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)


def test_cases_include_tensor_core_nodes():
    """The static path re-encodes the tensor-core operand maps for the
    scratch array: some case must exercise them."""
    dense = 0
    for net, tree, sl in _cases():
        h = tn.tn_plan(net.tensors, net.extents, net.open_modes, tree, sl)
        try:
            dense += sum(tn.tn_plan_node_class(h, s) == tn.TN_NODE_DENSE
                         for s in range(tn.tn_plan_num_steps(h)))
        finally:
            tn.tn_plan_destroy(h)
    assert dense >= 3


@pytest.mark.parametrize("idx", range(5))
def test_static_scratch_matches_oracle_and_tn_execute(idx):
    import torch
    net, tree, sl = _cases()[idx]
    dev = torch.device("cuda:0")
    plan = tn.Plan.from_network(net, tree, sl)
    assert plan.workspace_bytes <= 32 << 20
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    ptrs = [x.data_ptr() for x in leaves]
    stream = torch.cuda.current_stream(dev).cuda_stream
    ref = torch.zeros(plan.out_shape, dtype=torch.complex64, device=dev)
    plan.execute(leaves, ref)
    outs = []
    for _ in range(2):
        o = torch.full(plan.out_shape, complex(5.0, 5.0), dtype=torch.complex64, device=dev)
        tn.tn_execute_static(plan.handle, ptrs, o.data_ptr(), stream)
        outs.append(o)
    torch.cuda.synchronize(dev)
    tn.tn_plan_check(plan.handle)          # the static call's status word
    # tn_execute once more: its operand maps point back into the workspace
    again = torch.zeros(plan.out_shape, dtype=torch.complex64, device=dev)
    plan.execute(leaves, again)
    torch.cuda.synchronize(dev)
    plan.check()
    want = _oracle(net, tree, sl)
    first = ref.cpu().numpy().astype(np.complex128)
    assert_close(first, want, TOL_C64, "tn_execute vs oracle")
    for o in outs:
        got = o.cpu().numpy().astype(np.complex128)
        assert_close(got, want, TOL_C64, "static vs oracle")
        assert_close(got, first, 2 * TOL_C64, "static vs tn_execute")
    assert_close(again.cpu().numpy().astype(np.complex128), want, TOL_C64,
                 "tn_execute after static calls vs oracle")


def test_static_call_allocates_nothing():
    import torch
    net, tree, sl = _dense_chain()
    dev = torch.device("cuda:0")
    plan = tn.Plan.from_network(net, tree, sl)
    leaves = [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]
    ptrs = [x.data_ptr() for x in leaves]
    out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    # the first call loads the kernels and looks up the array's address
    tn.tn_execute_static(plan.handle, ptrs, out.data_ptr(), stream)
    torch.cuda.synchronize(dev)
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    reserved0 = torch.cuda.memory_reserved(dev)
    tn.tn_execute_static(plan.handle, ptrs, out.data_ptr(), stream)
    torch.cuda.synchronize(dev)
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert torch.cuda.memory_reserved(dev) == reserved0
    tn.tn_plan_check(plan.handle)
    want = _oracle(net, tree, sl)
    assert_close(out.cpu().numpy().astype(np.complex128), want, TOL_C64, "static vs oracle")


def test_static_scratch_rejects_large_plans():
    import torch
    # chain A[i,a] B[a,j] C[j,l]: the intermediate A.B has 2^24 entries
    # (128 MiB) and lives in the workspace, above the 32 MiB limit
    ext = [4096, 2, 4096, 2]
    tensors = [[0, 1], [1, 2], [2, 3]]
    open_modes = [0, 3]
    h = tn.tn_plan(tensors, ext, open_modes, [(0, 1), (3, 2)])
    try:
        assert tn.tn_plan_workspace_bytes(h) > 32 << 20
        dev = torch.device("cuda:0")
        # correctly sized buffers, so that nothing could go out of bounds
        leaves = [torch.zeros([ext[x] for x in t], dtype=torch.complex64, device=dev)
                  for t in tensors]
        out = torch.zeros([ext[x] for x in open_modes], dtype=torch.complex64, device=dev)
        with pytest.raises(tn.TNError) as e:
            tn.tn_execute_static(h, [x.data_ptr() for x in leaves], out.data_ptr(), 0)
        assert e.value.status == tn.TN_ENOMEM
        assert "static scratch" in str(e.value)
    finally:
        tn.tn_plan_destroy(h)
