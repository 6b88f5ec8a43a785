"""tn_execute_static: the entry point for callers that cannot allocate
device memory (for instance code that may not allocate after start-up, or a
plugin inside a runtime that owns all device memory).  It runs the same
kernels as tn_execute but on the library's fixed 32 MiB device scratch
array.  Checked here against tn_execute through the C ABI, on two calls in a
row (the array keeps the previous call's contents), and for the size limit.
This file sorts last so that a failure here never hides another test."""
import numpy as np
import pytest

import exact_tensor_network_gb300 as tn
from workloads import configs, greedy_tree, random_network, random_tiny_network, choose_slices
from workloads import largest_intermediate

from helpers import TOL_C64, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _cases():
    out = [configs.circuit_3x3_d4()]
    net = random_network(30, 4)
    tree = greedy_tree(net, 0)
    out.append((net, tree, choose_slices(net, tree, largest_intermediate(net, tree) // 4)[:2]))
    t = random_tiny_network(77)
    out.append((t, greedy_tree(t, 1), []))
    return out


@pytest.mark.parametrize("idx", range(3))
def test_static_scratch_matches_tn_execute(idx):
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
    want = ref.cpu().numpy().astype(np.complex128)
    for o in outs:
        assert_close(o.cpu().numpy().astype(np.complex128), want, TOL_C64, "static vs tn_execute")


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
