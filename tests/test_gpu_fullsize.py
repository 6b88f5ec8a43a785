"""Full-size checks with an exactly known value, and node-by-node checks of
the real data flow (needs a GB300 with ~120 GB free).

* <0|C' C|0> for a circuit C followed by its inverse C' in adjugate form
  (every stored gate U undone by adj(U) = det(U) U^-1, exactly representable)
  is exactly prod det(U), a closed form computed from the stored gates.  The
  network (no gate simplified away) is contracted as two half states of 2^30
  (5x6 grid, 10 cycles) and 2^32 (5x6 grid, 12 cycles; C_t 1.0e15, more
  than the 6x6 x 12-cycle amplitude workload) entries, joined by one dot
  product: the result must equal the closed form within the complex64
  tolerance.
* Every tensor-core node, and the largest nodes of the other classes, of
  the 6x6 x 12-cycle and 7x7 x 10-cycle workloads, the random 60-tensor
  network and the norm network: the first slice is run up to the node
  (tn_execute_prefix) and sampled rows of its two operands and the outputs
  they give are read back from the workspace (tn_plan_tensor_gather), as
  the node's kernel read and wrote them (formats, K-tiling, arena
  placement, the producer's epilogue); the outputs must equal fp64 dot
  products of the operand rows.
* On networks the oracle finishes, every node's full output and operands
  read back this way equal the oracle's own intermediate-free result
  through the product of the gathered operands, so the read-back itself is
  checked.
"""
import numpy as np
import pytest

import exact_tensor_network_gb300 as tn
import oracle
from workloads import configs

from helpers import TOL_C64, assert_close, check_node_sampled, max_rel_err, node_layout, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _free_bytes():
    import torch
    torch.cuda.empty_cache()
    return torch.cuda.mem_get_info(0)[0]


def exact_norm_value(circuit):
    """<0|C' C|0> with C' the adjugate-form inverse: C' C = prod det(U) over
    C's stored single-qubit gates (CZ has determinant 1 and is its own
    inverse), evaluated in fp64 from the stored complex64 entries."""
    v = 1.0 + 0.0j
    for g in circuit.gates:
        if g[0] == "u":
            u = np.asarray(g[2], dtype=np.complex128)
            v *= u[0, 0] * u[1, 1] - u[0, 1] * u[1, 0]
    return v


@pytest.mark.parametrize("shape", [(4, 4, 8), (5, 6, 10), (5, 6, 12)])
def test_norm_network_exact_value(shape):
    net, tree, _, circ = configs.circuit_norm(*shape)
    plan = tn.Plan.from_network(net, tree)
    if plan.workspace_bytes > _free_bytes() - (8 << 30):
        pytest.skip(f"needs {plan.workspace_bytes / 2**30:.0f} GiB of free device memory")
    want = exact_norm_value(circ)
    if shape == (4, 4, 8):
        ref = oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)
        assert abs(complex(ref) - want) < 1e-12     # the oracle agrees with the closed form
    del plan
    got, plan = run_gpu(net, tree)
    big = max(np.prod(plan.node_mnk(s)) for s in range(len(tree)))
    dense = sum(plan.node_class(s) == tn.TN_NODE_DENSE for s in range(len(tree)))
    assert dense >= 2
    if shape != (4, 4, 8):
        assert plan.peak >= 1 << 30 and big >= 1 << 36
    err = abs(complex(got) - want) / abs(want)
    print(f"norm {shape}: C_s 2^{np.log2(plan.peak):.0f}, C_t {plan.flops:.3e}, "
          f"|got - prod det| / |prod det| = {err:.3e}")
    assert err <= TOL_C64, f"<0|C' C|0> = {complex(got)}, exact {want}"


def _node_steps(plan, n_steps, extra=3):
    """Every tensor-core step, plus the largest `extra` steps (by m n k) of
    the other classes."""
    dense = [s for s in range(n_steps) if plan.node_class(s) == tn.TN_NODE_DENSE]
    # steps inside fused leaf subtrees keep their tensors in shared memory
    other = sorted((s for s in range(n_steps)
                    if plan.node_class(s) not in (tn.TN_NODE_DENSE, tn.TN_NODE_FUSED)),
                   key=lambda s: -int(np.prod(plan.node_mnk(s))))
    return dense + other[:extra]


def _leaves(net, dev):
    import torch
    return [torch.from_numpy(np.ascontiguousarray(d)).to(dev) for d in net.data]


@pytest.mark.parametrize("name", ["circuit_6x6_d12", "circuit_7x7_d10", "random_60", "norm_5x6_d10"])
def test_nodes_of_full_size_workloads(name):
    import torch
    if name == "norm_5x6_d10":
        net, tree, sl, _ = configs.circuit_norm(5, 6, 10)
    else:
        net, tree, sl = configs.by_name(name)
    plan = tn.Plan.from_network(net, tree, sl)
    if plan.workspace_bytes > _free_bytes() - (8 << 30):
        pytest.skip(f"needs {plan.workspace_bytes / 2**30:.0f} GiB of free device memory")
    dev = torch.device("cuda:0")
    leaves = _leaves(net, dev)
    out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    worst = 0.0
    for i, s in enumerate(_node_steps(plan, len(tree))):
        r, mnk = check_node_sampled(plan, net.extents, leaves, out, s, seed=100 + i)
        print(f"{name} step {s} {mnk} class {plan.node_class(s)}: sampled rel err {r:.2e}")
        worst = max(worst, r)
        assert r <= TOL_C64, f"{name} step {s} {mnk}: sampled max rel err {r:.3e}"
    # a full execute afterwards is unaffected by the prefix runs
    plan.execute(leaves, out)
    torch.cuda.synchronize(dev)
    plan.check()


def test_gathered_nodes_match_oracle_product():
    """random_60 (every step): the gathered operands give, in fp64, the
    gathered output of every node entry by entry, and the root's output
    equals the oracle's contraction."""
    import torch
    net, tree, _ = configs.random_60()
    dev = torch.device("cuda:0")
    plan = tn.Plan.from_network(net, tree)
    leaves = _leaves(net, dev)
    out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    fused = 0
    for s in range(len(tree)):
        a, b, c, m, n, k, offm, offn = node_layout(plan, s, net.extents)
        if plan.node_class(s) == tn.TN_NODE_FUSED:
            # its tensors live in a fused group's shared memory only
            fused += 1
            plan.execute_prefix(leaves, out, s)
            with pytest.raises(tn.TNError):
                plan.gather(a, torch.zeros(1, dtype=torch.int64, device=dev))
            continue
        if m * n * k > (1 << 26):
            continue
        plan.execute_prefix(leaves, out, s)
        A = plan.gather(a, torch.arange(m * k, device=dev)).cpu().numpy().reshape(m, k)
        B = plan.gather(b, torch.arange(n * k, device=dev)).cpu().numpy().reshape(n, k)
        I, J = np.meshgrid(np.arange(m), np.arange(n), indexing="ij")
        idx = torch.from_numpy((offm(I.ravel()) + offn(J.ravel())).astype(np.int64)).to(dev)
        C = plan.gather(c, idx).cpu().numpy().reshape(m, n)
        plan.check()
        ref = A.astype(np.complex128) @ B.astype(np.complex128).T
        assert_close(C.astype(np.complex128), ref, TOL_C64, f"step {s} ({m}x{n}x{k})")
    assert fused > 0
    plan.execute(leaves, out)
    torch.cuda.synchronize(dev)
    plan.check()
    ref = oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)
    assert_close(out.cpu().numpy().astype(np.complex128), ref, TOL_C64, "execute after prefix runs")


def test_gather_rejects_other_tensors():
    import torch
    net, tree, _ = configs.circuit_3x3_d4()
    dev = torch.device("cuda:0")
    plan = tn.Plan.from_network(net, tree)
    plan.set_fusion(False)                 # every step in the workspace
    leaves = _leaves(net, dev)
    out = torch.empty(plan.out_shape, dtype=torch.complex64, device=dev)
    idx = torch.zeros(1, dtype=torch.int64, device=dev)
    with pytest.raises(tn.TNError):        # no prefix run yet
        plan.gather(0, idx)
    plan.execute_prefix(leaves, out, 10)
    a, b = plan.pairs[10]
    other = next(t for t in range(net.n_tensors) if t not in (a, b))
    with pytest.raises(tn.TNError):
        plan.gather(other, idx)
    plan.gather(a, idx)
    plan.execute(leaves, out)              # a full execute ends the window
    with pytest.raises(tn.TNError):
        plan.gather(a, idx)
    torch.cuda.synchronize(dev)
    plan.check()
