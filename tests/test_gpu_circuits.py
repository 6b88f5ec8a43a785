"""Circuit workloads on the GPU (needs a GB300 with ~100 GB free).

The full-size circuits (6x6 x 12 cycles with 64 amplitudes, 7x7 x 10 cycles
sliced 8 ways) are far beyond the fp64 oracle (C_t ~ 6e14 / 7e14 flop), so
they are checked by:
  * scaled twins from the same generator and the same tree recipes, in full
    against the oracle and the state-vector simulator;
  * properties that hold at any size: two different trees (path
    independence) and two different slice sets give the same amplitudes;
  * the largest tensor-core node of each, rebuilt at full size as a
    two-leaf network with its exact mode layout and random entries, checked
    on 1024 sampled outputs recomputed in fp64 from the same leaves.
"""
import numpy as np
import pytest

import exact_tensor_network_gb300 as tn
import oracle
from oracle import planner
from oracle.statevector import amplitudes
from workloads import choose_slices, configs, greedy_tree, grid_circuit_network
from workloads.network import Network
from workloads.trees import largest_intermediate

from helpers import TOL_C64, assert_close, max_rel_err, run_gpu

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


def test_twin_of_6x6_recipe():
    """4x4 grid, 12 cycles, 6 open qubits, C3's tree recipe."""
    net, circ = grid_circuit_network(4, 4, 12, 2, n_open=6)
    tree = greedy_tree(net, 28, noise=0.6, alpha=0.25)
    got, _ = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), TOL_C64, "4x4 d12 twin vs oracle")
    assert_close(got, amplitudes(16, circ.gates, list(range(6))), TOL_C64, "vs statevector")


def test_twin_of_7x7_recipe_sliced():
    """5x5 grid, 10 cycles, scalar amplitude, C5's tree recipe, 3 slices."""
    net, circ = grid_circuit_network(5, 5, 10, 3)
    tree = greedy_tree(net, 11, noise=1.0, alpha=1.0)
    sl = choose_slices(net, tree, largest_intermediate(net, tree) // 8)[:3]
    got, plan = run_gpu(net, tree, sl)
    assert plan.num_slices >= 4
    assert_close(got, _ref(net, tree, sl), TOL_C64, "5x5 d10 sliced twin vs oracle")
    sv = amplitudes(25, circ.gates, [])
    assert abs(complex(got) - complex(sv)) <= TOL_C64 * abs(complex(sv))


def test_twin_with_large_nodes():
    """A deliberately wide tree on a 5x4 grid, 12 cycles: intermediates of
    2^20+ entries put several nodes on the tensor cores."""
    net, circ = grid_circuit_network(5, 4, 12, 2, n_open=4)
    tree = greedy_tree(net, 4, noise=1.0, alpha=0.0)
    p = tn.Plan.from_network(net, tree)
    got, _ = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), TOL_C64, "5x4 d12 wide tree vs oracle")
    assert_close(got, amplitudes(20, circ.gates, list(range(4))), TOL_C64, "vs statevector")


def test_6x6_d12_two_trees_agree():
    """Full size: the C_s = 2^31 tree against a second tree (C_s = 2^33,
    two modes sliced down to 2^31).  Each result is within the complex64
    tolerance of the exact value, so they agree within twice that."""
    net, tree, _ = configs.circuit_6x6_d12()
    a, pa = run_gpu(net, tree)
    tree2 = greedy_tree(net, 3, noise=0.3, alpha=0.5)
    sl2 = choose_slices(net, tree2, 1 << 31)
    b, pb = run_gpu(net, tree2, sl2)
    assert pb.num_slices > 1
    assert a.shape == (2,) * 6
    assert np.all(np.isfinite(a)) and np.abs(a).max() > 0
    assert_close(b, a, 2 * TOL_C64, "6x6 d12: second tree, sliced")
    # Porter-Thomas sanity (reported): over the random single-qubit gates of
    # the last layer, E |<x|C|0>|^2 = 2^-36 for every x, so the mean of
    # 2^36 |amp|^2 over the 64 amplitudes is about 1; the loose bound only
    # catches a gross scale error (the exact-value norm networks pin it)
    pt = float(np.mean(np.abs(a.astype(np.complex128)) ** 2) * 2.0 ** 36)
    print(f"6x6 d12: mean of 2^36 |amp|^2 over 64 amplitudes = {pt:.3f}")
    assert 0.05 < pt < 20


def test_7x7_d10_two_slicings_agree():
    """Full size: 3 sliced modes (C_s 2^32) against 4 (C_s <= 2^31)."""
    net, tree, sl3 = configs.circuit_7x7_d10()
    a, pa = run_gpu(net, tree, sl3)
    _, _, sl4 = configs.circuit_7x7_d10(target_log2=31)
    b, pb = run_gpu(net, tree, sl4)
    assert pa.num_slices == 8 and pb.num_slices > pa.num_slices
    assert np.isfinite(complex(a)) and abs(complex(a)) > 0
    assert_close(b, a, 2 * TOL_C64, "7x7 d10: two slice sets")


def _largest_dense_node(net, tree, slices):
    plan = tn.Plan.from_network(net, tree, slices)
    best = None
    for s in range(len(tree)):
        if plan.node_class(s) != tn.TN_NODE_DENSE:
            continue
        m, n, k = plan.node_mnk(s)
        if best is None or m * n * k > best[0]:
            best = (m * n * k, s)
    return best[1]


@pytest.mark.parametrize("name", ["circuit_6x6_d12", "circuit_7x7_d10"])
def test_largest_node_full_size_sampled(name):
    """The workload's largest tensor-core node at full size: same M, N, K
    extents and the same (possibly interleaved) output order, random N(0,1)
    entries; 1024 sampled outputs against fp64 dot products."""
    import torch
    net, tree, sl = configs.by_name(name, with_data=False)
    s = _largest_dense_node(net, tree, sl)
    op = planner.plan(net.tensors, net.extents, net.open_modes, tree, sl)
    nd = op.nodes[s]
    ext = net.extents
    M, N, K = nd.M, nd.N, nd.K
    out_order = op.orders[nd.out]
    modes = M + N + K
    remap = {x: i for i, x in enumerate(modes)}
    e2 = [ext[x] for x in modes]
    m, n, k = nd.m, nd.n, nd.k
    tensors = [[remap[x] for x in M + K], [remap[x] for x in N + K]]
    open_modes = [remap[x] for x in out_order]
    node_net = Network(tensors, e2, open_modes, None, f"{name}_node{s}")
    plan = tn.Plan.from_network(node_net, [(0, 1)])
    assert plan.node_class(0) == tn.TN_NODE_DENSE
    dev = torch.device("cuda:0")
    # seeded synthetic leaves, generated where they are used (tens of GiB)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(s))
    Ad = torch.randn((m, k), dtype=torch.complex64, device=dev, generator=gen)
    Bd = torch.randn((n, k), dtype=torch.complex64, device=dev, generator=gen)
    out = torch.empty(int(m * n), dtype=torch.complex64, device=dev)
    plan.execute([Ad, Bd], out)
    torch.cuda.synchronize()
    plan.check()
    rng = np.random.default_rng(s)
    rows = rng.integers(0, m, size=1024)
    cols = rng.integers(0, n, size=1024)
    A = Ad[torch.from_numpy(rows).to(dev)].cpu().numpy()     # sampled rows only
    B = Bd[torch.from_numpy(cols).to(dev)].cpu().numpy()
    del Ad, Bd
    # offsets of sampled (i, j) in the output order
    strides = {}
    acc = 1
    for x in reversed(open_modes):
        strides[x] = acc
        acc *= e2[x]

    def offset(idx, side):
        off = 0
        for x in reversed(side):
            d = e2[remap[x]]
            off += (idx % d) * strides[remap[x]]
            idx //= d
        return off
    ref = np.array([np.dot(A[t].astype(np.complex128), B[t].astype(np.complex128))
                    for t in range(len(rows))])
    offs = torch.tensor([offset(int(i), M) + offset(int(j), N) for i, j in zip(rows, cols)],
                        device=dev)
    sampled = out[offs].cpu().numpy()
    r = max_rel_err(sampled.astype(np.complex128), ref)
    assert r <= TOL_C64, f"{name} node {s} ({m}x{n}x{k}): sampled max rel err {r:.3e}"
