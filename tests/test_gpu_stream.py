"""Bandwidth-bound (stream) kernel and split-K vs the fp64 oracle (GB300).

Stream nodes have a side of at most 16 entries: gate-like (huge m, tiny n
and k), dot products (m = n = 1), outer products (k = 1), and the swapped
case where m is the small side.  Split-K cuts long k ranges across CTAs and
sums the partials in order; it is used by the stream kernel and the
general CUDA-core kernel when a node alone would not fill the GPU.
"""
import numpy as np
import pytest

import exact_tensor_network_gb300 as tn
import oracle
from workloads import greedy_tree, grid_circuit_network
from workloads.network import Network

from helpers import TOL_BF16, TOL_BF16X3, TOL_C64, assert_close, node_network, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _ref(net, tree):
    return oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)


@pytest.mark.parametrize("m,n,k,cls", [
    (32, 4, 65536, tn.TN_NODE_STREAM),      # split-K dot-like
    (4, 32, 65536, tn.TN_NODE_STREAM),      # swapped
    (1, 1, 262144, tn.TN_NODE_STREAM),      # dot product
    (1 << 20, 2, 2, tn.TN_NODE_STREAM),     # gate-like
    (1 << 16, 16, 16, tn.TN_NODE_STREAM),
    (3, 100000, 1, tn.TN_NODE_STREAM),      # outer product, swapped
    (1000, 7, 300, tn.TN_NODE_STREAM),
    (100003, 5, 3, tn.TN_NODE_STREAM),      # k <= 16, odd: rows kernel, scalar loads
    (70001, 13, 9, tn.TN_NODE_STREAM),      # k = 9 padded to 16
    (65536, 3, 8, tn.TN_NODE_STREAM),       # k = 8: 16-byte loads
    (1 << 18, 1, 4, tn.TN_NODE_STREAM),     # n = 1
    (33, 2, 1, tn.TN_NODE_STREAM),          # fewer rows than one pass
    (100, 90, 5000, tn.TN_NODE_SIMT),       # split SIMT tiles
    (70, 300, 1001, tn.TN_NODE_SIMT),       # k odd: not tensor-core eligible
    (17, 17, 17, tn.TN_NODE_SIMT),
])
def test_stream_and_split_nodes(m, n, k, cls):
    """Class expected with tiny batching off; then the same node under the
    default policy (where small ones go to the tiny-node kernel)."""
    net = node_network(m, n, k, m * 7 + n * 3 + k)
    p = tn.Plan.from_network(net, [(0, 1)], (), "tf32x3", tn.TN_POLICY_NO_TINY)
    assert p.node_class(0) == cls
    ref = _ref(net, [(0, 1)])
    got, _ = run_gpu(net, [(0, 1)], policy=tn.TN_POLICY_NO_TINY)
    assert_close(got, ref, TOL_C64, f"node {m}x{n}x{k}")
    got2, _ = run_gpu(net, [(0, 1)])
    assert_close(got2, ref, TOL_C64, f"node {m}x{n}x{k} default policy")


def test_split_root_with_slices_accumulates():
    net = node_network(32, 4, 4096, 5)
    # slice the contracted mode by replacing it with two modes of 64 each
    rng = np.random.default_rng(2)
    a = net.data[0].reshape(32, 64, 64)
    b = net.data[1].reshape(4, 64, 64)
    net2 = Network([[0, 2, 3], [1, 2, 3]], [32, 4, 64, 64], [0, 1], [a, b])
    got, plan = run_gpu(net2, [(0, 1)], slices=[2])
    assert plan.num_slices == 64
    assert_close(got, _ref(net2, [(0, 1)]), TOL_C64, "sliced split-K root")


@pytest.mark.parametrize("rows,cols,cycles,n_open", [(4, 4, 8, 0), (4, 5, 10, 4), (5, 5, 8, 2)])
def test_circuits(rows, cols, cycles, n_open):
    net, _ = grid_circuit_network(rows, cols, cycles, rows * cols + cycles, n_open=n_open)
    tree = greedy_tree(net, 0)
    got, _ = run_gpu(net, tree)
    assert_close(got, _ref(net, tree), TOL_C64, f"circuit {rows}x{cols} d{cycles}")


def test_gate_like_root_with_slices_accumulates():
    # A[i, x, z] B[j, x, z] -> root[i, j], z sliced: k = 4 per slice, so the
    # row-streaming kernel writes slice 0 and adds slices 1 and 2
    rng = np.random.default_rng(12)
    ext = [50001, 3, 4, 3]                 # i j x z
    def rnd(shape):
        return ((rng.standard_normal(shape) + 1j * rng.standard_normal(shape)) * 0.5).astype(np.complex64)
    net = Network([[0, 2, 3], [1, 2, 3]], ext, [0, 1], [rnd((50001, 4, 3)), rnd((3, 4, 3))])
    plan = tn.Plan.from_network(net, [(0, 1)], [3], "tf32x3", tn.TN_POLICY_NO_TINY)
    assert plan.node_class(0) == tn.TN_NODE_STREAM and plan.num_slices == 3
    got, _ = run_gpu(net, [(0, 1)], slices=[3], policy=tn.TN_POLICY_NO_TINY)
    assert_close(got, _ref(net, [(0, 1)]), TOL_C64, "sliced gate-like root")


def _rnd(rng, shape):
    return ((rng.standard_normal(shape) + 1j * rng.standard_normal(shape)) * 0.5).astype(np.complex64)


@pytest.mark.parametrize("m", [20, 8 * 152 * 8 + 3, 100003])
def test_gate16_rows_ragged(m):
    """n = k = 16 (four-lane rows, B in registers): row counts that leave a
    partial group of 8 rows and a partial last pass over the grid."""
    net = node_network(m, 16, 16, m + 11)
    p = tn.Plan.from_network(net, [(0, 1)], (), "tf32x3", tn.TN_POLICY_NO_TINY)
    assert p.node_class(0) == tn.TN_NODE_STREAM
    got, _ = run_gpu(net, [(0, 1)], policy=tn.TN_POLICY_NO_TINY)
    assert_close(got, _ref(net, [(0, 1)]), TOL_C64, f"gate16 m={m}")


def test_gate16_transposed_root():
    """n = k = 16 with the root's axes in the order (j, i): the entries of a
    row are not contiguous, so each lane stores its four outputs one by one
    through the separable offsets."""
    rng = np.random.default_rng(21)
    ext = [30001, 2, 2, 2, 2, 2, 2, 2, 2]   # i, j0..j3, x0..x3
    a = _rnd(rng, (30001, 2, 2, 2, 2))
    b = _rnd(rng, (2, 2, 2, 2, 2, 2, 2, 2))
    net = Network([[0, 5, 6, 7, 8], [1, 2, 3, 4, 5, 6, 7, 8]], ext, [1, 2, 3, 4, 0], [a, b])
    p = tn.Plan.from_network(net, [(0, 1)], (), "tf32x3", tn.TN_POLICY_NO_TINY)
    assert p.node_class(0) == tn.TN_NODE_STREAM
    got, _ = run_gpu(net, [(0, 1)], policy=tn.TN_POLICY_NO_TINY)
    assert_close(got, _ref(net, [(0, 1)]), TOL_C64, "gate16 transposed root")


@pytest.mark.parametrize("prec", ["tf32x3", "bf16x3", "bf16"])
def test_gate16_feeds_tensor_core_node(prec):
    """An n = k = 16 node whose output is an operand of a tensor-core node:
    the gate kernel writes the consumer's planar (K-tiled) format."""
    rng = np.random.default_rng(22)
    # modes: a(256) b(256) x(16) j(16) l(256)
    ext = [256, 256, 16, 16, 256]
    A = _rnd(rng, (256, 256, 16))
    B = _rnd(rng, (16, 16))
    D = _rnd(rng, (256, 16, 256))
    net = Network([[0, 1, 2], [3, 2], [1, 3, 4]], ext, [0, 4], [A, B, D])
    tree = [(0, 1), (3, 2)]
    p = tn.Plan.from_network(net, tree, (), prec, tn.TN_POLICY_NO_TINY)
    assert p.node_class(0) == tn.TN_NODE_STREAM and p.node_class(1) == tn.TN_NODE_DENSE
    got, _ = run_gpu(net, tree, precision=prec, policy=tn.TN_POLICY_NO_TINY)
    tol = {"tf32x3": TOL_C64, "bf16x3": TOL_BF16X3, "bf16": TOL_BF16}[prec]
    assert_close(got, _ref(net, tree), tol, f"gate16 -> dense ({prec})")


def test_gate16_root_with_slices_accumulates():
    """n = k = 16 root summed over three slices (write, then add twice)."""
    rng = np.random.default_rng(23)
    ext = [40000, 16, 16, 3]                 # i j x z
    net = Network([[0, 2, 3], [1, 2, 3]], ext, [0, 1], [_rnd(rng, (40000, 16, 3)), _rnd(rng, (16, 16, 3))])
    plan = tn.Plan.from_network(net, [(0, 1)], [3], "tf32x3", tn.TN_POLICY_NO_TINY)
    assert plan.node_class(0) == tn.TN_NODE_STREAM and plan.num_slices == 3
    got, _ = run_gpu(net, [(0, 1)], slices=[3], policy=tn.TN_POLICY_NO_TINY)
    assert_close(got, _ref(net, [(0, 1)]), TOL_C64, "sliced gate16 root")
