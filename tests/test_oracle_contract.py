"""Pins for the oracle contraction (no GPU).

The fp64 explicit-loop contraction is checked against things that do not
share its code or its route:
* the definition summed over every index assignment (brute force, no tree);
* state-vector simulation of the circuit that generated the network;
* unitarity (sum over all output bitstrings of |amp|^2 = 1);
* C^dagger C = identity, as a network with no simplification;
* path independence (two different trees);
* slicing (sum of sub-contractions = unsliced value, §1.1);
* a chain of matrices, whose value is a plain matrix product.
"""
import numpy as np
import pytest

import oracle
from oracle.brute import brute_force
from oracle.statevector import amplitudes
from workloads import (circuit_network, concat, greedy_tree, grid_circuit_network,
                       inverse_circuit, random_circuit, random_network,
                       random_tiny_network, choose_slices, largest_intermediate)
from workloads.network import Network


def _c(net, tree):
    return oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)


@pytest.mark.parametrize("seed", range(120))
def test_matches_brute_force(seed):
    net = random_tiny_network(seed)
    tree = greedy_tree(net, seed, noise=0.5)
    got = _c(net, tree)
    want = brute_force(net.tensors, net.extents, net.open_modes, net.data)
    assert got.shape == want.shape
    scale = max(1.0, float(np.abs(want).max()))
    assert np.abs(got - want).max() <= 1e-12 * scale


@pytest.mark.parametrize("rows,cols,cycles,n_open,seed", [
    (3, 3, 4, 0, 0), (3, 3, 4, 3, 1), (4, 4, 8, 0, 2), (3, 4, 6, 4, 3), (4, 4, 6, 6, 4)])
def test_matches_statevector(rows, cols, cycles, n_open, seed):
    net, circ = grid_circuit_network(rows, cols, cycles, seed, n_open=n_open)
    tree = greedy_tree(net, seed)
    got = _c(net, tree)
    want = amplitudes(rows * cols, circ.gates, list(range(n_open)))
    assert got.shape == want.shape
    assert np.abs(got - want).max() <= 1e-12


def test_unitarity_all_open():
    net, _ = grid_circuit_network(3, 3, 4, 7, n_open=9)
    got = _c(net, greedy_tree(net, 3))
    # the gates are stored in complex64, so each is unitary only to about
    # 1e-7; 45 of them leave the norm within a few 1e-6 of one
    assert abs(float(np.sum(np.abs(got) ** 2)) - 1.0) < 1e-5


def test_identity_network():
    c = random_circuit(3, 3, 4, 11)
    cc = concat(c, inverse_circuit(c))
    net = circuit_network(cc, [])
    v = _c(net, greedy_tree(net, 0))
    assert abs(complex(v) - 1.0) < 1e-6   # single-precision gate entries
    # two qubits open at both ends: the 4x4 identity
    net2 = circuit_network(cc, [0, 1], open_inputs=[0, 1])
    m = _c(net2, greedy_tree(net2, 1)).reshape(4, 4)
    assert np.abs(m - np.eye(4)).max() < 1e-6


def test_path_independence():
    net = random_network(40, 3)
    a = _c(net, greedy_tree(net, 0))
    b = _c(net, greedy_tree(net, 5, noise=0.8))
    assert np.abs(a - b).max() <= 1e-11 * np.abs(a).max()


@pytest.mark.parametrize("which", ["random", "circuit"])
def test_slicing_sums_to_unsliced(which):
    if which == "random":
        net = random_network(30, 2)
    else:
        net, _ = grid_circuit_network(4, 4, 6, 9, n_open=2)
    tree = greedy_tree(net, 0)
    full = _c(net, tree)
    sl = choose_slices(net, tree, largest_intermediate(net, tree) // 8)[:3]
    assert len(sl) >= 1
    parts = oracle.contract_sliced(net.tensors, net.extents, net.open_modes, net.data, tree, sl)
    assert np.abs(parts - full).max() <= 1e-11 * np.abs(full).max()


def test_matrix_chain_closed_form():
    rng = np.random.default_rng(0)
    dims = [3, 5, 2, 4, 6]
    mats = [(rng.standard_normal((dims[i], dims[i + 1])) +
             1j * rng.standard_normal((dims[i], dims[i + 1]))).astype(np.complex64)
            for i in range(4)]
    # modes 0..4 along the chain; mode 0 and 4 open
    tensors = [[i, i + 1] for i in range(4)]
    net = Network(tensors, dims, [0, 4], mats)
    want = mats[0].astype(np.complex128)
    for mtx in mats[1:]:
        want = want @ mtx.astype(np.complex128)
    for tree in ([(0, 1), (4, 2), (5, 3)], [(2, 3), (1, 4), (0, 5)], [(3, 2), (0, 1), (5, 4)]):
        got = _c(net, tree)
        assert np.abs(got - want).max() <= 1e-12 * np.abs(want).max()
    # transposed root order
    net_t = Network(tensors, dims, [4, 0], mats)
    assert np.abs(_c(net_t, [(0, 1), (4, 2), (5, 3)]) - want.T).max() <= 1e-12 * np.abs(want).max()


def test_single_leaf_and_scalars():
    rng = np.random.default_rng(1)
    d = (rng.standard_normal((2, 3, 4)) + 0j).astype(np.complex64)
    net = Network([[0, 1, 2]], [2, 3, 4], [2, 0, 1], [d])
    assert np.abs(_c(net, []) - np.transpose(d, (2, 0, 1))).max() == 0
    s = np.array(2.5 - 1j, dtype=np.complex64)
    net2 = Network([[], [0]], [3], [0], [s, d[0, :, 0].copy()])
    assert np.abs(_c(net2, [(0, 1)]) - s * d[0, :, 0]).max() < 1e-6


def test_adjugate_inverse_closed_form():
    """A circuit followed by its inverse written with adjugates is exactly
    prod det(U) times the identity (adj(U) U = det(U) I for each stored
    2x2 gate; CZ undoes itself).  The oracle, run on the half-state tree of
    that network, must give the closed form to fp64 rounding."""
    from workloads import configs
    net, tree, _, circ = configs.circuit_norm(4, 4, 8)
    want = 1.0 + 0.0j
    for g in circ.gates:
        if g[0] == "u":
            u = np.asarray(g[2], dtype=np.complex128)
            want *= u[0, 0] * u[1, 1] - u[0, 1] * u[1, 0]
    assert abs(abs(want) - 1.0) < 1e-5        # the stored gates are nearly unitary
    got = complex(oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree))
    assert abs(got - want) < 1e-12
    # the same network with the plain adjoint as inverse is only 1 to the
    # gates' complex64 rounding
    from workloads import inverse_circuit
    net2 = circuit_network(concat(circ, inverse_circuit(circ)), ())
    got2 = complex(oracle.contract(net2.tensors, net2.extents, net2.open_modes, net2.data, tree))
    assert 1e-9 < abs(got2 - 1.0) < 1e-5
