"""The named synthetic workloads (seeded; recipes in the module docs).

* ``circuit_3x3_d4``: 3x3 qubit grid, 4 cycles + final layer, CZ gates,
  amplitude <0..0|C|0..0>, greedy tree (seed 0).  75 leaves, 74 steps.
* ``random_60``: 60-tensor random network (orders 3..6, bond extents drawn
  from {2, 4}, N(0, 1/2) entries, 4 open modes, spatial locality radius
  0.4); the generator seed is the first s >= 1 whose greedy tree (seed 0)
  has its largest intermediate in [2**23, 2**24] elements.
* ``circuit_6x6_d12``: 6x6 grid, 12 cycles, 6 open qubits (64 amplitudes).
* ``gemm_m{a}_n{b}_k{c}``: one GEMM-aligned node with dimension-2 modes.
* ``circuit_7x7_d10``: 7x7 grid, 10 cycles, scalar amplitude, sliced.
* ``circuit_norm(rows, cols, cycles)``: <0|C' C|0> of a grid circuit and
  its inverse in adjugate form (value exactly prod det(U)), contracted as
  two half states joined by one dot product.
"""
from __future__ import annotations

import functools
from typing import List, Tuple

from .circuits import grid_circuit_network
from .network import Network, Tree
from .circuits import adjugate_circuit, circuit_network, concat, random_circuit
from .random_tn import gemm_network, random_network
from .trees import choose_slices, greedy_tree, largest_intermediate, split_tree

C2_LO, C2_HI = 1 << 23, 1 << 24


@functools.lru_cache(maxsize=None)
def random_60_seed(max_seed: int = 200) -> int:
    for s in range(1, max_seed):
        net = random_network(60, s, with_data=False)
        cs = largest_intermediate(net, greedy_tree(net, 0))
        if C2_LO <= cs <= C2_HI:
            return s
    raise RuntimeError("no seed gives the requested intermediate size")


def circuit_3x3_d4(n_open: int = 0) -> Tuple[Network, Tree, List[int]]:
    net, _ = grid_circuit_network(3, 3, 4, 0, n_open=n_open, name="circuit_3x3_d4")
    return net, greedy_tree(net, 0), []


def random_60(with_data: bool = True) -> Tuple[Network, Tree, List[int]]:
    s = random_60_seed()
    net = random_network(60, s, with_data=with_data, name=f"random_60_s{s}")
    return net, greedy_tree(net, 0), []


def circuit_6x6_d12(with_data: bool = True) -> Tuple[Network, Tree, List[int]]:
    """6x6 grid, 12 cycles, qubits 0..5 open (64 amplitudes), circuit seed 2.

    Tree: greedy with score |out| - 0.25 (|a| + |b|), multiplicative noise
    0.6, seed 28: the only tree with C_s <= 2^31 found by a search over
    alpha in {0.25, 0.5, 0.75} x noise in {0.1, 0.3, 0.6} x seeds 0..59
    (plain greedy gives 2^36).  C_s = 2^31, C_t = 5.9e14.
    """
    net, _ = grid_circuit_network(6, 6, 12, 2, n_open=6, name="circuit_6x6_d12")
    return net, greedy_tree(net, 28, noise=0.6, alpha=0.25), []


def circuit_7x7_d10(with_data: bool = True, target_log2: int = 32):
    """7x7 grid, 10 cycles, scalar amplitude <0..0|C|0..0>, circuit seed 3.

    Tree: greedy, alpha 1, noise 1.0, seed 11: the cheapest (smallest C_t)
    of the trees with an unsliced C_s of exactly 2^35 among alpha in
    {0.5, 1} x noise in {0, 0.3, 1} x seeds 0..23.  Slice modes: greedy
    choice down to C_s <= 2^target_log2 (2^32: 3 modes, 8 slices, no extra
    flops over the unsliced C_t of 7.27e14).
    """
    net, _ = grid_circuit_network(7, 7, 10, 3, n_open=0, name="circuit_7x7_d10")
    tree = greedy_tree(net, 11, noise=1.0, alpha=1.0)
    return net, tree, choose_slices(net, tree, 1 << target_log2)


# tree recipes of the half states (alpha, noise, seed), from a search over
# alpha in {1, 0.5, 0.25, 0} x noise in {0, 0.3, 0.6} x seeds 0..3 for the
# smallest largest intermediate (then the smallest C_t)
NORM_RECIPES = {(5, 6, 12): (0.0, 0.6, 3), (5, 6, 10): (1.0, 0.6, 3), (4, 4, 8): (1.0, 0.3, 0)}


def circuit_norm(rows: int, cols: int, cycles: int, seed: int = 2):
    """The network of <0..0|C' C|0..0> for a random grid circuit C (cycles
    as in the other circuits, final Haar layer included) followed by its
    inverse C' written with adjugates (adjugate_circuit): C' C is exactly
    prod det(U) over C's single-qubit gates times the identity, so the
    value is known exactly (a unit complex number up to the gates'
    complex64 rounding).  No gate is simplified away: the C half (inputs
    |0> and C's gates) and the C' half (C''s gates and the <0| projections)
    are each contracted by a greedy tree into the full state of rows x cols
    qubits, and the last step is their dot product over the qubit wires
    between C and C'.  Returns (net, tree, [], circuit C)."""
    c = random_circuit(rows, cols, cycles, seed)
    nq = rows * cols
    net = circuit_network(concat(c, adjugate_circuit(c)), (),
                          f"circuit_norm_{rows}x{cols}_d{cycles}")
    ng = len(c.gates)
    split = nq + ng   # |0> leaves and C's gates come first
    part_a, part_b = list(range(split)), list(range(split, net.n_tensors))
    alpha, noise, tseed = NORM_RECIPES.get((rows, cols, cycles), (1.0, 0.3, 0))
    modes = [x for t in part_a for x in net.tensors[t]]
    count = {}
    for x in modes:
        count[x] = count.get(x, 0) + 1
    sub = Network([net.tensors[t] for t in part_a], net.extents,
                  sorted(x for x, k in count.items() if k == 1), None)
    tree_a = greedy_tree(sub, tseed, noise=noise, alpha=alpha)
    # The C' half is the mirror image of the C half: gate i of C faces gate
    # ng - 1 - i of C' and the |0> input of qubit q the <0| projection of q,
    # with the same mode-sharing pattern, so the mirror of tree_a contracts
    # it through intermediates of the same sizes.
    # local index in the C' half of the mirror of leaf t of the C half
    def mirror(t):
        if t < nq:                  # |0> of qubit t -> <0| of qubit t
            return ng + t
        return ng - 1 - (t - nq)    # gate i of C -> gate ng - 1 - i of C'
    assert net.n_tensors == 2 * (nq + ng)
    local_b = [mirror(t) for t in part_a]
    tree_b = [(local_b[a] if a < split else a, local_b[b] if b < split else b) for a, b in tree_a]
    return net, split_tree(net, part_a, tree_a, part_b, tree_b), [], c


def gemm(lm: int, ln: int, lk: int, seed: int = 0, with_data: bool = True):
    net = gemm_network(lm, ln, lk, seed, with_data=with_data)
    return net, [(0, 1)], []


def by_name(name: str, with_data: bool = True):
    if name == "circuit_3x3_d4":
        return circuit_3x3_d4()
    if name == "random_60":
        return random_60(with_data)
    if name == "circuit_6x6_d12":
        return circuit_6x6_d12(with_data)
    if name == "circuit_7x7_d10":
        return circuit_7x7_d10(with_data)
    if name.startswith("gemm_"):
        fields = name.split("_")[1:]
        lm = int(fields[0][1:])
        ln = int(fields[1][1:])
        lk = int(fields[2][1:])
        return gemm(lm, ln, lk, with_data=with_data)
    raise KeyError(name)
