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
"""
from __future__ import annotations

import functools
from typing import List, Tuple

from .circuits import grid_circuit_network
from .network import Network, Tree
from .random_tn import gemm_network, random_network
from .trees import choose_slices, greedy_tree, largest_intermediate

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
