"""Seeded synthetic inputs (networks, trees, slice sets) for tests and bench.

Holds none of the contraction method's arithmetic: it draws random numbers,
builds leaf arrays and searches for trees.  Both the oracle and the CUDA
path consume its output; neither imports the other.
"""
from .network import Network, Tree, save, load  # noqa: F401
from .circuits import (Circuit, random_circuit, circuit_network,  # noqa: F401
                       grid_circuit_network, inverse_circuit, adjugate_circuit, concat)
from .random_tn import random_network, random_tiny_network, gemm_network  # noqa: F401
from .trees import (greedy_tree, choose_slices, largest_intermediate,  # noqa: F401
                    intermediate_modes, step_volume)
from . import configs  # noqa: F401
