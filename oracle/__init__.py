"""Oracle for the exact tensor-network contraction path.

TEST INFRASTRUCTURE.  Plain, slow, obviously correct CPU code that the GPU
path is checked against.  Only ``tests/``, the smoke check and the bench's
CPU-baseline leg may import it; the library never does, and this package
imports nothing of the library.

* ``planner``: lifetime ordering, node shapes, C_t, C_s, slice count.
* ``contract``: fp64 explicit-loop contraction along a tree (C, OpenMP).
* ``brute``: the definition summed over all index assignments (tiny only).
* ``statevector``: circuit amplitudes by state-vector simulation.
"""
from . import planner, brute, statevector  # noqa: F401
from .contract import contract, contract_sliced, slice_leaves, build, num_threads  # noqa: F401
