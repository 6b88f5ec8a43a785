"""Python side of the oracle contraction (fp64, explicit loops in C).

TEST INFRASTRUCTURE: used by the tests, the smoke check and the bench's CPU
baseline only.

``contract`` runs the plain C loops of ``contract.c`` over the tree in the
network's natural mode order.  ``contract_sliced`` follows §1.1 of "Crossing
the single-GPU memory wall" (slicing): for every assignment of the sliced
modes (lexicographic, first slice mode most significant) it fixes those
indices in the leaves that carry them, contracts the smaller network, and adds
the results in fp64.
"""
from __future__ import annotations

import ctypes
import hashlib
import itertools
import os
import subprocess
from typing import List, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "contract.c")
_BUILD = os.path.join(_HERE, "_build")
_lib = None


def build(force: bool = False) -> str:
    """Compile contract.c with gcc (-O2 -fopenmp) into oracle/_build."""
    with open(_SRC, "rb") as f:
        tag = hashlib.sha1(f.read()).hexdigest()[:12]
    out = os.path.join(_BUILD, f"liboracle_{tag}.so")
    if force or not os.path.exists(out):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC])
        os.replace(tmp, out)
    return out


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_contract.restype = ctypes.c_int
        lib.oracle_contract.argtypes = [
            ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
            ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_void_p),
            ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int,
            ctypes.POINTER(ctypes.c_int), ctypes.c_void_p]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def contract(tensors: Sequence[Sequence[int]], extents: Sequence[int],
             open_modes: Sequence[int], data: Sequence[np.ndarray],
             pairs: Sequence[Tuple[int, int]]) -> np.ndarray:
    """Exact (fp64) value of the network along ``pairs``; result shaped by
    the open modes in the order given."""
    lib = _load()
    n = len(tensors)
    leaves = [np.ascontiguousarray(np.asarray(d, dtype=np.complex128)) for d in data]
    for t, d in enumerate(leaves):
        want = tuple(int(extents[x]) for x in tensors[t])
        if d.shape != want and d.size != int(np.prod(want, dtype=np.int64)):
            raise ValueError(f"leaf {t} has shape {d.shape}, expected {want}")
    ranks = (ctypes.c_int * max(n, 1))(*[len(t) for t in tensors])
    flat = [x for t in tensors for x in t]
    modes = (ctypes.c_int * max(len(flat), 1))(*flat)
    ext = (ctypes.c_longlong * max(len(extents), 1))(*[int(e) for e in extents])
    ptrs = (ctypes.c_void_p * max(n, 1))(*[d.ctypes.data for d in leaves])
    pf = [i for p in pairs for i in p]
    pr = (ctypes.c_int * max(len(pf), 1))(*pf)
    op = (ctypes.c_int * max(len(open_modes), 1))(*open_modes)
    shape = tuple(int(extents[x]) for x in open_modes)
    out = np.zeros(shape, dtype=np.complex128)
    rc = lib.oracle_contract(n, ranks, modes, ext, ptrs, len(pairs), pr,
                             len(open_modes), op, out.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_contract failed with {rc}")
    return out


def slice_leaves(tensors: Sequence[Sequence[int]], data: Sequence[np.ndarray],
                 slices: Sequence[int], values: Sequence[int]):
    """Leaves of the sub-network with sliced mode slices[i] fixed to
    values[i]: the mode disappears from the tensors that carry it."""
    fix = dict(zip(slices, values))
    new_t: List[List[int]] = []
    new_d: List[np.ndarray] = []
    for ms, d in zip(tensors, data):
        idx = tuple(fix[x] if x in fix else slice(None) for x in ms)
        new_t.append([x for x in ms if x not in fix])
        new_d.append(np.asarray(d)[idx])
    return new_t, new_d


def contract_sliced(tensors, extents, open_modes, data, pairs, slices) -> np.ndarray:
    total = None
    ranges = [range(int(extents[x])) for x in slices]
    for vals in itertools.product(*ranges):
        t2, d2 = slice_leaves(tensors, data, slices, vals)
        part = contract(t2, extents, open_modes, d2, pairs)
        total = part if total is None else total + part
    return total
