"""Brute-force value of a small tensor network (no tree at all).

TEST INFRASTRUCTURE: tests only.

The value of a network is, for every assignment of the open modes, the sum
over every assignment of the closed modes of the product of all leaf entries
("Crossing the single-GPU memory wall", §1.1: each pairwise step sums the
shared modes; chaining the steps sums all closed modes of the product).  This
module evaluates that definition directly: each leaf is broadcast over the
full index space of all modes, the leaves are multiplied entry by entry in
complex128, and the closed axes are summed.  It is only usable while the full
index space is small (about 2**22 entries).
"""
from __future__ import annotations

from typing import Sequence

import numpy as np


def brute_force(tensors: Sequence[Sequence[int]], extents: Sequence[int],
                open_modes: Sequence[int], data: Sequence[np.ndarray]) -> np.ndarray:
    used = sorted({x for t in tensors for x in t} | set(open_modes))
    axis = {x: i for i, x in enumerate(used)}
    full = [int(extents[x]) for x in used]
    if int(np.prod(full, dtype=np.int64)) > (1 << 24):
        raise ValueError("index space too large for brute force")
    prod = np.ones(full, dtype=np.complex128)
    for ms, d in zip(tensors, data):
        d = np.asarray(d, dtype=np.complex128).reshape([int(extents[x]) for x in ms])
        # Move the leaf's axes into global mode order, then broadcast.
        order = sorted(range(len(ms)), key=lambda i: axis[ms[i]])
        d = np.transpose(d, order)
        shape = [1] * len(used)
        for i in order:
            shape[axis[ms[i]]] = int(extents[ms[i]])
        prod = prod * d.reshape(shape)
    closed = tuple(axis[x] for x in used if x not in set(open_modes))
    s = prod.sum(axis=closed) if closed else prod
    # Remaining axes are the open modes in ascending id; put them in open order.
    remaining = [x for x in used if x in set(open_modes)]
    perm = [remaining.index(x) for x in open_modes]
    return np.transpose(s, perm) if perm else s
