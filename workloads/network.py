"""Plain container for a tensor network, a contraction tree and a slice set.

This module only holds data and does file I/O; it computes nothing of the
contraction method.  Conventions (shared by every consumer):

* ``tensors[t]`` lists the mode ids of leaf ``t`` in its storage order;
  storage is row-major, the last listed mode varies fastest.
* ``extents[x]`` is the dimension of mode ``x``.
* ``open_modes`` are the modes left in the result, in the order of the
  result's axes (row-major, last fastest).  Every other mode is closed and
  appears in exactly two leaves; an open mode appears in exactly one.
* ``data[t]`` is a complex64 numpy array of shape
  ``[extents[x] for x in tensors[t]]``.
* A tree is a list of ``(a, b)`` pairs in SSA form: step ``s`` consumes the
  ids ``a`` and ``b`` (leaves are ``0..n-1``, the output of step ``s`` is
  ``n + s``); the last step produces the root.
"""
from __future__ import annotations

import dataclasses
import json
from typing import List, Optional, Sequence, Tuple

import numpy as np


@dataclasses.dataclass
class Network:
    tensors: List[List[int]]
    extents: List[int]
    open_modes: List[int]
    data: Optional[List[np.ndarray]] = None
    name: str = ""

    @property
    def n_tensors(self) -> int:
        return len(self.tensors)

    @property
    def n_modes(self) -> int:
        return len(self.extents)

    def shape(self, t: int) -> Tuple[int, ...]:
        return tuple(int(self.extents[x]) for x in self.tensors[t])

    def closed_modes(self) -> List[int]:
        op = set(self.open_modes)
        used = sorted({x for ms in self.tensors for x in ms})
        return [x for x in used if x not in op]

    def out_shape(self) -> Tuple[int, ...]:
        return tuple(int(self.extents[x]) for x in self.open_modes)

    def to_json(self) -> dict:
        return {
            "name": self.name,
            "tensors": [list(map(int, t)) for t in self.tensors],
            "extents": list(map(int, self.extents)),
            "open_modes": list(map(int, self.open_modes)),
        }


Tree = List[Tuple[int, int]]


def save(path: str, net: Network, tree: Optional[Tree] = None,
         slices: Optional[Sequence[int]] = None) -> None:
    """Write ``path``.json (structure) and ``path``.npz (leaf values)."""
    meta = net.to_json()
    meta["tree"] = [list(map(int, p)) for p in tree] if tree is not None else None
    meta["slices"] = list(map(int, slices)) if slices is not None else []
    with open(path + ".json", "w") as f:
        json.dump(meta, f)
    if net.data is not None:
        np.savez(path + ".npz", *net.data)


def load(path: str):
    with open(path + ".json") as f:
        meta = json.load(f)
    data = None
    try:
        z = np.load(path + ".npz")
        data = [z["arr_%d" % i] for i in range(len(meta["tensors"]))]
    except FileNotFoundError:
        pass
    net = Network(meta["tensors"], meta["extents"], meta["open_modes"], data,
                  meta.get("name", ""))
    tree = [tuple(p) for p in meta["tree"]] if meta.get("tree") else None
    return net, tree, meta.get("slices", [])
