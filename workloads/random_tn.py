"""Seeded random connected tensor networks with mixed bond dimensions.

Recipe: every tensor draws an order uniformly from [order_lo, order_hi];
``n_open`` distinct tensors give one of their axes to an open mode; a
spanning tree makes the graph connected; the remaining free axes are paired
at random between distinct, not yet adjacent, nearby tensors, and an axis
that finds no partner is dropped (that tensor's order falls by one).  Every mode
draws its extent uniformly from ``dims``; entries have independent
N(0, 1/2) real and imaginary parts (so E|z|^2 = 1).  Axis order within each
tensor is a random permutation.

Draws random numbers and builds arrays only; none of the contraction method.
"""
from __future__ import annotations

from typing import List, Sequence

import numpy as np

from .network import Network


def random_network(n: int, seed: int, order_lo: int = 3, order_hi: int = 6,
                   dims: Sequence[int] = (2, 4), n_open: int = 4,
                   radius: float = 0.4, name: str = "",
                   with_data: bool = True) -> Network:
    """Random connected network with spatial locality (see module doc).

    Tensors get uniform positions in the unit square.  A spanning tree is
    grown Prim-style (repeatedly join the closest outside tensor to an
    inside tensor that still has a free axis), which keeps the graph
    connected; every remaining free axis then pairs with a uniformly chosen
    tensor within distance ``radius`` that has a free axis and is not yet
    adjacent, else it is dropped.  ``radius`` sets the width of the graph:
    unrestricted pairing (radius >= sqrt 2) gives expander-like graphs whose
    best trees need intermediates far above 2**24 elements.
    """
    rng = np.random.default_rng(seed)
    pos = rng.random((n, 2))
    order = rng.integers(order_lo, order_hi + 1, size=n)
    free = [int(o) for o in order]
    modes_of: List[List[int]] = [[] for _ in range(n)]
    extents: List[int] = []
    adj = [set() for _ in range(n)]
    dist = np.linalg.norm(pos[:, None, :] - pos[None, :, :], axis=-1)

    def new_mode() -> int:
        extents.append(int(rng.choice(np.asarray(dims))))
        return len(extents) - 1

    def join(a: int, b: int) -> None:
        x = new_mode()
        modes_of[a].append(x)
        modes_of[b].append(x)
        free[a] -= 1
        free[b] -= 1
        adj[a].add(b)
        adj[b].add(a)

    open_modes = []
    for t in sorted(rng.choice(n, size=n_open, replace=False).tolist()):
        x = new_mode()
        modes_of[t].append(x)
        free[t] -= 1
        open_modes.append(x)
    rng.shuffle(open_modes)

    inside = [0]
    outside = set(range(1, n))
    while outside:
        best = None
        for i in inside:
            if free[i] <= 0:
                continue
            for j in sorted(outside):
                if best is None or dist[i, j] < best[0]:
                    best = (dist[i, j], i, j)
        _, i, j = best
        join(i, j)
        inside.append(j)
        outside.discard(j)

    stubs = [t for t in range(n) for _ in range(free[t])]
    rng.shuffle(stubs)
    for t in stubs:
        if free[t] <= 0:
            continue
        cand = [u for u in range(n) if u != t and free[u] > 0
                and u not in adj[t] and dist[t, u] <= radius]
        if not cand:
            continue
        join(t, int(cand[rng.integers(len(cand))]))

    tensors = []
    for t in range(n):
        ms = list(modes_of[t])
        rng.shuffle(ms)
        tensors.append(ms)
    data = None
    if with_data:
        data = []
        for ms in tensors:
            shp = tuple(extents[x] for x in ms)
            z = (rng.standard_normal(shp) + 1j * rng.standard_normal(shp)) * np.sqrt(0.5)
            data.append(z.astype(np.complex64))
    return Network(tensors, extents, open_modes, data, name or f"random_tn_{n}_s{seed}")


def random_tiny_network(seed: int, max_bits: int = 16) -> Network:
    """Tiny random network (total index space <= 2**max_bits) for brute-force
    checks: 2..5 tensors, extents 2..4, 0..3 open modes, possibly several
    modes between the same pair and possibly disconnected pieces."""
    rng = np.random.default_rng(seed)
    while True:
        n = int(rng.integers(2, 6))
        n_closed = int(rng.integers(1, 7))
        n_openm = int(rng.integers(0, 4))
        extents: List[int] = []
        tensors: List[List[int]] = [[] for _ in range(n)]
        for _ in range(n_closed):
            a, b = rng.choice(n, size=2, replace=False)
            x = len(extents)
            extents.append(int(rng.integers(2, 5)))
            tensors[a].append(x)
            tensors[b].append(x)
        open_modes = []
        for _ in range(n_openm):
            t = int(rng.integers(n))
            x = len(extents)
            extents.append(int(rng.integers(2, 5)))
            tensors[t].append(x)
            open_modes.append(x)
        total = float(np.prod([float(e) for e in extents]))
        if total > 2.0 ** max_bits:
            continue
        for ms in tensors:
            rng.shuffle(ms)
        rng.shuffle(open_modes)
        data = []
        for ms in tensors:
            shp = tuple(extents[x] for x in ms)
            z = (rng.standard_normal(shp) + 1j * rng.standard_normal(shp)) * np.sqrt(0.5)
            data.append(np.asarray(z, dtype=np.complex64).reshape(shp))
        return Network(tensors, extents, open_modes, data, f"tiny_{seed}")


def gemm_network(log2_m: int, log2_n: int, log2_k: int, seed: int,
                 with_data: bool = True, dtype=np.complex64) -> Network:
    """Two leaves with dimension-2 modes: A = [M || K], B = [N || K], result
    [M || N].  Modes are numbered M first, then N, then K.  Entries have
    independent N(0, 1) real and imaginary parts."""
    M = list(range(log2_m))
    N = list(range(log2_m, log2_m + log2_n))
    K = list(range(log2_m + log2_n, log2_m + log2_n + log2_k))
    extents = [2] * (log2_m + log2_n + log2_k)
    tensors = [M + K, N + K]
    data = None
    if with_data:
        rng = np.random.default_rng(seed)
        data = []
        for ms in tensors:
            shp = (1 << len(ms),)
            re = rng.standard_normal(shp, dtype=np.float32)
            im = rng.standard_normal(shp, dtype=np.float32)
            z = np.empty(shp, dtype=np.complex64)
            z.real = re
            z.imag = im
            data.append(z.reshape([2] * len(ms)))
    return Network(tensors, extents, M + N, data,
                   f"gemm_m2^{log2_m}_n2^{log2_n}_k2^{log2_k}_s{seed}")
