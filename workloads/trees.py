"""Seeded contraction-tree and slice-mode choosers (input tools).

The pages take their trees and slice sets from an external path finder; these
plain heuristics stand in for it.  A tree is an input to both the planner and
the oracle: they share the tree, not code.  Sizes here are plain products of
extents over mode sets, computed for the search only.
"""
from __future__ import annotations

import heapq
from typing import Dict, FrozenSet, List, Sequence, Tuple

import numpy as np

from .network import Network, Tree


def _prod(extents: Sequence[int], modes) -> int:
    p = 1
    for x in modes:
        p *= int(extents[x])
    return p


def greedy_tree(net: Network, seed: int, noise: float = 0.0,
                exclude: Sequence[int] = (), alpha: float = 1.0) -> Tree:
    """Repeatedly contract the pair of live tensors sharing a mode that
    minimises |out| - alpha (|a| + |b|) (ties broken by a seeded random key;
    with ``noise`` > 0 the score is also multiplied by a random factor in
    [1-noise, 1+noise] for positive scores).  Tensors with nothing in common
    are joined at the end, smallest first.  Modes in ``exclude`` are
    treated as absent (extent 1), as when they are sliced."""
    rng = np.random.default_rng(seed)
    ext = list(net.extents)
    for x in exclude:
        ext[x] = 1
    n = net.n_tensors
    live: Dict[int, FrozenSet[int]] = {t: frozenset(net.tensors[t]) for t in range(n)}
    owners: Dict[int, set] = {}
    for t, ms in live.items():
        for x in ms:
            owners.setdefault(x, set()).add(t)
    size = {t: _prod(ext, ms) for t, ms in live.items()}
    heap: List[Tuple[float, float, int, int]] = []

    def push(a: int, b: int) -> None:
        out = live[a] ^ live[b]
        score = float(_prod(ext, out)) - alpha * float(size[a] + size[b])
        if noise > 0.0:
            f = 1.0 + noise * (2.0 * rng.random() - 1.0)
            score = score * f if score > 0 else score / f
        heapq.heappush(heap, (score, rng.random(), min(a, b), max(a, b)))

    seen = set()
    for x, ts in owners.items():
        ts = sorted(ts)
        for i in range(len(ts)):
            for j in range(i + 1, len(ts)):
                if (ts[i], ts[j]) not in seen:
                    seen.add((ts[i], ts[j]))
                    push(ts[i], ts[j])
    tree: Tree = []
    next_id = n
    while len(live) > 1:
        pair = None
        while heap:
            _, _, a, b = heapq.heappop(heap)
            if a in live and b in live:
                pair = (a, b)
                break
        if pair is None:
            by_size = sorted(live, key=lambda t: (size[t], t))
            pair = (by_size[0], by_size[1])
        a, b = pair
        out = live[a] ^ live[b]
        c = next_id
        next_id += 1
        tree.append((a, b))
        for t in (a, b):
            for x in live[t]:
                owners[x].discard(t)
            del live[t]
        live[c] = out
        size[c] = _prod(ext, out)
        nb = set()
        for x in out:
            owners.setdefault(x, set()).add(c)
            nb |= owners[x]
        nb.discard(c)
        for t in nb:
            push(t, c)
    return tree


def intermediate_modes(net: Network, tree: Tree) -> List[FrozenSet[int]]:
    """Mode set of every step's output (closed modes meet in exactly two
    tensors, so the output keeps the symmetric difference)."""
    ms: List[FrozenSet[int]] = [frozenset(t) for t in net.tensors]
    outs = []
    for a, b in tree:
        c = ms[a] ^ ms[b]
        ms.append(c)
        outs.append(c)
    return outs


def largest_intermediate(net: Network, tree: Tree, exclude: Sequence[int] = ()) -> int:
    ext = list(net.extents)
    for x in exclude:
        ext[x] = 1
    return max([1] + [_prod(ext, c) for c in intermediate_modes(net, tree)])


def step_volume(net: Network, tree: Tree, exclude: Sequence[int] = ()) -> int:
    """Sum over steps of the product of extents over all modes the step
    touches (search score for slice choice)."""
    ext = list(net.extents)
    for x in exclude:
        ext[x] = 1
    ms: List[FrozenSet[int]] = [frozenset(t) for t in net.tensors]
    tot = 0
    for a, b in tree:
        tot += _prod(ext, ms[a] | ms[b])
        ms.append(ms[a] ^ ms[b])
    return tot


def choose_slices(net: Network, tree: Tree, target: int, max_modes: int = 64) -> List[int]:
    """Greedy slice choice: while some intermediate exceeds ``target``
    elements, slice the closed mode, among those present in every such
    intermediate (or, failing that, in the largest one), that gives the
    smallest step volume; ties go to the lowest mode id."""
    chosen: List[int] = []
    inter = intermediate_modes(net, tree)
    closed = set(net.closed_modes())
    while len(chosen) < max_modes:
        ext = list(net.extents)
        for x in chosen:
            ext[x] = 1
        big = [c for c in inter if _prod(ext, c) > target]
        if not big:
            break
        common = set.intersection(*[set(c) for c in big]) & closed
        common -= set(chosen)
        if not common:
            largest = max(big, key=lambda c: _prod(ext, c))
            common = (set(largest) & closed) - set(chosen)
        best = min(sorted(common), key=lambda x: step_volume(net, tree, chosen + [x]))
        chosen.append(best)
    return chosen


def split_tree(net: Network, part_a: Sequence[int], tree_a: Tree, part_b: Sequence[int],
               tree_b: Tree) -> Tree:
    """A tree of ``net`` that contracts the leaves ``part_a`` along
    ``tree_a`` (a tree of the sub-network of those leaves, in its own SSA
    numbering), then ``part_b`` along ``tree_b``, then joins the two
    results.  ``part_a`` + ``part_b`` must list every leaf once."""
    n = net.n_tensors
    assert sorted(list(part_a) + list(part_b)) == list(range(n))
    out: Tree = []

    def emit(part, sub_tree):
        ids = {i: int(t) for i, t in enumerate(part)}
        for s, (a, b) in enumerate(sub_tree):
            out.append((ids[a], ids[b]))
            ids[len(part) + s] = n + len(out) - 1
        return ids[len(part) + len(sub_tree) - 1] if sub_tree else ids[0]

    ra = emit(part_a, tree_a)
    rb = emit(part_b, tree_b)
    out.append((ra, rb))
    return out
