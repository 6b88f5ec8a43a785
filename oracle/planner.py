"""Oracle planner: GEMM-oriented lifetime ordering, node shapes, C_t and C_s.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
baseline may import this package; the product path never does.

Written from the page "Crossing the single-GPU memory wall: multi-GPU
large-scale tensor network contraction" (digest of arXiv 2606.01852):

* §1.1: a pairwise step A x B -> C keeps the modes M (from A) and N (from B)
  and sums over the shared modes K; m, n, k are the products of their
  extents.  The per-step cost formula was lost from the page; the FLOP count
  used here is 8 m n k (one complex multiply-add is 8 real flops), and the
  space of a step is |C| = m n elements.  C_t sums the step costs over the
  tree; C_s is the largest |C|.
* §1.1, slicing: fixing n_slice modes splits the contraction into
  prod(extents) independent sub-contractions whose results add up.
* §1.4, lifetime ordering: the root's order is given by the user; walking the
  steps from the last to the first, a step's output order is already known,
  and each operand takes the output's modes it owns, in the output's
  relative order, followed by the summed modes K.  The page leaves the order
  of K open; here K is ascending by mode id, the same list for A and B.
* §1.4 (emergent property): every tensor ends up sorted by remaining
  lifetime, long-lived modes first.  ``closed_form_orders`` writes that
  property as a sort key so a test can compare both.

Readings where the page is silent: the first id of a step pair is A (its
retained modes form M); open modes are never contracted; a mode id that a
sliced network no longer carries is removed from every tensor before
ordering.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

INF = float("inf")


class PlanError(ValueError):
    pass


@dataclasses.dataclass
class OracleNode:
    step: int
    a: int
    b: int
    out: int
    M: List[int]
    N: List[int]
    K: List[int]
    m: int
    n: int
    k: int
    flops: int


@dataclasses.dataclass
class OraclePlan:
    orders: Dict[int, List[int]]       # tensor id -> mode order
    nodes: List[OracleNode]
    C_t: int                           # per slice, times n_slices below
    C_t_total: int
    C_s: int
    n_slices: int
    slice_modes: List[int]
    death_step: Dict[int, float]


def _prod(extents: Sequence[int], modes: Sequence[int]) -> int:
    p = 1
    for x in modes:
        p *= int(extents[x])
    return p


def validate(tensors: Sequence[Sequence[int]], extents: Sequence[int],
             open_modes: Sequence[int], pairs: Sequence[Tuple[int, int]],
             slices: Sequence[int] = ()) -> None:
    n = len(tensors)
    nm = len(extents)
    count = [0] * nm
    for t in tensors:
        if len(set(t)) != len(t):
            raise PlanError("mode repeated within one tensor")
        for x in t:
            if not 0 <= x < nm:
                raise PlanError("mode id out of range")
            count[x] += 1
    for e in extents:
        if e <= 0:
            raise PlanError("extent must be positive")
    if len(set(open_modes)) != len(open_modes):
        raise PlanError("open mode listed twice")
    op = set(open_modes)
    for x in range(nm):
        want = 1 if x in op else 2
        if count[x] != want:
            raise PlanError(f"mode {x} appears in {count[x]} tensors, expected {want}")
    if len(pairs) != max(n - 1, 0):
        raise PlanError("tree must have n_tensors - 1 steps")
    used = [False] * (n + len(pairs))
    for s, (a, b) in enumerate(pairs):
        for i in (a, b):
            if not 0 <= i < n + s or used[i]:
                raise PlanError("tree reuses or forward-references an id")
            used[i] = True
        if a == b:
            raise PlanError("step contracts a tensor with itself")
    if len(set(slices)) != len(slices):
        raise PlanError("slice mode listed twice")
    for x in slices:
        if not 0 <= x < nm or x in op:
            raise PlanError("only closed modes can be sliced")


def tensor_modes(tensors, pairs, drop=()) -> List[List[int]]:
    """Mode sets (as lists) of leaves and step outputs; an output carries the
    modes of A and B that are not shared (summed)."""
    drop = set(drop)
    ms = [[x for x in t if x not in drop] for t in tensors]
    for a, b in pairs:
        sa, sb = set(ms[a]), set(ms[b])
        ms.append([x for x in ms[a] if x not in sb] + [x for x in ms[b] if x not in sa])
    return ms


def lifetime_orders(tensors, extents, open_modes, pairs, slices=()) -> Dict[int, List[int]]:
    """Reverse walk of §1.4: order(root) = open_modes; for each step from the
    last to the first, order(A) = [order(C) restricted to A] + K and
    order(B) = [order(C) restricted to B] + K, K ascending."""
    n = len(tensors)
    ms = tensor_modes(tensors, pairs, slices)
    root = n + len(pairs) - 1 if pairs else 0
    orders: Dict[int, List[int]] = {root: list(open_modes)}
    if not pairs:
        return orders
    for s in range(len(pairs) - 1, -1, -1):
        a, b = pairs[s]
        c = n + s
        oc = orders[c]
        sa, sb = set(ms[a]), set(ms[b])
        K = sorted(sa & sb)
        orders[a] = [x for x in oc if x in sa] + K
        orders[b] = [x for x in oc if x in sb] + K
    return orders


def death_steps(tensors, open_modes, pairs, slices=()) -> Dict[int, float]:
    """Index of the step that sums each closed mode; open modes live forever."""
    ms = tensor_modes(tensors, pairs, slices)
    d: Dict[int, float] = {x: INF for x in open_modes}
    for s, (a, b) in enumerate(pairs):
        for x in set(ms[a]) & set(ms[b]):
            d[x] = s
    return d


def closed_form_orders(tensors, open_modes, pairs, slices=()) -> Dict[int, List[int]]:
    """Every tensor's modes sorted by remaining lifetime (§1.4's emergent
    property): open modes first, in result order; then closed modes by the
    step that sums them, latest first; ties by ascending mode id."""
    n = len(tensors)
    ms = tensor_modes(tensors, pairs, slices)
    d = death_steps(tensors, open_modes, pairs, slices)
    rank = {x: i for i, x in enumerate(open_modes)}

    def key(x):
        if x in rank:
            return (0, rank[x], 0)
        return (1, -d[x], x)

    total = n + len(pairs)
    return {t: sorted(ms[t], key=key) for t in range(total)}


def plan(tensors, extents, open_modes, pairs, slices: Sequence[int] = ()) -> OraclePlan:
    validate(tensors, extents, open_modes, pairs, slices)
    n = len(tensors)
    sl = list(slices)
    orders = lifetime_orders(tensors, extents, open_modes, pairs, sl)
    ms = tensor_modes(tensors, pairs, sl)
    nodes: List[OracleNode] = []
    C_t = 0
    C_s = 0
    for s, (a, b) in enumerate(pairs):
        c = n + s
        sa, sb = set(ms[a]), set(ms[b])
        K = sorted(sa & sb)
        M = [x for x in orders[c] if x in sa]
        N = [x for x in orders[c] if x in sb]
        m, nn, k = _prod(extents, M), _prod(extents, N), _prod(extents, K)
        f = 8 * m * nn * k
        C_t += f
        C_s = max(C_s, m * nn)
        nodes.append(OracleNode(s, a, b, c, M, N, K, m, nn, k, f))
    if not pairs:
        C_s = _prod(extents, [x for x in tensors[0] if x not in set(sl)]) if tensors else 1
    n_sl = _prod(extents, sl)
    return OraclePlan(orders, nodes, C_t, C_t * n_sl, C_s, n_sl, sl,
                      death_steps(tensors, open_modes, pairs, sl))


def layout_class(node: OracleNode, out_order: Sequence[int]) -> str:
    """Whether C's order is [M || N], [N || M] or interleaves them."""
    mset = set(node.M)
    flags = [x in mset for x in out_order]
    if flags == sorted(flags, reverse=True):
        return "MN"
    if flags == sorted(flags):
        return "NM"
    return "riffle"
