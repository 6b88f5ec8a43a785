"""Seeded random quantum circuits on a 2-D qubit grid and their tensor networks.

The pages' benchmark circuits (Sycamore / Zuchongzhi-type grid circuits) are
not available; these synthetic circuits have the same structure: a grid of
qubits, Haar-random single-qubit gates on every qubit each cycle, and a layer
of CZ gates on one of four grid-edge patterns per cycle, cycling through
A B C D C D A B (A/B: horizontal edges starting at an even/odd column, C/D:
vertical edges starting at an even/odd row).  A final Haar layer follows the
last cycle.

The tensor network of ``<x|C|0...0>`` has one leaf per |0> input (order 1),
per single-qubit gate (order 2, axes [out, in]), per CZ (order 4, axes
[out_a, out_b, in_a, in_b]) and per <0| projection (order 1).  Qubits listed
as open keep their final wire as an open mode (result axes in that order).

This module draws random numbers and builds arrays; it contains none of the
contraction method.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence, Tuple

import numpy as np

from .network import Network

PATTERN = "ABCDCDAB"


@dataclasses.dataclass
class Circuit:
    rows: int
    cols: int
    # ("u", q, U[2x2]) or ("cz", qa, qb)
    gates: List[tuple]

    @property
    def n_qubits(self) -> int:
        return self.rows * self.cols


def haar_u2(rng: np.random.Generator) -> np.ndarray:
    """Haar-random 2x2 unitary: QR of a complex Ginibre matrix with the
    diagonal phases of R moved into Q (Mezzadri's recipe)."""
    z = (rng.standard_normal((2, 2)) + 1j * rng.standard_normal((2, 2))) / np.sqrt(2.0)
    q, r = np.linalg.qr(z)
    d = np.diag(r)
    return q * (d / np.abs(d))[None, :]


def cz_edges(rows: int, cols: int, kind: str) -> List[Tuple[int, int]]:
    e = []
    if kind in "AB":
        start = 0 if kind == "A" else 1
        for r in range(rows):
            for c in range(start, cols - 1, 2):
                e.append((r * cols + c, r * cols + c + 1))
    else:
        start = 0 if kind == "C" else 1
        for r in range(start, rows - 1, 2):
            for c in range(cols):
                e.append((r * cols + c, (r + 1) * cols + c))
    return e


def random_circuit(rows: int, cols: int, cycles: int, seed: int) -> Circuit:
    rng = np.random.default_rng(seed)
    gates: List[tuple] = []
    n = rows * cols
    for cyc in range(cycles):
        for q in range(n):
            gates.append(("u", q, haar_u2(rng).astype(np.complex64)))
        for a, b in cz_edges(rows, cols, PATTERN[cyc % len(PATTERN)]):
            gates.append(("cz", a, b))
    for q in range(n):
        gates.append(("u", q, haar_u2(rng).astype(np.complex64)))
    return Circuit(rows, cols, gates)


def inverse_circuit(c: Circuit) -> Circuit:
    """C^dagger as a gate list (reverse order, adjoint 1-qubit gates)."""
    inv = []
    for g in reversed(c.gates):
        if g[0] == "u":
            inv.append(("u", g[1], np.conj(g[2].T).astype(np.complex64)))
        else:
            inv.append(g)
    return Circuit(c.rows, c.cols, inv)


def adjugate_circuit(c: Circuit) -> Circuit:
    """The reverse circuit with every single-qubit gate U = [[a, b], [c, d]]
    replaced by its adjugate [[d, -b], [-c, a]] (= det(U) U^-1), and every
    CZ kept (CZ^-1 = CZ).  The adjugate of a stored complex64 gate is
    exactly representable (entries are only moved and negated), so the
    stored circuit followed by this one is exactly prod det(U) times the
    identity, whatever rounding the stored gates carry."""
    adj = []
    for g in reversed(c.gates):
        if g[0] == "u":
            u = np.asarray(g[2], dtype=np.complex64)
            v = np.array([[u[1, 1], -u[0, 1]], [-u[1, 0], u[0, 0]]], dtype=np.complex64)
            adj.append(("u", g[1], v))
        else:
            adj.append(g)
    return Circuit(c.rows, c.cols, adj)


def concat(c1: Circuit, c2: Circuit) -> Circuit:
    assert (c1.rows, c1.cols) == (c2.rows, c2.cols)
    return Circuit(c1.rows, c1.cols, list(c1.gates) + list(c2.gates))


def _cz_tensor() -> np.ndarray:
    t = np.zeros((2, 2, 2, 2), dtype=np.complex64)  # [out_a, out_b, in_a, in_b]
    for a in range(2):
        for b in range(2):
            t[a, b, a, b] = -1.0 if (a == 1 and b == 1) else 1.0
    return t


def circuit_network(c: Circuit, open_qubits: Sequence[int] = (),
                    name: str = "", bits: Sequence[int] = None,
                    open_inputs: Sequence[int] = ()) -> Network:
    """Tensor network of <bits|C|0..0> with ``open_qubits`` left open.

    ``bits`` (default all zero) gives the projected output value of every
    closed qubit.  ``open_inputs`` leaves the input wire of those qubits open
    too (no |0> leaf); the result axes are then the open outputs followed by
    the open inputs, each in the order given.
    """
    n = c.n_qubits
    bits = [0] * n if bits is None else list(bits)
    extents: List[int] = []
    tensors: List[List[int]] = []
    data: List[np.ndarray] = []

    def new_mode() -> int:
        extents.append(2)
        return len(extents) - 1

    wire = [new_mode() for _ in range(n)]
    in_open = list(open_inputs)
    in_modes = {q: wire[q] for q in in_open}
    for q in range(n):
        if q in in_modes:
            continue
        tensors.append([wire[q]])
        data.append(np.array([1.0, 0.0], dtype=np.complex64))
    cz = _cz_tensor()
    for g in c.gates:
        if g[0] == "u":
            q = g[1]
            o = new_mode()
            tensors.append([o, wire[q]])
            data.append(np.asarray(g[2], dtype=np.complex64).copy())
            wire[q] = o
        else:
            a, b = g[1], g[2]
            oa, ob = new_mode(), new_mode()
            tensors.append([oa, ob, wire[a], wire[b]])
            data.append(cz.copy())
            wire[a], wire[b] = oa, ob
    openset = set(open_qubits)
    for q in range(n):
        if q in openset:
            continue
        v = np.zeros(2, dtype=np.complex64)
        v[bits[q]] = 1.0
        tensors.append([wire[q]])
        data.append(v)
    open_modes = [wire[q] for q in open_qubits] + [in_modes[q] for q in in_open]
    return Network(tensors, extents, open_modes, data, name)


def grid_circuit_network(rows: int, cols: int, cycles: int, seed: int,
                         n_open: int = 0, name: str = "") -> Tuple[Network, Circuit]:
    """Amplitudes <x 0..0|C|0..0> with the first ``n_open`` qubits open
    (result axis i = qubit i, ascending)."""
    c = random_circuit(rows, cols, cycles, seed)
    net = circuit_network(c, list(range(n_open)),
                          name or f"circuit_{rows}x{cols}_d{cycles}_s{seed}")
    return net, c
