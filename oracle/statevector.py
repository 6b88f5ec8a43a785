"""Statevector simulation of the generating circuit (complex128).

TEST INFRASTRUCTURE: tests only.

An amplitude <x|C|0..0> of a circuit equals the value of the circuit's tensor
network (the pages' workloads are circuit tensor networks whose results are
amplitudes).  This module applies the gates one by one to the full 2**n state
vector, so it needs no tree and no tensor network at all.  Qubit q is axis q
of the state tensor.
"""
from __future__ import annotations

import numpy as np


def simulate(n_qubits: int, gates) -> np.ndarray:
    """State C|0..0> as an array of shape [2]*n.  ``gates`` holds
    ("u", q, U) with U[out, in] and ("cz", a, b)."""
    psi = np.zeros((2,) * n_qubits, dtype=np.complex128)
    psi[(0,) * n_qubits] = 1.0
    for g in gates:
        if g[0] == "u":
            q, u = g[1], np.asarray(g[2], dtype=np.complex128)
            psi = np.moveaxis(np.tensordot(u, psi, axes=([1], [q])), 0, q)
        else:
            a, b = g[1], g[2]
            idx = [slice(None)] * n_qubits
            idx[a] = 1
            idx[b] = 1
            psi[tuple(idx)] *= -1.0
    return psi


def amplitudes(n_qubits: int, gates, open_qubits, bits=None) -> np.ndarray:
    """<x_open, bits_rest|C|0..0> for all values of the open qubits, axes in
    the order of ``open_qubits``; closed qubits are fixed to ``bits`` (0)."""
    psi = simulate(n_qubits, gates)
    bits = [0] * n_qubits if bits is None else list(bits)
    idx = tuple(slice(None) if q in set(open_qubits) else bits[q] for q in range(n_qubits))
    sub = psi[idx]
    kept = [q for q in range(n_qubits) if q in set(open_qubits)]
    perm = [kept.index(q) for q in open_qubits]
    return np.transpose(sub, perm) if perm else sub
