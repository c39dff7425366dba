"""Offline OSCAR calibration: per-layer rotations R_K, R_V and clip thresholds.

This is the offline phase of OSCAR (gist.science technical summary, section
2.2 A; arXiv abstract: "fixed per-layer rotations and clipping thresholds"),
run once on calibration activations before serving.  It is not part of the
serving hot path, which only consumes its outputs (float32 R matrices and two
float32 clip values per layer).

Steps, for one layer with calibration queries q [T, Hq, d] and keys / values
k, v [T, Hkv, d]:
  C_Q = (1/N) sum over every query row of q^T q            (query-aware key target)
  C_S = (1/N) sum over query heads of (S V)^T (S V),       (score-aware value target)
        S = causal softmax(q k^T / sqrt(d)), query head h reads kv head h // (Hq/Hkv)
  U   = eigenvectors of C, descending eigenvalue, each column's largest-magnitude
        entry positive
  R   = U . H . P_br with H the 1/sqrt(d)-scaled Sylvester Hadamard matrix and
        (x P_br)_j = x_{bitreverse(j)}
  clip = 99.9th percentile (linear interpolation) of |x R| over the calibration rows.
"""
from __future__ import annotations

import numpy as np


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_ij = (-1)^popcount(i & j) / sqrt(d)."""
    i = np.arange(d)
    bits = np.bitwise_and(i[:, None], i[None, :])
    parity = np.zeros_like(bits)
    while bits.any():
        parity ^= bits & 1
        bits >>= 1
    return np.where(parity == 1, -1.0, 1.0) / np.sqrt(d)


def bitrev_indices(d: int) -> np.ndarray:
    n = int(np.log2(d))
    j = np.arange(d)
    out = np.zeros(d, dtype=np.int64)
    for b in range(n):
        out |= ((j >> b) & 1) << (n - 1 - b)
    return out


def rotation_from_basis(u: np.ndarray) -> np.ndarray:
    d = u.shape[0]
    return (u @ hadamard(d))[:, bitrev_indices(d)]


def sorted_eigvecs(c: np.ndarray) -> np.ndarray:
    w, u = np.linalg.eigh((c + c.T) / 2)
    u = u[:, np.argsort(w)[::-1]]
    idx = np.abs(u).argmax(axis=0)
    s = np.sign(u[idx, np.arange(u.shape[1])])
    s[s == 0] = 1
    return u * s


def key_target(q: np.ndarray) -> np.ndarray:
    rows = q.reshape(-1, q.shape[-1]).astype(np.float64)
    return rows.T @ rows / rows.shape[0]


def value_target(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    t, hq, d = q.shape
    grp = hq // k.shape[1]
    out = np.zeros((d, d))
    causal = np.triu(np.ones((t, t), dtype=bool), 1)
    for h in range(hq):
        qh = q[:, h].astype(np.float64)
        kh = k[:, h // grp].astype(np.float64)
        vh = v[:, h // grp].astype(np.float64)
        z = qh @ kh.T / np.sqrt(d)
        z[causal] = -np.inf
        z = np.exp(z - z.max(axis=1, keepdims=True))
        o = (z / z.sum(axis=1, keepdims=True)) @ vh
        out += o.T @ o
    return out / (t * hq)


def calibrate_layer(q: np.ndarray, k: np.ndarray, v: np.ndarray, hadamard_only: bool = False,
                    pct: float = 99.9) -> dict:
    """Rotations (float32, row-major [d, d]) and clip thresholds for one layer."""
    d = q.shape[-1]
    if hadamard_only:
        r_k = r_v = rotation_from_basis(np.eye(d))
    else:
        r_k = rotation_from_basis(sorted_eigvecs(key_target(q)))
        r_v = rotation_from_basis(sorted_eigvecs(value_target(q, k, v)))
    r_k32 = np.ascontiguousarray(r_k, dtype=np.float32)
    r_v32 = np.ascontiguousarray(r_v, dtype=np.float32)
    clip_k = np.float32(np.percentile(np.abs(k.reshape(-1, d).astype(np.float64) @ r_k32.astype(np.float64)), pct))
    clip_v = np.float32(np.percentile(np.abs(v.reshape(-1, d).astype(np.float64) @ r_v32.astype(np.float64)), pct))
    return {"R_K": r_k32, "R_V": r_v32, "clip_K": float(clip_k), "clip_V": float(clip_v)}
