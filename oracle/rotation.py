"""Offline calibration fixture of OSCAR, float64 (test infrastructure only).

Source: the OSCAR technical summaries on gist.science (Dutch and French pages),
section 2.2 "algorithm design", phase A "offline calibration":

* covariance targets C_Q = (1/N) sum_n q_n^T q_n (query-aware key target) and
  C_S = (1/N) V^T S^T S V (score-aware value target);
* an eigendecomposition of each gives the eigenbases U_Q and U_S;
* the composite rotations are R_K = U_Q H_Had P_br and R_V = U_S H_Had P_br;
* per-layer clip thresholds are estimated from rotated calibration activations.
The arXiv abstract (paperdot page) adds that rotations and clip thresholds are
fixed per layer.

Readings taken where the pages are silent (each listed in the design notes):
row-vector convention x' = x R; eigenvectors as columns sorted by descending
eigenvalue, each column's largest-magnitude entry made positive; H is the
natural-order Sylvester matrix scaled by 1/sqrt(d); (x P_br)_j = x_{br(j)};
one R_K and one R_V per layer shared by all KV heads (C_Q pools every query
head, C_S pools every query head's attention output); the clip threshold is the
99.9th percentile (linear interpolation) of |rotated calibration values|.
"""
from __future__ import annotations

import numpy as np


def sylvester_hadamard(d: int) -> np.ndarray:
    """Orthonormal Sylvester Hadamard matrix of order d (power of two), float64.

    Built by the doubling recursion H_{2n} = [[H_n, H_n], [H_n, -H_n]] from
    H_1 = [1], then scaled by 1/sqrt(d) so that H H^T = I.
    """
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(d)


def bit_reversal(d: int) -> np.ndarray:
    """br[j] = j with its log2(d) bits reversed."""
    nbits = d.bit_length() - 1
    if 1 << nbits != d:
        raise ValueError("d must be a power of two")
    out = np.zeros(d, dtype=np.int64)
    for j in range(d):
        r = 0
        for b in range(nbits):
            if j >> b & 1:
                r |= 1 << (nbits - 1 - b)
        out[j] = r
    return out


def bit_reversal_matrix(d: int) -> np.ndarray:
    """Permutation matrix P_br with (x P_br)_j = x_{br(j)}, i.e. P[br(j), j] = 1."""
    br = bit_reversal(d)
    p = np.zeros((d, d), dtype=np.float64)
    p[br, np.arange(d)] = 1.0
    return p


def query_covariance(q_rows: np.ndarray) -> np.ndarray:
    """C_Q = (1/N) sum_n q_n^T q_n over N query row vectors, float64 [d, d]."""
    q = np.asarray(q_rows, dtype=np.float64).reshape(-1, np.shape(q_rows)[-1])
    return q.T @ q / q.shape[0]


def causal_softmax_scores(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """S = causal softmax(q k^T / sqrt(d)) for one head: q, k [T, d] -> S [T, T]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    t, d = q.shape
    logits = q @ k.T / np.sqrt(d)
    mask = np.tril(np.ones((t, t), dtype=bool))
    logits = np.where(mask, logits, -np.inf)
    logits -= logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    return e / e.sum(axis=1, keepdims=True)


def score_covariance(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """C_S = (1/N) sum_h V_h^T S_h^T S_h V_h, float64 [d, d].

    q: [T, Hq, d]; k, v: [T, Hkv, d].  Query head h reads KV head
    h // (Hq/Hkv).  N = T * Hq, the number of attention-output rows pooled.
    """
    t, hq, d = q.shape
    hkv = k.shape[1]
    grp = hq // hkv
    acc = np.zeros((d, d), dtype=np.float64)
    for h in range(hq):
        kv = h // grp
        s = causal_softmax_scores(q[:, h, :], k[:, kv, :])
        sv = s @ np.asarray(v[:, kv, :], dtype=np.float64)
        acc += sv.T @ sv
    return acc / (t * hq)


def eigenbasis(c: np.ndarray) -> np.ndarray:
    """Eigenvectors of the symmetric matrix c as columns, by descending eigenvalue.

    Sign rule: the entry of largest magnitude in each column is made positive.
    """
    c = np.asarray(c, dtype=np.float64)
    c = 0.5 * (c + c.T)
    w, u = np.linalg.eigh(c)
    order = np.argsort(-w, kind="stable")
    u = u[:, order]
    piv = np.argmax(np.abs(u), axis=0)
    sign = np.sign(u[piv, np.arange(u.shape[1])])
    sign[sign == 0] = 1.0
    return u * sign[None, :]


def composite_rotation(u: np.ndarray) -> np.ndarray:
    """R = U . H_Had . P_br (float64)."""
    d = u.shape[0]
    return np.asarray(u, dtype=np.float64) @ sylvester_hadamard(d) @ bit_reversal_matrix(d)


def clip_threshold(x_rows: np.ndarray, r: np.ndarray, pct: float = 99.9) -> float:
    """99.9th percentile (linear interpolation) of |x R| over all rows and channels."""
    x = np.asarray(x_rows, dtype=np.float64).reshape(-1, r.shape[0])
    return float(np.percentile(np.abs(x @ np.asarray(r, dtype=np.float64)), pct))


def to_f32(x) -> np.ndarray:
    """Round a float64 array to the float32 values handed to the GPU path."""
    return np.asarray(x, dtype=np.float32)


def layer_fixture(q_cal: np.ndarray, k_cal: np.ndarray, v_cal: np.ndarray, u_identity: bool = False) -> dict:
    """Per-layer calibration artefacts from calibration activations.

    q_cal [T, Hq, d], k_cal / v_cal [T, Hkv, d].  Returns the float64 rotations,
    their float32 roundings (what both sides use for write and decode), and the
    float32 clip thresholds.  ``u_identity`` gives the data-oblivious
    Hadamard-only rotation R = H P (U = I) used as an ablation baseline.
    """
    d = q_cal.shape[-1]
    if u_identity:
        u_q = np.eye(d)
        u_s = np.eye(d)
    else:
        u_q = eigenbasis(query_covariance(q_cal.reshape(-1, d)))
        u_s = eigenbasis(score_covariance(q_cal, k_cal, v_cal))
    r_k = composite_rotation(u_q)
    r_v = composite_rotation(u_s)
    r_k32 = to_f32(r_k)
    r_v32 = to_f32(r_v)
    clip_k = np.float32(clip_threshold(k_cal, r_k32.astype(np.float64)))
    clip_v = np.float32(clip_threshold(v_cal, r_v32.astype(np.float64)))
    return {"R_K64": r_k, "R_V64": r_v, "R_K": r_k32, "R_V": r_v32,
            "clip_K": clip_k, "clip_V": clip_v, "U_Q": u_q, "U_S": u_s}


def head_fixture(q_cal: np.ndarray, k_cal: np.ndarray, v_cal: np.ndarray) -> dict:
    """Per-kv-head calibration artefacts (a variant of the pages' fixed per-layer rotation): kv head h
    gets R_K[h] = U_Q,h H P from the queries of its own query-head group and R_V[h] = U_S,h H P from
    its own attention outputs; the clip thresholds stay per layer, the 99.9th percentile of
    |x R_h| over every head.

    q_cal [T, Hq, d], k_cal / v_cal [T, Hkv, d] -> R_K, R_V [Hkv, d, d] (float64 and float32).
    """
    d = q_cal.shape[-1]
    hkv = k_cal.shape[1]
    grp = q_cal.shape[1] // hkv
    r_k, r_v = [], []
    for h in range(hkv):
        qh = q_cal[:, h * grp:(h + 1) * grp]
        r_k.append(composite_rotation(eigenbasis(query_covariance(qh.reshape(-1, d)))))
        r_v.append(composite_rotation(eigenbasis(score_covariance(qh, k_cal[:, h:h + 1], v_cal[:, h:h + 1]))))
    r_k, r_v = np.stack(r_k), np.stack(r_v)
    r_k32, r_v32 = to_f32(r_k), to_f32(r_v)
    rot_k = np.concatenate([np.asarray(k_cal[:, h], np.float64) @ r_k32[h].astype(np.float64) for h in range(hkv)])
    rot_v = np.concatenate([np.asarray(v_cal[:, h], np.float64) @ r_v32[h].astype(np.float64) for h in range(hkv)])
    clip_k = np.float32(np.percentile(np.abs(rot_k), 99.9))
    clip_v = np.float32(np.percentile(np.abs(rot_v), 99.9))
    return {"R_K64": r_k, "R_V64": r_v, "R_K": r_k32, "R_V": r_v32, "clip_K": clip_k, "clip_V": clip_v}
