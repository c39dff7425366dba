"""Decode attention over the mixed-precision paged cache, float64 (test infrastructure only).

Source: the OSCAR technical summaries on gist.science, section 2.2 B ("kernel
integration"): the serving kernel unpacks, dequantises and inverse-rotates the
INT2 history and computes attention over it, compatible with paged attention
and prefix caching; the arXiv abstract (paperdot page) describes fused decode
kernels.  History is stored after rotation, so the keys and values the model
attends to are K_hat = Y_K R_K^T and V_hat = Y_V R_V^T; sink and recent tokens
are stored unrotated in BF16.

``decode`` is the plain definition: reconstruct K_hat, V_hat, concatenate the
BF16 window, softmax(q K^T / sqrt(d)) V per query head, exact float64, with
max subtraction, no mask or soft-cap (every cached token is visible to the
token being decoded).  ``decode_fused`` is the serving-side rearrangement
(rotate q once, accumulate history in the rotated basis, apply R_V^T once);
the two must agree to rounding.  Query head h reads KV head h // (Hq/Hkv).
``extend`` is the chunked-prefill counterpart: new query tokens attend to a
cached prefix (as stored) and causally to their own chunk.
"""
from __future__ import annotations

import numpy as np

from . import quant
from .cache import CacheImage


def softmax_attention(q, k, v) -> np.ndarray:
    """Textbook attention for one query head: q [d], k, v [N, d] -> [d], float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    logits = k @ q / np.sqrt(q.shape[-1])
    logits = logits - logits.max()
    p = np.exp(logits)
    return (p / p.sum()) @ v


def token_sets(n: int, sink: int, recent: int):
    """(history tokens, window tokens) of a sequence of length n."""
    hist = np.arange(sink, max(sink, n - recent), dtype=np.int64)
    win = np.concatenate([np.arange(0, min(sink, n)), np.arange(max(sink, n - recent), n)]).astype(np.int64)
    return hist, win


def _gather(cache: CacheImage, layer: int, b: int, n: int, block_table, req_slot):
    g = cache.g
    hist, win = token_sets(n, g.sink, g.recent)
    bt = np.asarray(block_table)
    if hist.size:
        pages = bt[b, hist // g.page_size]
        ck, sk, zk, cv, sv, zv = cache.read_history(layer, pages, hist % g.page_size)
        yk = quant.dequantize(ck, sk, zk, g.group_size)   # [M, Hkv, d], rotated basis
        yv = quant.dequantize(cv, sv, zv, g.group_size)
    else:
        yk = np.zeros((0, g.n_kv_heads, g.head_dim))
        yv = np.zeros((0, g.n_kv_heads, g.head_dim))
    wk = np.zeros((win.size, g.n_kv_heads, g.head_dim))
    wv = np.zeros_like(wk)
    for i, t in enumerate(win):
        wk[i], wv[i] = cache.read_window(layer, int(req_slot[b]), int(t))
    return yk, yv, wk, wv


def unrotate(y, r) -> np.ndarray:
    """x_hat = y R^T for history rows y [n, Hkv, d]: r is [d, d] (shared by every kv head) or
    [Hkv, d, d] (head h rotated by r[h])."""
    y = np.asarray(y, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if r.ndim == 2:
        return y @ r.T
    return np.stack([y[:, h] @ r[h].T for h in range(y.shape[1])], axis=1)


def _head_rot(r, kv: int) -> np.ndarray:
    r = np.asarray(r, dtype=np.float64)
    return r if r.ndim == 2 else r[kv]


def decode(cache: CacheImage, layer: int, q, block_table, seq_lens, req_slot, r_k, r_v) -> np.ndarray:
    """Plain definition.  q [B, Hq, d] -> o [B, Hq, d] float64."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    g = cache.g
    grp = hq // g.n_kv_heads
    out = np.zeros((bsz, hq, d))
    for b in range(bsz):
        yk, yv, wk, wv = _gather(cache, layer, b, int(seq_lens[b]), block_table, req_slot)
        k_all = np.concatenate([unrotate(yk, r_k), wk], axis=0)
        v_all = np.concatenate([unrotate(yv, r_v), wv], axis=0)
        for h in range(hq):
            out[b, h] = softmax_attention(q[b, h], k_all[:, h // grp], v_all[:, h // grp])
    return out


def decode_fused(cache: CacheImage, layer: int, q, block_table, seq_lens, req_slot, r_k, r_v) -> np.ndarray:
    """Rotated-query form: q' = q R_K scores the history in the rotated basis, the
    history values accumulate in the rotated basis, and R_V^T is applied once."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    g = cache.g
    grp = hq // g.n_kv_heads
    out = np.zeros((bsz, hq, d))
    for b in range(bsz):
        yk, yv, wk, wv = _gather(cache, layer, b, int(seq_lens[b]), block_table, req_slot)
        for h in range(hq):
            kv = h // grp
            rk, rv = _head_rot(r_k, kv), _head_rot(r_v, kv)
            qr = q[b, h] @ rk
            s_h = yk[:, kv] @ qr / np.sqrt(d)
            s_w = wk[:, kv] @ q[b, h] / np.sqrt(d)
            m = max(s_h.max(initial=-np.inf), s_w.max(initial=-np.inf))
            p_h = np.exp(s_h - m)
            p_w = np.exp(s_w - m)
            l = p_h.sum() + p_w.sum()
            acc_rot = p_h @ yv[:, kv]
            acc_plain = p_w @ wv[:, kv]
            out[b, h] = (acc_plain + acc_rot @ rv.T) / l
    return out


def bf16_paged_decode(pool_bits, layer: int, q, block_table, seq_lens, page_size: int) -> np.ndarray:
    """Textbook decode over an all-BF16 paged cache.

    pool_bits: uint16 [L, num_pages, Hkv, 2, P, d] (K then V per page and head).
    Token t of request b is at page block_table[b][t // P], slot t % P.
    """
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = pool_bits.shape[2]
    grp = hq // hkv
    bt = np.asarray(block_table)
    out = np.zeros((bsz, hq, d))
    for b in range(bsz):
        n = int(seq_lens[b])
        t = np.arange(n)
        pages = bt[b, t // page_size]
        kk = quant.bits_to_f64(pool_bits[layer, pages, :, 0, t % page_size, :])  # [n, Hkv, d]
        vv = quant.bits_to_f64(pool_bits[layer, pages, :, 1, t % page_size, :])
        for h in range(hq):
            out[b, h] = softmax_attention(q[b, h], kk[:, h // grp], vv[:, h // grp])
    return out


def extend(cache: CacheImage, layer: int, q, k_new, v_new, cu_seqlens, prefix_lens, block_table, req_slot,
           r_k, r_v) -> np.ndarray:
    """Extend (chunked prefill) attention over the mixed cache: the plain definition, float64.

    Source: the OSCAR technical summaries on gist.science, section 2.2 B (the serving
    kernel covers paged attention and prefix caching over the INT2 history) and the
    same page's systems contribution (prefix reuse kept in the INT2 cache).  The pages
    do not spell out the extend step; the reading taken here is the usual one for a
    prefix cache: request b holds prefix_lens[b] cached tokens, in the form the cache
    stores them at that length (history dequantised and rotated back, sink and recent
    tokens in BF16), and brings a chunk of len_b = cu_seqlens[b+1] - cu_seqlens[b] new
    tokens at positions prefix_lens[b] + i.  Query i of the chunk attends to every
    cached token and to the chunk's tokens 0..i (causal), whose keys and values are the
    chunk's own inputs (k_new, v_new, already BF16-valued).  The chunk is written to
    the cache afterwards.

    q [T, Hq, d], k_new / v_new [T, Hkv, d] (T = cu_seqlens[-1]) -> o [T, Hq, d].
    """
    q = np.asarray(q, dtype=np.float64)
    k_new = np.asarray(k_new, dtype=np.float64)
    v_new = np.asarray(v_new, dtype=np.float64)
    total, hq, d = q.shape
    g = cache.g
    grp = hq // g.n_kv_heads
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = np.zeros((total, hq, d))
    for b in range(cu.size - 1):
        n_pre = int(prefix_lens[b])
        yk, yv, wk, wv = _gather(cache, layer, b, n_pre, block_table, req_slot)
        k_pre = np.concatenate([unrotate(yk, r_k), wk], axis=0)
        v_pre = np.concatenate([unrotate(yv, r_v), wv], axis=0)
        c0, c1 = int(cu[b]), int(cu[b + 1])
        k_all = np.concatenate([k_pre, k_new[c0:c1]], axis=0)   # query i sees the first n_pre + i + 1 rows
        v_all = np.concatenate([v_pre, v_new[c0:c1]], axis=0)
        for i in range(c1 - c0):
            n = k_pre.shape[0] + i + 1
            for h in range(hq):
                out[c0 + i, h] = softmax_attention(q[c0 + i, h], k_all[:n, h // grp], v_all[:n, h // grp])
    return out
