"""Paged mixed-precision KV-cache image and its write paths, float64 (test infrastructure only).

Source: the OSCAR technical summaries on gist.science, section 2.2 B
("mixed-precision layout"): a paged KV cache in which the first ("sink") and
the most recent tokens stay BF16 while the middle history is stored in INT2
after the fixed rotation and clipping; the arXiv abstract (paperdot page) adds
fused write kernels that keep the paged layout and prefix caching.

Readings (the pages are silent on all of these):

* token t of a sequence of length n is a sink token if t < S, recent if
  t >= max(S, n - W), history otherwise; n <= S + W means no history;
* a write that grows a sequence from n0 to n1 first moves the ring tokens that
  stop being recent, [max(S, n0-W), min(n0, n1-W)), into INT2 (quantising
  their stored BF16 values), then writes the new tokens;
* absolute-position paging: history token t lives in page
  block_table[b][t // P] at slot t % P;
* window slab: sink token t at slot t, recent token t at slot S + (t-S) mod W,
  so an evicted token's slot is the slot of the token that replaces it;
* per (layer, page, kv head) block: K codes [P][d/4] | K (scale, zero) BF16
  pairs [P][d/G][2] | V codes [P][d/4] | V (scale, zero) [P][d/G][2];
* history rows are quantised from the values the path received: float32
  inputs as float32, BF16 inputs as their BF16 values, evicted ring tokens as
  their stored BF16 values.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import quant


@dataclass(frozen=True)
class Geometry:
    num_layers: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    group_size: int
    sink: int
    recent: int
    num_pages: int
    max_requests: int

    @property
    def row_bytes(self) -> int:
        return self.head_dim // 4

    @property
    def sz_bytes(self) -> int:  # one token's (scale, zero) BF16 pairs
        return 4 * (self.head_dim // self.group_size)

    @property
    def k_codes_off(self) -> int:
        return 0

    @property
    def k_sz_off(self) -> int:
        return self.page_size * self.row_bytes

    @property
    def v_codes_off(self) -> int:
        return self.k_sz_off + self.page_size * self.sz_bytes

    @property
    def v_sz_off(self) -> int:
        return self.v_codes_off + self.page_size * self.row_bytes

    @property
    def block_bytes(self) -> int:
        return self.v_sz_off + self.page_size * self.sz_bytes

    @property
    def window(self) -> int:
        return self.sink + self.recent


def window_slot(t: int, sink: int, recent: int) -> int:
    return t if t < sink else sink + (t - sink) % recent


def is_history(t: int, n: int, sink: int, recent: int) -> bool:
    return sink <= t < n - recent


class CacheImage:
    """Host image of the INT2 page pool and the BF16 window slab."""

    def __init__(self, geom: Geometry, fill: int = 0):
        self.g = geom
        self.pool = np.full((geom.num_layers, geom.num_pages, geom.n_kv_heads, geom.block_bytes), fill, dtype=np.uint8)
        self.slab = np.zeros((geom.num_layers, geom.max_requests, geom.n_kv_heads, 2, geom.window, geom.head_dim),
                             dtype=np.uint16)

    # ------------------------------------------------------------ history
    def store_history(self, layer: int, pages, slots, kq: dict, vq: dict) -> None:
        """Write quantised rows (dicts from quantize_rows) for M tokens at (pages[m], slots[m])."""
        g = self.g
        pages = np.asarray(pages, dtype=np.int64)
        slots = np.asarray(slots, dtype=np.int64)
        if pages.size == 0:
            return
        if (pages < 0).any() or (pages >= g.num_pages).any():
            raise ValueError("history token on an unmapped or out-of-range page")
        h = np.arange(g.n_kv_heads)[None, :, None]
        for qd, c_off, s_off, offs in ((kq, g.k_codes_off, g.k_sz_off, quant.k_bit_offsets(g.head_dim)),
                                       (vq, g.v_codes_off, g.v_sz_off, quant.v_bit_offsets(g.head_dim))):
            rows = quant.pack_rows(qd["codes"], offs)                      # [M, H, d/4]
            sz = np.stack([quant.bf16_to_bits(qd["scale"]), quant.bf16_to_bits(qd["zero"])], axis=-1)
            szb = np.ascontiguousarray(sz.astype("<u2")).view(np.uint8).reshape(rows.shape[0], g.n_kv_heads, -1)
            col = c_off + slots[:, None, None] * g.row_bytes + np.arange(g.row_bytes)[None, None, :]
            self.pool[layer, pages[:, None, None], h, col] = rows
            col = s_off + slots[:, None, None] * g.sz_bytes + np.arange(g.sz_bytes)[None, None, :]
            self.pool[layer, pages[:, None, None], h, col] = szb

    def read_history(self, layer: int, pages, slots):
        """(codes_k, scale_k, zero_k, codes_v, scale_v, zero_v) for M tokens, natural channel order."""
        g = self.g
        pages = np.asarray(pages, dtype=np.int64)
        slots = np.asarray(slots, dtype=np.int64)
        h = np.arange(g.n_kv_heads)[None, :, None]
        out = []
        for c_off, s_off, offs in ((g.k_codes_off, g.k_sz_off, quant.k_bit_offsets(g.head_dim)),
                                   (g.v_codes_off, g.v_sz_off, quant.v_bit_offsets(g.head_dim))):
            col = c_off + slots[:, None, None] * g.row_bytes + np.arange(g.row_bytes)[None, None, :]
            codes = quant.unpack_rows(self.pool[layer, pages[:, None, None], h, col], offs)
            col = s_off + slots[:, None, None] * g.sz_bytes + np.arange(g.sz_bytes)[None, None, :]
            szb = np.ascontiguousarray(self.pool[layer, pages[:, None, None], h, col])
            sz = szb.view("<u2").reshape(pages.shape[0], g.n_kv_heads, -1, 2)
            out += [codes, quant.bits_to_f64(sz[..., 0]), quant.bits_to_f64(sz[..., 1])]
        return tuple(out)

    # ------------------------------------------------------------ window
    def store_window(self, layer: int, slot_req: int, t: int, k_bits, v_bits) -> None:
        s = window_slot(t, self.g.sink, self.g.recent)
        self.slab[layer, slot_req, :, 0, s, :] = k_bits
        self.slab[layer, slot_req, :, 1, s, :] = v_bits

    def read_window(self, layer: int, slot_req: int, t: int):
        s = window_slot(t, self.g.sink, self.g.recent)
        return (quant.bits_to_f64(self.slab[layer, slot_req, :, 0, s, :]),
                quant.bits_to_f64(self.slab[layer, slot_req, :, 1, s, :]))


def rotate_rows(x, r) -> np.ndarray:
    """y = x R for token rows x [M, H, d], float64.

    r is [d, d], the layer's rotation shared by every kv head (the pages' fixed per-layer
    rotation), or [H, d, d], one rotation per kv head (head h of every row uses r[h]).
    """
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if r.ndim == 2:
        return x @ r
    return np.stack([x[:, h] @ r[h] for h in range(x.shape[1])], axis=1)


def quantize_rows(x, r, clip: float, group: int) -> dict:
    """Rotate, clip and quantise token rows: x [M, H, d] (float64 values), r [d, d] or [H, d, d]
    (float32 values; see rotate_rows).

    y = x R (row-vector convention), y <- clamp(y, -c, c), then per-group INT2.
    """
    y = rotate_rows(x, r)
    c = float(np.float32(clip))
    y = np.clip(y, -c, c)
    codes, scale, zero, mn, rng3 = quant.quantize_groups(y, group)
    return {"y": y, "codes": codes, "scale": scale, "zero": zero, "mn": mn, "rng3": rng3}


def _bf16_bits_of_input(x) -> np.ndarray:
    """BF16 storage of an input value (RNE from its exact float value)."""
    return quant.bf16_to_bits(quant.bf16_round(np.asarray(x, dtype=np.float64)))


def write_kv(cache: CacheImage, layer: int, k, v, cu_seqlens, start_pos, r_k, r_v, clip_k, clip_v,
             block_table, req_slot) -> dict:
    """Varlen write of tokens [start_pos[b], start_pos[b] + len_b) for each request b.

    k, v: [sum len, Hkv, d] input values (float32 or BF16-valued).  Returns the
    quantisation diagnostics of every history row written, keyed for the
    near-boundary rule of the parity tests.
    """
    g = cache.g
    s_, w_ = g.sink, g.recent
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    hist_b, hist_t, xk, xv = [], [], [], []
    window_writes = []
    for b in range(len(start_pos)):
        t0 = int(start_pos[b])
        ln = int(cu_seqlens[b + 1]) - int(cu_seqlens[b])
        n1 = t0 + ln
        # 1) ring tokens that stop being recent are quantised from their stored BF16 values
        for e in range(max(s_, t0 - w_), min(t0, n1 - w_)):
            ke, ve = cache.read_window(layer, int(req_slot[b]), e)
            hist_b.append(b); hist_t.append(e); xk.append(ke); xv.append(ve)
        # 2) new tokens
        for i in range(ln):
            t = t0 + i
            row = int(cu_seqlens[b]) + i
            if is_history(t, n1, s_, w_):
                hist_b.append(b); hist_t.append(t); xk.append(k[row]); xv.append(v[row])
            else:
                window_writes.append((b, t, row))
    diag = {"b": np.asarray(hist_b, dtype=np.int64), "t": np.asarray(hist_t, dtype=np.int64)}
    if hist_b:
        kq = quantize_rows(np.stack(xk), r_k, clip_k, g.group_size)
        vq = quantize_rows(np.stack(xv), r_v, clip_v, g.group_size)
        bt = np.asarray(block_table)
        pages = bt[diag["b"], diag["t"] // g.page_size]
        slots = diag["t"] % g.page_size
        cache.store_history(layer, pages, slots, kq, vq)
        diag.update({"k": kq, "v": vq, "pages": pages, "slots": slots})
    for b, t, row in window_writes:
        cache.store_window(layer, int(req_slot[b]), t, _bf16_bits_of_input(k[row]), _bf16_bits_of_input(v[row]))
    return diag


def fork_prefix(cache: CacheImage, src_slot: int, dst_slot: int, src_pages, dst_pages, n: int) -> None:
    """Branch request dst off request src at src's current length n (every layer).

    Reading: a fork happens at a branch point, so the destination starts as an
    exact copy of the source's state at length n.  History pages that are full
    ([S, max(S, n-W)) covers them completely) are shared; the page holding the
    end of the history, if partial, is copied to the destination's own page
    (copy-on-write), since later evictions fill its remaining slots differently;
    the BF16 window (sink + recent ring) is copied.  ``src_pages`` and
    ``dst_pages`` are the two requests' block-table rows; dst_pages must already
    hold the shared page ids and a fresh id for the partial page.
    """
    g = cache.g
    h_end = max(g.sink, n - g.recent)
    full = h_end // g.page_size
    for i in range(full):
        if int(dst_pages[i]) != int(src_pages[i]):
            raise ValueError("full prefix pages must be shared")
    if h_end % g.page_size and h_end > g.sink:
        cache.pool[:, int(dst_pages[full])] = cache.pool[:, int(src_pages[full])]
    cache.slab[:, dst_slot] = cache.slab[:, src_slot]


def append_step(cache: CacheImage, layer: int, k_new, v_new, seq_lens_before, r_k, r_v, clip_k, clip_v,
                block_table, req_slot) -> dict:
    """One decode-step append per request: k_new, v_new [B, Hkv, d] at position seq_lens_before[b]."""
    bsz = len(seq_lens_before)
    cu = np.arange(bsz + 1, dtype=np.int64)
    return write_kv(cache, layer, k_new, v_new, cu, seq_lens_before, r_k, r_v, clip_k, clip_v, block_table, req_slot)
