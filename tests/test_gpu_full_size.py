"""Full-size workloads on the GPU, checked on samples the oracle computes one by one.

The cache is filled by the GPU write path (the tensor-core prefill for these BF16
inputs).  History rows are re-quantised by the oracle from their inputs (every row
of the batch-1 32K and 131K, batched and prefill cases; sampled rows in the
capacity case): codes, scales and zeros bit-exact up to the near-boundary rule,
with the exemptions counted over the whole case and listed.  Sampled requests
are decoded by the oracle from the GPU's own packed pages (identical caches),
against the GPU decode of the whole batch in one launch: max abs error <= 2e-3 and
mean abs error <= 2e-4 on unit-scale outputs.

Inputs are the synthetic workloads of the same shapes.  The requests of a case
draw on one seeded input stream per layer: request b takes the rows starting at
row 37*b (not a multiple of the page size, so no two requests hold the same page
contents and a page-table mix-up cannot hide).  The stream lives on the device
in BF16, each write reads its own slice, and the host keeps the float values to
re-quantise sampled rows.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import attention, cache
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def osc():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from int2_rotated_paged_oscar_gb300 import build
    build.build()
    import int2_rotated_paged_oscar_gb300 as m
    m.load()
    return m


ROW_SHIFT = 37


class Stream:
    """One seeded K/V input stream of a layer: host float32 values and device BF16 copies."""

    def __init__(self, wl, layer, n_rows, sub=0):
        self.k, self.v = syn.kv_tokens(wl, layer, n_rows, sub=sub)
        self.dk, self.dv = H.dev_input(self.k, "bf16"), H.dev_input(self.v, "bf16")

    def rows(self, r):
        return self.k[r], self.v[r]


def _write(osc, gc, layer, dk, dv, t0, n, bt_row, bt_stride, slot):
    """One request's write of tokens [t0, t0 + n) from device BF16 rows dk, dv [n, Hkv, d]."""
    fx = gc.fx[layer]
    osc.oscar_write_kv(gc.ctx, layer, dk, dv, osc.DTYPE_BF16, H.dev(np.array([0, n], np.int32)),
                       H.dev(np.array([t0], np.int32)), 1, n, H.dev(fx["R_K"]), H.dev(fx["R_V"]), fx["clip_K"],
                       fx["clip_V"], H.dev(np.asarray(bt_row, np.int32)[None]), bt_stride,
                       H.dev(np.array([slot], np.int32)))


def _prefill(osc, gc, layer, st, lens, bt):
    """Prefill of every request b into slot b: rows [37 b, 37 b + lens[b]) of the stream."""
    for b, n in enumerate(lens):
        o = ROW_SHIFT * b
        _write(osc, gc, layer, st.dk[o:o + n], st.dv[o:o + n], 0, n, bt[b], bt.shape[1], b)
    assert osc.oscar_check_status(gc.ctx) == 0


def _check_window(gc, layer, bt_row, n, slot, rows_of):
    """The BF16 sink and recent tokens of one request equal its inputs (BF16 values, stored exactly)."""
    img, _ = H.compact_request_image(gc, layer, bt_row, n, slot)
    _, win = attention.token_sets(n, gc.geom.sink, gc.geom.recent)
    for t in win:
        k, v = img.read_window(0, 0, int(t))
        xk, xv = rows_of(int(t))
        assert np.array_equal(k, xk) and np.array_equal(v, xv), f"window token {t} of slot {slot} differs"


def _sample_rows(rng, lens, geom, m, rows_of):
    """m random history rows (b, t, k_row, v_row); rows_of(b, t) gives the input rows of token t of request b."""
    out = []
    for _ in range(m):
        b = int(rng.integers(len(lens)))
        lo, hi = geom.sink, lens[b] - geom.recent
        if hi > lo:
            t = int(rng.integers(lo, hi))
            out.append((b, t) + tuple(rows_of(b, t)))
    return out


def _check_rows(gc, layer, bt, samples):
    """Sampled history rows of the GPU cache against the oracle's quantisation of their inputs.

    Only the pages the samples touch are read back: they form a compact pool, pages renumbered."""
    g = gc.geom
    diag = H.sampled_history_diag(g, bt, samples, gc.fx[layer])
    used, remap = np.unique(diag["pages"], return_inverse=True)
    cg = cache.Geometry(1, g.n_kv_heads, g.head_dim, g.page_size, g.group_size, g.sink, g.recent, len(used), 1)
    res = H.compare_history(H.gpu_pages(gc, layer, used)[None], cg, 0, dict(diag, pages=remap.reshape(-1)))
    assert res["elements"] == len(samples) * 2 * g.n_kv_heads * g.head_dim
    return res


def _check_all_rows(gc, layer, bt, lens, rows_for, case, chunk=8192):
    """Every history row of every request, re-quantised by the oracle from its inputs, against the GPU's
    pages (codes, scales and zeros bit-exact up to the near-boundary rule).  The exemption budget holds
    over the whole case and every exemption is listed.  rows_for(b, ts) gives the input rows of tokens
    ts of request b ([m, Hkv, d] each for K and V).  Chunks of rows go to a spawned process pool; the
    GPU's page blocks of each chunk are gathered on the device."""
    g = gc.geom
    fx = {k: gc.fx[layer][k] for k in ("R_K", "R_V", "clip_K", "clip_V")}
    fields = (g.num_layers, g.n_kv_heads, g.head_dim, g.page_size, g.group_size, g.sink, g.recent, g.num_pages,
              g.max_requests)
    futs = []
    pool = H.oracle_pool()
    for b, n in enumerate(lens):
        for t0 in range(g.sink, n - g.recent, chunk):
            ts = np.arange(t0, min(n - g.recent, t0 + chunk), dtype=np.int64)
            xk, xv = rows_for(b, ts)
            pages = np.asarray(bt[b], np.int64)[ts // g.page_size]
            used, remap = np.unique(pages, return_inverse=True)
            blocks = H.gpu_pages(gc, layer, used)
            futs.append(pool.submit(H.check_history_chunk, (fields, fx, b, ts, np.ascontiguousarray(xk),
                                                            np.ascontiguousarray(xv), blocks, remap.reshape(-1))))
    res = H.merge_results(f.result() for f in futs)
    assert res["elements"] == sum(max(0, n - g.recent - g.sink) for n in lens) * 2 * g.n_kv_heads * g.head_dim
    H.record_exemptions(case, res)
    H.check_budget(res)
    return res


def _decode_all(osc, gc, layer, q, bt, lens, slots, max_seq):
    """GPU decode of the whole batch in one call (the layer's clip was declared by its writes)."""
    import torch
    b = q.shape[0]
    ws_bytes = osc.oscar_decode_workspace_size(gc.cfg, b, max_seq)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty((b, q.shape[1], q.shape[2]), dtype=torch.float32, device="cuda")
    fx = gc.fx[layer]
    osc.oscar_decode_attn(gc.ctx, layer, H.dev_input(q, "bf16"), osc.DTYPE_BF16, out, osc.DTYPE_F32,
                          H.dev(np.asarray(bt, np.int32)), bt.shape[1], H.dev(np.asarray(lens, np.int32)),
                          H.dev(np.asarray(slots, np.int32)), b, max_seq, gc.geom.sink, gc.geom.recent,
                          H.dev(fx["R_K"]), H.dev(fx["R_V"]), ws, ws_bytes)
    assert osc.oscar_check_status(gc.ctx) == 0
    return out.cpu().numpy().astype(np.float64)


def _check_request(gc, layer, got_row, q_row, bt_row, n, slot, heads=None):
    """Oracle decode of one request from the GPU's own pages and window slot; heads restricts the check
    to some kv heads (and their q heads)."""
    fx = gc.fx[layer]
    img, bt_c = H.compact_request_image(gc, layer, bt_row, n, slot, heads)
    if heads is not None:
        gq = q_row.shape[0] // gc.geom.n_kv_heads
        sel = np.concatenate([np.arange(h * gq, (h + 1) * gq) for h in heads])
        q_row, got_row = q_row[sel], got_row[sel]
    want = attention.decode(img, 0, q_row[None], bt_c, [n], [0], fx["R_K"], fx["R_V"])[0]
    return H.assert_decode_close(got_row, want)


def _cache(wl, num_pages, max_requests, ppr, num_layers=1, layers=None):
    """Device cache of the workload's shape; the calibrated fixture (R_K, R_V, clips) of each used layer."""
    s = wl.shape
    geom = H.geometry(s, num_pages, max_requests, num_layers=num_layers)
    gc = H.make_gpu_cache(geom, s.n_q_heads, ppr)
    gc.fx = {layer: H.fixture(wl, layer) for layer in (range(num_layers) if layers is None else layers)}
    return geom, gc


def _single_request(osc, wl, n, case, heads=None, seed=0):
    """Batch-1 prefill of n tokens and one decode; every history row, the window and the decode are checked."""
    s = wl.shape
    ppr = syn.pages_for(n, s.page_size)
    geom, gc = _cache(wl, ppr, 1, ppr)
    try:
        st = Stream(wl, 0, n)
        bt = np.arange(ppr, dtype=np.int32)[None]
        _prefill(osc, gc, 0, st, [n], bt)
        rows_of = lambda b, t: st.rows(t)
        rng = np.random.default_rng(seed)
        samples = _sample_rows(rng, [n], geom, 64, rows_of)
        # the first and last history tokens and both ends of a page boundary
        for t in (geom.sink, 63, 64, n // 2, n - geom.recent - 1):
            samples.append((0, t) + tuple(st.rows(t)))
        _check_rows(gc, 0, bt, samples)
        _check_all_rows(gc, 0, bt, [n], lambda b, ts: (st.k[ts], st.v[ts]), case)
        _check_window(gc, 0, bt[0], n, 0, st.rows)
        q = syn.queries(wl, 0, 1)
        got = _decode_all(osc, gc, 0, q, bt, [n], [0], n)
        _check_request(gc, 0, got[0], q[0], bt[0], n, 0, heads)
    finally:
        gc.close()


def test_batch1_32k_full(osc):
    """Batch-1 decode at 32,768 tokens, 32 q / 8 kv heads, d=128, page 64; all heads checked."""
    _single_request(osc, syn.batch1_32k(), 32768, "batch1_32k", seed=100)


def test_long_131k_full(osc):
    """Batch-1 decode at 131,072 tokens; every history row and all eight kv heads (32 q heads) checked."""
    _single_request(osc, syn.long_131k(), 131072, "long_131k", seed=101)


def test_batched_ragged_b64_full(osc):
    """64 requests, lengths U[8K, 32K], 64 q / 8 kv heads, pages handed out in shuffled order, one decode
    launch for the batch; every history row of every request is checked, and the shortest, longest and
    two other requests are decoded by the oracle."""
    wl = syn.batched_ragged(64)
    s = wl.shape
    lens = list(wl.seq_lens)
    b = len(lens)
    ppr = syn.pages_for(max(lens), s.page_size)
    num_pages = b * ppr
    bt = syn.page_permutation(wl.seed, num_pages, shuffle=True).reshape(b, ppr).astype(np.int32)
    geom, gc = _cache(wl, num_pages, b, ppr)
    try:
        st = Stream(wl, 0, max(lens) + ROW_SHIFT * b)
        _prefill(osc, gc, 0, st, lens, bt)
        rows_of = lambda r, t: st.rows(ROW_SHIFT * r + t)
        rng = np.random.default_rng(102)
        _check_rows(gc, 0, bt, _sample_rows(rng, lens, geom, 128, rows_of))
        _check_all_rows(gc, 0, bt, lens, lambda r, ts: (st.k[ROW_SHIFT * r + ts], st.v[ROW_SHIFT * r + ts]),
                        "batched_ragged_b64")
        q = syn.queries(wl, 0, b)
        got = _decode_all(osc, gc, 0, q, bt, lens, list(range(b)), max(lens))
        for r in sorted({int(np.argmin(lens)), int(np.argmax(lens)), 17, 40}):
            _check_window(gc, 0, bt[r], lens[r], r, lambda t, r=r: rows_of(r, t))
            _check_request(gc, 0, got[r], q[r], bt[r], lens[r], r, heads=None if r in (17,) else [1, 6])
    finally:
        gc.close()


def test_prefill_8x32k_shared_prefix_and_appends(osc):
    """Eight requests of 32,768 tokens.  Requests 1-3 fork off request 0 after its 16,384-token prefix
    (whole history pages shared, the window slot copied) and each writes its own continuation; requests
    4-7 are independent.  Then 256 fused decode steps (append + attention) for all eight.  Every history
    row of every request (the prefill, the evicted rings and the appends) is checked."""
    import torch
    wl = syn.write_prefill()
    s = wl.shape
    n_full, b = wl.seq_lens[0], len(wl.seq_lens)
    n_pre, sharers, steps = wl.extra["prefix_tokens"], wl.extra["prefix_sharers"], wl.extra["appends"]
    n_end = n_full + steps
    ppr = syn.pages_for(n_end, s.page_size)
    geom, gc = _cache(wl, b * ppr, b, ppr)
    try:
        st = Stream(wl, 0, n_full + ROW_SHIFT * b)
        kn, vn = syn.kv_tokens(wl, 0, steps * b, sub=9)
        kn = kn.reshape(steps, b, s.n_kv_heads, s.head_dim)
        vn = vn.reshape(steps, b, s.n_kv_heads, s.head_dim)

        def rows_of(r, t):
            if t >= n_full:
                return kn[t - n_full, r], vn[t - n_full, r]
            if r < sharers and t < n_pre:
                return st.rows(t)
            return st.rows(ROW_SHIFT * r + t)

        # pages from the library's allocator: request 0's prefix, the forks, then every request's rest
        bts = -np.ones((b, ppr), np.int32)
        pre_pages = H.cache_pages_for(n_pre, geom)
        bts[0, :pre_pages] = osc.oscar_alloc_pages(gc.ctx, pre_pages)
        _write(osc, gc, 0, st.dk[:n_pre], st.dv[:n_pre], 0, n_pre, bts[0], ppr, 0)
        torch.cuda.synchronize()
        for r in range(1, sharers):
            bts[r] = osc.oscar_fork_prefix(gc.ctx, list(bts[0]), n_pre, 0, r, ppr)
        torch.cuda.synchronize()
        shared = bts[0, :pre_pages]
        for r in range(1, sharers):
            assert np.array_equal(bts[r, :pre_pages], shared) and np.all(bts[r, pre_pages:] == -1)
        assert all(osc.oscar_page_refcount(gc.ctx, int(p)) == sharers for p in shared)
        for r in range(b):
            have = int((bts[r] >= 0).sum())
            bts[r, have:] = osc.oscar_alloc_pages(gc.ctx, ppr - have)
        assert osc.oscar_free_page_count(gc.ctx) == b * ppr - (pre_pages + sharers * (ppr - pre_pages)
                                                               + (b - sharers) * ppr)
        assert len(np.unique(bts[:, pre_pages:])) == b * (ppr - pre_pages)
        for r in range(sharers):       # continuations: the ring of the prefix is evicted into INT2 first
            o = ROW_SHIFT * r
            _write(osc, gc, 0, st.dk[o + n_pre:o + n_full], st.dv[o + n_pre:o + n_full], n_pre, n_full - n_pre,
                   bts[r], ppr, r)
        for r in range(sharers, b):
            o = ROW_SHIFT * r
            _write(osc, gc, 0, st.dk[o:o + n_full], st.dv[o:o + n_full], 0, n_full, bts[r], ppr, r)
        assert osc.oscar_check_status(gc.ctx) == 0

        fx = gc.fx[0]
        ws_bytes = osc.oscar_decode_workspace_size(gc.cfg, b, n_end)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        out = torch.empty((b, s.n_q_heads, s.head_dim), dtype=torch.float32, device="cuda")
        q_all = syn.queries(wl, 0, steps * b, sub=7).reshape(steps, b, s.n_q_heads, s.head_dim)
        dq, dkn, dvn = H.dev_input(q_all, "bf16"), H.dev_input(kn, "bf16"), H.dev_input(vn, "bf16")
        lens_d = H.dev(n_full + 1 + np.repeat(np.arange(steps, dtype=np.int32)[:, None], b, axis=1))
        btd, slots = H.dev(bts), H.dev(np.arange(b, dtype=np.int32))
        rk, rv = H.dev(fx["R_K"]), H.dev(fx["R_V"])
        for i in range(steps):
            osc.oscar_decode_step(gc.ctx, 0, dkn[i], dvn[i], osc.DTYPE_BF16, dq[i], osc.DTYPE_BF16, out,
                                  osc.DTYPE_F32, btd, ppr, lens_d[i], slots, b, n_end, s.sink, s.recent, rk, rv,
                                  fx["clip_K"], fx["clip_V"], ws, ws_bytes)
        assert osc.oscar_check_status(gc.ctx) == 0
        assert all(osc.oscar_page_refcount(gc.ctx, int(p)) == sharers for p in shared)

        rng = np.random.default_rng(103)
        samples = _sample_rows(rng, [n_end] * b, geom, 128, rows_of)
        for r in (1, 3):               # the shared prefix and the ring the continuation evicted
            for t in (s.sink, 5000, n_pre - s.recent - 1, n_pre - s.recent, n_pre - 1, n_pre):
                samples.append((r, t) + tuple(rows_of(r, t)))
        for r in (0, 2, 6):            # tokens the appends evicted
            for t in (n_full - s.recent, n_full - 1, n_full + 10, n_end - s.recent - 1):
                samples.append((r, t) + tuple(rows_of(r, t)))
        _check_rows(gc, 0, bts, samples)

        def rows_for(r, ts):
            k = np.empty((ts.size, s.n_kv_heads, s.head_dim), np.float32)
            v = np.empty_like(k)
            app = ts >= n_full
            pre = ~app & (ts < n_pre) if r < sharers else np.zeros(ts.size, bool)
            own = ~app & ~pre
            k[app], v[app] = kn[ts[app] - n_full, r], vn[ts[app] - n_full, r]
            k[pre], v[pre] = st.k[ts[pre]], st.v[ts[pre]]
            k[own], v[own] = st.k[ROW_SHIFT * r + ts[own]], st.v[ROW_SHIFT * r + ts[own]]
            return k, v
        _check_all_rows(gc, 0, bts, [n_end] * b, rows_for, "prefill_8x32k_shared_prefix_256_appends")
        got = out.cpu().numpy().astype(np.float64)
        q_last = syn.as_input(q_all[steps - 1], "bf16")
        for r in (1, 5):
            _check_window(gc, 0, bts[r], n_end, r, lambda t, r=r: rows_of(r, t))
            _check_request(gc, 0, got[r], q_last[r], bts[r], n_end, r)
    finally:
        gc.close()


def test_capacity_28x100k_64_layers(osc):
    """28 requests x 100,000 tokens x 64 layers, 64 q / 8 kv heads: the whole INT2 cache is allocated on
    one GPU (a BF16 cache of the same tokens would not fit), layers 0 and 63 are written and decoded in
    one launch each (byte offsets past 2^32 into the pool), and sampled rows and requests are checked."""
    import torch
    wl = syn.capacity_28x100k(num_layers=64)
    s = wl.shape
    lens = list(wl.seq_lens)
    b, n = len(lens), max(lens)
    torch.cuda.empty_cache()
    total = torch.cuda.get_device_properties(0).total_memory
    g0 = H.geometry(s, 1, b, num_layers=s.num_layers)
    ppr = syn.pages_for(n, s.page_size)
    geom_bytes = s.num_layers * b * ppr * s.n_kv_heads * g0.block_bytes
    bf16_bytes = s.num_layers * b * n * s.n_kv_heads * s.head_dim * 2 * 2
    assert geom_bytes < 0.6 * total < bf16_bytes
    layers = (0, s.num_layers - 1)
    geom, gc = _cache(wl, b * ppr, b, ppr, num_layers=s.num_layers, layers=layers)
    try:
        assert osc.oscar_int2_pool_bytes(gc.cfg) == geom_bytes
        bt = np.arange(b * ppr, dtype=np.int32).reshape(b, ppr)
        for layer in layers:
            st = Stream(wl, layer, n + ROW_SHIFT * b)
            _prefill(osc, gc, layer, st, lens, bt)
            rows_of = lambda r, t: st.rows(ROW_SHIFT * r + t)
            rng = np.random.default_rng(104 + layer)
            _check_rows(gc, layer, bt, _sample_rows(rng, lens, geom, 64, rows_of))
            q = syn.queries(wl, layer, b)
            got = _decode_all(osc, gc, layer, q, bt, lens, list(range(b)), n)
            for r, heads in ((5, [0, 3]), (b - 1, [7])):
                _check_window(gc, layer, bt[r], n, r, lambda t, r=r: rows_of(r, t))
                _check_request(gc, layer, got[r], q[r], bt[r], n, r, heads)
            del st
    finally:
        gc.close()
