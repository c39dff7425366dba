"""GPU parity of extend (chunked prefill) attention over the mixed cache, against the oracle.

The prefix of every request is written by the GPU's own write path; the oracle then attends over
the GPU's cache image (pages and window slots read back), so these tests check the attention
kernel alone.  Every case spans several 64-key tiles and query tiles with ragged tails.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import attention, cache
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def osc():
    from int2_rotated_paged_oscar_gb300 import build
    build.build()
    import int2_rotated_paged_oscar_gb300 as m
    m.load()
    return m


def _setup(wl, fx, prefix, room=0):
    """GPU cache with each request's prefix written (request b in slot b, pages b*ppr ...); each request's
    block-table row maps room more tokens than its prefix."""
    s = wl.shape
    b = len(prefix)
    ppr = max(syn.pages_for(max(n + room, 1), s.page_size) for n in prefix) + 1
    bt = np.arange(b * ppr, dtype=np.int32).reshape(b, ppr)
    geom = H.geometry(s, b * ppr, b)
    gc = H.make_gpu_cache(geom, s.n_q_heads, ppr)
    if sum(prefix):
        import int2_rotated_paged_oscar_gb300 as osc
        ks, vs = zip(*[syn.kv_tokens(wl, 0, n, sub=i) for i, n in enumerate(prefix)])
        k = np.concatenate(ks)
        v = np.concatenate(vs)
        cu = np.concatenate([[0], np.cumsum(prefix)]).astype(np.int32)
        osc.oscar_write_kv(gc.ctx, 0, H.dev_input(k, wl.dtype), H.dev_input(v, wl.dtype), H.dtype_code(wl.dtype),
                           H.dev(cu), H.dev(np.zeros(b, np.int32)), b, int(cu[-1]), H.dev(fx["R_K"]),
                           H.dev(fx["R_V"]), fx["clip_K"], fx["clip_V"], H.dev(bt), ppr,
                           H.dev(np.arange(b, dtype=np.int32)))
        assert osc.oscar_check_status(gc.ctx) == 0
    return gc, geom, bt


def _image(gc, geom):
    img = cache.CacheImage(geom)
    img.pool, img.slab = gc.pool_np(), gc.slab_np()
    return img


@pytest.mark.parametrize("q_scale", [1.0, 0.25])
@pytest.mark.parametrize("shape,prefix,chunks,q_dtype,out_bf16", [
    (syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [1300, 0, 90, 700], [200, 150, 37, 64], "bf16", False),
    (syn.Shape(8, 4, 64, 16, 32, 4, 32, 1), [300, 35], [70, 9], "bf16", False),
    (syn.Shape(8, 8, 128, 32, 32, 0, 64, 1), [500, 64], [130, 1], "bf16", True),
    (syn.Shape(64, 8, 128, 64, 32, 4, 128, 1), [260], [40], "bf16", False),
    # edges: window exactly full (no history), one history token, sink only, an empty chunk
    (syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [132, 133, 4, 200], [17, 0, 5, 64], "bf16", False),
], ids=["d128_p64_gq4", "d64_p16_gq2", "d128_p32_gq1_nosink_bf16out", "d128_p64_gq8", "edges"])
def test_extend_parity(osc, shape, prefix, chunks, q_dtype, out_bf16, q_scale):
    wl = syn.Workload("ext", shape, [0], seed=31, dtype="bf16")
    fx = H.fixture(wl)
    gc, geom, bt = _setup(wl, fx, prefix)
    try:
        total = sum(chunks)
        k, v = syn.kv_tokens(wl, 0, total, sub=7)
        # BF16-valued (the workload's dtype); q x 0.25 spreads the weights (a peaky softmax hides errors)
        q = syn.queries(wl, 0, total, sub=8, scale=q_scale)
        cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
        slots = np.arange(len(prefix), dtype=np.int32)
        got = H.run_extend(gc, 0, q, q_dtype, k, v, cu, prefix, bt, slots, fx, out_bf16=out_bf16)
        # the unpacked-prefix form (the history dequantised once per call by a pre-pass, the attention CTAs
        # copying its tiles) runs the same operands through the same MMAs: identical outputs, also when the
        # workspace holds the tiles of the shorter prefixes only (the longest prefix unpacks its own)
        for form in (True, max(1, sorted(prefix)[-2] if len(prefix) > 1 else prefix[0] // 2)):
            got_u = H.run_extend(gc, 0, q, q_dtype, k, v, cu, prefix, bt, slots, fx, out_bf16=out_bf16,
                                 unpacked=form)
            assert np.array_equal(got_u, got), f"unpacked form {form}: {np.abs(got_u - got).max():.3e} apart"
        want = attention.extend(_image(gc, geom), 0, q, k, v, cu, prefix, bt, slots, fx["R_K"], fx["R_V"])
        if out_bf16:
            # a BF16 store rounds each element to 2^-9 of itself: one BF16 ulp of the element plus the
            # float32 bound (outlier channels reach tens of times the output RMS)
            rms = float(np.sqrt(np.mean(np.square(want))))
            err = np.abs(got - want)
            bound = 2.0 ** -8 * np.abs(want) + H.DECODE_MAX_ABS * rms
            assert np.all(np.isfinite(got)) and np.all(err <= bound), f"worst excess {float((err - bound).max()):.3e}"
            assert err.mean() <= 2e-3 * rms
        else:
            H.assert_decode_close(got, want)
    finally:
        gc.close()


@pytest.mark.parametrize("seed", range(10))
def test_extend_forms_agree_on_random_requests(osc, seed):
    """Random shapes, prefixes and chunks (seeded): the output is within the decode tolerance of the oracle
    attending over the GPU's cache image, and the form in which every CTA forms its tiles, the
    unpacked-prefix form with a workspace for every prefix, and one with a workspace for shorter prefixes
    only give identical outputs (the same operands through the same MMAs)."""
    rng = np.random.default_rng(1000 + seed)
    gq = int(rng.choice([1, 2, 4, 8]))
    hkv = int(rng.choice([2, 4, 8]))
    d = int(rng.choice([64, 128]))
    page = int(rng.choice([16, 32, 64]))
    sink = int(rng.choice([0, 4]))
    recent = int(rng.choice([32, 64, 128]))
    shape = syn.Shape(gq * hkv, hkv, d, page, 32, sink, recent, 1)
    b = int(rng.integers(1, 5))
    prefix = [int(x) for x in rng.integers(0, 1600, size=b)]
    chunks = [int(x) for x in rng.integers(0, 180, size=b)]
    chunks[int(rng.integers(0, b))] = int(rng.integers(1, 180))   # at least one query token
    wl = syn.Workload("ext_rand", shape, [0], seed=60 + seed, dtype="bf16")
    fx = H.fixture(wl)
    gc, geom, bt = _setup(wl, fx, prefix)
    try:
        total = sum(chunks)
        k, v = syn.kv_tokens(wl, 0, total, sub=13)
        q = syn.queries(wl, 0, total, sub=14, scale=0.5)
        cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
        slots = np.arange(b, dtype=np.int32)
        got = H.run_extend(gc, 0, q, "bf16", k, v, cu, prefix, bt, slots, fx)
        assert np.all(np.isfinite(got))
        want = attention.extend(_image(gc, geom), 0, q, k, v, cu, prefix, bt, slots, fx["R_K"], fx["R_V"])
        H.assert_decode_close(got, want)
        for form in (True, int(rng.integers(0, max(prefix) + 1))):
            got_u = H.run_extend(gc, 0, q, "bf16", k, v, cu, prefix, bt, slots, fx, unpacked=form)
            assert np.array_equal(got_u, got), (shape, prefix, chunks, form)
    finally:
        gc.close()


def test_extend_on_a_forked_prefix(osc):
    """Prefix caching end to end: request 0 writes a prefix, request 1 forks it (full history pages
    shared, the partial page copied, the window copied), and one extend call serves both with
    different chunks.  The oracle writes each request's prefix from scratch into its own pages."""
    shape = syn.Shape(32, 8, 128, 64, 32, 4, 128, 1)
    wl = syn.Workload("fork_ext", shape, [0], seed=41, dtype="bf16")
    fx = H.fixture(wl)
    n_pre, chunks = 1500, [90, 70]
    ppr = 30
    geom = H.geometry(shape, 64, 2)
    gc = H.make_gpu_cache(geom, shape.n_q_heads, ppr)
    try:
        ids = osc.oscar_alloc_pages(gc.ctx, syn.pages_for(n_pre, 64))
        bt0 = np.full(ppr, -1, np.int32)
        bt0[:len(ids)] = ids
        k, v = syn.kv_tokens(wl, 0, n_pre)
        osc.oscar_write_kv(gc.ctx, 0, H.dev_input(k, "bf16"), H.dev_input(v, "bf16"), osc.DTYPE_BF16,
                           H.dev(np.array([0, n_pre], np.int32)), H.dev(np.zeros(1, np.int32)), 1, n_pre,
                           H.dev(fx["R_K"]), H.dev(fx["R_V"]), fx["clip_K"], fx["clip_V"], H.dev(bt0[None]), ppr,
                           H.dev(np.array([0], np.int32)))
        import torch
        torch.cuda.synchronize()
        bt1 = np.array(osc.oscar_fork_prefix(gc.ctx, bt0, n_pre, 0, 1, ppr, stream=None), np.int32)
        shared = int(np.sum((bt1 == bt0) & (bt0 >= 0)))
        assert shared >= (n_pre - shape.recent - shape.sink) // 64 - 1, "full history pages are shared"
        bt = np.stack([bt0, bt1])
        total = sum(chunks)
        kc, vc = syn.kv_tokens(wl, 0, total, sub=9)
        q = syn.queries(wl, 0, total, sub=10)
        cu = np.array([0, chunks[0], total], np.int32)
        got = H.run_extend(gc, 0, q, "bf16", kc, vc, cu, [n_pre, n_pre], bt, [0, 1], fx)
        got_u = H.run_extend(gc, 0, q, "bf16", kc, vc, cu, [n_pre, n_pre], bt, [0, 1], fx, unpacked=True)
        assert np.array_equal(got_u, got), "the unpacked-prefix form reads the shared pages the same way"
        # oracle: both prefixes written from scratch into separate pages
        bt_o = np.stack([np.arange(ppr), ppr + np.arange(ppr)]).astype(np.int32)
        img = cache.CacheImage(H.geometry(shape, 2 * ppr, 2))
        for i in range(2):
            cache.write_kv(img, 0, k, v, [0, n_pre], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"],
                           bt_o[i:i + 1], [i])
        want = attention.extend(img, 0, q, kc, vc, cu, [n_pre, n_pre], bt_o, [0, 1], fx["R_K"], fx["R_V"])
        H.assert_decode_close(got, want)
    finally:
        gc.close()


def test_extend_flags_host_sizes_that_miss_a_chunk(osc):
    """A max_chunk below a request's chunk length sets OSCAR_DEV_BAD_LEN (no silent partial output);
    the context stays usable and a correct call afterwards reports no error."""
    import torch
    shape = syn.Shape(32, 8, 128, 64, 32, 4, 128, 1)
    wl = syn.Workload("badlen", shape, [0], seed=43, dtype="bf16")
    fx = H.fixture(wl)
    gc, geom, bt = _setup(wl, fx, [300])
    try:
        t = 100
        k, v = syn.kv_tokens(wl, 0, t, sub=3)
        q = syn.queries(wl, 0, t, sub=4)
        cu = np.array([0, t], np.int32)
        ws_bytes = osc.oscar_extend_workspace_size(gc.cfg, t)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        out = torch.zeros((t, shape.n_q_heads, shape.head_dim), dtype=torch.float32, device="cuda")
        osc.oscar_set_layer_clip(gc.ctx, 0, fx["clip_K"], fx["clip_V"])
        osc.oscar_extend_attn(gc.ctx, 0, H.dev_input(q, "bf16"), osc.DTYPE_BF16, H.dev_input(k, "bf16"),
                              H.dev_input(v, "bf16"), osc.DTYPE_BF16, out, osc.DTYPE_F32, H.dev(cu),
                              H.dev(np.array([300], np.int32)), 1, t, 40, H.dev(bt), bt.shape[1],
                              H.dev(np.zeros(1, np.int32)), H.dev(fx["R_K"]), H.dev(fx["R_V"]), ws, ws_bytes)
        assert osc.oscar_check_status(gc.ctx) & osc.DEV_BAD_LEN
        got = H.run_extend(gc, 0, q, "bf16", k, v, cu, [300], bt, [0], fx)   # asserts a clean status
        assert np.all(np.isfinite(got))
    finally:
        gc.close()


def test_extend_step_equals_extend_then_write(osc):
    """oscar_extend_step = oscar_extend_attn then oscar_write_kv of the chunk: the same outputs and the same
    cache bytes (pages and window slots), bit for bit; then a decode over the extended cache matches the oracle.
    The step runs with the unpacked-prefix workspace, the separate calls with the base one."""
    import torch
    shape = syn.Shape(32, 8, 128, 64, 32, 4, 128, 1)
    wl = syn.Workload("xstep", shape, [0], seed=47, dtype="bf16")
    fx = H.fixture(wl)
    prefix, chunks = [700, 150], [300, 90]
    outs, pools, slabs = [], [], []
    for fused in (False, True):
        gc, geom, bt = _setup(wl, fx, prefix, room=max(chunks))
        ppr = bt.shape[1]
        assert ppr * 64 >= max(p + c for p, c in zip(prefix, chunks))
        try:
            total = sum(chunks)
            k, v = syn.kv_tokens(wl, 0, total, sub=11)
            q = syn.queries(wl, 0, total, sub=12)
            cu = np.array([0, chunks[0], total], np.int32)
            ws_bytes = (osc.oscar_extend_workspace_size_unpacked(gc.cfg, total, 2, max(prefix), max(chunks)) if fused
                        else osc.oscar_extend_workspace_size(gc.cfg, total))
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
            out = torch.empty((total, shape.n_q_heads, shape.head_dim), dtype=torch.float32, device="cuda")
            args = (H.dev_input(q, "bf16"), osc.DTYPE_BF16, H.dev_input(k, "bf16"), H.dev_input(v, "bf16"),
                    osc.DTYPE_BF16, out, osc.DTYPE_F32, H.dev(cu), H.dev(np.array(prefix, np.int32)), 2, total,
                    max(chunks), H.dev(bt), ppr, H.dev(np.arange(2, dtype=np.int32)), H.dev(fx["R_K"]),
                    H.dev(fx["R_V"]))
            if fused:
                osc.oscar_extend_step(gc.ctx, 0, *args, fx["clip_K"], fx["clip_V"], ws, ws_bytes)
            else:
                osc.oscar_extend_attn(gc.ctx, 0, *args, ws, ws_bytes)
                q_d, _, k_d, v_d, _, _, _, cu_d, pre_d, _, _, _, bt_d, _, slots_d, rk_d, rv_d = args
                osc.oscar_write_kv(gc.ctx, 0, k_d, v_d, osc.DTYPE_BF16, cu_d, pre_d, 2, total, rk_d, rv_d,
                                   fx["clip_K"], fx["clip_V"], bt_d, ppr, slots_d)
            assert osc.oscar_check_status(gc.ctx) == 0
            outs.append(out.cpu().numpy())
            pools.append(gc.pool_np().copy())
            slabs.append(gc.slab_np().copy())
            if fused:
                n = [p + c for p, c in zip(prefix, chunks)]
                qd = syn.queries(wl, 0, 2, sub=13)
                got = H.run_decode(gc, 0, qd, "bf16", bt, n, [0, 1], fx)
                img = cache.CacheImage(geom)
                img.pool, img.slab = gc.pool_np(), gc.slab_np()
                want = attention.decode(img, 0, qd, bt, n, [0, 1], fx["R_K"], fx["R_V"])
                H.assert_decode_close(got, want)
        finally:
            gc.close()
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(pools[0], pools[1])
    assert np.array_equal(slabs[0], slabs[1])
