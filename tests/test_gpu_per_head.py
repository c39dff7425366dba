"""Per-kv-head rotations (configuration rotation_per_kv_head = 1, R_K and R_V [Hkv][d][d]) on the GPU.

The pages fix one rotation per layer ("fixed per-layer rotations", arXiv abstract; the calibration of
the gist.science summary, section 2.2 A, is per layer).  A rotation per kv head is a variant of ours:
each kv head calibrated on its own query group and attention outputs.  Two checks:
  * all per-head rotations equal to the layer's rotation: the cache bytes and every output are bit
    for bit those of the per-layer path (same kernels, same arithmetic per row; only where each row
    finds its rotation changes);
  * distinct per-head rotations: the write (BF16 rows on the tensor-core write, float32 rows on the
    CUDA-core write), appends, the fused step, decode and extend against the oracle on the same
    seeded inputs, with the tolerances of the per-layer tests.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import attention, cache, rotation
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


SHAPE = syn.Shape(32, 8, 128, 64, 32, 4, 128, 1)


def _head_fixture(wl):
    q = syn.queries(wl, 0, 256, calib=True)
    k, v = syn.kv_tokens(wl, 0, 256, calib=True)
    return rotation.head_fixture(q, k, v)


def _write(osc, gc, fx, k, v, dtype, lens, start, bt):
    b = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    osc.oscar_write_kv(gc.ctx, 0, H.dev_input(k, dtype), H.dev_input(v, dtype), H.dtype_code(dtype), H.dev(cu),
                       H.dev(np.asarray(start, np.int32)), b, int(cu[-1]), H.dev(fx["R_K"]), H.dev(fx["R_V"]),
                       fx["clip_K"], fx["clip_V"], H.dev(bt), bt.shape[1], H.dev(np.arange(b, dtype=np.int32)))
    assert osc.oscar_check_status(gc.ctx) == 0
    return cu


def _inputs(wl, lens, sub0=0):
    ks, vs = zip(*[syn.kv_tokens(wl, 0, n, sub=sub0 + i) for i, n in enumerate(lens)])
    return np.concatenate(ks), np.concatenate(vs)


def _run_step(osc, gc, fx, kn, vn, q, lens_after, bt, max_seq, ws, ws_bytes):
    import torch
    b = q.shape[0]
    out = torch.empty((b, SHAPE.n_q_heads, SHAPE.head_dim), dtype=torch.float32, device="cuda")
    osc.oscar_decode_step(gc.ctx, 0, H.dev_input(kn, "bf16"), H.dev_input(vn, "bf16"), osc.DTYPE_BF16,
                          H.dev_input(q, "bf16"), osc.DTYPE_BF16, out, osc.DTYPE_F32, H.dev(bt), bt.shape[1],
                          H.dev(np.asarray(lens_after, np.int32)), H.dev(np.arange(b, dtype=np.int32)), b, max_seq,
                          SHAPE.sink, SHAPE.recent, H.dev(fx["R_K"]), H.dev(fx["R_V"]), fx["clip_K"], fx["clip_V"], ws,
                          ws_bytes)
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"], ids=["tensor_core_write", "float32_write"])
def test_per_head_rotations_all_equal_match_the_per_layer_path_bit_for_bit(osc, dtype):
    import torch
    wl = syn.Workload("ph_eq", SHAPE, [0], seed=31, dtype=dtype)
    fx = H.fixture(wl)
    fx8 = dict(fx, R_K=np.ascontiguousarray(np.stack([fx["R_K"]] * SHAPE.n_kv_heads)),
               R_V=np.ascontiguousarray(np.stack([fx["R_V"]] * SHAPE.n_kv_heads)))
    lens = [1500, 700]
    ppr = syn.pages_for(max(lens) + 40, SHAPE.page_size)
    bt = np.arange(2 * ppr, dtype=np.int32).reshape(2, ppr)
    geom = H.geometry(SHAPE, 2 * ppr, 2)
    ga = H.make_gpu_cache(geom, SHAPE.n_q_heads, ppr)
    gb = H.make_gpu_cache(geom, SHAPE.n_q_heads, ppr, rotation_per_kv_head=1)
    try:
        k, v = _inputs(wl, lens)
        _write(osc, ga, fx, k, v, dtype, lens, [0, 0], bt)
        _write(osc, gb, fx8, k, v, dtype, lens, [0, 0], bt)
        assert np.array_equal(ga.pool_np(), gb.pool_np()) and np.array_equal(ga.slab_np(), gb.slab_np())
        max_seq = ppr * SHAPE.page_size
        ws_bytes = osc.oscar_decode_workspace_size(ga.cfg, 2, max_seq)
        wsa = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        wsb = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        cur = list(lens)
        for step in range(12):   # fused steps: the append and the query rotation
            kn, vn = syn.kv_tokens(wl, 0, 2, sub=400 + step)
            q = syn.queries(wl, 0, 2, sub=400 + step)
            after = [n + 1 for n in cur]
            oa = _run_step(osc, ga, fx, kn, vn, q, after, bt, max_seq, wsa, ws_bytes)
            ob = _run_step(osc, gb, fx8, kn, vn, q, after, bt, max_seq, wsb, ws_bytes)
            assert torch.equal(oa, ob), step
            cur = after
        assert osc.oscar_check_status(ga.ctx) == 0 and osc.oscar_check_status(gb.ctx) == 0
        assert np.array_equal(ga.pool_np(), gb.pool_np()) and np.array_equal(ga.slab_np(), gb.slab_np())
        # decode only and extend (a 40-token chunk over each request's cache)
        q = syn.queries(wl, 0, 2, sub=500)
        da = H.run_decode(ga, 0, q, "bf16", bt, cur, [0, 1], fx)
        db = H.run_decode(gb, 0, q, "bf16", bt, cur, [0, 1], fx8)
        assert np.array_equal(da, db)
        t = 40
        kc, vc = syn.kv_tokens(wl, 0, 2 * t, sub=501)
        kc, vc = syn.as_input(kc, "bf16"), syn.as_input(vc, "bf16")
        qx = syn.as_input(syn.queries(wl, 0, 2 * t, sub=502), "bf16")
        cu = np.array([0, t, 2 * t], np.int32)
        xa = H.run_extend(ga, 0, qx, "bf16", kc, vc, cu, cur, bt, [0, 1], fx)
        xb = H.run_extend(gb, 0, qx, "bf16", kc, vc, cu, cur, bt, [0, 1], fx8)
        assert np.array_equal(xa, xb)
        # the unpacked-prefix form too (its pre-pass forms the same tiles in either context)
        xb_u = H.run_extend(gb, 0, qx, "bf16", kc, vc, cu, cur, bt, [0, 1], fx8, unpacked=True)
        assert np.array_equal(xb_u, xa)
    finally:
        ga.close()
        gb.close()


@pytest.mark.parametrize("dtype", ["bf16", "f32"], ids=["tensor_core_write", "float32_write"])
def test_per_head_rotations_parity(osc, dtype):
    wl = syn.Workload("ph", SHAPE, [0], seed=32, dtype=dtype)
    fx = _head_fixture(wl)
    assert fx["R_K"].shape == (SHAPE.n_kv_heads, SHAPE.head_dim, SHAPE.head_dim)
    lens = [2000, 900]
    ppr = syn.pages_for(max(lens) + 80, SHAPE.page_size)
    bt = np.arange(2 * ppr, dtype=np.int32).reshape(2, ppr)
    geom = H.geometry(SHAPE, 2 * ppr, 2)
    img = cache.CacheImage(geom)
    gc = H.make_gpu_cache(geom, SHAPE.n_q_heads, ppr, rotation_per_kv_head=1)
    slots = np.arange(2, dtype=np.int32)
    try:
        k, v = _inputs(wl, lens, sub0=10)
        cu = _write(osc, gc, fx, k, v, dtype, lens, [0, 0], bt)
        diag = cache.write_kv(img, 0, k, v, cu, [0, 0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, slots)
        res = H.compare_history(gc.pool_np(), geom, 0, diag)
        assert res["elements"] == sum(n - SHAPE.sink - SHAPE.recent for n in lens) * 2 * 8 * 128
        H.compare_window(gc.slab_np(), img.slab, 0, range(2))
        # appends (each evicts a ring token into INT2 with its head's rotation)
        cur = list(lens)
        for step in range(30):
            kn, vn = (syn.as_input(x, "bf16") for x in syn.kv_tokens(wl, 0, 2, sub=200 + step))
            sl = np.array(cur, np.int32)
            d_app = cache.append_step(img, 0, kn, vn, sl, fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, slots)
            osc.oscar_append_step(gc.ctx, 0, H.dev_input(kn, "bf16"), H.dev_input(vn, "bf16"), osc.DTYPE_BF16,
                                  H.dev(sl), 2, H.dev(fx["R_K"]), H.dev(fx["R_V"]), fx["clip_K"], fx["clip_V"],
                                  H.dev(bt), ppr, H.dev(slots))
            cur = [n + 1 for n in cur]
        assert osc.oscar_check_status(gc.ctx) == 0
        H.compare_history(gc.pool_np(), geom, 0, d_app)
        H.compare_window(gc.slab_np(), img.slab, 0, range(2))
        # decode over the GPU's own cache against the oracle over the same cache image
        gimg = cache.CacheImage(geom)
        gimg.pool, gimg.slab = gc.pool_np(), gc.slab_np()
        for scale in (1.0, 0.25):
            q = syn.queries(wl, 0, 2, sub=300, scale=scale)
            got = H.run_decode(gc, 0, q, "bf16", bt, cur, slots, fx)
            want = attention.decode(gimg, 0, syn.as_input(q, "bf16"), bt, cur, slots, fx["R_K"], fx["R_V"])
            H.assert_decode_close(got, want)
        # extend: a chunk over each request's cache
        t = 48
        kc, vc = syn.kv_tokens(wl, 0, 2 * t, sub=301)
        kc, vc = syn.as_input(kc, "bf16"), syn.as_input(vc, "bf16")
        qx = syn.as_input(syn.queries(wl, 0, 2 * t, sub=302), "bf16")
        cux = np.array([0, t, 2 * t], np.int32)
        got = H.run_extend(gc, 0, qx, "bf16", kc, vc, cux, cur, bt, slots, fx)
        got_u = H.run_extend(gc, 0, qx, "bf16", kc, vc, cux, cur, bt, slots, fx, unpacked=True)
        assert np.array_equal(got_u, got), "unpacked-prefix form with a rotation per kv head"
        want = attention.extend(gimg, 0, qx, kc, vc, cux, cur, bt, slots, fx["R_K"], fx["R_V"])
        H.assert_decode_close(got, want)
    finally:
        gc.close()


@pytest.mark.parametrize("seed", range(6))
def test_per_head_random_requests(osc, seed):
    """Random shapes (GQA 1-8, d = 64 / 128, pages 16-64, with and without sink, windows 32-128), BF16 or
    float32 rows, 1-4 requests with distinct per-kv-head rotations: the write against the oracle under the
    near-boundary rule (window bit-exact), then decode and extend (the unpacked-prefix form) within the
    decode tolerance of the oracle over the GPU's cache; queries and chunk rows are BF16 values."""
    rng = np.random.default_rng(13000 + seed)
    gq, hkv = int(rng.choice([1, 2, 4, 8])), int(rng.choice([2, 4, 8]))
    d, page = int(rng.choice([64, 128])), int(rng.choice([16, 32, 64]))
    sink, recent = int(rng.choice([0, 4])), int(rng.choice([32, 64, 128]))
    dtype = str(rng.choice(["bf16", "f32"]))
    shape = syn.Shape(gq * hkv, hkv, d, page, 32, sink, recent, 1)
    b = int(rng.integers(1, 5))
    lens = [int(x) for x in rng.integers(1, 1500, size=b)]
    chunks = [int(x) for x in rng.integers(0, 150, size=b)]
    chunks[int(rng.integers(0, b))] = int(rng.integers(1, 150))
    wl = syn.Workload("ph_rand", shape, [0], seed=1400 + seed, dtype=dtype)
    fx = _head_fixture(wl)
    ppr = max(syn.pages_for(n + c + 1, page) for n, c in zip(lens, chunks)) + 1
    bt = np.arange(b * ppr, dtype=np.int32).reshape(b, ppr)
    geom = H.geometry(shape, b * ppr, b)
    img = cache.CacheImage(geom)
    gc = H.make_gpu_cache(geom, shape.n_q_heads, ppr, rotation_per_kv_head=1)
    slots = np.arange(b, dtype=np.int32)
    try:
        k, v = _inputs(wl, lens)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        diag = cache.write_kv(img, 0, k, v, cu, np.zeros(b, np.int32), fx["R_K"], fx["R_V"], fx["clip_K"],
                              fx["clip_V"], bt, slots)
        _write(osc, gc, fx, k, v, dtype, lens, [0] * b, bt)
        H.compare_history(gc.pool_np(), geom, 0, diag)
        H.compare_window(gc.slab_np(), img.slab, 0, range(b))
        gimg = cache.CacheImage(geom)
        gimg.pool, gimg.slab = gc.pool_np(), gc.slab_np()
        bf = lambda x: syn.as_input(x, "bf16")
        q = bf(syn.queries(wl, 0, b, sub=41, scale=0.5))
        got = H.run_decode(gc, 0, q, "bf16", bt, lens, list(range(b)), fx)
        H.assert_decode_close(got, attention.decode(gimg, 0, q, bt, lens, list(range(b)), fx["R_K"], fx["R_V"]))
        total = sum(chunks)
        kx, vx = (bf(x) for x in syn.kv_tokens(wl, 0, total, sub=42))
        qx = bf(syn.queries(wl, 0, total, sub=43, scale=0.5))
        cux = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
        gx = H.run_extend(gc, 0, qx, "bf16", kx, vx, cux, lens, bt, slots, fx, unpacked=True)
        H.assert_decode_close(gx, attention.extend(gimg, 0, qx, kx, vx, cux, lens, bt, slots, fx["R_K"], fx["R_V"]))
    finally:
        gc.close()
