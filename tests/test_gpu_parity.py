"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded inputs.

Write path: packed codes, scales and zeros bit-exact except elements within
1e-6 relative of a rounding boundary (at most 1e-4 of the elements, listed);
window slab bit-exact.  Decode: max abs error <= 2e-3 and mean abs error <=
2e-4 on unit-scale outputs, given identical packed caches (the oracle's cache
image is uploaded as the GPU cache).
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import attention, cache, quant
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


def _contiguous_bt(batch, pages_per_req, offset=0):
    return (offset + np.arange(batch * pages_per_req, dtype=np.int32)).reshape(batch, pages_per_req)


def _prefill_both(osc, wl, fx, lens, bt, num_pages, max_requests=None, start=None, fill=0):
    """Prefill requests with lengths `lens` on both sides; returns (gpu cache, oracle image, diag, k, v)."""
    s = wl.shape
    b = len(lens)
    geom = H.geometry(s, num_pages, max_requests or b)
    img = cache.CacheImage(geom, fill=fill)
    gc = H.make_gpu_cache(geom, s.n_q_heads, bt.shape[1], fill=fill)
    ks, vs = [], []
    for i, n in enumerate(lens):
        k, v = syn.kv_tokens(wl, 0, n, sub=i)
        ks.append(k)
        vs.append(v)
    k = np.concatenate(ks)
    v = np.concatenate(vs)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sp = np.zeros(b, np.int32) if start is None else np.asarray(start, np.int32)
    slots = np.arange(b, dtype=np.int32)
    diag = cache.write_kv(img, 0, k, v, cu, sp, fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, slots)
    osc.oscar_write_kv(gc.ctx, 0, H.dev_input(k, wl.dtype), H.dev_input(v, wl.dtype), H.dtype_code(wl.dtype),
                       H.dev(cu), H.dev(sp), b, int(cu[-1]), H.dev(fx["R_K"]), H.dev(fx["R_V"]), fx["clip_K"],
                       fx["clip_V"], H.dev(bt), bt.shape[1], H.dev(slots))
    assert osc.oscar_check_status(gc.ctx) == 0
    return gc, img, diag, k, v


# ---------------------------------------------------------------------------------------------- write path
@pytest.mark.parametrize("wl,lens", [
    (syn.tiny(), [512]),
    (syn.Workload("d128_ragged", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=1), [1000, 4133, 131, 70]),
    (syn.Workload("d64_p32_bf16", syn.Shape(8, 2, 64, 32, 32, 4, 16, 1), [0], seed=6), [300, 77]),
], ids=["tiny_f32", "d128_ragged_bf16", "d64_p32"])
def test_write_parity(osc, wl, lens):
    fx = H.fixture(wl)
    s = wl.shape
    ppr = max(syn.pages_for(n, s.page_size) for n in lens) + 1
    bt = _contiguous_bt(len(lens), ppr)
    gc, img, diag, _, _ = _prefill_both(osc, wl, fx, lens, bt, len(lens) * ppr)
    try:
        res = H.compare_history(gc.pool_np(), img.g, 0, diag)
        H.compare_window(gc.slab_np(), img.slab, 0, range(len(lens)))
        assert res["elements"] > 0
    finally:
        gc.close()


@pytest.mark.parametrize("seed", range(8))
def test_write_random_requests(osc, seed):
    """Random shapes (d = 64 / 128, pages 16-64, 2-8 kv heads, with and without sink, windows 32-128), BF16
    or float32 rows, the dense or the Hadamard-only rotation, 1-4 requests on pages handed out in reverse
    order: a prefill of random lengths, then an extend chunk of each request after its prefix (ring tokens
    evicted into history).  Codes, scales and zeros against the oracle under the near-boundary rule, window
    slots bit-exact."""
    rng = np.random.default_rng(7000 + seed)
    gq, hkv = int(rng.choice([1, 4])), int(rng.choice([2, 4, 8]))
    d, page = int(rng.choice([64, 128])), int(rng.choice([16, 32, 64]))
    sink, recent = int(rng.choice([0, 4])), int(rng.choice([32, 64, 128]))
    dtype = str(rng.choice(["bf16", "f32"]))
    had = bool(rng.integers(0, 2))
    shape = syn.Shape(gq * hkv, hkv, d, page, 32, sink, recent, 1)
    b = int(rng.integers(1, 5))
    lens = [int(x) for x in rng.integers(0, 1500, size=b)]
    lens[int(rng.integers(0, b))] = int(rng.integers(1, 1500))
    chunk = [int(x) for x in rng.integers(0, 300, size=b)]
    wl = syn.Workload("wr_rand", shape, [0], seed=900 + seed, dtype=dtype)
    fx = H.fixture(wl, u_identity=had)
    ppr = max(syn.pages_for(n + c + 1, page) for n, c in zip(lens, chunk)) + 1
    bt = np.arange(b * ppr, dtype=np.int32)[::-1].copy().reshape(b, ppr)
    geom = H.geometry(shape, b * ppr, b)
    img = cache.CacheImage(geom)
    gc = H.make_gpu_cache(geom, shape.n_q_heads, ppr)
    slots = np.arange(b, dtype=np.int32)
    try:
        for now, start, sub0 in ((lens, [0] * b, 0), (chunk, lens, 10)):
            k = np.concatenate([syn.kv_tokens(wl, 0, n, sub=sub0 + i)[0] for i, n in enumerate(now)])
            v = np.concatenate([syn.kv_tokens(wl, 0, n, sub=sub0 + i)[1] for i, n in enumerate(now)])
            cu = np.concatenate([[0], np.cumsum(now)]).astype(np.int32)
            sp = np.asarray(start, np.int32)
            diag = cache.write_kv(img, 0, k, v, cu, sp, fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, slots)
            if int(cu[-1]) == 0:
                continue
            if had:
                osc.oscar_write_kv_hadamard(gc.ctx, 0, H.dev_input(k, dtype), H.dev_input(v, dtype),
                                            H.dtype_code(dtype), H.dev(cu), H.dev(sp), b, int(cu[-1]), fx["clip_K"],
                                            fx["clip_V"], H.dev(bt), ppr, H.dev(slots))
            else:
                osc.oscar_write_kv(gc.ctx, 0, H.dev_input(k, dtype), H.dev_input(v, dtype), H.dtype_code(dtype),
                                   H.dev(cu), H.dev(sp), b, int(cu[-1]), H.dev(fx["R_K"]), H.dev(fx["R_V"]),
                                   fx["clip_K"], fx["clip_V"], H.dev(bt), ppr, H.dev(slots))
            assert osc.oscar_check_status(gc.ctx) == 0
            H.compare_history(gc.pool_np(), geom, 0, diag)
            H.compare_window(gc.slab_np(), img.slab, 0, range(b))
    finally:
        gc.close()


def test_naive_int2_identity_rotation(osc):
    """The pages' naive INT2 baseline (no rotation, R_K = R_V = I; clip from the unrotated calibration values)
    runs on the same kernels: write codes against the oracle, and decode against the oracle on the GPU's cache."""
    from oracle import rotation
    wl = syn.Workload("naive", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=11)
    s = wl.shape
    eye = np.eye(s.head_dim, dtype=np.float32)
    kc, vc = syn.kv_tokens(wl, 0, 256, calib=True)
    fx = {"R_K": eye, "R_V": eye, "clip_K": float(np.float32(rotation.clip_threshold(kc, eye))),
          "clip_V": float(np.float32(rotation.clip_threshold(vc, eye)))}
    lens = [2100, 600]
    ppr = max(syn.pages_for(n, s.page_size) for n in lens) + 1
    bt = _contiguous_bt(len(lens), ppr)
    gc, img, diag, _, _ = _prefill_both(osc, wl, fx, lens, bt, len(lens) * ppr)
    try:
        res = H.compare_history(gc.pool_np(), img.g, 0, diag, exact_ties=True)
        assert res["elements"] > 0
        H.compare_window(gc.slab_np(), img.slab, 0, range(len(lens)))
        q = syn.queries(wl, 0, len(lens))
        got = H.run_decode(gc, 0, q, "bf16", bt, lens, [0, 1], fx)
        gimg = cache.CacheImage(img.g)
        gimg.pool, gimg.slab = gc.pool_np(), gc.slab_np()
        want = attention.decode(gimg, 0, q, bt, lens, [0, 1], fx["R_K"], fx["R_V"])
        H.assert_decode_close(got, want)
    finally:
        gc.close()


@pytest.mark.parametrize("path", ["dense_bf16", "dense_f32", "hadamard_f32"])
def test_write_group_zero_rounded_past_the_clip(osc, path):
    """Groups held within a BF16 ulp of a clip that BF16 cannot represent (c = 1 + 0.75 * 2^-7): the zero
    rounds past the clip, (clip - z) / s is about -6, and every code is 0 (3 for the mirrored groups below
    -c) on both sides ([summary §2.2 B]: clip, then min/max INT2 with codes clamped to the four levels).
    The rotated rows are alpha (1.0 x16, 1.0078125 x16) and their negatives, alpha = 1 + 2^-8 + 2^-10: dense
    R = alpha I on BF16 rows (tensor cores) and on float32 rows, and the Hadamard-only write of float32 rows
    whose Hadamard rotation is that row (x = y R^T).  Even tokens carry the edge rows in K, odd tokens in V,
    and the other rows are the seeded workload."""
    shape = syn.Shape(32, 8, 128, 64, 32, 4, 128, 1)
    dtype = "bf16" if path == "dense_bf16" else "f32"
    wl = syn.Workload("clip_edge", shape, [0], seed=23, dtype=dtype)
    c = 1 + 0.75 * 2.0 ** -7
    alpha = 1 + 2.0 ** -8 + 2.0 ** -10
    row = np.repeat([1.0, 1.0078125], 16)
    edge = np.concatenate([row, row, -row, -row])
    if path == "hadamard_f32":
        had = H.fixture(wl, u_identity=True)
        r_k, r_v = had["R_K"], had["R_V"]
        xk, xv = (alpha * edge) @ np.asarray(r_k, np.float64).T, (alpha * edge) @ np.asarray(r_v, np.float64).T
    else:
        r_k = r_v = (alpha * np.eye(128)).astype(np.float32)
        xk = xv = edge
    fx = {"R_K": r_k, "R_V": r_v, "clip_K": c, "clip_V": c}
    n = 300
    k, v = syn.kv_tokens(wl, 0, n)
    k, v = np.array(k, np.float64), np.array(v, np.float64)
    k[0::2] = xk
    v[1::2] = xv
    k, v = k.astype(np.float32), v.astype(np.float32)
    ppr = syn.pages_for(n, shape.page_size) + 1
    bt = _contiguous_bt(1, ppr)
    geom = H.geometry(shape, ppr, 1)
    img = cache.CacheImage(geom)
    gc = H.make_gpu_cache(geom, shape.n_q_heads, ppr)
    cu, sp, slots = np.array([0, n], np.int32), np.zeros(1, np.int32), np.zeros(1, np.int32)
    try:
        diag = cache.write_kv(img, 0, k, v, cu, sp, r_k, r_v, c, c, bt, slots)
        for kv in ("k", "v"):
            z = diag[kv]["zero"]
            assert np.any(z == 1.0078125) and np.any(z == -1.0078125)
        if path == "hadamard_f32":
            osc.oscar_write_kv_hadamard(gc.ctx, 0, H.dev_input(k, dtype), H.dev_input(v, dtype), H.dtype_code(dtype),
                                        H.dev(cu), H.dev(sp), 1, n, c, c, H.dev(bt), ppr, H.dev(slots))
        else:
            osc.oscar_write_kv(gc.ctx, 0, H.dev_input(k, dtype), H.dev_input(v, dtype), H.dtype_code(dtype), H.dev(cu),
                               H.dev(sp), 1, n, H.dev(r_k), H.dev(r_v), c, c, H.dev(bt), ppr, H.dev(slots))
        assert osc.oscar_check_status(gc.ctx) == 0
        res = H.compare_history(gc.pool_np(), geom, 0, diag, exact_ties=(path == "dense_bf16"))
        assert res["elements"] > 0
        H.compare_window(gc.slab_np(), img.slab, 0, range(1))
    finally:
        gc.close()


def _hadamard_case(osc, shape, dtype, rph):
    """Data-oblivious rotation R = H P (U = I), written by oscar_write_kv_hadamard (BF16 rows: one exact
    +-1 plane on the tensor cores; float32 rows: the fast Walsh-Hadamard transform) against the oracle's
    dense R: three requests of ragged lengths (row counts not a multiple of a tile), then an extend chunk
    of each request after its prefix (eviction of ring tokens, then the write)."""
    wl = syn.Workload("had", shape, [0], seed=7, dtype=dtype)
    fx = H.fixture(wl, u_identity=True)
    lens = [700, 300, 37]
    s = wl.shape
    ppr = syn.pages_for(max(lens) + 200, s.page_size) + 1
    bt = _contiguous_bt(3, ppr)
    geom = H.geometry(s, 3 * ppr, 3)
    img = cache.CacheImage(geom)
    gc = H.make_gpu_cache(geom, s.n_q_heads, ppr, rotation_per_kv_head=rph)
    slots = np.arange(3, dtype=np.int32)

    def write(lens_now, start, sub0):
        k = np.concatenate([syn.kv_tokens(wl, 0, n, sub=sub0 + i)[0] for i, n in enumerate(lens_now)])
        v = np.concatenate([syn.kv_tokens(wl, 0, n, sub=sub0 + i)[1] for i, n in enumerate(lens_now)])
        cu = np.concatenate([[0], np.cumsum(lens_now)]).astype(np.int32)
        sp = np.asarray(start, np.int32)
        diag = cache.write_kv(img, 0, k, v, cu, sp, fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, slots)
        osc.oscar_write_kv_hadamard(gc.ctx, 0, H.dev_input(k, dtype), H.dev_input(v, dtype), H.dtype_code(dtype),
                                    H.dev(cu), H.dev(sp), 3, int(cu[-1]), fx["clip_K"], fx["clip_V"], H.dev(bt), ppr,
                                    H.dev(slots))
        assert osc.oscar_check_status(gc.ctx) == 0
        return diag

    try:
        diag = write(lens, [0, 0, 0], 0)
        H.compare_history(gc.pool_np(), geom, 0, diag)
        H.compare_window(gc.slab_np(), img.slab, 0, range(3))
        chunk = [90, 33, 150]
        diag = write(chunk, lens, 10)
        H.compare_history(gc.pool_np(), geom, 0, diag)
        H.compare_window(gc.slab_np(), img.slab, 0, range(3))
    finally:
        gc.close()


@pytest.mark.parametrize("shape", [syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), syn.Shape(8, 4, 64, 16, 32, 4, 32, 1),
                                   syn.Shape(24, 6, 128, 32, 32, 4, 64, 1)],
                         ids=["d128_p64", "d64_p16", "d128_p32_six_kv_heads"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_write_hadamard_only_parity(osc, shape, dtype):
    """The Hadamard-only write against the oracle (see _hadamard_case), one rotation per layer."""
    _hadamard_case(osc, shape, dtype, 0)


@pytest.mark.parametrize("shape", [syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), syn.Shape(8, 4, 64, 16, 32, 4, 32, 1)],
                         ids=["d128_p64", "d64_p16"])
def test_write_hadamard_only_parity_in_a_per_head_context(osc, shape):
    """The same with BF16 rows in a context that keeps a rotation per kv head: the tensor-core write then
    tiles each kv head's rows separately (a CTA per head, a 3-D row map), and the Hadamard rotation,
    the same for every head, must give the same codes."""
    _hadamard_case(osc, shape, "bf16", 1)


def test_append_and_extend_parity(osc):
    """Prefill, then an extend (evicting ring tokens), then single-token appends, on both sides."""
    wl = syn.Workload("app", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=8)
    fx = H.fixture(wl)
    s = wl.shape
    ppr = 20
    lens0 = [300, 140]
    bt = _contiguous_bt(2, ppr)
    gc, img, diag0, _, _ = _prefill_both(osc, wl, fx, lens0, bt, 2 * ppr)
    try:
        H.compare_history(gc.pool_np(), img.g, 0, diag0)
        # extend by 90 and 200 tokens
        ext = [90, 200]
        k = np.concatenate([syn.kv_tokens(wl, 0, n, sub=10 + i)[0] for i, n in enumerate(ext)])
        v = np.concatenate([syn.kv_tokens(wl, 0, n, sub=10 + i)[1] for i, n in enumerate(ext)])
        cu = np.array([0, ext[0], sum(ext)], np.int32)
        sp = np.array(lens0, np.int32)
        slots = np.arange(2, dtype=np.int32)
        diag1 = cache.write_kv(img, 0, k, v, cu, sp, fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, slots)
        osc.oscar_write_kv(gc.ctx, 0, H.dev_input(k, "bf16"), H.dev_input(v, "bf16"), osc.DTYPE_BF16, H.dev(cu),
                           H.dev(sp), 2, int(cu[-1]), H.dev(fx["R_K"]), H.dev(fx["R_V"]), fx["clip_K"], fx["clip_V"],
                           H.dev(bt), ppr, H.dev(slots))
        assert osc.oscar_check_status(gc.ctx) == 0
        H.compare_history(gc.pool_np(), img.g, 0, diag1)
        H.compare_window(gc.slab_np(), img.slab, 0, range(2))
        # 40 appends
        lens = [lens0[0] + ext[0], lens0[1] + ext[1]]
        for step in range(40):
            kn, vn = syn.kv_tokens(wl, 0, 2, sub=100 + step)
            sl = np.array(lens, np.int32)
            diag = cache.append_step(img, 0, kn, vn, sl, fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt,
                                     slots)
            osc.oscar_append_step(gc.ctx, 0, H.dev_input(kn, "bf16"), H.dev_input(vn, "bf16"), osc.DTYPE_BF16,
                                  H.dev(sl), 2, H.dev(fx["R_K"]), H.dev(fx["R_V"]), fx["clip_K"], fx["clip_V"],
                                  H.dev(bt), ppr, H.dev(slots))
            if step % 13 == 0 or step == 39:
                assert osc.oscar_check_status(gc.ctx) == 0
                H.compare_history(gc.pool_np(), img.g, 0, diag)
            lens = [n + 1 for n in lens]
        assert osc.oscar_check_status(gc.ctx) == 0
        H.compare_window(gc.slab_np(), img.slab, 0, range(2))
        # decode after the appends on the GPU's own cache, against the oracle on its own cache
        q = syn.queries(wl, 0, 2)
        want = attention.decode(img, 0, q, bt, lens, slots, fx["R_K"], fx["R_V"])
        got = H.run_decode(gc, 0, q, "bf16", bt, lens, slots, fx)
        H.assert_decode_close(got, want)
    finally:
        gc.close()


@pytest.mark.parametrize("shape,ppr,lens0,steps", [
    (syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), 24, [1300, 131], 70),   # crosses a page of evicted tokens
    (syn.Shape(8, 4, 64, 16, 32, 4, 32, 1), 24, [300, 35], 40),        # d = 64, 16-token pages, GQA 2
], ids=["d128_p64_gq4", "d64_p16_gq2"])
@pytest.mark.parametrize("form", ["three_kernels", "one_launch"])
def test_fused_decode_step_equals_append_then_decode(osc, shape, ppr, lens0, steps, form):
    """oscar_decode_step (the query rotation and the append in one grid; in the one-launch form the
    append alone, then the one decode kernel) leaves the same cache and output, bit for bit, as
    oscar_append_step followed by oscar_decode_attn in the same form; checked against the oracle at
    the end.  The second request is one token short of evicting at the first step."""
    import torch
    wl = syn.Workload("step", shape, [0], seed=12)
    fx = H.fixture(wl)
    bt = _contiguous_bt(2, ppr)
    ga, img, _, _, _ = _prefill_both(osc, wl, fx, lens0, bt, 2 * ppr)
    gb, _, _, _, _ = _prefill_both(osc, wl, fx, lens0, bt, 2 * ppr)
    code = osc.DECODE_ONE_LAUNCH if form == "one_launch" else osc.DECODE_THREE_KERNELS
    osc.oscar_set_decode_form(ga.ctx, code)
    osc.oscar_set_decode_form(gb.ctx, code)
    try:
        hq, d = shape.n_q_heads, shape.head_dim
        slots = np.arange(2, dtype=np.int32)
        max_seq = shape.page_size * ppr
        ws_bytes = osc.oscar_decode_workspace_size(ga.cfg, 2, max_seq)
        wsa = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        wsb = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        rk, rv, btd, sld = H.dev(fx["R_K"]), H.dev(fx["R_V"]), H.dev(bt), H.dev(slots)
        lens = list(lens0)
        for step in range(steps):
            kn, vn = syn.kv_tokens(wl, 0, 2, sub=300 + step)
            q = syn.queries(wl, 0, 2, sub=300 + step)
            before = H.dev(np.array(lens, np.int32))
            after = H.dev(np.array(lens, np.int32) + 1)
            kd, vd, qd = H.dev_input(kn, "bf16"), H.dev_input(vn, "bf16"), H.dev_input(q, "bf16")
            oa = torch.empty((2, hq, d), dtype=torch.float32, device="cuda")
            ob = torch.empty_like(oa)
            osc.oscar_append_step(ga.ctx, 0, kd, vd, osc.DTYPE_BF16, before, 2, rk, rv, fx["clip_K"], fx["clip_V"],
                                  btd, ppr, sld)
            osc.oscar_decode_attn(ga.ctx, 0, qd, osc.DTYPE_BF16, oa, osc.DTYPE_F32, btd, ppr, after, sld, 2, max_seq,
                                  shape.sink, shape.recent, rk, rv, wsa, ws_bytes)
            osc.oscar_decode_step(gb.ctx, 0, kd, vd, osc.DTYPE_BF16, qd, osc.DTYPE_BF16, ob, osc.DTYPE_F32, btd, ppr,
                                  after, sld, 2, max_seq, shape.sink, shape.recent, rk, rv, fx["clip_K"],
                                  fx["clip_V"], wsb, ws_bytes)
            assert torch.equal(oa, ob), step
            cache.append_step(img, 0, kn, vn, np.array(lens, np.int32), fx["R_K"], fx["R_V"], fx["clip_K"],
                              fx["clip_V"], bt, slots)
            lens = [n + 1 for n in lens]
        assert osc.oscar_check_status(ga.ctx) == 0 and osc.oscar_check_status(gb.ctx) == 0
        assert np.array_equal(ga.pool_np(), gb.pool_np())
        assert np.array_equal(ga.slab_np(), gb.slab_np())
        want = attention.decode(img, 0, q, bt, lens, slots, fx["R_K"], fx["R_V"])
        H.assert_decode_close(ob.cpu().numpy().astype(np.float64), want)
    finally:
        ga.close()
        gb.close()


@pytest.mark.parametrize("seed", range(6))
def test_fused_decode_step_random_requests(osc, seed):
    """Random shapes (GQA 1-8, d = 64 / 128, pages 16-64, with and without sink, windows 32-128), 1-5
    requests and 5-30 fused decode steps in a random decode form: after every step the appended rows
    against the oracle's append under the near-boundary rule, and every seventh step's output within the
    decode tolerance of the oracle decoding the GPU's own cache (the tolerance is stated for identical
    caches); window slots bit-exact at the end."""
    import torch
    rng = np.random.default_rng(11000 + seed)
    gq, hkv = int(rng.choice([1, 2, 4, 8])), int(rng.choice([2, 4, 8]))
    d, page = int(rng.choice([64, 128])), int(rng.choice([16, 32, 64]))
    sink, recent = int(rng.choice([0, 4])), int(rng.choice([32, 64, 128]))
    shape = syn.Shape(gq * hkv, hkv, d, page, 32, sink, recent, 1)
    b = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.integers(1, 1500, size=b)]
    steps = int(rng.integers(5, 31))
    one = bool(rng.integers(0, 2))
    wl = syn.Workload("step_rand", shape, [0], seed=1200 + seed)
    fx = H.fixture(wl)
    ppr = max(syn.pages_for(n + steps + 1, page) for n in lens) + 1
    bt = _contiguous_bt(b, ppr)
    gc, img, _, _, _ = _prefill_both(osc, wl, fx, lens, bt, b * ppr)
    osc.oscar_set_decode_form(gc.ctx, osc.DECODE_ONE_LAUNCH if one else osc.DECODE_THREE_KERNELS)
    try:
        slots = np.arange(b, dtype=np.int32)
        max_seq = page * ppr
        ws_bytes = osc.oscar_decode_workspace_size(gc.cfg, b, max_seq)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        rk, rv, btd, sld = H.dev(fx["R_K"]), H.dev(fx["R_V"]), H.dev(bt), H.dev(slots)
        appended = []   # exemptions are budgeted over all steps' appended rows
        for step in range(steps):
            kn, vn = syn.kv_tokens(wl, 0, b, sub=300 + step)
            q = syn.queries(wl, 0, b, sub=300 + step, scale=0.5)
            out = torch.empty((b, shape.n_q_heads, d), dtype=torch.float32, device="cuda")
            osc.oscar_decode_step(gc.ctx, 0, H.dev_input(kn, "bf16"), H.dev_input(vn, "bf16"), osc.DTYPE_BF16,
                                  H.dev_input(q, "bf16"), osc.DTYPE_BF16, out, osc.DTYPE_F32, btd, ppr,
                                  H.dev(np.array(lens, np.int32) + 1), sld, b, max_seq, sink, recent, rk, rv,
                                  fx["clip_K"], fx["clip_V"], ws, ws_bytes)
            assert osc.oscar_check_status(gc.ctx) == 0
            diag = cache.append_step(img, 0, kn, vn, np.array(lens, np.int32), fx["R_K"], fx["R_V"], fx["clip_K"],
                                     fx["clip_V"], bt, slots)
            appended.append(H.compare_history(gc.pool_np(), img.g, 0, diag, enforce_budget=False))
            lens = [n + 1 for n in lens]
            if step % 7 == 6 or step == steps - 1:
                gimg = cache.CacheImage(img.g)
                gimg.pool, gimg.slab = gc.pool_np(), gc.slab_np()
                want = attention.decode(gimg, 0, q, bt, lens, slots, fx["R_K"], fx["R_V"])
                H.assert_decode_close(out.cpu().numpy().astype(np.float64), want)
        H.check_budget(H.merge_results(appended))
        H.compare_window(gc.slab_np(), img.slab, 0, range(b))
    finally:
        gc.close()


def test_prefill_plus_appends_matches_direct_prefill_on_gpu(osc):
    wl = syn.Workload("chain", syn.Shape(16, 8, 128, 64, 32, 4, 128, 1), [0], seed=9)
    fx = H.fixture(wl)
    n0, extra = 400, 70
    ppr = 10
    bt = _contiguous_bt(1, ppr)
    k, v = syn.kv_tokens(wl, 0, n0 + extra)
    geom = H.geometry(wl.shape, ppr, 1)
    a = H.make_gpu_cache(geom, 16, ppr)
    b = H.make_gpu_cache(geom, 16, ppr)
    try:
        args = (H.dev(fx["R_K"]), H.dev(fx["R_V"]), fx["clip_K"], fx["clip_V"], H.dev(bt), ppr, H.dev(np.zeros(1, np.int32)))
        osc.oscar_write_kv(a.ctx, 0, H.dev_input(k[:n0], "bf16"), H.dev_input(v[:n0], "bf16"), osc.DTYPE_BF16,
                           H.dev(np.array([0, n0], np.int32)), H.dev(np.zeros(1, np.int32)), 1, n0, *args)
        for i in range(extra):
            osc.oscar_append_step(a.ctx, 0, H.dev_input(k[n0 + i][None], "bf16"), H.dev_input(v[n0 + i][None], "bf16"),
                                  osc.DTYPE_BF16, H.dev(np.array([n0 + i], np.int32)), 1, *args)
        osc.oscar_write_kv(b.ctx, 0, H.dev_input(k, "bf16"), H.dev_input(v, "bf16"), osc.DTYPE_BF16,
                           H.dev(np.array([0, n0 + extra], np.int32)), H.dev(np.zeros(1, np.int32)), 1, n0 + extra,
                           *args)
        assert osc.oscar_check_status(a.ctx) == 0 and osc.oscar_check_status(b.ctx) == 0
        # the BF16 window is a plain copy on both paths
        assert np.array_equal(a.slab_np(), b.slab_np())
        # history: the prefill runs on the tensor cores, the appends on CUDA cores, so the two caches may
        # differ only where a rotated value sits at a rounding boundary; both must match the oracle's
        # single prefill under the near-boundary rule
        img = cache.CacheImage(geom)
        diag = cache.write_kv(img, 0, k, v, [0, n0 + extra], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"],
                              bt, [0])
        H.compare_history(a.pool_np(), geom, 0, diag)
        H.compare_history(b.pool_np(), geom, 0, diag)
        # rows the prefill wrote in both caches are identical: same rows, same kernel
        pa, pb = a.pool_np(), b.pool_np()
        first_appended_page = (n0 - 128) // 64
        assert np.array_equal(pa[:, :first_appended_page], pb[:, :first_appended_page])
    finally:
        a.close()
        b.close()


# ---------------------------------------------------------------------------------------------- decode
def _decode_case(osc, wl, lens, q_scale=1.0, shuffle=False, fill=0xFF):
    """Oracle-built cache uploaded to the GPU; GPU decode vs oracle decode."""
    fx = H.fixture(wl)
    s = wl.shape
    b = len(lens)
    ppr = max(syn.pages_for(n, s.page_size) for n in lens) + 1
    num_pages = b * ppr
    order = syn.page_permutation(wl.seed, num_pages, shuffle=shuffle)
    bt = order.reshape(b, ppr).astype(np.int32)
    geom = H.geometry(s, num_pages, b)
    img = cache.CacheImage(geom, fill=fill)
    for i, n in enumerate(lens):
        k, v = syn.kv_tokens(wl, 0, n, sub=i)
        cache.write_kv(img, 0, k, v, [0, n], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt[i:i + 1], [i])
    q = syn.queries(wl, 0, b, scale=q_scale)
    want = attention.decode(img, 0, q, bt, lens, np.arange(b), fx["R_K"], fx["R_V"])
    gc = H.make_gpu_cache(geom, s.n_q_heads, ppr)
    try:
        gc.upload(img)
        got = H.run_decode(gc, 0, q, wl.dtype, bt, lens, np.arange(b), fx)
        return got, want
    finally:
        gc.close()


@pytest.mark.parametrize("q_scale", [1.0, 0.25])
def test_decode_parity_tiny(osc, q_scale):
    got, want = _decode_case(osc, syn.tiny(), [512], q_scale)
    H.assert_decode_close(got, want)


@pytest.mark.parametrize("q_scale", [1.0, 0.25])
def test_decode_parity_batch1_gq4(osc, q_scale):
    wl = syn.Workload("b1", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=1)
    got, want = _decode_case(osc, wl, [6000], q_scale)
    H.assert_decode_close(got, want)


def test_decode_parity_gq8_ragged_shuffled(osc):
    wl = syn.Workload("b4", syn.Shape(64, 8, 128, 64, 32, 4, 128, 1), [0], seed=2)
    got, want = _decode_case(osc, wl, [3000, 133, 1029, 64 * 9 + 132], shuffle=True)
    H.assert_decode_close(got, want)


@pytest.mark.parametrize("lens", [[1], [4], [100], [132], [133], [134], [197], [4 + 128 + 64]])
def test_decode_edge_lengths(osc, lens):
    """No history, a single history token, history ending exactly at a page boundary."""
    wl = syn.Workload("edge", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=3)
    got, want = _decode_case(osc, wl, lens)
    H.assert_decode_close(got, want)


def test_decode_gq1_gq2_d64(osc):
    for shape in (syn.Shape(4, 4, 64, 16, 32, 4, 32, 1), syn.Shape(8, 4, 64, 32, 32, 2, 20, 1)):
        wl = syn.Workload("small", shape, [0], seed=4, dtype="f32")
        got, want = _decode_case(osc, wl, [700, 333])
        H.assert_decode_close(got, want)


@pytest.mark.parametrize("seed", range(10))
def test_decode_random_requests(osc, seed):
    """Random shapes (GQA 1-8, d = 64 / 128, pages 16-64, with and without sink, windows 32-128) and 1-6
    requests of random lengths up to 5,000 tokens, written by the GPU and decoded with q x 1 or x 0.25:
    within the decode tolerance of the oracle attending over the GPU's own cache image."""
    rng = np.random.default_rng(9000 + seed)
    gq, hkv = int(rng.choice([1, 2, 4, 8])), int(rng.choice([2, 4, 8]))
    d, page = int(rng.choice([64, 128])), int(rng.choice([16, 32, 64]))
    sink, recent = int(rng.choice([0, 4])), int(rng.choice([32, 64, 128]))
    shape = syn.Shape(gq * hkv, hkv, d, page, 32, sink, recent, 1)
    b = int(rng.integers(1, 7))
    lens = [int(x) for x in rng.integers(1, 5000, size=b)]
    q_scale = float(rng.choice([1.0, 0.25]))
    wl = syn.Workload("dec_rand", shape, [0], seed=800 + seed, dtype="bf16")
    fx = H.fixture(wl)
    ppr = max(syn.pages_for(n, page) for n in lens) + 1
    bt = _contiguous_bt(b, ppr)
    geom = H.geometry(shape, b * ppr, b)
    gc = H.make_gpu_cache(geom, shape.n_q_heads, ppr)
    try:
        ks, vs = zip(*[syn.kv_tokens(wl, 0, n, sub=i) for i, n in enumerate(lens)])
        k, v = np.concatenate(ks), np.concatenate(vs)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        slots = np.arange(b, dtype=np.int32)
        osc.oscar_write_kv(gc.ctx, 0, H.dev_input(k, "bf16"), H.dev_input(v, "bf16"), osc.DTYPE_BF16, H.dev(cu),
                           H.dev(np.zeros(b, np.int32)), b, int(cu[-1]), H.dev(fx["R_K"]), H.dev(fx["R_V"]),
                           fx["clip_K"], fx["clip_V"], H.dev(bt), ppr, H.dev(slots))
        assert osc.oscar_check_status(gc.ctx) == 0
        q = syn.queries(wl, 0, b, sub=31, scale=q_scale)
        got = H.run_decode(gc, 0, q, "bf16", bt, lens, list(range(b)), fx)
        gimg = cache.CacheImage(geom)
        gimg.pool, gimg.slab = gc.pool_np(), gc.slab_np()
        want = attention.decode(gimg, 0, q, bt, lens, list(range(b)), fx["R_K"], fx["R_V"])
        H.assert_decode_close(got, want)
    finally:
        gc.close()


def test_decode_independent_of_split_count(osc):
    """A larger max_seq changes the split plan but not the result (beyond summation order)."""
    wl = syn.Workload("split", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=5)
    fx = H.fixture(wl)
    n = 5000
    ppr = 200
    bt = _contiguous_bt(1, ppr)
    geom = H.geometry(wl.shape, ppr, 1)
    img = cache.CacheImage(geom)
    k, v = syn.kv_tokens(wl, 0, n)
    cache.write_kv(img, 0, k, v, [0, n], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, [0])
    q = syn.queries(wl, 0, 1)
    gc = H.make_gpu_cache(geom, 32, ppr)
    try:
        gc.upload(img)
        a = H.run_decode(gc, 0, q, "bf16", bt, [n], [0], fx, max_seq=n)
        b = H.run_decode(gc, 0, q, "bf16", bt, [n], [0], fx, max_seq=ppr * 64)
        rms = np.sqrt(np.mean(a ** 2))
        # each split keeps its own softmax reference, so the bf16 hi/lo split of p*scale rounds
        # differently (~2^-16 relative per weight); a merging bug would show at O(1)
        assert np.abs(a - b).max() / rms < 2e-4
    finally:
        gc.close()


def test_bad_page_sets_status_without_fault(osc):
    wl = syn.Workload("bad", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=6)
    fx = H.fixture(wl)
    geom = H.geometry(wl.shape, 8, 1)
    gc = H.make_gpu_cache(geom, 32, 8)
    try:
        bt = np.array([[0, 1, 2, 99, 4, 5, 6, 7]], np.int32)   # page 99 does not exist
        import torch
        ws_bytes = osc.oscar_decode_workspace_size(gc.cfg, 1, 500)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        out = torch.empty((1, 32, 128), dtype=torch.float32, device="cuda")
        q = H.dev_input(syn.queries(wl, 0, 1), "bf16")
        with pytest.raises(osc.OscarError):   # no clip threshold declared for the layer yet
            osc.oscar_decode_attn(gc.ctx, 0, q, osc.DTYPE_BF16, out, osc.DTYPE_F32, H.dev(bt), 8,
                                  H.dev(np.array([500], np.int32)), H.dev(np.zeros(1, np.int32)), 1, 500, 4, 128,
                                  H.dev(fx["R_K"]), H.dev(fx["R_V"]), ws, ws_bytes)
        osc.oscar_set_layer_clip(gc.ctx, 0, fx["clip_K"], fx["clip_V"])
        osc.oscar_decode_attn(gc.ctx, 0, q, osc.DTYPE_BF16, out, osc.DTYPE_F32, H.dev(bt), 8,
                              H.dev(np.array([500], np.int32)), H.dev(np.zeros(1, np.int32)), 1, 500, 4, 128,
                              H.dev(fx["R_K"]), H.dev(fx["R_V"]), ws, ws_bytes)
        bits = osc.oscar_check_status(gc.ctx)
        assert bits & osc.DEV_BAD_PAGE
        assert osc.oscar_check_status(gc.ctx) == 0    # cleared after reading
        # a sequence length beyond max_seq is flagged, not read
        osc.oscar_decode_attn(gc.ctx, 0, q, osc.DTYPE_BF16, out, osc.DTYPE_F32, H.dev(bt), 8,
                              H.dev(np.array([600], np.int32)), H.dev(np.zeros(1, np.int32)), 1, 500, 4, 128,
                              H.dev(fx["R_K"]), H.dev(fx["R_V"]), ws, ws_bytes)
        assert osc.oscar_check_status(gc.ctx) & osc.DEV_BAD_LEN
        with pytest.raises(osc.OscarError):   # sink/recent must match the cache
            osc.oscar_decode_attn(gc.ctx, 0, q, osc.DTYPE_BF16, out, osc.DTYPE_F32, H.dev(bt), 8,
                                  H.dev(np.array([500], np.int32)), H.dev(np.zeros(1, np.int32)), 1, 500, 4, 64,
                                  H.dev(fx["R_K"]), H.dev(fx["R_V"]), ws, ws_bytes)
    finally:
        gc.close()


# ---------------------------------------------------------------------------------------------- prefix fork
def test_fork_prefix_then_diverge(osc):
    wl = syn.Workload("fork", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=7)
    fx = H.fixture(wl)
    n_pre, n = 1000, 1700
    ppr = 30
    geom = H.geometry(wl.shape, 80, 2)
    gc = H.make_gpu_cache(geom, 32, ppr)
    img = cache.CacheImage(geom)
    try:
        ids = osc.oscar_alloc_pages(gc.ctx, syn.pages_for(n, 64))
        bt0 = np.full(ppr, -1, np.int32)
        bt0[:len(ids)] = ids
        k, v = syn.kv_tokens(wl, 0, n)
        k2, v2 = syn.kv_tokens(wl, 0, n, sub=1)
        args = (H.dev(fx["R_K"]), H.dev(fx["R_V"]), fx["clip_K"], fx["clip_V"])
        osc.oscar_write_kv(gc.ctx, 0, H.dev_input(k[:n_pre], "bf16"), H.dev_input(v[:n_pre], "bf16"), osc.DTYPE_BF16,
                           H.dev(np.array([0, n_pre], np.int32)), H.dev(np.zeros(1, np.int32)), 1, n_pre, *args,
                           H.dev(bt0[None]), ppr, H.dev(np.array([0], np.int32)))
        import torch
        torch.cuda.synchronize()
        bt1 = np.array(osc.oscar_fork_prefix(gc.ctx, bt0, n_pre, 0, 1, ppr, stream=None), np.int32)
        need = syn.pages_for(n, 64)
        have = int((bt1 >= 0).sum())
        bt1[have:need] = osc.oscar_alloc_pages(gc.ctx, need - have)
        bt = np.stack([bt0, bt1])
        for i, (kk, vv) in enumerate(((k, v), (k2, v2))):
            osc.oscar_write_kv(gc.ctx, 0, H.dev_input(kk[n_pre:], "bf16"), H.dev_input(vv[n_pre:], "bf16"),
                               osc.DTYPE_BF16, H.dev(np.array([0, n - n_pre], np.int32)),
                               H.dev(np.array([n_pre], np.int32)), 1, n - n_pre, *args, H.dev(bt[i:i + 1]), ppr,
                               H.dev(np.array([i], np.int32)))
        assert osc.oscar_check_status(gc.ctx) == 0
        # oracle: both requests written from scratch (request 1 = shared prefix + its own suffix)
        k2[:n_pre], v2[:n_pre] = k[:n_pre], v[:n_pre]
        bt_o = np.stack([np.arange(ppr), ppr + np.arange(ppr)]).astype(np.int32)
        geom2 = H.geometry(wl.shape, 2 * ppr, 2)
        img = cache.CacheImage(geom2)
        for i, (kk, vv) in enumerate(((k, v), (k2, v2))):
            cache.write_kv(img, 0, kk, vv, [0, n], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"],
                           bt_o[i:i + 1], [i])
        q = syn.queries(wl, 0, 2)
        want = attention.decode(img, 0, q, bt_o, [n, n], [0, 1], fx["R_K"], fx["R_V"])
        got = H.run_decode(gc, 0, q, "bf16", bt, [n, n], [0, 1], fx)
        H.assert_decode_close(got, want)
    finally:
        gc.close()


# ---------------------------------------------------------------------------------------------- BF16 comparison kernel
@pytest.mark.parametrize("hq,lens", [(32, [3000]), (64, [700, 64, 1, 1500])])
def test_bf16_paged_decode_parity(osc, hq, lens):
    import torch
    rng = np.random.default_rng(11)
    hkv, d, p = 8, 128, 64
    b = len(lens)
    ppr = max(syn.pages_for(n, p) for n in lens)
    num_pages = b * ppr + 3
    wl = syn.Workload("bf", syn.Shape(hq, hkv, d, p, 32, 4, 128, 1), [0], seed=12)
    pool = np.zeros((1, num_pages, hkv, 2, p, d), np.uint16)
    bt = (3 + rng.permutation(b * ppr)).astype(np.int32).reshape(b, ppr)
    for i, n in enumerate(lens):
        k, v = syn.kv_tokens(wl, 0, n, sub=i)
        t = np.arange(n)
        pool[0, bt[i, t // p], :, 0, t % p] = syn.to_bf16_bits(k)
        pool[0, bt[i, t // p], :, 1, t % p] = syn.to_bf16_bits(v)
    q = syn.queries(wl, 0, b)
    want = attention.bf16_paged_decode(pool, 0, q, bt, lens, p)
    geom = H.geometry(wl.shape, num_pages, b)
    gc = H.make_gpu_cache(geom, hq, ppr)
    try:
        ws_bytes = osc.oscar_bf16_decode_workspace_size(gc.cfg, b, max(lens))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        out = torch.empty((b, hq, d), dtype=torch.float32, device="cuda")
        pool_d = torch.from_numpy(pool.reshape(-1).view(np.int16)).cuda()
        osc.oscar_bf16_decode_attn(gc.ctx, 0, pool_d, H.dev_input(q, "bf16"), osc.DTYPE_BF16, out, osc.DTYPE_F32,
                                   H.dev(bt), ppr, H.dev(np.asarray(lens, np.int32)), b, max(lens), ws, ws_bytes)
        assert osc.oscar_check_status(gc.ctx) == 0
        H.assert_decode_close(out.cpu().numpy().astype(np.float64), want)
    finally:
        gc.close()


def test_read_pages_copies_the_blocks(osc):
    """oscar_read_pages returns exactly the pool's blocks of the requested pages (any order), and rejects
    page ids out of range."""
    wl = syn.Workload("rp", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=3)
    fx = H.fixture(wl)
    bt = _contiguous_bt(1, 12)
    gc, img, diag, _, _ = _prefill_both(osc, wl, fx, [600], bt, 12)
    try:
        ids = [5, 0, 3]
        got = osc.oscar_read_pages(gc.ctx, gc.cfg, 0, ids)
        assert np.array_equal(got, gc.pool_np()[0, ids])
        with pytest.raises(osc.OscarError):
            osc.oscar_read_pages(gc.ctx, gc.cfg, 0, [12])
    finally:
        gc.close()


def test_bounded_wait_timeout_sets_status_and_context_stays_usable(osc):
    """The failure path without a GPU fault: a wait on a barrier that nothing arrives on runs out after
    20 ms and sets OSCAR_DEV_TIMEOUT; reading the status clears it, and the context then writes and
    decodes correctly."""
    wl = syn.tiny()
    fx = H.fixture(wl)
    bt = _contiguous_bt(1, 40)
    s = wl.shape
    geom = H.geometry(s, 40, 1)
    gc = H.make_gpu_cache(geom, s.n_q_heads, 40)
    try:
        osc.oscar_selftest_wait_timeout(gc.ctx, 20000)
        assert osc.oscar_check_status(gc.ctx) & osc.DEV_TIMEOUT
        assert osc.oscar_check_status(gc.ctx) == 0
    finally:
        gc.close()
    gc, img, diag, _, _ = _prefill_both(osc, wl, fx, [512], bt, 40)
    try:
        H.compare_history(gc.pool_np(), img.g, 0, diag)
        q = syn.queries(wl, 0, 1)
        got = H.run_decode(gc, 0, q, "f32", bt, [512], [0], fx)
        gimg = cache.CacheImage(img.g)
        gimg.pool, gimg.slab = gc.pool_np(), gc.slab_np()
        H.assert_decode_close(got, attention.decode(gimg, 0, q, bt, [512], [0], fx["R_K"], fx["R_V"]))
    finally:
        gc.close()
