"""The one-launch decode form on the GPU.

In the one-launch form (oscar_set_decode_form ONE_LAUNCH) a decode is a single kernel:
the split CTAs form the rotated query themselves and the last CTA of each (request, kv
head) to finish merges that pair's partials and applies R_V^T (fused decode kernel of the
arXiv abstract; summary section 2.2 B: query rotated once, R_V^T once per output row).
The CTAs meet through per-(request, kv head) counters owned by the context, which each
launch must leave at zero.  These tests check which form runs, that both forms match the
oracle and each other on the same inputs, across many back-to-back launches with changing
grids and lengths (a counter left off zero would merge too early or never), inside a CUDA
graph, and after a launch that flagged a bad page.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import attention, cache
from tests import harness as H

pytestmark = pytest.mark.gpu

SHAPE = syn.Shape(32, 8, 128, 64, 32, 4, 128, 1)


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


def _image(wl, lens, ppr, shuffle=True):
    fx = H.fixture(wl)
    b = len(lens)
    order = syn.page_permutation(wl.seed, b * ppr, shuffle=shuffle)
    bt = order.reshape(b, ppr).astype(np.int32)
    geom = H.geometry(wl.shape, b * ppr, b)
    img = cache.CacheImage(geom)
    for i, n in enumerate(lens):
        k, v = syn.kv_tokens(wl, 0, n, sub=i)
        cache.write_kv(img, 0, k, v, [0, n], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt[i:i + 1], [i])
    return fx, bt, geom, img


class _Decoder:
    """Device-resident arguments of repeated decode calls on one cache."""

    def __init__(self, osc, gc, fx, bt, batch, max_seq):
        import torch
        self.osc, self.gc, self.batch, self.max_seq = osc, gc, batch, max_seq
        self.ws_bytes = osc.oscar_decode_workspace_size(gc.cfg, batch, max_seq)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.bt = H.dev(bt)
        self.ppr = bt.shape[1]
        self.rk, self.rv = H.dev(fx["R_K"]), H.dev(fx["R_V"])
        self.slots = H.dev(np.arange(batch, dtype=np.int32))
        osc.oscar_set_layer_clip(gc.ctx, 0, fx["clip_K"], fx["clip_V"])
        osc.oscar_set_decode_form(gc.ctx, osc.DECODE_ONE_LAUNCH)

    def __call__(self, q_dev, lens_dev, out):
        g = self.gc.geom
        self.osc.oscar_decode_attn(self.gc.ctx, 0, q_dev, self.osc.DTYPE_BF16, out, self.osc.DTYPE_F32, self.bt,
                                   self.ppr, lens_dev, self.slots, self.batch, self.max_seq, g.sink, g.recent,
                                   self.rk, self.rv, self.ws, self.ws_bytes)


@pytest.mark.parametrize("batch", [1, 4, 8])
def test_both_forms_match_the_oracle_and_each_other(osc, batch):
    """Each form launches what it says (one kernel, or q_rotate + split-K + combine; the
    automatic form is one of the two), both match the oracle, and they agree with each other
    to the rounding of the rotated query's summation order."""
    import torch
    wl = syn.Workload("lc", SHAPE, [0], seed=41)
    lens = [900 + 37 * i for i in range(batch)]
    fx, bt, geom, img = _image(wl, lens, syn.pages_for(max(lens), SHAPE.page_size) + 1)
    gc = H.make_gpu_cache(geom, SHAPE.n_q_heads, bt.shape[1])
    try:
        gc.upload(img)
        dec = _Decoder(osc, gc, fx, bt, batch, max(lens))
        q = syn.queries(wl, 0, batch)
        want = attention.decode(img, 0, syn.as_input(q, "bf16"), bt, lens, np.arange(batch), fx["R_K"], fx["R_V"])
        got = {}
        for form, launches in ((osc.DECODE_ONE_LAUNCH, (1,)), (osc.DECODE_THREE_KERNELS, (3,)),
                               (osc.DECODE_AUTO, (1, 3))):
            osc.oscar_set_decode_form(gc.ctx, form)
            out = torch.empty((batch, 32, 128), dtype=torch.float32, device="cuda")
            c0 = osc.oscar_launch_count(gc.ctx)
            dec(H.dev_input(q, "bf16"), H.dev(np.asarray(lens, np.int32)), out)
            assert osc.oscar_launch_count(gc.ctx) - c0 in launches, form
            assert osc.oscar_check_status(gc.ctx) == 0
            got[form] = out.cpu().numpy().astype(np.float64)
            H.assert_decode_close(got[form], want)
        # the forms sum q' = q R_K in different orders (float32, ~1e-7 relative); through scores of
        # keys with outlier channels (|k| ~ 100) that moves outputs by a few 1e-4 of their RMS at most,
        # where a merging mistake would show at O(1)
        a, b = got[osc.DECODE_ONE_LAUNCH], got[osc.DECODE_THREE_KERNELS]
        assert np.abs(a - b).max() / np.sqrt(np.mean(b ** 2)) < 1e-3
        with pytest.raises(osc.OscarError):
            osc.oscar_set_decode_form(gc.ctx, 7)
    finally:
        gc.close()


def test_back_to_back_launches_with_changing_grids(osc):
    """24 one-launch decodes on one context, each with its own lengths and max_seq (so its own
    grid and partial count), queued without synchronising; every output matches the oracle."""
    import torch
    wl = syn.Workload("b2b", SHAPE, [0], seed=42)
    lens_full = [7000, 2600]
    ppr = syn.pages_for(max(lens_full), SHAPE.page_size) + 1
    fx, bt, geom, img = _image(wl, lens_full, ppr)
    gc = H.make_gpu_cache(geom, SHAPE.n_q_heads, ppr)
    rng = np.random.default_rng(7)
    try:
        gc.upload(img)
        cases = []
        for i in range(24):
            lens = [int(rng.integers(1, lens_full[0] + 1)), int(rng.integers(1, lens_full[1] + 1))]
            max_seq = int(rng.choice([max(lens), lens_full[0], ppr * SHAPE.page_size]))
            q = syn.queries(wl, 0, 2, sub=100 + i)
            dec = _Decoder(osc, gc, fx, bt, 2, max_seq)
            out = torch.empty((2, 32, 128), dtype=torch.float32, device="cuda")
            dec(H.dev_input(q, "bf16"), H.dev(np.asarray(lens, np.int32)), out)
            cases.append((lens, q, out, dec))
        assert osc.oscar_check_status(gc.ctx) == 0
        for lens, q, out, _ in cases:
            want = attention.decode(img, 0, syn.as_input(q, "bf16"), bt, lens, np.arange(2), fx["R_K"], fx["R_V"])
            H.assert_decode_close(out.cpu().numpy().astype(np.float64), want)
    finally:
        gc.close()


def test_graph_replays_are_bit_identical(osc):
    """A CUDA graph of 6 one-launch decodes replayed 5 times reproduces the eager outputs bit for bit."""
    import torch
    wl = syn.Workload("graph", SHAPE, [0], seed=43)
    lens = [5000]
    ppr = syn.pages_for(lens[0], SHAPE.page_size) + 1
    fx, bt, geom, img = _image(wl, lens, ppr)
    gc = H.make_gpu_cache(geom, SHAPE.n_q_heads, ppr)
    try:
        gc.upload(img)
        dec = _Decoder(osc, gc, fx, bt, 1, lens[0])
        qs = [H.dev_input(syn.queries(wl, 0, 1, sub=200 + i), "bf16") for i in range(6)]
        lens_d = H.dev(np.asarray(lens, np.int32))
        outs = [torch.empty((1, 32, 128), dtype=torch.float32, device="cuda") for _ in range(6)]

        def run():
            for q, o in zip(qs, outs):
                dec(q, lens_d, o)

        run()
        torch.cuda.synchronize()
        eager = [o.clone() for o in outs]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        for _ in range(5):
            for o in outs:
                o.zero_()
            g.replay()
            torch.cuda.synchronize()
            for e, o in zip(eager, outs):
                assert torch.equal(e, o)
        assert osc.oscar_check_status(gc.ctx) == 0
        want = attention.decode(img, 0, syn.as_input(syn.queries(wl, 0, 1, sub=200), "bf16"), bt, lens, [0],
                                fx["R_K"], fx["R_V"])
        H.assert_decode_close(eager[0].cpu().numpy().astype(np.float64), want)
    finally:
        gc.close()


def test_correct_after_a_flagged_launch(osc):
    """A launch that meets a bad page id flags it (no fault); the next launch on the context is right."""
    import torch
    wl = syn.Workload("flag", SHAPE, [0], seed=44)
    lens = [3000]
    ppr = syn.pages_for(lens[0], SHAPE.page_size) + 1
    fx, bt, geom, img = _image(wl, lens, ppr)
    gc = H.make_gpu_cache(geom, SHAPE.n_q_heads, ppr)
    try:
        gc.upload(img)
        bad = bt.copy()
        bad[0, 5] = geom.num_pages + 3
        q = syn.queries(wl, 0, 1)
        out = torch.empty((1, 32, 128), dtype=torch.float32, device="cuda")
        _Decoder(osc, gc, fx, bad, 1, lens[0])(H.dev_input(q, "bf16"), H.dev(np.asarray(lens, np.int32)), out)
        assert osc.oscar_check_status(gc.ctx) & osc.DEV_BAD_PAGE
        got = H.run_decode(gc, 0, q, "bf16", bt, lens, [0], fx)
        want = attention.decode(img, 0, syn.as_input(q, "bf16"), bt, lens, [0], fx["R_K"], fx["R_V"])
        H.assert_decode_close(got, want)
    finally:
        gc.close()
