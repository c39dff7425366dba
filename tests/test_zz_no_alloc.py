"""The allocation-free decode entry point against the regular one.

oscar_decode_attn_noalloc exists for callers that cannot allocate device
memory (an engine whose allocator owns every byte, a plugin that must not call
cudaMalloc because it can synchronise the device, a serving loop that may not
allocate after start-up).  It keeps its scratch in a file-scope device array
inside the library instead of a caller workspace.  This file is collected last
so that a run stopping at the first failure has already run every other test;
it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import cache
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


def test_noalloc_decode_matches_workspace_decode_twice(osc):
    import torch
    wl = syn.Workload("noalloc", syn.Shape(32, 8, 128, 64, 32, 4, 128, 1), [0], seed=13)
    fx = H.fixture(wl)
    lens = [3000, 700]
    b = len(lens)
    ppr = max(syn.pages_for(n, 64) for n in lens) + 1
    bt = np.arange(b * ppr, dtype=np.int32).reshape(b, ppr)
    geom = H.geometry(wl.shape, b * ppr, b)
    img = cache.CacheImage(geom, fill=0xFF)
    for i, n in enumerate(lens):
        k, v = syn.kv_tokens(wl, 0, n, sub=i)
        cache.write_kv(img, 0, k, v, [0, n], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt[i:i + 1], [i])
    gc = H.make_gpu_cache(geom, 32, ppr)
    try:
        gc.upload(img)
        osc.oscar_set_layer_clip(gc.ctx, 0, fx["clip_K"], fx["clip_V"])
        max_seq = max(lens)
        args_common = dict(bt=H.dev(bt), lens=H.dev(np.asarray(lens, np.int32)), slots=H.dev(np.arange(b, dtype=np.int32)),
                           rk=H.dev(fx["R_K"]), rv=H.dev(fx["R_V"]))
        qs = [syn.queries(wl, 0, b), syn.queries(wl, 0, b, scale=0.25)]
        # reference: the regular entry point with a caller workspace
        ws_bytes = osc.oscar_decode_workspace_size(gc.cfg, b, max_seq)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        want = []
        for q in qs:
            out = torch.empty((b, 32, 128), dtype=torch.float32, device="cuda")
            osc.oscar_decode_attn(gc.ctx, 0, H.dev_input(q, "bf16"), osc.DTYPE_BF16, out, osc.DTYPE_F32,
                                  args_common["bt"], ppr, args_common["lens"], args_common["slots"], b, max_seq, 4, 128,
                                  args_common["rk"], args_common["rv"], ws, ws_bytes)
            want.append(out.cpu().numpy().astype(np.float64))
        # two calls in a row through the allocation-free entry point
        for q, w in zip(qs, want):
            out = torch.full((b, 32, 128), float("nan"), dtype=torch.float32, device="cuda")
            osc.oscar_decode_attn_noalloc(gc.ctx, 0, H.dev_input(q, "bf16"), osc.DTYPE_BF16, out, osc.DTYPE_F32,
                                          args_common["bt"], ppr, args_common["lens"], args_common["slots"], b,
                                          max_seq, 4, 128, args_common["rk"], args_common["rv"])
            assert osc.oscar_check_status(gc.ctx) == 0
            H.assert_decode_close(out.cpu().numpy().astype(np.float64), w)
        # sizes beyond the fixed scratch are rejected before any launch
        big = torch.empty((512, 32, 128), dtype=torch.float32, device="cuda")
        with pytest.raises(osc.OscarError) as ei:
            osc.oscar_decode_attn_noalloc(gc.ctx, 0, big, osc.DTYPE_F32, big, osc.DTYPE_F32, args_common["bt"], ppr,
                                          args_common["lens"], args_common["slots"], 512, ppr * 64, 4, 128,
                                          args_common["rk"], args_common["rv"])
        assert ei.value.status == osc.ERR_INVALID and "scratch" in str(ei.value)
    finally:
        gc.close()
