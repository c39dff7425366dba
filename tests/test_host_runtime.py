"""Host runtime of liboscar.so on the CPU: symbol exports, validation, page allocator, fork, planning.

These tests call no kernel; they need the library built but no GPU.
"""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def osc():
    from int2_rotated_paged_oscar_gb300 import build
    build.build()
    import int2_rotated_paged_oscar_gb300 as m
    m.load()
    return m


def _cfg(osc, **kw):
    base = dict(num_layers=2, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=64, sink=4, recent=128,
                max_requests=4, max_pages_per_req=600, num_pages=64)
    base.update(kw)
    return osc.make_config(**base)


def test_every_header_symbol_is_exported(osc):
    header = open(os.path.join(ROOT, "include", "oscar.h")).read()
    decl = r"^\s*(?:oscar_status|size_t|int32_t|int64_t|const char\s*\*)\s*(oscar_[a-z0-9_]+)\s*\("
    names = set(re.findall(decl, header, flags=re.M))
    assert len(names) >= 25
    lib = osc.load()
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing
    assert set(osc._SIGS) == names, set(osc._SIGS) ^ names


def test_binding_argument_counts_match_the_header(osc):
    """Each ctypes signature has as many arguments as its C prototype (a dropped or extra argument in the
    binding would shift every later one)."""
    header = open(os.path.join(ROOT, "include", "oscar.h")).read()
    header = re.sub(r"/\*.*?\*/", "", header, flags=re.S)
    proto = r"^\s*(?:oscar_status|size_t|int32_t|int64_t|const char\s*\*)\s*(oscar_[a-z0-9_]+)\s*\(([^;]*?)\)\s*;"
    counts = {}
    for name, params in re.findall(proto, header, flags=re.M | re.S):
        params = params.strip()
        counts[name] = 0 if params in ("", "void") else params.count(",") + 1
    assert set(counts) == set(osc._SIGS)
    bad = {n: (counts[n], len(osc._SIGS[n][1])) for n in counts if counts[n] != len(osc._SIGS[n][1])}
    assert not bad, bad


def test_version_and_sizes(osc):
    assert "sm_103a" in osc.oscar_version()
    c = _cfg(osc)
    assert osc.oscar_page_block_bytes(c) == 6144
    assert osc.oscar_int2_pool_bytes(c) == 2 * 64 * 8 * 6144
    assert osc.oscar_window_slab_bytes(c) == 2 * 4 * 8 * 2 * 132 * 128 * 2
    tiny = _cfg(osc, head_dim=64, page_size=16, n_q_heads=4, n_kv_heads=2, recent=32, num_layers=1)
    assert osc.oscar_page_block_bytes(tiny) == 16 * 48


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=96), -5), (dict(page_size=8), -5), (dict(group_size=64), -5), (dict(n_q_heads=24), -5),
    (dict(n_q_heads=12, n_kv_heads=8), -5), (dict(recent=0), -1), (dict(num_pages=0), -1), (dict(sink=-1), -1),
])
def test_config_validation(osc, bad, code):
    c = _cfg(osc, **bad)
    with pytest.raises(osc.OscarError) as ei:
        osc.oscar_create(c)
    assert ei.value.status == code
    assert osc.oscar_int2_pool_bytes(c) == 0


def test_allocator_refcounts_and_exhaustion(osc):
    c = _cfg(osc, num_pages=8)
    ctx = osc.oscar_create(c)
    try:
        ids = osc.oscar_alloc_pages(ctx, 5)
        assert ids == [0, 1, 2, 3, 4]
        assert osc.oscar_free_page_count(ctx) == 3
        with pytest.raises(osc.OscarError) as ei:
            osc.oscar_alloc_pages(ctx, 4)
        assert ei.value.status == osc.ERR_OOM
        osc.oscar_ref_pages(ctx, [1, 1])
        assert osc.oscar_page_refcount(ctx, 1) == 3
        osc.oscar_unref_pages(ctx, [1, 1, 1, 2])
        assert osc.oscar_page_refcount(ctx, 1) == 0 and osc.oscar_free_page_count(ctx) == 5
        with pytest.raises(osc.OscarError):
            osc.oscar_unref_pages(ctx, [1])          # already free
        with pytest.raises(osc.OscarError):
            osc.oscar_ref_pages(ctx, [7])            # never allocated
        again = osc.oscar_alloc_pages(ctx, 2)
        assert set(again) <= {1, 2, 5, 6, 7}
    finally:
        osc.oscar_destroy(ctx)


def test_pages_needed(osc):
    c = _cfg(osc)
    assert osc.oscar_pages_needed(c, 100) == 0
    assert osc.oscar_pages_needed(c, 132) == 0
    assert osc.oscar_pages_needed(c, 133) == 1          # token 4 is history, page 0
    assert osc.oscar_pages_needed(c, 32768) == (32768 - 128 - 1) // 64 + 1


def test_fork_prefix_shares_full_pages_and_copies_partial(osc):
    c = _cfg(osc, num_pages=32, max_pages_per_req=16, page_size=16, head_dim=64, n_q_heads=4, n_kv_heads=2,
             recent=8)
    ctx = osc.oscar_create(c)
    try:
        src = osc.oscar_alloc_pages(ctx, 4)   # prefix of 64 tokens: history [4, 56) -> pages 0..2 full, 3 partial
        dst = osc.oscar_fork_prefix(ctx, src, 64, 0, 1, 16)
        assert dst[:3] == src[:3]
        assert dst[3] not in src and dst[3] >= 0
        assert all(x == -1 for x in dst[4:])
        for p in src[:3]:
            assert osc.oscar_page_refcount(ctx, p) == 2
        assert osc.oscar_page_refcount(ctx, src[3]) == 1
        assert osc.oscar_page_refcount(ctx, dst[3]) == 1
        # page-aligned history end: no copy, nothing allocated
        free_before = osc.oscar_free_page_count(ctx)
        dst2 = osc.oscar_fork_prefix(ctx, src, 8 + 48, 0, 2, 16)   # history [4, 48): 3 full pages
        assert dst2[:3] == src[:3] and dst2[3] == -1
        assert osc.oscar_free_page_count(ctx) == free_before
        with pytest.raises(osc.OscarError):
            osc.oscar_fork_prefix(ctx, src, 64, 1, 1, 16)          # same slot
    finally:
        osc.oscar_destroy(ctx)


def test_fault_injection_alloc_failure(osc):
    """OSCAR_FAULT_ALLOC_FAIL_AFTER makes the allocator fail after n pages (host-side fault injection)."""
    code = (
        "import int2_rotated_paged_oscar_gb300 as o\n"
        "c=o.make_config(num_layers=1,n_q_heads=8,n_kv_heads=8,head_dim=128,page_size=64,sink=4,recent=128,"
        "max_requests=1,max_pages_per_req=8,num_pages=32)\n"
        "x=o.oscar_create(c)\n"
        "o.oscar_alloc_pages(x,3)\n"
        "try:\n    o.oscar_alloc_pages(x,1)\nexcept o.OscarError as e:\n    print('OOM', e.status)\n")
    env = dict(os.environ, OSCAR_FAULT_ALLOC_FAIL_AFTER="3", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, cwd=ROOT)
    assert "OOM -2" in r.stdout, r.stdout + r.stderr


def test_kernel_calls_need_device_buffers(osc):
    c = _cfg(osc)
    ctx = osc.oscar_create(c)   # host-only context
    try:
        with pytest.raises(osc.OscarError) as ei:
            osc.oscar_append_step(ctx, 0, 1, 1, osc.DTYPE_BF16, 1, 1, 1, 1, 1.0, 1.0, 1, 1, 1, stream=0)
        assert ei.value.status == osc.ERR_INVALID
    finally:
        osc.oscar_destroy(ctx)


def test_layer_clip_declaration(osc):
    """Clip thresholds feed the f16 operand exponent of the decode MMAs: the range is validated on the host."""
    ctx = osc.oscar_create(_cfg(osc))   # host-only context: the declaration is host state
    try:
        osc.oscar_set_layer_clip(ctx, 0, 3.5, 120.0)
        osc.oscar_set_layer_clip(ctx, 1, 2.0 ** -80, 16383.0)
        for clip_k, clip_v, code in ((0.0, 1.0, osc.ERR_INVALID), (1.0, -2.0, osc.ERR_INVALID),
                                     (16384.0, 1.0, osc.ERR_UNSUPPORTED), (1.0, float("inf"), osc.ERR_INVALID),
                                     (2.0 ** -90, 1.0, osc.ERR_UNSUPPORTED)):
            with pytest.raises(osc.OscarError) as ei:
                osc.oscar_set_layer_clip(ctx, 0, clip_k, clip_v)
            assert ei.value.status == code, (clip_k, clip_v)
        with pytest.raises(osc.OscarError) as ei:
            osc.oscar_set_layer_clip(ctx, 2, 1.0, 1.0)   # layer out of range
        assert ei.value.status == osc.ERR_INVALID
    finally:
        osc.oscar_destroy(ctx)


def test_workspace_planning(osc):
    c = _cfg(osc, num_layers=1, num_pages=600)
    small = osc.oscar_decode_workspace_size(c, 1, 100)          # window only
    big = osc.oscar_decode_workspace_size(c, 1, 32768)
    batched = osc.oscar_decode_workspace_size(_cfg(osc, n_q_heads=64, num_pages=600), 64, 32768)
    assert 0 < small < big < batched
    assert osc.oscar_bf16_decode_workspace_size(c, 1, 32768) > 0


def test_extend_unpacked_workspace_planning(osc):
    """The unpacked-prefix extend workspace: the base size plus, per (request, kv head), one 43,008-byte
    operand image (d = 128) per 64 positions of INT2 history (sink 4, window 128), of the window slots
    and of the chunk (the attention grid's query tiles of 32 tokens at GQA 4, rounded up to 64 keys)."""
    c = _cfg(osc, num_layers=1, num_pages=600)
    tile = 128 * 64 * 2 + 64 * 128 + 128 * 64 * 2 + 16 * 128
    assert tile == 43008
    base = osc.oscar_extend_workspace_size(c, 2048)
    base256 = (base + 255) // 256 * 256

    def tiles(max_prefix, max_chunk):
        hist_end = max(4, max_prefix - 128)
        hist = (hist_end - 1) // 64 - 4 // 64 + 1 if hist_end > 4 else 0
        chunk = ((max_chunk + 31) // 32 * 32 + 63) // 64
        return hist + (4 + 128 + 63) // 64 + chunk

    for batch, max_prefix, max_chunk in [(1, 0, 1), (4, 32768, 2048), (3, 133, 65), (2, 132, 64), (8, 200, 0)]:
        got = osc.oscar_extend_workspace_size_unpacked(c, 2048, batch, max_prefix, max_chunk)
        assert got == base256 + batch * 8 * tiles(max_prefix, max_chunk) * tile, (batch, max_prefix, max_chunk)
    # 64 more history tokens: one more tile per (request, kv head)
    a = osc.oscar_extend_workspace_size_unpacked(c, 2048, 4, 32768, 2048)
    b = osc.oscar_extend_workspace_size_unpacked(c, 2048, 4, 32768 + 64, 2048)
    assert b - a == 4 * 8 * tile
    for bad in [(-1, 100, 64), (1, -1, 64), (1, 100, -1)]:
        with pytest.raises(osc.OscarError) as ei:
            osc.oscar_extend_workspace_size_unpacked(c, 2048, *bad)
        assert ei.value.status == osc.ERR_INVALID


def test_calibration_matches_oracle_fixture():
    """The product's offline calibration and the oracle fixture are independent code; they must agree."""
    import numpy as np
    import synthetic as syn
    from int2_rotated_paged_oscar_gb300 import calibrate
    from oracle import rotation
    wl = syn.batch1_32k()
    q = syn.queries(wl, 0, 128, calib=True)
    k, v = syn.kv_tokens(wl, 0, 128, calib=True)
    a = calibrate.calibrate_layer(q, k, v)
    b = rotation.layer_fixture(q, k, v)
    assert np.abs(a["R_K"].astype(np.float64) - b["R_K64"]).max() < 1e-6
    assert np.abs(a["R_V"].astype(np.float64) - b["R_V64"]).max() < 1e-6
    assert abs(a["clip_K"] - float(b["clip_K"])) <= 1e-6 * float(b["clip_K"])
    assert abs(a["clip_V"] - float(b["clip_V"])) <= 1e-6 * float(b["clip_V"])
    h = calibrate.calibrate_layer(q, k, v, hadamard_only=True)
    assert np.array_equal(h["R_K"], rotation.layer_fixture(q, k, v, u_identity=True)["R_K"])
