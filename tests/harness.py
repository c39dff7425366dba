"""Test helpers: drive the CUDA path through the C ABI and compare with the oracle.

Only tests import this module.  Oracle outputs may feed the CUDA path (for
example an oracle-built cache image uploaded for decode parity); nothing from
the CUDA path ever feeds the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import synthetic as syn
from oracle import attention, cache, quant, rotation

# decode tolerance on unit-scale outputs (errors divided by the RMS of the oracle output)
DECODE_MAX_ABS = 2e-3
DECODE_MEAN_ABS = 2e-4
# near-boundary rule for packed codes
BOUNDARY_REL = 1e-6
EXEMPT_FRACTION = 1e-4


def torch_mod():
    import torch
    return torch


def geometry(shape: syn.Shape, num_pages: int, max_requests: int, num_layers: int = 1) -> cache.Geometry:
    return cache.Geometry(num_layers, shape.n_kv_heads, shape.head_dim, shape.page_size, shape.group_size,
                          shape.sink, shape.recent, num_pages, max_requests)


def fixture(wl: syn.Workload, layer: int = 0, n_cal: int = 256, u_identity: bool = False) -> dict:
    q = syn.queries(wl, layer, n_cal, calib=True)
    k, v = syn.kv_tokens(wl, layer, n_cal, calib=True)
    return rotation.layer_fixture(q, k, v, u_identity=u_identity)


@dataclass
class GpuCache:
    """Device buffers + context for one cache geometry."""
    cfg: object
    ctx: int
    pool: object
    slab: object
    geom: cache.Geometry

    def close(self):
        import int2_rotated_paged_oscar_gb300 as osc
        osc.oscar_destroy(self.ctx)

    def pool_np(self) -> np.ndarray:
        g = self.geom
        return self.pool.cpu().numpy().reshape(g.num_layers, g.num_pages, g.n_kv_heads, g.block_bytes)

    def slab_np(self) -> np.ndarray:
        g = self.geom
        return self.slab.cpu().numpy().view(np.uint16).reshape(
            g.num_layers, g.max_requests, g.n_kv_heads, 2, g.window, g.head_dim)

    def upload(self, img: cache.CacheImage):
        torch = torch_mod()
        self.pool.copy_(torch.from_numpy(img.pool.reshape(-1)))
        self.slab.copy_(torch.from_numpy(img.slab.reshape(-1).view(np.int16)))


def make_gpu_cache(geom: cache.Geometry, n_q_heads: int, max_pages_per_req: int, fill: int = 0,
                   rotation_per_kv_head: int = 0) -> GpuCache:
    torch = torch_mod()
    import int2_rotated_paged_oscar_gb300 as osc
    cfg = osc.make_config(num_layers=geom.num_layers, n_q_heads=n_q_heads, n_kv_heads=geom.n_kv_heads,
                          head_dim=geom.head_dim, page_size=geom.page_size, group_size=geom.group_size,
                          sink=geom.sink, recent=geom.recent, max_requests=geom.max_requests,
                          max_pages_per_req=max_pages_per_req, num_pages=geom.num_pages,
                          rotation_per_kv_head=rotation_per_kv_head)
    nbytes = osc.oscar_int2_pool_bytes(cfg)
    assert nbytes == geom.num_layers * geom.num_pages * geom.n_kv_heads * geom.block_bytes
    pool = torch.full((nbytes,), fill, dtype=torch.uint8, device="cuda")
    slab = torch.zeros((osc.oscar_window_slab_bytes(cfg) // 2,), dtype=torch.int16, device="cuda")
    ctx = osc.oscar_create(cfg, pool, slab)
    return GpuCache(cfg, ctx, pool, slab, geom)


def dev(x, dtype=None):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def dev_input(x: np.ndarray, dtype: str):
    """Upload float32 input values in their storage type (bf16 bit patterns or float32)."""
    torch = torch_mod()
    if dtype == "bf16":
        bits = syn.to_bf16_bits(x)
        return torch.from_numpy(bits.view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def dtype_code(dtype: str) -> int:
    import int2_rotated_paged_oscar_gb300 as osc
    return osc.DTYPE_BF16 if dtype == "bf16" else osc.DTYPE_F32


# ------------------------------------------------------------------ write parity with the near-boundary rule
def _near_bf16_boundary(x: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """True where x lies within 1e-6 * max(|x|, ref) of a BF16 rounding boundary.

    ref is the magnitude x is computed from: a rotated value carries an absolute error set by the
    magnitude of the values, so a group minimum close to zero is judged on the scale of its group
    (the reference the per-element rule uses), and (max - min) / 3 on max(|max|, |min|), since a
    narrow group of large values (a clipped group) has a range that is a small difference of large
    numbers.
    """
    x = np.asarray(x, dtype=np.float64)
    w = BOUNDARY_REL * np.maximum(np.abs(x), np.asarray(ref, dtype=np.float64))
    return quant.bf16_round(x + w) != quant.bf16_round(x - w)


def _near_code_boundary(y: np.ndarray, scale: np.ndarray, zero: np.ndarray, group: int) -> np.ndarray:
    d = y.shape[-1]
    yg = y.reshape(y.shape[:-1] + (d // group, group))
    s = scale[..., None]
    z = zero[..., None]
    near = np.zeros(yg.shape, dtype=bool)
    for k in range(3):
        yb = z + (k + 0.5) * s
        near |= np.abs(yg - yb) <= BOUNDARY_REL * np.maximum(np.abs(yb), s)
    return near.reshape(y.shape)


def _exact_ties(y: np.ndarray, scale: np.ndarray, zero: np.ndarray, group: int) -> np.ndarray:
    """True where y sits exactly on a code boundary z + (k + 1/2) s (all three BF16-grid values, exact in fp64)."""
    d = y.shape[-1]
    yg = np.asarray(y, np.float64).reshape(y.shape[:-1] + (d // group, group))
    s = np.asarray(scale, np.float64)[..., None]
    z = np.asarray(zero, np.float64)[..., None]
    ties = np.zeros(yg.shape, dtype=bool)
    for k in range(3):
        ties |= (yg - z) == (k + 0.5) * s
    return ties.reshape(y.shape)


def compare_history(gpu_pool: np.ndarray, geom: cache.Geometry, layer: int, diag: dict,
                    exact_ties: bool = False, enforce_budget: bool = True) -> dict:
    """Check GPU history rows against the oracle write diagnostics; returns counts, raises on violation.

    Every element that is not bit-identical to the oracle is an exemption and is listed:
    * a code that differs where the group's scale and zero agree (kind "K" / "V"): allowed only within
      1e-6 relative of a decision boundary;
    * a scale or a zero that differs (kinds "K-scale", "K-zero", ...): allowed only when the pre-rounding
      value lies within 1e-6 relative of a BF16 rounding boundary; the group's codes must then equal a
      re-quantisation with the GPU's own scale and zero, and each of them that differs from the oracle's
      own code is listed too (kind "K-group-code", ...).
    The exemptions may make up at most 1e-4 of the codes compared (enforce_budget; callers that compare
    a case in several pieces check the budget over the whole case with check_budget).

    exact_ties: the rotated values are exact on both sides (R = I on BF16 inputs), so a value can sit
    exactly halfway between two codes; there both codes have the same error s/2, both are correct, and
    such elements are checked for that and not counted against the exemption budget.
    """
    if "k" not in diag:
        return {"elements": 0, "exempt": 0, "list": []}
    gimg = cache.CacheImage(geom)
    gimg.pool = gpu_pool
    ck, sk, zk, cv, sv, zv = gimg.read_history(layer, diag["pages"], diag["slots"])
    G = geom.group_size
    total, exempt_list = 0, []
    for name, qd, gc, gs, gz in (("K", diag["k"], ck, sk, zk), ("V", diag["v"], cv, sv, zv)):
        y = qd["y"]
        same_s, same_z = gs == qd["scale"], gz == qd["zero"]
        same_sz = same_s & same_z
        # the zero is rounded from the group minimum, the scale from (max - min) / 3: each is judged
        # relative to the magnitude of the values it is computed from (min; max and min)
        mag = np.maximum(np.abs(qd["mn"]), np.abs(qd["mn"] + 3.0 * qd["rng3"]))
        group_exempt = _near_bf16_boundary(qd["mn"], qd["rng3"]) | _near_bf16_boundary(qd["rng3"], mag)
        bad_groups = ~same_sz & ~group_exempt
        if bad_groups.any():
            lines = []
            for r, h, gi in np.argwhere(bad_groups)[:5]:
                mn, r3 = float(qd["mn"][r, h, gi]), float(qd["rng3"][r, h, gi])
                lines.append(f"(b {int(diag['b'][r])}, t {int(diag['t'][r])}, head {h}, group {gi}): "
                             f"min {mn!r} rng/3 {r3!r}; oracle s {float(qd['scale'][r, h, gi])!r} "
                             f"z {float(qd['zero'][r, h, gi])!r}; gpu s {float(gs[r, h, gi])!r} "
                             f"z {float(gz[r, h, gi])!r}; group y {qd['y'][r, h, gi * G:(gi + 1) * G].tolist()}")
            raise AssertionError(f"{name}: scale/zero differ outside the boundary rule: " + "; ".join(lines))
        # expected codes: oracle codes where (s, z) agree, else re-quantised with the GPU's own (s, z)
        in_same = np.repeat(same_sz, G, axis=-1)
        want = np.where(in_same, qd["codes"], quant.quantize_with(y, gs, gz, G))
        near = _near_code_boundary(y, gs, gz, G)
        diff = gc != want
        bad = diff & ~near
        if bad.any():
            idx = np.argwhere(bad)[:5]
            raise AssertionError(f"{name}: {int(bad.sum())} codes differ away from a rounding boundary, e.g. "
                                 f"{idx.tolist()}")
        total += gc.size
        if exact_ties:
            tie = _exact_ties(y, gs, gz, G) & diff
            if tie.any():
                sg = np.repeat(np.asarray(gs, np.float64), G, axis=-1)
                zg = np.repeat(np.asarray(gz, np.float64), G, axis=-1)
                err = np.abs(zg + gc.astype(np.float64) * sg - y)
                assert np.all(err[tie] == 0.5 * sg[tie]), f"{name}: a tie took a code that is not one of its two nearest"
            diff = diff & ~tie
        b_of, t_of = diag["b"], diag["t"]
        for i in np.argwhere(diff & in_same):
            exempt_list.append((name, int(b_of[i[0]]), int(t_of[i[0]]), int(i[1]), int(i[2])))
        for kind, mask in (("-scale", ~same_s), ("-zero", ~same_z)):
            for i in np.argwhere(mask):  # (row, head, group)
                exempt_list.append((name + kind, int(b_of[i[0]]), int(t_of[i[0]]), int(i[1]), int(i[2])))
        for i in np.argwhere((gc != qd["codes"]) & ~in_same):
            exempt_list.append((name + "-group-code", int(b_of[i[0]]), int(t_of[i[0]]), int(i[1]), int(i[2])))
    res = {"elements": total, "exempt": len(exempt_list), "list": exempt_list}
    if enforce_budget:
        check_budget(res)
    return res


def check_budget(res: dict) -> None:
    """At most 1e-4 of the compared codes may be exemptions (no slack)."""
    assert res["exempt"] <= EXEMPT_FRACTION * res["elements"], \
        f"too many exemptions: {res['exempt']} of {res['elements']} codes"


def merge_results(results) -> dict:
    out = {"elements": 0, "exempt": 0, "list": []}
    for r in results:
        out["elements"] += r["elements"]
        out["exempt"] += r["exempt"]
        out["list"] += r["list"]
    return out


def check_history_chunk(job) -> dict:
    """Worker of a spawned process pool: the oracle quantises one chunk of history rows of request b
    (tokens ts, input rows xk / xv [m, Hkv, d]) and compares them with the GPU's page blocks holding
    those rows (blocks [k, Hkv, block bytes], remap[m] = the row's block)."""
    geom_fields, fx, b, ts, xk, xv, blocks, remap = job
    g = cache.Geometry(*geom_fields)
    kq = cache.quantize_rows(xk, fx["R_K"], fx["clip_K"], g.group_size)
    vq = cache.quantize_rows(xv, fx["R_V"], fx["clip_V"], g.group_size)
    cg = cache.Geometry(1, g.n_kv_heads, g.head_dim, g.page_size, g.group_size, g.sink, g.recent, blocks.shape[0], 1)
    diag = {"b": np.full(ts.size, b, np.int64), "t": ts, "k": kq, "v": vq, "pages": remap,
            "slots": ts % g.page_size}
    return compare_history(blocks[None], cg, 0, diag, enforce_budget=False)


_ORACLE_POOL = None


def oracle_pool():
    """Process pool for oracle work (spawned, one BLAS thread per worker)."""
    global _ORACLE_POOL
    if _ORACLE_POOL is None:
        import concurrent.futures as cf
        import multiprocessing as mp
        import os
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"   # read by the workers' numpy at import
        n = max(1, min(16, len(os.sched_getaffinity(0))))
        _ORACLE_POOL = cf.ProcessPoolExecutor(n, mp_context=mp.get_context("spawn"))
    return _ORACLE_POOL


# exemption records of this test session: (case, elements, exemptions by kind); printed at the end
EXEMPTION_LOG = []


def record_exemptions(case: str, res: dict) -> None:
    """Log a case's exemption counts (shown in the pytest summary) and, when OSCAR_EXEMPTION_DIR is set,
    write every exemption (kind, request, token, kv head, channel or group) to <dir>/<case>.txt."""
    import collections
    import os
    kinds = collections.Counter(e[0] for e in res["list"])
    EXEMPTION_LOG.append((case, res["elements"], res["exempt"], dict(sorted(kinds.items()))))
    d = os.environ.get("OSCAR_EXEMPTION_DIR")
    if d:
        os.makedirs(d, exist_ok=True)
        with open(os.path.join(d, f"exemptions_{case}.txt"), "w") as f:
            f.write(f"# {case}: {res['exempt']} exemptions of {res['elements']} codes compared\n")
            f.write("# kind request token kv_head channel_or_group\n")
            for e in res["list"]:
                f.write(" ".join(str(v) for v in e) + "\n")


def compare_window(gpu_slab: np.ndarray, oracle_slab: np.ndarray, layer: int, slots):
    for s in slots:
        assert np.array_equal(gpu_slab[layer, s], oracle_slab[layer, s]), f"window slab of request slot {s} differs"


def decode_errors(got: np.ndarray, want: np.ndarray):
    rms = float(np.sqrt(np.mean(np.square(want))))
    e = np.abs(np.asarray(got, dtype=np.float64) - want) / max(rms, 1e-30)
    return float(e.max()), float(e.mean())


def assert_decode_close(got, want, max_abs=DECODE_MAX_ABS, mean_abs=DECODE_MEAN_ABS):
    assert np.all(np.isfinite(got)), "non-finite decode output"
    mx, mn = decode_errors(got, want)
    assert mx <= max_abs and mn <= mean_abs, f"decode error max {mx:.3e} (<= {max_abs}), mean {mn:.3e} (<= {mean_abs})"
    return mx, mn


def run_decode(gc: GpuCache, layer, q: np.ndarray, q_dtype: str, bt: np.ndarray, seq_lens, req_slot, fx,
               max_seq=None, out_bf16=False):
    torch = torch_mod()
    import int2_rotated_paged_oscar_gb300 as osc
    b = q.shape[0]
    max_seq = int(max(seq_lens)) if max_seq is None else max_seq
    ws_bytes = osc.oscar_decode_workspace_size(gc.cfg, b, max_seq)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    qd = dev_input(q, q_dtype)
    out = torch.empty((b, q.shape[1], q.shape[2]), dtype=torch.bfloat16 if out_bf16 else torch.float32, device="cuda")
    bt_d = dev(bt.astype(np.int32))
    # an uploaded image carries no write call: declare the layer's clip thresholds
    osc.oscar_set_layer_clip(gc.ctx, layer, fx["clip_K"], fx["clip_V"])
    osc.oscar_decode_attn(gc.ctx, layer, qd, dtype_code(q_dtype), out, osc.DTYPE_BF16 if out_bf16 else osc.DTYPE_F32,
                          bt_d, bt.shape[1], dev(np.asarray(seq_lens, np.int32)), dev(np.asarray(req_slot, np.int32)),
                          b, max_seq, gc.geom.sink, gc.geom.recent, dev(fx["R_K"]), dev(fx["R_V"]), ws, ws_bytes)
    status = osc.oscar_check_status(gc.ctx)
    assert status == 0, f"device status {status}"
    return out.float().cpu().numpy().astype(np.float64)


# ------------------------------------------------------------------ full-size cases: sampled checks
def sampled_history_diag(geom: cache.Geometry, bt: np.ndarray, samples, fx) -> dict:
    """Oracle write diagnostics (as cache.write_kv returns) for sampled history rows.

    samples: list of (b, t, k_row [Hkv, d], v_row [Hkv, d]) with the input values of token t of request b.
    """
    b = np.array([s[0] for s in samples], dtype=np.int64)
    t = np.array([s[1] for s in samples], dtype=np.int64)
    xk = np.stack([s[2] for s in samples]).astype(np.float64)
    xv = np.stack([s[3] for s in samples]).astype(np.float64)
    kq = cache.quantize_rows(xk, fx["R_K"], fx["clip_K"], geom.group_size)
    vq = cache.quantize_rows(xv, fx["R_V"], fx["clip_V"], geom.group_size)
    pages = bt[b, t // geom.page_size]
    return {"b": b, "t": t, "k": kq, "v": vq, "pages": pages, "slots": t % geom.page_size}


def gpu_pages(gc: GpuCache, layer: int, pages) -> np.ndarray:
    """Pool blocks [len(pages), Hkv, block] of one layer, gathered on the device."""
    torch = torch_mod()
    g = gc.geom
    view = gc.pool.view(g.num_layers, g.num_pages, g.n_kv_heads * g.block_bytes)[layer]
    idx = torch.as_tensor(np.asarray(pages, dtype=np.int64), device=view.device)
    return view.index_select(0, idx).cpu().numpy().reshape(len(pages), g.n_kv_heads, g.block_bytes)


def compact_request_image(gc: GpuCache, layer: int, bt_row, n: int, slot: int, heads=None):
    """An oracle CacheImage holding one request of the GPU cache (its pages renumbered 0..k-1, one
    request slot), optionally restricted to some kv heads.  Returns (image, block_table [1, k])."""
    g = gc.geom
    heads = list(range(g.n_kv_heads)) if heads is None else list(heads)
    k = cache_pages_for(n, g)
    pages = np.asarray(bt_row[:k], dtype=np.int64)
    geom = cache.Geometry(1, len(heads), g.head_dim, g.page_size, g.group_size, g.sink, g.recent, max(k, 1), 1)
    img = cache.CacheImage(geom)
    if k:
        img.pool[0] = gpu_pages(gc, layer, pages)[:, heads]
    torch = torch_mod()
    slab = gc.slab.view(g.num_layers, g.max_requests, g.n_kv_heads, 2, g.window, g.head_dim)[layer, slot]
    img.slab[0, 0] = slab[heads].cpu().numpy().view(np.uint16)
    return img, np.arange(max(k, 1), dtype=np.int32)[None]


def cache_pages_for(n: int, g: cache.Geometry) -> int:
    """Pages holding the history of a request of length n (absolute-position paging)."""
    h_end = max(g.sink, n - g.recent)
    return 0 if h_end <= g.sink else (h_end - 1) // g.page_size + 1


def run_extend(gc: GpuCache, layer, q: np.ndarray, q_dtype: str, k_new: np.ndarray, v_new: np.ndarray, cu, prefix,
               bt: np.ndarray, req_slot, fx, out_bf16=False, max_chunk=None, unpacked=False):
    """oscar_extend_attn on the GPU cache; k_new / v_new BF16-valued float arrays [T, Hkv, d].  unpacked: a
    workspace of the unpacked-prefix form (the prefix dequantised once by a pre-pass), sized for the longest
    prefix (True) or for prefixes of at most that many tokens (an int: longer ones unpack their own tiles)."""
    torch = torch_mod()
    import int2_rotated_paged_oscar_gb300 as osc
    cu = np.asarray(cu, np.int32)
    total = int(cu[-1])
    b = cu.size - 1
    max_chunk = int(np.diff(cu).max()) if max_chunk is None else max_chunk
    if unpacked is not False:   # True: sized for the longest prefix; an int: for prefixes up to that length
        cap = int(max(prefix)) if unpacked is True else int(unpacked)
        ws_bytes = osc.oscar_extend_workspace_size_unpacked(gc.cfg, total, b, cap, max_chunk)
    else:
        ws_bytes = osc.oscar_extend_workspace_size(gc.cfg, total)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty((total, q.shape[1], q.shape[2]), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                      device="cuda")
    osc.oscar_set_layer_clip(gc.ctx, layer, fx["clip_K"], fx["clip_V"])
    osc.oscar_extend_attn(gc.ctx, layer, dev_input(q, q_dtype), dtype_code(q_dtype), dev_input(k_new, "bf16"),
                          dev_input(v_new, "bf16"), osc.DTYPE_BF16, out, osc.DTYPE_BF16 if out_bf16 else osc.DTYPE_F32,
                          dev(cu), dev(np.asarray(prefix, np.int32)), b, total, max_chunk, dev(bt.astype(np.int32)),
                          bt.shape[1], dev(np.asarray(req_slot, np.int32)), dev(fx["R_K"]), dev(fx["R_V"]), ws,
                          ws_bytes)
    status = osc.oscar_check_status(gc.ctx)
    assert status == 0, f"device status {status}"
    return out.float().cpu().numpy().astype(np.float64)
