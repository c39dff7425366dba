"""GB300-native OSCAR INT2 rotated paged KV cache: Python binding of liboscar.so.

The compute path is the CUDA library built from ``csrc/`` (see include/oscar.h
for the C ABI).  This module only marshals arguments: it exposes every C entry
point under the same name, raises :class:`OscarError` on a non-zero status, and
offers ``ptr()`` / ``stream_ptr()`` helpers for torch tensors and streams.
There is no fallback: importing the binding without a built library, or calling
a kernel entry point without a GPU, fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from . import calibrate  # noqa: F401  (offline calibration tooling)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboscar.so")

OK, ERR_INVALID, ERR_OOM, ERR_CUDA, ERR_DEVICE, ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5
DTYPE_F32, DTYPE_BF16 = 0, 1
DECODE_AUTO, DECODE_THREE_KERNELS, DECODE_ONE_LAUNCH = 0, 1, 2
DEV_BAD_PAGE, DEV_TIMEOUT, DEV_BAD_LEN, DEV_BAD_SLOT = 1, 2, 4, 8


class OscarError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"oscar status {status}: {message}")
        self.status = status


class oscar_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "n_q_heads", "n_kv_heads", "head_dim", "page_size", "group_size", "sink", "recent",
        "max_requests", "max_pages_per_req", "num_pages", "rotation_per_kv_head")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def make_config(**kw) -> oscar_config:
    c = oscar_config()
    c.group_size = 32
    for k, v in kw.items():
        setattr(c, k, int(v))
    return c


_c_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_f32 = ctypes.c_float
_cfgp = ctypes.POINTER(oscar_config)

# name -> (restype, argtypes); every entry point declared in include/oscar.h
_SIGS = {
    "oscar_last_error": (ctypes.c_char_p, []),
    "oscar_version": (ctypes.c_char_p, []),
    "oscar_int2_pool_bytes": (ctypes.c_size_t, [_cfgp]),
    "oscar_window_slab_bytes": (ctypes.c_size_t, [_cfgp]),
    "oscar_page_block_bytes": (ctypes.c_size_t, [_cfgp]),
    "oscar_create": (_i32, [_cfgp, _vp, _vp, ctypes.POINTER(_vp)]),
    "oscar_destroy": (_i32, [_vp]),
    "oscar_alloc_pages": (_i32, [_vp, _i32, _c_i32p]),
    "oscar_ref_pages": (_i32, [_vp, _c_i32p, _i32]),
    "oscar_unref_pages": (_i32, [_vp, _c_i32p, _i32]),
    "oscar_page_refcount": (_i32, [_vp, _i32, _c_i32p]),
    "oscar_free_page_count": (_i32, [_vp, _c_i32p]),
    "oscar_pages_needed": (_i32, [_cfgp, _i32]),
    "oscar_read_pages": (_i32, [_vp, _i32, _c_i32p, _i32, _vp]),
    "oscar_fork_prefix": (_i32, [_vp, _c_i32p, _c_i32p, _i32, _i32, _i32, _vp]),
    "oscar_write_kv": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _f32, _f32, _vp, _i32,
                              _vp, _vp]),
    "oscar_write_kv_hadamard": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _f32, _f32, _vp, _i32,
                                       _vp, _vp]),
    "oscar_set_layer_clip": (_i32, [_vp, _i32, _f32, _f32]),
    "oscar_append_step": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _f32, _f32, _vp, _i32, _vp, _vp]),
    "oscar_decode_workspace_size": (_i32, [_cfgp, _i32, _i32, ctypes.POINTER(ctypes.c_size_t)]),
    "oscar_decode_attn": (_i32, [_vp, _i32, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                                 _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "oscar_decode_step": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _vp, _i32, _i32,
                                 _i32, _i32, _vp, _vp, _f32, _f32, _vp, ctypes.c_size_t, _vp]),
    "oscar_decode_attn_noalloc": (_i32, [_vp, _i32, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _vp, _i32, _i32, _i32,
                                         _i32, _vp, _vp, _vp]),
    "oscar_extend_workspace_size": (_i32, [_cfgp, _i32, ctypes.POINTER(ctypes.c_size_t)]),
    "oscar_extend_workspace_size_unpacked": (_i32, [_cfgp, _i32, _i32, _i32, _i32, ctypes.POINTER(ctypes.c_size_t)]),
    "oscar_extend_step": (_i32, [_vp, _i32, _vp, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _vp,
                                 _i32, _vp, _vp, _vp, _f32, _f32, _vp, ctypes.c_size_t, _vp]),
    "oscar_extend_attn": (_i32, [_vp, _i32, _vp, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _vp,
                                 _i32, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "oscar_bf16_decode_workspace_size": (_i32, [_cfgp, _i32, _i32, ctypes.POINTER(ctypes.c_size_t)]),
    "oscar_bf16_decode_attn": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _i32, _i32, _vp,
                                      ctypes.c_size_t, _vp]),
    "oscar_selftest_wait_timeout": (_i32, [_vp, _i32, _vp]),
    "oscar_check_status": (_i32, [_vp, _vp, _c_i32p]),
    "oscar_set_decode_form": (_i32, [_vp, _i32]),
    "oscar_set_timing": (_i32, [_vp, _i32]),
    "oscar_kernel_time": (_i32, [_vp, ctypes.c_char_p, ctypes.POINTER(ctypes.c_double), _c_i32p]),
    "oscar_reset_timing": (_i32, [_vp]),
    "oscar_launch_count": (ctypes.c_int64, [_vp]),
}

_lib: Optional[ctypes.CDLL] = None


def load() -> ctypes.CDLL:
    """Load liboscar.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OscarError(ERR_INVALID, f"{LIB_PATH} is not built; run __graft_entry__.build() or "
                                          "python int2_rotated_paged_oscar_gb300/build.py")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int) -> None:
    if status != OK:
        raise OscarError(status, load().oscar_last_error().decode())


def ptr(x) -> Optional[int]:
    """Device (or host) address of a torch tensor / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def stream_ptr(stream=None) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i32_array(seq: Sequence[int]):
    arr = (ctypes.c_int32 * len(seq))(*[int(v) for v in seq])
    return arr


# ------------------------------------------------------------------ thin wrappers (same names as the C ABI)
def oscar_version() -> str:
    return load().oscar_version().decode()


def oscar_int2_pool_bytes(cfg: oscar_config) -> int:
    return load().oscar_int2_pool_bytes(ctypes.byref(cfg))


def oscar_window_slab_bytes(cfg: oscar_config) -> int:
    return load().oscar_window_slab_bytes(ctypes.byref(cfg))


def oscar_page_block_bytes(cfg: oscar_config) -> int:
    return load().oscar_page_block_bytes(ctypes.byref(cfg))


def oscar_create(cfg: oscar_config, int2_pool=None, window_slab=None) -> int:
    out = ctypes.c_void_p()
    _check(load().oscar_create(ctypes.byref(cfg), ptr(int2_pool), ptr(window_slab), ctypes.byref(out)))
    return out.value


def oscar_destroy(ctx: int) -> None:
    _check(load().oscar_destroy(ctx))


def oscar_alloc_pages(ctx: int, n: int):
    arr = (ctypes.c_int32 * max(n, 1))()
    _check(load().oscar_alloc_pages(ctx, n, arr))
    return [arr[i] for i in range(n)]


def oscar_ref_pages(ctx: int, ids: Sequence[int]) -> None:
    _check(load().oscar_ref_pages(ctx, _i32_array(ids), len(ids)))


def oscar_unref_pages(ctx: int, ids: Sequence[int]) -> None:
    _check(load().oscar_unref_pages(ctx, _i32_array(ids), len(ids)))


def oscar_page_refcount(ctx: int, page: int) -> int:
    out = ctypes.c_int32()
    _check(load().oscar_page_refcount(ctx, page, ctypes.byref(out)))
    return out.value


def oscar_free_page_count(ctx: int) -> int:
    out = ctypes.c_int32()
    _check(load().oscar_free_page_count(ctx, ctypes.byref(out)))
    return out.value


def oscar_pages_needed(cfg: oscar_config, seq_len: int) -> int:
    return load().oscar_pages_needed(ctypes.byref(cfg), seq_len)


def oscar_read_pages(ctx: int, cfg: oscar_config, layer: int, ids: Sequence[int]):
    """The INT2 blocks of pages ``ids`` of ``layer`` as a host uint8 array [len(ids), n_kv_heads, block bytes]
    (``cfg`` is the context's configuration; it gives the array's shape)."""
    import numpy as np
    bb = oscar_page_block_bytes(cfg)
    out = np.empty((len(ids), cfg.n_kv_heads, bb), np.uint8)
    _check(load().oscar_read_pages(ctx, layer, _i32_array(list(ids)), len(ids), out.ctypes.data))
    return out


def oscar_fork_prefix(ctx: int, src_bt: Sequence[int], n: int, src_slot: int, dst_slot: int, max_pages: int,
                      stream=0):
    dst = (ctypes.c_int32 * max_pages)()
    src = _i32_array(list(src_bt) + [-1] * (max_pages - len(src_bt)))
    _check(load().oscar_fork_prefix(ctx, src, dst, n, src_slot, dst_slot, stream_ptr(stream) if stream != 0 else None))
    return [dst[i] for i in range(max_pages)]


def oscar_write_kv(ctx, layer, K, V, dtype, cu_seqlens, start_pos, batch, total_tokens, R_K, R_V, clip_K, clip_V,
                   block_table, bt_stride, req_slot, stream=None) -> None:
    _check(load().oscar_write_kv(ctx, layer, ptr(K), ptr(V), dtype, ptr(cu_seqlens), ptr(start_pos), batch,
                                 total_tokens, ptr(R_K), ptr(R_V), float(clip_K), float(clip_V), ptr(block_table),
                                 bt_stride, ptr(req_slot), stream_ptr(stream)))


def oscar_write_kv_hadamard(ctx, layer, K, V, dtype, cu_seqlens, start_pos, batch, total_tokens, clip_K, clip_V,
                            block_table, bt_stride, req_slot, stream=None) -> None:
    _check(load().oscar_write_kv_hadamard(ctx, layer, ptr(K), ptr(V), dtype, ptr(cu_seqlens), ptr(start_pos), batch,
                                          total_tokens, float(clip_K), float(clip_V), ptr(block_table), bt_stride,
                                          ptr(req_slot), stream_ptr(stream)))


def oscar_append_step(ctx, layer, K_new, V_new, dtype, seq_lens_before, batch, R_K, R_V, clip_K, clip_V,
                      block_table, bt_stride, req_slot, stream=None) -> None:
    _check(load().oscar_append_step(ctx, layer, ptr(K_new), ptr(V_new), dtype, ptr(seq_lens_before), batch,
                                    ptr(R_K), ptr(R_V), float(clip_K), float(clip_V), ptr(block_table), bt_stride,
                                    ptr(req_slot), stream_ptr(stream)))


def oscar_set_layer_clip(ctx, layer, clip_K, clip_V) -> None:
    _check(load().oscar_set_layer_clip(ctx, layer, float(clip_K), float(clip_V)))


def oscar_decode_workspace_size(cfg: oscar_config, batch: int, max_seq: int) -> int:
    out = ctypes.c_size_t()
    _check(load().oscar_decode_workspace_size(ctypes.byref(cfg), batch, max_seq, ctypes.byref(out)))
    return out.value


def oscar_bf16_decode_workspace_size(cfg: oscar_config, batch: int, max_seq: int) -> int:
    out = ctypes.c_size_t()
    _check(load().oscar_bf16_decode_workspace_size(ctypes.byref(cfg), batch, max_seq, ctypes.byref(out)))
    return out.value


def oscar_decode_attn(ctx, layer, q, q_dtype, out, out_dtype, block_table, bt_stride, seq_lens, req_slot, batch,
                      max_seq, sink, recent, R_K, R_V, workspace, ws_bytes, stream=None) -> None:
    _check(load().oscar_decode_attn(ctx, layer, ptr(q), q_dtype, ptr(out), out_dtype, ptr(block_table), bt_stride,
                                    ptr(seq_lens), ptr(req_slot), batch, max_seq, sink, recent, ptr(R_K), ptr(R_V),
                                    ptr(workspace), ws_bytes, stream_ptr(stream)))


def oscar_decode_step(ctx, layer, K_new, V_new, kv_dtype, q, q_dtype, out, out_dtype, block_table, bt_stride,
                      seq_lens, req_slot, batch, max_seq, sink, recent, R_K, R_V, clip_K, clip_V, workspace, ws_bytes,
                      stream=None) -> None:
    _check(load().oscar_decode_step(ctx, layer, ptr(K_new), ptr(V_new), kv_dtype, ptr(q), q_dtype, ptr(out),
                                    out_dtype, ptr(block_table), bt_stride, ptr(seq_lens), ptr(req_slot), batch,
                                    max_seq, sink, recent, ptr(R_K), ptr(R_V), float(clip_K), float(clip_V),
                                    ptr(workspace), ws_bytes, stream_ptr(stream)))


def oscar_decode_attn_noalloc(ctx, layer, q, q_dtype, out, out_dtype, block_table, bt_stride, seq_lens, req_slot,
                              batch, max_seq, sink, recent, R_K, R_V, stream=None) -> None:
    """oscar_decode_attn without a workspace: scratch is the library's own 8 MiB device array (see oscar.h)."""
    _check(load().oscar_decode_attn_noalloc(ctx, layer, ptr(q), q_dtype, ptr(out), out_dtype, ptr(block_table),
                                            bt_stride, ptr(seq_lens), ptr(req_slot), batch, max_seq, sink, recent,
                                            ptr(R_K), ptr(R_V), stream_ptr(stream)))


def oscar_extend_workspace_size(cfg: oscar_config, total_tokens: int) -> int:
    out = ctypes.c_size_t()
    _check(load().oscar_extend_workspace_size(ctypes.byref(cfg), total_tokens, ctypes.byref(out)))
    return out.value


def oscar_extend_workspace_size_unpacked(cfg: oscar_config, total_tokens: int, batch: int, max_prefix: int,
                                         max_chunk: int) -> int:
    out = ctypes.c_size_t()
    _check(load().oscar_extend_workspace_size_unpacked(ctypes.byref(cfg), total_tokens, batch, max_prefix, max_chunk,
                                                       ctypes.byref(out)))
    return out.value


def oscar_extend_attn(ctx, layer, q, q_dtype, K_new, V_new, kv_dtype, out, out_dtype, cu_seqlens, prefix_lens, batch,
                      total_tokens, max_chunk, block_table, bt_stride, req_slot, R_K, R_V, workspace, ws_bytes,
                      stream=None) -> None:
    _check(load().oscar_extend_attn(ctx, layer, ptr(q), q_dtype, ptr(K_new), ptr(V_new), kv_dtype, ptr(out),
                                    out_dtype, ptr(cu_seqlens), ptr(prefix_lens), batch, total_tokens, max_chunk,
                                    ptr(block_table), bt_stride, ptr(req_slot), ptr(R_K), ptr(R_V), ptr(workspace),
                                    ws_bytes, stream_ptr(stream)))


def oscar_extend_step(ctx, layer, q, q_dtype, K_new, V_new, kv_dtype, out, out_dtype, cu_seqlens, prefix_lens, batch,
                      total_tokens, max_chunk, block_table, bt_stride, req_slot, R_K, R_V, clip_K, clip_V, workspace,
                      ws_bytes, stream=None) -> None:
    _check(load().oscar_extend_step(ctx, layer, ptr(q), q_dtype, ptr(K_new), ptr(V_new), kv_dtype, ptr(out),
                                    out_dtype, ptr(cu_seqlens), ptr(prefix_lens), batch, total_tokens, max_chunk,
                                    ptr(block_table), bt_stride, ptr(req_slot), ptr(R_K), ptr(R_V), float(clip_K),
                                    float(clip_V), ptr(workspace), ws_bytes, stream_ptr(stream)))


def oscar_bf16_decode_attn(ctx, layer, bf16_pool, q, q_dtype, out, out_dtype, block_table, bt_stride, seq_lens,
                           batch, max_seq, workspace, ws_bytes, stream=None) -> None:
    _check(load().oscar_bf16_decode_attn(ctx, layer, ptr(bf16_pool), ptr(q), q_dtype, ptr(out), out_dtype,
                                         ptr(block_table), bt_stride, ptr(seq_lens), batch, max_seq, ptr(workspace),
                                         ws_bytes, stream_ptr(stream)))


def oscar_selftest_wait_timeout(ctx, limit_us: int, stream=None) -> None:
    _check(load().oscar_selftest_wait_timeout(ctx, int(limit_us), stream_ptr(stream)))


def oscar_check_status(ctx, stream=None) -> int:
    bits = ctypes.c_int32()
    st = load().oscar_check_status(ctx, stream_ptr(stream), ctypes.byref(bits))
    if st not in (OK, ERR_DEVICE):
        _check(st)
    return bits.value


def oscar_set_decode_form(ctx, form: int) -> None:
    _check(load().oscar_set_decode_form(ctx, int(form)))


def oscar_set_timing(ctx, enable: bool) -> None:
    _check(load().oscar_set_timing(ctx, 1 if enable else 0))


def oscar_kernel_time(ctx, name: str):
    ms = ctypes.c_double()
    n = ctypes.c_int32()
    _check(load().oscar_kernel_time(ctx, name.encode(), ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def oscar_reset_timing(ctx) -> None:
    _check(load().oscar_reset_timing(ctx))


def oscar_launch_count(ctx) -> int:
    return load().oscar_launch_count(ctx)
