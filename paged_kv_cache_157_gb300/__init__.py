"""paged_kv_cache_157_gb300: paged KV-cache decode attention for GB300 (sm_103a).

Thin ctypes binding over ``libkvc.so`` (C ABI in ``include/kvc.h``). The
functions below only marshal arguments: tensors become device pointers and
sizes, the current torch stream becomes the ``cudaStream_t``. Every step of
the computation runs in the library's CUDA kernels; there is no Python or
CPU fallback, and a missing library raises ``KvcLibraryMissing``.

``raw()`` returns the loaded ``ctypes.CDLL`` for callers that want the C
functions directly.
"""

from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "KvcError", "KvcLibraryMissing", "raw", "lib_path", "symbols",
    "append", "append_latent", "decode_workspace_size", "decode_attention", "decode_attention_static",
    "decode_attention_window", "copy_blocks", "append_fp8", "decode_attention_fp8",
    "append_int8", "decode_attention_int8",
    "decode_mla_workspace_size", "decode_attention_mla", "set_option", "get_option",
    "get_error_flags", "BlockPool", "slots_from_tables",
    "F32", "F16", "BF16", "FLAG_BAD_BLOCK", "FLAG_BAD_LEN", "FLAG_BAD_SLOT", "FLAG_TIMEOUT", "FLAG_WORKSPACE",
    "new_decode_workspace",
    "OPT_CHECKED", "OPT_BLOCKS_PER_CTA", "OPT_MAX_CTAS", "OPT_GQA_ENGINE", "OPT_DYNAMIC_SHARE", "OPT_DYNAMIC_CHUNK",
    "OPT_WAIT_POLLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libkvc.so")

F32, F16, BF16 = 0, 1, 2
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_NO_BLOCKS, ERR_CUDA, ERR_OUT_OF_RANGE, ERR_WORKSPACE = range(7)
FLAG_BAD_BLOCK, FLAG_BAD_LEN, FLAG_BAD_SLOT, FLAG_TIMEOUT, FLAG_WORKSPACE = 0x1, 0x2, 0x4, 0x8, 0x10
OPT_CHECKED, OPT_BLOCKS_PER_CTA, OPT_MAX_CTAS, OPT_GQA_ENGINE, OPT_DYNAMIC_SHARE, OPT_DYNAMIC_CHUNK, OPT_WAIT_POLLS = \
    0, 1, 2, 3, 4, 5, 6

# Every exported symbol of include/kvc.h with (restype, argtypes).
_vp, _i32, _i64, _f32, _sz, _u32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, \
    ctypes.POINTER(ctypes.c_uint32)
_i64p, _szp, _i32p = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_int32)


class PoolStats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("free_blocks", ctypes.c_int64), ("unique_blocks", ctypes.c_int64),
                ("table_entries", ctypes.c_int64), ("useful_tokens", ctypes.c_int64), ("live_seqs", ctypes.c_int64),
                ("block_size", ctypes.c_int32)]


SIGNATURES = {
    "kvc_abi_version": (_i32, []),
    "kvc_status_string": (ctypes.c_char_p, [_i32]),
    "kvc_last_error_message": (ctypes.c_char_p, []),
    "kvc_set_option": (_i32, [_i32, _i64]),
    "kvc_get_option": (_i32, [_i32, _i64p]),
    "kvc_set_checked": (_i32, [_i32]),
    "kvc_get_error_flags": (_i32, [_vp, _u32p]),
    "kvc_append": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _vp]),
    "kvc_append_latent": (_i32, [_vp, _vp, _i64, _vp, _i64, _i32, _i32, _i32, _i32, _vp]),
    "kvc_decode_workspace_size": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _szp]),
    "kvc_decode_attention": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _f32, _i32, _i32, _i32, _i32, _i64, _i32,
                                    _vp, _i32, _vp, _sz, _vp]),
    "kvc_decode_attention_static": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _f32, _i32, _i32, _i32, _i32, _i64,
                                           _i32, _vp, _i32, _vp]),
    "kvc_decode_attention_window": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _f32, _i32, _i32, _i32, _i32, _i64,
                                           _i32, _i32, _vp, _i32, _vp, _sz, _vp]),
    "kvc_decode_attention_multi": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _f32, _i32, _i32, _i32, _i32,
                                          _i64, _i32, _vp, _i32, _vp, _sz, _vp]),
    "kvc_decode_shared_prefix_workspace_size": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _szp]),
    "kvc_decode_attention_shared_prefix": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _vp, _f32, _i32,
                                                  _i32, _i32, _i32, _i64, _i32, _vp, _i32, _vp, _sz, _vp]),
    "kvc_decode_mla_workspace_size": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _szp]),
    "kvc_decode_attention_mla": (_i32, [_vp, _vp, _vp, _i32, _vp, _i32, _f32, _i32, _i32, _i32, _i32, _i64, _i32, _vp,
                                        _i32, _vp, _sz, _vp]),
    "kvc_pool_create": (_i32, [_i64, _i32, ctypes.POINTER(_vp)]),
    "kvc_pool_destroy": (None, [_vp]),
    "kvc_seq_add": (_i32, [_vp, _i64p]),
    "kvc_seq_fork": (_i32, [_vp, _i64, _i64p]),
    "kvc_seq_reserve": (_i32, [_vp, _i64, _i64, _vp]),
    "kvc_seq_reserve_cow": (_i32, [_vp, _i64, _i64, _vp, _vp]),
    "kvc_seq_reserve_batch": (_i32, [_vp, _vp, _i32, _i64, _vp]),
    "kvc_copy_blocks": (_i32, [_vp, _i64, _i64, _vp, _i64, _vp]),
    "kvc_append_fp8": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _vp]),
    "kvc_decode_attention_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _f32, _i32, _i32, _i32, _i32,
                                        _i64, _vp, _i32, _vp, _sz, _vp]),
    "kvc_append_int8": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _vp]),
    "kvc_decode_attention_int8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _f32, _i32, _i32, _i32, _i32,
                                         _i64, _vp, _i32, _vp, _sz, _vp]),
    "kvc_seq_free": (_i32, [_vp, _i64]),
    "kvc_seq_length": (_i32, [_vp, _i64, _i64p]),
    "kvc_block_refcount": (_i32, [_vp, _i64, _i32p]),
    "kvc_build_block_tables": (_i32, [_vp, _vp, _i32, _vp, _i32, _vp]),
    "kvc_pool_get_stats": (_i32, [_vp, ctypes.POINTER(PoolStats)]),
    "kvc_slots_from_tables": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _i64, _vp]),
}


def symbols():
    return sorted(SIGNATURES)


class KvcError(RuntimeError):
    def __init__(self, status: int, call: str, message: str):
        super().__init__(f"{call}: status {status} ({message})")
        self.status = status


class KvcLibraryMissing(ImportError):
    pass


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return _LIB_PATH


def raw() -> ctypes.CDLL:
    """Loads libkvc.so (built by ``build_lib.build()``) and declares its symbols."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise KvcLibraryMissing(
                    f"{_LIB_PATH} is missing: build it with `python -m paged_kv_cache_157_gb300.build_lib` "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int, call: str):
    if status != OK:
        lib = raw()
        raise KvcError(status, call, lib.kvc_last_error_message().decode(errors="replace"))


# ------------------------------------------------------------------ tensors

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    m = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        torch = _torch()
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(getattr(stream, "cuda_stream", stream)))


def _require(t, name, dtype=None, contiguous=True, cuda=True):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


# ---------------------------------------------------------------- options

def set_option(opt: int, value: int):
    _check(raw().kvc_set_option(opt, int(value)), "kvc_set_option")


def get_option(opt: int) -> int:
    v = ctypes.c_int64()
    _check(raw().kvc_get_option(opt, ctypes.byref(v)), "kvc_get_option")
    return v.value


def get_error_flags(stream=None) -> int:
    f = ctypes.c_uint32()
    _check(raw().kvc_get_error_flags(_stream(stream), ctypes.byref(f)), "kvc_get_error_flags")
    return f.value


# ---------------------------------------------------------------- compute

def append(k, v, slot_mapping, k_cache, v_cache, stream=None):
    """kvc_append: k, v [T, Hkv, D]; slot_mapping int64 [T]; caches [num_blocks, Hkv, bs, D]."""
    torch = _torch()
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n)
    _require(slot_mapping, "slot_mapping", torch.int64)
    nb, hkv, bs, d = k_cache.shape
    _check(raw().kvc_append(_ptr(k), _ptr(v), _ptr(slot_mapping), slot_mapping.numel(), _ptr(k_cache), _ptr(v_cache),
                            nb, bs, hkv, d, _dtype_code(k_cache), _stream(stream)), "kvc_append")


def append_latent(c, slot_mapping, latent_cache, d_c, stream=None):
    """kvc_append_latent: c [T, d_c + d_r]; latent_cache [num_blocks, bs, d_c + d_r]."""
    torch = _torch()
    _require(c, "c")
    _require(latent_cache, "latent_cache")
    _require(slot_mapping, "slot_mapping", torch.int64)
    nb, bs, w = latent_cache.shape
    _check(raw().kvc_append_latent(_ptr(c), _ptr(slot_mapping), slot_mapping.numel(), _ptr(latent_cache), nb, bs,
                                   d_c, w - d_c, _dtype_code(latent_cache), _stream(stream)), "kvc_append_latent")


def decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq) -> int:
    n = ctypes.c_size_t()
    _check(raw().kvc_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                           ctypes.byref(n)), "kvc_decode_workspace_size")
    return n.value


def new_decode_workspace(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq, device="cuda"):
    """Zero-filled uint8 workspace of the size kvc_decode_workspace_size asks for."""
    torch = _torch()
    n = decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq)
    return torch.zeros(max(n, 1), dtype=torch.uint8, device=device)


def decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace=None, stream=None,
                     window=None):
    """kvc_decode_attention (or kvc_decode_attention_window when ``window`` is given). q/out [B, Hq, D];
    caches [num_blocks, Hkv, bs, D]; block_tables int32 [B, max_blocks]; context_lens int32 [B]; workspace:
    a zero-filled uint8 tensor (see new_decode_workspace) that later calls keep zeroed, or None; window:
    attend only the newest ``window`` rows of every sequence."""
    torch = _torch()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _require(t, n)
    _require(block_tables, "block_tables", torch.int32)
    _require(context_lens, "context_lens", torch.int32)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, hq, d) or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("shape mismatch")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        _require(workspace, "workspace")
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    if window is not None:
        _check(raw().kvc_decode_attention_window(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                                 block_tables.shape[1], _ptr(context_lens), B, float(scale), hq, hkv,
                                                 d, bs, nb, int(window), _dtype_code(k_cache), _ptr(out),
                                                 _dtype_code(out), ws_ptr, ws_bytes, _stream(stream)),
               "kvc_decode_attention_window")
        return
    _check(raw().kvc_decode_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                      block_tables.shape[1], _ptr(context_lens), B, float(scale), hq, hkv, d, bs, nb,
                                      _dtype_code(k_cache), _ptr(out), _dtype_code(out), ws_ptr, ws_bytes,
                                      _stream(stream)), "kvc_decode_attention")


def new_multi_workspace(batch, n_tokens, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                        device="cuda"):
    """Zero-filled workspace for decode_attention_multi (the decode size query with n_tokens * n_q_heads)."""
    return new_decode_workspace(batch, n_tokens * n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                device)


def decode_attention_multi(q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace=None,
                           stream=None):
    """kvc_decode_attention_multi: q/out [B, T, Hq, D], the T newest rows of every sequence are its new tokens
    (already appended; context_lens count them) and token t attends rows 0 .. n - T + t. Workspace: a
    zero-filled uint8 tensor from new_multi_workspace, or None."""
    torch = _torch()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _require(t, n)
    _require(block_tables, "block_tables", torch.int32)
    _require(context_lens, "context_lens", torch.int32)
    B, T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, T, hq, d) or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("shape mismatch")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        _require(workspace, "workspace")
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(raw().kvc_decode_attention_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                            block_tables.shape[1], _ptr(context_lens), B, T, float(scale), hq, hkv,
                                            d, bs, nb, _dtype_code(k_cache), _ptr(out), _dtype_code(out), ws_ptr,
                                            ws_bytes, _stream(stream)), "kvc_decode_attention_multi")


def shared_prefix_workspace(batch, group_size, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                            device="cuda"):
    """Zero-filled uint8 workspace of the size kvc_decode_shared_prefix_workspace_size asks for."""
    torch = _torch()
    n = ctypes.c_size_t()
    _check(raw().kvc_decode_shared_prefix_workspace_size(batch, group_size, n_q_heads, n_kv_heads, head_dim,
                                                         block_size, max_blocks_per_seq, ctypes.byref(n)),
           "kvc_decode_shared_prefix_workspace_size")
    return torch.zeros(max(n.value, 1), dtype=torch.uint8, device=device)


def decode_attention_shared_prefix(q, k_cache, v_cache, block_tables, context_lens, group_size, prefix_lens, scale,
                                   out, workspace, stream=None):
    """kvc_decode_attention_shared_prefix: q/out [B, Hq, D]; sequences [g*group_size, (g+1)*group_size) share
    their first prefix_lens[g] rows (int32 device tensor [B / group_size]); workspace from
    shared_prefix_workspace."""
    torch = _torch()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out"), (workspace, "workspace")):
        _require(t, n)
    _require(block_tables, "block_tables", torch.int32)
    _require(context_lens, "context_lens", torch.int32)
    _require(prefix_lens, "prefix_lens", torch.int32)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, hq, d) or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("shape mismatch")
    if prefix_lens.numel() * group_size != B:
        raise ValueError("prefix_lens must hold one entry per group of group_size sequences")
    _check(raw().kvc_decode_attention_shared_prefix(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                                    block_tables.shape[1], _ptr(context_lens), B, int(group_size),
                                                    _ptr(prefix_lens), float(scale), hq, hkv, d, bs, nb,
                                                    _dtype_code(k_cache), _ptr(out), _dtype_code(out),
                                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                                    _stream(stream)), "kvc_decode_attention_shared_prefix")


def decode_attention_static(q, k_cache, v_cache, block_tables, context_lens, scale, out, stream=None):
    """kvc_decode_attention_static: the same decode with the library's built-in scratch, for callers that
    cannot allocate device memory (see include/kvc.h). Calls that may overlap on the GPU must not be issued
    concurrently: they share one scratch array."""
    torch = _torch()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _require(t, n)
    _require(block_tables, "block_tables", torch.int32)
    _require(context_lens, "context_lens", torch.int32)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, hq, d) or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("shape mismatch")
    _check(raw().kvc_decode_attention_static(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                             block_tables.shape[1], _ptr(context_lens), B, float(scale), hq, hkv, d,
                                             bs, nb, _dtype_code(k_cache), _ptr(out), _dtype_code(out),
                                             _stream(stream)), "kvc_decode_attention_static")


def decode_mla_workspace_size(batch, n_q_heads, d_c, d_r, block_size, max_blocks_per_seq) -> int:
    n = ctypes.c_size_t()
    _check(raw().kvc_decode_mla_workspace_size(batch, n_q_heads, d_c, d_r, block_size, max_blocks_per_seq,
                                               ctypes.byref(n)), "kvc_decode_mla_workspace_size")
    return n.value


def decode_attention_mla(q_absorbed, latent_cache, block_tables, context_lens, scale, d_c, out, workspace=None,
                         stream=None):
    """kvc_decode_attention_mla. q_absorbed [B, H, d_c + d_r]; latent_cache [num_blocks, bs, d_c + d_r];
    out [B, H, d_c]."""
    torch = _torch()
    for t, n in ((q_absorbed, "q_absorbed"), (latent_cache, "latent_cache"), (out, "out")):
        _require(t, n)
    _require(block_tables, "block_tables", torch.int32)
    _require(context_lens, "context_lens", torch.int32)
    B, h, w = q_absorbed.shape
    nb, bs, w2 = latent_cache.shape
    if w2 != w or tuple(out.shape) != (B, h, d_c):
        raise ValueError("shape mismatch")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        _require(workspace, "workspace")
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(raw().kvc_decode_attention_mla(_ptr(q_absorbed), _ptr(latent_cache), _ptr(block_tables),
                                          block_tables.shape[1], _ptr(context_lens), B, float(scale), h, d_c, w - d_c,
                                          bs, nb, _dtype_code(latent_cache), _ptr(out), _dtype_code(out), ws_ptr,
                                          ws_bytes, _stream(stream)), "kvc_decode_attention_mla")


# ------------------------------------------------------------------ pool

class BlockPool:
    """Host-side refcounted block pool (kvc_pool_*). Not thread-safe."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = raw()
        h = ctypes.c_void_p()
        _check(self._lib.kvc_pool_create(num_blocks, block_size, ctypes.byref(h)), "kvc_pool_create")
        self._h = h
        self.block_size = block_size
        self.num_blocks = num_blocks

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.kvc_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self) -> int:
        s = ctypes.c_int64()
        _check(self._lib.kvc_seq_add(self._h, ctypes.byref(s)), "kvc_seq_add")
        return s.value

    def fork(self, parent: int) -> int:
        s = ctypes.c_int64()
        _check(self._lib.kvc_seq_fork(self._h, parent, ctypes.byref(s)), "kvc_seq_fork")
        return s.value

    def reserve(self, seq: int, n_new: int):
        buf = (ctypes.c_int64 * max(1, n_new))()
        _check(self._lib.kvc_seq_reserve(self._h, seq, n_new, buf), "kvc_seq_reserve")
        return list(buf[:n_new])

    def reserve_batch(self, seqs, n_new: int):
        """kvc_seq_reserve_batch: n_new slots for each of the distinct sequences `seqs`, all or nothing.
        Returns one list of slots per sequence."""
        n = len(seqs)
        ids = (ctypes.c_int64 * max(1, n))(*seqs)
        buf = (ctypes.c_int64 * max(1, n * n_new))()
        _check(self._lib.kvc_seq_reserve_batch(self._h, ids, n, n_new, buf), "kvc_seq_reserve_batch")
        return [list(buf[i * n_new:(i + 1) * n_new]) for i in range(n)]

    def reserve_cow(self, seq: int, n_new: int):
        """kvc_seq_reserve_cow: (slots, copy) with copy = (shared block, fresh block) or None."""
        buf = (ctypes.c_int64 * max(1, n_new))()
        pair = (ctypes.c_int64 * 2)()
        _check(self._lib.kvc_seq_reserve_cow(self._h, seq, n_new, buf, pair), "kvc_seq_reserve_cow")
        copy = None if pair[0] < 0 else (int(pair[0]), int(pair[1]))
        return [int(buf[i]) for i in range(n_new)], copy

    def free(self, seq: int):
        _check(self._lib.kvc_seq_free(self._h, seq), "kvc_seq_free")

    def length(self, seq: int) -> int:
        n = ctypes.c_int64()
        _check(self._lib.kvc_seq_length(self._h, seq, ctypes.byref(n)), "kvc_seq_length")
        return n.value

    def refcount(self, block: int) -> int:
        r = ctypes.c_int32()
        _check(self._lib.kvc_block_refcount(self._h, block, ctypes.byref(r)), "kvc_block_refcount")
        return r.value

    def tables(self, seqs, max_blocks: int):
        """Returns (rows: list of lists of int, lens: list of int)."""
        n = len(seqs)
        ids = (ctypes.c_int64 * max(1, n))(*seqs)
        tab = (ctypes.c_int32 * max(1, n * max_blocks))()
        lens = (ctypes.c_int32 * max(1, n))()
        _check(self._lib.kvc_build_block_tables(self._h, ids, n, tab, max_blocks, lens), "kvc_build_block_tables")
        rows = [list(tab[i * max_blocks:(i + 1) * max_blocks]) for i in range(n)]
        return rows, list(lens[:n])

    def stats(self) -> dict:
        st = PoolStats()
        _check(self._lib.kvc_pool_get_stats(self._h, ctypes.byref(st)), "kvc_pool_get_stats")
        return {f: getattr(st, f) for f, _ in PoolStats._fields_}


def slots_from_tables(block_tables, block_size: int, rows, positions):
    """Host helper (kvc_slots_from_tables): block_tables is a CPU int32 tensor [R, max_blocks]."""
    torch = _torch()
    bt = block_tables.to(torch.int32).contiguous().cpu()
    r = torch.as_tensor(rows, dtype=torch.int32).contiguous()
    p = torch.as_tensor(positions, dtype=torch.int64).contiguous()
    out = torch.empty(p.numel(), dtype=torch.int64)
    _check(raw().kvc_slots_from_tables(_ptr(bt), bt.shape[0], bt.shape[1], block_size, _ptr(r), _ptr(p), p.numel(),
                                       _ptr(out)), "kvc_slots_from_tables")
    return out


def decode_attention_window(q, k_cache, v_cache, block_tables, context_lens, scale, window, out, workspace=None,
                            stream=None):
    """kvc_decode_attention_window: decode over the newest ``window`` rows of every sequence."""
    decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace, stream, window=window)


def copy_blocks(cache, pairs, stream=None):
    """kvc_copy_blocks: block pairs[i, 1] of ``cache`` (a pool tensor [num_blocks, ...]) becomes a copy of
    block pairs[i, 0]. pairs: int64 device tensor [n, 2]."""
    torch = _torch()
    _require(cache, "cache")
    _require(pairs, "pairs", torch.int64)
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be [n, 2]")
    nb = cache.shape[0]
    block_bytes = cache[0].numel() * cache.element_size()
    _check(raw().kvc_copy_blocks(_ptr(cache), nb, block_bytes, _ptr(pairs), pairs.shape[0], _stream(stream)),
           "kvc_copy_blocks")


def _append_q8(fn, code_dtype, k, v, slot_mapping, k_cache, v_cache, v_scale, k_scale, stream):
    torch = _torch()
    for t, n in ((k, "k"), (v, "v")):
        _require(t, n)
    _require(slot_mapping, "slot_mapping", torch.int64)
    _require(k_cache, "k_cache", code_dtype)
    _require(v_cache, "v_cache", code_dtype)
    _require(v_scale, "v_scale", torch.float32)
    _require(k_scale, "k_scale", torch.float32)
    T, hkv, d = k.shape
    nb, hkv2, bs, d2 = k_cache.shape
    if (hkv2, d2) != (hkv, d) or tuple(v_scale.shape) != (nb, hkv, bs) or tuple(k_scale.shape) != (hkv, d):
        raise ValueError("shape mismatch")
    _check(getattr(raw(), fn)(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache), _ptr(v_scale),
                              _ptr(k_scale), nb, bs, hkv, d, _dtype_code(k), _stream(stream)), fn)


def _decode_q8(fn, code_dtype, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
               workspace, stream):
    torch = _torch()
    _require(q, "q", torch.bfloat16)
    _require(out, "out")
    _require(k_cache, "k_cache", code_dtype)
    _require(v_cache, "v_cache", code_dtype)
    _require(k_scale, "k_scale", torch.float32)
    _require(v_scale, "v_scale", torch.float32)
    _require(block_tables, "block_tables", torch.int32)
    _require(context_lens, "context_lens", torch.int32)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != d or tuple(out.shape) != (B, hq, d) or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("shape mismatch")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        _require(workspace, "workspace")
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(getattr(raw(), fn)(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                              _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, float(scale), hq, hkv,
                              d, bs, nb, _ptr(out), _dtype_code(out), ws_ptr, ws_bytes, _stream(stream)), fn)


def append_fp8(k, v, slot_mapping, k_cache, v_cache, v_scale, k_scale, stream=None):
    """kvc_append_fp8. k/v [T, Hkv, D] (f32/f16/bf16); k_cache/v_cache uint8 [num_blocks, Hkv, bs, D];
    v_scale fp32 [num_blocks, Hkv, bs] (written); k_scale fp32 [Hkv, D]."""
    _append_q8("kvc_append_fp8", _torch().uint8, k, v, slot_mapping, k_cache, v_cache, v_scale, k_scale, stream)


def decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
                         workspace=None, stream=None):
    """kvc_decode_attention_fp8: q bf16 [B, Hq, D] over FP8 caches written by append_fp8."""
    _decode_q8("kvc_decode_attention_fp8", _torch().uint8, q, k_cache, v_cache, k_scale, v_scale, block_tables,
               context_lens, scale, out, workspace, stream)


def append_int8(k, v, slot_mapping, k_cache, v_cache, v_scale, k_scale, stream=None):
    """kvc_append_int8. k/v [T, Hkv, D] (f32/f16/bf16); k_cache/v_cache int8 [num_blocks, Hkv, bs, D];
    v_scale fp32 [num_blocks, Hkv, bs] (written); k_scale fp32 [Hkv, D]."""
    _append_q8("kvc_append_int8", _torch().int8, k, v, slot_mapping, k_cache, v_cache, v_scale, k_scale, stream)


def decode_attention_int8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
                          workspace=None, stream=None):
    """kvc_decode_attention_int8: q bf16 [B, Hq, D] over INT8 caches written by append_int8."""
    _decode_q8("kvc_decode_attention_int8", _torch().int8, q, k_cache, v_cache, k_scale, v_scale, block_tables,
               context_lens, scale, out, workspace, stream)
