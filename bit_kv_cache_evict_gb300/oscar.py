"""Thin ctypes binding of liboscar (include/oscar.h), same call names.

Argument marshalling only: every step of the hot path runs in the CUDA
kernels of liboscar.so.  There is no CPU fallback: if the library is missing
or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "liboscar.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "oscar.h")

OSCAR_OK, OSCAR_ERR_INVALID_ARG, OSCAR_ERR_UNSUPPORTED, OSCAR_ERR_OUT_OF_PAGES, OSCAR_ERR_WORKSPACE, \
    OSCAR_ERR_CUDA = range(6)
OSCAR_STATUS_BAD_PAGE, OSCAR_STATUS_BAD_POS, OSCAR_STATUS_TIMEOUT = 1, 2, 4
BLOCK_BYTES = 6144


class OscarError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class oscar_shape(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("quant_group", ctypes.c_int32), ("sink", ctypes.c_int32),
                ("recent", ctypes.c_int32), ("page_size", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32)]


def make_shape(num_q_heads: int, num_kv_heads: int, head_dim: int = 128, quant_group: int = 32, sink: int = 64,
               recent: int = 256, page_size: int = 64) -> oscar_shape:
    return oscar_shape(head_dim, quant_group, sink, recent, page_size, num_q_heads, num_kv_heads)


_LIB = None
_P = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """Load liboscar.so (built in-tree by ``build.build()``); raise if absent."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"liboscar.so not built ({LIB_PATH}); run bit_kv_cache_evict_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        S = ctypes.POINTER(oscar_shape)
        L.oscar_block_bytes.restype = ctypes.c_size_t
        L.oscar_block_bytes.argtypes = [S]
        L.oscar_status_string.restype = ctypes.c_char_p
        L.oscar_status_string.argtypes = [ctypes.c_int]
        L.oscar_last_cuda_error.restype = ctypes.c_int
        L.oscar_pool_layout.restype = ctypes.c_int
        L.oscar_pool_layout.argtypes = [S, ctypes.c_int32, _P, _P, ctypes.c_int32, ctypes.c_uint64, ctypes.c_int32,
                                        _P, _P, _P]
        I32, PP = ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p)
        L.oscar_pages_create.restype = ctypes.c_int
        L.oscar_pages_create.argtypes = [I32, PP]
        L.oscar_pages_destroy.restype = None
        L.oscar_pages_destroy.argtypes = [_P]
        for fn in ("oscar_pages_alloc", "oscar_pages_retain", "oscar_pages_release"):
            getattr(L, fn).restype = ctypes.c_int
            getattr(L, fn).argtypes = [_P, I32, _P]
        L.oscar_pages_refcount.restype = I32
        L.oscar_pages_refcount.argtypes = [_P, I32]
        L.oscar_pages_free_count.restype = I32
        L.oscar_pages_free_count.argtypes = [_P]
        L.oscar_pages_prepare_write.restype = ctypes.c_int
        L.oscar_pages_prepare_write.argtypes = [_P, I32, _P, _P, _P, I32, I32, _P, _P, _P]
        L.oscar_pages_copy.restype = ctypes.c_int
        L.oscar_pages_copy.argtypes = [S, I32, _P, _P, _P, _P, I32, _P]
        L.oscar_radix_create.restype = ctypes.c_int
        L.oscar_radix_create.argtypes = [_P, PP]
        L.oscar_radix_destroy.restype = None
        L.oscar_radix_destroy.argtypes = [_P]
        L.oscar_radix_insert.restype = ctypes.c_int
        L.oscar_radix_insert.argtypes = [_P, _P, I32, _P, I32]
        L.oscar_radix_match.restype = ctypes.c_int
        L.oscar_radix_match.argtypes = [_P, _P, I32, I32, _P, _P]
        L.oscar_radix_evict.restype = ctypes.c_int
        L.oscar_radix_evict.argtypes = [_P, I32, _P]
        L.oscar_radix_cached_pages.restype = I32
        L.oscar_radix_cached_pages.argtypes = [_P]
        L.oscar_evict_quantize.restype = ctypes.c_int
        L.oscar_evict_quantize.argtypes = [S, ctypes.c_int32, _P, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P]
        L.oscar_decode_attn.restype = ctypes.c_int
        L.oscar_decode_attn.argtypes = [S, ctypes.c_int32, _P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_int32, _P,
                                        _P, ctypes.c_float, _P, _P, ctypes.POINTER(ctypes.c_size_t), _P, _P]
        L.oscar_decode_attn_noalloc.restype = ctypes.c_int
        L.oscar_decode_attn_noalloc.argtypes = [S, ctypes.c_int32, _P, _P, _P, _P, _P, ctypes.c_int32,
                                                ctypes.c_int32, _P, _P, ctypes.c_float, _P, _P, _P]
        L.oscar_time_next_int2.restype = None
        L.oscar_time_next_int2.argtypes = [_P, _P]
        L.oscar_evict_quantize_codebook.restype = ctypes.c_int
        L.oscar_evict_quantize_codebook.argtypes = [S, ctypes.c_int32, _P, ctypes.c_int32, _P, _P, _P, _P, _P, _P,
                                                    _P, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P,
                                                    _P]
        L.oscar_decode_attn_codebook.restype = ctypes.c_int
        L.oscar_decode_attn_codebook.argtypes = [S, ctypes.c_int32, _P, _P, _P, _P, _P, ctypes.c_int32,
                                                 ctypes.c_int32, _P, _P, _P, ctypes.c_float, _P, _P,
                                                 ctypes.POINTER(ctypes.c_size_t), _P, _P]
        L.oscar_evict_quantize_boost.restype = ctypes.c_int
        L.oscar_evict_quantize_boost.argtypes = [S, ctypes.c_int32, _P, ctypes.c_int32, _P, _P, _P, _P, _P, _P,
                                                 _P, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P]
        L.oscar_decode_attn_boost.restype = ctypes.c_int
        L.oscar_decode_attn_boost.argtypes = [S, ctypes.c_int32, _P, _P, _P, _P, _P, _P, ctypes.c_int32,
                                              ctypes.c_int32, _P, _P, ctypes.c_float, _P, _P,
                                              ctypes.POINTER(ctypes.c_size_t), _P, _P]
        L.oscar_calibrate_codebook.restype = ctypes.c_int
        L.oscar_calibrate_codebook.argtypes = [S, ctypes.c_int32, _P, _P, _P, _P, _P, ctypes.POINTER(ctypes.c_size_t),
                                               _P]
        L.oscar_calibrate_clip.restype = ctypes.c_int
        L.oscar_calibrate_clip.argtypes = [S, ctypes.c_int32, _P, _P, _P, ctypes.c_int32, _P, _P, _P,
                                           ctypes.POINTER(ctypes.c_size_t), _P]
        L.oscar_calibrate_rotation.restype = ctypes.c_int
        L.oscar_calibrate_rotation.argtypes = [S, ctypes.c_int32, _P, ctypes.c_int32, _P, ctypes.c_float, _P, _P,
                                               _P, ctypes.POINTER(ctypes.c_size_t), _P, _P]
        _LIB = L
    return _LIB


def declared_functions() -> list[str]:
    """Entry points declared in include/oscar.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(oscar_\w+)\s*\(", text, re.M)))


def _check(fn: str, st: int) -> None:
    if st != OSCAR_OK:
        msg = lib().oscar_status_string(st).decode()
        if st == OSCAR_ERR_CUDA:
            msg += f" (cudaError {lib().oscar_last_cuda_error()})"
        raise OscarError(fn, st, msg)


def _dptr(t, what: str, dtype=None, align: int = 1):
    """Device pointer of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what}: expected a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def block_bytes(shape: oscar_shape) -> int:
    return int(lib().oscar_block_bytes(ctypes.byref(shape)))


def oscar_pool_layout(shape: oscar_shape, hist_capacity, prefix_group=None, shared_hist_tokens: int = 0,
                      perm_seed: int = 0, max_pages: int | None = None):
    """Host page-table layout.  Returns (page_table int32 [B][max_pages],
    num_pages, pool_bytes)."""
    cap = np.ascontiguousarray(hist_capacity, np.int32)
    B = cap.shape[0]
    if max_pages is None:
        max_pages = max(1, int((int(cap.max(initial=0)) + shape.page_size - 1) // shape.page_size))
    pg = None if prefix_group is None else np.ascontiguousarray(prefix_group, np.int32)
    table = np.zeros((B, max_pages), np.int32)
    n = ctypes.c_int32(0)
    nbytes = ctypes.c_uint64(0)
    st = lib().oscar_pool_layout(ctypes.byref(shape), B, cap.ctypes.data_as(_P),
                                 None if pg is None else pg.ctypes.data_as(_P), shared_hist_tokens,
                                 ctypes.c_uint64(perm_seed), max_pages, table.ctypes.data_as(_P), ctypes.byref(n),
                                 ctypes.byref(nbytes))
    _check("oscar_pool_layout", st)
    return table, int(n.value), int(nbytes.value)


def oscar_evict_quantize(shape: oscar_shape, src_kv, dst_seq, dst_pos, U, clip, pool, page_table, batch: int,
                         max_pages: int, num_pages: int, src_row=None, new_kv=None, dev_status=None,
                         stream=None) -> None:
    """Fused rotate/clip/quantise/pack of dst_seq.numel() token rows into the
    pool (see include/oscar.h).  src_kv: bf16 [rows][Hk][2][d]."""
    import torch
    n_tok = int(dst_seq.numel())
    st = lib().oscar_evict_quantize(
        ctypes.byref(shape), n_tok, _dptr(src_kv, "src_kv", torch.bfloat16), int(src_kv.shape[0]),
        _dptr(src_row, "src_row", torch.int32), _dptr(dst_seq, "dst_seq", torch.int32),
        _dptr(dst_pos, "dst_pos", torch.int32), _dptr(new_kv, "new_kv", torch.bfloat16),
        _dptr(U, "U", torch.float32), _dptr(clip, "clip", torch.float32), _dptr(pool, "pool", torch.uint8),
        _dptr(page_table, "page_table", torch.int32), batch, max_pages, num_pages,
        _dptr(dev_status, "dev_status", torch.int32), _stream_ptr(stream))
    _check("oscar_evict_quantize", st)


def oscar_time_next_int2(ev_start, ev_stop) -> None:
    """Measurement hook: the next oscar_decode_attn on this thread records the
    two (already recorded once, timing-enabled) torch.cuda.Event objects
    around its INT2 split-K kernel."""
    lib().oscar_time_next_int2(ctypes.c_void_p(ev_start.cuda_event), ctypes.c_void_p(ev_stop.cuda_event))


def oscar_decode_workspace_bytes(shape: oscar_shape, batch: int, max_pages: int) -> int:
    ws = ctypes.c_size_t(0)
    st = lib().oscar_decode_attn(ctypes.byref(shape), batch, None, None, None, None, None, max_pages, 0, None,
                                 None, ctypes.c_float(1.0), None, None, ctypes.byref(ws), None, None)
    _check("oscar_decode_attn", st)
    return int(ws.value)


def oscar_decode_attn(shape: oscar_shape, q, bf16_kv, bf16_len, pool, page_table, max_pages: int, num_pages: int,
                      hist_len, U, sm_scale: float, out, workspace, dev_status=None, stream=None) -> None:
    """Decode attention over sink + INT2 history + recent (see
    include/oscar.h).  ``workspace``: CUDA uint8 tensor of at least
    oscar_decode_workspace_bytes(shape, batch, max_pages) bytes."""
    import torch
    B = int(q.shape[0])
    ws = ctypes.c_size_t(int(workspace.numel()))
    st = lib().oscar_decode_attn(
        ctypes.byref(shape), B, _dptr(q, "q", torch.bfloat16), _dptr(bf16_kv, "bf16_kv", torch.bfloat16),
        _dptr(bf16_len, "bf16_len", torch.int32), _dptr(pool, "pool", torch.uint8),
        _dptr(page_table, "page_table", torch.int32), max_pages, num_pages, _dptr(hist_len, "hist_len", torch.int32),
        _dptr(U, "U", torch.float32), ctypes.c_float(sm_scale), _dptr(out, "out", torch.float32),
        _dptr(workspace, "workspace", torch.uint8), ctypes.byref(ws), _dptr(dev_status, "dev_status", torch.int32),
        _stream_ptr(stream))
    _check("oscar_decode_attn", st)


NOALLOC_SCRATCH_BYTES = 64 << 20


def oscar_decode_attn_noalloc(shape: oscar_shape, q, bf16_kv, bf16_len, pool, page_table, max_pages: int,
                              num_pages: int, hist_len, U, sm_scale: float, out, dev_status=None,
                              stream=None) -> None:
    """oscar_decode_attn for callers that cannot allocate device memory: the
    scratch is the library's fixed 64 MiB device array (see include/oscar.h
    for the limits, the first-call set-up and why overlapping calls race)."""
    import torch
    B = int(q.shape[0])
    st = lib().oscar_decode_attn_noalloc(
        ctypes.byref(shape), B, _dptr(q, "q", torch.bfloat16), _dptr(bf16_kv, "bf16_kv", torch.bfloat16),
        _dptr(bf16_len, "bf16_len", torch.int32), _dptr(pool, "pool", torch.uint8),
        _dptr(page_table, "page_table", torch.int32), max_pages, num_pages, _dptr(hist_len, "hist_len", torch.int32),
        _dptr(U, "U", torch.float32), ctypes.c_float(sm_scale), _dptr(out, "out", torch.float32),
        _dptr(dev_status, "dev_status", torch.int32), _stream_ptr(stream))
    _check("oscar_decode_attn_noalloc", st)


def oscar_calibrate_workspace_bytes(shape: oscar_shape, n_q: int) -> int:
    ws = ctypes.c_size_t(0)
    st = lib().oscar_calibrate_rotation(ctypes.byref(shape), n_q, None, 1, None, ctypes.c_float(1.0), None, None,
                                        None, ctypes.byref(ws), None, None)
    _check("oscar_calibrate_rotation", st)
    return int(ws.value)


def oscar_calibrate_rotation(shape: oscar_shape, q, kv, sm_scale: float, U, workspace, eigvals=None,
                             dev_status=None, stream=None) -> None:
    """Offline calibration of U from calibration queries q [n_q][Hq][d] and
    tokens kv [n_t][Hk][2][d] (bf16 CUDA tensors) into U [Hk][2][d][d]
    (fp32); see include/oscar.h."""
    import torch
    ws = ctypes.c_size_t(int(workspace.numel()))
    st = lib().oscar_calibrate_rotation(
        ctypes.byref(shape), int(q.shape[0]), _dptr(q, "q", torch.bfloat16), int(kv.shape[0]),
        _dptr(kv, "kv", torch.bfloat16), ctypes.c_float(sm_scale), _dptr(U, "U", torch.float32),
        _dptr(eigvals, "eigvals", torch.float32), _dptr(workspace, "workspace", torch.uint8), ctypes.byref(ws),
        _dptr(dev_status, "dev_status", torch.int32), _stream_ptr(stream))
    _check("oscar_calibrate_rotation", st)


def oscar_calibrate_clip_workspace_bytes(shape: oscar_shape, n_t: int = 1, n_grid: int = 1) -> int:
    need = ctypes.c_size_t(0)
    st = lib().oscar_calibrate_clip(ctypes.byref(shape), n_t, None, None, None, n_grid, None, None, None,
                                    ctypes.byref(need), None)
    _check("oscar_calibrate_clip", st)
    return int(need.value)


def oscar_calibrate_clip(shape: oscar_shape, kv, U, grid, clip, workspace=None, mse=None, stream=None) -> None:
    """Offline clip-ratio search: for each (KV head, K/V) the ratio of grid
    (fp32 CUDA tensor) with the least reconstruction error of the rotated
    calibration tokens kv [n_t][Hk][2][d] under the eviction's quantiser;
    see include/oscar.h.  ``workspace`` defaults to a fresh tensor."""
    import torch
    n_grid = int(grid.numel())
    if workspace is None:
        workspace = torch.zeros(oscar_calibrate_clip_workspace_bytes(shape, int(kv.shape[0]), n_grid),
                                dtype=torch.uint8, device=kv.device)
    ws = ctypes.c_size_t(int(workspace.numel()))
    st = lib().oscar_calibrate_clip(
        ctypes.byref(shape), int(kv.shape[0]), _dptr(kv, "kv", torch.bfloat16), _dptr(U, "U", torch.float32),
        _dptr(grid, "grid", torch.float32), n_grid, _dptr(clip, "clip", torch.float32),
        _dptr(mse, "mse", torch.float32), _dptr(workspace, "workspace", torch.uint8), ctypes.byref(ws),
        _stream_ptr(stream))
    _check("oscar_calibrate_clip", st)


def oscar_evict_quantize_codebook(shape: oscar_shape, src_kv, dst_seq, dst_pos, U, clip, codebook, pool, page_table,
                                  batch: int, max_pages: int, num_pages: int, src_row=None, new_kv=None,
                                  dev_status=None, stream=None) -> None:
    """oscar_evict_quantize with the Lloyd-Max levels {0, a, 3 - a, 3}
    (codebook: fp32 [Hk][2] inner levels a); see include/oscar.h."""
    import torch
    n_tok = int(dst_seq.numel())
    st = lib().oscar_evict_quantize_codebook(
        ctypes.byref(shape), n_tok, _dptr(src_kv, "src_kv", torch.bfloat16), int(src_kv.shape[0]),
        _dptr(src_row, "src_row", torch.int32), _dptr(dst_seq, "dst_seq", torch.int32),
        _dptr(dst_pos, "dst_pos", torch.int32), _dptr(new_kv, "new_kv", torch.bfloat16),
        _dptr(U, "U", torch.float32), _dptr(clip, "clip", torch.float32),
        _dptr(codebook, "codebook", torch.float32), _dptr(pool, "pool", torch.uint8),
        _dptr(page_table, "page_table", torch.int32), batch, max_pages, num_pages,
        _dptr(dev_status, "dev_status", torch.int32), _stream_ptr(stream))
    _check("oscar_evict_quantize_codebook", st)


def oscar_decode_attn_codebook(shape: oscar_shape, q, bf16_kv, bf16_len, pool, page_table, max_pages: int,
                               num_pages: int, hist_len, U, codebook, sm_scale: float, out, workspace,
                               dev_status=None, stream=None) -> None:
    """oscar_decode_attn reading the history with the Lloyd-Max levels
    (codebook: fp32 [Hk][2]).  The workspace size is
    oscar_decode_workspace_bytes's."""
    import torch
    B = int(q.shape[0])
    ws = ctypes.c_size_t(int(workspace.numel()))
    st = lib().oscar_decode_attn_codebook(
        ctypes.byref(shape), B, _dptr(q, "q", torch.bfloat16), _dptr(bf16_kv, "bf16_kv", torch.bfloat16),
        _dptr(bf16_len, "bf16_len", torch.int32), _dptr(pool, "pool", torch.uint8),
        _dptr(page_table, "page_table", torch.int32), max_pages, num_pages, _dptr(hist_len, "hist_len", torch.int32),
        _dptr(U, "U", torch.float32), _dptr(codebook, "codebook", torch.float32), ctypes.c_float(sm_scale),
        _dptr(out, "out", torch.float32), _dptr(workspace, "workspace", torch.uint8), ctypes.byref(ws),
        _dptr(dev_status, "dev_status", torch.int32), _stream_ptr(stream))
    _check("oscar_decode_attn_codebook", st)


def _host_i32(a):
    import numpy as np
    return np.ascontiguousarray(a, np.int32)


def _np_ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None and a.size else None


class Pages:
    """Refcounted history pages with copy-on-write (host logic of the C ABI's
    oscar_pages_* calls; see include/oscar.h)."""

    def __init__(self, num_pages: int):
        h = ctypes.c_void_p()
        _check("oscar_pages_create", lib().oscar_pages_create(int(num_pages), ctypes.byref(h)))
        self._h = h

    def close(self) -> None:
        if self._h:
            lib().oscar_pages_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, n: int):
        import numpy as np
        out = np.zeros(max(int(n), 0), np.int32)
        _check("oscar_pages_alloc", lib().oscar_pages_alloc(self._h, int(n), _np_ptr(out)))
        return out

    def retain(self, pages) -> None:
        a = _host_i32(pages)
        _check("oscar_pages_retain", lib().oscar_pages_retain(self._h, a.size, _np_ptr(a)))

    def release(self, pages) -> None:
        a = _host_i32(pages)
        _check("oscar_pages_release", lib().oscar_pages_release(self._h, a.size, _np_ptr(a)))

    def refcount(self, page: int) -> int:
        return int(lib().oscar_pages_refcount(self._h, int(page)))

    def free_count(self) -> int:
        return int(lib().oscar_pages_free_count(self._h))

    def prepare_write(self, seq, page_index, page_table):
        """Make the target pages of page_table (numpy int32 [batch][max_pages],
        updated in place) private; returns (copy_src, copy_dst)."""
        import numpy as np
        sq, pi = _host_i32(seq), _host_i32(page_index)
        assert page_table.dtype == np.int32 and page_table.flags.c_contiguous
        src = np.zeros(max(sq.size, 1), np.int32)
        dst = np.zeros(max(sq.size, 1), np.int32)
        n = ctypes.c_int32(0)
        st = lib().oscar_pages_prepare_write(self._h, sq.size, _np_ptr(sq), _np_ptr(pi),
                                             page_table.ctypes.data_as(ctypes.c_void_p), page_table.shape[0],
                                             page_table.shape[1], _np_ptr(src), _np_ptr(dst), ctypes.byref(n))
        _check("oscar_pages_prepare_write", st)
        return src[:n.value].copy(), dst[:n.value].copy()


class Radix:
    """Radix prefix cache over history pages (the C ABI's oscar_radix_*; see
    include/oscar.h).  Keeps a reference to its Pages allocator."""

    def __init__(self, pages: Pages):
        h = ctypes.c_void_p()
        _check("oscar_radix_create", lib().oscar_radix_create(pages._h, ctypes.byref(h)))
        self._h, self.pages = h, pages

    def close(self) -> None:
        if self._h:
            lib().oscar_radix_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def insert(self, tokens, pages) -> None:
        t, p = _host_i32(tokens), _host_i32(pages)
        _check("oscar_radix_insert", lib().oscar_radix_insert(self._h, _np_ptr(t), t.size, _np_ptr(p), p.size))

    def match(self, tokens, max_pages: int):
        """Page ids of the longest cached prefix (one reference each for the caller)."""
        import numpy as np
        t = _host_i32(tokens)
        out = np.zeros(max(int(max_pages), 1), np.int32)
        n = ctypes.c_int32(0)
        _check("oscar_radix_match", lib().oscar_radix_match(self._h, _np_ptr(t), t.size, int(max_pages),
                                                            _np_ptr(out), ctypes.byref(n)))
        return out[:n.value].copy()

    def evict(self, n_pages: int) -> int:
        n = ctypes.c_int32(0)
        _check("oscar_radix_evict", lib().oscar_radix_evict(self._h, int(n_pages), ctypes.byref(n)))
        return int(n.value)

    def cached_pages(self) -> int:
        return int(lib().oscar_radix_cached_pages(self._h))


def oscar_pages_copy(shape: oscar_shape, copy_src, copy_dst, pool, boost, num_pages: int, stream=None) -> None:
    """Copy the pool blocks (and boost records) of copy_src pages to copy_dst
    pages on the device (host index arrays)."""
    import torch
    src, dst = _host_i32(copy_src), _host_i32(copy_dst)
    assert src.size == dst.size
    st = lib().oscar_pages_copy(ctypes.byref(shape), src.size, _np_ptr(src), _np_ptr(dst),
                                _dptr(pool, "pool", torch.uint8), _dptr(boost, "boost", torch.uint8), num_pages,
                                _stream_ptr(stream))
    _check("oscar_pages_copy", st)


BOOST_N = 8
BOOST_BLOCK_BYTES = 1024        # per (page, KV head): 64 tokens x 8 entries x 2 bytes


def oscar_evict_quantize_boost(shape: oscar_shape, src_kv, dst_seq, dst_pos, U, clip, pool, boost, page_table,
                               batch: int, max_pages: int, num_pages: int, src_row=None, new_kv=None,
                               dev_status=None, stream=None) -> None:
    """oscar_evict_quantize plus the K channel-boost records (boost: uint8
    [num_pages * Hk * BOOST_BLOCK_BYTES]); see include/oscar.h."""
    import torch
    n_tok = int(dst_seq.numel())
    st = lib().oscar_evict_quantize_boost(
        ctypes.byref(shape), n_tok, _dptr(src_kv, "src_kv", torch.bfloat16), int(src_kv.shape[0]),
        _dptr(src_row, "src_row", torch.int32), _dptr(dst_seq, "dst_seq", torch.int32),
        _dptr(dst_pos, "dst_pos", torch.int32), _dptr(new_kv, "new_kv", torch.bfloat16),
        _dptr(U, "U", torch.float32), _dptr(clip, "clip", torch.float32), _dptr(pool, "pool", torch.uint8),
        _dptr(boost, "boost", torch.uint8), _dptr(page_table, "page_table", torch.int32), batch, max_pages,
        num_pages, _dptr(dev_status, "dev_status", torch.int32), _stream_ptr(stream))
    _check("oscar_evict_quantize_boost", st)


def oscar_decode_attn_boost(shape: oscar_shape, q, bf16_kv, bf16_len, pool, boost, page_table, max_pages: int,
                            num_pages: int, hist_len, U, sm_scale: float, out, workspace, dev_status=None,
                            stream=None) -> None:
    """oscar_decode_attn with the boosted K values.  The workspace size is
    oscar_decode_workspace_bytes's."""
    import torch
    B = int(q.shape[0])
    ws = ctypes.c_size_t(int(workspace.numel()))
    st = lib().oscar_decode_attn_boost(
        ctypes.byref(shape), B, _dptr(q, "q", torch.bfloat16), _dptr(bf16_kv, "bf16_kv", torch.bfloat16),
        _dptr(bf16_len, "bf16_len", torch.int32), _dptr(pool, "pool", torch.uint8), _dptr(boost, "boost", torch.uint8),
        _dptr(page_table, "page_table", torch.int32), max_pages, num_pages, _dptr(hist_len, "hist_len", torch.int32),
        _dptr(U, "U", torch.float32), ctypes.c_float(sm_scale), _dptr(out, "out", torch.float32),
        _dptr(workspace, "workspace", torch.uint8), ctypes.byref(ws), _dptr(dev_status, "dev_status", torch.int32),
        _stream_ptr(stream))
    _check("oscar_decode_attn_boost", st)


def oscar_calibrate_codebook(shape: oscar_shape, kv, U, clip, codebook, workspace=None, stream=None) -> None:
    """Lloyd-Max fit of the codebook inner levels a [Hk][2] (fp32 CUDA tensor,
    out) from calibration tokens kv [n_t][Hk][2][d]; see include/oscar.h."""
    import torch
    n_t = int(kv.shape[0])
    if workspace is None:
        need = ctypes.c_size_t(0)
        st = lib().oscar_calibrate_codebook(ctypes.byref(shape), n_t, None, None, None, None, None,
                                            ctypes.byref(need), None)
        _check("oscar_calibrate_codebook", st)
        workspace = torch.zeros(int(need.value), dtype=torch.uint8, device=kv.device)
    ws = ctypes.c_size_t(int(workspace.numel()))
    st = lib().oscar_calibrate_codebook(
        ctypes.byref(shape), n_t, _dptr(kv, "kv", torch.bfloat16), _dptr(U, "U", torch.float32),
        _dptr(clip, "clip", torch.float32), _dptr(codebook, "codebook", torch.float32),
        _dptr(workspace, "workspace", torch.uint8), ctypes.byref(ws), _stream_ptr(stream))
    _check("oscar_calibrate_codebook", st)
