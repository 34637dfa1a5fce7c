"""ctypes wrapper around the float64 C oracle (oscar_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The product library never
imports this package.  See oscar_oracle.c for the method sources and the
readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oscar_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboscar_oracle.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_OUT_OF_PAGES = 0, 1, 2, 3


def build(force: bool = False, defines: tuple[str, ...] = (), out: str | None = None) -> str:
    """Compile the oracle with gcc (-O2, OpenMP).  ``defines`` lets a test
    build a variant of the oracle into ``out`` (never the default path)."""
    target = out or _LIB_PATH
    if not force and not defines and os.path.exists(target) and \
            os.path.getmtime(target) >= os.path.getmtime(_SRC):
        return target
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-Wextra", "-Wno-unused-parameter"]
    cmd += [f"-D{d}" for d in defines]
    cmd += [_SRC, "-o", target + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(target + ".tmp", target)
    return target


@dataclasses.dataclass(frozen=True)
class Shape:
    head_dim: int = 128
    quant_group: int = 32
    sink: int = 64
    recent: int = 256
    page_size: int = 64
    num_q_heads: int = 4
    num_kv_heads: int = 1


class _CShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("head_dim", "quant_group", "sink", "recent", "page_size", "num_q_heads", "num_kv_heads")]


def _cshape(s: Shape) -> _CShape:
    return _CShape(s.head_dim, s.quant_group, s.sink, s.recent, s.page_size, s.num_q_heads, s.num_kv_heads)


_P = ctypes.c_void_p


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """Loaded oracle library.  All arrays are numpy, C-contiguous."""

    def __init__(self, path: str | None = None):
        self.lib = ctypes.CDLL(path or build())
        L = self.lib
        L.oracle_bitrev.restype = ctypes.c_int
        L.oracle_bitrev.argtypes = [ctypes.c_int, ctypes.c_int]
        L.oracle_hadamard.argtypes = [ctypes.c_int, _P]
        L.oracle_build_R.argtypes = [ctypes.c_int, _P, _P]
        L.oracle_f16_from_f64.restype = ctypes.c_uint16
        L.oracle_f16_from_f64.argtypes = [ctypes.c_double]
        L.oracle_f64_from_f16.restype = ctypes.c_double
        L.oracle_f64_from_f16.argtypes = [ctypes.c_uint16]
        L.oracle_f64_from_bf16.restype = ctypes.c_double
        L.oracle_f64_from_bf16.argtypes = [ctypes.c_uint16]
        L.oracle_pack4.restype = ctypes.c_uint8
        L.oracle_pack4.argtypes = [_P]
        L.oracle_unpack4.argtypes = [ctypes.c_uint8, _P]
        L.oracle_quantize_vec.argtypes = [ctypes.c_int, ctypes.c_int, _P, ctypes.c_double, _P, _P, _P, _P, _P, _P]
        L.oracle_dequantize_vec.argtypes = [ctypes.c_int, ctypes.c_int, _P, _P, _P, _P]
        L.oracle_block_bytes.restype = ctypes.c_size_t
        L.oracle_block_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.oracle_evict.restype = ctypes.c_int
        L.oracle_evict.argtypes = [ctypes.POINTER(_CShape), ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P,
                                   ctypes.c_int, _P, _P, _P]
        L.oracle_decode.restype = ctypes.c_int
        L.oracle_decode.argtypes = [ctypes.POINTER(_CShape), ctypes.c_int, _P, _P, _P, _P, _P, ctypes.c_int,
                                    _P, _P, ctypes.c_double, _P, _P]
        L.oracle_decode_segmented.restype = ctypes.c_int
        L.oracle_decode_segmented.argtypes = [ctypes.POINTER(_CShape), ctypes.c_int, _P, _P, _P, _P, _P,
                                              ctypes.c_int, _P, _P, ctypes.c_double, _P]
        L.oracle_pool_layout.restype = ctypes.c_int
        L.oracle_pool_layout.argtypes = [ctypes.POINTER(_CShape), ctypes.c_int, _P, _P, ctypes.c_int,
                                         ctypes.c_uint64, ctypes.c_int, _P, _P, _P]
        L.oracle_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_int, _P]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]

    # -- scalar helpers -------------------------------------------------
    def bitrev(self, j: int, nbits: int) -> int:
        return self.lib.oracle_bitrev(j, nbits)

    def hadamard(self, d: int) -> np.ndarray:
        H = np.zeros((d, d), np.float64)
        self.lib.oracle_hadamard(d, _ptr(H))
        return H

    def build_R(self, U: np.ndarray) -> np.ndarray:
        U = np.ascontiguousarray(U, np.float64)
        d = U.shape[0]
        R = np.zeros((d, d), np.float64)
        self.lib.oracle_build_R(d, _ptr(U), _ptr(R))
        return R

    def f16_from_f64(self, x) -> np.ndarray:
        x = np.asarray(x, np.float64).ravel()
        return np.array([self.lib.oracle_f16_from_f64(float(v)) for v in x], np.uint16)

    def f64_from_f16(self, h) -> np.ndarray:
        h = np.asarray(h, np.uint16).ravel()
        return np.array([self.lib.oracle_f64_from_f16(int(v)) for v in h], np.float64)

    def f64_from_bf16(self, b) -> np.ndarray:
        b = np.asarray(b, np.uint16).ravel()
        return np.array([self.lib.oracle_f64_from_bf16(int(v)) for v in b], np.float64)

    def pack4(self, codes) -> int:
        c = np.ascontiguousarray(codes, np.uint8)
        return int(self.lib.oracle_pack4(_ptr(c)))

    def unpack4(self, byte: int) -> np.ndarray:
        c = np.zeros(4, np.uint8)
        self.lib.oracle_unpack4(byte, _ptr(c))
        return c

    def quantize_vec(self, y: np.ndarray, g: int, clip: float):
        y = np.ascontiguousarray(y, np.float64)
        d = y.shape[0]
        ng = d // g
        codes = np.zeros(d, np.uint8)
        s16 = np.zeros(ng, np.uint16)
        z16 = np.zeros(ng, np.uint16)
        u = np.zeros(d, np.float64)
        sp = np.zeros(ng, np.float64)
        zp = np.zeros(ng, np.float64)
        self.lib.oracle_quantize_vec(d, g, _ptr(y), float(clip), _ptr(codes), _ptr(s16), _ptr(z16),
                                     _ptr(u), _ptr(sp), _ptr(zp))
        return codes, s16, z16, u, sp, zp

    def dequantize_vec(self, codes, s16, z16, g: int) -> np.ndarray:
        codes = np.ascontiguousarray(codes, np.uint8)
        s16 = np.ascontiguousarray(s16, np.uint16)
        z16 = np.ascontiguousarray(z16, np.uint16)
        out = np.zeros(codes.shape[0], np.float64)
        self.lib.oracle_dequantize_vec(codes.shape[0], g, _ptr(codes), _ptr(s16), _ptr(z16), _ptr(out))
        return out

    def block_bytes(self, d: int, g: int, page: int) -> int:
        return int(self.lib.oracle_block_bytes(d, g, page))

    # -- hot-path steps ---------------------------------------------------
    def evict(self, shape: Shape, src_kv: np.ndarray, dst_seq, dst_pos, U: np.ndarray, clip: np.ndarray,
              pool: np.ndarray, page_table: np.ndarray, max_pages: int, src_row=None, want_aux=False):
        """Quantise n_tok token-vectors into ``pool`` (modified in place).
        src_kv: uint16 bf16 bits [rows][Hk][2][d]; U float64 [Hk][2][d][d];
        clip [Hk][2].  Returns (u, s_pre, z_pre) when want_aux."""
        dst_seq = np.ascontiguousarray(dst_seq, np.int32)
        dst_pos = np.ascontiguousarray(dst_pos, np.int32)
        n = dst_seq.shape[0]
        src_kv = np.ascontiguousarray(src_kv, np.uint16)
        U = np.ascontiguousarray(U, np.float64)
        clip = np.ascontiguousarray(clip, np.float64)
        page_table = np.ascontiguousarray(page_table, np.int32)
        assert pool.dtype == np.uint8 and pool.flags.c_contiguous
        sr = None if src_row is None else np.ascontiguousarray(src_row, np.int32)
        Hk, d, ng = shape.num_kv_heads, shape.head_dim, shape.head_dim // shape.quant_group
        u = sp = zp = None
        if want_aux:
            u = np.zeros((n, Hk, 2, d), np.float64)
            sp = np.zeros((n, Hk, 2, ng), np.float64)
            zp = np.zeros((n, Hk, 2, ng), np.float64)
        cs = _cshape(shape)
        rc = self.lib.oracle_evict(ctypes.byref(cs), n, _ptr(src_kv), _ptr(sr), _ptr(dst_seq), _ptr(dst_pos),
                                   _ptr(U), _ptr(clip), _ptr(pool), _ptr(page_table), max_pages,
                                   _ptr(u), _ptr(sp), _ptr(zp))
        if rc != OK:
            raise ValueError(f"oracle_evict failed: {rc}")
        return (u, sp, zp) if want_aux else None

    def decode(self, shape: Shape, q, bf16_kv, bf16_len, pool, page_table, max_pages, hist_len, U,
               sm_scale: float, unit_mask=None, segmented=False) -> np.ndarray:
        q = np.ascontiguousarray(q, np.uint16)
        B = q.shape[0]
        bf16_kv = np.ascontiguousarray(bf16_kv, np.uint16)
        bf16_len = np.ascontiguousarray(bf16_len, np.int32)
        hist_len = np.ascontiguousarray(hist_len, np.int32)
        U = np.ascontiguousarray(U, np.float64)
        pool = None if pool is None else np.ascontiguousarray(pool, np.uint8)
        page_table = None if page_table is None else np.ascontiguousarray(page_table, np.int32)
        out = np.zeros((B, shape.num_q_heads, shape.head_dim), np.float64)
        cs = _cshape(shape)
        if segmented:
            rc = self.lib.oracle_decode_segmented(ctypes.byref(cs), B, _ptr(q), _ptr(bf16_kv), _ptr(bf16_len),
                                                  _ptr(pool), _ptr(page_table), max_pages, _ptr(hist_len),
                                                  _ptr(U), float(sm_scale), _ptr(out))
        else:
            um = None if unit_mask is None else np.ascontiguousarray(unit_mask, np.uint8)
            rc = self.lib.oracle_decode(ctypes.byref(cs), B, _ptr(q), _ptr(bf16_kv), _ptr(bf16_len),
                                        _ptr(pool), _ptr(page_table), max_pages, _ptr(hist_len), _ptr(U),
                                        float(sm_scale), _ptr(um), _ptr(out))
        if rc != OK:
            raise ValueError(f"oracle_decode failed: {rc}")
        return out

    def pool_layout(self, shape: Shape, hist_capacity, prefix_group=None, shared_hist_tokens: int = 0,
                    perm_seed: int = 0, max_pages: int | None = None):
        cap = np.ascontiguousarray(hist_capacity, np.int32)
        B = cap.shape[0]
        if max_pages is None:
            max_pages = max(1, int((cap.max(initial=0) + shape.page_size - 1) // shape.page_size))
        pg = None if prefix_group is None else np.ascontiguousarray(prefix_group, np.int32)
        table = np.zeros((B, max_pages), np.int32)
        npages = ctypes.c_int32(0)
        nbytes = ctypes.c_uint64(0)
        cs = _cshape(shape)
        rc = self.lib.oracle_pool_layout(ctypes.byref(cs), B, _ptr(cap), _ptr(pg), shared_hist_tokens,
                                         ctypes.c_uint64(perm_seed), max_pages, _ptr(table),
                                         ctypes.byref(npages), ctypes.byref(nbytes))
        return rc, table, int(npages.value), int(nbytes.value)

    def splitmix64(self, seed: int, n: int) -> np.ndarray:
        out = np.zeros(n, np.uint64)
        self.lib.oracle_splitmix64(ctypes.c_uint64(seed), n, _ptr(out))
        return out

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.oracle_set_num_threads(n)


_INSTANCE: Oracle | None = None


def get() -> Oracle:
    global _INSTANCE
    if _INSTANCE is None:
        _INSTANCE = Oracle()
    return _INSTANCE
