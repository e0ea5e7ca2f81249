"""Oracle for head-segmented paged attention. TEST INFRASTRUCTURE ONLY.

Python side of the plain fp64 C++ oracle in ``segkv_oracle.cpp``: the page
model (kept sets, page ids), attention over explicit per-head key sets, the
attention mass each key receives, and the rotary re-alignment. The token
selection and FFN of sparse FFN routing are in ``sparse_ffn.py``.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
it; the library never imports it. See the C++ file for the sources and the
readings of the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "segkv_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, INVALID_ARG, OUT_OF_PAGES, EVICTED = 0, -1, -2, -3
GLOBAL, LOCAL = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with the host compiler (fp64, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        _lib.orc_state_create.restype = P
        _lib.orc_state_create.argtypes = [I, I, P, P, I, I, I, I]
        _lib.orc_state_destroy.argtypes = [P]
        _lib.orc_free_pages.argtypes = [P]
        _lib.orc_seq_len.argtypes = [P, I, I]
        _lib.orc_append.argtypes = [P, I, P, P, I]
        _lib.orc_trim.argtypes = [P, I, P, I]
        _lib.orc_free_seq.argtypes = [P, I]
        _lib.orc_import.argtypes = [P, I, I, I, P]
        _lib.orc_segment.argtypes = [P, I, I, I, P, P, P, P, I, P]
        att = [I, I, I, ctypes.c_double, P, P, P, P, P, P, P, P, I, P, P, I64]
        _lib.orc_attention.argtypes = att + [P, P]
        _lib.orc_attention_blocked.argtypes = att + [I, P, P]
        _lib.orc_rope.argtypes = [P, I64, I, I, I, ctypes.c_double, P]
        _lib.orc_attn_mass.argtypes = [I, I, I, ctypes.c_double, P, P, P, P, P, I, P, P, I, P,
                                       I64, I64, P]
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


class PageModel:
    """Kept sets and page ids of every (layer, KV head, sequence) segment."""

    def __init__(self, num_layers, num_kv_heads, head_class, window, page_size, max_seqs,
                 max_seq_len, num_pages):
        hc = np.ascontiguousarray(np.asarray(head_class, dtype=np.uint8).reshape(-1))
        win = _i32(window)
        self.L, self.H, self.P, self.S = num_layers, num_kv_heads, page_size, max_seqs
        self._h = lib().orc_state_create(num_layers, num_kv_heads, _ptr(hc), _ptr(win), page_size,
                                         max_seqs, max_seq_len, num_pages)
        if not self._h:
            raise ValueError("invalid page model parameters")

    def __del__(self):
        if getattr(self, "_h", None):
            lib().orc_state_destroy(self._h)
            self._h = None

    def append(self, layer, cu_seqlens, seq_ids) -> int:
        cu, ids = _i32(cu_seqlens), _i32(seq_ids)
        return lib().orc_append(self._h, layer, _ptr(cu), _ptr(ids), len(ids))

    def trim(self, layer, seq_ids) -> int:
        ids = _i32(seq_ids)
        return lib().orc_trim(self._h, layer, _ptr(ids), len(ids))

    def free_seq(self, seq) -> int:
        return lib().orc_free_seq(self._h, seq)

    def import_segment(self, layer, seq, n, starts) -> int:
        st = _i32(starts)
        return lib().orc_import(self._h, layer, seq, n, _ptr(st))

    def free_pages(self) -> int:
        return lib().orc_free_pages(self._h)

    def seq_len(self, layer, seq) -> int:
        return lib().orc_seq_len(self._h, layer, seq)

    def segment(self, layer, head, seq):
        """(start, length, first logical page, [page ids in logical order])."""
        cap = 1 << 16
        ids = np.zeros(cap, dtype=np.int32)
        s, n, f, c = (np.zeros(1, dtype=np.int32) for _ in range(4))
        rc = lib().orc_segment(self._h, layer, head, seq, _ptr(s), _ptr(n), _ptr(f), _ptr(ids),
                               cap, _ptr(c))
        if rc != OK:
            raise ValueError(f"orc_segment failed: {rc}")
        return int(s[0]), int(n[0]), int(f[0]), ids[:int(c[0])].tolist()


def _bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor (CPU)."""
    import torch
    return np.ascontiguousarray(t.detach().to("cpu").contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def attention(q, k, v, row_seq, row_pos, kv_off, kv_len, head_class, window, seg_start,
              rows=None, scale=None, block=None):
    """fp64 attention of the listed query tokens.

    q: bf16 [Nq, Hq, D]; k, v: bf16 [sum kv_len, Hkv, D] (logical sequences);
    row_seq/row_pos: per query token, its sequence index and position;
    kv_off/kv_len: per sequence, first row in k/v and tracked length;
    head_class: [Hkv]; seg_start: [num_seqs, Hkv] first kept key.
    Returns (status, o [nrows, Hq, D] fp64, lse [nrows, Hq] fp64).
    With block=b the key set is reduced in blocks of b and merged.
    """
    nq, hq, d = q.shape
    hkv = k.shape[1]
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    rs, rp = _i32(row_seq), _i32(row_pos)
    ko = np.ascontiguousarray(np.asarray(kv_off, dtype=np.int64))
    kl = _i32(kv_len)
    hc = np.ascontiguousarray(np.asarray(head_class, dtype=np.uint8))
    ss = _i32(seg_start).reshape(-1)
    rows = np.arange(nq, dtype=np.int64) if rows is None else np.ascontiguousarray(
        np.asarray(rows, dtype=np.int64))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((len(rows), hq, d), dtype=np.float64)
    lse = np.zeros((len(rows), hq), dtype=np.float64)
    args = [hq, hkv, d, ctypes.c_double(scale), _ptr(qb), _ptr(rs), _ptr(rp), _ptr(ko), _ptr(kl),
            _ptr(kb), _ptr(vb), _ptr(hc), int(window), _ptr(ss), _ptr(rows),
            ctypes.c_int64(len(rows))]
    if block is None:
        rc = lib().orc_attention(*args, _ptr(o), _ptr(lse))
    else:
        rc = lib().orc_attention_blocked(*args, int(block), _ptr(o), _ptr(lse))
    return rc, o, lse


def rope(x, pos, rotary_dim, style, base):
    """fp64 rotary rotation of rows x [rows, d] by pos[row] positions (see
    orc_rope). x may be bf16 (widened exactly) or float; returns fp64."""
    import torch
    if hasattr(x, "dtype") and x.dtype == torch.bfloat16:
        xs = x.to(torch.float64).numpy()
    else:
        xs = np.asarray(x, dtype=np.float64)
    shape = xs.shape
    v = np.ascontiguousarray(xs.reshape(-1, shape[-1]).copy())
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.float64).reshape(-1),
                                             (v.shape[0],)) if np.ndim(pos) == 0 else
                             np.asarray(pos, dtype=np.float64).reshape(-1))
    rc = lib().orc_rope(_ptr(v), ctypes.c_int64(v.shape[0]), v.shape[1], rotary_dim, style,
                        ctypes.c_double(base), _ptr(p))
    if rc != OK:
        raise ValueError("orc_rope: bad arguments")
    return v.reshape(shape)


def attn_mass(q, k, row_seq, row_pos, kv_off, kv_len, head_class, window, seg_start, scale=None):
    """fp64 attention mass each key receives from the listed query tokens
    (see orc_attn_mass): returns (status, mass [Hkv, sum kv_len]); key j of
    sequence b is column kv_off[b] + j."""
    nq, hq, d = q.shape
    hkv = k.shape[1]
    qb, kb = _bf16_bits(q), _bf16_bits(k)
    ko = np.ascontiguousarray(np.asarray(kv_off, dtype=np.int64))
    kl = _i32(kv_len)
    hc = np.ascontiguousarray(np.asarray(head_class, dtype=np.uint8))
    ss = _i32(seg_start).reshape(-1)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    nkeys = k.shape[0]
    mass = np.zeros((hkv, nkeys), dtype=np.float64)
    rc = lib().orc_attn_mass(hq, hkv, d, ctypes.c_double(scale), _ptr(qb), _ptr(_i32(row_seq)),
                             _ptr(_i32(row_pos)), _ptr(ko), _ptr(kl), len(kl), _ptr(kb), _ptr(hc),
                             int(window), _ptr(ss), ctypes.c_int64(nq), ctypes.c_int64(nkeys),
                             _ptr(mass))
    return rc, mass
