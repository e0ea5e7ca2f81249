"""Head-segmented paged KV attention for one GB300 (sm_103a).

Python binding of the C ABI in include/segkv.h: argument marshalling only.
Every step of the path runs in libsegkv.so (host planner + CUDA kernels);
PyTorch supplies device memory and streams. Importing this package without a
built library raises ImportError: there is no fallback path.

The module-level ``segkv_*`` functions mirror the C entry points one to one
and return the C status code; :class:`SegKV` wraps them and raises
:class:`SegKVError` on failure.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsegkv.so")

SEGKV_GLOBAL, SEGKV_LOCAL = 0, 1
SEGKV_OK = 0
SEGKV_ERR_INVALID_ARG = -1
SEGKV_ERR_OUT_OF_PAGES = -2
SEGKV_ERR_EVICTED = -3
SEGKV_ERR_CUDA = -4
SEGKV_ERR_DEVICE_TIMEOUT = -5
SEGKV_WS_PREFILL, SEGKV_WS_DECODE = 0, 1
SEGKV_ROPE_INTERLEAVED, SEGKV_ROPE_HALF = 0, 1
SEGKV_WINDOW_INCLUSIVE, SEGKV_WINDOW_FA = 0, 1

SYMBOLS = ["segkv_create", "segkv_destroy", "segkv_append", "segkv_prefill_attn",
           "segkv_decode_attn", "segkv_trim", "segkv_free_seq", "segkv_workspace_size",
           "segkv_get_segment", "segkv_seq_len", "segkv_stats", "segkv_status",
           "segkv_last_error", "segkv_set_debug", "segkv_decode_attn_noalloc", "segkv_rope_shift",
           "segkv_export_size", "segkv_export", "segkv_import", "segkv_set_window_convention",
           "segkv_decode_attn_multi", "segkv_sparse_ffn", "segkv_ffn_workspace_size", "segkv_attn_mass",
           "segkv_topk_tokens", "segkv_plan_decode", "segkv_plan_prefill", "segkv_plan_mass",
           "segkv_exp2_check"]
NOALLOC_SCRATCH_BYTES = 8 << 20


class SegKVStats(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int64), ("pages_in_use", ctypes.c_int64),
                ("pages_global", ctypes.c_int64), ("pages_local", ctypes.c_int64),
                ("kept_tokens", ctypes.c_int64), ("upload_bytes", ctypes.c_int64)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libsegkv.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "segkv_create": [ctypes.POINTER(P), I, I, I, I, P, P, I, I, I, P, P, I64, ctypes.c_float],
        "segkv_destroy": [P],
        "segkv_append": [P, I, P, P, P, P, I, P],
        "segkv_prefill_attn": [P, I, P, P, P, P, I, P, P, P, SZ, P],
        "segkv_decode_attn": [P, I, P, P, P, I, P, P, SZ, P],
        "segkv_trim": [P, I, P, I],
        "segkv_free_seq": [P, I],
        "segkv_workspace_size": [P, I, I64, I, ctypes.POINTER(SZ)],
        "segkv_get_segment": [P, I, I, I, P, P, P, P, I, P],
        "segkv_seq_len": [P, I, I, P],
        "segkv_stats": [P, ctypes.POINTER(SegKVStats)],
        "segkv_status": [P, P],
        "segkv_last_error": [P],
        "segkv_set_debug": [P, I],
        "segkv_decode_attn_noalloc": [P, I, P, P, P, I, P, P],
        "segkv_rope_shift": [P, I, I, ctypes.c_int32, ctypes.c_double, I, I, ctypes.c_uint64, P],
        "segkv_export_size": [P, I, I, ctypes.POINTER(SZ)],
        "segkv_set_window_convention": [P, I],
        "segkv_decode_attn_multi": [P, I, P, I, P, P, I, P, P, P, SZ, P],
        "segkv_sparse_ffn": [P, P, P, ctypes.c_int64, P, I, P, P, P, I, I, P, SZ, P],
        "segkv_attn_mass": [P, I, P, P, P, P, I, P, P, P],
        "segkv_topk_tokens": [P, P, P, I, P, P, P, P],
        "segkv_ffn_workspace_size": [I, I, I, P],
        "segkv_export": [P, I, I, P, SZ, P, P],
        "segkv_import": [P, I, I, P, SZ, P, P],
        "segkv_plan_decode": [P, I, I, P, P, I, I, P, I, P, I, P, P],
        "segkv_plan_prefill": [P, I, P, P, P, I, I, P, I, P, P],
        "segkv_plan_mass": [P, I, P, P, P, I, I, P, I, P, I, P, P],
        "segkv_exp2_check": [P, P, P, I, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_char_p if name == "segkv_last_error" else ctypes.c_int
    return lib


_lib = _load()


class SegKVError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"segkv error {code}: {msg}")
        self.code = code


def _ptr(t):
    """Device/host pointer of a tensor or numpy array (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _host_i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _stream_ptr(stream):
    if stream is None:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- C entry points, same names -------------------------------------------------

def segkv_create(num_layers, num_q_heads, num_kv_heads, head_dim, head_class, window, page_size,
                 max_seqs, max_seq_len, k_pool, v_pool, num_pages, softmax_scale=0.0):
    """Returns (status, handle)."""
    hc = np.ascontiguousarray(np.asarray(head_class, dtype=np.uint8).reshape(-1))
    win = _host_i32(window)
    h = ctypes.c_void_p()
    rc = _lib.segkv_create(ctypes.byref(h), num_layers, num_q_heads, num_kv_heads, head_dim,
                           hc.ctypes.data, win.ctypes.data, page_size, max_seqs, max_seq_len,
                           _ptr(k_pool), _ptr(v_pool), int(num_pages), float(softmax_scale))
    return rc, h


def segkv_destroy(h):
    return _lib.segkv_destroy(h)


def segkv_append(h, layer, k, v, cu_seqlens, seq_ids, stream=None):
    cu, ids = _host_i32(cu_seqlens), _host_i32(seq_ids)
    return _lib.segkv_append(h, layer, _ptr(k), _ptr(v), cu.ctypes.data, ids.ctypes.data, len(ids),
                             _stream_ptr(stream))


def segkv_prefill_attn(h, layer, q, cu_seqlens, q_pos, seq_ids, o, lse=None, workspace=None,
                       workspace_bytes=0, stream=None):
    cu, qp, ids = _host_i32(cu_seqlens), _host_i32(q_pos), _host_i32(seq_ids)
    return _lib.segkv_prefill_attn(h, layer, _ptr(q), cu.ctypes.data, qp.ctypes.data,
                                   ids.ctypes.data, len(ids), _ptr(o), _ptr(lse), _ptr(workspace),
                                   workspace_bytes, _stream_ptr(stream))


def segkv_decode_attn(h, layer, q, seq_lens, seq_ids, o, workspace, workspace_bytes=None,
                      stream=None):
    sl, ids = _host_i32(seq_lens), _host_i32(seq_ids)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return _lib.segkv_decode_attn(h, layer, _ptr(q), sl.ctypes.data, ids.ctypes.data, len(ids),
                                  _ptr(o), _ptr(workspace), workspace_bytes, _stream_ptr(stream))


def segkv_decode_attn_noalloc(h, layer, q, seq_lens, seq_ids, o, stream=None):
    """Decode with the library's fixed scratch instead of a workspace, for
    callers that cannot allocate when they decode."""
    sl, ids = _host_i32(seq_lens), _host_i32(seq_ids)
    return _lib.segkv_decode_attn_noalloc(h, layer, _ptr(q), sl.ctypes.data, ids.ctypes.data,
                                          len(ids), _ptr(o), _stream_ptr(stream))


def segkv_rope_shift(h, layer, seq, delta, base, rotary_dim, style, head_mask=(1 << 64) - 1,
                     stream=None):
    return _lib.segkv_rope_shift(h, layer, seq, int(delta), float(base), rotary_dim, style,
                                 head_mask, _stream_ptr(stream))


def segkv_export_size(h, layer, seq):
    b = ctypes.c_size_t()
    rc = _lib.segkv_export_size(h, layer, seq, ctypes.byref(b))
    return rc, b.value


def segkv_export(h, layer, seq, out, header, stream=None):
    """header: host int32 numpy array of length 1 + Hkv, filled by the call."""
    nbytes = 0 if out is None else out.numel() * out.element_size()
    return _lib.segkv_export(h, layer, seq, _ptr(out), nbytes, header.ctypes.data,
                             _stream_ptr(stream))


def segkv_import(h, layer, seq, src, header, stream=None):
    hd = _host_i32(header)
    nbytes = 0 if src is None else src.numel() * src.element_size()
    return _lib.segkv_import(h, layer, seq, _ptr(src), nbytes, hd.ctypes.data, _stream_ptr(stream))


def segkv_set_window_convention(h, convention):
    return _lib.segkv_set_window_convention(h, convention)


def segkv_decode_attn_multi(h, layer, q, T, seq_lens, seq_ids, o, lse=None, workspace=None,
                            workspace_bytes=None, stream=None):
    sl, ids = _host_i32(seq_lens), _host_i32(seq_ids)
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _lib.segkv_decode_attn_multi(h, layer, _ptr(q), T, sl.ctypes.data, ids.ctypes.data,
                                        len(ids), _ptr(o), _ptr(lse), _ptr(workspace),
                                        workspace_bytes, _stream_ptr(stream))


def segkv_attn_mass(h, layer, q, cu_seqlens, q_pos, seq_ids, lse, mass, stream=None):
    cu, qp, ids = _host_i32(cu_seqlens), _host_i32(q_pos), _host_i32(seq_ids)
    return _lib.segkv_attn_mass(h, layer, _ptr(q), cu.ctypes.data, qp.ctypes.data, ids.ctypes.data,
                                len(ids), _ptr(lse), _ptr(mass), _stream_ptr(stream))


def segkv_topk_tokens(h, mass, cu_seqlens, k, score, idx, stream=None):
    cu, kk = _host_i32(cu_seqlens), _host_i32(k)
    return _lib.segkv_topk_tokens(h, _ptr(mass), cu.ctypes.data, len(kk), kk.ctypes.data,
                                  _ptr(score), _ptr(idx), _stream_ptr(stream))


def segkv_ffn_workspace_size(m, d_model, d_ff):
    b = ctypes.c_size_t(0)
    rc = _lib.segkv_ffn_workspace_size(m, d_model, d_ff, ctypes.byref(b))
    return rc, b.value


def segkv_sparse_ffn(h, x, residual, idx, m, w_gate, w_up, w_down, workspace,
                     workspace_bytes=None, stream=None):
    """residual[idx[r]] += SwiGLU FFN(x[idx[r]]) for r < m (idx None: every row)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    n_rows, d_model = x.shape
    d_ff = w_gate.shape[0]
    return _lib.segkv_sparse_ffn(h, _ptr(x), _ptr(residual), n_rows, _ptr(idx), m, _ptr(w_gate),
                                 _ptr(w_up), _ptr(w_down), d_model, d_ff, _ptr(workspace),
                                 workspace_bytes, _stream_ptr(stream))


def segkv_trim(h, layer, seq_ids):
    ids = _host_i32(seq_ids)
    return _lib.segkv_trim(h, layer, ids.ctypes.data, len(ids))


def segkv_free_seq(h, seq_id):
    return _lib.segkv_free_seq(h, seq_id)


def segkv_workspace_size(h, kind, n_tokens, n_seqs):
    b = ctypes.c_size_t()
    rc = _lib.segkv_workspace_size(h, kind, n_tokens, n_seqs, ctypes.byref(b))
    return rc, b.value


def segkv_get_segment(h, layer, head, seq, max_ids=1 << 20):
    s, n, f, c = (ctypes.c_int32() for _ in range(4))
    ids = np.zeros(max_ids, dtype=np.int32)
    rc = _lib.segkv_get_segment(h, layer, head, seq, ctypes.byref(s), ctypes.byref(n),
                                ctypes.byref(f), ids.ctypes.data, max_ids, ctypes.byref(c))
    return rc, (s.value, n.value, f.value, ids[:c.value].tolist())


def segkv_seq_len(h, layer, seq):
    n = ctypes.c_int32()
    rc = _lib.segkv_seq_len(h, layer, seq, ctypes.byref(n))
    return rc, n.value


def segkv_stats(h):
    st = SegKVStats()
    rc = _lib.segkv_stats(h, ctypes.byref(st))
    return rc, {f: getattr(st, f) for f, _ in SegKVStats._fields_}


def segkv_status(h, stream=None):
    return _lib.segkv_status(h, _stream_ptr(stream))


def segkv_last_error(h=None):
    m = _lib.segkv_last_error(h)
    return m.decode() if m else ""


def segkv_exp2_check(x, y_poly, y_mufu, stream=None):
    """The softmax's two base-2 exponentials over device fp32 x (test hook):
    the FMA-pipe cubic into y_poly, the hardware ex2 into y_mufu."""
    return _lib.segkv_exp2_check(_ptr(x), _ptr(y_poly), _ptr(y_mufu), int(x.numel()),
                                 _stream_ptr(stream))


def segkv_plan_decode(h, layer, T, seq_lens, seq_ids, num_ctas=0):
    """The decode work plan (host only). Returns (rc, units [n_units, 8] int32,
    cta_begin [n_ctas + 1] int32); unit columns: sequence index, KV head,
    local, k0, k1, first unit of its pair, units of its pair, newest query
    position."""
    sl, ids = _host_i32(seq_lens), _host_i32(seq_ids)
    nu, nc = ctypes.c_int(0), ctypes.c_int(0)
    rc = _lib.segkv_plan_decode(h, layer, T, sl.ctypes.data, ids.ctypes.data, len(ids), num_ctas, None,
                                0, None, 0, ctypes.byref(nu), ctypes.byref(nc))
    if len(ids) == 0 or (rc != 0 and nu.value == 0):
        return rc, np.zeros((0, 8), np.int32), np.zeros(1, np.int32)
    units = np.zeros((nu.value, 8), np.int32)
    cta = np.zeros(nc.value + 1, np.int32)
    rc = _lib.segkv_plan_decode(h, layer, T, sl.ctypes.data, ids.ctypes.data, len(ids), num_ctas,
                                units.ctypes.data, nu.value, cta.ctypes.data, nc.value, ctypes.byref(nu),
                                ctypes.byref(nc))
    return rc, units, cta


def segkv_plan_prefill(h, layer, cu_seqlens, q_pos, seq_ids, num_ctas=0):
    """The prefill work plan (host only). Returns (rc, units [n_units, 8] int32
    in claim order, n_ctas); unit columns: first token, tokens, KV head, local,
    kt0, kt1, lowest and highest key seen. CTA c runs unit c first and then
    claims the next unclaimed unit each time it finishes one."""
    cu, qp, ids = _host_i32(cu_seqlens), _host_i32(q_pos), _host_i32(seq_ids)
    nu, nc = ctypes.c_int(0), ctypes.c_int(0)
    rc = _lib.segkv_plan_prefill(h, layer, cu.ctypes.data, qp.ctypes.data, ids.ctypes.data, len(ids),
                                 num_ctas, None, 0, ctypes.byref(nu), ctypes.byref(nc))
    if len(ids) == 0 or (rc != 0 and nu.value == 0):
        return rc, np.zeros((0, 8), np.int32), 0
    units = np.zeros((nu.value, 8), np.int32)
    rc = _lib.segkv_plan_prefill(h, layer, cu.ctypes.data, qp.ctypes.data, ids.ctypes.data, len(ids),
                                 num_ctas, units.ctypes.data, nu.value, ctypes.byref(nu), ctypes.byref(nc))
    return rc, units, nc.value


def segkv_plan_mass(h, layer, cu_seqlens, q_pos, seq_ids, num_ctas=0):
    """The attention-mass work plan (host only). Returns (rc, units [n_units, 12]
    int32, cta_begin [n_ctas + 1] int32); unit columns: first token, chunk
    length, first position, KV head, local, key tile, qt0, qt1, piece, pieces,
    first partial slot, key-tile counter."""
    cu, qp, ids = _host_i32(cu_seqlens), _host_i32(q_pos), _host_i32(seq_ids)
    nu, nc = ctypes.c_int(0), ctypes.c_int(0)
    rc = _lib.segkv_plan_mass(h, layer, cu.ctypes.data, qp.ctypes.data, ids.ctypes.data, len(ids),
                              num_ctas, None, 0, None, 0, ctypes.byref(nu), ctypes.byref(nc))
    if len(ids) == 0 or (rc != 0 and nu.value == 0):
        return rc, np.zeros((0, 12), np.int32), np.zeros(1, np.int32)
    units = np.zeros((nu.value, 12), np.int32)
    cta = np.zeros(nc.value + 1, np.int32)
    rc = _lib.segkv_plan_mass(h, layer, cu.ctypes.data, qp.ctypes.data, ids.ctypes.data, len(ids),
                              num_ctas, units.ctypes.data, nu.value, cta.ctypes.data, nc.value,
                              ctypes.byref(nu), ctypes.byref(nc))
    return rc, units, cta


def segkv_set_debug(h, flags):
    return _lib.segkv_set_debug(h, flags)


# ---- convenience wrapper -----------------------------------------------------------

class SegKV:
    """A segment-table handle over caller-owned K/V page pools.

    Pools are bf16 [num_pages, page_size, head_dim] each; pass none for a
    host-only handle (page tables only, no kernels).
    """

    def __init__(self, num_layers, num_q_heads, num_kv_heads, head_dim, head_class, window,
                 page_size, max_seqs, max_seq_len, k_pool=None, v_pool=None, num_pages=None,
                 softmax_scale=0.0):
        if num_pages is None:
            if k_pool is None:
                raise ValueError("num_pages is required for a host-only handle")
            num_pages = k_pool.shape[0]
        self.k_pool, self.v_pool = k_pool, v_pool
        self.num_layers, self.hq, self.hkv, self.head_dim = (num_layers, num_q_heads,
                                                             num_kv_heads, head_dim)
        self.page_size, self.num_pages = page_size, num_pages
        rc, h = segkv_create(num_layers, num_q_heads, num_kv_heads, head_dim, head_class, window,
                             page_size, max_seqs, max_seq_len, k_pool, v_pool, num_pages,
                             softmax_scale)
        if rc != SEGKV_OK:
            raise SegKVError(rc, segkv_last_error(None))
        self._h = h

    def _check(self, rc):
        if rc != SEGKV_OK:
            raise SegKVError(rc, segkv_last_error(self._h))
        return rc

    def close(self):
        if getattr(self, "_h", None):
            segkv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def append(self, layer, k, v, cu_seqlens, seq_ids, stream=None):
        return self._check(segkv_append(self._h, layer, k, v, cu_seqlens, seq_ids, stream))

    def prefill_attn(self, layer, q, cu_seqlens, q_pos, seq_ids, o, lse=None, stream=None):
        return self._check(segkv_prefill_attn(self._h, layer, q, cu_seqlens, q_pos, seq_ids, o,
                                              lse, None, 0, stream))

    def workspace_size(self, kind, n_tokens, n_seqs):
        rc, b = segkv_workspace_size(self._h, kind, n_tokens, n_seqs)
        self._check(rc)
        return b

    def decode_attn(self, layer, q, seq_lens, seq_ids, o, workspace, stream=None):
        return self._check(segkv_decode_attn(self._h, layer, q, seq_lens, seq_ids, o, workspace,
                                             None, stream))

    def decode_attn_noalloc(self, layer, q, seq_lens, seq_ids, o, stream=None):
        return self._check(segkv_decode_attn_noalloc(self._h, layer, q, seq_lens, seq_ids, o,
                                                     stream))

    def rope_shift(self, layer, seq, delta, base=10000.0, rotary_dim=None, style=SEGKV_ROPE_HALF,
                   head_mask=(1 << 64) - 1, stream=None):
        rd = self.head_dim if rotary_dim is None else rotary_dim
        return self._check(segkv_rope_shift(self._h, layer, seq, delta, base, rd, style, head_mask,
                                            stream))

    def export_segment(self, layer, seq, stream=None):
        """Returns (buffer, header): the kept K/V rows packed for transfer."""
        import torch
        rc, nbytes = segkv_export_size(self._h, layer, seq)
        self._check(rc)
        header = np.zeros(1 + self.hkv, dtype=np.int32)
        dev = self.k_pool.device if self.k_pool is not None else "cpu"
        buf = torch.empty(max(nbytes // 2, 8), dtype=torch.bfloat16, device=dev)
        self._check(segkv_export(self._h, layer, seq, buf if self.k_pool is not None else None,
                                 header, stream))
        return buf[: nbytes // 2], header

    def import_segment(self, layer, seq, buf, header, stream=None):
        return self._check(segkv_import(self._h, layer, seq, buf, header, stream))

    def set_window_convention(self, convention):
        return self._check(segkv_set_window_convention(self._h, convention))

    def decode_attn_multi(self, layer, q, T, seq_lens, seq_ids, o, lse=None, workspace=None,
                          stream=None):
        return self._check(segkv_decode_attn_multi(self._h, layer, q, T, seq_lens, seq_ids, o, lse,
                                                   workspace, None, stream))

    def attn_mass(self, layer, q, cu_seqlens, q_pos, seq_ids, lse, mass, stream=None):
        return self._check(segkv_attn_mass(self._h, layer, q, cu_seqlens, q_pos, seq_ids, lse,
                                           mass, stream))

    def topk_tokens(self, mass, cu_seqlens, k, score, idx, stream=None):
        return self._check(segkv_topk_tokens(self._h, mass, cu_seqlens, k, score, idx, stream))

    def sparse_ffn(self, x, residual, idx, w_gate, w_up, w_down, workspace=None, stream=None):
        """residual[idx] += SwiGLU FFN(x[idx]) (idx None: every row). Allocates
        the workspace when none is given."""
        m = x.shape[0] if idx is None else idx.numel()
        if workspace is None:
            rc, b = segkv_ffn_workspace_size(m, x.shape[1], w_gate.shape[0])
            self._check(rc)
            import torch
            workspace = torch.empty(b, dtype=torch.uint8, device=x.device)
        return self._check(segkv_sparse_ffn(self._h, x, residual, idx, m, w_gate, w_up, w_down,
                                            workspace, None, stream))

    def trim(self, layer, seq_ids):
        return self._check(segkv_trim(self._h, layer, seq_ids))

    def free_seq(self, seq):
        return self._check(segkv_free_seq(self._h, seq))

    def segment(self, layer, head, seq):
        rc, seg = segkv_get_segment(self._h, layer, head, seq)
        self._check(rc)
        return seg

    def seq_len(self, layer, seq):
        rc, n = segkv_seq_len(self._h, layer, seq)
        self._check(rc)
        return n

    def stats(self):
        rc, st = segkv_stats(self._h)
        self._check(rc)
        return st

    def status(self, stream=None):
        return segkv_status(self._h, stream)

    def set_debug(self, flags):
        return self._check(segkv_set_debug(self._h, flags))
