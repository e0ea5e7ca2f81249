"""Shared helpers for the GPU parity tests: build a segment cache through the
C ABI, mirror every call on the oracle's page model, and compare outputs with
the oracle's fp64 attention."""
from __future__ import annotations

import numpy as np
import torch

import head_segmented_paged_gb300 as S
import oracle
from head_segmented_paged_gb300 import inputs as I

# Output bar, as stated for the method: max-abs <= 1e-2 and mean-abs <= 1e-3
# of the bf16 GPU output against the fp64 oracle, element by element.
MAX_ABS = 1e-2
MEAN_ABS = 1e-3

# Every comparison's flat max-abs and mean-abs, in call order; the test
# session prints them at its end (tests/conftest.py).
RECORDS: list = []


def bf16_half_ulp(x):
    """Half a unit in the last place of bf16 (8 significant bits) at |x|:
    2^(floor(log2 |x|) - 8) for normal values."""
    a = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)


def check_close(o_gpu, o_ref, what="", output_rounding=False):
    """Assert the flat bar: max |o_gpu - o_ref| <= 1e-2, mean <= 1e-3.

    output_rounding=True is for a named case whose outputs reach |o| >= 4,
    where the bf16 half-ulp of the returned value alone (2^-6 from 4 on)
    exceeds 1e-2: each element may then also carry exactly the bf16
    half-ulp of its oracle value. No case uses it unless it names it."""
    g = o_gpu.detach().to("cpu", torch.float64).numpy() if torch.is_tensor(o_gpu) else \
        np.asarray(o_gpu, np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - o_ref)
    bound = MAX_ABS + (bf16_half_ulp(o_ref) if output_rounding else 0.0)
    mx, mean = float(err.max()), float(err.mean())
    RECORDS.append((what, mx, mean, err.size, output_rounding))
    worst = np.argmax(err - bound)
    assert (err <= bound).all(), (f"{what}: max err {mx:.3e} "
                                  f"at {np.unravel_index(worst, err.shape)}, ref "
                                  f"{o_ref.reshape(-1)[worst]:.4f}")
    assert mean <= MEAN_ABS, f"{what}: mean err {mean:.3e}"
    return mx, mean


class Cache:
    """A library handle with NaN-filled pools plus the oracle's mirror."""

    def __init__(self, num_layers, hq, hkv, d, head_class, window, page_size, max_seqs,
                 max_seq_len, num_pages, poison=True):
        fill = float("nan") if poison else 0.0
        self.kp = torch.full((num_pages, page_size, d), fill, dtype=torch.bfloat16, device="cuda")
        self.vp = torch.full((num_pages, page_size, d), fill, dtype=torch.bfloat16, device="cuda")
        self.h = S.SegKV(num_layers, hq, hkv, d, head_class, window, page_size, max_seqs,
                         max_seq_len, self.kp, self.vp)
        self.m = oracle.PageModel(num_layers, hkv, head_class, window, page_size, max_seqs,
                                  max_seq_len, num_pages)
        self.L, self.hq, self.hkv, self.d, self.P = num_layers, hq, hkv, d, page_size
        self.head_class, self.window = head_class, window
        self.max_seqs = max_seqs
        # logical K/V per (layer, seq), CPU bf16 [n, hkv, d]
        self.k_log = {}
        self.v_log = {}

    def append(self, layer, k, v, cu, seq_ids):
        rc_m = self.m.append(layer, cu, seq_ids)
        rc = S.segkv_append(self.h.handle, layer, k, v, cu, seq_ids)
        assert rc == rc_m, (rc, rc_m, S.segkv_last_error(self.h.handle))
        if rc == 0:
            kc, vc = k.cpu(), v.cpu()
            for i, b in enumerate(seq_ids):
                sl = slice(int(cu[i]), int(cu[i + 1]))
                key = (layer, b)
                self.k_log[key] = torch.cat([self.k_log.get(key, kc[:0]), kc[sl]])
                self.v_log[key] = torch.cat([self.v_log.get(key, vc[:0]), vc[sl]])
        return rc

    def trim(self, layer, seq_ids):
        assert self.m.trim(layer, seq_ids) == self.h.trim(layer, seq_ids) == 0

    def free_seq(self, b):
        assert self.m.free_seq(b) == 0
        self.h.free_seq(b)
        for l in range(self.L):
            self.k_log.pop((l, b), None)
            self.v_log.pop((l, b), None)

    def check_tables(self, layer):
        for b in range(self.max_seqs):
            for hd in range(self.hkv):
                assert self.h.segment(layer, hd, b) == self.m.segment(layer, hd, b), (layer, hd, b)

    def check_pages(self, layer, seqs):
        """Every kept key/value row, read back through the page table, equals
        the appended row bit for bit."""
        kp, vp = self.kp.cpu(), self.vp.cpu()
        for b in seqs:
            kl, vl = self.k_log[(layer, b)], self.v_log[(layer, b)]
            for hd in range(self.hkv):
                s, ln, first, ids = self.m.segment(layer, hd, b)
                if ln == 0:
                    continue
                pos = torch.arange(s, s + ln)
                pid = torch.tensor(ids)[pos // self.P - first]
                slot = pos % self.P
                assert torch.equal(kp[pid, slot].view(torch.int16), kl[pos, hd].view(torch.int16))
                assert torch.equal(vp[pid, slot].view(torch.int16), vl[pos, hd].view(torch.int16))

    def oracle_attention(self, layer, q, seq_ids, q_seq_index, q_pos, rows=None):
        """fp64 oracle over this cache's logical K/V and the model's kept starts."""
        ks, vs, offs, lens = [], [], [], []
        off = 0
        for b in seq_ids:
            kb = self.k_log[(layer, b)]
            ks.append(kb)
            vs.append(self.v_log[(layer, b)])
            offs.append(off)
            lens.append(kb.shape[0])
            off += kb.shape[0]
        seg_start = np.array([[self.m.segment(layer, hd, b)[0] for hd in range(self.hkv)]
                              for b in seq_ids], dtype=np.int32)
        return oracle.attention(q.cpu(), torch.cat(ks), torch.cat(vs), q_seq_index, q_pos, offs,
                                lens, self.head_class[layer], self.window[layer], seg_start,
                                rows=rows)


def prefill_case(w: I.Workload, layer=0, num_pages=None, poison=True, max_seq_len=None):
    """Append every sequence of a workload in one call; return cache and inputs."""
    q, k, v, cu, qp = I.prefill_tensors(w, layer)
    P = w.page_size
    need = sum((n + P - 1) // P for n in w.seq_lens) * w.hkv
    c = Cache(w.num_layers, w.hq, w.hkv, w.head_dim, w.head_class, w.window, P,
              len(w.seq_lens), max_seq_len or max(w.seq_lens), num_pages or need + 8,
              poison=poison)
    ids = list(range(len(w.seq_lens)))
    assert c.append(layer, k.cuda(), v.cuda(), cu, ids) == 0
    return c, q, cu, qp, ids


def oracle_mass(c: Cache, layer, q, seq_ids, q_seq_index, q_pos):
    """fp64 attention mass each logical key of the listed sequences receives
    from the query rows q (row i of sequence q_seq_index[i] at q_pos[i]):
    returns (status, mass [Hkv, sum of lengths], offsets per sequence)."""
    ks, offs, lens = [], [], []
    off = 0
    for b in seq_ids:
        kb = c.k_log[(layer, b)]
        ks.append(kb)
        offs.append(off)
        lens.append(kb.shape[0])
        off += kb.shape[0]
    seg_start = np.array([[c.m.segment(layer, hd, b)[0] for hd in range(c.hkv)]
                          for b in seq_ids], dtype=np.int32)
    rc, m = oracle.attn_mass(q.cpu(), torch.cat(ks), q_seq_index, q_pos, offs, lens,
                             c.head_class[layer], c.window[layer], seg_start)
    return rc, m, offs
