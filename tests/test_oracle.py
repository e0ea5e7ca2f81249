"""Pins for the oracle's attention, independent of the oracle itself.

Each check ties the oracle to something outside it: a dense masked attention
written separately (an explicit L x L boolean mask and a masked softmax, the
layout the RedKnot summary page, section "3. 算法上省了字节，工程上没省算力",
says the method removes while computing the same thing), closed forms, and the
split invariance behind the online-softmax merge (KV-cache architecture page,
section 5.2).
"""
import numpy as np
import pytest
import torch

import oracle
from head_segmented_paged_gb300 import inputs as I


def dense_masked(q, k, v, mask, scale):
    """Brute force: [L, D] per head pair with an explicit boolean mask [L, L]."""
    s = scale * (q @ k.T)
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    z = p.sum(axis=1, keepdims=True)
    return (p / z) @ v, (m + np.log(z))[:, 0]


def make_mask(L, local, W):
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    m = j <= i
    if local:
        m &= j >= i - W + 1
    return m


def run_single_seq(q, k, v, head_class, W, seg_start=None, block=None):
    L = q.shape[0]
    hkv = k.shape[1]
    ss = np.zeros((1, hkv), np.int32) if seg_start is None else seg_start
    return oracle.attention(q, k, v, np.zeros(L, np.int32), np.arange(L, dtype=np.int32), [0], [L],
                            head_class, W, ss, block=block)


def as64(t):
    return t.to(torch.float64).numpy()


@pytest.fixture(scope="module")
def tiny():
    w = I.tiny_256()
    q, k, v, cu, qp = I.prefill_tensors(w)
    return w, q, k, v


def test_tiny_matches_dense_masked_bruteforce(tiny):
    w, q, k, v = tiny
    rc, o, lse = run_single_seq(q, k, v, w.head_class[0], w.window[0])
    assert rc == oracle.OK
    G = w.group
    scale = 1 / np.sqrt(w.head_dim)
    for hq in range(w.hq):
        h = hq // G
        mask = make_mask(256, w.head_class[0][h] == I.LOCAL, w.window[0])
        ref, rl = dense_masked(as64(q[:, hq]), as64(k[:, h]), as64(v[:, h]), mask, scale)
        np.testing.assert_allclose(o[:, hq], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, hq], rl, rtol=0, atol=1e-12)


def test_global_head_is_dense_causal(tiny):
    w, q, k, v = tiny
    rc, o, _ = run_single_seq(q, k, v, [I.GLOBAL, I.GLOBAL], 32)
    assert rc == oracle.OK
    scale = 1 / np.sqrt(64)
    for hq in range(8):
        h = hq // 4
        ref, _ = dense_masked(as64(q[:, hq]), as64(k[:, h]), as64(v[:, h]),
                              make_mask(256, False, 0), scale)
        np.testing.assert_allclose(o[:, hq], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("W", [256, 257, 10000])
def test_local_head_with_window_ge_L_is_dense_causal(tiny, W):
    w, q, k, v = tiny
    rc_g, og, _ = run_single_seq(q, k, v, [I.GLOBAL, I.GLOBAL], W)
    rc_l, ol, _ = run_single_seq(q, k, v, [I.LOCAL, I.LOCAL], W)
    assert rc_g == rc_l == oracle.OK
    np.testing.assert_allclose(ol, og, rtol=0, atol=1e-13)


def test_window_one_returns_own_value(tiny):
    w, q, k, v = tiny
    rc, o, lse = run_single_seq(q, k, v, [I.LOCAL, I.LOCAL], 1)
    assert rc == oracle.OK
    for hq in range(8):
        np.testing.assert_array_equal(o[:, hq], as64(v[:, hq // 4]))
    # one key: lse is that key's scaled score
    sc = (as64(q[:, 0]) * as64(k[:, 0])).sum(1) / 8.0
    np.testing.assert_allclose(lse[:, 0], sc, rtol=0, atol=1e-12)


def test_constant_values_give_that_constant(tiny):
    w, q, k, _ = tiny
    v = torch.full_like(k, 0.375)
    rc, o, _ = run_single_seq(q, k, v, w.head_class[0], w.window[0])
    assert rc == oracle.OK
    np.testing.assert_allclose(o, 0.375, rtol=0, atol=1e-14)


@pytest.mark.parametrize("hc,W", [([I.GLOBAL, I.LOCAL], 32), ([I.LOCAL, I.LOCAL], 5)])
def test_identical_keys_average_visible_values(tiny, hc, W):
    w, q, _, v = tiny
    k = torch.zeros_like(v)
    k[:] = v[7:8]  # every key the same row
    rc, o, lse = run_single_seq(q, k, v, hc, W)
    assert rc == oracle.OK
    vv = as64(v)
    for hq in range(8):
        h = hq // 4
        local = hc[h] == I.LOCAL
        for p in (0, 1, 4, 5, 31, 32, 100, 255):
            lo = max(0, p - W + 1) if local else 0
            np.testing.assert_allclose(o[p, hq], vv[lo:p + 1, h].mean(0), rtol=0, atol=1e-12)
            cnt = p + 1 - lo
            sc = (as64(q[p, hq]) * as64(k[0, h])).sum() / 8.0
            assert abs(lse[p, hq] - (sc + np.log(cnt))) < 1e-12


@pytest.mark.parametrize("block", [1, 7, 16, 64, 1000])
def test_blocked_merge_equals_direct(tiny, block):
    w, q, k, v = tiny
    rc, o, lse = run_single_seq(q, k, v, w.head_class[0], w.window[0])
    rcb, ob, lseb = run_single_seq(q, k, v, w.head_class[0], w.window[0], block=block)
    assert rc == rcb == oracle.OK
    np.testing.assert_allclose(ob, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lseb, lse, rtol=0, atol=1e-12)


def test_sinks_and_scale_match_bruteforce():
    w = I.llama70b_varlen()
    w.seq_lens = [200, 77]
    w.sink_positions = [[0, 50], [3]]
    w.window = [16]
    q, k, v, cu, qp = I.prefill_tensors(w)
    hc = w.head_class[0]
    row_seq = np.repeat(np.arange(2), w.seq_lens)
    rc, o, _ = oracle.attention(q, k, v, row_seq, qp.numpy(), [0, 200], w.seq_lens, hc, 16,
                                np.zeros((2, 8), np.int32), scale=0.3)
    assert rc == oracle.OK
    for b, (off, L) in enumerate([(0, 200), (200, 77)]):
        for hq in (0, 9, 63):
            h = hq // 8
            ref, _ = dense_masked(as64(q[off:off + L, hq]), as64(k[off:off + L, h]),
                                  as64(v[off:off + L, h]), make_mask(L, hc[h] == I.LOCAL, 16), 0.3)
            np.testing.assert_allclose(o[off:off + L, hq], ref, rtol=0, atol=1e-12)


def test_evicted_and_out_of_range_queries_are_errors(tiny):
    w, q, k, v = tiny
    ss = np.array([[0, 200]], np.int32)  # local head keeps only from 200
    L = 256
    rows_ok = np.arange(231, 256)         # needs keys >= p-31 >= 200
    rc, _, _ = oracle.attention(q, k, v, np.zeros(L, np.int32), np.arange(L, dtype=np.int32),
                                [0], [L], w.head_class[0], 32, ss, rows=rows_ok)
    assert rc == oracle.OK
    rc, _, _ = oracle.attention(q, k, v, np.zeros(L, np.int32), np.arange(L, dtype=np.int32),
                                [0], [L], w.head_class[0], 32, ss, rows=[230])
    assert rc == oracle.EVICTED
    rc, _, _ = oracle.attention(q, k, v, np.zeros(L, np.int32), np.full(L, 256, np.int32),
                                [0], [L], w.head_class[0], 32, np.zeros((1, 2), np.int32), rows=[0])
    assert rc == oracle.INVALID_ARG


def test_kept_start_changes_nothing_while_needed_keys_are_kept(tiny):
    # Keys below the kept start are never visible to queries that are allowed.
    w, q, k, v = tiny
    L = 256
    rows = np.arange(240, 256)
    base = oracle.attention(q, k, v, np.zeros(L, np.int32), np.arange(L, dtype=np.int32), [0], [L],
                            w.head_class[0], 32, np.zeros((1, 2), np.int32), rows=rows)
    trimmed = oracle.attention(q, k, v, np.zeros(L, np.int32), np.arange(L, dtype=np.int32), [0],
                               [L], w.head_class[0], 32, np.array([[0, 209]], np.int32), rows=rows)
    assert base[0] == trimmed[0] == oracle.OK
    np.testing.assert_array_equal(base[1], trimmed[1])
