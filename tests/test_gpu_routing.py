"""Sparse FFN routing through the C ABI: attention mass per token, top-k
token choice, and the routed FFN, against the oracle.

Mass tolerance, derived from the arithmetic: scores are fp32 dot products of
exact bf16 inputs; the LSE comes from the prefill kernel, whose softmax
denominator has relative error below 7.5e-5 (the polynomial exp2 at D=64; far
less at D=128) plus fp32 summation; exp2 on the MUFU unit is within 2^-22;
the per-key sums are fp32. Each mass is within 2e-4 relative of the fp64
oracle, plus 1e-6 absolute for keys whose mass underflows.
The top-k choice is an integer decision: it is compared bit for bit with the
oracle's choice taken on the same fp32 scores.
"""
import numpy as np
import pytest
import torch

import head_segmented_paged_gb300 as S
from head_segmented_paged_gb300 import inputs as I
import oracle
from harness import Cache, oracle_mass
from oracle import sparse_ffn as F

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-4, 1e-6


def chunk_mass(c, layer, q, cu, qp, ids):
    """Prefill the chunk (for its LSE) and compute its mass on the GPU."""
    tot = int(cu[-1])
    o = torch.empty((tot, c.hq, c.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((c.hq, tot), dtype=torch.float32, device="cuda")
    qd = q.cuda()
    assert S.segkv_prefill_attn(c.h.handle, layer, qd, cu, qp, ids, o, lse) == 0
    mass = torch.full((c.hkv, tot), float("nan"), dtype=torch.float32, device="cuda")
    c.h.attn_mass(layer, qd, cu, qp, ids, lse, mass)
    assert c.h.status() == 0
    return mass.cpu().numpy()


def check_mass(c, layer, q, cu, qp, ids, got):
    seq_index = np.repeat(np.arange(len(ids)), np.diff(cu)).astype(np.int32)
    rc, ref, offs = oracle_mass(c, layer, q, ids, seq_index, np.asarray(qp, np.int32))
    assert rc == 0
    for i, b in enumerate(ids):
        t0, t1 = int(cu[i]), int(cu[i + 1])
        if t1 == t0:
            continue
        a = int(qp[t0])
        want = ref[:, offs[i] + a: offs[i] + a + (t1 - t0)]
        g = got[:, t0:t1]
        assert np.isfinite(g).all()
        bad = np.abs(g - want) > RTOL * np.abs(want) + ATOL
        assert not bad.any(), (b, np.argwhere(bad)[:5], g[bad][:5], want[bad][:5])


@pytest.mark.parametrize("G,d,P,W,lens", [(4, 64, 16, 32, [256]),
                                          (4, 128, 64, 100, [700, 130, 1]),
                                          (8, 128, 32, 64, [300, 257]),
                                          (1, 64, 16, 40, [200])])
def test_mass_whole_prefill_matches_oracle(G, d, P, W, lens):
    hkv = 2
    hq = hkv * G
    tot = sum(lens)
    q = I.normal_bf16(71, 1, (tot, hq, d))
    k = I.normal_bf16(71, 2, (tot, hkv, d))
    v = I.normal_bf16(71, 3, (tot, hkv, d))
    pages = sum((n + P - 1) // P for n in lens) * hkv + 4
    c = Cache(1, hq, hkv, d, [[I.GLOBAL, I.LOCAL]], [W], P, len(lens), max(lens), pages)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ids = list(range(len(lens)))
    assert c.append(0, k.cuda(), v.cuda(), cu, ids) == 0
    qp = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    got = chunk_mass(c, 0, q, cu, qp, ids)
    check_mass(c, 0, q, cu, qp, ids, got)
    # each query's probabilities sum to one and all its keys are in the chunk
    np.testing.assert_allclose(got.sum(axis=1), G * tot, rtol=1e-4)
    # fixed summation order: a second call repeats every bit
    again = chunk_mass(c, 0, q, cu, qp, ids)
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))


def test_mass_second_chunk_sees_cached_keys():
    # chunk 2 starts at position 300: its queries also attend to cached keys
    # (changing their softmax), but only chunk keys receive a mass entry
    hkv, G, d, P, W = 2, 4, 128, 64, 96
    c = Cache(1, hkv * G, hkv, d, [[I.LOCAL, I.GLOBAL]], [W], P, 1, 1024, 40)
    k1 = I.normal_bf16(72, 1, (300, hkv, d))
    assert c.append(0, k1.cuda(), k1.cuda(), [0, 300], [0]) == 0
    k2 = I.normal_bf16(72, 2, (230, hkv, d))
    assert c.append(0, k2.cuda(), k2.cuda(), [0, 230], [0]) == 0
    q = I.normal_bf16(72, 3, (230, hkv * G, d))
    cu = np.array([0, 230], np.int32)
    qp = np.arange(300, 530, dtype=np.int32)
    got = chunk_mass(c, 0, q, cu, qp, [0])
    check_mass(c, 0, q, cu, qp, [0], got)


def test_mass_refuses_non_consecutive_positions():
    hkv, G, d, P, W = 2, 4, 64, 16, 32
    c = Cache(1, hkv * G, hkv, d, [[I.GLOBAL, I.LOCAL]], [W], P, 1, 256, 40)
    k = I.normal_bf16(73, 1, (100, hkv, d))
    assert c.append(0, k.cuda(), k.cuda(), [0, 100], [0]) == 0
    q = torch.zeros((3, hkv * G, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((hkv * G, 3), device="cuda")
    mass = torch.zeros((hkv, 3), device="cuda")
    rc = S.segkv_attn_mass(c.h.handle, 0, q, [0, 3], [5, 7, 8], [0], lse, mass)
    assert rc == S.SEGKV_ERR_INVALID_ARG


def run_topk(h, mass_np, cu, k):
    tot = mass_np.shape[1]
    mass = torch.tensor(mass_np, device="cuda")
    score = torch.full((tot,), float("nan"), device="cuda")
    idx = torch.full((max(1, sum(k)),), -1, dtype=torch.int32, device="cuda")
    h.topk_tokens(mass, cu, k, score, idx)
    assert h.status() == 0
    return score.cpu().numpy(), idx.cpu().numpy()[:sum(k)]


def fp32_score(mass_np):
    s = mass_np[0].astype(np.float32).copy()
    for hh in range(1, mass_np.shape[0]):
        s = (s + mass_np[hh]).astype(np.float32)
    return s


@pytest.mark.parametrize("lens,ks,levels", [([1000], [250], 7), ([1], [1], 3),
                                            ([50, 0, 300, 17], [50, 0, 1, 0], 4),
                                            ([100000], [25000], 1000), ([4096, 513], [0, 513], 2),
                                            ([20000], [7], 5)])
def test_topk_matches_oracle_bit_for_bit(lens, ks, levels):
    kp = torch.empty((8, 16, 64), dtype=torch.bfloat16, device="cuda")
    h = S.SegKV(1, 8, 2, 64, [[0, 1]], [32], 16, 1, 64, kp, kp.clone())
    rng = np.random.default_rng(sum(lens) + levels)
    tot = sum(lens)
    # few distinct values per head, so the summed scores tie often
    mass = (rng.integers(0, levels, (2, tot)) * 0.375).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    score, idx = run_topk(h, mass, cu, ks)
    want_score = fp32_score(mass)
    assert np.array_equal(score.view(np.uint32), want_score.view(np.uint32))
    off = 0
    for i, kk in enumerate(ks):
        want = F.topk_tokens(want_score[cu[i]:cu[i + 1]].astype(np.float64), kk) + cu[i]
        assert np.array_equal(idx[off:off + kk], want), (i, idx[off:off + kk][:10], want[:10])
        off += kk


def score_tolerance(ref_mass):
    """Per-token bound on |GPU score - fp64 score|: the per-head mass bound
    summed over the KV heads, plus fp32 rounding of that sum."""
    return (RTOL * np.abs(ref_mass) + ATOL).sum(axis=0) + 2.0 ** -22 * ref_mass.sum(axis=0)


def check_valid_topk(idx, ref_score, tol, k):
    """idx must be a valid top-k of the fp64 scores within the tolerance:
    k distinct positions, and no unchosen token's score exceeds a chosen
    token's by more than both tolerances (several sets are correct where
    scores sit within the tolerance of the k-th largest)."""
    n = ref_score.shape[0]
    assert idx.shape == (k,) and len(np.unique(idx)) == k
    assert ((0 <= idx) & (idx < n)).all() and (np.diff(idx) > 0).all()
    chosen = np.zeros(n, bool)
    chosen[idx] = True
    if 0 < k < n:
        lo = (ref_score[chosen] + tol[chosen]).min()
        hi = (ref_score[~chosen] - tol[~chosen]).max()
        assert lo >= hi, (lo, hi)
    return chosen


def test_routing_end_to_end():
    # chunk -> prefill (LSE) -> mass -> top-k -> FFN on the chosen rows
    hkv, G, d, P, W = 2, 4, 128, 64, 128
    n, dm, dff, kk = 640, 256, 512, 160
    c = Cache(1, hkv * G, hkv, d, [[I.GLOBAL, I.LOCAL]], [W], P, 1, 1024, 40)
    k = I.normal_bf16(74, 1, (n, hkv, d))
    assert c.append(0, k.cuda(), k.cuda(), [0, n], [0]) == 0
    q = I.normal_bf16(74, 2, (n, hkv * G, d))
    cu = np.array([0, n], np.int32)
    qp = np.arange(n, dtype=np.int32)
    mass = chunk_mass(c, 0, q, cu, qp, [0])
    check_mass(c, 0, q, cu, qp, [0], mass)
    score, idx = run_topk(c.h, mass, cu, [kk])
    # stage check: the choice on the GPU's own fp32 scores, bit for bit
    assert np.array_equal(idx, F.topk_tokens(fp32_score(mass).astype(np.float64), kk))
    # end to end: the choice is a valid top-k of the oracle's fp64 scores
    rc, ref_mass, _ = oracle_mass(c, 0, q, [0], np.zeros(n, np.int32), qp)
    assert rc == 0
    ref_score = ref_mass.sum(axis=0)
    check_valid_topk(idx, ref_score, score_tolerance(ref_mass), kk)
    sel_ref = F.topk_tokens(ref_score, kk)  # the oracle's own choice
    w = I.FfnWorkload("t", n, dm, dff, kk, 5)
    x, r, wg, wu, wd = I.ffn_tensors(w, device="cuda")
    out = r.clone()
    c.h.sparse_ffn(x, out, torch.tensor(idx, dtype=torch.int32, device="cuda"), wg, wu, wd)
    assert c.h.status() == 0
    host = [t.to(torch.float64).cpu().numpy() for t in (x, r, wg, wu, wd)]
    got = out.to(torch.float64).cpu().numpy()
    sig_w = host[4] ** 2

    def check_rows(rows, ref, hh_rows):
        sig = 2.0 ** -8 / np.sqrt(3) * np.sqrt((hh_rows ** 2) @ sig_w.T)
        err = np.abs(got[rows] - ref[rows])
        assert (err <= 2.0 ** -8 * np.abs(ref[rows]) + 6 * sig + 1e-3).all()

    # the oracle FFN on the oracle's own choice, on every row both choose
    ref_o, hh_o = F.sparse_ffn(host[0], host[1], sel_ref, *host[2:])
    both = np.intersect1d(idx, sel_ref)
    check_rows(both, ref_o, hh_o[np.searchsorted(sel_ref, both)])
    # rows where the two valid choices differ: the oracle FFN on the GPU's set
    ref_g, hh_g = F.sparse_ffn(host[0], host[1], idx, *host[2:])
    only = np.setdiff1d(idx, sel_ref)
    check_rows(only, ref_g, hh_g[np.searchsorted(idx, only)])
    rest = np.setdiff1d(np.arange(n), idx)
    assert np.array_equal(got[rest], host[1][rest])  # residual identity, bit for bit


def test_mass_mistral_8k_conserves_probability():
    # full-size chunk (8192 tokens, 32/8 heads): every query's probabilities
    # sum to one, so each KV head's masses add up to G x 8192
    w = I.mistral_8k()
    q, k, v, cu, qp = I.prefill_tensors(w, 0, device="cuda")
    P = w.page_size
    pages = (w.seq_lens[0] // P + 2) * w.hkv
    kp = torch.empty((pages, P, w.head_dim), dtype=torch.bfloat16, device="cuda")
    h = S.SegKV(1, w.hq, w.hkv, w.head_dim, w.head_class, w.window, P, 1, w.seq_lens[0], kp,
                torch.empty_like(kp))
    h.append(0, k, v, cu, [0])
    n = w.seq_lens[0]
    o = torch.empty((n, w.hq, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.hq, n), device="cuda")
    h.prefill_attn(0, q, cu, qp, [0], o, lse)
    mass = torch.empty((w.hkv, n), device="cuda")
    h.attn_mass(0, q, cu, qp, [0], lse, mass)
    assert h.status() == 0
    m = mass.cpu().numpy().astype(np.float64)
    assert (m >= 0).all()
    np.testing.assert_allclose(m.sum(axis=1), w.group * n, rtol=1e-4)
    # element by element against the oracle's fp64 mass, every key
    rc, ref = oracle.attn_mass(q.cpu(), k.cpu(), np.zeros(n, np.int32), qp.numpy(), [0], [n],
                               w.head_class[0], w.window[0], np.zeros((1, w.hkv), np.int32))
    assert rc == 0
    bad = np.abs(m - ref) > RTOL * np.abs(ref) + ATOL
    assert not bad.any(), (np.argwhere(bad)[:5], m[bad][:5], ref[bad][:5])
    # the top-k of a quarter of the chunk is a valid top-k of the fp64 scores
    kk = n // 4
    score = torch.empty((n,), device="cuda")
    idx = torch.empty((kk,), dtype=torch.int32, device="cuda")
    h.topk_tokens(mass, cu, [kk], score, idx)
    assert h.status() == 0
    check_valid_topk(idx.cpu().numpy().astype(np.int64), ref.sum(axis=0), score_tolerance(ref), kk)
