"""Pins of the sparse-FFN routing oracle (attention mass, top-k, SwiGLU FFN).

Each pin ties the oracle to something outside it: a separately written dense
masked-softmax computation, conservation of probability, closed forms for
identical keys and for W = 1, a threshold formulation of top-k, and a
hand-derived FFN example (tests/golden/sparse_ffn_example.json).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import sparse_ffn as F
from head_segmented_paged_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sparse_ffn_example.json")


def dense_mass(q, k, head_class, window, lens):
    """Column sums of the masked softmax matrices, built with an explicit
    boolean L x L mask per head (no key lists): [Hkv, sum lens]."""
    qd = q.to(torch.float64).numpy()
    kd = k.to(torch.float64).numpy()
    hq, hkv, d = qd.shape[1], kd.shape[1], qd.shape[2]
    G = hq // hkv
    out = np.zeros((hkv, kd.shape[0]))
    off = 0
    for n in lens:
        pos = np.arange(n)
        for qh in range(hq):
            h = qh // G
            mask = pos[None, :] <= pos[:, None]
            if head_class[h] != oracle.GLOBAL:
                mask &= pos[None, :] >= pos[:, None] - window + 1
            s = qd[off:off + n, qh] @ kd[off:off + n, h].T / math.sqrt(d)
            s = np.where(mask, s, -np.inf)
            s -= s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=1, keepdims=True)
            out[h, off:off + n] += p.sum(axis=0)
        off += n
    return out


def run_mass(q, k, head_class, window, lens):
    row_seq = np.concatenate([np.full(n, b) for b, n in enumerate(lens)])
    row_pos = np.concatenate([np.arange(n) for n in lens])
    off = np.concatenate([[0], np.cumsum(lens)[:-1]])
    rc, m = oracle.attn_mass(q, k, row_seq, row_pos, off, lens, head_class, window,
                             np.zeros((len(lens), k.shape[1]), np.int32))
    assert rc == 0
    return m


@pytest.mark.parametrize("lens,window", [([256], 32), ([70, 130], 16), ([40], 1)])
def test_mass_matches_dense_masked_softmax(lens, window):
    hq, hkv, d = 8, 2, 64
    tot = sum(lens)
    q = I.normal_bf16(61, 1, (tot, hq, d))
    k = I.normal_bf16(61, 2, (tot, hkv, d))
    hc = [oracle.GLOBAL, oracle.LOCAL]
    got = run_mass(q, k, hc, window, lens)
    np.testing.assert_allclose(got, dense_mass(q, k, hc, window, lens), rtol=0, atol=1e-12)


def test_mass_conserves_probability():
    # every query's probabilities sum to 1, and every visible key is in the
    # listed sequence: the masses of a KV head add up to G x queries
    hq, hkv, d, lens = 12, 3, 32, [50, 90]
    q = I.normal_bf16(62, 1, (sum(lens), hq, d))
    k = I.normal_bf16(62, 2, (sum(lens), hkv, d))
    m = run_mass(q, k, [oracle.LOCAL, oracle.GLOBAL, oracle.LOCAL], 7, lens)
    np.testing.assert_allclose(m.sum(axis=1), 4 * sum(lens), rtol=0, atol=1e-9)


def test_mass_identical_keys_closed_form():
    # identical keys: a query spreads its mass evenly over its visible keys,
    # 1/(p+1) each on a global head and 1/min(p+1, W) on a local head
    hq, hkv, d, n, W = 4, 2, 16, 40, 6
    q = I.normal_bf16(63, 1, (n, hq, d))
    row = I.normal_bf16(63, 2, (1, 1, d))
    k = row.expand(n, hkv, d).contiguous()
    m = run_mass(q, k, [oracle.GLOBAL, oracle.LOCAL], W, [n])
    G = 2
    glob = [G * sum(1.0 / (p + 1) for p in range(j, n)) for j in range(n)]
    loc = [G * sum(1.0 / min(p + 1, W) for p in range(j, min(n, j + W))) for j in range(n)]
    np.testing.assert_allclose(m[0], glob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(m[1], loc, rtol=0, atol=1e-12)


def test_mass_window_one_is_self():
    hq, hkv, d, n = 6, 3, 16, 25
    q = I.normal_bf16(64, 1, (n, hq, d))
    k = I.normal_bf16(64, 2, (n, hkv, d))
    m = run_mass(q, k, [oracle.LOCAL] * 3, 1, [n])
    np.testing.assert_array_equal(m, np.full((3, n), 2.0))


def topk_threshold(score, k):
    """Top-k by threshold: the k-th largest value v; everything above v plus
    the lowest positions equal to v."""
    score = np.asarray(score, dtype=np.float64)
    if k == 0:
        return np.zeros(0, np.int64)
    v = np.sort(score)[::-1][k - 1]
    above = np.nonzero(score > v)[0]
    equal = np.nonzero(score == v)[0][:k - len(above)]
    return np.sort(np.concatenate([above, equal]))


def test_topk_hand_example_and_special_cases():
    s = [0.5, 2.0, 2.0, 1.0, 0.5]
    assert F.topk_tokens(s, 3).tolist() == [1, 2, 3]
    assert F.topk_tokens(s, 1).tolist() == [1]          # tie 1 vs 2: lower position
    assert F.topk_tokens(s, 4).tolist() == [0, 1, 2, 3]  # tie 0 vs 4
    assert F.topk_tokens(s, 0).tolist() == []
    assert F.topk_tokens(s, 5).tolist() == [0, 1, 2, 3, 4]
    assert F.topk_tokens([1.0] * 6, 2).tolist() == [0, 1]
    assert F.topk_tokens(np.arange(10.0), 3).tolist() == [7, 8, 9]
    with pytest.raises(ValueError):
        F.topk_tokens(s, 6)


def test_topk_matches_threshold_formulation():
    rng = np.random.default_rng(5)
    for trial in range(40):
        n = int(rng.integers(1, 300))
        # few distinct values, so ties are common
        s = rng.integers(0, max(2, n // 7), n).astype(np.float32).astype(np.float64) * 0.25
        k = int(rng.integers(0, n + 1))
        np.testing.assert_array_equal(F.topk_tokens(s, k), topk_threshold(s, k))


def load_golden():
    fx = json.load(open(GOLDEN))
    env = {"ln3": math.log(3.0), "sig": lambda t: 1.0 / (1.0 + math.exp(-t)), "__builtins__": {}}
    ev = lambda a: np.array([[eval(v, env) if isinstance(v, str) else v for v in r] for r in a])
    return fx, ev


def test_ffn_hand_derived_example():
    fx, ev = load_golden()
    out, h = F.sparse_ffn(ev(fx["x"]), ev(fx["residual"]), fx["idx"], ev(fx["w_gate"]),
                          ev(fx["w_up"]), ev(fx["w_down"]))
    np.testing.assert_allclose(h, ev(fx["expected_h"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(out, ev(fx["expected_out"]), rtol=0, atol=1e-14)


def test_ffn_silu_closed_forms():
    # d_ff = 1, u = 1, W_down picks h: y = [silu(g), 0]
    ln3 = math.log(3.0)
    g = np.array([ln3, -ln3, 0.0, 2.0])
    x = np.stack([g, np.ones(4)], axis=1)
    out, _ = F.sparse_ffn(x, np.zeros((4, 2)), [0, 1, 2, 3], [[1.0, 0.0]], [[0.0, 1.0]], [[1.0], [0.0]])
    want = [0.75 * ln3, -0.25 * ln3, 0.0, 2.0 * math.exp(2) / (1 + math.exp(2))]
    np.testing.assert_allclose(out[:, 0], want, rtol=0, atol=1e-15)
    assert not out[:, 1].any()


def test_ffn_identity_path_and_linearity():
    rng = np.random.default_rng(9)
    n, dm, dff = 20, 8, 12
    x, r = rng.standard_normal((n, dm)), rng.standard_normal((n, dm))
    wg, wu, wd = (rng.standard_normal(s) for s in ((dff, dm), (dff, dm), (dm, dff)))
    idx = [3, 7, 8, 15]
    out, _ = F.sparse_ffn(x, r, idx, wg, wu, wd)
    rest = np.setdiff1d(np.arange(n), idx)
    np.testing.assert_array_equal(out[rest], r[rest])            # identity path, bit for bit
    out0, _ = F.sparse_ffn(x, r, idx, wg, wu, np.zeros_like(wd))
    np.testing.assert_array_equal(out0, r)                       # W_down = 0
    out2, _ = F.sparse_ffn(x, r, idx, wg, wu, 2 * wd)
    np.testing.assert_allclose(out2 - r, 2 * (out - r), rtol=0, atol=1e-12)  # linear in W_down
    empty, _ = F.sparse_ffn(x, r, [], wg, wu, wd)
    np.testing.assert_array_equal(empty, r)
