"""CUDA path vs the oracle, element by element, through the C ABI.

Pools start NaN-filled, so any read of a slot outside a segment's kept range
(freed page, unwritten tail, stale head) would surface as a non-finite or
wrong output.
"""
import numpy as np
import pytest
import torch

import head_segmented_paged_gb300 as S
from head_segmented_paged_gb300 import inputs as I
from harness import Cache, check_close, prefill_case

pytestmark = pytest.mark.gpu


def run_prefill(c, layer, q, cu, qp, ids, lse=True):
    tot = q.shape[0]
    o = torch.full((tot, c.hq, c.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    l = torch.full((c.hq, tot), float("nan"), dtype=torch.float32, device="cuda") if lse else None
    rc = S.segkv_prefill_attn(c.h.handle, layer, q.cuda(), cu, qp, ids, o, l)
    assert rc == 0, S.segkv_last_error(c.h.handle)
    assert c.h.status() == 0
    torch.cuda.synchronize()
    return o, l


def q_index(cu):
    cu = [int(x) for x in cu]
    return np.repeat(np.arange(len(cu) - 1), np.diff(cu))


def test_tiny_256_tables_pages_and_attention():
    w = I.tiny_256()
    c, q, cu, qp, ids = prefill_case(w)
    c.check_tables(0)
    c.check_pages(0, ids)
    o, lse = run_prefill(c, 0, q, cu, qp, ids)
    rc, ref, ref_lse = c.oracle_attention(0, q, ids, q_index(cu), qp.numpy())
    assert rc == 0
    check_close(o, ref, "tiny-256")
    np.testing.assert_allclose(lse.cpu().numpy().T, ref_lse, atol=1e-3, rtol=0)


@pytest.mark.parametrize("P", [8, 16, 64, 128, 256])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
def test_ragged_varlen_page_sizes(P, G):
    hkv = 2
    w = I.Workload("ragged", 1, G * hkv, hkv, 128, P, [[I.GLOBAL, I.LOCAL]], [100],
                   [700, 129, 1000, 1], seed=3)
    c, q, cu, qp, ids = prefill_case(w)
    c.check_tables(0)
    c.check_pages(0, ids)
    o, lse = run_prefill(c, 0, q, cu, qp, ids)
    rc, ref, ref_lse = c.oracle_attention(0, q, ids, q_index(cu), qp.numpy())
    assert rc == 0
    # Named output-rounding case, G=4 (the same seeded data at every P): one
    # element with oracle value -2.1046 comes back as -2.0938, 1.09e-2 away.
    # The bf16 grid spacing there is 2^-6, so the fp32 result before the
    # output rounding was at least 3.0e-3 off (P is rounded to bf16 for the
    # P V MMA).
    check_close(o, ref, f"ragged P={P} G={G}", output_rounding=(G == 4))
    np.testing.assert_allclose(lse.cpu().numpy().T, ref_lse, atol=1e-3, rtol=0)


def test_prefill_repeats_bit_for_bit_whichever_cta_runs_a_unit():
    """CTAs claim units at run time, so which CTA runs a unit changes from call
    to call; a unit's result must not. Many short sequences (small units,
    claimed last) beside two long ones, run five times and compared bit for
    bit; the first run also against the oracle."""
    hkv = 4
    lens = [1500, 3000] + [int(x) for x in np.random.default_rng(11).integers(1, 200, size=60)]
    w = I.Workload("claims", 1, 4 * hkv, hkv, 128, 64, [[I.GLOBAL, I.LOCAL, I.LOCAL, I.LOCAL]], [300],
                   lens, seed=11)
    c, q, cu, qp, ids = prefill_case(w)
    o0, l0 = run_prefill(c, 0, q, cu, qp, ids)
    for _ in range(4):
        o, l = run_prefill(c, 0, q, cu, qp, ids)
        assert torch.equal(o, o0) and torch.equal(l, l0)
    rc, ref, ref_lse = c.oracle_attention(0, q, ids, q_index(cu), qp.numpy())
    assert rc == 0
    check_close(o0, ref, "claimed units")
    np.testing.assert_allclose(l0.cpu().numpy().T, ref_lse, atol=1e-3, rtol=0)


def test_head_dim_64_many_heads():
    w = I.Workload("d64", 1, 16, 4, 64, 32, [[I.LOCAL, I.GLOBAL, I.LOCAL, I.LOCAL]], [7],
                   [300, 45], seed=5)
    c, q, cu, qp, ids = prefill_case(w)
    o, _ = run_prefill(c, 0, q, cu, qp, ids)
    rc, ref, _ = c.oracle_attention(0, q, ids, q_index(cu), qp.numpy())
    assert rc == 0
    check_close(o, ref, "d64")


def test_chunked_prefill_with_lazy_eviction_and_poisoned_stale_heads():
    """Chunks of one sequence appended and attended in turn: local heads drop
    old pages between chunks; the stale head of each local segment's first
    page is overwritten with NaN before attention."""
    hq, hkv, d, P, W = 16, 4, 128, 64, 150
    hc = [[I.LOCAL, I.GLOBAL, I.LOCAL, I.LOCAL]]
    n = 1100
    c = Cache(1, hq, hkv, d, hc, [W], P, 2, 4096, 200)
    g = torch.Generator().manual_seed(0)
    allq = I.normal_bf16(11, 1, (n, hq, d))
    allk = I.normal_bf16(11, 2, (n, hkv, d))
    allv = I.normal_bf16(11, 3, (n, hkv, d))
    bounds = [0, 97, 300, 301, 650, 1100]
    for a, b in zip(bounds[:-1], bounds[1:]):
        cu = [0, b - a]
        assert c.append(0, allk[a:b].cuda(), allv[a:b].cuda(), cu, [1]) == 0
        c.check_tables(0)
        # poison slots below the kept start inside each local segment's first page
        for hd in range(hkv):
            s, ln, first, ids = c.m.segment(0, hd, 1)
            if ids and s % P:
                c.kp[ids[0], : s % P] = float("nan")
                c.vp[ids[0], : s % P] = float("nan")
        qp = torch.arange(a, b, dtype=torch.int32)
        o, _ = run_prefill(c, 0, allq[a:b], cu, qp, [1])
        rc, ref, _ = c.oracle_attention(0, allq[a:b], [1], np.zeros(b - a, np.int32), qp.numpy())
        assert rc == 0
        check_close(o, ref, f"chunk {a}:{b}")


def test_evicted_queries_are_rejected():
    w = I.tiny_256()
    c, q, cu, qp, ids = prefill_case(w, num_pages=64, max_seq_len=512)
    k1 = I.normal_bf16(9, 9, (1, 2, 64)).cuda()
    assert c.append(0, k1, k1, [0, 1], [0]) == 0  # local head drops keys < 225
    o = torch.empty((256, 8, 64), dtype=torch.bfloat16, device="cuda")
    rc = S.segkv_prefill_attn(c.h.handle, 0, q.cuda(), cu, qp, ids, o)
    assert rc == S.SEGKV_ERR_EVICTED
    # position 255 needs key 224, already dropped; 256 needs 225.. only
    o1 = torch.empty((1, 8, 64), dtype=torch.bfloat16, device="cuda")
    assert S.segkv_prefill_attn(c.h.handle, 0, q[-1:].cuda(), [0, 1], [255], [0], o1) == \
        S.SEGKV_ERR_EVICTED
    qp2 = torch.tensor([256], dtype=torch.int32)
    o2, _ = run_prefill(c, 0, q[-1:], [0, 1], qp2, [0])
    rc, ref, _ = c.oracle_attention(0, q[-1:], [0], np.zeros(1, np.int32), qp2.numpy())
    assert rc == 0
    check_close(o2, ref, "after eviction")


def test_out_of_order_and_repeated_query_positions():
    w = I.Workload("perm", 1, 8, 2, 128, 64, [[I.GLOBAL, I.LOCAL]], [40], [500], seed=2)
    c, q, cu, qp, ids = prefill_case(w)
    perm = torch.tensor([499, 0, 3, 3, 250, 128, 127, 64, 63, 400, 1, 2] * 3, dtype=torch.int32)
    qq = I.normal_bf16(4, 4, (perm.numel(), 8, 128))
    o, _ = run_prefill(c, 0, qq, [0, perm.numel()], perm, [0])
    rc, ref, _ = c.oracle_attention(0, qq, [0], np.zeros(perm.numel(), np.int32), perm.numpy())
    assert rc == 0
    check_close(o, ref, "permuted q_pos")


def test_empty_calls_are_noops():
    w = I.tiny_256()
    c, q, cu, qp, ids = prefill_case(w)
    o = torch.empty((0, 8, 64), dtype=torch.bfloat16, device="cuda")
    assert S.segkv_prefill_attn(c.h.handle, 0, q.cuda(), [0, 0], [], [0], o) == 0
    assert S.segkv_append(c.h.handle, 0, q.cuda(), q.cuda(), [0, 0], [0]) == 0
    assert c.m.append(0, [0, 0], [0]) == 0
    c.check_tables(0)
    assert c.h.status() == 0


# both head dims of the prefill kernel: the MMA issuer's wait expires, then
# every other warp's bounded wait sees the block's abort flag and returns
@pytest.mark.parametrize("d", [64, 128])
def test_device_timeout_path_reports_status_and_context_survives(d):
    w = I.tiny_256() if d == 64 else I.Workload("tiny128", 1, 8, 2, 128, 16, [[I.GLOBAL, I.LOCAL]],
                                                 [32], [256], seed=0)
    c, q, cu, qp, ids = prefill_case(w)
    c.h.set_debug(1)
    o = torch.empty((256, 8, d), dtype=torch.bfloat16, device="cuda")
    assert S.segkv_prefill_attn(c.h.handle, 0, q.cuda(), cu, qp, ids, o) == 0
    assert c.h.status() == S.SEGKV_ERR_DEVICE_TIMEOUT
    assert c.h.status() == 0  # cleared
    o2, _ = run_prefill(c, 0, q, cu, qp, ids)
    rc, ref, _ = c.oracle_attention(0, q, ids, q_index(cu), qp.numpy())
    check_close(o2, ref, "after timeout")


def decode_run(c, layer, reqs, steps, seed):
    """Append one token per request per step, decode, compare every step."""
    B = len(reqs)
    ws_bytes = c.h.workspace_size(S.SEGKV_WS_DECODE, B, B)
    ws = torch.empty(ws_bytes // 4 + 64, dtype=torch.float32, device="cuda")
    for st in range(steps):
        qd = I.normal_bf16(seed, 100 + st, (B, c.hq, c.d))
        kd = I.normal_bf16(seed, 200 + st, (B, c.hkv, c.d))
        vd = I.normal_bf16(seed, 300 + st, (B, c.hkv, c.d))
        cu = list(range(B + 1))
        assert c.append(layer, kd.cuda(), vd.cuda(), cu, reqs) == 0
        lens = [c.m.seq_len(layer, b) for b in reqs]
        o = torch.full((B, c.hq, c.d), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = S.segkv_decode_attn(c.h.handle, layer, qd.cuda(), lens, reqs, o, ws)
        assert rc == 0, S.segkv_last_error(c.h.handle)
        assert c.h.status() == 0
        rc, ref, _ = c.oracle_attention(layer, qd, reqs, np.arange(B, dtype=np.int32),
                                        np.array(lens, np.int32) - 1)
        assert rc == 0
        check_close(o, ref, f"decode step {st}")
    c.check_tables(layer)
    c.check_pages(layer, reqs)


@pytest.mark.parametrize("G,P,d", [(4, 64, 128), (8, 16, 128), (1, 128, 64), (16, 32, 64)])
def test_decode_ragged_with_ring_eviction(G, P, d):
    hkv = 2
    lens = [1, 63, 64, 65, 600, 1500, 2047, 3000]
    w = I.Workload("dec", 1, G * hkv, hkv, d, P, [[I.LOCAL, I.GLOBAL]], [300], lens, seed=7)
    c, q, cu, qp, ids = prefill_case(w, num_pages=2000, max_seq_len=4096)
    decode_run(c, 0, ids, steps=6, seed=8)
    # trim then keep decoding: the next token's keys are all still there
    c.trim(0, ids)
    c.check_tables(0)
    decode_run(c, 0, ids, steps=3, seed=9)


def test_decode_subset_of_sequences_and_free_reuse():
    hkv, G, d, P = 2, 4, 128, 64
    c = Cache(1, hkv * G, hkv, d, [[I.GLOBAL, I.LOCAL]], [128], P, 4, 2048, 300)
    for b, n in zip(range(4), [200, 900, 50, 1300]):
        k = I.normal_bf16(1, 10 + b, (n, hkv, d))
        v = I.normal_bf16(1, 20 + b, (n, hkv, d))
        assert c.append(0, k.cuda(), v.cuda(), [0, n], [b]) == 0
    decode_run(c, 0, [3, 1], steps=3, seed=2)
    c.free_seq(1)
    k = I.normal_bf16(1, 30, (700, hkv, d))
    assert c.append(0, k.cuda(), k.cuda(), [0, 700], [1]) == 0
    c.check_tables(0)
    decode_run(c, 0, [0, 1, 2, 3], steps=3, seed=3)


@pytest.mark.parametrize("d,P", [(128, 16), (64, 64)])
def test_window_one_local_heads_return_their_own_value(d, P):
    """A local head with W = 1 sees only its own key, so its softmax weight is
    1 and its output is that key's V row exactly. Prefill, then trim (which
    leaves the local segments with no key), then decode steps that append and
    read a single key per local segment."""
    hkv, G, n = 2, 4, 300
    w = I.Workload("w1", 1, G * hkv, hkv, d, P, [[I.GLOBAL, I.LOCAL]], [1], [n], seed=21)
    c, q, cu, qp, ids = prefill_case(w, num_pages=200, max_seq_len=512)
    o, lse = run_prefill(c, 0, q, cu, qp, ids)
    rc, ref, _ = c.oracle_attention(0, q, ids, q_index(cu), qp.numpy())
    assert rc == 0
    check_close(o, ref, "prefill W=1")
    v_local = c.v_log[(0, ids[0])][:, 1]  # [n, d] bf16
    for g in range(G):
        assert torch.equal(o[:, G + g].cpu().contiguous().view(torch.int16),
                           v_local.contiguous().view(torch.int16))
    np.testing.assert_allclose(lse[G:].cpu().numpy(),  # one key: LSE = its scaled score
                               (q[:, G:].double() * c.k_log[(0, ids[0])][:, 1:2].double()).sum(-1).T.numpy()
                               / np.sqrt(d), atol=1e-3, rtol=1e-4)
    c.trim(0, ids)
    s, ln, _, pages = c.m.segment(0, 1, ids[0])
    # no key kept (the next query needs only its own); only the page that will
    # receive the next key stays held when position n falls inside it
    assert (s, ln) == (n, 0) and len(pages) == (1 if n % P else 0)
    c.check_tables(0)
    decode_run(c, 0, ids, steps=3, seed=22)
