"""Parity at the benchmark's full sizes, on sampled query rows.

The CUDA path runs each workload exactly as bench.py times it (same shapes,
page sizes, head classes, launch configuration); the oracle recomputes a
sample of rows: the first and last 64 positions, +-2 around window starts,
key-tile and page edges (strided at 128K), and 512 random positions. Large
inputs are drawn by the shared seeded generator on the GPU and copied to the
host for the oracle, so both sides read identical values.
"""
import numpy as np
import pytest
import torch

import head_segmented_paged_gb300 as S
from head_segmented_paged_gb300 import inputs as I
from harness import check_close
import oracle

pytestmark = pytest.mark.gpu


def sample_positions(n, W, P, edge_stride=1, seed=0):
    s = set(range(min(64, n))) | set(range(max(0, n - 64), n))
    for c in (W - 1, W, 2 * W):
        s |= {p for p in range(c - 2, c + 3) if 0 <= p < n}
    for e in range(0, n, P * edge_stride):
        s |= {p for p in range(e - 2, e + 3) if 0 <= p < n}
    for e in range(0, n, 128 * edge_stride):
        s |= {p for p in range(e - 2, e + 3) if 0 <= p < n}
    rng = np.random.default_rng(seed)
    s |= set(rng.integers(0, n, 512).tolist())
    return np.array(sorted(s), dtype=np.int64)


def gen_layer(w, layer_set, lens, device="cuda"):
    tot = sum(lens)
    sc = w.qk_scale_inputs
    q = I.normal_bf16(w.seed, I.tensor_stream(I._Q, layer_set), (tot, w.hq, w.head_dim), sc, device)
    k = I.normal_bf16(w.seed, I.tensor_stream(I._K, layer_set), (tot, w.hkv, w.head_dim), sc, device)
    v = I.normal_bf16(w.seed, I.tensor_stream(I._V, layer_set), (tot, w.hkv, w.head_dim), sc, device)
    return q, k, v


def run_prefill_case(w, head_class, window, q, k, v, lens, rows_per_seq, edge_stride=1,
                     output_rounding=False):
    P, D = w.page_size, w.head_dim
    pages = sum((n + P - 1) // P for n in lens) * w.hkv + 8
    kp = torch.full((pages, P, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    h = S.SegKV(1, w.hq, w.hkv, D, [head_class], [window], P, len(lens), max(lens), kp, vp)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ids = list(range(len(lens)))
    h.append(0, k, v, cu, ids)
    q_pos = np.concatenate([np.arange(n, dtype=np.int32) for n in lens])
    o = torch.empty((int(cu[-1]), w.hq, D), dtype=torch.bfloat16, device="cuda")
    h.prefill_attn(0, q, cu, q_pos, ids, o)
    assert h.status() == 0
    torch.cuda.synchronize()
    kc, vc = k.cpu(), v.cpu()
    for b, n in enumerate(lens):
        pos = rows_per_seq(n)
        tok = cu[b] + pos
        qs = q[torch.as_tensor(tok, device="cuda")].cpu()
        rc, ref, _ = oracle.attention(qs, kc[cu[b]:cu[b + 1]], vc[cu[b]:cu[b + 1]],
                                      np.zeros(len(pos), np.int32), pos.astype(np.int32), [0], [n],
                                      head_class, window, np.zeros((1, w.hkv), np.int32))
        assert rc == 0
        check_close(o[torch.as_tensor(tok, device="cuda")], ref, f"{w.name} seq {b}",
                    output_rounding=output_rounding)
    h.close()


def test_mistral_8k_prefill_sampled():
    w = I.mistral_8k()
    q, k, v = gen_layer(w, 0, w.seq_lens)
    run_prefill_case(w, w.head_class[0], w.window[0], q, k, v, w.seq_lens,
                     lambda n: sample_positions(n, w.window[0], w.page_size))


def test_llama70b_varlen_with_sinks_sampled():
    # Named output-rounding case: key rows scaled x8 concentrate attention on
    # single keys, so outputs reach |o| >= 4 (one sampled element is -4.40),
    # where the bf16 half-ulp of the returned value is 2^-6 = 0.0156 > 1e-2.
    w = I.llama70b_varlen()
    q, k, v = gen_layer(w, 0, w.seq_lens)
    off = 0
    for b, n in enumerate(w.seq_lens):  # 1% of key rows x8, as the workload specifies
        idx = torch.tensor(w.sink_positions[b], dtype=torch.int64, device="cuda") + off
        k[idx] = k[idx] * 8
        off += n
    run_prefill_case(w, w.head_class[0], w.window[0], q, k, v, w.seq_lens,
                     lambda n: sample_positions(n, w.window[0], w.page_size, edge_stride=8),
                     output_rounding=True)


@pytest.mark.parametrize("kind", ["shallow", "deep_g1", "deep_g0", "dense"])
def test_128k_layer_sampled(kind):
    w = I.long_128k_64layer(all_global=(kind == "dense"))
    if kind == "dense":
        layer = 8
    else:
        want = {"shallow": lambda l, g: l < 8, "deep_g1": lambda l, g: l >= 8 and g == 1,
                "deep_g0": lambda l, g: l >= 8 and g == 0}[kind]
        layer = next(l for l in range(64)
                     if want(l, sum(1 for c in w.head_class[l] if c == I.GLOBAL)))
    q, k, v = gen_layer(w, layer % 4, w.seq_lens)
    n = w.seq_lens[0]

    def rows(n):
        pos = sample_positions(n, w.window[layer], w.page_size, edge_stride=64)
        return pos if kind != "dense" else pos[:: max(1, len(pos) // 96)]

    run_prefill_case(w, w.head_class[layer], w.window[layer], q, k, v, [n], rows)


def test_ragged_decode_full_steps():
    w = I.ragged_decode(steps=4)
    B, P, D = len(w.seq_lens), w.page_size, w.head_dim
    q, k, v = gen_layer(w, 0, w.seq_lens)
    del q
    pages = sum((n + 8) // P + 2 for n in w.seq_lens) * w.hkv + 64
    kp = torch.full((pages, P, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    h = S.SegKV(1, w.hq, w.hkv, D, w.head_class, w.window, P, B, max(w.seq_lens) + 8, kp, vp)
    m = oracle.PageModel(1, w.hkv, w.head_class, w.window, P, B, max(w.seq_lens) + 8, pages)
    cu = np.concatenate([[0], np.cumsum(w.seq_lens)]).astype(np.int32)
    ids = list(range(B))
    h.append(0, k, v, cu, ids)
    assert m.append(0, cu, ids) == 0
    h.trim(0, ids)
    assert m.trim(0, ids) == 0
    kc, vc = k.cpu(), v.cpu()
    klog = [kc[cu[b]:cu[b + 1]] for b in range(B)]
    vlog = [vc[cu[b]:cu[b + 1]] for b in range(B)]
    ws = torch.empty(h.workspace_size(S.SEGKV_WS_DECODE, B, B) // 4 + 64, device="cuda")
    one = np.arange(B + 1, dtype=np.int32)
    for st in range(w.decode_steps):
        qd, kd, vd = I.decode_step_tensors(w, st, device="cuda")
        h.append(0, kd, vd, one, ids)
        assert m.append(0, one, ids) == 0
        for b in range(B):
            klog[b] = torch.cat([klog[b], kd[b:b + 1].cpu()])
            vlog[b] = torch.cat([vlog[b], vd[b:b + 1].cpu()])
        lens = [m.seq_len(0, b) for b in ids]
        o = torch.full((B, w.hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        h.decode_attn(0, qd, lens, ids, o, ws)
        assert h.status() == 0
        offs = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
        seg = np.array([[m.segment(0, hd, b)[0] for hd in range(w.hkv)] for b in ids], np.int32)
        rc, ref, _ = oracle.attention(qd.cpu(), torch.cat(klog), torch.cat(vlog),
                                      np.arange(B, dtype=np.int32),
                                      np.array(lens, np.int32) - 1, offs, lens,
                                      w.head_class[0], w.window[0], seg)
        assert rc == 0
        check_close(o, ref, f"ragged decode step {st}")
    for hd in range(w.hkv):
        for b in ids:
            assert h.segment(0, hd, b) == m.segment(0, hd, b)
    h.close()


def test_ragged_decode_four_tokens_full():
    # The benchmark's four-token leg: the ragged-decode contexts, four new
    # tokens per request appended in one call, 4 x 4 = 16 query rows per KV head
    # on the tensor-core decode kernel (split pairs, merge kernel, LSE).
    w = I.ragged_decode(steps=1)
    B, P, D, T = len(w.seq_lens), w.page_size, w.head_dim, 4
    q, k, v = gen_layer(w, 0, w.seq_lens)
    del q
    pages = sum((n + T + 8) // P + 2 for n in w.seq_lens) * w.hkv + 64
    kp = torch.full((pages, P, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    h = S.SegKV(1, w.hq, w.hkv, D, w.head_class, w.window, P, B, max(w.seq_lens) + T + 8, kp, vp)
    m = oracle.PageModel(1, w.hkv, w.head_class, w.window, P, B, max(w.seq_lens) + T + 8, pages)
    cu = np.concatenate([[0], np.cumsum(w.seq_lens)]).astype(np.int32)
    ids = list(range(B))
    h.append(0, k, v, cu, ids)
    assert m.append(0, cu, ids) == 0
    h.trim(0, ids)
    assert m.trim(0, ids) == 0
    kt = I.normal_bf16(w.seed, I.tensor_stream(I._KD, 1, 9999), (B * T, w.hkv, D), device="cuda")
    vt = I.normal_bf16(w.seed, I.tensor_stream(I._VD, 1, 9999), (B * T, w.hkv, D), device="cuda")
    qt = I.normal_bf16(w.seed, I.tensor_stream(I._QD, 1, 9999), (B * T, w.hq, D), device="cuda")
    cut = np.arange(0, B * T + 1, T, dtype=np.int32)
    h.append(0, kt, vt, cut, ids)
    assert m.append(0, cut, ids) == 0
    lens = [m.seq_len(0, b) for b in ids]
    o = torch.full((B * T, w.hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.hq, B * T), dtype=torch.float32, device="cuda")
    ws = torch.empty(h.workspace_size(S.SEGKV_WS_DECODE, B * T, B) // 4 + 64, device="cuda")
    h.decode_attn_multi(0, qt, T, lens, ids, o, lse, ws)
    assert h.status() == 0
    kc, vc, ktc, vtc = k.cpu(), v.cpu(), kt.cpu(), vt.cpu()
    klog = torch.cat([torch.cat([kc[cu[b]:cu[b + 1]], ktc[T * b:T * b + T]]) for b in ids])
    vlog = torch.cat([torch.cat([vc[cu[b]:cu[b + 1]], vtc[T * b:T * b + T]]) for b in ids])
    offs = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    seg = np.array([[m.segment(0, hd, b)[0] for hd in range(w.hkv)] for b in ids], np.int32)
    row_seq = np.repeat(np.arange(B), T).astype(np.int32)
    row_pos = np.concatenate([np.arange(n - T, n) for n in lens]).astype(np.int32)
    rc, ref, ref_lse = oracle.attention(qt.cpu(), klog, vlog, row_seq, row_pos, offs, lens,
                                        w.head_class[0], w.window[0], seg)
    assert rc == 0
    check_close(o, ref, "four-token ragged decode")
    np.testing.assert_allclose(lse.cpu().numpy().T, ref_lse, atol=1e-3, rtol=0)
    h.close()
