"""Decode variants: several query tokens per sequence, and the
FlashAttention window convention, against the oracle."""
import numpy as np
import pytest
import torch

import head_segmented_paged_gb300 as S
from head_segmented_paged_gb300 import inputs as I
from harness import Cache, check_close

pytestmark = pytest.mark.gpu


# T * G in {1, 2, 4, 8, 16} runs on a decode kernel (8 or 16 rows of 128 dims
# on the tensor-core one, fewer on the CUDA-core one), the rest on the prefill
# kernel
@pytest.mark.parametrize("T,G", [(1, 4), (4, 4), (2, 8), (4, 2), (16, 1), (2, 1),
                                 (1, 8), (1, 16), (8, 1), (3, 4), (7, 8), (16, 2),
                                 (1, 1), (1, 2)])
def test_multi_query_decode_matches_oracle(T, G):
    multi_query_case(T, G, 128)


# at 64 dims every T * G of 1 to 16 runs on the CUDA-core decode kernel
@pytest.mark.parametrize("T,G", [(1, 1), (1, 2), (2, 2), (1, 8), (1, 16), (4, 4)])
def test_multi_query_decode_head_dim_64(T, G):
    multi_query_case(T, G, 64)


def multi_query_case(T, G, d):
    hkv, P, W = 4, 64, 200
    hc = [[I.GLOBAL, I.LOCAL, I.LOCAL, I.LOCAL]]
    lens0 = [3000, 64, 700, 1500, 20]
    c = Cache(1, hkv * G, hkv, d, hc, [W], P, len(lens0), 4096, 600)
    ids = list(range(len(lens0)))
    for b, n in enumerate(lens0):
        k = I.normal_bf16(51, 10 + b, (n, hkv, d))
        v = I.normal_bf16(51, 20 + b, (n, hkv, d))
        assert c.append(0, k.cuda(), v.cuda(), [0, n], [b]) == 0
    c.trim(0, ids)
    # T new tokens per sequence, appended in one call
    B = len(ids)
    kd = I.normal_bf16(52, 1, (B * T, hkv, d))
    vd = I.normal_bf16(52, 2, (B * T, hkv, d))
    assert c.append(0, kd.cuda(), vd.cuda(), [T * i for i in range(B + 1)], ids) == 0
    lens = [c.m.seq_len(0, b) for b in ids]
    q = I.normal_bf16(52, 3, (B * T, hkv * G, d))
    o = torch.full((B * T, hkv * G, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hkv * G, B * T), dtype=torch.float32, device="cuda")
    wsb = c.h.workspace_size(S.SEGKV_WS_DECODE, B * T, B)
    assert (wsb > 0) == (T * G in (1, 2, 4, 8, 16))
    ws = torch.empty(wsb // 4 + 64, device="cuda") if wsb else None
    c.h.decode_attn_multi(0, q.cuda(), T, lens, ids, o, lse, ws)
    assert c.h.status() == 0
    row_seq = np.repeat(np.arange(B), T).astype(np.int32)
    row_pos = np.concatenate([np.arange(n - T, n) for n in lens]).astype(np.int32)
    rc, ref, ref_lse = c.oracle_attention(0, q, ids, row_seq, row_pos)
    assert rc == 0
    check_close(o, ref, f"multi-query decode T={T}")
    np.testing.assert_allclose(lse.cpu().numpy().T, ref_lse, atol=1e-3, rtol=0)
    if T == 1:  # equals the split-KV decode path
        ws = torch.empty(c.h.workspace_size(S.SEGKV_WS_DECODE, B, B) // 4 + 64, device="cuda")
        o1 = torch.empty_like(o)
        c.h.decode_attn(0, q.cuda(), lens, ids, o1, ws)
        check_close(o1, ref, "split-KV decode")
    # a too-large T is refused, and so is a short workspace
    assert S.segkv_decode_attn_multi(c.h.handle, 0, q.cuda(), 100, lens, ids, o) == \
        S.SEGKV_ERR_INVALID_ARG
    if wsb:
        assert S.segkv_decode_attn_multi(c.h.handle, 0, q.cuda(), T, lens, ids, o, None, ws,
                                         256) == S.SEGKV_ERR_INVALID_ARG


def test_fa_window_convention_prefill_and_decode():
    # FlashAttention window (W, 0) covers W+1 keys: the library handle is made
    # with W and switched to that convention; the oracle mirror uses the
    # inclusive window W+1.
    hkv, d, P, W = 2, 64, 16, 31
    c = Cache(1, 8, hkv, d, [[I.GLOBAL, I.LOCAL]], [W + 1], P, 1, 512, 64)
    c.h.close()
    c.h = S.SegKV(1, 8, hkv, d, [[I.GLOBAL, I.LOCAL]], [W], P, 1, 512, c.kp, c.vp)
    c.h.set_window_convention(S.SEGKV_WINDOW_FA)
    w = I.tiny_256()
    q, k, v, cu, qp = I.prefill_tensors(w)
    assert c.append(0, k.cuda(), v.cuda(), cu, [0]) == 0
    o = torch.empty((256, 8, d), dtype=torch.bfloat16, device="cuda")
    assert S.segkv_prefill_attn(c.h.handle, 0, q.cuda(), cu, qp, [0], o) == 0
    rc, ref, _ = c.oracle_attention(0, q, [0], np.zeros(256, np.int32), qp.numpy())
    assert rc == 0
    check_close(o, ref, "FA-window prefill")
    # decode after one more token: local head keeps keys p-W .. p
    kd = I.normal_bf16(53, 1, (1, hkv, d))
    assert c.append(0, kd.cuda(), kd.cuda(), [0, 1], [0]) == 0
    c.check_tables(0)
    qd = I.normal_bf16(53, 2, (1, 8, d))
    ws = torch.empty(c.h.workspace_size(S.SEGKV_WS_DECODE, 1, 1) // 4 + 64, device="cuda")
    od = torch.empty((1, 8, d), dtype=torch.bfloat16, device="cuda")
    c.h.decode_attn(0, qd.cuda(), [257], [0], od, ws)
    rc, ref, _ = c.oracle_attention(0, qd, [0], np.zeros(1, np.int32), np.array([256], np.int32))
    assert rc == 0
    check_close(od, ref, "FA-window decode")


@pytest.mark.parametrize("P", [8, 16, 128, 256])
@pytest.mark.parametrize("d", [64, 128])
def test_single_token_decode_page_sizes(P, d):
    """Single-token split-KV decode after a prefill append, a trim and one
    decode append, for the smallest and largest page sizes the library takes."""
    hkv, G, W = 2, 4, 150
    hc = [[I.GLOBAL, I.LOCAL]]
    lens0 = [1000, 9, 300, 257]
    c = Cache(1, hkv * G, hkv, d, hc, [W], P, len(lens0), 2048, 2048 // P * 2 * len(lens0) + 64)
    ids = list(range(len(lens0)))
    for b, n in enumerate(lens0):
        k = I.normal_bf16(61, 10 + b, (n, hkv, d))
        v = I.normal_bf16(61, 20 + b, (n, hkv, d))
        assert c.append(0, k.cuda(), v.cuda(), [0, n], [b]) == 0
    c.trim(0, ids)
    B = len(ids)
    kd = I.normal_bf16(62, 1, (B, hkv, d))
    vd = I.normal_bf16(62, 2, (B, hkv, d))
    assert c.append(0, kd.cuda(), vd.cuda(), list(range(B + 1)), ids) == 0
    c.check_tables(0)
    lens = [c.m.seq_len(0, b) for b in ids]
    q = I.normal_bf16(62, 3, (B, hkv * G, d))
    o = torch.full((B, hkv * G, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(c.h.workspace_size(S.SEGKV_WS_DECODE, B, B) // 4 + 64, device="cuda")
    c.h.decode_attn(0, q.cuda(), lens, ids, o, ws)
    assert c.h.status() == 0
    rc, ref, _ = c.oracle_attention(0, q, ids, np.arange(B, dtype=np.int32),
                                    np.array([n - 1 for n in lens], np.int32))
    assert rc == 0
    check_close(o, ref, f"decode P={P} d={d}")
