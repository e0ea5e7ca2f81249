"""The no-allocation decode entry point against the regular one.

segkv_decode_attn_noalloc serves callers that cannot allocate device memory
when they decode (no per-call workspace): it keeps its split partials in a
fixed array inside the library. It runs the same plan and kernels as
segkv_decode_attn, only with another partials buffer, so its outputs must
equal that call's bit for bit on the same cache, on consecutive calls, and
match the fp64 oracle within the output bar; it must refuse a call whose
partials do not fit. This file is collected last.
"""
import numpy as np
import pytest
import torch

import head_segmented_paged_gb300 as S
from head_segmented_paged_gb300 import inputs as I
from harness import Cache, check_close

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    hkv, G, d, P = 8, 4, 128, 64
    lens = [3000, 700, 65, 12000, 1]
    hc = [[I.GLOBAL] + [I.LOCAL] * 7]
    c = Cache(1, hkv * G, hkv, d, hc, [1024], P, len(lens), 16384, 2600)
    for b, n in enumerate(lens):
        k = I.normal_bf16(5, 10 + b, (n, hkv, d))
        v = I.normal_bf16(5, 20 + b, (n, hkv, d))
        assert c.append(0, k.cuda(), v.cuda(), [0, n], [b]) == 0
    ids = list(range(len(lens)))
    B = len(ids)
    ws = torch.empty(c.h.workspace_size(S.SEGKV_WS_DECODE, B, B) // 4 + 64, device="cuda")
    for step in range(2):
        kd = I.normal_bf16(6, 100 + step, (B, hkv, d)).cuda()
        vd = I.normal_bf16(6, 200 + step, (B, hkv, d)).cuda()
        assert c.append(0, kd, vd, list(range(B + 1)), ids) == 0
        qd = I.normal_bf16(6, 300 + step, (B, hkv * G, d)).cuda()
        cur = [c.m.seq_len(0, b) for b in ids]
        o_ref = torch.full((B, hkv * G, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        o_na = torch.full_like(o_ref, float("nan"))
        assert S.segkv_decode_attn(c.h.handle, 0, qd, cur, ids, o_ref, ws) == 0
        rc = S.segkv_decode_attn_noalloc(c.h.handle, 0, qd, cur, ids, o_na)
        assert rc == 0, S.segkv_last_error(c.h.handle)
        assert c.h.status() == 0
        assert torch.equal(o_na.view(torch.int16), o_ref.view(torch.int16)), f"step {step}"
        rc, ref, _ = c.oracle_attention(0, qd.cpu(), ids, np.arange(B, dtype=np.int32),
                                        np.array(cur, np.int32) - 1)
        assert rc == 0
        check_close(o_na, ref, f"no-alloc decode step {step}")


def test_noalloc_decode_refuses_plans_beyond_its_scratch():
    # 512 one-token sequences x 8 KV heads: up to 4096 + 2*SMs split units of
    # 2 KiB each, more than the 8 MiB the entry point holds.
    hkv, G, d, P, B = 8, 4, 128, 16, 512
    hc = [[I.GLOBAL] + [I.LOCAL] * 7]
    kp = torch.zeros((B * hkv + 8, P, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    h = S.SegKV(1, hkv * G, hkv, d, hc, [64], P, B, 64, kp, vp)
    kv = torch.zeros((B, hkv, d), dtype=torch.bfloat16, device="cuda")
    h.append(0, kv, kv, list(range(B + 1)), list(range(B)))
    q = torch.zeros((B, hkv * G, d), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    rc = S.segkv_decode_attn_noalloc(h.handle, 0, q, [1] * B, list(range(B)), o)
    assert rc == S.SEGKV_ERR_INVALID_ARG
    assert "no-alloc" in S.segkv_last_error(h.handle)
    # a smaller call on the same handle still works
    assert S.segkv_decode_attn_noalloc(h.handle, 0, q[:64], [1] * 64, list(range(64)),
                                       o[:64]) == 0
    assert h.status() == 0
    h.close()
