"""Segment export/import (prefill/decode transfer) through the C ABI.

The exported buffer must hold exactly each head's kept K and V rows; an
import into another handle must reproduce the oracle page model's tables,
the same page contents and the same attention outputs as the source.
"""
import numpy as np
import pytest
import torch

import head_segmented_paged_gb300 as S
from head_segmented_paged_gb300 import inputs as I
from harness import Cache, check_close

pytestmark = pytest.mark.gpu


def build_source():
    hkv, G, d, P, W = 8, 4, 128, 64, 256
    hc = [[I.GLOBAL] + [I.LOCAL] * 7]
    c = Cache(1, hkv * G, hkv, d, hc, [W], P, 3, 4096, 700)
    for b, n in enumerate([1500, 2300, 90]):
        k = I.normal_bf16(41, 10 + b, (n, hkv, d))
        v = I.normal_bf16(41, 20 + b, (n, hkv, d))
        assert c.append(0, k.cuda(), v.cuda(), [0, n], [b]) == 0
    c.trim(0, [0, 1, 2])
    return c


def test_export_holds_exactly_the_kept_rows_and_is_smaller_than_dense():
    c = build_source()
    buf, hdr = c.h.export_segment(0, 1)
    n = c.m.seq_len(0, 1)
    assert hdr[0] == n
    got = buf.cpu().view(-1, c.d)
    row = 0
    kept = 0
    for hd in range(c.hkv):
        s = c.m.segment(0, hd, 1)[0]
        assert hdr[1 + hd] == s
        ln = n - s
        kl, vl = c.k_log[(0, 1)][s:, hd], c.v_log[(0, 1)][s:, hd]
        assert torch.equal(got[row:row + ln].view(torch.int16), kl.view(torch.int16))
        assert torch.equal(got[row + ln:row + 2 * ln].view(torch.int16), vl.view(torch.int16))
        row += 2 * ln
        kept += ln
    assert got.shape[0] == row
    dense = n * c.hkv * c.d * 2 * 2
    assert buf.numel() * 2 == kept * c.d * 2 * 2
    # one global head keeps 2300 keys, seven local heads keep W-1 = 255 each
    assert dense / (buf.numel() * 2) == pytest.approx(8 * 2300 / (2300 + 7 * 255))


def test_import_into_another_handle_reproduces_tables_pages_and_attention():
    a = build_source()
    buf, hdr = a.h.export_segment(0, 1)
    # target with other residents, so page ids differ from the source's
    b = Cache(1, a.hq, a.hkv, a.d, a.head_class, a.window, a.P, 4, 4096, 500)
    k = I.normal_bf16(42, 1, (700, a.hkv, a.d))
    assert b.append(0, k.cuda(), k.cuda(), [0, 700], [0]) == 0
    rc = S.segkv_import(b.h.handle, 0, 0, buf, hdr)
    assert rc == S.SEGKV_ERR_INVALID_ARG  # seq 0 is not empty
    assert b.m.import_segment(0, 2, int(hdr[0]), hdr[1:].tolist()) == 0
    b.h.import_segment(0, 2, buf, hdr)
    b.k_log[(0, 2)] = a.k_log[(0, 1)].clone()
    b.v_log[(0, 2)] = a.v_log[(0, 1)].clone()
    b.check_tables(0)
    b.check_pages(0, [2])
    # one more token on both sides, then decode: identical outputs
    kd = I.normal_bf16(43, 2, (1, a.hkv, a.d))
    vd = I.normal_bf16(43, 3, (1, a.hkv, a.d))
    qd = I.normal_bf16(43, 4, (1, a.hq, a.d))
    assert a.append(0, kd.cuda(), vd.cuda(), [0, 1], [1]) == 0
    assert b.append(0, kd.cuda(), vd.cuda(), [0, 1], [2]) == 0
    n = a.m.seq_len(0, 1)
    outs = []
    for c, seq in ((a, 1), (b, 2)):
        ws = torch.empty(c.h.workspace_size(S.SEGKV_WS_DECODE, 1, 1) // 4 + 64, device="cuda")
        o = torch.empty((1, c.hq, c.d), dtype=torch.bfloat16, device="cuda")
        c.h.decode_attn(0, qd.cuda(), [n], [seq], o, ws)
        assert c.h.status() == 0
        outs.append(o.cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    rc, ref, _ = b.oracle_attention(0, qd, [2], np.zeros(1, np.int32), np.array([n - 1], np.int32))
    assert rc == 0
    check_close(outs[1], ref, "decode after import")


def test_import_without_room_changes_nothing():
    a = build_source()
    buf, hdr = a.h.export_segment(0, 1)
    small = Cache(1, a.hq, a.hkv, a.d, a.head_class, a.window, a.P, 2, 4096, 20)
    before = [small.h.segment(0, hd, 1) for hd in range(a.hkv)]
    rc = S.segkv_import(small.h.handle, 0, 1, buf, hdr)
    assert rc == S.SEGKV_ERR_OUT_OF_PAGES
    assert small.m.import_segment(0, 1, int(hdr[0]), hdr[1:].tolist()) == S.SEGKV_ERR_OUT_OF_PAGES
    assert [small.h.segment(0, hd, 1) for hd in range(a.hkv)] == before
    assert small.h.stats()["pages_in_use"] == 0
