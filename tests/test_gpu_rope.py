"""Rotary re-alignment of cached keys vs the oracle's fp64 rotation.

Selected heads' kept keys must equal the oracle's rotation of the appended
keys within bf16 rounding; everything else (other heads, V, other
sequences, dimensions beyond rotary_dim, slots below a local head's kept
start) must be unchanged bit for bit.
"""
import numpy as np
import pytest
import torch

import head_segmented_paged_gb300 as S
import oracle
from head_segmented_paged_gb300 import inputs as I
from harness import Cache

pytestmark = pytest.mark.gpu


def gather_rows(pool, c, layer, hd, b):
    s, ln, first, ids = c.m.segment(layer, hd, b)
    pos = torch.arange(s, s + ln)
    pid = torch.tensor(ids)[pos // c.P - first]
    return pool[pid, pos % c.P].to(torch.float64).numpy(), s


@pytest.mark.parametrize("style,rd,mask,delta", [(0, 128, 0xFF, 12345), (1, 96, 0b101, -777),
                                                 (0, 36, 0xF, 999), (1, 36, 0b11, -5),
                                                 (1, 128, 0b10, 131000)])
def test_rope_shift_matches_oracle(style, rd, mask, delta):
    hkv, d, P, W = 4, 128, 64, 300
    hc = [[I.GLOBAL, I.LOCAL, I.LOCAL, I.GLOBAL]]
    c = Cache(1, hkv * 4, hkv, d, hc, [W], P, 3, 4096, 400)
    for b, n in enumerate([900, 1500, 70]):
        k = I.normal_bf16(21, 10 + b, (n, hkv, d))
        v = I.normal_bf16(21, 20 + b, (n, hkv, d))
        assert c.append(0, k.cuda(), v.cuda(), [0, n], [b]) == 0
    one = I.normal_bf16(21, 30, (1, hkv, d))
    assert c.append(0, one.cuda(), one.cuda(), [0, 1], [1]) == 0  # local heads of seq 1 evict
    kp0, vp0 = c.kp.cpu().clone(), c.vp.cpu().clone()
    c.h.rope_shift(0, 1, delta, 10000.0, rd, style, mask)
    assert c.h.status() == 0
    kp1, vp1 = c.kp.cpu(), c.vp.cpu()
    assert torch.equal(vp0.view(torch.int16), vp1.view(torch.int16))
    for b in (0, 2):
        for hd in range(hkv):
            a, _ = gather_rows(kp0, c, 0, hd, b)
            z, _ = gather_rows(kp1, c, 0, hd, b)
            np.testing.assert_array_equal(a, z)
    for hd in range(hkv):
        before, s = gather_rows(kp0, c, 0, hd, 1)
        after, _ = gather_rows(kp1, c, 0, hd, 1)
        if not (mask >> hd) & 1:
            np.testing.assert_array_equal(before, after)
            continue
        klog = c.k_log[(0, 1)][s:, hd]
        assert np.array_equal(klog.to(torch.float64).numpy(), before)
        ref = oracle.rope(klog, delta, rd, style, 10000.0)
        err = np.abs(after - ref)
        assert (err <= 2.0 ** -8 * np.abs(ref) + 1e-6).all(), err.max()
        np.testing.assert_array_equal(after[:, rd:], before[:, rd:])


def test_rope_shift_then_inverse_is_near_identity():
    # Rotating by +delta then -delta returns the keys within two bf16 roundings,
    # each bounded by half an ulp of the rotated pair (at most 2^-8 of its norm).
    hkv, d, P = 2, 64, 16
    c = Cache(1, 8, hkv, d, [[I.GLOBAL, I.LOCAL]], [40], P, 1, 512, 64)
    k = I.normal_bf16(3, 1, (200, hkv, d))
    assert c.append(0, k.cuda(), k.cuda(), [0, 200], [0]) == 0
    before, _ = gather_rows(c.kp.cpu(), c, 0, 0, 0)
    c.h.rope_shift(0, 0, 5000, 500000.0, 64, S.SEGKV_ROPE_INTERLEAVED)
    c.h.rope_shift(0, 0, -5000, 500000.0, 64, S.SEGKV_ROPE_INTERLEAVED)
    after, _ = gather_rows(c.kp.cpu(), c, 0, 0, 0)
    pair_norm = np.repeat(np.hypot(before[:, 0::2], before[:, 1::2]), 2, axis=1)
    assert (np.abs(after - before) <= 2.0 ** -7 * pair_norm + 2e-6).all()
    assert S.segkv_rope_shift(c.h.handle, 0, 0, 1, 10000.0, 63, 0) == S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_rope_shift(c.h.handle, 0, 0, 1, 10000.0, 130, 0) == S.SEGKV_ERR_INVALID_ARG
