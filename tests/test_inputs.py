"""Seeded input generator: splitmix64 stream, fp64 -> bf16 rounding, recipes."""
import math

import numpy as np
import pytest
import torch

from head_segmented_paged_gb300 import inputs as I


def test_splitmix64_published_first_output():
    # splitmix64 seeded with 0 outputs 0xE220A8397B1DCDAF first (Vigna's
    # reference implementation, the usual known-answer value).
    z = I._mix(torch.tensor([I._GAMMA], dtype=torch.int64))
    assert (int(z.item()) & I._MASK64) == 0xE220A8397B1DCDAF


def test_torch_stream_matches_uint64_arithmetic():
    # The int64 torch version must equal well-defined uint64 numpy arithmetic.
    key = I.stream_key(0, 12345)
    i = np.arange(1, 5001, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + i * np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    t = I.raw_u64(0, 12345, 5000).numpy().view(np.uint64)
    assert np.array_equal(t, z)


def test_bf16_round_nearest_even_exact_cases():
    one = 1.0
    x = torch.tensor([one + 2 ** -8,            # midpoint 1 | 1+2^-7 -> even (1)
                      one + 3 * 2 ** -8,        # midpoint 1+2^-7 | 1+2^-6 -> even (1+2^-6)
                      one + 2 ** -8 + 2 ** -40,  # just above the midpoint -> up
                      -(one + 2 ** -8 + 2 ** -40),
                      one + 2 ** -8 - 2 ** -40,  # just below -> down
                      3.0, -0.15625], dtype=torch.float64)
    y = I.f64_to_bf16_rne(x).to(torch.float64).tolist()
    assert y == [1.0, 1 + 2 ** -6, 1 + 2 ** -7, -(1 + 2 ** -7), 1.0, 3.0, -0.15625]


def test_bf16_round_matches_single_rounding_of_fp32_values():
    # For values exact in fp32 the one-step rounding equals torch's fp32->bf16.
    g = torch.Generator().manual_seed(1)
    f = torch.randn(100000, generator=g, dtype=torch.float32) * 3
    a = I.f64_to_bf16_rne(f.to(torch.float64))
    b = f.to(torch.bfloat16)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_normal_moments_and_determinism():
    x = I.normal_bf16(0, 7, (1 << 20,)).to(torch.float64)
    assert abs(x.mean().item()) < 5e-3
    assert abs(x.std().item() - 1.0) < 5e-3
    y = I.normal_bf16(0, 7, (1 << 20,), chunk=1 << 16).to(torch.float64)
    assert torch.equal(x, y)
    z = I.normal_bf16(0, 8, (1 << 20,)).to(torch.float64)
    assert not torch.equal(x, z)


def test_recipes_shapes():
    w = I.tiny_256()
    assert (w.hq, w.hkv, w.head_dim, w.page_size, w.window, w.seq_lens) == (8, 2, 64, 16, [32], [256])
    w2 = I.mistral_8k()
    assert sum(1 for c in w2.head_class[0] if c == I.GLOBAL) == 1 and w2.window == [1024]
    assert math.isclose(w2.qk_scale_inputs, 1 / math.sqrt(128))
    w3 = I.llama70b_varlen()
    assert len(w3.seq_lens) == 4 and all(16384 <= n <= 32768 for n in w3.seq_lens)
    for n, s in zip(w3.seq_lens, w3.sink_positions):
        assert len(s) == round(0.01 * n) and len(set(s)) == len(s) and max(s) < n
    w4 = I.long_128k_64layer()
    assert w4.num_layers == 64 and w4.seq_lens == [131072] and w4.page_size == 128
    for l in range(8):
        assert w4.head_class[l] == [I.LOCAL] * 8 and w4.window[l] == 4096
    for l in range(8, 64):
        assert w4.window[l] == 1024 and sum(c == I.GLOBAL for c in w4.head_class[l]) in (0, 1)
    w5 = I.ragged_decode()
    assert len(w5.seq_lens) == 32 and all(2048 <= n < 32768 for n in w5.seq_lens)


def test_sink_rows_scaled_by_8():
    w = I.llama70b_varlen()
    w.seq_lens = [300, 200]
    w.sink_positions = [[3, 100], [0]]
    q, k, v, cu, qp = I.prefill_tensors(w)
    w.sink_positions = []
    _, k0, _, _, _ = I.prefill_tensors(w)
    assert torch.equal(k[3].float(), 8 * k0[3].float())
    assert torch.equal(k[300].float(), 8 * k0[300].float())
    assert torch.equal(k[4], k0[4])


def test_row_subset_matches_full_draw():
    full = I.normal_bf16(3, 44, (50, 3, 8))
    rows = [0, 7, 49, 7]
    sub = I.normal_bf16_rows(3, 44, (50, 3, 8), rows)
    assert torch.equal(sub.view(torch.int16), full[rows].view(torch.int16))
