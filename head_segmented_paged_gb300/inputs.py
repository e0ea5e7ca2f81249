"""Seeded synthetic inputs for segmented paged attention.

This module only draws numbers and lays out workloads; it holds none of the
attention or paging arithmetic, so both the CUDA path and the CPU oracle can
consume the same buffers.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) run in counter mode, one independent stream
per (seed, stream id). Two 53-bit uniforms feed one Box-Muller draw in fp64;
the fp64 value (times an optional fp64 scale) is rounded straight to bf16 with
round-to-nearest-even by integer arithmetic on its bit pattern, so no fp32
double rounding occurs.

Workload recipes follow the shapes the RedKnot summary page describes for
long-context prefill and decode (page "让 KV Cache「按头分家」", sections
"头分类稀疏" and "系统收益"): 8K-128K contexts, GQA models with
a small share of global heads and sliding-window local heads.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_MASK64 = (1 << 64) - 1


def _s64(c: int) -> int:
    """Unsigned 64-bit constant as a two's complement int64."""
    c &= _MASK64
    return c - (1 << 64) if c >= (1 << 63) else c


_GAMMA = _s64(0x9E3779B97F4A7C15)
_M1 = _s64(0xBF58476D1CE4E5B9)
_M2 = _s64(0x94D049BB133111EB)


def _lsr(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 viewed as uint64."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _M1
    z = (z ^ _lsr(z, 27)) * _M2
    return z ^ _lsr(z, 31)


def _mix_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """Key of one independent splitmix64 stream."""
    return _mix_int((seed * 0x100000001B3) ^ _mix_int(stream + 0x632BE59BD9B4E019))


def raw_u64(seed: int, stream: int, count: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """Draws offset .. offset+count-1 of a stream, as int64 bit patterns."""
    key = _s64(stream_key(seed, stream))
    i = torch.arange(offset + 1, offset + count + 1, dtype=torch.int64, device=device)
    return _mix(key + i * _GAMMA)


def uniform01(seed: int, stream: int, count: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """fp64 uniforms in [0, 1) with 53 random bits each."""
    x = _lsr(raw_u64(seed, stream, count, device, offset), 11)
    return x.to(torch.float64) * (2.0 ** -53)


def f64_to_bf16_rne(x: torch.Tensor) -> torch.Tensor:
    """Round fp64 to bf16, nearest-even, in one step (normal range)."""
    bits = x.view(torch.int64)
    sign = bits & _s64(1 << 63)
    mag = bits & ((1 << 63) - 1)
    lsb = (mag >> 45) & 1
    mag = (mag + ((1 << 44) - 1) + lsb) & ~((1 << 45) - 1)
    y = (mag | sign).view(torch.float64)
    return y.to(torch.float32).to(torch.bfloat16)


def _normal_range(seed: int, stream: int, start: int, count: int, scale: float, device):
    """Elements start .. start+count-1 of the normal stream, as bf16."""
    u = uniform01(seed, stream, 2 * count, device, offset=2 * start).view(count, 2)
    z = torch.sqrt(-2.0 * torch.log1p(-u[:, 0])) * torch.cos((2.0 * math.pi) * u[:, 1])
    if scale != 1.0:
        z = z * scale
    return f64_to_bf16_rne(z)


def normal_bf16(seed: int, stream: int, shape, scale: float = 1.0, device="cpu",
                chunk: int | None = None) -> torch.Tensor:
    """N(0,1)*scale drawn in fp64 and rounded once to bf16."""
    n = 1
    for s in shape:
        n *= int(s)
    if chunk is None:  # cache-sized chunks on the host, large ones on a GPU
        chunk = (1 << 26) if torch.device(device).type == "cuda" else (1 << 20)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for c0 in range(0, n, chunk):
        c = min(chunk, n - c0)
        out[c0:c0 + c] = _normal_range(seed, stream, c0, c, scale, device)
    return out.view(*shape)


def normal_bf16_rows(seed: int, stream: int, shape, rows, scale: float = 1.0) -> torch.Tensor:
    """Only the listed leading-index rows of normal_bf16(seed, stream, shape),
    bit for bit, without drawing the rest."""
    inner = 1
    for s in shape[1:]:
        inner *= int(s)
    out = torch.empty((len(rows), inner), dtype=torch.bfloat16)
    for i, r in enumerate(rows):
        out[i] = _normal_range(seed, stream, int(r) * inner, inner, scale, "cpu")
    return out.view(len(rows), *shape[1:])


def randint_list(seed: int, stream: int, count: int, lo: int, hi: int) -> list[int]:
    """count integers uniform in [lo, hi] (inclusive), by 53-bit uniforms."""
    u = uniform01(seed, stream, count).tolist()
    span = hi - lo + 1
    return [lo + min(span - 1, int(v * span)) for v in u]


def sample_without_replacement(seed: int, stream: int, n: int, k: int) -> list[int]:
    """k distinct values of range(n), by a partial Fisher-Yates shuffle."""
    perm = list(range(n))
    u = uniform01(seed, stream, k).tolist()
    for i in range(k):
        j = i + min(n - i - 1, int(u[i] * (n - i)))
        perm[i], perm[j] = perm[j], perm[i]
    return perm[:k]


GLOBAL, LOCAL = 0, 1


@dataclass
class Workload:
    """One synthetic workload: geometry, head classes and sequence lengths."""
    name: str
    num_layers: int
    hq: int
    hkv: int
    head_dim: int
    page_size: int
    head_class: list  # [L][Hkv] of GLOBAL/LOCAL
    window: list      # [L]
    seq_lens: list    # per sequence
    qk_scale_inputs: float = 1.0   # input distribution scale for Q/K/V
    sink_positions: list = field(default_factory=list)  # per sequence, K rows x8
    decode_steps: int = 0
    seed: int = 0

    @property
    def group(self) -> int:
        return self.hq // self.hkv


# stream ids: (tensor kind, layer) -> stream; kinds are fixed small integers
_Q, _K, _V, _QD, _KD, _VD = 1, 2, 3, 4, 5, 6


def tensor_stream(kind: int, layer: int, extra: int = 0) -> int:
    return (kind << 40) | (layer << 20) | extra


def tiny_256() -> Workload:
    """1 layer, 8 query / 2 KV heads, D=64, one 256-token sequence; KV head 0
    global, KV head 1 local with window 32; pages of 16 tokens."""
    return Workload("tiny-256", 1, 8, 2, 64, 16, [[GLOBAL, LOCAL]], [32], [256])


def mistral_8k(seed: int = 0) -> Workload:
    """Mistral-7B-shaped single layer: 32/8 heads, D=128, 8192 tokens, one
    seeded global KV head, 7 local heads with window 1024, pages of 64."""
    g = randint_list(seed, 100, 1, 0, 7)[0]
    hc = [[GLOBAL if h == g else LOCAL for h in range(8)]]
    return Workload("mistral-8k", 1, 32, 8, 128, 64, hc, [1024], [8192],
                    qk_scale_inputs=1.0 / math.sqrt(128.0), seed=seed)


def llama70b_varlen(seed: int = 0) -> Workload:
    """Llama-3.3-70B-shaped varlen prefill: 64/8 heads, D=128, 4 sequences of
    16K-32K tokens, one seeded global KV head, window 2048, pages of 64, and
    round(1% of each length) key rows scaled by 8 (attention sinks)."""
    lens = randint_list(seed, 200, 4, 16384, 32768)
    g = randint_list(seed, 201, 1, 0, 7)[0]
    hc = [[GLOBAL if h == g else LOCAL for h in range(8)]]
    sinks = []
    for b, n in enumerate(lens):
        k = int(round(0.01 * n))
        sinks.append(sorted(sample_without_replacement(seed, 210 + b, n, k)))
    return Workload("llama70b-varlen", 1, 64, 8, 128, 64, hc, [2048], lens,
                    sink_positions=sinks, seed=seed)


def long_128k_64layer(seed: int = 0, all_global: bool = False) -> Workload:
    """64 layers x (64/8 heads, D=128), one 131072-token sequence, pages of 128.
    Layers 0-7: all heads local, window 4096. Layers 8-63: global fraction
    f ~ U[0.03, 0.17], g = round-half-even(8 f) global KV heads drawn without
    replacement, window 1024. all_global=True gives the dense full-causal path
    of the same shape."""
    L = 64
    f = uniform01(seed, 300, L).tolist()
    hc, win = [], []
    for l in range(L):
        if all_global:
            hc.append([GLOBAL] * 8)
            win.append(131072)
            continue
        if l < 8:
            hc.append([LOCAL] * 8)
            win.append(4096)
            continue
        frac = 0.03 + 0.14 * f[l]
        g = int(round(frac * 8))  # Python round() is half-even
        glob = set(sample_without_replacement(seed, 400 + l, 8, g))
        hc.append([GLOBAL if h in glob else LOCAL for h in range(8)])
        win.append(1024)
    return Workload("128k-64layer-dense" if all_global else "128k-64layer", L, 64, 8, 128,
                    128, hc, win, [131072], seed=seed)


def ragged_decode(seed: int = 0, steps: int = 128) -> Workload:
    """32 requests with context lengths floor(exp(U[ln 2048, ln 32768])),
    32/8 heads, D=128, 1 seeded global + 7 local heads (window 1024), pages of
    64, one decode token per request per step."""
    u = uniform01(seed, 500, 32).tolist()
    lens = [int(math.floor(math.exp(math.log(2048) + v * (math.log(32768) - math.log(2048)))))
            for v in u]
    g = randint_list(seed, 501, 1, 0, 7)[0]
    hc = [[GLOBAL if h == g else LOCAL for h in range(8)]]
    return Workload("ragged-decode", 1, 32, 8, 128, 64, hc, [1024], lens,
                    decode_steps=steps, seed=seed)


def prefill_tensors(w: Workload, layer: int = 0, device="cpu"):
    """Packed Q [sum n, Hq, D], K and V [sum n, Hkv, D] (bf16) for a full
    prefill of every sequence, plus cu_seqlens and q_pos (int32, CPU)."""
    tot = sum(w.seq_lens)
    s = w.qk_scale_inputs
    q = normal_bf16(w.seed, tensor_stream(_Q, layer), (tot, w.hq, w.head_dim), s, device)
    k = normal_bf16(w.seed, tensor_stream(_K, layer), (tot, w.hkv, w.head_dim), s, device)
    v = normal_bf16(w.seed, tensor_stream(_V, layer), (tot, w.hkv, w.head_dim), s, device)
    cu = [0]
    for n in w.seq_lens:
        cu.append(cu[-1] + n)
    if w.sink_positions:
        for b, pos in enumerate(w.sink_positions):
            if pos:
                idx = torch.tensor(pos, dtype=torch.int64, device=device) + cu[b]
                k[idx] = k[idx] * 8  # x8 is exact in bf16
    cu_t = torch.tensor(cu, dtype=torch.int32)
    q_pos = torch.cat([torch.arange(n, dtype=torch.int32) for n in w.seq_lens])
    return q, k, v, cu_t, q_pos


def decode_step_tensors(w: Workload, step: int, device="cpu"):
    """One decode step: q [B, Hq, D] and the new token's k, v [B, Hkv, D]."""
    B = len(w.seq_lens)
    s = w.qk_scale_inputs
    q = normal_bf16(w.seed, tensor_stream(_QD, 0, step), (B, w.hq, w.head_dim), s, device)
    k = normal_bf16(w.seed, tensor_stream(_KD, 0, step), (B, w.hkv, w.head_dim), s, device)
    v = normal_bf16(w.seed, tensor_stream(_VD, 0, step), (B, w.hkv, w.head_dim), s, device)
    return q, k, v


# ---- sparse FFN routing -------------------------------------------------------
_X, _RES, _WG, _WU, _WD = 7, 8, 9, 10, 11


@dataclass
class FfnWorkload:
    """One FFN layer over a prefill chunk: n tokens, hidden d_model, FFN
    width d_ff, m chosen tokens. Synthetic: x and the residual are N(0,1)
    (the FFN input is a normalised hidden state), weights N(0,1)/sqrt(fan_in)."""
    name: str
    n: int
    d_model: int
    d_ff: int
    m: int
    seed: int = 0


def mistral_ffn(seed: int = 0) -> FfnWorkload:
    """Mistral-7B FFN shape (hidden 4096, SwiGLU width 14336) over the 8192
    tokens of the Mistral-shaped prefill, a quarter of them chosen."""
    return FfnWorkload("mistral-ffn-8k", 8192, 4096, 14336, 2048, seed)


def ffn_tensors(w: FfnWorkload, device="cpu"):
    """x, residual [n, d_model]; w_gate, w_up [d_ff, d_model]; w_down [d_model, d_ff] (bf16)."""
    x = normal_bf16(w.seed, tensor_stream(_X, 0), (w.n, w.d_model), 1.0, device)
    r = normal_bf16(w.seed, tensor_stream(_RES, 0), (w.n, w.d_model), 1.0, device)
    wg = normal_bf16(w.seed, tensor_stream(_WG, 0), (w.d_ff, w.d_model), w.d_model ** -0.5, device)
    wu = normal_bf16(w.seed, tensor_stream(_WU, 0), (w.d_ff, w.d_model), w.d_model ** -0.5, device)
    wd = normal_bf16(w.seed, tensor_stream(_WD, 0), (w.d_model, w.d_ff), w.d_ff ** -0.5, device)
    return x, r, wg, wu, wd
