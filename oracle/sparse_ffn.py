"""Oracle for sparse FFN token routing. TEST INFRASTRUCTURE ONLY.

RedKnot summary page, section "稀疏 FFN（Sparse FFN）": only the top-k tokens
by attention score go through the dense FFN; every other token takes the
residual identity path. The page gives neither the score, the FFN form nor
the tie rule; the readings taken here:
  * a token's score is the attention mass it receives as a key (see
    ``oracle.attn_mass``), summed over the KV heads;
  * top-k: the k largest scores, ties to the lower position; the chosen
    positions are returned in ascending order;
  * the FFN is the gated SwiGLU MLP of the models the page names:
    FFN(x) = W_down (silu(W_gate x) * (W_up x)), silu(g) = g / (1 + e^-g),
    added to the residual stream of the chosen rows only.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this module; the library never imports it.
"""
from __future__ import annotations

import numpy as np


def topk_tokens(score, k):
    """Positions of the k largest values of score (1-D), ties to the lower
    position, in ascending order. score is compared exactly as given."""
    score = np.asarray(score, dtype=np.float64)
    n = score.shape[0]
    if not 0 <= k <= n:
        raise ValueError("k out of range")
    order = sorted(range(n), key=lambda t: (-score[t], t))
    return np.array(sorted(order[:k]), dtype=np.int64)


def silu(g):
    return g / (1.0 + np.exp(-g))


def swiglu_rows(x, w_gate, w_up, w_down):
    """fp64 SwiGLU FFN of the rows of x [m, d_model]: returns (y [m, d_model],
    h [m, d_ff]) with h = silu(x W_gate^T) * (x W_up^T) and y = h W_down^T."""
    x = np.asarray(x, dtype=np.float64)
    g = x @ np.asarray(w_gate, dtype=np.float64).T
    u = x @ np.asarray(w_up, dtype=np.float64).T
    h = silu(g) * u
    return h @ np.asarray(w_down, dtype=np.float64).T, h


def sparse_ffn(x, residual, idx, w_gate, w_up, w_down):
    """residual + FFN(x) on the rows idx, residual unchanged elsewhere (fp64).
    Returns (out [n, d_model], h [len(idx), d_ff])."""
    out = np.array(residual, dtype=np.float64, copy=True)
    idx = np.asarray(idx, dtype=np.int64)
    if len(idx) == 0:
        return out, np.zeros((0, np.asarray(w_gate).shape[0]))
    y, h = swiglu_rows(np.asarray(x, dtype=np.float64)[idx], w_gate, w_up, w_down)
    out[idx] += y
    return out, h
