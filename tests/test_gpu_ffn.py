"""Sparse FFN (gather -> SwiGLU GEMM -> W_down GEMM -> scatter-add into the
residual) through the C ABI, against the fp64 oracle.

Tolerance, derived from the arithmetic: inputs and weights are exact bf16,
accumulation is fp32 (error well under 1e-3 here), the hidden activation h is
rounded to bf16 (unit roundoff 2^-8) before W_down, and the result is rounded
once to bf16. With the rounding errors of h independent and uniform, the
error of y_d has standard deviation sigma_d = 2^-8/sqrt(3) *
sqrt(sum_f (W_down[d,f] h_f)^2). Each element must satisfy
|gpu - ref| <= 2^-8 |ref| + 6 sigma_d + 1e-3, and the mean error must stay
below 2^-8 times the mean |ref|.
"""
import numpy as np
import pytest
import torch

import head_segmented_paged_gb300 as S
from head_segmented_paged_gb300 import inputs as I
from oracle import sparse_ffn as F

pytestmark = pytest.mark.gpu


def handle():
    kp = torch.empty((4, 16, 64), dtype=torch.bfloat16, device="cuda")
    return S.SegKV(1, 8, 2, 64, [[0, 1]], [32], 16, 1, 64, kp, kp.clone())


def check_ffn(got, ref, h, wd, rows, what):
    got = got.to(torch.float64).cpu().numpy()[rows]
    ref = ref[rows]
    sig = 2.0 ** -8 / np.sqrt(3) * np.sqrt((h ** 2) @ (wd.astype(np.float64) ** 2).T)
    bound = 2.0 ** -8 * np.abs(ref) + 6 * sig + 1e-3
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements out of bound, worst {err.max()}"
    assert err.mean() <= 2.0 ** -8 * np.abs(ref).mean(), f"{what}: mean error {err.mean()}"


def run_case(n, d_model, d_ff, m, seed, dense=False):
    w = I.FfnWorkload("t", n, d_model, d_ff, m, seed)
    x, r, wg, wu, wd = I.ffn_tensors(w, device="cuda")
    h = handle()
    if dense:
        idx = None
        sel = np.arange(n)
    else:
        g = torch.Generator().manual_seed(seed)
        sel = np.sort(torch.randperm(n, generator=g)[:m].numpy())
        idx = torch.tensor(sel, dtype=torch.int32, device="cuda")
    out = r.clone()
    h.sparse_ffn(x, out, idx, wg, wu, wd)
    assert h.status() == 0
    xc, rc_, wgc, wuc, wdc = (t.to(torch.float64).cpu().numpy() for t in (x, r, wg, wu, wd))
    ref, hh = F.sparse_ffn(xc, rc_, sel, wgc, wuc, wdc)
    check_ffn(out, ref, hh, wdc, sel, f"ffn n={n} dm={d_model} dff={d_ff} m={m}")
    rest = np.setdiff1d(np.arange(n), sel)
    assert torch.equal(out[torch.as_tensor(rest, device="cuda")].view(torch.int16),
                       r[torch.as_tensor(rest, device="cuda")].view(torch.int16))
    return out, r, (x, wg, wu, wd), sel, h


@pytest.mark.parametrize("n,d_model,d_ff,m", [(300, 256, 512, 150), (130, 320, 384, 129),
                                               (64, 192, 128, 1), (513, 512, 1024, 513)])
def test_sparse_ffn_small_shapes(n, d_model, d_ff, m):
    # ragged row tiles, a d_model that is not a multiple of the 256-column tile,
    # a single row and every row chosen
    run_case(n, d_model, d_ff, m, seed=n)


def test_dense_equals_all_rows_chosen():
    out_s, r, (x, wg, wu, wd), sel, h = run_case(200, 256, 256, 200, seed=3)
    out_d = r.clone()
    h.sparse_ffn(x, out_d, None, wg, wu, wd)
    assert h.status() == 0
    assert torch.equal(out_d.view(torch.int16), out_s.view(torch.int16))


def test_mistral_shape_reduced_rows():
    run_case(1024, 4096, 14336, 256, seed=11)


def test_mistral_full_size_sampled_rows():
    # the benchmark's workload; the oracle recomputes 48 of the chosen rows
    w = I.mistral_ffn()
    x, r, wg, wu, wd = I.ffn_tensors(w, device="cuda")
    h = handle()
    g = torch.Generator().manual_seed(1)
    sel = np.sort(torch.randperm(w.n, generator=g)[:w.m].numpy())
    idx = torch.tensor(sel, dtype=torch.int32, device="cuda")
    out = r.clone()
    h.sparse_ffn(x, out, idx, wg, wu, wd)
    assert h.status() == 0
    pick = sel[np.linspace(0, len(sel) - 1, 48).astype(int)]
    xc = x[torch.as_tensor(pick, device="cuda")].to(torch.float64).cpu().numpy()
    rc_ = r[torch.as_tensor(pick, device="cuda")].to(torch.float64).cpu().numpy()
    wgc, wuc, wdc = (t.to(torch.float64).cpu().numpy() for t in (wg, wu, wd))
    ref, hh = F.sparse_ffn(xc, rc_, np.arange(len(pick)), wgc, wuc, wdc)
    got = out[torch.as_tensor(pick, device="cuda")]
    check_ffn(got, ref, hh, wdc, np.arange(len(pick)), "mistral ffn sampled")


def test_bad_index_is_reported_and_skipped():
    w = I.FfnWorkload("t", 100, 128, 128, 3, 5)
    x, r, wg, wu, wd = I.ffn_tensors(w, device="cuda")
    h = handle()
    idx = torch.tensor([5, 100, 7], dtype=torch.int32, device="cuda")  # 100 is out of range
    out = r.clone()
    h.sparse_ffn(x, out, idx, wg, wu, wd)
    assert h.status() == S.SEGKV_ERR_INVALID_ARG
    assert h.status() == 0  # cleared
    keep = [i for i in range(100) if i not in (5, 7)]
    assert torch.equal(out[keep].view(torch.int16), r[keep].view(torch.int16))
