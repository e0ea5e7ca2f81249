"""C ABI without a GPU: exported symbols, and the host-side segment allocator
and page-table builder compared bit-exactly with the oracle's page model.

A host-only handle (no pools) runs the library's real planner and tables but
launches nothing, so the allocator can be checked on any machine.
"""
import ctypes
import os
import random
import re

import numpy as np
import pytest

import head_segmented_paged_gb300 as S
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^\s*(?:int|const char\*)\s+(segkv_\w+)\s*\(", txt, re.M))
    return names


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert {"segkv_create", "segkv_append", "segkv_prefill_attn", "segkv_decode_attn"} <= names
    lib = ctypes.CDLL(S.LIB_PATH)
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert names <= set(S.SYMBOLS)


def host_handle(L, H, hc, W, P, Smax, max_len, pages, hq=None):
    hq = hq or H * 4
    return S.SegKV(L, hq, H, 64, hc, W, P, Smax, max_len, num_pages=pages)


def same_state(h, m, L, H, Smax):
    for l in range(L):
        for b in range(Smax):
            assert h.seq_len(l, b) == m.seq_len(l, b)
            for hd in range(H):
                assert h.segment(l, hd, b) == m.segment(l, hd, b), (l, hd, b)
    st = h.stats()
    assert st["num_pages"] - st["pages_in_use"] == m.free_pages()


def test_worked_examples_match_golden_and_oracle():
    import json
    ex = json.load(open(os.path.join(ROOT, "tests", "golden", "page_model_examples.json")))
    for e in ex["examples"]:
        s = e["setup"]
        h = host_handle(s["num_layers"], s["num_kv_heads"], s["head_class"], s["window"],
                        s["page_size"], s["max_seqs"], s["max_seq_len"], s["num_pages"])
        m = oracle.PageModel(s["num_layers"], s["num_kv_heads"], s["head_class"], s["window"],
                             s["page_size"], s["max_seqs"], s["max_seq_len"], s["num_pages"])
        for st in e["steps"]:
            if st["op"] == "append":
                rc = S.segkv_append(h.handle, st["layer"], None, None, st["cu_seqlens"],
                                    st["seq_ids"])
                rm = m.append(st["layer"], st["cu_seqlens"], st["seq_ids"])
            elif st["op"] == "trim":
                rc = S.segkv_trim(h.handle, st["layer"], st["seq_ids"])
                rm = m.trim(st["layer"], st["seq_ids"])
            elif st["op"] == "import":
                hdr = [st["n"]] + list(st["starts"])
                rc = S.segkv_import(h.handle, st["layer"], st["seq"], None, hdr)
                rm = m.import_segment(st["layer"], st["seq"], st["n"], st["starts"])
            else:
                rc = S.segkv_free_seq(h.handle, st["seq"])
                rm = m.free_seq(st["seq"])
            assert rc == rm == st["status"]
            for x in st.get("expect", []):
                got = h.segment(x["layer"], x["head"], x["seq"])
                assert got == (x["start"], x["len"], x["first_page"], x["ids"])
            same_state(h, m, s["num_layers"], s["num_kv_heads"], s["max_seqs"])


@pytest.mark.parametrize("seed", range(8))
def test_random_scripts_bit_exact_with_oracle(seed):
    rnd = random.Random(100 + seed)
    L, H, Smax = rnd.choice([1, 2]), rnd.choice([1, 2, 4]), rnd.choice([1, 3, 5])
    P = rnd.choice([8, 16, 32, 64, 128, 256])
    hc = [[rnd.randint(0, 1) for _ in range(H)] for _ in range(L)]
    W = [rnd.choice([1, 5, 33, 100, 1000]) for _ in range(L)]
    max_len = rnd.choice([300, 1000, 2048])
    pages = rnd.choice([10, 50, 200, 5000])
    h = host_handle(L, H, hc, W, P, Smax, max_len, pages)
    m = oracle.PageModel(L, H, hc, W, P, Smax, max_len, pages)
    for _ in range(150):
        op = rnd.random()
        l = rnd.randrange(L)
        if op < 0.65:
            ids = rnd.sample(range(Smax), rnd.randint(1, Smax))
            ts = [rnd.choice([0, 1, 1, 3, 8, 31, 64, 200]) for _ in ids]
            cu = np.concatenate([[0], np.cumsum(ts)]).astype(np.int32)
            rc = S.segkv_append(h.handle, l, None, None, cu, ids)
            assert rc == m.append(l, cu, ids)
        elif op < 0.85:
            ids = rnd.sample(range(Smax), rnd.randint(1, Smax))
            tl = rnd.choice([-1, l])
            assert S.segkv_trim(h.handle, tl, ids) == m.trim(tl, ids) == 0
        elif op < 0.93:
            b = rnd.randrange(Smax)
            assert S.segkv_free_seq(h.handle, b) == m.free_seq(b) == 0
        else:  # import a transferred segment set, valid or not
            b = rnd.randrange(Smax)
            n = rnd.choice([0, 1, 17, 100, 300, max_len + 1])
            starts = [rnd.randint(0, max(n, 0)) if rnd.random() < 0.5 else 0 for _ in range(H)]
            rc = S.segkv_import(h.handle, l, b, None, [n] + starts)
            assert rc == m.import_segment(l, b, n, starts)
        same_state(h, m, L, H, Smax)


def test_out_of_pages_and_bad_args_are_transactional():
    h = host_handle(1, 2, [[0, 1]], [8], 16, 2, 256, 10)
    assert S.segkv_append(h.handle, 0, None, None, [0, 64], [0]) == 0  # 8 pages
    before = [h.segment(0, hd, b) for hd in range(2) for b in range(2)]
    assert S.segkv_append(h.handle, 0, None, None, [0, 32], [1]) == S.SEGKV_ERR_OUT_OF_PAGES
    assert S.segkv_append(h.handle, 0, None, None, [0, 300], [1]) == S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_append(h.handle, 0, None, None, [0, 1, 2], [1, 1]) == S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_append(h.handle, 1, None, None, [0, 1], [1]) == S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_append(h.handle, 0, None, None, [0, 1], [2]) == S.SEGKV_ERR_INVALID_ARG
    assert "max_seq" in S.segkv_last_error(h.handle) or S.segkv_last_error(h.handle)
    after = [h.segment(0, hd, b) for hd in range(2) for b in range(2)]
    assert before == after


def test_create_rejects_bad_shapes():
    ok = dict(num_layers=1, num_q_heads=8, num_kv_heads=2, head_dim=64, head_class=[0, 1],
              window=[4], page_size=16, max_seqs=1, max_seq_len=64, k_pool=None, v_pool=None,
              num_pages=8)
    rc, h = S.segkv_create(**ok)
    assert rc == 0
    S.segkv_destroy(h)
    for bad in [dict(head_dim=96), dict(page_size=24), dict(page_size=4), dict(num_q_heads=6),
                dict(window=[0]), dict(head_class=[0, 2]), dict(num_pages=0),
                dict(num_q_heads=64, num_kv_heads=2)]:
        rc, _ = S.segkv_create(**{**ok, **bad})
        assert rc == S.SEGKV_ERR_INVALID_ARG, bad
        assert S.segkv_last_error(None)


def test_workspace_size_and_host_only_attention_refused():
    h = host_handle(1, 2, [[0, 1]], [8], 16, 4, 1000, 100)
    assert h.workspace_size(S.SEGKV_WS_PREFILL, 100, 4) == 0
    ws = h.workspace_size(S.SEGKV_WS_DECODE, 0, 4)
    G, D, units = 4, 64, 4 * 2 * (2 + 1)
    assert ws >= units * G * D * 4 + units * G * 8
    # T query tokens per sequence: T * G rows per KV head; past 16 rows the
    # prefill kernel serves the call and needs none
    assert h.workspace_size(S.SEGKV_WS_DECODE, 4, 4) == ws
    assert h.workspace_size(S.SEGKV_WS_DECODE, 16, 4) >= 4 * ws - 1024
    assert h.workspace_size(S.SEGKV_WS_DECODE, 12, 4) == 0  # 12 rows
    assert h.workspace_size(S.SEGKV_WS_DECODE, 32, 4) == 0  # 32 rows
    rc = S.segkv_prefill_attn(h.handle, 0, None, [0, 1], [0], [0], None)
    assert rc == S.SEGKV_ERR_INVALID_ARG


def test_stats_count_pages_by_class():
    h = host_handle(1, 2, [[0, 1]], [16], 16, 1, 512, 100)
    h.append(0, None, None, [0, 100], [0])
    st = h.stats()
    assert st["pages_global"] == 7 and st["pages_local"] == 7 and st["kept_tokens"] == 200
    h.trim(0, [0])
    st = h.stats()
    # local head keeps positions 85..99: pages 5 and 6
    assert st["pages_local"] == 2 and st["kept_tokens"] == 100 + 15


def test_fa_window_convention_equals_inclusive_window_plus_one():
    # FlashAttention's window (W, 0) covers W+1 keys; the kept sets and pages
    # must equal those of the inclusive reading with W+1 (oracle page model).
    rnd = random.Random(7)
    W, P = 20, 8
    fa = host_handle(1, 2, [[0, 1]], [W], P, 2, 500, 300)
    fa.set_window_convention(S.SEGKV_WINDOW_FA)
    m = oracle.PageModel(1, 2, [[0, 1]], [W + 1], P, 2, 500, 300)
    for _ in range(60):
        ids = rnd.sample(range(2), rnd.randint(1, 2))
        ts = [rnd.choice([1, 3, 9, 30]) for _ in ids]
        cu = np.concatenate([[0], np.cumsum(ts)]).astype(np.int32)
        assert S.segkv_append(fa.handle, 0, None, None, cu, ids) == m.append(0, cu, ids)
        if rnd.random() < 0.3:
            assert S.segkv_trim(fa.handle, 0, ids) == m.trim(0, ids)
        same_state(fa, m, 1, 2, 2)
    # only while empty
    assert S.segkv_set_window_convention(fa.handle, S.SEGKV_WINDOW_INCLUSIVE) == \
        S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_set_window_convention(fa.handle, 7) == S.SEGKV_ERR_INVALID_ARG


def test_plain_c_caller_compiles_against_the_header_and_runs(tmp_path):
    """`tests/c/abi_host_check.c` includes `include/segkv.h` from C99 (strict,
    warnings as errors), links the library and drives a host-only handle:
    append, trim, segment and page counts, a decode plan's key coverage, and
    refused calls that change nothing."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_host_check")
    lib_dir = os.path.dirname(S.LIB_PATH)
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_host_check.c"), S.LIB_PATH, f"-Wl,-rpath,{lib_dir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
