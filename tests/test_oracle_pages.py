"""Pins for the oracle's page model: hand-derived states and invariants.

The kept sets follow the RedKnot summary page (sections "头分类稀疏" and
"SegPagedAttention"); the allocator order and eviction timing are the
readings stated in tests/golden/page_model_examples.json.
"""
import json
import os
import random

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_model_examples.json")


def _examples():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


def apply_step(m, st):
    if st["op"] == "append":
        return m.append(st["layer"], st["cu_seqlens"], st["seq_ids"])
    if st["op"] == "trim":
        return m.trim(st["layer"], st["seq_ids"])
    if st["op"] == "free_seq":
        return m.free_seq(st["seq"])
    if st["op"] == "import":
        return m.import_segment(st["layer"], st["seq"], st["n"], st["starts"])
    raise ValueError(st["op"])


@pytest.mark.parametrize("ex", _examples(), ids=lambda e: e["name"])
def test_hand_derived_examples(ex):
    s = ex["setup"]
    m = oracle.PageModel(s["num_layers"], s["num_kv_heads"], s["head_class"], s["window"],
                         s["page_size"], s["max_seqs"], s["max_seq_len"], s["num_pages"])
    for st in ex["steps"]:
        assert apply_step(m, st) == st["status"], st
        if "free_pages" in st:
            assert m.free_pages() == st["free_pages"], st
        for e in st.get("expect", []):
            got = m.segment(e["layer"], e["head"], e["seq"])
            assert got == (e["start"], e["len"], e["first_page"], e["ids"]), (st, e)


def check_invariants(m, L, H, S, P, W, hc, num_pages, lens, starts):
    held = []
    for l in range(L):
        for b in range(S):
            n = m.seq_len(l, b)
            assert n == lens[l][b]
            for h in range(H):
                s, ln, first, ids = m.segment(l, h, b)
                assert s + ln == n
                assert s == starts[l][h][b]
                # exactly the pages floor(s/P) .. floor((n-1)/P): every page that
                # holds a kept key, plus a partly filled page the next token uses
                want = 0 if n == 0 else max(0, (n - 1) // P - s // P + 1)
                assert len(ids) == want
                if want:
                    assert first == s // P
                held.extend(ids)
    assert len(held) == len(set(held)), "a page id is held twice"
    assert all(0 <= i < num_pages for i in held)
    assert m.free_pages() + len(held) == num_pages


@pytest.mark.parametrize("seed", range(6))
def test_random_scripts_keep_invariants(seed):
    rnd = random.Random(seed)
    L, H, S, P = 2, 3, 3, rnd.choice([4, 8, 16])
    hc = [[rnd.randint(0, 1) for _ in range(H)] for _ in range(L)]
    W = [rnd.choice([1, 3, 8, 20]) for _ in range(L)]
    num_pages = rnd.choice([20, 60, 400])
    max_len = 200
    m = oracle.PageModel(L, H, hc, W, P, S, max_len, num_pages)
    lens = [[0] * S for _ in range(L)]
    starts = [[[0] * S for _ in range(H)] for _ in range(L)]
    for _ in range(120):
        op = rnd.random()
        l = rnd.randrange(L)
        if op < 0.6:
            k = rnd.randint(1, S)
            ids = rnd.sample(range(S), k)
            ts = [rnd.choice([0, 1, 1, 2, 5, 17, 40]) for _ in ids]
            cu = [0]
            for t in ts:
                cu.append(cu[-1] + t)
            before = m.free_pages()
            rc = m.append(l, cu, ids)
            if any(lens[l][b] + t > max_len for b, t in zip(ids, ts)):
                assert rc == oracle.INVALID_ARG
                assert m.free_pages() == before
                continue
            if rc == oracle.OUT_OF_PAGES:
                assert m.free_pages() == before
                continue
            assert rc == oracle.OK
            for b, t in zip(ids, ts):
                a = lens[l][b]
                for h in range(H):
                    if hc[l][h] == 1:
                        starts[l][h][b] = max(starts[l][h][b], a - W[l] + 1, 0)
                lens[l][b] = a + t
        elif op < 0.8:
            ids = rnd.sample(range(S), rnd.randint(1, S))
            tl = rnd.choice([-1, l])
            assert m.trim(tl, ids) == oracle.OK
            for ll in (range(L) if tl == -1 else [tl]):
                for b in ids:
                    for h in range(H):
                        if hc[ll][h] == 1:
                            starts[ll][h][b] = max(starts[ll][h][b], lens[ll][b] - W[ll] + 1, 0)
        else:
            b = rnd.randrange(S)
            assert m.free_seq(b) == oracle.OK
            for ll in range(L):
                lens[ll][b] = 0
                for h in range(H):
                    starts[ll][h][b] = 0
        check_invariants(m, L, H, S, P, W, hc, num_pages, lens, starts)


def test_lowest_free_ids_first_after_scattered_frees():
    # Pages freed in any order come back lowest id first.
    m = oracle.PageModel(1, 1, [[0]], [4], 4, 4, 64, 16)
    for b in range(4):
        assert m.append(0, [0, 16], [b]) == oracle.OK  # 4 pages each: ids 4b..4b+3
    assert m.free_pages() == 0
    assert m.free_seq(2) == oracle.OK
    assert m.free_seq(0) == oracle.OK
    assert m.append(0, [0, 5, 10], [2, 0]) == oracle.OK
    assert m.segment(0, 0, 2)[3] == [0, 1]
    assert m.segment(0, 0, 0)[3] == [2, 3]


def test_invalid_arguments_change_nothing():
    m = oracle.PageModel(1, 2, [[0, 1]], [8], 4, 2, 32, 64)
    assert m.append(0, [0, 4], [5]) == oracle.INVALID_ARG        # seq out of range
    assert m.append(0, [0, 4, 8], [1, 1]) == oracle.INVALID_ARG  # duplicate seq
    assert m.append(0, [0, 40], [0]) == oracle.INVALID_ARG       # beyond max length
    assert m.append(1, [0, 4], [0]) == oracle.INVALID_ARG        # bad layer
    assert m.append(0, [1, 4], [0]) == oracle.INVALID_ARG        # cu_seqlens[0] != 0
    assert m.free_pages() == 64
    assert m.segment(0, 0, 0) == (0, 0, 0, [])
