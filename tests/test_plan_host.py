"""Work plans on the host, without a GPU.

`segkv_plan_decode` returns the plan a decode call would launch: the
(sequence, KV head) key ranges cut stream-K style into units, grouped by CTA.
The checks pin what the plan must be for the kernels to be right and
balanced:
- every kept key a query row needs is in exactly one unit;
- a pair's units are consecutive and in key order, and carry the pair's
  bookkeeping;
- each CTA's cost (keys + a charge per unit + a charge per split piece) stays
  within one unit's charges of the most loaded CTA.

`segkv_plan_prefill` returns the prefill plan: one unit per (KV head, chunk of
two Q tiles' tokens), with the chunk's key range, in the order the kernel's
CTAs claim them (CTA c runs unit c first, then each CTA that finishes a unit
takes the next unclaimed one). The checks pin that every (chunk, head)
appears once with the right key range, and the claim order exactly:
descending key tiles, ties in building order.

`segkv_plan_mass` returns the attention-mass plan: one unit per (KV head, key
tile of a chunk) over the query tiles that see its keys, long ones cut into
pieces with their own partial-sum slots, dealt by LPT. The checks pin the
query-tile ranges against the visibility rule, the pieces and slots, and the
exact LPT order.
"""
import numpy as np
import pytest

import head_segmented_paged_gb300 as S
import oracle

GLOBAL, LOCAL = 0, 1


def unit_cost(d, rows):
    # the tensor-core decode kernel (8 or 16 rows of 128 dims) is priced apart
    return 64 if d == 128 and rows in (8, 16) else 128


def split_cost(d, rows):
    return 128 if d == 128 and rows in (8, 16) else 256


def host_handle(hq, hkv, d, hc, W, P, max_seqs, max_len, pages):
    return S.SegKV(1, hq, hkv, d, [hc], [W], P, max_seqs, max_len, num_pages=pages)


def fill(h, lens):
    for b, n in enumerate(lens):
        rc = S.segkv_append(h.handle, 0, None, None, np.array([0, n], np.int32),
                            np.array([b], np.int32))
        assert rc == 0


def check_plan(units, cta, lens, hc, W, T, d, G, num_ctas):
    rows = T * G
    n_units = units.shape[0]
    assert cta[0] == 0 and cta[-1] == n_units and (np.diff(cta) >= 1).all()
    assert len(cta) - 1 <= num_ctas
    hkv = len(hc)
    # each CTA boundary splits at most one range, so the workspace bound
    # (one partial slot per pair plus one per CTA) always holds
    assert n_units <= len(lens) * hkv + (len(cta) - 1) - 1
    # coverage, order and bookkeeping per (sequence index, head)
    for i, n in enumerate(lens):
        for hd in range(hkv):
            sel = np.nonzero((units[:, 0] == i) & (units[:, 1] == hd))[0]
            assert len(sel) >= 1
            assert (np.diff(sel) == 1).all(), "a pair's units are consecutive"
            lo = max(0, n - T - W + 1) if hc[hd] == LOCAL else 0
            assert units[sel[0], 3] == lo and units[sel[-1], 4] == n
            assert (units[sel[1:], 3] == units[sel[:-1], 4]).all(), "pieces tile the range"
            assert (units[sel, 4] > units[sel, 3]).all()
            assert (units[sel, 5] == sel[0]).all() and (units[sel, 6] == len(sel)).all()
            assert (units[sel, 2] == hc[hd]).all() and (units[sel, 7] == n - 1).all()
    # the tensor-core kernel streams whole 128-key tiles: its work is priced in
    # tiles, and a split pair is cut only at tile boundaries
    tiled = d == 128 and rows in (8, 16)
    q = 128 if tiled else 1
    if tiled:
        inner = units[:, 5] != np.arange(len(units))  # not the first piece of its pair
        assert (units[inner, 3] % 128 == 0).all(), "cuts fall on tile boundaries"
    work = ((units[:, 4] - 1) // 128 - units[:, 3] // 128 + 1) * 128 if tiled else units[:, 4] - units[:, 3]
    # balance: a CTA closes only when the next unit's charges and one quantum
    # of work no longer fit
    U = unit_cost(d, rows)
    SPLIT_COST = split_cost(d, rows)
    costs = []
    for c in range(len(cta) - 1):
        us = units[cta[c]:cta[c + 1]]
        split = us[:, 6] > 1
        costs.append(int(work[cta[c]:cta[c + 1]].sum()) + U * len(us) + SPLIT_COST * int(split.sum()))
    costs = np.array(costs)
    assert (costs[:-1] >= costs.max() - U - SPLIT_COST - q).all(), costs


@pytest.mark.parametrize("hq,hkv,d,T", [(32, 8, 128, 1), (32, 8, 128, 4), (64, 8, 128, 2),
                                        (8, 2, 64, 1), (16, 2, 64, 3)])
@pytest.mark.parametrize("num_ctas", [152, 16, 1])
def test_decode_plan_covers_each_needed_key_once_and_balances(hq, hkv, d, T, num_ctas):
    G = hq // hkv
    hc = [GLOBAL] + [LOCAL] * (hkv - 1)
    W, P = 300, 64
    rng = np.random.default_rng(hq * 7 + T)
    lens = [int(x) for x in rng.integers(T, 6000, size=24)] + [T, T + 1, 4097]
    h = host_handle(hq, hkv, d, hc, W, P, len(lens), 8192, 16 * 1024)
    fill(h, lens)
    ids = list(range(len(lens)))
    rc, units, cta = S.segkv_plan_decode(h.handle, 0, T, lens, ids, num_ctas)
    assert rc == 0, S.segkv_last_error(h.handle)
    check_plan(units, cta, lens, hc, W, T, d, G, num_ctas)


def test_decode_plan_after_trim_and_on_a_subset_of_sequences():
    hq, hkv, d = 32, 8, 128
    hc = [LOCAL, GLOBAL, LOCAL, LOCAL, LOCAL, LOCAL, LOCAL, LOCAL]
    W, P = 1024, 64
    lens = [2048, 32768, 5000, 1, 1023, 1024, 1025]
    h = host_handle(hq, hkv, d, hc, W, P, len(lens), 40000, 12000)
    fill(h, lens)
    assert h.trim(0, list(range(len(lens)))) == 0
    # one new token each, then plan for a subset in a shuffled order
    for b in range(len(lens)):
        assert S.segkv_append(h.handle, 0, None, None, np.array([0, 1], np.int32),
                              np.array([b], np.int32)) == 0
    ids = [5, 1, 3, 0]
    sub = [lens[b] + 1 for b in ids]
    rc, units, cta = S.segkv_plan_decode(h.handle, 0, 1, sub, ids, 152)
    assert rc == 0, S.segkv_last_error(h.handle)
    check_plan(units, cta, sub, hc, W, 1, d, hq // hkv, 152)


def test_decode_plan_matches_the_oracle_page_model_key_sets():
    """The keys a plan streams for each (sequence, head) are those the oracle's
    page model keeps and the query sees."""
    hq, hkv, d, W, P = 16, 2, 64, 40, 16
    hc = [GLOBAL, LOCAL]
    lens = [10, 100, 333]
    h = host_handle(hq, hkv, d, hc, W, P, len(lens), 1024, 512)
    m = oracle.PageModel(1, hkv, [hc], [W], P, len(lens), 1024, 512)
    for b, n in enumerate(lens):
        cu = np.array([0, n], np.int32)
        assert S.segkv_append(h.handle, 0, None, None, cu, np.array([b], np.int32)) == 0
        assert m.append(0, cu, [b]) == 0
    assert h.trim(0, [0, 1, 2]) == 0 and m.trim(0, [0, 1, 2]) == 0
    # the next token of each sequence, then its decode
    one = np.array([0, 1, 2, 3], np.int32)
    assert S.segkv_append(h.handle, 0, None, None, one, np.array([0, 1, 2], np.int32)) == 0
    assert m.append(0, one, [0, 1, 2]) == 0
    lens = [n + 1 for n in lens]
    rc, units, cta = S.segkv_plan_decode(h.handle, 0, 1, lens, [0, 1, 2], 4)
    assert rc == 0, S.segkv_last_error(h.handle)
    for i, n in enumerate(lens):
        for hd in range(hkv):
            s, ln, _, _ = m.segment(0, hd, i)
            sel = (units[:, 0] == i) & (units[:, 1] == hd)
            k0, k1 = units[sel, 3].min(), units[sel, 4].max()
            # the query at n - 1 sees [max(0, n - W), n) on a local head, all keys on a global one
            want = max(0, n - W) if hc[hd] == LOCAL else 0
            assert (k0, k1) == (want, n)
            assert s <= k0 and s + ln == n  # every streamed key is kept


def test_decode_plan_errors():
    h = host_handle(8, 2, 64, [GLOBAL, LOCAL], 16, 16, 2, 512, 64)
    fill(h, [100, 5])
    assert S.segkv_plan_decode(h.handle, 0, 1, [99, 5], [0, 1], 8)[0] == S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_plan_decode(h.handle, 0, 6, [100, 5], [0, 1], 8)[0] == S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_plan_decode(h.handle, 1, 1, [100, 5], [0, 1], 8)[0] == S.SEGKV_ERR_INVALID_ARG
    assert h.trim(0, [0]) == 0  # the local head keeps only what position 100 needs
    assert S.segkv_plan_decode(h.handle, 0, 3, [100], [0], 8)[0] == S.SEGKV_ERR_EVICTED
    rc, units, cta = S.segkv_plan_decode(h.handle, 0, 1, [], [], 8)
    assert rc == 0 and units.shape == (0, 8)


# ---------------------------------------------------------------- prefill
@pytest.mark.parametrize("G,hkv", [(1, 2), (4, 8), (8, 8), (16, 2)])
@pytest.mark.parametrize("num_ctas", [152, 7])
def test_prefill_plan_tiles_every_token_and_head_once_longest_first(G, hkv, num_ctas):
    hq, d, P = G * hkv, 128, 64
    hc = [GLOBAL if hd % 4 == 1 else LOCAL for hd in range(hkv)]
    W = 700
    rng = np.random.default_rng(G * 31 + num_ctas)
    lens = [int(x) for x in rng.integers(1, 3000, size=6)] + [1, 4096]
    h = host_handle(hq, hkv, d, hc, W, P, len(lens), 8192, 4 * 8192)
    fill(h, lens)
    # chunked queries: the second half of each sequence, positions shuffled within it
    cu, qp = [0], []
    for n in lens:
        pos = np.arange(n // 2, n, dtype=np.int32)
        rng.shuffle(pos)
        qp.extend(pos.tolist())
        cu.append(cu[-1] + len(pos))
    ids = list(range(len(lens)))
    rc, units, grid = S.segkv_plan_prefill(h.handle, 0, cu, qp, ids, num_ctas)
    assert rc == 0, S.segkv_last_error(h.handle)
    assert grid == min(num_ctas, units.shape[0])
    unit_tok = 2 * (128 // G)
    qp = np.array(qp)
    # every (token chunk, head) exactly once, with the chunk's key range
    seen = set()
    for u in units:
        tok0, ntok, hd, local, kt0, kt1, klo, khi = (int(v) for v in u)
        i = int(np.searchsorted(cu, tok0, side="right")) - 1
        assert (tok0 - cu[i]) % unit_tok == 0 and ntok == min(unit_tok, cu[i + 1] - tok0)
        pos = qp[tok0:tok0 + ntok]
        assert local == (hc[hd] == LOCAL)
        assert khi == pos.max() and klo == (max(0, pos.min() - W + 1) if local else 0)
        assert (kt0, kt1) == (klo // 128, khi // 128)
        assert (tok0, hd) not in seen
        seen.add((tok0, hd))
    want = {(t0, hd) for i in range(len(lens)) for t0 in range(cu[i], cu[i + 1], unit_tok)
            for hd in range(hkv)}
    assert seen == want
    # claimed longest first
    tiles = units[:, 5] - units[:, 4] + 1
    assert (np.diff(tiles) <= 0).all()


def test_prefill_plan_errors():
    h = host_handle(8, 2, 64, [GLOBAL, LOCAL], 16, 16, 2, 512, 64)
    fill(h, [100, 5])
    assert S.segkv_plan_prefill(h.handle, 0, [0, 2], [99, 100], [0], 8)[0] == S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_plan_prefill(h.handle, 0, [0, 1], [0], [3], 8)[0] == S.SEGKV_ERR_INVALID_ARG
    assert h.trim(0, [0]) == 0
    assert S.segkv_plan_prefill(h.handle, 0, [0, 1], [50], [0], 8)[0] == S.SEGKV_ERR_EVICTED
    rc, units, grid = S.segkv_plan_prefill(h.handle, 0, [0], [], [], 8)
    assert rc == 0 and units.shape == (0, 8) and grid == 0


def claim_order(units):
    """The claim order replayed from its definition: units in building order
    (token chunk, then KV head), stably sorted by key tiles, longest first."""
    build = sorted(range(len(units)), key=lambda x: (int(units[x][0]), int(units[x][2])))
    return sorted(build, key=lambda x: -int(units[x][5] - units[x][4]))


@pytest.mark.parametrize("G,hkv,num_ctas", [(4, 8, 152), (8, 8, 7), (1, 2, 3)])
def test_prefill_plan_is_exactly_the_claim_order(G, hkv, num_ctas):
    hq, d, P, W = G * hkv, 128, 64, 500
    hc = [GLOBAL] + [LOCAL] * (hkv - 1)
    rng = np.random.default_rng(G + 5 * hkv + num_ctas)
    lens = [int(x) for x in rng.integers(1, 5000, size=5)]
    h = host_handle(hq, hkv, d, hc, W, P, len(lens), 8192, 4 * 8192)
    fill(h, lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    qp = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    rc, units, grid = S.segkv_plan_prefill(h.handle, 0, cu, qp, list(range(len(lens))), num_ctas)
    assert rc == 0, S.segkv_last_error(h.handle)
    assert grid == min(num_ctas, len(units))
    assert claim_order(units) == list(range(len(units)))


def test_plans_on_a_reused_handle_match_fresh_handles():
    """A handle keeps its plan storage from call to call: a large plan, then a
    small one, then the large one again must each equal the plan a fresh
    handle makes."""
    hq, hkv, d, W, P = 32, 8, 128, 1024, 64
    hc = [GLOBAL] + [LOCAL] * 7
    rng = np.random.default_rng(99)
    lens = [int(x) for x in rng.integers(2048, 20000, size=12)]
    small = [0, 5]

    def make():
        h = host_handle(hq, hkv, d, hc, W, P, len(lens), 20480, 80000)
        fill(h, lens)
        return h

    def dec(h, ids, T):
        rc, u, c = S.segkv_plan_decode(h.handle, 0, T, [lens[b] for b in ids], ids, 152)
        assert rc == 0
        return u, c

    def pre(h, ids):
        cu = np.concatenate([[0], np.cumsum([256 for _ in ids])]).astype(np.int32)
        qp = np.concatenate([np.arange(lens[b] - 256, lens[b]) for b in ids]).astype(np.int32)
        rc, u, c = S.segkv_plan_prefill(h.handle, 0, cu, qp, ids, 152)
        assert rc == 0
        return u, c

    every = list(range(len(lens)))
    calls = [(dec, every, 1), (dec, small, 4), (dec, every, 4), (pre, every, None), (pre, small, None),
             (pre, every, None), (dec, every, 1)]
    reused = make()
    for fn, ids, T in calls:
        args = (ids,) if T is None else (ids, T)
        u1, c1 = fn(reused, *args)
        u2, c2 = fn(make(), *args)
        assert np.array_equal(u1, u2) and np.array_equal(c1, c2)


# ---------------------------------------------------------------- attention mass
def mass_case(G, hkv, W, chunks, prior, num_ctas, seed):
    """Host-only handle; sequence b holds prior[b] tokens, then its chunk of
    chunks[b] tokens is appended and planned."""
    hq, d, P = G * hkv, 128, 64
    hc = [GLOBAL if hd % 3 == 0 else LOCAL for hd in range(hkv)]
    n = len(chunks)
    h = host_handle(hq, hkv, d, hc, W, P, n, 16384, 8 * 16384)
    for b in range(n):
        if prior[b]:
            fill_one = np.array([0, prior[b]], np.int32)
            assert S.segkv_append(h.handle, 0, None, None, fill_one, np.array([b], np.int32)) == 0
    rng = np.random.default_rng(seed)
    ids = rng.permutation(n).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum([chunks[b] for b in ids])]).astype(np.int32)
    assert S.segkv_append(h.handle, 0, None, None, cu, ids) == 0
    qp = np.concatenate([np.arange(prior[b], prior[b] + chunks[b]) for b in ids]).astype(np.int32)
    rc, units, cta = S.segkv_plan_mass(h.handle, 0, cu, qp, ids, num_ctas)
    assert rc == 0, S.segkv_last_error(h.handle)
    return h, hc, ids, cu, units, cta


@pytest.mark.parametrize("G,hkv,W,num_ctas", [(4, 8, 300, 152), (8, 4, 1024, 16), (1, 2, 64, 5),
                                              (16, 2, 5000, 152)])
def test_mass_plan_covers_every_seeing_query_tile_once(G, hkv, W, num_ctas):
    chunks, prior = [700, 4096, 1, 129, 2500], [0, 1000, 37, 5000, 300]
    h, hc, ids, cu, units, cta = mass_case(G, hkv, W, chunks, prior, num_ctas, G + hkv)
    tpt = 128 // G
    assert cta[0] == 0 and cta[-1] == units.shape[0] and (np.diff(cta) >= 1).all()
    assert len(cta) - 1 == min(num_ctas, units.shape[0])
    # group the pieces by (chunk, head, key tile)
    tiles = {}
    for u in units:
        tok0, ntok, a, hd, local, kt, qt0, qt1, piece, npc, part0, tid = (int(v) for v in u)
        tiles.setdefault((tok0, hd, kt), []).append((piece, npc, qt0, qt1, part0, tid))
        assert local == (hc[hd] == LOCAL)
    slots, counters = [], []
    for i, b in enumerate(ids):
        a, T = prior[b], chunks[b]
        for hd in range(hkv):
            for kt in range(a // 128, (a + T - 1) // 128 + 1):
                ps = sorted(tiles.pop((int(cu[i]), hd, kt)))
                npc = len(ps)
                assert [p[0] for p in ps] == list(range(npc)) and all(p[1] == npc for p in ps)
                # pieces tile a contiguous run of query tiles
                assert all(ps[x][3] + 1 == ps[x + 1][2] for x in range(npc - 1))
                lens = [p[3] - p[2] + 1 for p in ps]
                assert min(lens) >= 1 and max(lens) - min(lens) <= 1
                # from the definition: query p (a <= p < a+T) sees key j iff
                # j <= p, and j >= p - W + 1 on a local head
                j = np.arange(max(a, 128 * kt), min(a + T, 128 * (kt + 1)))[:, None]
                p = np.arange(a, a + T)[None, :]
                vis = (j <= p) & ((hc[hd] == GLOBAL) | (j >= p - W + 1))
                seeing = np.nonzero(vis.any(axis=0))[0]  # chunk-relative query tokens
                assert ps[0][2] == seeing[0] // tpt and ps[-1][3] == seeing[-1] // tpt
                if npc > 1:
                    assert len({p[4] for p in ps}) == 1 and len({p[5] for p in ps}) == 1
                    slots.append((ps[0][4], npc))
                    counters.append(ps[0][5])
                else:
                    assert ps[0][4] == 0 and ps[0][5] == 0
    assert not tiles, "no unit outside the chunks' key tiles"
    # split key tiles own disjoint runs of partial slots and distinct counters
    slots.sort()
    assert all(slots[x][0] + slots[x][1] == slots[x + 1][0] for x in range(len(slots) - 1))
    assert (not slots or slots[0][0] == 0) and sorted(counters) == list(range(len(counters)))


@pytest.mark.parametrize("num_ctas", [152, 7])
def test_mass_plan_is_exactly_the_lpt_schedule(num_ctas):
    chunks, prior = [3000, 640, 9000], [100, 0, 2000]
    h, hc, ids, cu, units, cta = mass_case(4, 8, 700, chunks, prior, num_ctas, 3)
    # building order: chunk (call order), KV head, key tile, piece; then a
    # stable sort on query tiles, longest first; least loaded list, lowest
    # index on ties; a unit costs its query tiles + 1
    build = sorted(range(len(units)), key=lambda x: tuple(int(v) for v in units[x][[0, 3, 5, 8]]))
    order = sorted(build, key=lambda x: -int(units[x][7] - units[x][6]))
    grid = min(num_ctas, len(units))
    loads = np.zeros(grid, np.int64)
    lists = [[] for _ in range(grid)]
    for x in order:
        c = int(np.argmin(loads))
        lists[c].append(x)
        loads[c] += int(units[x][7] - units[x][6]) + 2
    assert len(cta) - 1 == grid
    for c in range(grid):
        assert (units[cta[c]:cta[c + 1]] == units[lists[c]]).all(), c


def test_mass_plan_errors():
    h = host_handle(8, 2, 64, [GLOBAL, LOCAL], 16, 16, 2, 512, 64)
    fill(h, [100, 5])
    # positions of a chunk must be consecutive and inside the sequence
    assert S.segkv_plan_mass(h.handle, 0, [0, 2], [10, 12], [0], 8)[0] == S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_plan_mass(h.handle, 0, [0, 2], [99, 100], [0], 8)[0] == S.SEGKV_ERR_INVALID_ARG
    assert S.segkv_plan_mass(h.handle, 0, [0, 1], [0], [3], 8)[0] == S.SEGKV_ERR_INVALID_ARG
    assert h.trim(0, [0]) == 0
    assert S.segkv_plan_mass(h.handle, 0, [0, 1], [50], [0], 8)[0] == S.SEGKV_ERR_EVICTED
    rc, units, cta = S.segkv_plan_mass(h.handle, 0, [0], [], [], 8)
    assert rc == 0 and units.shape == (0, 12)
