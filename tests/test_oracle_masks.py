"""Pins for the mask side of the oracle (no GPU).

Each test checks the oracle against something other than itself: masks built
by hand from their textual definition, closed-form counts, hand-worked tile
tables and localised bounds, and brute force on small inputs.
"""
import os

import numpy as np
import pytest

from fm_inputs import masks as gen
from fm_inputs.configs import TINY_DOCS, dual_chunk_map
from oracle import masks as om


def _read_golden(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- predicate

def _doc_id(S, lengths):
    out = np.empty(S, dtype=int)
    for n, (s, e) in enumerate(gen.doc_spans(lengths)):
        out[s:e] = n
    return out


def _visible_from_rule(S, rule):
    V = np.zeros((S, S), dtype=bool)
    for i in range(S):
        for j in range(S):
            V[i, j] = rule(i, j)
    return V


@pytest.mark.parametrize("S", [64, 200])
def test_causal_and_window_by_hand(S):
    V = _visible_from_rule(S, lambda i, j: j <= i)
    assert np.array_equal(~om.dense_mask(*gen.causal(S), S), V)
    w = 17
    V = _visible_from_rule(S, lambda i, j: 0 <= i - j < w)
    assert np.array_equal(~om.dense_mask(*gen.sliding_window(S, w), S), V)


def test_documents_by_hand():
    S = 150
    lengths = [40, 1, 59, 50]
    doc = _doc_id(S, lengths)
    V = _visible_from_rule(S, lambda i, j: doc[i] == doc[j] and j <= i)
    assert np.array_equal(~om.dense_mask(*gen.causal_document(S, lengths), S), V)
    V = _visible_from_rule(S, lambda i, j: doc[i] == doc[j])
    assert np.array_equal(~om.dense_mask(*gen.bidirectional_document(S, lengths), S), V)
    starts = {n: s for n, (s, e) in enumerate(gen.doc_spans(lengths))}
    plen = {n: (e - s) // 2 for n, (s, e) in enumerate(gen.doc_spans(lengths))}
    V = _visible_from_rule(S, lambda i, j: doc[i] == doc[j]
                           and (j < starts[doc[j]] + plen[doc[j]] or j <= i))
    assert np.array_equal(~om.dense_mask(*gen.prefix_document(S, lengths), S), V)


def test_prefix_lm_by_hand():
    S, P = 96, 30
    V = _visible_from_rule(S, lambda i, j: j < P or j <= i)
    assert np.array_equal(~om.dense_mask(*gen.prefix_lm(S, P), S), V)


def test_share_question_by_hand():
    S = 300
    rng = np.random.default_rng(3)
    groups = gen.share_question_spans(S, rng, question=20, answers=3, lo=10, hi=40)
    seg = np.empty(S, dtype=int)
    grp = np.empty(S, dtype=int)
    isq = np.zeros(S, dtype=bool)
    n = 0
    for g, (gs, ge, segs) in enumerate(groups):
        for s, e, q in segs:
            seg[s:e] = n
            grp[s:e] = g
            isq[s:e] = q
            n += 1
    V = _visible_from_rule(S, lambda i, j: j <= i and (seg[i] == seg[j] or (isq[j] and grp[i] == grp[j])))
    M = om.dense_mask(*gen.share_question(S, np.random.default_rng(3), question=20, answers=3,
                                          lo=10, hi=40), S)
    assert np.array_equal(~M, V)


def test_other_families_by_hand():
    S = 256
    # global + sliding
    G, w = 8, 40
    V = _visible_from_rule(S, lambda i, j: j < G or i < G or 0 <= i - j < w)
    assert np.array_equal(~om.dense_mask(*gen.global_sliding(S, G, w), S), V)
    # qk-sparse
    qs, qe, ks, ke = gen.qk_sparse_ranges(S)
    V = _visible_from_rule(S, lambda i, j: j <= i and not (qs <= i < qe) and not (ks <= j < ke))
    assert np.array_equal(~om.dense_mask(*gen.qk_sparse(S), S), V)
    # causal blockwise
    F = S - S // 8
    lengths = [50, 70, 40, F - 160]
    blk = _doc_id(F, lengths)
    V = _visible_from_rule(S, lambda i, j: j <= i and (i >= F or (j < F and blk[i] == blk[j])))
    assert np.array_equal(~om.dense_mask(*gen.causal_blockwise(S, lengths), S), V)
    # causal document intersected with a window
    lengths = [100, 30, 126]
    doc = _doc_id(S, lengths)
    V = _visible_from_rule(S, lambda i, j: doc[i] == doc[j] and 0 <= i - j < 25)
    assert np.array_equal(~om.dense_mask(*gen.causal_document_window(S, lengths, 25), S), V)


def test_block_sparse_by_hand():
    S, blk = 1024, 128
    nQ = S // blk
    n = int(round(0.3 * nQ))
    rng = np.random.default_rng(5)
    starts = [int(rng.integers(0, nQ - n + 1)) for _ in range(nQ)]
    V = _visible_from_rule(S, lambda i, j: starts[j // blk] <= i // blk < starts[j // blk] + n)
    M = om.dense_mask(*gen.block_sparse(S, np.random.default_rng(5)), S)
    assert np.array_equal(~M, V)


# ---------------------------------------------------------------- counts

def test_visible_counts_closed_forms(golden_dir):
    for name, S, want in _read_golden(os.path.join(golden_dir, "visible_counts.txt")):
        S, want = int(S), int(want)
        if name == "tiny_causal_document":
            b = gen.causal_document(S, TINY_DOCS)
        else:
            b = gen.make_mask(name, S)
        assert om.visible_count(*b, S) == want, name
        if S <= 4096:
            assert int((~om.dense_mask(*b, S)).sum()) == want, name


@pytest.mark.parametrize("name", ["causal_document", "share_question", "random_eviction",
                                  "qk_sparse", "global_sliding", "prefix_document"])
def test_visible_count_matches_dense(name):
    S = 1000
    b = gen.make_mask(name, S, seed=1)
    assert om.visible_count(*b, S) == int((~om.dense_mask(*b, S)).sum())


# ---------------------------------------------------------------- tiles

def test_tiny_tile_table_golden(golden_dir):
    want = np.array([[int(x) for x in r] for r in _read_golden(os.path.join(golden_dir, "tiny_tile_table.txt"))])
    got = om.tile_table_one(*gen.causal_document(256, TINY_DOCS), 256)
    assert np.array_equal(got, want)


def test_tile_table_causal_closed_form():
    S = 1024
    t = om.tile_table_one(*gen.causal(S), S)
    n = S // 128
    want = np.full((n, n), om.EMPTY)
    want[np.tril_indices(n, -1)] = om.FULL
    want[np.diag_indices(n)] = om.PARTIAL
    assert np.array_equal(t, want)
    assert np.all(om.tile_table_one(*gen.full(S), S) == om.FULL)


def test_block_sparse_has_no_partial_tiles():
    S = 4096
    t = om.tile_table_one(*gen.block_sparse(S, np.random.default_rng(0)), S)
    assert not np.any(t == om.PARTIAL)
    assert abs(np.mean(t == om.FULL) - 0.3) < 0.02


@pytest.mark.parametrize("S,Bq,Bk", [(512, 128, 128), (300, 128, 128), (333, 64, 32), (1000, 128, 64)])
@pytest.mark.parametrize("name", ["causal", "causal_document", "share_question", "random_eviction",
                                  "qk_sparse", "global_sliding", "prefix_lm", "bidirectional_document",
                                  "causal_blockwise", "prefix_document", "sliding_window"])
def test_tile_table_is_sound(name, S, Bq, Bk):
    """EMPTY tiles hide every entry, FULL tiles hide none (ragged tails included)."""
    b = gen.make_mask(name, S, seed=2, window=37, n_global=5) if name in ("sliding_window", "global_sliding") \
        else gen.make_mask(name, S, seed=2)
    M = om.dense_mask(*b, S)
    t = om.tile_table_one(*b, S, Bq, Bk)
    for qi in range(t.shape[0]):
        for kj in range(t.shape[1]):
            blk = M[qi * Bq:(qi + 1) * Bq, kj * Bk:(kj + 1) * Bk]
            if t[qi, kj] == om.EMPTY:
                assert blk.all()
            elif t[qi, kj] == om.FULL:
                assert not blk.any()


def test_tile_rule_planted_mistake_is_caught():
    """A rule that uses r0 + Bq instead of the clipped r1 on the ragged last
    q-tile still is sound, but one that swaps the cover test's r0 and r1 is not:
    the soundness check must reject it."""
    S = 300
    b = gen.causal_document(S, [70, 130, 100])
    M = om.dense_mask(*b, S)
    lts, lte, uts, ute = (np.asarray(x) for x in b)

    def wrong_table():
        nQ = nK = -(-S // 128)
        t = np.empty((nQ, nK), dtype=np.uint8)
        for qi in range(nQ):
            r0, r1 = qi * 128, min(S, qi * 128 + 128)
            for kj in range(nK):
                c = slice(kj * 128, min(S, kj * 128 + 128))
                cov = any(np.all((s[c] <= r1) & (e[c] >= r0)) for s, e in ((lts, lte), (uts, ute)))
                mis = all(np.all(s[c] >= r1) or np.all(e[c] <= r0) for s, e in ((lts, lte), (uts, ute)))
                t[qi, kj] = om.EMPTY if cov else (om.FULL if mis else om.PARTIAL)
        return t

    t = wrong_table()
    bad = False
    for qi in range(t.shape[0]):
        for kj in range(t.shape[1]):
            blk = M[qi * 128:(qi + 1) * 128, kj * 128:(kj + 1) * 128]
            if t[qi, kj] == om.EMPTY and not blk.all():
                bad = True
    assert bad


def test_lists_and_unit_order():
    S, H = 2048, 3
    b = gen.make_mask("causal_document", S, seed=4)
    bounds = np.stack([np.stack([np.asarray(x)[None]]) for x in b])  # [4][1][1][S]
    t = om.tile_table(bounds, S)
    rc, rl = om.row_lists(t)
    cc, cl = om.col_lists(t)
    assert rc.sum() == cc.sum() == np.count_nonzero(t)
    for (bb, hm, qi), lst in rl.items():
        ks = [k for k, _ in lst]
        assert ks == sorted(ks)
        assert all(t[bb, hm, qi, k] == c for k, c in lst)
    order = om.unit_order(rc, H)
    nT = rc.shape[2]
    assert sorted(order.tolist()) == list(range(H * nT))
    cost = [rc[0, 0, u % nT] for u in order]
    head = [u // nT for u in order]
    for a in range(len(order) - 1):
        assert head[a] < head[a + 1] or (head[a] == head[a + 1] and (
            cost[a] > cost[a + 1] or (cost[a] == cost[a + 1] and order[a] < order[a + 1])))


def test_unit_order_for_shared_kv_heads_by_hand():
    """Units of K/V heads shared by G = 2 query heads: a unit's cost sums its
    two query heads' counts.  counts [1][4][3] (per-head masks):
        query head 0: 1 3 0    query head 1: 2 0 0    -> unit head 0 costs 3 3 0
        query head 2: 0 1 1    query head 3: 0 0 2    -> unit head 1 costs 0 1 3
    so the order is 0, 1, 2 (ties by index) then 3+2, 3+1, 3+0."""
    counts = np.array([[[1, 3, 0], [2, 0, 0], [0, 1, 1], [0, 0, 2]]], dtype=np.int32)
    assert om.unit_order(counts, 4, 2).tolist() == [0, 1, 2, 5, 4, 3]
    # one mask for all heads: each unit costs G times its column
    one = np.array([[[1, 3, 2]]], dtype=np.int32)
    assert om.unit_order(one, 4, 2).tolist() == [1, 2, 0, 4, 5, 3]
    assert om.unit_order(one, 4, 1).tolist() == [1, 2, 0, 4, 5, 3, 7, 8, 6, 10, 11, 9]


def _table_of(b, S):
    bounds = np.stack([np.stack([np.asarray(x)[None]]) for x in b])  # [4][1][1][S]
    return om.tile_table(bounds, S)


def test_col_lists_by_hand():
    """Column lists in order and with their classes, worked out by hand.

    From a hand-written table (rows = q-tiles, columns = k-tiles):
        q0: FULL    PARTIAL EMPTY
        q1: EMPTY   PARTIAL FULL
        q2: PARTIAL EMPTY   PARTIAL
    column 0 holds q-tiles 0 (FULL), 2 (PARTIAL); column 1 q-tiles 0, 1
    (both PARTIAL); column 2 q-tiles 1 (FULL), 2 (PARTIAL).  The table is not
    symmetric, so returning row lists for column lists fails.

    Then from a mask: causal documents [0, 200) and [200, 384), S = 384, by
    hand.  (q0, k0), (q1, k1), (q2, k2) hold the diagonal (PARTIAL); (q1, k0)
    has rows 128..199 that see every key of k0 and rows 200..255 in the next
    document (PARTIAL); (q2, k0): every key of k0 is in document 0, whose lower
    interval [200, 384) covers rows 256..383 (EMPTY); (q2, k1): keys 128..199
    are hidden from rows 256..383, keys 200..255 are seen by all of them
    (PARTIAL); the tiles above the diagonal are covered by the upper
    interval [0, j) (EMPTY).  Column lists: k0 -> q0, q1; k1 -> q1, q2;
    k2 -> q2."""
    P, F, E = om.PARTIAL, om.FULL, om.EMPTY
    table = np.array([[[[F, P, E], [E, P, F], [P, E, P]]]], dtype=np.uint8)
    cc, cl = om.col_lists(table)
    assert cc.tolist() == [[[2, 2, 2]]]
    assert cl == {(0, 0, 0): [(0, F), (2, P)],
                  (0, 0, 1): [(0, P), (1, P)],
                  (0, 0, 2): [(1, F), (2, P)]}
    derived = _table_of(gen.causal_document(384, [200, 184]), 384)
    assert derived.tolist() == [[[[P, E, E], [P, P, E], [E, P, P]]]]
    cc, cl = om.col_lists(derived)
    assert cc.tolist() == [[[2, 2, 1]]]
    assert cl == {(0, 0, 0): [(0, P), (1, P)],
                  (0, 0, 1): [(1, P), (2, P)],
                  (0, 0, 2): [(2, P)]}


@pytest.mark.parametrize("name", ["causal_document", "qk_sparse", "random_eviction", "share_question"])
def test_pair_lists_are_unions_of_rows(name):
    S = 1100  # nQ = 9: the last pair has one row; the last k-tile is ragged
    t = _table_of(gen.make_mask(name, S, seed=2), S)
    nQ, nK = t.shape[2], t.shape[3]
    rc, rl = om.row_lists(t)
    n, c, pl = om.pair_lists(t, S)
    assert n.shape == (1, 1, (nQ + 1) // 2)
    for p in range((nQ + 1) // 2):
        rows = [q for q in (2 * p, 2 * p + 1) if q < nQ]
        want = sorted(set(k for q in rows for k, _ in rl[(0, 0, q)]))
        got = pl[(0, 0, p)]
        assert [k for k, _, _ in got] == want
        assert c[0, 0, p] == sum(rc[0, 0, q] for q in rows)
        for k, ca, cb in got:
            for q, cls in zip((2 * p, 2 * p + 1), (ca, cb)):
                tab = int(t[0, 0, q, k]) if q < nQ else om.EMPTY
                if tab != om.EMPTY and k == nK - 1:
                    tab = om.PARTIAL
                assert cls == tab


# ---------------------------------------------------------------- localisation

def test_localize_golden(golden_dir):
    rows = _read_golden(os.path.join(golden_dir, "localize_s16.txt"))
    S = 16
    cmap = dual_chunk_map(S, 2)
    b = np.stack([np.asarray(x)[None, None] for x in gen.causal(S)])  # [4][1][1][16]
    got = {r: om.localize_bounds(b, cmap[r]) for r in range(2)}
    r = None
    for row in rows:
        if row[0] == "rank":
            r = int(row[1])
            continue
        t = ["lts", "lte", "uts", "ute"].index(row[0])
        assert got[r][t, 0, 0].tolist() == [int(x) for x in row[1:]], (r, row[0])


def _check_localized_rows(b, S, chunks):
    G = om.chunk_rows(chunks)
    loc = om.localize_bounds(np.stack([np.asarray(x)[None, None] for x in b]), chunks)
    Ml = om.dense_mask(*(loc[t, 0, 0] for t in range(4)), len(G))
    Mg = om.dense_mask(*b, S)[G]
    assert np.array_equal(Ml, Mg)
    assert loc.min() >= 0 and loc.max() <= len(G)


@pytest.mark.parametrize("name", ["causal", "causal_document", "share_question", "sliding_window",
                                  "global_sliding", "qk_sparse", "random_eviction", "prefix_lm",
                                  "bidirectional_document", "block_sparse"])
def test_localize_dual_chunk_brute_force(name):
    S = 256
    b = gen.make_mask(name, S, seed=1) if name not in ("sliding_window", "global_sliding") \
        else gen.make_mask(name, S, seed=1, window=40, n_global=6)
    for R in (1, 2, 4):
        for chunks in dual_chunk_map(S, R):
            _check_localized_rows(b, S, chunks)


def test_localize_random_chunks_brute_force():
    rng = np.random.default_rng(9)
    S = 200
    for trial in range(40):
        b = gen.make_mask(["causal_document", "random_eviction", "qk_sparse"][trial % 3], S, seed=trial)
        cuts = np.sort(rng.choice(np.arange(1, S), size=2 * int(rng.integers(1, 5)), replace=False))
        pairs = cuts.reshape(-1, 2)
        chunks = [(int(a), int(e - a)) for a, e in pairs]
        _check_localized_rows(b, S, chunks)


def test_localize_rejects_unsorted_chunks():
    b = np.stack([np.asarray(x)[None, None] for x in gen.causal(64)])
    with pytest.raises(ValueError):
        om.localize_bounds(b, [(32, 16), (0, 16)])
    with pytest.raises(ValueError):
        om.localize_bounds(b, [(0, 20), (10, 16)])


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_bounds_are_the_block_diagonal_mask(causal):
    """A packed batch's bounds give exactly the block-diagonal mask built
    entry by entry from the sequence boundaries (zero-length sequences too)."""
    cu = [0, 5, 5, 17, 18, 40]
    total = cu[-1]
    seq = np.empty(total, dtype=int)
    for s_, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        seq[a:b] = s_
    want = np.zeros((total, total), dtype=bool)  # True = hidden
    for i in range(total):
        for j in range(total):
            want[i, j] = seq[i] != seq[j] or (causal and j > i)
    b = om.varlen_bounds(cu, causal)
    assert np.array_equal(om.dense_mask(*b, total), want)
    # the same as a document mask of those lengths (the input generators')
    lengths = [y - x for x, y in zip(cu[:-1], cu[1:]) if y > x]
    g = (gen.causal_document if causal else gen.bidirectional_document)(total, lengths)
    assert np.array_equal(om.dense_mask(*g, total), want)
