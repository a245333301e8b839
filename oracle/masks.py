"""Mask-side oracle: predicate, visible counts, tile rule, work lists, unit
order and localisation.  Plain numpy / Python, no blocking beyond what each
definition states.  Test infrastructure only (see ``oracle/__init__.py``).

Bounds arrive as an int array ``[4][B][Hm][Skv]`` (LTS, LTE, UTS, UTE) or, for
one (batch, mask head), as four vectors of length Skv.
"""
from __future__ import annotations

import numpy as np

EMPTY, PARTIAL, FULL = 0, 1, 2


# --------------------------------------------------------------------------
# the predicate
# --------------------------------------------------------------------------

def dense_mask(lts, lte, uts, ute, Sq: int, rows=None) -> np.ndarray:
    """Boolean matrix M[i][j], True where key column j is hidden from query row i:
    ``LTS[j] <= i < LTE[j]`` or ``UTS[j] <= i < UTE[j]``.

    The column-wise sparse form keeps, per key column, bounds along the query
    axis (FlashMask-3 page, introduction and «Ключевые факты»: four bound
    vectors, O(n) memory); the two half-open intervals are the reading of those
    four vectors used throughout this library.  ``rows`` selects a subset of
    query rows (default all Sq)."""
    i = np.arange(Sq) if rows is None else np.asarray(rows)
    i = i[:, None]
    lts, lte, uts, ute = (np.asarray(x)[None, :] for x in (lts, lte, uts, ute))
    return ((lts <= i) & (i < lte)) | ((uts <= i) & (i < ute))


def _interval_len(a, b, Sq):
    a = np.clip(a, 0, Sq)
    b = np.clip(b, 0, Sq)
    return np.maximum(b - a, 0)


def visible_count(lts, lte, uts, ute, Sq: int) -> int:
    """N_u = sum over columns of (Sq - |[LTS,LTE) U [UTS,UTE)|), by exact
    integer interval arithmetic (|A u B| = |A| + |B| - |A n B|).  This is the
    number of score entries the masked attention actually evaluates, the
    quantity the effective-throughput figure counts."""
    lts, lte, uts, ute = (np.asarray(x, dtype=np.int64) for x in (lts, lte, uts, ute))
    a = _interval_len(lts, lte, Sq)
    b = _interval_len(uts, ute, Sq)
    c = _interval_len(np.maximum(lts, uts), np.minimum(lte, ute), Sq)
    return int(np.sum(Sq - (a + b - c)))


def visible_count_all(bounds, Sq: int, H: int) -> int:
    """Total visible entries over all batches and query heads (bounds [4][B][Hm][Skv])."""
    bounds = np.asarray(bounds)
    _, B, Hm, _ = bounds.shape
    tot = 0
    for b in range(B):
        for hm in range(Hm):
            n = visible_count(*(bounds[t, b, hm] for t in range(4)), Sq)
            tot += n * (H if Hm == 1 else 1)
    return tot


# --------------------------------------------------------------------------
# tile classification, column by column
# --------------------------------------------------------------------------

def tile_table_one(lts, lte, uts, ute, Sq: int, Bq: int = 128, Bk: int = 128) -> np.ndarray:
    """Empty / full / partial class of every (q-tile, k-tile) for one mask head.

    Rule (tiles are rows [r0, r1) with r1 = min(r0 + Bq, Sq), and the valid
    key columns of one k-block).  For interval X in {lower, upper}:
      X covers the tile  iff every column has start <= r0 and end >= r1;
      X misses the tile  iff every column has start >= r1, or every column has
                          end <= r0.
    EMPTY iff either interval covers; FULL iff both miss; else PARTIAL.
    Skipping empty tiles and dropping mask work on full ones is the
    "fewer non-matmul operations" step of the FlashAttention-2 page
    («Три способа повысить загрузку GPU»).  Here each test is an ``all`` over
    the columns of the block, not a min/max summary."""
    Skv = len(lts)
    nQ, nK = -(-Sq // Bq), -(-Skv // Bk)
    lts, lte, uts, ute = (np.asarray(x, dtype=np.int64) for x in (lts, lte, uts, ute))
    r0 = np.arange(nQ, dtype=np.int64) * Bq
    r1 = np.minimum(r0 + Bq, Sq)
    r0c, r1c = r0[:, None], r1[:, None]
    out = np.empty((nQ, nK), dtype=np.uint8)
    for kj in range(nK):
        c = slice(kj * Bk, min(Skv, (kj + 1) * Bk))
        covers = np.zeros(nQ, dtype=bool)
        misses = np.ones(nQ, dtype=bool)
        for s, e in ((lts[c], lte[c]), (uts[c], ute[c])):
            s, e = s[None, :], e[None, :]
            covers |= np.all((s <= r0c) & (e >= r1c), axis=1)
            misses &= np.all(s >= r1c, axis=1) | np.all(e <= r0c, axis=1)
        out[:, kj] = np.where(covers, EMPTY, np.where(misses, FULL, PARTIAL))
    return out


def tile_table(bounds, Sq: int, Bq: int = 128, Bk: int = 128) -> np.ndarray:
    """uint8 table [B][Hm][nQ][nK] for bounds [4][B][Hm][Skv]."""
    bounds = np.asarray(bounds)
    _, B, Hm, _ = bounds.shape
    tabs = [[tile_table_one(*(bounds[t, b, hm] for t in range(4)), Sq, Bq, Bk)
             for hm in range(Hm)] for b in range(B)]
    return np.array(tabs, dtype=np.uint8)


def row_lists(table: np.ndarray):
    """Per (b, hm, qi): ascending k-tile indices of the non-empty tiles, and
    their classes.  Returns (counts [B][Hm][nQ], list of lists)."""
    B, Hm, nQ, nK = table.shape
    counts = np.zeros((B, Hm, nQ), dtype=np.int32)
    lists = {}
    for b in range(B):
        for hm in range(Hm):
            for qi in range(nQ):
                ks = [kj for kj in range(nK) if table[b, hm, qi, kj] != EMPTY]
                counts[b, hm, qi] = len(ks)
                lists[(b, hm, qi)] = [(kj, int(table[b, hm, qi, kj])) for kj in ks]
    return counts, lists


def col_lists(table: np.ndarray):
    """Per (b, hm, kj): ascending q-tile indices of the non-empty tiles."""
    B, Hm, nQ, nK = table.shape
    counts = np.zeros((B, Hm, nK), dtype=np.int32)
    lists = {}
    for b in range(B):
        for hm in range(Hm):
            for kj in range(nK):
                qs = [qi for qi in range(nQ) if table[b, hm, qi, kj] != EMPTY]
                counts[b, hm, kj] = len(qs)
                lists[(b, hm, kj)] = [(qi, int(table[b, hm, qi, kj])) for qi in qs]
    return counts, lists


def pair_lists(table: np.ndarray, Skv: int, Bk: int = 128):
    """Forward work units of two q-tiles: rows 2p and 2p+1 of one (b, hm) (the
    second absent when nQ is odd) walk their k-tiles together, so that each
    K/V tile is loaded once for both; the forward pass gives each warp group
    its own queries and shares K and V (FlashAttention-2 page, «Три способа
    повысить загрузку GPU», third point).  A pair's list is the union of the
    two rows' non-empty k-tiles, ascending, each entry carrying the tile's
    class in row 2p and in row 2p+1 (EMPTY where that row skips it).  A
    non-empty last k-tile that is ragged (Skv not a multiple of Bk) is given
    the class PARTIAL: its columns past Skv are masked element by element.
    Returns (counts [B][Hm][nP] = entries, costs [B][Hm][nP] = non-empty tiles
    of both rows, dict (b, hm, p) -> [(kj, class_a, class_b), ...])."""
    B, Hm, nQ, nK = table.shape
    nP = -(-nQ // 2)
    ragged = Skv % Bk != 0
    counts = np.zeros((B, Hm, nP), dtype=np.int32)
    costs = np.zeros((B, Hm, nP), dtype=np.int32)
    lists = {}
    for b in range(B):
        for hm in range(Hm):
            for p in range(nP):
                ent = []
                for kj in range(nK):
                    cls = []
                    for qi in (2 * p, 2 * p + 1):
                        c = int(table[b, hm, qi, kj]) if qi < nQ else EMPTY
                        if c != EMPTY and ragged and kj == nK - 1:
                            c = PARTIAL
                        cls.append(c)
                    if cls[0] != EMPTY or cls[1] != EMPTY:
                        ent.append((kj, cls[0], cls[1]))
                counts[b, hm, p] = len(ent)
                costs[b, hm, p] = sum((ca != EMPTY) + (cb != EMPTY) for _, ca, cb in ent)
                lists[(b, hm, p)] = ent
    return counts, costs, lists


def unit_order(counts: np.ndarray, H: int, G: int = 1) -> np.ndarray:
    """Work units (b, h, tile), numbered u = (b*Hu + h)*nT + tile with Hu = H / G,
    ordered by (b, h) ascending and, within one (b, h), by cost (non-empty
    tiles of the unit's q-tile pair, k-tile column or q-tile row) descending,
    ties by tile ascending.  Within a head this is the
    longest-processing-time-first order that balances units by work rather
    than by position (the sparsity-aware balancing the FlashMask-3 page names
    in «Ключевые факты», applied to one GPU's work units); keeping heads in
    order makes the units that run at the same time share one head.
    ``counts`` is [B][Hm][nT]; query head h reads mask head 0 if Hm == 1 else h.
    G > 1: the units belong to K/V heads shared by G query heads (grouped-query
    attention; unit head h covers query heads h*G .. h*G+G-1) and a unit's cost
    is the sum of its query heads' counts."""
    B, Hm, nT = counts.shape
    Hu = H // G
    units = []
    for b in range(B):
        for h in range(Hu):
            for t in range(nT):
                cost = sum(int(counts[b, 0 if Hm == 1 else h * G + j, t]) for j in range(G))
                u = (b * Hu + h) * nT + t
                units.append(((b, h), -cost, u))
    units.sort()
    return np.array([u for _, _, u in units], dtype=np.int32)


# --------------------------------------------------------------------------
# packed variable-length batches
# --------------------------------------------------------------------------

def varlen_bounds(cu_seqlens, causal: bool) -> np.ndarray:
    """Bounds [4][total] of a packed batch: sequence s holds rows and keys
    [cu[s], cu[s+1]) of one axis of length total = cu[-1], and a row sees only
    keys of its own sequence (and, if causal, only keys at or before it).  So
    key j of sequence [a, b) is seen by rows [j, b) (causal) or [a, b): the
    lower hidden interval is [b, total), the upper one [0, j) or [0, a).
    Sequences of length 0 hold nothing.  This is the FlashAttention-2 page's
    fixed-token batch («Как понимать заявленное ускорение»: 16K tokens per
    batch) written in the column-bound form of the FlashMask-3 page."""
    cu = [int(x) for x in cu_seqlens]
    total = cu[-1]
    out = np.empty((4, total), dtype=np.int64)
    for a, b in zip(cu[:-1], cu[1:]):
        for j in range(a, b):
            out[:, j] = (b, total, 0, j if causal else a)
    return out


# --------------------------------------------------------------------------
# localisation to a rank's query chunks
# --------------------------------------------------------------------------

def chunk_rows(chunks) -> np.ndarray:
    """G: local query row -> global query row, for chunks (global_start, length)
    listed in local order."""
    return np.concatenate([np.arange(g, g + C) for g, C in chunks]) if chunks else np.zeros(0, int)


def localize_value(x: int, chunks) -> int:
    """Local image of one bound value x: clip x into each chunk, shift it by
    that chunk's local offset, and take the max over the chunks that start at
    or before x (0 if none) - the clip, shift, max of the FlashMask-3 page
    (introduction and «Ключевые факты»).  For chunks in ascending global order
    this is the number of local rows whose global row is < x."""
    best = 0
    off = 0
    for g, C in chunks:
        if g <= x:
            best = max(best, off + min(x - g, C))
        off += C
    return best


def chunks_ascending(chunks) -> bool:
    """True iff the chunks are non-empty, non-overlapping and listed in
    ascending global order (the condition under which an interval's preimage is
    an interval)."""
    end = -1
    for g, C in chunks:
        if C <= 0 or g < 0 or g < end:
            return False
        end = g + C
    return True


def localize_bounds(bounds, chunks) -> np.ndarray:
    """Apply ``localize_value`` to every entry of bounds [4][B][Hm][Skv]; the
    key axis is left unchanged (each rank keeps every key)."""
    if not chunks_ascending(chunks):
        raise ValueError("chunks must be non-empty and in ascending global order")
    bounds = np.asarray(bounds)
    flat = bounds.reshape(-1)
    cache = {}
    out = np.empty_like(flat)
    for n, x in enumerate(flat.tolist()):
        v = cache.get(x)
        if v is None:
            v = localize_value(x, chunks)
            cache[x] = v
        out[n] = v
    return out.reshape(bounds.shape).astype(np.int32)
