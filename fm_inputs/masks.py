"""Seeded generators of structured masks in the column-wise sparse form.

Every generator returns four int32 vectors ``(lts, lte, uts, ute)`` of length S
(one entry per key column j).  Key column j is hidden from query row i when
``lts[j] <= i < lte[j]`` or ``uts[j] <= i < ute[j]`` (the FlashMask-3 page,
"FlashMask ... four bound vectors along the query axis"; the exact predicate is
the one the attention library documents in ``include/fm.h``).

An interval that hides nothing is written in one canonical form: the lower
interval as ``[S, S)`` and the upper one as ``[0, 0)``.  Keeping empties
canonical keeps per-block min/max summaries tight.

These are input builders only: they draw document lengths, window sizes and
random choices and write bound values.  They evaluate no attention, mask
predicate, tile rule or localisation; both the CPU oracle and the CUDA library
consume what they return.

The mask families are those the FlashMask-3 page lists in its introduction
(document, prefix-LM, share-question, sliding window, block-sparse), widened to
the twelve-mask suite of the 32K workload.  The pages fix none of the
parameters; each choice made here is stated in the function's docstring.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "empty_bounds", "doc_lengths_uniform", "doc_lengths_loguniform", "doc_spans",
    "full", "causal", "sliding_window", "causal_document", "bidirectional_document",
    "prefix_lm", "prefix_document", "share_question", "causal_blockwise",
    "random_eviction", "global_sliding", "qk_sparse", "block_sparse",
    "causal_document_window", "MASKS_32K", "make_mask",
]


def empty_bounds(S: int):
    """All-visible bounds: lower interval [S,S), upper interval [0,0)."""
    lts = np.full(S, S, dtype=np.int64)
    lte = np.full(S, S, dtype=np.int64)
    uts = np.zeros(S, dtype=np.int64)
    ute = np.zeros(S, dtype=np.int64)
    return lts, lte, uts, ute


def _pack(lts, lte, uts, ute):
    return tuple(np.ascontiguousarray(x, dtype=np.int32) for x in (lts, lte, uts, ute))


def doc_lengths_uniform(S: int, lo: int, hi: int, rng) -> list[int]:
    """Integer lengths drawn from U[lo, hi] in order until they sum to >= S;
    the last one is cut so the lengths sum to exactly S."""
    out, tot = [], 0
    while tot < S:
        L = int(rng.integers(lo, hi + 1))
        L = min(L, S - tot)
        out.append(L)
        tot += L
    return out


def doc_lengths_loguniform(S: int, lo: int, hi: int, rng) -> list[int]:
    """Lengths round(exp(U[ln lo, ln hi])) drawn until they reach S; last one cut."""
    out, tot = [], 0
    while tot < S:
        L = int(round(float(np.exp(rng.uniform(np.log(lo), np.log(hi))))))
        L = max(1, min(L, S - tot))
        out.append(L)
        tot += L
    return out


def doc_spans(lengths) -> list[tuple[int, int]]:
    """Half-open [start, end) spans of consecutive documents."""
    spans, s = [], 0
    for L in lengths:
        spans.append((s, s + L))
        s += L
    return spans


# --------------------------------------------------------------------------
# the mask families
# --------------------------------------------------------------------------

def full(S: int, **_):
    """No key is hidden from any query."""
    return _pack(*empty_bounds(S))


def causal(S: int, **_):
    """Row i sees key j iff j <= i: the upper interval hides rows [0, j)."""
    lts, lte, uts, ute = empty_bounds(S)
    ute[:] = np.arange(S)
    return _pack(lts, lte, uts, ute)


def sliding_window(S: int, window: int, **_):
    """Causal band: row i sees key j iff 0 <= i - j < window.
    Upper interval [0, j); lower interval [min(j+window, S), S)."""
    j = np.arange(S)
    lts, lte, uts, ute = empty_bounds(S)
    ute[:] = j
    lts[:] = np.minimum(j + window, S)
    return _pack(lts, lte, uts, ute)


def causal_document(S: int, lengths, **_):
    """Causal attention inside each document [s, e): key j is seen by rows
    j..e-1.  Upper interval [0, j); lower interval [e, S)."""
    lts, lte, uts, ute = empty_bounds(S)
    for s, e in doc_spans(lengths):
        ute[s:e] = np.arange(s, e)
        lts[s:e] = e
    return _pack(lts, lte, uts, ute)


def bidirectional_document(S: int, lengths, **_):
    """Full attention inside each document [s, e): upper [0, s), lower [e, S)."""
    lts, lte, uts, ute = empty_bounds(S)
    for s, e in doc_spans(lengths):
        ute[s:e] = s
        lts[s:e] = e
    return _pack(lts, lte, uts, ute)


def prefix_lm(S: int, prefix: int, **_):
    """Keys j < prefix are seen by every row; later keys are causal."""
    lts, lte, uts, ute = empty_bounds(S)
    j = np.arange(S)
    ute[prefix:] = j[prefix:]
    return _pack(lts, lte, uts, ute)


def prefix_document(S: int, lengths, **_):
    """Per document [s, e) with prefix p = floor((e - s) / 2): prefix keys are
    seen by the whole document, the rest causally within it (the prefix length
    is a choice; the pages give none)."""
    lts, lte, uts, ute = empty_bounds(S)
    for s, e in doc_spans(lengths):
        p = (e - s) // 2
        lts[s:e] = e
        ute[s:s + p] = s
        ute[s + p:e] = np.arange(s + p, e)
    return _pack(lts, lte, uts, ute)


def share_question_spans(S: int, rng, question: int = 2048, answers: int = 8,
                         lo: int = 512, hi: int = 4096):
    """Groups of one question followed by ``answers`` answers with lengths
    U[lo, hi], repeated until S; the last segment is cut at S.
    Returns a list of (group_start, group_end, [(seg_start, seg_end, is_q)])."""
    groups, pos = [], 0
    while pos < S:
        gs = pos
        segs = []
        qe = min(pos + question, S)
        segs.append((pos, qe, True))
        pos = qe
        for _ in range(answers):
            if pos >= S:
                break
            L = int(rng.integers(lo, hi + 1))
            e = min(pos + L, S)
            segs.append((pos, e, False))
            pos = e
        groups.append((gs, pos, segs))
    return groups


def share_question(S: int, rng, question: int = 2048, answers: int = 8,
                   lo: int = 512, hi: int = 4096, **_):
    """Question tokens are causal among themselves and seen by every answer of
    their group; answer tokens are causal within their own answer only."""
    lts, lte, uts, ute = empty_bounds(S)
    for gs, ge, segs in share_question_spans(S, rng, question, answers, lo, hi):
        for s, e, is_q in segs:
            ute[s:e] = np.arange(s, e)
            lts[s:e] = ge if is_q else e
    return _pack(lts, lte, uts, ute)


def causal_blockwise(S: int, lengths, **_):
    """Blocks from ``lengths`` cover the first S - S//8 tokens; each is causal
    within itself.  The final block (the last S//8 tokens) attends causally to
    everything before it.  Non-final block [s, e): upper [0, j), lower
    [e, S - S//8).  Final block: upper [0, j)."""
    F = S - S // 8
    assert sum(lengths) == F
    lts, lte, uts, ute = empty_bounds(S)
    j = np.arange(S)
    ute[:] = j
    for s, e in doc_spans(lengths):
        if e < F:
            lts[s:e] = e
            lte[s:e] = F
    return _pack(lts, lte, uts, ute)


def random_eviction(S: int, rng, p: float = 0.5, **_):
    """Causal, and each key j < S-1 is evicted with probability p from row
    e_j ~ U[j+1, S-1] on: lower interval [e_j, S)."""
    lts, lte, uts, ute = empty_bounds(S)
    j = np.arange(S)
    ute[:] = j
    coin = rng.random(S) < p
    ev = rng.integers(np.minimum(j + 1, S - 1), S)  # in [j+1, S-1] (or S-1 at the end)
    sel = coin & (j + 1 <= S - 1)
    lts[sel] = ev[sel]
    return _pack(lts, lte, uts, ute)


def global_sliding(S: int, n_global: int = 64, window: int = 4096, **_):
    """The first n_global tokens attend to and are attended by everything;
    other keys j are seen by rows [j, j + window) and by the global rows.
    Keys j >= G: upper [G, j), lower [min(j + window, S), S)."""
    lts, lte, uts, ute = empty_bounds(S)
    j = np.arange(S)
    G = n_global
    uts[G:] = G
    ute[G:] = j[G:]
    lts[G:] = np.minimum(j[G:] + window, S)
    # a key with j == G has an upper interval [G, G): write it canonically
    e = ute <= uts
    uts[e] = 0
    ute[e] = 0
    return _pack(lts, lte, uts, ute)


def qk_sparse_ranges(S: int):
    """Dropped query rows [S/4, S/4 + S/16) and key columns [S/2, S/2 + S/16)."""
    qs, qe = S // 4, S // 4 + S // 16
    ks, ke = S // 2, S // 2 + S // 16
    return qs, qe, ks, ke


def qk_sparse(S: int, **_):
    """Causal, with the query rows and key columns of ``qk_sparse_ranges``
    dropped: a dropped column is hidden from all rows, a dropped row sees
    no key.  This produces fully masked rows and fully masked columns."""
    qs, qe, ks, ke = qk_sparse_ranges(S)
    lts, lte, uts, ute = empty_bounds(S)
    j = np.arange(S)
    ute[:] = j
    a = j < qs
    lts[a] = qs
    lte[a] = qe
    b = (j >= qs) & (j < qe)
    ute[b] = np.maximum(j[b], qe)
    ute[ks:ke] = S
    return _pack(lts, lte, uts, ute)


def block_sparse(S: int, rng, density: float = 0.3, block: int = 128, **_):
    """Per key block, the visible query blocks are one contiguous run of
    n = round(density * nQ) blocks starting at a seeded uniform block a:
    upper [0, block*a), lower [block*(a+n), S)."""
    nQ = -(-S // block)
    nK = nQ
    n = int(round(density * nQ))
    lts, lte, uts, ute = empty_bounds(S)
    for kb in range(nK):
        a = int(rng.integers(0, nQ - n + 1))
        j0, j1 = kb * block, min(S, (kb + 1) * block)
        ute[j0:j1] = min(block * a, S)
        lts[j0:j1] = min(block * (a + n), S)
    e = ute <= uts
    uts[e] = 0
    ute[e] = 0
    return _pack(lts, lte, uts, ute)


def causal_document_window(S: int, lengths, window: int, **_):
    """Causal document mask intersected with a causal sliding window:
    key j is seen by rows j .. min(e, j + window) - 1."""
    lts, lte, uts, ute = empty_bounds(S)
    for s, e in doc_spans(lengths):
        j = np.arange(s, e)
        ute[s:e] = j
        lts[s:e] = np.minimum(e, j + window)
    return _pack(lts, lte, uts, ute)


# --------------------------------------------------------------------------
# named masks with their seeded parameters
# --------------------------------------------------------------------------

MASKS_32K = [
    "causal", "sliding_window", "causal_document", "bidirectional_document",
    "prefix_lm", "prefix_document", "share_question", "causal_blockwise",
    "random_eviction", "global_sliding", "qk_sparse", "block_sparse",
]


def make_mask(name: str, S: int, seed: int = 0, **params):
    """Build a named mask of length S from a fresh ``default_rng(seed)``.

    Parameters not given take the defaults of the workloads: window S//8
    (512 at 4K, 4096 at 32K), prefix S//4 (1024 at 4K), documents U[256, 2048].
    """
    rng = np.random.default_rng(seed)
    if name == "full":
        return full(S)
    if name == "causal":
        return causal(S)
    if name == "sliding_window":
        return sliding_window(S, params.get("window", max(1, S // 8)))
    if name == "prefix_lm":
        return prefix_lm(S, params.get("prefix", S // 4))
    if name in ("causal_document", "bidirectional_document", "prefix_document"):
        lengths = params.get("lengths")
        if lengths is None:
            lengths = doc_lengths_uniform(S, params.get("lo", 256), params.get("hi", 2048), rng)
        fn = {"causal_document": causal_document,
              "bidirectional_document": bidirectional_document,
              "prefix_document": prefix_document}[name]
        return fn(S, lengths)
    if name == "share_question":
        return share_question(S, rng)
    if name == "causal_blockwise":
        F = S - S // 8
        return causal_blockwise(S, doc_lengths_uniform(F, 256, 2048, rng))
    if name == "random_eviction":
        return random_eviction(S, rng)
    if name == "global_sliding":
        return global_sliding(S, params.get("n_global", 64), params.get("window", 4096))
    if name == "qk_sparse":
        return qk_sparse(S)
    if name == "block_sparse":
        return block_sparse(S, rng, params.get("density", 0.3))
    if name == "causal_document_window":
        lengths = params.get("lengths")
        if lengths is None:
            lengths = doc_lengths_loguniform(S, 1024, 32768, rng)
        return causal_document_window(S, lengths, params.get("window", 8192))
    raise KeyError(name)
