"""The five synthetic workloads, with every free parameter written down.

All tensors are bf16 N(0,1) drawn with seed 0; scale = 1/sqrt(d); one mask
head (Hm = 1) shared by all heads.  Masks are built by ``fm_inputs.masks``.
The pages publish their benchmark suite only by name (twelve structured masks
at 4K..128K on one H100, on the FlashMask-3 page's results paragraph); these
seeded shapes stand in for it.
"""
from __future__ import annotations

from dataclasses import dataclass, field

TINY_DOCS = [80, 100, 76]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    d: int
    masks: tuple
    mask_params: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return self.d ** -0.5


TINY = Workload("tiny", 1, 2, 256, 64, ("causal_document",), {"lengths": TINY_DOCS})

SWEEP_4K = Workload("sweep_4k", 4, 16, 4096, 128,
                    ("full", "causal", "sliding_window", "causal_document", "prefix_lm"))

SUITE_32K = Workload("suite_32k", 1, 32, 32768, 128, (
    "causal", "sliding_window", "causal_document", "bidirectional_document",
    "prefix_lm", "prefix_document", "share_question", "causal_blockwise",
    "random_eviction", "global_sliding", "qk_sparse", "block_sparse"))

LONG_128K = Workload("long_128k", 1, 8, 131072, 128, ("causal_document_window",),
                     {"window": 8192})

# 8 chunks of 8192 tokens; simulated rank r holds chunks r and 7 - r (dual chunk)
LOCALIZE_64K = Workload("localize_64k", 1, 16, 65536, 128, ("causal_document",))
LOCALIZE_RANKS = 4
LOCALIZE_CHUNK = 8192


def dual_chunk_map(S: int, ranks: int):
    """Split S into 2*ranks equal chunks; rank r gets chunks r and 2*ranks-1-r,
    in ascending global order.  Returns per rank a list of (global_start, length)."""
    n = 2 * ranks
    C = S // n
    assert C * n == S
    out = []
    for r in range(ranks):
        ids = sorted((r, n - 1 - r))
        out.append([(i * C, C) for i in ids])
    return out


WORKLOADS = {w.name: w for w in (TINY, SWEEP_4K, SUITE_32K, LONG_128K, LOCALIZE_64K)}
