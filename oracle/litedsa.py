"""CPU oracle for LiteDSA candidate packing (test infrastructure only).

Only tests (and the smoke check) may import this module; it shares no code
with the CUDA path.

LiteTopK arXiv abstract: LiteDSA packs the overlapping candidates of
neighbouring query tokens into a shared key/value list for joint attention and
uses per-query masks to keep each token's own top-k membership.  Reading taken
(the abstract gives no more detail): consecutive queries form groups of G; the
shared list of a group is the ascending set union of the valid (>= 0) key
indices its queries selected, and query t's mask has bit j set iff entry j of
its group's list is among t's own selected keys.
"""
from __future__ import annotations

import numpy as np


def pack(topk_idx: np.ndarray, group: int):
    """Returns (union [n_groups, G*k] int32 padded with -1, lengths [n_groups],
    masks [T, ceil(G*k/32)] uint32, bit j of word j//32 = list entry j)."""
    topk_idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = topk_idx.shape
    n_groups = (T + group - 1) // group
    max_u = group * k
    words = (max_u + 31) // 32
    union = np.full((n_groups, max_u), -1, dtype=np.int32)
    lens = np.zeros(n_groups, dtype=np.int32)
    masks = np.zeros((T, words), dtype=np.uint32)
    for g in range(n_groups):
        rows = topk_idx[g * group: min(T, (g + 1) * group)]
        u = np.unique(rows[rows >= 0])                       # sorted set union
        union[g, : u.size] = u
        lens[g] = u.size
        for r, row in enumerate(rows):
            sel = row[row >= 0]
            j = np.searchsorted(u, sel)                      # position in the list
            np.bitwise_or.at(masks[g * group + r], j // 32, (np.uint32(1) << (j % 32).astype(np.uint32)))
    return union, lens, masks


def unpack_row(union_row: np.ndarray, length: int, mask_row: np.ndarray) -> np.ndarray:
    """Key indices a query's mask selects from its group's list (ascending)."""
    j = np.arange(length)
    bits = (mask_row[j // 32] >> (j % 32).astype(np.uint32)) & 1
    return union_row[:length][bits.astype(bool)]
