"""CPU oracle for the block table of a batch given in flat token-slot form.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use it.
It shares no code with the C-ABI library.

Source: sglang PR 30105 digest, "Fix 2: draft_extend_v2 re-routed to
unified_attention". The draft-extend pass builds a 2D page table from the
batch's flat metadata and takes each sequence's KV length as the difference of
consecutive ``kv_indptr`` entries (``seqused_k = kv_indptr[1:] - kv_indptr[:-1]``),
then calls the same attention as target verify with
``max_seqlen_k = page_table width * page size``.

Reading, where the digest does not show the page-table builder: ``kv_indices``
holds the KV-cache token slot of every token (slot = page * 16 + position in
the page), sequence b's tokens at ``kv_indices[kv_indptr[b]:kv_indptr[b+1]]``.
Entry p of row b is the page of that sequence's tokens [16p, 16p + 16), i.e.
``kv_indices[kv_indptr[b] + 16 p] // 16``. It is only a faithful page if the
slots of those tokens are one page in order. Status bits report what does not
fit:
  1  a page's slots are not one aligned page in order;
  2  a sequence has more pages than the table is wide (the row keeps the first);
  4  ``kv_indptr`` is negative, decreases, or passes the end of ``kv_indices``
     (that row is all padding and its length 0).
"""

from __future__ import annotations

import numpy as np

PAGE = 16
BAD_PAGE, TRUNCATED, BAD_INDPTR = 1, 2, 4


def sequence_range(indptr, b):
    """Token range [start, end) of sequence b in kv_indices."""
    return indptr[b], indptr[b + 1]


def pages_needed(n):
    """Pages holding n tokens."""
    return -(-n // PAGE)


def page_of(first_slot):
    """Page of a token slot."""
    return first_slot // PAGE


def block_table_from_indptr(kv_indptr, kv_indices, width: int, pad_page: int = 0):
    """Returns (block_table [B, width] int32, seqused_k [B] int32, status int)."""
    indptr = [int(x) for x in np.asarray(kv_indptr).reshape(-1)]
    slots = np.asarray(kv_indices, dtype=np.int64).reshape(-1)
    nnz = len(slots)
    B = len(indptr) - 1
    table = np.full((B, width), pad_page, dtype=np.int32)
    seqused = np.zeros(B, dtype=np.int32)
    status = 0
    for b in range(B):
        start, end = sequence_range(indptr, b)
        if start < 0 or end < start or end > nnz:
            status |= BAD_INDPTR
            continue
        n = end - start
        seqused[b] = n
        pages = pages_needed(n)
        if pages > width:
            status |= TRUNCATED
        for p in range(min(pages, width)):
            page_slots = slots[start + PAGE * p: start + min(PAGE * p + PAGE, n)]
            first = int(page_slots[0])
            expected = first + np.arange(len(page_slots))
            if first < 0 or first % PAGE != 0 or not np.array_equal(page_slots, expected):
                status |= BAD_PAGE
            table[b, p] = page_of(first) if first >= 0 else pad_page
    return table, seqused, status
