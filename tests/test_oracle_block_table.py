"""Pins of the block-table oracle (oracle/block_table.py) to facts outside it.

* Round trip: a random paged layout (page permutation, ragged lengths) is
  expanded to flat token slots by code written here (slot = page * 16 +
  position), and the oracle must give back exactly the original table,
  lengths and no status bit.
* A hand example with its table written out.
* Each status bit on a case built to trigger it.
* Planted mistakes in the oracle's steps (on the CPU) each break a pin.
"""
import numpy as np
import pytest

import oracle.block_table as obt

PAD = -7


def expand(rows, lengths):
    """Flat (kv_indptr, kv_indices) of sequences whose pages are rows[b]."""
    indptr, slots = [0], []
    for pages, n in zip(rows, lengths):
        for t in range(n):
            slots.append(pages[t // 16] * 16 + t % 16)
        indptr.append(indptr[-1] + n)
    return np.array(indptr, dtype=np.int64), np.array(slots, dtype=np.int64)


def random_layout(rng):
    B = int(rng.integers(0, 7))
    lengths = [int(rng.choice([0, 1, 15, 16, 17, 32, 33, int(rng.integers(1, 400))])) for _ in range(B)]
    npages = [-(-n // 16) for n in lengths]
    perm = rng.permutation(sum(npages) + 5)
    rows, k = [], 0
    for m in npages:
        rows.append([int(x) for x in perm[k:k + m]])
        k += m
    width = max(npages + [0]) + int(rng.integers(0, 4))
    return rows, lengths, width


def check_round_trip(seed):
    rng = np.random.default_rng(seed)
    rows, lengths, width = random_layout(rng)
    indptr, slots = expand(rows, lengths)
    table, seqused, status = obt.block_table_from_indptr(indptr, slots, width, PAD)
    assert status == 0
    assert seqused.tolist() == lengths
    for b, pages in enumerate(rows):
        assert table[b, :len(pages)].tolist() == pages
        assert (table[b, len(pages):] == PAD).all()


@pytest.mark.parametrize("seed", range(40))
def test_round_trip(seed):
    check_round_trip(seed)


def test_hand_example():
    # seq 0: 20 tokens on pages 7, 3; seq 1: empty; seq 2: 16 tokens on page 0
    slots = list(range(112, 128)) + list(range(48, 52)) + list(range(0, 16))
    table, seqused, status = obt.block_table_from_indptr([0, 20, 20, 36], slots, 3, PAD)
    assert table.tolist() == [[7, 3, PAD], [PAD, PAD, PAD], [0, PAD, PAD]]
    assert seqused.tolist() == [20, 0, 16]
    assert status == 0


def test_status_bits():
    good = list(range(112, 128)) + list(range(48, 52))
    # first slot of a page not a multiple of 16: the entry is still its page
    t, _, st = obt.block_table_from_indptr([0, 20], [113] + good[1:], 2, PAD)
    assert st == obt.BAD_PAGE and t[0].tolist() == [7, 3]
    # two slots of a page swapped
    bad = list(good)
    bad[4], bad[5] = bad[5], bad[4]
    assert obt.block_table_from_indptr([0, 20], bad, 2, PAD)[2] == obt.BAD_PAGE
    # a partial last page out of order
    bad = list(good)
    bad[18], bad[19] = bad[19], bad[18]
    assert obt.block_table_from_indptr([0, 20], bad, 2, PAD)[2] == obt.BAD_PAGE
    # more pages than the table is wide: the row keeps the first ones
    t, s, st = obt.block_table_from_indptr([0, 20], good, 1, PAD)
    assert st == obt.TRUNCATED and t.tolist() == [[7]] and s.tolist() == [20]
    # kv_indptr decreasing / negative / past the end: padding and length 0
    for indptr in ([0, 20, 10], [-1, 20, 20], [0, 20, 25]):
        t, s, st = obt.block_table_from_indptr(indptr, good, 2, PAD)
        assert st & obt.BAD_INDPTR
        bad_rows = [b for b in range(2) if not (0 <= indptr[b] <= indptr[b + 1] <= len(good))]
        for b in bad_rows:
            assert (t[b] == PAD).all() and s[b] == 0


def _range_off_by_one(indptr, b):
    return indptr[b] + 1, indptr[b + 1]


def _pages_floor(n):
    return n // 16


def _page_plus_one(first_slot):
    return first_slot // 16 + 1


@pytest.mark.parametrize("name,fake", [("sequence_range", _range_off_by_one),
                                       ("pages_needed", _pages_floor),
                                       ("page_of", _page_plus_one)])
def test_planted_mistakes_are_caught(monkeypatch, name, fake):
    monkeypatch.setattr(obt, name, fake)
    failures = 0
    for seed in range(40):
        try:
            check_round_trip(seed)
        except AssertionError:
            failures += 1
    try:
        test_hand_example()
    except AssertionError:
        failures += 1
    assert failures > 0
