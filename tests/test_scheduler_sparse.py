"""Host schedule of the block-sparse variant (no GPU).

The variant only adds iteration over selected key blocks (TLX porta
l'attenzione jagged su Blackwell oltre FA4 con un terzo del codice, section
"The turning point"); the library's reading: 128-key blocks per sequence, a
selection per (sequence, head), mask uint8 [NB, H].  Checked here against a
plain restatement: the forward's per-pair lists of selected blocks, the
forward items (unchanged) and their costs, and the backward's split of key
tiles into work items (selected) and zeroed tiles (unselected).
"""
import pytest
import torch

import jfa_inputs


@pytest.fixture(scope="module")
def jfa():
    import bwd_jagged_flashattention_gb300 as jfa
    jfa.build()
    return jfa


def _restate(offsets, mask, H):
    """Per (b, h): selected block indices and how many hold 128 keys."""
    lens = (offsets[1:] - offsets[:-1]).tolist()
    sel, g = {}, 0
    for b, L in enumerate(lens):
        n = (L + 127) // 128
        for h in range(H):
            blocks = [i for i in range(n) if mask[g + i, h]]
            sel[(b, h)] = (blocks, sum(1 for i in blocks if L - 128 * i >= 128))
        g += n
    return sel


CASES = [
    # lengths, Lq, H, broadcast_q, ratio
    ([300, 129, 0, 257, 50, 1000], 256, 4, True, 0.5),
    ([300, 129, 0, 257, 50, 1000], 384, 2, True, 0.0),
    ([300, 129, 0, 257, 50, 1000], 130, 2, True, 1.0),
    ([260, 140, 1, 513], 0, 2, False, 0.5),
]


@pytest.mark.parametrize("case", CASES)
def test_forward_selection_tables(jfa, case):
    lengths, Lq, H, bq, ratio = case
    off = jfa_inputs.offsets_from_lengths(torch.tensor(lengths))
    mask = jfa_inputs.kv_block_mask(off, H, ratio, seed=len(lengths))
    items, starts, sel, blocks, zero = jfa.host_schedule_sparse(off, mask, Lq, H, bq, False, 8)
    ref = _restate(off, mask, H)
    assert len(zero) == 0
    for (b, h), (blk, nfull) in ref.items():
        o, n, f, _ = sel[b * H + h].tolist()
        assert n == len(blk) and f == nfull
        assert blocks[o:o + n].tolist() == blk
    # the forward items are the dense ones: every (b, h, query-tile pair) once
    dense, _ = jfa.host_schedule(off, Lq, H, bq, False, False, 8, policy=jfa.SCHED_GREEDY)
    key = lambda t: sorted(map(tuple, t.tolist()))
    assert key(items) == key(dense)
    assert starts[-1] == len(items)


@pytest.mark.parametrize("case", CASES)
def test_backward_split_into_items_and_zero_tiles(jfa, case):
    lengths, Lq, H, bq, ratio = case
    off = jfa_inputs.offsets_from_lengths(torch.tensor(lengths))
    mask = jfa_inputs.kv_block_mask(off, H, ratio, seed=len(lengths) + 1)
    items, starts, sel, blocks, zero = jfa.host_schedule_sparse(off, mask, Lq, H, bq, True, 8)
    offl = off.tolist()
    want_items, want_zero, g = set(), set(), 0
    for b in range(len(lengths)):
        n = (lengths[b] + 127) // 128
        for h in range(H):
            for t in range(n):
                if mask[g + t, h]:
                    want_items.add((b, h, t))
                else:
                    row0 = offl[b] + 128 * t
                    want_zero.add((row0, min(128, offl[b + 1] - row0), h))
        g += n
    got_items = {(int(w[0]), int(w[3]) & 0xFF, (int(w[3]) >> 8) & 0x7FFFFF) for w in items}
    assert got_items == want_items and len(items) == len(want_items)
    assert {tuple(z[:3]) for z in zero.tolist()} == want_zero and len(zero) == len(want_zero)
    assert starts[-1] == len(items)


def test_forward_costs_follow_the_selection(jfa):
    """The greedy deal weighs items by their selected blocks: with only
    sequence 0 selected (8 blocks: cost 2 * 8 + 1) and 15 sequences with
    nothing selected (cost 1 each), each head's two CTAs split 1 / 15 items,
    where the dense costs (sequences of 4 blocks, cost 9) split them evenly."""
    lengths = [1024] + [512] * 15
    H, P = 4, 8                                    # head groups of P / H = 2 CTAs
    off = jfa_inputs.offsets_from_lengths(torch.tensor(lengths))
    mask = torch.zeros(jfa_inputs.num_kv_blocks(off), H, dtype=torch.uint8)
    mask[:8] = 1                                   # all blocks of sequence 0, every head
    items, starts, sel, blocks, zero = jfa.host_schedule_sparse(off, mask, 256, H, True, False, P)
    counts = sorted((starts[1:] - starts[:-1]).tolist())
    assert counts == [1] * H + [15] * H
    for p in range(P):
        if starts[p + 1] - starts[p] == 1:
            assert int(items[starts[p]][0]) == 0
    _, dense_starts = jfa.host_schedule(off, 256, H, True, False, False, P, policy=jfa.SCHED_GREEDY)
    assert max((dense_starts[1:] - dense_starts[:-1]).tolist()) <= 9
