"""Split-KV in the host schedule of the broadcast-Q forward (no GPU).

A query tile of one (sequence, head) whose key loop alone costs more than
1.5x an average CTA's share is cut into key chunks of about half that share; the
chunks are single-tile items b = -(slot + 1) whose kv_start / kv_len cover
their keys, and one group record per split tile lists its slots.  Checked
here: the pages' workloads never split (their longest items are below the
average share); a skewed batch does, every split tile's keys are covered
exactly once in order, slots are used once each, the group records match the
chunks, and the deal becomes balanced.
"""
import pytest
import torch

import jfa_inputs


@pytest.fixture(scope="module")
def jfa():
    import bwd_jagged_flashattention_gb300 as jfa
    jfa.build()
    return jfa


def _loads(items, starts, P):
    """Per-CTA cost in blocks (+1 per item), the scheduler's own cost model."""
    loads = []
    for p in range(P):
        tot = 0
        for w in items[starts[p]:starts[p + 1]].tolist():
            b, k0, L, packed = w
            packed &= 0xFFFFFFFF
            tiles = 1 + (packed >> 31)
            tot += tiles * ((L + 127) // 128) + 1
        loads.append(tot)
    return loads


@pytest.mark.parametrize("name", ["ads_bwd", "extreme"])
def test_pages_workloads_do_not_split(jfa, name):
    x = jfa_inputs.make(name)
    items, starts, groups, slots = jfa.host_schedule_split(x["offsets"], x["Lq"], x["H"], 152)
    assert len(groups) == 0 and slots == 0
    assert (items[:, 0] >= 0).all()


@pytest.mark.parametrize("Lq", [128, 256, 300])
def test_skewed_batch_splits_and_covers_every_key_once(jfa, Lq):
    lengths = [20000, 5, 300, 0, 129, 1000]
    H, P = 2, 152
    off = jfa_inputs.offsets_from_lengths(torch.tensor(lengths))
    items, starts, groups, slots = jfa.host_schedule_split(off, Lq, H, P)
    assert 0 < slots <= jfa.SPLIT_MAX_SLOTS and len(groups) > 0
    chunk = {}                                        # slot -> (kv_start, kv_len, h, tile)
    for b, k0, L, packed in items.tolist():
        packed &= 0xFFFFFFFF
        if b < 0:
            assert packed >> 31 == 0                  # one query tile per chunk
            chunk[-b - 1] = (k0, L, packed & 0xFF, (packed >> 8) & 0x7FFFFF)
    assert sorted(chunk) == list(range(slots))        # every slot exactly once
    offl = off.tolist()
    seen = set()
    for b, slot0, n, packed in groups.tolist():
        h, tile = packed & 0xFF, packed >> 8
        assert (b, h, tile) not in seen
        seen.add((b, h, tile))
        pos = offl[b]
        for s in range(slot0, slot0 + n):             # chunks tile the sequence's keys in order
            k0, L, hh, tt = chunk[s]
            assert (hh, tt) == (h, tile) and k0 == pos and L > 0
            pos += L
        assert pos == offl[b + 1]
    # the split tiles are those of items costing more than 1.5x the average share with at
    # least two chunks (restated: cost = tiles * blocks + 1; chunk = max(4, avg // 2))
    nt = (Lq + 127) // 128
    costs = []
    for b, L in enumerate(lengths):
        for h in range(H):
            for m in range(0, nt, 2):
                tiles = 2 if m + 1 < nt else 1
                costs.append((b, h, m, tiles, tiles * ((L + 127) // 128) + 1))
    avg = sum(c[-1] for c in costs) // P
    chunk = max(4, avg // 2)
    want = {(b, h, m + t) for b, h, m, tiles, c in costs
            if 2 * c > 3 * avg and -(-((lengths[b] + 127) // 128) // chunk) >= 2 for t in range(tiles)}
    assert seen == want and {(0, h, 0) for h in range(H)} <= seen
    # whole items keep their tiles; no (b, h, tile) appears both whole and split
    for b, k0, L, packed in items.tolist():
        packed &= 0xFFFFFFFF
        if b >= 0:
            tile, two = (packed >> 8) & 0x7FFFFF, packed >> 31
            for t in range(tile, tile + 1 + two):
                assert (b, packed & 0xFF, t) not in seen


def test_split_balances_the_deal(jfa):
    lengths = [65536] + [512] * 31
    H, Lq, P = 4, 128, 152
    off = jfa_inputs.offsets_from_lengths(torch.tensor(lengths))
    items, starts, groups, slots = jfa.host_schedule_split(off, Lq, H, P)
    loads = _loads(items, starts, P)
    avg = sum(loads) / P
    assert max(loads) <= 2.5 * avg + 2
    whole, whole_starts = jfa.host_schedule(off, Lq, H, True, False, False, P, policy=jfa.SCHED_GREEDY)
    assert max(_loads(whole, whole_starts, P)) >= 512  # without split one CTA holds a 512-block item


def test_profiling_case_does_not_split(jfa):
    """Items at most 1.5x the average share stay whole (the first 256 ads sequences)."""
    x = jfa_inputs.make("ads_bwd")
    off = x["offsets"][:257].clone()
    _, _, groups, slots = jfa.host_schedule_split(off, 256, 4, 152)
    assert len(groups) == 0


def test_slot_first_blocks(jfa):
    """Each split slot's first key block, numbered over all sequences' 128-key
    blocks in order (what the MXFP8 forward looks its V scales up by): the
    chunk's start row minus its sequence's start, in blocks, plus the blocks
    of all earlier sequences."""
    lengths = [20000, 5, 300, 0, 129, 1000, 1, 9000]
    off = torch.tensor([0] + list(torch.tensor(lengths).cumsum(0)), dtype=torch.int32)
    items, _, groups, slots, slot_blocks = jfa.host_schedule_split(off, 256, 2, 152, with_slot_blocks=True)
    assert slots > 0
    first_block = [0]
    for L in lengths:
        first_block.append(first_block[-1] + (L + 127) // 128)
    seen = 0
    for g in groups.tolist():
        b, slot0, n = g[0], g[1], g[2]
        for c in range(n):
            slot = slot0 + c
            it = [r for r in items.tolist() if r[0] == -(slot + 1)]
            assert len(it) == 1
            kv_start = it[0][1]
            assert (kv_start - int(off[b])) % 128 == 0
            assert int(slot_blocks[slot]) == first_block[b] + (kv_start - int(off[b])) // 128
            seen += 1
    assert seen == slots
