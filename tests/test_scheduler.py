"""Host tile scheduler: cost-descending (LPT) order dealt zigzag to CTAs.

The pages: tiles are sorted on the host by KV workload, descending, and
handed to the SMs in a zigzag pattern (Meta's TLX Jagged Flash Attention
Beats FA4 on Blackwell With 3x Less Code, section "Optimizations layered on
top").  These tests need no GPU.
"""
import pytest
import torch

import jfa_inputs


@pytest.fixture(scope="module")
def jfa():
    import bwd_jagged_flashattention_gb300 as jfa
    jfa.build()
    return jfa


def _decode(items):
    b, start, length, packed = items.unbind(1)
    packed = packed.to(torch.int64) & 0xFFFFFFFF
    h = packed & 0xFF
    tile = (packed >> 8) & 0x7FFFFF
    two = packed >> 31
    return b, start, length, h, tile, two


def _cost(length, tile, two, Lq, broadcast_q, causal, is_bwd):
    """The documented cost model, restated: 128x128 block products + 1."""
    nkv = (length + 127) // 128
    if not is_bwd:
        c = 0
        for t in range(int(two) + 1):
            m = int(tile) + t
            c += min(m + 1, int(nkv)) if causal else int(nkv)
        return c + 1
    nq = (Lq + 127) // 128 if broadcast_q else int(nkv)
    return (nq - int(tile) if causal else nq) + 1


@pytest.mark.parametrize("name,is_bwd", [("tiny", 0), ("tiny", 1), ("ads_fwd", 0), ("ads_bwd", 1),
                                         ("extreme", 0), ("extreme", 1)])
def test_every_item_exactly_once(jfa, name, is_bwd):
    w = jfa_inputs.WORKLOADS[name]
    g = torch.Generator().manual_seed(5)
    L = jfa_inputs.draw_lengths(w.lengths, w.B, g)
    off = jfa_inputs.offsets_from_lengths(L)
    P = 152
    items, starts = jfa.host_schedule(off, w.Lq, w.H, w.broadcast_q, w.causal, bool(is_bwd), P)
    b, start, length, h, tile, two = _decode(items)
    seen = set()
    for i in range(items.shape[0]):
        key = (int(b[i]), int(h[i]), int(tile[i]))
        assert key not in seen
        seen.add(key)
        assert int(start[i]) == int(off[b[i]]) and int(length[i]) == int(off[b[i] + 1] - off[b[i]])
    expect = set()
    for bb in range(w.B):
        Lk = int(off[bb + 1] - off[bb])
        nkv = (Lk + 127) // 128
        for hh in range(w.H):
            if is_bwd:
                expect |= {(bb, hh, n) for n in range(nkv)}
            else:
                nq = (w.Lq + 127) // 128 if w.broadcast_q else nkv
                expect |= {(bb, hh, m) for m in range(0, nq, 2)}
    assert seen == expect
    assert int(starts[0]) == 0 and int(starts[-1]) == items.shape[0]
    assert torch.all(starts[1:] >= starts[:-1])


def test_lpt_zigzag_bound(jfa):
    """Sorted zigzag dealing stays within the LPT-style bound on the makespan."""
    w = jfa_inputs.WORKLOADS["extreme"]
    g = torch.Generator().manual_seed(6)
    off = jfa_inputs.offsets_from_lengths(jfa_inputs.draw_lengths(w.lengths, w.B, g))
    P = 152
    items, starts = jfa.host_schedule(off, w.Lq, w.H, True, False, False, P)
    b, start, length, h, tile, two = _decode(items)
    cost = [_cost(int(length[i]), int(tile[i]), int(two[i]), w.Lq, True, False, False) for i in range(len(b))]
    loads = [sum(cost[int(starts[p]):int(starts[p + 1])]) for p in range(P)]
    total, biggest = sum(cost), max(cost)
    lower = max(total / P, biggest)
    assert max(loads) <= 4 / 3 * lower + biggest
    # and it clearly beats the round-robin deal in generation order
    items_n, starts_n = jfa.host_schedule(off, w.Lq, w.H, True, False, False, P, policy=1)
    bn, sn, ln, hn, tn, twon = _decode(items_n)
    cost_n = [_cost(int(ln[i]), int(tn[i]), int(twon[i]), w.Lq, True, False, False) for i in range(len(bn))]
    loads_n = [sum(cost_n[int(starts_n[p]):int(starts_n[p + 1])]) for p in range(P)]
    assert max(loads) <= max(loads_n)


def test_zigzag_hand_example(jfa):
    """Six sequences, one head, P = 3 CTAs, broadcast Lq = 128 (one q tile).

    KV lengths 128*[1,5,3,6,2,4] give costs [2,6,4,7,3,5] (blocks + 1).
    Sorted descending: b = 3(7), 1(6), 5(5), 2(4), 4(3), 0(2).
    Zigzag: round 0 -> CTAs 0,1,2; round 1 -> CTAs 2,1,0.
    CTA 0: b3, b0; CTA 1: b1, b4; CTA 2: b5, b2.
    """
    L = torch.tensor([1, 5, 3, 6, 2, 4]) * 128
    off = jfa_inputs.offsets_from_lengths(L)
    items, starts = jfa.host_schedule(off, 128, 1, True, False, False, 3)
    b = items[:, 0].tolist()
    assert starts.tolist() == [0, 2, 4, 6]
    assert b == [3, 0, 1, 4, 5, 2]


def test_causal_costs_and_pairs(jfa):
    """Jagged causal forward pairs q tiles; the later tile of a pair sees one more KV block."""
    off = torch.tensor([0, 1000], dtype=torch.int32)      # 8 q tiles -> 4 items per head
    items, starts = jfa.host_schedule(off, 0, 2, False, True, False, 4)
    b, start, length, h, tile, two = _decode(items)
    assert sorted(int(t) for t in tile[h == 0]) == [0, 2, 4, 6]
    assert torch.all(two == 1)
    costs = [_cost(1000, int(tile[i]), 1, 0, False, True, False) for i in range(len(tile))]
    assert costs == sorted(costs, reverse=True) or len(set(starts.tolist())) > 1


@pytest.mark.parametrize("name,is_bwd", [("ads_fwd", 0), ("ads_bwd", 1), ("extreme", 0), ("extreme", 1)])
def test_broadcast_deal_per_head_group(jfa, name, is_bwd):
    """Broadcast Q with H dividing P: head h's items go to CTAs h, h+H, ...
    (G = P/H of them), dealt by the same cost sort and zigzag within the group; each
    CTA reads one head's Q tiles, in runs grouped by query tile, keeping the
    deal order (cost descending) inside a run."""
    w = jfa_inputs.WORKLOADS[name]
    g = torch.Generator().manual_seed(7)
    off = jfa_inputs.offsets_from_lengths(jfa_inputs.draw_lengths(w.lengths, w.B, g))
    P = 152
    assert P % w.H == 0
    G = P // w.H
    items, starts = jfa.host_schedule(off, w.Lq, w.H, True, False, bool(is_bwd), P)
    b, start, length, h, tile, two = _decode(items)
    cost = [_cost(int(length[i]), int(tile[i]), int(two[i]), w.Lq, True, False, bool(is_bwd)) for i in range(len(b))]
    for p in range(P):
        s, e = int(starts[p]), int(starts[p + 1])
        assert set(h[s:e].tolist()) <= {p % w.H}
        # runs of equal Q key: the forward's first query tile (the backward's
        # tile field is a key/value tile, and its Q key is the head alone)
        k = [0] * (e - s) if is_bwd else tile[s:e].tolist()
        assert k == sorted(k)
        for i in range(s + 1, e):
            if k[i - s] == k[i - 1 - s]:
                assert cost[i] <= cost[i - 1]
    # per-CTA loads equal the deal restated here: per head, stable cost sort
    # of the (b, tile) generation order, zigzag over the head's G CTAs
    loads = [0] * P
    for hh in range(w.H):
        gen = []
        for bb in range(w.B):
            Lk = int(off[bb + 1] - off[bb])
            nkv = (Lk + 127) // 128
            nq = (w.Lq + 127) // 128
            if is_bwd:
                gen += [_cost(Lk, n, 0, w.Lq, True, False, True) for n in range(nkv)]
            else:
                gen += [_cost(Lk, m, 1 if m + 1 < nq else 0, w.Lq, True, False, False) for m in range(0, nq, 2)]
        order = sorted(range(len(gen)), key=lambda i: -gen[i])
        for pos, o in enumerate(order):
            r, lane = divmod(pos, G)
            loads[((G - 1 - lane) if (r & 1) else lane) * w.H + hh] += gen[o]
    assert loads == [sum(cost[int(starts[p]):int(starts[p + 1])]) for p in range(P)]


def _greedy_restated(off, Lq, H, broadcast_q, causal, is_bwd, P):
    """The greedy longest-processing-time deal, restated: stable cost-descending
    sort of the (b, h, tile) generation order, then each item to the CTA of its
    group with the least cost so far (ties: lowest lane); per head group of
    P/H CTAs {h, h+H, ...} in broadcast mode when H divides P.  Returns the
    per-CTA item multisets as sorted lists of (b, h, tile)."""
    import heapq
    gen = []
    for bb in range(len(off) - 1):
        Lk = int(off[bb + 1] - off[bb])
        nkv = (Lk + 127) // 128
        for hh in range(H):
            if is_bwd:
                gen += [(bb, hh, n, _cost(Lk, n, 0, Lq, broadcast_q, causal, True)) for n in range(nkv)]
            else:
                nq = (Lq + 127) // 128 if broadcast_q else nkv
                gen += [(bb, hh, m, _cost(Lk, m, 1 if m + 1 < nq else 0, Lq, broadcast_q, causal, False))
                        for m in range(0, nq, 2)]
    order = sorted(range(len(gen)), key=lambda i: -gen[i][3])
    by_head = broadcast_q and H > 1 and P % H == 0
    groups = H if by_head else 1
    G = P // groups
    heaps = [[(0, lane) for lane in range(G)] for _ in range(groups)]
    owned = [[] for _ in range(P)]
    for o in order:
        bb, hh, t, c = gen[o]
        g = hh if by_head else 0
        load, lane = heapq.heappop(heaps[g])
        heapq.heappush(heaps[g], (load + c, lane))
        owned[lane * H + g if by_head else lane].append((bb, hh, t))
    return [sorted(x) for x in owned]


@pytest.mark.parametrize("name,is_bwd", [("ads_bwd", 0), ("ads_bwd", 1), ("extreme", 0), ("dense_llm", 0),
                                         ("dense_llm", 1), ("tiny", 0)])
def test_greedy_deal_matches_restatement(jfa, name, is_bwd):
    w = jfa_inputs.WORKLOADS[name]
    g = torch.Generator().manual_seed(11)
    off = jfa_inputs.offsets_from_lengths(jfa_inputs.draw_lengths(w.lengths, min(w.B, 256), g))
    P = 152
    Lq = w.Lq if w.broadcast_q else 0
    items, starts = jfa.host_schedule(off, Lq, w.H, w.broadcast_q, w.causal, bool(is_bwd), P,
                                      policy=jfa.SCHED_GREEDY)
    b, start, length, h, tile, two = _decode(items)
    got = [sorted((int(b[i]), int(h[i]), int(tile[i])) for i in range(int(starts[p]), int(starts[p + 1])))
           for p in range(P)]
    assert got == _greedy_restated(off, Lq, w.H, w.broadcast_q, w.causal, bool(is_bwd), P)
    # the allocation-free builder deals the same items in the same order
    items2, starts2 = jfa.host_schedule(off, Lq, w.H, w.broadcast_q, w.causal, bool(is_bwd), P, noalloc=True)
    assert torch.equal(items, items2) and torch.equal(starts, starts2)


def test_greedy_balances_the_ads_forward(jfa):
    """On the ads forward the greedy deal keeps the busiest CTA within 5% of
    the mean load, where the zigzag deal leaves it about 30% above."""
    w = jfa_inputs.WORKLOADS["ads_bwd"]
    off = jfa_inputs.make("ads_bwd")["offsets"]
    P = 152

    def ratio(policy):
        items, starts = jfa.host_schedule(off, w.Lq, w.H, True, False, False, P, policy=policy)
        b, start, length, h, tile, two = _decode(items)
        cost = [_cost(int(length[i]), int(tile[i]), int(two[i]), w.Lq, True, False, False) for i in range(len(b))]
        loads = [sum(cost[int(starts[p]):int(starts[p + 1])]) for p in range(P)]
        return max(loads) / (sum(loads) / P)

    assert ratio(jfa.SCHED_GREEDY) < 1.05
    assert ratio(jfa.SCHED_ZIGZAG) > 1.2


@pytest.mark.parametrize("name,causal", [("ads_bwd", False), ("extreme", False), ("tiny", True)])
def test_clc_list_is_cost_sorted_generation_order(jfa, name, causal):
    """Cluster Launch Control backward: one slice holding every item, largest
    cost first, equal costs in generation order (sequence, head, key tile) --
    not grouped by head, since the CTAs that run together take consecutive
    entries -- built in linear time (the extreme workload's tens of thousands
    of items well inside a second)."""
    import time
    w = jfa_inputs.WORKLOADS[name]
    L = jfa_inputs.draw_lengths(w.lengths, w.B, torch.Generator().manual_seed(6))
    off = jfa_inputs.offsets_from_lengths(L)
    t0 = time.perf_counter()
    items, starts = jfa.host_schedule(off, w.Lq, w.H, w.broadcast_q, causal, True, 1, policy=jfa.SCHED_CLC)
    took = time.perf_counter() - t0
    b, start, length, h, tile, two = _decode(items)
    n = items.shape[0]
    assert starts.tolist() == [0, n]
    gen = [(bb, hh, t) for bb in range(w.B) for hh in range(w.H)
           for t in range((int(off[bb + 1] - off[bb]) + 127) // 128)]
    assert n == len(gen)
    cost = {g: _cost(int(off[g[0] + 1] - off[g[0]]), g[2], 0, w.Lq, w.broadcast_q, causal, True) for g in gen}
    expect = sorted(gen, key=lambda g: -cost[g])  # stable: ties keep generation order
    got = list(zip(b.tolist(), h.tolist(), tile.tolist()))
    assert got == expect
    assert took < 1.0, f"CLC list build took {took:.2f} s for {n} items"


def test_clc_policy_is_backward_single_slice_only(jfa):
    off = jfa_inputs.offsets_from_lengths(torch.tensor([300, 5, 129], dtype=torch.int32))
    with pytest.raises(jfa.JFAError):
        jfa.host_schedule(off, 256, 2, True, False, True, 152, policy=jfa.SCHED_CLC)
    with pytest.raises(jfa.JFAError):
        jfa.host_schedule(off, 256, 2, True, False, False, 1, policy=jfa.SCHED_CLC)


@pytest.mark.parametrize("name,P", [("ads_bwd", 152), ("extreme", 152), ("tiny", 8), ("ads_bwd", 150)])
def test_queue_schedule_layout(jfa, name, P):
    """Backward queues: with broadcast Q and H | P one queue per head (else
    one), each longest-first and stable, every item once, bounds in
    cta_start[0..G], the G take counters after them zero."""
    w = jfa_inputs.WORKLOADS[name]
    L = jfa_inputs.draw_lengths(w.lengths, w.B, torch.Generator().manual_seed(7))
    off = jfa_inputs.offsets_from_lengths(L)
    items, starts = jfa.host_schedule(off, w.Lq, w.H, w.broadcast_q, w.causal, True, P, policy=jfa.SCHED_QUEUE)
    G = w.H if (w.broadcast_q and 1 < w.H <= 255 and P % w.H == 0) else 1
    st = starts.tolist()
    assert st[0] == 0 and st[G] == items.shape[0] and st[G + 1:2 * G + 1] == [0] * G
    b, start, length, h, tile, two = _decode(items)
    gen = [(bb, hh, t) for bb in range(w.B) for hh in range(w.H)
           for t in range((int(off[bb + 1] - off[bb]) + 127) // 128)]
    assert sorted(zip(b.tolist(), h.tolist(), tile.tolist())) == sorted(gen)
    for g in range(G):
        lo, hi = st[g], st[g + 1]
        part = list(zip(b[lo:hi].tolist(), h[lo:hi].tolist(), tile[lo:hi].tolist()))
        if G > 1:
            assert all(hh == g for _, hh, _ in part)
        mine = [x for x in gen if G == 1 or x[1] == g]
        cost = {x: _cost(int(off[x[0] + 1] - off[x[0]]), x[2], 0, w.Lq, w.broadcast_q, w.causal, True) for x in mine}
        assert part == sorted(mine, key=lambda x: -cost[x])


def test_queue_policy_is_backward_only(jfa):
    off = jfa_inputs.offsets_from_lengths(torch.tensor([300, 5, 129], dtype=torch.int32))
    with pytest.raises(jfa.JFAError):
        jfa.host_schedule(off, 256, 2, True, False, False, 8, policy=jfa.SCHED_QUEUE)
