"""Pins for the oracle's block-sparse variant, against things other than itself.

The pages describe the variant in one sentence: it only adds iteration over
selected key blocks and leaves the rest of the kernel as it is (TLX porta
l'attenzione jagged su Blackwell oltre FA4 con un terzo del codice, section
"The turning point").  Reading taken (the oracle's header states it): blocks
of 128 keys counted from each sequence's start; a selection applies to one
(sequence, head) pair; mask layout uint8 [NB, H] with
NB = sum_b ceil(len_b / 128).

* gathered dense: for every (sequence, head), attention over only the keys of
  the selected blocks, computed as a small dense problem in torch fp64 with
  autograd -- an independent computation (no masking, no -inf, library
  softmax, reverse-mode AD) whose gradients are scattered back;
* exact special cases: a pair with no selected block has O = 0, LSE = -inf
  and no gradient; keys of unselected blocks get exactly zero dK and dV;
* an all-ones mask reproduces the dense oracle bit for bit (broadcast dQ up
  to the order in which the oracle's threads add their partial sums).
"""
import math

import pytest
import torch

import jfa_inputs
import oracle


def gathered_dense(q, k, v, do, offsets, Lq, broadcast_q, causal, scale, mask):
    """(o, lse, dq, dk, dv) in the oracle's layouts, one small dense problem per (b, h)."""
    offsets = [int(x) for x in offsets]
    B = len(offsets) - 1
    N = offsets[-1]
    H, D = k.shape[1], k.shape[2]
    q, k, v, do = (t.to(torch.float64) for t in (q, k, v, do))
    o_out = torch.zeros((B, Lq, H, D) if broadcast_q else (N, H, D), dtype=torch.float64)
    lse_out = torch.full((B, H, Lq) if broadcast_q else (H, N), -math.inf, dtype=torch.float64)
    dq_out = torch.zeros_like(q)
    dk_out = torch.zeros_like(k)
    dv_out = torch.zeros_like(v)
    bstart = 0
    for b in range(B):
        s0, Lk = offsets[b], offsets[b + 1] - offsets[b]
        nblk = (Lk + 127) // 128
        for h in range(H):
            keys = [j for j in range(Lk) if mask[bstart + j // 128, h]]
            rows = range(Lq) if broadcast_q else range(Lk)
            if not keys or len(rows) == 0:
                continue
            idx = torch.tensor(keys)
            qb = (q[:, h] if broadcast_q else q[s0:s0 + Lk, h]).clone().requires_grad_(True)
            kb = k[s0 + idx, h].clone().requires_grad_(True)
            vb = v[s0 + idx, h].clone().requires_grad_(True)
            dob = do[b, :, h] if broadcast_q else do[s0:s0 + Lk, h]
            s = scale * qb @ kb.T
            if causal:
                pos = torch.arange(len(rows))[:, None]
                s = s.masked_fill(idx[None, :] > pos, -math.inf)
            live = torch.isfinite(s).any(dim=1)          # rows with at least one visible key
            s_live = s[live]
            lse = torch.logsumexp(s_live, dim=1)
            o = torch.softmax(s_live, dim=1) @ vb
            gq, gk, gv = torch.autograd.grad((o * dob[live]).sum(), (qb, kb, vb), allow_unused=True)
            live_rows = torch.nonzero(live).flatten()
            if broadcast_q:
                o_out[b, live_rows, h] = o.detach()
                lse_out[b, h, live_rows] = lse.detach()
                dq_out[:, h] += gq
            else:
                o_out[s0 + live_rows, h] = o.detach()
                lse_out[h, s0 + live_rows] = lse.detach()
                dq_out[s0:s0 + Lk, h] += gq
            dk_out[s0 + idx, h] = gk
            dv_out[s0 + idx, h] = gv
        bstart += nblk
    return o_out, lse_out, dq_out, dk_out, dv_out


def _inputs(B, Lq, H, D, lengths, broadcast_q, causal, seed):
    x = jfa_inputs.custom(B, Lq, H, D, lengths, broadcast_q, causal, seed=seed)
    g = torch.Generator().manual_seed(2000 + seed)
    for name in ("q", "k", "v", "do"):
        x[name] = torch.randn(x[name].shape, generator=g, dtype=torch.float64)
    return x


def _oracle(x, mask):
    a = (x["q"], x["k"], x["v"])
    o, lse = oracle.fwd(*a, x["offsets"], x["Lq"], x["broadcast_q"], x["causal"], x["scale"], kv_block_mask=mask)
    dq, dk, dv = oracle.bwd(*a, x["do"], x["offsets"], x["Lq"], x["broadcast_q"], x["causal"], x["scale"],
                            kv_block_mask=mask)
    return o, lse, dq, dk, dv


def _close(a, b, tol=1e-10):
    fin = torch.isfinite(b)
    assert torch.equal(torch.isfinite(a), fin), "non-finite pattern differs"
    assert torch.equal(a[~fin], b[~fin])
    if fin.any():
        err = (a[fin] - b[fin]).abs().max().item()
        assert err <= tol, f"max abs err {err}"


CASES = [
    # B, Lq, H, D, lengths, broadcast_q, causal
    (5, 5, 2, 8, [300, 129, 0, 257, 50], True, False),
    (3, 130, 1, 4, [256, 384, 1], True, False),
    (2, 0, 2, 8, [260, 140], False, False),
    (2, 0, 2, 4, [300, 129], False, True),
]


def _masks(offsets, H, seed):
    """Random selections plus the edge patterns: none, tail only, first block only, all."""
    nb = jfa_inputs.num_kv_blocks(offsets)
    rand = jfa_inputs.kv_block_mask(offsets, H, 0.5, seed)
    none_first = rand.clone()
    none_first[:, 0] = 0                                   # head 0 sees no key in any sequence
    lens = (offsets[1:] - offsets[:-1]).tolist()
    tail = torch.zeros(nb, H, dtype=torch.uint8)
    first = torch.zeros(nb, H, dtype=torch.uint8)
    g = 0
    for L in lens:
        n = (L + 127) // 128
        if n:
            tail[g + n - 1] = 1                            # the (possibly ragged) last block
            first[g] = 1
        g += n
    return {"random": rand, "head0_empty": none_first, "tail_only": tail, "first_only": first,
            "all": torch.ones(nb, H, dtype=torch.uint8)}


@pytest.mark.parametrize("case", CASES)
def test_block_sparse_equals_gathered_dense(case):
    B, Lq, H, D, lengths, bq, causal = case
    x = _inputs(B, Lq, H, D, lengths, bq, causal, seed=sum(lengths) % 97)
    for name, mask in _masks(x["offsets"], H, seed=len(lengths)).items():
        got = _oracle(x, mask)
        ref = gathered_dense(x["q"], x["k"], x["v"], x["do"], x["offsets"], x["Lq"], bq, causal, x["scale"], mask)
        for a, b, what in zip(got, ref, ("o", "lse", "dq", "dk", "dv")):
            try:
                _close(a, b)
            except AssertionError as e:
                raise AssertionError(f"{name}/{what}: {e}") from None


def test_unselected_keys_get_exact_zeros():
    x = _inputs(3, 7, 2, 8, [300, 129, 257], True, False, seed=5)
    mask = jfa_inputs.kv_block_mask(x["offsets"], 2, 0.5, 9)
    mask[:, 1] = 0                                         # head 1 selects nothing at all
    o, lse, dq, dk, dv = _oracle(x, mask)
    assert torch.all(o[:, :, 1] == 0) and torch.all(lse[:, 1] == -math.inf)
    assert torch.all(dq[:, 1] == 0) and torch.all(dk[:, 1] == 0) and torch.all(dv[:, 1] == 0)
    off = x["offsets"].tolist()
    g = 0
    for b in range(3):
        n = (off[b + 1] - off[b] + 127) // 128
        for blk in range(n):
            rows = slice(off[b] + 128 * blk, min(off[b + 1], off[b] + 128 * (blk + 1)))
            if not mask[g + blk, 0]:
                assert torch.all(dk[rows, 0] == 0) and torch.all(dv[rows, 0] == 0)
            else:  # (dK can vanish: a block whose one key is a row's only visible key gets dS = 0)
                assert dv[rows, 0].abs().sum() > 0
        g += n


def test_all_ones_mask_is_the_dense_oracle():
    x = _inputs(4, 9, 2, 8, [129, 0, 300, 77], True, False, seed=11)
    ones = torch.ones(jfa_inputs.num_kv_blocks(x["offsets"]), 2, dtype=torch.uint8)
    dense = _oracle(x, None)
    sparse = _oracle(x, ones)
    for what, a, b in zip(("o", "lse", "dq", "dk", "dv"), dense, sparse):
        if what == "dq":  # broadcast dQ sums per-thread buffers in scheduling order: last-bit differences
            _close(a, b, tol=1e-12)
        else:
            assert torch.equal(a, b), what


def test_mask_shape_is_checked():
    x = _inputs(2, 3, 2, 4, [130, 5], True, False, seed=1)
    with pytest.raises(ValueError):
        _oracle(x, torch.ones(2, 2, dtype=torch.uint8))    # NB is 3 here


MASK_MUTATIONS = {
    # key j read as belonging to block (j + 1) / 128
    "block_index_off_by_one": ("} else if (sel && !sel[(int64_t)(j / 128) * sel_stride]) {",
                               "} else if (sel && !sel[(int64_t)((j + 1) / 128) * sel_stride]) {"),
    # mask read head-major ([H, NB]) instead of block-major ([NB, H])
    "mask_layout_transposed": ("} else if (sel && !sel[(int64_t)(j / 128) * sel_stride]) {",
                               "} else if (sel && !sel[(int64_t)(j / 128)]) {"),
}


@pytest.mark.parametrize("name", sorted(MASK_MUTATIONS))
def test_pins_reject_mask_mutant(tmp_path, name):
    before, after = MASK_MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert src.count(before) == 1
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(before, after))
    mut = oracle.Oracle(oracle.compile_source(str(path), str(tmp_path / f"lib{name}.so")))
    x = _inputs(5, 5, 2, 8, [300, 129, 0, 257, 50], True, False, seed=4)
    mask = jfa_inputs.kv_block_mask(x["offsets"], 2, 0.5, 3)
    a = (x["q"], x["k"], x["v"])
    o, lse = mut.fwd(*a, x["offsets"], x["Lq"], True, False, x["scale"], kv_block_mask=mask)
    ref = gathered_dense(x["q"], x["k"], x["v"], x["do"], x["offsets"], x["Lq"], True, False, x["scale"], mask)
    with pytest.raises(AssertionError):
        _close(o, ref[0])
        _close(lse, ref[1])
