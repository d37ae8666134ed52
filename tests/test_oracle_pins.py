"""Pins for the fp64 oracle: it is checked here against things other than itself.

* brute force: padded dense attention with key masking, torch fp64 on the CPU,
  gradients from torch.autograd (a different computation: dense padded
  matrices, library softmax, reverse-mode AD instead of the closed-form
  gradient formulas);
* a hand-derived worked example (tests/golden/worked_example_2x2.txt);
* closed forms (one key; zero queries), invariants (rows of P sum to one via
  constant V; sum_j dV_j = sum_i dO_i; sum_j dK_j = 0; key permutation;
  key shift);
* central finite differences of L = <dO, O>;
* broadcast-Q: dQ equals the sum over sequences of single-sequence dQ, and
  O/LSE equal the single-sequence results;
* causal jagged with one sequence equals torch's scaled_dot_product_attention.

The operation is the one the pages define: FlashAttention run directly on
packed Q/K/V plus an offsets tensor ("Why attention in GEM needed a rewrite",
Meta's TLX Jagged Flash Attention Beats FA4 on Blackwell With 3x Less Code),
with a broadcast Q whose gradient is summed over the batch (Meta's 3.2K-line
Triton kernel outruns FlashAttention-4 on jagged Blackwell attention, second
paragraph).
"""
import math
import os

import pytest
import torch

import jfa_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# Independent brute force: padded dense attention, torch fp64 + autograd.
# ----------------------------------------------------------------------------
def brute_force(q, k, v, do, offsets, Lq, broadcast_q, causal, scale):
    """Returns (o, lse, dq, dk, dv) in the oracle's layouts, computed densely.

    Every non-empty sequence is padded to the longest one; padded keys get a
    -inf mask.  Sequences with no keys are skipped (their outputs stay zero,
    LSE -inf), matching the empty-row convention.
    """
    offsets = [int(x) for x in offsets]
    B = len(offsets) - 1
    N = offsets[-1]
    H, D = k.shape[1], k.shape[2]
    q = q.detach().to(torch.float64).clone().requires_grad_(True)
    k = k.detach().to(torch.float64).clone().requires_grad_(True)
    v = v.detach().to(torch.float64).clone().requires_grad_(True)
    do = do.to(torch.float64)
    lens = [offsets[b + 1] - offsets[b] for b in range(B)]
    Lmax = max(lens) if lens else 0
    Lqmax = Lq if broadcast_q else Lmax
    o_out = torch.zeros((B, Lq, H, D) if broadcast_q else (N, H, D), dtype=torch.float64)
    lse_out = torch.full((B, H, Lq) if broadcast_q else (H, N), -math.inf, dtype=torch.float64)
    if Lmax == 0:
        return o_out, lse_out, torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    # Padded [B, H, L, D] views (differentiable gathers); padded keys are masked.
    kmask = torch.zeros(B, Lmax, dtype=torch.bool)
    for b in range(B):
        kmask[b, :lens[b]] = True
    kpad = torch.stack([torch.nn.functional.pad(k[offsets[b]:offsets[b + 1]].permute(1, 0, 2),
                                                (0, 0, 0, Lmax - lens[b])) for b in range(B)])
    vpad = torch.stack([torch.nn.functional.pad(v[offsets[b]:offsets[b + 1]].permute(1, 0, 2),
                                                (0, 0, 0, Lmax - lens[b])) for b in range(B)])
    if broadcast_q:
        qpad = q.permute(1, 0, 2).unsqueeze(0).expand(B, H, Lq, D)
    else:
        qpad = torch.stack([torch.nn.functional.pad(q[offsets[b]:offsets[b + 1]].permute(1, 0, 2),
                                                    (0, 0, 0, Lmax - lens[b])) for b in range(B)])
    s = torch.einsum("bhid,bhjd->bhij", qpad, kpad) * scale
    mask = kmask[:, None, None, :].expand(B, H, Lqmax, Lmax)
    if causal:
        i = torch.arange(Lqmax)[:, None]
        j = torch.arange(Lmax)[None, :]
        mask = mask & (j <= i)[None, None]
    s = s.masked_fill(~mask, -math.inf)
    nonempty = torch.tensor([L > 0 for L in lens])
    s_safe = torch.where(nonempty[:, None, None, None], s, torch.zeros_like(s))
    p = torch.softmax(s_safe, dim=-1)
    lse = torch.logsumexp(s_safe, dim=-1)
    o = torch.einsum("bhij,bhjd->bhid", p, vpad)
    # scatter back into the oracle's layouts
    loss = 0.0
    for b in range(B):
        if lens[b] == 0:
            continue
        if broadcast_q:
            ob = o[b].permute(1, 0, 2)                     # [Lq, H, D]
            o_out[b] = ob.detach()
            lse_out[b] = lse[b].detach()
            loss = loss + (ob * do[b]).sum()
        else:
            L = lens[b]
            ob = o[b, :, :L].permute(1, 0, 2)              # [L, H, D]
            o_out[offsets[b]:offsets[b + 1]] = ob.detach()
            lse_out[:, offsets[b]:offsets[b + 1]] = lse[b, :, :L].detach()
            loss = loss + (ob * do[offsets[b]:offsets[b + 1]]).sum()
    dq, dk, dv = torch.autograd.grad(loss, (q, k, v), allow_unused=True)
    dq = torch.zeros_like(q) if dq is None else dq
    return o_out, lse_out, dq, dk, dv


def _run_oracle(x, causal=None):
    causal = x["causal"] if causal is None else causal
    o, lse = oracle.fwd(x["q"], x["k"], x["v"], x["offsets"], x["Lq"], x["broadcast_q"], causal, x["scale"])
    dq, dk, dv = oracle.bwd(x["q"], x["k"], x["v"], x["do"], x["offsets"], x["Lq"], x["broadcast_q"],
                            causal, x["scale"])
    return o, lse, dq, dk, dv


def _f64_inputs(B, Lq, H, D, lengths, broadcast_q, causal, seed):
    x = jfa_inputs.custom(B, Lq, H, D, lengths, broadcast_q, causal, seed=seed)
    # fp64 (not bf16) values so the comparison exercises the full fp64 path
    g = torch.Generator().manual_seed(1000 + seed)
    for name in ("q", "k", "v", "do"):
        x[name] = torch.randn(x[name].shape, generator=g, dtype=torch.float64)
    return x


def _close(a, b, tol):
    a, b = a.to(torch.float64), b.to(torch.float64)
    fin = torch.isfinite(b)
    assert torch.equal(torch.isfinite(a), fin), "non-finite pattern differs"
    assert torch.equal(a[~fin], b[~fin])
    if fin.any():
        err = (a[fin] - b[fin]).abs().max().item()
        assert err <= tol, f"max abs err {err} > {tol}"


CASES = [
    # B, Lq, H, D, lengths, broadcast_q, causal
    (3, 5, 2, 4, [3, 1, 7], True, False),
    (4, 8, 1, 8, [0, 5, 2, 9], True, False),
    (3, 0, 2, 4, [4, 1, 6], False, False),
    (3, 0, 2, 4, [4, 1, 6], False, True),
    (2, 0, 1, 16, [16, 11], False, True),
    (5, 3, 3, 2, [2, 2, 0, 1, 5], True, False),
]


@pytest.mark.parametrize("case", CASES)
def test_brute_force(case):
    B, Lq, H, D, lengths, bq, causal = case
    x = _f64_inputs(B, Lq, H, D, lengths, bq, causal, seed=len(lengths) + sum(lengths))
    got = _run_oracle(x)
    ref = brute_force(x["q"], x["k"], x["v"], x["do"], x["offsets"], Lq, bq, causal, x["scale"])
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), got, ref):
        _close(a, b, 1e-12)


def _parse_golden(path):
    env = {"ln": math.log}
    vals = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, rhs = (t.strip() for t in line.split("=", 1))
        rows = [[eval(c, {"__builtins__": {}}, env) for c in r.split(",")] for r in rhs.split(";")]
        vals[key] = torch.tensor(rows, dtype=torch.float64)
    return vals


def test_worked_example_golden():
    g = _parse_golden(os.path.join(GOLDEN, "worked_example_2x2.txt"))
    scale = float(g["scale"].item())
    q, k, v, do = (g[n].reshape(2, 1, 2) for n in ("q", "k", "v", "do"))
    off = torch.tensor([0, 2], dtype=torch.int32)
    # jagged self-attention, one sequence
    o, lse = oracle.fwd(q, k, v, off, 0, False, False, scale)
    dq, dk, dv = oracle.bwd(q, k, v, do, off, 0, False, False, scale)
    _close(o.reshape(2, 2), g["o"], 1e-14)
    _close(lse.reshape(2), g["lse"].reshape(2), 1e-14)
    _close(dq.reshape(2, 2), g["dq"], 1e-14)
    _close(dk.reshape(2, 2), g["dk"], 1e-14)
    _close(dv.reshape(2, 2), g["dv"], 1e-14)
    # broadcast-Q, the same sequence twice: outputs repeat, dQ doubles
    off2 = torch.tensor([0, 2, 4], dtype=torch.int32)
    k2, v2 = torch.cat([k, k]), torch.cat([v, v])
    do2 = torch.stack([do, do])                              # [B=2, Lq=2, H=1, D=2]
    o, lse = oracle.fwd(q, k2, v2, off2, 2, True, False, scale)
    dq, dk, dv = oracle.bwd(q, k2, v2, do2, off2, 2, True, False, scale)
    for b in range(2):
        _close(o[b].reshape(2, 2), g["o"], 1e-14)
        _close(lse[b].reshape(2), g["lse"].reshape(2), 1e-14)
        _close(dk[2 * b:2 * b + 2].reshape(2, 2), g["dk"], 1e-14)
        _close(dv[2 * b:2 * b + 2].reshape(2, 2), g["dv"], 1e-14)
    _close(dq.reshape(2, 2), 2 * g["dq"], 1e-14)


def test_single_key_closed_form():
    """Lk = 1: O_i = v_0, LSE_i = s_i0, dS = 0 so dQ = dK = 0, dV_0 = sum_i dO_i."""
    x = _f64_inputs(3, 6, 2, 8, [1, 1, 1], True, False, seed=7)
    o, lse, dq, dk, dv = _run_oracle(x)
    for b in range(3):
        _close(o[b], x["v"][b].unsqueeze(0).expand(6, 2, 8), 1e-14)
        s = x["scale"] * torch.einsum("ihd,hd->hi", x["q"], x["k"][b])
        _close(lse[b], s, 1e-13)
        _close(dv[b], x["do"][b].sum(0), 1e-13)
    _close(dq, torch.zeros_like(dq), 1e-14)
    _close(dk, torch.zeros_like(dk), 1e-14)


def test_zero_query_closed_form():
    """q = 0: uniform weights, O_i = mean_j v_j, LSE_i = ln Lk."""
    x = _f64_inputs(3, 4, 2, 8, [5, 2, 9], True, False, seed=8)
    x["q"] = torch.zeros_like(x["q"])
    o, lse = oracle.fwd(x["q"], x["k"], x["v"], x["offsets"], 4, True, False, x["scale"])
    off = x["offsets"].tolist()
    for b in range(3):
        mean = x["v"][off[b]:off[b + 1]].mean(0)
        _close(o[b], mean.unsqueeze(0).expand(4, 2, 8), 1e-14)
        _close(lse[b], torch.full((2, 4), math.log(off[b + 1] - off[b]), dtype=torch.float64), 1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_invariants(causal):
    lengths = [6, 1, 9, 4]
    x = _f64_inputs(4, 0, 2, 8, lengths, False, causal, seed=9)
    off = x["offsets"].tolist()
    # constant V (per head) => O = that constant: the rows of P sum to one
    c = torch.randn(2, 8, dtype=torch.float64)
    o, _ = oracle.fwd(x["q"], x["k"], c.expand_as(x["v"]).contiguous(), x["offsets"], 0, False, causal,
                      x["scale"])
    _close(o, c.expand_as(o), 1e-13)
    _, _, dq, dk, dv = _run_oracle(x)
    for b in range(4):
        sl = slice(off[b], off[b + 1])
        _close(dv[sl].sum(0), x["do"][sl].sum(0), 1e-12)          # sum_j dV_j = sum_i dO_i
        _close(dk[sl].sum(0), torch.zeros(2, 8, dtype=torch.float64), 1e-12)  # sum_j dS_ij = 0


def test_key_permutation_and_shift():
    x = _f64_inputs(2, 5, 2, 8, [7, 4], True, False, seed=10)
    o, lse, dq, dk, dv = _run_oracle(x)
    perm = torch.cat([torch.randperm(7, generator=torch.Generator().manual_seed(3)),
                      7 + torch.randperm(4, generator=torch.Generator().manual_seed(4))])
    y = dict(x, k=x["k"][perm].contiguous(), v=x["v"][perm].contiguous())
    o2, lse2, dq2, dk2, dv2 = _run_oracle(y)
    _close(o2, o, 1e-13)
    _close(lse2, lse, 1e-13)
    _close(dq2, dq, 1e-12)
    _close(dk2, dk[perm], 1e-12)
    _close(dv2, dv[perm], 1e-12)
    # adding one vector to every key of a sequence shifts each score row by a constant
    shift = torch.randn(1, 2, 8, dtype=torch.float64)
    y = dict(x, k=(x["k"] + shift).contiguous())
    o3, lse3 = oracle.fwd(y["q"], y["k"], y["v"], y["offsets"], 5, True, False, y["scale"])
    _close(o3, o, 1e-12)
    delta = x["scale"] * torch.einsum("ihd,hd->hi", x["q"], shift[0])
    _close(lse3, lse + delta.unsqueeze(0), 1e-12)


@pytest.mark.parametrize("bq,causal", [(True, False), (False, False), (False, True)])
def test_finite_differences(bq, causal):
    """dQ, dK, dV equal central differences of L = sum <dO, O> (h = 1e-6)."""
    lengths = [3, 5]
    x = _f64_inputs(2, 4 if bq else 0, 1, 4, lengths, bq, causal, seed=11)
    _, _, dq, dk, dv = _run_oracle(x)

    def loss(q, k, v):
        o, _ = oracle.fwd(q, k, v, x["offsets"], x["Lq"], bq, causal, x["scale"])
        return float((o * x["do"]).sum())

    h = 1e-6
    g = torch.Generator().manual_seed(12)
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        t = x[name]
        for _ in range(6):
            idx = tuple(int(torch.randint(0, s, (1,), generator=g)) for s in t.shape)
            tp, tm = t.clone(), t.clone()
            tp[idx] += h
            tm[idx] -= h
            args = {n: x[n] for n in ("q", "k", "v")}
            lp = loss(**dict(args, **{name: tp}))
            lm = loss(**dict(args, **{name: tm}))
            fd = (lp - lm) / (2 * h)
            an = float(grad[idx])
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, idx, fd, an)


def test_broadcast_equals_per_sequence_sum():
    lengths = [5, 0, 3, 8]
    x = _f64_inputs(4, 6, 2, 8, lengths, True, False, seed=13)
    o, lse, dq, dk, dv = _run_oracle(x)
    off = x["offsets"].tolist()
    dq_sum = torch.zeros_like(dq)
    for b in range(4):
        sl = slice(off[b], off[b + 1])
        one = torch.tensor([0, off[b + 1] - off[b]], dtype=torch.int32)
        ob, lb = oracle.fwd(x["q"], x["k"][sl], x["v"][sl], one, 6, True, False, x["scale"])
        dqb, dkb, dvb = oracle.bwd(x["q"], x["k"][sl], x["v"][sl], x["do"][b:b + 1], one, 6, True, False,
                                   x["scale"])
        _close(o[b:b + 1], ob, 0.0)
        _close(lse[b:b + 1], lb, 0.0)
        _close(dk[sl], dkb, 0.0)
        _close(dv[sl], dvb, 0.0)
        dq_sum += dqb
    _close(dq, dq_sum, 1e-12)


def test_causal_single_sequence_matches_sdpa():
    L, H, D = 13, 2, 8
    x = _f64_inputs(1, 0, H, D, [L], False, True, seed=14)
    o, lse = oracle.fwd(x["q"], x["k"], x["v"], x["offsets"], 0, False, True, x["scale"])
    q, k, v = (x[n].permute(1, 0, 2).unsqueeze(0) for n in ("q", "k", "v"))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=x["scale"])
    _close(o, ref[0].permute(1, 0, 2), 1e-13)


def test_empty_sequences():
    """Lk = 0: O rows are zero, LSE is -inf, and the sequence adds nothing to dQ."""
    x = _f64_inputs(3, 4, 1, 4, [0, 3, 0], True, False, seed=15)
    o, lse, dq, dk, dv = _run_oracle(x)
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    assert torch.all(lse[0] == -math.inf) and torch.all(lse[2] == -math.inf)
    y = dict(x, offsets=torch.tensor([0, 3], dtype=torch.int32), do=x["do"][1:2])
    dq1, _, _ = oracle.bwd(y["q"], y["k"], y["v"], y["do"], y["offsets"], 4, True, False, y["scale"])
    _close(dq, dq1, 0.0)
    # B = 0 is a valid, empty call
    z = jfa_inputs.custom(0, 4, 1, 4, [], True, False)
    o, lse = oracle.fwd(z["q"], z["k"], z["v"], z["offsets"], 4, True, False, z["scale"])
    assert o.numel() == 0 and lse.numel() == 0


def test_bf16_inputs_widen_exactly():
    """The bf16 entry widens inputs exactly: it equals the fp64 entry on the same values."""
    x = jfa_inputs.make("tiny")
    a = _run_oracle(x)
    y = {**x, **{n: x[n].to(torch.float64) for n in ("q", "k", "v", "do")}}
    b = _run_oracle(y)
    # per-(sequence, head) outputs are computed in a fixed order: exact;
    # the broadcast dQ batch sum depends on the OpenMP thread split: rounding only
    for name, u, w in zip(("o", "lse", "dq", "dk", "dv"), a, b):
        _close(u, w, 1e-12 if name == "dq" else 0.0)


def test_workload_generator_recipe():
    """The workloads carry the stated shapes and length distributions."""
    t = jfa_inputs.make("tiny")
    L = (t["offsets"][1:] - t["offsets"][:-1])
    assert t["q"].shape == (32, 2, 64) and t["q"].dtype == torch.bfloat16
    assert int(L.min()) >= 1 and int(L.max()) <= 64
    g = torch.Generator().manual_seed(3)
    L = jfa_inputs.draw_lengths(jfa_inputs.WORKLOADS["ads_bwd"].lengths, 512, g)
    assert int(L.min()) >= 8 and int(L.max()) <= 4096
    assert 180 <= float(L.float().median()) <= 330
    L = jfa_inputs.draw_lengths(jfa_inputs.WORKLOADS["extreme"].lengths, 2048, g)
    assert int((L >= 4096).sum()) == 205 and int((L <= 32).sum()) == 1843
