"""GPU parity at the five workloads' full sizes, in the launch configuration
bench.py times (one persistent CTA per SM, the host LPT + zigzag schedule,
one workspace reused by the forward and the backward).

Where the fp64 oracle can afford the whole workload it checks every element
(tiny; ads forward; ads forward+backward).  Elsewhere it checks sampled
outputs it can compute on their own: whole sequences x heads (sliced out of
the same inputs) for O, LSE, dK, dV and the per-sequence dQ, and, for the
broadcast dQ that sums over every sequence, every head over the whole batch.
"""
import pytest
import torch

import jfa_inputs
import oracle
from tests.gpu_util import check_all, check_grad, check_o_lse, gpu_fwd_bwd, oracle_fwd_bwd

pytestmark = pytest.mark.gpu


def _slice_heads(x, h):
    y = dict(x)
    for n in ("q", "k", "v", "do"):
        if n in x:
            y[n] = x[n][..., h:h + 1, :].contiguous()
    return y


def _sub_batch(x, seqs):
    """A batch of the chosen sequences only (the oracle runs them on their own)."""
    off = x["offsets"].tolist()
    ks, vs, qs, dos, lens = [], [], [], [], []
    for b in seqs:
        sl = slice(off[b], off[b + 1])
        ks.append(x["k"][sl])
        vs.append(x["v"][sl])
        lens.append(off[b + 1] - off[b])
        if x["broadcast_q"]:
            dos.append(x["do"][b:b + 1])
        else:
            qs.append(x["q"][sl])
            dos.append(x["do"][sl])
    y = dict(x, B=len(seqs), k=torch.cat(ks), v=torch.cat(vs), do=torch.cat(dos),
             offsets=jfa_inputs.offsets_from_lengths(torch.tensor(lens)))
    y["N"] = int(y["offsets"][-1])
    if not x["broadcast_q"]:
        y["q"] = torch.cat(qs)
    return y


def _gather_outputs(x, got, seqs, h):
    """The GPU outputs of the chosen sequences and head, in the sub-batch's layout."""
    off = x["offsets"].tolist()
    o, lse, dk, dv, dq = [], [], [], [], []
    for b in seqs:
        sl = slice(off[b], off[b + 1])
        dk.append(got["dk"][sl, h:h + 1])
        dv.append(got["dv"][sl, h:h + 1])
        if x["broadcast_q"]:
            o.append(got["o"][b:b + 1, :, h:h + 1])
            lse.append(got["lse"][b:b + 1, h:h + 1])
        else:
            o.append(got["o"][sl, h:h + 1])
            lse.append(got["lse"][h:h + 1, sl])
            dq.append(got["dq"][sl, h:h + 1])
    res = {"o": torch.cat(o), "lse": torch.cat(lse, dim=0 if x["broadcast_q"] else 1), "dk": torch.cat(dk),
           "dv": torch.cat(dv)}
    if not x["broadcast_q"]:
        res["dq"] = torch.cat(dq)
    return res


def _check_sampled(x, got, seqs, heads, what):
    for h in heads:
        y = _slice_heads(_sub_batch(x, seqs), h)
        ref = oracle_fwd_bwd(y)
        g = _gather_outputs(x, got, seqs, h)
        check_o_lse(g["o"], g["lse"], ref["o"], ref["lse"], f"{what} h={h}")
        check_grad(g["dk"], ref["dk"], f"{what} h={h} dK")
        check_grad(g["dv"], ref["dv"], f"{what} h={h} dV")
        if not x["broadcast_q"]:
            check_grad(g["dq"], ref["dq"], f"{what} h={h} dQ")


def test_tiny_full():
    x = jfa_inputs.make("tiny")
    check_all(x, gpu_fwd_bwd(x), oracle_fwd_bwd(x), "tiny")


def test_ads_forward_full():
    x = jfa_inputs.make("ads_fwd")
    got = gpu_fwd_bwd(x, backward=False)
    ref = oracle_fwd_bwd(x, backward=False)
    check_all(x, got, ref, "ads forward", backward=False)


def test_ads_forward_backward_full():
    x = jfa_inputs.make("ads_bwd")
    got = gpu_fwd_bwd(x)
    ref = oracle_fwd_bwd(x)
    check_all(x, got, ref, "ads fwd+bwd")


def test_dense_llm_sampled():
    x = jfa_inputs.make("dense_llm")
    got = gpu_fwd_bwd(x)
    L = (x["offsets"][1:] - x["offsets"][:-1])
    order = torch.argsort(L).tolist()
    # the shortest sequence on every head; the median and the longest on two heads
    _check_sampled(x, got, [order[0]], range(x["H"]), "dense-llm shortest")
    _check_sampled(x, got, [order[len(order) // 2], order[-1]], [0, x["H"] - 1], "dense-llm median+longest")


def test_extreme_sampled():
    x = jfa_inputs.make("extreme")
    got = gpu_fwd_bwd(x)
    # broadcast dQ sums over all 2048 sequences: check every head over the whole batch
    for h in range(x["H"]):
        y = _slice_heads(x, h)
        dq_ref, _, _ = oracle.bwd(y["q"], y["k"], y["v"], y["do"], y["offsets"], y["Lq"], True, False, y["scale"],
                                  want_dkv=False)
        check_grad(got["dq"][:, h:h + 1], dq_ref, f"extreme dQ head {h}")
    L = (x["offsets"][1:] - x["offsets"][:-1])
    order = torch.argsort(L).tolist()
    seqs = order[:3] + order[len(order) // 2: len(order) // 2 + 2] + order[-2:]
    _check_sampled(x, got, seqs, [0, 1], "extreme sampled sequences")
