"""The useful-work accounting behind bench.py's TFLOPS and roofline figures
(CPU only): pair counts against brute-force counting of visible (query, key)
pairs, FLOPs from the pair counts, algorithmic bytes against the sizes of
the tensors each kernel must read and write, and the block-sparse accounting
against the dense one where the mask selects everything or nothing."""
import pytest
import torch

import bench
import jfa_inputs


def _brute_pairs(lengths, Lq, broadcast_q, causal):
    n = 0
    for L in lengths:
        rows = Lq if broadcast_q else L
        for i in range(rows):
            for j in range(L):
                n += 0 if (causal and j > i) else 1
    return n


CASES = [([3, 0, 130, 1], 5, True, False), ([7, 129, 0, 2], 0, False, True), ([40, 1, 300], 0, False, False)]


@pytest.mark.parametrize("lengths,Lq,bq,causal", CASES)
def test_pairs_and_flops(lengths, Lq, bq, causal):
    x = jfa_inputs.custom(len(lengths), Lq, 2, 64, lengths, bq, causal, seed=1)
    acc = bench.accounting(x)
    pairs = _brute_pairs(lengths, Lq, bq, causal)
    assert acc["pairs"] == pairs
    assert acc["flops_fwd"] == 4.0 * 64 * 2 * pairs          # two products of 2*D flops per pair and head
    assert acc["flops_bwd"] == 2.5 * acc["flops_fwd"]         # five products, counting the S recompute


@pytest.mark.parametrize("lengths,Lq,bq,causal", CASES)
def test_bytes_are_the_tensors_moved(lengths, Lq, bq, causal):
    x = jfa_inputs.custom(len(lengths), Lq, 2, 64, lengths, bq, causal, seed=1)
    acc = bench.accounting(x)
    nbytes = lambda t: t.numel() * t.element_size()
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o_bytes = nbytes(do)                                      # O has dO's shape and dtype
    stat = (len(lengths) * 2 * Lq if bq else 2 * x["N"]) * 4  # LSE / Delta, fp32
    assert acc["bytes_fwd"] == nbytes(q) + nbytes(k) + nbytes(v) + o_bytes + stat
    assert acc["bytes_pre"] == 2 * o_bytes + stat
    dq_bytes = 2 * nbytes(q)                                  # fp32 dQ
    assert acc["bytes_bwd"] == (nbytes(q) + nbytes(k) + nbytes(v) + nbytes(do) + 2 * stat
                                + nbytes(k) + nbytes(v) + dq_bytes)


def test_sparse_accounting_matches_dense_at_the_extremes():
    x = jfa_inputs.custom(4, 64, 2, 64, [300, 0, 129, 40], True, False, seed=2)
    nb = jfa_inputs.num_kv_blocks(x["offsets"])
    dense = bench.accounting(x)
    full = bench.accounting_sparse(x, torch.ones(nb, 2, dtype=torch.uint8))
    for key in ("pairs", "flops_fwd", "flops_bwd", "bytes_fwd", "bytes_bwd"):
        assert full[key] == pytest.approx(dense[key])
    assert full["bytes_zero"] == 0 and full["selected_fraction"] == 1.0
    none = bench.accounting_sparse(x, torch.zeros(nb, 2, dtype=torch.uint8))
    assert none["flops_fwd"] == 0 and none["selected_fraction"] == 0.0
    assert none["bytes_zero"] == 2 * 2 * x["N"] * 2 * 64      # every dK and dV row written as zeros


def test_make_inputs_lengths_override():
    """bench.py --lengths SPEC: the workload's shapes with the given KV
    lengths ("N" or "NxR" entries), for the fwd+bwd step and the MXFP8
    forward alike."""
    import argparse
    args = argparse.Namespace(workload="extreme", lengths="300,5x3,0,129")
    x = bench.make_inputs(args)
    w = jfa_inputs.WORKLOADS["extreme"]
    assert x["B"] == 6 and x["offsets"].tolist() == [0, 300, 305, 310, 315, 315, 444]
    assert (x["Lq"], x["H"], x["D"]) == (w.Lq, w.H, w.D) and x["broadcast_q"] == w.broadcast_q
    assert "do" in x and x["workload"].endswith("300,5x3,0,129")
    fwd_only = bench.make_inputs(args, backward=False)
    assert "do" not in fwd_only and fwd_only["offsets"].tolist() == x["offsets"].tolist()
    plain = bench.make_inputs(argparse.Namespace(workload="tiny", lengths=None))
    assert plain["B"] == jfa_inputs.WORKLOADS["tiny"].B
