"""GPU parity of the block-sparse variant (jfa_fwd_block_sparse /
jfa_bwd_block_sparse through the C ABI) against the fp64 oracle's
block-sparse entry points, on seeded inputs.

The variant only adds iteration over selected key blocks (TLX porta
l'attenzione jagged su Blackwell oltre FA4 con un terzo del codice, section
"The turning point"); reading: 128-key blocks per sequence, one selection per
(sequence, head), mask uint8 [NB, H].  Tolerances are the dense contract's
(O/LSE max-abs 2e-2 and rel-L2 1e-2; gradients rel-L2 2e-2); keys of
unselected blocks must get exactly zero dK and dV, and an all-ones mask must
reproduce the dense kernels bit for bit (dQ up to its atomic summation order).
"""
import pytest
import torch

import jfa_inputs
import oracle
from tests.gpu_util import check_grad, check_o_lse, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _gpu(x, mask, backward=True):
    import bwd_jagged_flashattention_gb300 as jfa
    y = to_dev(x)
    H, D = x["k"].shape[1], x["k"].shape[2]
    Lq = x["Lq"] if x["broadcast_q"] else 0
    ws = jfa.new_workspace(x["B"], x["N"], Lq, H, D, x["broadcast_q"], False, y["q"].device)
    o, lse = jfa.fwd_block_sparse(y["q"], y["k"], y["v"], y["offsets_dev"], mask, broadcast_q=x["broadcast_q"],
                                  scale=x["scale"], offsets_host=x["offsets"], workspace=ws)
    out = {"o": o, "lse": lse}
    if backward:
        # dK/dV start as NaN so that a tile the library forgets to write is caught
        dk = torch.full(x["k"].shape, float("nan"), dtype=torch.bfloat16, device=y["q"].device)
        dv = torch.full(x["v"].shape, float("nan"), dtype=torch.bfloat16, device=y["q"].device)
        dq, dk, dv = jfa.bwd_block_sparse(y["q"], y["k"], y["v"], o, lse, y["do"], y["offsets_dev"], mask,
                                          broadcast_q=x["broadcast_q"], scale=x["scale"], offsets_host=x["offsets"],
                                          workspace=ws, dk=dk, dv=dv)
        out.update(dq=dq, dk=dk, dv=dv)
    assert jfa.device_status(ws) == 0
    return {k_: v_.cpu() for k_, v_ in out.items()}


def _oracle(x, mask):
    a = (x["q"], x["k"], x["v"])
    o, lse = oracle.fwd(*a, x["offsets"], x["Lq"], x["broadcast_q"], False, x["scale"], kv_block_mask=mask)
    dq, dk, dv = oracle.bwd(*a, x["do"], x["offsets"], x["Lq"], x["broadcast_q"], False, x["scale"],
                            kv_block_mask=mask)
    return o, lse, dq, dk, dv


def _unselected_rows(offsets, mask, h):
    rows, g = [], 0
    off = offsets.tolist()
    for b in range(len(off) - 1):
        n = (off[b + 1] - off[b] + 127) // 128
        for t in range(n):
            if not mask[g + t, h]:
                rows.extend(range(off[b] + 128 * t, min(off[b + 1], off[b] + 128 * (t + 1))))
        g += n
    return torch.tensor(rows, dtype=torch.int64)


def _check(x, mask, what):
    got = _gpu(x, mask)
    o, lse, dq, dk, dv = _oracle(x, mask)
    check_o_lse(got["o"], got["lse"], o, lse, what)
    check_grad(got["dq"], dq, what + " dQ")
    check_grad(got["dk"], dk, what + " dK")
    check_grad(got["dv"], dv, what + " dV")
    for h in range(x["k"].shape[1]):
        rows = _unselected_rows(x["offsets"], mask, h)
        if rows.numel():
            assert torch.all(got["dk"][rows, h] == 0) and torch.all(got["dv"][rows, h] == 0), what


def _masks(offsets, H, seed):
    nb = jfa_inputs.num_kv_blocks(offsets)
    rand = jfa_inputs.kv_block_mask(offsets, H, 0.5, seed)
    head0_empty = rand.clone()
    head0_empty[:, 0] = 0
    tail = torch.zeros(nb, H, dtype=torch.uint8)
    g = 0
    for L in (offsets[1:] - offsets[:-1]).tolist():
        n = (L + 127) // 128
        if n:
            tail[g + n - 1] = 1
        g += n
    return {"random": rand, "head0_empty": head0_empty, "tail_only": tail,
            "none": torch.zeros(nb, H, dtype=torch.uint8)}


LENGTHS = [300, 0, 129, 700, 1, 128, 257, 64]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lq", [129, 256, 300])
def test_broadcast_block_sparse(D, Lq):
    x = jfa_inputs.custom(len(LENGTHS), Lq, 2, D, LENGTHS, True, False, seed=D + Lq)
    for name, mask in _masks(x["offsets"], 2, seed=Lq).items():
        _check(x, mask, f"broadcast D={D} Lq={Lq} {name}")


@pytest.mark.parametrize("D", [64, 128])
def test_jagged_block_sparse(D):
    x = jfa_inputs.custom(len(LENGTHS), 0, 2, D, LENGTHS, False, False, seed=3 + D)
    for name, mask in _masks(x["offsets"], 2, seed=D).items():
        _check(x, mask, f"jagged D={D} {name}")


def test_all_ones_mask_matches_dense_kernels():
    import bwd_jagged_flashattention_gb300 as jfa
    from tests.gpu_util import gpu_fwd_bwd
    # enough sequences of <= 4 blocks that the dense forward splits nothing (split-KV chunks
    # are merged in fp32, so a split tile's bf16 O may differ in the last bit)
    lengths = [300, 0, 129, 500, 1, 128, 257, 64] * 24
    x = jfa_inputs.custom(len(lengths), 256, 4, 128, lengths, True, False, seed=21)
    assert len(jfa.host_schedule_split(x["offsets"], 256, 4, jfa.num_ctas())[2]) == 0
    ones = torch.ones(jfa.num_kv_blocks(x["offsets"]), 4, dtype=torch.uint8)
    dense = gpu_fwd_bwd(x)
    sparse = _gpu(x, ones)
    for k_ in ("o", "lse", "dk", "dv"):
        assert torch.equal(dense[k_], sparse[k_]), k_
    assert rel_l2(sparse["dq"], dense["dq"].to(torch.float64)) <= 1e-5


def test_ads_like_half_selected():
    """The ads shape at a smaller batch (B=48, Lq=256, H=4, D=128, lognormal
    lengths) with half of the (block, head) pairs selected."""
    lengths = jfa_inputs.draw_lengths("lognormal:256:1.0:8:4096", 48, torch.Generator().manual_seed(5))
    x = jfa_inputs.custom(48, 256, 4, 128, lengths.tolist(), True, False, seed=5)
    mask = jfa_inputs.kv_block_mask(x["offsets"], 4, 0.5, seed=5)
    _check(x, mask, "ads-like 0.5")


def test_mask_shape_is_checked():
    import bwd_jagged_flashattention_gb300 as jfa
    x = jfa_inputs.custom(2, 32, 2, 64, [130, 5], True, False, seed=1)
    with pytest.raises(ValueError):
        _gpu(x, torch.ones(2, 2, dtype=torch.uint8), backward=False)


@pytest.mark.parametrize("policy", ["clc", "queue"])
@pytest.mark.parametrize("bq", [True, False])
def test_block_sparse_backward_dealt_at_run_time(policy, bq):
    """The block-sparse backward with its selected key tiles dealt at run
    time (Cluster Launch Control, or the per-head-group queues), the
    unselected ones zeroed as in the static deal."""
    import bwd_jagged_flashattention_gb300 as jfa
    x = jfa_inputs.custom(len(LENGTHS), 256 if bq else 0, 2, 128, LENGTHS, bq, False, seed=11 + bq)
    jfa.set_schedule_policy(bwd_policy=jfa.SCHED_CLC if policy == "clc" else jfa.SCHED_QUEUE)
    try:
        for name, mask in _masks(x["offsets"], 2, seed=5).items():
            _check(x, mask, f"{policy} broadcast={bq} {name}")
    finally:
        jfa.set_schedule_policy()
