"""GPU parity of the MXFP8 forward (P V as block-scaled E4M3 on the tensor
cores, P quantized on the fly) and of the V quantizer, through the C ABI,
against the fp64 oracle.

- quantize_v_mxfp8: codes and scales bit-exact (exact fp32 arithmetic on bf16
  inputs decides every byte on both sides).
- fwd_mxfp8: O within max-abs 2e-2 plus the oracle's per-element slack (a
  quantization decision within 1e-4 of a boundary may fall either way in the
  kernel's fp32 logits; the slack is that choice's effect on O), relative L2
  <= 1e-2; LSE, which does not depend on the quantization, with the bf16
  forward's max-abs 2e-2 and relative L2 1e-2.  Each side runs on its own
  quantized V, after the two were found equal.
"""
import pytest
import torch

import jfa_inputs
import oracle
from tests.gpu_util import rel_l2, to_dev

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_L2 = 2e-2, 1e-2


def _gpu_quant(x):
    import bwd_jagged_flashattention_gb300 as jfa
    v8, vs = jfa.quantize_v_mxfp8(x["v"].cuda(), x["offsets"].cuda(), offsets_host=x["offsets"])
    torch.cuda.synchronize()
    return v8, vs


def _gpu_fwd(x, v8, vs):
    import bwd_jagged_flashattention_gb300 as jfa
    y = to_dev(x)
    H, D = x["k"].shape[1], x["k"].shape[2]
    Lq = x["Lq"] if x["broadcast_q"] else 0
    ws = jfa.new_workspace(x["B"], x["N"], Lq, H, D, x["broadcast_q"], x["causal"], y["q"].device)
    o, lse = jfa.fwd_mxfp8(y["q"], y["k"], v8, vs, y["offsets_dev"], broadcast_q=x["broadcast_q"],
                           causal=x["causal"], scale=x["scale"], offsets_host=x["offsets"], workspace=ws)
    assert jfa.device_status(ws) == 0
    return o.cpu(), lse.cpu()


def check_mx(o, lse, o_ref, lse_ref, slack, what, mass=None):
    """mass (optional): sum_j |pq_j v_j| / l per element, for inputs far from unit scale, where the bound
    becomes the bf16 rounding of O (2^-9 |O|, doubled) plus fp32 accumulation (1e-4 of the mass)."""
    o, lse = o.to(torch.float64), lse.to(torch.float64)
    assert torch.isfinite(o).all(), f"{what}: non-finite O"
    if o.numel():
        bound = O_MAX_ABS if mass is None else 2.0 ** -8 * o_ref.abs() + 1e-4 * mass
        excess = ((o - o_ref).abs() - slack - bound).max().item()
        assert excess <= 0, f"{what}: O error beyond bound and slack by {excess}"
        r = rel_l2(o, o_ref)
        assert r <= O_REL_L2, f"{what}: O rel-L2 {r}"
    inf_ref = torch.isinf(lse_ref)
    assert torch.equal(torch.isinf(lse), inf_ref), f"{what}: LSE -inf pattern differs"
    fin = ~inf_ref
    if fin.any():
        e = (lse[fin] - lse_ref[fin]).abs().max().item()
        assert e <= O_MAX_ABS, f"{what}: LSE max-abs {e}"
        assert rel_l2(lse[fin], lse_ref[fin]) <= O_REL_L2


def run_case(x, what, scaled=False):
    v8, vs = _gpu_quant(x)
    r8, rs = oracle.quantize_v_mxfp8(x["v"], x["offsets"])
    assert torch.equal(v8.cpu(), r8), f"{what}: E4M3 codes differ at {(v8.cpu() != r8).sum().item()} places"
    assert torch.equal(vs.cpu(), rs), f"{what}: E8M0 scales differ at {(vs.cpu() != rs).sum().item()} places"
    o, lse = _gpu_fwd(x, v8, vs)
    orc = oracle._default()
    args = (x["offsets"], x["Lq"], x["broadcast_q"], x["causal"], x["scale"])
    o_ref, lse_ref, slack = orc.fwd_mxfp8(x["q"], x["k"], r8, rs, *args, want_slack=True)
    mass = orc.fwd_mxfp8(x["q"], x["k"], r8 & 0x7F, rs, *args)[0] if scaled else None  # |V| codes
    check_mx(o, lse, o_ref, lse_ref, slack, what, mass)
    return o_ref, slack


CASES = {
    "broadcast_d128_tails": (8, 256, 2, 128, [300, 5, 128, 129, 0, 1000, 64, 2000], True, False),
    "broadcast_d64_ragged_q": (5, 300, 3, 64, [1, 200, 513, 0, 77], True, False),
    "jagged_causal_d128": (5, 0, 2, 128, [1, 130, 300, 0, 257], False, True),
    "jagged_d64": (3, 0, 2, 64, [50, 1000, 3], False, False),
    "jagged_causal_d64_long": (2, 0, 1, 64, [1500, 40], False, True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_mxfp8_parity(name):
    B, Lq, H, D, lengths, bq, causal = CASES[name]
    x = jfa_inputs.custom(B, Lq, H, D, lengths, bq, causal, seed=B + Lq + D, backward=False)
    run_case(x, name)


def test_mxfp8_wide_logits_rescale():
    """Large logits (scaled Q): the running max jumps by more than 2^8 between blocks, so O is rescaled
    in TMEM, and many chunks sit far below the row maximum (small shared exponents)."""
    x = jfa_inputs.custom(4, 256, 2, 128, [700, 129, 1, 520], True, False, seed=3, backward=False)
    ramp = torch.linspace(0.2, 3.0, x["N"]).to(torch.bfloat16)[:, None, None]
    x["k"] = (x["k"].to(torch.float32) * ramp).to(torch.bfloat16)
    x["q"] = (x["q"].to(torch.float32) * 3.0).to(torch.bfloat16)
    run_case(x, "wide logits")


def test_mxfp8_v_dynamic_range():
    """V whose magnitudes vary by 2^+-40 from row to row, with zero and tiny (subnormal bf16) rows:
    every chunk gets its own scale; all-zero chunks get code 0."""
    x = jfa_inputs.custom(3, 128, 2, 128, [257, 64, 130], True, False, seed=4, backward=False)
    g = torch.Generator().manual_seed(9)
    ex = torch.randint(-40, 41, (x["N"], 1, 1), generator=g).to(torch.float32)
    v = x["v"].to(torch.float32) * torch.exp2(ex)
    v[10:50] = 0.0
    v[60:62] = 1e-39
    v[63] = -0.0
    x["v"] = v.to(torch.bfloat16)
    run_case(x, "V dynamic range", scaled=True)


def test_mxfp8_close_to_bf16_forward():
    """The MXFP8 forward's O stays close to the bf16 forward's (E4M3 P and V: about 2^-4 relative per
    weight, averaged over the keys): relative L2 below 5e-2 on an ads-like batch."""
    import bwd_jagged_flashattention_gb300 as jfa
    x = jfa_inputs.custom(16, 256, 2, 128, [384, 1000, 50, 129] * 4, True, False, seed=5, backward=False)
    v8, vs = _gpu_quant(x)
    o_mx, _ = _gpu_fwd(x, v8, vs)
    y = to_dev(x)
    o_bf, _ = jfa.fwd(y["q"], y["k"], y["v"], y["offsets_dev"], broadcast_q=True, scale=x["scale"],
                      offsets_host=x["offsets"])
    assert rel_l2(o_mx.to(torch.float64), o_bf.cpu().to(torch.float64)) < 5e-2


def test_mxfp8_ads_full_size_sampled():
    """The ads workload at full size, in the bench's launch configuration: the whole batch is quantized and
    run on the GPU; whole sequences (all heads) are checked against the oracle run on those sequences only,
    and the quantized V of those sequences bit-exactly."""
    x = jfa_inputs.make("ads_bwd", backward=False)
    v8, vs = _gpu_quant(x)
    o, lse = _gpu_fwd(x, v8, vs)
    off = x["offsets"].tolist()
    lens = [off[b + 1] - off[b] for b in range(x["B"])]
    order = sorted(range(x["B"]), key=lambda b: lens[b])
    seqs = sorted({order[0], order[len(order) // 2], order[-1], 7, 300})
    blk = [0]
    for L in lens:
        blk.append(blk[-1] + (L + 127) // 128)
    sub_len = [lens[b] for b in seqs]
    sub = dict(x, B=len(seqs), offsets=jfa_inputs.offsets_from_lengths(torch.tensor(sub_len)),
               k=torch.cat([x["k"][off[b]:off[b + 1]] for b in seqs]),
               v=torch.cat([x["v"][off[b]:off[b + 1]] for b in seqs]))
    sub["N"] = int(sub["offsets"][-1])
    r8, rs = oracle.quantize_v_mxfp8(sub["v"], sub["offsets"])
    g8 = torch.cat([v8[off[b]:off[b + 1]].cpu() for b in seqs])
    gs = torch.cat([vs[blk[b]:blk[b + 1]].cpu() for b in seqs])
    assert torch.equal(g8, r8) and torch.equal(gs, rs)
    o_ref, lse_ref, slack = oracle._default().fwd_mxfp8(sub["q"], sub["k"], r8, rs, sub["offsets"], x["Lq"], True,
                                                        False, x["scale"], want_slack=True)
    check_mx(o[seqs], lse[seqs], o_ref, lse_ref, slack, "ads full size, sampled sequences")


def test_mxfp8_empty_batch_and_sequences():
    import bwd_jagged_flashattention_gb300 as jfa
    x = jfa_inputs.custom(3, 128, 2, 64, [0, 0, 0], True, False, seed=1, backward=False)
    y = to_dev(x)
    v8 = torch.zeros((0, 2, 64), dtype=torch.uint8, device="cuda")
    vs = torch.zeros((0, 2, 64, 4), dtype=torch.uint8, device="cuda")
    o, lse = jfa.fwd_mxfp8(y["q"], y["k"], v8, vs, y["offsets_dev"], broadcast_q=True, scale=x["scale"],
                           offsets_host=x["offsets"])
    assert torch.all(o.cpu() == 0) and torch.all(torch.isinf(lse.cpu()))


def test_mxfp8_dense_llm_sampled():
    """The dense-LLM workload (jagged causal self-attention, 32 sequences of 512..8192 keys, H=16, D=128) at full
    size: the whole batch is quantized and run on the GPU; the shortest sequence is checked on every head and
    the longest on one head against the oracle run on just those rows, with their quantized V bit-exact."""
    x = jfa_inputs.make("dense_llm", backward=False)
    v8, vs = _gpu_quant(x)
    o, lse = _gpu_fwd(x, v8, vs)
    v8, vs = v8.cpu(), vs.cpu()
    off = x["offsets"].tolist()
    lens = [off[b + 1] - off[b] for b in range(x["B"])]
    blk = [0]
    for L in lens:
        blk.append(blk[-1] + (L + 127) // 128)
    order = sorted(range(x["B"]), key=lambda b: lens[b])
    for b, h0, h1 in ((order[0], 0, x["H"]), (order[-1], 0, 1)):
        rows = slice(off[b], off[b + 1])
        sub = dict(x, B=1, N=lens[b], offsets=torch.tensor([0, lens[b]], dtype=torch.int32),
                   q=x["q"][rows, h0:h1].contiguous(), k=x["k"][rows, h0:h1].contiguous(),
                   v=x["v"][rows, h0:h1].contiguous())
        r8, rs = oracle.quantize_v_mxfp8(sub["v"], sub["offsets"])
        assert torch.equal(v8[rows, h0:h1], r8) and torch.equal(vs[blk[b]:blk[b + 1], h0:h1], rs)
        o_ref, lse_ref, slack = oracle._default().fwd_mxfp8(sub["q"], sub["k"], r8, rs, sub["offsets"], 0, False,
                                                            True, x["scale"], want_slack=True)
        check_mx(o[rows, h0:h1], lse[h0:h1, rows], o_ref, lse_ref, slack, f"dense-LLM sequence {b} heads {h0}:{h1}")


@pytest.mark.parametrize("D,Lq", [(128, 256), (64, 300), (128, 128)])
def test_mxfp8_split_kv(D, Lq):
    """Split-KV in the MXFP8 forward: a skewed broadcast batch whose long
    sequence's query tiles the host cuts into key chunks; each chunk finds
    its V scales through its slot's first key block, writes fp32 partials,
    and the merge pass combines them.  Checked against the oracle's MXFP8
    forward like the unsplit cases (a chunk quantizes P exactly as the
    whole tile would: the shared exponents do not depend on the running
    max)."""
    import bwd_jagged_flashattention_gb300 as jfa
    lengths = [20000, 5, 300, 0, 129, 1000, 1]
    x = jfa_inputs.custom(len(lengths), Lq, 2, D, lengths, True, False, seed=D + Lq + 7, backward=False)
    _, _, groups, slots = jfa.host_schedule_split(x["offsets"], x["Lq"], x["H"], jfa.num_ctas())
    assert len(groups) > 0, "the batch must exercise split-KV"
    run_case(x, f"MXFP8 split-KV D={D} Lq={Lq} ({len(groups)} tiles, {slots} chunks)")
