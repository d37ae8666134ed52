"""Shared helpers of the GPU parity tests: run the CUDA path through the
C ABI (via the thin binding) and compare with the fp64 oracle."""
import math

import torch

import oracle

# Tolerances (stated with the forward/backward contract):
#   O and LSE: max-abs <= 2e-2 and relative L2 <= 1e-2
#   dQ, dK, dV: relative L2 <= 2e-2
O_MAX_ABS, O_REL_L2 = 2e-2, 1e-2
G_REL_L2 = 2e-2


def rel_l2(a, ref):
    a, ref = a.to(torch.float64), ref.to(torch.float64)
    den = ref.norm().item()
    num = (a - ref).norm().item()
    return num / den if den > 0 else num


def check_o_lse(o, lse, o_ref, lse_ref, what=""):
    o, lse = o.cpu().to(torch.float64), lse.cpu().to(torch.float64)
    assert torch.isfinite(o).all(), f"{what}: non-finite O"
    err = (o - o_ref).abs().max().item() if o.numel() else 0.0
    assert err <= O_MAX_ABS, f"{what}: O max-abs {err}"
    if o.numel():
        r = rel_l2(o, o_ref)
        assert r <= O_REL_L2, f"{what}: O rel-L2 {r}"
    inf_ref = torch.isinf(lse_ref)
    assert torch.equal(torch.isinf(lse), inf_ref), f"{what}: LSE -inf pattern differs"
    assert torch.equal(lse[inf_ref], lse_ref[inf_ref])
    fin = ~inf_ref
    if fin.any():
        e = (lse[fin] - lse_ref[fin]).abs().max().item()
        assert e <= O_MAX_ABS, f"{what}: LSE max-abs {e}"
        r = rel_l2(lse[fin], lse_ref[fin])
        assert r <= O_REL_L2, f"{what}: LSE rel-L2 {r}"


def check_grad(g, ref, what):
    g = g.cpu().to(torch.float64)
    assert torch.isfinite(g).all(), f"{what}: non-finite gradient"
    if ref.numel() == 0:
        return
    if ref.norm().item() == 0:
        assert g.abs().max().item() <= 1e-6, f"{what}: expected zeros"
        return
    r = rel_l2(g, ref)
    assert r <= G_REL_L2, f"{what}: rel-L2 {r}"


def to_dev(x, device="cuda"):
    y = dict(x)
    for n in ("q", "k", "v", "do"):
        if n in x:
            y[n] = x[n].to(device)
    y["offsets_dev"] = x["offsets"].to(device)
    return y


def gpu_fwd_bwd(x, backward=True):
    import bwd_jagged_flashattention_gb300 as jfa
    y = to_dev(x)
    B, N = x["B"], x["N"]
    H, D = x["k"].shape[1], x["k"].shape[2]
    Lq = x["Lq"] if x["broadcast_q"] else 0
    ws = jfa.new_workspace(B, N, Lq, H, D, x["broadcast_q"], x["causal"], y["q"].device)
    o, lse = jfa.fwd(y["q"], y["k"], y["v"], y["offsets_dev"], broadcast_q=x["broadcast_q"], causal=x["causal"],
                     scale=x["scale"], offsets_host=x["offsets"], workspace=ws)
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv = jfa.bwd(y["q"], y["k"], y["v"], o, lse, y["do"], y["offsets_dev"], broadcast_q=x["broadcast_q"],
                             causal=x["causal"], scale=x["scale"], offsets_host=x["offsets"], workspace=ws)
        out.update(dq=dq, dk=dk, dv=dv)
    status = jfa.device_status(ws)
    assert status == 0, f"device status {status}"
    return {k_: v_.cpu() for k_, v_ in out.items()}


def oracle_fwd_bwd(x, backward=True, want_dkv=True):
    o, lse = oracle.fwd(x["q"], x["k"], x["v"], x["offsets"], x["Lq"], x["broadcast_q"], x["causal"], x["scale"])
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv = oracle.bwd(x["q"], x["k"], x["v"], x["do"], x["offsets"], x["Lq"], x["broadcast_q"],
                                x["causal"], x["scale"], want_dkv=want_dkv)
        out.update(dq=dq, dk=dk, dv=dv)
    return out


def check_all(x, got, ref, what, backward=True):
    check_o_lse(got["o"], got["lse"], ref["o"], ref["lse"], what)
    if backward:
        check_grad(got["dq"], ref["dq"], what + " dQ")
        if ref.get("dk") is not None:
            check_grad(got["dk"], ref["dk"], what + " dK")
            check_grad(got["dv"], ref["dv"], what + " dV")
