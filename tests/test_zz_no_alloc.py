"""jfa_fwd_static_scratch: the forward entry point for callers that cannot
allocate memory (an engine plugin that may not call cudaMalloc while it runs,
a program confined to a fixed memory pool).  It keeps its scratch in a
fixed-size array in device memory that the library owns, so the caller
passes only inputs and outputs.

Two calls in a row (a large batch, then a small one, so the second call runs
over whatever the first left in the shared array) must each match the
workspace-based jfa_fwd on the same inputs, within the forward tolerance the
other tests use.  A batch beyond the array's limit is rejected up front.

The file is named so pytest collects it last."""
import ctypes

import pytest
import torch

import jfa_inputs
from tests.gpu_util import check_o_lse

pytestmark = pytest.mark.gpu


def _entry():
    import bwd_jagged_flashattention_gb300 as jfa
    f = jfa.lib().jfa_fwd_static_scratch
    vp, ci = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ctypes.c_float, vp, vp, vp]
    f.restype = ci
    return jfa, f


def _static_fwd(f, x, q, k, v):
    B, H, D = x["B"], x["H"], x["D"]
    Lq = x["Lq"] if x["broadcast_q"] else 0
    N = x["N"]
    o = torch.full((B, Lq, H, D) if x["broadcast_q"] else (N, H, D), float("nan"), dtype=torch.bfloat16,
                   device="cuda")
    lse = torch.full((B, H, Lq) if x["broadcast_q"] else (H, N), float("nan"), dtype=torch.float32, device="cuda")
    off = x["offsets"].to(torch.int32).contiguous()
    st = f(q.data_ptr(), k.data_ptr() if k.numel() else None, v.data_ptr() if v.numel() else None, off.data_ptr(),
           B, Lq, H, D, int(x["broadcast_q"]), int(x["causal"]), x["scale"], o.data_ptr(), lse.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    return st, o, lse


def _case(x):
    return x, tuple(x[n].cuda() for n in ("q", "k", "v"))


def test_static_scratch_matches_workspace_forward():
    jfa, f = _entry()
    g = torch.Generator().manual_seed(31)
    lengths = jfa_inputs.draw_lengths("lognormal:256:1.0:8:4096", 96, g).tolist()
    cases = [_case(jfa_inputs.custom(96, 256, 4, 128, lengths, True, False, seed=31)),
             _case(jfa_inputs.make("tiny")),
             _case(jfa_inputs.custom(4, 0, 2, 128, [300, 1, 129, 700], False, True, seed=32))]
    for x, (q, k, v) in cases:
        st, o, lse = _static_fwd(f, x, q, k, v)
        assert st == jfa.JFA_OK, jfa.status_string(st)
        o_ref, lse_ref = jfa.fwd(q, k, v, x["offsets"].cuda(), broadcast_q=x["broadcast_q"], causal=x["causal"],
                                 scale=x["scale"], offsets_host=x["offsets"])
        torch.cuda.synchronize()
        check_o_lse(o.cpu(), lse.cpu(), o_ref.cpu().to(torch.float64), lse_ref.cpu().to(torch.float64),
                    f"static-scratch forward {x['workload']} B={x['B']}")


def test_static_scratch_rejects_oversized_batch():
    jfa, f = _entry()
    # 65,536 sequences x 1 head x one q-tile pair each exceeds the 65,264-item scratch.
    B = 65536
    off = torch.arange(B + 1, dtype=torch.int32)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = f(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), off.data_ptr(), B, 1, 1, 64, 1, 0, 0.125,
           dummy.data_ptr(), dummy.data_ptr(), None)
    assert st == jfa.JFA_ERR_WORKSPACE
