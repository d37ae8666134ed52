"""jfa_fwd_static_scratch: the forward entry point for callers that cannot
allocate memory (an engine plugin that may not call cudaMalloc while it runs,
a program confined to a fixed memory pool).  It keeps its scratch in a
fixed-size array in device memory that the library owns, so the caller
passes only inputs and outputs.

Calls in a row (a large batch, then smaller ones, so each later call runs
over whatever the previous one left in the shared array) must each match the
workspace-based jfa_fwd on the same inputs, and the fp64 oracle, within the
forward tolerance the other tests use; the array's status word must read 0
after them.  One batch holds a broadcast sequence long enough that jfa_fwd
splits its key loop while this entry point (which never splits) walks it
whole.  A batch beyond the array's limit is rejected up front, and so is a
call on a stream that is capturing.

The file is named so pytest collects it last."""
import ctypes

import pytest
import torch

import jfa_inputs
from tests.gpu_util import check_o_lse, oracle_fwd_bwd

pytestmark = pytest.mark.gpu


def _entry():
    import bwd_jagged_flashattention_gb300 as jfa
    f = jfa.lib().jfa_fwd_static_scratch
    vp, ci = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ctypes.c_float, vp, vp, vp]
    f.restype = ci
    st = jfa.lib().jfa_static_scratch_status
    st.argtypes = [vp]
    st.restype = ci
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
             _case(jfa_inputs.custom(4, 0, 2, 128, [300, 1, 129, 700], False, True, seed=32)),
             # one 65,536-key sequence among short ones: jfa_fwd splits it, this entry point does not
             _case(jfa_inputs.custom(16, 128, 1, 128, [65536] + [200] * 15, True, False, seed=33))]
    for x, (q, k, v) in cases:
        st, o, lse = _static_fwd(f, x, q, k, v)
        assert st == jfa.JFA_OK, jfa.status_string(st)
        o_ref, lse_ref = jfa.fwd(q, k, v, x["offsets"].cuda(), broadcast_q=x["broadcast_q"], causal=x["causal"],
                                 scale=x["scale"], offsets_host=x["offsets"])
        torch.cuda.synchronize()
        what = f"static-scratch forward {x['workload']} B={x['B']}"
        check_o_lse(o.cpu(), lse.cpu(), o_ref.cpu().to(torch.float64), lse_ref.cpu().to(torch.float64),
                    what + " vs jfa_fwd")
        if x["B"] <= 16:  # small enough for the fp64 oracle in seconds
            ref = oracle_fwd_bwd(x, backward=False)
            check_o_lse(o.cpu(), lse.cpu(), ref["o"], ref["lse"], what + " vs oracle")
    status = jfa.lib().jfa_static_scratch_status(torch.cuda.current_stream().cuda_stream)
    assert status == jfa.JFA_OK, jfa.status_string(status)


def test_static_scratch_refuses_capturing_stream():
    jfa, f = _entry()
    x, (q, k, v) = _case(jfa_inputs.make("tiny"))
    st0, _, _ = _static_fwd(f, x, q, k, v)  # first call on the device: the address look-up, outside capture
    assert st0 == jfa.JFA_OK
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        graph.capture_begin()
        try:
            st, _, _ = _static_fwd(f, x, q, k, v)
        finally:
            graph.capture_end()
    assert st == jfa.JFA_ERR_UNSUPPORTED


def test_static_scratch_rejects_oversized_batch():
    jfa, f = _entry()
    # 65,536 sequences x 1 head x one q-tile pair each exceeds the 65,264-item scratch.
    B = 65536
    off = torch.arange(B + 1, dtype=torch.int32)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = f(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), off.data_ptr(), B, 1, 1, 64, 1, 0, 0.125,
           dummy.data_ptr(), dummy.data_ptr(), None)
    assert st == jfa.JFA_ERR_WORKSPACE
