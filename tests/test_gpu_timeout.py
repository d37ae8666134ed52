"""The kernels' failure path, exercised without a GPU fault.

Every barrier wait in the kernels is bounded; when one runs out, the kernel
records JFA_ERR_DEVICE_TIMEOUT in its status word, makes the CTA's other waits
give up, frees its tensor memory and returns.  Here a self-test kernel waits
on a barrier nothing ever completes, under a 1 ms limit (a second wait has a
2 s limit and can only return early through the CTA's abort flag).  The test
checks that the call returns promptly, that the status word reports the
timeout (and is cleared by the read), and that the same device then runs the
attention passes correctly, including with a short wait limit in force.
"""
import time

import pytest
import torch

import jfa_inputs
from tests.gpu_util import check_all, gpu_fwd_bwd, oracle_fwd_bwd

pytestmark = pytest.mark.gpu


def test_wait_timeout_returns_and_reports():
    import bwd_jagged_flashattention_gb300 as jfa
    L = jfa.lib()
    x = jfa_inputs.make("tiny")
    ws = jfa.new_workspace(x["B"], x["N"], x["Lq"], x["H"], x["D"], True, False, torch.device("cuda"))
    assert jfa.device_status(ws) == jfa.JFA_OK
    out = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = L.jfa_selftest_timeout(1_000_000, ws.data_ptr(), out.data_ptr(), stream)
    assert rc == 0
    status = jfa.device_status(ws)  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status == jfa.JFA_ERR_DEVICE_TIMEOUT
    assert out.tolist() == [0, 0], "both waits must have given up"
    assert elapsed < 1.0, f"the second wait should have left on the abort flag, not its 2 s limit ({elapsed:.3f} s)"
    assert jfa.device_status(ws) == jfa.JFA_OK  # the read cleared the word
    # the same device, right after: a normal forward + backward, checked against the oracle
    check_all(x, gpu_fwd_bwd(x), oracle_fwd_bwd(x), "tiny after a timeout")


def test_short_wait_limit_leaves_normal_calls_intact():
    import bwd_jagged_flashattention_gb300 as jfa
    x = jfa_inputs.custom(6, 200, 2, 128, [300, 7, 128, 1, 999, 250], True, False, seed=41)
    jfa.set_wait_limit(10_000_000)  # 10 ms: legitimate waits last microseconds
    try:
        got = gpu_fwd_bwd(x)  # asserts the status word is clear
    finally:
        jfa.set_wait_limit(0)
    check_all(x, got, oracle_fwd_bwd(x), "broadcast with a 10 ms wait limit")
