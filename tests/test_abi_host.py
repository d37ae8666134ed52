"""The C-ABI library builds, loads and exports every symbol include/*.h
declares, and rejects invalid arguments on the host before any GPU work.
No call here launches a kernel or needs a GPU."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def jfa():
    import bwd_jagged_flashattention_gb300 as jfa
    jfa.build()
    return jfa


def _declared_functions():
    names = set()
    for h in ("jfa.h", "jfa_selftest.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(jfa_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(jfa):
    declared = _declared_functions()
    assert declared, "no declarations parsed"
    lib = jfa.lib()
    for name in declared:
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert declared <= set(jfa.EXPORTED) | {"jfa_host_build_schedule"}


def test_status_strings(jfa):
    for code, name in enumerate(["JFA_OK", "JFA_ERR_INVALID_ARG", "JFA_ERR_UNSUPPORTED", "JFA_ERR_WORKSPACE",
                                 "JFA_ERR_CUDA", "JFA_ERR_DEVICE_TIMEOUT"]):
        assert jfa.status_string(code) == name


def test_workspace_bytes(jfa):
    lib = jfa.lib()
    a = lib.jfa_workspace_bytes(512, 190000, 256, 4, 128, 1, 0)
    assert a > 0 and a % 256 == 0
    # Delta [B,H,Lq] fp32 is part of it
    assert a >= 512 * 4 * 256 * 4
    assert lib.jfa_workspace_bytes(4, 100, 32, 2, 96, 1, 0) == 0          # unsupported D
    assert lib.jfa_workspace_bytes(-1, 100, 32, 2, 64, 1, 0) == 0
    j = lib.jfa_workspace_bytes(32, 139000, 0, 16, 128, 0, 1)
    assert j >= 16 * 139000 * 4
    # The boundary's form: (B, total_len, Lq, H, D, broadcast_q, causal), no is_bwd
    # flag (one workspace serves both passes).  total_len sizes the jagged
    # Delta [H, N]: 1000 more rows need at least 1000 * H * 4 more bytes.
    assert len(lib.jfa_workspace_bytes.argtypes) == 7
    j2 = lib.jfa_workspace_bytes(32, 140000, 0, 16, 128, 0, 1)
    assert j2 - j >= 1000 * 16 * 4
    # Broadcast Delta [B, H, Lq]: doubling Lq adds at least B * H * Lq * 4 bytes.
    a2 = lib.jfa_workspace_bytes(512, 190000, 512, 4, 128, 1, 0)
    assert a2 - a >= 512 * 4 * 256 * 4


# Fake, never-dereferenced device addresses: validation must reject these
# calls before touching them.
P16 = 1 << 20
WS = 1 << 24


def _fwd(lib, offsets, B=2, Lq=32, H=2, D=64, bq=1, causal=0, scale=0.125, q=P16, o=P16, lse=P16, ws=WS,
         ws_bytes=1 << 30):
    off = torch.tensor(offsets, dtype=torch.int32)
    return lib.jfa_fwd(ctypes.c_void_p(q), ctypes.c_void_p(P16), ctypes.c_void_p(P16), None,
                       ctypes.c_void_p(off.data_ptr()), B, Lq, H, D, bq, causal, scale, ctypes.c_void_p(o),
                       ctypes.c_void_p(lse), ctypes.c_void_p(ws), ws_bytes, None)


def test_fwd_argument_errors(jfa):
    lib = jfa.lib()
    ok_off = [0, 3, 7]
    assert _fwd(lib, ok_off, D=96) == jfa.JFA_ERR_UNSUPPORTED
    assert _fwd(lib, ok_off, H=256) == jfa.JFA_ERR_UNSUPPORTED
    assert _fwd(lib, ok_off, causal=1) == jfa.JFA_ERR_UNSUPPORTED      # causal with broadcast Q
    assert _fwd(lib, [1, 3, 7]) == jfa.JFA_ERR_INVALID_ARG            # offsets[0] != 0
    assert _fwd(lib, [0, 5, 4]) == jfa.JFA_ERR_INVALID_ARG            # decreasing offsets
    assert _fwd(lib, ok_off, B=-1) == jfa.JFA_ERR_INVALID_ARG
    assert _fwd(lib, ok_off, scale=float("nan")) == jfa.JFA_ERR_INVALID_ARG
    assert _fwd(lib, ok_off, ws_bytes=16) == jfa.JFA_ERR_WORKSPACE
    assert _fwd(lib, ok_off, ws=WS + 8) == jfa.JFA_ERR_WORKSPACE        # misaligned workspace
    assert _fwd(lib, ok_off, q=P16 + 2) == jfa.JFA_ERR_UNSUPPORTED      # TMA needs 16-byte alignment
    assert _fwd(lib, ok_off, q=0) == jfa.JFA_ERR_INVALID_ARG            # null input
    assert _fwd(lib, [0, 1 << 24, 1 << 24]) == jfa.JFA_ERR_UNSUPPORTED  # sequence longer than 2^23
    # neither offsets copy given
    assert lib.jfa_fwd(None, None, None, None, None, 2, 32, 2, 64, 1, 0, 0.1, None, None, None, 0,
                       None) == jfa.JFA_ERR_INVALID_ARG


def test_bwd_argument_errors(jfa):
    lib = jfa.lib()
    off = torch.tensor([0, 3, 7], dtype=torch.int32)
    p = ctypes.c_void_p(P16)

    def call(D=64, bq=1, causal=0, dq=P16, ws_bytes=1 << 30):
        return lib.jfa_bwd(p, p, p, p, p, p, None, ctypes.c_void_p(off.data_ptr()), 2, 32, 2, D, bq, causal, 0.1,
                           ctypes.c_void_p(dq), p, p, ctypes.c_void_p(WS), ws_bytes, None)
    assert call(D=32) == jfa.JFA_ERR_UNSUPPORTED
    assert call(causal=1) == jfa.JFA_ERR_UNSUPPORTED
    assert call(dq=P16 + 4) == jfa.JFA_ERR_UNSUPPORTED
    assert call(ws_bytes=100) == jfa.JFA_ERR_WORKSPACE
    assert call(dq=0) == jfa.JFA_ERR_INVALID_ARG


def test_device_status_rejects_null(jfa):
    assert jfa.lib().jfa_device_status(None, None) == jfa.JFA_ERR_INVALID_ARG


def test_product_path_has_no_cpu_fallback():
    """The package never imports the oracle and raises when its library is missing."""
    pkg = os.path.join(ROOT, "bwd_jagged_flashattention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "jfa_oracle" not in text, f
    src = open(os.path.join(pkg, "__init__.py")).read()
    assert "raise ImportError" in src


def test_block_sparse_argument_errors(jfa):
    """The block-sparse entries check their mask and share the dense checks (no GPU needed)."""
    lib = jfa.lib()
    off = torch.tensor([0, 3, 300], dtype=torch.int32)
    mask = torch.ones(jfa.num_kv_blocks(off), 2, dtype=torch.uint8)
    p = ctypes.c_void_p(P16)
    mp = ctypes.c_void_p(mask.data_ptr())

    def fwd(m=mp, D=64, ws_bytes=1 << 30):
        return lib.jfa_fwd_block_sparse(p, p, p, None, ctypes.c_void_p(off.data_ptr()), m, 2, 32, 2, D, 1, 0.1, p, p,
                                        ctypes.c_void_p(WS), ws_bytes, None)

    def bwd(m=mp, D=64):
        return lib.jfa_bwd_block_sparse(p, p, p, p, p, p, None, ctypes.c_void_p(off.data_ptr()), m, 2, 32, 2, D, 1,
                                        0.1, p, p, p, ctypes.c_void_p(WS), 1 << 30, None)
    assert fwd(m=None) == jfa.JFA_ERR_INVALID_ARG
    assert bwd(m=None) == jfa.JFA_ERR_INVALID_ARG
    assert fwd(D=96) == jfa.JFA_ERR_UNSUPPORTED
    assert bwd(D=96) == jfa.JFA_ERR_UNSUPPORTED
    assert fwd(ws_bytes=64) == jfa.JFA_ERR_WORKSPACE


def test_num_kv_blocks(jfa):
    off = torch.tensor([0, 0, 1, 128, 257, 1000], dtype=torch.int32)
    assert jfa.num_kv_blocks(off) == 0 + 1 + 1 + 2 + 6
    assert jfa.lib().jfa_num_kv_blocks(None, 3) == -1


def test_mxfp8_argument_errors(jfa):
    """The MXFP8 entries check their scale pointer, alignment and workspace before any launch (no GPU needed)."""
    lib = jfa.lib()
    off = torch.tensor([0, 3, 300], dtype=torch.int32)
    p = ctypes.c_void_p(P16)
    offp = ctypes.c_void_p(off.data_ptr())

    def fwd(vs=p, D=64, ws_bytes=1 << 30, causal=0):
        return lib.jfa_fwd_mxfp8(p, p, p, vs, None, offp, 2, 32, 2, D, 1, causal, 0.1, p, p, ctypes.c_void_p(WS),
                                 ws_bytes, None)

    def quant(v=p, D=64, dev=p, ws_bytes=1 << 20, vs=p):
        return lib.jfa_quantize_v_mxfp8(v, dev, offp, 2, 2, D, p, vs, ctypes.c_void_p(WS), ws_bytes, None)
    assert fwd(vs=None) == jfa.JFA_ERR_INVALID_ARG
    assert fwd(vs=ctypes.c_void_p(P16 + 4)) == jfa.JFA_ERR_UNSUPPORTED  # scales must be 16-byte aligned
    assert fwd(D=96) == jfa.JFA_ERR_UNSUPPORTED
    assert fwd(causal=1) == jfa.JFA_ERR_UNSUPPORTED                      # causal with broadcast Q
    assert fwd(ws_bytes=64) == jfa.JFA_ERR_WORKSPACE
    assert quant(D=96) == jfa.JFA_ERR_UNSUPPORTED
    assert quant(dev=None) == jfa.JFA_ERR_INVALID_ARG                    # the kernel reads device offsets
    assert quant(v=None) == jfa.JFA_ERR_INVALID_ARG
    assert quant(vs=ctypes.c_void_p(P16 + 8)) == jfa.JFA_ERR_UNSUPPORTED
    assert quant(ws_bytes=256) == jfa.JFA_ERR_WORKSPACE                  # needs 256 + 4 (B + 1) bytes


def test_schedule_policy_values(jfa):
    """Deal policies: 0 zigzag, 1 round-robin, 2 greedy for either pass; 3 (Cluster
    Launch Control) and 4 (per-head-group queues) for the backward only;
    anything else is rejected."""
    lib = jfa.lib()
    try:
        for f in (0, 1, 2):
            for b in (0, 1, 2, 3, 4):
                assert lib.jfa_set_schedule_policy(f, b) == jfa.JFA_OK
        assert lib.jfa_set_schedule_policy(3, 0) == jfa.JFA_ERR_INVALID_ARG
        assert lib.jfa_set_schedule_policy(4, 0) == jfa.JFA_ERR_INVALID_ARG
        assert lib.jfa_set_schedule_policy(0, 5) == jfa.JFA_ERR_INVALID_ARG
        assert lib.jfa_set_schedule_policy(-1, 0) == jfa.JFA_ERR_INVALID_ARG
    finally:
        jfa.set_schedule_policy()


def test_wait_limit_setter(jfa):
    lib = jfa.lib()
    assert lib.jfa_set_wait_limit(1_000_000) == jfa.JFA_OK
    assert lib.jfa_set_wait_limit(0) == jfa.JFA_OK  # back to the 4 s default
