"""Jagged Flash Attention for GB300 (sm_103a): thin Python binding over libjfa.so.

Every step of the computation runs in the library's CUDA kernels; this module
only marshals torch tensors (device memory and the current stream) into the
C ABI declared in ``include/jfa.h``.  There is no CPU fallback: if the
library is missing or a call fails, an exception is raised.

The operation is FlashAttention applied directly to packed, unpadded Q/K/V
with an int32 offsets tensor ("Why attention in GEM needed a rewrite", Meta's
TLX Jagged Flash Attention Beats FA4 on Blackwell With 3x Less Code), with an
optional broadcast Q whose gradient is summed over the batch (Meta's 3.2K-line
Triton kernel outruns FlashAttention-4 on jagged Blackwell attention, second
paragraph).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libjfa.so")

JFA_OK, JFA_ERR_INVALID_ARG, JFA_ERR_UNSUPPORTED, JFA_ERR_WORKSPACE, JFA_ERR_CUDA, JFA_ERR_DEVICE_TIMEOUT = range(6)

# Every symbol include/jfa.h and include/jfa_selftest.h declare.
EXPORTED = ("jfa_workspace_bytes", "jfa_fwd", "jfa_bwd", "jfa_device_status", "jfa_status_string",
            "jfa_num_ctas", "jfa_profile_enable", "jfa_profile_read", "jfa_selftest_mma", "jfa_fwd_static_scratch",
            "jfa_static_scratch_status", "jfa_set_schedule_policy", "jfa_set_wait_limit", "jfa_selftest_timeout",
            "jfa_fwd_block_sparse", "jfa_bwd_block_sparse", "jfa_num_kv_blocks", "jfa_fwd_mxfp8",
            "jfa_quantize_v_mxfp8")

_lock = threading.Lock()
_lib = None


class JFAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def build(force: bool = False) -> str:
    from . import buildlib as _b
    return _b.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                  "(python bwd_jagged_flashattention_gb300/buildlib.py)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32p, ci, cf, sz = (ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_int,
                                    ctypes.c_float, ctypes.c_size_t)
            L.jfa_workspace_bytes.argtypes = [ci, ci, ci, ci, ci, ci, ci]
            L.jfa_workspace_bytes.restype = sz
            L.jfa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, vp, vp, vp, sz, vp]
            L.jfa_fwd.restype = ci
            L.jfa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, vp, vp, vp, vp, sz, vp]
            L.jfa_bwd.restype = ci
            if hasattr(L, "jfa_fwd_block_sparse"):  # (absent only from builds that predate it)
                L.jfa_fwd_block_sparse.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp, vp, vp, sz,
                                                   vp]
                L.jfa_fwd_block_sparse.restype = ci
                L.jfa_bwd_block_sparse.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp, vp,
                                                   vp, vp, sz, vp]
                L.jfa_bwd_block_sparse.restype = ci
                L.jfa_num_kv_blocks.argtypes = [vp, ci]
                L.jfa_num_kv_blocks.restype = ctypes.c_int64
            if hasattr(L, "jfa_fwd_mxfp8"):  # (absent only from builds that predate it)
                L.jfa_fwd_mxfp8.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, vp, vp, vp, sz, vp]
                L.jfa_fwd_mxfp8.restype = ci
                L.jfa_quantize_v_mxfp8.argtypes = [vp, vp, vp, ci, ci, ci, vp, vp, vp, sz, vp]
                L.jfa_quantize_v_mxfp8.restype = ci
            L.jfa_device_status.argtypes = [vp, vp]
            L.jfa_device_status.restype = ci
            L.jfa_status_string.argtypes = [ci]
            L.jfa_status_string.restype = ctypes.c_char_p
            L.jfa_set_wait_limit.argtypes = [ctypes.c_ulonglong]
            L.jfa_set_wait_limit.restype = ci
            L.jfa_selftest_timeout.argtypes = [ctypes.c_ulonglong, vp, vp, vp]
            L.jfa_selftest_timeout.restype = ci
            L.jfa_set_schedule_policy.argtypes = [ci, ci]
            L.jfa_set_schedule_policy.restype = ci
            L.jfa_num_ctas.argtypes = []
            L.jfa_num_ctas.restype = ci
            L.jfa_profile_enable.argtypes = [ci]
            L.jfa_profile_enable.restype = ci
            L.jfa_profile_read.argtypes = [vp, vp, ci]
            L.jfa_profile_read.restype = ci
            L.jfa_selftest_mma.argtypes = [ci, vp, vp, vp, vp, vp]
            L.jfa_selftest_mma.restype = ci
            L.jfa_host_build_schedule.argtypes = [vp, ci, ci, ci, ci, ci, ci, ci, ci, vp, vp, ctypes.c_longlong]
            ll = ctypes.c_longlong
            if hasattr(L, "jfa_host_build_schedule_split"):
                L.jfa_host_build_schedule_split.argtypes = [vp, ci, ci, ci, ci, vp, vp, ll, vp, ctypes.POINTER(ll), vp]
                L.jfa_host_build_schedule_split.restype = ll
            if hasattr(L, "jfa_host_build_schedule_sparse"):
                L.jfa_host_build_schedule_sparse.argtypes = [vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, ll, vp, vp, vp,
                                                             ll, ctypes.POINTER(ll)]
                L.jfa_host_build_schedule_sparse.restype = ll
            L.jfa_host_build_schedule.restype = ctypes.c_longlong
            if hasattr(L, "jfa_host_build_schedule_noalloc"):  # host-only test entry
                L.jfa_host_build_schedule_noalloc.argtypes = [vp, ci, ci, ci, ci, ci, ci, ci, vp, vp,
                                                              ctypes.c_longlong]
                L.jfa_host_build_schedule_noalloc.restype = ctypes.c_longlong
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().jfa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != JFA_OK:
        raise JFAError(status, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else None


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def workspace_bytes(B: int, total_len: int, Lq: int, H: int, D: int, broadcast_q: bool, causal: bool) -> int:
    n = lib().jfa_workspace_bytes(B, total_len, Lq, H, D, int(broadcast_q), int(causal))
    if n == 0:
        raise JFAError(JFA_ERR_UNSUPPORTED, "jfa_workspace_bytes")
    return int(n)


def new_workspace(B: int, total_len: int, Lq: int, H: int, D: int, broadcast_q: bool, causal: bool,
                  device) -> torch.Tensor:
    """A workspace for these sizes; the status word at its start is zeroed."""
    ws = torch.empty(workspace_bytes(B, total_len, Lq, H, D, broadcast_q, causal), dtype=torch.uint8,
                     device=device)
    ws[:256].zero_()
    return ws


def _host_offsets(offsets, offsets_host):
    if offsets_host is None:
        offsets_host = offsets.detach().to("cpu", torch.int32)
    offsets_host = offsets_host.to(torch.int32).contiguous()
    assert offsets_host.device.type == "cpu"
    return offsets_host


def fwd(q, k, v, offsets, Lq: int | None = None, broadcast_q: bool = True, causal: bool = False,
        scale: float | None = None, offsets_host=None, workspace=None, out=None, lse=None):
    """O (bf16) and LSE (fp32).  q [Lq,H,D] (broadcast) or [N,H,D]; k, v [N,H,D]."""
    assert q.is_cuda and q.dtype == torch.bfloat16 and k.dtype == torch.bfloat16 and v.dtype == torch.bfloat16
    H, D = k.shape[1], k.shape[2]
    offsets_host = _host_offsets(offsets, offsets_host)
    B = offsets_host.numel() - 1
    N = int(offsets_host[-1]) if B > 0 else 0
    Lq = q.shape[0] if broadcast_q else 0
    o_shape = (B, Lq, H, D) if broadcast_q else (N, H, D)
    lse_shape = (B, H, Lq) if broadcast_q else (H, N)
    out = torch.empty(o_shape, dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device) if lse is None else lse
    if workspace is None:
        workspace = new_workspace(B, N, Lq, H, D, broadcast_q, causal, q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    offsets_dev = offsets if (offsets is not None and offsets.is_cuda) else None
    st = lib().jfa_fwd(_ptr(q.contiguous()), _ptr(k.contiguous()), _ptr(v.contiguous()),
                       _ptr(offsets_dev), ctypes.c_void_p(offsets_host.data_ptr()),
                       B, Lq, H, D, int(broadcast_q), int(causal), sc, _ptr(out), _ptr(lse),
                       _ptr(workspace), workspace.numel(), _stream(q.device))
    _check(st, "jfa_fwd")
    return out, lse


def bwd(q, k, v, o, lse, do, offsets, broadcast_q: bool = True, causal: bool = False,
        scale: float | None = None, offsets_host=None, workspace=None, dq=None, dk=None, dv=None):
    """dQ (fp32, shaped like q), dK and dV (bf16, [N,H,D])."""
    H, D = k.shape[1], k.shape[2]
    offsets_host = _host_offsets(offsets, offsets_host)
    B = offsets_host.numel() - 1
    N = int(offsets_host[-1]) if B > 0 else 0
    Lq = q.shape[0] if broadcast_q else 0
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.bfloat16, device=q.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.bfloat16, device=q.device) if dv is None else dv
    if workspace is None:
        workspace = new_workspace(B, N, Lq, H, D, broadcast_q, causal, q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    offsets_dev = offsets if (offsets is not None and offsets.is_cuda) else None
    st = lib().jfa_bwd(_ptr(q.contiguous()), _ptr(k.contiguous()), _ptr(v.contiguous()), _ptr(o.contiguous()),
                       _ptr(lse.contiguous()), _ptr(do.contiguous()), _ptr(offsets_dev),
                       ctypes.c_void_p(offsets_host.data_ptr()), B, Lq, H, D, int(broadcast_q), int(causal), sc,
                       _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), _stream(q.device))
    _check(st, "jfa_bwd")
    return dq, dk, dv


def num_kv_blocks(offsets_host) -> int:
    """NB = sum_b ceil(len_b / 128), the row count of a block-sparse mask."""
    off = offsets_host.detach().to("cpu", torch.int32).contiguous()
    n = int(lib().jfa_num_kv_blocks(ctypes.c_void_p(off.data_ptr()), off.numel() - 1))
    if n < 0:
        raise JFAError(JFA_ERR_INVALID_ARG, "jfa_num_kv_blocks")
    return n


def _host_mask(kv_block_mask, offsets_host, H):
    mask = kv_block_mask.detach().to("cpu", torch.uint8).contiguous()
    nb = num_kv_blocks(offsets_host)
    if tuple(mask.shape) != (nb, H):
        raise ValueError(f"kv_block_mask must be uint8 [{nb}, {H}] (key blocks x heads), got {tuple(mask.shape)}")
    return mask


def fwd_block_sparse(q, k, v, offsets, kv_block_mask, broadcast_q: bool = True, scale: float | None = None,
                     offsets_host=None, workspace=None, out=None, lse=None):
    """Block-sparse O and LSE: only the key blocks kv_block_mask (host uint8 [NB, H]) selects."""
    assert q.is_cuda and q.dtype == torch.bfloat16 and k.dtype == torch.bfloat16 and v.dtype == torch.bfloat16
    H, D = k.shape[1], k.shape[2]
    offsets_host = _host_offsets(offsets, offsets_host)
    mask = _host_mask(kv_block_mask, offsets_host, H)
    B = offsets_host.numel() - 1
    N = int(offsets_host[-1]) if B > 0 else 0
    Lq = q.shape[0] if broadcast_q else 0
    out = torch.empty((B, Lq, H, D) if broadcast_q else (N, H, D), dtype=torch.bfloat16,
                      device=q.device) if out is None else out
    lse = torch.empty((B, H, Lq) if broadcast_q else (H, N), dtype=torch.float32,
                      device=q.device) if lse is None else lse
    if workspace is None:
        workspace = new_workspace(B, N, Lq, H, D, broadcast_q, False, q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    offsets_dev = offsets if (offsets is not None and offsets.is_cuda) else None
    st = lib().jfa_fwd_block_sparse(_ptr(q.contiguous()), _ptr(k.contiguous()), _ptr(v.contiguous()),
                                    _ptr(offsets_dev), ctypes.c_void_p(offsets_host.data_ptr()),
                                    ctypes.c_void_p(mask.data_ptr()), B, Lq, H, D, int(broadcast_q), sc, _ptr(out),
                                    _ptr(lse), _ptr(workspace), workspace.numel(), _stream(q.device))
    _check(st, "jfa_fwd_block_sparse")
    return out, lse


def bwd_block_sparse(q, k, v, o, lse, do, offsets, kv_block_mask, broadcast_q: bool = True,
                     scale: float | None = None, offsets_host=None, workspace=None, dq=None, dk=None, dv=None):
    """Block-sparse dQ, dK, dV (unselected keys get zero dK and dV)."""
    H, D = k.shape[1], k.shape[2]
    offsets_host = _host_offsets(offsets, offsets_host)
    mask = _host_mask(kv_block_mask, offsets_host, H)
    B = offsets_host.numel() - 1
    N = int(offsets_host[-1]) if B > 0 else 0
    Lq = q.shape[0] if broadcast_q else 0
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.bfloat16, device=q.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.bfloat16, device=q.device) if dv is None else dv
    if workspace is None:
        workspace = new_workspace(B, N, Lq, H, D, broadcast_q, False, q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    offsets_dev = offsets if (offsets is not None and offsets.is_cuda) else None
    st = lib().jfa_bwd_block_sparse(_ptr(q.contiguous()), _ptr(k.contiguous()), _ptr(v.contiguous()),
                                    _ptr(o.contiguous()), _ptr(lse.contiguous()), _ptr(do.contiguous()),
                                    _ptr(offsets_dev), ctypes.c_void_p(offsets_host.data_ptr()),
                                    ctypes.c_void_p(mask.data_ptr()), B, Lq, H, D, int(broadcast_q), sc, _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), _stream(q.device))
    _check(st, "jfa_bwd_block_sparse")
    return dq, dk, dv


def quantize_v_mxfp8(v, offsets, offsets_host=None, workspace=None, v8=None, v_scale=None):
    """MXFP8 V for fwd_mxfp8: E4M3 codes (uint8 [N,H,D]) and E8M0 scales (uint8 [NB,H,D,4]) of bf16 v."""
    assert v.is_cuda and v.dtype == torch.bfloat16 and offsets is not None and offsets.is_cuda
    N, H, D = v.shape
    offsets_host = _host_offsets(offsets, offsets_host)
    B = offsets_host.numel() - 1
    nb = num_kv_blocks(offsets_host)
    v8 = torch.empty((N, H, D), dtype=torch.uint8, device=v.device) if v8 is None else v8
    v_scale = torch.empty((nb, H, D, 4), dtype=torch.uint8, device=v.device) if v_scale is None else v_scale
    if workspace is None:
        workspace = torch.empty(256 + 4 * (B + 1), dtype=torch.uint8, device=v.device)
    st = lib().jfa_quantize_v_mxfp8(_ptr(v.contiguous()), _ptr(offsets), ctypes.c_void_p(offsets_host.data_ptr()),
                                    B, H, D, _ptr(v8), _ptr(v_scale), _ptr(workspace), workspace.numel(),
                                    _stream(v.device))
    _check(st, "jfa_quantize_v_mxfp8")
    return v8, v_scale


def fwd_mxfp8(q, k, v8, v_scale, offsets, broadcast_q: bool = True, causal: bool = False,
              scale: float | None = None, offsets_host=None, workspace=None, out=None, lse=None):
    """MXFP8 forward: O (bf16) and LSE (fp32) with P V in MXFP8; v8 / v_scale from quantize_v_mxfp8."""
    assert q.is_cuda and q.dtype == torch.bfloat16 and k.dtype == torch.bfloat16 and v8.dtype == torch.uint8
    H, D = k.shape[1], k.shape[2]
    offsets_host = _host_offsets(offsets, offsets_host)
    B = offsets_host.numel() - 1
    N = int(offsets_host[-1]) if B > 0 else 0
    nb = num_kv_blocks(offsets_host)
    if tuple(v8.shape) != (N, H, D) or tuple(v_scale.shape) != (nb, H, D, 4) or v_scale.dtype != torch.uint8:
        raise ValueError(f"v8 must be uint8 [{N}, {H}, {D}] and v_scale uint8 [{nb}, {H}, {D}, 4]")
    Lq = q.shape[0] if broadcast_q else 0
    out = torch.empty((B, Lq, H, D) if broadcast_q else (N, H, D), dtype=torch.bfloat16,
                      device=q.device) if out is None else out
    lse = torch.empty((B, H, Lq) if broadcast_q else (H, N), dtype=torch.float32,
                      device=q.device) if lse is None else lse
    if workspace is None:
        workspace = new_workspace(B, N, Lq, H, D, broadcast_q, causal, q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    offsets_dev = offsets if (offsets is not None and offsets.is_cuda) else None
    st = lib().jfa_fwd_mxfp8(_ptr(q.contiguous()), _ptr(k.contiguous()), _ptr(v8.contiguous()),
                             _ptr(v_scale.contiguous()), _ptr(offsets_dev), ctypes.c_void_p(offsets_host.data_ptr()),
                             B, Lq, H, D, int(broadcast_q), int(causal), sc, _ptr(out), _ptr(lse), _ptr(workspace),
                             workspace.numel(), _stream(q.device))
    _check(st, "jfa_fwd_mxfp8")
    return out, lse


def device_status(workspace, device=None) -> int:
    """Synchronises the current stream and returns (and clears) the kernels' status word."""
    device = workspace.device if device is None else device
    return int(lib().jfa_device_status(_ptr(workspace), _stream(device)))


def profile_enable(on: bool = True) -> None:
    _check(lib().jfa_profile_enable(int(on)), "jfa_profile_enable")


PROFILE_KINDS = ("fwd", "bwd_pre", "bwd", "zero_tiles", "fwd_merge", "quant_v")


def profile_read() -> dict:
    """Per-kernel event-timed totals since the previous read: {kernel: (ms, launches)}."""
    n = len(PROFILE_KINDS)
    ms, cnt = (ctypes.c_double * n)(), (ctypes.c_int * n)()
    _check(lib().jfa_profile_read(ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(cnt, ctypes.c_void_p), n),
           "jfa_profile_read")
    return {k: (ms[i], cnt[i]) for i, k in enumerate(PROFILE_KINDS)}


def num_ctas() -> int:
    return int(lib().jfa_num_ctas())


# deal policies (SCHED_CLC, SCHED_QUEUE: backward only)
SCHED_ZIGZAG, SCHED_NAIVE, SCHED_GREEDY, SCHED_CLC, SCHED_QUEUE = 0, 1, 2, 3, 4


def host_schedule(offsets_host, Lq: int, H: int, broadcast_q: bool, causal: bool, is_bwd: bool, P: int,
                  policy: int = SCHED_ZIGZAG, noalloc: bool = False):
    """The host scheduler alone (no GPU): returns (items int32 [n,4], cta_start int32 [P+1]).
    noalloc=True runs the allocation-free builder (always the greedy deal)."""
    off = offsets_host.to(torch.int32).contiguous()
    B = off.numel() - 1
    N = int(off[-1]) if B > 0 else 0
    cap = H * (N // 128 + B) + H * B * ((max(Lq, 0) + 255) // 256) + 1
    items = torch.zeros((cap, 4), dtype=torch.int32)
    # P + 1 CTA bounds; a queue schedule writes 2G + 1 <= 2H + 1 entries
    starts = torch.zeros(max(P + 1, 2 * H + 1), dtype=torch.int32)
    if noalloc:
        n = lib().jfa_host_build_schedule_noalloc(ctypes.c_void_p(off.data_ptr()), B, Lq, H, int(broadcast_q),
                                                  int(causal), int(is_bwd), P, ctypes.c_void_p(items.data_ptr()),
                                                  ctypes.c_void_p(starts.data_ptr()), cap)
    else:
        n = lib().jfa_host_build_schedule(ctypes.c_void_p(off.data_ptr()), B, Lq, H, int(broadcast_q),
                                          int(causal), int(is_bwd), P, policy, ctypes.c_void_p(items.data_ptr()),
                                          ctypes.c_void_p(starts.data_ptr()), cap)
    if n < 0:
        raise JFAError(JFA_ERR_WORKSPACE, "jfa_host_build_schedule")
    return items[:n].clone(), (starts if policy == SCHED_QUEUE else starts[:P + 1].clone())


def set_wait_limit(ns: int = 0) -> None:
    """Limit of one barrier wait inside the kernels, in ns, for later launches (0: the 4 s default)."""
    _check(lib().jfa_set_wait_limit(int(ns)), "jfa_set_wait_limit")


def set_schedule_policy(fwd_policy: int = None, bwd_policy: int = None) -> None:
    """How later calls deal their sorted items to the CTAs (a measurement aid; defaults: greedy / zigzag)."""
    _check(lib().jfa_set_schedule_policy(SCHED_GREEDY if fwd_policy is None else int(fwd_policy),
                                         SCHED_ZIGZAG if bwd_policy is None else int(bwd_policy)),
           "jfa_set_schedule_policy")


def host_schedule_split(offsets_host, Lq: int, H: int, P: int, with_slot_blocks: bool = False):
    """The broadcast-Q forward schedule with split-KV (no GPU): (items [n,4], cta_start [P+1],
    groups [n_groups,4] = (b, first slot, chunks, h | tile << 8), slot count); with_slot_blocks
    adds each slot's first key block over all sequences (int32 [slots])."""
    off = offsets_host.to(torch.int32).contiguous()
    B = off.numel() - 1
    N = int(off[-1]) if B > 0 else 0
    cap = H * (N // 128 + B) + H * B * ((max(Lq, 0) + 255) // 256) + 1
    items = torch.zeros((cap, 4), dtype=torch.int32)
    starts = torch.zeros(P + 1, dtype=torch.int32)
    groups = torch.zeros((SPLIT_MAX_SLOTS, 4), dtype=torch.int32)
    counts = (ctypes.c_longlong * 2)()
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    slot_blocks = torch.zeros(SPLIT_MAX_SLOTS, dtype=torch.int32)
    n = lib().jfa_host_build_schedule_split(vp(off), B, Lq, H, P, vp(items), vp(starts), cap, vp(groups), counts,
                                            vp(slot_blocks) if with_slot_blocks else None)
    if n < 0:
        raise JFAError(JFA_ERR_WORKSPACE, "jfa_host_build_schedule_split")
    out = (items[:n].clone(), starts, groups[:counts[0]].clone(), int(counts[1]))
    return out + (slot_blocks[:counts[1]].clone(),) if with_slot_blocks else out


SPLIT_MAX_SLOTS = 512  # split-KV partial slots per call (the library's workspace bound)


def host_schedule_sparse(offsets_host, kv_block_mask, Lq: int, H: int, broadcast_q: bool, is_bwd: bool, P: int):
    """The block-sparse host schedule alone (no GPU): (items [n,4], cta_start [P+1], sel [B*H,4]
    = (list offset, selected, full selected, 0), blocks [n_blocks], zero tiles [n_zero,4] =
    (row0, rows, h, 0))."""
    off = offsets_host.to(torch.int32).contiguous()
    B = off.numel() - 1
    N = int(off[-1]) if B > 0 else 0
    mask = _host_mask(kv_block_mask, off, H)
    cap_items = H * (N // 128 + B) + H * B * ((max(Lq, 0) + 255) // 256) + 1
    cap = H * (N // 128 + B) + 1
    items = torch.zeros((cap_items, 4), dtype=torch.int32)
    starts = torch.zeros(P + 1, dtype=torch.int32)
    sel = torch.zeros((max(B * H, 1), 4), dtype=torch.int32)
    blocks = torch.zeros(cap, dtype=torch.int32)
    zero = torch.zeros((cap, 4), dtype=torch.int32)
    counts = (ctypes.c_longlong * 2)()
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    n = lib().jfa_host_build_schedule_sparse(vp(off), B, Lq, H, int(broadcast_q), int(is_bwd), P, vp(mask),
                                             vp(items), vp(starts), cap_items, vp(sel), vp(blocks), vp(zero), cap,
                                             counts)
    if n < 0:
        raise JFAError(JFA_ERR_WORKSPACE, "jfa_host_build_schedule_sparse")
    return (items[:n].clone(), starts, sel[:B * H].clone(), blocks[:counts[0]].clone(),
            zero[:counts[1]].clone())


def selftest_mma(mode: int, a, b):
    """One 128x128x128 tcgen05 product (see include/jfa_selftest.h); returns (C fp32, status word)."""
    c = torch.empty((128, 128), dtype=torch.float32, device=a.device)
    status = torch.zeros(1, dtype=torch.int32, device=a.device)
    st = lib().jfa_selftest_mma(mode, _ptr(a.contiguous()), _ptr(b.contiguous()), _ptr(c), _ptr(status),
                                _stream(a.device))
    if st != 0:
        raise JFAError(st, "jfa_selftest_mma")
    return c, status
