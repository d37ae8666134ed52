"""fp64 CPU oracle for Jagged Flash Attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never does; the two share no
code.  The arithmetic lives in ``jfa_oracle.c`` (plain C, fp64, OpenMP) and
follows the definition written at the top of that file: per sequence and
head, softmax(scale * Q K^T) V with its analytic gradients, looping over the
offsets tensor ("Why attention in GEM needed a rewrite", Meta's TLX Jagged
Flash Attention Beats FA4 on Blackwell With 3x Less Code); broadcast-Q sums
dQ over the batch (Meta's 3.2K-line Triton kernel outruns FlashAttention-4 on
jagged Blackwell attention, second paragraph).

Every function here is pinned by ``tests/test_oracle_pins.py`` (brute force
against padded dense attention with torch autograd in fp64, invariants,
closed forms, a hand-derived worked example under ``tests/golden/``, central
finite differences, and the broadcast dQ batch sum).  The block-sparse
variant (``kv_block_mask``) is pinned by ``tests/test_oracle_block_sparse.py``
(dense attention over only the gathered selected keys, per sequence and head,
with torch autograd; exact zeros and -inf for empty selections; planted mask
bugs).  The MXFP8 variant (``quantize_v_mxfp8``, ``fwd_mxfp8`` and the
E4M3 / E8M0 helpers) is pinned by ``tests/test_oracle_mxfp8.py`` (the E4M3
format's landmarks, brute-force nearest-even rounding, the MX exponent's
top-binade property, brute-force V and P quantization, equality with the plain
oracle where quantization is lossless, planted mistakes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jfa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libjfa_oracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """Compile one oracle source file into a shared library at ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    # -ffp-contract=off keeps every multiply and add a separately rounded fp64 op.
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp) if stale.  Returns the .so path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _offsets_arg(offsets):
    offsets = offsets.detach().cpu().to(torch.int32).contiguous()
    return offsets, ctypes.cast(offsets.data_ptr(), ctypes.POINTER(ctypes.c_int32))


def _mask_arg(mask, offsets, H):
    """uint8 [NB, H] block mask (checked against the offsets) and its pointer."""
    mask = mask.detach().cpu().to(torch.uint8).contiguous()
    lens = offsets[1:] - offsets[:-1]
    nb = int(((lens.to(torch.int64) + 127) // 128).sum())
    if tuple(mask.shape) != (nb, H):
        raise ValueError(f"kv_block_mask must be [{nb}, {H}], got {tuple(mask.shape)}")
    return mask, ctypes.cast(mask.data_ptr(), ctypes.POINTER(ctypes.c_uint8))


def _inputs(*ts):
    """All-bf16 inputs pass as raw bf16 (widened exactly in C); anything else as fp64."""
    ts = [t.detach().cpu().contiguous() for t in ts]
    if all(t.dtype == torch.bfloat16 for t in ts):
        return ts, 1
    return [t.to(torch.float64).contiguous() for t in ts], 0


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        vp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
        ci, cd = ctypes.c_int, ctypes.c_double
        lib.jfa_oracle_fwd.argtypes = [vp, vp, vp, ci, i32p, ci, ci, ci, ci, ci, ci, cd, vp, vp]
        lib.jfa_oracle_fwd.restype = None
        lib.jfa_oracle_bwd.argtypes = [vp, vp, vp, vp, ci, i32p, ci, ci, ci, ci, ci, ci, cd, vp, vp, vp]
        lib.jfa_oracle_bwd.restype = None
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.jfa_oracle_fwd_block_sparse.argtypes = [vp, vp, vp, ci, i32p, ci, ci, ci, ci, ci, ci, cd, u8p, vp, vp]
        lib.jfa_oracle_fwd_block_sparse.restype = None
        lib.jfa_oracle_bwd_block_sparse.argtypes = [vp, vp, vp, vp, ci, i32p, ci, ci, ci, ci, ci, ci, cd, u8p,
                                                    vp, vp, vp]
        lib.jfa_oracle_bwd_block_sparse.restype = None
        lib.jfa_oracle_max_threads.argtypes = []
        lib.jfa_oracle_max_threads.restype = ci
        # MXFP8 variant (present in every build of jfa_oracle.c)
        i64 = ctypes.c_int64
        lib.jfa_oracle_e4m3_encode_array.argtypes = [vp, i64, vp]
        lib.jfa_oracle_e4m3_encode_array.restype = None
        lib.jfa_oracle_e4m3_value_array.argtypes = [vp, i64, vp]
        lib.jfa_oracle_e4m3_value_array.restype = None
        lib.jfa_oracle_mx_exponent.argtypes = [cd]
        lib.jfa_oracle_mx_exponent.restype = ci
        lib.jfa_oracle_mx_quantize_p.argtypes = [vp, ci, vp, vp]
        lib.jfa_oracle_mx_quantize_p.restype = None
        lib.jfa_oracle_quantize_v_mxfp8.argtypes = [vp, i32p, ci, ci, ci, vp, vp]
        lib.jfa_oracle_quantize_v_mxfp8.restype = None
        lib.jfa_oracle_fwd_mxfp8.argtypes = [vp, vp, vp, vp, ci, i32p, ci, ci, ci, ci, ci, ci, cd, vp, vp, vp]
        lib.jfa_oracle_fwd_mxfp8.restype = None
        self.lib = lib
        self.path = path

    def max_threads(self) -> int:
        return int(self.lib.jfa_oracle_max_threads())

    def fwd(self, q, k, v, offsets, Lq: int, broadcast_q: bool, causal: bool, scale: float,
            want_o: bool = True, want_lse: bool = True, kv_block_mask=None):
        """O (fp64, [B,Lq,H,D] or [N,H,D]) and LSE (fp64, [B,H,Lq] or [H,N]).

        kv_block_mask: optional uint8 [NB, H] (NB = sum_b ceil(len_b / 128));
        a zero entry hides that 128-key block of that head (block-sparse)."""
        offsets, off_p = _offsets_arg(offsets)
        B = offsets.numel() - 1
        N = int(offsets[-1]) if B > 0 else 0
        H, D = k.shape[1], k.shape[2]
        (qq, kk, vv), bf = _inputs(q, k, v)
        o = torch.zeros((B, Lq, H, D) if broadcast_q else (N, H, D), dtype=torch.float64) if want_o else None
        lse = torch.zeros((B, H, Lq) if broadcast_q else (H, N), dtype=torch.float64) if want_lse else None
        args = (_ptr(qq), _ptr(kk), _ptr(vv), bf, off_p, B, Lq, H, D, int(broadcast_q), int(causal), float(scale))
        if kv_block_mask is None:
            self.lib.jfa_oracle_fwd(*args, _ptr(o), _ptr(lse))
        else:
            mask, mask_p = _mask_arg(kv_block_mask, offsets, H)
            self.lib.jfa_oracle_fwd_block_sparse(*args, mask_p, _ptr(o), _ptr(lse))
        return o, lse

    def bwd(self, q, k, v, do, offsets, Lq: int, broadcast_q: bool, causal: bool, scale: float,
            want_dq: bool = True, want_dkv: bool = True, kv_block_mask=None):
        """dQ (fp64, shaped like Q), dK and dV (fp64, [N,H,D]) for upstream gradient dO.

        kv_block_mask: as for fwd()."""
        offsets, off_p = _offsets_arg(offsets)
        B = offsets.numel() - 1
        N = int(offsets[-1]) if B > 0 else 0
        H, D = k.shape[1], k.shape[2]
        (qq, kk, vv, dd), bf = _inputs(q, k, v, do)
        dq = torch.zeros(tuple(q.shape), dtype=torch.float64) if want_dq else None
        dk = torch.zeros((N, H, D), dtype=torch.float64) if want_dkv else None
        dv = torch.zeros((N, H, D), dtype=torch.float64) if want_dkv else None
        args = (_ptr(qq), _ptr(kk), _ptr(vv), _ptr(dd), bf, off_p, B, Lq, H, D, int(broadcast_q), int(causal),
                float(scale))
        if kv_block_mask is None:
            self.lib.jfa_oracle_bwd(*args, _ptr(dq), _ptr(dk), _ptr(dv))
        else:
            mask, mask_p = _mask_arg(kv_block_mask, offsets, H)
            self.lib.jfa_oracle_bwd_block_sparse(*args, mask_p, _ptr(dq), _ptr(dk), _ptr(dv))
        return dq, dk, dv

    # ---- MXFP8 variant (definitions at the end of jfa_oracle.c) ----
    def e4m3_encode(self, x):
        """Nearest E4M3 codes (uint8) to the finite values x (ties to even, saturating at 448)."""
        x = torch.as_tensor(x, dtype=torch.float64).contiguous()
        out = torch.empty(x.shape, dtype=torch.uint8)
        self.lib.jfa_oracle_e4m3_encode_array(_ptr(x), x.numel(), _ptr(out))
        return out

    def e4m3_value(self, codes):
        """Values (fp64; NaN for S.1111.111) of E4M3 codes."""
        codes = torch.as_tensor(codes, dtype=torch.uint8).contiguous()
        out = torch.empty(codes.shape, dtype=torch.float64)
        self.lib.jfa_oracle_e4m3_value_array(_ptr(codes), codes.numel(), _ptr(out))
        return out

    def mx_exponent(self, amax: float) -> int:
        """Shared exponent X of an MX block whose largest magnitude is amax."""
        return int(self.lib.jfa_oracle_mx_exponent(float(amax)))

    def mx_quantize_p(self, x, want_slack: bool = False):
        """Quantized weights 2^X E4M3(2^(x - X)) of one row of log2-domain logits x (chunks of 32 from 0)."""
        x = torch.as_tensor(x, dtype=torch.float64).contiguous()
        pq = torch.empty_like(x)
        sl = torch.empty_like(x) if want_slack else None
        self.lib.jfa_oracle_mx_quantize_p(_ptr(x), x.numel(), _ptr(pq), _ptr(sl))
        return (pq, sl) if want_slack else pq

    def quantize_v_mxfp8(self, v, offsets):
        """MXFP8 V: E4M3 codes [N,H,D] (uint8) and E8M0 scales [NB,H,D,4] (uint8) from bf16 V [N,H,D]."""
        offsets, off_p = _offsets_arg(offsets)
        B = offsets.numel() - 1
        v = v.detach().cpu().contiguous()
        if v.dtype != torch.bfloat16:
            raise ValueError("V must be bf16")
        N, H, D = v.shape
        lens = (offsets[1:] - offsets[:-1]).to(torch.int64)
        nb = int(((lens + 127) // 128).sum())
        v8 = torch.zeros((N, H, D), dtype=torch.uint8)
        vs = torch.zeros((nb, H, D, 4), dtype=torch.uint8)
        self.lib.jfa_oracle_quantize_v_mxfp8(_ptr(v), off_p, B, H, D, _ptr(v8), _ptr(vs))
        return v8, vs

    def fwd_mxfp8(self, q, k, v8, v_scale, offsets, Lq: int, broadcast_q: bool, causal: bool, scale: float,
                  want_slack: bool = False):
        """MXFP8 forward (P V with P quantized per 32 keys, V given as E4M3 codes + E8M0 scales):
        O (fp64), LSE (fp64) and, with want_slack, the per-element slack of O."""
        offsets, off_p = _offsets_arg(offsets)
        B = offsets.numel() - 1
        N = int(offsets[-1]) if B > 0 else 0
        H, D = k.shape[1], k.shape[2]
        (qq, kk), bf = _inputs(q, k)
        v8 = v8.detach().cpu().to(torch.uint8).contiguous()
        v_scale = v_scale.detach().cpu().to(torch.uint8).contiguous()
        lens = (offsets[1:] - offsets[:-1]).to(torch.int64)
        nb = int(((lens + 127) // 128).sum())
        if tuple(v8.shape) != (N, H, D) or tuple(v_scale.shape) != (nb, H, D, 4):
            raise ValueError("v8 must be [N,H,D] and v_scale [NB,H,D,4]")
        shape = (B, Lq, H, D) if broadcast_q else (N, H, D)
        o = torch.zeros(shape, dtype=torch.float64)
        lse = torch.zeros((B, H, Lq) if broadcast_q else (H, N), dtype=torch.float64)
        sl = torch.zeros(shape, dtype=torch.float64) if want_slack else None
        self.lib.jfa_oracle_fwd_mxfp8(_ptr(qq), _ptr(kk), _ptr(v8), _ptr(v_scale), bf, off_p, B, Lq, H, D,
                                      int(broadcast_q), int(causal), float(scale), _ptr(o), _ptr(lse), _ptr(sl))
        return (o, lse, sl) if want_slack else (o, lse)


def _default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def max_threads() -> int:
    return _default().max_threads()


def fwd(*args, **kwargs):
    return _default().fwd(*args, **kwargs)


def bwd(*args, **kwargs):
    return _default().bwd(*args, **kwargs)


def quantize_v_mxfp8(*args, **kwargs):
    return _default().quantize_v_mxfp8(*args, **kwargs)


def fwd_mxfp8(*args, **kwargs):
    return _default().fwd_mxfp8(*args, **kwargs)
