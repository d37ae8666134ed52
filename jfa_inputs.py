"""Seeded synthetic workloads for Jagged Flash Attention.

This module only draws random numbers: it holds none of the attention
arithmetic, so both the fp64 oracle (``oracle/``) and the CUDA path
(``bwd_jagged_flashattention_gb300``) can take their inputs from it without
sharing any of the method's code.

The five workloads follow the shapes the pages describe: jagged user
sequences packed contiguously with an offsets tensor ("Why attention in GEM
needed a rewrite", Meta's TLX Jagged Flash Attention Beats FA4 on Blackwell
With 3x Less Code), a single dense Q broadcast over every sequence (Meta's
3.2K-line Triton kernel outruns FlashAttention-4 on jagged Blackwell
attention, second paragraph), and dense LLM-style causal self-attention
(TLX porta l'attenzione jagged su Blackwell oltre FA4, introduction).
No dataset is involved; these inputs stand in for the GEM workloads.

Recipe (all on the CPU, ``torch.Generator().manual_seed(seed)``):
  1. sequence lengths (int64, then int32 offsets = exclusive prefix sum),
  2. Q, K, V as fp32 N(0,1), rounded to bf16 (round-to-nearest-even),
  3. dO as fp32 N(0,1) rounded to bf16 (backward workloads only).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Lq: int            # broadcast Q rows; ignored (per-sequence) when not broadcast_q
    H: int
    D: int
    broadcast_q: bool
    causal: bool
    lengths: str       # length recipe: "uniform:a:b", "lognormal:median:sigma:lo:hi", "skew:frac:a:b:c:d"
    backward: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# The five workloads, in order. Index i (1-based) is also the default seed.
WORKLOADS = {
    "tiny": Workload("tiny", B=4, Lq=32, H=2, D=64, broadcast_q=True, causal=False,
                     lengths="uniform:1:64"),
    "ads_fwd": Workload("ads_fwd", B=512, Lq=256, H=4, D=128, broadcast_q=True, causal=False,
                        lengths="lognormal:256:1.0:8:4096", backward=False),
    "ads_bwd": Workload("ads_bwd", B=512, Lq=256, H=4, D=128, broadcast_q=True, causal=False,
                        lengths="lognormal:256:1.0:8:4096"),
    "dense_llm": Workload("dense_llm", B=32, Lq=0, H=16, D=128, broadcast_q=False, causal=True,
                          lengths="uniform:512:8192"),
    "extreme": Workload("extreme", B=2048, Lq=128, H=2, D=128, broadcast_q=True, causal=False,
                        lengths="skew:0.1:1:32:4096:16384"),
}
WORKLOAD_ORDER = ["tiny", "ads_fwd", "ads_bwd", "dense_llm", "extreme"]


def default_seed(name: str) -> int:
    return WORKLOAD_ORDER.index(name) + 1


def draw_lengths(recipe: str, B: int, gen: torch.Generator) -> torch.Tensor:
    """Per-sequence KV lengths (int64 [B]) from a recipe string."""
    kind, *args = recipe.split(":")
    if kind == "uniform":
        lo, hi = int(args[0]), int(args[1])
        return torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64)
    if kind == "lognormal":
        median, sigma, lo, hi = float(args[0]), float(args[1]), int(args[2]), int(args[3])
        x = torch.empty(B, dtype=torch.float64).log_normal_(math.log(median), sigma, generator=gen)
        return x.round().clamp_(lo, hi).to(torch.int64)
    if kind == "skew":
        frac, slo, shi, llo, lhi = float(args[0]), *(int(a) for a in args[1:])
        n_long = int(round(frac * B))
        short = torch.randint(slo, shi + 1, (B - n_long,), generator=gen, dtype=torch.int64)
        long_ = torch.randint(llo, lhi + 1, (n_long,), generator=gen, dtype=torch.int64)
        perm = torch.randperm(B, generator=gen)
        return torch.cat([short, long_])[perm]
    if kind == "fixed":
        vals = [int(a) for a in args[0].split(",")]
        assert len(vals) == B
        return torch.tensor(vals, dtype=torch.int64)
    raise ValueError(f"unknown length recipe {recipe!r}")


def offsets_from_lengths(lengths: torch.Tensor) -> torch.Tensor:
    off = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    off[1:] = torch.cumsum(lengths.to(torch.int64), 0)
    assert int(off[-1]) < 2**31, "total length must fit int32"
    return off.to(torch.int32)


def _normal_bf16(shape, gen) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make(w: Workload | str, seed: int | None = None, lengths: torch.Tensor | None = None,
         backward: bool | None = None) -> dict:
    """Draw one batch of CPU tensors for workload ``w``.

    Returns a dict with: offsets int32 [B+1], q bf16 ([Lq,H,D] broadcast or
    [N,H,D] jagged), k, v bf16 [N,H,D], do bf16 (output-shaped, backward only),
    and the scalar fields B, Lq, H, D, broadcast_q, causal, scale, N.
    """
    if isinstance(w, str):
        if seed is None:
            seed = default_seed(w)
        w = WORKLOADS[w]
    gen = torch.Generator().manual_seed(0 if seed is None else seed)
    if lengths is None:
        lengths = draw_lengths(w.lengths, w.B, gen)
    offsets = offsets_from_lengths(lengths)
    N = int(offsets[-1])
    qrows = w.Lq if w.broadcast_q else N
    q = _normal_bf16((qrows, w.H, w.D), gen)
    k = _normal_bf16((N, w.H, w.D), gen)
    v = _normal_bf16((N, w.H, w.D), gen)
    out = dict(workload=w.name, offsets=offsets, q=q, k=k, v=v, B=w.B, Lq=w.Lq, H=w.H, D=w.D,
               broadcast_q=w.broadcast_q, causal=w.causal, scale=w.scale, N=N)
    if w.backward if backward is None else backward:
        oshape = (w.B, w.Lq, w.H, w.D) if w.broadcast_q else (N, w.H, w.D)
        out["do"] = _normal_bf16(oshape, gen)
    return out


def custom(B: int, Lq: int, H: int, D: int, lengths, broadcast_q: bool, causal: bool,
           seed: int = 0, backward: bool = True) -> dict:
    """Same recipe as :func:`make` for an explicit list of sequence lengths."""
    lengths = torch.as_tensor(list(lengths), dtype=torch.int64)
    assert lengths.numel() == B
    w = Workload("custom", B=B, Lq=Lq, H=H, D=D, broadcast_q=broadcast_q, causal=causal,
                 lengths="fixed:" + ",".join(str(int(x)) for x in lengths) if B else "fixed:",
                 backward=backward)
    return make(w, seed=seed, lengths=lengths, backward=backward)


def num_kv_blocks(offsets: torch.Tensor) -> int:
    """Number of 128-key blocks over all sequences: sum_b ceil(len_b / 128)."""
    lens = (offsets[1:] - offsets[:-1]).to(torch.int64)
    return int(((lens + 127) // 128).sum())


def kv_block_mask(offsets: torch.Tensor, H: int, ratio: float, seed: int = 0) -> torch.Tensor:
    """Seeded block selection for the block-sparse variant: uint8 [NB, H],
    each (128-key block, head) selected independently with probability
    `ratio` (a Bernoulli draw from its own generator)."""
    gen = torch.Generator().manual_seed(10_000 + seed)
    nb = num_kv_blocks(offsets)
    return (torch.rand((nb, H), generator=gen) < ratio).to(torch.uint8)
