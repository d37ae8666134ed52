"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, element by element, at sizes the oracle finishes in
seconds that still span several tiles and ragged tails, plus the edge cases
(empty sequences, single keys, tile boundaries, both head dimensions)."""
import pytest
import torch

import jfa_inputs
from tests.gpu_util import check_all, gpu_fwd_bwd, oracle_fwd_bwd

pytestmark = pytest.mark.gpu


def _run(x, what, backward=True):
    got = gpu_fwd_bwd(x, backward)
    ref = oracle_fwd_bwd(x, backward)
    check_all(x, got, ref, what, backward)


def test_tiny_workload():
    _run(jfa_inputs.make("tiny"), "tiny")


EDGE_LENGTHS = [1, 127, 128, 129, 255, 256, 257]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lq", [1, 32, 128, 129, 256])
def test_broadcast_tile_edges(D, Lq):
    x = jfa_inputs.custom(len(EDGE_LENGTHS), Lq, 2, D, EDGE_LENGTHS, True, False, seed=Lq + D)
    _run(x, f"broadcast D={D} Lq={Lq}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_jagged_tile_edges(D, causal):
    lengths = EDGE_LENGTHS + [300, 513]
    x = jfa_inputs.custom(len(lengths), 0, 2, D, lengths, False, causal, seed=7 + D + causal)
    _run(x, f"jagged D={D} causal={causal}")


def test_empty_sequences_broadcast():
    lengths = [0, 5, 0, 0, 130, 0]
    x = jfa_inputs.custom(len(lengths), 40, 2, 128, lengths, True, False, seed=3)
    _run(x, "broadcast with empty sequences")


def test_all_empty_but_one():
    lengths = [0, 0, 0, 200, 0]
    for bq in (True, False):
        x = jfa_inputs.custom(len(lengths), 130 if bq else 0, 1, 64, lengths, bq, False, seed=4)
        _run(x, f"all empty but one (broadcast={bq})")


def test_all_empty():
    x = jfa_inputs.custom(3, 16, 2, 64, [0, 0, 0], True, False, seed=5)
    _run(x, "all sequences empty")


def test_ads_like_small():
    """The ads broadcast-Q recipe (lognormal lengths, Lq=256, H=4, D=128) on 24 sequences."""
    w = jfa_inputs.WORKLOADS["ads_bwd"]
    g = torch.Generator().manual_seed(11)
    L = jfa_inputs.draw_lengths(w.lengths, 24, g)
    x = jfa_inputs.custom(24, 256, 4, 128, L.tolist(), True, False, seed=11)
    _run(x, "ads-like small")


def test_dense_llm_like_small():
    """Causal jagged self-attention (H=2, D=128) with lengths spanning many tiles."""
    x = jfa_inputs.custom(3, 0, 2, 128, [600, 1500, 777], False, True, seed=12)
    _run(x, "dense-llm-like small")


def test_extreme_like_small():
    """Length skew: many 1..32-key sequences and a few 4096+ ones (Lq=128, H=2)."""
    g = torch.Generator().manual_seed(13)
    L = jfa_inputs.draw_lengths("skew:0.1:1:32:4096:5000", 40, g)
    x = jfa_inputs.custom(40, 128, 2, 128, L.tolist(), True, False, seed=13)
    _run(x, "extreme-like small")


def test_repeat_determinism():
    """O, LSE, dK and dV are bitwise repeatable; dQ (atomic adds) within rounding."""
    x = jfa_inputs.custom(6, 200, 2, 128, [300, 7, 128, 1, 999, 250], True, False, seed=21)
    a = gpu_fwd_bwd(x)
    b = gpu_fwd_bwd(x)
    for n in ("o", "lse", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n
    assert (a["dq"] - b["dq"]).abs().max().item() <= 1e-4 * max(1.0, a["dq"].abs().max().item())


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lq", [64, 128])
def test_broadcast_one_query_tile_many_items(D, Lq):
    """Broadcast Q of a single query tile (Lq <= 128) with many key-tile
    items per CTA (60 sequences of up to 3000 keys over the SMs): every item
    reuses the CTA's resident Q tile, and every CTA walks several items
    through the single-buffered K/V; dK / dV / dQ against the oracle."""
    g = torch.Generator().manual_seed(Lq + D)
    lengths = torch.randint(1, 3000, (60,), generator=g).tolist()
    x = jfa_inputs.custom(len(lengths), Lq, 2, D, lengths, True, False, seed=Lq * D)
    _run(x, f"broadcast one query tile D={D} Lq={Lq}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bq", [True, False])
def test_many_items_per_cta_with_empty_sequences(D, bq):
    """Several items per CTA (700 short sequences over the SMs), with empty
    sequences between them: each CTA's K/V ring (4 slots at D = 128, 8 at
    D = 64) wraps across items, so a V tile and the next item's first K share
    a barrier phase and a release, with empty items skipped in between; the
    backward walks several key tiles per CTA the same way."""
    g = torch.Generator().manual_seed(31 + D + bq)
    pool = torch.tensor([0, 0, 1, 5, 64, 127, 128, 129, 200, 256, 300])
    lengths = pool[torch.randint(0, len(pool), (700,), generator=g)].tolist()
    x = jfa_inputs.custom(len(lengths), 64 if bq else 0, 1, D, lengths, bq, False, seed=41 + D)
    _run(x, f"many items per CTA D={D} broadcast={bq}")
