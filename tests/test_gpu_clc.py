"""The backward with its items dealt at run time: by Cluster Launch Control,
or from per-head-group queues.

With jfa_set_schedule_policy(bwd=3) the backward launches one CTA per item of
the longest-first list; every resident CTA, as it starts an item, asks the
hardware to cancel a CTA that has not started yet and takes over that item
(the pages name Cluster Launch Control among the primitives that keep SMs
busy under length skew: Meta's TLX Jagged Flash Attention Beats FA4 on
Blackwell With 3x Less Code, sections "What TLX changes" and "Optimizations
layered on top").  Each case must match the fp64 oracle as the static
schedule does, and the status word must stay clear.
"""
import pytest
import torch

import jfa_inputs
from tests.gpu_util import check_all, gpu_fwd_bwd, oracle_fwd_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["clc", "queue"])
def clc_backward(request):
    """The backward dealt at run time: by Cluster Launch Control, or by the
    persistent CTAs taking items from their head group's queue."""
    import bwd_jagged_flashattention_gb300 as jfa
    jfa.set_schedule_policy(bwd_policy=jfa.SCHED_CLC if request.param == "clc" else jfa.SCHED_QUEUE)
    yield jfa
    jfa.set_schedule_policy()


def _lengths(recipe, B, seed):
    return jfa_inputs.draw_lengths(recipe, B, torch.Generator().manual_seed(seed)).tolist()


CASES = [
    ("tiny", lambda: jfa_inputs.make("tiny")),
    ("broadcast tile edges", lambda: jfa_inputs.custom(7, 129, 2, 128, [1, 127, 128, 129, 255, 256, 257], True,
                                                        False, seed=51)),
    ("ads-like", lambda: jfa_inputs.custom(24, 256, 4, 128, _lengths("lognormal:256:1.0:8:4096", 24, 52), True,
                                           False, seed=52)),
    ("skewed", lambda: jfa_inputs.custom(40, 128, 2, 128, _lengths("skew:0.1:1:32:4096:5000", 40, 53), True,
                                         False, seed=53)),
    ("jagged causal D=64", lambda: jfa_inputs.custom(5, 0, 2, 64, [600, 1, 129, 300, 777], False, True, seed=54)),
    ("with empty sequences", lambda: jfa_inputs.custom(6, 40, 2, 128, [0, 5, 0, 0, 130, 0], True, False, seed=55)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_clc_backward_matches_oracle(clc_backward, name, make):
    x = make()
    check_all(x, gpu_fwd_bwd(x), oracle_fwd_bwd(x), f"CLC backward: {name}")


def test_clc_backward_full_ads(clc_backward):
    """The ads workload at full size (7,000+ CTAs in the grid, 152 resident)."""
    x = jfa_inputs.make("ads_bwd")
    check_all(x, gpu_fwd_bwd(x), oracle_fwd_bwd(x), "CLC backward: ads")
