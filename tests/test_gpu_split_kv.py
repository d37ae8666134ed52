"""GPU parity of split-KV in the broadcast-Q forward: batches skewed enough
that the host splits the long sequences' query tiles into key chunks (fp32
partial O / LSE per chunk, merged by the merge kernel), checked against the
fp64 oracle with the dense contract's tolerances; the backward then runs on
the merged O and LSE."""
import pytest
import torch

import jfa_inputs
from tests.gpu_util import check_all, gpu_fwd_bwd, oracle_fwd_bwd

pytestmark = pytest.mark.gpu


def _splits(x):
    import bwd_jagged_flashattention_gb300 as jfa
    _, _, groups, slots = jfa.host_schedule_split(x["offsets"], x["Lq"], x["H"], jfa.num_ctas())
    return len(groups), slots


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lq", [128, 256, 300])
def test_skewed_broadcast_split_kv(D, Lq):
    lengths = [20000, 5, 300, 0, 129, 1000, 1]
    x = jfa_inputs.custom(len(lengths), Lq, 2, D, lengths, True, False, seed=D + Lq)
    groups, slots = _splits(x)
    assert groups > 0, "the batch must exercise split-KV"
    check_all(x, gpu_fwd_bwd(x), oracle_fwd_bwd(x), f"split-KV D={D} Lq={Lq} ({groups} tiles, {slots} chunks)")


def test_one_very_long_sequence():
    """A single 100K-key sequence among short ones (the case split-KV is for)."""
    lengths = [100000] + [64] * 15
    x = jfa_inputs.custom(len(lengths), 128, 4, 128, lengths, True, False, seed=9)
    groups, slots = _splits(x)
    assert groups == 4 and slots > 100
    check_all(x, gpu_fwd_bwd(x), oracle_fwd_bwd(x), f"100K keys ({slots} chunks)")
