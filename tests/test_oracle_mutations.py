"""The oracle's pins are sensitive: plant a plausible mistake in a copy of the
oracle's C source (on the CPU, in a temporary directory) and check that the
brute-force pin of tests/test_oracle_pins.py rejects every mutant.

Each mutation is one of the slips the pins are meant to catch: a dropped term,
a wrong sign, a wrong operand, an off-by-one mask, a dropped scale.
"""
import os

import pytest
import torch

import oracle
from tests.test_oracle_pins import CASES, _f64_inputs, brute_force

SRC = os.path.join(os.path.dirname(oracle.__file__), "jfa_oracle.c")

MUTATIONS = {
    "delta_drops_P": ("delta += s[j] * dp[j];", "delta += dp[j];"),
    "dS_sign": ("const double ds = p * (dp[j] - delta);", "const double ds = p * (dp[j] + delta);"),
    "dK_drops_scale": ("dkacc[(int64_t)j * D + d] += scale * ds * qi[d];", "dkacc[(int64_t)j * D + d] += ds * qi[d];"),
    "dQ_uses_V": ("dqi[d] += scale * ds * kmat[(int64_t)j * D + d];", "dqi[d] += scale * ds * vmat[(int64_t)j * D + d];"),
    "dV_uses_dS": ("dvacc[(int64_t)j * D + d] += p * doi[d];", "dvacc[(int64_t)j * D + d] += ds * doi[d];"),
    "causal_off_by_one": ("if (causal && j > i) {", "if (causal && j >= i) {"),
    "lse_drops_max": ("return m + log(acc);", "return log(acc);"),
    "scores_drop_scale": ("s[j] = scale * dot(qi, kmat + (int64_t)j * D, D);", "s[j] = dot(qi, kmat + (int64_t)j * D, D);"),
    "jagged_q_row_ignores_offset": ("return broadcast_q ? (int64_t)i : (int64_t)off[b] + i;", "return (int64_t)i;"),
    "lse_layout_transposed": ("return broadcast_q ? ((int64_t)b * H + h) * Lq + i : (int64_t)h * N + off[b] + i;",
                              "return broadcast_q ? ((int64_t)i * H + h) * B0 + b : (int64_t)h * N + off[b] + i;"),
}


def _mutant(tmp_path, name):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    src = src.replace(before, after)
    if "B0" in after:
        # the transposed-layout mutant needs B in scope; give it the batch size via a global
        src = src.replace("static int64_t lse_index(", "static int B0 = 1;\nstatic int64_t lse_index(")
        src = src.replace("    const int N = B > 0 ? offsets[B] : 0;\n    const int64_t pairs = (int64_t)B * H;\n#pragma omp parallel\n",
                          "    const int N = B > 0 ? offsets[B] : 0;\n    const int64_t pairs = (int64_t)B * H;\n    B0 = B;\n#pragma omp parallel\n")
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    return oracle.Oracle(oracle.compile_source(str(path), str(tmp_path / f"lib{name}.so")))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutant(tmp_path, name):
    mut = _mutant(tmp_path, name)
    worst = 0.0
    for case in CASES:
        B, Lq, H, D, lengths, bq, causal = case
        x = _f64_inputs(B, Lq, H, D, lengths, bq, causal, seed=len(lengths) + sum(lengths))
        o, lse = mut.fwd(x["q"], x["k"], x["v"], x["offsets"], Lq, bq, causal, x["scale"])
        dq, dk, dv = mut.bwd(x["q"], x["k"], x["v"], x["do"], x["offsets"], Lq, bq, causal, x["scale"])
        ref = brute_force(x["q"], x["k"], x["v"], x["do"], x["offsets"], Lq, bq, causal, x["scale"])
        for a, b in zip((o, lse, dq, dk, dv), ref):
            fin = torch.isfinite(a) & torch.isfinite(b)
            if not torch.equal(torch.isfinite(a), torch.isfinite(b)):
                worst = float("inf")
            elif fin.any():
                worst = max(worst, (a[fin] - b[fin]).abs().max().item())
    assert worst > 1e-6, f"mutant {name} survived the brute-force pin (max err {worst})"
