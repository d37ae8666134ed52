"""Pins of the oracle's MXFP8 variant (CPU only).

The MXFP8 forward quantizes P to FP8 on the fly with its scale factors next
to it (TLX porta l'attenzione jagged su Blackwell oltre FA4 con un terzo del
codice, section "The turning point"); the oracle's reading of that sentence
is written at the MXFP8 part of oracle/jfa_oracle.c.  What pins it here,
independently of the oracle's own arithmetic:

- E4M3 values: the format's published landmarks (1.0, the largest normal 448,
  the smallest normal 2^-6 and subnormal 2^-9, NaN), strict monotonicity, and
  every code surviving encode(value(code)).
- E4M3 rounding: for random and midpoint inputs, the encoder's choice equals a
  brute-force search for the nearest finite E4M3 value (ties to the even
  code), saturating at 448.
- The MX shared exponent: the block's largest magnitude divided by 2^X lands
  in E4M3's top binade [256, 512) -- checked as a property, X found by search.
- V quantization and P quantization against brute force built from the two
  checks above (sequence-relative chunks of 32, scale code X + 127).
- The quantized P equals what an online softmax with an integer running
  maximum produces block by block (the schedule a kernel runs), whatever
  the order in which the maximum grows.
- The MXFP8 forward equals the plain attention oracle where quantization is
  lossless (V exactly representable, every weight 1.5 * 2^k), has the bf16
  forward's LSE, and matches a brute-force restatement on small random cases.
- Planted mistakes in a copy of the oracle's source (rounding ties away,
  ceil for floor, shifted exponent, missing saturation, swapped chunk scales,
  chunks counted from the packed row instead of the sequence) are each
  rejected by at least one pin.
"""
import math
import os

import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "jfa_oracle.c")


@pytest.fixture(scope="module")
def orc():
    return oracle._default()


def _finite_table(orc):
    codes = torch.arange(256, dtype=torch.int64).to(torch.uint8)
    vals = orc.e4m3_value(codes)
    keep = torch.isfinite(vals)
    return codes[keep].to(torch.int64), vals[keep]


def brute_e4m3(orc, x):
    """Nearest finite E4M3 value to each x by exhaustive search (ties: even code), clamped to +-448."""
    codes, vals = _finite_table(orc)
    x = torch.as_tensor(x, dtype=torch.float64).reshape(-1)
    xc = x.clamp(-448.0, 448.0)
    dist = (vals[None, :] - xc[:, None]).abs()
    best = dist.min(dim=1, keepdim=True).values
    cand = (dist == best)
    # among equally near candidates prefer an even code; keep the sign of x for zero
    even = (codes % 2 == 0)[None, :]
    pick = torch.where((cand & even).any(dim=1, keepdim=True), cand & even, cand)
    res = torch.gather(vals[None, :].expand_as(dist), 1, pick.to(torch.int64).argmax(dim=1, keepdim=True)).squeeze(1)
    return torch.where(res == 0, torch.copysign(torch.zeros_like(res), x), res)


def mx_exponent_by_search(amax):
    """The integer X with 256 <= amax / 2^X < 512, found by stepping (no logarithm)."""
    X = 0
    while amax / 2.0 ** X >= 512:
        X += 1
    while amax / 2.0 ** X < 256:
        X -= 1
    return max(-127, min(127, X))


# ---------------------------------------------------------------------------
# pins, each a function of an oracle instance (reused on planted mutants)
# ---------------------------------------------------------------------------
def pin_e4m3_landmarks(orc):
    v = orc.e4m3_value(torch.tensor([0x38, 0x7E, 0x08, 0x01, 0x00, 0x80, 0xFE, 0x07], dtype=torch.uint8))
    assert v.tolist()[:5] == [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, 0.0]
    assert math.copysign(1.0, v[5].item()) < 0 and v[6].item() == -448.0 and v[7].item() == 7 * 2.0 ** -9
    assert torch.isnan(orc.e4m3_value(torch.tensor([0x7F, 0xFF], dtype=torch.uint8))).all()
    pos = orc.e4m3_value(torch.arange(0x7F, dtype=torch.int64).to(torch.uint8))
    assert (pos[1:] > pos[:-1]).all()
    neg = orc.e4m3_value(torch.arange(0x80, 0xFF, dtype=torch.int64).to(torch.uint8))
    assert torch.equal(neg.abs(), pos)


def pin_e4m3_round_trip(orc):
    codes, vals = _finite_table(orc)
    assert torch.equal(orc.e4m3_encode(vals).to(torch.int64), codes)


def pin_e4m3_nearest_even(orc):
    g = torch.Generator().manual_seed(5)
    mag = torch.exp2(torch.empty(20000, dtype=torch.float64).uniform_(-13, 9.3, generator=g))
    sign = torch.where(torch.rand(20000, generator=g) < 0.5, -1.0, 1.0).to(torch.float64)
    _, vals = _finite_table(orc)
    pos = vals[vals > 0].sort().values
    mids = torch.cat([(pos[1:] + pos[:-1]) / 2, torch.tensor([2.0 ** -10])])
    x = torch.cat([sign * mag, mids, -mids, torch.tensor([448.0, 449.0, 463.9, 464.0, 470.0, 1e6, 0.0, -0.0])])
    got = orc.e4m3_value(orc.e4m3_encode(x))
    want = brute_e4m3(orc, x)
    assert torch.equal(got, want)
    assert torch.equal(torch.signbit(got), torch.signbit(x))


def pin_mx_exponent(orc):
    g = torch.Generator().manual_seed(6)
    for a in torch.exp2(torch.empty(2000, dtype=torch.float64).uniform_(-110, 110, generator=g)).tolist():
        X = orc.mx_exponent(a)
        assert 256 <= a / 2.0 ** X < 512, (a, X)
    for a in [1.0, 256.0, 511.999, 512.0, 2.0 ** -8, 3.0]:
        assert orc.mx_exponent(a) == mx_exponent_by_search(a)
    assert orc.mx_exponent(0.0) == -127


def _seqs(lengths):
    off = [0]
    for L in lengths:
        off.append(off[-1] + L)
    return torch.tensor(off, dtype=torch.int32)


def pin_quantize_v(orc):
    lengths = [5, 0, 37, 128, 129, 300]
    off = _seqs(lengths)
    N, H, D = int(off[-1]), 2, 8
    g = torch.Generator().manual_seed(7)
    v = (torch.randn(N, H, D, generator=g) * torch.exp2(torch.randint(-6, 7, (N, 1, 1), generator=g))).to(torch.bfloat16)
    v[40:45] = 0  # an all-zero chunk somewhere
    v8, vs = orc.quantize_v_mxfp8(v, off)
    vd = v.to(torch.float64)
    nb = 0
    for b, L in enumerate(lengths):
        o0 = int(off[b])
        for n in range((L + 127) // 128):
            for c in range(4):
                j0, j1 = 128 * n + 32 * c, min(128 * n + 32 * c + 32, L)
                for h in range(H):
                    for d in range(D):
                        code = int(vs[nb + n, h, d, c])
                        if j0 >= j1:
                            assert code == 0
                            continue
                        col = vd[o0 + j0:o0 + j1, h, d]
                        amax = col.abs().max().item()
                        X = mx_exponent_by_search(amax) if amax > 0 else -127
                        assert code == X + 127, (b, n, c, h, d)
                        want = brute_e4m3(orc, col / 2.0 ** X)
                        got = orc.e4m3_value(v8[o0 + j0:o0 + j1, h, d])
                        assert torch.equal(got, want), (b, n, c, h, d)
        nb += (L + 127) // 128
    assert vs.shape[0] == nb


def brute_quantize_p(orc, x):
    """Per chunk of 32 from index 0: X from the top-binade property of max 2^x, brute-force rounding."""
    x = torch.as_tensor(x, dtype=torch.float64)
    out = torch.zeros_like(x)
    for c0 in range(0, x.numel(), 32):
        xs = x[c0:c0 + 32]
        fin = torch.isfinite(xs)
        if not fin.any():
            continue
        mx = xs[fin].max().item()
        X = 0
        while mx - X >= 9:
            X += 1
        while mx - X < 8:
            X -= 1
        y = torch.where(fin, torch.exp2(xs - X), torch.zeros_like(xs))
        out[c0:c0 + 32] = brute_e4m3(orc, y) * 2.0 ** X
    return out


def pin_quantize_p(orc):
    g = torch.Generator().manual_seed(8)
    for n in [1, 31, 32, 33, 64, 100, 200]:
        for trial in range(3):
            x = torch.empty(n, dtype=torch.float64).uniform_(-20, 12, generator=g)
            x[torch.rand(n, generator=g) < 0.15] = -math.inf
            got = orc.mx_quantize_p(x)
            want = brute_quantize_p(orc, x)
            assert torch.allclose(got, want, rtol=1e-12, atol=0), (n, trial)


def _lossless_inputs(orc, lengths, Lq, H, broadcast_q, seed):
    """D = 2 inputs whose log2-domain logits are exactly (up to fp64 rounding) 0.585 + integers, so every
    weight 2^(x - X) is 1.5 * 2^k, and V whose every 32-key chunk has amax in [1, 2) built from E4M3 values:
    MXFP8 quantization of both P and V is then lossless."""
    g = torch.Generator().manual_seed(seed)
    off = _seqs(lengths)
    N, D = int(off[-1]), 2
    alpha = math.log2(1.5)
    ln2 = math.log(2.0)
    scale = 1.0
    nq = Lq if broadcast_q else N
    cq = torch.randint(0, 3, (nq, H), generator=g).to(torch.float64)
    q = torch.stack([torch.ones(nq, H, dtype=torch.float64), cq], dim=-1)
    gk = torch.randint(-6, 1, (N, H), generator=g).to(torch.float64)
    hk = torch.randint(-2, 1, (N, H), generator=g).to(torch.float64)
    k = torch.stack([(alpha + gk) * ln2, hk * ln2], dim=-1)
    # V: E4M3 values of magnitude <= 1.75, one entry of magnitude 1 or 1.5 per 32-key chunk
    codes, vals = _finite_table(orc)
    small = vals[(vals.abs() <= 1.75) & (vals.abs() >= 2.0 ** -3)]
    v = small[torch.randint(0, small.numel(), (N, H, D), generator=g)]
    for b, L in enumerate(lengths):
        for j0 in range(0, L, 32):
            v[int(off[b]) + j0, :, :] = torch.where(torch.rand(H, D, generator=g) < 0.5, 1.0, -1.5).to(torch.float64)
    return q, k, v.to(torch.bfloat16), off, scale


def pin_fwd_lossless(orc):
    for lengths, Lq, bq, causal in [([0, 1, 40, 130, 300], 3, True, False), ([33, 0, 129, 64], 0, False, True),
                                    ([200, 7], 0, False, False)]:
        H = 2
        q, k, v, off, scale = _lossless_inputs(orc, lengths, Lq, H, bq, seed=len(lengths) + Lq)
        v8, vs = orc.quantize_v_mxfp8(v, off)
        assert torch.equal(orc.e4m3_value(v8) * 0 + 1, torch.ones(v8.shape, dtype=torch.float64))  # all finite
        o, lse = orc.fwd_mxfp8(q, k, v8, vs, off, Lq, bq, causal, scale)
        o_ref, lse_ref = orc.fwd(q, k, v.to(torch.float64), off, Lq, bq, causal, scale)
        assert torch.allclose(o, o_ref, rtol=0, atol=1e-12), (lengths, (o - o_ref).abs().max())
        assert torch.equal(torch.isfinite(lse), torch.isfinite(lse_ref))
        fin = torch.isfinite(lse_ref)
        assert torch.allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-12)


def pin_fwd_brute_force(orc):
    for lengths, Lq, bq, causal in [([70, 0, 33], 5, True, False), ([45, 130], 0, False, True)]:
        H, D = 2, 4
        g = torch.Generator().manual_seed(11)
        off = _seqs(lengths)
        N = int(off[-1])
        q = torch.randn(Lq if bq else N, H, D, generator=g).to(torch.bfloat16)
        k = torch.randn(N, H, D, generator=g).to(torch.bfloat16)
        v = torch.randn(N, H, D, generator=g).to(torch.bfloat16)
        scale = 0.9
        v8, vs = orc.quantize_v_mxfp8(v, off)
        o, lse = orc.fwd_mxfp8(q, k, v8, vs, off, Lq, bq, causal, scale)
        qd, kd = q.to(torch.float64), k.to(torch.float64)
        nb = 0
        for b, L in enumerate(lengths):
            o0 = int(off[b])
            # dequantized V of this sequence from its codes and chunk scales
            vdeq = torch.zeros(L, H, D, dtype=torch.float64)
            for j in range(L):
                sc = vs[nb + j // 128, :, :, (j % 128) // 32].to(torch.float64) - 127
                vdeq[j] = orc.e4m3_value(v8[o0 + j]) * torch.exp2(sc)
            nb += (L + 127) // 128
            for h in range(H):
                rows = range(Lq if bq else L)
                for i in rows:
                    qi = qd[i if bq else o0 + i, h]
                    s = scale * (kd[o0:o0 + L, h] @ qi)
                    if causal:
                        s[i + 1:] = -math.inf
                    x = s / math.log(2.0)
                    orow = (b, i, h) if bq else (o0 + i, h)
                    if L == 0 or not torch.isfinite(x).any():
                        assert torch.all(o[orow] == 0)
                        continue
                    R = math.floor(x[torch.isfinite(x)].max().item())
                    pq = brute_quantize_p(orc, x - R)
                    den = torch.exp2(x - R).sum()
                    want = (pq[:, None] * vdeq[:, h]).sum(0) / den
                    assert torch.allclose(o[orow], want, rtol=1e-9, atol=1e-12), (b, h, i)


def pin_lse_is_the_bf16_forwards(orc):
    lengths, H, D = [50, 0, 140], 2, 8
    g = torch.Generator().manual_seed(12)
    off = _seqs(lengths)
    N = int(off[-1])
    q = torch.randn(6, H, D, generator=g).to(torch.bfloat16)
    k = torch.randn(N, H, D, generator=g).to(torch.bfloat16)
    v = torch.randn(N, H, D, generator=g).to(torch.bfloat16)
    v8, vs = orc.quantize_v_mxfp8(v, off)
    _, lse = orc.fwd_mxfp8(q, k, v8, vs, off, 6, True, False, 0.3)
    _, lse_ref = orc.fwd(q, k, v, off, 6, True, False, 0.3)
    assert torch.equal(lse, lse_ref)


def online_quantize_p(orc, x, threshold=8.0):
    """The schedule a kernel runs: 128-key blocks in order, a running maximum kept at an integer m (the
    ceiling of the first block's maximum, raised to the ceiling of a new maximum only when that exceeds m by
    more than `threshold`), and per 32-key chunk the exponent e = floor(chunk max - m) - 8 applied to
    2^(x - m); returns the absolute weights 2^(m + e) E4M3(2^(x - m - e)) for every key."""
    x = torch.as_tensor(x, dtype=torch.float64)
    out = torch.zeros_like(x)
    m = None
    for j0 in range(0, x.numel(), 128):
        blk = x[j0:j0 + 128]
        fin = torch.isfinite(blk)
        if fin.any():
            bm = blk[fin].max().item()
            if m is None:
                m = math.ceil(bm)
            elif bm > m + threshold:
                m = math.ceil(bm)
        if m is None:
            continue
        for c0 in range(0, blk.numel(), 32):
            ch = blk[c0:c0 + 32]
            cf = torch.isfinite(ch)
            if not cf.any():
                continue
            e = math.floor(ch[cf].max().item() - m) - 8
            y = torch.where(cf, torch.exp2(ch - m - e), torch.zeros_like(ch))
            out[j0 + c0:j0 + c0 + 32] = orc.e4m3_value(orc.e4m3_encode(y)) * 2.0 ** (m + e)
    return out


def pin_online_schedule_invariance(orc):
    """The oracle's quantized P (one exponent per chunk from floor(chunk max) - 8) is what an online softmax
    with an integer running max produces, whatever the order in which the maximum grows: rows whose maxima
    rise over the blocks (so the running max is stale or raised), fall, or jump by more than 8."""
    g = torch.Generator().manual_seed(14)
    for trial in range(12):
        n = int(torch.randint(1, 700, (1,), generator=g))
        ramp = torch.linspace(0, float(torch.empty(1).uniform_(-30, 30, generator=g)), n, dtype=torch.float64)
        x = torch.empty(n, dtype=torch.float64).uniform_(-12, 4, generator=g) + ramp
        x[torch.rand(n, generator=g) < 0.1] = -math.inf
        want = orc.mx_quantize_p(x)
        got = online_quantize_p(orc, x)
        assert torch.allclose(got, want, rtol=1e-12, atol=0), trial


PINS = [pin_e4m3_landmarks, pin_e4m3_round_trip, pin_e4m3_nearest_even, pin_mx_exponent, pin_quantize_v,
        pin_quantize_p, pin_online_schedule_invariance, pin_fwd_lossless, pin_fwd_brute_force,
        pin_lse_is_the_bf16_forwards]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


def test_slack_marks_boundaries_only(orc):
    """Far from any boundary the slack is 0; a logit 1e-6 from a rounding midpoint or a chunk maximum 1e-6
    from an integer gets a slack of the other side's change."""
    g = torch.Generator().manual_seed(13)
    x = torch.empty(64, dtype=torch.float64).uniform_(-6, 0, generator=g)
    x[0] = 0.5
    _, sl = orc.mx_quantize_p(x, want_slack=True)
    near = (sl > 0).sum().item()
    assert near <= 2  # random logits: almost never within 1e-4
    # chunk maximum 0.5 gives X = -8; 2^(x + 8) = 272 (1 + 1e-7) sits just above the midpoint of the
    # E4M3 values 256 and 288, so the other side is one step (32 * 2^-8) down
    _, sl = orc.mx_quantize_p(torch.tensor([0.5, math.log2(272.0 * (1 + 1e-7)) - 8]), want_slack=True)
    assert sl[1].item() == pytest.approx(32 * 2.0 ** -8) and sl[0].item() == 0
    # chunk maximum 1e-6 below an integer: on the other side X is one higher, and the maximum (saturated
    # to 448 here) becomes 256 of the coarser scale; elements inside a binade keep their absolute grid
    _, sl = orc.mx_quantize_p(torch.tensor([1.0 - 1e-6, -2.3]), want_slack=True)
    assert sl[0].item() == pytest.approx(2.0 - 1.75) and sl[1].item() == 0


MUTATIONS = {
    "rounding_ties_away": ("const double r = ldexp(nearbyint(ldexp(a, -q)), q);",
                           "const double r = ldexp(round(ldexp(a, -q)), q);"),
    "p_exponent_ceil": ("const double f = floor(mx);", "const double f = ceil(mx);"),
    "mx_exponent_off_by_one": ("int X = ex - 1 - 8;", "int X = ex - 8;"),
    "no_saturation": ("if (a >= 448.0) return sign | 0x7E;", "if (a >= 480.0) return sign | 0x7E;"),
    "chunk_scales_swapped": ("v_scale[(((bstart[b] + j / 128) * H + h) * (int64_t)D + d) * 4 + (j % 128) / 32];",
                             "v_scale[(((bstart[b] + j / 128) * H + h) * (int64_t)D + d) * 4 + 3 - (j % 128) / 32];"),
    "v_chunks_from_packed_row": ("const int j0 = 128 * n + 32 * c, j1 = j0 + 32 < Lk ? j0 + 32 : Lk;",
                                 "const int j0 = 128 * n + 32 * c - offsets[b] % 32 > 0 ? 128 * n + 32 * c - offsets[b] % 32 : 0,"
                                 " j1 = 128 * n + 32 * c + 32 - offsets[b] % 32 < Lk ? 128 * n + 32 * c + 32 - offsets[b] % 32 : Lk;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mxfp8_mutant(tmp_path, name):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(before, after))
    mut = oracle.Oracle(oracle.compile_source(str(path), str(tmp_path / f"lib{name}.so")))
    failed = []
    for pin in PINS:
        try:
            pin(mut)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin rejects the {name} mutant"
