"""Pins for the CPU oracle against things other than itself.

Each test ties one oracle function to a fact the oracle cannot produce on its
own: a value worked by hand from the format definitions (golden files), a
library routine (torch's float8/bf16 casts, scipy's expit, integer matmul),
a closed form, an invariant, or brute force on tiny inputs.  The set is chosen
so that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one test.
"""

import itertools
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------- formats

def test_e2m1_table_matches_spec():
    rows = _read_golden("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        v = O.e2m1_value(int(code, 16))
        want = float(val)
        assert v == want and math.copysign(1.0, v) == math.copysign(1.0, want), (code, v, want)


def test_e4m3_table_matches_torch_float8():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = O.E4M3_LUT
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(ours[ok]))


def test_nvfp4_hand_worked_examples():
    rows = _read_golden("nvfp4_examples.txt")
    assert len(rows) >= 10
    for code, scale, ts, val in rows:
        c = int(code, 16)
        codes = np.array([[c | (c << 4)] * 8], dtype=np.uint8)  # 16 elements, both nibbles
        scales = np.array([[int(scale, 16)]], dtype=np.uint8)
        got = O.dequant_nvfp4(codes, scales, float(ts))
        assert got.shape == (1, 16)
        want = float(val)
        if math.isnan(want):
            assert np.all(np.isnan(got))
        else:
            assert np.allclose(got, want, rtol=1e-15, atol=0), (code, scale, got[0, 0], want)
            assert np.all(np.signbit(got) == (math.copysign(1.0, want) < 0))


def test_dequant_nibble_order_and_block_boundaries():
    # row of 32 elements: byte j = (hi=code of element 2j+1, lo=code of element 2j)
    codes = np.zeros((1, 16), dtype=np.uint8)
    codes[0, 0] = 0x71          # element 0 -> code 1 (0.5), element 1 -> code 7 (6)
    codes[0, 7] = 0x20          # element 14 -> 0, element 15 -> code 2 (1)
    codes[0, 8] = 0x0A          # element 16 -> code A (-1), element 17 -> 0
    scales = np.array([[0x38, 0x40]], dtype=np.uint8)  # block 0 x1, block 1 x2
    w = O.dequant_nvfp4(codes, scales, 1.0)[0]
    assert w[0] == 0.5 and w[1] == 6.0 and w[15] == 1.0 and w[14] == 0.0
    assert w[16] == -2.0 and w[17] == 0.0
    assert np.count_nonzero(w) == 4


# --------------------------------------------------------------------------- rounding

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(1_000_000).astype(np.float32) * np.float32(3.0)
    # exact halfway cases: bf16 value + half an ulp, both parities
    base = rng.standard_normal(20000).astype(np.float32)
    b = (base.view(np.uint32) & np.uint32(0xFFFF0000))
    half = (b | np.uint32(0x8000)).view(np.float32)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, 1e-40, -1e-40, 3.3895e38, 1.0, 65504.0],
                        dtype=np.float32)
    allv = np.concatenate([x, half, specials])
    ours = O.f64_to_bf16_bits(allv.astype(np.float64))
    ref = torch.from_numpy(allv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    nanb = O.f64_to_bf16_bits(np.array([np.nan]))
    assert np.isnan(O.bf16_bits_to_f64(nanb))[0]


def test_round_f32_is_nearest_even():
    one = 1.0
    ulp = 2.0 ** -23
    assert O.round_f32(one + ulp / 2) == one            # tie to even (1.0)
    assert O.round_f32(one + 1.5 * ulp) == one + 2 * ulp  # tie to even (odd -> up)
    assert O.round_f32(one + 0.51 * ulp) == one + ulp


def _exact_round_to_f32(q):
    """Nearest fp32 (ties to even) of a rational, by exact integer arithmetic."""
    from fractions import Fraction
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(Fraction(q))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                       # subnormals share the smallest exponent's spacing
    scaled = a / Fraction(2) ** (e - 23)   # significand with 23 fraction bits
    m, rem = divmod(scaled.numerator, scaled.denominator)
    twice = 2 * rem
    if twice > scaled.denominator or (twice == scaled.denominator and m % 2 == 1):
        m += 1
    return sign * float(Fraction(m) * Fraction(2) ** (e - 23))


def test_round_sum_f32_equals_exact_rational_rounding():
    from fractions import Fraction
    rng = np.random.default_rng(12)
    cases = []
    # a sum whose float64 rounding lands on an fp32 midpoint: fsum alone would tie to even
    cases.append([1.0, 2.0 ** -8, 2.0 ** -24, 2.0 ** -60])
    cases.append([1.0, 2.0 ** -8, 2.0 ** -24, -(2.0 ** -60)])
    cases.append([1.0, 2.0 ** -24])                     # an exact midpoint: ties to even
    cases.append([1.0, 3 * 2.0 ** -24])                 # an exact midpoint, odd side
    cases.append([2.0 ** 60, 1.0, -(2.0 ** 60)])        # cancellation
    cases.append([1e-45, 1e-46])                        # fp32 subnormal range
    for _ in range(300):
        n = int(rng.integers(2, 40))
        t = O.round_bf16(rng.standard_normal(n)) * O.round_bf16(rng.standard_normal(n))
        t *= np.exp2(rng.integers(-30, 30, size=n))
        cases.append(list(t))
    for _ in range(300):  # sums placed on an fp32 midpoint, nudged by a tiny term either way
        base = float(np.float32(rng.standard_normal()))
        ulp = float(np.spacing(np.float32(base)))
        tiny = float(rng.choice([-1.0, 0.0, 1.0])) * abs(base) * 2.0 ** -70
        cases.append([base, ulp / 2, tiny])
    for terms in cases:
        want = _exact_round_to_f32(sum(Fraction(x) for x in terms))
        got = O.round_sum_f32(terms)
        assert got == want, (terms, got, want)


def test_router_logits_round_the_exact_sum_not_a_float64_sum():
    """logit = bf16(fp32(S)) of the exact sum S = 1 + 2^-8 + 2^-24 + 2^-60.  fp32(S) is
    1 + 2^-8 + 2^-23 (S is just above the fp32 midpoint 1 + 2^-8 + 2^-24), whose bf16
    rounding is 1 + 2^-7.  A float64 sum loses the 2^-60 term, lands on the midpoint,
    ties to 1 + 2^-8 in fp32 and to 1.0 in bf16."""
    x = np.array([[1.0, 2.0 ** -8, 2.0 ** -24, 2.0 ** -60]])
    W = np.ones((1, 4))
    assert O.router_logits(x, W)[0, 0] == 1.0 + 2.0 ** -7
    naive = O.round_bf16(O.round_f32(((1.0 + 2.0 ** -8) + 2.0 ** -24) + 2.0 ** -60))
    assert naive == 1.0  # the pin separates the exact definition from a float64 sum
    # the same terms spread over 2048 columns and 3 experts, in another order
    big = np.zeros((2, 2048))
    big[0, [5, 700, 1500, 2047]] = [2.0 ** -60, 2.0 ** -24, 1.0, 2.0 ** -8]
    big[1, 0] = 3.0
    Wb = np.zeros((3, 2048))
    Wb[1, :] = 1.0
    Wb[2, 0] = 2.0
    got = O.router_logits(big, Wb)
    assert got[0, 1] == 1.0 + 2.0 ** -7 and got[0, 0] == 0.0 and got[0, 2] == 0.0
    assert got[1, 1] == 3.0 and got[1, 2] == 6.0


def test_router_logits_match_exact_rounding_on_random_rows():
    from fractions import Fraction
    rng = np.random.default_rng(13)
    xh = O.round_bf16(rng.standard_normal((3, 256)))
    W = O.round_bf16(rng.standard_normal((8, 256)) / 16)
    got = O.router_logits(xh, W)
    for t in range(3):
        for e in range(8):
            s = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xh[t], W[e]))
            assert got[t, e] == O.round_bf16(_exact_round_to_f32(s))


# --------------------------------------------------------------------------- GEMV special cases

def _int_nvfp4(rng, n, k):
    """Codes in {0, +1, -1} with scale 1.0: every weight is a small integer."""
    vals = rng.integers(-1, 2, size=(n, k))
    code = np.where(vals == 1, 0x2, np.where(vals == -1, 0xA, 0x0)).astype(np.uint8)
    codes = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    scales = np.full((n, k // 16), 0x38, dtype=np.uint8)
    return vals, codes, scales


def test_gate_up_and_down_exact_on_integer_weights():
    rng = np.random.default_rng(2)
    H, I = 256, 64
    vals_gu, c_gu, s_gu = _int_nvfp4(rng, 2 * I, H)
    vals_d, c_d, s_d = _int_nvfp4(rng, H, I)
    x = rng.integers(-3, 4, size=(5, H))
    h = rng.integers(-2, 3, size=(5, I))
    g, u = O.expert_gate_up(x.astype(np.float64), O.dequant_nvfp4(c_gu, s_gu, 1.0))
    ref = x @ vals_gu.T  # int64 matmul
    assert np.array_equal(g, ref[:, :I].astype(np.float64))
    assert np.array_equal(u, ref[:, I:].astype(np.float64))
    d = O.expert_down(h.astype(np.float64), O.dequant_nvfp4(c_d, s_d, 1.0))
    assert np.array_equal(d, (h @ vals_d.T).astype(np.float64))


def test_router_logits_exact_on_integers_and_transposition():
    rng = np.random.default_rng(3)
    W = rng.integers(-4, 5, size=(16, 64))
    x = rng.integers(-2, 3, size=(3, 64))
    got = O.router_logits(x.astype(np.float64), W.astype(np.float64))
    assert got.shape == (3, 16)
    assert np.array_equal(got, (x @ W.T).astype(np.float64))  # |values| < 256: exact in bf16


def test_bf16_expert_matches_torch_matmul():
    rng = np.random.default_rng(4)
    wgu = torch.randn(2 * 64, 512, generator=torch.Generator().manual_seed(5)).mul(0.02).to(torch.bfloat16)
    x = torch.randn(3, 512, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    bits = wgu.view(torch.int16).numpy().view(np.uint16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    g, u = O.expert_gate_up(O.bf16_bits_to_f64(xb), O.bf16_bits_to_f64(bits))
    ref = torch.matmul(x.double(), wgu.double().T).float().double().numpy()
    assert np.array_equal(np.concatenate([g, u], axis=1), ref)
    del rng


# --------------------------------------------------------------------------- routing

def _brute_force_topk(s, k):
    """The unique k-subset S with (s_i > s_j) or (s_i == s_j and i < j) for all i in S, j not in S."""
    n = len(s)
    found = []
    for sub in itertools.combinations(range(n), k):
        S = set(sub)
        if all((s[i] > s[j]) or (s[i] == s[j] and i < j) for i in S for j in range(n) if j not in S):
            found.append(sub)
    assert len(found) == 1
    S = found[0]
    return sorted(S, key=lambda i: (-s[i], i))


@pytest.mark.parametrize("n,k", [(8, 2), (10, 3), (9, 6)])
def test_topk_matches_brute_force_with_ties(n, k):
    rng = np.random.default_rng(10 + n)
    for trial in range(300):
        if trial % 2:
            s = rng.integers(0, 4, size=n).astype(np.float64) / 4.0   # many ties
        else:
            s = rng.random(n)
        got = list(O.topk_desc(s[None, :], k)[0])
        assert got == _brute_force_topk(list(s), k), (s, got)


def test_sigmoid_and_routing_weights():
    lg = np.array([[0.0, 40.0, -40.0, 1.0, -1.0, 2.5, 3.0, -0.5, 0.25]])
    s = O.sigmoid_scores(lg)
    ref = expit(lg).astype(np.float32).astype(np.float64)
    assert np.array_equal(s, ref)
    assert s[0, 0] == 0.5 and s[0, 1] == 1.0
    rng = np.random.default_rng(7)
    logits = O.round_bf16(rng.standard_normal((64, 256)))
    s, ids, w, gap = O.route(logits, 6)
    assert ids.shape == (64, 6) and w.shape == (64, 6)
    for t in range(64):
        assert len(set(ids[t])) == 6
        sel = s[t, ids[t]]
        assert np.all(np.diff(sel) <= 0)                      # descending
        assert abs(np.sum(w[t]) - 1.0) <= 6 * 2.0 ** -24       # renormalised
        assert np.allclose(w[t], sel / sel.sum(), rtol=2 ** -23, atol=0)
        srt = np.sort(s[t])[::-1]
        assert gap[t] == srt[5] - srt[6]


def test_forced_ids_replace_selection():
    logits = O.round_bf16(np.linspace(-1, 1, 16))[None, :]
    s, ids, w, _ = O.route(logits, 6, forced={0: [0, 1, 2, 3, 4, 5]})
    assert list(ids[0]) == [0, 1, 2, 3, 4, 5]
    assert np.isclose(w[0].sum(), 1.0)


# --------------------------------------------------------------------------- SiLU and RMSNorm

def test_silu_mul_closed_forms():
    g = O.round_f32(np.array([0.0, 1.0, -1.0, 3.5, -20.0, 12.0]))
    assert np.all(O.silu_mul(g, np.zeros_like(g)) == 0.0)
    assert O.silu_mul(np.array([0.0]), np.array([5.0]))[0] == 0.0
    got = O.silu_mul(g, np.ones_like(g))
    ref = torch.from_numpy((g * expit(g)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, ref)
    # the gate is the argument of silu, the up projection the multiplier
    assert O.silu_mul(np.array([2.0]), np.array([3.0]))[0] != O.silu_mul(np.array([3.0]), np.array([2.0]))[0]


def test_rmsnorm_constant_vector_closed_form():
    for c in [0.5, 1.0, 3.0, 0.0078125, 100.0]:
        y = np.full((1, 2048), c)
        got = O.rmsnorm(y, np.ones(2048))
        want = c / math.sqrt(c * c + 1e-6)
        ulp = 2.0 ** (math.floor(math.log2(want)) - 7)
        assert np.all(np.abs(got - want) <= ulp), (c, got[0, 0], want)
        assert np.all(got == got[0, 0])


def test_rmsnorm_matches_torch_fp64():
    gen = torch.Generator().manual_seed(11)
    y = torch.randn(4, 2048, generator=gen).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(2048, generator=gen)).to(torch.bfloat16)
    yd, wd = y.double(), w.double()
    ref = (yd * torch.rsqrt(yd.pow(2).mean(-1, keepdim=True) + 1e-6) * wd).float().to(torch.bfloat16).double()
    got = O.rmsnorm(yd.numpy(), wd.numpy())
    diff = np.abs(got - ref.numpy())
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref.numpy()), 1e-30))) - 7)
    assert np.all(diff <= ulp)
    assert np.mean(diff == 0) > 0.99


# --------------------------------------------------------------------------- whole-layer invariants

def _tiny_layer(rng, H=64, I=32, E=16, norm=False, scale_range=(0x30, 0x40)):
    n = E + 1
    lw = O.LayerView(
        router_w=O.round_bf16(rng.standard_normal((E, H)) / math.sqrt(H)),
        norm_w=O.round_bf16(1 + 0.1 * rng.standard_normal(H)) if norm else None,
        fmt="nvfp4",
        gu_codes=rng.integers(0, 256, size=(n, 2 * I, H // 2), dtype=np.uint8),
        gu_scales=rng.integers(scale_range[0], scale_range[1] + 1, size=(n, 2 * I, H // 16), dtype=np.uint8),
        dn_codes=rng.integers(0, 256, size=(n, H, I // 2), dtype=np.uint8),
        dn_scales=rng.integers(scale_range[0], scale_range[1] + 1, size=(n, H, I // 16), dtype=np.uint8),
        tensor_scales=np.full((n, 2), 0.05),
    )
    return lw


def test_unselected_experts_contribute_exactly_nothing():
    rng = np.random.default_rng(20)
    lw = _tiny_layer(rng)
    x = O.round_bf16(rng.standard_normal((4, 64)))
    r = O.moe_layer(x, lw)
    sel = set(r["ids"].ravel().tolist())
    bad = O.LayerView(lw.router_w, None, "nvfp4", lw.gu_codes.copy(), lw.gu_scales.copy(),
                      lw.dn_codes.copy(), lw.dn_scales.copy(), lw.tensor_scales)
    for e in range(16):
        if e not in sel:
            bad.gu_scales[e] = 0x7F  # NaN
            bad.dn_scales[e] = 0x7F
            bad.gu_codes[e] = rng.integers(0, 256, size=bad.gu_codes[e].shape, dtype=np.uint8)
    r2 = O.moe_layer(x, bad)
    assert np.array_equal(r["y"], r2["y"])
    # poisoning a selected expert does change the output (the test can fail)
    e0 = int(r["ids"][0, 0])
    bad.dn_scales[e0] = 0x7F
    bad.drop_cache()
    assert np.isnan(O.moe_layer(x, bad)["y"][0]).any()


def test_identical_routed_experts_and_zero_shared_give_one_expert():
    rng = np.random.default_rng(21)
    lw = _tiny_layer(rng)
    for e in range(1, 16):
        lw.gu_codes[e] = lw.gu_codes[0]
        lw.gu_scales[e] = lw.gu_scales[0]
        lw.dn_codes[e] = lw.dn_codes[0]
        lw.dn_scales[e] = lw.dn_scales[0]
    lw.dn_scales[16] = 0x00  # shared expert's down projection is all zeros
    x = O.round_bf16(rng.standard_normal((6, 64)))
    r = O.moe_layer(x, lw)
    wgu, wd = lw.expert(0)
    g, u = O.expert_gate_up(x, wgu)
    want = O.round_bf16(O.expert_down(O.silu_mul(g, u), wd))
    diff = np.abs(r["y"] - want)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 1e-30))) - 7)
    assert np.all(diff <= ulp)                 # sum of weights is 1 up to fp32 rounding
    assert np.mean(diff == 0) > 0.99


def test_shared_expert_added_with_weight_one():
    rng = np.random.default_rng(22)
    lw = _tiny_layer(rng)
    lw.dn_scales[:16] = 0x00  # every routed expert outputs zero
    x = O.round_bf16(rng.standard_normal((3, 64)))
    r = O.moe_layer(x, lw)
    wgu, wd = lw.expert(16)
    g, u = O.expert_gate_up(x, wgu)
    want = O.round_bf16(O.expert_down(O.silu_mul(g, u), wd))
    assert np.array_equal(r["y"], want)
    assert np.any(want != 0)


def test_routed_weights_scale_expert_outputs():
    # two experts active per token is impossible with top-6 over 16, so check linearity:
    # doubling every routed expert's down projection (scale byte +1 exponent) with the
    # shared expert zeroed doubles y exactly.
    rng = np.random.default_rng(23)
    lw = _tiny_layer(rng)
    lw.dn_scales[16] = 0x00
    x = O.round_bf16(rng.standard_normal((3, 64)))
    y1 = O.moe_layer(x, lw)["y"]
    lw.dn_scales[:16] = lw.dn_scales[:16] + 0x08  # E4M3 exponent +1 (range stays normal)
    lw.drop_cache()
    y2 = O.moe_layer(x, lw)["y"]
    assert np.array_equal(y2, 2 * y1)


def test_prefill_equals_per_token_decode():
    rng = np.random.default_rng(24)
    lw = _tiny_layer(rng, norm=True)
    x = O.round_bf16(rng.standard_normal((40, 64)))
    a = O.moe_prefill(x, lw)
    lw.drop_cache()
    b = O.moe_layer(x, lw)
    assert np.array_equal(a["ids"], b["ids"])
    assert np.array_equal(a["y"], b["y"])


def test_stack_chains_through_norm_without_residual():
    rng = np.random.default_rng(25)
    l0 = _tiny_layer(rng, norm=False)
    l1 = _tiny_layer(rng, norm=True)
    x = O.round_bf16(rng.standard_normal((2, 64)))
    y, outs = O.moe_stack(x, [l0, l1])
    y0 = O.moe_layer(x, l0)["y"]
    assert np.array_equal(outs[1]["x_hat"], O.rmsnorm(y0, l1.norm_w))
    assert np.array_equal(y, O.moe_layer(y0, l1)["y"])


def test_full_size_layer_from_generator():
    import synth
    d = synth.gen_layer(0, 0, device="cpu")
    lw = O.layer_from_tensors(d)
    x = synth.gen_x(0, 1)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    r = O.moe_layer(O.bf16_bits_to_f64(xb), lw)
    assert r["y"].shape == (1, 2048) and np.all(np.isfinite(r["y"]))
    assert len(set(r["ids"][0].tolist())) == 6
    rms = np.sqrt(np.mean(r["y"] ** 2))
    assert 1e-3 < rms < 1e4


# --------------------------------------------------------------------------- dense GEMV

def test_dense_gemv_exact_on_integer_weights_and_transposition():
    """Codes in {0, +-1} with scale 1 and tensor scale 1: every product is a small
    integer, the fp32 sums are exact, and y must equal an int64 matmul (this also
    catches a transposed operand: N != K below)."""
    rng = np.random.default_rng(21)
    N, K = 48, 256
    vals, codes, scales = _int_nvfp4(rng, N, K)
    x = rng.integers(-3, 4, size=(5, K))
    y = O.dense_gemv(x.astype(np.float64), codes, scales, 1.0)
    assert y.shape == (5, N)
    ref = x @ vals.T
    assert np.all(np.abs(ref) < 256)  # exact in bf16
    assert np.array_equal(y, ref.astype(np.float64))


def test_dense_gemv_rounds_once_to_bf16_and_applies_the_tensor_scale():
    """Hand-worked row: 16 elements of code 0x7 (6.0) with block scale 0x40 (2.0) and
    tensor scale 0.5 give weights of 6; x = 1 at 16 columns sums to 96 (exact).  A
    second row of 0x1 (0.5) codes against x = 17 at one column gives 0.5 * 2 * 0.5 *
    17 = 8.5, and x = 257 at one column of weight 1 gives 257, which rounds to 256 in
    bf16 (ties to even)."""
    K = 256
    codes = np.zeros((3, K // 2), dtype=np.uint8)
    scales = np.full((3, K // 16), 0x38, dtype=np.uint8)  # 1.0
    codes[0, :8] = 0x77
    scales[0, 0] = 0x40
    codes[1, 0] = 0x01                                      # element 0 = 0.5
    scales[1, 0] = 0x40
    codes[2, 0] = 0x02                                      # element 0 = 1.0
    x = np.zeros((1, K))
    x[0, :16] = 1.0
    y = O.dense_gemv(x, codes, scales, 0.5)
    assert y[0, 0] == 96.0
    x2 = np.zeros((1, K))
    x2[0, 0] = 17.0
    assert O.dense_gemv(x2, codes, scales, 0.5)[0, 1] == 8.5
    x3 = np.zeros((1, K))
    x3[0, 0] = 257.0
    assert O.dense_gemv(x3, codes, scales, 1.0)[0, 2] == 256.0
