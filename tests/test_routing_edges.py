"""GPU routing edge cases against the CPU oracle, through the C ABI.

* Exact ties.  Experts with identical router rows have identical logits for
  every token; the selection takes the lower expert index, as the oracle does.
  Inside the band where logit order equals score order both sides select by the
  same exact bf16 logits, so the ids must agree bit for bit, tie-breaks
  included, and some ties must straddle the 6th place.
* Logits outside that band.  Scaling the activations by 64 or by 2^-14 (a
  sublayer without RMSNorm) pushes the top logits above 8 or below 2^-12:
  decode then selects on the fp32 sigmoid scores, and the prefill router
  computes every logit exactly instead of only the candidates'.  The scores
  then tie widely (they saturate, or crowd around 1/2), so the oracle accepts
  any valid selection; prefill must still agree with decode exactly.
"""

import numpy as np
import pytest
import torch

import oracle as O
import synth
from flint_testlib import bf16_to_f64, check_layer, check_prefill, compare_routing
from moe_decode_router_gb300 import flint_moe as F

pytestmark = pytest.mark.gpu

# (a, b): expert b gets expert a's router row
TIED = [(3, 200), (5, 6), (17, 18), (40, 41), (64, 65), (90, 91), (100, 255), (120, 121),
        (130, 131), (150, 151), (160, 161), (170, 171), (180, 181), (190, 191), (210, 211), (7, 250)]


@pytest.fixture(scope="module")
def dev():
    F.load_library()
    return torch.device("cuda:0")


def _pack(plain, dev):
    L = F.pack_layer(plain, device=dev)
    torch.cuda.synchronize()
    return O.layer_from_tensors(plain), L


@pytest.fixture(scope="module")
def tied_layer(dev):
    plain = dict(synth.gen_layer(0, 0, device="cpu"))
    wr = plain["router_w"].clone()
    for a, b in TIED:
        wr[b] = wr[a]
    plain["router_w"] = wr
    return _pack(plain, dev)


@pytest.fixture(scope="module")
def plain_layer(dev):
    plain = synth.gen_layer(0, 0, device="cpu")
    assert plain["norm_w"] is None  # the scaling reaches the router unchanged
    return _pack(plain, dev)


def oracle_routing(x, lw):
    logits = O.router_logits(bf16_to_f64(x), lw.router_w)
    s, ids, w, gap = O.route(logits)
    return logits, dict(ids=ids, gap=gap, scores=s)


def in_fast_band(logits):
    """Per token: do the 7 largest logits lie where logit order is score order."""
    top = -np.sort(-logits, axis=1)[:, :7]
    return np.all((np.abs(top) >= 2.0 ** -12) & (top > -80) & (top < 8), axis=1)


def straddling_ties(ids):
    """Number of (token, pair) where exactly one expert of a tied pair is selected."""
    n = 0
    for row in ids:
        sel = set(int(i) for i in row)
        n += sum((a in sel) != (b in sel) for a, b in TIED)
    return n


def decode(L, x, dev):
    B = x.shape[0]
    xd = x.to(dev)
    y = torch.empty_like(xd)
    ids = torch.full((B, 6), -1, dtype=torch.int32, device=dev)
    w = torch.zeros((B, 6), dtype=torch.float32, device=dev)
    F.decode_layer(L, xd, y, F.alloc_workspace(F.W_NVFP4), ids, w)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    return y, ids.cpu().numpy(), w.cpu().numpy()


def prefill(L, x, dev):
    T = x.shape[0]
    xd = x.to(dev)
    y = torch.full_like(xd, float("nan"))
    ids = torch.full((T, 6), -1, dtype=torch.int32, device=dev)
    w = torch.zeros((T, 6), dtype=torch.float32, device=dev)
    F.prefill_layer(L, xd, y, F.alloc_workspace(F.W_NVFP4, T, device=dev), ids, w)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    return y, ids.cpu().numpy(), w.cpu().numpy()


def test_decode_exact_ties_break_to_lower_index(tied_layer, dev):
    lw, L = tied_layer
    for i in range(8):
        x = synth.gen_x(0, 8, index=300 + i)
        logits, ref = oracle_routing(x, lw)
        assert in_fast_band(logits).all()
        y, ids, w = decode(L, x, dev)
        assert np.array_equal(ids, ref["ids"]), (ids, ref["ids"])
        check_layer(bf16_to_f64(x), lw, bf16_to_f64(y), ids, w)


def test_prefill_exact_ties_break_to_lower_index(tied_layer, dev):
    lw, L = tied_layer
    x = synth.gen_x(0, 512, index=310)
    logits, ref = oracle_routing(x, lw)
    assert in_fast_band(logits).all()
    y, ids, w = prefill(L, x, dev)
    assert np.array_equal(ids, ref["ids"])
    assert straddling_ties(ref["ids"]) > 0  # some ties decided the 6th place
    st = check_prefill(x, lw, y, ids, w)
    print("ties straddling the 6th place:", straddling_ties(ids), st)


@pytest.mark.parametrize("scale", [64.0, 2.0 ** -14])
def test_decode_logits_outside_the_fast_band(plain_layer, dev, scale):
    lw, L = plain_layer
    x = synth.gen_x(0, 8, index=320) * scale  # exact in bf16: a power of two
    logits, _ = oracle_routing(x, lw)
    assert not in_fast_band(logits).any()
    y, ids, w = decode(L, x, dev)
    _, st = check_layer(bf16_to_f64(x), lw, bf16_to_f64(y), ids, w)
    print(f"scale {scale}:", st)


@pytest.mark.parametrize("scale", [64.0, 2.0 ** -14])
def test_prefill_logits_outside_the_fast_band(plain_layer, dev, scale):
    lw, L = plain_layer
    x = synth.gen_x(0, 96, index=330) * scale
    logits, ref = oracle_routing(x, lw)
    assert not in_fast_band(logits).any()
    y, ids, w = prefill(L, x, dev)
    compare_routing(ref, ids)
    # both paths select on exact bf16 logits with the same top-6: decode's
    # choice on the first 8 tokens must be prefill's, bit for bit
    _, ids_d, w_d = decode(L, x[:8], dev)
    assert np.array_equal(ids[:8], ids_d) and np.array_equal(w[:8], w_d)
    st = check_prefill(x, lw, y, ids, w)
    print(f"scale {scale}:", st)
