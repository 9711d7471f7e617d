"""Host-side check of the selection shortcut used by the expert kernels' top-6.

The kernels select the top-6 experts by an integer key built from the bf16
logit and the expert index, and fall back to comparing fp32 sigmoid scores
unless all 7 best candidates lie in the band 2^-12 <= |logit|, -80 < logit < 8.
The shortcut is exact only if, inside that band, the correctly rounded fp32
sigmoid is strictly increasing on the bf16 grid with a margin larger than the
error of CUDA's expf-based evaluation.  Both facts are checked here: the
margin exhaustively over every bf16 value, the selection by emulating it
against the oracle's definition.
"""

import numpy as np

import oracle as O


def _all_bf16_values():
    b = np.arange(65536, dtype=np.uint32)
    f = (b << 16).view(np.float32)
    return np.unique(f[np.isfinite(f)].astype(np.float64))


def test_sigmoid_margin_on_bf16_grid_inside_band():
    vals = _all_bf16_values()
    s = O.sigmoid_scores(vals).astype(np.float32)
    ulp = np.spacing(s).astype(np.float64)
    band = (np.abs(vals) >= 2.0 ** -12) & (vals > -80) & (vals < 8)
    idx = np.nonzero(band)[0]
    idx = idx[idx > 0]
    gap = (s[idx].astype(np.float64) - s[idx - 1].astype(np.float64)) / ulp[idx]
    assert gap.min() >= 4.0          # each value beats the next smaller bf16 value by >= 4 ulps
    # and the band is needed: just outside it distinct logits share a score
    outside = np.nonzero((vals > 0) & (vals < 2.0 ** -14))[0]
    assert np.any(s[outside][1:] == s[outside][:-1])


def _fast_select(bits):
    ordk = np.where(bits & 0x8000, (~bits) & 0xFFFF, bits | 0x8000).astype(np.int64)
    key = (ordk << 16) | (255 - np.arange(256))
    top = np.argsort(-key)[:7]
    mag = bits[top] & 0x7FFF
    band = (mag >= 0x3980) & np.where(bits[top] & 0x8000, mag < 0x42A0, mag < 0x4100)
    return top[:6], bool(band.all())


def test_key_selection_equals_sigmoid_topk_when_in_band():
    rng = np.random.default_rng(0)
    used = 0
    for trial in range(4000):
        kind = trial % 4
        if kind == 0:
            v = rng.standard_normal(256)
        elif kind == 1:
            v = rng.standard_normal(256) * 6
        elif kind == 2:
            v = np.round(rng.standard_normal(256) * 4) / 4   # many equal logits
        else:
            v = rng.standard_normal(256) * 1e-4               # near the excluded band
        bits = O.f64_to_bf16_bits(v).astype(np.int64)
        sel, ok = _fast_select(bits)
        ref = O.topk_desc(O.sigmoid_scores(O.bf16_bits_to_f64(bits))[None, :], 6)[0]
        if ok:
            used += 1
            assert list(sel) == list(ref), (trial, sel, ref)
    assert used > 1000
