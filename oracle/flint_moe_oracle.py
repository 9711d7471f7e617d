"""Plain, slow, obviously-correct CPU definition of the Flint MoE sublayer.

TEST INFRASTRUCTURE: imported only by tests/, __graft_entry__.smoke() and the
CPU-baseline / reference arm of bench.py.  Nothing on the product path calls it.

What is computed (sources: "Day-0 Support for Flint on vLLM", hot.jian.ing
translation, sections "Model architecture" and "Optimizations"; the
yuxiaoba.github.io English commentary, section "Only 14 of 49 layers retain
full-history KV"):

  * a pre-norm MoE sublayer with hidden size 2048, 256 routed experts chosen
    by sigmoid top-6, and one always-on shared expert;
  * expert weights stored as NVIDIA NVFP4 blocks and run weight-only
    (W4A16): activations stay bf16 ("Model architecture", the paragraph on the
    GGUF NVFP4 checkpoint);
  * every kernel follows the reference implementation's rounding points
    (same paragraph, and "Optimizations": norm and SiLU kernels that follow
    the reference rounding).

The pages do not print the rounding points.  This oracle declares them
(readings, listed in the design notes): dot products accumulate exactly and
are rounded once to fp32; bf16 rounding (round-to-nearest-even, via fp32)
after the RMSNorm, after the router logits, after SiLU(gate)*up and after the
weighted combine.  Where a rounded sum decides an integer result (the router
logits that feed top-6, the RMSNorm scale) the oracle rounds the exact sum
itself (``round_sum_f32``); the expert GEMVs, whose results are only compared
within a tolerance, sum in fp64 before the one fp32 rounding.  Routing weights are the selected sigmoid scores
divided by their sum; the shared expert is added with weight 1; there is no
residual inside the sublayer.

All arithmetic is numpy float64 unless a step is declared fp32.  Arrays
holding bf16 data are passed either as float64 values or as uint16 bit
patterns (see ``bf16_bits_to_f64``).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "H", "E", "INTER", "TOP_K", "BLOCK", "RMS_EPS",
    "e2m1_value", "e4m3fn_value", "E2M1_LUT", "E4M3_LUT",
    "bf16_bits_to_f64", "round_f32", "round_bf16", "f64_to_bf16_bits", "round_sum_f32",
    "dequant_nvfp4", "rmsnorm", "router_logits", "sigmoid_scores",
    "topk_desc", "route", "silu_mul", "expert_gate_up", "expert_down",
    "LayerView", "layer_from_tensors", "moe_layer", "moe_stack", "moe_prefill", "dense_gemv",
]

H = 2048
E = 256
INTER = 512
TOP_K = 6
BLOCK = 16
RMS_EPS = 1e-6


# ----------------------------------------------------------------------------
# Number formats.  NVFP4 = blocks of 16 E2M1 codes sharing one E4M3 scale byte,
# plus one fp32 per-tensor scale ("Model architecture": the NVFP4 checkpoint's
# blocks use NVIDIA's NVFP4 format).  The element formats are the OCP
# Microscaling ones: E2M1 = sign, 2 exponent bits (bias 1), 1 mantissa bit, no
# inf/nan; E4M3FN = sign, 4 exponent bits (bias 7), 3 mantissa bits, no inf,
# S.1111.111 = NaN.
# ----------------------------------------------------------------------------

def e2m1_value(code):
    """Value of a 4-bit E2M1 code (bit 3 sign, bits 2..1 exponent, bit 0 mantissa)."""
    code = np.asarray(code, dtype=np.int64) & 0xF
    sign = np.where(code & 0x8, -1.0, 1.0)
    exp = (code >> 1) & 0x3
    man = (code & 0x1).astype(np.float64)
    # exponent field 0 is subnormal: man * 2^(1 - bias) * 2^-1 = man / 2
    mag = np.where(exp == 0, man * 0.5, (1.0 + man * 0.5) * np.exp2(exp.astype(np.float64) - 1.0))
    return sign * mag


def e4m3fn_value(byte):
    """Value of an OCP E4M3FN byte (bit 7 sign, bits 6..3 exponent, bits 2..0 mantissa)."""
    byte = np.asarray(byte, dtype=np.int64) & 0xFF
    sign = np.where(byte & 0x80, -1.0, 1.0)
    exp = (byte >> 3) & 0xF
    man = (byte & 0x7).astype(np.float64)
    sub = man / 8.0 * 2.0 ** (1 - 7)
    nrm = (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    val = sign * np.where(exp == 0, sub, nrm)
    return np.where((exp == 0xF) & ((byte & 0x7) == 0x7), np.nan, val)


E2M1_LUT = e2m1_value(np.arange(16))
E4M3_LUT = e4m3fn_value(np.arange(256))


# ----------------------------------------------------------------------------
# Rounding points
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits):
    """bf16 bit patterns (uint16/int16) -> float64 values (exact)."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_f32(x):
    """Round float64 values to the nearest fp32 (ties to even); returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """float64 -> fp32 (RNE) -> bf16 (RNE) bit patterns (uint16).  NaN stays NaN."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint32)
    nan = np.isnan(f)
    r = np.where(nan, ((u >> np.uint64(16)).astype(np.uint32) | np.uint32(0x40)), r)
    return r.astype(np.uint16)


def round_bf16(x):
    """Round float64 values to bf16 through fp32 (each step ties-to-even)."""
    return bf16_bits_to_f64(f64_to_bf16_bits(x))


def round_sum_f32(terms):
    """The fp32 value nearest the exact sum of `terms` (float64 values), ties to even.

    math.fsum gives d, the float64 nearest the exact sum S.  Rounding d to fp32
    gives the fp32 nearest S except where d is exactly halfway between two fp32
    values while S is not (double rounding): S < m implies d <= m for every
    fp32 midpoint m, since m is itself a float64.  In that case the sign of the
    exact residual S - d (fsum of the terms and -d, whose sign is exact) picks
    the side.
    """
    terms = [float(t) for t in np.ravel(terms)]
    d = math.fsum(terms)
    f = np.float32(d)
    if float(f) == d or not np.isfinite(f):
        return float(f)
    if float(f) < d:
        lo, hi = f, np.nextafter(f, np.float32(np.inf))
    else:
        lo, hi = np.nextafter(f, np.float32(-np.inf)), f
    if d - float(lo) != float(hi) - d:
        return float(f)
    r = math.fsum(terms + [-d])
    if r > 0:
        return float(hi)
    if r < 0:
        return float(lo)
    return float(f)


# ----------------------------------------------------------------------------
# NVFP4 dequantisation
# ----------------------------------------------------------------------------

def dequant_nvfp4(codes, scales, tensor_scale):
    """Element [n, k] = e2m1(code[n, k]) * e4m3(scale[n, k // 16]) * tensor_scale.

    codes  uint8 [N, K/2]: byte j holds element 2j in its low nibble and 2j+1 in
           its high nibble (the plain NVFP4 layout the packer reads);
    scales uint8 [N, K/16]: one E4M3 byte per 16 consecutive elements of a row.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    n, kh = codes.shape
    vals = np.empty((n, 2 * kh), dtype=np.float64)
    vals[:, 0::2] = E2M1_LUT[codes & 0xF]
    vals[:, 1::2] = E2M1_LUT[codes >> 4]
    blk = np.repeat(E4M3_LUT[scales], BLOCK, axis=1)
    assert blk.shape == vals.shape
    return vals * blk * float(tensor_scale)


# ----------------------------------------------------------------------------
# Sublayer steps
# ----------------------------------------------------------------------------

def rmsnorm(y, w, eps=RMS_EPS):
    """Pre-norm between stacked sublayers ("Model architecture": a 49-layer pre-norm
    MoE; "Optimizations": norm kernels that follow the reference rounding).

    Declared steps: mean of squares = exact sum / H rounded once to fp32;
    r = 1 / sqrt(mean + eps) with each fp32 operation correctly rounded;
    x_hat = bf16( fp32( fp32(y * r) * w ) ).
    y [B, H] and w [H] hold bf16 values as float64.
    """
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    # the exact sum of the exact squares, rounded once to fp32; / H is exact (H = 2^11)
    ss = np.array([round_sum_f32(row * row) for row in y])
    ms = (ss / y.shape[-1]).astype(np.float32)
    r = np.float32(1.0) / np.sqrt(ms + np.float32(eps))
    t = y.astype(np.float32) * r[:, None]
    xh = t * np.asarray(w, dtype=np.float64).astype(np.float32)[None, :]
    return round_bf16(xh.astype(np.float64))


def router_logits(xh, router_w):
    """Router GEMV over the 256 experts: logit = bf16(fp32(sum_k x_hat[k] * W_r[e, k])),
    the sum exact before its one rounding to fp32.

    Products of bf16 values are exact in float64.  A float64 matrix product
    approximates each sum S within gamma * sum|products| for any summation
    order (gamma = n * 2^-53 / (1 - n * 2^-53), taken here as (n + 2) * 2^-52);
    where every value of that interval rounds to the same fp32, that fp32 is
    the rounding of S.  The few sums whose interval holds an fp32 rounding
    boundary are rounded exactly with ``round_sum_f32``.
    """
    xh = np.atleast_2d(np.asarray(xh, np.float64))
    w = np.asarray(router_w, np.float64)
    approx = xh @ w.T
    bound = (np.abs(xh) @ np.abs(w).T) * ((xh.shape[1] + 2) * 2.0 ** -52)
    with np.errstate(over="ignore"):
        lo = (approx - bound).astype(np.float32)
        hi = (approx + bound).astype(np.float32)
    out = lo.astype(np.float64)
    for t, e in zip(*np.nonzero(lo != hi)):
        out[t, e] = round_sum_f32(xh[t] * w[e])
    return round_bf16(out)


def sigmoid_scores(logits):
    """Sigmoid scores ("sigmoid top-6" in "Model architecture"), rounded to fp32."""
    lg = np.asarray(logits, dtype=np.float64)
    return round_f32(1.0 / (1.0 + np.exp(-lg)))


def topk_desc(scores, k):
    """Indices of the k largest scores per row, in descending score order.

    Ties go to the lower expert index (a reading: the pages do not say).
    """
    scores = np.atleast_2d(np.asarray(scores, dtype=np.float64))
    out = np.empty((scores.shape[0], k), dtype=np.int64)
    idx = np.arange(scores.shape[1])
    for t in range(scores.shape[0]):
        order = np.lexsort((idx, -scores[t]))  # primary: -score, secondary: index
        out[t] = order[:k]
    return out


def route(logits, k=TOP_K, forced=None):
    """Sigmoid top-k routing with the selected scores renormalised to sum to 1.

    Returns (scores fp32 [B,E], ids [B,k], weights fp32 [B,k], gap [B]) where gap is
    the difference between the k-th and (k+1)-th largest score.  `forced` maps a
    token to an id list that replaces its selection (used where a near-tie makes
    several selections correct).
    """
    s = sigmoid_scores(logits)
    ids = topk_desc(s, k)
    srt = -np.sort(-s, axis=1)
    gap = srt[:, k - 1] - srt[:, k]
    if forced:
        for t, sel in forced.items():
            ids[t] = np.asarray(sel, dtype=np.int64)
    sel = np.take_along_axis(s, ids, axis=1)
    w = round_f32(sel / np.sum(sel, axis=1, keepdims=True))
    return s, ids, w, gap


def silu_mul(g, u):
    """h = bf16( silu(g) * u ) with silu(g) = g / (1 + exp(-g)) ("Optimizations": SiLU
    kernels that follow the reference rounding)."""
    g = np.asarray(g, dtype=np.float64)
    return round_bf16(g / (1.0 + np.exp(-g)) * np.asarray(u, dtype=np.float64))


def expert_gate_up(xh, w_gu):
    """g, u = fp32(x_hat . W_gate^T), fp32(x_hat . W_up^T); w_gu [2I, H] (gate rows first)."""
    gu = round_f32(np.atleast_2d(np.asarray(xh, np.float64)) @ np.asarray(w_gu, np.float64).T)
    i = w_gu.shape[0] // 2
    return gu[:, :i], gu[:, i:]


def expert_down(h, w_d):
    """d = fp32(h . W_down^T); w_d [H, I]."""
    return round_f32(np.atleast_2d(np.asarray(h, np.float64)) @ np.asarray(w_d, np.float64).T)


# ----------------------------------------------------------------------------
# Layer weights
# ----------------------------------------------------------------------------

class LayerView:
    """Read-only view of one sublayer's weights with lazily dequantised experts.

    Fields: router_w f64 [E, H]; norm_w f64 [H] or None; fmt 'nvfp4' | 'bf16'.
    nvfp4: gu_codes/gu_scales/dn_codes/dn_scales uint8, tensor_scales f64 [E+1, 2].
    bf16:  gu_bits uint16 [E+1, 2I, H], dn_bits uint16 [E+1, H, I].
    Expert E (= 256) is the shared expert.
    """

    def __init__(self, router_w, norm_w=None, fmt="nvfp4", gu_codes=None, gu_scales=None,
                 dn_codes=None, dn_scales=None, tensor_scales=None, gu_bits=None, dn_bits=None):
        self.router_w = np.asarray(router_w, dtype=np.float64)
        self.norm_w = None if norm_w is None else np.asarray(norm_w, dtype=np.float64)
        self.fmt = fmt
        self.gu_codes, self.gu_scales = gu_codes, gu_scales
        self.dn_codes, self.dn_scales = dn_codes, dn_scales
        self.tensor_scales = None if tensor_scales is None else np.asarray(tensor_scales, np.float64)
        self.gu_bits, self.dn_bits = gu_bits, dn_bits
        self._cache: dict = {}

    @property
    def n_experts_total(self):
        src = self.gu_codes if self.fmt == "nvfp4" else self.gu_bits
        return src.shape[0]

    def expert(self, e):
        """(W_gate_up f64 [2I, H], W_down f64 [H, I]) of expert e."""
        if e not in self._cache:
            if self.fmt == "nvfp4":
                wgu = dequant_nvfp4(self.gu_codes[e], self.gu_scales[e], self.tensor_scales[e, 0])
                wd = dequant_nvfp4(self.dn_codes[e], self.dn_scales[e], self.tensor_scales[e, 1])
            else:
                wgu = bf16_bits_to_f64(self.gu_bits[e])
                wd = bf16_bits_to_f64(self.dn_bits[e])
            self._cache[e] = (wgu, wd)
        return self._cache[e]

    def drop_cache(self):
        self._cache.clear()


def _bf16_tensor_to_bits(t):
    import torch  # plain CPU plumbing: read a bf16 tensor's bit pattern
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def layer_from_tensors(d):
    """Build a LayerView from the dict of tensors drawn by ``synth.gen_layer``."""
    rw = bf16_bits_to_f64(_bf16_tensor_to_bits(d["router_w"]))
    nw = None if d.get("norm_w") is None else bf16_bits_to_f64(_bf16_tensor_to_bits(d["norm_w"]))
    if "gu_codes" in d:
        return LayerView(rw, nw, "nvfp4",
                         gu_codes=d["gu_codes"].cpu().numpy(), gu_scales=d["gu_scales"].cpu().numpy(),
                         dn_codes=d["dn_codes"].cpu().numpy(), dn_scales=d["dn_scales"].cpu().numpy(),
                         tensor_scales=d["tensor_scales"].cpu().numpy())
    return LayerView(rw, nw, "bf16", gu_bits=_bf16_tensor_to_bits(d["gu_w"]),
                     dn_bits=_bf16_tensor_to_bits(d["dn_w"]))


# ----------------------------------------------------------------------------
# The sublayer, token by token (decode definition)
# ----------------------------------------------------------------------------

def moe_layer(x, lw: LayerView, forced=None, eps=RMS_EPS):
    """One MoE sublayer for a batch of independent tokens, computed token by token.

    x [B, H] holds bf16 values (float64).  Steps ("Model architecture" and the
    low-latency path description in "Optimizations"):
      x_hat = RMSNorm(x) if the layer has a norm weight, else x;
      logits = router GEMV; sigmoid; top-6; renormalise;
      for each selected expert and the shared expert:
          h = bf16(silu(g) * u),  d = fp32(h . W_down^T);
      y = bf16( sum_j w_j d_j + d_shared ).
    Returns a dict with y, x_hat, logits, scores, ids, weights, gap.
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    xh = rmsnorm(x, lw.norm_w, eps) if lw.norm_w is not None else x
    logits = router_logits(xh, lw.router_w)
    s, ids, w, gap = route(logits, TOP_K, forced)
    shared = lw.n_experts_total - 1
    y = np.empty_like(x)
    for t in range(x.shape[0]):
        acc = 0.0
        for j in range(TOP_K):
            wgu, wd = lw.expert(int(ids[t, j]))
            g, u = expert_gate_up(xh[t], wgu)
            d = expert_down(silu_mul(g, u), wd)[0]
            acc = acc + w[t, j] * d
        wgu, wd = lw.expert(shared)
        g, u = expert_gate_up(xh[t], wgu)
        acc = acc + expert_down(silu_mul(g, u), wd)[0]
        y[t] = round_bf16(acc)
    return dict(y=y, x_hat=xh, logits=logits, scores=s, ids=ids, weights=w, gap=gap)


def moe_stack(x, layers, forced_per_layer=None):
    """Chained sublayers: layer i+1 reads layer i's output through its own RMSNorm.

    No residual is added (a reading: the workload describes the output of one
    sublayer feeding the next after an RMSNorm).  Returns the final y and the
    per-layer results.
    """
    y = np.atleast_2d(np.asarray(x, dtype=np.float64))
    outs = []
    for i, lw in enumerate(layers):
        forced = None if forced_per_layer is None else forced_per_layer.get(i)
        r = moe_layer(y, lw, forced)
        outs.append(r)
        y = r["y"]
    return y, outs


# ----------------------------------------------------------------------------
# The sublayer over many tokens, grouped by expert (prefill definition)
# ----------------------------------------------------------------------------

def moe_prefill(x, lw: LayerView, eps=RMS_EPS):
    """The same sublayer for T tokens, computed expert by expert.

    ("Optimizations": the small-batch MoE kernels also gave the largest prefill
    gain; the prefill is the 8,192-token case.)  Tokens are bucketed by the
    expert they chose, each expert runs once over its bucket, and the weighted
    results are scattered back.  Per token it equals ``moe_layer``; the loop
    structure differs on purpose so each checks the other's indexing.
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    T = x.shape[0]
    xh = rmsnorm(x, lw.norm_w, eps) if lw.norm_w is not None else x
    logits = router_logits(xh, lw.router_w)
    s, ids, w, gap = route(logits, TOP_K)
    acc = np.zeros_like(x)
    n_total = lw.n_experts_total
    for e in range(n_total):
        if e == n_total - 1:
            toks = np.arange(T)
            wt = np.ones(T)
        else:
            tt, jj = np.nonzero(ids == e)
            if tt.size == 0:
                continue
            toks, wt = tt, w[tt, jj]
        wgu, wd = lw.expert(e)
        g, u = expert_gate_up(xh[toks], wgu)
        d = expert_down(silu_mul(g, u), wd)
        np.add.at(acc, toks, wt[:, None] * d)
        lw._cache.pop(e, None)
    return dict(y=round_bf16(acc), x_hat=xh, logits=logits, scores=s, ids=ids, weights=w, gap=gap)


# ----------------------------------------------------------------------------
# Small-batch dense GEMV on NVFP4 weights
# ----------------------------------------------------------------------------

def dense_gemv(x, codes, scales, tensor_scale):
    """y = bf16( fp32( x . W^T ) ), W = dequant_nvfp4(codes, scales, tensor_scale).

    ("Optimizations": a small-batch dense GEMV on the same NVFP4 weights.)
    x [B, K] holds bf16 values; codes uint8 [N, K/2] and scales uint8 [N, K/16]
    in the plain NVFP4 layout.  The dot products are summed in float64 and
    rounded once to fp32, then to bf16.
    """
    w = dequant_nvfp4(codes, scales, tensor_scale)
    return round_bf16(round_f32(np.atleast_2d(np.asarray(x, np.float64)) @ w.T))
