"""Seeded synthetic tensors with the shapes and distributions of the Flint MoE workloads.

Shapes follow the model description in "Day-0 Support for Flint on vLLM"
(section "Model architecture": hidden size 2048, 256 routed experts with
sigmoid top-6 plus one shared expert).  The expert intermediate size (512) is
not printed on the pages; it is the value consistent with the stated 40B total
parameters and is the assumption the workloads are quoted with.

Distributions (per workload):
  x             ~ N(0, 1), rounded to bf16, shape [B, 2048]
  router W      ~ N(0, 1/2048), bf16 [256, 2048]
  NVFP4 experts: E2M1 codes uniform over all 16 codes (each nibble of a
                 uniform random byte), E4M3 block scales uniform over the 49
                 E4M3 encodings 0x18..0x48 (values 2^-4 .. 2^2), one FP32
                 per-tensor scale 0.02 for gate/up and one for down
  BF16 experts  ~ N(0, 0.02), bf16
  RMSNorm weight ~ 1 + N(0, 0.1), bf16 (layers 1.. of a stack)

Plain NVFP4 layout produced here (the input format of the packer):
  gate/up codes  uint8 [257, 1024, 1024]  rows 0..511 gate, 512..1023 up;
                 byte j of a row holds elements 2j (low nibble) and 2j+1
  gate/up scales uint8 [257, 1024, 128]   one E4M3 byte per 16 elements
  down codes     uint8 [257, 2048, 256]
  down scales    uint8 [257, 2048, 32]
  tensor scales  fp32  [257, 2]           (gate/up, down)
Expert index 256 is the shared expert.

Every tensor is drawn from its own torch.Generator seeded from
(workload seed, layer, tensor id).  The stream depends on the device the
generator runs on: a CUDA-drawn layer differs from a CPU-drawn one with the
same seed, so a check always feeds the oracle the very tensors the GPU used.
"""

from __future__ import annotations

import torch

H = 2048
E = 256
N_SHARED = 1
INTER = 512
TOP_K = 6
N_LAYERS = 47
BLOCK = 16
SCALE_LO, SCALE_HI = 0x18, 0x48  # E4M3 encodings of 2^-4 and 2^2
TENSOR_SCALE = 0.02

# name -> (layers, batch, weight format); index = position in the workload list
CONFIGS = {
    0: dict(name="layer_b1_nvfp4", layers=1, batch=1, weights="nvfp4", norm=False),
    1: dict(name="stack47_b1_nvfp4", layers=N_LAYERS, batch=1, weights="nvfp4", norm=True),
    2: dict(name="stack47_b8_nvfp4", layers=N_LAYERS, batch=8, weights="nvfp4", norm=True),
    3: dict(name="stack47_b8_bf16", layers=N_LAYERS, batch=8, weights="bf16", norm=True),
    4: dict(name="prefill8192_nvfp4", layers=1, batch=8192, weights="nvfp4", norm=False),
}

_TENSOR_IDS = {
    "x": 1, "router_w": 2, "gu_codes": 3, "gu_scales": 4, "dn_codes": 5,
    "dn_scales": 6, "norm_w": 7, "gu_bf16": 8, "dn_bf16": 9,
    "dense_codes": 10, "dense_scales": 11, "dense_x": 12,
}

# Dense NVFP4 matrices (the small-batch dense GEMV): the same element
# distributions as the expert weights; the seed offset keeps them apart from
# every workload's layers.
DENSE_SEED = 0xD3E5


def config_seed(cfg: int) -> int:
    return 0xF117 + int(cfg)


def _mix(*vals: int) -> int:
    """splitmix64 finaliser folded over the key; gives a 63-bit torch seed."""
    h = 0x9E3779B97F4A7C15
    for v in vals:
        h = (h ^ (int(v) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        h = (h + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = h
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        h = z ^ (z >> 31)
    return h & 0x7FFFFFFFFFFFFFFF


def _gen(seed: int, layer: int, tensor: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(seed, layer, _TENSOR_IDS[tensor]))
    return g


def gen_x(cfg: int, batch: int, index: int = 0, device="cpu") -> torch.Tensor:
    """x ~ N(0,1) as bf16 [batch, H]; `index` selects one of several seeded inputs."""
    g = _gen(config_seed(cfg), 100000 + index, "x", device)
    return torch.randn(batch, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def gen_layer(cfg: int, layer: int, device="cpu", weights: str | None = None,
              norm: bool | None = None, n_experts_total: int = E + N_SHARED) -> dict:
    """All tensors of one MoE sublayer in the plain (unpacked) layout.

    Returns a dict of torch tensors on `device`:
      router_w bf16 [E, H]; tensor_scales fp32 [E+1, 2];
      nvfp4: gu_codes, gu_scales, dn_codes, dn_scales (uint8, layouts above)
      bf16:  gu_w bf16 [E+1, 2*INTER, H], dn_w bf16 [E+1, H, INTER]
      norm_w bf16 [H] or None.
    """
    c = CONFIGS[cfg]
    weights = weights or c["weights"]
    if norm is None:
        norm = c["norm"] and layer > 0
    s = config_seed(cfg)
    n = n_experts_total
    out: dict = {}
    g = _gen(s, layer, "router_w", device)
    out["router_w"] = (torch.randn(E, H, generator=g, device=device) * (1.0 / H) ** 0.5).to(torch.bfloat16)
    if weights == "nvfp4":
        def rbytes(name, shape, lo=0, hi=256):
            gg = _gen(s, layer, name, device)
            return torch.randint(lo, hi, shape, generator=gg, device=device, dtype=torch.uint8)
        out["gu_codes"] = rbytes("gu_codes", (n, 2 * INTER, H // 2))
        out["gu_scales"] = rbytes("gu_scales", (n, 2 * INTER, H // BLOCK), SCALE_LO, SCALE_HI + 1)
        out["dn_codes"] = rbytes("dn_codes", (n, H, INTER // 2))
        out["dn_scales"] = rbytes("dn_scales", (n, H, INTER // BLOCK), SCALE_LO, SCALE_HI + 1)
        out["tensor_scales"] = torch.full((n, 2), TENSOR_SCALE, dtype=torch.float32, device=device)
    elif weights == "bf16":
        g1 = _gen(s, layer, "gu_bf16", device)
        out["gu_w"] = (torch.randn(n, 2 * INTER, H, generator=g1, device=device) * 0.02).to(torch.bfloat16)
        g2 = _gen(s, layer, "dn_bf16", device)
        out["dn_w"] = (torch.randn(n, H, INTER, generator=g2, device=device) * 0.02).to(torch.bfloat16)
        out["tensor_scales"] = None
    else:
        raise ValueError(weights)
    if norm:
        g = _gen(s, layer, "norm_w", device)
        out["norm_w"] = (1.0 + 0.1 * torch.randn(H, generator=g, device=device)).to(torch.bfloat16)
    else:
        out["norm_w"] = None
    return out


def gen_dense(N: int, K: int, index: int = 0, device="cpu") -> dict:
    """A plain NVFP4 matrix [N][K]: codes uint8 [N, K/2] (uniform bytes), E4M3
    block scales uint8 [N, K/16] (uniform over 0x18..0x48), tensor scale 0.02."""
    g1 = _gen(DENSE_SEED, index, "dense_codes", device)
    g2 = _gen(DENSE_SEED, index, "dense_scales", device)
    return {
        "codes": torch.randint(0, 256, (N, K // 2), generator=g1, device=device, dtype=torch.uint8),
        "scales": torch.randint(SCALE_LO, SCALE_HI + 1, (N, K // BLOCK), generator=g2, device=device,
                                dtype=torch.uint8),
        "tensor_scale": TENSOR_SCALE,
    }


def gen_dense_x(B: int, K: int, index: int = 0, device="cpu") -> torch.Tensor:
    """x ~ N(0,1) as bf16 [B, K] for the dense GEMV."""
    g = _gen(DENSE_SEED, 100000 + index, "dense_x", device)
    return torch.randn(B, K, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
