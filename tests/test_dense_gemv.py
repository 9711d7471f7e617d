"""The small-batch dense GEMV on packed NVFP4 weights against the oracle, through the C ABI.

Shapes span one 16-row tile (N = 16) to 6144 rows, K from one 256-column
slice to 8192, a ragged last unit of slices (K = 2304: 9 slices, one
8-slice bulk copy and one of a single slice), and the B * K limit of the
staged activations (B = 8 at K = 4096, B = 4 at K = 8192).
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import synth
from flint_testlib import bf16_to_f64, check_output
from moe_decode_router_gb300 import flint_moe as F


def _pack(N, K, index, dev):
    d = synth.gen_dense(N, K, index=index, device="cpu")
    w = F.pack_dense(d["codes"], d["scales"], d["tensor_scale"], device=dev)
    torch.cuda.synchronize()
    return d, w


@pytest.mark.gpu
@pytest.mark.parametrize("N,K,B", [(16, 256, 1), (2048, 2048, 1), (2048, 2048, 3), (2048, 2048, 8),
                                   (6144, 2048, 8), (2064, 2304, 5), (512, 4096, 8), (4096, 8192, 4)])
def test_dense_gemv_matches_oracle(N, K, B):
    F.load_library()
    dev = torch.device("cuda:0")
    d, w = _pack(N, K, index=N + K, dev=dev)
    x = synth.gen_dense_x(B, K, index=B).to(dev)
    y = torch.full((B, N), float("nan"), dtype=torch.bfloat16, device=dev)
    F.dense_gemv(w, x, y)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    ref = O.dense_gemv(bf16_to_f64(x), d["codes"].numpy(), d["scales"].numpy(), d["tensor_scale"])
    st = check_output(bf16_to_f64(y), ref)
    print(f"N={N} K={K} B={B} {st}")
    # deterministic: a second call gives the same bits
    y2 = torch.empty_like(y)
    F.dense_gemv(w, x, y2)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.gpu
def test_dense_gemv_integer_weights_exact():
    """Codes in {0, +-1}, scale 1, tensor scale 1, integer x: the GPU result is the
    exact integer product (fp32 accumulation of small integers is exact)."""
    F.load_library()
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(5)
    N, K, B = 256, 1024, 8
    vals = rng.integers(-1, 2, size=(N, K))
    code = np.where(vals == 1, 0x2, np.where(vals == -1, 0xA, 0x0)).astype(np.uint8)
    codes = torch.from_numpy((code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8))
    scales = torch.full((N, K // 16), 0x38, dtype=torch.uint8)
    w = F.pack_dense(codes, scales, 1.0, device=dev)
    xi = rng.integers(-2, 3, size=(B, K))
    x = torch.from_numpy(xi.astype(np.float32)).to(torch.bfloat16).to(dev)
    y = torch.empty((B, N), dtype=torch.bfloat16, device=dev)
    F.dense_gemv(w, x, y)
    torch.cuda.synchronize()
    ref = xi @ vals.T
    assert np.all(np.abs(ref) <= 256)
    assert np.array_equal(bf16_to_f64(y), ref.astype(np.float64))


FAKE = 0x7F0000000000


@pytest.mark.skipif(torch.cuda.is_available(), reason="passes fake device addresses")
def test_dense_rejects_bad_arguments_on_host():
    lib = F.load_library()
    assert lib.flint_moe_dense_packed_bytes(2048, 2048) == 2048 * 2048 * 9 // 16
    assert lib.flint_moe_dense_packed_bytes(2040, 2048) == 0   # N not a multiple of 16
    assert lib.flint_moe_dense_packed_bytes(2048, 2000) == 0   # K not a multiple of 256
    assert lib.flint_moe_dense_packed_bytes(2048, 65536) == 0  # K above 32768

    def gemv(N=2048, K=2048, B=1, x=FAKE + (1 << 32), y=FAKE + (2 << 32), w=FAKE, ts=1.0):
        return lib.flint_moe_dense_gemv(w, N, K, ts, x, B, y, None)

    assert gemv(N=2040) == F.FLINT_MOE_ERR_UNSUPPORTED
    assert gemv(B=9) == F.FLINT_MOE_ERR_UNSUPPORTED
    assert gemv(K=8192, B=5) == F.FLINT_MOE_ERR_UNSUPPORTED      # B * K above 32768
    assert gemv(B=0) == F.FLINT_MOE_ERR_INVALID_ARG
    assert gemv(x=FAKE + (1 << 32) + 8) == F.FLINT_MOE_ERR_INVALID_ARG  # misaligned
    assert gemv(ts=float("inf")) == F.FLINT_MOE_ERR_INVALID_ARG
    assert gemv(y=FAKE + (1 << 32) + 1024) == F.FLINT_MOE_ERR_INVALID_ARG  # y overlaps x
    assert gemv(y=FAKE + 4096) == F.FLINT_MOE_ERR_INVALID_ARG  # y overlaps the packed matrix
    rc = lib.flint_moe_pack_dense(FAKE, FAKE + (1 << 32), 2048, 2048, FAKE + (2 << 32), 1000, None)
    assert rc == F.FLINT_MOE_ERR_WORKSPACE
