"""GPU parity of the medium-batch decode path (9..64 tokens) against the CPU oracle.

Same entry points as the decode path (flint_moe_decode_layer / _stack); past 8
tokens they run the expert-grouped kernels.  Full-size shapes; the batches
cover one partial chunk of 8 (9, 17), whole chunks (16, 32, 40, 64), experts
chosen by more than 8 tokens (several slot-chunks of one expert) and the
shared expert's 8 slot-chunks at 64 tokens.
"""

import numpy as np
import pytest
import torch

import oracle as O
import synth
from flint_testlib import bf16_to_f64, check_layer
from moe_decode_router_gb300 import flint_moe as F

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    F.load_library()
    return torch.device("cuda:0")


def _pack(plain, dev):
    L = F.pack_layer(plain, device=dev)
    torch.cuda.synchronize()
    return L


@pytest.fixture(scope="module")
def layer_cfg0(dev):
    plain = synth.gen_layer(0, 0, device="cpu")
    return plain, O.layer_from_tensors(plain), _pack(plain, dev)


@pytest.fixture(scope="module")
def layer_norm(dev):
    plain = synth.gen_layer(1, 1, device="cpu")
    assert plain["norm_w"] is not None
    return plain, O.layer_from_tensors(plain), _pack(plain, dev)


@pytest.fixture(scope="module")
def ws(dev):
    return F.alloc_workspace(F.W_NVFP4, max_tokens=F.MAX_MEDIUM_BATCH, device=dev)


def run_layer(L, x, dev, ws):
    B = x.shape[0]
    xd = x.to(dev)
    y = torch.empty_like(xd)
    ids = torch.full((B, 6), -1, dtype=torch.int32, device=dev)
    w = torch.zeros((B, 6), dtype=torch.float32, device=dev)
    F.decode_layer(L, xd, y, ws, ids, w)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    return y, ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("B", [9, 16, 17, 32, 40, 64])
def test_medium_layer_matches_oracle(layer_cfg0, dev, ws, B):
    _, lw, L = layer_cfg0
    x = synth.gen_x(0, B, index=200 + B)
    y, ids, w = run_layer(L, x, dev, ws)
    _, st = check_layer(bf16_to_f64(x), lw, bf16_to_f64(y), ids, w)
    print(f"B={B} distinct experts {len(set(ids.ravel().tolist()))} {st}")


@pytest.mark.parametrize("B", [12, 64])
def test_medium_layer_with_rmsnorm_matches_oracle(layer_norm, dev, ws, B):
    _, lw, L = layer_norm
    x = synth.gen_x(1, B, index=300 + B)
    y, ids, w = run_layer(L, x, dev, ws)
    check_layer(bf16_to_f64(x), lw, bf16_to_f64(y), ids, w)


def test_medium_is_deterministic(layer_cfg0, dev, ws):
    _, _, L = layer_cfg0
    x = synth.gen_x(0, 64, index=7)
    y1, i1, w1 = run_layer(L, x, dev, ws)
    y2, i2, w2 = run_layer(L, x, dev, ws)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert np.array_equal(i1, i2) and np.array_equal(w1, w2)


def test_medium_experts_shared_by_many_tokens(layer_cfg0, dev, ws):
    """20 copies of one token plus 21 others: the copies' 6 experts each serve
    at least 20 tokens (three slot-chunks of one expert: 8, 8 and the rest)."""
    _, lw, L = layer_cfg0
    x = torch.cat([synth.gen_x(0, 1, index=8).repeat(20, 1), synth.gen_x(0, 21, index=9)])
    y, ids, w = run_layer(L, x, dev, ws)
    assert np.all(ids[:20] == ids[0]) and np.all(w[:20] == w[0])
    yv = bf16_to_f64(y)
    assert np.all(yv[:20] == yv[0])
    _, st = check_layer(bf16_to_f64(x), lw, yv, ids, w)
    print(st)


def test_medium_all_tokens_identical(layer_cfg0, dev, ws):
    """64 identical tokens: 6 routed experts with 64 tokens each (8 slot-chunks
    apiece) and the shared expert's 8."""
    _, lw, L = layer_cfg0
    x = synth.gen_x(0, 1, index=10).repeat(64, 1)
    y, ids, w = run_layer(L, x, dev, ws)
    assert np.all(ids == ids[0])
    yv = bf16_to_f64(y)
    assert np.all(yv == yv[0])
    check_layer(bf16_to_f64(x[:1]), lw, yv[:1], ids[:1], w[:1])


def test_medium_unselected_experts_are_never_read(layer_cfg0, dev, ws):
    plain, lw, L = layer_cfg0
    x = synth.gen_x(0, 24, index=11)
    y_ref, ids, _ = run_layer(L, x, dev, ws)
    sel = set(ids.ravel().tolist())
    assert len(sel) < 256
    bad = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in plain.items()}
    for e in range(256):
        if e not in sel:
            bad["gu_scales"][e] = 0x7F  # E4M3 NaN
            bad["dn_scales"][e] = 0x7F
    y_bad, ids_b, _ = run_layer(_pack(bad, dev), x, dev, ws)
    assert np.array_equal(ids, ids_b)
    assert torch.equal(y_ref.view(torch.int16), y_bad.view(torch.int16))


def test_medium_stack_teacher_forced(dev, ws):
    plains = [synth.gen_layer(1, i, device="cpu") for i in range(3)]
    Ls = [_pack(p, dev) for p in plains]
    lws = [O.layer_from_tensors(p) for p in plains]
    B = 24
    x = synth.gen_x(1, B, index=12).to(dev)
    y = torch.empty_like(x)
    ids = torch.full((3, B, 6), -1, dtype=torch.int32, device=dev)
    w = torch.zeros((3, B, 6), dtype=torch.float32, device=dev)
    ys = torch.empty((3, B, 2048), dtype=torch.bfloat16, device=dev)
    F.decode_stack(Ls, x, y, ws, ids, w, ys)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    assert torch.equal(y.view(torch.int16), ys[-1].view(torch.int16))
    idn, wn = ids.cpu().numpy(), w.cpu().numpy()
    for i in range(3):
        x_in = bf16_to_f64(x.cpu()) if i == 0 else bf16_to_f64(ys[i - 1].cpu())
        check_layer(x_in, lws[i], bf16_to_f64(ys[i].cpu()), idn[i], wn[i])
    # the stack (one cached graph, no per-layer outputs) equals per-layer calls
    y2 = torch.empty_like(x)
    F.decode_stack(Ls, x, y2, ws)
    cur = x
    for L in Ls:
        nxt = torch.empty_like(cur)
        F.decode_layer(L, cur, nxt, ws)
        cur = nxt
    torch.cuda.synchronize()
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    assert torch.equal(cur.view(torch.int16), y.view(torch.int16))


def test_medium_rejections(layer_cfg0, dev, ws):
    _, _, L = layer_cfg0
    x = synth.gen_x(0, 65, index=13).to(dev)
    y = torch.empty_like(x)
    with pytest.raises(F.FlintMoeError) as ei:
        F.decode_layer(L, x, y, ws)
    assert ei.value.status == F.FLINT_MOE_ERR_UNSUPPORTED
    small = F.alloc_workspace(F.W_NVFP4, max_tokens=8, device=dev)
    if small.numel() < F.workspace_bytes(F.W_NVFP4, 64):
        with pytest.raises(F.FlintMoeError) as ei:
            F.decode_layer(L, x[:16], y[:16], small)
        assert ei.value.status == F.FLINT_MOE_ERR_WORKSPACE
