"""The prefill call at its largest accepted size, T = 2^20 tokens (about 33 GB
of device memory with the workspace), through the C ABI.  Every token must get
six distinct experts and a finite output row; the routing and output rows of
8,192 contiguous tokens in the middle, the last 256-token tile, the first token
and 29 random ones are checked against the oracle."""

import numpy as np
import pytest
import torch

import oracle as O
import synth
from flint_testlib import check_prefill
from moe_decode_router_gb300 import flint_moe as F

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

T_MAX = 1 << 20


def test_prefill_at_the_token_limit():
    F.load_library()
    dev = torch.device("cuda:0")
    need = F.workspace_bytes(F.W_NVFP4, T_MAX) + 2 * T_MAX * 2048 * 2 + T_MAX * 6 * 8 + (1 << 30)
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip(f"needs {need / 2**30:.1f} GiB of free device memory, {free / 2**30:.1f} free")
    plain = synth.gen_layer(0, 0, device="cpu")
    lw = O.layer_from_tensors(plain)
    L = F.pack_layer(plain, device=dev)
    x = synth.gen_x(0, T_MAX, index=400, device=dev)
    y = torch.full_like(x, float("nan"))
    ids = torch.full((T_MAX, 6), -1, dtype=torch.int32, device=dev)
    w = torch.zeros((T_MAX, 6), dtype=torch.float32, device=dev)
    ws = F.alloc_workspace(F.W_NVFP4, T_MAX, device=dev)
    F.prefill_layer(L, x, y, ws, ids, w)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    idc = ids.cpu().numpy()
    srt = np.sort(idc, axis=1)
    assert (srt[:, 0] >= 0).all() and (srt[:, -1] < 256).all()
    assert (srt[:, 1:] != srt[:, :-1]).all()  # six distinct experts per token
    assert bool(torch.isfinite(y).all())
    rng = np.random.default_rng(11)
    block = np.arange(T_MAX // 2 - 4096, T_MAX // 2 + 4096)  # 8,192 contiguous rows (32 shared-expert tiles)
    last_tile = np.arange(T_MAX - 256, T_MAX)
    sample = np.unique(np.concatenate([[0, T_MAX - 1], block, last_tile, rng.choice(T_MAX, 29, replace=False)]))
    sel = torch.from_numpy(sample).to(dev)
    st = check_prefill(x[sel].cpu(), lw, y[sel], idc[sample], w[sel].cpu().numpy())
    print(f"T={T_MAX} sampled {len(sample)} rows {st}")
    del ws, x, y
    torch.cuda.empty_cache()
