"""flint_moe_decode_layer_noalloc: the decode call for callers that cannot allocate.

Some callers cannot hand the library a device workspace (no cudaMalloc in
their context, or every device allocation owned by someone else).  The
no-allocation entry point uses a scratch array built into the library
instead.  This file checks that it gives bit for bit the result of the
workspace-based flint_moe_decode_layer on two calls in a row (the second
call finds the first call's leftovers in the shared scratch; the first goes
straight through the C ABI, the second through the Python wrapper), and that
a batch beyond the built-in scratch, or overlapping buffers, are refused on
the host.

Collected last on purpose (file name), so a stop-at-first-failure run has
already run every other test before this one.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth
from flint_testlib import bf16_to_f64, check_output
from moe_decode_router_gb300 import flint_moe as F


@pytest.mark.gpu
@pytest.mark.parametrize("kernel", [F.DECODE_CHAINED, F.DECODE_PERSISTENT], ids=["chained", "persistent"])
def test_noalloc_matches_workspace_call_twice_in_a_row(kernel):
    lib = F.load_library()
    F.set_decode_kernel(kernel)
    dev = torch.device("cuda:0")
    plain = synth.gen_layer(0, 0, device="cpu")
    L = F.pack_layer(plain, device=dev)
    torch.cuda.synchronize()
    ws = F.alloc_workspace(F.W_NVFP4, 8, device=dev)
    # different batches: the second call finds the first call's leftovers in the
    # shared scratch; it goes through the Python wrapper and its tensor checks
    for B, index, raw_call in ((8, 91, True), (3, 92, False)):
        x = synth.gen_x(0, B, index=index).to(dev)
        y_ref = torch.empty_like(x)
        ids_ref = torch.empty((B, 6), dtype=torch.int32, device=dev)
        w_ref = torch.empty((B, 6), dtype=torch.float32, device=dev)
        F.decode_layer(L, x, y_ref, ws, ids_ref, w_ref)
        y = torch.empty_like(x)
        ids = torch.full((B, 6), -1, dtype=torch.int32, device=dev)
        w = torch.zeros((B, 6), dtype=torch.float32, device=dev)
        if raw_call:
            d = F.dims(F.W_NVFP4)
            Lc = L.c_struct()
            rc = lib.flint_moe_decode_layer_noalloc(ctypes.byref(d), ctypes.byref(Lc), x.data_ptr(), B,
                                                    y.data_ptr(), ids.data_ptr(), w.data_ptr(),
                                                    torch.cuda.current_stream().cuda_stream)
            assert rc == F.FLINT_MOE_OK
        else:
            F.decode_layer_noalloc(L, x, y, ids, w)
        torch.cuda.synchronize()
        assert F.device_error() == 0
        assert np.array_equal(ids.cpu().numpy(), ids_ref.cpu().numpy())
        assert np.array_equal(w.cpu().numpy(), w_ref.cpu().numpy())
        # the decode path is deterministic: same kernels, same inputs, same bits
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
        check_output(bf16_to_f64(y), bf16_to_f64(y_ref))
    F.set_decode_kernel(F.DECODE_CHAINED)


@pytest.mark.skipif(torch.cuda.is_available(), reason="passes fake device addresses")
def test_noalloc_rejects_batches_beyond_its_scratch():
    lib = F.load_library()
    d = F.dims(F.W_NVFP4)
    fake = 0x7F0000000000  # never dereferenced: the batch check fails first
    Lc = F.Layer(fake, fake + 256, fake + 512, None)
    rc = lib.flint_moe_decode_layer_noalloc(ctypes.byref(d), ctypes.byref(Lc), fake + 1024, 9, fake + 2048,
                                            None, None, None)
    assert rc == F.FLINT_MOE_ERR_WORKSPACE


@pytest.mark.skipif(torch.cuda.is_available(), reason="passes fake device addresses")
def test_noalloc_rejects_overlapping_buffers_on_the_host():
    lib = F.load_library()
    d = F.dims(F.W_NVFP4)
    fake = 0x7F0000000000  # never dereferenced: the overlap check fails first
    Lc = F.Layer(fake, fake + (1 << 32), fake + (1 << 33), None)
    x = fake + (1 << 34)
    # B = 2: activations are 8,192 bytes; y starts inside x
    rc = lib.flint_moe_decode_layer_noalloc(ctypes.byref(d), ctypes.byref(Lc), x, 2, x + 4096, None, None, None)
    assert rc == F.FLINT_MOE_ERR_INVALID_ARG
    # topk_ids inside y
    rc = lib.flint_moe_decode_layer_noalloc(ctypes.byref(d), ctypes.byref(Lc), x, 2, x + 8192, x + 8192 + 64, None,
                                            None)
    assert rc == F.FLINT_MOE_ERR_INVALID_ARG
