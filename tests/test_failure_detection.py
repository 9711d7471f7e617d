"""Failure detection on the decode path, without a GPU fault: a wait that runs out.

The persistent NVFP4 decode kernel's thread blocks (selected with
flint_moe_set_decode_kernel) wait for logits, h and y
that the other blocks of the same call write.  Every such wait is bounded
(flint_moe_set_wait_limit, about one second by default).  With a limit of one
cycle, a wait that is not satisfied at its first look gives up: it sets bit 32
of the device error word and raises the call's abort flag, and every block
then returns (after its own bulk copies have landed).  The test checks that
the call ends, that flint_moe_device_status maps the word to
FLINT_MOE_ERR_TIMEOUT, and that the context stays usable: the next call with
the default limit gives the same bits as before.  Nothing here faults or
hangs the GPU; the waits that run out are on data words, which no bulk copy
targets.
"""

import numpy as np
import pytest
import torch

import synth
from moe_decode_router_gb300 import flint_moe as F

pytestmark = pytest.mark.gpu

ERR_POLL = 32


def test_wait_that_runs_out_abandons_the_call_and_reports_timeout():
    F.load_library()
    dev = torch.device("cuda:0")
    Ls = [F.pack_layer(synth.gen_layer(1, i, device="cpu"), device=dev) for i in range(3)]
    torch.cuda.synchronize()
    x = synth.gen_x(1, 8, index=500).to(dev)
    ws = F.alloc_workspace(F.W_NVFP4, 8, device=dev)
    y_ref = torch.empty_like(x)
    F.set_decode_kernel(F.DECODE_PERSISTENT)
    F.decode_stack(Ls, x, y_ref, ws)
    torch.cuda.synchronize()
    assert F.device_status() == F.FLINT_MOE_OK

    F.set_decode_kernel(F.DECODE_PERSISTENT)
    F.set_wait_limit(1)
    try:
        words = []
        for _ in range(5):
            y = torch.full_like(x, float("nan"))
            F.decode_stack(Ls, x, y, ws)
            torch.cuda.synchronize()  # the kernel returned
            word = F.device_error(reset=False)
            st = F.device_status(reset=True)
            words.append(word)
            assert st in (F.FLINT_MOE_OK, F.FLINT_MOE_ERR_TIMEOUT), (st, word)
            if st == F.FLINT_MOE_ERR_TIMEOUT:
                assert word & ERR_POLL
                break
        print("error words seen with a one-cycle limit:", words)
        assert words[-1] & ERR_POLL, words
    finally:
        F.set_wait_limit(0)

    y2 = torch.empty_like(x)
    F.decode_stack(Ls, x, y2, ws)
    torch.cuda.synchronize()
    F.set_decode_kernel(F.DECODE_CHAINED)
    assert F.device_status() == F.FLINT_MOE_OK
    assert torch.equal(y2.view(torch.int16), y_ref.view(torch.int16))
    assert bool(torch.isfinite(y2.float()).all())
