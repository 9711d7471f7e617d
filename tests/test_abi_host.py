"""The C-ABI library builds, loads, exports every declared symbol, and rejects bad
arguments on the host before touching a GPU (no compute call is made here)."""

import ctypes
import os
import re

import pytest

from moe_decode_router_gb300 import flint_moe as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flint_moe.h")


@pytest.fixture(scope="module")
def lib():
    return F.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flint_moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_four_calls_and_helpers():
    names = declared_functions()
    for n in ("flint_moe_pack_weights", "flint_moe_decode_layer", "flint_moe_decode_stack",
              "flint_moe_prefill_layer", "flint_moe_packed_bytes", "flint_moe_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(F.EXPORTED)


def test_packed_and_workspace_sizes(lib):
    assert F.packed_bytes(F.W_NVFP4) == 257 * 1_769_472
    assert F.packed_bytes(F.W_BF16) == 257 * 6_291_456
    ws = F.workspace_bytes(F.W_NVFP4, 8)
    assert ws > 0 and ws % 256 == 0
    assert F.workspace_bytes(F.W_NVFP4, 1) == ws
    assert F.workspace_bytes(F.W_NVFP4, 64) > ws                   # medium-batch tables, h and partials
    assert F.workspace_bytes(F.W_NVFP4, 65) >= F.workspace_bytes(F.W_NVFP4, 64)  # covers every smaller call
    assert F.workspace_bytes(F.W_BF16, 9) == 0                     # 9..64 tokens: NVFP4 only
    bad = F.Dims(4096, 256, 1, 512, 6, 0, 1e-6)
    assert lib.flint_moe_packed_bytes(ctypes.byref(bad)) == 0
    assert lib.flint_moe_workspace_bytes(ctypes.byref(bad), 8) == 0


FAKE = 0x7f0000000000  # 256-aligned address never dereferenced: validation fails first

# The calls below pass fake device addresses that must be refused on the host.
# Where a GPU is visible, a call whose arguments were wrongly valid would launch
# kernels on them, so these tests run only where no GPU is visible.
no_gpu_only = pytest.mark.skipif(__import__("torch").cuda.is_available(),
                                 reason="host-validation tests pass fake device addresses")


def _layer(**kw):
    base = dict(router_w=FAKE, experts=FAKE + 256, tensor_scales=FAKE + 512, norm_w=None)
    base.update(kw)
    return F.Layer(base["router_w"], base["experts"], base["tensor_scales"], base["norm_w"])


def _decode(lib, d=None, L=None, x=FAKE + 1024, B=1, y=FAKE + 2048, ws=FAKE + 4096, ws_bytes=None):
    d = d or F.dims()
    L = L or _layer()
    ws_bytes = F.workspace_bytes() if ws_bytes is None else ws_bytes
    return lib.flint_moe_decode_layer(ctypes.byref(d), ctypes.byref(L), x, B, y, None, None, ws, ws_bytes, None)


@no_gpu_only
def test_decode_rejects_bad_arguments_on_host(lib):
    assert _decode(lib, B=65) == F.FLINT_MOE_ERR_UNSUPPORTED       # beyond the medium-batch cap
    assert _decode(lib, B=9) == F.FLINT_MOE_ERR_WORKSPACE          # 9..64 tokens need the medium workspace
    assert _decode(lib, B=9, d=F.dims(F.W_BF16), L=_layer(tensor_scales=None)) == F.FLINT_MOE_ERR_UNSUPPORTED
    assert _decode(lib, B=0) == F.FLINT_MOE_ERR_INVALID_ARG
    assert _decode(lib, x=None) == F.FLINT_MOE_ERR_INVALID_ARG
    assert _decode(lib, x=FAKE + 1032) == F.FLINT_MOE_ERR_INVALID_ARG  # not 16-byte aligned
    assert _decode(lib, y=FAKE + 1024) == F.FLINT_MOE_ERR_INVALID_ARG  # y aliases x
    assert _decode(lib, ws=FAKE + 4112) == F.FLINT_MOE_ERR_INVALID_ARG  # ws not 256-byte aligned
    assert _decode(lib, ws_bytes=1024) == F.FLINT_MOE_ERR_WORKSPACE
    assert _decode(lib, L=_layer(router_w=None)) == F.FLINT_MOE_ERR_INVALID_ARG
    assert _decode(lib, L=_layer(tensor_scales=None)) == F.FLINT_MOE_ERR_INVALID_ARG  # NVFP4 needs scales
    assert _decode(lib, d=F.Dims(2048, 128, 1, 512, 6, 0, 1e-6)) == F.FLINT_MOE_ERR_UNSUPPORTED
    assert _decode(lib, d=F.Dims(2048, 256, 1, 512, 8, 0, 1e-6)) == F.FLINT_MOE_ERR_UNSUPPORTED
    assert _decode(lib, d=F.Dims(2048, 256, 1, 512, 6, 7, 1e-6)) == F.FLINT_MOE_ERR_UNSUPPORTED
    assert _decode(lib, d=F.Dims(2048, 256, 1, 512, 6, 0, float("nan"))) == F.FLINT_MOE_ERR_INVALID_ARG
    # byte ranges: B = 1 activations are 4096 bytes; x, y and the workspace must not share any
    far = FAKE + (1 << 30)
    assert _decode(lib, x=FAKE, y=FAKE + 4080, ws=far) == F.FLINT_MOE_ERR_INVALID_ARG    # y overlaps x
    assert _decode(lib, x=FAKE, y=FAKE + 8192, ws=FAKE + 8192 + 3840) == F.FLINT_MOE_ERR_INVALID_ARG  # ws overlaps y
    assert _decode(lib, x=far + 4096, y=FAKE, ws=far) == F.FLINT_MOE_ERR_INVALID_ARG     # ws overlaps x


@no_gpu_only
def test_stack_and_pack_reject_bad_arguments_on_host(lib):
    d = F.dims()
    arr = (F.Layer * 2)(_layer(), _layer(router_w=None))
    ws_b = F.workspace_bytes()
    rc = lib.flint_moe_decode_stack(ctypes.byref(d), arr, 2, FAKE + 1024, 1, FAKE + 2048, None, None, None,
                                    FAKE + 4096, ws_b, None)
    assert rc == F.FLINT_MOE_ERR_INVALID_ARG
    arr = (F.Layer * 1)(_layer())
    rc = lib.flint_moe_decode_stack(ctypes.byref(d), arr, 0, FAKE + 1024, 1, FAKE + 2048, None, None, None,
                                    FAKE + 4096, ws_b, None)
    assert rc == F.FLINT_MOE_ERR_INVALID_ARG
    rc = lib.flint_moe_decode_stack(ctypes.byref(d), arr, 1, FAKE + 1024, 65, FAKE + 2048, None, None, None,
                                    FAKE + 4096, ws_b, None)
    assert rc == F.FLINT_MOE_ERR_UNSUPPORTED
    rc = lib.flint_moe_decode_stack(ctypes.byref(d), arr, 1, FAKE + 1024, 12, FAKE + 2048, None, None, None,
                                    FAKE + 4096, ws_b, None)
    assert rc == F.FLINT_MOE_ERR_WORKSPACE  # 12 tokens need the medium-batch workspace
    # NVFP4 pack needs both scale tensors; BF16 pack must not get any
    rc = lib.flint_moe_pack_weights(ctypes.byref(d), FAKE, None, FAKE + 256, FAKE + 512, FAKE + 1024,
                                    F.packed_bytes(), None)
    assert rc == F.FLINT_MOE_ERR_INVALID_ARG
    db = F.dims(F.W_BF16)
    rc = lib.flint_moe_pack_weights(ctypes.byref(db), FAKE, FAKE + 16, FAKE + 256, None, FAKE + 1024,
                                    F.packed_bytes(F.W_BF16), None)
    assert rc == F.FLINT_MOE_ERR_INVALID_ARG
    rc = lib.flint_moe_pack_weights(ctypes.byref(d), FAKE, FAKE + 16, FAKE + 256, FAKE + 512, FAKE + 1024,
                                    100, None)
    assert rc == F.FLINT_MOE_ERR_WORKSPACE


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5):
        assert lib.flint_moe_status_string(st)
    assert lib.flint_moe_status_string(-99) == b"unknown status"


@no_gpu_only
def test_prefill_rejects_bad_arguments_on_host(lib):
    d = F.dims()
    ws_b = F.workspace_bytes(F.W_NVFP4, 8192)
    assert ws_b >= F.workspace_bytes(F.W_NVFP4, 8) and ws_b % 256 == 0
    assert F.workspace_bytes(F.W_BF16, 9) == 0  # prefill takes NVFP4 weights only

    def call(dd=None, T=8192, x=FAKE + 1024, y=FAKE + 2048, ws=FAKE + 4096, n=ws_b, L=None):
        return lib.flint_moe_prefill_layer(ctypes.byref(dd or d), ctypes.byref(L or _layer()), x, T, y, None,
                                           None, ws, n, None)

    assert call(T=0) == F.FLINT_MOE_ERR_INVALID_ARG
    assert call(T=(1 << 20) + 1) == F.FLINT_MOE_ERR_UNSUPPORTED
    assert call(dd=F.dims(F.W_BF16)) == F.FLINT_MOE_ERR_UNSUPPORTED
    assert call(n=ws_b - 256) == F.FLINT_MOE_ERR_WORKSPACE
    assert call(y=FAKE + 1024) == F.FLINT_MOE_ERR_INVALID_ARG
    assert call(x=FAKE + 1032) == F.FLINT_MOE_ERR_INVALID_ARG
    assert call(ws=FAKE + 4112) == F.FLINT_MOE_ERR_INVALID_ARG
    assert call(L=_layer(tensor_scales=None)) == F.FLINT_MOE_ERR_INVALID_ARG
    act = 8192 * 2048 * 2
    far = FAKE + (1 << 36)
    assert call(x=FAKE, y=FAKE + act - 16, ws=far) == F.FLINT_MOE_ERR_INVALID_ARG       # y overlaps x
    assert call(x=FAKE, y=FAKE + act, ws=FAKE + 2 * act - 256) == F.FLINT_MOE_ERR_INVALID_ARG  # ws overlaps y


@no_gpu_only
def test_outputs_must_not_overlap_any_other_buffer(lib):
    """Every buffer a call writes (y, workspace, ids, weights out, per-layer outputs) is
    checked against every other buffer of the call, weights included.  The fake
    buffers below lie 2^32 bytes apart, so the unmodified set would pass the host
    checks; every call changes exactly one address to create one overlap, and so
    is refused before anything is launched.  The unmodified set is never called."""
    G = 1 << 32
    base = FAKE + (1 << 40)
    RW, EX, TS, NW, X, Y, WS, IDS, WO, YS = (base + k * G for k in range(10))
    d = F.dims()
    ws_b = F.workspace_bytes()

    def layer(**kw):
        a = dict(router_w=RW, experts=EX, tensor_scales=TS, norm_w=NW)
        a.update(kw)
        return F.Layer(a["router_w"], a["experts"], a["tensor_scales"], a["norm_w"])

    def dec(x=X, y=Y, ws=WS, ids=IDS, w=WO, L=None):
        return lib.flint_moe_decode_layer(ctypes.byref(d), ctypes.byref(L or layer()), x, 2, y, ids, w, ws, ws_b,
                                          None)

    bad = [
        dict(ids=Y + 4096),                 # ids inside y (B = 2: 8,192 bytes)
        dict(w=X + 16),                     # weights out inside x
        dict(ids=WS + 256),                 # ids inside the workspace
        dict(w=IDS + 32),                   # ids (48 bytes) and weights out share bytes
        dict(y=EX + 4096),                  # y inside the packed experts
        dict(w=TS + 512),                   # weights out on the tensor scales
        dict(ids=NW + 4064),                # ids overlapping the end of the norm weight (4,096 bytes)
        dict(ws=RW + (1 << 20) - 256),      # workspace starting in the last bytes of the router weights
    ]
    for kw in bad:
        assert dec(**kw) == F.FLINT_MOE_ERR_INVALID_ARG, kw

    arr = (F.Layer * 2)(layer(), layer(router_w=RW + (1 << 24)))

    def stack(ids=IDS, w=WO, ys=YS, y=Y):
        return lib.flint_moe_decode_stack(ctypes.byref(d), arr, 2, X, 1, y, ids, w, ys, WS, ws_b, None)

    assert stack(ys=Y + 4096 - 16) == F.FLINT_MOE_ERR_INVALID_ARG   # ys overlaps y
    assert stack(ys=X - 8192 + 16) == F.FLINT_MOE_ERR_INVALID_ARG   # ys (2 layers x 4,096 bytes) reaches into x
    assert stack(ids=WS + ws_b - 16) == F.FLINT_MOE_ERR_INVALID_ARG  # ids overlaps the workspace's end
    assert stack(w=IDS + 32) == F.FLINT_MOE_ERR_INVALID_ARG          # 2 layers x 6 ids = 48 bytes
    assert stack(y=RW + (1 << 24) + 64) == F.FLINT_MOE_ERR_INVALID_ARG  # y on the second layer's router

    pre_ws = F.workspace_bytes(F.W_NVFP4, 64)
    rc = lib.flint_moe_prefill_layer(ctypes.byref(d), ctypes.byref(layer()), X, 64, Y, Y + 100 * 1024, None, WS,
                                     pre_ws, None)
    assert rc == F.FLINT_MOE_ERR_INVALID_ARG  # ids inside y (64 x 2048 x 2 = 256 KiB)


def test_wait_limit_and_status_helpers_exist(lib):
    assert lib.flint_moe_set_wait_limit(0) == F.FLINT_MOE_OK
    assert lib.flint_moe_set_wait_limit(123456) == F.FLINT_MOE_OK
    assert lib.flint_moe_set_wait_limit(-1) == F.FLINT_MOE_OK  # restores the default
