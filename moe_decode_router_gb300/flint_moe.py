"""ctypes binding of libflint_moe.so (include/flint_moe.h), same entry-point names.

Argument marshalling only: tensors are passed as device pointers, the stream
is torch's current CUDA stream unless one is given.  Every computation runs in
the library's CUDA kernels; there is no fallback path.  If the library cannot
be built or loaded the import-time call ``load_library`` raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

FLINT_MOE_OK = 0
FLINT_MOE_ERR_INVALID_ARG = -1
FLINT_MOE_ERR_UNSUPPORTED = -2
FLINT_MOE_ERR_WORKSPACE = -3
FLINT_MOE_ERR_CUDA = -4
FLINT_MOE_ERR_TIMEOUT = -5

W_NVFP4 = 0
W_BF16 = 1

DECODE_CHAINED = 0
DECODE_PERSISTENT = 1

HIDDEN, N_EXPERTS, N_SHARED, INTER, TOP_K = 2048, 256, 1, 512, 6
MAX_DECODE_BATCH = 8
MAX_MEDIUM_BATCH = 64  # decode calls with 9..64 tokens take the medium-batch kernels (NVFP4)


class FlintMoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib().flint_moe_status_string(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


class Dims(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("n_shared", ctypes.c_int),
        ("inter", ctypes.c_int), ("top_k", ctypes.c_int), ("weight_dtype", ctypes.c_int),
        ("rms_eps", ctypes.c_float),
    ]


class Layer(ctypes.Structure):
    _fields_ = [
        ("router_w", ctypes.c_void_p), ("experts", ctypes.c_void_p),
        ("tensor_scales", ctypes.c_void_p), ("norm_w", ctypes.c_void_p),
    ]


_LIB = None
_LOCK = threading.Lock()

_SIGS = {
    "flint_moe_packed_bytes": (ctypes.c_size_t, [ctypes.POINTER(Dims)]),
    "flint_moe_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Dims), ctypes.c_int]),
    "flint_moe_pack_weights": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_void_p]),
    "flint_moe_decode_layer": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(Layer), ctypes.c_void_p,
                                              ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "flint_moe_decode_stack": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(Layer), ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_void_p]),
    "flint_moe_prefill_layer": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(Layer), ctypes.c_void_p,
                                               ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "flint_moe_decode_layer_noalloc": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(Layer), ctypes.c_void_p,
                                                      ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                      ctypes.c_void_p]),
    "flint_moe_dense_packed_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int]),
    "flint_moe_pack_dense": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "flint_moe_dense_gemv": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "flint_moe_release": (ctypes.c_int, []),
    "flint_moe_device_error": (ctypes.c_int, [ctypes.c_int]),
    "flint_moe_device_status": (ctypes.c_int, [ctypes.c_int]),
    "flint_moe_set_wait_limit": (ctypes.c_int, [ctypes.c_longlong]),
    "flint_moe_set_decode_kernel": (ctypes.c_int, [ctypes.c_int]),
    "flint_moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

EXPORTED = tuple(_SIGS)


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads (building first if needed) the in-tree libflint_moe.so."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libflint_moe.so not found at {path}; build it with "
                               "python -m moe_decode_router_gb300.build")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
        return lib


def _lib():
    return _LIB if _LIB is not None else load_library()


def dims(weight_dtype: int = W_NVFP4, rms_eps: float = 1e-6) -> Dims:
    return Dims(HIDDEN, N_EXPERTS, N_SHARED, INTER, TOP_K, weight_dtype, rms_eps)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _expect(t, name, dtype, shape):
    """Marshalling check of one tensor argument: dtype, shape (None = any length
    of a 1-D tensor), contiguity, and residence on the current CUDA device.  The
    C ABI receives bare pointers and cannot check these; a wrong shape would make
    the kernels read or write outside the tensor."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is None:
        if t.dim() != 1:
            raise ValueError(f"{name}: expected a 1-D byte buffer, got shape {tuple(t.shape)}")
    elif tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if not t.is_cuda or t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name}: must be on the current CUDA device")


def _rows(x, name="x") -> int:
    """Token count of an activation tensor [rows][HIDDEN]."""
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(x).__name__}")
    if x.dim() != 2:
        raise ValueError(f"{name}: expected [tokens][{HIDDEN}], got shape {tuple(x.shape)}")
    return int(x.shape[0])


def _check_io(x, y, topk_ids, topk_w, layers=None):
    rows = _rows(x)
    _expect(x, "x", torch.bfloat16, (rows, HIDDEN))
    _expect(y, "y", torch.bfloat16, (rows, HIDDEN))
    lead = () if layers is None else (layers,)
    if topk_ids is not None:
        _expect(topk_ids, "topk_ids", torch.int32, lead + (rows, TOP_K))
    if topk_w is not None:
        _expect(topk_w, "topk_w", torch.float32, lead + (rows, TOP_K))
    return rows


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(rc: int, where: str):
    if rc != FLINT_MOE_OK:
        raise FlintMoeError(rc, where)


def packed_bytes(weight_dtype: int = W_NVFP4) -> int:
    d = dims(weight_dtype)
    return int(_lib().flint_moe_packed_bytes(ctypes.byref(d)))


def workspace_bytes(weight_dtype: int = W_NVFP4, max_tokens: int = MAX_DECODE_BATCH) -> int:
    d = dims(weight_dtype)
    return int(_lib().flint_moe_workspace_bytes(ctypes.byref(d), int(max_tokens)))


def pack_weights(gate_up, gate_up_scales, down, down_scales, packed, weight_dtype=W_NVFP4, stream=None):
    ne = N_EXPERTS + N_SHARED
    if weight_dtype == W_NVFP4:
        _expect(gate_up, "gate_up", torch.uint8, (ne, 2 * INTER, HIDDEN // 2))
        _expect(gate_up_scales, "gate_up_scales", torch.uint8, (ne, 2 * INTER, HIDDEN // 16))
        _expect(down, "down", torch.uint8, (ne, HIDDEN, INTER // 2))
        _expect(down_scales, "down_scales", torch.uint8, (ne, HIDDEN, INTER // 16))
    else:
        _expect(gate_up, "gate_up", torch.bfloat16, (ne, 2 * INTER, HIDDEN))
        _expect(down, "down", torch.bfloat16, (ne, HIDDEN, INTER))
    _expect(packed, "packed", torch.uint8, None)
    d = dims(weight_dtype)
    rc = _lib().flint_moe_pack_weights(ctypes.byref(d), _ptr(gate_up), _ptr(gate_up_scales), _ptr(down),
                                       _ptr(down_scales), _ptr(packed), packed.numel() * packed.element_size(),
                                       _stream(stream))
    _check(rc, "flint_moe_pack_weights")


class FlintLayer:
    """Device tensors of one sublayer: router weight, packed experts, scales, norm."""

    def __init__(self, router_w, experts, tensor_scales=None, norm_w=None, weight_dtype=W_NVFP4):
        self.router_w = router_w
        self.experts = experts
        self.tensor_scales = tensor_scales
        self.norm_w = norm_w
        self.weight_dtype = weight_dtype

    def c_struct(self) -> Layer:
        _expect(self.router_w, "router_w", torch.bfloat16, (N_EXPERTS, HIDDEN))
        _expect(self.experts, "experts", torch.uint8, None)
        if self.tensor_scales is not None:
            _expect(self.tensor_scales, "tensor_scales", torch.float32, (N_EXPERTS + N_SHARED, 2))
        if self.norm_w is not None:
            _expect(self.norm_w, "norm_w", torch.bfloat16, (HIDDEN,))
        return Layer(_ptr(self.router_w), _ptr(self.experts), _ptr(self.tensor_scales), _ptr(self.norm_w))


def pack_layer(plain: dict, device="cuda", stream=None) -> FlintLayer:
    """Packs one sublayer's plain tensors (as drawn by the input generator) on `device`."""
    fmt = W_NVFP4 if "gu_codes" in plain else W_BF16
    packed = torch.empty(packed_bytes(fmt), dtype=torch.uint8, device=device)
    if fmt == W_NVFP4:
        args = [plain[k].to(device).contiguous() for k in ("gu_codes", "gu_scales", "dn_codes", "dn_scales")]
        pack_weights(args[0], args[1], args[2], args[3], packed, fmt, stream)
        ts = plain["tensor_scales"].to(device=device, dtype=torch.float32).contiguous()
    else:
        gu = plain["gu_w"].to(device).contiguous()
        dn = plain["dn_w"].to(device).contiguous()
        pack_weights(gu, None, dn, None, packed, fmt, stream)
        args = [gu, dn]
        ts = None
    nw = None if plain.get("norm_w") is None else plain["norm_w"].to(device).contiguous()
    layer = FlintLayer(plain["router_w"].to(device).contiguous(), packed, ts, nw, fmt)
    layer._keepalive = args  # plain inputs must live until the pack kernel ran
    return layer


def decode_layer(layer: FlintLayer, x, y, ws, topk_ids=None, topk_w=None, rms_eps=1e-6, stream=None):
    d = dims(layer.weight_dtype, rms_eps)
    L = layer.c_struct()
    B = _check_io(x, y, topk_ids, topk_w)
    _expect(ws, "ws", torch.uint8, None)
    rc = _lib().flint_moe_decode_layer(ctypes.byref(d), ctypes.byref(L), _ptr(x), B, _ptr(y), _ptr(topk_ids),
                                       _ptr(topk_w), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "flint_moe_decode_layer")


def decode_layer_noalloc(layer: FlintLayer, x, y, topk_ids=None, topk_w=None, rms_eps=1e-6, stream=None):
    """decode_layer with the library's built-in scratch instead of a caller workspace.

    For callers that cannot allocate device memory.  Calls on one device share
    that scratch, so they must not overlap on the GPU.
    """
    d = dims(layer.weight_dtype, rms_eps)
    L = layer.c_struct()
    B = _check_io(x, y, topk_ids, topk_w)
    rc = _lib().flint_moe_decode_layer_noalloc(ctypes.byref(d), ctypes.byref(L), _ptr(x), B, _ptr(y),
                                               _ptr(topk_ids), _ptr(topk_w), _stream(stream))
    _check(rc, "flint_moe_decode_layer_noalloc")


def decode_stack(layers, x, y, ws, ids_per_layer=None, w_per_layer=None, ys_per_layer=None, rms_eps=1e-6,
                 stream=None):
    fmt = layers[0].weight_dtype
    d = dims(fmt, rms_eps)
    arr = (Layer * len(layers))(*[l.c_struct() for l in layers])
    B = _check_io(x, y, ids_per_layer, w_per_layer, layers=len(layers))
    if ys_per_layer is not None:
        _expect(ys_per_layer, "ys_per_layer", torch.bfloat16, (len(layers), B, HIDDEN))
    _expect(ws, "ws", torch.uint8, None)
    rc = _lib().flint_moe_decode_stack(ctypes.byref(d), arr, len(layers), _ptr(x), B, _ptr(y),
                                       _ptr(ids_per_layer), _ptr(w_per_layer), _ptr(ys_per_layer), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "flint_moe_decode_stack")


def prefill_layer(layer: FlintLayer, x, y, ws, topk_ids=None, topk_w=None, rms_eps=1e-6, stream=None):
    d = dims(layer.weight_dtype, rms_eps)
    L = layer.c_struct()
    T = _check_io(x, y, topk_ids, topk_w)
    _expect(ws, "ws", torch.uint8, None)
    rc = _lib().flint_moe_prefill_layer(ctypes.byref(d), ctypes.byref(L), _ptr(x), T, _ptr(y),
                                        _ptr(topk_ids), _ptr(topk_w), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream))
    _check(rc, "flint_moe_prefill_layer")


class DenseNVFP4:
    """A packed NVFP4 matrix [N][K] with its fp32 tensor scale, for dense_gemv."""

    def __init__(self, packed, N, K, tensor_scale):
        self.packed, self.N, self.K, self.tensor_scale = packed, int(N), int(K), float(tensor_scale)


def dense_packed_bytes(N: int, K: int) -> int:
    return int(_lib().flint_moe_dense_packed_bytes(int(N), int(K)))


def pack_dense(codes, scales, tensor_scale: float, device="cuda", stream=None) -> DenseNVFP4:
    """Packs a plain NVFP4 matrix (codes uint8 [N][K/2], scales uint8 [N][K/16])."""
    if not isinstance(codes, torch.Tensor) or codes.dim() != 2:
        raise ValueError("codes: expected a 2-D uint8 tensor [N][K/2]")
    N, K = int(codes.shape[0]), int(codes.shape[1]) * 2
    codes = codes.to(device).contiguous()
    scales = scales.to(device).contiguous()
    _expect(codes, "codes", torch.uint8, (N, K // 2))
    _expect(scales, "scales", torch.uint8, (N, K // 16))
    n = dense_packed_bytes(N, K)
    if n == 0:
        raise FlintMoeError(FLINT_MOE_ERR_UNSUPPORTED, "flint_moe_dense_packed_bytes")
    packed = torch.empty(n, dtype=torch.uint8, device=device)
    rc = _lib().flint_moe_pack_dense(_ptr(codes), _ptr(scales), N, K, _ptr(packed), n, _stream(stream))
    _check(rc, "flint_moe_pack_dense")
    w = DenseNVFP4(packed, N, K, tensor_scale)
    w._keepalive = (codes, scales)  # inputs must live until the pack kernel ran
    return w


def dense_gemv(w: DenseNVFP4, x, y, stream=None):
    """y[B][N] = bf16(tensor_scale * x[B][K] @ W^T) on the packed NVFP4 matrix."""
    B = _rows(x)
    _expect(x, "x", torch.bfloat16, (B, w.K))
    _expect(y, "y", torch.bfloat16, (B, w.N))
    _expect(w.packed, "packed", torch.uint8, None)
    rc = _lib().flint_moe_dense_gemv(_ptr(w.packed), w.N, w.K, w.tensor_scale, _ptr(x), B, _ptr(y), _stream(stream))
    _check(rc, "flint_moe_dense_gemv")


def release():
    _check(_lib().flint_moe_release(), "flint_moe_release")


def device_error(reset: bool = True) -> int:
    rc = _lib().flint_moe_device_error(1 if reset else 0)
    if rc < 0:
        raise FlintMoeError(rc, "flint_moe_device_error")
    return rc


def device_status(reset: bool = True) -> int:
    """The device error word mapped to a status: FLINT_MOE_OK, FLINT_MOE_ERR_TIMEOUT
    (a bounded device wait gave up) or FLINT_MOE_ERR_CUDA."""
    return int(_lib().flint_moe_device_status(1 if reset else 0))


def set_decode_kernel(kernel: int = DECODE_CHAINED):
    """Decode kernels of later NVFP4 calls: DECODE_CHAINED (default) or DECODE_PERSISTENT."""
    _check(_lib().flint_moe_set_decode_kernel(int(kernel)), "flint_moe_set_decode_kernel")


def set_wait_limit(cycles: int = 0):
    """Cycle limit of later NVFP4 decode calls' waits on data of their other thread
    blocks; 0 restores the default (about one second)."""
    _check(_lib().flint_moe_set_wait_limit(int(cycles)), "flint_moe_set_wait_limit")


def alloc_workspace(weight_dtype=W_NVFP4, max_tokens=MAX_DECODE_BATCH, device="cuda"):
    n = workspace_bytes(weight_dtype, max_tokens)
    if n == 0:
        raise FlintMoeError(FLINT_MOE_ERR_UNSUPPORTED, "flint_moe_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)
