"""GB300 (sm_103a) Flint MoE sublayer: C-ABI CUDA library plus a thin binding.

The compute path is libflint_moe.so (csrc/, declared in include/flint_moe.h);
``flint_moe`` marshals torch tensors into its entry points.
"""

from .flint_moe import (  # noqa: F401
    W_NVFP4,
    W_BF16,
    FlintLayer,
    FlintMoeError,
    alloc_workspace,
    decode_layer,
    decode_stack,
    device_error,
    load_library,
    pack_layer,
    pack_weights,
    packed_bytes,
    prefill_layer,
    release,
    workspace_bytes,
)
