"""GB300-native fused MoE expert layer.

The compute path is libmoe_layer.so (hand-written CUDA for sm_103a) behind the
C ABI declared in include/moe_layer.h; ``binding`` marshals torch tensors to
it and ``layer.MoELayer`` issues the calls of one layer in order.  Importing
this package does not load the library; ``load()`` does, and raises if it has
not been built.
"""
from .binding import (  # noqa: F401
    EXPORTED, LIB_PATH, MOE_BF16, MOE_DEVERR_CAPACITY, MOE_DEVERR_ID_RANGE, MOE_DEVERR_INTERNAL, MOE_DEVERR_TIMEOUT,
    MOE_E4M3, MOE_F32,
    MOE_IMPL_AUTO, MOE_IMPL_SIMT, MOE_IMPL_TCGEN05, MOE_IMPL_TCGEN05_MIXED, MOE_IMPL_TCGEN05_PAIR,
    MOE_IMPL_TCGEN05_SWAP_AB,
    MOE_LAYOUT_BATCHED,
    MOE_LAYOUT_CONTIGUOUS, MOE_W1_GATE_UP, MOE_W1_INTERLEAVE16, MOE_W_TILED, MoEError, load, moe_batched_topk_reduce, moe_batched_weight_reduce, moe_experts_fused,
    moe_experts_fused_workspace_size,
    moe_gemm1_swiglu, moe_gemm2, moe_max_padded_rows, moe_permute_align, moe_permute_align_static, moe_permute_workspace_size,
    moe_route_permute_align, moe_tile_weights,
    moe_topk_route, moe_unpermute_topk_reduce, moe_version, mxfp8_quantize_block32)


def MoELayer(*args, **kwargs):
    from .layer import MoELayer as _L
    return _L(*args, **kwargs)
