"""The whole expert layer as the library's calls in order on one stream.

``MoELayer`` owns the device buffers of one layer shape, allocated once (the
workspace_shapes() idea of the "Fused MoE Modular Kernel" design doc: the
intermediates are declared up front and reused), and ``forward`` issues

    moe_topk_route -> moe_permute_align -> moe_gemm1_swiglu -> moe_gemm2
        -> moe_unpermute_topk_reduce          (contiguous layout)

or, for the batched layout,

    moe_gemm1_swiglu -> moe_gemm2 (route weight in the epilogue)

with no host synchronisation.  Every step runs in libmoe_layer's kernels.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class MoELayer:
    def __init__(self, T: int, K: int, I: int, E: int, top_k: int, act_dtype=torch.bfloat16, block_m: int = 1,
                 layout: int = B.MOE_LAYOUT_CONTIGUOUS, max_tokens: int = 0, impl: int = B.MOE_IMPL_AUTO,
                 weight_in_gemm2: bool = True, device="cuda"):
        self.T, self.K, self.I, self.E, self.top_k = T, K, I, E, top_k
        self.block_m, self.layout, self.max_tokens, self.impl = block_m, layout, max_tokens, impl
        self.weight_in_gemm2 = weight_in_gemm2
        self.act_dtype = act_dtype
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.err = torch.zeros(1, **i32)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        if layout == B.MOE_LAYOUT_CONTIGUOUS:
            self.rows_cap = B.moe_max_padded_rows(T, top_k, E, block_m)
            self.ids = torch.empty((T, top_k), **i32)
            self.weights = torch.empty((T, top_k), dtype=torch.float32, device=dev)
            self.row_route = torch.empty(max(self.rows_cap, 1), **i32)
            self.route_row = torch.empty((T, top_k), **i32)
            self.workspace = torch.empty(max(B.moe_permute_workspace_size(T, top_k, E), 256), dtype=torch.uint8,
                                         device=dev)
            self.x_perm = torch.empty((self.rows_cap, K), dtype=act_dtype, device=dev)
            self.h = torch.empty((self.rows_cap, I), dtype=act_dtype, device=dev)
            self.y = torch.empty((T * top_k, K), dtype=act_dtype, device=dev)
            self.out = torch.empty((T, K), dtype=act_dtype, device=dev)
        else:
            self.rows_cap = E * max_tokens
            self.h = torch.empty((E, max_tokens, I), dtype=act_dtype, device=dev)
            self.out = torch.empty((E, max_tokens, K), dtype=act_dtype, device=dev)

    def forward(self, x: torch.Tensor, w1: torch.Tensor, w2: torch.Tensor, logits: Optional[torch.Tensor] = None,
                topk_ids: Optional[torch.Tensor] = None, topk_weights: Optional[torch.Tensor] = None,
                w1_scale=None, w2_scale=None, w1_layout: int = B.MOE_W1_GATE_UP,
                expert_num_tokens: Optional[torch.Tensor] = None, row_weights: Optional[torch.Tensor] = None,
                stream=None, gemm1_events=None) -> torch.Tensor:
        """Runs the layer; ``gemm1_events`` = (start, end) CUDA events recorded around the gate/up GEMM."""
        if self.layout == B.MOE_LAYOUT_BATCHED:
            return self._forward_batched(x, w1, w2, expert_num_tokens, row_weights, w1_scale, w2_scale, w1_layout,
                                         stream, gemm1_events)
        if logits is not None:
            B.moe_topk_route(logits, self.top_k, True, self.ids, self.weights, stream=stream)
            ids, weights = self.ids, self.weights
        else:
            ids, weights = topk_ids, topk_weights
        B.moe_permute_align(ids, self.E, B.MOE_LAYOUT_CONTIGUOUS, self.block_m, 0, x=x, x_out=self.x_perm,
                            rows_cap=self.rows_cap, expert_counts=self.counts, expert_offsets=self.offsets,
                            row_route=self.row_route, route_row=self.route_row, workspace=self.workspace,
                            err_word=self.err, stream=stream)
        if gemm1_events is not None:
            gemm1_events[0].record(stream)
        B.moe_gemm1_swiglu(self.x_perm, self.counts, self.offsets, w1, self.I, w1_scale=w1_scale,
                           w1_layout=w1_layout, impl=self.impl, h=self.h, err_word=self.err, stream=stream)
        if gemm1_events is not None:
            gemm1_events[1].record(stream)
        B.moe_gemm2(self.h, self.counts, self.offsets, w2, self.T * self.top_k, w2_scale=w2_scale,
                    row_route=self.row_route, route_weights=weights if self.weight_in_gemm2 else None,
                    impl=self.impl, y=self.y, err_word=self.err, stream=stream)
        B.moe_unpermute_topk_reduce(self.y, ids, self.E, None if self.weight_in_gemm2 else weights, out=self.out,
                                    stream=stream)
        return self.out

    def _forward_batched(self, xb, w1, w2, counts, row_weights, w1_scale, w2_scale, w1_layout, stream,
                         gemm1_events=None):
        if gemm1_events is not None:
            gemm1_events[0].record(stream)
        B.moe_gemm1_swiglu(xb, counts, None, w1, self.I, layout=B.MOE_LAYOUT_BATCHED, max_tokens=self.max_tokens,
                           w1_scale=w1_scale, w1_layout=w1_layout, impl=self.impl, h=self.h, err_word=self.err,
                           stream=stream)
        if gemm1_events is not None:
            gemm1_events[1].record(stream)
        if self.weight_in_gemm2:
            B.moe_gemm2(self.h, counts, None, w2, self.rows_cap, layout=B.MOE_LAYOUT_BATCHED,
                        max_tokens=self.max_tokens, w2_scale=w2_scale, route_weights=row_weights, impl=self.impl,
                        y=self.out, err_word=self.err, stream=stream)
        else:
            B.moe_gemm2(self.h, counts, None, w2, self.rows_cap, layout=B.MOE_LAYOUT_BATCHED,
                        max_tokens=self.max_tokens, w2_scale=w2_scale, impl=self.impl, y=self.out,
                        err_word=self.err, stream=stream)
            B.moe_batched_weight_reduce(self.out, counts, row_weights, out=self.out, stream=stream)
        return self.out

    def device_errors(self, reset: bool = True) -> int:
        """Device error bits (MOE_DEVERR_*) accumulated since the last reset (synchronises)."""
        v = int(self.err.item())
        if reset:
            self.err.zero_()
        return v
