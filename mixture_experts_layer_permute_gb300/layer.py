"""The whole expert layer as the library's calls in order on one stream.

``MoELayer`` owns the device buffers of one layer shape, allocated once (the
workspace_shapes() idea of the "Fused MoE Modular Kernel" design doc: the
intermediates are declared up front and reused), and ``forward`` issues

    moe_route_permute_align (moe_topk_route + moe_permute_align) -> moe_gemm1_swiglu -> moe_gemm2
        -> moe_unpermute_topk_reduce          (contiguous layout)

with, for MXFP8 weights and ``act_quant=True``, the activations quantised on
the fly so that both GEMMs run block-scaled MXFP8 x MXFP8:

    ... moe_permute_align -> mxfp8_quantize_block32 (x rows) -> moe_gemm1_swiglu (h written as MXFP8
        by its epilogue) -> moe_gemm2 -> moe_unpermute_topk_reduce

or, for the batched layout fed with expert-major rows (T = 0),

    moe_gemm1_swiglu -> moe_gemm2 (route weight in the epilogue)
        [-> moe_batched_weight_reduce when the weight is not fused]

or, for the batched layout fed with tokens (T > 0),

    moe_route_permute_align (batched rows, capacity max_tokens)
        -> moe_gemm1_swiglu -> moe_gemm2 -> moe_batched_topk_reduce (token order)

Given ``topk_ids``/``topk_weights`` instead of router logits, moe_permute_align
takes the place of moe_route_permute_align.  There is no host synchronisation,
and every step runs in libmoe_layer's kernels.
The marshalled argument lists of the C calls are kept between calls with the
same tensors and stream, so a decode step spends a few microseconds per call
on the host; ``capture`` records one forward into a CUDA graph whose replay
re-runs the layer on the same tensors (new inputs are copied into them).
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


def _p(t):
    return None if t is None else t.data_ptr()


class MoELayer:
    def __init__(self, T: int, K: int, I: int, E: int, top_k: int, act_dtype=torch.bfloat16, block_m: int = 1,
                 layout: int = B.MOE_LAYOUT_CONTIGUOUS, max_tokens: int = 0, impl: int = B.MOE_IMPL_AUTO,
                 weight_in_gemm2: bool = True, device="cuda", act_quant: bool = False,
                 fused_experts: bool = True):
        self.T, self.K, self.I, self.E, self.top_k = T, K, I, E, top_k
        if act_quant and layout != B.MOE_LAYOUT_CONTIGUOUS:
            raise ValueError("act_quant (MXFP8 activations) is implemented for the contiguous layout")
        if act_quant and (K % 32 or I % 32):
            raise ValueError("act_quant needs K and I multiples of 32")
        self.act_quant = act_quant
        # GEMM 1 + GEMM 2 in one launch (moe_experts_fused) where the contiguous bf16 plan runs swap-AB tiles
        dev0 = torch.device(device)
        tc_device = dev0.type == "cuda" and torch.cuda.get_device_capability(dev0)[0] >= 10
        self.fused_experts = (fused_experts and tc_device and layout == B.MOE_LAYOUT_CONTIGUOUS and not act_quant
                              and impl in (B.MOE_IMPL_AUTO, B.MOE_IMPL_TCGEN05_SWAP_AB) and K % 128 == 0
                              and I % 64 == 0)
        self.block_m, self.layout, self.max_tokens, self.impl = block_m, layout, max_tokens, impl
        self.weight_in_gemm2 = weight_in_gemm2
        self.act_dtype = act_dtype
        self.lib = B.load()
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
            if self.fused_experts:
                self.fused_ws = torch.empty(max(B.moe_experts_fused_workspace_size(self.rows_cap, E), 256),
                                            dtype=torch.uint8, device=dev)
            if act_quant:
                u8 = dict(dtype=torch.uint8, device=dev)
                self.x_codes = torch.empty((self.rows_cap, K), **u8)
                self.x_scales = torch.empty((self.rows_cap, K // 32), **u8)
                self.h_codes = torch.empty((self.rows_cap, I), **u8)
                self.h_scales = torch.empty((self.rows_cap, I // 32), **u8)
        elif T > 0:   # batched rows, token input and output
            self.rows_cap = E * max_tokens
            self.ids = torch.empty((T, top_k), **i32)
            self.weights = torch.empty((T, top_k), dtype=torch.float32, device=dev)
            self.row_route = torch.empty(max(self.rows_cap, 1), **i32)
            self.route_row = torch.empty((T, top_k), **i32)
            self.workspace = torch.empty(max(B.moe_permute_workspace_size(T, top_k, E), 256), dtype=torch.uint8,
                                         device=dev)
            self.x_perm = torch.empty((max(self.rows_cap, 1), K), dtype=act_dtype, device=dev)
            self.h = torch.empty((E, max_tokens, I), dtype=act_dtype, device=dev)
            self.y = torch.empty((E, max_tokens, K), dtype=act_dtype, device=dev)
            self.out = torch.empty((T, K), dtype=act_dtype, device=dev)
        else:
            self.rows_cap = E * max_tokens
            self.h = torch.empty((E, max_tokens, I), dtype=act_dtype, device=dev)
            self.out = torch.empty((E, max_tokens, K), dtype=act_dtype, device=dev)
        self._plan_key = None
        self._plan = None

    # ---------------------------------------------------------------- planning
    def _check_inputs(self, x, w1, w2, logits, topk_ids, topk_weights, w1_scale, w2_scale, counts, row_weights):
        for t in (x, w1, w2, logits, topk_ids, topk_weights, w1_scale, w2_scale, counts, row_weights):
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise ValueError("MoELayer.forward takes contiguous device tensors")
        if w1.shape[0] != self.E or w2.shape[0] != self.E:
            raise ValueError("weight expert count does not match the layer")
        if logits is not None and tuple(logits.shape) != (self.T, self.E):
            raise ValueError(f"logits must be ({self.T}, {self.E})")
        if self.layout == B.MOE_LAYOUT_CONTIGUOUS or self.T > 0:
            if tuple(x.shape) != (self.T, self.K) or x.dtype != self.act_dtype:
                raise ValueError(f"x must be ({self.T}, {self.K}) {self.act_dtype}")
        elif tuple(x.shape) != (self.E, self.max_tokens, self.K):
            raise ValueError(f"x must be ({self.E}, {self.max_tokens}, {self.K})")

    def _build_plan(self, x, w1, w2, logits, topk_ids, topk_weights, w1_scale, w2_scale, w1_layout, counts,
                    row_weights, stream):
        lib = self.lib
        adt = B.dtype_code(x)
        wdt = B.dtype_code(w1, e4m3=w1_scale is not None)
        I, K, E, T, k = self.I, self.K, self.E, self.T, self.top_k
        # MOE_W_TILED: W1 and W2 both from moe_tile_weights (the fused decode launch, CTA-pair tiles, or MXFP8
        # codes on swap-AB tiles)
        w2_layout = B.MOE_W_TILED if w1_layout == B.MOE_W_TILED else B.MOE_W1_GATE_UP
        calls = []
        if self.layout == B.MOE_LAYOUT_BATCHED and T > 0:
            return self._token_batched_plan(x, w1, w2, logits, topk_ids, topk_weights, w1_scale, w2_scale,
                                            w1_layout, adt, wdt, stream)
        if self.layout == B.MOE_LAYOUT_BATCHED:
            mt = self.max_tokens
            calls.append((lib.moe_gemm1_swiglu, (x.data_ptr(), adt, None, self.layout, counts.data_ptr(), None, mt,
                                                 self.rows_cap, E, K, I, w1.data_ptr(), _p(w1_scale), wdt,
                                                 w1_layout, self.impl, self.h.data_ptr(), adt, None,
                                                 self.err.data_ptr(), stream), "gemm1"))
            rw = row_weights if self.weight_in_gemm2 else None
            calls.append((lib.moe_gemm2, (self.h.data_ptr(), adt, None, self.layout, counts.data_ptr(), None, mt,
                                          self.rows_cap, E, K, I, w2.data_ptr(), _p(w2_scale), wdt, w2_layout,
                                          None, _p(rw),
                                          self.impl, self.out.data_ptr(), adt, self.rows_cap, self.err.data_ptr(),
                                          stream), "gemm2"))
            if not self.weight_in_gemm2:
                calls.append((lib.moe_batched_weight_reduce, (self.out.data_ptr(), adt, counts.data_ptr(),
                                                              _p(row_weights), E, mt, K, self.out.data_ptr(), adt,
                                                              stream), "reduce"))
            return calls
        perm_args = (self.layout, self.block_m, 0, x.data_ptr(), adt, K, self.x_perm.data_ptr(), self.rows_cap,
                     self.counts.data_ptr(), self.offsets.data_ptr(), self.row_route.data_ptr(),
                     self.route_row.data_ptr(), self.workspace.data_ptr(), self.workspace.numel(),
                     self.err.data_ptr(), stream)
        if logits is not None:   # routing, placement and gather (one launch for decode-sized batches)
            calls.append((lib.moe_route_permute_align, (logits.data_ptr(), T, E, k, 1, self.ids.data_ptr(),
                                                        self.weights.data_ptr()) + perm_args, "route_permute"))
            ids, weights = self.ids, self.weights
        else:
            ids, weights = topk_ids, topk_weights
            calls.append((lib.moe_permute_align, (ids.data_ptr(), T, k, E) + perm_args, "permute"))
        if self.act_quant:
            if wdt != B.MOE_E4M3:
                raise ValueError("act_quant needs MXFP8 (E4M3 + scales) weights")
            calls.append((lib.mxfp8_quantize_block32, (self.x_perm.data_ptr(), adt, self.rows_cap, K,
                                                       self.x_codes.data_ptr(), self.x_scales.data_ptr(), stream),
                          "quant_x"))
            a1, a1dt, a1s = self.x_codes.data_ptr(), B.MOE_E4M3, self.x_scales.data_ptr()
        else:
            a1, a1dt, a1s = self.x_perm.data_ptr(), adt, None
        swap_regime = self.impl == B.MOE_IMPL_TCGEN05_SWAP_AB or self.rows_cap // max(E, 1) < 64
        if (self.fused_experts and swap_regime and adt == B.MOE_BF16 and wdt == B.MOE_BF16
                and self.weight_in_gemm2):
            calls.append((lib.moe_experts_fused, (self.x_perm.data_ptr(), adt, self.counts.data_ptr(),
                                                  self.offsets.data_ptr(), self.rows_cap, E, K, I, w1.data_ptr(),
                                                  w1_layout, w2.data_ptr(), wdt, self.row_route.data_ptr(),
                                                  weights.data_ptr(), self.h.data_ptr(), self.y.data_ptr(), adt,
                                                  T * k, self.fused_ws.data_ptr(), self.fused_ws.numel(),
                                                  self.err.data_ptr(), stream), "gemm1"))
            calls.append((lib.moe_unpermute_topk_reduce, (self.y.data_ptr(), adt, ids.data_ptr(), None, T, k, E,
                                                          K, self.out.data_ptr(), adt, stream), "reduce"))
            return calls
        if self.act_quant:   # GEMM 1's epilogue writes h as MXFP8 (codes + scales)
            hout, hdt, hs = self.h_codes.data_ptr(), B.MOE_E4M3, self.h_scales.data_ptr()
        else:
            hout, hdt, hs = self.h.data_ptr(), adt, None
        calls.append((lib.moe_gemm1_swiglu, (a1, a1dt, a1s, self.layout, self.counts.data_ptr(),
                                             self.offsets.data_ptr(), 0, self.rows_cap, E, K, I, w1.data_ptr(),
                                             _p(w1_scale), wdt, w1_layout, self.impl, hout, hdt, hs,
                                             self.err.data_ptr(), stream), "gemm1"))
        a2, a2dt, a2s = hout, hdt, hs
        rw = weights if self.weight_in_gemm2 else None
        calls.append((lib.moe_gemm2, (a2, a2dt, a2s, self.layout, self.counts.data_ptr(),
                                      self.offsets.data_ptr(), 0, self.rows_cap, E, K, I, w2.data_ptr(),
                                      _p(w2_scale), wdt, w2_layout, self.row_route.data_ptr(), _p(rw), self.impl,
                                      self.y.data_ptr(), adt, T * k, self.err.data_ptr(), stream), "gemm2"))
        calls.append((lib.moe_unpermute_topk_reduce, (self.y.data_ptr(), adt, ids.data_ptr(),
                                                      None if self.weight_in_gemm2 else weights.data_ptr(), T, k,
                                                      E, K, self.out.data_ptr(), adt, stream), "reduce"))
        return calls

    def _token_batched_plan(self, x, w1, w2, logits, topk_ids, topk_weights, w1_scale, w2_scale, w1_layout, adt,
                            wdt, stream):
        lib = self.lib
        I, K, E, T, k, mt = self.I, self.K, self.E, self.T, self.top_k, self.max_tokens
        calls = []
        perm_args = (self.layout, 1, mt, x.data_ptr(), adt, K, self.x_perm.data_ptr(), self.rows_cap,
                     self.counts.data_ptr(), self.offsets.data_ptr(), self.row_route.data_ptr(),
                     self.route_row.data_ptr(), self.workspace.data_ptr(), self.workspace.numel(),
                     self.err.data_ptr(), stream)
        if logits is not None:
            calls.append((lib.moe_route_permute_align, (logits.data_ptr(), T, E, k, 1, self.ids.data_ptr(),
                                                        self.weights.data_ptr()) + perm_args, "route_permute"))
            ids, weights = self.ids, self.weights
        else:
            ids, weights = topk_ids, topk_weights
            calls.append((lib.moe_permute_align, (ids.data_ptr(), T, k, E) + perm_args, "permute"))
        calls.append((lib.moe_gemm1_swiglu, (self.x_perm.data_ptr(), adt, None, self.layout, self.counts.data_ptr(), None,
                                             mt, self.rows_cap, E, K, I, w1.data_ptr(), _p(w1_scale), wdt,
                                             w1_layout, self.impl, self.h.data_ptr(), adt, None,
                                             self.err.data_ptr(), stream), "gemm1"))
        w2_layout = B.MOE_W_TILED if w1_layout == B.MOE_W_TILED else B.MOE_W1_GATE_UP
        calls.append((lib.moe_gemm2, (self.h.data_ptr(), adt, None, self.layout, self.counts.data_ptr(), None, mt,
                                      self.rows_cap, E, K, I, w2.data_ptr(), _p(w2_scale), wdt, w2_layout, None, None,
                                      self.impl, self.y.data_ptr(), adt, self.rows_cap, self.err.data_ptr(),
                                      stream), "gemm2"))
        calls.append((lib.moe_batched_topk_reduce, (self.y.data_ptr(), adt, self.rows_cap,
                                                    self.route_row.data_ptr(), weights.data_ptr(), T, k, K,
                                                    self.out.data_ptr(), adt, self.err.data_ptr(), stream),
                      "reduce"))
        return calls

    # ---------------------------------------------------------------- running
    def forward(self, x: torch.Tensor, w1: torch.Tensor, w2: torch.Tensor, logits: Optional[torch.Tensor] = None,
                topk_ids: Optional[torch.Tensor] = None, topk_weights: Optional[torch.Tensor] = None,
                w1_scale=None, w2_scale=None, w1_layout: int = B.MOE_W1_GATE_UP,
                expert_num_tokens: Optional[torch.Tensor] = None, row_weights: Optional[torch.Tensor] = None,
                stream=None, gemm1_events=None) -> torch.Tensor:
        """Runs the layer on `stream` (default: the current stream) and returns the output buffer.

        Contiguous layout, or batched layout with T > 0: x (T, K) and either router `logits` (T, E) or
        `topk_ids`/`topk_weights` (T, top_k); routes beyond max_tokens per expert are dropped (batched).
        Batched layout with T = 0: x (E, max_tokens, K), `expert_num_tokens` (E,), optional `row_weights`
        (E, max_tokens).
        ``w1_layout``: MOE_W1_GATE_UP or MOE_W1_INTERLEAVE16 for row-major W1, or MOE_W_TILED when W1 and W2 come
        from moe_tile_weights (bf16: the fused decode launch, or CTA-pair tiles where there are many rows per
        expert; MXFP8 codes: the swap-AB tiles, scales as stored; the library refuses other plans with
        MOE_ERR_UNSUPPORTED).
        ``gemm1_events`` = (start, end) CUDA events recorded around the gate/up GEMM.
        """
        s = stream if stream is not None else torch.cuda.current_stream()
        key = (_p(x), _p(w1), _p(w2), _p(logits), _p(topk_ids), _p(topk_weights), _p(w1_scale), _p(w2_scale),
               w1_layout, _p(expert_num_tokens), _p(row_weights), s.cuda_stream)
        if key != self._plan_key:
            self._check_inputs(x, w1, w2, logits, topk_ids, topk_weights, w1_scale, w2_scale, expert_num_tokens,
                               row_weights)
            self._plan = self._build_plan(x, w1, w2, logits, topk_ids, topk_weights, w1_scale, w2_scale, w1_layout,
                                          expert_num_tokens, row_weights, s.cuda_stream)
            self._plan_key = key
        for fn, args, name in self._plan:
            if gemm1_events is not None and name == "gemm1":
                gemm1_events[0].record(s)
            rc = fn(*args)
            if rc != B.MOE_OK:
                B._check(rc)
            if gemm1_events is not None and name == "gemm1":
                gemm1_events[1].record(s)
        return self.out

    def capture(self, x: torch.Tensor, w1: torch.Tensor, w2: torch.Tensor, before=None, after=None,
                **kwargs) -> torch.cuda.CUDAGraph:
        """Records one forward on (x, w1, w2, **kwargs) into a CUDA graph and returns it.

        ``graph.replay()`` then runs route/permute/GEMMs/reduce on the same tensors; write new inputs into
        them (or let ``before`` do it) and read ``self.out`` after the replay.  ``before`` and ``after`` are
        optional callables recorded around the forward, e.g. the copies of a step's inputs from pinned host
        buffers and of its output back.  One eager forward runs first (it builds the call plan and sets up the
        library on the device).
        """
        self.forward(x, w1, w2, **kwargs)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            if before is not None:
                before()
            self.forward(x, w1, w2, **kwargs)
            if after is not None:
                after()
        return graph

    def launches_per_forward(self) -> int:
        """Kernels one forward launches (for launch accounting)."""
        if self.layout == B.MOE_LAYOUT_BATCHED and self.T == 0:
            return 2 if self.weight_in_gemm2 else 3
        R = self.T * self.top_k
        routed = any(name == "route_permute" for _, _, name in (self._plan or []))
        if routed and 1 <= self.T <= 128 and R <= 1024:
            front = 1                                                 # route + permute + gather in one launch
        else:
            front = (1 if routed else 0) + (1 if R <= 1024 else 2) + 1   # route, permute, gather
        n = front + 3                                                 # gemm1 gemm2 reduce
        if any(name == "gemm1" and fn is self.lib.moe_experts_fused for fn, _, name in (self._plan or [])):
            n -= 1                                                    # GEMM 1 + GEMM 2 in one launch
        if self.act_quant:
            n += 1                                                    # quantise x rows (h: in GEMM 1)
        return n

    def device_errors(self, reset: bool = True) -> int:
        """Device error bits (MOE_DEVERR_*) accumulated since the last reset (synchronises)."""
        v = int(self.err.item())
        if reset:
            self.err.zero_()
        return v
