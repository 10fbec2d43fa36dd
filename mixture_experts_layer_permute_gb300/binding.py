"""ctypes binding of libmoe_layer.so: argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of the layer itself: it turns torch tensors into device pointers,
sizes and element-type codes, passes the current CUDA stream, allocates
outputs that the caller did not supply, and raises MoEError when the library
reports a failure.  If the library is missing, ``load()`` raises -- there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_layer.so")

# values of include/moe_layer.h
MOE_OK = 0
MOE_F32, MOE_BF16, MOE_E4M3 = 0, 1, 2
MOE_LAYOUT_CONTIGUOUS, MOE_LAYOUT_BATCHED = 0, 1
MOE_W1_GATE_UP, MOE_W1_INTERLEAVE16, MOE_W_TILED = 0, 1, 2
MOE_IMPL_AUTO, MOE_IMPL_TCGEN05, MOE_IMPL_TCGEN05_SWAP_AB, MOE_IMPL_SIMT, MOE_IMPL_TCGEN05_MIXED = 0, 1, 2, 3, 4
MOE_IMPL_TCGEN05_PAIR = 5
MOE_DEVERR_ID_RANGE, MOE_DEVERR_CAPACITY, MOE_DEVERR_TIMEOUT, MOE_DEVERR_INTERNAL = 1, 2, 4, 8

EXPORTED = [
    "moe_last_error", "moe_version", "moe_max_padded_rows", "moe_permute_workspace_size", "moe_topk_route",
    "moe_permute_align", "moe_permute_align_static", "moe_route_permute_align", "moe_gemm1_swiglu", "moe_gemm2", "moe_unpermute_topk_reduce",
    "moe_batched_weight_reduce", "moe_batched_topk_reduce", "mxfp8_quantize_block32",
    "moe_experts_fused_workspace_size", "moe_experts_fused", "moe_tile_weights",
]


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libmoe_layer status {status}: {msg}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None):
    """Loads libmoe_layer.so (built by build.py / __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libmoe_layer.so not found at {p}: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sig = {
            "moe_last_error": (ctypes.c_char_p, []),
            "moe_version": (I32, []),
            "moe_max_padded_rows": (I64, [I64, I32, I32, I32]),
            "moe_permute_workspace_size": (SZ, [I64, I32, I32]),
            "moe_experts_fused_workspace_size": (SZ, [I64, I32]),
            "moe_experts_fused": (I32, [P, I32, P, P, I64, I32, I64, I64, P, I32, P, I32, P, P, P, P, I32, I64, P,
                                        SZ, P, P]),
            "moe_topk_route": (I32, [P, I64, I32, I32, I32, P, P, P]),
            "moe_tile_weights": (I32, [P, I32, I32, I32, I32, I64, I64, P, P]),
            "moe_permute_align": (I32, [P, I64, I32, I32, I32, I32, I32, P, I32, I64, P, I64, P, P, P, P, P, SZ,
                                        P, P]),
            "moe_route_permute_align": (I32, [P, I64, I32, I32, I32, P, P, I32, I32, I32, P, I32, I64, P, I64, P,
                                              P, P, P, P, SZ, P, P]),
            "moe_permute_align_static": (I32, [P, I64, I32, I32, I32, I32, I32, P, I32, I64, P, I64, P, P, P, P,
                                               P, P]),
            "moe_gemm1_swiglu": (I32, [P, I32, P, I32, P, P, I32, I64, I32, I64, I64, P, P, I32, I32, I32, P,
                                       I32, P, P, P]),
            "moe_gemm2": (I32, [P, I32, P, I32, P, P, I32, I64, I32, I64, I64, P, P, I32, I32, P, P, I32, P, I32,
                                I64, P, P]),
            "moe_unpermute_topk_reduce": (I32, [P, I32, P, P, I64, I32, I32, I64, P, I32, P]),
            "moe_batched_weight_reduce": (I32, [P, I32, P, P, I32, I32, I64, P, I32, P]),
            "moe_batched_topk_reduce": (I32, [P, I32, I64, P, P, I64, I32, I64, P, I32, P, P]),
            "mxfp8_quantize_block32": (I32, [P, I32, I64, I64, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int):
    if status != MOE_OK:
        raise MoEError(status, load().moe_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe_layer takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libmoe_layer takes contiguous tensors")
    return t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def dtype_code(t: torch.Tensor, e4m3: bool = False) -> int:
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.uint8 and e4m3:
        return MOE_E4M3
    raise TypeError(f"unsupported element type {t.dtype}")


_TORCH = {MOE_F32: torch.float32, MOE_BF16: torch.bfloat16}


# ----------------------------------------------------------------------------
# the C entry points
# ----------------------------------------------------------------------------

def moe_version() -> int:
    return load().moe_version()


def moe_max_padded_rows(T: int, top_k: int, E: int, block_m: int) -> int:
    return load().moe_max_padded_rows(T, top_k, E, block_m)


def moe_permute_workspace_size(T: int, top_k: int, E: int) -> int:
    return load().moe_permute_workspace_size(T, top_k, E)


def moe_topk_route(logits, top_k, renormalize=True, topk_ids=None, topk_weights=None, stream=None):
    T, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    if topk_weights is None:
        topk_weights = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    _check(load().moe_topk_route(_ptr(logits), T, E, top_k, int(bool(renormalize)), _ptr(topk_ids),
                                 _ptr(topk_weights), _stream(stream)))
    return topk_ids, topk_weights


def moe_permute_align(topk_ids, E, layout=MOE_LAYOUT_CONTIGUOUS, block_m=1, max_tokens=0, x=None, x_out=None,
                      rows_cap=None, expert_counts=None, expert_offsets=None, row_route=None, route_row=None,
                      workspace=None, err_word=None, stream=None):
    """Returns dict(counts, offsets, row_route, route_row, x_out)."""
    T, top_k = topk_ids.shape
    dev = topk_ids.device
    if rows_cap is None:
        rows_cap = (moe_max_padded_rows(T, top_k, E, block_m) if layout == MOE_LAYOUT_CONTIGUOUS
                    else E * max_tokens)
    if expert_counts is None:
        expert_counts = torch.empty(E, dtype=torch.int32, device=dev)
    if expert_offsets is None:
        expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if row_route is None:
        row_route = torch.empty(max(rows_cap, 1), dtype=torch.int32, device=dev)
    if route_row is None:
        route_row = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(moe_permute_workspace_size(T, top_k, E), dtype=torch.uint8, device=dev)
    K, x_dtype = 0, MOE_BF16
    if x is not None:
        K = x.shape[-1]
        x_dtype = dtype_code(x)
        if x_out is None:
            x_out = torch.empty((rows_cap, K), dtype=x.dtype, device=dev)
    _check(load().moe_permute_align(
        _ptr(topk_ids), T, top_k, E, layout, block_m, max_tokens, _ptr(x), x_dtype, K, _ptr(x_out), rows_cap,
        _ptr(expert_counts), _ptr(expert_offsets), _ptr(row_route), _ptr(route_row), _ptr(workspace),
        workspace.numel(), _ptr(err_word), _stream(stream)))
    return dict(counts=expert_counts, offsets=expert_offsets, row_route=row_route, route_row=route_row,
                x_out=x_out, rows_cap=rows_cap)


def moe_tile_weights(w, which, w1_layout=MOE_W1_GATE_UP, out=None, stream=None):
    """Offline re-layout of W1 (which=1, (E, 2I, K) in w1_layout) or W2 (which=2, (E, K, I)) into the
    tile-contiguous layout the GEMMs read with MOE_W_TILED: bf16 weights, or E4M3 codes (uint8; W1 in the
    interleave-16 layout, the E8M0 scales unchanged).  Returns a tensor of w's shape holding the tiled bytes."""
    E, rows, cols = w.shape
    if out is None:
        out = torch.empty_like(w)
    _check(load().moe_tile_weights(_ptr(w), dtype_code(w, e4m3=True), which, w1_layout, E, rows, cols, _ptr(out),
                                   _stream(stream)))
    return out


def moe_route_permute_align(logits, top_k, E=None, renormalize=True, layout=MOE_LAYOUT_CONTIGUOUS, block_m=1,
                            max_tokens=0, x=None, x_out=None, rows_cap=None, topk_ids=None, topk_weights=None,
                            expert_counts=None, expert_offsets=None, row_route=None, route_row=None, workspace=None,
                            err_word=None, stream=None):
    """moe_topk_route then moe_permute_align in one call (one launch for decode-sized batches).
    Returns dict(topk_ids, topk_weights, counts, offsets, row_route, route_row, x_out)."""
    T, E_logits = logits.shape
    E = E_logits if E is None else E
    dev = logits.device
    if rows_cap is None:
        rows_cap = (moe_max_padded_rows(T, top_k, E, block_m) if layout == MOE_LAYOUT_CONTIGUOUS
                    else E * max_tokens)
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((T, top_k), dtype=torch.float32, device=dev)
    if expert_counts is None:
        expert_counts = torch.empty(E, dtype=torch.int32, device=dev)
    if expert_offsets is None:
        expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if row_route is None:
        row_route = torch.empty(max(rows_cap, 1), dtype=torch.int32, device=dev)
    if route_row is None:
        route_row = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(moe_permute_workspace_size(T, top_k, E), dtype=torch.uint8, device=dev)
    K, x_dtype = 0, MOE_BF16
    if x is not None:
        K = x.shape[-1]
        x_dtype = dtype_code(x)
        if x_out is None:
            x_out = torch.empty((rows_cap, K), dtype=x.dtype, device=dev)
    _check(load().moe_route_permute_align(
        _ptr(logits), T, E, top_k, int(bool(renormalize)), _ptr(topk_ids), _ptr(topk_weights), layout, block_m,
        max_tokens, _ptr(x), x_dtype, K, _ptr(x_out), rows_cap, _ptr(expert_counts), _ptr(expert_offsets),
        _ptr(row_route), _ptr(route_row), _ptr(workspace), workspace.numel(), _ptr(err_word), _stream(stream)))
    return dict(topk_ids=topk_ids, topk_weights=topk_weights, counts=expert_counts, offsets=expert_offsets,
                row_route=row_route, route_row=route_row, x_out=x_out, rows_cap=rows_cap)


def moe_permute_align_static(topk_ids, E, layout=MOE_LAYOUT_CONTIGUOUS, block_m=1, max_tokens=0, x=None,
                             x_out=None, rows_cap=None, expert_counts=None, expert_offsets=None, row_route=None,
                             route_row=None, err_word=None, stream=None):
    """moe_permute_align with the library's built-in scratch instead of a workspace (no allocation in the
    library).  Returns dict(counts, offsets, row_route, route_row, x_out)."""
    T, top_k = topk_ids.shape
    dev = topk_ids.device
    if rows_cap is None:
        rows_cap = (moe_max_padded_rows(T, top_k, E, block_m) if layout == MOE_LAYOUT_CONTIGUOUS
                    else E * max_tokens)
    if expert_counts is None:
        expert_counts = torch.empty(E, dtype=torch.int32, device=dev)
    if expert_offsets is None:
        expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if row_route is None:
        row_route = torch.empty(max(rows_cap, 1), dtype=torch.int32, device=dev)
    if route_row is None:
        route_row = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    K, x_dtype = 0, MOE_BF16
    if x is not None:
        K = x.shape[-1]
        x_dtype = dtype_code(x)
        if x_out is None:
            x_out = torch.empty((rows_cap, K), dtype=x.dtype, device=dev)
    _check(load().moe_permute_align_static(
        _ptr(topk_ids), T, top_k, E, layout, block_m, max_tokens, _ptr(x), x_dtype, K, _ptr(x_out), rows_cap,
        _ptr(expert_counts), _ptr(expert_offsets), _ptr(row_route), _ptr(route_row), _ptr(err_word),
        _stream(stream)))
    return dict(counts=expert_counts, offsets=expert_offsets, row_route=row_route, route_row=route_row,
                x_out=x_out, rows_cap=rows_cap)


def moe_gemm1_swiglu(a, expert_counts, expert_offsets, w1, I, layout=MOE_LAYOUT_CONTIGUOUS, max_tokens=0,
                     w1_scale=None, w1_layout=MOE_W1_GATE_UP, impl=MOE_IMPL_AUTO, h=None, h_dtype=None,
                     err_word=None, stream=None, a_scale=None, h_scale=None):
    """a_scale: E8M0 scales when `a` holds E4M3 codes (uint8) of MXFP8 activations.
    h_dtype=MOE_E4M3: h is written as MXFP8 (E4M3 codes + E8M0 scales); returns (h, h_scale) then."""
    E = w1.shape[0]
    K = w1.shape[-1]
    rows_cap = a.shape[0] if layout == MOE_LAYOUT_CONTIGUOUS else E * max_tokens
    a_dt = dtype_code(a, e4m3=a_scale is not None)
    if h_dtype is None:
        h_dtype = MOE_BF16 if a_dt == MOE_E4M3 else a_dt
    shape = (rows_cap, I) if layout == MOE_LAYOUT_CONTIGUOUS else (E, max_tokens, I)
    if h is None:
        h = torch.empty(shape, dtype=torch.uint8 if h_dtype == MOE_E4M3 else _TORCH[h_dtype], device=a.device)
    if h_dtype == MOE_E4M3 and h_scale is None:
        h_scale = torch.empty(shape[:-1] + (I // 32,), dtype=torch.uint8, device=a.device)
    _check(load().moe_gemm1_swiglu(
        _ptr(a), a_dt, _ptr(a_scale), layout, _ptr(expert_counts), _ptr(expert_offsets), max_tokens, rows_cap, E, K,
        I,
        _ptr(w1), _ptr(w1_scale), dtype_code(w1, e4m3=w1_scale is not None), w1_layout, impl, _ptr(h), h_dtype,
        _ptr(h_scale), _ptr(err_word), _stream(stream)))
    return (h, h_scale) if h_dtype == MOE_E4M3 else h


def moe_gemm2(h, expert_counts, expert_offsets, w2, y_rows, layout=MOE_LAYOUT_CONTIGUOUS, max_tokens=0,
              w2_scale=None, row_route=None, route_weights=None, impl=MOE_IMPL_AUTO, y=None, y_dtype=None,
              err_word=None, stream=None, h_scale=None, w2_layout=MOE_W1_GATE_UP):
    """h_scale: E8M0 scales when `h` holds E4M3 codes (uint8) of an MXFP8 intermediate.
    w2_layout: MOE_W1_GATE_UP (row-major) or MOE_W_TILED (W2 from moe_tile_weights)."""
    E, K, I = w2.shape
    rows_cap = h.shape[0] if layout == MOE_LAYOUT_CONTIGUOUS else E * max_tokens
    h_dt = dtype_code(h, e4m3=h_scale is not None)
    if y_dtype is None:
        y_dtype = MOE_BF16 if h_dt == MOE_E4M3 else h_dt
    if y is None:
        shape = (y_rows, K) if layout == MOE_LAYOUT_CONTIGUOUS else (E, max_tokens, K)
        y = torch.empty(shape, dtype=_TORCH[y_dtype], device=h.device)
    _check(load().moe_gemm2(
        _ptr(h), h_dt, _ptr(h_scale), layout, _ptr(expert_counts), _ptr(expert_offsets), max_tokens, rows_cap, E,
        K, I,
        _ptr(w2), _ptr(w2_scale), dtype_code(w2, e4m3=w2_scale is not None), w2_layout, _ptr(row_route),
        _ptr(route_weights), impl, _ptr(y), y_dtype, y_rows, _ptr(err_word), _stream(stream)))
    return y


def moe_experts_fused_workspace_size(rows_cap: int, E: int) -> int:
    return load().moe_experts_fused_workspace_size(rows_cap, E)


def moe_experts_fused(a, expert_counts, expert_offsets, w1, w2, I, row_route, y_rows, route_weights=None,
                      w1_layout=MOE_W1_GATE_UP, h=None, y=None, y_dtype=None, workspace=None, err_word=None,
                      stream=None):
    """GEMM 1 + GEMM 2 in one launch (bf16, contiguous layout, swap-AB tiles).  Returns (h, y)."""
    E, K, _ = w2.shape
    rows_cap = a.shape[0]
    if y_dtype is None:
        y_dtype = dtype_code(a)
    if h is None:
        h = torch.empty((rows_cap, I), dtype=torch.bfloat16, device=a.device)
    if y is None:
        y = torch.empty((y_rows, K), dtype=_TORCH[y_dtype], device=a.device)
    if workspace is None:
        workspace = torch.empty(max(moe_experts_fused_workspace_size(rows_cap, E), 256), dtype=torch.uint8,
                                device=a.device)
    _check(load().moe_experts_fused(
        _ptr(a), dtype_code(a), _ptr(expert_counts), _ptr(expert_offsets), rows_cap, E, K, I, _ptr(w1), w1_layout,
        _ptr(w2), dtype_code(w2), _ptr(row_route), _ptr(route_weights), _ptr(h), _ptr(y), y_dtype, y_rows,
        _ptr(workspace), workspace.numel(), _ptr(err_word), _stream(stream)))
    return h, y


def moe_unpermute_topk_reduce(y, topk_ids, E, topk_weights=None, out=None, out_dtype=None, stream=None):
    T, top_k = topk_ids.shape
    K = y.shape[-1]
    if out_dtype is None:
        out_dtype = dtype_code(y)
    if out is None:
        out = torch.empty((T, K), dtype=_TORCH[out_dtype], device=y.device)
    _check(load().moe_unpermute_topk_reduce(_ptr(y), dtype_code(y), _ptr(topk_ids), _ptr(topk_weights), T, top_k,
                                            E, K, _ptr(out), out_dtype, _stream(stream)))
    return out


def moe_batched_weight_reduce(y, expert_num_tokens, row_weights=None, out=None, out_dtype=None, stream=None):
    E, max_tokens, K = y.shape
    if out_dtype is None:
        out_dtype = dtype_code(y)
    if out is None:
        out = torch.empty((E, max_tokens, K), dtype=_TORCH[out_dtype], device=y.device)
    _check(load().moe_batched_weight_reduce(_ptr(y), dtype_code(y), _ptr(expert_num_tokens), _ptr(row_weights),
                                            E, max_tokens, K, _ptr(out), out_dtype, _stream(stream)))
    return out


def moe_batched_topk_reduce(y, route_row, topk_weights=None, out=None, out_dtype=None, err_word=None,
                            stream=None):
    """y: (E, max_tokens, K) or (rows, K); route_row: (T, top_k) or (T*top_k,) with top_k given by
    topk_weights when it is flat."""
    K = y.shape[-1]
    rows = y.numel() // K
    if route_row.dim() == 2:
        T, top_k = route_row.shape
    else:
        T, top_k = topk_weights.shape
    if out_dtype is None:
        out_dtype = dtype_code(y)
    if out is None:
        out = torch.empty((T, K), dtype=_TORCH[out_dtype], device=y.device)
    _check(load().moe_batched_topk_reduce(_ptr(y), dtype_code(y), rows, _ptr(route_row), _ptr(topk_weights), T,
                                          top_k, K, _ptr(out), out_dtype, _ptr(err_word), _stream(stream)))
    return out


def mxfp8_quantize_block32(x, codes=None, scales=None, stream=None):
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (cols // 32,), dtype=torch.uint8, device=x.device)
    _check(load().mxfp8_quantize_block32(_ptr(x), dtype_code(x), rows, cols, _ptr(codes), _ptr(scales),
                                         _stream(stream)))
    return codes, scales
