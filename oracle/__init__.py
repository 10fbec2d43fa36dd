"""CPU oracle for the fused MoE expert layer -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 reference written in C (``moe_oracle.c``) and wrapped here
with ctypes and numpy.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The CUDA library never imports, links or calls anything in this package, and
this package never imports the CUDA library.

Arrays are numpy arrays.  bf16 values travel as ``np.uint16`` bit patterns,
E4M3 codes and E8M0 scales as ``np.uint8``.  Every function cites, in its
docstring, the passage of the sources it follows (see ``moe_oracle.c`` for the
full list of sources and readings).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoe_oracle.so")

F32, BF16, E4M3, F64 = 0, 1, 2, 3
ERR_ID_RANGE, ERR_CAPACITY = 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE semantics: no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fvisibility=hidden", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        sig = {
            "oracle_bf16_to_double": (D, [ctypes.c_uint16]),
            "oracle_round_f32": (ctypes.c_float, [D]),
            "oracle_double_to_bf16": (ctypes.c_uint16, [D]),
            "oracle_e4m3_to_double": (D, [ctypes.c_uint8]),
            "oracle_double_to_e4m3": (ctypes.c_uint8, [D]),
            "oracle_e8m0_to_double": (D, [ctypes.c_uint8]),
            "oracle_mxfp8_scale_code": (ctypes.c_uint8, [D]),
            "oracle_mxfp8_quantize": (I32, [P, I32, I64, I64, P, P]),
            "oracle_mxfp8_dequantize": (I32, [P, P, I64, I64, P]),
            "oracle_topk_route": (I32, [P, I64, I32, I32, I32, P, P]),
            "oracle_permute_contiguous": (I32, [P, I64, I32, I32, I32, P, P, P, P]),
            "oracle_permute_batched": (I32, [P, I64, I32, I32, I32, P, P, P]),
            "oracle_expert_gate_up": (I32, [P, I32, I64, P, P, P, I32, I32, I32, I64, I64, P, I32]),
            "oracle_expert_down": (I32, [P, I32, I64, P, P, P, I32, I32, I64, I64, P, I32]),
            "oracle_topk_reduce": (I32, [P, I32, P, P, I64, I32, I64, P, I32]),
            "oracle_batched_topk_reduce": (I32, [P, I32, I64, P, P, I64, I32, I64, P, I32]),
            "oracle_moe_layer": (I32, [P, I32, I64, I64, I64, I32, I32, P, P, P, P, P, P, I32, I32, I32, I32,
                                       P, I32]),
            "oracle_moe_layer_batched": (I32, [P, I32, I32, I64, P, P, I64, I64, P, P, P, P, I32, I32, I32, I32,
                                               P, I32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def _dtype_code(a: np.ndarray, e4m3: bool = False) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.uint8 and e4m3:
        return E4M3
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle: unsupported element type {a.dtype}")


def _c(a):
    """Contiguous array and its address (None -> NULL)."""
    if a is None:
        return None, None
    a = np.ascontiguousarray(a)
    return a, a.ctypes.data


_OUT_NP = {F32: np.float32, BF16: np.uint16, E4M3: np.uint8, F64: np.float64}


# ----------------------------------------------------------------------------
# scalar codecs
# ----------------------------------------------------------------------------

def bf16_to_double(h: int) -> float:
    return _load().oracle_bf16_to_double(h)


def double_to_bf16(v: float) -> int:
    return _load().oracle_double_to_bf16(v)


def round_f32(v: float) -> float:
    return _load().oracle_round_f32(v)


def e4m3_to_double(c: int) -> float:
    return _load().oracle_e4m3_to_double(c)


def double_to_e4m3(v: float) -> int:
    return _load().oracle_double_to_e4m3(v)


def e8m0_to_double(c: int) -> float:
    return _load().oracle_e8m0_to_double(c)


def mxfp8_scale_code(blockmax: float) -> int:
    """Scale code of one block ("Cake MegaMoE" PR analysis, section 2, _quantize_mxfp8_block32 "After")."""
    return _load().oracle_mxfp8_scale_code(blockmax)


# ----------------------------------------------------------------------------
# the layer's steps
# ----------------------------------------------------------------------------

def mxfp8_quantize(x: np.ndarray):
    """Block-32 MXFP8 quantisation along the last axis.  Returns (codes u8, scales u8)."""
    x, px = _c(x)
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    cols = x.shape[-1]
    codes = np.empty(x.shape, np.uint8)
    scales = np.empty(x.shape[:-1] + (cols // 32,), np.uint8)
    rc = _load().oracle_mxfp8_quantize(px, _dtype_code(x), rows, cols, codes.ctypes.data, scales.ctypes.data)
    if rc != 0:
        raise ValueError("oracle: cols must be a multiple of 32")
    return codes, scales


def mxfp8_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Decoded MXFP8 values in fp64: E4M3(code) * 2^(scale - 127), one scale per 32 along the last axis."""
    codes, pc = _c(np.asarray(codes, np.uint8))
    scales, ps = _c(np.asarray(scales, np.uint8))
    cols = codes.shape[-1]
    rows = codes.size // cols if cols else 0
    out = np.empty(codes.shape, np.float64)
    if _load().oracle_mxfp8_dequantize(pc, ps, rows, cols, out.ctypes.data) != 0:
        raise ValueError("oracle: cols must be a multiple of 32")
    return out


def _quant_h_mode(quant_h) -> int:
    """quant_h: False (no intermediate quantisation), True or "f32" (h rounded to binary32 first), "bf16"."""
    if quant_h is False or quant_h is None or quant_h == 0:
        return 0
    if quant_h == "bf16":
        return 2
    return 1


def topk_route(logits: np.ndarray, top_k: int, renormalize: bool = True):
    """Top-k routing ("Fused MoE Modular Kernel", How-To: select_experts / topk ids)."""
    logits, pl = _c(np.asarray(logits, np.float32))
    T, E = logits.shape
    ids = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float32)
    rc = _load().oracle_topk_route(pl, T, E, top_k, int(renormalize), ids.ctypes.data, w.ctypes.data)
    if rc != 0:
        raise ValueError("oracle: bad top_k")
    return ids, w


def permute_contiguous(ids: np.ndarray, E: int, block_m: int = 1):
    """Contiguous-layout permute ("Fused MoE Modular Kernel", apply(): Permute).

    Returns dict(counts, offsets, sorted_route, route_row, err).
    """
    ids, pi = _c(np.asarray(ids, np.int32))
    T, k = ids.shape
    cap = T * k + E * (block_m - 1)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    sorted_route = np.full(max(cap, 1), -7, np.int32)
    route_row = np.empty(T * k, np.int32)
    err = _load().oracle_permute_contiguous(pi, T, k, E, block_m, counts.ctypes.data, offsets.ctypes.data,
                                            sorted_route.ctypes.data, route_row.ctypes.data)
    return dict(counts=counts, offsets=offsets, sorted_route=sorted_route[: offsets[E]].copy(),
                route_row=route_row.reshape(T, k), err=err)


def permute_batched(ids: np.ndarray, E: int, max_tokens: int):
    """Batched-layout permute ("Fused MoE Modular Kernel", Introduction: Batched format)."""
    ids, pi = _c(np.asarray(ids, np.int32))
    T, k = ids.shape
    ent = np.empty(E, np.int32)
    row_route = np.empty(E * max_tokens, np.int32)
    route_row = np.empty(T * k, np.int32)
    err = _load().oracle_permute_batched(pi, T, k, E, max_tokens, ent.ctypes.data, row_route.ctypes.data,
                                         route_row.ctypes.data)
    return dict(expert_num_tokens=ent, row_route=row_route.reshape(E, max_tokens),
                route_row=route_row.reshape(T, k), err=err)


def expert_gate_up(x, row_expert, w1, w1_scale=None, w1_layout=0, I=None, out=F64):
    """h = silu(x W1_gate^T) * (x W1_up^T) per row ("Fused MoE Modular Kernel", apply(): W1, Act + Mul)."""
    x, px = _c(x)
    re_, pre = _c(np.asarray(row_expert, np.int32))
    w1, pw = _c(w1)
    s1, ps = _c(w1_scale)
    E, two_i, K = w1.shape
    I = two_i // 2
    n = x.shape[0]
    h = np.empty((n, I), _OUT_NP[out])
    _load().oracle_expert_gate_up(px, _dtype_code(x), n, pre, pw, ps, _dtype_code(w1, e4m3=True), w1_layout,
                                  E, K, I, h.ctypes.data, out)
    return h


def expert_down(h, row_expert, w2, w2_scale=None, out=F64):
    """y = h W2^T per row ("Fused MoE Modular Kernel", apply(): Matmul with W2)."""
    h, ph = _c(h)
    re_, pre = _c(np.asarray(row_expert, np.int32))
    w2, pw = _c(w2)
    s2, ps = _c(w2_scale)
    E, K, I = w2.shape
    n = h.shape[0]
    y = np.empty((n, K), _OUT_NP[out])
    _load().oracle_expert_down(ph, _dtype_code(h), n, pre, pw, ps, _dtype_code(w2, e4m3=True), E, K, I,
                               y.ctypes.data, out)
    return y


def topk_reduce(y_slots, ids, weights=None, out=F64):
    """Ordered weight-and-reduce over the top-k slots ("Fused MoE Modular Kernel", TopKWeightAndReduce;
    "Cake MegaMoE" PR analysis, section 3: ordered Top-K reduce)."""
    y_slots, py = _c(y_slots)
    ids, pi = _c(np.asarray(ids, np.int32))
    w, pw = _c(None if weights is None else np.asarray(weights, np.float32))
    T, k = ids.shape
    K = y_slots.shape[-1]
    o = np.empty((T, K), _OUT_NP[out])
    _load().oracle_topk_reduce(py, _dtype_code(y_slots), pi, pw, T, k, K, o.ctypes.data, out)
    return o


def batched_topk_reduce(y_rows, route_row, weights=None, out=F64):
    """Batched-format weight-and-reduce into token order ("Fused MoE Modular Kernel", TopKWeightAndReduce,
    NaiveBatched): out[t] = sum_j w[t,j] * y_rows[route_row[t,j]] over rows != -1, j increasing.
    y_rows: (E, max_tokens, K) or (rows, K); route_row: (T, k).  Returns (out, err_bits)."""
    y_rows, py = _c(y_rows)
    rr, pr = _c(np.asarray(route_row, np.int32))
    w, pw = _c(None if weights is None else np.asarray(weights, np.float32))
    T, k = rr.shape
    K = y_rows.shape[-1]
    rows = y_rows.size // K if K else 0
    o = np.empty((T, K), _OUT_NP[out])
    err = _load().oracle_batched_topk_reduce(py, _dtype_code(y_rows), rows, pr, pw, T, k, K, o.ctypes.data, out)
    return o, err


def moe_layer(x, ids, weights, w1, w2, w1_scale=None, w2_scale=None, w1_layout=0, quant_h=False, out=F64,
              quant_x=False):
    """The whole contiguous layer; returns (out, err_bits).  quant_x: x rows MXFP8-quantised before W1;
    quant_h: see _quant_h_mode."""
    x, px = _c(x)
    ids, pi = _c(np.asarray(ids, np.int32))
    w, pw = _c(None if weights is None else np.asarray(weights, np.float32))
    w1, p1 = _c(w1)
    w2, p2 = _c(w2)
    s1, ps1 = _c(w1_scale)
    s2, ps2 = _c(w2_scale)
    T, K = x.shape
    E, two_i, _ = w1.shape
    k = ids.shape[1]
    o = np.empty((T, K), _OUT_NP[out])
    err = _load().oracle_moe_layer(px, _dtype_code(x), T, K, two_i // 2, E, k, pi, pw, p1, ps1, p2, ps2,
                                   _dtype_code(w1, e4m3=True), w1_layout, int(bool(quant_x)), _quant_h_mode(quant_h),
                                   o.ctypes.data, out)
    return o, err


def moe_layer_batched(xb, expert_num_tokens, weights, w1, w2, w1_scale=None, w2_scale=None, w1_layout=0,
                      quant_h=False, out=F64, out_init=None, quant_x=False):
    """The whole batched layer with naive-batched weight application; rows >= count keep out_init."""
    xb, px = _c(xb)
    ent, pe = _c(np.asarray(expert_num_tokens, np.int32))
    w, pw = _c(None if weights is None else np.asarray(weights, np.float32))
    w1, p1 = _c(w1)
    w2, p2 = _c(w2)
    s1, ps1 = _c(w1_scale)
    s2, ps2 = _c(w2_scale)
    E, maxT, K = xb.shape
    two_i = w1.shape[1]
    if out_init is None:
        o = np.zeros((E, maxT, K), _OUT_NP[out])
    else:
        o = np.array(out_init, dtype=_OUT_NP[out], copy=True)
    err = _load().oracle_moe_layer_batched(px, _dtype_code(xb), E, maxT, pe, pw, K, two_i // 2, p1, ps1, p2, ps2,
                                           _dtype_code(w1, e4m3=True), w1_layout, int(bool(quant_x)),
                                           _quant_h_mode(quant_h), o.ctypes.data, out)
    return o, err
