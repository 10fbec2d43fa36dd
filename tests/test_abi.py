"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host (no kernel is launched)."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_permute_gb300 as m
from mixture_experts_layer_permute_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return m.load()


def _declared():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"MOE_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(m.EXPORTED)


def test_every_entry_point_has_a_python_wrapper():
    for n in m.EXPORTED:
        if n.startswith("moe_") or n.startswith("mxfp8_"):
            if n in ("moe_last_error",):
                continue
            assert callable(getattr(m, n, None)), n


def test_library_is_built_for_sm103a():
    # the build passes exactly one -gencode for sm_103a
    assert build_mod.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_version_and_sizes(lib):
    assert m.moe_version() >> 16 == 1
    assert m.moe_max_padded_rows(4096, 8, 128, 128) == 4096 * 8 + 128 * 127
    assert m.moe_max_padded_rows(0, 8, 128, 1) == 0
    assert m.moe_max_padded_rows(1, 0, 1, 1) == -1
    assert m.moe_permute_workspace_size(4096, 8, 128) >= 4096 * 8 * 4


def _status(fn, *args):
    return fn(*args), lib_error()


def lib_error():
    return m.load().moe_last_error().decode()


@pytest.mark.parametrize("args,expect", [
    ((None, 4, 8, 9, 1, None, None, None), 1),        # top_k > E
    ((None, 4, 2000, 2, 1, None, None, None), 1),     # E > 1024
    ((None, -1, 8, 2, 1, None, None, None), 1),       # T < 0
    ((None, 4, 8, 2, 1, None, None, None), 1),        # null pointers
])
def test_route_validation(lib, args, expect):
    assert lib.moe_topk_route(*args) == expect
    assert lib_error().startswith("moe_topk_route")


def test_route_T0_is_a_no_op(lib):
    assert lib.moe_topk_route(None, 0, 8, 2, 1, None, None, None) == 0


def test_permute_validation(lib):
    fake = ctypes.c_void_p(0x1000)      # never dereferenced: validation fails first
    # rows_cap too small for the padding
    rc = lib.moe_permute_align(fake, 4, 2, 8, 0, 16, 0, None, 1, 0, None, 8, fake, fake, fake, fake, fake,
                               1 << 20, None, None)
    assert rc == 1 and "rows_cap" in lib_error()
    # workspace too small
    rc = lib.moe_permute_align(fake, 4, 2, 8, 0, 1, 0, None, 1, 0, None, 8, fake, fake, fake, fake, fake, 0,
                               None, None)
    assert rc == 4
    # misaligned workspace
    rc = lib.moe_permute_align(fake, 4, 2, 8, 0, 1, 0, None, 1, 0, None, 8, fake, fake, fake, fake,
                               ctypes.c_void_p(0x1004), 1 << 20, None, None)
    assert rc == 3
    # batched rows_cap must be E*max_tokens
    rc = lib.moe_permute_align(fake, 4, 2, 8, 1, 1, 16, None, 1, 0, None, 100, fake, fake, fake, fake, fake,
                               1 << 20, None, None)
    assert rc == 1
    # gather with a K that breaks 16-byte rows
    rc = lib.moe_permute_align(fake, 4, 2, 8, 0, 1, 0, fake, 1, 12, fake, 8, fake, fake, fake, fake, fake,
                               1 << 20, None, None)
    assert rc == 3


def test_route_permute_validation(lib):
    fake = ctypes.c_void_p(0x1000)      # never dereferenced: validation fails first

    def call(T=4, E=8, k=2, layout=0, bm=1, mt=0, x=None, K=0, x_out=None, rows_cap=8, ws=fake, ws_bytes=1 << 20,
             logits=fake):
        return lib.moe_route_permute_align(logits, T, E, k, 1, fake, fake, layout, bm, mt, x, 1, K, x_out,
                                           rows_cap, fake, fake, fake, fake, ws, ws_bytes, None, None)
    assert call(k=9) == 1 and lib_error().startswith("moe_route_permute_align")      # top_k > E
    assert call(k=33, E=64) == 1                                                      # top_k > 32
    assert call(E=2000) == 1                                                          # E > 1024
    assert call(bm=16) == 1 and "rows_cap" in lib_error()                             # rows_cap too small
    assert call(ws_bytes=0) == 4                                                      # workspace too small
    assert call(ws=ctypes.c_void_p(0x1004)) == 3                                      # misaligned workspace
    assert call(layout=1, mt=16, rows_cap=100) == 1                                   # batched rows_cap
    assert call(x=fake, K=12, x_out=fake) == 3                                        # 24-byte rows
    assert call(logits=None) == 1 and "null" in lib_error()                           # no logits


def test_tile_weights_validation(lib):
    fake, other = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x40000000)
    assert lib.moe_tile_weights(fake, 0, 1, 0, 2, 256, 128, other, None) == 2      # fp32 weights
    assert lib.moe_tile_weights(fake, 1, 3, 0, 2, 256, 128, other, None) == 1      # which
    assert lib.moe_tile_weights(fake, 1, 1, 7, 2, 256, 128, other, None) == 1      # w1_layout
    assert lib.moe_tile_weights(fake, 1, 2, 0, 2, 200, 128, other, None) == 3      # rows % 128
    assert lib.moe_tile_weights(fake, 1, 2, 0, 2, 256, 96, other, None) == 3       # cols % 64
    assert lib.moe_tile_weights(fake, 1, 2, 0, 2, 256, 128, ctypes.c_void_p(0x100100), None) == 1   # overlap
    assert lib.moe_tile_weights(None, 1, 2, 0, 2, 256, 128, other, None) == 1      # null
    assert lib.moe_tile_weights(ctypes.c_void_p(0x100008), 1, 2, 0, 2, 256, 128, other, None) == 3  # alignment
    # E4M3 codes: W1 only in the interleave-16 layout (the scales keep the stored row order), 128-code columns
    assert lib.moe_tile_weights(fake, 2, 1, 0, 2, 256, 128, other, None) == 2      # [gate; up] codes
    assert "interleave-16" in lib_error()
    assert lib.moe_tile_weights(fake, 2, 2, 0, 2, 256, 64, other, None) == 3       # cols % 128
    assert lib.moe_tile_weights(fake, 2, 1, 1, 2, 256, 192, other, None) == 3     # cols % 128 (W1)


def test_gemm_validation(lib):
    fake = ctypes.c_void_p(0x1000)
    # K not a multiple of 32
    rc = lib.moe_gemm1_swiglu(fake, 1, None, 0, fake, fake, 0, 64, 4, 100, 64, fake, None, 1, 0, 0, fake, 1, None, None, None)
    assert rc == 3 and "multiples of 32" in lib_error()
    # E4M3 weights without scales
    rc = lib.moe_gemm1_swiglu(fake, 1, None, 0, fake, fake, 0, 64, 4, 128, 64, fake, None, 2, 0, 0, fake, 1, None, None, None)
    assert rc == 1
    # misaligned activations
    rc = lib.moe_gemm1_swiglu(ctypes.c_void_p(0x1002), 1, None, 0, fake, fake, 0, 64, 4, 128, 64, fake, None, 1, 0, 0,
                              fake, 1, None, None, None)
    assert rc == 3
    # contiguous gemm2 needs row_route
    rc = lib.moe_gemm2(fake, 1, None, 0, fake, fake, 0, 64, 4, 128, 64, fake, None, 1, 0, None, None, 0, fake, 1, 10, None,
                       None)
    assert rc == 1 and "row_route" in lib_error()
    # unknown layout
    rc = lib.moe_gemm2(fake, 1, None, 7, fake, fake, 0, 64, 4, 128, 64, fake, None, 1, 0, fake, None, 0, fake, 1, 10, None,
                       None)
    assert rc == 1
    # E4M3 activations: scales required, E4M3 weights required, normal tiles refused
    rc = lib.moe_gemm1_swiglu(fake, 2, None, 0, fake, fake, 0, 64, 4, 128, 64, fake, fake, 2, 0, 0, fake, 1, None, None,
                              None)
    assert rc == 1 and "scales" in lib_error()
    rc = lib.moe_gemm1_swiglu(fake, 2, fake, 0, fake, fake, 0, 64, 4, 128, 64, fake, None, 1, 0, 0, fake, 1, None, None,
                              None)
    assert rc == 2 and "E4M3 weights" in lib_error()
    rc = lib.moe_gemm1_swiglu(fake, 2, ctypes.c_void_p(0x1001), 0, fake, fake, 0, 64, 4, 128, 64, fake, fake, 2, 0,
                              0, fake, 1, None, None, None)
    assert rc == 3
    rc = lib.moe_gemm2(fake, 2, fake, 0, fake, fake, 0, 64, 4, 128, 128, fake, fake, 2, 0, fake, None, 1, fake, 1, 10,
                       None, None)
    assert rc == 2 and "swap-AB" in lib_error()
    # E4M3 h needs its scale output
    rc = lib.moe_gemm1_swiglu(fake, 2, fake, 0, fake, fake, 0, 64, 4, 128, 64, fake, fake, 2, 0, 0, fake, 2, None,
                              None, None)
    assert rc == 1 and "h_scale" in lib_error()


def test_reduce_and_quant_validation(lib):
    fake = ctypes.c_void_p(0x1000)
    assert lib.moe_unpermute_topk_reduce(fake, 1, fake, None, 4, 2, 8, 12, fake, 1, None) == 3   # K % 8
    assert lib.moe_unpermute_topk_reduce(fake, 2, fake, None, 4, 2, 8, 16, fake, 1, None) == 2   # E4M3 y
    assert lib.moe_batched_weight_reduce(fake, 1, fake, None, 0, 4, 16, fake, 1, None) == 1      # E = 0
    assert lib.moe_batched_topk_reduce(fake, 1, 64, fake, None, 4, 2, 12, ctypes.c_void_p(0x2000), 1, None,
                                       None) == 3                                                # K % 8
    assert lib.moe_batched_topk_reduce(fake, 1, 64, fake, None, 4, 2, 16, fake, 1, None, None) == 1  # out == y
    assert lib.moe_batched_topk_reduce(fake, 1, 64, None, None, 4, 2, 16, ctypes.c_void_p(0x2000), 1, None,
                                       None) == 1                                                # no route_row
    assert lib.moe_batched_topk_reduce(None, 1, 0, None, None, 0, 2, 16, None, 1, None, None) == 0   # T = 0
    assert lib.mxfp8_quantize_block32(fake, 1, 4, 33, fake, fake, None) == 3                     # cols % 32
    assert lib.mxfp8_quantize_block32(fake, 2, 4, 32, fake, fake, None) == 2                     # E4M3 input
    assert lib.mxfp8_quantize_block32(None, 1, 0, 32, None, None, None) == 0                     # empty: no-op


def test_route_counts_that_overflow_are_rejected(lib):
    # T*top_k would overflow int64 (or reach 2^31): every entry point rejects it before forming the product
    fake = ctypes.c_void_p(0x1000)      # never dereferenced: validation fails first
    huge = 2 ** 61
    assert m.moe_max_padded_rows(huge, 8, 128, 1) == -1
    assert m.moe_max_padded_rows(2 ** 28, 8, 128, 1) == -1          # exactly 2^31 routes
    assert m.moe_max_padded_rows(2 ** 28 - 1, 8, 128, 1) == (2 ** 28 - 1) * 8
    assert m.moe_max_padded_rows(4, 2000, 8, 1) == -1               # top_k > 1024
    assert m.moe_permute_workspace_size(huge, 8, 128) == 0
    assert m.moe_permute_workspace_size(4, 8, 2000) == 0
    rc = lib.moe_permute_align(fake, huge, 8, 128, 0, 1, 0, None, 1, 0, None, 8, fake, fake, fake, fake, fake,
                               1 << 20, None, None)
    assert rc == 1 and "2^31" in lib_error()
    rc = lib.moe_permute_align_static(fake, huge, 8, 128, 0, 1, 0, None, 1, 0, None, 8, fake, fake, fake, fake,
                                      None, None)
    assert rc == 1 and "2^31" in lib_error()
    assert lib.moe_unpermute_topk_reduce(fake, 1, fake, None, huge, 8, 128, 16, fake, 1, None) == 1
    assert lib.moe_batched_topk_reduce(fake, 1, 64, fake, None, huge, 8, 16, ctypes.c_void_p(0x2000), 1, None,
                                       None) == 1


def test_permute_static_validation(lib):
    # the entry point without a workspace: its own early checks run on the host, with nothing launched and no
    # pointer read (the pointers below are never dereferenced)
    fake = ctypes.c_void_p(0x1000)

    def call(T=4, k=2, E=8, layout=0, bm=1, mt=0, rows_cap=8):
        return lib.moe_permute_align_static(fake, T, k, E, layout, bm, mt, None, 1, 0, None, rows_cap, fake, fake,
                                            fake, fake, None, None)
    for bad in (dict(T=-1), dict(k=0), dict(k=1025), dict(E=0), dict(E=1025)):
        assert call(**bad) == 1, bad
        assert lib_error().startswith("moe_permute_align_static")
    # a routing whose scratch exceeds the built-in array: refused with the limit in the message
    rc = call(T=70000, k=8, E=128, rows_cap=70000 * 8)
    assert rc == 4
    assert "2097152" in lib_error() and "moe_permute_align" in lib_error()


def test_tiled_weight_layout_validation(lib):
    fake = ctypes.c_void_p(0x1000)      # never dereferenced: validation fails first
    # moe_gemm2: an unknown W2 layout
    rc = lib.moe_gemm2(fake, 1, None, 0, fake, fake, 0, 64, 4, 256, 128, fake, None, 1, 7, fake, None, 0, fake, 1,
                       10, None, None)
    assert rc == 1 and "w2_layout" in lib_error()
    # tile-contiguous weights on an implementation other than the CTA-pair tiles
    rc = lib.moe_gemm2(fake, 1, None, 0, fake, fake, 0, 64, 4, 256, 128, fake, None, 1, 2, fake, None,
                       m.MOE_IMPL_TCGEN05_SWAP_AB, fake, 1, 10, None, None)
    assert rc == 2 and "CTA-pair" in lib_error()
    rc = lib.moe_gemm1_swiglu(fake, 1, None, 0, fake, fake, 0, 64, 4, 256, 128, fake, None, 1, 2, m.MOE_IMPL_SIMT,
                              fake, 1, None, None, None)
    assert rc == 2 and "CTA-pair" in lib_error()
