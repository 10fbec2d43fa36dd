"""GPU parity: every call of the C ABI against the CPU oracle on the same seeded inputs.

Bit-exact: routing ids, permutation (counts, offsets, rows, inverse map),
gathered rows, MXFP8 codes and scales, device error bits.  Floats: the
tolerances of tests/helpers.py (rel-RMS and max-abs relative to max|ref|,
1e-5 for fp32, 2e-2 for bf16).  Sizes span several tiles and ragged tails;
full-size workloads are checked on sampled tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_permute_gb300 import workloads as wl
from helpers import TOL_BF16, TOL_F32, assert_close, compact_experts, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
IMPLS_BF16 = ["tcgen05", "swap_ab", "mixed", "pair", "simt"]


def _impl(m, name):
    return {"tcgen05": m.MOE_IMPL_TCGEN05, "swap_ab": m.MOE_IMPL_TCGEN05_SWAP_AB, "simt": m.MOE_IMPL_SIMT,
            "mixed": m.MOE_IMPL_TCGEN05_MIXED, "pair": m.MOE_IMPL_TCGEN05_PAIR, "auto": m.MOE_IMPL_AUTO}[name]


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k,renorm", [(16, 8, 2, True), (64, 128, 8, True), (4096, 128, 8, True),
                                          (33, 512, 8, True), (100, 40, 5, False), (7, 1024, 32, True),
                                          (5, 3, 3, False)])
def test_route_bit_exact(moe, T, E, k, renorm):
    w = wl.scaled(wl.decode(T), E=E, top_k=k)
    logits = wl.router_logits(w, seed=T + E)
    if E == 40:
        logits = torch.round(logits * 2) / 2          # exact ties: lower index must win
    ids, wts = moe.moe_topk_route(logits.to(DEV), k, renormalize=renorm)
    rids, rw = oracle.topk_route(logits.numpy(), k, renormalize=renorm)
    assert np.array_equal(ids.cpu().numpy(), rids)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("E", [64, 1024])
def test_route_signed_zeros_and_infinities(moe, E):
    """-0 and +0 compare equal, so among zero logits the lower index wins whatever the signs; -inf logits are
    chosen last and get weight 0."""
    T, k = 8, 5
    g = torch.Generator().manual_seed(E)
    logits = -torch.rand((T, E), generator=g) - 1.0          # every other logit <= -1
    for t in range(T):
        pos = torch.randperm(E, generator=g)[:3]
        logits[t, torch.randperm(E, generator=g)[: E // 2]] = float("-inf")
        logits[t, pos] = torch.tensor([-0.0 if (n + t) % 2 == 0 else 0.0 for n in range(3)])
    if E == 1024:
        logits[:, 3:] = float("-inf")                          # three finite logits: two -inf ones are chosen
        logits[:, :3] = torch.tensor([-0.0, -1.5, 0.0])
    for renorm in (True, False):
        ids, wts = moe.moe_topk_route(logits.to(DEV), k, renormalize=renorm)
        rids, rw = oracle.topk_route(logits.numpy(), k, renormalize=renorm)
        assert np.array_equal(ids.cpu().numpy(), rids)
        np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=1e-6, atol=1e-7)
        res = moe.moe_route_permute_align(logits.to(DEV), k, renormalize=renorm)
        assert torch.equal(res["topk_ids"], ids)
        assert torch.equal(res["topk_weights"].view(torch.int32), wts.view(torch.int32))


def test_route_zipf_prefill(moe):
    w = wl.prefill()
    logits = wl.router_logits(w, 0)
    ids, wts = moe.moe_topk_route(logits.to(DEV), w.top_k)
    rids, rw = oracle.topk_route(logits.numpy(), w.top_k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=1e-6, atol=1e-7)


# ----------------------------------------------------------------------------
# permute / align
# ----------------------------------------------------------------------------

def _ids(T, k, E, seed, pad=0.0, bad=0):
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    if pad:
        ids[torch.rand(T, k, generator=g) < pad] = -1
    if bad:
        flat = ids.view(-1)
        pos = torch.randperm(flat.numel(), generator=g)[:bad]
        flat[pos[: bad // 2]] = E + 3
        flat[pos[bad // 2:]] = -5
    return ids


@pytest.mark.parametrize("T,k,E,bm,pad", [(16, 2, 8, 1, 0.0), (64, 8, 128, 1, 0.1), (128, 8, 128, 16, 0.0),
                                          (4096, 8, 128, 128, 0.05), (9000, 8, 64, 4, 0.2),
                                          (3, 1, 1, 1, 0.0), (1, 8, 1024, 128, 0.0)])
def test_permute_contiguous_bit_exact(moe, T, k, E, bm, pad):
    ids = _ids(T, k, E, seed=T * 7 + E, pad=pad) if E >= k else torch.zeros(T, k, dtype=torch.int32)
    K = 64
    x = wl._normal((T, K), 1.0, 5, "x", 0, "cpu", torch.bfloat16)
    res = moe.moe_permute_align(ids.to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, bm, x=x.to(DEV))
    ref = oracle.permute_contiguous(ids.numpy(), E, bm)
    off = res["offsets"].cpu().numpy()
    assert np.array_equal(res["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(off, ref["offsets"])
    rows = off[E]
    assert np.array_equal(res["row_route"][:rows].cpu().numpy(), ref["sorted_route"])
    assert np.array_equal(res["route_row"].cpu().numpy(), ref["route_row"])
    # gathered rows are the token rows, bit for bit
    xo = res["x_out"][:rows].cpu()
    valid = ref["sorted_route"] >= 0
    src = torch.from_numpy(ref["sorted_route"][valid] // k).long()
    assert torch.equal(xo[torch.from_numpy(valid)].view(torch.int16), x[src].view(torch.int16))


def test_permute_chunked_rounds(moe):
    """More routes than 64 chunks x 1024: each CTA takes several rounds."""
    T, k, E = 12000, 8, 96
    ids = _ids(T, k, E, seed=3, pad=0.1)
    res = moe.moe_permute_align(ids.to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 8)
    ref = oracle.permute_contiguous(ids.numpy(), E, 8)
    rows = ref["offsets"][E]
    assert np.array_equal(res["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(res["row_route"][:rows].cpu().numpy(), ref["sorted_route"])
    assert np.array_equal(res["route_row"].cpu().numpy(), ref["route_row"])


@pytest.mark.parametrize("T", [40, 3000])
def test_permute_bad_ids_flagged(moe, T):
    E, k = 16, 4
    ids = _ids(T, k, E, seed=9, pad=0.1, bad=10)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = moe.moe_permute_align(ids.to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, err_word=err)
    ref = oracle.permute_contiguous(ids.numpy(), E, 1)
    assert int(err.item()) == moe.MOE_DEVERR_ID_RANGE == ref["err"]
    assert np.array_equal(res["route_row"].cpu().numpy(), ref["route_row"])
    assert np.array_equal(res["counts"].cpu().numpy(), ref["counts"])


@pytest.mark.parametrize("T,k,E,cap", [(50, 4, 8, 32), (2000, 2, 16, 200), (100, 2, 4, 0)])
def test_permute_batched_bit_exact(moe, T, k, E, cap):
    ids = _ids(T, k, E, seed=T + cap, pad=0.1)
    K = 32
    x = wl._normal((T, K), 1.0, 6, "x", 0, "cpu", torch.float32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = moe.moe_permute_align(ids.to(DEV), E, moe.MOE_LAYOUT_BATCHED, 1, cap, x=x.to(DEV), err_word=err)
    ref = oracle.permute_batched(ids.numpy(), E, cap)
    assert int(err.item()) == ref["err"]
    assert np.array_equal(res["counts"].cpu().numpy(), ref["expert_num_tokens"])
    assert np.array_equal(res["offsets"].cpu().numpy(), np.arange(E + 1) * cap)
    assert np.array_equal(res["row_route"][:E * cap].cpu().numpy(), ref["row_route"].reshape(-1))
    assert np.array_equal(res["route_row"].cpu().numpy(), ref["route_row"])
    xo = res["x_out"].cpu().reshape(E, cap, K) if cap else None
    for e in range(E):
        for q in range(ref["expert_num_tokens"][e]):
            r = ref["row_route"][e, q]
            assert torch.equal(xo[e, q], x[r // k])


# ----------------------------------------------------------------------------
# routing + placement + gather in one call
# ----------------------------------------------------------------------------

# T, E, k, renormalize, layout, block_m, max_tokens, x dtype (None: no gather), K
ROUTE_PERMUTE_CASES = [
    (1, 128, 8, True, "contiguous", 1, 0, torch.bfloat16, 4096),     # decode T = 1 at full K: one launch
    (64, 128, 8, True, "contiguous", 1, 0, torch.bfloat16, 4096),    # decode T = 64
    (128, 128, 8, True, "contiguous", 16, 0, torch.bfloat16, 256),   # 1024 routes, padded rows: still one launch
    (129, 128, 8, True, "contiguous", 1, 0, torch.bfloat16, 256),    # one token more: the separate launches
    (33, 40, 5, False, "contiguous", 4, 0, torch.float32, 96),       # exact ties, plain softmax, fp32 rows
    (7, 1024, 32, True, "contiguous", 1, 0, torch.bfloat16, 64),     # 32 logits per lane
    (20, 32, 1, True, "contiguous", 128, 0, torch.bfloat16, 8),      # top_k = 1, 16-byte rows, wide padding
    (5, 3, 3, True, "contiguous", 1, 0, None, 0),                    # top_k = E, no gather
    (100, 16, 4, True, "batched", 1, 12, torch.bfloat16, 64),        # capacity drops routes (one launch)
    (2000, 64, 4, True, "batched", 1, 200, torch.bfloat16, 32),      # batched, separate launches
]


@pytest.mark.parametrize("T,E,k,renorm,layout,bm,cap,xdt,K", ROUTE_PERMUTE_CASES)
def test_route_permute_bit_exact(moe, T, E, k, renorm, layout, bm, cap, xdt, K):
    """moe_route_permute_align against the oracle's routing and placement, and bit-identical to
    moe_topk_route followed by moe_permute_align."""
    w = wl.scaled(wl.decode(T), E=E, top_k=k)
    logits = wl.router_logits(w, seed=T + E)
    if E == 40:
        logits = torch.round(logits * 2) / 2          # exact ties: lower index must win
    x = wl._normal((T, K), 1.0, 5, "x", 0, "cpu", xdt) if xdt is not None else None
    lay = moe.MOE_LAYOUT_CONTIGUOUS if layout == "contiguous" else moe.MOE_LAYOUT_BATCHED
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    xd = x.to(DEV) if x is not None else None
    res = moe.moe_route_permute_align(logits.to(DEV), k, renormalize=renorm, layout=lay, block_m=bm,
                                      max_tokens=cap, x=xd, err_word=err)
    rids, rw = oracle.topk_route(logits.numpy(), k, renormalize=renorm)
    assert np.array_equal(res["topk_ids"].cpu().numpy(), rids)
    np.testing.assert_allclose(res["topk_weights"].cpu().numpy(), rw, rtol=1e-6, atol=1e-7)

    # the separate calls give the same bits
    ids2, w2 = moe.moe_topk_route(logits.to(DEV), k, renormalize=renorm)
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    sep = moe.moe_permute_align(ids2, E, lay, bm, cap, x=xd, err_word=err2)
    assert torch.equal(res["topk_ids"], ids2)
    assert torch.equal(res["topk_weights"].view(torch.int32), w2.view(torch.int32))
    for key in ("counts", "offsets", "route_row"):
        assert torch.equal(res[key], sep[key]), key
    assert int(err.item()) == int(err2.item())

    if lay == moe.MOE_LAYOUT_CONTIGUOUS:
        ref = oracle.permute_contiguous(rids, E, bm)
        rows = int(ref["offsets"][E])
        assert np.array_equal(res["counts"].cpu().numpy(), ref["counts"])
        assert np.array_equal(res["offsets"].cpu().numpy(), ref["offsets"])
        assert np.array_equal(res["row_route"][:rows].cpu().numpy(), ref["sorted_route"])
        route_of_row = ref["sorted_route"]
    else:
        ref = oracle.permute_batched(rids, E, cap)
        rows = E * cap
        assert np.array_equal(res["counts"].cpu().numpy(), ref["expert_num_tokens"])
        assert np.array_equal(res["offsets"].cpu().numpy(), np.arange(E + 1) * cap)
        assert np.array_equal(res["row_route"][:rows].cpu().numpy(), ref["row_route"].reshape(-1))
        route_of_row = ref["row_route"].reshape(-1)
    assert np.array_equal(res["route_row"].cpu().numpy(), ref["route_row"])
    assert int(err.item()) == ref["err"]
    assert torch.equal(res["row_route"][:rows], sep["row_route"][:rows])
    if x is not None:
        # every routed row is its token's row, bit for bit
        valid = route_of_row >= 0
        src = torch.from_numpy(route_of_row[valid] // k).long()
        xo = res["x_out"][:rows].cpu()[torch.from_numpy(valid)]
        bits = torch.int16 if xdt == torch.bfloat16 else torch.int32
        assert torch.equal(xo.view(bits), x[src].view(bits))


def test_route_permute_empty(moe):
    """T = 0: no routes, every count and offset is zero."""
    logits = torch.empty((0, 16), dtype=torch.float32, device=DEV)
    res = moe.moe_route_permute_align(logits, 2, x=torch.empty((0, 64), dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert res["topk_ids"].shape == (0, 2)
    assert not torch.any(res["counts"]) and not torch.any(res["offsets"])


# ----------------------------------------------------------------------------
# MXFP8 quantisation
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_mxfp8_quantize_bit_exact(moe, dtype):
    g = torch.Generator().manual_seed(1)
    x = torch.randn(300, 512, generator=g) * 0.02
    x[0, :64] = 0.0                                        # zero blocks
    x[1, :32] = -0.0
    x[2, :32] *= 1e-36                                      # clamps the code at 0
    x[3, :32] = 448.0                                       # exact boundary: code 127
    x[4, :32] = torch.randn(32, generator=g) * 1e30         # large
    x[5] = torch.exp(torch.randn(512, generator=g) * 8)     # wide dynamic range inside blocks
    x[6, 5] = 1.75 * 2.0 ** -120                            # f exactly 1.75 in a tiny block
    x = x.to(dtype)
    codes, scales = moe.mxfp8_quantize_block32(x.to(DEV))
    rc, rs = oracle.mxfp8_quantize(wl.to_numpy(x))
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


# ----------------------------------------------------------------------------
# reduce
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("ydt,odt,weighted", [(torch.bfloat16, torch.bfloat16, True),
                                              (torch.float32, torch.float32, True),
                                              (torch.bfloat16, torch.float32, False)])
def test_topk_reduce(moe, ydt, odt, weighted):
    T, k, K, E = 37, 8, 4096, 64
    g = torch.Generator().manual_seed(2)
    ids = _ids(T, k, E, seed=4, pad=0.2)
    ids[5] = -1                                            # a token made only of padding
    y = torch.randn(T * k, K, generator=g).to(ydt)
    w = torch.rand(T, k, generator=g)
    out = moe.moe_unpermute_topk_reduce(y.to(DEV), ids.to(DEV), E, w.to(DEV) if weighted else None,
                                        out_dtype=moe.MOE_F32 if odt == torch.float32 else moe.MOE_BF16)
    ref = oracle.topk_reduce(wl.to_numpy(y), ids.numpy(), w.numpy() if weighted else None)
    tol = TOL_F32 if (ydt == torch.float32 and odt == torch.float32) else TOL_BF16
    assert_close(to_f64(out), ref, tol, "topk_reduce")
    o5 = out[5].cpu()
    assert torch.all(o5 == 0) and not torch.any(torch.signbit(o5.float()))   # +0.0
    again = moe.moe_unpermute_topk_reduce(y.to(DEV), ids.to(DEV), E, w.to(DEV) if weighted else None,
                                          out_dtype=moe.MOE_F32 if odt == torch.float32 else moe.MOE_BF16)
    assert torch.equal(out.view(torch.uint8), again.view(torch.uint8))       # fixed order: same bits


def test_batched_weight_reduce(moe):
    E, maxT, K = 6, 40, 256
    g = torch.Generator().manual_seed(3)
    counts = torch.tensor([0, 40, 7, 13, 1, 39], dtype=torch.int32)
    y = torch.randn(E, maxT, K, generator=g).to(torch.bfloat16)
    w = torch.rand(E, maxT, generator=g)
    out = torch.full((E, maxT, K), 7.0, dtype=torch.bfloat16, device=DEV)
    moe.moe_batched_weight_reduce(y.to(DEV), counts.to(DEV), w.to(DEV), out=out)
    out = out.cpu()
    for e in range(E):
        c = int(counts[e])
        ref = y[e, :c].double() * w[e, :c].double()[:, None]
        assert_close(to_f64(out[e, :c]), ref.numpy(), TOL_BF16, "batched weight")
        assert torch.all(out[e, c:] == 7.0)


@pytest.mark.parametrize("ydt,odt,weighted", [(torch.bfloat16, torch.bfloat16, True),
                                              (torch.float32, torch.float32, True),
                                              (torch.bfloat16, torch.float32, False)])
def test_batched_topk_reduce(moe, ydt, odt, weighted):
    """Token-order reduce of the batched layout through route_row; capacity drops, padding, +0.0."""
    T, k, E, maxT, K = 300, 6, 16, 100, 1024
    ids = _ids(T, k, E, seed=9, pad=0.1)
    ids[7] = -1                                            # a token made only of padding
    res = oracle.permute_batched(ids.numpy(), E, maxT)      # hot experts overflow: drops
    assert res["err"] == oracle.ERR_CAPACITY
    rr = res["route_row"]
    g = torch.Generator().manual_seed(6)
    y = torch.randn(E, maxT, K, generator=g).to(ydt)
    w = torch.rand(T, k, generator=g)
    odc = moe.MOE_F32 if odt == torch.float32 else moe.MOE_BF16
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = moe.moe_batched_topk_reduce(y.to(DEV), torch.from_numpy(rr).to(DEV), w.to(DEV) if weighted else None,
                                      out_dtype=odc, err_word=err)
    ref, rerr = oracle.batched_topk_reduce(wl.to_numpy(y), rr, w.numpy() if weighted else None)
    assert rerr == 0 and int(err.item()) == 0
    tol = TOL_F32 if (ydt == torch.float32 and odt == torch.float32) else TOL_BF16
    assert_close(to_f64(out), ref, tol, "batched topk reduce")
    o7 = out[7].cpu()
    assert torch.all(o7 == 0) and not torch.any(torch.signbit(o7.float()))   # +0.0
    again = moe.moe_batched_topk_reduce(y.to(DEV), torch.from_numpy(rr).to(DEV), w.to(DEV) if weighted else None,
                                        out_dtype=odc)
    assert torch.equal(out.view(torch.uint8), again.view(torch.uint8))       # fixed order: same bits
    # a row index past the buffer is reported and skipped
    bad = rr.copy()
    bad[3, 0] = E * maxT
    moe.moe_batched_topk_reduce(y.to(DEV), torch.from_numpy(bad).to(DEV), None, out_dtype=odc, err_word=err)
    assert int(err.item()) == moe.MOE_DEVERR_ID_RANGE


@pytest.mark.parametrize("impl", ["tcgen05", "swap_ab", "simt"])
@pytest.mark.parametrize("maxT", [64, 24])
def test_layer_batched_token_order(moe, impl, maxT):
    """route -> batched permute (+gather) -> GEMM 1 -> GEMM 2 (no weight) -> token-order reduce equals the
    contiguous oracle layer with the routes dropped for capacity removed."""
    T, k, E, K, I = 96, 4, 8, 512, 256
    w = wl.scaled(wl.tiny(), T=T, K=K, I=I, E=E, top_k=k, x_std=1.0, w_std=0.05)
    x = wl.activations(w, 3).to(torch.bfloat16)
    W1 = wl.expert_weights(w, "W1", 3).to(torch.bfloat16)
    W2 = wl.expert_weights(w, "W2", 3).to(torch.bfloat16)
    ids, wts = moe.moe_topk_route(wl.router_logits(w, 3).to(DEV), k)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa = moe.moe_permute_align(ids, E, layout=moe.MOE_LAYOUT_BATCHED, max_tokens=maxT, x=x.to(DEV),
                               err_word=err)
    h = moe.moe_gemm1_swiglu(pa["x_out"], pa["counts"], pa["offsets"], W1.to(DEV), I,
                             layout=moe.MOE_LAYOUT_BATCHED, max_tokens=maxT, impl=_impl(moe, impl))
    yb = moe.moe_gemm2(h.reshape(E * maxT, I), pa["counts"], pa["offsets"], W2.to(DEV), E * maxT,
                       layout=moe.MOE_LAYOUT_BATCHED, max_tokens=maxT, impl=_impl(moe, impl))
    out = moe.moe_batched_topk_reduce(yb, pa["route_row"], wts)
    torch.cuda.synchronize()
    rr = pa["route_row"].cpu().numpy()
    ids_kept = np.where(rr >= 0, ids.cpu().numpy(), -1).astype(np.int32)
    if maxT == 24:
        assert int(err.item()) == moe.MOE_DEVERR_CAPACITY and (ids_kept < 0).any()
    ref, _ = oracle.moe_layer(wl.to_numpy(x), ids_kept, wts.cpu().numpy(), wl.to_numpy(W1), wl.to_numpy(W2))
    assert_close(to_f64(out), ref, TOL_BF16, f"batched token-order layer {impl}")


# ----------------------------------------------------------------------------
# grouped GEMMs
# ----------------------------------------------------------------------------

GEMM_SHAPES = [  # T, k, E, K, I, block_m
    (96, 4, 8, 512, 256, 1),
    (300, 2, 16, 256, 384, 128),
    (600, 1, 2, 256, 256, 1),        # ~300 rows per expert: several m-tiles / two token segments
    (5, 8, 128, 512, 128, 1),        # decode-like: a few tokens per expert
    (700, 2, 6, 256, 128, 1),        # skewed below: full tiles, long and short tails, tiny experts
]


def _routed(T, k, E, K, seed):
    w = wl.scaled(wl.decode(T), T=T, K=K, E=E, top_k=k)
    logits = wl.router_logits(w, seed)
    if E == 6:   # a steep per-expert bias: counts from hundreds down to a handful
        logits = logits + torch.tensor([6.0, 4.0, 2.5, 1.0, -1.0, -3.0])
    ids, weights = oracle.topk_route(logits.numpy(), k)
    x = wl.activations(w, seed)
    return w, x, ids, weights


@pytest.mark.parametrize("impl", IMPLS_BF16)
@pytest.mark.parametrize("shape", GEMM_SHAPES)
@pytest.mark.parametrize("w1_layout", [0, 1])
def test_gemm1_swiglu(moe, impl, shape, w1_layout):
    T, k, E, K, I, bm = shape
    w, x, ids, _ = _routed(T, k, E, K, seed=T + E)
    wI = wl.scaled(w, I=I)
    W1 = wl.expert_weights(wI, "W1", 1)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, bm, x=x.to(DEV))
    h = moe.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], W1.to(DEV), I, w1_layout=w1_layout,
                             impl=_impl(moe, impl))
    flat = ids.reshape(-1)
    href = oracle.expert_gate_up(wl.to_numpy(x)[np.arange(T * k) // k], flat, wl.to_numpy(W1),
                                 w1_layout=w1_layout)
    rr = res["route_row"].cpu().numpy().reshape(-1)
    got = to_f64(h.cpu()[torch.from_numpy(rr).long()])
    assert_close(got, href, TOL_BF16, f"gemm1 {impl}")


@pytest.mark.parametrize("impl", IMPLS_BF16)
@pytest.mark.parametrize("shape", GEMM_SHAPES)
@pytest.mark.parametrize("weighted", [True, False])
def test_gemm2(moe, impl, shape, weighted):
    T, k, E, K, I, bm = shape
    w, _, ids, weights = _routed(T, k, E, K, seed=T + 2 * E)
    wI = wl.scaled(w, I=I)
    W2 = wl.expert_weights(wI, "W2", 2)
    R = T * k
    hsrc = wl._normal((R, I), 1.0, 7, "h", 0, "cpu", torch.bfloat16)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, bm)
    rr = res["route_row"].view(-1).long()
    hperm = torch.zeros((res["rows_cap"], I), dtype=torch.bfloat16, device=DEV)
    hperm[rr] = hsrc.to(DEV)                                   # test plumbing: rows placed as routed
    wt = torch.from_numpy(weights).to(DEV).reshape(-1)
    y = moe.moe_gemm2(hperm, res["counts"], res["offsets"], W2.to(DEV), R, row_route=res["row_route"],
                      route_weights=wt if weighted else None, impl=_impl(moe, impl))
    yref = oracle.expert_down(wl.to_numpy(hsrc), ids.reshape(-1), wl.to_numpy(W2))
    if weighted:
        yref = yref * weights.reshape(-1, 1).astype(np.float64)
    assert_close(to_f64(y.cpu()), yref, TOL_BF16, f"gemm2 {impl}")


@pytest.mark.parametrize("impl", ["tcgen05", "pair", "auto"])
@pytest.mark.parametrize("maxT", [300, 256, 140])
@pytest.mark.parametrize("w1_layout", [0, 1])
def test_gemms_batched_layout(moe, impl, maxT, w1_layout):
    """Batched (E, max_tokens, K) rows with counts above 128 and 256: normal tiles of 256 rows, the second
    half full, ragged or empty, both W1 layouts, GEMM 2 with the per-row weight."""
    E, K, I = 5, 256, 256
    w = wl.scaled(wl.tiny(), T=1, K=K, I=I, E=E, top_k=1, x_std=1.0, w_std=0.05)
    g = torch.Generator().manual_seed(maxT + w1_layout)
    counts = torch.tensor([maxT, maxT - 1, 129, 128, 7][:E], dtype=torch.int32).clamp(max=maxT)
    x = wl._normal((E, maxT, K), 1.0, 11, "x", 0, "cpu", torch.bfloat16)
    rw = torch.rand((E, maxT), generator=g)
    W1 = wl.expert_weights(w, "W1", 4).to(torch.bfloat16)
    W2 = wl.expert_weights(w, "W2", 4).to(torch.bfloat16)
    offs = torch.arange(E + 1, dtype=torch.int32) * maxT
    h = moe.moe_gemm1_swiglu(x.to(DEV).reshape(E * maxT, K), counts.to(DEV), offs.to(DEV), W1.to(DEV), I,
                             layout=moe.MOE_LAYOUT_BATCHED, max_tokens=maxT, w1_layout=w1_layout,
                             impl=_impl(moe, impl))
    y = moe.moe_gemm2(h, counts.to(DEV), offs.to(DEV), W2.to(DEV), E * maxT, layout=moe.MOE_LAYOUT_BATCHED,
                      max_tokens=maxT, route_weights=rw.to(DEV).reshape(-1), impl=_impl(moe, impl))
    torch.cuda.synchronize()
    hc, yc = h.cpu().reshape(E, maxT, I), y.cpu().reshape(E, maxT, K)
    for e in range(E):
        c = int(counts[e])
        ids = np.full(c, e, dtype=np.int32)
        href = oracle.expert_gate_up(wl.to_numpy(x[e, :c]), ids, wl.to_numpy(W1), w1_layout=w1_layout)
        assert_close(to_f64(hc[e, :c]), href, TOL_BF16, f"batched gemm1 expert {e}")
        yref = oracle.expert_down(wl.to_numpy(hc[e, :c]), ids, wl.to_numpy(W2))
        yref = yref * rw[e, :c].numpy().astype(np.float64)[:, None]
        assert_close(to_f64(yc[e, :c]), yref, TOL_BF16, f"batched gemm2 expert {e}")


@pytest.mark.parametrize("w1_layout", [0, 1])
def test_pair_tiles_ragged_segments(moe, w1_layout):
    """CTA-pair tiles on experts of 257, 255, 33 and 1 tokens (a full 256-token segment plus a 1-token one, N
    rounded up to 32 tokens, one token), several 256-row weight tiles per expert: GEMM 1 and GEMM 2 (weighted,
    scattered to the routes) against the oracle, and run-to-run bit identity."""
    counts = [257, 255, 33, 1]
    E, K, I = len(counts), 512, 384
    g = torch.Generator().manual_seed(31)
    ids = torch.cat([torch.full((c,), e, dtype=torch.int32) for e, c in enumerate(counts)])
    ids = ids[torch.randperm(ids.numel(), generator=g)].reshape(-1, 1)
    T = ids.shape[0]
    w = wl.scaled(wl.decode(T), T=T, K=K, I=I, E=E, top_k=1, w_std=0.05)
    x = wl.activations(w, 31)
    W1 = wl.expert_weights(w, "W1", 31)
    W2 = wl.expert_weights(w, "W2", 31)
    wts = torch.rand(T, 1, generator=g)
    res = moe.moe_permute_align(ids.to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 128, x=x.to(DEV))
    pair = moe.MOE_IMPL_TCGEN05_PAIR
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    h = moe.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], W1.to(DEV), I, w1_layout=w1_layout,
                             impl=pair, err_word=err)
    y = moe.moe_gemm2(h, res["counts"], res["offsets"], W2.to(DEV), T, row_route=res["row_route"],
                      route_weights=wts.reshape(-1).to(DEV), impl=pair, err_word=err)
    y2 = moe.moe_gemm2(h, res["counts"], res["offsets"], W2.to(DEV), T, row_route=res["row_route"],
                       route_weights=wts.reshape(-1).to(DEV), impl=pair, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    flat = ids.reshape(-1).numpy()
    href = oracle.expert_gate_up(wl.to_numpy(x), flat, wl.to_numpy(W1), w1_layout=w1_layout)
    rr = res["route_row"].cpu().reshape(-1).long()
    assert_close(to_f64(h.cpu()[rr]), href, TOL_BF16, "pair gemm1")
    yref = oracle.expert_down(wl.to_numpy(h.cpu()[rr]), flat, wl.to_numpy(W2)) * wts.numpy().astype(np.float64)
    assert_close(to_f64(y.cpu()), yref, TOL_BF16, "pair gemm2")


@pytest.mark.parametrize("w1_layout", [0, 1])
@pytest.mark.parametrize("layout", ["contiguous", "batched"])
def test_pair_tiles_tiled_weights(moe, w1_layout, layout):
    """CTA-pair tiles on tile-contiguous W1 and W2 (moe_tile_weights, MOE_W_TILED) give h and y bit for bit equal
    to the row-major weights (same tiles, same accumulation order)."""
    E, K, I = 4, 512, 384
    pair = moe.MOE_IMPL_TCGEN05_PAIR
    w = wl.scaled(wl.decode(64), T=300, K=K, I=I, E=E, top_k=2, w_std=0.05)
    W1 = wl.expert_weights(w, "W1", 41).to(DEV)
    W2 = wl.expert_weights(w, "W2", 41).to(DEV)
    W1t, W2t = moe.moe_tile_weights(W1, 1, w1_layout), moe.moe_tile_weights(W2, 2)
    if layout == "contiguous":
        _, x, ids, weights = _routed(300, 2, E, K, seed=41)
        res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 128, x=x.to(DEV))
        a, counts, offs, kw = res["x_out"], res["counts"], res["offsets"], {}
        g2 = dict(row_route=res["row_route"], route_weights=torch.from_numpy(weights).to(DEV).reshape(-1))
        y_rows = 600
    else:
        maxT = 200
        counts = torch.tensor([200, 131, 77, 0], dtype=torch.int32, device=DEV)
        offs = torch.arange(E + 1, dtype=torch.int32, device=DEV) * maxT
        a = wl._normal((E * maxT, K), 1.0, 41, "x", 0, DEV, torch.bfloat16)
        kw = dict(layout=moe.MOE_LAYOUT_BATCHED, max_tokens=maxT)
        g2 = dict(route_weights=torch.rand(E * maxT, generator=torch.Generator().manual_seed(41)).to(DEV))
        y_rows = E * maxT
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for W1x, W2x, l1, l2 in ((W1, W2, w1_layout, moe.MOE_W1_GATE_UP), (W1t, W2t, moe.MOE_W_TILED, moe.MOE_W_TILED)):
        h = moe.moe_gemm1_swiglu(a, counts, offs, W1x, I, w1_layout=l1, impl=pair, err_word=err, **kw)
        y = moe.moe_gemm2(h, counts, offs, W2x, y_rows, w2_layout=l2, impl=pair, err_word=err, **kw, **g2)
        outs.append((h, y))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    (h1, y1), (h2, y2) = outs
    if layout == "contiguous":
        rr = res["route_row"].view(-1).long()
        assert torch.equal(h1[rr].view(torch.int16), h2[rr].view(torch.int16))
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    else:
        for e in range(E):
            c = int(counts[e])
            rows = slice(e * maxT, e * maxT + c)
            assert torch.equal(h1.reshape(-1, I)[rows].view(torch.int16), h2.reshape(-1, I)[rows].view(torch.int16))
            assert torch.equal(y1.reshape(-1, K)[rows].view(torch.int16), y2.reshape(-1, K)[rows].view(torch.int16))


def test_pair_tiles_refuse_other_shapes(moe):
    """Shapes outside the CTA-pair tiles (weight rows per expert not a multiple of 256) are refused with nothing
    launched; MOE_IMPL_AUTO never picks them there."""
    E, K, I = 2, 256, 64                      # GEMM 1: 2I = 128 weight rows per expert
    x = torch.zeros((8, K), dtype=torch.bfloat16, device=DEV)
    counts = torch.tensor([4, 4], dtype=torch.int32, device=DEV)
    offs = torch.tensor([0, 4, 8], dtype=torch.int32, device=DEV)
    W1 = torch.zeros((E, 2 * I, K), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_gemm1_swiglu(x, counts, offs, W1, I, impl=moe.MOE_IMPL_TCGEN05_PAIR)
    assert ei.value.status == 2 and "256" in str(ei.value)


E4M3_SHAPES = [  # T, k, E, K, I
    (96, 4, 8, 512, 256),            # ~48 tokens per expert
    (300, 1, 2, 256, 128),           # ~150 tokens per expert: three 64-token segments
    (5, 8, 64, 512, 128),            # decode-like
    (40, 2, 4, 384, 384),            # three k slices in both GEMMs (the second MMA issuer takes one)
    # 16 or fewer rows per expert on average: 32-token tiles with four MMA warps
    (90, 1, 6, 384, 256),            # steep bias: the first expert needs several 32-token tiles; 3 k slices
    (64, 2, 16, 256, 384),           # GEMM 2 with three k slices
]


def _e4m3_weights(moe, W):
    """Quantise fp32 weights with the library (codes are checked bit-exact elsewhere) and by the oracle."""
    W = W.clone()
    W[0, 3, :64] = 0.0                                  # an all-zero block and zero codes
    W[0, 5, :32] *= 1e-3                                # subnormal codes next to normal ones
    W[0, 5, 7] = 2.0
    codes, scales = moe.mxfp8_quantize_block32(W.to(DEV))
    rc, rs = oracle.mxfp8_quantize(W.numpy())
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)
    return codes, scales, rc, rs


@pytest.mark.parametrize("impl", ["swap_ab", "auto", "simt"])
@pytest.mark.parametrize("shape", E4M3_SHAPES)
@pytest.mark.parametrize("w1_layout", [0, 1])
def test_gemm1_swiglu_e4m3(moe, impl, shape, w1_layout):
    T, k, E, K, I = shape
    w, x, ids, _ = _routed(T, k, E, K, seed=T + 3 * E)
    W1 = wl.expert_weights(wl.scaled(w, I=I, weight="mxfp8"), "W1", 5)
    c1, s1, rc1, rs1 = _e4m3_weights(moe, W1)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    h = moe.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], c1, I, w1_scale=s1,
                             w1_layout=w1_layout, impl=_impl(moe, impl))
    href = oracle.expert_gate_up(wl.to_numpy(x)[np.arange(T * k) // k], ids.reshape(-1), rc1, w1_scale=rs1,
                                 w1_layout=w1_layout)
    rr = res["route_row"].cpu().numpy().reshape(-1)
    assert_close(to_f64(h.cpu()[torch.from_numpy(rr).long()]), href, TOL_BF16, f"gemm1 e4m3 {impl}")


@pytest.mark.parametrize("impl", ["swap_ab", "auto"])
@pytest.mark.parametrize("maxT", [12, 48])
def test_gemms_batched_layout_e4m3(moe, impl, maxT):
    """MXFP8 weights on the batched (E, max_tokens, K) layout: max_tokens = 12 runs the 32-token tiles with four
    MMA warps (16 or fewer rows per expert), 48 the 64-token tiles with two; full, ragged, empty and one-token
    experts, GEMM 2 with the per-row weight."""
    E, K, I = 5, 256, 256
    w = wl.scaled(wl.tiny(), T=1, K=K, I=I, E=E, top_k=1, x_std=1.0, w_std=0.05, weight="mxfp8")
    counts = torch.tensor([maxT, maxT - 1, maxT // 2 + 1, 0, 1], dtype=torch.int32)
    x = wl._normal((E, maxT, K), 1.0, 17, "x", 0, "cpu", torch.bfloat16)
    rw = torch.rand((E, maxT), generator=torch.Generator().manual_seed(maxT))
    c1, s1, rc1, rs1 = _e4m3_weights(moe, wl.expert_weights(w, "W1", 8))
    c2, s2, rc2, rs2 = _e4m3_weights(moe, wl.expert_weights(w, "W2", 8))
    offs = torch.arange(E + 1, dtype=torch.int32) * maxT
    kw = dict(layout=moe.MOE_LAYOUT_BATCHED, max_tokens=maxT, impl=_impl(moe, impl))
    h = moe.moe_gemm1_swiglu(x.to(DEV).reshape(E * maxT, K), counts.to(DEV), offs.to(DEV), c1, I, w1_scale=s1, **kw)
    y = moe.moe_gemm2(h, counts.to(DEV), offs.to(DEV), c2, E * maxT, w2_scale=s2,
                      route_weights=rw.to(DEV).reshape(-1), **kw)
    torch.cuda.synchronize()
    hc, yc = h.cpu().reshape(E, maxT, I), y.cpu().reshape(E, maxT, K)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        ids = np.full(c, e, dtype=np.int32)
        href = oracle.expert_gate_up(wl.to_numpy(x[e, :c]), ids, rc1, w1_scale=rs1)
        assert_close(to_f64(hc[e, :c]), href, TOL_BF16, f"batched e4m3 gemm1 expert {e}")
        yref = oracle.expert_down(wl.to_numpy(hc[e, :c]), ids, rc2, w2_scale=rs2)
        yref = yref * rw[e, :c].numpy().astype(np.float64)[:, None]
        assert_close(to_f64(yc[e, :c]), yref, TOL_BF16, f"batched e4m3 gemm2 expert {e}")


@pytest.mark.parametrize("impl", ["swap_ab", "auto", "simt"])
@pytest.mark.parametrize("shape", E4M3_SHAPES)
def test_gemm2_e4m3(moe, impl, shape):
    T, k, E, K, I = shape
    w, _, ids, weights = _routed(T, k, E, K, seed=T + 4 * E)
    W2 = wl.expert_weights(wl.scaled(w, I=I, weight="mxfp8"), "W2", 6)
    c2, s2, rc2, rs2 = _e4m3_weights(moe, W2)
    R = T * k
    hsrc = wl._normal((R, I), 1.0, 8, "h", 0, "cpu", torch.bfloat16)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1)
    hperm = torch.zeros((res["rows_cap"], I), dtype=torch.bfloat16, device=DEV)
    hperm[res["route_row"].view(-1).long()] = hsrc.to(DEV)
    wt = torch.from_numpy(weights).to(DEV).reshape(-1)
    y = moe.moe_gemm2(hperm, res["counts"], res["offsets"], c2, R, w2_scale=s2, row_route=res["row_route"],
                      route_weights=wt, impl=_impl(moe, impl))
    yref = oracle.expert_down(wl.to_numpy(hsrc), ids.reshape(-1), rc2, w2_scale=rs2)
    yref = yref * weights.reshape(-1, 1).astype(np.float64)
    assert_close(to_f64(y.cpu()), yref, TOL_BF16, f"gemm2 e4m3 {impl}")


def _exp_classes(n):
    """Power-of-two exponents for n weight units or output columns: whole 64-unit blocks at 2^0, 2^30 and 2^48
    in turn (so some 128-row weight tiles hold ordinary scales only and others large ones), and every fifth unit
    of the 2^0 blocks at 2^40 (large scale codes next to ordinary ones in one warp)."""
    s = np.array([0, 30, 48])[(np.arange(n) // 64) % 3]
    s[(s == 0) & (np.arange(n) % 5 == 2)] = 40
    return s


@pytest.mark.parametrize("shape", [(96, 4, 8, 512, 256), (5, 8, 64, 512, 256)])   # 64- / 32-token tiles
@pytest.mark.parametrize("impl", ["swap_ab", "simt"])
@pytest.mark.parametrize("w1_layout", [0, 1])
def test_e4m3_large_scale_codes(moe, shape, impl, w1_layout):
    """E8M0 scale codes above 134, for which the decoding's factor 2^(sc-7) leaves bf16's range and is applied as
    2^(sc-127) then 2^120, beside ordinary codes in the same tiles and warps (the MXFP8 block format, "Cake
    MegaMoE EP16" FlashInfer PR 5148 analysis, section 2): W1 units and W2 output columns scaled by 2^0, 2^30,
    2^40 and 2^48 (scale codes about 116 to 164), each class compared with the oracle on its own columns."""
    T, k, E, K, I = shape
    w, x, ids, weights = _routed(T, k, E, K, seed=T + 5 * E)
    wm = wl.scaled(w, I=I, weight="mxfp8")
    W1 = wl.expert_weights(wm, "W1", 9)
    units = np.arange(2 * I)
    units = units % I if w1_layout == 0 else 16 * (units // 32) + units % 16   # the unit of each W1 row
    s1 = _exp_classes(I)
    W1 *= torch.from_numpy(2.0 ** s1[units]).float()[None, :, None]
    W2 = wl.expert_weights(wm, "W2", 9)
    s2 = _exp_classes(K)
    W2 *= torch.from_numpy(2.0 ** s2).float()[None, :, None]
    c1, sc1, rc1, rs1 = _e4m3_weights(moe, W1)
    c2, sc2, rc2, rs2 = _e4m3_weights(moe, W2)
    assert rs1.max() > 134 and rs1.min() <= 134 and rs2.max() > 134
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    h = moe.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], c1, I, w1_scale=sc1,
                             w1_layout=w1_layout, impl=_impl(moe, impl))
    rr = res["route_row"].view(-1).long()
    href = oracle.expert_gate_up(wl.to_numpy(x)[np.arange(T * k) // k], ids.reshape(-1), rc1, w1_scale=rs1,
                                 w1_layout=w1_layout)
    # GEMM 2 on ordinary h rows (h above reaches 2^96, which times 2^48 would leave bf16's range)
    hsrc = wl._normal((T * k, I), 1.0, 10, "h", 0, "cpu", torch.bfloat16)
    hperm = torch.zeros((res["rows_cap"], I), dtype=torch.bfloat16, device=DEV)
    hperm[rr] = hsrc.to(DEV)
    wt = torch.from_numpy(weights).to(DEV).reshape(-1)
    y = moe.moe_gemm2(hperm, res["counts"], res["offsets"], c2, T * k, w2_scale=sc2, row_route=res["row_route"],
                      route_weights=wt, impl=_impl(moe, impl))
    yref = oracle.expert_down(wl.to_numpy(hsrc), ids.reshape(-1), rc2, w2_scale=rs2)
    yref = yref * weights.reshape(-1, 1).astype(np.float64)
    hg, yg = to_f64(h[rr].cpu()), to_f64(y.cpu())
    for c in np.unique(s1):
        cols = np.nonzero(s1 == c)[0]
        assert_close(hg[:, cols], href[:, cols], TOL_BF16, f"gemm1 e4m3 {impl} units at 2^{c}")
    for c in np.unique(s2):
        cols = np.nonzero(s2 == c)[0]
        assert_close(yg[:, cols], yref[:, cols], TOL_BF16, f"gemm2 e4m3 {impl} columns at 2^{c}")


MX_SHAPES = E4M3_SHAPES + [(700, 2, 6, 256, 128)]   # + skewed: full, long and short token segments


def _mx_rows(moe, a):
    """MXFP8 rows (codes, scales) of bf16 rows `a` on the GPU, checked bit-exact against the oracle."""
    codes, scales = moe.mxfp8_quantize_block32(a.to(DEV))
    rc, rs = oracle.mxfp8_quantize(wl.to_numpy(a.cpu()))
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)
    return codes, scales, rc, rs


@pytest.mark.parametrize("impl", ["swap_ab", "auto", "simt"])
@pytest.mark.parametrize("shape", MX_SHAPES)
@pytest.mark.parametrize("w1_layout", [0, 1])
def test_gemm1_swiglu_mxf8(moe, impl, shape, w1_layout):
    """MXFP8 activations x MXFP8 weights (block-scaled tcgen05 MMA) against the oracle on the decoded values."""
    T, k, E, K, I = shape
    w, x, ids, _ = _routed(T, k, E, K, seed=T + 5 * E)
    W1 = wl.expert_weights(wl.scaled(w, I=I, weight="mxfp8", w_std=0.05), "W1", 9)
    c1, s1, rc1, rs1 = _e4m3_weights(moe, W1)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    xc, xs, _, _ = _mx_rows(moe, res["x_out"])
    h = moe.moe_gemm1_swiglu(xc, res["counts"], res["offsets"], c1, I, w1_scale=s1, a_scale=xs,
                             w1_layout=w1_layout, impl=_impl(moe, impl))
    xr = wl.to_numpy(x)[np.arange(T * k) // k]
    xq = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(xr))          # the rows the GPU multiplied
    href = oracle.expert_gate_up(xq, ids.reshape(-1), rc1, w1_scale=rs1, w1_layout=w1_layout)
    rr = res["route_row"].cpu().numpy().reshape(-1)
    assert_close(to_f64(h.cpu()[torch.from_numpy(rr).long()]), href, TOL_BF16, f"gemm1 mxf8 {impl}")


@pytest.mark.parametrize("impl", ["swap_ab", "simt"])
@pytest.mark.parametrize("shape", MX_SHAPES)
def test_gemm2_mxf8(moe, impl, shape):
    T, k, E, K, I = shape
    w, _, ids, weights = _routed(T, k, E, K, seed=T + 6 * E)
    W2 = wl.expert_weights(wl.scaled(w, I=I, weight="mxfp8", w_std=0.05), "W2", 10)
    c2, s2, rc2, rs2 = _e4m3_weights(moe, W2)
    R = T * k
    hsrc = wl._normal((R, I), 1.0, 11, "h", 0, "cpu", torch.bfloat16)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1)
    hperm = torch.zeros((res["rows_cap"], I), dtype=torch.bfloat16, device=DEV)
    hperm[res["route_row"].view(-1).long()] = hsrc.to(DEV)
    hc, hs, _, _ = _mx_rows(moe, hperm)
    wt = torch.from_numpy(weights).to(DEV).reshape(-1)
    y = moe.moe_gemm2(hc, res["counts"], res["offsets"], c2, R, w2_scale=s2, h_scale=hs, row_route=res["row_route"],
                      route_weights=wt, impl=_impl(moe, impl))
    hq = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(wl.to_numpy(hsrc)))
    yref = oracle.expert_down(hq, ids.reshape(-1), rc2, w2_scale=rs2)
    yref = yref * weights.reshape(-1, 1).astype(np.float64)
    assert_close(to_f64(y.cpu()), yref, TOL_BF16, f"gemm2 mxf8 {impl}")


@pytest.mark.parametrize("act", ["bf16", "mxfp8"])
@pytest.mark.parametrize("shape", [(5, 8, 64, 512, 128), (96, 4, 8, 512, 256), (64, 2, 16, 384, 384)])
@pytest.mark.parametrize("impl", ["swap_ab", "auto"])
def test_e4m3_tiled_codes_bit_identical(moe, act, shape, impl):
    """E4M3 codes re-laid out by moe_tile_weights (interleave-16 W1, W2; scales as stored) give the same h and y,
    bit for bit, as the codes as stored: bf16 activations on both E4M3 tile forms (the first and last shape run
    the 32-token tiles, the second the 64-token ones), MXFP8 activations on the block-scaled tiles."""
    T, k, E, K, I = shape
    w, x, ids, weights = _routed(T, k, E, K, seed=T + 9 * E)
    W1 = wl.expert_weights(wl.scaled(w, I=I, weight="mxfp8"), "W1", 12)
    W2 = wl.expert_weights(wl.scaled(w, I=I, weight="mxfp8"), "W2", 12)
    c1, s1 = moe.mxfp8_quantize_block32(W1.to(DEV))
    c2, s2 = moe.mxfp8_quantize_block32(W2.to(DEV))
    c1t = moe.moe_tile_weights(c1, 1, moe.MOE_W1_INTERLEAVE16)
    c2t = moe.moe_tile_weights(c2, 2)
    assert not torch.equal(c1t, c1)                            # the layout did change
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    R = T * k
    wt = torch.from_numpy(weights).to(DEV).reshape(-1)
    a, a_scale = res["x_out"], None
    if act == "mxfp8":
        a, a_scale = moe.mxfp8_quantize_block32(a)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for w1x, w2x, l1, l2 in ((c1, c2, moe.MOE_W1_INTERLEAVE16, moe.MOE_W1_GATE_UP),
                             (c1t, c2t, moe.MOE_W_TILED, moe.MOE_W_TILED)):
        h = moe.moe_gemm1_swiglu(a, res["counts"], res["offsets"], w1x, I, w1_scale=s1, a_scale=a_scale,
                                 w1_layout=l1, impl=_impl(moe, impl), err_word=err)
        h2, h2s = (h, None) if act == "bf16" else moe.mxfp8_quantize_block32(h)
        y = moe.moe_gemm2(h2, res["counts"], res["offsets"], w2x, R, w2_scale=s2, h_scale=h2s,
                          row_route=res["row_route"], route_weights=wt, w2_layout=l2, impl=_impl(moe, impl),
                          err_word=err)
        outs.append((h, y))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    (h1, y1), (h2_, y2) = outs
    rr = res["route_row"].view(-1).long()
    assert torch.equal(h1[rr].view(torch.int16), h2_[rr].view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    if act == "bf16":   # and the tiled result against the oracle
        rc1, rs1 = oracle.mxfp8_quantize(W1.numpy())
        href = oracle.expert_gate_up(wl.to_numpy(x)[np.arange(R) // k], ids.reshape(-1), rc1, w1_scale=rs1,
                                     w1_layout=moe.MOE_W1_INTERLEAVE16)
        assert_close(to_f64(h2_.cpu()[rr.cpu()]), href, TOL_BF16, "gemm1 e4m3 tiled codes")


@pytest.mark.parametrize("impl", ["swap_ab", "simt"])
@pytest.mark.parametrize("shape", MX_SHAPES)
@pytest.mark.parametrize("w1_layout", [0, 1])
def test_gemm1_mxf8_fused_h_quant(moe, impl, shape, w1_layout):
    """h written as MXFP8 by GEMM 1's epilogue equals, bit for bit, mxfp8_quantize_block32 of the bf16 h the
    same GEMM writes otherwise (codes and scales of every valid row)."""
    T, k, E, K, I = shape
    w, x, ids, _ = _routed(T, k, E, K, seed=T + 7 * E)
    W1 = wl.expert_weights(wl.scaled(w, I=I, weight="mxfp8", w_std=0.05), "W1", 13)
    c1, s1, _, _ = _e4m3_weights(moe, W1)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    xc, xs = moe.mxfp8_quantize_block32(res["x_out"])
    kw = dict(w1_scale=s1, a_scale=xs, w1_layout=w1_layout, impl=_impl(moe, impl))
    h = moe.moe_gemm1_swiglu(xc, res["counts"], res["offsets"], c1, I, **kw)
    rc, rs = moe.mxfp8_quantize_block32(h)
    hc, hs = moe.moe_gemm1_swiglu(xc, res["counts"], res["offsets"], c1, I, h_dtype=moe.MOE_E4M3, **kw)
    rows = res["route_row"].view(-1).long()
    assert torch.equal(hc[rows], rc[rows]) and torch.equal(hs[rows], rs[rows])
    assert int((hs[rows] > 0).sum()) > 0


def test_mxf8_refuses_normal_tiles(moe):
    T, k, E, K, I = 64, 2, 4, 256, 128
    w, x, ids, _ = _routed(T, k, E, K, seed=12)
    W1 = wl.expert_weights(wl.scaled(w, I=I, weight="mxfp8"), "W1", 7)
    c1, s1 = moe.mxfp8_quantize_block32(W1.to(DEV))
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    xc, xs = moe.mxfp8_quantize_block32(res["x_out"])
    for impl in (moe.MOE_IMPL_TCGEN05, moe.MOE_IMPL_TCGEN05_MIXED):
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_gemm1_swiglu(xc, res["counts"], res["offsets"], c1, I, w1_scale=s1, a_scale=xs, impl=impl)
        assert ei.value.status == 2


def test_e4m3_normal_tiles_unsupported_but_auto_works(moe):
    T, k, E, K, I = 64, 2, 4, 256, 128
    w, x, ids, _ = _routed(T, k, E, K, seed=11)
    W1 = wl.expert_weights(wl.scaled(w, I=I, weight="mxfp8"), "W1", 7)
    c1, s1 = moe.mxfp8_quantize_block32(W1.to(DEV))
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], c1, I, w1_scale=s1,
                             impl=moe.MOE_IMPL_TCGEN05)
    assert ei.value.status == 2


def test_gemm_unsupported_shape_falls_back_under_auto(moe):
    """K not a multiple of 64: AUTO uses the CUDA-core tiles; forcing tcgen05 reports UNSUPPORTED."""
    T, k, E, K, I = 20, 2, 4, 96, 64
    w, x, ids, _ = _routed(T, k, E, K, seed=1)
    W1 = wl.expert_weights(wl.scaled(w, I=I), "W1", 1)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], W1.to(DEV), I,
                             impl=moe.MOE_IMPL_TCGEN05)
    assert ei.value.status == 2
    h = moe.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], W1.to(DEV), I, impl=moe.MOE_IMPL_AUTO)
    href = oracle.expert_gate_up(wl.to_numpy(x)[np.arange(T * k) // k], ids.reshape(-1), wl.to_numpy(W1))
    rr = res["route_row"].cpu().numpy().reshape(-1)
    assert_close(to_f64(h.cpu()[torch.from_numpy(rr).long()]), href, TOL_BF16, "auto fallback")


# ----------------------------------------------------------------------------
# whole layer
# ----------------------------------------------------------------------------

def test_layer_tiny_fp32(moe):
    """The fp32 configuration: T=16, K=128, I=256, E=8, top_k=2 -- tolerance 1e-5."""
    w = wl.tiny()
    x, logits = wl.activations(w, 0), wl.router_logits(w, 0)
    W1, W2 = wl.expert_weights(w, "W1", 0), wl.expert_weights(w, "W2", 0)
    for weight_in_gemm2 in (True, False):
        layer = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, act_dtype=torch.float32,
                             weight_in_gemm2=weight_in_gemm2, device=DEV)
        out = layer.forward(x.to(DEV), W1.to(DEV), W2.to(DEV), logits=logits.to(DEV))
        ids, weights = oracle.topk_route(logits.numpy(), w.top_k)
        assert np.array_equal(layer.ids.cpu().numpy(), ids)
        ref, _ = oracle.moe_layer(x.numpy(), ids, weights, W1.numpy(), W2.numpy())
        assert_close(to_f64(out.cpu()), ref, TOL_F32, "tiny fp32 layer")
        assert layer.device_errors() == 0


@pytest.mark.parametrize("impl", IMPLS_BF16 + ["auto"])
@pytest.mark.parametrize("bm", [1, 128])
@pytest.mark.parametrize("seed", [3, 1, 2])
def test_layer_bf16_small(moe, impl, bm, seed):
    w = wl.scaled(wl.decode(64), T=200, K=512, I=256, E=16, top_k=4)
    x, logits = wl.activations(w, seed), wl.router_logits(w, seed)
    W1, W2 = wl.expert_weights(w, "W1", seed), wl.expert_weights(w, "W2", seed)
    layer = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, block_m=bm, impl=_impl(moe, impl), device=DEV)
    out = layer.forward(x.to(DEV), W1.to(DEV), W2.to(DEV), logits=logits.to(DEV))
    ids, weights = oracle.topk_route(logits.numpy(), w.top_k)
    ref, _ = oracle.moe_layer(wl.to_numpy(x), ids, weights, wl.to_numpy(W1), wl.to_numpy(W2))
    assert_close(to_f64(out.cpu()), ref, TOL_BF16, f"layer {impl} bm={bm}")
    first = out.clone()
    layer.forward(x.to(DEV), W1.to(DEV), W2.to(DEV), logits=logits.to(DEV))
    assert torch.equal(first.view(torch.int16), out.view(torch.int16))          # run-to-run identical
    assert layer.device_errors() == 0


@pytest.mark.parametrize("T,layout", [(128, "contiguous"), (129, "contiguous"), (100, "batched"),
                                      (129, "batched")])
def test_layer_routing_launch_boundary(moe, T, layout):
    """Router logits in, on both sides of the one-launch routing limit (T <= 128, 1024 routes): the layer matches
    the oracle and issues the launches launches_per_forward() counts (1 or 4 before the GEMMs)."""
    k, E = 8, 32
    w = wl.scaled(wl.decode(64), T=T, K=256, I=128, E=E, top_k=k)
    x, logits = wl.activations(w, 12), wl.router_logits(w, 12)
    W1, W2 = wl.expert_weights(w, "W1", 12), wl.expert_weights(w, "W2", 12)
    lay = moe.MOE_LAYOUT_CONTIGUOUS if layout == "contiguous" else moe.MOE_LAYOUT_BATCHED
    mt = 48 if layout == "batched" else 0                    # batched: some routes dropped for capacity
    layer = moe.MoELayer(T, w.K, w.I, E, k, layout=lay, max_tokens=mt, device=DEV)
    out = layer.forward(x.to(DEV), W1.to(DEV), W2.to(DEV), logits=logits.to(DEV))
    torch.cuda.synchronize()
    ids, weights = oracle.topk_route(logits.numpy(), k)
    assert np.array_equal(layer.ids.cpu().numpy(), ids)
    if layout == "batched":
        kept = layer.route_row.cpu().numpy() >= 0
        ids = np.where(kept, ids, -1).astype(np.int32)
    ref, _ = oracle.moe_layer(wl.to_numpy(x), ids, weights, wl.to_numpy(W1), wl.to_numpy(W2))
    assert_close(to_f64(out.cpu()), ref, TOL_BF16, f"layer T={T} {layout}")
    names = [name for _, _, name in layer._plan]
    assert names[0] == "route_permute"
    front = 1 if T <= 128 else 1 + 2 + 1                     # route, permute (two launches above 1024 routes), gather
    gemms = 1 if any(fn is layer.lib.moe_experts_fused for fn, _, _ in layer._plan) else 2
    assert layer.launches_per_forward() == front + gemms + 1


def test_layer_padding_tokens(moe):
    """Tokens whose slots are all padding (id -1, weight 0) come out as +0.0."""
    w = wl.scaled(wl.decode(64), T=24, K=256, I=128, E=8, top_k=2)
    x = wl.activations(w, 4)
    ids, weights = oracle.topk_route(wl.router_logits(w, 4).numpy(), w.top_k)
    ids_t, w_t = wl.padding_tokens(torch.from_numpy(ids), torch.from_numpy(weights), 8)
    x_all = torch.cat([x, wl._normal((8, w.K), 1.0, 9, "xp", 0, "cpu", torch.bfloat16)])
    ids_t[3, 1], w_t[3, 1] = -1, 0.0
    W1, W2 = wl.expert_weights(w, "W1", 4), wl.expert_weights(w, "W2", 4)
    T = x_all.shape[0]
    for impl in ("tcgen05", "swap_ab"):
        layer = moe.MoELayer(T, w.K, w.I, w.E, w.top_k, impl=_impl(moe, impl), device=DEV)
        out = layer.forward(x_all.to(DEV), W1.to(DEV), W2.to(DEV), topk_ids=ids_t.to(DEV),
                            topk_weights=w_t.to(DEV)).cpu()
        ref, _ = oracle.moe_layer(wl.to_numpy(x_all), ids_t.numpy(), w_t.numpy(), wl.to_numpy(W1),
                                  wl.to_numpy(W2))
        assert_close(to_f64(out), ref, TOL_BF16, "padding")
        assert torch.all(out[-8:] == 0) and not torch.any(torch.signbit(out[-8:].float()))


def test_layer_decode_full_size_sampled(moe):
    """Decode configuration at full size (K=4096, I=1536, E=128, top_k=8), T=8; oracle on 2 tokens."""
    w = wl.decode(8)
    x, logits = wl.activations(w, 0, DEV), wl.router_logits(w, 0, DEV)
    W1, W2 = wl.expert_weights(w, "W1", 0, DEV), wl.expert_weights(w, "W2", 0, DEV)
    for impl in ("auto", "tcgen05"):
        layer = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, impl=_impl(moe, impl), device=DEV)
        out = layer.forward(x, W1, W2, logits=logits)
        ids, weights = oracle.topk_route(logits.cpu().numpy(), w.top_k)
        assert np.array_equal(layer.ids.cpu().numpy(), ids)
        for t in (0, 5):
            cids, (w1h, w2h, _, _) = compact_experts(ids[t:t + 1], W1, W2)
            ref, _ = oracle.moe_layer(wl.to_numpy(x[t:t + 1]), cids, weights[t:t + 1], w1h, w2h)
            assert_close(to_f64(out[t:t + 1]), ref, TOL_BF16, f"decode token {t} {impl}")


def test_layer_prefill_full_size_sampled(moe):
    """Skewed prefill at full size (T=4096, bm=128); oracle on 2 tokens, one of them routed to the hottest expert."""
    w = wl.prefill()
    x, logits = wl.activations(w, 0, DEV), wl.router_logits(w, 0, DEV)
    W1, W2 = wl.expert_weights(w, "W1", 0, DEV), wl.expert_weights(w, "W2", 0, DEV)
    layer = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, block_m=w.block_m, device=DEV)
    out = layer.forward(x, W1, W2, logits=logits)
    ids, weights = oracle.topk_route(logits.cpu().numpy(), w.top_k)
    assert np.array_equal(layer.ids.cpu().numpy(), ids)
    ref_perm = oracle.permute_contiguous(ids, w.E, w.block_m)
    assert np.array_equal(layer.offsets.cpu().numpy(), ref_perm["offsets"])
    assert np.array_equal(layer.row_route[:ref_perm["offsets"][-1]].cpu().numpy(), ref_perm["sorted_route"])
    for t in (0, 4095):
        cids, (w1h, w2h, _, _) = compact_experts(ids[t:t + 1], W1, W2)
        ref, _ = oracle.moe_layer(wl.to_numpy(x[t:t + 1]), cids, weights[t:t + 1], w1h, w2h)
        assert_close(to_f64(out[t:t + 1]), ref, TOL_BF16, f"prefill token {t}")
    assert layer.device_errors() == 0


def _mxfp8_weights(moe, w, which, seed):
    rows = 2 * w.I if which == "W1" else w.K
    cols = w.K if which == "W1" else w.I
    codes = torch.empty((w.E, rows, cols), dtype=torch.uint8, device=DEV)
    scales = torch.empty((w.E, rows, cols // 32), dtype=torch.uint8, device=DEV)
    for e in range(w.E):
        Wf = wl.expert_weights(w, which, seed, DEV, experts=[e])[0]
        moe.mxfp8_quantize_block32(Wf, codes=codes[e], scales=scales[e])
    return codes, scales


def test_layer_mxfp8_full_size_sampled(moe):
    """MXFP8 weights (E=512, K=7168, I=2048, interleave-16 W1, affine routing); oracle on 2 tokens."""
    w = wl.mxfp8()
    x = wl.activations(w, 0, DEV)
    ids_t, w_t = wl.affine_routing(w)
    c1, s1 = _mxfp8_weights(moe, w, "W1", 0)
    c2, s2 = _mxfp8_weights(moe, w, "W2", 0)
    # the GPU codes of one expert equal the oracle's codes of the same fp32 draw
    W1e = wl.expert_weights(w, "W1", 0, DEV, experts=[19])[0].cpu()
    rc, rs = oracle.mxfp8_quantize(W1e.numpy())
    assert np.array_equal(c1[19].cpu().numpy(), rc) and np.array_equal(s1[19].cpu().numpy(), rs)
    layer = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, device=DEV)
    out = layer.forward(x, c1, c2, topk_ids=ids_t.to(DEV), topk_weights=w_t.to(DEV), w1_scale=s1, w2_scale=s2,
                        w1_layout=moe.MOE_W1_INTERLEAVE16)
    ids = ids_t.numpy()
    for t in (0, 511):
        cids, (w1h, w2h, s1h, s2h) = compact_experts(ids[t:t + 1], c1, c2, s1, s2)
        ref, _ = oracle.moe_layer(wl.to_numpy(x[t:t + 1]), cids, w_t[t:t + 1].numpy(), w1h, w2h, w1_scale=s1h,
                                  w2_scale=s2h, w1_layout=1)
        assert_close(to_f64(out[t:t + 1]), ref, TOL_BF16, f"mxfp8 token {t}")


@pytest.mark.parametrize("impl", ["auto", "simt"])
def test_layer_mxf8_activations_small(moe, impl):
    """Whole layer with MXFP8 weights and activations quantised on the fly (x rows and h), against the oracle
    with the same quantisation points (x from its stored bf16 values, h rounded to bf16 first)."""
    T, k, E, K, I = 80, 4, 8, 512, 256
    w = wl.scaled(wl.decode(T), T=T, K=K, I=I, E=E, top_k=k, weight="mxfp8", w_std=0.05)
    x, logits = wl.activations(w, 2), wl.router_logits(w, 2)
    c1, s1, rc1, rs1 = _e4m3_weights(moe, wl.expert_weights(w, "W1", 2))
    c2, s2, rc2, rs2 = _e4m3_weights(moe, wl.expert_weights(w, "W2", 2))
    layer = moe.MoELayer(T, K, I, E, k, act_quant=True, impl=_impl(moe, impl), device=DEV)
    out = layer.forward(x.to(DEV), c1, c2, logits=logits.to(DEV), w1_scale=s1, w2_scale=s2)
    assert layer.device_errors() == 0
    ids, wts = oracle.topk_route(logits.numpy(), k)
    ref, _ = oracle.moe_layer(wl.to_numpy(x), ids, wts, rc1, rc2, w1_scale=rs1, w2_scale=rs2, quant_x=True,
                              quant_h="bf16")
    assert_close(to_f64(out), ref, TOL_BF16, f"layer mxf8 activations {impl}")


def test_layer_mxfp8_act_quant_full_size_sampled(moe):
    """MXFP8 workload (E=512, K=7168, I=2048, interleave-16 W1, affine routing) with activations quantised on the
    fly, as the benchmark's mxfp8_act workload runs it; oracle on 2 tokens."""
    w = wl.mxfp8()
    x = wl.activations(w, 0, DEV)
    ids_t, w_t = wl.affine_routing(w)
    c1, s1 = _mxfp8_weights(moe, w, "W1", 0)
    c2, s2 = _mxfp8_weights(moe, w, "W2", 0)
    layer = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, act_quant=True, device=DEV)
    out = layer.forward(x, c1, c2, topk_ids=ids_t.to(DEV), topk_weights=w_t.to(DEV), w1_scale=s1, w2_scale=s2,
                        w1_layout=moe.MOE_W1_INTERLEAVE16)
    assert layer.device_errors() == 0
    ids = ids_t.numpy()
    for t in (0, 511):
        cids, (w1h, w2h, s1h, s2h) = compact_experts(ids[t:t + 1], c1, c2, s1, s2)
        ref, _ = oracle.moe_layer(wl.to_numpy(x[t:t + 1]), cids, w_t[t:t + 1].numpy(), w1h, w2h, w1_scale=s1h,
                                  w2_scale=s2h, w1_layout=1, quant_x=True, quant_h="bf16")
        assert_close(to_f64(out[t:t + 1]), ref, TOL_BF16, f"mxfp8 act-quant token {t}")


@pytest.mark.parametrize("garbage", ["nan", "big"])
def test_layer_batched_full_size_sampled(moe, garbage):
    """Batched layout (E=32, max_tokens=256, K=6144, I=4096); garbage rows ignored; oracle on sampled rows."""
    w = wl.batched(garbage)
    xb, counts, rw = wl.batched_inputs(w, 0, DEV)
    W1, W2 = wl.expert_weights(w, "W1", 0, DEV), wl.expert_weights(w, "W2", 0, DEV)
    layer = moe.MoELayer(0, w.K, w.I, w.E, 1, layout=moe.MOE_LAYOUT_BATCHED, max_tokens=w.max_tokens, device=DEV)
    layer.out.fill_(3.0)
    out = layer.forward(xb, W1, W2, expert_num_tokens=counts, row_weights=rw)
    cnt = counts.cpu().numpy()
    for e in (int(np.argmax(cnt)), int(np.argmin(np.where(cnt > 0, cnt, 999)))):
        c = int(cnt[e])
        rows = sorted({0, c - 1, c // 2})
        sub = xb[e, rows][None]                             # (1, len(rows), K)
        ref, _ = oracle.moe_layer_batched(wl.to_numpy(sub), np.array([len(rows)], np.int32),
                                          rw[e, rows][None].cpu().numpy(), wl.to_numpy(W1[e:e + 1]),
                                          wl.to_numpy(W2[e:e + 1]))
        assert_close(to_f64(out[e, rows]), ref[0], TOL_BF16, f"batched expert {e}")
        if c < w.max_tokens:
            assert torch.all(out[e, c:] == 3.0)             # rows beyond the count untouched
    assert torch.isfinite(out.float()).sum() > 0


def test_layer_batched_tokens_full_size_sampled(moe):
    """Batched layout fed with tokens at full size (T=1024, top_k=4, E=32, max_tokens=256, K=6144, I=4096),
    as the benchmark runs it: permutation bit-exact, oracle on 2 sampled tokens."""
    w = wl.batched_tokens()
    x, logits = wl.activations(w, 0, DEV), wl.router_logits(w, 0, DEV)
    W1, W2 = wl.expert_weights(w, "W1", 0, DEV), wl.expert_weights(w, "W2", 0, DEV)
    layer = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, layout=moe.MOE_LAYOUT_BATCHED, max_tokens=w.max_tokens,
                         device=DEV)
    out = layer.forward(x, W1, W2, logits=logits)
    ids, weights = oracle.topk_route(logits.cpu().numpy(), w.top_k)
    assert np.array_equal(layer.ids.cpu().numpy(), ids)
    ref_perm = oracle.permute_batched(ids, w.E, w.max_tokens)
    assert np.array_equal(layer.counts.cpu().numpy(), ref_perm["expert_num_tokens"])
    assert np.array_equal(layer.route_row.cpu().numpy(), ref_perm["route_row"])
    assert layer.device_errors() == ref_perm["err"]
    for t in (0, 1023):
        cids, (w1h, w2h, _, _) = compact_experts(ids[t:t + 1], W1, W2)
        ref, _ = oracle.moe_layer(wl.to_numpy(x[t:t + 1]), cids, weights[t:t + 1], w1h, w2h)
        assert_close(to_f64(out[t:t + 1]), ref, TOL_BF16, f"batched_tokens token {t}")


# ----------------------------------------------------------------------------
# GEMM 1 + GEMM 2 in one launch
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(5, 8, 64, 512, 128, 0), (96, 4, 8, 512, 256, 1), (700, 2, 6, 256, 128, 0),
                                   (1, 8, 128, 1024, 192, 1)])
def test_experts_fused_matches_two_launches(moe, shape):
    """moe_experts_fused equals moe_gemm1_swiglu + moe_gemm2 on swap-AB tiles bit for bit (same tiles, same
    accumulation order) and the oracle within tolerance; run twice (the workspace is cleared by each call)."""
    T, k, E, K, I, w1_layout = shape
    w, x, ids, weights = _routed(T, k, E, K, seed=T + 9 * E)
    ws = wl.scaled(w, I=I, w_std=0.05)
    W1 = wl.expert_weights(ws, "W1", 14).to(torch.bfloat16)
    W2 = wl.expert_weights(ws, "W2", 14).to(torch.bfloat16)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    R = T * k
    wt = torch.from_numpy(weights).to(DEV).reshape(-1)
    swap = moe.MOE_IMPL_TCGEN05_SWAP_AB
    h2 = moe.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], W1.to(DEV), I, w1_layout=w1_layout,
                              impl=swap)
    y2 = moe.moe_gemm2(h2, res["counts"], res["offsets"], W2.to(DEV), R, row_route=res["row_route"],
                       route_weights=wt, impl=swap)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        h1, y1 = moe.moe_experts_fused(res["x_out"], res["counts"], res["offsets"], W1.to(DEV), W2.to(DEV), I,
                                       res["row_route"], R, route_weights=wt, w1_layout=w1_layout, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    ref, _ = oracle.moe_layer(wl.to_numpy(x), ids, weights, wl.to_numpy(W1), wl.to_numpy(W2), w1_layout=w1_layout)
    # y holds w * FFN per (token, slot); summing the slots reproduces the layer
    out = moe.moe_unpermute_topk_reduce(y1, torch.from_numpy(ids).to(DEV), E)
    assert_close(to_f64(out), ref, TOL_BF16, "fused experts")


def _tiled_reference(w, which, w1_layout):
    """Test plumbing: the tile-contiguous layout built with numpy indexing from its definition."""
    E, rows, cols = w.shape
    if which == 1 and w1_layout == 0:
        I = rows // 2
        order = []
        for b in range(rows // 128):
            for r in range(128):
                unit = 64 * b + 16 * (r // 32) + r % 16
                order.append(I + unit if (r // 16) % 2 else unit)
        w = w[:, order, :]
    t = w.reshape(E, rows // 128, 128, cols // 64, 64).permute(0, 1, 3, 2, 4)
    return t.contiguous().reshape(E, rows, cols)


@pytest.mark.parametrize("which,w1_layout,shape", [(1, 0, (3, 256, 192)), (1, 1, (3, 256, 192)),
                                                   (2, 0, (2, 384, 128)), (1, 0, (1, 3072, 4096))])
def test_tile_weights_layout(moe, which, w1_layout, shape):
    """moe_tile_weights writes exactly the documented layout (bit for bit)."""
    w = wl._normal(shape, 1.0, 21, "w", 0, "cpu", torch.bfloat16)
    t = moe.moe_tile_weights(w.to(DEV), which, w1_layout)
    torch.cuda.synchronize()
    ref = _tiled_reference(w, which, w1_layout)
    assert torch.equal(t.cpu().view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("shape", [(5, 8, 64, 512, 128, 0), (96, 4, 8, 512, 256, 1), (700, 2, 6, 256, 128, 0)])
def test_experts_fused_tiled_weights(moe, shape):
    """moe_experts_fused on tile-contiguous W1 and W2 (MOE_W_TILED) gives the same h and y, bit for bit, as on
    the row-major weights (same tiles, same accumulation order)."""
    T, k, E, K, I, w1_layout = shape
    w, x, ids, weights = _routed(T, k, E, K, seed=T + 11 * E)
    ws = wl.scaled(w, I=I, w_std=0.05)
    W1 = wl.expert_weights(ws, "W1", 15).to(torch.bfloat16).to(DEV)
    W2 = wl.expert_weights(ws, "W2", 15).to(torch.bfloat16).to(DEV)
    W1t, W2t = moe.moe_tile_weights(W1, 1, w1_layout), moe.moe_tile_weights(W2, 2)
    res = moe.moe_permute_align(torch.from_numpy(ids).to(DEV), E, moe.MOE_LAYOUT_CONTIGUOUS, 1, x=x.to(DEV))
    R = T * k
    wt = torch.from_numpy(weights).to(DEV).reshape(-1)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    h1, y1 = moe.moe_experts_fused(res["x_out"], res["counts"], res["offsets"], W1, W2, I, res["row_route"], R,
                                   route_weights=wt, w1_layout=w1_layout, err_word=err)
    h2, y2 = moe.moe_experts_fused(res["x_out"], res["counts"], res["offsets"], W1t, W2t, I, res["row_route"], R,
                                   route_weights=wt, w1_layout=moe.MOE_W_TILED, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rr = res["route_row"].view(-1).long()
    assert torch.equal(h1[rr].view(torch.int16), h2[rr].view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_layer_decode_tiled_weights_full_size(moe):
    """The decode layer at full size on tile-contiguous weights equals the layer on row-major weights bit for
    bit; so does a prefill-sized layer (CTA-pair tiles), and single-SM normal tiles refuse tiled weights."""
    w = wl.decode(64)
    x, logits = wl.activations(w, 1, DEV), wl.router_logits(w, 1, DEV)
    W1, W2 = wl.expert_weights(w, "W1", 1, DEV), wl.expert_weights(w, "W2", 1, DEV)
    W1t, W2t = moe.moe_tile_weights(W1, 1), moe.moe_tile_weights(W2, 2)
    layer = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, device=DEV)
    out_a = layer.forward(x, W1, W2, logits=logits).clone()
    out_b = layer.forward(x, W1t, W2t, logits=logits, w1_layout=moe.MOE_W_TILED)
    torch.cuda.synchronize()
    assert layer.device_errors() == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    xb = wl._normal((4096, w.K), 1.0, 3, "x", 0, DEV, torch.bfloat16)
    lb = wl._normal((4096, w.E), 1.0, 3, "l", 0, DEV, torch.float32)
    big = moe.MoELayer(4096, w.K, w.I, w.E, w.top_k, block_m=128, device=DEV)     # CTA-pair tiles
    big_a = big.forward(xb, W1, W2, logits=lb).clone()
    big_b = big.forward(xb, W1t, W2t, logits=lb, w1_layout=moe.MOE_W_TILED)
    torch.cuda.synchronize()
    assert big.device_errors() == 0
    assert torch.equal(big_a.view(torch.int16), big_b.view(torch.int16))
    normal = moe.MoELayer(4096, w.K, w.I, w.E, w.top_k, block_m=128, impl=moe.MOE_IMPL_TCGEN05, device=DEV)
    with pytest.raises(moe.MoEError):
        normal.forward(xb, W1t, W2t, logits=lb, w1_layout=moe.MOE_W_TILED)


def test_layer_decode_fused_experts_full_size(moe):
    """Decode configuration at full size with GEMM 1 + GEMM 2 in one launch: equals the two-launch layer bit for
    bit, sampled tokens against the oracle."""
    w = wl.decode(32)
    x, logits = wl.activations(w, 0, DEV), wl.router_logits(w, 0, DEV)
    W1, W2 = wl.expert_weights(w, "W1", 0, DEV), wl.expert_weights(w, "W2", 0, DEV)
    a = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, fused_experts=False, device=DEV)
    b = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, fused_experts=True, device=DEV)
    out_a = a.forward(x, W1, W2, logits=logits).clone()
    out_b = b.forward(x, W1, W2, logits=logits)
    assert b.launches_per_forward() == a.launches_per_forward() - 1
    assert b.device_errors() == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    ids, weights = oracle.topk_route(logits.cpu().numpy(), w.top_k)
    for t in (0, 31):
        cids, (w1h, w2h, _, _) = compact_experts(ids[t:t + 1], W1, W2)
        ref, _ = oracle.moe_layer(wl.to_numpy(x[t:t + 1]), cids, weights[t:t + 1], w1h, w2h)
        assert_close(to_f64(out_b[t:t + 1]), ref, TOL_BF16, f"fused decode token {t}")


def test_layer_capture_replays_with_new_inputs(moe):
    """MoELayer.capture: the graph re-runs the whole layer on the same tensors; inputs copied in from pinned host
    buffers by the recorded `before` and the output read back by `after` come out as an eager forward's."""
    w = wl.scaled(wl.decode(16), T=16, K=512, I=256, E=16, top_k=4)
    W1, W2 = wl.expert_weights(w, "W1", 1, DEV), wl.expert_weights(w, "W2", 1, DEV)
    hx = torch.empty((w.T, w.K), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((w.T, w.E), dtype=torch.float32).pin_memory()
    dx = torch.empty((w.T, w.K), dtype=torch.bfloat16, device=DEV)
    dl = torch.empty((w.T, w.E), dtype=torch.float32, device=DEV)
    layer = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, device=DEV)
    ho = torch.empty((w.T, w.K), dtype=torch.bfloat16).pin_memory()
    hx.copy_(wl.activations(w, 1))
    hl.copy_(wl.router_logits(w, 1))
    g = layer.capture(dx, W1, W2, logits=dl,
                      before=lambda: (dx.copy_(hx, non_blocking=True), dl.copy_(hl, non_blocking=True)),
                      after=lambda: ho.copy_(layer.out, non_blocking=True))
    eager = moe.MoELayer(w.T, w.K, w.I, w.E, w.top_k, device=DEV)
    for seed in (2, 3):                          # new inputs between replays
        hx.copy_(wl.activations(w, seed))
        hl.copy_(wl.router_logits(w, seed))
        g.replay()
        torch.cuda.synchronize()
        ref = eager.forward(hx.to(DEV), W1, W2, logits=hl.to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(ho.view(torch.int16), ref.cpu().view(torch.int16))
