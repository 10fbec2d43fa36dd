"""Pins for the CPU oracle, each against something other than the oracle itself.

Every test here runs on the CPU.  The pins are: hand-worked values from the
pages (tests/golden/, each file cites its passage), library routines
(scipy softmax, numpy stable argsort, torch float8 / bfloat16 casts, torch
fp64 matmul and silu), closed forms and invariants, and brute force on tiny
inputs.  They are chosen so that a dropped term, a wrong sign or index, or a
transposed operand anywhere in the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from mixture_experts_layer_permute_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _num(tok):
    return float.fromhex(tok) if tok.startswith(("0x", "-0x")) else float(tok)


# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------

def test_mxfp8_scale_codes_golden(oracle_mod):
    for blockmax, code in _read_golden("mxfp8_scale_codes.txt"):
        assert oracle_mod.mxfp8_scale_code(_num(blockmax)) == int(code), blockmax


def test_e4m3_encodings_golden(oracle_mod):
    for value, code in _read_golden("e4m3_encodings.txt"):
        assert oracle_mod.double_to_e4m3(_num(value)) == int(code, 16), value


def test_e4m3_decode_table_matches_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    # every finite code encodes back to itself (except -0 -> 0x80 which is itself)
    for c in range(256):
        if not nan[c]:
            assert oracle_mod.double_to_e4m3(got[c]) == c


def test_e4m3_encode_matches_torch_in_range(oracle_mod):
    g = torch.Generator().manual_seed(3)
    v = (torch.randn(4000, generator=g, dtype=torch.float64) * 100).clamp(-448, 448)
    v = torch.cat([v, torch.randn(1000, generator=g, dtype=torch.float64) * 0.01])
    # torch casts float32 -> float8_e4m3fn with round-to-nearest-even
    v32 = v.to(torch.float32)
    ref = v32.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.double_to_e4m3(float(a)) for a in v32.tolist()], dtype=np.uint8)
    assert np.array_equal(ref, got)


def test_bf16_round_matches_torch(oracle_mod):
    g = torch.Generator().manual_seed(4)
    v = torch.randn(5000, generator=g, dtype=torch.float32) * torch.exp(torch.randn(5000, generator=g) * 10)
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.double_to_bf16(float(a)) for a in v.tolist()], dtype=np.uint16)
    assert np.array_equal(ref, got)
    # decode is exact
    back = np.array([oracle_mod.bf16_to_double(int(h)) for h in got])
    assert np.array_equal(back, v.to(torch.bfloat16).to(torch.float64).numpy())


def test_mxfp8_quantize_properties(oracle_mod):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(16, 256, generator=g) * 0.02
    x[3, 32:64] = 0.0                     # an all-zero block
    x[5, :32] *= 1e-37                    # a block whose code clamps at 0? (it is tiny but above 448*2^-127)
    codes, scales = oracle_mod.mxfp8_quantize(x.numpy())
    assert scales[3, 1] == 0 and np.all(codes[3, 32:64] == 0)
    xd = x.numpy().astype(np.float64)
    for r in range(16):
        for b in range(8):
            blk = xd[r, 32 * b:32 * b + 32]
            m = np.abs(blk).max()
            s = int(scales[r, b])
            if m == 0:
                continue
            # code is the smallest c with m <= 448 * 2^c (frexp-exact check, no logarithms)
            c = s - 127
            assert m <= math.ldexp(448.0, c) and (s == 0 or m > math.ldexp(448.0, c - 1))
            dec = np.array([oracle_mod.e4m3_to_double(int(q)) for q in codes[r, 32 * b:32 * b + 32]])
            # each element is the nearest E4M3 value of x/scale (the library cast decides)
            ref = torch.tensor(blk / math.ldexp(1.0, c), dtype=torch.float32).to(torch.float8_e4m3fn)
            assert np.array_equal(ref.view(torch.uint8).numpy(), codes[r, 32 * b:32 * b + 32])
            # round-trip error within half a unit in the last place of E4M3
            err = np.abs(dec * math.ldexp(1.0, c) - blk)
            ulp = np.array([math.ldexp(1.0, max(math.frexp(abs(a) / math.ldexp(1.0, c))[1] - 1, -6) - 3)
                            if a != 0 else math.ldexp(1.0, -9) for a in blk]) * math.ldexp(1.0, c)
            assert np.all(err <= ulp / 2 + 1e-300)


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------

def _tie_logits(T, E, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.round(torch.randn(T, E, generator=g) * 2) / 2).numpy()   # many exact ties


def test_route_brute_force_selection_with_ties(oracle_mod):
    logits = _tie_logits(64, 16, 0)
    ids, w = oracle_mod.topk_route(logits, 4)
    for t in range(64):
        order = sorted(range(16), key=lambda e: (-logits[t, e], e))
        assert list(ids[t]) == order[:4]
        assert len(set(ids[t])) == 4


def test_route_signed_zeros_and_minus_infinity(oracle_mod):
    """-0 and +0 are equal logits (the lower index wins between them); -inf logits rank last, tie among
    themselves by index, and get weight 0 (exp(-inf) = 0) with or without renormalisation."""
    g = torch.Generator().manual_seed(3)
    logits = (-torch.rand(16, 12, generator=g) - 1.0).numpy().astype(np.float32)
    logits[:, 7:] = -np.inf
    for t in range(16):
        zeros = torch.randperm(7, generator=g)[:3].numpy()
        logits[t, zeros] = [-0.0, 0.0, -0.0] if t % 2 else [0.0, -0.0, 0.0]
    for renorm in (True, False):
        ids, w = oracle_mod.topk_route(logits, 9, renormalize=renorm)
        for t in range(16):
            order = sorted(range(12), key=lambda e: (-float(logits[t, e]), e))   # Python: -0.0 == 0.0
            assert list(ids[t]) == order[:9]
            assert np.all(w[t, 7:] == 0) and np.all(w[t, :7] > 0)
            fin = logits[t, :7].astype(np.float64)
            p = np.exp(fin - fin.max())
            denom = p[ids[t, :7]].sum() if renorm else p.sum()
            assert np.allclose(w[t, :7], p[ids[t, :7]] / denom, rtol=2e-7, atol=0)


def test_route_weights_renormalised_softmax(oracle_mod):
    g = torch.Generator().manual_seed(1)
    logits = torch.randn(32, 128, generator=g).numpy()
    ids, w = oracle_mod.topk_route(logits, 8, renormalize=True)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-6)
    # softmax over all experts, take the chosen, renormalise (library softmax)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    chosen = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    ref = chosen / chosen.sum(1, keepdims=True)
    assert np.allclose(w, ref, rtol=2e-7, atol=0)
    # selection agrees with torch.topk where logits are distinct
    tv, ti = torch.topk(torch.from_numpy(logits), 8, dim=1)
    assert np.array_equal(ti.numpy(), ids)


def test_route_no_renorm_and_topk_equals_E(oracle_mod):
    g = torch.Generator().manual_seed(2)
    logits = torch.randn(8, 16, generator=g).numpy()
    ids, w = oracle_mod.topk_route(logits, 3, renormalize=False)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(p, ids.astype(np.int64), axis=1), rtol=2e-7)
    ids_all, w_all = oracle_mod.topk_route(logits, 16, renormalize=True)
    assert np.allclose(np.take_along_axis(p, ids_all.astype(np.int64), axis=1), w_all, rtol=2e-7)


# ----------------------------------------------------------------------------
# permute / align
# ----------------------------------------------------------------------------

def _random_ids(T, k, E, seed, pad_frac=0.0):
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    if pad_frac:
        mask = torch.rand(T, k, generator=g) < pad_frac
        ids[mask] = -1
    return ids.numpy()


@pytest.mark.parametrize("block_m", [1, 4, 128])
def test_permute_equals_stable_argsort(oracle_mod, block_m):
    T, k, E = 50, 3, 7
    ids = _random_ids(T, k, E, 10 + block_m, pad_frac=0.2)
    res = oracle_mod.permute_contiguous(ids, E, block_m)
    flat = ids.reshape(-1)
    valid = flat >= 0
    assert res["err"] == 0
    assert res["counts"].sum() == valid.sum()
    assert np.array_equal(res["counts"], np.bincount(flat[valid], minlength=E))
    order = np.argsort(np.where(valid, flat, E), kind="stable")[: valid.sum()]   # library stable sort
    pad = lambda c: (c + block_m - 1) // block_m * block_m
    assert np.array_equal(res["offsets"], np.concatenate([[0], np.cumsum([pad(c) for c in res["counts"]])]))
    pos = 0
    for e in range(E):
        seg = res["sorted_route"][res["offsets"][e]:res["offsets"][e + 1]]
        c = res["counts"][e]
        assert np.array_equal(seg[:c], order[pos:pos + c])
        assert np.all(seg[c:] == -1)
        pos += c
    rr = res["route_row"].reshape(-1)
    assert np.all(rr[~valid] == -1)
    assert np.array_equal(res["sorted_route"][rr[valid]], np.nonzero(valid)[0])


def test_permute_flags_out_of_range_ids(oracle_mod):
    ids = np.array([[0, 5], [-1, 1], [-2, 2]], np.int32)
    res = oracle_mod.permute_contiguous(ids, 3, 1)
    assert res["err"] == oracle_mod.ERR_ID_RANGE
    assert list(res["counts"]) == [1, 1, 1]
    assert res["route_row"][0, 1] == -1 and res["route_row"][2, 0] == -1


def test_permute_then_unpermute_is_identity(oracle_mod):
    """Identity expert, top_k = 1, weight 1: the layer must return x bit-exactly."""
    T, K, E = 37, 16, 5
    g = torch.Generator().manual_seed(11)
    x = torch.randn(T, K, generator=g).to(torch.bfloat16)
    xn = wl.to_numpy(x)
    ids = torch.randint(0, E, (T, 1), generator=g, dtype=torch.int32).numpy()
    res = oracle_mod.permute_contiguous(ids, E, 8)
    x_perm = np.zeros((res["offsets"][E], K), np.uint16)
    valid = res["sorted_route"] >= 0
    x_perm[valid] = xn[res["sorted_route"][valid] // 1]          # gather (top_k = 1)
    y_slots = x_perm[res["route_row"].reshape(-1)]                  # unpermute
    out = oracle_mod.topk_reduce(y_slots, ids, np.ones((T, 1), np.float32), out=oracle_mod.BF16)
    assert np.array_equal(out, xn)


def test_permute_batched_ranks_and_capacity(oracle_mod):
    ids = np.array([[0, 1], [1, 0], [0, 2], [0, -1]], np.int32)
    res = oracle_mod.permute_batched(ids, 3, 2)
    # routes r = 2t + j go to experts 0,1,1,0,0,2,0,-1: expert 0 has 4 routes, capacity 2
    assert res["err"] == oracle_mod.ERR_CAPACITY
    assert list(res["expert_num_tokens"]) == [2, 2, 1]
    assert list(res["row_route"][0]) == [0, 3]           # routes in increasing index
    assert list(res["row_route"][1]) == [1, 2]
    assert list(res["row_route"][2]) == [5, -1]
    assert res["route_row"][2, 0] == -1                  # route 4 dropped by capacity
    assert res["route_row"][3, 0] == -1                  # dropped by capacity
    assert res["route_row"][3, 1] == -1                  # padding


# ----------------------------------------------------------------------------
# expert FFN and the layer
# ----------------------------------------------------------------------------

def _tiny_inputs(seed=0, T=12, K=64, I=32, E=6, k=3, dtype=torch.float32, x_std=1.0, w_std=0.2):
    """Small layer inputs; std large enough that silu is far from linear (g ~ N(0, 1.6^2))."""
    w = wl.scaled(wl.tiny(), T=T, K=K, I=I, E=E, top_k=k, x_std=x_std, w_std=w_std)
    x = wl.activations(w, seed).to(dtype)
    W1 = wl.expert_weights(w, "W1", seed).to(dtype)
    W2 = wl.expert_weights(w, "W2", seed).to(dtype)
    logits = wl.router_logits(w, seed)
    return w, x, W1, W2, logits


def _dense_reference(x, ids, weights, W1g, W1u, W2):
    """Dense all-experts computation masked by top-k (torch fp64, a different loop nest)."""
    x = x.double()
    out = torch.zeros(x.shape, dtype=torch.float64)
    for e in range(W2.shape[0]):
        h = F.silu(x @ W1g[e].double().T) * (x @ W1u[e].double().T)
        y = h @ W2[e].double().T
        m = ((torch.from_numpy(ids) == e).double() * torch.from_numpy(weights).double()).sum(1)
        out += m[:, None] * y
    return out.numpy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_layer_equals_dense_masked_reference(oracle_mod, dtype):
    w, x, W1, W2, logits = _tiny_inputs(dtype=dtype)
    ids, weights = oracle_mod.topk_route(logits.numpy(), w.top_k)
    out, err = oracle_mod.moe_layer(wl.to_numpy(x), ids, weights, wl.to_numpy(W1), wl.to_numpy(W2))
    assert err == 0
    ref = _dense_reference(x.float(), ids, weights, W1[:, :w.I].float(), W1[:, w.I:].float(), W2.float())
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-15)
    # a swapped gate/up would not match
    bad = _dense_reference(x.float(), ids, weights, W1[:, w.I:].float(), W1[:, :w.I].float(), W2.float())
    assert np.linalg.norm(out - bad) > 0.1 * np.linalg.norm(out)


def test_topk1_unit_weight_is_single_expert_ffn(oracle_mod):
    w, x, W1, W2, _ = _tiny_inputs(seed=3)
    e = 4
    ids = np.full((w.T, 1), e, np.int32)
    out, _ = oracle_mod.moe_layer(wl.to_numpy(x), ids, np.ones((w.T, 1), np.float32), wl.to_numpy(W1),
                                  wl.to_numpy(W2))
    xd = x.double()
    ref = (F.silu(xd @ W1[e, :w.I].double().T) * (xd @ W1[e, w.I:].double().T)) @ W2[e].double().T
    assert np.allclose(out, ref.numpy(), rtol=1e-10, atol=1e-15)


def test_interleave16_layout_matches_standard_layout(oracle_mod):
    """W1 in the interleave-16 layout (rows built from the golden table) gives the same layer bit for bit."""
    w, x, W1, W2, logits = _tiny_inputs(seed=4, I=32)
    table = _read_golden("interleave16_rows.txt")
    W1i = torch.empty_like(W1)
    for first, last, half, unit in table:
        first, last, half, unit = int(first), int(last), int(half), int(unit)
        src = half * w.I + unit
        W1i[:, first:last + 1] = W1[:, src:src + (last - first + 1)]
    ids, weights = oracle_mod.topk_route(logits.numpy(), w.top_k)
    a, _ = oracle_mod.moe_layer(wl.to_numpy(x), ids, weights, wl.to_numpy(W1), wl.to_numpy(W2), w1_layout=0)
    b, _ = oracle_mod.moe_layer(wl.to_numpy(x), ids, weights, wl.to_numpy(W1i), wl.to_numpy(W2), w1_layout=1)
    assert np.array_equal(a, b)
    h = oracle_mod.expert_gate_up(wl.to_numpy(x), np.zeros(w.T, np.int32), wl.to_numpy(W1i), w1_layout=1)
    xd = x.double()
    ref = F.silu(xd @ W1[0, :w.I].double().T) * (xd @ W1[0, w.I:].double().T)
    assert np.allclose(h, ref.numpy(), rtol=1e-12)


def _torch_dequant(codes, scales):
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
    s = torch.pow(2.0, torch.from_numpy(scales.astype(np.float64)) - 127.0)
    return v * s.repeat_interleave(32, dim=-1)


def test_mxfp8_weights_layer_equals_dequantised_reference(oracle_mod):
    w, x, W1, W2, logits = _tiny_inputs(seed=5, dtype=torch.float32)
    c1, s1 = oracle_mod.mxfp8_quantize(W1.numpy())
    c2, s2 = oracle_mod.mxfp8_quantize(W2.numpy())
    ids, weights = oracle_mod.topk_route(logits.numpy(), w.top_k)
    out, _ = oracle_mod.moe_layer(wl.to_numpy(x), ids, weights, c1, c2, w1_scale=s1, w2_scale=s2)
    D1, D2 = _torch_dequant(c1, s1), _torch_dequant(c2, s2)
    ref = _dense_reference(x, ids, weights, D1[:, :w.I], D1[:, w.I:], D2)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-15)
    # quantisation really happened: weights moved by up to a few percent
    assert not np.allclose(D1.numpy(), W1.double().numpy(), rtol=1e-3)


def test_quantised_intermediate(oracle_mod):
    w, x, W1, W2, logits = _tiny_inputs(seed=6, I=64)
    ids, weights = oracle_mod.topk_route(logits.numpy(), w.top_k)
    out, _ = oracle_mod.moe_layer(wl.to_numpy(x), ids, weights, wl.to_numpy(W1), wl.to_numpy(W2), quant_h=True)
    # reference: h in fp32, scale per 32 from the exact rule, element cast by torch, dequantised, then W2
    xd = x.double()
    ref = torch.zeros(w.T, w.K, dtype=torch.float64)
    for t in range(w.T):
        for j in range(w.top_k):
            e = int(ids[t, j])
            h = (F.silu(xd[t] @ W1[e, :w.I].double().T) * (xd[t] @ W1[e, w.I:].double().T)).float()
            hq = torch.empty(w.I, dtype=torch.float64)
            for b in range(w.I // 32):
                blk = h[32 * b:32 * b + 32]
                m = float(blk.abs().max())
                c = math.frexp(m / 448.0)[1]
                while m > math.ldexp(448.0, c):
                    c += 1
                while m <= math.ldexp(448.0, c - 1):
                    c -= 1
                sc = math.ldexp(1.0, c)
                hq[32 * b:32 * b + 32] = (blk.double() / sc).float().to(torch.float8_e4m3fn).double() * sc
            ref[t] += float(weights[t, j]) * (hq @ W2[e].double().T)
    assert np.allclose(out, ref.numpy(), rtol=1e-9, atol=1e-15)


def _py_mx_roundtrip(v):
    """Block-32 MXFP8 quantise-dequantise of a 1-D tensor: the exact scale rule written out, the element cast
    done by torch's float8_e4m3fn."""
    out = torch.empty(v.numel(), dtype=torch.float64)
    for b in range(v.numel() // 32):
        blk = v[32 * b:32 * b + 32].double()
        m = float(blk.abs().max())
        if m == 0.0:
            out[32 * b:32 * b + 32] = 0.0
            continue
        c = math.frexp(m / 448.0)[1]
        while m > math.ldexp(448.0, c):
            c += 1
        while m <= math.ldexp(448.0, c - 1):
            c -= 1
        sc = math.ldexp(1.0, c)
        out[32 * b:32 * b + 32] = (blk / sc).to(torch.float8_e4m3fn).double() * sc
    return out


def test_mxfp8_dequantize_matches_torch(oracle_mod):
    g = torch.Generator().manual_seed(21)
    codes = torch.randint(0, 256, (7, 96), generator=g, dtype=torch.int32)
    codes[(codes & 0x7F) == 0x7F] = 0x12                 # no NaN codes
    codes = codes.to(torch.uint8).numpy()
    scales = torch.randint(100, 160, (7, 3), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    got = oracle_mod.mxfp8_dequantize(codes, scales)
    assert np.array_equal(got, _torch_dequant(codes, scales).numpy())


@pytest.mark.parametrize("w1_layout", [0, 1])
def test_expert_gemms_decode_every_scale_code(oracle_mod, w1_layout):
    """The oracle's W1 and W2 products on E4M3 codes with E8M0 scale codes drawn over the whole range 0..254 (the
    MXFP8 block format, "Cake MegaMoE EP16" FlashInfer PR 5148 analysis, section 2: value = code x 2^(scale-127)),
    against a dense fp64 product of the weights decoded by torch's float8_e4m3fn and ldexp: every block's factor,
    from 2^-127 to 2^127, reaches the sums the GPU tests compare with."""
    g = torch.Generator().manual_seed(23)
    E, K, I, n = 2, 96, 32, 5
    c1 = torch.randint(0, 256, (E, 2 * I, K), generator=g, dtype=torch.int32)
    c1[(c1 & 0x7F) == 0x7F] = 0x31                         # no NaN codes
    c1 = c1.to(torch.uint8).numpy()
    s1 = torch.randint(0, 255, (E, 2 * I, K // 32), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    c2 = torch.randint(0, 256, (E, K, I), generator=g, dtype=torch.int32)
    c2[(c2 & 0x7F) == 0x7F] = 0x2C
    c2 = c2.to(torch.uint8).numpy()
    s2 = torch.randint(0, 255, (E, K, I // 32), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    assert s1.min() < 7 and s1.max() > 240                  # both ends of the factor range
    x = torch.randn((n, K), generator=g, dtype=torch.float64)
    ids = np.array([0, 1, 1, 0, 1], np.int32)
    h = oracle_mod.expert_gate_up(x.numpy(), ids, c1, w1_scale=s1, w1_layout=w1_layout)
    D1 = _torch_dequant(c1, s1)
    units = np.arange(2 * I)
    gate_rows = units[:I] if w1_layout == 0 else np.array([32 * (u // 16) + u % 16 for u in range(I)])
    up_rows = units[I:] if w1_layout == 0 else gate_rows + 16
    for r in range(n):
        e = int(ids[r])
        ref = F.silu(D1[e, gate_rows] @ x[r]) * (D1[e, up_rows] @ x[r])
        assert np.allclose(h[r], ref.numpy(), rtol=1e-12, atol=0), r
    hin = torch.randn((n, I), generator=g, dtype=torch.float64)
    y = oracle_mod.expert_down(hin.numpy(), ids, c2, w2_scale=s2)
    D2 = _torch_dequant(c2, s2)
    for r in range(n):
        ref = D2[int(ids[r])] @ hin[r]
        assert np.allclose(y[r], ref.numpy(), rtol=1e-12, atol=0), r


def test_quantised_activations_and_bf16_intermediate(oracle_mod):
    """quant_x: each x row MXFP8 round-tripped before W1; quant_h="bf16": h rounded to bf16, then round-tripped
    before W2 -- against torch fp64 matmuls with the round trips written out (torch float8 casts)."""
    w, x, W1, W2, logits = _tiny_inputs(seed=8, I=64, dtype=torch.bfloat16)
    c1, s1 = oracle_mod.mxfp8_quantize(W1.float().numpy())
    c2, s2 = oracle_mod.mxfp8_quantize(W2.float().numpy())
    ids, weights = oracle_mod.topk_route(logits.numpy(), w.top_k)
    out, _ = oracle_mod.moe_layer(wl.to_numpy(x), ids, weights, c1, c2, w1_scale=s1, w2_scale=s2, quant_x=True,
                                  quant_h="bf16")
    D1, D2 = _torch_dequant(c1, s1), _torch_dequant(c2, s2)
    ref = torch.zeros(w.T, w.K, dtype=torch.float64)
    for t in range(w.T):
        xq = _py_mx_roundtrip(x[t].double())
        for j in range(w.top_k):
            e = int(ids[t, j])
            h = F.silu(xq @ D1[e, :w.I].T) * (xq @ D1[e, w.I:].T)
            hq = _py_mx_roundtrip(h.to(torch.bfloat16).double())
            ref[t] += float(weights[t, j]) * (hq @ D2[e].T)
    assert np.allclose(out, ref.numpy(), rtol=1e-9, atol=1e-15)
    plain, _ = oracle_mod.moe_layer(wl.to_numpy(x), ids, weights, c1, c2, w1_scale=s1, w2_scale=s2)
    assert not np.allclose(out, plain, rtol=1e-3)          # the round trips changed the result


def test_padding_slots_contribute_nothing(oracle_mod):
    w, x, W1, W2, logits = _tiny_inputs(seed=7)
    ids, weights = oracle_mod.topk_route(logits.numpy(), w.top_k)
    ids_p, w_p = ids.copy(), weights.copy()
    ids_p[::2, 1] = -1
    w_p[::2, 1] = 0.0
    ids_p[5, :] = -1               # a token made only of padding
    w_p[5, :] = 0.0
    a, _ = oracle_mod.moe_layer(wl.to_numpy(x), ids_p, w_p, wl.to_numpy(W1), wl.to_numpy(W2))
    # the same layer with the padding slots removed: drop slot 1 (weight 0 anyway) on even tokens
    keep = np.zeros_like(a)
    for t in range(w.T):
        for j in range(w.top_k):
            if ids_p[t, j] >= 0:
                one, _ = oracle_mod.moe_layer(wl.to_numpy(x)[t:t + 1], ids_p[t:t + 1, j:j + 1],
                                              w_p[t:t + 1, j:j + 1], wl.to_numpy(W1), wl.to_numpy(W2))
                keep[t] += one[0]
    assert np.allclose(a, keep, rtol=1e-12, atol=0)
    assert np.all(a[5] == 0.0) and not np.any(np.signbit(a[5]))   # +0.0, never -0.0
    outb, _ = oracle_mod.moe_layer(wl.to_numpy(x), ids_p, w_p, wl.to_numpy(W1), wl.to_numpy(W2),
                                   out=oracle_mod.BF16)
    assert np.all(outb[5] == 0)


def test_topk_reduce_matches_einsum(oracle_mod):
    g = torch.Generator().manual_seed(8)
    T, k, K = 9, 4, 24
    y = torch.randn(T, k, K, generator=g).to(torch.bfloat16)
    ids = _random_ids(T, k, 6, 8, pad_frac=0.3)
    w = torch.rand(T, k, generator=g).numpy()
    out = oracle_mod.topk_reduce(wl.to_numpy(y), ids, w)
    mask = (ids >= 0).astype(np.float64)
    ref = np.einsum("tj,tjk->tk", mask * w.astype(np.float64), y.double().numpy())
    assert np.allclose(out, ref, rtol=1e-13, atol=1e-15)
    out_nw = oracle_mod.topk_reduce(wl.to_numpy(y), ids, None)
    assert np.allclose(out_nw, np.einsum("tj,tjk->tk", mask, y.double().numpy()), rtol=1e-13, atol=1e-15)


def test_batched_layer_naive_weight(oracle_mod):
    w = wl.scaled(wl.batched(), E=4, max_tokens=8, K=64, I=32)
    xb, counts, rw = wl.batched_inputs(w, seed=1)
    W1 = wl.expert_weights(w, "W1", 1)
    W2 = wl.expert_weights(w, "W2", 1)
    sentinel = np.full((w.E, w.max_tokens, w.K), 12345.0)
    out, err = oracle_mod.moe_layer_batched(wl.to_numpy(xb), counts.numpy(), rw.numpy(), wl.to_numpy(W1),
                                            wl.to_numpy(W2), out_init=sentinel)
    assert err == 0
    for e in range(w.E):
        c = int(counts[e])
        xd = xb[e, :c].double()
        ref = (F.silu(xd @ W1[e, :w.I].double().T) * (xd @ W1[e, w.I:].double().T)) @ W2[e].double().T
        ref = ref * rw[e, :c].double()[:, None]
        assert np.allclose(out[e, :c], ref.numpy(), rtol=1e-10, atol=1e-15)
        assert np.all(out[e, c:] == 12345.0)            # rows beyond the count untouched
        assert np.all(np.isfinite(out[e, :c]))           # garbage rows never read


def _batched_gather(xn, row_route, k):
    """(E, max_tokens, K) rows of x for each batched row (zeros where no route)."""
    E, maxT = row_route.shape
    xb = np.zeros((E, maxT, xn.shape[1]), xn.dtype)
    valid = row_route >= 0
    xb[valid] = xn[row_route[valid] // k]
    return xb


def test_batched_reduce_path_equals_contiguous_layer(oracle_mod):
    """Batched permute -> per-(expert, row) FFN without weights -> token-order reduce through route_row equals
    the contiguous layer, which loops over (token, slot) instead."""
    w, x, W1, W2, logits = _tiny_inputs(seed=4, T=14, K=64, I=32, E=5, k=3)
    ids, wts = oracle_mod.topk_route(logits.numpy(), w.top_k)
    xn = x.numpy()
    res = oracle_mod.permute_batched(ids, w.E, w.T * w.top_k)      # capacity never reached
    assert res["err"] == 0
    xb = _batched_gather(xn, res["row_route"], w.top_k)
    yb, err = oracle_mod.moe_layer_batched(xb, res["expert_num_tokens"], None, W1.numpy(), W2.numpy())
    assert err == 0
    out, err = oracle_mod.batched_topk_reduce(yb, res["route_row"], wts)
    assert err == 0
    ref, _ = oracle_mod.moe_layer(xn, ids, wts, W1.numpy(), W2.numpy())
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-15)
    assert np.abs(ref).max() > 0.1


def test_batched_reduce_identity_and_capacity(oracle_mod):
    """Identity expert, top_k = 1, weight 1: x comes back bit-exactly; routes dropped for capacity add
    nothing, a token left with no route gives +0.0, rows outside the buffer are reported."""
    T, K, E, maxT = 29, 16, 4, 6
    g = torch.Generator().manual_seed(5)
    x = torch.randn(T, K, generator=g).to(torch.bfloat16)
    xn = wl.to_numpy(x)
    ids = torch.randint(0, E, (T, 1), generator=g, dtype=torch.int32).numpy()
    big = oracle_mod.permute_batched(ids, E, T)
    xb = _batched_gather(xn, big["row_route"], 1)
    out, err = oracle_mod.batched_topk_reduce(xb, big["route_row"], np.ones((T, 1), np.float32),
                                              out=oracle_mod.BF16)
    assert err == 0 and np.array_equal(out, xn)
    small = oracle_mod.permute_batched(ids, E, maxT)             # some experts overflow
    assert small["err"] == oracle_mod.ERR_CAPACITY
    xb = _batched_gather(xn, small["row_route"], 1)
    out, err = oracle_mod.batched_topk_reduce(xb, small["route_row"], None, out=oracle_mod.F32)
    dropped = small["route_row"][:, 0] < 0
    assert dropped.any() and (~dropped).any()
    kept_ref = xn[~dropped].astype(np.uint32) << 16
    assert np.array_equal(out[~dropped].view(np.uint32), kept_ref)
    assert np.all(out[dropped].view(np.uint32) == 0)              # +0.0, not -0.0
    bad = small["route_row"].copy()
    bad[0, 0] = E * maxT                                          # one past the buffer
    _, err = oracle_mod.batched_topk_reduce(xb, bad, None)
    assert err == oracle_mod.ERR_ID_RANGE


def test_affine_routing_golden_and_balance():
    rows = _read_golden("affine_routing.txt")
    ids, wts = wl.affine_routing(wl.mxfp8())
    for row in rows:
        t = int(row[0])
        assert [int(v) for v in row[1:]] == ids[t].tolist()
    counts = torch.bincount(ids.reshape(-1).long(), minlength=512)
    assert torch.all(counts == 8)                         # every expert gets the same load
    assert torch.all(wts == 0.125)
    assert all(len(set(r)) == 8 for r in ids.tolist())    # no duplicate expert within a token
