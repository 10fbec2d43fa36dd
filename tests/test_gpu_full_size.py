"""Every configuration at full size, exactly as bench.py times it, against the CPU oracle.

Each workload is built by bench.py's own ``Instance`` (the same seeded draws, the same
``MoELayer`` plan and weight layout: for the decode passes tile-contiguous weights and
GEMM 1 + GEMM 2 in one launch), run once, and its output compared with the oracle
element by element at the stated tolerance (bf16 / MXFP8: 2e-2, fp32: 1e-5, both on
rel-RMS and on max-abs relative to max |ref|), token by token.  The whole computation
being checked is the decomposition of "Fused MoE Modular Kernel", apply(): permute,
W1 + act-and-mul, W2, unpermute with the top-k weight-and-reduce.

What is compared:

* decode sweep T = 1, 8, 32, 64 (K=4096, I=1536, E=128, top_k=8): all 105 tokens (840 routes);
* prefill with skewed routing (T=4096, block_m=128, normal 128-row tiles): for every touched
  expert the token of the first route of its last 128-row tile and the token of its last route
  (so every ragged last tile, the coldest experts and expert 0's last tile), topped up with the
  first tokens to at least 64;
* MXFP8 weights (E=512, K=7168, I=2048, interleave-16 W1, affine routing): tokens 0..63, whose
  512 routes reach every expert once (each expert's 8 routes share one tile);
* the same with activations quantised on the fly (block-scaled MXFP8 x MXFP8 GEMMs);
* batched (E=32, max_tokens=256, K=6144, I=4096, garbage rows): every expert's first and last
  valid row, rows past each count untouched;
* batched_tokens (T=1024, top_k=4): each expert's first and last kept route;
* tiny fp32: all 16 tokens at 1e-5.

The oracle runs one plain call per token on a thread pool over the host cores (its C calls
release the GIL); the routing ids and the permutation are also compared bit for bit.
"""
import gc

import numpy as np
import pytest
import torch

import bench
import oracle
from mixture_experts_layer_permute_gb300 import workloads as wl

from helpers import TOL_BF16, TOL_F32, assert_close, compact_experts, oracle_map, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _oracle_built():
    oracle.build()


def _release():
    """Returns the device memory of the workload just checked (the next one is built from scratch)."""
    gc.collect()
    torch.cuda.empty_cache()


def _check_tokens(out_host, refs, tokens, tol, what):
    for t, ref in zip(tokens, refs):
        assert_close(out_host[t:t + 1], ref, tol, f"{what} token {t}")


def _routing_exact(inst, w):
    """Routing ids (oracle.topk_route on the same logits) and the contiguous permutation, bit for bit."""
    ids, weights = oracle.topk_route(inst.logits.cpu().numpy(), w.top_k)
    L = inst.layer
    assert np.array_equal(L.ids.cpu().numpy(), ids)
    perm = oracle.permute_contiguous(ids, w.E, w.block_m)
    assert np.array_equal(L.counts.cpu().numpy(), perm["counts"])
    assert np.array_equal(L.offsets.cpu().numpy(), perm["offsets"])
    assert np.array_equal(L.row_route[:perm["offsets"][-1]].cpu().numpy(), perm["sorted_route"])
    assert np.array_equal(L.route_row.cpu().numpy().reshape(-1), perm["route_row"].reshape(-1))
    return ids, weights


def test_decode_sweep_every_token(moe):
    """The benchmarked decode passes, every token: fused experts launch on tile-contiguous weights."""
    w1h = w2h = None
    for T in (1, 8, 32, 64):
        w = wl.decode(T)
        inst = bench.Instance(w, 0, DEV)
        assert inst.fused() and inst.w1_layout == moe.MOE_W_TILED     # the plan bench.py times
        out = inst.forward()
        torch.cuda.synchronize()
        assert inst.layer.device_errors() == 0
        ids, weights = _routing_exact(inst, w)
        if w1h is None:     # the same draw for every pass (seed 0, same sizes)
            w1h, w2h = wl.to_numpy(inst.W1), wl.to_numpy(inst.W2)
        x = wl.to_numpy(inst.x)
        got = to_f64(out)
        refs = oracle_map(lambda t: oracle.moe_layer(x[t:t + 1], ids[t:t + 1], weights[t:t + 1], w1h, w2h)[0],
                          range(T))
        _check_tokens(got, refs, range(T), TOL_BF16, f"decode T={T}")
        del inst, out
        _release()


@pytest.mark.parametrize("seed", [1, 2])
def test_decode_t64_other_seeds(moe, seed):
    """The T=64 decode pass (the largest of the sweep) drawn from seeds 1 and 2: every token."""
    w = wl.decode(64)
    inst = bench.Instance(w, seed, DEV)
    assert inst.fused() and inst.w1_layout == moe.MOE_W_TILED
    out = inst.forward()
    torch.cuda.synchronize()
    assert inst.layer.device_errors() == 0
    ids, weights = _routing_exact(inst, w)
    x, w1h, w2h = wl.to_numpy(inst.x), wl.to_numpy(inst.W1), wl.to_numpy(inst.W2)
    refs = oracle_map(lambda t: oracle.moe_layer(x[t:t + 1], ids[t:t + 1], weights[t:t + 1], w1h, w2h)[0],
                      range(w.T))
    _check_tokens(to_f64(out), refs, range(w.T), TOL_BF16, f"decode T=64 seed {seed}")
    del inst, out
    _release()


def _prefill_tokens(ids, E, block_m, k, at_least=64):
    routes = ids.reshape(-1)
    tokens = set()
    for e in range(E):
        r = np.nonzero(routes == e)[0]            # expert e's rows, in row order (stable placement)
        if r.size == 0:
            continue
        last_tile = ((r.size - 1) // block_m) * block_m
        tokens.add(int(r[last_tile]) // k)
        tokens.add(int(r[-1]) // k)
    t = 0
    while len(tokens) < at_least:
        tokens.add(t)
        t += 1
    return sorted(tokens)


@pytest.mark.parametrize("seed", [0, 1])
def test_prefill_tail_tiles(moe, seed):
    """Skewed prefill: tokens covering every touched expert's ragged last 128-row tile and its coldest experts."""
    w = wl.prefill()
    inst = bench.Instance(w, seed, DEV)
    out = inst.forward()
    torch.cuda.synchronize()
    assert inst.layer.device_errors() == 0
    ids, weights = _routing_exact(inst, w)
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    tokens = _prefill_tokens(ids, w.E, w.block_m, w.top_k)
    assert len(tokens) >= 64
    touched = [e for e in range(w.E) if counts[e] > 0]
    cold = sorted(touched, key=lambda e: counts[e])[:8]
    assert all(any(e in ids[t] for t in tokens) for e in cold)             # the coldest experts are hit
    assert 0 in ids[tokens]                                                 # and the hottest one
    x = wl.to_numpy(inst.x)
    w1h, w2h = wl.to_numpy(inst.W1), wl.to_numpy(inst.W2)
    got = to_f64(out)
    refs = oracle_map(lambda t: oracle.moe_layer(x[t:t + 1], ids[t:t + 1], weights[t:t + 1], w1h, w2h)[0], tokens)
    _check_tokens(got, refs, tokens, TOL_BF16, "prefill")
    del inst, out
    _release()


@pytest.mark.parametrize("name", ["mxfp8", "mxfp8_act"])
def test_mxfp8_every_expert(moe, name):
    """MXFP8 weights (and, for mxfp8_act, activations quantised on the fly): tokens 0..63 reach all 512 experts."""
    w = wl.mxfp8() if name == "mxfp8" else wl.mxfp8_act()
    inst = bench.Instance(w, 0, DEV)
    out = inst.forward()
    torch.cuda.synchronize()
    assert inst.layer.device_errors() == 0
    ids, wts = inst.ids.cpu().numpy(), inst.tw.cpu().numpy()
    assert len({int(e) for e in ids[:64].reshape(-1)}) == w.E
    x = wl.to_numpy(inst.x)
    got = to_f64(out)
    quant = dict(quant_x=True, quant_h="bf16") if w.act_quant else {}
    for g in range(8):                           # 8 tokens (64 experts) at a time: bounded host memory
        tokens = list(range(8 * g, 8 * g + 8))
        cids, (w1h, w2h, s1h, s2h) = compact_experts(ids[tokens], inst.W1, inst.W2, inst.s1, inst.s2)
        refs = oracle_map(lambda i: oracle.moe_layer(x[tokens[i]:tokens[i] + 1], cids[i:i + 1],
                                                     wts[tokens[i]:tokens[i] + 1], w1h, w2h, w1_scale=s1h,
                                                     w2_scale=s2h, w1_layout=w.w1_layout, **quant)[0],
                          range(len(tokens)))
        _check_tokens(got, refs, tokens, TOL_BF16, name)
        del w1h, w2h, s1h, s2h
    del inst, out
    _release()


def test_batched_first_and_last_rows(moe):
    """Batched layout: every expert's first and last valid row; garbage rows ignored, rows past the count
    untouched."""
    w = wl.batched("nan")
    inst = bench.Instance(w, 0, DEV)
    inst.layer.out.fill_(3.0)
    out = inst.forward()
    torch.cuda.synchronize()
    cnt = inst.counts.cpu().numpy()
    xb = wl.to_numpy(inst.xb)
    rw = inst.rw.cpu().numpy()
    w1h, w2h = wl.to_numpy(inst.W1), wl.to_numpy(inst.W2)
    experts = [e for e in range(w.E) if cnt[e] > 0]

    def ref_rows(e):
        rows = sorted({0, int(cnt[e]) - 1})
        r, _ = oracle.moe_layer_batched(xb[e:e + 1, rows], np.array([len(rows)], np.int32), rw[e:e + 1, rows],
                                        w1h[e:e + 1], w2h[e:e + 1])
        return rows, r[0]
    results = oracle_map(ref_rows, experts)
    for e, (rows, ref) in zip(experts, results):
        assert_close(to_f64(out[e, rows]), ref, TOL_BF16, f"batched expert {e} rows {rows}")
    for e in range(w.E):
        if cnt[e] < w.max_tokens:
            assert torch.all(out[e, int(cnt[e]):] == 3.0)
    del inst, out
    _release()


def test_batched_tokens_first_and_last_routes(moe):
    """Batched layout fed with tokens: each expert's first and last kept route, permutation bit-exact."""
    w = wl.batched_tokens()
    inst = bench.Instance(w, 0, DEV)
    out = inst.forward()
    torch.cuda.synchronize()
    L = inst.layer
    ids, weights = oracle.topk_route(inst.logits.cpu().numpy(), w.top_k)
    assert np.array_equal(L.ids.cpu().numpy(), ids)
    perm = oracle.permute_batched(ids, w.E, w.max_tokens)
    assert np.array_equal(L.counts.cpu().numpy(), perm["expert_num_tokens"])
    assert np.array_equal(L.route_row.cpu().numpy(), perm["route_row"])
    assert perm["err"] == 0 and L.device_errors() == 0          # no route dropped for capacity
    routes = ids.reshape(-1)
    tokens = set()
    for e in range(w.E):
        r = np.nonzero(routes == e)[0]
        if r.size:
            tokens.update((int(r[0]) // w.top_k, int(r[-1]) // w.top_k))
    tokens = sorted(tokens)
    x = wl.to_numpy(inst.x)
    w1h, w2h = wl.to_numpy(inst.W1), wl.to_numpy(inst.W2)
    refs = oracle_map(lambda t: oracle.moe_layer(x[t:t + 1], ids[t:t + 1], weights[t:t + 1], w1h, w2h)[0], tokens)
    _check_tokens(to_f64(out), refs, tokens, TOL_BF16, "batched_tokens")
    del inst, out
    _release()


def test_tiny_fp32_every_token(moe):
    """The fp32 configuration (T=16, K=128, I=256, E=8, top_k=2), every token at 1e-5."""
    w = wl.tiny()
    inst = bench.Instance(w, 0, DEV)
    out = inst.forward()
    torch.cuda.synchronize()
    ids, weights = _routing_exact(inst, w)
    ref, err = oracle.moe_layer(wl.to_numpy(inst.x), ids, weights, wl.to_numpy(inst.W1), wl.to_numpy(inst.W2))
    assert err == 0
    _check_tokens(to_f64(out), [ref[t:t + 1] for t in range(w.T)], range(w.T), TOL_F32, "tiny")
