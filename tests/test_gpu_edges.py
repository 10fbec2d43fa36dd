"""GPU edge cases of the whole layer against the oracle: an empty batch, tokens made only of padding, a single
expert, top_k = E, the smallest contraction the tensor-core tiles take (with the fallback to the CUDA-core tiles
where a tile does not fit), and run-to-run identity of each."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_permute_gb300 import workloads as wl
from helpers import TOL_BF16, assert_close, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
IMPLS = {"auto": 0, "tcgen05": 1, "swap_ab": 2, "simt": 3}


def _layer_vs_oracle(moe, T, K, I, E, k, impl, seed, ids=None, weights=None):
    w = wl.scaled(wl.decode(max(T, 1)), T=T, K=K, I=I, E=E, top_k=k, w_std=0.05)
    x = wl.activations(w, seed)
    W1, W2 = wl.expert_weights(w, "W1", seed), wl.expert_weights(w, "W2", seed)
    layer = moe.MoELayer(T, K, I, E, k, impl=IMPLS[impl], device=DEV)
    if ids is None:
        logits = wl.router_logits(w, seed)
        out = layer.forward(x.to(DEV), W1.to(DEV), W2.to(DEV), logits=logits.to(DEV))
        ids, weights = oracle.topk_route(logits.numpy(), k)
    else:
        out = layer.forward(x.to(DEV), W1.to(DEV), W2.to(DEV), topk_ids=torch.from_numpy(ids).to(DEV),
                            topk_weights=torch.from_numpy(weights).to(DEV))
    first = out.clone()
    out2 = layer.forward(x.to(DEV), W1.to(DEV), W2.to(DEV), topk_ids=torch.from_numpy(ids).to(DEV),
                         topk_weights=torch.from_numpy(weights).to(DEV))
    torch.cuda.synchronize()
    assert layer.device_errors() == 0
    assert torch.equal(first.view(torch.int16), out2.view(torch.int16))       # run-to-run identical
    ref, _ = oracle.moe_layer(wl.to_numpy(x), ids, weights, wl.to_numpy(W1), wl.to_numpy(W2))
    return first.cpu(), ref


@pytest.mark.parametrize("impl", ["auto", "swap_ab", "simt"])
def test_empty_batch(moe, impl):
    """T = 0: every call is a no-op and the layer returns an empty output."""
    E, K, I, k = 8, 256, 128, 2
    w = wl.scaled(wl.decode(1), T=0, K=K, I=I, E=E, top_k=k)
    layer = moe.MoELayer(0, K, I, E, k, impl=IMPLS[impl], device=DEV)
    x = torch.empty((0, K), dtype=torch.bfloat16, device=DEV)
    logits = torch.empty((0, E), dtype=torch.float32, device=DEV)
    W1, W2 = wl.expert_weights(w, "W1", 0, DEV), wl.expert_weights(w, "W2", 0, DEV)
    out = layer.forward(x, W1, W2, logits=logits)
    torch.cuda.synchronize()
    assert out.shape == (0, K) and layer.device_errors() == 0


@pytest.mark.parametrize("impl", ["tcgen05", "swap_ab", "simt"])
def test_all_slots_padding(moe, impl):
    """Every slot is padding (id -1): nothing is computed and every output is +0.0."""
    T, K, I, E, k = 40, 256, 128, 8, 4
    ids = np.full((T, k), -1, np.int32)
    weights = np.zeros((T, k), np.float32)
    out, ref = _layer_vs_oracle(moe, T, K, I, E, k, impl, 5, ids, weights)
    assert torch.all(out == 0) and not torch.any(torch.signbit(out.float()))
    assert np.all(ref == 0)


@pytest.mark.parametrize("impl", ["auto", "tcgen05", "swap_ab", "simt"])
def test_single_expert(moe, impl):
    """E = 1, top_k = 1: the layer is one dense FFN with weight 1."""
    out, ref = _layer_vs_oracle(moe, 70, 256, 128, 1, 1, impl, 6)
    assert_close(to_f64(out), ref, TOL_BF16, f"single expert {impl}")


@pytest.mark.parametrize("impl", ["auto", "swap_ab", "simt"])
def test_topk_equals_experts(moe, impl):
    """top_k = E: every token visits every expert with the plain softmax weights."""
    out, ref = _layer_vs_oracle(moe, 33, 256, 128, 4, 4, impl, 7)
    assert_close(to_f64(out), ref, TOL_BF16, f"top_k = E {impl}")


@pytest.mark.parametrize("impl", ["auto", "swap_ab"])
def test_smallest_contraction(moe, impl):
    """K = I = 64: one k-block per tile; GEMM 2's 64 output rows do not fill a 128-row swap-AB tile, so AUTO
    runs it on the CUDA-core tiles and forcing swap-AB reports MOE_ERR_UNSUPPORTED."""
    if impl == "swap_ab":
        with pytest.raises(moe.MoEError) as ei:
            _layer_vs_oracle(moe, 20, 64, 64, 4, 2, impl, 8)
        assert ei.value.status == 2
        return
    out, ref = _layer_vs_oracle(moe, 20, 64, 64, 4, 2, impl, 8)
    assert_close(to_f64(out), ref, TOL_BF16, "K = I = 64")
