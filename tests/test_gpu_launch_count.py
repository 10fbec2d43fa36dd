"""The kernel launches of one MoELayer forward, counted by the CUDA activity trace (torch.profiler), equal
MoELayer.launches_per_forward(), the count bench.py reports as gpu_launches; every traced kernel of the forward
is one of the library's own."""
import pytest
import torch

from mixture_experts_layer_permute_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _trace_warmed_up():
    """The first profiler session of a process can come back without device activity while the tracer starts."""
    from torch.profiler import ProfilerActivity, profile
    a = torch.ones(1024, device=DEV)
    for _ in range(2):
        with profile(activities=[ProfilerActivity.CUDA]):
            (a * 2).sum().item()


def _library_kernels(fn):
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    kernels = [n for n in names if "moe::" in n or "_ZN3moe" in n]
    others = [n for n in names if n not in kernels and "emcpy" not in n and "emset" not in n]
    return kernels, others


CASES = [  # T, K, I, E, top_k, layout, max_tokens, block_m, routed by logits
    (8, 256, 128, 16, 4, "contiguous", 0, 1, True),       # decode: route+permute+gather, fused experts, reduce
    (129, 256, 128, 32, 8, "contiguous", 0, 1, True),     # separate routing launches, two permute launches
    (300, 256, 256, 4, 2, "contiguous", 0, 128, True),    # normal tiles, two GEMM launches
    (40, 256, 128, 8, 2, "contiguous", 0, 1, False),      # ids given: no routing launch
    (100, 256, 128, 16, 4, "batched", 48, 1, True),       # batched rows from tokens
    (0, 256, 128, 8, 1, "batched", 64, 1, False),         # batched rows given
]


@pytest.mark.parametrize("T,K,I,E,k,layout,mt,bm,routed", CASES)
def test_launches_per_forward_matches_trace(moe, T, K, I, E, k, layout, mt, bm, routed):
    lay = moe.MOE_LAYOUT_CONTIGUOUS if layout == "contiguous" else moe.MOE_LAYOUT_BATCHED
    w = wl.scaled(wl.decode(64), T=max(T, 1), K=K, I=I, E=E, top_k=k)
    W1, W2 = wl.expert_weights(w, "W1", 2, DEV), wl.expert_weights(w, "W2", 2, DEV)
    layer = moe.MoELayer(T, K, I, E, k, layout=lay, max_tokens=mt, block_m=bm, device=DEV)
    if layout == "batched" and T == 0:
        g = torch.Generator().manual_seed(5)
        xb = wl._normal((E, mt, K), 1.0, 5, "xb", 0, DEV, torch.bfloat16)
        counts = torch.randint(0, mt + 1, (E,), generator=g, dtype=torch.int32).to(DEV)
        kw = dict(expert_num_tokens=counts)
        x = xb
    else:
        x = wl.activations(w, 2, DEV)
        if routed:
            kw = dict(logits=wl.router_logits(w, 2, DEV))
        else:
            ids = torch.stack([torch.randperm(E)[:k] for _ in range(T)]).to(torch.int32).to(DEV)
            kw = dict(topk_ids=ids, topk_weights=torch.full((T, k), 1.0 / k, device=DEV))
    layer.forward(x, W1, W2, **kw)              # builds the plan; first calls set up tensor maps
    kernels, others = _library_kernels(lambda: layer.forward(x, W1, W2, **kw))
    if not kernels and not others:
        pytest.skip("no CUDA activity trace in this PyTorch build")
    assert not others, others
    assert len(kernels) == layer.launches_per_forward(), kernels
