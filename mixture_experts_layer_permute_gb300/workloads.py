"""Seeded synthetic inputs for the fused MoE expert layer.

This module draws random numbers and lays them out; it holds none of the
layer's arithmetic (no routing, permutation, quantisation or matmul).  Both the
CUDA path and the CPU oracle take their inputs from here, so that each side
sees the identical arrays.

Each tensor is drawn from its own ``torch.Generator`` seeded from
``(seed, tensor name, expert)``, so one expert's slice can be regenerated on its
own and any tensor can be drawn on the CPU or on a CUDA device (the two devices
give different streams of numbers; a workload is always drawn on one device
and copied from there).

The workloads are the five synthetic configurations of the layer:

* ``tiny``      fp32, T=16, K=128, I=256, E=8, top_k=2, x and W ~ N(0, 0.02),
                router logits ~ N(0, 1).
* ``decode``    bf16, T in {1, 8, 32, 64}, K=4096, I=1536, E=128, top_k=8,
                x ~ N(0, 1), W ~ N(0, 0.02), logits ~ N(0, 1).
* ``prefill``   bf16, T=4096, same sizes, logits ~ N(0, 1) plus a per-expert bias
                2 log(1/(e+1)) (Zipf-like load), rows padded to 128 per expert.
* ``mxfp8``     T=512, K=7168, I=2048, E=512, top_k=8, x bf16 ~ N(0, 1), W drawn
                fp32 ~ N(0, 0.02) (each side quantises it), W1 rows in the
                gate/up interleave-16 layout, topk_ids[t, j] = ((8t + j) 73 + 19)
                mod 512 and weights 1/8 (the balanced routing pattern of the
                "Cake MegaMoE" PR analysis, section 1 "After").
* ``mxfp8_act`` the mxfp8 workload with x rows and h quantised to MXFP8 on the
                fly (E4M3 codes, one E8M0 scale per 32).
* ``batched``   (E=32, max_tokens=256, K=6144) activations, I=4096,
                expert_num_tokens uniform in [0, 256], rows beyond the count
                filled with garbage (NaN or +-1e30), per-row weights U(0, 1).
* ``batched_tokens``  the batched layout fed with tokens: T=1024, top_k=4,
                the same E, max_tokens, K and I, x ~ N(0, 1), logits ~ N(0, 1)
                (about 128 routes per expert, far from the capacity).
"""
from __future__ import annotations

import dataclasses
import zlib

import torch

BF16, F32 = "bf16", "f32"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens (batched: unused, see E * max_tokens)
    K: int                 # hidden
    I: int                 # intermediate per expert
    E: int                 # experts
    top_k: int
    act: str = BF16        # activation / output element type
    weight: str = BF16     # "f32", "bf16" or "mxfp8"
    layout: str = "contiguous"
    routing: str = "softmax"     # "softmax", "zipf", "affine" or "given"
    w1_layout: int = 0           # 0: [gate; up], 1: gate/up interleave-16
    block_m: int = 1             # per-expert row padding of the contiguous layout
    max_tokens: int = 0          # batched layout capacity
    x_std: float = 1.0
    w_std: float = 0.02
    garbage: str = "nan"         # batched: fill of rows beyond the count
    act_quant: bool = False      # activations (x rows, h) quantised to MXFP8 on the fly

    @property
    def routes(self) -> int:
        return self.T * self.top_k


def tiny() -> Workload:
    return Workload("tiny_fp32", T=16, K=128, I=256, E=8, top_k=2, act=F32, weight=F32, x_std=0.02)


def decode(T: int) -> Workload:
    return Workload(f"decode_T{T}", T=T, K=4096, I=1536, E=128, top_k=8)


def prefill() -> Workload:
    return Workload("prefill_skewed", T=4096, K=4096, I=1536, E=128, top_k=8, routing="zipf", block_m=128)


def mxfp8() -> Workload:
    return Workload("mxfp8_weights", T=512, K=7168, I=2048, E=512, top_k=8, weight="mxfp8", routing="affine",
                    w1_layout=1)


def mxfp8_act() -> Workload:
    """The mxfp8 workload with its activations quantised on the fly (block-scaled MXFP8 x MXFP8 GEMMs)."""
    return dataclasses.replace(mxfp8(), name="mxfp8_act_quant", act_quant=True)


def batched(garbage: str = "nan") -> Workload:
    return Workload("batched", T=0, K=6144, I=4096, E=32, top_k=1, layout="batched", routing="given",
                    max_tokens=256, garbage=garbage)


def batched_tokens() -> Workload:
    return Workload("batched_tokens", T=1024, K=6144, I=4096, E=32, top_k=4, layout="batched_tokens",
                    max_tokens=256)


def scaled(w: Workload, **changes) -> Workload:
    """Same recipe at other sizes (for tests that must finish in seconds)."""
    return dataclasses.replace(w, **changes)


# ----------------------------------------------------------------------------
# drawing
# ----------------------------------------------------------------------------

def _gen(seed: int, name: str, index: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + zlib.crc32(name.encode()) * 7919 + index) % (2 ** 63))
    return g


def _normal(shape, std, seed, name, index, device, dtype):
    g = _gen(seed, name, index, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _tdtype(kind: str):
    return torch.float32 if kind in (F32, "mxfp8") else torch.bfloat16


def expert_weights(w: Workload, which: str, seed: int = 0, device="cpu", experts=None) -> torch.Tensor:
    """W1 (E, 2I, K) or W2 (E, K, I), drawn expert by expert.

    For "mxfp8" workloads the values are returned in fp32, before quantisation.
    ``experts`` selects a subset (the slice is identical to the full draw's).
    """
    shape = (2 * w.I, w.K) if which == "W1" else (w.K, w.I)
    ids = range(w.E) if experts is None else list(experts)
    dt = _tdtype(w.weight)
    out = torch.empty((len(ids),) + shape, dtype=dt, device=device)
    for n, e in enumerate(ids):
        out[n] = _normal(shape, w.w_std, seed, which, e, device, dt)
    return out


def activations(w: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    """x: (T, K) for the contiguous layout."""
    return _normal((w.T, w.K), w.x_std, seed, "x", 0, device, _tdtype(w.act))


def router_logits(w: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    """(T, E) fp32 router logits; the "zipf" recipe adds 2 log(1/(e+1)) per expert."""
    logits = _normal((w.T, w.E), 1.0, seed, "logits", 0, device, torch.float32)
    if w.routing == "zipf":
        rank = torch.arange(1, w.E + 1, device=device, dtype=torch.float32)
        logits = logits + 2.0 * torch.log(1.0 / rank)
    return logits


def affine_routing(w: Workload, device="cpu"):
    """topk_ids[t, j] = ((t*8 + j)*73 + 19) mod E with weights 1/top_k."""
    t = torch.arange(w.T, device=device, dtype=torch.int64)[:, None]
    j = torch.arange(w.top_k, device=device, dtype=torch.int64)[None, :]
    ids = (((t * w.top_k + j) * 73 + 19) % w.E).to(torch.int32)
    weights = torch.full((w.T, w.top_k), 1.0 / w.top_k, device=device, dtype=torch.float32)
    return ids, weights


def batched_inputs(w: Workload, seed: int = 0, device="cpu"):
    """(xb (E, max_tokens, K), expert_num_tokens (E,), row weights (E, max_tokens))."""
    g = _gen(seed, "counts", 0, "cpu")
    counts = torch.randint(0, w.max_tokens + 1, (w.E,), generator=g, dtype=torch.int32)
    xb = _normal((w.E, w.max_tokens, w.K), w.x_std, seed, "xb", 0, device, _tdtype(w.act))
    fill = float("nan") if w.garbage == "nan" else 1.0e30
    rows = torch.arange(w.max_tokens)[None, :] >= counts[:, None].long()
    if w.garbage != "nan":
        sign = torch.where(torch.arange(w.K) % 2 == 0, 1.0, -1.0)
        garbage = (sign * fill).to(xb.dtype).to(device)
    else:
        garbage = torch.full((w.K,), fill, dtype=xb.dtype, device=device)
    xb[rows.to(device)] = garbage
    gw = _gen(seed, "row_weights", 0, device)
    weights = torch.rand((w.E, w.max_tokens), generator=gw, device=device, dtype=torch.float32)
    return xb, counts.to(device), weights


def padding_tokens(ids: torch.Tensor, weights: torch.Tensor, n_pad_tokens: int):
    """Append tokens whose every slot is padding (expert id -1, weight 0)."""
    pad_ids = torch.full((n_pad_tokens, ids.shape[1]), -1, dtype=ids.dtype, device=ids.device)
    pad_w = torch.zeros((n_pad_tokens, weights.shape[1]), dtype=weights.dtype, device=weights.device)
    return torch.cat([ids, pad_ids]), torch.cat([weights, pad_w])


def max_padded_rows(routes: int, E: int, block_m: int) -> int:
    """Upper bound on sum_e ceil(count_e / block_m) * block_m."""
    return routes + E * (block_m - 1)


def to_numpy(t: torch.Tensor):
    """numpy view for the oracle: bf16 as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def touched_bytes_per_expert(w: Workload) -> int:
    """Weight bytes one expert occupies (W1 + W2, with scales for mxfp8)."""
    n = 3 * w.I * w.K
    if w.weight == "mxfp8":
        return n + n // 32
    return n * (4 if w.weight == F32 else 2)
