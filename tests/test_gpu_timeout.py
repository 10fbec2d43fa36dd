"""Failure detection on the GPU without a fault: a pipeline wait that runs out.

A child process sets MOE_TEST_SKIP_FIRST_COPY=1, so CTA 0 of the tcgen05 GEMM never
issues its first weight copy and that stage's barrier never completes (a flag nothing
sets).  The bounded wait gives up after ~2 s: the kernel must report
MOE_DEVERR_TIMEOUT in err_word, free its tensor memory and return, leaving the CUDA
context usable -- the same process then runs routing and checks it against the oracle.
In the fused experts launch the GEMM 2 tiles that wait on CTA 0's unfinished GEMM 1
tile give up the same way (their wait on the segment counter is bounded too).  The
batched case runs the 256-row normal tiles (one accumulator, 8 epilogue warps); the
E4M3 case the MXFP8-weight tiles whose converter warps wait on the code ring (E4M3N: their 32-token form
with four MMA warps, two per slice); the MX
case the block-scaled MXFP8 kernel (gemm_mx_kernel), whose MMA waits on the ring
while its scale writers run ahead; the PAIR case the CTA-pair tiles, where the leader CTA's MMA waits
on a stage whose bytes (counted for both CTAs) never all arrive, and both CTAs of every pair must
still meet at their closing cluster barrier and free their tensor memory.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, time
sys.path.insert(0, {root!r})
import numpy as np, torch
import mixture_experts_layer_permute_gb300 as m
import oracle
from mixture_experts_layer_permute_gb300 import workloads as wl
E = 16 if "{impl}" == "E4M3N" else 4   # 8 rows per expert: the 32-token MXFP8-weight tiles with four MMA warps
w = wl.scaled(wl.decode(64), T=64, K=256, I=128, E=E, top_k=2)
x, logits = wl.activations(w, 0).cuda(), wl.router_logits(w, 0)
W1 = wl.expert_weights(w, "W1", 0).cuda()
W2 = wl.expert_weights(w, "W2", 0).cuda()
ids, _ = m.moe_topk_route(logits.cuda(), 2)
if "{impl}" == "BATCHED":   # batched rows: 256-row normal tiles
    res = m.moe_permute_align(ids, E, m.MOE_LAYOUT_BATCHED, 1, 64, x=x)
else:
    res = m.moe_permute_align(ids, E, m.MOE_LAYOUT_CONTIGUOUS, 1, x=x)
err = torch.zeros(1, dtype=torch.int32, device="cuda")
t0 = time.time()
if "{impl}" in ("E4M3", "E4M3N", "MX"):   # MXFP8 weights: E4M3 codes + E8M0 scales
    W1c, W1s = m.mxfp8_quantize_block32(W1)
if "{impl}" == "BATCHED":
    m.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], W1, 128, layout=m.MOE_LAYOUT_BATCHED,
                       max_tokens=64, impl=m.MOE_IMPL_TCGEN05, err_word=err)
elif "{impl}" in ("E4M3", "E4M3N"):   # bf16 activations x MXFP8 weights: converter warps decode into TMEM
    m.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], W1c, 128, w1_scale=W1s,
                       impl=m.MOE_IMPL_TCGEN05_SWAP_AB, err_word=err)
elif "{impl}" == "MX":          # MXFP8 activations x MXFP8 weights: block-scaled MMA (gemm_mx_kernel)
    xc, xs = m.mxfp8_quantize_block32(res["x_out"])
    m.moe_gemm1_swiglu(xc, res["counts"], res["offsets"], W1c, 128, w1_scale=W1s, a_scale=xs,
                       impl=m.MOE_IMPL_TCGEN05_SWAP_AB, err_word=err)
elif "{impl}" == "FUSED":
    m.moe_experts_fused(res["x_out"], res["counts"], res["offsets"], W1, W2, 128, res["row_route"], 128,
                        err_word=err)
else:
    m.moe_gemm1_swiglu(res["x_out"], res["counts"], res["offsets"], W1, 128, impl=getattr(m, "MOE_IMPL_{impl}"),
                       err_word=err)
torch.cuda.synchronize()
dt = time.time() - t0
print("ERR", int(err.item()), "SECONDS", round(dt, 2))
ids2, w2 = m.moe_topk_route(logits.cuda(), 2)          # the context still works
rids, rw = oracle.topk_route(logits.numpy(), 2)
print("ROUTE_OK", bool(np.array_equal(ids2.cpu().numpy(), rids)))
"""


@pytest.mark.parametrize("impl", ["TCGEN05", "TCGEN05_SWAP_AB", "FUSED", "BATCHED", "E4M3", "E4M3N", "MX",
                                  "TCGEN05_PAIR"])
def test_gemm_wait_runs_out_and_reports(moe, impl):
    env = dict(os.environ, MOE_TEST_SKIP_FIRST_COPY="1")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, impl=impl)], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    fields = dict(zip(r.stdout.split()[::2], r.stdout.split()[1::2]))
    assert int(fields["ERR"]) & moe.MOE_DEVERR_TIMEOUT
    assert 1.0 <= float(fields["SECONDS"]) <= 30.0
    assert fields["ROUTE_OK"] == "True"
