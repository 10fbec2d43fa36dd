"""moe_permute_align_static: the permute step for callers that cannot allocate device memory.

Such callers (a plugin inside a framework that owns all device memory, a request
path where cudaMalloc/cudaFree and the device synchronisation they can cause are
not allowed, a deployment with a memory budget fixed at start-up) cannot pass a
workspace.  This entry point uses scratch built into the library instead.  Its
results must equal moe_permute_align's -- integer work, so bit for bit -- on two
calls in a row that share (and reuse) that built-in scratch.  The file is named so
that pytest collects it last.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _ids(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    ids[torch.rand(T, k, generator=g) < 0.05] = -1
    return ids


def _same(a, b, rows):
    assert torch.equal(a["counts"], b["counts"])
    assert torch.equal(a["offsets"], b["offsets"])
    assert torch.equal(a["row_route"][:rows], b["row_route"][:rows])
    assert torch.equal(a["route_row"], b["route_row"])


def test_static_scratch_matches_workspace_version_twice(moe):
    # several CTAs (more than 1024 routes), so the scratch is really used; then a different routing
    for T, k, E, bm, seed in ((4096, 8, 128, 128, 1), (3000, 4, 64, 1, 2)):
        ids = _ids(T, k, E, seed).to(DEV)
        x = torch.randn(T, 256, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16).to(DEV)
        ref = moe.moe_permute_align(ids, E, moe.MOE_LAYOUT_CONTIGUOUS, bm, x=x)
        got = moe.moe_permute_align_static(ids, E, moe.MOE_LAYOUT_CONTIGUOUS, bm, x=x)
        torch.cuda.synchronize()
        rows = int(ref["offsets"][E].item())
        _same(got, ref, rows)
        valid = ref["row_route"][:rows] >= 0
        assert torch.equal(got["x_out"][:rows][valid].view(torch.int16), ref["x_out"][:rows][valid].view(torch.int16))


def test_static_scratch_batched_and_limit(moe):
    ids = _ids(2000, 2, 16, 3).to(DEV)
    ref = moe.moe_permute_align(ids, 16, moe.MOE_LAYOUT_BATCHED, 1, 200)
    got = moe.moe_permute_align_static(ids, 16, moe.MOE_LAYOUT_BATCHED, 1, 200)
    _same(got, ref, 16 * 200)
    # a routing whose scratch exceeds the built-in 2 MiB is refused, with nothing launched
    big = torch.zeros((70000, 8), dtype=torch.int32, device=DEV)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_permute_align_static(big, 128, moe.MOE_LAYOUT_CONTIGUOUS, 1)
    assert ei.value.status == 4 and "2097152" in str(ei.value)


def test_static_small_routing_with_bad_ids_sets_the_same_error_bits(moe):
    # at most 1024 routes take the one-CTA placement, which never touches the scratch; ids outside [-1, E) must
    # be skipped and flagged exactly as moe_permute_align does
    T, k, E = 100, 8, 32
    ids = _ids(T, k, E, 4)
    ids[3, 1], ids[50, 7], ids[99, 0] = E, -7, 1000
    ids = ids.to(DEV)
    x = torch.randn(T, 128, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16).to(DEV)
    errs = []
    outs = []
    for fn in (moe.moe_permute_align, moe.moe_permute_align_static):
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        outs.append(fn(ids, E, moe.MOE_LAYOUT_CONTIGUOUS, 4, x=x, err_word=err))
        errs.append(err)
    torch.cuda.synchronize()
    ref, got = outs
    rows = int(ref["offsets"][E].item())
    _same(got, ref, rows)
    assert int(errs[0].item()) == int(errs[1].item()) == moe.MOE_DEVERR_ID_RANGE
    assert int((ref["route_row"] >= 0).sum().item()) == int(((ids >= 0) & (ids < E)).sum().item())
