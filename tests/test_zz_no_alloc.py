"""The planner entry point that allocates nothing (bep_plan_noalloc).

It exists for callers that cannot call cudaMalloc when they plan: services
whose device memory is handed out once at start-up and may not grow, and
embedders that do not own the allocator or cannot keep a bep_ctx. Its scratch
is a static 2 MiB device array inside the library, shared by every call, so
these tests check that calls in a row (the second on a routing with a different
replica layout, then ones of other sizes, up to the largest the array holds)
each give exactly what bep_plan gives through a context, and that a bad
routing is reported through the caller's error word.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import moe_expert_dispatch_online_gb300 as bep
import synth


def _outputs(cfg, dev):
    return (torch.full((cfg.R, cfg.E + cfg.B + 1), -7, dtype=torch.int32, device=dev),
            torch.full((cfg.R, cfg.B), -7, dtype=torch.int32, device=dev),
            torch.full((cfg.R, cfg.S, cfg.K), -7, dtype=torch.int32, device=dev),
            torch.full((1,), -7.0, dtype=torch.float64, device=dev))


def _with_context(cfg, topk):
    with bep.Context(cfg) as ctx:
        cu, se, dest, mv = _outputs(cfg, topk.device)
        bep.bep_plan(ctx, topk, cu, se, dest, mv)
        assert bep.bep_status(ctx) == 0
        return cu.cpu(), se.cpu(), dest.cpu(), mv.cpu()


def _no_alloc(cfg, topk):
    cu, se, dest, mv = _outputs(cfg, topk.device)
    err = torch.full((1,), 12345, dtype=torch.int32, device=topk.device)
    bep.bep_plan_noalloc(cfg, topk, cu, se, dest, mv, err)
    torch.cuda.synchronize()
    return cu.cpu(), se.cpu(), dest.cpu(), mv.cpu(), int(err.item())


@pytest.mark.gpu
def test_plan_noalloc_matches_plan_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bep.load()
    dev = torch.device("cuda")
    cases = [("train_r8_e64", 10.0), ("train_r8_e64", 0.2), ("bench_r8_e384", 20.0)]
    for name, target in cases:
        wl = synth.WORKLOADS[name]
        cfg = bep.Config(wl.R, wl.E, wl.B, wl.K, wl.S, wl.H, wl.Hp, wl.mode)
        topk = torch.from_numpy(synth.routing(wl, target, 0)).to(dev)
        ref = _with_context(cfg, topk)
        got = _no_alloc(cfg, topk)
        assert got[4] == 0, f"{name} {target}: device error bits {got[4]}"
        for a, b, what in zip(got[:4], ref, ("cu_seqlens", "slot_expert", "dest", "maxvio")):
            assert torch.equal(a, b), f"{name} {target}: {what} differs"


@pytest.mark.gpu
def test_plan_noalloc_at_the_largest_size_that_fits():
    """R=8, E=384, B=48, K=8: the chunk table grows with ceil(S/256), and S=43008
    (168 chunks per rank) is the largest S whose tables fit in the 2 MiB array."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bep.load()
    dev = torch.device("cuda")
    R, E, B, K, S = 8, 384, 48, 8, 43008
    cfg = bep.Config(R, E, B, K, S, 7168, 2048, bep.BEP_TRAIN)
    topk = torch.from_numpy(synth.gumbel_topk(R, S, K, synth.zipf_popularity(E, 0.9), 5)).to(dev)
    for _ in range(2):
        ref = _with_context(cfg, topk)
        got = _no_alloc(cfg, topk)
        assert got[4] == 0
        for a, b in zip(got[:4], ref):
            assert torch.equal(a, b)


@pytest.mark.gpu
def test_plan_noalloc_reports_a_bad_routing_in_the_error_word():
    """An expert id outside [0, E) sets BEP_DERR_EXPERT_ID in device_err and leaves
    an empty plan (dest = -1); the next call with a good routing clears the word
    and plans normally."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bep.load()
    dev = torch.device("cuda")
    wl = synth.WORKLOADS["train_r8_e64"]
    cfg = bep.Config(wl.R, wl.E, wl.B, wl.K, wl.S, wl.H, wl.Hp, wl.mode)
    good = synth.routing(wl, 1.0, 0)
    bad = good.copy()
    bad[2, 5, 1] = wl.E
    got = _no_alloc(cfg, torch.from_numpy(bad).to(dev))
    assert got[4] & bep.BEP_DERR_EXPERT_ID
    assert (got[2] == -1).all()
    ref = _with_context(cfg, torch.from_numpy(good).to(dev))
    got = _no_alloc(cfg, torch.from_numpy(good).to(dev))
    assert got[4] == 0
    for a, b in zip(got[:4], ref):
        assert torch.equal(a, b)


def _call(lib, c):
    cu = (ctypes.c_int32 * 16)()
    mv = (ctypes.c_double * 1)()
    err = (ctypes.c_int32 * 4)()
    return lib.bep_plan_noalloc(ctypes.byref(c), ctypes.addressof(cu), ctypes.addressof(cu),
                                ctypes.addressof(cu), ctypes.addressof(cu), ctypes.addressof(mv),
                                ctypes.addressof(err), None)


def test_plan_noalloc_rejects_sizes_past_the_array_before_any_device_work():
    """One token past the largest S that fits (43008 at R=8, E=384) is refused on the
    host with BEP_ERR_SIZE; so is a far larger batch. The configurations are valid
    otherwise (make_dims accepts them), so only the scratch limit refuses them."""
    lib = bep.load()
    for S in (43009, 65536):
        assert _call(lib, bep._Config(8, 384, 48, 8, S, 7168, 2048, bep.BEP_TRAIN)) == bep.BEP_ERR_SIZE


def test_plan_noalloc_rejects_an_inconsistent_configuration():
    lib = bep.load()
    assert _call(lib, bep._Config(8, 383, 48, 8, 64, 7168, 2048, bep.BEP_TRAIN)) == bep.BEP_ERR_SIZE
    assert _call(lib, bep._Config(8, 384, 40, 8, 64, 7168, 2048, bep.BEP_TRAIN)) == bep.BEP_ERR_MODE
