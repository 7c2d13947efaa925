"""The planner entry point that allocates nothing (bep_plan_noalloc).

It exists for callers that cannot call cudaMalloc when they plan (code running
under CUDA-graph stream capture, services with a fixed memory pool, embedders
without a bep_ctx). Its scratch is a static device array inside the library,
shared by every call, so these tests check that two calls in a row (the
second on a routing with a different replica layout, then one of another
size) each give exactly what bep_plan gives through a context.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
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


def test_plan_noalloc_rejects_oversized_config_before_any_device_work():
    lib = bep.load()
    # E * R * ceil(S/256) * 4 bytes of chunk counts alone exceed the 2 MiB array
    c = bep._Config(8, 384, 48, 8, 65536, 7168, 2048, bep.BEP_TRAIN)
    cu = (ctypes.c_int32 * 16)()
    mv = (ctypes.c_double * 1)()
    err = (ctypes.c_int32 * 4)()
    rc = lib.bep_plan_noalloc(ctypes.byref(c), ctypes.addressof(cu), ctypes.addressof(cu),
                              ctypes.addressof(cu), ctypes.addressof(cu), ctypes.addressof(mv),
                              ctypes.addressof(err), None)
    assert rc == bep.BEP_ERR_SIZE
    bad = bep._Config(8, 383, 48, 8, 64, 7168, 2048, bep.BEP_TRAIN)   # E % R != 0
    rc = lib.bep_plan_noalloc(ctypes.byref(bad), ctypes.addressof(cu), ctypes.addressof(cu),
                              ctypes.addressof(cu), ctypes.addressof(cu), ctypes.addressof(mv),
                              ctypes.addressof(err), None)
    assert rc == bep.BEP_ERR_SIZE
    assert np.all(np.frombuffer(err, dtype=np.int32) == 0)   # nothing was written
