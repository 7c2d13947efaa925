"""The weight layout of the pages' memory contract on one GPU: the "VM group
GEMM" that addresses each rank's [E+B, H, H'] weights by row index alone, and
the weight store whose per-rank views alias the home rows and one prefetch-slot
pool shared by every layer (CUDA virtual memory management)."""
import ctypes

import numpy as np
import pytest
import torch

import elementwise as ew
import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def setup(bep, name, target):
    wl = synth.WORKLOADS[name]
    topk = synth.routing(wl, target, 0)
    cfg = bep.Config(wl.R, wl.E, wl.B, wl.K, wl.S, wl.H, wl.Hp, wl.mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, DEV)
    bep.bep_plan(ctx, torch.from_numpy(topk).to(DEV), buf.cu_seqlens, buf.slot_expert, buf.dest,
                 buf.maxvio)
    return wl, cfg, ctx, buf


def test_vm_gemm_equals_grouped_gemm_on_materialised_views(lib):
    bep = lib
    wl, cfg, ctx, buf = setup(bep, "train_r8_e64", 10.0)
    w_home = synth.weights_device((wl.E, wl.H, wl.Hp), 201)
    w_slots = torch.zeros((wl.R, wl.B, wl.H, wl.Hp), dtype=torch.bfloat16, device=DEV)
    bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots)
    bep.bep_dispatch(ctx, synth.tokens_device((wl.R, wl.S, wl.H), 202), buf.dest, buf.recv)
    views = torch.cat([w_home.unsqueeze(0).expand(wl.R, -1, -1, -1), w_slots], dim=1).contiguous()
    y_ref = torch.empty_like(buf.y)
    bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, y_ref)
    bep.bep_grouped_gemm_vm(ctx, buf.cu_seqlens, buf.recv, views, buf.y)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    assert torch.equal(buf.y.view(torch.int16), y_ref.view(torch.int16))


def test_weight_store_aliases_and_shares_the_pool_across_layers(lib):
    bep = lib
    wl, cfg, ctx, buf = setup(bep, "grad_r8_e64", 10.0)    # expert rows of 4 MiB
    store = bep.WeightStore(cfg, layers=2)
    x = synth.tokens_device((wl.R, wl.S, wl.H), 211)
    bep.bep_dispatch(ctx, x, buf.dest, buf.recv)
    slots = store.slots()
    for layer in range(2):
        home = store.home(layer)
        w = synth.weights_device((wl.E, wl.H, wl.Hp), 212 + layer)
        home.copy_(w)                                   # write through the home alias
        views = store.views(layer)
        for u in range(wl.R):                           # ... seen through every rank's view
            assert torch.equal(views[u, :wl.E].view(torch.int16), w.view(torch.int16))
        bep.bep_prefetch_weight(ctx, buf.slot_expert, home, slots)   # the shared pool
        torch.cuda.synchronize()
        se = buf.slot_expert.cpu().numpy()
        for u in range(wl.R):
            for j in range(wl.B):
                if se[u, j] >= 0:
                    assert torch.equal(views[u, wl.E + j].view(torch.int16),
                                       w[se[u, j]].view(torch.int16))
        y_ref = torch.empty_like(buf.y)
        bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, home, slots, y_ref)
        bep.bep_grouped_gemm_vm(ctx, buf.cu_seqlens, buf.recv, views, buf.y)
        torch.cuda.synchronize()
        assert bep.bep_status(ctx) == 0
        assert torch.equal(buf.y.view(torch.int16), y_ref.view(torch.int16))
        # and against the oracle on a few segments' rows
        ref = oracle.plan(synth.routing(wl, 10.0, 0), wl.E, wl.B, wl.mode)
        C = wl.C
        inv = np.empty(wl.R * C, np.int64)
        inv[ref.dest.ravel()] = np.arange(wl.R * wl.S * wl.K) // wl.K
        for u in (0, wl.R - 1):
            for rho in range(wl.E + wl.B):
                a, b = int(ref.cu[u, rho]), int(ref.cu[u, rho + 1])
                if b == a or not (rho >= wl.E or rho == u * (wl.E // wl.R)):
                    continue
                rows = np.array([u * C + a, u * C + b - 1])
                xr = x.view(-1, wl.H)[torch.from_numpy(inv[rows]).to(DEV)]
                e = oracle.weight_row_of(rho, u, wl.E, ref.slot_expert)
                want = oracle.gemm_rows(xr.view(torch.int16).cpu().numpy().view(np.uint16),
                                        w[e].view(torch.int16).cpu().numpy().view(np.uint16))
                got = oracle.bf16_to_f32(buf.y[torch.from_numpy(rows).to(DEV)].view(torch.int16)
                                         .cpu().numpy().view(np.uint16)).astype(np.float64)
                assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 2e-2
                ew.fwd(got, want,
                       oracle.bf16_to_f32(xr.view(torch.int16).cpu().numpy().view(np.uint16)),
                       oracle.bf16_to_f32(w[e].view(torch.int16).cpu().numpy().view(np.uint16)),
                       f"rank {u} row {rho}")
    del slots, home, views
    store.close()


def test_weight_store_needs_granular_blocks(lib):
    bep = lib
    wl = synth.WORKLOADS["tiny_r2_e8"]                   # 8 home rows of 16 KB: not a 2 MiB block
    c = bep._Config(wl.R, wl.E, wl.B, wl.K, wl.S, wl.H, wl.Hp, wl.mode)
    h = ctypes.c_void_p()
    assert bep.load().bep_weights_create(ctypes.byref(c), 1, ctypes.byref(h)) == bep.BEP_ERR_SIZE
    assert not h.value
