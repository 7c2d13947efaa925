"""Failure detection on the GPU without a fault: invalid indices that the
kernels' own checks turn into BEP_DERR_BOUNDS (nothing written outside the
outputs, guard regions intact), a bounded wait that runs out and reports
BEP_DERR_TIMEOUT, and a context that stays usable afterwards."""
import time

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


class Guarded:
    PAD = 65536

    def __init__(self, shape, dtype, fill=0):
        n = int(np.prod(shape))
        esz = torch.empty((), dtype=dtype).element_size()
        self.pad = self.PAD // esz
        self.raw = torch.empty(n + 2 * self.pad, dtype=dtype, device=DEV)
        self.raw.view(torch.uint8).fill_(0xA5)
        self.t = self.raw[self.pad:self.pad + n].view(shape)
        self.t.view(torch.uint8).fill_(fill)

    def intact(self):
        b = self.raw.view(torch.uint8)
        nb = self.pad * self.raw.element_size()
        return bool((b[:nb] == 0xA5).all().item() and (b[-nb:] == 0xA5).all().item())


def planned(bep, name="train_r8_e64", target=10.0):
    wl = synth.WORKLOADS[name]
    cfg = bep.Config(wl.R, wl.E, wl.B, wl.K, wl.S, wl.H, wl.Hp, wl.mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, DEV)
    topk = synth.routing(wl, target, 0)
    bep.bep_plan(ctx, torch.from_numpy(topk).to(DEV), buf.cu_seqlens, buf.slot_expert, buf.dest,
                 buf.maxvio)
    assert bep.bep_status(ctx) == 0
    return wl, ctx, buf, topk


def test_bounded_wait_runs_out_and_context_stays_usable(lib):
    bep = lib
    wl, ctx, buf, topk = planned(bep)
    t0 = time.perf_counter()
    bep.bep_wait_selftest(ctx, 20000)            # 20 ms on a barrier nothing signals
    st = bep.bep_status(ctx)
    dt = time.perf_counter() - t0
    assert st & bep.BEP_DERR_TIMEOUT
    assert 0.015 < dt < 5.0
    bep.bep_clear_status(ctx)
    bep.bep_plan(ctx, torch.from_numpy(topk).to(DEV), buf.cu_seqlens, buf.slot_expert, buf.dest,
                 buf.maxvio)
    assert bep.bep_status(ctx) == 0
    ref = oracle.plan(topk, wl.E, wl.B, wl.mode)
    np.testing.assert_array_equal(buf.dest.cpu().numpy(), ref.dest)


def test_bad_dest_in_token_kernels(lib):
    bep = lib
    wl, ctx, buf, topk = planned(bep)
    dest = buf.dest.clone()
    dest[2, 5, 1] = wl.R * wl.C            # one past the receive space
    dest[4, 9, 0] = -3
    gates = torch.from_numpy(synth.gates_host(wl.R, wl.S, wl.K, 1)).to(DEV)
    y = synth.tokens_device((wl.R * wl.C, wl.Hp), 2)
    dout = synth.tokens_device((wl.R, wl.S, wl.Hp), 3)
    calls = [
        ("combine", (wl.R, wl.S, wl.Hp), torch.bfloat16,
         lambda o: bep.bep_combine(ctx, y, dest, gates, o)),
        ("combine_bwd", (wl.R * wl.C, wl.Hp), torch.bfloat16,
         lambda o: bep.bep_combine_bwd(ctx, dout, dest, gates, o)),
        ("dispatch_bwd", (wl.R, wl.S, wl.Hp), torch.bfloat16, None),
        ("dgates", (wl.R, wl.S, wl.K), torch.float32,
         lambda o: bep.bep_combine_dgates(ctx, dout, y, dest, o)),
    ]
    for name, shape, dtype, fn in calls:
        if fn is None:      # dispatch backward reads H-wide rows
            drecv = synth.tokens_device((wl.R * wl.C, wl.H), 4)
            g = Guarded((wl.R, wl.S, wl.H), dtype)
            bep.bep_dispatch_bwd(ctx, drecv, dest, g.t)
        else:
            g = Guarded(shape, dtype)
            fn(g.t)
        st = bep.bep_status(ctx)
        assert st & bep.BEP_DERR_BOUNDS, name
        assert g.intact(), name
        bep.bep_clear_status(ctx)


def test_bad_cu_seqlens_in_gemms(lib):
    bep = lib
    wl, ctx, buf, topk = planned(bep)
    cu = buf.cu_seqlens.clone()
    cu[3, 10] = cu[3, 11] + 5               # a segment that ends before it starts
    cu[6, -1] = wl.C + 128                  # a rank that runs past its rows
    w_home = synth.weights_device((wl.E, wl.H, wl.Hp), 5)
    w_slots = torch.zeros((wl.R, wl.B, wl.H, wl.Hp), dtype=torch.bfloat16, device=DEV)
    recv = synth.tokens_device((wl.R * wl.C, wl.H), 6)
    dy = synth.tokens_device((wl.R * wl.C, wl.Hp), 7)
    for name in ("fwd", "dx", "dw"):
        if name == "fwd":
            g = Guarded((wl.R * wl.C, wl.Hp), torch.bfloat16, fill=0x11)
            bep.bep_grouped_gemm(ctx, cu, recv, w_home, w_slots, g.t)
        elif name == "dx":
            g = Guarded((wl.R * wl.C, wl.H), torch.bfloat16, fill=0x11)
            bep.bep_grouped_gemm_dx(ctx, cu, dy, w_home, w_slots, g.t)
        else:
            g = Guarded((wl.E, wl.H, wl.Hp), torch.float32, fill=0)
            red = torch.zeros((wl.R, wl.B, wl.H, wl.Hp), dtype=torch.float32, device=DEV)
            bep.bep_grouped_gemm_dw(ctx, cu, recv, dy, g.t, red)
        st = bep.bep_status(ctx)
        assert st & bep.BEP_DERR_BOUNDS, name
        assert g.intact(), name
        # an inconsistent table is refused as a whole: nothing is written
        assert (g.t.view(torch.uint8) == (0x11 if name != "dw" else 0)).all().item(), name
        bep.bep_clear_status(ctx)


def test_bad_slot_map(lib):
    bep = lib
    wl, ctx, buf, topk = planned(bep, "grad_r8_e64")
    se = buf.slot_expert.clone()
    used = (se >= 0).nonzero()
    assert len(used) > 0
    u, j = used[0].tolist()
    se[u, j] = wl.E + 7                      # an expert that does not exist
    w_home = synth.weights_device((wl.E, wl.H, wl.Hp), 8)
    slots = Guarded((wl.R, wl.B, wl.H, wl.Hp), torch.bfloat16)
    bep.bep_prefetch_weight(ctx, se, w_home, slots.t)
    assert bep.bep_status(ctx) & bep.BEP_DERR_BOUNDS
    assert slots.intact()
    assert not slots.t[u, j].view(torch.int16).any().item()   # the bad slot was skipped
    bep.bep_clear_status(ctx)
    g = Guarded((wl.E, wl.H, wl.Hp), torch.float32)
    red = torch.ones((wl.R, wl.B, wl.H, wl.Hp), dtype=torch.float32, device=DEV)
    bep.bep_reduce_grad(ctx, se, g.t, red)
    assert bep.bep_status(ctx) & bep.BEP_DERR_BOUNDS
    assert g.intact()
    assert (red[u, j] == 1).all().item()                      # not consumed
