"""Run-to-run determinism: the whole chain -- plan, prefetch_weight, dispatch,
grouped GEMM, combine, combine backward, gate gradient, dispatch backward, dX and
dW GEMMs, reduce_grad -- queued twice on the same inputs gives the same bits in
every output. Nothing in the path has an unspecified order (no floating-point
atomics; dW adds each gradient element once per launch)."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def chain(bep, wl, topk, inputs):
    R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
    cfg = bep.Config(R, E, B, K, S, H, Hp, wl.mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, DEV, with_grad=True)
    x, gates, dout, w_home, g0, red0 = inputs
    w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=DEV)
    g, red = g0.clone(), red0.clone()
    dg = torch.empty((R, S, K), dtype=torch.float32, device=DEV)
    drecv = torch.empty((R * S * K, H), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((R, S, H), dtype=torch.bfloat16, device=DEV)
    bep.bep_plan(ctx, topk, buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio)
    bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots)
    bep.bep_dispatch(ctx, x, buf.dest, buf.recv)
    bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y)
    bep.bep_combine(ctx, buf.y, buf.dest, gates, buf.out)
    bep.bep_combine_bwd(ctx, dout, buf.dest, gates, buf.dy)
    bep.bep_combine_dgates(ctx, dout, buf.y, buf.dest, dg)
    bep.bep_grouped_gemm_dx(ctx, buf.cu_seqlens, buf.dy, w_home, w_slots, drecv)
    bep.bep_dispatch_bwd(ctx, drecv, buf.dest, dx)
    bep.bep_grouped_gemm_dw(ctx, buf.cu_seqlens, buf.recv, buf.dy, g, red)
    bep.bep_reduce_grad(ctx, buf.slot_expert, g, red)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    outs = dict(cu=buf.cu_seqlens, dest=buf.dest, slots=buf.slot_expert, w_slots=w_slots,
                recv=buf.recv, y=buf.y, out=buf.out, dy=buf.dy, dg=dg, drecv=drecv, dx=dx,
                g=g, red=red)
    return {k: v.contiguous().view(torch.uint8).clone() for k, v in outs.items()}


@pytest.mark.parametrize("name,target", [("train_r8_e64", 10.0), ("grad_r8_e64", 10.0)])
def test_whole_chain_is_bitwise_deterministic(lib, name, target):
    bep = lib
    wl = synth.WORKLOADS[name]
    topk = torch.from_numpy(synth.routing(wl, target, 0)).to(DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(3)
    inputs = (synth.tokens_device((wl.R, wl.S, wl.H), 61),
              torch.from_numpy(synth.gates_host(wl.R, wl.S, wl.K, 62)).to(DEV),
              synth.tokens_device((wl.R, wl.S, wl.Hp), 63),
              synth.weights_device((wl.E, wl.H, wl.Hp), 64),
              torch.empty((wl.E, wl.H, wl.Hp), dtype=torch.float32, device=DEV).normal_(0, 1e-2, generator=gen),
              torch.empty((wl.R, wl.B, wl.H, wl.Hp), dtype=torch.float32, device=DEV).normal_(0, 1e-3, generator=gen))
    a = chain(bep, wl, topk, inputs)
    b = chain(bep, wl, topk, inputs)
    for k in a:
        assert torch.equal(a[k], b[k]), k
