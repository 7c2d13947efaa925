"""Run-to-run determinism: the whole chain -- plan, prefetch_weight, dispatch,
grouped GEMM, combine, combine backward, gate gradient, dispatch backward, dX and
dW GEMMs, reduce_grad -- queued twice on the same inputs, or replayed from one
CUDA graph, gives the same bits in every output. Nothing in the path has an unspecified order (no floating-point
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


def test_whole_chain_in_one_cuda_graph_matches_eager(lib):
    """The same chain captured once in a CUDA graph on a side stream -- the dW GEMM's
    launch on clusters of two CTAs included -- and replayed on two new routings gives
    the bits that queueing it eagerly on each routing gives. The gradients start from
    the same values on every replay (their copies are part of the graph)."""
    bep = lib
    wl = synth.WORKLOADS["train_r8_e64"]
    R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
    gen = torch.Generator(device=DEV)
    gen.manual_seed(5)
    inputs = (synth.tokens_device((R, S, H), 71),
              torch.from_numpy(synth.gates_host(R, S, K, 72)).to(DEV),
              synth.tokens_device((R, S, Hp), 73),
              synth.weights_device((E, H, Hp), 74),
              torch.empty((E, H, Hp), dtype=torch.float32, device=DEV).normal_(0, 1e-2, generator=gen),
              torch.empty((R, B, H, Hp), dtype=torch.float32, device=DEV).normal_(0, 1e-3, generator=gen))
    x, gates, dout, w_home, g0, red0 = inputs
    routings = {t: torch.from_numpy(synth.routing(wl, t, 1)).to(DEV) for t in (10.0, 0.2)}
    warm = torch.from_numpy(synth.routing(wl, 1.0, 0)).to(DEV)
    eager = {t: chain(bep, wl, topk, inputs) for t, topk in routings.items()}

    ctx = bep.Context(bep.Config(R, E, B, K, S, H, Hp, wl.mode))
    buf = bep.Buffers(ctx.cfg, DEV, with_grad=True)
    topk_d = torch.zeros((R, S, K), dtype=torch.int32, device=DEV)
    w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=DEV)
    g, red = torch.empty_like(g0), torch.empty_like(red0)
    dg = torch.empty((R, S, K), dtype=torch.float32, device=DEV)
    drecv = torch.empty((R * S * K, H), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((R, S, H), dtype=torch.bfloat16, device=DEV)

    def queue():
        g.copy_(g0)
        red.copy_(red0)
        bep.bep_plan(ctx, topk_d, buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio)
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

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        topk_d.copy_(warm)
        queue()                      # warm-up outside the capture, on a third routing
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        queue()
    for t, topk in routings.items():
        topk_d.copy_(topk)
        graph.replay()
        torch.cuda.synchronize()
        assert bep.bep_status(ctx) == 0
        outs = dict(cu=buf.cu_seqlens, dest=buf.dest, slots=buf.slot_expert, w_slots=w_slots,
                    recv=buf.recv, y=buf.y, out=buf.out, dy=buf.dy, dg=dg, drecv=drecv, dx=dx,
                    g=g, red=red)
        for k, v in outs.items():
            if k == "w_slots":   # unused slots keep whatever an earlier routing put there
                used = eager[t]["slots"].view(torch.int32).view(R, B) >= 0
                a = v.view(torch.int16).view(R, B, -1)[used]
                b = eager[t][k].view(torch.int16).view(R, B, -1)[used]
                assert torch.equal(a, b), (t, k)
                continue
            assert torch.equal(v.contiguous().view(torch.uint8), eager[t][k]), (t, k)
