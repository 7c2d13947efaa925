"""Two contexts at once: the whole chains of two workloads -- plan, prefetch_weight,
dispatch, grouped GEMM, combine, combine backward, gate gradient, dX GEMM,
dispatch backward, overwriting and accumulating dW, reduce_grad -- queued call by
call in turn on two CUDA streams, so that their kernels can run side by side,
give the bits each chain gives alone on the default stream. Nothing is shared
between contexts, and every call runs on the stream it is given."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def make_chain(bep, name, target, seed):
    """The chain's calls, each taking a stream, and the tensors they write."""
    wl = synth.WORKLOADS[name]
    R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
    cfg = bep.Config(R, E, B, K, S, H, Hp, wl.mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, DEV, with_grad=True)
    topk = torch.from_numpy(synth.routing(wl, target, 0)).to(DEV)
    x = synth.tokens_device((R, S, H), seed + 1)
    gates = torch.from_numpy(synth.gates_host(R, S, K, seed + 2)).to(DEV)
    dout = synth.tokens_device((R, S, Hp), seed + 3)
    w_home = synth.weights_device((E, H, Hp), seed + 4)
    w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    g_first = torch.empty((E, H, Hp), dtype=torch.float32, device=DEV)
    g = torch.empty((E, H, Hp), dtype=torch.float32, device=DEV).normal_(0, 1e-2, generator=gen)
    red = torch.zeros((R, B, H, Hp), dtype=torch.float32, device=DEV)
    red_first = torch.zeros((R, B, H, Hp), dtype=torch.float32, device=DEV)
    dg = torch.empty((R, S, K), dtype=torch.float32, device=DEV)
    drecv = torch.empty((R * S * K, H), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((R, S, H), dtype=torch.bfloat16, device=DEV)
    calls = [
        lambda s: bep.bep_plan(ctx, topk, buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio, s),
        lambda s: bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots, s),
        lambda s: bep.bep_dispatch(ctx, x, buf.dest, buf.recv, s),
        lambda s: bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y, s),
        lambda s: bep.bep_combine(ctx, buf.y, buf.dest, gates, buf.out, s),
        lambda s: bep.bep_combine_bwd(ctx, dout, buf.dest, gates, buf.dy, s),
        lambda s: bep.bep_combine_dgates(ctx, dout, buf.y, buf.dest, dg, s),
        lambda s: bep.bep_grouped_gemm_dx(ctx, buf.cu_seqlens, buf.dy, w_home, w_slots, drecv, s),
        lambda s: bep.bep_dispatch_bwd(ctx, drecv, buf.dest, dx, s),
        lambda s: bep.bep_grouped_gemm_dw_overwrite(ctx, buf.cu_seqlens, buf.recv, buf.dy, g_first,
                                                    red_first, s),
        lambda s: bep.bep_grouped_gemm_dw(ctx, buf.cu_seqlens, buf.recv, buf.dy, g, red, s),
        lambda s: bep.bep_reduce_grad(ctx, buf.slot_expert, g, red, s),
    ]
    outs = dict(cu=buf.cu_seqlens, dest=buf.dest, slots=buf.slot_expert, w_slots=w_slots,
                recv=buf.recv, y=buf.y, out=buf.out, dy=buf.dy, dg=dg, drecv=drecv, dx=dx,
                g_first=g_first, red_first=red_first, g=g, red=red)
    snapshot = {k: v.clone() for k, v in outs.items() if k in ("g", "red")}

    def reset():
        """Put the accumulated gradients back to their starting values."""
        for k, v in snapshot.items():
            outs[k].copy_(v)

    return ctx, calls, outs, reset


def bits(outs):
    return {k: v.contiguous().view(torch.uint8).clone() for k, v in outs.items()}


def test_two_contexts_on_two_streams_match_each_alone(lib):
    bep = lib
    a = make_chain(bep, "train_r8_e64", 10.0, 700)
    b = make_chain(bep, "grad_r8_e64", 10.0, 800)
    alone = []
    for ctx, calls, outs, reset in (a, b):
        for call in calls:
            call(None)
        torch.cuda.synchronize()
        assert bep.bep_status(ctx) == 0
        alone.append(bits(outs))
        reset()
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for call_a, call_b in zip(a[1], b[1]):
        call_a(sa)
        call_b(sb)
    torch.cuda.synchronize()
    for (ctx, _, outs, _), want in zip((a, b), alone):
        assert bep.bep_status(ctx) == 0
        got = bits(outs)
        for k in want:
            assert torch.equal(got[k], want[k]), k
