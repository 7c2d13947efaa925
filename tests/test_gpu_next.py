"""GPU parity for the rows beyond the forward/backward step: the gate gradient
of the combine, the SM-budgeted token kernels, and a second (down) projection
that shares the first projection's plan and prefetch slot map."""
import numpy as np
import pytest
import torch

import elementwise as ew
import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
RTOL = 2e-2


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(DEV).view(
        torch.bfloat16)


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def setup(bep, name, target, **kw):
    wl = synth.WORKLOADS[name]
    topk = synth.routing(wl, target, 0)
    ref = oracle.plan(topk, wl.E, wl.B, wl.mode)
    d = dict(R=wl.R, E=wl.E, B=wl.B, K=wl.K, S=wl.S, H=wl.H, Hp=wl.Hp, mode=wl.mode)
    d.update(kw)
    cfg = bep.Config(**d)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, DEV)
    bep.bep_plan(ctx, torch.from_numpy(topk).to(DEV), buf.cu_seqlens, buf.slot_expert, buf.dest,
                 buf.maxvio)
    np.testing.assert_array_equal(buf.dest.cpu().numpy(), ref.dest)
    return wl, ref, ctx, buf


@pytest.mark.parametrize("name,target,D", [("tiny_r2_e8", None, 64), ("train_r8_e64", 10.0, 512),
                                           ("grad_r8_e64", 10.0, 2048)])
def test_combine_dgates(lib, name, target, D):
    bep = lib
    wl, ref, ctx, buf = setup(bep, name, target)
    y = synth.tokens_host((wl.R * wl.C, D), 101)
    dout = synth.tokens_host((wl.R, wl.S, D), 102)
    dg_ref = oracle.combine_dgates(dout, y, ref.dest)
    dg = torch.empty((wl.R, wl.S, wl.K), dtype=torch.float32, device=DEV)
    bep.bep_combine_dgates(ctx, dev_u16(dout), dev_u16(y), buf.dest, dg)
    assert bep.bep_status(ctx) == 0
    got = dg.cpu().numpy().astype(np.float64)
    # fp32 accumulation of D products: error <= D * 2^-24 * sum |products| (loose form)
    yf, df = oracle.bf16_to_f32(y).astype(np.float64), oracle.bf16_to_f32(dout).astype(np.float64)
    mag = np.einsum("rtc,rtkc->rtk", np.abs(df), np.abs(yf[ref.dest]))
    assert (np.abs(got - dg_ref) <= D * 2.0 ** -24 * mag + 1e-30).all()
    assert np.linalg.norm(got - dg_ref) / np.linalg.norm(dg_ref) <= 1e-5


@pytest.mark.parametrize("sms", [1, 32])
def test_comm_sm_budget_gives_identical_results(lib, sms):
    bep = lib
    wl, ref, ctx, buf = setup(bep, "train_r8_e64", 10.0)
    x = synth.tokens_device((wl.R, wl.S, wl.H), 111)
    y = synth.tokens_device((wl.R * wl.C, wl.Hp), 112)
    gates = torch.from_numpy(synth.gates_host(wl.R, wl.S, wl.K, 113)).to(DEV)
    dout = synth.tokens_device((wl.R, wl.S, wl.Hp), 114)

    def run():
        recv = torch.empty((wl.R * wl.C, wl.H), dtype=torch.bfloat16, device=DEV)
        out = torch.empty((wl.R, wl.S, wl.Hp), dtype=torch.bfloat16, device=DEV)
        dy = torch.empty((wl.R * wl.C, wl.Hp), dtype=torch.bfloat16, device=DEV)
        dx = torch.empty((wl.R, wl.S, wl.H), dtype=torch.bfloat16, device=DEV)
        dg = torch.empty((wl.R, wl.S, wl.K), dtype=torch.float32, device=DEV)
        bep.bep_dispatch(ctx, x, buf.dest, recv)
        bep.bep_combine(ctx, y, buf.dest, gates, out)
        bep.bep_combine_bwd(ctx, dout, buf.dest, gates, dy)
        bep.bep_dispatch_bwd(ctx, recv, buf.dest, dx)
        bep.bep_combine_dgates(ctx, dout, y, buf.dest, dg)
        torch.cuda.synchronize()
        return [t.clone() for t in (recv, out, dy, dx, dg)]

    full = run()
    bep.bep_set_comm_sms(ctx, sms)
    capped = run()
    bep.bep_set_comm_sms(ctx, 0)
    assert bep.bep_status(ctx) == 0
    for a, b in zip(full, capped):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    np.testing.assert_array_equal(host_u16(capped[0]), oracle.dispatch(host_u16(x), ref.dest))


def test_second_projection_shares_the_plan(lib):
    """Up projection [E+B, H, H'] then down projection [E+B, H', H] on the same
    cu_seqlens and slot map (a second context with H and H' swapped), then the
    combine on H-wide rows; against the oracle's chain."""
    bep = lib
    wl, ref, ctx, buf = setup(bep, "train_r8_e64", 10.0)
    R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
    ctx2 = bep.Context(bep.Config(R, E, B, K, S, Hp, H, wl.mode))
    x = synth.tokens_host((R, S, H), 121)
    w_up = synth.weights_host((E, H, Hp), 122)
    w_dn = synth.weights_host((E, Hp, H), 123)
    gates = synth.gates_host(R, S, K, 124)
    # oracle chain
    recv_ref = oracle.dispatch(x, ref.dest)
    up_slots = oracle.prefetch(w_up, ref.slot_expert, np.zeros((R, B, H, Hp), np.uint16))
    dn_slots = oracle.prefetch(w_dn, ref.slot_expert, np.zeros((R, B, Hp, H), np.uint16))
    y1 = oracle.f32_to_bf16(oracle.grouped_gemm(recv_ref, w_up, up_slots, ref.cu, E))
    y2 = oracle.f32_to_bf16(oracle.grouped_gemm(y1, w_dn, dn_slots, ref.cu, E))
    out_ref = oracle.bf16_to_f32(oracle.combine(y2, ref.dest, gates)).astype(np.float64)
    # library chain
    w_up_d, w_dn_d = dev_u16(w_up), dev_u16(w_dn)
    up_s = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=DEV)
    dn_s = torch.zeros((R, B, Hp, H), dtype=torch.bfloat16, device=DEV)
    bep.bep_prefetch_weight(ctx, buf.slot_expert, w_up_d, up_s)
    bep.bep_prefetch_weight(ctx2, buf.slot_expert, w_dn_d, dn_s)
    bep.bep_dispatch(ctx, dev_u16(x), buf.dest, buf.recv)
    bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_up_d, up_s, buf.y)
    y2d = torch.empty((R * S * K, H), dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm(ctx2, buf.cu_seqlens, buf.y, w_dn_d, dn_s, y2d)
    out = torch.empty((R, S, H), dtype=torch.bfloat16, device=DEV)
    bep.bep_combine(ctx, y2d, buf.dest, torch.from_numpy(gates).to(DEV), out)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0 and bep.bep_status(ctx2) == 0
    got = oracle.bf16_to_f32(host_u16(out)).astype(np.float64)
    assert np.linalg.norm(got - out_ref) / np.linalg.norm(out_ref) <= RTOL
    # the down projection alone, element by element, on the library's own first output
    y1_gpu = host_u16(buf.y)
    y2_ref = oracle.grouped_gemm(y1_gpu, w_dn, dn_slots, ref.cu, E)
    wd = oracle.bf16_to_f32(w_dn).astype(np.float64)
    wds = oracle.bf16_to_f32(dn_slots).astype(np.float64)
    worst = ew.gemm_table("fwd", oracle.bf16_to_f32(host_u16(y2d)).astype(np.float64), y2_ref,
                          oracle.bf16_to_f32(y1_gpu).astype(np.float64), ref.cu, E, S * K,
                          lambda u, rho: wd[rho] if rho < E else wds[u, rho - E])
    print(f"down projection: {worst}")
