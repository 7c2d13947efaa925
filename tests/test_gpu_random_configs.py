"""The whole chain on seeded random configurations against the oracle.

Each case draws R, E/R, K, S, H, H', the mode and B, and a routing from a
random Dirichlet popularity, so that the shapes reach paths the named workloads
do not: R = 1 and odd R, K = 1, one token per rank, every N tile width of the
forward and dX GEMMs, H and H' that are and are not multiples of 256 (dW on SM
pairs or on single CTAs), inference with and without overflow rows.

Checked through the C ABI:
  plan (cu_seqlens, slot map, dest, maxvio), prefetch, dispatch, combine
  backward, dispatch backward and reduce_grad bit for bit;
  forward and dX GEMMs per segment, dW per weight row (training; both the
  accumulating and the overwriting form), and the combined output, each within
  2e-2 relative of binary64; the three GEMMs also element by element against
  the fp32-accumulation bound of ``elementwise``.
"""
import numpy as np
import pytest
import torch

import elementwise as ew
import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
RTOL = 2e-2
N_CASES = 40


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(DEV).view(
        torch.bfloat16)


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.choice([1, 2, 3, 4, 5, 8]))
    G = int(rng.integers(1, 9))
    E = R * G
    K = int(rng.integers(1, min(8, E) + 1))
    S = int(rng.choice([1, 7, 64, 129, 300]))
    H = 64 * int(rng.choice([1, 2, 3, 4, 8, 12]))
    Hp = 64 * int(rng.choice([1, 2, 3, 4, 8]))
    mode = 1 if (G >= 2 and rng.random() < 0.35) else 0
    B = (1 if rng.random() < 0.5 else int(rng.integers(1, G))) if mode == 1 else G
    alpha = float(rng.choice([0.3, 1.0, 10.0]))
    pop = rng.dirichlet(np.full(E, alpha))
    if mode == 1 and rng.random() < 0.7:
        # equally hot experts on home group 0: the ranks it feeds need more of its experts
        # than they have slots, and the rest overflow onto the home rows
        pop[:G] = 200.0 * pop.sum() / E
    pop = np.maximum(pop, 1e-9)
    topk = synth.gumbel_topk(R, S, K, pop / pop.sum(), 2000 + seed)
    return dict(R=R, E=E, B=B, K=K, S=S, H=H, Hp=Hp, mode=mode), topk


def rel(got, ref):
    return np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_whole_chain_on_random_config(lib, seed):
    c, topk = draw(seed)
    run_chain(lib, c, topk, seed)


# Near the library's limits (R <= 64, E <= 2048, K <= 32): many ranks, thousands of
# experts, a wide top-K, and an inference batch whose hot group forces overflow rows.
LIMIT_CASES = [
    dict(R=64, E=2048, B=32, K=32, S=8, H=64, Hp=64, mode=0),
    dict(R=16, E=512, B=32, K=16, S=32, H=128, Hp=128, mode=0),
    dict(R=16, E=512, B=2, K=16, S=32, H=128, Hp=64, mode=1),
]


@pytest.mark.parametrize("case", range(len(LIMIT_CASES)))
def test_whole_chain_near_size_limits(lib, case):
    c = LIMIT_CASES[case]
    G = c["E"] // c["R"]
    rng = np.random.default_rng(77 + case)
    pop = rng.dirichlet(np.full(c["E"], 0.5))
    if c["mode"] == 1:
        pop[:G] = 200.0 * pop.sum() / c["E"]
    topk = synth.gumbel_topk(c["R"], c["S"], c["K"], pop / pop.sum(), 3000 + case)
    run_chain(lib, c, topk, 100 + case)


def run_chain(bep, c, topk, seed):
    R, E, B, K, S, H, Hp, mode = (c[k] for k in ("R", "E", "B", "K", "S", "H", "Hp", "mode"))
    C = S * K
    ref = oracle.plan(topk, E, B, mode)
    assert oracle.check_plan(topk, E, B, mode, ref.cu, ref.slot_expert, ref.dest) == 0

    cfg = bep.Config(R, E, B, K, S, H, Hp, mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, DEV, with_grad=True)
    x = synth.tokens_host((R, S, H), 10 + seed)
    gates = synth.gates_host(R, S, K, 20 + seed)
    w_home = synth.weights_host((E, H, Hp), 30 + seed)
    dout = synth.tokens_host((R, S, Hp), 40 + seed)
    w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=DEV)
    w_home_d, gates_d = dev_u16(w_home), torch.from_numpy(gates).to(DEV)

    # forward: plan, prefetch, dispatch, grouped GEMM, combine
    bep.forward(ctx, buf, torch.from_numpy(topk).to(DEV), dev_u16(x), gates_d, w_home_d, w_slots)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0, c
    np.testing.assert_array_equal(buf.cu_seqlens.cpu().numpy(), ref.cu)
    np.testing.assert_array_equal(buf.slot_expert.cpu().numpy(), ref.slot_expert)
    np.testing.assert_array_equal(buf.dest.cpu().numpy(), ref.dest)
    assert float(buf.maxvio.item()) == ref.maxvio
    slots_ref = oracle.prefetch(w_home, ref.slot_expert, np.zeros((R, B, H, Hp), np.uint16))
    used = ref.slot_expert >= 0
    np.testing.assert_array_equal(host_u16(w_slots)[used], slots_ref[used])
    recv_ref = oracle.dispatch(x, ref.dest)
    np.testing.assert_array_equal(host_u16(buf.recv), recv_ref)
    y_ref = oracle.grouped_gemm(recv_ref, w_home, slots_ref, ref.cu, E)
    y = oracle.bf16_to_f32(host_u16(buf.y)).astype(np.float64)
    segs = [(u, rho, int(ref.cu[u, rho]), int(ref.cu[u, rho + 1]))
            for u in range(R) for rho in range(E + B) if ref.cu[u, rho + 1] > ref.cu[u, rho]]
    for u, rho, a, b in segs:
        assert rel(y[u * C + a:u * C + b], y_ref[u * C + a:u * C + b]) <= RTOL, (c, u, rho)
    wh = oracle.bf16_to_f32(w_home).astype(np.float64)
    ws = oracle.bf16_to_f32(slots_ref).astype(np.float64)
    weight = lambda u, rho: wh[rho] if rho < E else ws[u, rho - E]      # noqa: E731
    recv_f = oracle.bf16_to_f32(recv_ref).astype(np.float64)
    ew.gemm_table("fwd", y, y_ref, recv_f, ref.cu, E, C, weight)
    out_ref = oracle.bf16_to_f32(oracle.combine(oracle.f32_to_bf16(y_ref), ref.dest, gates))
    assert rel(oracle.bf16_to_f32(host_u16(buf.out)).astype(np.float64), out_ref) <= RTOL, c
    # the combine itself, bit for bit, on the GPU's own Y
    np.testing.assert_array_equal(host_u16(buf.out), oracle.combine(host_u16(buf.y), ref.dest, gates))

    # backward: combine backward, dX GEMM, dispatch backward
    bep.bep_combine_bwd(ctx, dev_u16(dout), buf.dest, gates_d, buf.dy)
    drecv = torch.empty((R * C, H), dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm_dx(ctx, buf.cu_seqlens, buf.dy, w_home_d, w_slots, drecv)
    dx = torch.empty((R, S, H), dtype=torch.bfloat16, device=DEV)
    bep.bep_dispatch_bwd(ctx, drecv, buf.dest, dx)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0, c
    dy_ref = oracle.combine_bwd(dout, ref.dest, gates)
    np.testing.assert_array_equal(host_u16(buf.dy), dy_ref)
    dr_ref = oracle.grouped_gemm_dx(dy_ref, w_home, slots_ref, ref.cu, E)
    dr = oracle.bf16_to_f32(host_u16(drecv)).astype(np.float64)
    for u, rho, a, b in segs:
        assert rel(dr[u * C + a:u * C + b], dr_ref[u * C + a:u * C + b]) <= RTOL, (c, u, rho)
    dy_f = oracle.bf16_to_f32(dy_ref).astype(np.float64)
    ew.gemm_table("dx", dr, dr_ref, dy_f, ref.cu, E, C, weight)
    np.testing.assert_array_equal(host_u16(dx), oracle.dispatch_bwd(host_u16(drecv), ref.dest))

    if mode == 0 and H % 128 != 0:
        # the weight gradient needs whole 128-row blocks of H: refused on the host
        g = torch.zeros((E, H, Hp), dtype=torch.float32, device=DEV)
        red = torch.zeros((R, B, H, Hp), dtype=torch.float32, device=DEV)
        with pytest.raises(bep.BepError):
            bep.bep_grouped_gemm_dw(ctx, buf.cu_seqlens, buf.recv, buf.dy, g, red)
        with pytest.raises(bep.BepError):
            bep.bep_grouped_gemm_dw_overwrite(ctx, buf.cu_seqlens, buf.recv, buf.dy, g, red)
    elif mode == 0:
        # dW into the gradients, then reduce_grad folds the replica rows into the home rows
        g0 = synth.normal_host((E, H, Hp), 50 + seed, 0.5)
        red0 = synth.normal_host((R, B, H, Hp), 60 + seed, 0.5)
        g, red = torch.from_numpy(g0).to(DEV), torch.from_numpy(red0).to(DEV)
        bep.bep_grouped_gemm_dw(ctx, buf.cu_seqlens, buf.recv, buf.dy, g, red)
        torch.cuda.synchronize()
        assert bep.bep_status(ctx) == 0, c
        d_home, d_slots = oracle.grouped_gemm_dw(recv_ref, dy_ref, ref.cu, E, B, H, Hp)
        gh, rh = g.cpu().numpy(), red.cpu().numpy()
        for e in range(E):
            if d_home[e].any():
                err = np.linalg.norm(gh[e] - (g0[e] + d_home[e])) / np.linalg.norm(d_home[e])
                assert err <= RTOL, (c, e, err)
            else:
                np.testing.assert_array_equal(gh[e], g0[e])
        for u in range(R):
            for j in range(B):
                if d_slots[u, j].any():
                    err = np.linalg.norm(rh[u, j] - (red0[u, j] + d_slots[u, j])) / np.linalg.norm(d_slots[u, j])
                    assert err <= RTOL, (c, u, j, err)
                else:
                    np.testing.assert_array_equal(rh[u, j], red0[u, j])
        ew.dw_table(gh, rh, d_home, d_slots, recv_f, dy_f, ref.cu, E, C, g0, red0)
        # the overwriting form on poisoned buffers: home rows written (zeros where the home
        # segment is empty), used slots written, the other slots untouched
        gw = torch.full((E, H, Hp), 7.0, dtype=torch.float32, device=DEV)
        rw = torch.full((R, B, H, Hp), 7.0, dtype=torch.float32, device=DEV)
        bep.bep_grouped_gemm_dw_overwrite(ctx, buf.cu_seqlens, buf.recv, buf.dy, gw, rw)
        torch.cuda.synchronize()
        assert bep.bep_status(ctx) == 0, c
        gwh, rwh = gw.cpu().numpy(), rw.cpu().numpy()
        for e in range(E):
            if d_home[e].any():
                err = np.linalg.norm(gwh[e] - d_home[e]) / np.linalg.norm(d_home[e])
                assert err <= RTOL, (c, e, err)
            else:
                assert (gwh[e] == 0).all(), (c, e)
        for u in range(R):
            for j in range(B):
                if ref.slot_expert[u, j] >= 0:
                    err = np.linalg.norm(rwh[u, j] - d_slots[u, j]) / np.linalg.norm(d_slots[u, j])
                    assert err <= RTOL, (c, u, j, err)
                else:
                    assert (rwh[u, j] == 7.0).all(), (c, u, j)
        ew.dw_table(gwh, rwh, d_home, d_slots, recv_f, dy_f, ref.cu, E, C)
        del gw, rw
        g_ref, red_ref = gh.copy(), rh.copy()
        oracle.reduce_grad(g_ref, red_ref, ref.slot_expert)
        bep.bep_reduce_grad(ctx, buf.slot_expert, g, red)
        torch.cuda.synchronize()
        assert bep.bep_status(ctx) == 0, c
        np.testing.assert_array_equal(g.cpu().numpy(), g_ref)
        np.testing.assert_array_equal(red.cpu().numpy(), red_ref)
