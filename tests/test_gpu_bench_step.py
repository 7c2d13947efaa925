"""The whole step at the full S=8192, E=384 size, queued exactly as the benchmark
queues it (plan, prefetch_weight, dispatch, grouped GEMM, combine, combine
backward, reduce_grad on one side stream), checked against the oracle on
sampled outputs the oracle computes one by one:
  - the plan, in full, bit-exact;
  - prefetch_weight: 8 rows of every slot, bit-exact (oracle copy of those rows);
  - combine backward: 1024 sampled tokens' K destination rows, bit-exact;
  - reduce_grad: 8 rows of every expert gradient and every slot, bit-exact
    (fp32 adds in ascending rank order), plus properties over all elements: every
    consumed slot is zero, every unused slot and every untouched expert unchanged;
  - combine after the GEMM: 48 sampled tokens within the GEMM tolerance of the
    oracle chain (binary64 GEMM rows rounded to bf16, then the oracle combine)."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
GEMM_RTOL = 2e-2


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_sum(t):
    """Order-free fingerprint of a tensor's bit patterns (int64 sum of 32-bit words)."""
    return int(t.contiguous().view(torch.int32).to(torch.int64).sum().item())


@pytest.fixture(scope="module")
def step(lib):
    bep = lib
    torch.cuda.empty_cache()
    wl = synth.WORKLOADS["bench_r8_e384"]
    R, S, K, E, B, H, Hp = wl.R, wl.S, wl.K, wl.E, wl.B, wl.H, wl.Hp
    topk = synth.routing(wl, 10.0, 0)
    ref = oracle.plan(topk, E, B, wl.mode)
    cfg = bep.Config(R, E, B, K, S, H, Hp, wl.mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, DEV, with_grad=True)
    x = synth.tokens_device((R, S, H), 1)
    gates = synth.gates_host(R, S, K, 1)
    dout = synth.tokens_device((R, S, Hp), 2)
    w_home = synth.weights_device((E, H, Hp), 3)
    w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(5)
    g_home = torch.empty((E, H, Hp), dtype=torch.float32, device=DEV).normal_(0.0, 1e-2, generator=gen)
    red = torch.empty((R, B, H, Hp), dtype=torch.float32, device=DEV).normal_(0.0, 1e-3, generator=gen)

    hs = np.sort(np.random.default_rng(7).choice(H, size=8, replace=False))
    hs_t = torch.from_numpy(hs).to(DEV)
    before = {
        "g_rows": g_home[:, hs_t, :].cpu().numpy(),
        "red_rows": red[:, :, hs_t, :].cpu().numpy(),
        "g_sums": [bits_sum(g_home[e]) for e in range(E)],
        "red_sums": [[bits_sum(red[u, j]) for j in range(B)] for u in range(R)],
    }
    stream = torch.cuda.Stream(device=DEV)
    gates_d = torch.from_numpy(gates).to(DEV)
    topk_d = torch.from_numpy(topk).to(DEV)
    torch.cuda.synchronize()
    bep.bep_plan(ctx, topk_d, buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio, stream)
    bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots, stream)
    bep.bep_dispatch(ctx, x, buf.dest, buf.recv, stream)
    bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y, stream)
    bep.bep_combine(ctx, buf.y, buf.dest, gates_d, buf.out, stream)
    bep.bep_combine_bwd(ctx, dout, buf.dest, gates_d, buf.dy, stream)
    bep.bep_reduce_grad(ctx, buf.slot_expert, g_home, red, stream)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx, stream) == 0
    yield dict(wl=wl, ref=ref, buf=buf, x=x, gates=gates, dout=dout, w_home=w_home,
               w_slots=w_slots, g_home=g_home, red=red, hs=hs, hs_t=hs_t, before=before)
    del buf, x, dout, w_home, w_slots, g_home, red
    torch.cuda.empty_cache()


def test_plan(step):
    buf, ref = step["buf"], step["ref"]
    np.testing.assert_array_equal(buf.dest.cpu().numpy(), ref.dest)
    np.testing.assert_array_equal(buf.cu_seqlens.cpu().numpy(), ref.cu)
    np.testing.assert_array_equal(buf.slot_expert.cpu().numpy(), ref.slot_expert)
    assert (ref.slot_expert >= 0).sum() >= 10         # the maxvio-10 routing uses 14 slots


def test_prefetch_weight_sampled_rows(step):
    wl, ref, hs_t = step["wl"], step["ref"], step["hs_t"]
    home_rows = host_u16(step["w_home"][:, hs_t, :])                 # [E, 8, H'] input rows
    want = np.zeros((wl.R, wl.B, len(step["hs"]), wl.Hp), np.uint16)
    oracle.prefetch(home_rows, ref.slot_expert, want)
    got = host_u16(step["w_slots"][:, :, hs_t, :])
    np.testing.assert_array_equal(got, want)


def test_combine_bwd_sampled_tokens(step):
    wl, ref = step["wl"], step["ref"]
    K = wl.K
    toks = np.random.default_rng(3).choice(wl.R * wl.S, size=1024, replace=False)
    d = ref.dest.reshape(-1, K)[toks]
    dout_rows = host_u16(step["dout"].view(-1, wl.Hp)[torch.from_numpy(toks).to(DEV)])
    local = np.arange(len(toks) * K, dtype=np.int32).reshape(1, len(toks), K)
    g = step["gates"].reshape(-1, K)[toks].reshape(1, len(toks), K)
    want = oracle.combine_bwd(dout_rows.reshape(1, len(toks), wl.Hp), local, g)
    got = host_u16(step["buf"].dy[torch.from_numpy(d.ravel().astype(np.int64)).to(DEV)])
    np.testing.assert_array_equal(got, want)


def test_reduce_grad_sampled_rows_and_whole_buffers(step):
    wl, ref, hs_t, before = step["wl"], step["ref"], step["hs_t"], step["before"]
    g_rows = np.ascontiguousarray(before["g_rows"])        # [E, 8, H'] fp32, before the call
    red_rows = np.ascontiguousarray(before["red_rows"])    # [R, B, 8, H']
    oracle.reduce_grad(g_rows, red_rows, ref.slot_expert)
    got_g = step["g_home"][:, hs_t, :].cpu().numpy()
    got_red = step["red"][:, :, hs_t, :].cpu().numpy()
    np.testing.assert_array_equal(got_g.view(np.uint32), g_rows.view(np.uint32))
    np.testing.assert_array_equal(got_red.view(np.uint32), red_rows.view(np.uint32))
    se = ref.slot_expert
    touched = set(int(e) for e in se[se >= 0])
    for u in range(wl.R):
        for j in range(wl.B):
            if se[u, j] >= 0:
                assert not step["red"][u, j].view(torch.int32).any().item(), (u, j)
            else:
                assert bits_sum(step["red"][u, j]) == before["red_sums"][u][j], (u, j)
    for e in range(wl.E):
        if e not in touched:
            assert bits_sum(step["g_home"][e]) == before["g_sums"][e], e


def test_combine_after_gemm_sampled_tokens(step):
    wl, ref = step["wl"], step["ref"]
    R, S, K, E, H, Hp, C = wl.R, wl.S, wl.K, wl.E, wl.H, wl.Hp, wl.C
    toks = np.random.default_rng(4).choice(R * S, size=48, replace=False)
    x_rows = host_u16(step["x"].view(-1, H)[torch.from_numpy(toks).to(DEV)])   # [n, H]
    d = ref.dest.reshape(-1, K)[toks]
    # the weight row serving each (token, k): its receive row's segment on its rank
    by_expert = {}
    for i in range(len(toks)):
        for k in range(K):
            u, r = divmod(int(d[i, k]), C)
            rho = int(np.searchsorted(ref.cu[u], r, side="right") - 1)
            e = oracle.weight_row_of(rho, u, E, ref.slot_expert)
            by_expert.setdefault(e, []).append((i, k))
    y_ref = np.zeros((len(toks) * K, Hp), np.uint16)
    for e, pairs in by_expert.items():
        rows = np.array([i for i, _ in pairs])
        y = oracle.gemm_rows(x_rows[rows], host_u16(step["w_home"][e]))
        yb = oracle.f32_to_bf16(y.astype(np.float32))
        for (i, k), v in zip(pairs, yb):
            y_ref[i * K + k] = v
    local = np.arange(len(toks) * K, dtype=np.int32).reshape(1, len(toks), K)
    g = step["gates"].reshape(-1, K)[toks].reshape(1, len(toks), K)
    want = oracle.bf16_to_f32(oracle.combine(y_ref, local, g)[0]).astype(np.float64)
    got = oracle.bf16_to_f32(
        host_u16(step["buf"].out.view(-1, Hp)[torch.from_numpy(toks).to(DEV)])).astype(np.float64)
    for i in range(len(toks)):
        err = np.linalg.norm(got[i] - want[i]) / max(np.linalg.norm(want[i]), 1e-30)
        assert err <= GEMM_RTOL, (int(toks[i]), err)
