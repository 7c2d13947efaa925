"""Exact pins of the three grouped GEMMs, bit for bit, on inputs where bf16 x bf16
products summed in fp32 are exact:
  - forward and input gradient with permutation weights: W_e[h, h'] = 1 where
    h = (h' + shift_e) mod H, else 0. Each output is a single input element, so
    Y[row] is recv[row] with its columns permuted, and dRecv[row] scatters dY[row]
    back; any slip in weight-row selection (home row, prefetch slot, overflow),
    operand orientation or segment bounds shows as a wrong bit pattern;
  - weight gradient with one-hot receive rows and small-integer dY: dW[h, :] is an
    integer sum of the dY rows whose one-hot column is h (well below 2^24).
The oracle (binary64) computes the expected values, which are exactly
representable; the closed forms above are asserted too. Small workload in full,
and the S=8192, E=384 workload on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16_ONE = 0x3F80


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(DEV).view(
        torch.bfloat16)


def nz(a):
    """bf16 bit patterns with -0 written as +0: a sum of signed zeros may carry either sign."""
    a = np.array(a, np.uint16)
    a[a == 0x8000] = 0
    return a


def shifts(E, H):
    return (np.arange(E, dtype=np.int64) * 37 + 5) % H


def perm_weights_device(E, H, Hp):
    """[E, H, H'] bf16 with a single 1.0 per column: row (h' + shift_e) mod H."""
    w = torch.zeros((E, H, Hp), dtype=torch.bfloat16, device=DEV)
    sh = torch.from_numpy(shifts(E, H)).to(DEV)
    cols = torch.arange(Hp, device=DEV)
    e_idx = torch.arange(E, device=DEV)[:, None].expand(E, Hp)
    rows = (cols[None, :] + sh[:, None]) % H
    w[e_idx, rows, cols[None, :].expand(E, Hp)] = 1.0
    return w


def planned(bep, name, target):
    wl = synth.WORKLOADS[name]
    topk = synth.routing(wl, target, 0)
    ref = oracle.plan(topk, wl.E, wl.B, wl.mode)
    cfg = bep.Config(wl.R, wl.E, wl.B, wl.K, wl.S, wl.H, wl.Hp, wl.mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, DEV, with_grad=True)
    bep.bep_plan(ctx, torch.from_numpy(topk).to(DEV), buf.cu_seqlens, buf.slot_expert, buf.dest,
                 buf.maxvio)
    np.testing.assert_array_equal(buf.cu_seqlens.cpu().numpy(), ref.cu)
    np.testing.assert_array_equal(buf.slot_expert.cpu().numpy(), ref.slot_expert)
    return wl, ref, ctx, buf


def weight_rows_of_receive_rows(ref, wl):
    """For every receive row, the home expert whose weights serve its segment."""
    C, E = wl.C, wl.E
    out = np.empty(wl.R * C, np.int64)
    for u in range(wl.R):
        for rho in range(E + wl.B):
            a, b = int(ref.cu[u, rho]), int(ref.cu[u, rho + 1])
            if b > a:
                out[u * C + a:u * C + b] = oracle.weight_row_of(rho, u, E, ref.slot_expert)
    return out


def test_forward_permutation_weights_exact(lib):
    bep = lib
    wl, ref, ctx, buf = planned(bep, "train_r8_e64", 10.0)
    H, Hp = wl.H, wl.Hp
    x = synth.tokens_host((wl.R, wl.S, H), 501)
    w_home = perm_weights_device(wl.E, H, Hp)
    w_slots = torch.zeros((wl.R, wl.B, H, Hp), dtype=torch.bfloat16, device=DEV)
    bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots)
    bep.bep_dispatch(ctx, dev_u16(x), buf.dest, buf.recv)
    bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    recv_ref = oracle.dispatch(x, ref.dest)
    w_home_h = host_u16(w_home)
    w_slots_h = oracle.prefetch(w_home_h, ref.slot_expert,
                                np.zeros((wl.R, wl.B, H, Hp), np.uint16))
    y_ref = oracle.f32_to_bf16(oracle.grouped_gemm(recv_ref, w_home_h, w_slots_h, ref.cu, wl.E)
                               .astype(np.float32))
    # the closed form: a column permutation of the receive rows
    e_of = weight_rows_of_receive_rows(ref, wl)
    cols = (np.arange(Hp)[None, :] + shifts(wl.E, H)[e_of][:, None]) % H
    np.testing.assert_array_equal(nz(y_ref), nz(np.take_along_axis(recv_ref, cols, axis=1)))
    np.testing.assert_array_equal(nz(host_u16(buf.y)), nz(y_ref))


def test_input_gradient_permutation_weights_exact(lib):
    bep = lib
    wl, ref, ctx, buf = planned(bep, "train_r8_e64", 1.0)
    H, Hp = wl.H, wl.Hp
    dy = synth.tokens_host((wl.R * wl.C, Hp), 502)
    w_home = perm_weights_device(wl.E, H, Hp)
    w_slots = torch.zeros((wl.R, wl.B, H, Hp), dtype=torch.bfloat16, device=DEV)
    bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots)
    drecv = torch.empty((wl.R * wl.C, H), dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm_dx(ctx, buf.cu_seqlens, dev_u16(dy), w_home, w_slots, drecv)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    w_home_h = host_u16(w_home)
    w_slots_h = oracle.prefetch(w_home_h, ref.slot_expert,
                                np.zeros((wl.R, wl.B, H, Hp), np.uint16))
    d_ref = oracle.f32_to_bf16(oracle.grouped_gemm_dx(dy, w_home_h, w_slots_h, ref.cu, wl.E)
                               .astype(np.float32))
    # the closed form: dY scattered to columns (h' + shift) mod H, zero elsewhere
    e_of = weight_rows_of_receive_rows(ref, wl)
    want = np.zeros((wl.R * wl.C, H), np.uint16)
    cols = (np.arange(Hp)[None, :] + shifts(wl.E, H)[e_of][:, None]) % H
    np.put_along_axis(want, cols, dy, axis=1)
    np.testing.assert_array_equal(nz(d_ref), nz(want))
    np.testing.assert_array_equal(nz(host_u16(drecv)), nz(want))


def one_hot_rows(n, H, seed):
    c = np.random.default_rng(seed).integers(0, H, size=n)
    a = np.zeros((n, H), np.uint16)
    a[np.arange(n), c] = BF16_ONE
    return a, c


def small_int_bf16(shape, seed):
    v = np.random.default_rng(seed).integers(-8, 9, size=shape).astype(np.float32)
    return oracle.f32_to_bf16(v), v


def test_weight_gradient_one_hot_rows_exact(lib):
    bep = lib
    wl, ref, ctx, buf = planned(bep, "train_r8_e64", 10.0)
    H, Hp, n = wl.H, wl.Hp, wl.R * wl.C
    recv, c = one_hot_rows(n, H, 503)
    dy, dy_f = small_int_bf16((n, Hp), 504)
    g0 = np.random.default_rng(505).integers(-4, 5, size=(wl.E, H, Hp)).astype(np.float32)
    red0 = np.random.default_rng(506).integers(-4, 5, size=(wl.R, wl.B, H, Hp)).astype(np.float32)
    g = torch.from_numpy(g0).to(DEV)
    red = torch.from_numpy(red0).to(DEV)
    bep.bep_grouped_gemm_dw(ctx, buf.cu_seqlens, dev_u16(recv), dev_u16(dy), g, red)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    d_home, d_slots = oracle.grouped_gemm_dw(recv, dy, ref.cu, wl.E, wl.B, H, Hp)
    # the closed form for one home row: the dY rows of its segments, binned by one-hot column
    e = int(np.argmax([np.abs(d_home[i]).sum() for i in range(wl.E)]))
    want_e = np.zeros((H, Hp))
    for u in range(wl.R):
        a, b = int(ref.cu[u, e]), int(ref.cu[u, e + 1])
        np.add.at(want_e, c[u * wl.C + a:u * wl.C + b], dy_f[u * wl.C + a:u * wl.C + b])
    np.testing.assert_array_equal(d_home[e], want_e)
    np.testing.assert_array_equal(g.cpu().numpy(), (g0 + d_home).astype(np.float32))
    np.testing.assert_array_equal(red.cpu().numpy(), (red0 + d_slots).astype(np.float32))


@pytest.mark.parametrize("target", [0.2, 1.0, 10.0, 20.0])
def test_forward_and_weight_gradient_exact_at_bench_size_sampled(lib, target):
    """S=8192, E=384: forward with permutation weights on sampled rows of every rank's
    first, last and remote segments; weight gradient with one-hot rows on sampled
    rows of sampled home experts and slots."""
    bep = lib
    torch.cuda.empty_cache()
    wl, ref, ctx, buf = planned(bep, "bench_r8_e384", target)
    R, C, E, B, H, Hp = wl.R, wl.C, wl.E, wl.B, wl.H, wl.Hp
    n = R * C
    rng = np.random.default_rng(507)
    x = synth.tokens_device((R, wl.S, H), 508)
    w_home = perm_weights_device(E, H, Hp)
    w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=DEV)
    bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots)
    bep.bep_dispatch(ctx, x, buf.dest, buf.recv)
    bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    inv = np.empty(n, np.int64)
    inv[ref.dest.ravel()] = np.arange(R * wl.S * wl.K) // wl.K      # receive row -> token
    sh = shifts(E, H)
    w_cache = {}
    for u in range(R):
        segs = [rho for rho in range(E + B) if ref.cu[u, rho + 1] > ref.cu[u, rho]]
        remote = [rho for rho in segs if rho >= E or rho // (E // R) != u]
        for rho in sorted(set(segs[:1] + segs[-1:] + remote[:6])):
            a, b = int(ref.cu[u, rho]), int(ref.cu[u, rho + 1])
            rows = np.array(sorted(set([a, b - 1] + list(rng.integers(a, b, size=2)))), np.int64)
            gi = u * C + rows
            e = oracle.weight_row_of(rho, u, E, ref.slot_expert)
            if e not in w_cache:
                w_cache.clear()
                w_cache[e] = host_u16(w_home[e])
            a_rows = host_u16(x.view(-1, H)[torch.from_numpy(inv[gi]).to(DEV)])
            y_ref = oracle.f32_to_bf16(oracle.gemm_rows(a_rows, w_cache[e]).astype(np.float32))
            np.testing.assert_array_equal(nz(y_ref), nz(a_rows[:, (np.arange(Hp) + sh[e]) % H]))
            np.testing.assert_array_equal(nz(host_u16(buf.y[torch.from_numpy(gi).to(DEV)])), nz(y_ref))
    del x, w_home, w_slots
    torch.cuda.empty_cache()

    # weight gradient: one-hot receive rows, small-integer dY, zero-initialised gradients
    c = torch.randint(0, H, (n,), generator=torch.Generator(device=DEV).manual_seed(509), device=DEV)
    recv = torch.zeros((n, H), dtype=torch.bfloat16, device=DEV)
    recv[torch.arange(n, device=DEV), c] = 1.0
    dy = torch.randint(-8, 9, (n, Hp), generator=torch.Generator(device=DEV).manual_seed(510),
                       device=DEV).to(torch.bfloat16)
    g = torch.zeros((E, H, Hp), dtype=torch.float32, device=DEV)
    red = torch.zeros((R, B, H, Hp), dtype=torch.float32, device=DEV)
    bep.bep_grouped_gemm_dw(ctx, buf.cu_seqlens, recv, dy, g, red)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    c_h = c.cpu().numpy()
    del recv
    segs = [(u, rho) for u in range(R) for rho in range(E + B) if ref.cu[u, rho + 1] > ref.cu[u, rho]]
    home = [s for s in segs if s[1] < E]
    slots = [s for s in segs if s[1] >= E]
    pick = [home[i] for i in rng.choice(len(home), size=6, replace=False)] + slots[:6]
    for u, rho in pick:
        a, b = u * C + int(ref.cu[u, rho]), u * C + int(ref.cu[u, rho + 1])
        hs = np.unique(np.concatenate([c_h[a:a + 2], rng.integers(0, H, size=2)]))
        # rows hs of this segment's dW = (its receive rows restricted to columns hs)^T dY:
        # the oracle's weight gradient on those columns of the one-hot rows
        seg_recv = np.zeros((b - a, len(hs)), np.uint16)
        hit = np.searchsorted(hs, c_h[a:b])
        on = (hit < len(hs)) & (hs[np.minimum(hit, len(hs) - 1)] == c_h[a:b])
        seg_recv[np.nonzero(on)[0], hit[on]] = BF16_ONE
        seg_dy = host_u16(dy[a:b])
        cu1 = np.array([[0, b - a]], np.int32)
        dw, _ = oracle.grouped_gemm_dw(seg_recv, seg_dy, cu1, 1, 0, len(hs), Hp)
        hs_t = torch.from_numpy(hs).to(DEV)
        got = (g[rho, hs_t] if rho < E else red[u, rho - E, hs_t]).cpu().numpy()
        np.testing.assert_array_equal(got, dw[0].astype(np.float32))
    del dy, g, red
    torch.cuda.empty_cache()


@pytest.mark.parametrize("target", [1.0, 20.0])
def test_overflow_rows_exact_at_inference_size_sampled(lib, target):
    """S=512, B=4 < E/R, hot experts on group 0 (maxvio 1 and 20): segments of remote
    experts beyond the B slots are overflow rows that read the home weights in place.
    Forward and input gradient with permutation weights, exact on sampled rows of
    every rank's overflow, slot and first home segments."""
    bep = lib
    torch.cuda.empty_cache()
    wl, ref, ctx, buf = planned(bep, "infer_r8_e384_b4", target)
    R, C, E, B, H, Hp, G = wl.R, wl.C, wl.E, wl.B, wl.H, wl.Hp, wl.E // wl.R
    rng = np.random.default_rng(511)
    x = synth.tokens_device((R, wl.S, H), 512)
    dy = synth.tokens_device((R * C, Hp), 513)
    w_home = perm_weights_device(E, H, Hp)
    w_slots = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=DEV)
    bep.bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots)
    bep.bep_dispatch(ctx, x, buf.dest, buf.recv)
    bep.bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y)
    drecv = torch.empty((R * C, H), dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm_dx(ctx, buf.cu_seqlens, dy, w_home, w_slots, drecv)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    inv = np.empty(R * C, np.int64)
    inv[ref.dest.ravel()] = np.arange(R * wl.S * wl.K) // wl.K
    sh = shifts(E, H)
    overflow_seen = 0
    for u in range(R):
        segs = [rho for rho in range(E + B) if ref.cu[u, rho + 1] > ref.cu[u, rho]]
        overflow = [rho for rho in segs if rho < E and rho // G != u]
        slots = [rho for rho in segs if rho >= E]
        home = [rho for rho in segs if rho < E and rho // G == u]
        overflow_seen += len(overflow)
        for rho in overflow[:6] + slots[:2] + home[:1]:
            a, b = int(ref.cu[u, rho]), int(ref.cu[u, rho + 1])
            rows = np.array(sorted(set([a, b - 1] + list(rng.integers(a, b, size=2)))), np.int64)
            gi = torch.from_numpy(u * C + rows).to(DEV)
            e = oracle.weight_row_of(rho, u, E, ref.slot_expert)
            w = host_u16(w_home[e])
            a_rows = host_u16(x.view(-1, H)[torch.from_numpy(inv[u * C + rows]).to(DEV)])
            y_ref = oracle.f32_to_bf16(oracle.gemm_rows(a_rows, w).astype(np.float32))
            np.testing.assert_array_equal(nz(y_ref), nz(a_rows[:, (np.arange(Hp) + sh[e]) % H]))
            np.testing.assert_array_equal(nz(host_u16(buf.y[gi])), nz(y_ref))
            dy_rows = host_u16(dy[gi])
            d_ref = oracle.f32_to_bf16(oracle.gemm_rows(dy_rows, np.ascontiguousarray(w.T))
                                       .astype(np.float32))
            np.testing.assert_array_equal(nz(host_u16(drecv[gi])), nz(d_ref))
    assert overflow_seen > 0      # the routing does produce overflow rows
    del x, dy, w_home, w_slots, drecv
    torch.cuda.empty_cache()
