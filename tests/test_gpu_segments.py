"""The three grouped GEMMs on hand-made cu_seqlens tables whose segment lengths
cover every residue of a segment end against the kernels' blocking: the 16-row
K step and 64-row K block of the weight-gradient GEMM (its last block issues
only the steps it holds and zeroes the rest of the last step), and the 128-row
M tile of the forward and input-gradient GEMMs (rows past a segment end belong
to the next segment and must not be written). Compared per segment / weight
row with the binary64 oracle (relative Frobenius, and every element against the
fp32-accumulation bound of ``elementwise``); rows outside every segment keep
their contents."""
import numpy as np
import pytest
import torch

import elementwise as ew
import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
RTOL = 2e-2

# R=2, E=8, B=4 (training), K=2, S=1024: C=2048 slots per rank; H=256, H'=128
R, E, B, K, S, H, HP = 2, 8, 4, 2, 1024, 256, 128
C = S * K
LENGTHS = [
    [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12],                  # rank 0: 78 rows
    [13, 14, 15, 16, 63, 64, 65, 127, 128, 129, 257, 0],      # rank 1: 891 rows
]


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(DEV).view(
        torch.bfloat16)


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def table():
    cu = np.zeros((R, E + B + 1), np.int32)
    for u in range(R):
        cu[u, 1:] = np.cumsum(LENGTHS[u])
    assert cu[:, -1].max() <= C
    return cu


def context(bep, h=H, hp=HP):
    return bep.Context(bep.Config(R, E, B, K, S, h, hp, 0))


def covered(cu):
    """Boolean mask over the R*C receive rows that lie inside some segment."""
    m = np.zeros(R * C, bool)
    for u in range(R):
        m[u * C:u * C + int(cu[u, -1])] = True
    return m


def test_lengths_cover_every_residue():
    flat = [n for row in LENGTHS for n in row if n > 0]
    assert {n % 16 for n in flat} == set(range(16))
    assert {n % 64 for n in flat} >= {0, 1, 15, 16, 63}
    assert {n % 128 for n in flat} >= {0, 1, 127}


def test_forward_on_ragged_segments(lib):
    bep = lib
    ctx = context(bep)
    cu = table()
    recv = synth.tokens_host((R * C, H), 301)
    w_home = synth.weights_host((E, H, HP), 302)
    w_slots = synth.weights_host((R, B, H, HP), 303)
    y = torch.full((R * C, HP), -7.0, dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm(ctx, torch.from_numpy(cu).to(DEV), dev_u16(recv), dev_u16(w_home),
                         dev_u16(w_slots), y)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    ref = oracle.grouped_gemm(recv, w_home, w_slots, cu, E)
    got = oracle.bf16_to_f32(host_u16(y)).astype(np.float64)
    for u in range(R):
        for rho in range(E + B):
            a, b = u * C + int(cu[u, rho]), u * C + int(cu[u, rho + 1])
            if a == b:
                continue
            err = np.linalg.norm(got[a:b] - ref[a:b]) / max(np.linalg.norm(ref[a:b]), 1e-30)
            assert err <= RTOL, (u, rho, b - a, err)
    assert (got[~covered(cu)] == -7.0).all()
    wh, ws = oracle.bf16_to_f32(w_home).astype(np.float64), oracle.bf16_to_f32(w_slots).astype(np.float64)
    worst = ew.gemm_table("fwd", got, ref, oracle.bf16_to_f32(recv).astype(np.float64), cu, E, C,
                          lambda u, rho: wh[rho] if rho < E else ws[u, rho - E])
    print(f"forward on ragged segments: {worst}")


def test_input_gradient_on_ragged_segments(lib):
    bep = lib
    ctx = context(bep)
    cu = table()
    dy = synth.tokens_host((R * C, HP), 311)
    w_home = synth.weights_host((E, H, HP), 312)
    w_slots = synth.weights_host((R, B, H, HP), 313)
    drecv = torch.full((R * C, H), 3.0, dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm_dx(ctx, torch.from_numpy(cu).to(DEV), dev_u16(dy), dev_u16(w_home),
                            dev_u16(w_slots), drecv)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    ref = oracle.grouped_gemm_dx(dy, w_home, w_slots, cu, E)
    got = oracle.bf16_to_f32(host_u16(drecv)).astype(np.float64)
    for u in range(R):
        for rho in range(E + B):
            a, b = u * C + int(cu[u, rho]), u * C + int(cu[u, rho + 1])
            if a == b:
                continue
            err = np.linalg.norm(got[a:b] - ref[a:b]) / max(np.linalg.norm(ref[a:b]), 1e-30)
            assert err <= RTOL, (u, rho, b - a, err)
    assert (got[~covered(cu)] == 3.0).all()
    wh, ws = oracle.bf16_to_f32(w_home).astype(np.float64), oracle.bf16_to_f32(w_slots).astype(np.float64)
    worst = ew.gemm_table("dx", got, ref, oracle.bf16_to_f32(dy).astype(np.float64), cu, E, C,
                          lambda u, rho: wh[rho] if rho < E else ws[u, rho - E])
    print(f"input gradient on ragged segments: {worst}")


@pytest.mark.parametrize("H, HP", [(256, 128), (512, 256)])
@pytest.mark.parametrize("poison", [False, True])
def test_weight_gradient_on_ragged_segments(lib, poison, H, HP):
    """poison=True fills the receive rows outside every segment with +inf: a tail
    step that read them unzeroed would turn a gradient row non-finite. H=512,
    H'=256 runs the weight gradient on SM pairs (256 x 256 tiles, each CTA
    zeroing the tail rows of its own halves); H=256, H'=128 on single CTAs."""
    bep = lib
    ctx = context(bep, H, HP)
    cu = table()
    recv = synth.tokens_host((R * C, H), 321)
    dy = synth.tokens_host((R * C, HP), 322)
    if poison:
        out = ~covered(cu)
        recv[out] = 0x7F80          # bf16 +inf
        dy[out] = 0x7F80
    g0 = synth.normal_host((E, H, HP), 323, 0.5)
    red0 = synth.normal_host((R, B, H, HP), 324, 0.5)
    g = torch.from_numpy(g0).to(DEV)
    red = torch.from_numpy(red0).to(DEV)
    bep.bep_grouped_gemm_dw(ctx, torch.from_numpy(cu).to(DEV), dev_u16(recv), dev_u16(dy), g, red)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    d_home, d_slots = oracle.grouped_gemm_dw(recv, dy, cu, E, B, H, HP)
    gh, rh = g.cpu().numpy().astype(np.float64), red.cpu().numpy().astype(np.float64)
    assert np.isfinite(gh).all() and np.isfinite(rh).all()
    for e in range(E):
        if not d_home[e].any():
            np.testing.assert_array_equal(gh[e], g0[e])
            continue
        err = np.linalg.norm(gh[e] - (g0[e] + d_home[e])) / np.linalg.norm(d_home[e])
        assert err <= RTOL, (e, err)
    for u in range(R):
        for j in range(B):
            if not d_slots[u, j].any():
                np.testing.assert_array_equal(rh[u, j], red0[u, j])
                continue
            err = np.linalg.norm(rh[u, j] - (red0[u, j] + d_slots[u, j])) / np.linalg.norm(d_slots[u, j])
            assert err <= RTOL, (u, j, err)
    worst = ew.dw_table(gh, rh, d_home, d_slots, oracle.bf16_to_f32(recv).astype(np.float64),
                        oracle.bf16_to_f32(dy).astype(np.float64), cu, E, C, g0, red0)
    print(f"weight gradient on ragged segments (H={H}, poison={poison}): {worst}")


def test_weight_gradient_on_many_tiny_segments_sm_pairs(lib):
    """dW on SM pairs (H=512, H'=256) over random tables where most segments hold
    1-15 rows: long runs of units that are a single tail block each, so up to the
    ring's six tail stages are in flight at once and every tail barrier is reused
    many times. Compared per weight row with the binary64 oracle."""
    bep = lib
    R_, E_, B_, K_, S_, H_, HP_ = 4, 64, 16, 4, 96, 512, 256
    C_ = S_ * K_
    rng = np.random.default_rng(17)
    cu = np.zeros((R_, E_ + B_ + 1), np.int32)
    for u in range(R_):
        lens = rng.choice([0, 1, 2, 3, 5, 7, 9, 12, 15, 17, 33], size=E_ + B_,
                          p=[.2, .15, .1, .1, .1, .1, .05, .05, .05, .05, .05])
        while lens.sum() > C_:
            lens[rng.integers(E_ + B_)] //= 2
        cu[u, 1:] = np.cumsum(lens)
    ctx = bep.Context(bep.Config(R_, E_, B_, K_, S_, H_, HP_, 0))
    recv = synth.tokens_host((R_ * C_, H_), 331)
    dy = synth.tokens_host((R_ * C_, HP_), 332)
    g0 = synth.normal_host((E_, H_, HP_), 333, 0.5)
    red0 = synth.normal_host((R_, B_, H_, HP_), 334, 0.5)
    g = torch.from_numpy(g0).to(DEV)
    red = torch.from_numpy(red0).to(DEV)
    bep.bep_grouped_gemm_dw(ctx, torch.from_numpy(cu).to(DEV), dev_u16(recv), dev_u16(dy), g, red)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    d_home, d_slots = oracle.grouped_gemm_dw(recv, dy, cu, E_, B_, H_, HP_)
    gh, rh = g.cpu().numpy().astype(np.float64), red.cpu().numpy().astype(np.float64)
    for e in range(E_):
        if not d_home[e].any():
            np.testing.assert_array_equal(gh[e], g0[e])
            continue
        err = np.linalg.norm(gh[e] - (g0[e] + d_home[e])) / np.linalg.norm(d_home[e])
        assert err <= RTOL, (e, err)
    for u in range(R_):
        for j in range(B_):
            if not d_slots[u, j].any():
                np.testing.assert_array_equal(rh[u, j], red0[u, j])
                continue
            err = np.linalg.norm(rh[u, j] - (red0[u, j] + d_slots[u, j])) / np.linalg.norm(d_slots[u, j])
            assert err <= RTOL, (u, j, err)
    worst = ew.dw_table(gh, rh, d_home, d_slots, oracle.bf16_to_f32(recv).astype(np.float64),
                        oracle.bf16_to_f32(dy).astype(np.float64), cu, E_, C_, g0, red0)
    print(f"weight gradient on tiny segments: {worst}")
