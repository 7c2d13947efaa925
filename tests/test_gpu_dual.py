"""The forward GEMM's two-m-tile units, on hand-made cu_seqlens tables.

Segments of 768 rows or more run in a launch of their own with two 128-row
m-tiles per unit sharing each weight stage; the other segments run in the usual
one-m-tile launch. Every two-m-tile unit runs both m-tiles at M=128: a unit's
second m-tile may be ragged, down to one row, or lie wholly past the segment end,
on rows whose results are never stored (the next segment's, or past the end of
the tensor). These tables mix both kinds with every tail case: an even number of
m-tiles, an odd number (the last unit's second m-tile lies past the segment), a
second m-tile of at most 64 rows, a first m-tile of at most 64 rows, a segment
that ends at the end of the tensor, and short segments. Compared with the binary64 oracle in full (relative Frobenius per
segment and every element against the fp32-accumulation bound), exactly with
permutation weights, rows outside every segment untouched, and the
two-pointer GEMM equal bit for bit to the VM GEMM on materialised views. The
input-gradient GEMM takes the same two launches and is checked the same way."""
import numpy as np
import pytest
import torch

import elementwise as ew
import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
RTOL = 2e-2

# R=2, E=4 (2 home experts per rank), B=2, K=2, S=4096: C=8192 rows per rank.
# H=2048 (the reduction length) and H'=256 (one 256-column tile): the conditions
# under which the two-m-tile launch runs. MIN_ROWS is its threshold.
R, E, B, K, S, H, HP = 2, 4, 2, 2, 4096, 2048, 256
C = S * K
MIN_ROWS = 768
LENGTHS = [
    [2048, 2177, 1500, 2100, 300, 64],      # 16 m-tiles; 1-row second tile; short; 52-row unit
    [2113, 2276, 0, 1, 1752, 2050],         # 65-row one-tile unit; 100-row second tile; 1; 2-row unit
]


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(DEV).view(
        torch.bfloat16)


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def nz(a):
    """bf16 bit patterns with -0 written as +0: a sum of signed zeros may carry either sign."""
    a = np.array(a, np.uint16)
    a[a == 0x8000] = 0
    return a


def table():
    cu = np.zeros((R, E + B + 1), np.int32)
    for u in range(R):
        cu[u, 1:] = np.cumsum(LENGTHS[u])
    assert cu[:, -1].max() <= C
    return cu


def covered(cu):
    m = np.zeros(R * C, bool)
    for u in range(R):
        m[u * C:u * C + int(cu[u, -1])] = True
    return m


def test_lengths_reach_both_launches():
    assert table()[:, -1].max() <= C
    flat = [n for row in LENGTHS for n in row if n > 0]
    long_ = [n for n in flat if n >= MIN_ROWS]
    assert any((n + 127) // 128 % 2 == 0 for n in long_)     # even m-tile count
    assert any((n + 127) // 128 % 2 == 1 for n in long_)     # odd: a second m-tile past the segment
    assert any(0 < n % 256 - 128 <= 64 for n in long_)       # second m-tile <= 64 rows
    assert any(0 < n % 256 <= 64 for n in long_)             # first m-tile <= 64 rows
    assert any(MIN_ROWS <= n < 2048 for n in long_)          # long, below the earlier 2,048 threshold
    assert any(0 < n < MIN_ROWS for n in flat)               # the one-m-tile launch
    assert table()[-1, -1] == C and LENGTHS[-1][-1] >= MIN_ROWS   # ends at the end of the tensor


def test_forward_two_mtile_units_against_binary64(lib):
    bep = lib
    ctx = bep.Context(bep.Config(R, E, B, K, S, H, HP, 0))
    cu = table()
    recv = synth.tokens_host((R * C, H), 701)
    w_home = synth.weights_host((E, H, HP), 702)
    w_slots = synth.weights_host((R, B, H, HP), 703)
    y = torch.full((R * C, HP), -5.0, dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm(ctx, torch.from_numpy(cu).to(DEV), dev_u16(recv), dev_u16(w_home),
                         dev_u16(w_slots), y)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    ref = oracle.grouped_gemm(recv, w_home, w_slots, cu, E)
    got = oracle.bf16_to_f32(host_u16(y)).astype(np.float64)
    for u, rho, a, b in ew.segments(cu, E, C):
        err = np.linalg.norm(got[a:b] - ref[a:b]) / max(np.linalg.norm(ref[a:b]), 1e-30)
        assert err <= RTOL, (u, rho, b - a, err)
    wh = oracle.bf16_to_f32(w_home).astype(np.float64)
    ws = oracle.bf16_to_f32(w_slots).astype(np.float64)
    worst = ew.gemm_table("fwd", got, ref, oracle.bf16_to_f32(recv).astype(np.float64), cu, E, C,
                          lambda u, rho: wh[rho] if rho < E else ws[u, rho - E])
    assert (got[~covered(cu)] == -5.0).all()
    print(f"two-m-tile forward: {worst}")


def test_forward_two_mtile_units_exact_and_equal_to_vm(lib):
    """Permutation weights (one 1.0 per column, a shift per weight row): every output
    is one input element, so a wrong m-tile, accumulator, row or weight row shows."""
    bep = lib
    ctx = bep.Context(bep.Config(R, E, B, K, S, H, HP, 0))
    cu = table()
    cu_d = torch.from_numpy(cu).to(DEV)
    recv = synth.tokens_host((R * C, H), 711)

    def perm(shift):
        w = np.zeros((H, HP), np.float32)
        w[(np.arange(HP) + shift) % H, np.arange(HP)] = 1.0
        return oracle.f32_to_bf16(w)
    w_home = np.stack([perm(37 * e + 5) for e in range(E)])
    w_slots = np.stack([np.stack([perm(37 * (E + u * B + j) + 5) for j in range(B)]) for u in range(R)])
    y = torch.zeros((R * C, HP), dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm(ctx, cu_d, dev_u16(recv), dev_u16(w_home), dev_u16(w_slots), y)
    # the same weights as R materialised [E+B, H, H'] views, through the VM GEMM
    views = np.concatenate([np.concatenate([w_home, w_slots[u]], axis=0)[None] for u in range(R)])
    y_vm = torch.zeros_like(y)
    bep.bep_grouped_gemm_vm(ctx, cu_d, dev_u16(recv), dev_u16(views), y_vm)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    want = oracle.f32_to_bf16(oracle.grouped_gemm(recv, w_home, w_slots, cu, E).astype(np.float32))
    got = host_u16(y)
    for u, rho, a, b in ew.segments(cu, E, C):
        shift = 37 * (rho if rho < E else E + u * B + (rho - E)) + 5
        cols = (np.arange(HP) + shift) % H
        np.testing.assert_array_equal(nz(want[a:b]), nz(recv[a:b][:, cols]))
    np.testing.assert_array_equal(nz(got), nz(want))
    assert torch.equal(y.view(torch.int16), y_vm.view(torch.int16))


# The input gradient dRecv = dY W^T runs the same two launches when H (its N) is a multiple
# of 256 and H' (its reduction length) is at least 2048: H=256, H'=2048 on the same tables.
H_DX, HP_DX = 256, 2048


def test_input_gradient_two_mtile_units_against_binary64(lib):
    bep = lib
    ctx = bep.Context(bep.Config(R, E, B, K, S, H_DX, HP_DX, 0))
    cu = table()
    dy = synth.tokens_host((R * C, HP_DX), 721)
    w_home = synth.weights_host((E, H_DX, HP_DX), 722)
    w_slots = synth.weights_host((R, B, H_DX, HP_DX), 723)
    drecv = torch.full((R * C, H_DX), 3.0, dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm_dx(ctx, torch.from_numpy(cu).to(DEV), dev_u16(dy), dev_u16(w_home),
                            dev_u16(w_slots), drecv)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    ref = oracle.grouped_gemm_dx(dy, w_home, w_slots, cu, E)
    got = oracle.bf16_to_f32(host_u16(drecv)).astype(np.float64)
    for u, rho, a, b in ew.segments(cu, E, C):
        err = np.linalg.norm(got[a:b] - ref[a:b]) / max(np.linalg.norm(ref[a:b]), 1e-30)
        assert err <= RTOL, (u, rho, b - a, err)
    wh = oracle.bf16_to_f32(w_home).astype(np.float64)
    ws = oracle.bf16_to_f32(w_slots).astype(np.float64)
    worst = ew.gemm_table("dx", got, ref, oracle.bf16_to_f32(dy).astype(np.float64), cu, E, C,
                          lambda u, rho: wh[rho] if rho < E else ws[u, rho - E])
    assert (got[~covered(cu)] == 3.0).all()
    print(f"two-m-tile input gradient: {worst}")


def test_input_gradient_two_mtile_units_exact(lib):
    """One 1.0 per weight row h, at column sigma(h) = (8h + shift) mod H' (distinct per h):
    every dRecv[row, h] is the single element dY[row, sigma(h)]."""
    bep = lib
    ctx = bep.Context(bep.Config(R, E, B, K, S, H_DX, HP_DX, 0))
    cu = table()
    dy = synth.tokens_host((R * C, HP_DX), 731)

    def perm(shift):
        w = np.zeros((H_DX, HP_DX), np.float32)
        w[np.arange(H_DX), (8 * np.arange(H_DX) + shift) % HP_DX] = 1.0
        return oracle.f32_to_bf16(w)
    w_home = np.stack([perm(41 * e + 3) for e in range(E)])
    w_slots = np.stack([np.stack([perm(41 * (E + u * B + j) + 3) for j in range(B)]) for u in range(R)])
    drecv = torch.zeros((R * C, H_DX), dtype=torch.bfloat16, device=DEV)
    bep.bep_grouped_gemm_dx(ctx, torch.from_numpy(cu).to(DEV), dev_u16(dy), dev_u16(w_home),
                            dev_u16(w_slots), drecv)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    want = oracle.f32_to_bf16(oracle.grouped_gemm_dx(dy, w_home, w_slots, cu, E).astype(np.float32))
    for u, rho, a, b in ew.segments(cu, E, C):
        shift = 41 * (rho if rho < E else E + u * B + (rho - E)) + 3
        cols = (8 * np.arange(H_DX) + shift) % HP_DX
        np.testing.assert_array_equal(nz(want[a:b]), nz(dy[a:b][:, cols]))
    np.testing.assert_array_equal(nz(host_u16(drecv)), nz(want))
