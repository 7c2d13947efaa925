"""The weight gradient written instead of added (bep_grouped_gemm_dw_overwrite),
through the C ABI, against the binary64 oracle:

  g_home[e]       = recv[seg]^T dY[seg] of e's home segment, zeros when it is empty
  red[u][j]       = recv[seg]^T dY[seg] of every non-empty slot segment
  other red slots   keep their contents

on hand-made training tables (home rows only on their home rank, ragged lengths,
empty home segments, +inf in every receive row outside the segments) on single
CTAs (H'=128) and on SM pairs (H=512, H'=256); the sums equal, value for value,
those the accumulating call adds onto zeros; a table that is not a training
plan's is refused; S*K = 0 zeroes the home rows. Written rows are also checked
element by element against the fp32-accumulation bound of ``elementwise``."""
import numpy as np
import pytest
import torch

import elementwise as ew
import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
RTOL = 2e-2
POISON = 12345.0

# R=2, E=8 (4 home experts per rank), B=4, K=2, S=1024: C=2048 slots per rank.
# Rank 0 owns experts 0-3, rank 1 experts 4-7: each rank's other home rows stay
# empty, as in every training plan. Experts 2 and 5 have empty home segments.
R, E, B, K, S = 2, 8, 4, 2, 1024
G = E // R
C = S * K
LENGTHS = [
    [1, 15, 0, 64, 0, 0, 0, 0, 17, 63, 128, 0],
    [0, 0, 0, 0, 2, 0, 129, 257, 16, 65, 0, 33],
]


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(DEV).view(
        torch.bfloat16)


def table(lengths=LENGTHS):
    cu = np.zeros((R, E + B + 1), np.int32)
    for u in range(R):
        cu[u, 1:] = np.cumsum(lengths[u])
    assert cu[:, -1].max() <= C
    return cu


def inputs(cu, H, HP):
    recv = synth.tokens_host((R * C, H), 421)
    dy = synth.tokens_host((R * C, HP), 422)
    inside = np.zeros(R * C, bool)
    for u in range(R):
        inside[u * C:u * C + int(cu[u, -1])] = True
    recv[~inside] = 0x7F80      # bf16 +inf: a tail step that read them unzeroed shows
    dy[~inside] = 0x7F80
    return recv, dy


@pytest.mark.parametrize("H, HP", [(256, 128), (512, 256)])
def test_overwrite_matches_oracle_on_training_table(lib, H, HP):
    bep = lib
    ctx = bep.Context(bep.Config(R, E, B, K, S, H, HP, 0))
    cu = table()
    recv, dy = inputs(cu, H, HP)
    g = torch.full((E, H, HP), POISON, dtype=torch.float32, device=DEV)
    red = torch.full((R, B, H, HP), POISON, dtype=torch.float32, device=DEV)
    bep.bep_grouped_gemm_dw_overwrite(ctx, torch.from_numpy(cu).to(DEV), dev_u16(recv), dev_u16(dy),
                                      g, red)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    d_home, d_slots = oracle.grouped_gemm_dw(recv, dy, cu, E, B, H, HP)
    gh, rh = g.cpu().numpy().astype(np.float64), red.cpu().numpy().astype(np.float64)
    for e in range(E):
        u = e // G
        if cu[u, e + 1] == cu[u, e]:
            assert (gh[e] == 0.0).all(), e           # empty home segment: written as zeros
            continue
        err = np.linalg.norm(gh[e] - d_home[e]) / np.linalg.norm(d_home[e])
        assert err <= RTOL, (e, err)
    for u in range(R):
        for j in range(B):
            if cu[u, E + j + 1] == cu[u, E + j]:
                assert (rh[u, j] == POISON).all(), (u, j)   # slot without tokens: not written
                continue
            err = np.linalg.norm(rh[u, j] - d_slots[u, j]) / np.linalg.norm(d_slots[u, j])
            assert err <= RTOL, (u, j, err)
    worst = ew.dw_table(gh, rh, d_home, d_slots, oracle.bf16_to_f32(recv).astype(np.float64),
                        oracle.bf16_to_f32(dy).astype(np.float64), cu, E, C)
    print(f"overwriting dW (H={H}): {worst}")


@pytest.mark.parametrize("H, HP", [(256, 128), (512, 256)])
def test_overwrite_equals_accumulating_onto_zeros(lib, H, HP):
    """Both calls take the same K order, so the written sums are the values the
    accumulating call adds onto zero buffers (x + 0 = x; == treats -0 and +0 alike)."""
    bep = lib
    ctx = bep.Context(bep.Config(R, E, B, K, S, H, HP, 0))
    cu = torch.from_numpy(table()).to(DEV)
    recv, dy = inputs(table(), H, HP)
    recv_d, dy_d = dev_u16(recv), dev_u16(dy)
    g_add = torch.zeros((E, H, HP), dtype=torch.float32, device=DEV)
    red_add = torch.zeros((R, B, H, HP), dtype=torch.float32, device=DEV)
    bep.bep_grouped_gemm_dw(ctx, cu, recv_d, dy_d, g_add, red_add)
    g_set = torch.full((E, H, HP), POISON, dtype=torch.float32, device=DEV)
    red_set = torch.zeros((R, B, H, HP), dtype=torch.float32, device=DEV)
    bep.bep_grouped_gemm_dw_overwrite(ctx, cu, recv_d, dy_d, g_set, red_set)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    assert torch.equal(g_set, g_add)
    assert torch.equal(red_set, red_add)


def test_overwrite_refuses_a_home_row_on_another_rank(lib):
    bep = lib
    H, HP = 256, 128
    ctx = bep.Context(bep.Config(R, E, B, K, S, H, HP, 0))
    bad = [list(LENGTHS[0]), list(LENGTHS[1])]
    bad[0][5] = 3            # expert 5 lives on rank 1: rank 0 must not use row 5
    cu = table(bad)
    recv, dy = inputs(cu, H, HP)
    g = torch.full((E, H, HP), POISON, dtype=torch.float32, device=DEV)
    red = torch.full((R, B, H, HP), POISON, dtype=torch.float32, device=DEV)
    bep.bep_grouped_gemm_dw_overwrite(ctx, torch.from_numpy(cu).to(DEV), dev_u16(recv), dev_u16(dy),
                                      g, red)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == bep.BEP_DERR_BOUNDS
    assert (g == POISON).all() and (red == POISON).all()     # nothing written


def test_overwrite_with_no_tokens_zeroes_the_home_rows(lib):
    bep = lib
    H, HP = 256, 128
    ctx = bep.Context(bep.Config(R, E, B, K, 0, H, HP, 0))
    g = torch.full((E, H, HP), POISON, dtype=torch.float32, device=DEV)
    red = torch.full((R, B, H, HP), POISON, dtype=torch.float32, device=DEV)
    empty_bf16 = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    empty_dy = torch.empty((0, HP), dtype=torch.bfloat16, device=DEV)
    cu = torch.zeros((R, E + B + 1), dtype=torch.int32, device=DEV)
    bep.bep_grouped_gemm_dw_overwrite(ctx, cu, empty_bf16, empty_dy, g, red)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    assert (g == 0).all()
    assert (red == POISON).all()


def test_overwrite_then_reduce_grad_gives_the_whole_gradient(lib):
    """A planned training step: the overwriting dW and reduce_grad leave in g_home
    what zeroed buffers, the accumulating dW and reduce_grad leave there."""
    bep = lib
    wl = synth.WORKLOADS["grad_r8_e64"]
    topk = synth.routing(wl, 10.0, 0)
    ref = oracle.plan(topk, wl.E, wl.B, wl.mode)
    cfg = bep.Config(wl.R, wl.E, wl.B, wl.K, wl.S, wl.H, wl.Hp, wl.mode)
    ctx = bep.Context(cfg)
    buf = bep.Buffers(cfg, DEV)
    bep.bep_plan(ctx, torch.from_numpy(topk).to(DEV), buf.cu_seqlens, buf.slot_expert, buf.dest,
                 buf.maxvio)
    x = synth.tokens_host((wl.R, wl.S, wl.H), 431)
    dy = dev_u16(synth.tokens_host((wl.R * wl.C, wl.Hp), 432))
    bep.bep_dispatch(ctx, dev_u16(x), buf.dest, buf.recv)
    shape_g, shape_r = (wl.E, wl.H, wl.Hp), (wl.R, wl.B, wl.H, wl.Hp)
    g_add = torch.zeros(shape_g, dtype=torch.float32, device=DEV)
    red_add = torch.zeros(shape_r, dtype=torch.float32, device=DEV)
    bep.bep_grouped_gemm_dw(ctx, buf.cu_seqlens, buf.recv, dy, g_add, red_add)
    bep.bep_reduce_grad(ctx, buf.slot_expert, g_add, red_add)
    g_set = torch.full(shape_g, POISON, dtype=torch.float32, device=DEV)
    red_set = torch.zeros(shape_r, dtype=torch.float32, device=DEV)
    bep.bep_grouped_gemm_dw_overwrite(ctx, buf.cu_seqlens, buf.recv, dy, g_set, red_set)
    bep.bep_reduce_grad(ctx, buf.slot_expert, g_set, red_set)
    torch.cuda.synchronize()
    assert bep.bep_status(ctx) == 0
    assert int((buf.slot_expert >= 0).sum()) > 0          # the routing plans replicas
    np.testing.assert_array_equal(buf.cu_seqlens.cpu().numpy(), ref.cu)
    assert torch.equal(g_set, g_add)
    assert (red_set == 0).all() and (red_add == 0).all()
