"""CPU checks of the element-wise GEMM error bound the GPU tests apply: an fp32
accumulation of bf16 products, in several orders and with truncating adds,
stays inside it, and the mistakes a kernel can make (a wrong column, a row of
the next segment, a dropped K block) fall outside it."""
import numpy as np
import pytest
import torch

import elementwise as ew
import oracle
import synth


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _truncate_f32(x):
    """Round a float64 array toward zero to fp32."""
    f = x.astype(np.float32)
    over = np.abs(f.astype(np.float64)) > np.abs(x)
    f[over] = np.nextafter(f[over], np.float32(0))
    return f


def _accumulate(a, w, order, truncating, block=16):
    """fp32 sum over k of a[:, k] w[k, :] (products exact), in a given block order."""
    m, n = a.shape
    acc = np.zeros((m, w.shape[1]), np.float32)
    for k0 in order:
        part = (a[:, k0:k0 + block].astype(np.float64) @ w[k0:k0 + block].astype(np.float64))
        s = acc.astype(np.float64) + _truncate_f32(part).astype(np.float64)
        acc = _truncate_f32(s) if truncating else s.astype(np.float32)
    return acc


@pytest.mark.parametrize("truncating", [False, True])
def test_fp32_accumulation_stays_inside_the_bound(truncating):
    n, m, hp = 1024, 24, 48
    a = oracle.bf16_to_f32(synth.tokens_host((m, n), 1))
    w = oracle.bf16_to_f32(synth.weights_host((n, hp), 2))
    ref = a.astype(np.float64) @ w.astype(np.float64)
    rng = np.random.default_rng(3)
    for order in (range(0, n, 16), range(n - 16, -1, -16), rng.permutation(np.arange(0, n, 16))):
        got = _bf16(_accumulate(a, w, order, truncating))
        err, frac = ew.fwd(got, ref, a, w)
        assert frac < 1.0


def test_kernel_mistakes_fall_outside_the_bound():
    n, m, hp = 512, 16, 32
    a = oracle.bf16_to_f32(synth.tokens_host((m + 1, n), 4))
    w = oracle.bf16_to_f32(synth.weights_host((n, hp), 5))
    ref = a[:m].astype(np.float64) @ w.astype(np.float64)
    good = _bf16(_accumulate(a[:m], w, range(0, n, 16), False))
    ew.fwd(good, ref, a[:m], w)
    bad_col = good.copy()
    bad_col[:, [3, 4]] = bad_col[:, [4, 3]]                    # two output columns swapped
    bad_row = good.copy()
    bad_row[-1] = _bf16(a[m:m + 1] @ w)[0]                     # the next segment's row
    dropped = _bf16(_accumulate(a[:m], w, range(0, n - 64, 16), False))   # last K block lost
    for bad in (bad_col, bad_row, dropped):
        with pytest.raises(AssertionError):
            ew.fwd(bad, ref, a[:m], w)


def test_weight_gradient_bound_admits_the_add_and_catches_a_lost_segment():
    rows, h, hp = 300, 8, 16
    a = oracle.bf16_to_f32(synth.tokens_host((rows, h), 6)).astype(np.float64)
    g = oracle.bf16_to_f32(synth.tokens_host((rows, hp), 7)).astype(np.float64)
    base = synth.normal_host((h, hp), 8, 0.5).astype(np.float64)
    half = rows // 2
    parts = [(a[:half], g[:half]), (a[half:], g[half:])]
    ref = base + a.T @ g
    got = base.astype(np.float32)
    for pa, pg in parts:                                       # two segments, two fp32 adds
        got = (got.astype(np.float64) + (pa.T @ pg).astype(np.float32)).astype(np.float32)
    ew.dw(got, ref, parts, base)
    lost = (base + (a[:half].T @ g[:half])).astype(np.float32)
    with pytest.raises(AssertionError):
        ew.dw(lost, ref, parts, base)
