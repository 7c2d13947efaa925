"""Element-wise error bound for the grouped GEMMs (bf16 operands, fp32 accumulation).

Every output element of the forward and input-gradient GEMMs is an n-term dot
product y = sum_i a_i w_i of bf16 values, accumulated in fp32 and rounded once
to bf16. Products of two bf16 values are exact in fp32; each of the n - 1
additions may lose up to one fp32 ulp whatever the adder's rounding mode, so
the fp32 sum carries at most gamma_(n-1) * sum_i |a_i w_i| of error, in any
summation order (the standard bound for a sum of n terms, taken with unit
roundoff 2^-23 so that a truncating accumulator is admitted too). Rounding to
bf16 (8 significant bits) then adds at most 2^-8 of the fp32 sum, so

    |y_gpu - y| <= 2^-8 |y| + (1 + 2^-8) gamma_(n-1) sum_i |a_i w_i|,

and 1.01 * n * 2^-23 exceeds (1 + 2^-8) gamma_(n-1) for every n up to 50,000
(the forward and dX sums here have n = H or H', at most 7168).
The rounding term alone can come close to its share of the bound (a sum just
above a power of two), so a ratio near 1 on small n is expected, not a warning.
A weight gradient stays in fp32 and is added onto the buffer once per
segment: 2^-23 (|y| + |g0|) more per add, and no bf16 rounding; there
1.01 * n * 2^-23 exceeds (1 + 2^-23) gamma_(n-1) for every n up to 80,000, and
no weight row sums more than R*S = 65,536 rows.

``check`` compares every element of a GPU result with the binary64 oracle
against that bound and returns the largest absolute error and the largest
error as a fraction of its element's bound, for the test to print.
"""
import numpy as np

FP32_U = 2.0 ** -23
BF16_OUT = 2.0 ** -8


def bf16_bound(ref, absprod, n):
    """Bound for a bf16 output of an n-term fp32 dot product."""
    return BF16_OUT * np.abs(ref) + 1.01 * n * FP32_U * absprod + 1e-30


def fp32_bound(ref, absprod, n, base=None, adds=1):
    """Bound for an fp32 output (a weight gradient) whose partial sums are added
    onto `base` in `adds` fp32 additions (one per segment sharing the row)."""
    b = 1.01 * n * FP32_U * absprod + adds * FP32_U * (np.abs(ref) + absprod) + 1e-30
    if base is not None:
        b = b + adds * FP32_U * np.abs(base)
    return b


def fwd(got, ref, a, w, what=""):
    """Forward GEMM rows: a [m, H] and w [H, H'] as float arrays, ref = a @ w."""
    return check(got, ref, bf16_bound(ref, np.abs(a) @ np.abs(w), a.shape[1]), what)


def dx(got, ref, dy, w, what=""):
    """Input-gradient rows: dy [m, H'], w [H, H'], ref = dy @ w.T."""
    return check(got, ref, bf16_bound(ref, np.abs(dy) @ np.abs(w).T, dy.shape[1]), what)


def dw(got, ref, parts, base=None, what=""):
    """A weight-gradient row block: parts is a list of (a [m, h], dy [m, H'])
    segment operands whose a^T dy sum is ref (minus base)."""
    absprod = sum(np.abs(a).T @ np.abs(g) for a, g in parts)
    n = sum(a.shape[0] for a, _ in parts)
    return check(got, ref, fp32_bound(ref, absprod, n, base, adds=len(parts)), what)


def check(got, ref, bound, what=""):
    """Assert |got - ref| <= bound element by element; return (max abs err, max err/bound)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    ratio = err / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    if not worst <= 1.0:
        i = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
        raise AssertionError(f"{what}: element {i} got {got[i]!r} want {ref[i]!r} "
                             f"err {err[i]:.3e} > bound {bound[i]:.3e}")
    return (float(err.max()) if err.size else 0.0), worst


class Worst:
    """Running maxima over a test's checks, printed at its end."""

    def __init__(self):
        self.abs = 0.0
        self.frac = 0.0
        self.frob = 0.0

    def add(self, pair, frob=0.0):
        self.abs = max(self.abs, pair[0])
        self.frac = max(self.frac, pair[1])
        self.frob = max(self.frob, frob)

    def __str__(self):
        return (f"worst segment rel Frobenius {self.frob:.3e}; max element error "
                f"{self.abs:.3e} ({self.frac:.3f} of its bound)")


def segments(cu, E, C):
    """(u, rho, first, end) in global receive rows for every non-empty segment."""
    R = cu.shape[0]
    for u in range(R):
        for rho in range(cu.shape[1] - 1):
            a, b = int(cu[u, rho]), int(cu[u, rho + 1])
            if b > a:
                yield u, rho, u * C + a, u * C + b


def gemm_table(kind, got, ref, rows_f, cu, E, C, weight):
    """Every segment of a forward ("fwd") or input-gradient ("dx") result, element by
    element. rows_f are the A operand's rows (receive rows or dY) as floats and
    weight(u, rho) the float [H, H'] matrix that serves segment rho on rank u."""
    worst = Worst()
    one = fwd if kind == "fwd" else dx
    for u, rho, a, b in segments(cu, E, C):
        worst.add(one(got[a:b], ref[a:b], rows_f[a:b], weight(u, rho), f"{kind} rank {u} row {rho}"))
    return worst


def dw_table(g_got, red_got, d_home, d_slots, recv_f, dy_f, cu, E, C, g0=None, red0=None):
    """Every written weight-gradient row block, element by element: home row e
    against g0[e] + d_home[e] (or d_home[e] alone when g0 is None: the overwriting
    form), slot (u, j) against red0[u, j] + d_slots[u, j]."""
    parts = {}
    for u, rho, a, b in segments(cu, E, C):
        key = rho if rho < E else (u, rho - E)
        parts.setdefault(key, []).append((recv_f[a:b], dy_f[a:b]))
    worst = Worst()
    for key, p in parts.items():
        if isinstance(key, tuple):
            u, j = key
            base = None if red0 is None else red0[u, j]
            want = d_slots[u, j] if base is None else base + d_slots[u, j]
            worst.add(dw(red_got[u, j], want, p, base, f"slot {u},{j}"))
        else:
            base = None if g0 is None else g0[key]
            want = d_home[key] if base is None else base + d_home[key]
            worst.add(dw(g_got[key], want, p, base, f"home row {key}"))
    return worst
