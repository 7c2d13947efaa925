"""Oracle for balanced expert-parallel dispatch -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU restatement of what the hot path computes, written from the
MoonEP announcement pages (see ``oracle.cpp`` for the page citations and the
step-by-step rule). Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with the CUDA library and never imports it.

Pieces:
  * ``liboracle.so`` (plain C++, single thread, ``-ffp-contract=off``):
    histogram, maxvio, the planning rule, the plan-validity checker, dispatch,
    combine, combine backward, prefetch and reduce_grad.
  * ``liboracle_omp.so``: the same source built with ``-fopenmp``, loaded
    instead when ``ORACLE_OPENMP=1`` is set before the first call. Its per-token
    loops run on every core and give the same bits; only the CPU baseline's
    all-core leg uses it.
  * ``grouped_gemm`` (numpy, binary64): the expert GEMM per segment, from
    bf16 inputs, with numpy's matmul as the one library step.

Parity status: every function is pinned by the ``-m "not gpu"`` tests
(closed forms, brute force on tiny inputs, library routines for special
cases, hand-worked examples). The pages leave the planner's choice among
valid plans open ("near-optimal"); the oracle follows one documented rule (a
reading of the pages), pinned to that rule by plans worked out by hand from
its definition, and to validity by ``check_plan`` and by brute force over
every parent function on small cases. Whether MoonEP's own planner makes the
same choice cannot be decided from the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_SERIAL = os.path.join(_HERE, "liboracle.so")
_LIB_OMP = os.path.join(_HERE, "liboracle_omp.so")
_LIB = _LIB_OMP if os.environ.get("ORACLE_OPENMP") == "1" else _LIB_SERIAL
_lock = threading.Lock()
_lib = None

MODE_TRAIN = 0
MODE_INFER = 1

ERRORS = {
    0: "ok",
    -1: "expert id out of range",
    -2: "duplicate expert id in one token",
    -3: "inconsistent configuration",
    -4: "plan infeasible",
}


def _compile(lib: str, openmp: bool, force: bool) -> str:
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(_SRC):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
               "-Wno-unknown-pragmas"] + (["-fopenmp"] if openmp else []) + ["-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


def build(force: bool = False, openmp: bool | None = None) -> str:
    """Compile the oracle with the host C++ compiler: the single-threaded
    ``liboracle.so`` (openmp=False), the OpenMP ``liboracle_omp.so`` (True), or
    the one this process loads (None)."""
    if openmp is None:
        openmp = _LIB == _LIB_OMP
    return _compile(_LIB_OMP if openmp else _LIB_SERIAL, openmp, force)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i32p = ctypes.POINTER(ctypes.c_int32)
            i64p = ctypes.POINTER(ctypes.c_int64)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            ci, c64 = ctypes.c_int, ctypes.c_int64
            sig = {
                "oracle_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "oracle_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "oracle_f32_to_bf16_array": (None, [f32p, c64, u16p]),
                "oracle_histogram": (ci, [i32p, ci, ci, ci, ci, i64p]),
                "oracle_maxvio": (ctypes.c_double, [i64p, ci, c64]),
                "oracle_tree": (ci, [ci, i64p, c64, i32p, i64p, i32p]),
                "oracle_plan": (ci, [ci, ci, ci, ci, ci, ci, i32p, i32p, i32p, i32p, i32p,
                                     i64p, f64p]),
                "oracle_check_plan": (ci, [ci, ci, ci, ci, ci, ci, i32p, i32p, i32p, i32p]),
                "oracle_dispatch": (None, [u16p, i32p, ci, ci, ci, ci, u16p]),
                "oracle_combine": (None, [u16p, i32p, f32p, ci, ci, ci, ci, u16p]),
                "oracle_combine_bwd": (None, [u16p, i32p, f32p, ci, ci, ci, ci, u16p]),
                "oracle_dispatch_bwd": (None, [u16p, i32p, ci, ci, ci, ci, u16p]),
                "oracle_combine_dgates": (None, [u16p, u16p, i32p, ci, ci, ci, ci, f64p]),
                "oracle_prefetch": (None, [u16p, i32p, ci, ci, c64, u16p]),
                "oracle_reduce_grad": (None, [f32p, f32p, i32p, ci, ci, ci, c64]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle error {code}: {ERRORS.get(code, '?')}")
        self.code = code


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, by definition (upper half of binary32)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_scalar(f: float) -> int:
    return int(_load().oracle_f32_to_bf16(ctypes.c_float(f)))


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns, round to nearest even."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_f32_to_bf16_array(_ptr(a, ctypes.c_float), a.size, _ptr(out, ctypes.c_uint16))
    return out


def histogram(topk: np.ndarray, E: int) -> np.ndarray:
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    R, S, K = topk.shape
    T = np.zeros(E, dtype=np.int64)
    rc = _load().oracle_histogram(_ptr(topk, ctypes.c_int32), R, S, K, E, _ptr(T, ctypes.c_int64))
    if rc:
        raise OracleError(rc)
    return T


def maxvio(T: np.ndarray, rsk: int) -> float:
    T = np.ascontiguousarray(T, dtype=np.int64)
    return float(_load().oracle_maxvio(_ptr(T, ctypes.c_int64), len(T), int(rsk)))


def tree(L, C: int):
    """The planning rule's tree step alone: (parent, inflow, order) per rank."""
    L = np.ascontiguousarray(L, dtype=np.int64)
    R = len(L)
    parent = np.zeros(R, np.int32)
    inflow = np.zeros(R, np.int64)
    order = np.zeros(R, np.int32)
    rc = _load().oracle_tree(R, _ptr(L, ctypes.c_int64), int(C), _ptr(parent, ctypes.c_int32),
                             _ptr(inflow, ctypes.c_int64), _ptr(order, ctypes.c_int32))
    if rc:
        raise OracleError(rc)
    return parent, inflow, order


class Plan:
    __slots__ = ("cu", "slot_expert", "dest", "parent", "inflow", "maxvio")


def plan(topk: np.ndarray, E: int, B: int, mode: int) -> Plan:
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    R, S, K = topk.shape
    p = Plan()
    p.cu = np.zeros((R, E + B + 1), np.int32)
    p.slot_expert = np.zeros((R, B), np.int32)
    p.dest = np.zeros((R, S, K), np.int32)
    p.parent = np.zeros(R, np.int32)
    p.inflow = np.zeros(R, np.int64)
    mv = ctypes.c_double(0.0)
    rc = _load().oracle_plan(R, E, B, K, S, mode, _ptr(topk, ctypes.c_int32),
                             _ptr(p.cu, ctypes.c_int32), _ptr(p.slot_expert, ctypes.c_int32),
                             _ptr(p.dest, ctypes.c_int32), _ptr(p.parent, ctypes.c_int32),
                             _ptr(p.inflow, ctypes.c_int64), ctypes.byref(mv))
    if rc:
        raise OracleError(rc)
    p.maxvio = mv.value
    return p


def check_plan(topk, E, B, mode, cu, slot_expert, dest) -> int:
    """0 if (cu, slot_expert, dest) is a valid plan for topk, else the failed invariant."""
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    R, S, K = topk.shape
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    se = np.ascontiguousarray(slot_expert, dtype=np.int32)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    return int(_load().oracle_check_plan(R, E, B, K, S, mode, _ptr(topk, ctypes.c_int32),
                                         _ptr(cu, ctypes.c_int32), _ptr(se, ctypes.c_int32),
                                         _ptr(dest, ctypes.c_int32)))


def dispatch(x: np.ndarray, dest: np.ndarray) -> np.ndarray:
    """x: uint16 (bf16 bits) [R,S,H]; dest [R,S,K] -> recv [R*S*K, H]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    R, S, H = x.shape
    K = dest.shape[2]
    recv = np.zeros((R * S * K, H), np.uint16)
    _load().oracle_dispatch(_ptr(x, ctypes.c_uint16), _ptr(dest, ctypes.c_int32), R, S, K, H,
                            _ptr(recv, ctypes.c_uint16))
    return recv


def combine(y: np.ndarray, dest: np.ndarray, gates: np.ndarray) -> np.ndarray:
    """y: uint16 [R*S*K, D]; dest, gates [R,S,K] -> out uint16 [R,S,D]."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float32)
    R, S, K = dest.shape
    D = y.shape[1]
    out = np.zeros((R, S, D), np.uint16)
    _load().oracle_combine(_ptr(y, ctypes.c_uint16), _ptr(dest, ctypes.c_int32),
                           _ptr(gates, ctypes.c_float), R, S, K, D, _ptr(out, ctypes.c_uint16))
    return out


def combine_bwd(dout: np.ndarray, dest: np.ndarray, gates: np.ndarray) -> np.ndarray:
    """dout uint16 [R,S,D] -> dy uint16 [R*S*K, D]."""
    dout = np.ascontiguousarray(dout, dtype=np.uint16)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float32)
    R, S, K = dest.shape
    D = dout.shape[2]
    dy = np.zeros((R * S * K, D), np.uint16)
    _load().oracle_combine_bwd(_ptr(dout, ctypes.c_uint16), _ptr(dest, ctypes.c_int32),
                               _ptr(gates, ctypes.c_float), R, S, K, D, _ptr(dy, ctypes.c_uint16))
    return dy


def prefetch(w_home: np.ndarray, slot_expert: np.ndarray, w_slots: np.ndarray) -> np.ndarray:
    """Copies home rows into the used slots of w_slots [R,B,H,H'] (in place, returned)."""
    w_home = np.ascontiguousarray(w_home, dtype=np.uint16)
    se = np.ascontiguousarray(slot_expert, dtype=np.int32)
    assert w_slots.flags["C_CONTIGUOUS"] and w_slots.dtype == np.uint16
    R, B = se.shape
    hhp = int(np.prod(w_home.shape[1:]))
    _load().oracle_prefetch(_ptr(w_home, ctypes.c_uint16), _ptr(se, ctypes.c_int32), R, B, hhp,
                            _ptr(w_slots, ctypes.c_uint16))
    return w_slots


def reduce_grad(g_home: np.ndarray, red: np.ndarray, slot_expert: np.ndarray) -> None:
    """In place: g_home [E,H,H'] fp32 += replica grads from red [R,B,H,H'] fp32; red slots zeroed."""
    assert g_home.flags["C_CONTIGUOUS"] and g_home.dtype == np.float32
    assert red.flags["C_CONTIGUOUS"] and red.dtype == np.float32
    se = np.ascontiguousarray(slot_expert, dtype=np.int32)
    R, B = se.shape
    E = g_home.shape[0]
    hhp = int(np.prod(g_home.shape[1:]))
    _load().oracle_reduce_grad(_ptr(g_home, ctypes.c_float), _ptr(red, ctypes.c_float),
                               _ptr(se, ctypes.c_int32), R, B, E, hhp)


def segment_of_rows(cu: np.ndarray, C: int, rows: np.ndarray) -> np.ndarray:
    """For global receive rows i (rank u = i // C), the segment row index rho."""
    rows = np.asarray(rows, dtype=np.int64)
    u = rows // C
    pos = rows % C
    out = np.empty(len(rows), np.int64)
    for n in range(len(rows)):
        out[n] = np.searchsorted(cu[u[n]], pos[n], side="right") - 1
    return out


def grouped_gemm(recv: np.ndarray, w_home: np.ndarray, w_slots: np.ndarray, cu: np.ndarray,
                 E: int, rows=None) -> np.ndarray:
    """Expert GEMM in binary64 ([P4] "The memory contract": one [E+B, H, H'] weight
    tensor addressed by row index; cu_seqlens selects the active rows).

    For rank u and row rho with a non-empty segment, Y[u, seg] = recv[u, seg] @ W_rho,
    W_rho = w_home[rho] if rho < E else w_slots[u, rho - E]. Inputs are bf16 bit
    patterns (uint16); the product is formed in float64 from the exact bf16 values.

    rows=None computes every row (small cases); otherwise only the listed global
    receive rows, returned in that order.
    """
    R = cu.shape[0]
    nrow_total, H = recv.shape
    C = nrow_total // R
    Hp = w_home.shape[2]
    if rows is None:
        y = np.zeros((nrow_total, Hp), np.float64)
        for u in range(R):
            for rho in range(cu.shape[1] - 1):
                a, b = int(cu[u, rho]), int(cu[u, rho + 1])
                if b == a:
                    continue
                w = w_home[rho] if rho < E else w_slots[u, rho - E]
                A = bf16_to_f32(recv[u * C + a:u * C + b]).astype(np.float64)
                W = bf16_to_f32(w).astype(np.float64)
                y[u * C + a:u * C + b] = A @ W
        return y
    rows = np.asarray(rows, dtype=np.int64)
    seg = segment_of_rows(cu, C, rows)
    y = np.zeros((len(rows), Hp), np.float64)
    wcache = {}
    for n, (i, rho) in enumerate(zip(rows, seg)):
        u = int(i // C)
        key = (u, int(rho)) if rho >= E else (-1, int(rho))
        if key not in wcache:
            w = w_home[rho] if rho < E else w_slots[u, rho - E]
            wcache[key] = bf16_to_f32(np.asarray(w)).astype(np.float64)
        y[n] = bf16_to_f32(recv[i]).astype(np.float64) @ wcache[key]
    return y


def gemm_rows(a_rows: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = a @ W in binary64 for bf16 bit-pattern inputs a [n, H], W [H, H']."""
    A = bf16_to_f32(np.asarray(a_rows)).astype(np.float64)
    W = bf16_to_f32(np.asarray(w)).astype(np.float64)
    return A @ W


def weight_row_of(rho: int, u: int, E: int, slot_expert: np.ndarray) -> int:
    """The home expert whose weights serve segment row rho on rank u: rho itself for
    rho < E, else the expert prefetch_weight copied into slot rho - E."""
    return int(rho) if rho < E else int(slot_expert[u, rho - E])


def dispatch_bwd(drecv: np.ndarray, dest: np.ndarray) -> np.ndarray:
    """drecv uint16 [R*S*K, H], dest [R,S,K] -> dx uint16 [R,S,H] (sum of the K rows, fp32, in k order)."""
    drecv = np.ascontiguousarray(drecv, dtype=np.uint16)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    R, S, K = dest.shape
    H = drecv.shape[1]
    dx = np.zeros((R, S, H), np.uint16)
    _load().oracle_dispatch_bwd(_ptr(drecv, ctypes.c_uint16), _ptr(dest, ctypes.c_int32), R, S, K,
                                H, _ptr(dx, ctypes.c_uint16))
    return dx


def combine_dgates(dout: np.ndarray, y: np.ndarray, dest: np.ndarray) -> np.ndarray:
    """dg [R,S,K] float64: <dOut[r,t], Y[dest[r,t,k]]>."""
    dout = np.ascontiguousarray(dout, dtype=np.uint16)
    y = np.ascontiguousarray(y, dtype=np.uint16)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    R, S, K = dest.shape
    D = y.shape[1]
    dg = np.zeros((R, S, K), np.float64)
    _load().oracle_combine_dgates(_ptr(dout, ctypes.c_uint16), _ptr(y, ctypes.c_uint16),
                                  _ptr(dest, ctypes.c_int32), R, S, K, D,
                                  _ptr(dg, ctypes.c_double))
    return dg


def grouped_gemm_dx(dy: np.ndarray, w_home: np.ndarray, w_slots: np.ndarray, cu: np.ndarray,
                    E: int) -> np.ndarray:
    """Input gradient of the expert GEMM, binary64: for every non-empty segment,
    dRecv[u, seg] = dY[u, seg] @ W(u, rho)^T (W(u, rho) as in grouped_gemm)."""
    R = cu.shape[0]
    nrow_total = dy.shape[0]
    C = nrow_total // R
    H = w_home.shape[1]
    out = np.zeros((nrow_total, H), np.float64)
    for u in range(R):
        for rho in range(cu.shape[1] - 1):
            a, b = int(cu[u, rho]), int(cu[u, rho + 1])
            if b == a:
                continue
            w = w_home[rho] if rho < E else w_slots[u, rho - E]
            G = bf16_to_f32(dy[u * C + a:u * C + b]).astype(np.float64)
            W = bf16_to_f32(w).astype(np.float64)
            out[u * C + a:u * C + b] = G @ W.T
    return out


def grouped_gemm_dw(recv: np.ndarray, dy: np.ndarray, cu: np.ndarray, E: int, B: int,
                    H: int, Hp: int):
    """Weight gradient of the expert GEMM, binary64, per non-empty segment:
    dW(u, rho) = recv[u, seg]^T @ dY[u, seg]. Returns (d_home [E,H,H'], d_slots [R,B,H,H']),
    summing the segments that share a weight row (a home row's segments on every rank)."""
    R = cu.shape[0]
    C = recv.shape[0] // R
    d_home = np.zeros((E, H, Hp), np.float64)
    d_slots = np.zeros((R, B, H, Hp), np.float64)
    for u in range(R):
        for rho in range(cu.shape[1] - 1):
            a, b = int(cu[u, rho]), int(cu[u, rho + 1])
            if b == a:
                continue
            A = bf16_to_f32(recv[u * C + a:u * C + b]).astype(np.float64)
            G = bf16_to_f32(dy[u * C + a:u * C + b]).astype(np.float64)
            if rho < E:
                d_home[rho] += A.T @ G
            else:
                d_slots[u, rho - E] += A.T @ G
    return d_home, d_slots
