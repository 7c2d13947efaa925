"""Balanced expert-parallel dispatch for one GB300 (sm_103a) -- Python binding.

A thin ctypes layer over ``libbep.so`` (C ABI in ``include/bep.h``): it checks
tensors and passes raw device pointers and the current CUDA stream. Every step
of the path runs in the library's CUDA kernels; there is no fallback. If the
library is missing or cannot be loaded, every call raises.

The calls keep the C names (``bep_create``, ``bep_plan``, ``bep_prefetch_weight``,
``bep_dispatch``, ``bep_grouped_gemm``, ``bep_combine``, ``bep_combine_bwd``,
``bep_reduce_grad``, ``bep_status``); :class:`Context` owns a ``bep_ctx``.
PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbep.so")

BEP_OK = 0
BEP_ERR_ARG = -1
BEP_ERR_ALIGN = -2
BEP_ERR_MODE = -3
BEP_ERR_SIZE = -4
BEP_ERR_CUDA = -5
BEP_DERR_EXPERT_ID = 1
BEP_DERR_DUP_ID = 2
BEP_DERR_INFEASIBLE = 4
BEP_DERR_BOUNDS = 8
BEP_DERR_TIMEOUT = 16
BEP_TRAIN = 0
BEP_INFER = 1

# every entry point declared in include/bep.h
SYMBOLS = ("bep_create", "bep_destroy", "bep_plan", "bep_plan_noalloc", "bep_prefetch_weight",
           "bep_dispatch", "bep_grouped_gemm", "bep_combine", "bep_combine_bwd",
           "bep_combine_dgates", "bep_dispatch_bwd", "bep_grouped_gemm_dx", "bep_grouped_gemm_dw",
           "bep_grouped_gemm_dw_overwrite",
           "bep_grouped_gemm_vm", "bep_weights_create", "bep_weights_get",
           "bep_weights_destroy", "bep_reduce_grad", "bep_set_comm_sms", "bep_wait_selftest",
           "bep_status", "bep_clear_status", "bep_strerror")

_lib = None
_lock = threading.Lock()


class BepError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {code} ({strerror(code)})")


class _Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("R", "E", "B", "K", "S", "H", "Hp", "mode")]


def load(path: str = LIB_PATH):
    """Loads libbep.so (raises if it is absent: build it with ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"libbep.so not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, i32, p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p
        sig = {
            "bep_create": (ctypes.c_int, [ctypes.POINTER(_Config), ctypes.POINTER(vp)]),
            "bep_destroy": (None, [vp]),
            "bep_plan": (ctypes.c_int, [vp, p, p, p, p, p, vp]),
            "bep_plan_noalloc": (ctypes.c_int, [ctypes.POINTER(_Config), p, p, p, p, p, p, vp]),
            "bep_prefetch_weight": (ctypes.c_int, [vp, p, p, p, vp]),
            "bep_dispatch": (ctypes.c_int, [vp, p, p, p, vp]),
            "bep_grouped_gemm": (ctypes.c_int, [vp, p, p, p, p, p, vp]),
            "bep_combine": (ctypes.c_int, [vp, p, p, p, i32, p, vp]),
            "bep_combine_bwd": (ctypes.c_int, [vp, p, p, p, i32, p, vp]),
            "bep_grouped_gemm_vm": (ctypes.c_int, [vp, p, p, p, p, vp]),
            "bep_weights_create": (ctypes.c_int, [ctypes.POINTER(_Config), i32,
                                                  ctypes.POINTER(vp)]),
            "bep_weights_get": (ctypes.c_int, [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                               ctypes.POINTER(vp)]),
            "bep_weights_destroy": (None, [vp]),
            "bep_combine_dgates": (ctypes.c_int, [vp, p, p, p, i32, p, vp]),
            "bep_set_comm_sms": (ctypes.c_int, [vp, i32]),
            "bep_wait_selftest": (ctypes.c_int, [vp, i32, vp]),
            "bep_dispatch_bwd": (ctypes.c_int, [vp, p, p, p, vp]),
            "bep_grouped_gemm_dx": (ctypes.c_int, [vp, p, p, p, p, p, vp]),
            "bep_grouped_gemm_dw": (ctypes.c_int, [vp, p, p, p, p, p, vp]),
            "bep_grouped_gemm_dw_overwrite": (ctypes.c_int, [vp, p, p, p, p, p, vp]),
            "bep_reduce_grad": (ctypes.c_int, [vp, p, p, p, vp]),
            "bep_status": (ctypes.c_int, [vp, ctypes.POINTER(i32), vp]),
            "bep_clear_status": (ctypes.c_int, [vp, vp]),
            "bep_strerror": (ctypes.c_char_p, [i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def strerror(code: int) -> str:
    try:
        return load().bep_strerror(int(code)).decode()
    except ImportError:
        return "?"


def _check(rc: int, where: str):
    if rc != BEP_OK:
        raise BepError(rc, where)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _ptr(t, dtypes, name, optional=False):
    import torch
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _numel(t, n, name):
    if t is not None and t.numel() != n:
        raise ValueError(f"{name} has {t.numel()} elements, expected {n}")


def _bf16():
    import torch
    return (torch.bfloat16, torch.int16, torch.uint16)


def _i32():
    import torch
    return (torch.int32,)


def _f32():
    import torch
    return (torch.float32,)


@dataclass(frozen=True)
class Config:
    R: int
    E: int
    B: int
    K: int
    S: int
    H: int
    Hp: int
    mode: int = BEP_TRAIN

    @property
    def G(self):
        return self.E // self.R

    @property
    def C(self):
        return self.S * self.K


class Context:
    """Owns a bep_ctx (planning / scheduling workspace on the current device)."""

    def __init__(self, cfg: Config):
        lib = load()
        c = _Config(cfg.R, cfg.E, cfg.B, cfg.K, cfg.S, cfg.H, cfg.Hp, cfg.mode)
        h = ctypes.c_void_p()
        _check(lib.bep_create(ctypes.byref(c), ctypes.byref(h)), "bep_create")
        self.cfg = cfg
        self.handle = h

    def close(self):
        if self.handle:
            load().bep_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


def bep_create(cfg: Config) -> Context:
    return Context(cfg)


def bep_plan(ctx: Context, topk, cu_seqlens, slot_expert, dest, maxvio, stream=None):
    import torch
    c = ctx.cfg
    _numel(topk, c.R * c.S * c.K, "topk")
    _numel(dest, c.R * c.S * c.K, "dest")
    _numel(cu_seqlens, c.R * (c.E + c.B + 1), "cu_seqlens")
    _numel(slot_expert, c.R * c.B, "slot_expert")
    _numel(maxvio, 1, "maxvio")
    _check(load().bep_plan(ctx.handle, _ptr(topk, _i32(), "topk"),
                           _ptr(cu_seqlens, _i32(), "cu_seqlens"),
                           _ptr(slot_expert, _i32(), "slot_expert"), _ptr(dest, _i32(), "dest"),
                           _ptr(maxvio, (torch.float64,), "maxvio"), _stream(stream)), "bep_plan")


def bep_plan_noalloc(cfg: Config, topk, cu_seqlens, slot_expert, dest, maxvio, device_err,
                     stream=None):
    """bep_plan without a context and without allocating (scratch in a static device
    array inside the library); device_err receives this call's BEP_DERR_* bits."""
    import torch
    c = cfg
    _numel(topk, c.R * c.S * c.K, "topk")
    _numel(dest, c.R * c.S * c.K, "dest")
    _numel(cu_seqlens, c.R * (c.E + c.B + 1), "cu_seqlens")
    _numel(slot_expert, c.R * c.B, "slot_expert")
    _numel(maxvio, 1, "maxvio")
    _numel(device_err, 1, "device_err")
    cc = _Config(c.R, c.E, c.B, c.K, c.S, c.H, c.Hp, c.mode)
    _check(load().bep_plan_noalloc(ctypes.byref(cc), _ptr(topk, _i32(), "topk"),
                                   _ptr(cu_seqlens, _i32(), "cu_seqlens"),
                                   _ptr(slot_expert, _i32(), "slot_expert"),
                                   _ptr(dest, _i32(), "dest"),
                                   _ptr(maxvio, (torch.float64,), "maxvio"),
                                   _ptr(device_err, _i32(), "device_err"), _stream(stream)),
           "bep_plan_noalloc")


def bep_prefetch_weight(ctx: Context, slot_expert, w_home, w_slots, stream=None):
    c = ctx.cfg
    _numel(slot_expert, c.R * c.B, "slot_expert")
    _numel(w_home, c.E * c.H * c.Hp, "w_home")
    _numel(w_slots, c.R * c.B * c.H * c.Hp, "w_slots")
    _check(load().bep_prefetch_weight(ctx.handle, _ptr(slot_expert, _i32(), "slot_expert"),
                                      _ptr(w_home, _bf16(), "w_home"),
                                      _ptr(w_slots, _bf16(), "w_slots"), _stream(stream)),
           "bep_prefetch_weight")


def bep_dispatch(ctx: Context, x, dest, recv, stream=None):
    c = ctx.cfg
    _numel(x, c.R * c.S * c.H, "x")
    _numel(dest, c.R * c.S * c.K, "dest")
    _numel(recv, c.R * c.C * c.H, "recv")
    _check(load().bep_dispatch(ctx.handle, _ptr(x, _bf16(), "x"), _ptr(dest, _i32(), "dest"),
                               _ptr(recv, _bf16(), "recv"), _stream(stream)), "bep_dispatch")


def bep_grouped_gemm(ctx: Context, cu_seqlens, recv, w_home, w_slots, y, stream=None):
    c = ctx.cfg
    _numel(cu_seqlens, c.R * (c.E + c.B + 1), "cu_seqlens")
    _numel(recv, c.R * c.C * c.H, "recv")
    _numel(w_home, c.E * c.H * c.Hp, "w_home")
    _numel(w_slots, c.R * c.B * c.H * c.Hp, "w_slots")
    _numel(y, c.R * c.C * c.Hp, "y")
    _check(load().bep_grouped_gemm(ctx.handle, _ptr(cu_seqlens, _i32(), "cu_seqlens"),
                                   _ptr(recv, _bf16(), "recv"), _ptr(w_home, _bf16(), "w_home"),
                                   _ptr(w_slots, _bf16(), "w_slots"), _ptr(y, _bf16(), "y"),
                                   _stream(stream)), "bep_grouped_gemm")


def bep_combine(ctx: Context, y, dest, gates, out, stream=None):
    c = ctx.cfg
    D = int(y.shape[-1])
    _numel(y, c.R * c.C * D, "y")
    _numel(dest, c.R * c.S * c.K, "dest")
    _numel(gates, c.R * c.S * c.K, "gates")
    _numel(out, c.R * c.S * D, "out")
    _check(load().bep_combine(ctx.handle, _ptr(y, _bf16(), "y"), _ptr(dest, _i32(), "dest"),
                              _ptr(gates, _f32(), "gates"), D, _ptr(out, _bf16(), "out"),
                              _stream(stream)), "bep_combine")


def bep_combine_bwd(ctx: Context, dout, dest, gates, dy, stream=None):
    c = ctx.cfg
    D = int(dout.shape[-1])
    _numel(dout, c.R * c.S * D, "dout")
    _numel(dest, c.R * c.S * c.K, "dest")
    _numel(gates, c.R * c.S * c.K, "gates")
    _numel(dy, c.R * c.C * D, "dy")
    _check(load().bep_combine_bwd(ctx.handle, _ptr(dout, _bf16(), "dout"),
                                  _ptr(dest, _i32(), "dest"), _ptr(gates, _f32(), "gates"), D,
                                  _ptr(dy, _bf16(), "dy"), _stream(stream)), "bep_combine_bwd")


def bep_grouped_gemm_vm(ctx: Context, cu_seqlens, recv, w_views, y, stream=None):
    """The grouped GEMM with each rank's weights as one [E+B, H, H'] tensor: w_views
    is [R, E+B, H, H'] (a WeightStore view or any tensor laid out that way)."""
    c = ctx.cfg
    _numel(cu_seqlens, c.R * (c.E + c.B + 1), "cu_seqlens")
    _numel(recv, c.R * c.C * c.H, "recv")
    _numel(w_views, c.R * (c.E + c.B) * c.H * c.Hp, "w_views")
    _numel(y, c.R * c.C * c.Hp, "y")
    _check(load().bep_grouped_gemm_vm(ctx.handle, _ptr(cu_seqlens, _i32(), "cu_seqlens"),
                                      _ptr(recv, _bf16(), "recv"),
                                      _ptr(w_views, _bf16(), "w_views"), _ptr(y, _bf16(), "y"),
                                      _stream(stream)), "bep_grouped_gemm_vm")


class WeightStore:
    """bep_weights: per layer home rows [E, H, H'], one prefetch-slot pool [R, B, H, H']
    shared by all layers, and per layer R aliased [E+B, H, H'] views (no copies).
    Tensors returned by home()/slots()/views() alias device memory the store owns:
    keep the store alive while they are used."""

    def __init__(self, cfg: Config, layers: int = 1):
        lib = load()
        c = _Config(cfg.R, cfg.E, cfg.B, cfg.K, cfg.S, cfg.H, cfg.Hp, cfg.mode)
        h = ctypes.c_void_p()
        _check(lib.bep_weights_create(ctypes.byref(c), int(layers), ctypes.byref(h)),
               "bep_weights_create")
        self.cfg, self.layers, self.handle = cfg, layers, h

    def _ptrs(self, layer):
        home, slots, views = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        _check(load().bep_weights_get(self.handle, int(layer), ctypes.byref(home),
                                      ctypes.byref(slots), ctypes.byref(views)),
               "bep_weights_get")
        return home.value, slots.value, views.value

    def _tensor(self, addr, shape):
        import torch
        n = 1
        for s_ in shape:
            n *= s_
        # zero-copy view of device memory the store owns, through the CUDA array interface
        class _Arr:
            __cuda_array_interface__ = {"shape": (n,), "typestr": "<i2", "data": (addr, False),
                                        "version": 3, "strides": None}
        return torch.as_tensor(_Arr(), device="cuda").view(torch.bfloat16).view(*shape)

    def home(self, layer):
        c = self.cfg
        return self._tensor(self._ptrs(layer)[0], (c.E, c.H, c.Hp))

    def slots(self):
        c = self.cfg
        return self._tensor(self._ptrs(0)[1], (c.R, c.B, c.H, c.Hp))

    def views(self, layer):
        c = self.cfg
        return self._tensor(self._ptrs(layer)[2], (c.R, c.E + c.B, c.H, c.Hp))

    def close(self):
        if self.handle:
            load().bep_weights_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bep_combine_dgates(ctx: Context, dout, y, dest, dgates, stream=None):
    c = ctx.cfg
    D = int(dout.shape[-1])
    _numel(dout, c.R * c.S * D, "dout")
    _numel(y, c.R * c.C * D, "y")
    _numel(dest, c.R * c.S * c.K, "dest")
    _numel(dgates, c.R * c.S * c.K, "dgates")
    _check(load().bep_combine_dgates(ctx.handle, _ptr(dout, _bf16(), "dout"), _ptr(y, _bf16(), "y"),
                                     _ptr(dest, _i32(), "dest"), D, _ptr(dgates, _f32(), "dgates"),
                                     _stream(stream)), "bep_combine_dgates")


def bep_set_comm_sms(ctx: Context, sms: int):
    _check(load().bep_set_comm_sms(ctx.handle, int(sms)), "bep_set_comm_sms")


def bep_wait_selftest(ctx: Context, timeout_us: int, stream=None):
    """Runs the bounded-wait failure path once: sets BEP_DERR_TIMEOUT after timeout_us."""
    _check(load().bep_wait_selftest(ctx.handle, int(timeout_us), _stream(stream)),
           "bep_wait_selftest")


def bep_dispatch_bwd(ctx: Context, drecv, dest, dx, stream=None):
    c = ctx.cfg
    _numel(drecv, c.R * c.C * c.H, "drecv")
    _numel(dest, c.R * c.S * c.K, "dest")
    _numel(dx, c.R * c.S * c.H, "dx")
    _check(load().bep_dispatch_bwd(ctx.handle, _ptr(drecv, _bf16(), "drecv"),
                                   _ptr(dest, _i32(), "dest"), _ptr(dx, _bf16(), "dx"),
                                   _stream(stream)), "bep_dispatch_bwd")


def bep_grouped_gemm_dx(ctx: Context, cu_seqlens, dy, w_home, w_slots, drecv, stream=None):
    c = ctx.cfg
    _numel(cu_seqlens, c.R * (c.E + c.B + 1), "cu_seqlens")
    _numel(dy, c.R * c.C * c.Hp, "dy")
    _numel(w_home, c.E * c.H * c.Hp, "w_home")
    _numel(w_slots, c.R * c.B * c.H * c.Hp, "w_slots")
    _numel(drecv, c.R * c.C * c.H, "drecv")
    _check(load().bep_grouped_gemm_dx(ctx.handle, _ptr(cu_seqlens, _i32(), "cu_seqlens"),
                                      _ptr(dy, _bf16(), "dy"), _ptr(w_home, _bf16(), "w_home"),
                                      _ptr(w_slots, _bf16(), "w_slots"),
                                      _ptr(drecv, _bf16(), "drecv"), _stream(stream)),
           "bep_grouped_gemm_dx")


def _grouped_gemm_dw(name, ctx, cu_seqlens, recv, dy, g_home, red, stream):
    c = ctx.cfg
    _numel(cu_seqlens, c.R * (c.E + c.B + 1), "cu_seqlens")
    _numel(recv, c.R * c.C * c.H, "recv")
    _numel(dy, c.R * c.C * c.Hp, "dy")
    _numel(g_home, c.E * c.H * c.Hp, "g_home")
    _numel(red, c.R * c.B * c.H * c.Hp, "red")
    _check(getattr(load(), name)(ctx.handle, _ptr(cu_seqlens, _i32(), "cu_seqlens"),
                                 _ptr(recv, _bf16(), "recv"), _ptr(dy, _bf16(), "dy"),
                                 _ptr(g_home, _f32(), "g_home"), _ptr(red, _f32(), "red"),
                                 _stream(stream)), name)


def bep_grouped_gemm_dw(ctx: Context, cu_seqlens, recv, dy, g_home, red, stream=None):
    """g_home[e] / red[u][j] += recv[seg]^T @ dy[seg] for every non-empty segment."""
    _grouped_gemm_dw("bep_grouped_gemm_dw", ctx, cu_seqlens, recv, dy, g_home, red, stream)


def bep_grouped_gemm_dw_overwrite(ctx: Context, cu_seqlens, recv, dy, g_home, red, stream=None):
    """g_home[e] = its home segment's recv^T @ dy (zeros when empty) for every expert;
    red[u][j] = recv[seg]^T @ dy[seg] for every non-empty slot segment."""
    _grouped_gemm_dw("bep_grouped_gemm_dw_overwrite", ctx, cu_seqlens, recv, dy, g_home, red,
                     stream)


def bep_reduce_grad(ctx: Context, slot_expert, g_home, red, stream=None):
    c = ctx.cfg
    _numel(slot_expert, c.R * c.B, "slot_expert")
    _numel(g_home, c.E * c.H * c.Hp, "g_home")
    _numel(red, c.R * c.B * c.H * c.Hp, "red")
    _check(load().bep_reduce_grad(ctx.handle, _ptr(slot_expert, _i32(), "slot_expert"),
                                  _ptr(g_home, _f32(), "g_home"), _ptr(red, _f32(), "red"),
                                  _stream(stream)), "bep_reduce_grad")


def bep_status(ctx: Context, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(load().bep_status(ctx.handle, ctypes.byref(v), _stream(stream)), "bep_status")
    return int(v.value)


def bep_clear_status(ctx: Context, stream=None):
    _check(load().bep_clear_status(ctx.handle, _stream(stream)), "bep_clear_status")


class Buffers:
    """Device tensors of one MoE projection step, allocated once (static shapes)."""

    def __init__(self, cfg: Config, device="cuda", with_grad=False, D_bwd=None):
        import torch
        R, S, K, E, B, H, Hp = cfg.R, cfg.S, cfg.K, cfg.E, cfg.B, cfg.H, cfg.Hp
        dev = torch.device(device)
        self.cu_seqlens = torch.zeros((R, E + B + 1), dtype=torch.int32, device=dev)
        self.slot_expert = torch.full((R, B), -1, dtype=torch.int32, device=dev)
        self.dest = torch.zeros((R, S, K), dtype=torch.int32, device=dev)
        self.maxvio = torch.zeros(1, dtype=torch.float64, device=dev)
        self.recv = torch.empty((R * S * K, H), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((R * S * K, Hp), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((R, S, Hp), dtype=torch.bfloat16, device=dev)
        if with_grad:
            D = Hp if D_bwd is None else D_bwd
            self.dy = torch.empty((R * S * K, D), dtype=torch.bfloat16, device=dev)


def forward(ctx: Context, buf: Buffers, topk, x, gates, w_home, w_slots, stream=None):
    """plan -> prefetch_weight -> dispatch -> grouped_gemm -> combine, all queued on one stream."""
    bep_plan(ctx, topk, buf.cu_seqlens, buf.slot_expert, buf.dest, buf.maxvio, stream)
    bep_prefetch_weight(ctx, buf.slot_expert, w_home, w_slots, stream)
    bep_dispatch(ctx, x, buf.dest, buf.recv, stream)
    bep_grouped_gemm(ctx, buf.cu_seqlens, buf.recv, w_home, w_slots, buf.y, stream)
    bep_combine(ctx, buf.y, buf.dest, gates, buf.out, stream)
    return buf.out


def backward_fold(ctx: Context, buf: Buffers, dout, gates, slot_expert, g_home, red, stream=None):
    """combine backward (dy) and reduce_grad of the replica gradients into the home rows."""
    bep_combine_bwd(ctx, dout, buf.dest, gates, buf.dy, stream)
    bep_reduce_grad(ctx, slot_expert, g_home, red, stream)
    return buf.dy
