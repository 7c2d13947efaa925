"""Seeded synthetic inputs for balanced expert-parallel dispatch.

This module serves the oracle and the CUDA path alike and holds none of the
method's arithmetic: it draws routings, tokens, weights and gates, and nothing
else. Recipes (stated once more in the design notes):

* routing: every token picks K distinct experts by Gumbel-top-K over a
  popularity vector p (Plackett-Luce sampling without replacement); the k order
  is the order of the perturbed scores, highest first;
* popularity: Zipf (p_e proportional to (e+1)^-s, expert 0 hottest) or
  Dirichlet(alpha) drawn as normalised Gamma(alpha) variates; alpha per
  (workload, maxvio target, seed) comes from ``alpha_table.json``, which the
  calibration script beside the tests writes;
* ``hot_group``: the largest popularities are moved onto one home group's
  experts (inference workload with overflow);
* tokens: bf16 of U[-1, 1]; weights: bf16 of N(0, 0.02); gates: softmax over
  each token's K logits drawn N(0, 1), in fp32; reduce buffers: N(0, 1e-3).

Generators come in two flavours: numpy on the host (small cases, oracle
inputs) and torch on a CUDA device (bench-sized tensors, GB of weights).
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))

MODE_TRAIN = 0
MODE_INFER = 1


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    S: int
    E: int
    K: int
    H: int
    Hp: int
    B: int
    mode: int
    hot_group: bool = False

    @property
    def C(self):
        return self.S * self.K


# The five workloads of the balanced-dispatch study, by what they are.
WORKLOADS = {
    # tiny training case, Zipf(1.2) popularity
    "tiny_r2_e8": Workload("tiny_r2_e8", R=2, S=64, E=8, K=2, H=128, Hp=64, B=4, mode=MODE_TRAIN),
    # training, 8 ranks, 64 experts
    "train_r8_e64": Workload("train_r8_e64", R=8, S=1024, E=64, K=4, H=1024, Hp=512, B=8,
                             mode=MODE_TRAIN),
    # bench-shaped training: S=8192/rank, E=384, K=8, H=7168, H'=2048, B=48
    "bench_r8_e384": Workload("bench_r8_e384", R=8, S=8192, E=384, K=8, H=7168, Hp=2048, B=48,
                              mode=MODE_TRAIN),
    # inference with overflow, hot experts on one home rank, B=4 < E/R
    "infer_r8_e384_b4": Workload("infer_r8_e384_b4", R=8, S=512, E=384, K=8, H=7168, Hp=2048,
                                 B=4, mode=MODE_INFER, hot_group=True),
    # backward fold: reduce_grad on [E+B, 2048, 1024] fp32 and combine backward
    "grad_r8_e64": Workload("grad_r8_e64", R=8, S=1024, E=64, K=4, H=2048, Hp=1024, B=8,
                            mode=MODE_TRAIN),
    # the bench's expert shape (H=7168, H'=2048) on a few GB: profiling captures
    "gemm_probe_r4_e16": Workload("gemm_probe_r4_e16", R=4, S=2048, E=16, K=8, H=7168, Hp=2048,
                                  B=4, mode=MODE_TRAIN),
    # about 1,700 rows per segment, like the bench-shaped workload's ~1,400: profiling
    # of the weight-gradient GEMM, whose cost grows with the number of segments
    "dw_probe_r4_e16_s1024": Workload("dw_probe_r4_e16_s1024", R=4, S=1024, E=16, K=8, H=7168,
                                      Hp=2048, B=4, mode=MODE_TRAIN),
}

MAXVIO_TARGETS = {
    "tiny_r2_e8": (None,),
    "train_r8_e64": (0.2, 1.0, 10.0),
    "bench_r8_e384": (0.2, 1.0, 10.0, 20.0),
    "infer_r8_e384_b4": (1.0, 20.0),
    "grad_r8_e64": (10.0,),
    "gemm_probe_r4_e16": (None,),
    "dw_probe_r4_e16_s1024": (None,),
}


# ----------------------------------------------------------------------------
# popularity and routing
# ----------------------------------------------------------------------------
def zipf_popularity(E: int, s: float = 1.2) -> np.ndarray:
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-s)
    return p / p.sum()


def dirichlet_popularity(E: int, alpha: float, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64([seed, 0x5eed]))
    g = rng.standard_gamma(alpha, size=E)
    g = np.maximum(g, np.finfo(np.float64).tiny)
    return g / g.sum()


def concentrate_on_group(p: np.ndarray, R: int, group: int = 0) -> np.ndarray:
    """Reorder p so the E/R largest popularities sit on home group `group`'s experts."""
    E = len(p)
    G = E // R
    order = np.argsort(-p, kind="stable")
    out = np.empty_like(p)
    hot = order[:G]
    cold = order[G:]
    out[group * G:(group + 1) * G] = p[hot]
    rest = [e for e in range(E) if not (group * G <= e < (group + 1) * G)]
    out[rest] = p[cold]
    return out


def gumbel_topk(R: int, S: int, K: int, p: np.ndarray, seed: int, block: int = 8192) -> np.ndarray:
    """topk [R,S,K] int32: each token draws K distinct experts from popularity p
    (Plackett-Luce, realised as the K largest log p_e + Gumbel noise)."""
    E = len(p)
    logp = np.log(np.maximum(p, 1e-300))
    rng = np.random.Generator(np.random.PCG64([seed, 0x70c]))
    n = R * S
    out = np.empty((n, K), np.int32)
    for a in range(0, n, block):
        b = min(n, a + block)
        u = rng.random((b - a, E))
        score = logp[None, :] - np.log(-np.log(np.clip(u, 1e-300, 1.0 - 1e-16)))
        idx = np.argpartition(-score, K - 1, axis=1)[:, :K]
        sc = np.take_along_axis(score, idx, axis=1)
        o = np.argsort(-sc, axis=1, kind="stable")
        out[a:b] = np.take_along_axis(idx, o, axis=1)
    return out.reshape(R, S, K)


def round_robin_topk(R: int, S: int, K: int, E: int) -> np.ndarray:
    """topk[r,t,k] = ((r*S + t)*K + k) mod E: K consecutive ids per token
    (distinct when K <= E)."""
    i = np.arange(R * S * K, dtype=np.int64)
    return (i % E).astype(np.int32).reshape(R, S, K)


def _alpha_table():
    path = os.path.join(_HERE, "alpha_table.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        return json.load(f)


def alpha_for(workload: str, target: float, seed: int) -> float:
    tab = _alpha_table()
    key = f"{workload}|{target:g}|{seed}"
    if key not in tab:
        raise KeyError(f"no calibrated alpha for {key}; run tests/golden/calibrate_alpha.py")
    return float(tab[key])


def routing(wl: Workload, target, seed: int, alpha: float | None = None) -> np.ndarray:
    """The workload's routing at a maxvio target (None: Zipf(1.2) popularity)."""
    if target is None:
        p = zipf_popularity(wl.E, 1.2)
    else:
        a = alpha if alpha is not None else alpha_for(wl.name, target, seed)
        p = dirichlet_popularity(wl.E, a, seed)
        if wl.hot_group:
            p = concentrate_on_group(p, wl.R, 0)
    return gumbel_topk(wl.R, wl.S, wl.K, p, seed)


# ----------------------------------------------------------------------------
# values (host)
# ----------------------------------------------------------------------------
def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def tokens_host(shape, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64([seed, 0x70e]))
    return _to_bf16_bits(rng.uniform(-1.0, 1.0, size=shape).astype(np.float32))


def weights_host(shape, seed: int, std: float = 0.02) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64([seed, 0x3e1]))
    return _to_bf16_bits((rng.standard_normal(size=shape) * std).astype(np.float32))


def gates_host(R: int, S: int, K: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64([seed, 0x9a7]))
    z = rng.standard_normal(size=(R, S, K)).astype(np.float32)
    z = z - z.max(axis=2, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=2, keepdims=True)).astype(np.float32)


def normal_host(shape, seed: int, std: float) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64([seed, 0xf32]))
    return (rng.standard_normal(size=shape) * std).astype(np.float32)


def reduce_buffer_host(R, B, H, Hp, slot_expert: np.ndarray, seed: int, std=1e-3) -> np.ndarray:
    """red [R,B,H,H'] fp32: N(0, std) in the slots the plan uses, zero elsewhere."""
    red = np.zeros((R, B, H, Hp), np.float32)
    for u in range(R):
        for j in range(B):
            if slot_expert[u, j] >= 0:
                red[u, j] = normal_host((H, Hp), seed * 1000003 + u * B + j, std)
    return red


# ----------------------------------------------------------------------------
# values (device; bench-sized)
# ----------------------------------------------------------------------------
def tokens_device(shape, seed: int, device="cuda"):
    import torch
    g = torch.Generator(device=device).manual_seed(seed * 7919 + 1)
    t = torch.empty(shape, dtype=torch.float32, device=device).uniform_(-1.0, 1.0, generator=g)
    return t.to(torch.bfloat16)


def weights_device(shape, seed: int, std: float = 0.02, device="cuda", chunk_rows: int = 16):
    """bf16 N(0, std) drawn in row chunks to bound the fp32 temporary."""
    import torch
    g = torch.Generator(device=device).manual_seed(seed * 7919 + 2)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for a in range(0, shape[0], chunk_rows):
        b = min(shape[0], a + chunk_rows)
        tmp = torch.empty((b - a, flat.shape[1]), dtype=torch.float32, device=device)
        tmp.normal_(0.0, std, generator=g)
        flat[a:b].copy_(tmp)
        del tmp
    return out
