"""Pins for the oracle, on the CPU: every oracle function is checked against
something other than itself -- hand-worked examples, closed forms, brute force
on tiny inputs, and special cases that reduce to a library routine."""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 rounding
def _torch_bf16_bits(f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_matches_torch_on_random_bit_patterns():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # ties and near-ties on every exponent, subnormals, the overflow edge, infinities
    specials = []
    for hi in (0x0000, 0x0001, 0x0080, 0x3f80, 0x3f81, 0x7f7f, 0x7f7e, 0x8001, 0xbf80, 0xff7f):
        for lo in (0x0000, 0x7fff, 0x8000, 0x8001, 0xffff):
            specials.append((hi << 16) | lo)
    specials += [0x7f800000, 0xff800000]
    bits = np.concatenate([bits, np.array(specials, np.uint32)])
    f = bits.view(np.float32)
    keep = ~np.isnan(f)  # NaN payloads are outside the parity contract
    f = f[keep]
    ours = np.array([oracle.f32_to_bf16_scalar(float(v)) for v in f], np.uint16)
    np.testing.assert_array_equal(ours, _torch_bf16_bits(f))


def test_bf16_widening_is_exact():
    h = np.arange(0, 2**16, dtype=np.uint16)
    ours = oracle.bf16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    finite = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[finite].view(np.uint32), ref[finite].view(np.uint32))


# ---------------------------------------------------------------- histogram / maxvio
def test_histogram_matches_bincount():
    wl = synth.WORKLOADS["train_r8_e64"]
    topk = synth.gumbel_topk(wl.R, wl.S, wl.K, synth.zipf_popularity(wl.E, 1.0), seed=3)
    np.testing.assert_array_equal(oracle.histogram(topk, wl.E),
                                  np.bincount(topk.ravel(), minlength=wl.E))


def test_histogram_rejects_bad_ids():
    topk = np.zeros((1, 2, 2), np.int32)
    topk[0, 0] = [0, 1]
    topk[0, 1] = [2, 2]
    with pytest.raises(oracle.OracleError) as ei:
        oracle.histogram(topk, 4)
    assert ei.value.code == -2
    topk[0, 1] = [2, 4]
    with pytest.raises(oracle.OracleError) as ei:
        oracle.histogram(topk, 4)
    assert ei.value.code == -1
    topk[0, 1] = [-1, 3]
    with pytest.raises(oracle.OracleError) as ei:
        oracle.histogram(topk, 4)
    assert ei.value.code == -1


@pytest.mark.parametrize("R,S,K,E", [(2, 64, 2, 8), (8, 1024, 4, 64), (8, 6144, 8, 384)])
def test_maxvio_round_robin_is_zero(R, S, K, E):
    topk = synth.round_robin_topk(R, S, K, E)
    assert (R * S * K) % E == 0
    assert oracle.maxvio(oracle.histogram(topk, E), R * S * K) == 0.0


@pytest.mark.parametrize("R,S,K,E", [(2, 64, 2, 8), (8, 1024, 4, 64), (8, 512, 8, 384)])
def test_maxvio_all_tokens_same_experts_is_E_over_K_minus_1(R, S, K, E):
    # every token picks experts 0..K-1: T_0 = R*S, Tbar = R*S*K/E -> E/K - 1
    topk = np.broadcast_to(np.arange(K, dtype=np.int32), (R, S, K)).copy()
    mv = oracle.maxvio(oracle.histogram(topk, E), R * S * K)
    assert mv == E / K - 1


def test_maxvio_single_rounding():
    # T = [3, 0, 0], RSK = 3: (3*3 - 3)/3 = 2 exactly; T=[2,1,0]: (3*2-3)/3 = 1
    assert oracle.maxvio(np.array([3, 0, 0]), 3) == 2.0
    assert oracle.maxvio(np.array([2, 1, 0]), 3) == 1.0
    # 1/3 - 1 shape: E=7, T_max=5, RSK=21 -> (35-21)/21 = 2/3 rounded once
    assert oracle.maxvio(np.array([5, 4, 3, 3, 2, 2, 2]), 21) == 14.0 / 21.0
    assert oracle.maxvio(np.zeros(4, np.int64), 0) == 0.0


# ---------------------------------------------------------------- the tree
def test_tree_worked_examples():
    with open(os.path.join(GOLD, "tree_worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        parent, inflow, order = oracle.tree(c["L"], c["C"])
        assert parent.tolist() == c["parent"], c
        assert inflow.tolist() == c["inflow"], c
        assert order.tolist() == c["order"], c


def _forest_flows(parent, L, C):
    """Brute-force feasibility of a parent function: returns inflow per node or None.
    Flow into u from its parent must equal C*|subtree(u)| - sum L over the subtree
    (so every node ends with exactly C), be >= 0, and every node must keep a
    non-negative number of its own slots (give no more than it owns)."""
    R = len(parent)
    # acyclic?
    for u in range(R):
        seen, v = set(), u
        while v != -1:
            if v in seen:
                return None
            seen.add(v)
            v = parent[v]
    children = [[c for c in range(R) if parent[c] == u] for u in range(R)]

    def sub(u):
        out = [u]
        for c in children[u]:
            out += sub(c)
        return out

    inflow = [0] * R
    for u in range(R):
        s = sub(u)
        need = C * len(s) - sum(L[v] for v in s)
        if parent[u] == -1:
            if need != 0:
                return None
        else:
            if need < 0:
                return None
            inflow[u] = need
    for u in range(R):
        give = sum(inflow[c] for c in children[u])
        if L[u] - give < 0:
            return None
        if L[u] - give + inflow[u] != C:
            return None
    return inflow


def _all_loads(R, C):
    total = R * C
    for L in itertools.product(range(total + 1), repeat=R - 1):
        last = total - sum(L)
        if last >= 0:
            yield list(L) + [last]


@pytest.mark.parametrize("R,C", [(2, 3), (3, 2), (3, 3), (4, 2)])
def test_tree_valid_on_every_load_vector_brute_force(R, C):
    parents = list(itertools.product(range(-1, R), repeat=R))
    parents = [p for p in parents if all(p[u] != u for u in range(R))]
    for L in _all_loads(R, C):
        feasible = [p for p in parents if _forest_flows(list(p), L, C) is not None]
        assert feasible, L                      # a one-parent-per-rank plan always exists
        parent, inflow, _ = oracle.tree(L, C)
        flows = _forest_flows(parent.tolist(), L, C)
        assert flows is not None, (L, parent)   # the rule's plan is one of them
        assert list(inflow) == flows


def test_tree_valid_on_random_loads():
    rng = np.random.default_rng(1)
    for trial in range(3000):
        R = int(rng.integers(2, 9))
        C = int(rng.integers(1, 50))
        # random composition of R*C into R parts, some extreme
        if trial % 5 == 0:
            L = np.zeros(R, np.int64)
            L[rng.integers(R)] = R * C
        else:
            cuts = np.sort(rng.integers(0, R * C + 1, size=R - 1))
            L = np.diff(np.concatenate([[0], cuts, [R * C]]))
        parent, inflow, _ = oracle.tree(L, C)
        flows = _forest_flows(parent.tolist(), L.tolist(), C)
        assert flows is not None and list(inflow) == flows, (L, parent)


# ---------------------------------------------------------------- the plan
def test_plan_worked_examples():
    with open(os.path.join(GOLD, "plan_worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        topk = np.array(c["topk"], np.int32)
        p = oracle.plan(topk, c["E"], c["B"], c["mode"])
        assert p.maxvio == c["maxvio"], c["name"]
        assert p.parent.tolist() == c["parent"], c["name"]
        assert p.inflow.tolist() == c["inflow"], c["name"]
        assert p.slot_expert.tolist() == c["slot_expert"], c["name"]
        assert p.cu.tolist() == c["cu"], c["name"]
        assert p.dest.tolist() == c["dest"], c["name"]
        assert oracle.check_plan(topk, c["E"], c["B"], c["mode"], p.cu, p.slot_expert, p.dest) == 0


def _py_check(topk, E, B, mode, cu, se, dest):
    """Independent pure-Python restatement of plan validity (tiny inputs)."""
    R, S, K = topk.shape
    G, C = E // R, S * K
    if any(cu[u][0] != 0 or cu[u][-1] != C for u in range(R)):
        return False
    flat = dest.ravel().tolist()
    if sorted(flat) != list(range(R * C)):
        return False
    groups = [set() for _ in range(R)]
    for i, d in enumerate(flat):
        e = int(topk.ravel()[i])
        u, pos = divmod(d, C)
        row = max(r for r in range(E + B) if cu[u][r] <= pos and pos < cu[u][r + 1])
        if row < E:
            if row != e:
                return False
            if e // G != u and mode == 0:
                return False
        elif se[u][row - E] != e:
            return False
        if e // G != u:
            groups[u].add(e // G)
    return all(len(g) <= 1 for g in groups)


def _enumerate_routings(R, S, K, E):
    tok_choices = list(itertools.permutations(range(E), K))
    for combo in itertools.product(tok_choices, repeat=R * S):
        yield np.array(combo, np.int32).reshape(R, S, K)


@pytest.mark.parametrize("R,S,K,E,B,mode", [
    (2, 2, 1, 4, 2, 0), (2, 2, 1, 4, 1, 1), (3, 2, 1, 3, 1, 0),
    (2, 2, 2, 4, 2, 0), (2, 2, 2, 4, 1, 1),
])
def test_plan_valid_on_every_micro_routing(R, S, K, E, B, mode):
    n = 0
    for topk in _enumerate_routings(R, S, K, E):
        p = oracle.plan(topk, E, B, mode)
        assert oracle.check_plan(topk, E, B, mode, p.cu, p.slot_expert, p.dest) == 0, topk
        if n % 7 == 0:  # the pure-Python checker is slow; sample it
            assert _py_check(topk, E, B, mode, p.cu, p.slot_expert, p.dest), topk
        T = np.bincount(topk.ravel(), minlength=E)
        assert p.maxvio == (E * T.max() - topk.size) / topk.size
        n += 1
    assert n == len(list(itertools.permutations(range(E), K))) ** (R * S)


@pytest.mark.parametrize("R,S,K,E", [(2, 64, 2, 8), (8, 1024, 4, 64), (8, 6144, 8, 384)])
def test_balanced_routing_is_stable_argsort(R, S, K, E):
    """Round-robin routing loads every group with exactly C: no replicas, every
    slot stays home, and dest is the stable argsort position of its expert id."""
    topk = synth.round_robin_topk(R, S, K, E)
    p = oracle.plan(topk, E, E // R, 0)
    assert (p.parent == -1).all() and (p.slot_expert == -1).all()
    flat = topk.ravel()
    order = np.argsort(flat, kind="stable")
    expect = np.empty_like(order)
    expect[order] = np.arange(len(order))
    np.testing.assert_array_equal(p.dest.ravel(), expect)
    counts = np.bincount(flat, minlength=E).reshape(R, E // R)
    for u in range(R):
        lens = np.diff(p.cu[u])
        np.testing.assert_array_equal(lens[u * (E // R):(u + 1) * (E // R)], counts[u])
        assert lens.sum() == S * K


@pytest.mark.parametrize("name,target", [("train_r8_e64", 0.2), ("train_r8_e64", 10.0),
                                         ("tiny_r2_e8", None)])
def test_plan_valid_on_workloads(name, target):
    wl = synth.WORKLOADS[name]
    topk = synth.routing(wl, target, 0, alpha=None if target is None else
                         {0.2: 3000.0, 10.0: 0.05}[target])
    p = oracle.plan(topk, wl.E, wl.B, wl.mode)
    assert oracle.check_plan(topk, wl.E, wl.B, wl.mode, p.cu, p.slot_expert, p.dest) == 0
    # training: at most one remote group per rank and B = E/R
    G = wl.E // wl.R
    for u in range(wl.R):
        used = p.slot_expert[u][p.slot_expert[u] >= 0]
        assert len({int(e) // G for e in used}) <= 1
        if len(used):
            assert {int(e) // G for e in used} == {int(p.parent[u])}


def test_infer_overflow_reads_home_rows():
    wl = synth.WORKLOADS["infer_r8_e384_b4"]
    topk = synth.routing(wl, 20.0, 0, alpha=0.02)
    p = oracle.plan(topk, wl.E, wl.B, wl.mode)
    assert oracle.check_plan(topk, wl.E, wl.B, wl.mode, p.cu, p.slot_expert, p.dest) == 0
    G = wl.E // wl.R
    n_overflow = 0
    for u in range(wl.R):
        lens = np.diff(p.cu[u])
        for e in range(wl.E):
            if e // G != u and lens[e] > 0:
                n_overflow += 1
                assert e not in p.slot_expert[u]
                # overflow only happens once every slot is taken
                assert (p.slot_expert[u] >= 0).all()
    assert n_overflow > 0


def test_check_plan_catches_planted_mistakes():
    wl = synth.WORKLOADS["tiny_r2_e8"]
    topk = synth.routing(wl, None, 0)
    p = oracle.plan(topk, wl.E, wl.B, wl.mode)
    ok = lambda cu, se, d: oracle.check_plan(topk, wl.E, wl.B, wl.mode, cu, se, d)  # noqa: E731
    assert ok(p.cu, p.slot_expert, p.dest) == 0
    d = p.dest.copy().ravel()
    d[0], d[1] = d[1], d[0]                    # two different experts swap places
    assert ok(p.cu, p.slot_expert, d.reshape(p.dest.shape)) == 3
    d = p.dest.copy().ravel()
    flat = topk.ravel()
    i, j = np.flatnonzero(flat == flat[0])[:2]
    d[j] = d[i]                                # two slots of one expert, one place
    assert ok(p.cu, p.slot_expert, d.reshape(p.dest.shape)) == 2
    d = p.dest.copy().ravel()
    d[3] = wl.R * wl.C                         # outside the receive space
    assert ok(p.cu, p.slot_expert, d.reshape(p.dest.shape)) == 2
    cu = p.cu.copy()
    cu[1, -1] += 1                             # a rank off by one slot
    assert ok(cu, p.slot_expert, p.dest) == 1
    se = p.slot_expert.copy()
    used = np.argwhere(se >= 0)
    u, j = used[0]
    se[u, j] = (se[u, j] + 1) % wl.E           # a slot naming the wrong expert
    assert ok(p.cu, se, p.dest) in (3, 6)


# ---------------------------------------------------------------- dispatch / combine
def _small_problem(seed=0, R=2, S=37, K=4, E=16, H=40, B=None, mode=0, D=24):
    B = E // R if B is None else B
    topk = synth.gumbel_topk(R, S, K, synth.zipf_popularity(E, 1.1), seed)
    p = oracle.plan(topk, E, B, mode)
    x = synth.tokens_host((R, S, H), seed)
    g = synth.gates_host(R, S, K, seed)
    y = synth.tokens_host((R * S * K, D), seed + 100)
    return topk, p, x, g, y


def test_dispatch_is_scatter_of_repeated_rows():
    topk, p, x, g, y = _small_problem()
    R, S, H = x.shape
    K = topk.shape[2]
    recv = oracle.dispatch(x, p.dest)
    expect = np.zeros_like(recv)
    expect[p.dest.ravel()] = np.repeat(x.reshape(R * S, H), K, axis=0)
    np.testing.assert_array_equal(recv, expect)


def test_dispatch_combine_round_trip_is_identity():
    """gates = 1/K with K a power of two: out = sum_k x/K = x exactly."""
    topk, p, x, g, y = _small_problem(K=4)
    K = topk.shape[2]
    recv = oracle.dispatch(x, p.dest)
    gates = np.full(topk.shape, 1.0 / K, np.float32)
    out = oracle.combine(recv, p.dest, gates)
    np.testing.assert_array_equal(out, x)


def test_combine_one_hot_gates_select_a_row():
    topk, p, x, g, y = _small_problem()
    R, S, K = topk.shape
    rng = np.random.default_rng(5)
    hot = rng.integers(0, K, size=(R, S))
    gates = np.zeros(topk.shape, np.float32)
    gates[np.arange(R)[:, None], np.arange(S)[None, :], hot] = 1.0
    out = oracle.combine(y, p.dest, gates)
    pick = np.take_along_axis(p.dest, hot[:, :, None], axis=2)[:, :, 0]
    np.testing.assert_array_equal(out, y[pick])


def test_combine_single_k_matches_torch_product():
    topk, p, x, g, y = _small_problem(K=1)
    out = oracle.combine(y, p.dest, g)
    yf = torch.from_numpy(oracle.bf16_to_f32(y))
    ref = (torch.from_numpy(g)[..., 0:1] * yf[torch.from_numpy(p.dest[..., 0]).long()])
    np.testing.assert_array_equal(out, _torch_bf16_bits(ref.numpy()))


def test_combine_exact_on_dyadic_values():
    """Gates 2^-j and small-integer Y: every partial sum is exact in fp32, so the
    result is the exact weighted sum (computed here in float64), then bf16."""
    topk, p, x, g, y = _small_problem(K=4, D=16)
    R, S, K = topk.shape
    rng = np.random.default_rng(7)
    gates = (2.0 ** -rng.integers(0, 4, size=topk.shape)).astype(np.float32)
    yv = rng.integers(-8, 9, size=y.shape).astype(np.float32)
    ybits = _torch_bf16_bits(yv)
    out = oracle.combine(ybits, p.dest, gates)
    exact = (gates[..., None].astype(np.float64) *
             yv[p.dest].astype(np.float64)).sum(axis=2)
    np.testing.assert_array_equal(out, _torch_bf16_bits(exact.astype(np.float32)))


def test_combine_within_fp32_bound_of_exact():
    topk, p, x, g, y = _small_problem(K=8, E=32, D=64)
    out = oracle.bf16_to_f32(oracle.combine(y, p.dest, g)).astype(np.float64)
    yf = oracle.bf16_to_f32(y).astype(np.float64)
    exact = (g[..., None].astype(np.float64) * yf[p.dest]).sum(axis=2)
    # one bf16 rounding (2^-8 relative) dominates K fp32 roundings
    bound = 2.0 ** -8 * np.abs(exact) + 8 * 2.0 ** -23 * (np.abs(g[..., None]) * np.abs(yf[p.dest])).sum(2)
    assert (np.abs(out - exact) <= bound + 1e-30).all()


def test_combine_bwd_matches_torch():
    topk, p, x, g, y = _small_problem(D=24)
    R, S, K = topk.shape
    dout = synth.tokens_host((R, S, 24), 9)
    dy = oracle.combine_bwd(dout, p.dest, g)
    prod = torch.from_numpy(g)[..., None] * torch.from_numpy(oracle.bf16_to_f32(dout))[:, :, None, :]
    ref = np.zeros_like(dy)
    ref[p.dest.ravel()] = _torch_bf16_bits(prod.numpy()).reshape(R * S * K, 24)
    np.testing.assert_array_equal(dy, ref)


# ---------------------------------------------------------------- prefetch / reduce_grad
def _expert_pattern(e, H, Hp):
    """A weight row that spells out its own expert id: element (h, h') is the
    integer (e*131 + h*7 + h'*3) mod 251, exact in bf16 (every integer below 256 is)."""
    h = np.arange(H)[:, None]
    hp = np.arange(Hp)[None, :]
    return _torch_bf16_bits(((e * 131 + h * 7 + hp * 3) % 251).astype(np.float32))


@pytest.mark.parametrize("seed,R,E,S,K", [(0, 2, 16, 37, 4), (1, 4, 16, 60, 3), (2, 8, 32, 50, 4)])
def test_prefetch_slots_hold_their_parents_experts(seed, R, E, S, K):
    """Training mode ([P4] "The memory contract"): B = E/R and a replica of expert e
    on rank u sits in slot j = e - parent(u)*G, so slot j of a rank that takes
    replicas must hold expert parent(u)*G + j. Every home row is filled with a
    pattern that encodes its expert id; the expected slot contents are that
    pattern evaluated at the expert the training rule names -- not an index into
    w_home -- and every slot the plan leaves unused keeps its sentinel bits."""
    G, B, H, Hp = E // R, E // R, 6, 10
    topk = synth.gumbel_topk(R, S, K, synth.zipf_popularity(E, 1.6), seed)
    p = oracle.plan(topk, E, B, oracle.MODE_TRAIN)
    assert (p.slot_expert >= 0).any()
    w_home = np.stack([_expert_pattern(e, H, Hp) for e in range(E)])
    sentinel = np.uint16(0x7FC1)      # a NaN pattern no pattern element can take
    w_slots = np.full((R, B, H, Hp), sentinel, np.uint16)
    oracle.prefetch(w_home, p.slot_expert, w_slots)
    for u in range(R):
        # the slots a rank's segment rows E..E+B-1 actually use (cu_seqlens)
        used_rows = [j for j in range(B) if p.cu[u, E + j + 1] > p.cu[u, E + j]]
        assert used_rows == [j for j in range(B) if p.slot_expert[u, j] >= 0]
        for j in range(B):
            if j in used_rows:
                assert p.parent[u] >= 0
                np.testing.assert_array_equal(w_slots[u, j],
                                              _expert_pattern(p.parent[u] * G + j, H, Hp))
            else:
                assert (w_slots[u, j] == sentinel).all()


def test_prefetch_inference_slots_hold_the_top_counted_remote_experts():
    """Inference mode (B < E/R): a rank's slots hold, in ascending id, the B remote
    experts with the most of its token-slots ([P4] "The memory contract", with the
    overflow reading), and each such slot's contents are that expert's pattern."""
    R, S, K, E, B, H, Hp = 4, 80, 4, 32, 2, 4, 8
    G = E // R
    pop = np.full(E, 1e-6)
    pop[:G] = np.linspace(1.0, 2.0, G)
    topk = synth.gumbel_topk(R, S, K, pop / pop.sum(), 3)
    p = oracle.plan(topk, E, B, oracle.MODE_INFER)
    w_home = np.stack([_expert_pattern(e, H, Hp) for e in range(E)])
    w_slots = np.zeros((R, B, H, Hp), np.uint16)
    oracle.prefetch(w_home, p.slot_expert, w_slots)
    C = S * K
    moved = 0
    for u in range(R):
        # count, from dest and topk alone, the token-slots of each remote expert on rank u
        on_u = (p.dest // C) == u
        cnt = np.bincount(topk[on_u].ravel(), minlength=E)
        remote = [e for e in range(E) if cnt[e] > 0 and e // G != u]
        top = sorted(sorted(remote, key=lambda e: (-cnt[e], e))[:B])
        moved += len(top)
        for j, e in enumerate(top):
            np.testing.assert_array_equal(w_slots[u, j], _expert_pattern(e, H, Hp))
        for j in range(len(top), B):
            assert not w_slots[u, j].any()
    assert moved > 0


def test_reduce_grad_integer_values_exact_and_zeroed():
    R, B, E, H, Hp = 4, 3, 12, 5, 7
    rng = np.random.default_rng(2)
    se = np.full((R, B), -1, np.int32)
    # ranks 1..3 hold replicas of group 0's experts (0,1,2) in various slots
    se[1] = [0, 1, -1]
    se[2] = [0, -1, 2]
    se[3] = [-1, 1, 2]
    G0 = rng.integers(-100, 100, size=(E, H, Hp)).astype(np.float32)
    red = np.zeros((R, B, H, Hp), np.float32)
    for u in range(R):
        for j in range(B):
            if se[u, j] >= 0:
                red[u, j] = rng.integers(-50, 50, size=(H, Hp))
    Gx = G0.copy()
    redx = red.copy()
    oracle.reduce_grad(Gx, redx, se)
    expect = G0.astype(np.float64).copy()
    for u in range(R):
        for j in range(B):
            if se[u, j] >= 0:
                expect[se[u, j]] += red[u, j]
    np.testing.assert_array_equal(Gx, expect.astype(np.float32))
    assert not redx.any()
    np.testing.assert_array_equal(Gx[3:], G0[3:])   # experts without replicas untouched


def test_reduce_grad_ascending_rank_order():
    """fp32 addition is not associative: with G=1, red_r1 = 2^24, red_r2 = -2^24
    the ascending-rank order gives (1 + 2^24) - 2^24 = 0 (1 is lost to rounding),
    the opposite order would give 1."""
    R, B, E = 3, 1, 3
    se = np.array([[-1], [0], [0]], np.int32)
    G = np.array([[[1.0]], [[0.0]], [[0.0]]], np.float32)
    red = np.array([[[[0.0]]], [[[2.0 ** 24]]], [[[-(2.0 ** 24)]]]], np.float32)
    oracle.reduce_grad(G, red, se)
    assert G[0, 0, 0] == 0.0
    # (1 - 2^24) is exact, then + 2^24 = 1
    G = np.array([[[1.0]], [[0.0]], [[0.0]]], np.float32)
    red = np.array([[[[0.0]]], [[[-(2.0 ** 24)]]], [[[2.0 ** 24]]]], np.float32)
    oracle.reduce_grad(G, red, se)
    assert G[0, 0, 0] == 1.0


# ---------------------------------------------------------------- grouped GEMM
def test_grouped_gemm_shift_matrices_select_the_right_row():
    """W_rho[h, j] = 1 iff j == (h + shift(rho)) mod H' with a distinct shift per
    weight row (home rows and every rank's slots): each output element is a
    short exact sum of bf16 inputs, computed here by index arithmetic."""
    R, S, K, E, H, Hp = 2, 29, 2, 8, 24, 8
    B = E // R
    topk = synth.gumbel_topk(R, S, K, synth.zipf_popularity(E, 1.3), 4)
    p = oracle.plan(topk, E, B, 0)
    x = synth.tokens_host((R, S, H), 3)
    recv = oracle.dispatch(x, p.dest)

    def shift_w(s):
        w = np.zeros((H, Hp), np.float32)
        w[np.arange(H), (np.arange(H) + s) % Hp] = 1.0
        return _torch_bf16_bits(w)

    w_home = np.stack([shift_w(e) for e in range(E)])
    w_slots = np.stack([np.stack([shift_w(E + u * B + j) for j in range(B)]) for u in range(R)])
    y = oracle.grouped_gemm(recv, w_home, w_slots, p.cu, E)
    C = S * K
    rf = oracle.bf16_to_f32(recv).astype(np.float64)
    for i in range(R * C):
        u, pos = divmod(i, C)
        rho = int(np.searchsorted(p.cu[u], pos, side="right") - 1)
        s = rho if rho < E else E + u * B + (rho - E)
        expect = np.zeros(Hp)
        for h in range(H):
            expect[(h + s) % Hp] += rf[i, h]
        np.testing.assert_array_equal(y[i], expect)
    # the sampled-row variant agrees with the full one
    rows = np.array([0, 5, C - 1, C, R * C - 1])
    np.testing.assert_array_equal(oracle.grouped_gemm(recv, w_home, w_slots, p.cu, E, rows=rows),
                                  y[rows])


def test_grouped_gemm_brute_force_tiny():
    R, S, K, E, H, Hp = 2, 5, 2, 4, 6, 3
    topk = synth.gumbel_topk(R, S, K, synth.zipf_popularity(E, 2.0), 1)
    p = oracle.plan(topk, E, E // R, 0)
    recv = synth.tokens_host((R * S * K, H), 8)
    w_home = synth.weights_host((E, H, Hp), 2, std=0.5)
    w_slots = synth.weights_host((R, E // R, H, Hp), 3, std=0.5)
    y = oracle.grouped_gemm(recv, w_home, w_slots, p.cu, E)
    C = S * K
    for i in range(R * C):
        u, pos = divmod(i, C)
        rho = max(r for r in range(E + E // R) if p.cu[u][r] <= pos < p.cu[u][r + 1])
        w = w_home[rho] if rho < E else w_slots[u, rho - E]
        for j in range(Hp):
            acc = 0.0
            for h in range(H):
                acc += float(oracle.bf16_to_f32(recv[i:i + 1, h])[0]) * \
                       float(oracle.bf16_to_f32(w[h:h + 1, j])[0])
            assert abs(y[i, j] - acc) <= 1e-12 * (1 + abs(acc))


# ---------------------------------------------------------------- backward pieces
def test_dispatch_bwd_k1_is_the_inverse_permutation():
    topk, p, x, g, y = _small_problem(K=1, H=40)
    R, S, H = x.shape
    recv = oracle.dispatch(x, p.dest)
    np.testing.assert_array_equal(oracle.dispatch_bwd(recv, p.dest), x)


def test_dispatch_bwd_of_dispatch_is_K_times_x():
    """Each token is copied to K rows; summing them back gives K*x, exact for K a
    power of two (a scaling by 2^j), computed here by torch."""
    topk, p, x, g, y = _small_problem(K=4, H=40)
    recv = oracle.dispatch(x, p.dest)
    dx = oracle.dispatch_bwd(recv, p.dest)
    ref = torch.from_numpy(oracle.bf16_to_f32(x) * 4.0)
    np.testing.assert_array_equal(dx, _torch_bf16_bits(ref.numpy()))


def test_dispatch_bwd_exact_on_dyadic_values():
    topk, p, x, g, y = _small_problem(K=4, H=16)
    rng = np.random.default_rng(3)
    v = rng.integers(-64, 65, size=(topk.size, 16)).astype(np.float32) / 8.0
    drecv = _torch_bf16_bits(v)
    dx = oracle.dispatch_bwd(drecv, p.dest)
    exact = v[p.dest].astype(np.float64).sum(axis=2)
    np.testing.assert_array_equal(dx, _torch_bf16_bits(exact.astype(np.float32)))


def test_combine_dgates_one_hot_dout_reads_one_element():
    """dg[t,k] = <dOut[t], Y[dest[t,k]]> ([P4] "The core idea": the gradient of the
    gate weight). With dOut[t] one-hot at column c_t the dot product is the single
    element Y[dest[t,k], c_t], exactly."""
    topk, p, x, g, y = _small_problem(K=3, D=8, S=5)
    R, S, K = topk.shape
    D = y.shape[1]
    c = np.random.default_rng(11).integers(0, D, size=(R, S))
    dout = np.zeros((R, S, D), np.uint16)
    dout[np.arange(R)[:, None], np.arange(S)[None, :], c] = 0x3F80      # bf16 1.0
    dg = oracle.combine_dgates(dout, y, p.dest)
    yf = oracle.bf16_to_f32(y)
    for r in range(R):
        for t in range(S):
            for k in range(K):
                assert dg[r, t, k] == float(yf[p.dest[r, t, k], c[r, t]])


def test_combine_dgates_is_the_adjoint_of_combine():
    """Combine is linear in the gates: out[t] = sum_k g[t,k] Y[dest[t,k]]. So
    sum_{t,k} g[t,k] * dg[t,k] = <dOut, out> for any gates. The right side is
    formed here as one fp64 tensor contraction of the gathered rows, with small
    dyadic values so that both sides are exact sums."""
    topk, p, x, _, _ = _small_problem(K=4, D=12, S=9, R=2)
    R, S, K = topk.shape
    rng = np.random.default_rng(12)
    yv = rng.integers(-16, 17, size=(R * S * K, 12)).astype(np.float32) / 4
    dv = rng.integers(-16, 17, size=(R, S, 12)).astype(np.float32) / 8
    gv = rng.integers(-8, 9, size=(R, S, K)).astype(np.float64)
    dg = oracle.combine_dgates(_torch_bf16_bits(dv), _torch_bf16_bits(yv), p.dest)
    out = np.einsum("rsk,rskd->rsd", gv, yv[p.dest].astype(np.float64))
    assert (gv * dg).sum() == (dv.astype(np.float64) * out).sum()
    # and gate by gate: a one-hot gate vector isolates one dg entry
    for r, t, k in [(0, 0, 0), (1, 8, 3), (0, 4, 2)]:
        e = np.zeros_like(gv)
        e[r, t, k] = 1.0
        out = np.einsum("rsk,rskd->rsd", e, yv[p.dest].astype(np.float64))
        assert dg[r, t, k] == (dv.astype(np.float64) * out).sum()


def _shift_weights(E, R, B, H, Hp):
    def shift_w(s):
        w = np.zeros((H, Hp), np.float32)
        w[np.arange(H), (np.arange(H) + s) % Hp] = 1.0
        return _torch_bf16_bits(w)
    w_home = np.stack([shift_w(e) for e in range(E)])
    w_slots = np.stack([np.stack([shift_w(E + u * B + j) for j in range(B)]) for u in range(R)])
    return w_home, w_slots


def test_grouped_gemm_dx_shift_matrices():
    """dRecv = dY @ W^T with W_rho[h, j] = [j == (h + s_rho) mod H']: each output
    element picks dY[i, (h + s_rho) mod H'], a distinct shift per weight row."""
    R, S, K, E, H, Hp = 2, 23, 2, 8, 16, 8
    B = E // R
    topk = synth.gumbel_topk(R, S, K, synth.zipf_popularity(E, 1.3), 5)
    p = oracle.plan(topk, E, B, 0)
    w_home, w_slots = _shift_weights(E, R, B, H, Hp)
    dy = synth.tokens_host((R * S * K, Hp), 6)
    dr = oracle.grouped_gemm_dx(dy, w_home, w_slots, p.cu, E)
    C = S * K
    df = oracle.bf16_to_f32(dy).astype(np.float64)
    for i in range(R * C):
        u, pos = divmod(i, C)
        rho = int(np.searchsorted(p.cu[u], pos, side="right") - 1)
        s = rho if rho < E else E + u * B + (rho - E)
        np.testing.assert_array_equal(dr[i], df[i, (np.arange(H) + s) % Hp])


def test_grouped_gemm_dw_brute_force_tiny():
    R, S, K, E, H, Hp = 2, 6, 2, 4, 5, 3
    B = E // R
    topk = synth.gumbel_topk(R, S, K, synth.zipf_popularity(E, 2.0), 2)
    p = oracle.plan(topk, E, B, 0)
    recv = synth.tokens_host((R * S * K, H), 7)
    dy = synth.tokens_host((R * S * K, Hp), 8)
    d_home, d_slots = oracle.grouped_gemm_dw(recv, dy, p.cu, E, B, H, Hp)
    C = S * K
    rf, df = oracle.bf16_to_f32(recv), oracle.bf16_to_f32(dy)
    ref_home = np.zeros((E, H, Hp))
    ref_slots = np.zeros((R, B, H, Hp))
    for i in range(R * C):
        u, pos = divmod(i, C)
        rho = max(r for r in range(E + B) if p.cu[u][r] <= pos < p.cu[u][r + 1])
        for h in range(H):
            for j in range(Hp):
                v = float(rf[i, h]) * float(df[i, j])
                if rho < E:
                    ref_home[rho, h, j] += v
                else:
                    ref_slots[u, rho - E, h, j] += v
    np.testing.assert_allclose(d_home, ref_home, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(d_slots, ref_slots, rtol=1e-12, atol=1e-14)


def test_grouped_gemm_dw_one_hot_rows_are_outer_products():
    """recv rows that are one-hot at column h(i) make dW(rho)[h, :] the sum of the
    dY rows of the segment whose one-hot column is h -- exact."""
    R, S, K, E, H, Hp = 2, 17, 2, 8, 6, 4
    B = E // R
    topk = synth.gumbel_topk(R, S, K, synth.zipf_popularity(E, 1.1), 9)
    p = oracle.plan(topk, E, B, 0)
    n = R * S * K
    hot = np.arange(n) % H
    recv = np.zeros((n, H), np.float32)
    recv[np.arange(n), hot] = 1.0
    dyv = np.random.default_rng(4).integers(-8, 9, size=(n, Hp)).astype(np.float32)
    d_home, d_slots = oracle.grouped_gemm_dw(_torch_bf16_bits(recv), _torch_bf16_bits(dyv), p.cu,
                                             E, B, H, Hp)
    C = S * K
    ref_home = np.zeros_like(d_home)
    ref_slots = np.zeros_like(d_slots)
    for i in range(n):
        u, pos = divmod(i, C)
        rho = int(np.searchsorted(p.cu[u], pos, side="right") - 1)
        tgt = ref_home[rho] if rho < E else ref_slots[u, rho - E]
        tgt[hot[i]] += dyv[i]
    np.testing.assert_array_equal(d_home, ref_home)
    np.testing.assert_array_equal(d_slots, ref_slots)


def test_sampled_gemm_helpers_agree_with_the_whole_gemm():
    """The helpers the bench-size parity tests use to check sampled rows --
    segment_of_rows, weight_row_of and gemm_rows (and grouped_gemm's rows= form) --
    give, row for row, what the whole grouped GEMM (pinned above by shift matrices
    and brute force) gives, on an inference batch whose hot group overflows, so
    home, slot and overflow segments all occur. segment_of_rows is also checked
    against a plain search of cu_seqlens."""
    R, E, B, K, S, H, Hp = 2, 16, 2, 2, 64, 64, 48
    G = E // R
    pop = np.full(E, 1.0)
    pop[:G] = 200.0                                       # group 0's experts all hot
    topk = synth.gumbel_topk(R, S, K, pop / pop.sum(), 11)
    ref = oracle.plan(topk, E, B, 1)
    assert oracle.check_plan(topk, E, B, 1, ref.cu, ref.slot_expert, ref.dest) == 0
    C = S * K
    x = synth.tokens_host((R, S, H), 12)
    recv = oracle.dispatch(x, ref.dest)
    w_home = synth.weights_host((E, H, Hp), 13)
    w_slots = oracle.prefetch(w_home, ref.slot_expert, np.zeros((R, B, H, Hp), np.uint16))
    y = oracle.grouped_gemm(recv, w_home, w_slots, ref.cu, E)
    rows, segs = [], []
    overflow = slot = 0
    for u in range(R):
        for rho in range(E + B):
            a, b = int(ref.cu[u, rho]), int(ref.cu[u, rho + 1])
            if b > a:
                rows += range(u * C + a, u * C + b)
                segs += [rho] * (b - a)
                overflow += int(rho < E and rho // G != u)
                slot += int(rho >= E)
    assert overflow > 0 and slot > 0                      # every kind of segment is present
    rows = np.array(rows)
    np.testing.assert_array_equal(oracle.segment_of_rows(ref.cu, C, rows), segs)
    np.testing.assert_allclose(oracle.grouped_gemm(recv, w_home, w_slots, ref.cu, E, rows=rows),
                               y[rows], rtol=1e-12, atol=1e-12)
    for i, rho in zip(rows, segs):
        e = oracle.weight_row_of(rho, i // C, E, ref.slot_expert)
        np.testing.assert_allclose(oracle.gemm_rows(recv[i:i + 1], w_home[e])[0], y[i],
                                   rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- the OpenMP build
def test_openmp_build_gives_the_same_bits(tmp_path):
    """The CPU baseline's all-core leg loads the same oracle source built with
    -fopenmp: its data stages must give exactly the single-threaded bits."""
    import subprocess
    import sys
    try:
        oracle.build(openmp=True)
    except Exception as exc:   # noqa: BLE001
        pytest.skip(f"no OpenMP compiler here: {exc}")
    topk, p, x, g, y = _small_problem(S=300, K=4, H=48, D=40)
    w_home = synth.weights_host((16, 6, 10), 3)
    red0 = synth.normal_host((2, 8, 6, 10), 4, 1.0)
    np.savez(tmp_path / "in.npz", dest=p.dest, x=x, g=g, y=y, se=p.slot_expert, w_home=w_home,
             red0=red0)
    code = f"""
import numpy as np, sys
sys.path.insert(0, {os.path.dirname(os.path.dirname(os.path.abspath(__file__)))!r})
import oracle
d = np.load({str(tmp_path / 'in.npz')!r})
g_home = np.zeros((16, 6, 10), np.float32); red = d['red0'].copy()
oracle.reduce_grad(g_home, red, d['se'])
np.savez({str(tmp_path / 'out.npz')!r},
         recv=oracle.dispatch(d['x'], d['dest']), out=oracle.combine(d['y'], d['dest'], d['g']),
         dy=oracle.combine_bwd(d['x'][..., :40], d['dest'], d['g']),
         dx=oracle.dispatch_bwd(oracle.dispatch(d['x'], d['dest']), d['dest']),
         slots=oracle.prefetch(d['w_home'], d['se'], np.zeros((2, 8, 6, 10), np.uint16)),
         g_home=g_home, red=red)
"""
    env = dict(os.environ, ORACLE_OPENMP="1", OMP_NUM_THREADS="4")
    subprocess.run([sys.executable, "-c", code], env=env, check=True)
    got = np.load(tmp_path / "out.npz")
    g_home = np.zeros((16, 6, 10), np.float32)
    red = red0.copy()
    oracle.reduce_grad(g_home, red, p.slot_expert)
    recv = oracle.dispatch(x, p.dest)
    want = dict(recv=recv, out=oracle.combine(y, p.dest, g),
                dy=oracle.combine_bwd(x[..., :40].copy(), p.dest, g),
                dx=oracle.dispatch_bwd(recv, p.dest),
                slots=oracle.prefetch(w_home, p.slot_expert, np.zeros((2, 8, 6, 10), np.uint16)),
                g_home=g_home, red=red)
    for k, v in want.items():
        np.testing.assert_array_equal(got[k], v, err_msg=k)
