// Oracle for balanced expert-parallel dispatch: TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU restatement of what the hot path computes,
// written from the MoonEP announcement pages. Only the test suite, the smoke
// check and the benchmark's CPU-baseline leg may load this library; the
// product path never does. It shares no code, header or table with the CUDA
// library.
//
// Sources (page title / host, then section):
//   [P1] "Moonshot AI libera MoonEP ..." (noticiai.com.br): "O problema que o
//        MoonEP resolve", "A ideia central", "O contrato de memoria".
//   [P2] "Moonshot AI Open-Sources MoonEP: A Perfectly Balanced Expert
//        Parallelism Library for MoE Training" (spaxe.top): the paragraphs on
//        the memory contract, gradients and reduce_grad.
//   [P4] "Moonshot AI open-sources MoonEP" (ai-maestro.online): "The problem
//        MoonEP targets", "The core idea: dynamic redundant experts", "The
//        memory contract".
//
// The pages fix the metric (maxvio), the invariant (every rank receives exactly
// S*K token-slots), the replica source constraint (training: replicas come from
// at most one remote home group, B = E/R), the overflow rule (inference: B < E/R,
// extra remote experts are read from the home rows [0,E)), the row layout of the
// [E+B, H, H'] weight tensor, and reduce_grad (fold the replica gradients into
// the home rows, zero the consumed slots). They do NOT state the planning
// algorithm ("near-optimal"); this file implements one deterministic rule,
// stated in plan_tree() below, a reading of the pages. The tests pin this
// file's plans to that rule (plans worked out by hand from its definition);
// whether MoonEP's own planner makes the same choice among valid plans cannot
// be decided from the pages. Validity of a plan is pinned by
// oracle_check_plan(), which is independent of the rule, and by brute force.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared (no FMA contraction,
// so every fused multiply-add below is the explicit std::fma call). The same
// source built with -fopenmp as well runs the per-token loops of the data
// stages on every core (the "omp parallel for" lines below; without -fopenmp
// the compiler ignores them). Each iteration writes its own outputs only, so
// both builds give the same bits; the CPU baseline times both.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <deque>
#include <utility>
#include <vector>

namespace {

enum {
    OR_OK = 0,
    OR_ERR_EXPERT_ID = -1,   // a top-K id outside [0, E)
    OR_ERR_DUP_ID = -2,      // the same expert twice in one token's top-K
    OR_ERR_CONFIG = -3,      // inconsistent sizes / mode
    OR_ERR_INFEASIBLE = -4,  // a rank did not end with exactly S*K slots
};

enum { MODE_TRAIN = 0, MODE_INFER = 1 };

// bf16 <-> fp32, from the formats' definitions: bf16 is the upper half of an
// IEEE binary32 word. Narrowing rounds to nearest, ties to even, on the 16
// discarded bits (a carry out of the mantissa correctly bumps the exponent,
// and finite values past the largest bf16 become infinity).
float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) {           // NaN stays NaN (quiet bit set)
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

// ---------------------------------------------------------------------------
// Planning rule (the build's documented choice; the pages only say the GPU
// planner is "near-optimal", [P4] "The core idea", property 2).
//
// Group g (home rank g, experts [g*G, (g+1)*G)) carries load L_g; every rank
// must end with C = S*K slots. x_g = L_g - C.
//   donors     : {g : x_g > 0}, by x descending, ties by lower g
//   recipients : deque of {(g, -x_g) : x_g < 0}, by deficit descending, ties lower g
//   repeat while the deque is not empty:
//       pop (u, D) from the front; d = current donor;
//       parent[u] = d; d sends D slots to u; x_d -= D;
//       if x_d < 0: d now lacks -x_d slots: push (d, -x_d) to the FRONT, next donor
//       if x_d == 0: next donor
// Every rank gets at most one parent, so a rank's replicas come from at most
// one remote home group ([P4] "The memory contract": training needs B = E/R
// because the planner duplicates experts from at most one remote group).
// ---------------------------------------------------------------------------
struct Edge { int donor; int child; int64_t flow; };

int plan_tree(int R, const int64_t* L, int64_t C, std::vector<int>& parent,
              std::vector<int64_t>& inflow, std::vector<Edge>& edges) {
    parent.assign(R, -1);
    inflow.assign(R, 0);
    edges.clear();
    std::vector<int64_t> x(R);
    std::vector<int> donors;
    std::vector<std::pair<int, int64_t>> recv;
    for (int g = 0; g < R; ++g) {
        x[g] = L[g] - C;
        if (x[g] > 0) donors.push_back(g);
        if (x[g] < 0) recv.push_back({g, -x[g]});
    }
    std::stable_sort(donors.begin(), donors.end(),
                     [&](int a, int b) { return x[a] > x[b]; });
    std::stable_sort(recv.begin(), recv.end(),
                     [](const std::pair<int, int64_t>& a, const std::pair<int, int64_t>& b) {
                         return a.second > b.second;
                     });
    std::deque<std::pair<int, int64_t>> queue(recv.begin(), recv.end());
    size_t di = 0;
    while (!queue.empty()) {
        if (di >= donors.size()) return OR_ERR_INFEASIBLE;  // cannot happen when sum x == 0
        std::pair<int, int64_t> top = queue.front();
        queue.pop_front();
        int u = top.first;
        int64_t D = top.second;
        int d = donors[di];
        parent[u] = d;
        inflow[u] = D;
        edges.push_back({d, u, D});
        x[d] -= D;
        if (x[d] < 0) {
            queue.push_front({d, -x[d]});
            ++di;
        } else if (x[d] == 0) {
            ++di;
        }
    }
    return OR_OK;
}

int check_config(int R, int E, int B, int K, int S, int mode) {
    if (R < 1 || E < 1 || K < 1 || S < 0 || B < 0) return OR_ERR_CONFIG;
    if (E % R != 0 || K > E) return OR_ERR_CONFIG;
    int G = E / R;
    if (mode == MODE_TRAIN && B != G) return OR_ERR_CONFIG;
    if (mode == MODE_INFER && !(B >= 1 && B < G)) return OR_ERR_CONFIG;
    if (mode != MODE_TRAIN && mode != MODE_INFER) return OR_ERR_CONFIG;
    return OR_OK;
}

}  // namespace

extern "C" {

float oracle_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }
uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }
void oracle_f32_to_bf16_array(const float* f, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(f[i]);
}

// T_e = #{(r,t,k) : topk[r,t,k] = e}. Also validates the routing: ids in
// [0,E) and pairwise distinct within a token (top-K picks K different experts).
int oracle_histogram(const int32_t* topk, int R, int S, int K, int E, int64_t* T) {
    for (int e = 0; e < E; ++e) T[e] = 0;
    int64_t ntok = (int64_t)R * S;
    for (int64_t i = 0; i < ntok; ++i) {
        const int32_t* ids = topk + i * K;
        for (int k = 0; k < K; ++k) {
            if (ids[k] < 0 || ids[k] >= E) return OR_ERR_EXPERT_ID;
            for (int k2 = 0; k2 < k; ++k2)
                if (ids[k2] == ids[k]) return OR_ERR_DUP_ID;
        }
        for (int k = 0; k < K; ++k) T[ids[k]] += 1;
    }
    return OR_OK;
}

// maxvio = max_e (T_e / Tbar) - 1 with Tbar = R*S*K / E, the expected count
// under perfect balance ([P4] "The problem MoonEP targets"). Written as
// (E*max_e T_e - RSK) / RSK: the numerator and denominator are exact
// integers, so the result carries exactly one binary64 rounding. An empty
// batch (RSK = 0) is defined as perfectly balanced, 0.
double oracle_maxvio(const int64_t* T, int E, int64_t RSK) {
    if (RSK == 0) return 0.0;
    int64_t mx = 0;
    for (int e = 0; e < E; ++e) mx = std::max(mx, T[e]);
    return (double)((int64_t)E * mx - RSK) / (double)RSK;
}

// The tree step alone (for brute-force pins): parent[R] (-1 = none),
// inflow[R] (slots received from the parent), and edge order: order[u] = the
// index at which u received its parent (-1 = none).
int oracle_tree(int R, const int64_t* L, int64_t C, int32_t* parent, int64_t* inflow,
                int32_t* order) {
    std::vector<int> par;
    std::vector<int64_t> inf;
    std::vector<Edge> edges;
    int64_t total = 0;
    for (int g = 0; g < R; ++g) total += L[g];
    if (total != (int64_t)R * C) return OR_ERR_CONFIG;
    int rc = plan_tree(R, L, C, par, inf, edges);
    for (int g = 0; g < R; ++g) {
        parent[g] = par[g];
        inflow[g] = inf[g];
        order[g] = -1;
    }
    for (size_t i = 0; i < edges.size(); ++i) order[edges[i].child] = (int32_t)i;
    return rc;
}

// The whole plan. Outputs:
//   cu[R][E+B+1]      per rank, exclusive offsets of the row segments
//                     0..E+B-1 (cu[u][0] = 0, cu[u][E+B] = C)
//   slot_expert[R][B] the expert held by each prefetch slot, -1 if unused
//   dest[R][S][K]     flat slot index into the [R*C] receive space
//   parent[R], inflow[R], maxvio (diagnostics)
//
// Step order:
//  1. histogram, group loads L_g;
//  2. the tree (plan_tree);
//  3. group g's slots listed expert by expert, the group's experts in
//     ascending token count (ties: lower id), each expert's slots in (r, t)
//     order: home g keeps the first C - inflow[g], each child takes the next
//     `flow` entries in the order the children were assigned. The tail that
//     moves therefore holds the group's largest experts, so each child's range
//     touches few experts and few replicas are needed ("a small number of
//     redundant experts", [P4] "The core idea");
//  4. rows: a home slot of expert e uses row e. A replica on child u:
//     TRAIN: slot j = e - parent[u]*G, row E + j.
//     INFER: u's remote experts ranked by slot count descending, ties by
//     lower id; the top B get slots 0..B-1 in ascending expert id; the rest
//     overflow and stay on row e, a home row in [0,E) whose weights the GEMM
//     reads in place ([P4] "The memory contract": overflow weights are read
//     from the home rank);
//  5. on every rank, segments in ascending row order, tokens inside a
//     segment in (r, t) order; dest = u*C + position.
int oracle_plan(int R, int E, int B, int K, int S, int mode, const int32_t* topk,
                int32_t* cu, int32_t* slot_expert, int32_t* dest, int32_t* parent_out,
                int64_t* inflow_out, double* maxvio) {
    int rc = check_config(R, E, B, K, S, mode);
    if (rc) return rc;
    const int G = E / R;
    const int64_t C = (int64_t)S * K;
    const int64_t RSK = (int64_t)R * C;
    const int NROW = E + B;

    // 1. histogram and loads
    std::vector<int64_t> T(E);
    rc = oracle_histogram(topk, R, S, K, E, T.data());
    if (rc) return rc;
    *maxvio = oracle_maxvio(T.data(), E, RSK);
    std::vector<int64_t> L(R, 0);
    for (int e = 0; e < E; ++e) L[e / G] += T[e];

    // 2. tree
    std::vector<int> parent;
    std::vector<int64_t> inflow;
    std::vector<Edge> edges;
    rc = plan_tree(R, L.data(), C, parent, inflow, edges);
    if (rc) return rc;
    for (int g = 0; g < R; ++g) {
        parent_out[g] = parent[g];
        inflow_out[g] = inflow[g];
    }

    // 3. per-expert slot lists in (r, t) order (k never ties: ids are distinct
    //    per token), then owner of each slot.
    std::vector<std::vector<int64_t>> by_expert(E);
    for (int64_t i = 0; i < RSK; ++i) by_expert[topk[i]].push_back(i);
    std::vector<int> owner(RSK, -1);
    for (int g = 0; g < R; ++g) {
        // ranges over group g's list: [0, keep) -> g, then one per child
        std::vector<std::pair<int64_t, int>> bounds;  // (end position, owner)
        int64_t pos = C - inflow[g];
        bounds.push_back({pos, g});
        for (const Edge& ed : edges)
            if (ed.donor == g) {
                pos += ed.flow;
                bounds.push_back({pos, ed.child});
            }
        if (pos != L[g]) return OR_ERR_INFEASIBLE;
        std::vector<int> ex;
        for (int e = g * G; e < (g + 1) * G; ++e) ex.push_back(e);
        std::stable_sort(ex.begin(), ex.end(),
                         [&](int a, int b2) { return T[a] < T[b2]; });  // stable: ties keep lower id first
        int64_t q = 0;
        size_t b = 0;
        for (int e : ex)
            for (int64_t i : by_expert[e]) {
                while (q >= bounds[b].first) ++b;
                owner[i] = bounds[b].second;
                ++q;
            }
    }

    // 4. rows
    for (int64_t v = 0; v < (int64_t)R * B; ++v) slot_expert[v] = -1;
    std::vector<int> row(RSK, -1);
    for (int u = 0; u < R; ++u) {
        // remote experts held on u, with their slot counts
        std::vector<int64_t> cnt(E, 0);
        for (int64_t i = 0; i < RSK; ++i)
            if (owner[i] == u && topk[i] / G != u) cnt[topk[i]] += 1;
        std::vector<int> slot_of(E, -1);
        if (mode == MODE_TRAIN) {
            for (int e = 0; e < E; ++e)
                if (cnt[e] > 0) {
                    if (e / G != parent[u]) return OR_ERR_INFEASIBLE;
                    slot_of[e] = e - parent[u] * G;
                }
        } else {
            std::vector<int> cand;
            for (int e = 0; e < E; ++e)
                if (cnt[e] > 0) cand.push_back(e);
            std::stable_sort(cand.begin(), cand.end(), [&](int a, int b2) {
                return cnt[a] > cnt[b2];   // stable: equal counts keep ascending id
            });
            if ((int)cand.size() > B) cand.resize(B);
            std::sort(cand.begin(), cand.end());
            for (size_t j = 0; j < cand.size(); ++j) slot_of[cand[j]] = (int)j;
        }
        for (int e = 0; e < E; ++e)
            if (slot_of[e] >= 0) slot_expert[(int64_t)u * B + slot_of[e]] = e;
        for (int64_t i = 0; i < RSK; ++i) {
            if (owner[i] != u) continue;
            int e = topk[i];
            if (e / G == u || slot_of[e] < 0) row[i] = e;       // home row, or overflow
            else row[i] = E + slot_of[e];
        }
    }

    // 5. segments and destinations
    for (int u = 0; u < R; ++u) {
        std::vector<std::pair<int, int64_t>> mine;  // (row, flat index)
        for (int64_t i = 0; i < RSK; ++i)
            if (owner[i] == u) mine.push_back({row[i], i});
        if ((int64_t)mine.size() != C) return OR_ERR_INFEASIBLE;
        std::sort(mine.begin(), mine.end());
        int32_t* cuu = cu + (int64_t)u * (NROW + 1);
        for (int rr = 0; rr <= NROW; ++rr) cuu[rr] = 0;
        for (int64_t p = 0; p < C; ++p) {
            dest[mine[p].second] = (int32_t)((int64_t)u * C + p);
            cuu[mine[p].first + 1] += 1;
        }
        for (int rr = 0; rr < NROW; ++rr) cuu[rr + 1] += cuu[rr];
    }
    return OR_OK;
}

// Validity of ANY plan, independent of the rule above. Returns 0, or the
// number of the first invariant that fails:
//   1  cu[u] starts at 0, never decreases, ends at C (exactly S*K per rank)
//   2  dest is a bijection onto [0, R*C)
//   3  every (r,t,k) lands on a row serving its routed expert: row e itself,
//      or a slot row whose slot_expert is e
//   4  TRAIN: B == E/R, every row used on u is local (u's own experts or its
//      slots) and u's slots come from at most one remote group
//   5  INFER: B < E/R; overflow rows are home rows in [0,E); remote experts
//      (slots and overflow) come from at most one remote group
//   6  slot_expert entries are -1 or in [0,E), distinct per rank, and every
//      non-empty slot segment names an expert
int oracle_check_plan(int R, int E, int B, int K, int S, int mode, const int32_t* topk,
                      const int32_t* cu, const int32_t* slot_expert, const int32_t* dest) {
    if (check_config(R, E, B, K, S, mode)) return 4;
    const int G = E / R;
    const int64_t C = (int64_t)S * K;
    const int64_t RSK = (int64_t)R * C;
    const int NROW = E + B;
    for (int u = 0; u < R; ++u) {
        const int32_t* cuu = cu + (int64_t)u * (NROW + 1);
        if (cuu[0] != 0 || cuu[NROW] != C) return 1;
        for (int rr = 0; rr < NROW; ++rr)
            if (cuu[rr + 1] < cuu[rr]) return 1;
    }
    for (int u = 0; u < R; ++u) {
        std::vector<int> seen;
        for (int j = 0; j < B; ++j) {
            int e = slot_expert[(int64_t)u * B + j];
            if (e < -1 || e >= E) return 6;
            if (e >= 0) {
                if (std::find(seen.begin(), seen.end(), e) != seen.end()) return 6;
                seen.push_back(e);
            }
            const int32_t* cuu = cu + (int64_t)u * (NROW + 1);
            if (cuu[E + j + 1] > cuu[E + j] && e < 0) return 6;
        }
    }
    std::vector<char> hit(RSK, 0);
    std::vector<int> remote_group(R, -1);
    for (int64_t i = 0; i < RSK; ++i) {
        int64_t d = dest[i];
        if (d < 0 || d >= RSK || hit[d]) return 2;
        hit[d] = 1;
        int u = (int)(d / C);
        int64_t pos = d % C;
        const int32_t* cuu = cu + (int64_t)u * (NROW + 1);
        int rr = (int)(std::upper_bound(cuu, cuu + NROW + 1, (int32_t)pos) - cuu) - 1;
        int e = topk[i];
        int home = e / G;
        if (rr < E) {
            if (rr != e) return 3;
            if (home != u) {                 // an expert served on a home row of another rank
                if (mode == MODE_TRAIN) return 4;
            }
        } else {
            if (slot_expert[(int64_t)u * B + (rr - E)] != e) return 3;
        }
        if (home != u) {
            if (remote_group[u] == -1) remote_group[u] = home;
            else if (remote_group[u] != home) return mode == MODE_TRAIN ? 4 : 5;
        }
    }
    return 0;
}

// recv[dest[r,t,k], :] = x[r,t,:], a bit copy of each bf16 row
// ([P4] "The core idea", property 3: tokens are written directly into their
// expert-grouped positions).
void oracle_dispatch(const uint16_t* x, const int32_t* dest, int R, int S, int K, int H,
                     uint16_t* recv) {
    int64_t ntok = (int64_t)R * S;
#pragma omp parallel for schedule(static)
    for (int64_t tok = 0; tok < ntok; ++tok)
        for (int k = 0; k < K; ++k) {
            int64_t d = dest[tok * K + k];
            std::memcpy(recv + d * H, x + tok * H, sizeof(uint16_t) * (size_t)H);
        }
}

// out[r,t,c] = bf16_rne(acc), acc = 0; for k = 0..K-1: acc = fma(g[r,t,k], Y[dest[r,t,k], c], acc)
// fp32 accumulation in ascending k, one bf16 rounding at the end.
void oracle_combine(const uint16_t* y, const int32_t* dest, const float* gates, int R, int S,
                    int K, int D, uint16_t* out) {
    int64_t ntok = (int64_t)R * S;
#pragma omp parallel for schedule(static)
    for (int64_t tok = 0; tok < ntok; ++tok)
        for (int c = 0; c < D; ++c) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t d = dest[tok * K + k];
                acc = std::fma(gates[tok * K + k], bf16_to_f32(y[d * D + c]), acc);
            }
            out[tok * D + c] = f32_to_bf16_rne(acc);
        }
}

// Backward of the weighted combine with respect to Y:
// dY[dest[r,t,k], c] = bf16_rne( fp32( g[r,t,k] * dOut[r,t,c] ) ).
void oracle_combine_bwd(const uint16_t* dout, const int32_t* dest, const float* gates, int R,
                        int S, int K, int D, uint16_t* dy) {
    int64_t ntok = (int64_t)R * S;
#pragma omp parallel for schedule(static)
    for (int64_t tok = 0; tok < ntok; ++tok)
        for (int k = 0; k < K; ++k) {
            int64_t d = dest[tok * K + k];
            float g = gates[tok * K + k];
            for (int c = 0; c < D; ++c) {
                float p = g * bf16_to_f32(dout[tok * D + c]);
                dy[d * D + c] = f32_to_bf16_rne(p);
            }
        }
}

// Backward of the dispatch (a copy of each token to K rows): the token's
// gradient is the sum of its K receive-row gradients,
// dx[r,t,c] = bf16_rne(acc), acc = 0; for k = 0..K-1: acc = acc + dRecv[dest[r,t,k], c]
// (fp32 adds in ascending k).
void oracle_dispatch_bwd(const uint16_t* drecv, const int32_t* dest, int R, int S, int K, int H,
                         uint16_t* dx) {
    int64_t ntok = (int64_t)R * S;
#pragma omp parallel for schedule(static)
    for (int64_t tok = 0; tok < ntok; ++tok)
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t d = dest[tok * K + k];
                acc = acc + bf16_to_f32(drecv[d * H + c]);
            }
            dx[tok * H + c] = f32_to_bf16_rne(acc);
        }
}

// Gradient of the combine with respect to the gates:
// dg[r,t,k] = sum_c dOut[r,t,c] * Y[dest[r,t,k], c], accumulated in binary64.
void oracle_combine_dgates(const uint16_t* dout, const uint16_t* y, const int32_t* dest, int R,
                           int S, int K, int D, double* dg) {
    int64_t ntok = (int64_t)R * S;
#pragma omp parallel for schedule(static)
    for (int64_t tok = 0; tok < ntok; ++tok)
        for (int k = 0; k < K; ++k) {
            int64_t d = dest[tok * K + k];
            double acc = 0.0;
            for (int c = 0; c < D; ++c)
                acc += (double)bf16_to_f32(dout[tok * D + c]) * (double)bf16_to_f32(y[d * D + c]);
            dg[tok * K + k] = acc;
        }
}

// prefetch_weight: slots[u][j] <- W_home[slot_expert[u][j]] for every used
// slot ([P4] "The memory contract": rows [E, E+B) are local prefetch slots).
void oracle_prefetch(const uint16_t* w_home, const int32_t* slot_expert, int R, int B,
                     int64_t HHp, uint16_t* w_slots) {
    for (int u = 0; u < R; ++u)
        for (int j = 0; j < B; ++j) {
            int e = slot_expert[(int64_t)u * B + j];
            if (e < 0) continue;
            uint16_t* dst = w_slots + ((int64_t)u * B + j) * HHp;
            const uint16_t* src = w_home + (int64_t)e * HHp;
            // the row in 64 KiB pieces (one piece per iteration of the parallel build)
            const int64_t piece = 32768;
#pragma omp parallel for schedule(static)
            for (int64_t i = 0; i < HHp; i += piece)
                std::memcpy(dst + i, src + i,
                            sizeof(uint16_t) * (size_t)(HHp - i < piece ? HHp - i : piece));
        }
}

// reduce_grad ([P2], [P4] "The memory contract"): each home expert e
// gathers its replica gradients from every rank's reduce buffer, in
// ascending rank order, into its fp32 parameter gradient, and the consumed
// slots are zeroed.
//   for e in [0,E): for r = 0..R-1: for j with slot_expert[r][j] == e:
//       G[e] += red[r][j];  red[r][j] = 0
void oracle_reduce_grad(float* G, float* red, const int32_t* slot_expert, int R, int B, int E,
                        int64_t HHp) {
    for (int e = 0; e < E; ++e)
        for (int r = 0; r < R; ++r)
            for (int j = 0; j < B; ++j) {
                if (slot_expert[(int64_t)r * B + j] != e) continue;
                float* g = G + (int64_t)e * HHp;
                float* s = red + ((int64_t)r * B + j) * HHp;
#pragma omp parallel for schedule(static)
                for (int64_t i = 0; i < HHp; ++i) {
                    g[i] = g[i] + s[i];
                    s[i] = 0.0f;
                }
            }
}

}  // extern "C"
