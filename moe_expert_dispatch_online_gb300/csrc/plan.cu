// Online planner for balanced expert-parallel dispatch (sm_103a).
//
// MoonEP pages: "The core idea: dynamic redundant experts" (ai-maestro.online):
// a small number of redundant experts is planned on the GPU from the current
// router output so that every rank receives exactly S*K token-slots; "The
// problem MoonEP targets": maxvio = max_e(T_e/Tbar) - 1; "The memory contract":
// training duplicates experts from at most one remote home group per rank
// (B = E/R), inference (B < E/R) reads overflow experts from their home rows.
//
// The planning rule (the pages call the planner "near-optimal" and give no
// algorithm; this is the library's deterministic choice):
//   x_g = L_g - C for every home group g (L_g = tokens routed to g's experts).
//   Donors (x > 0) by x descending, recipients (x < 0) in a deque by deficit
//   descending, ties by lower g. Pop a recipient, attach it to the current
//   donor; a donor that overshoots re-enters at the front of the deque with
//   its new deficit and the next donor takes over.
//   Group g's slots are listed expert by expert, the experts in ascending
//   token count (ties: lower id), each expert's slots in (rank, token) order:
//   g keeps the first C - inflow_g, each child takes the next `flow` in
//   assignment order. The moving tail holds the group's largest experts, so a
//   child's range touches few experts and few replicas are planned. A replica of expert e on child u sits in slot e - parent(u)*G
//   (training) or, for inference, in one of B slots given to u's B most-loaded
//   remote experts (ties: lower id; slots in ascending id) with the rest
//   overflowing onto home row e.
//   Each rank's segments follow ascending row order, tokens in (rank, token)
//   order inside a segment.
//
// Kernels, all on one stream, no host synchronisation:
//   plan_hist  : one CTA per 256-token chunk: validates ids, counts experts per
//                chunk in shared memory                          -> off[E][NC]
//   plan_scan  : one CTA per expert: exclusive scan over chunks    -> off, T[E]
//   plan_solve : one CTA: maxvio, group loads, the tree, expert pieces, slot
//                map, segment lengths, cu_seqlens, piece bases
//   plan_dest  : one CTA per chunk: rank of every (token,k) among same-expert
//                entries (warp __match_any_sync + per-warp shared counters),
//                then dest = piece base + position in the expert's list.

#include <math.h>

#include "bep_internal.cuh"

namespace bep {
namespace {

constexpr int kHistThreads = 256;
constexpr int kScanThreads = 256;
constexpr int kSolveThreads = 1024;
constexpr int kDestWarps = kChunkTokens / 32;   // 8 warps, 32 tokens each

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Exclusive scan of one value per thread across the block; returns the
// exclusive prefix and writes the block total to *total. s_warp: >= 32 ints.
__device__ int block_excl_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    int incl = warp_incl_scan(v, lane);
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? s_warp[lane] : 0;
        int wi = warp_incl_scan(w, lane);
        if (lane < nwarps) s_warp[lane] = wi - w;
        if (lane == 31) s_warp[32] = wi;
    }
    __syncthreads();
    int out = s_warp[warp] + incl - v;
    *total = s_warp[32];
    __syncthreads();
    return out;
}

// In-place exclusive scan of a shared array of n ints; returns the total.
__device__ int block_excl_scan_array(int* a, int n, int* s_warp) {
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += a[i];
    int total;
    int run = block_excl_scan(sum, s_warp, &total);
    for (int i = lo; i < hi; ++i) {
        int v = a[i];
        a[i] = run;
        run += v;
    }
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kHistThreads) plan_hist_kernel(Dims d, const int32_t* __restrict__ topk,
                                                                 Workspace ws) {
    extern __shared__ int32_t s_cnt[];   // [E]
    const int c = blockIdx.x;
    const int r = c / d.NCH;
    const int t0 = (c % d.NCH) * kChunkTokens;
    const int ntok = min(kChunkTokens, d.S - t0);
    for (int e = threadIdx.x; e < d.E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    int bad = 0;
    if ((int)threadIdx.x < ntok) {
        const int32_t* ids = topk + ((int64_t)r * d.S + t0 + threadIdx.x) * d.K;
        for (int k = 0; k < d.K; ++k) {
            const int v = ids[k];
            if (v < 0 || v >= d.E) {
                bad |= BEP_DERR_EXPERT_ID;
                continue;
            }
            for (int k2 = 0; k2 < k; ++k2)
                if (ids[k2] == v) bad |= BEP_DERR_DUP_ID;
            atomicAdd(&s_cnt[v], 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < d.E; e += blockDim.x) ws.off[(int64_t)e * d.NC + c] = s_cnt[e];
    if (bad) {
        set_status(ws.status, bad);
        set_status(ws.plan_err, bad);
    }
}

__global__ void __launch_bounds__(kScanThreads) plan_scan_kernel(Dims d, Workspace ws) {
    __shared__ int s_warp[33];
    const int e = blockIdx.x;
    int32_t* row = ws.off + (int64_t)e * d.NC;
    const int per = (d.NC + blockDim.x - 1) / blockDim.x;
    const int lo = min(d.NC, (int)threadIdx.x * per), hi = min(d.NC, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += row[i];
    int total;
    int run = block_excl_scan(sum, s_warp, &total);
    for (int i = lo; i < hi; ++i) {
        int v = row[i];
        row[i] = run;
        run += v;
    }
    if (threadIdx.x == 0) ws.T[e] = total;
}

__global__ void __launch_bounds__(kSolveThreads) plan_solve_kernel(Dims d, Workspace ws,
                                                                   int32_t* __restrict__ cu,
                                                                   int32_t* __restrict__ slot_expert,
                                                                   double* __restrict__ maxvio) {
    extern __shared__ int32_t sm[];
    int32_t* sT = sm;              // [E]
    int32_t* sGS = sT + d.E;       // [E]  start of expert e inside its group's list
    int32_t* sNP = sGS + d.E;      // [E+1] piece counts, then first piece
    __shared__ int s_warp[33];
    __shared__ int64_t sL[kMaxR];
    __shared__ int sParent[kMaxR];
    __shared__ int64_t sInflow[kMaxR];
    __shared__ int sEdgeDonor[kMaxR], sEdgeChild[kMaxR];
    __shared__ int64_t sEdgeFlow[kMaxR];
    __shared__ int sRangeFirst[kMaxR + 1];
    __shared__ int64_t sRangeEnd[2 * kMaxR];
    __shared__ int sRangeOwner[2 * kMaxR];
    __shared__ int sMax, sFail;

    const int tid = threadIdx.x, nth = blockDim.x;
    const int R = d.R, E = d.E, B = d.B, G = d.G, NROW = d.NROW;
    const int64_t C = d.C;

    if (*(volatile int32_t*)ws.plan_err) {
        // routing rejected by plan_hist: publish an empty plan
        for (int i = tid; i < R * (NROW + 1); i += nth) cu[i] = 0;
        for (int i = tid; i < R * B; i += nth) slot_expert[i] = -1;
        if (tid == 0) *maxvio = nan("");
        return;
    }

    // 1. counts, maxvio ([P4] "The problem MoonEP targets")
    if (tid == 0) {
        sMax = 0;
        sFail = 0;
    }
    __syncthreads();
    int mx = 0;
    for (int e = tid; e < E; e += nth) {
        const int v = ws.T[e];
        sT[e] = v;
        mx = max(mx, v);
    }
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) atomicMax(&sMax, mx);
    for (int i = tid; i < R * NROW; i += nth) ws.lens[i] = 0;
    for (int i = tid; i < R * B; i += nth) slot_expert[i] = -1;
    __syncthreads();
    if (tid == 0) {
        const int64_t rsk = (int64_t)R * C;
        *maxvio = rsk ? (double)((int64_t)E * sMax - rsk) / (double)rsk : 0.0;
    }

    // 2. group loads, and each expert's start inside its group's list: the tokens
    //    of the group's experts with a smaller count, or an equal count and a lower id
    for (int e = tid; e < E; e += nth) {
        const int g0 = (e / G) * G;
        const int te = sT[e];
        int64_t start = 0;
        for (int f = g0; f < g0 + G; ++f) {
            const int tf = sT[f];
            if (tf < te || (tf == te && f < e)) start += tf;
        }
        sGS[e] = (int32_t)start;
    }
    if (tid < R) {
        int64_t run = 0;
        for (int e = tid * G; e < (tid + 1) * G; ++e) run += sT[e];
        sL[tid] = run;
    }
    __syncthreads();

    // 3. the tree (serial over R <= 64 ranks) and each group's ranges
    if (tid == 0) {
        int64_t x[kMaxR];
        int donors[kMaxR], rq[kMaxR];
        int64_t rdef[kMaxR];
        int nd = 0, nr = 0;
        for (int g = 0; g < R; ++g) {
            x[g] = sL[g] - C;
            sParent[g] = -1;
            sInflow[g] = 0;
            if (x[g] > 0) {      // stable insertion by x descending
                int p = nd++;
                while (p > 0 && x[donors[p - 1]] < x[g]) {
                    donors[p] = donors[p - 1];
                    --p;
                }
                donors[p] = g;
            } else if (x[g] < 0) {  // stable insertion by deficit descending
                int p = nr++;
                while (p > 0 && rdef[p - 1] < -x[g]) {
                    rq[p] = rq[p - 1];
                    rdef[p] = rdef[p - 1];
                    --p;
                }
                rq[p] = g;
                rdef[p] = -x[g];
            }
        }
        int head = 0, di = 0, ne = 0;
        while (head < nr) {
            const int u = rq[head];
            const int64_t D = rdef[head];
            ++head;
            if (di >= nd) {
                sFail = 1;
                break;
            }
            const int dn = donors[di];
            sParent[u] = dn;
            sInflow[u] = D;
            sEdgeDonor[ne] = dn;
            sEdgeChild[ne] = u;
            sEdgeFlow[ne] = D;
            ++ne;
            x[dn] -= D;
            if (x[dn] < 0) {      // overshoot: dn now lacks -x, served next
                --head;
                rq[head] = dn;
                rdef[head] = -x[dn];
                ++di;
            } else if (x[dn] == 0) {
                ++di;
            }
        }
        int idx = 0;
        for (int g = 0; g < R; ++g) {
            sRangeFirst[g] = idx;
            int64_t pos = C - sInflow[g];
            sRangeEnd[idx] = pos;
            sRangeOwner[idx] = g;
            ++idx;
            for (int i = 0; i < ne; ++i)
                if (sEdgeDonor[i] == g) {
                    pos += sEdgeFlow[i];
                    sRangeEnd[idx] = pos;
                    sRangeOwner[idx] = sEdgeChild[i];
                    ++idx;
                }
            if (pos != sL[g]) sFail = 1;
        }
        sRangeFirst[R] = idx;
    }
    __syncthreads();

    // 4. pieces: the intersection of each expert's run with its group's ranges
    for (int e = tid; e < E; e += nth) {
        const int g = e / G;
        const int64_t a = sGS[e], b = a + sT[e];
        int n = 0;
        int64_t lo = 0;
        for (int i = sRangeFirst[g]; i < sRangeFirst[g + 1]; ++i) {
            const int64_t hi = sRangeEnd[i];
            if (i64max(a, lo) < i64min(b, hi)) ++n;
            lo = hi;
        }
        sNP[e] = n;
    }
    __syncthreads();
    const int npieces = block_excl_scan_array(sNP, E, s_warp);
    if (tid == 0) sNP[E] = npieces;
    __syncthreads();
    for (int e = tid; e < E; e += nth) {
        const int g = e / G;
        const int64_t a = sGS[e], b = a + sT[e];
        int idx = sNP[e];
        int64_t lo = 0;
        for (int i = sRangeFirst[g]; i < sRangeFirst[g + 1]; ++i) {
            const int64_t hi = sRangeEnd[i];
            const int64_t s0 = i64max(a, lo), s1 = i64min(b, hi);
            if (s0 < s1) {
                const int owner = sRangeOwner[i];
                ws.pstart[idx] = (int32_t)(s0 - a);
                ws.plen[idx] = (int32_t)(s1 - s0);
                ws.prank[idx] = owner;
                int row;
                if (owner == g) row = e;                                    // home row
                else if (d.mode == BEP_TRAIN) row = E + (e - g * G);        // slot of the donor group
                else row = -1;                                              // decided in step 5
                ws.prow[idx] = row;
                if (owner != g && d.mode == BEP_TRAIN) slot_expert[owner * B + (e - g * G)] = e;
                ++idx;
            }
            lo = hi;
        }
        ws.pfirst[e] = sNP[e];
    }
    if (tid == 0) ws.pfirst[E] = npieces;
    __syncthreads();

    // 5. inference: top-B remote experts of each child get slots, the rest overflow.
    //    One warp per child u of group g. A child's range is contiguous in g's list and
    //    each expert's run is contiguous, so expert e has at most one piece on u. Each of
    //    B rounds picks the unselected piece with the most slots, ties to the lower expert
    //    id (a warp argmax over the lanes' own bests, each lane scanning its experts in
    //    ascending id); then the selected experts take slots E+0.. in ascending id and the
    //    others overflow onto their home rows.
    if (d.mode == BEP_INFER) {
        const int lane = tid & 31, warp = tid >> 5, nwarps = nth >> 5;
        for (int u = warp; u < R; u += nwarps) {
            const int g = sParent[u];
            if (g < 0) continue;
            auto piece_on_u = [&](int e) -> int {
                for (int i = ws.pfirst[e]; i < ws.pfirst[e + 1]; ++i)
                    if (ws.prank[i] == u) return i;
                return -1;
            };
            for (int j = 0; j < B; ++j) {
                int bl = -1, be = 0x7fffffff, bi = -1;
                for (int e = g * G + lane; e < (g + 1) * G; e += 32) {
                    const int i = piece_on_u(e);
                    if (i >= 0 && ws.prow[i] == -1 && ws.plen[i] > bl) {
                        bl = ws.plen[i];
                        be = e;
                        bi = i;
                    }
                }
                for (int o = 16; o > 0; o >>= 1) {
                    const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (ol > bl || (ol == bl && oe < be)) {
                        bl = ol;
                        be = oe;
                        bi = oi;
                    }
                }
                if (bl < 0) break;          // the same on every lane
                if (lane == 0) ws.prow[bi] = -2;   // selected
                __syncwarp();
            }
            int jrun = 0;
            for (int base = g * G; base < (g + 1) * G; base += 32) {
                const int e = base + lane;
                const int i = e < (g + 1) * G ? piece_on_u(e) : -1;
                const bool sel = i >= 0 && ws.prow[i] == -2;
                const unsigned m = __ballot_sync(0xffffffffu, sel);
                if (i >= 0) {
                    if (sel) {
                        const int jj = jrun + __popc(m & ((1u << lane) - 1u));
                        ws.prow[i] = E + jj;
                        slot_expert[u * B + jj] = e;
                    } else {
                        ws.prow[i] = e;   // overflow: the GEMM reads home row e
                    }
                }
                jrun += __popc(m);
            }
        }
        __syncthreads();
    }

    // 6. segment lengths (at most one piece per (rank, row)), cu_seqlens per rank
    for (int i = tid; i < npieces; i += nth) ws.lens[ws.prank[i] * NROW + ws.prow[i]] = ws.plen[i];
    __syncthreads();
    {
        const int lane = tid & 31, warp = tid >> 5, nwarps = nth >> 5;
        for (int u = warp; u < R; u += nwarps) {
            int run = 0;
            for (int base = 0; base < NROW; base += 32) {
                const int rr = base + lane;
                const int v = rr < NROW ? ws.lens[u * NROW + rr] : 0;
                const int incl = warp_incl_scan(v, lane);
                if (rr < NROW) cu[u * (NROW + 1) + rr] = run + incl - v;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) {
                cu[u * (NROW + 1) + NROW] = run;
                if (run != C) sFail = 1;
            }
        }
    }
    __syncthreads();
    // 7. dest base of every piece
    for (int i = tid; i < npieces; i += nth) {
        const int u = ws.prank[i];
        ws.pbase[i] = (int32_t)(u * C + cu[u * (NROW + 1) + ws.prow[i]] - ws.pstart[i]);
    }
    if (tid == 0 && sFail) {
        set_status(ws.status, BEP_DERR_INFEASIBLE);
        set_status(ws.plan_err, BEP_DERR_INFEASIBLE);
    }
}

__global__ void __launch_bounds__(kDestWarps * 32) plan_dest_kernel(Dims d, Workspace ws,
                                                                     const int32_t* __restrict__ topk,
                                                                     int32_t* __restrict__ dest) {
    extern __shared__ int32_t sm[];
    int32_t* s_cnt = sm;                            // [8][E] per-warp counts, then warp bases
    int32_t* s_lr = sm + kDestWarps * d.E;          // [256*K] rank inside the warp's entries
    const int c = blockIdx.x;
    const int r = c / d.NCH;
    const int t0 = (c % d.NCH) * kChunkTokens;
    const int ntok = min(kChunkTokens, d.S - t0);
    const int64_t tok0 = (int64_t)r * d.S + t0;
    const int K = d.K, E = d.E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    if (*(volatile int32_t*)ws.plan_err) {
        for (int q = threadIdx.x; q < ntok * K; q += blockDim.x) dest[tok0 * K + q] = -1;
        return;
    }
    for (int i = threadIdx.x; i < kDestWarps * E; i += blockDim.x) s_cnt[i] = 0;
    __syncthreads();

    // phase 1: each warp ranks its 32 tokens' entries in (token, k) order
    const int wtok = max(0, min(32, ntok - warp * 32));
    const int n_ent = wtok * K;
    const int32_t* wids = topk + (tok0 + warp * 32) * K;
    int32_t* wcnt = s_cnt + warp * E;
    int32_t* wlr = s_lr + warp * 32 * K;
    for (int base = 0; base < 32 * K; base += 32) {
        const int q = base + lane;
        const bool valid = q < n_ent;
        const int e = valid ? wids[q] : -1;
        const unsigned mask = __match_any_sync(0xffffffffu, e);
        const int lr = __popc(mask & ((1u << lane) - 1u));
        int prev = 0;
        if (valid) {
            prev = wcnt[e];
            wlr[q] = prev + lr;
        }
        __syncwarp();
        if (valid && lr == 0) wcnt[e] = prev + __popc(mask);
        __syncwarp();
    }
    __syncthreads();

    // phase 2: warp bases = chunk offset + counts of the earlier warps
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = ws.off[(int64_t)e * d.NC + c];
        for (int w = 0; w < kDestWarps; ++w) {
            const int v = s_cnt[w * E + e];
            s_cnt[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();

    // phase 3: position in the expert's list -> piece -> dest
    for (int q = lane; q < n_ent; q += 32) {
        const int e = wids[q];
        const int p = wcnt[e] + wlr[q];
        int i = ws.pfirst[e];
        const int iend = ws.pfirst[e + 1];
        while (i + 1 < iend && p >= ws.pstart[i] + ws.plen[i]) ++i;
        dest[(tok0 + warp * 32) * K + q] = ws.pbase[i] + p;
    }
}

}  // namespace

cudaError_t plan_setup(int device) {
    (void)device;
    cudaError_t err;
    err = cudaFuncSetAttribute(plan_dest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (kDestWarps * kMaxE + kChunkTokens * kMaxK) * 4);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(plan_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (3 * kMaxE + 1) * 4);
    return err;
}

cudaError_t launch_plan(const Dims& d, const Workspace& ws, const int32_t* topk, int32_t* cu,
                        int32_t* slot_expert, int32_t* dest, double* maxvio, cudaStream_t st) {
    cudaError_t err = cudaMemsetAsync(ws.plan_err, 0, sizeof(int32_t), st);
    if (err != cudaSuccess) return err;
    if (d.NC > 0) {
        plan_hist_kernel<<<d.NC, kHistThreads, d.E * 4, st>>>(d, topk, ws);
    }
    plan_scan_kernel<<<d.E, kScanThreads, 0, st>>>(d, ws);
    plan_solve_kernel<<<1, kSolveThreads, (3 * d.E + 1) * 4, st>>>(d, ws, cu, slot_expert, maxvio);
    if (d.NC > 0) {
        plan_dest_kernel<<<d.NC, kDestWarps * 32, (kDestWarps * d.E + kChunkTokens * d.K) * 4, st>>>(
            d, ws, topk, dest);
    }
    return cudaGetLastError();
}

}  // namespace bep

// ---------------------------------------------------------------------------
// Planner entry point that allocates nothing (declared in include/bep.h).
//
// Some callers cannot call cudaMalloc when they plan: services whose device
// memory is handed out once at start-up and may not grow afterwards, and
// embedders (plug-ins inside a host framework that owns the allocator, or
// code that cannot keep a bep_ctx alive between calls). This variant takes the
// configuration directly and keeps the planner's scratch tables in a
// file-scope device array that every GPU loading the library reserves until
// the process exits.
//
// Host code must not hand the array's symbol to a kernel: on the host it is a
// stand-in, not a device address. The device address is fetched with
// cudaGetSymbolAddress once per CUDA context, on the first call made in that
// context (normally a device's primary context), which also sets the planner
// kernels' shared-memory limits. That first call should therefore come
// before any stream capture. The cache is keyed on the context's unique id,
// so a device reset or a second context on the same device repeats the
// set-up instead of reusing an address from a context that no longer exists.
// Every call shares the one array: calls whose work overlaps on the GPU
// (other streams, other threads) race on it and must be serialised by the
// caller.
#include <cuda.h>

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)2 << 20;   // 2 MiB
constexpr int kNoAllocMaxContexts = 64;

__device__ __align__(256) int32_t g_plan_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

// One entry per CUDA context that has called bep_plan_noalloc: the context's
// unique id (cuCtxGetId) and the array's device address in it.
struct NoAllocEntry {
    unsigned long long ctx_id;
    int32_t* addr;
};
std::mutex g_noalloc_mutex;
NoAllocEntry g_noalloc[kNoAllocMaxContexts] = {};
int g_noalloc_n = 0;      // entries in use
int g_noalloc_next = 0;   // when all are in use, the one to replace next (oldest first)

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The current context's unique id, through the driver entry points the runtime
// hands out (no link against libcuda). Returns false if there is none yet.
bool current_ctx_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (!get_current || !get_id) {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault,
                                             &qa) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
                cudaSuccess ||
            qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess || !a || !b)
            return false;
        get_current = reinterpret_cast<CtxGetCurrentFn>(a);
        get_id = reinterpret_cast<CtxGetIdFn>(b);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Scratch bytes the planner needs for d (the same tables bep_create carves).
size_t noalloc_bytes(const bep::Dims& d) {
    const size_t E = d.E, R = d.R, NC = d.NC, NROW = d.NROW, NP = (size_t)d.E + d.R;
    auto rnd = [](size_t n) { return (n * sizeof(int32_t) + 255) & ~(size_t)255; };
    return rnd(1) + rnd(E * (NC > 0 ? NC : 1)) + rnd(E) + rnd(R * NROW) + rnd(E + 1) + 5 * rnd(NP);
}

int32_t* carve_i32(char*& p, size_t n) {
    int32_t* out = reinterpret_cast<int32_t*>(p);
    p += (n * sizeof(int32_t) + 255) & ~(size_t)255;
    return out;
}

}  // namespace

extern "C" int bep_plan_noalloc(const bep_config* cfg, const int32_t* topk, int32_t* cu_seqlens,
                                int32_t* slot_expert, int32_t* dest, double* maxvio,
                                int32_t* device_err, void* stream) {
    if (!cfg || !cu_seqlens || !maxvio || !device_err) return BEP_ERR_ARG;
    bep::Dims d;
    const int rc = bep::make_dims(cfg, &d);
    if (rc) return rc;
    if (d.R * d.B > 0 && !slot_expert) return BEP_ERR_ARG;
    if (d.C > 0 && (!topk || !dest)) return BEP_ERR_ARG;
    auto al = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
    if (!al(topk, 4) || !al(cu_seqlens, 4) || !al(slot_expert, 4) || !al(dest, 4) ||
        !al(maxvio, 8) || !al(device_err, 4))
        return BEP_ERR_ALIGN;
    if (noalloc_bytes(d) > kNoAllocScratchBytes) return BEP_ERR_SIZE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BEP_ERR_CUDA;
    int32_t* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        unsigned long long id = 0;
        bool known = current_ctx_id(&id);
        if (known) {
            for (int i = 0; i < g_noalloc_n; ++i)
                if (g_noalloc[i].ctx_id == id) base = g_noalloc[i].addr;
        }
        if (!base) {
            // First call in this context: look the array up (this also makes the
            // device's primary context current if none was), set the kernels up.
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || !p) return BEP_ERR_CUDA;
            if (bep::plan_setup(dev) != cudaSuccess) return BEP_ERR_CUDA;
            if (!known && !current_ctx_id(&id)) return BEP_ERR_CUDA;
            int slot = -1;
            for (int i = 0; i < g_noalloc_n; ++i)
                if (g_noalloc[i].ctx_id == id) slot = i;
            if (slot < 0) {
                if (g_noalloc_n < kNoAllocMaxContexts) {
                    slot = g_noalloc_n++;
                } else {
                    slot = g_noalloc_next;
                    g_noalloc_next = (g_noalloc_next + 1) % kNoAllocMaxContexts;
                }
            }
            g_noalloc[slot] = {id, static_cast<int32_t*>(p)};
            base = g_noalloc[slot].addr;
        }
    }

    // The planner's tables, carved from the static array in bep_create's order. Only the
    // per-call error word must start at zero (launch_plan clears it); every other table is
    // fully rewritten by the kernels before it is read.
    char* p = reinterpret_cast<char*>(base);
    bep::Workspace ws = {};
    ws.status = device_err;
    ws.plan_err = carve_i32(p, 1);
    ws.off = carve_i32(p, (size_t)d.E * (d.NC > 0 ? d.NC : 1));
    ws.T = carve_i32(p, d.E);
    ws.lens = carve_i32(p, (size_t)d.R * d.NROW);
    ws.pfirst = carve_i32(p, (size_t)d.E + 1);
    ws.pstart = carve_i32(p, (size_t)d.E + d.R);
    ws.plen = carve_i32(p, (size_t)d.E + d.R);
    ws.prank = carve_i32(p, (size_t)d.E + d.R);
    ws.prow = carve_i32(p, (size_t)d.E + d.R);
    ws.pbase = carve_i32(p, (size_t)d.E + d.R);

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(device_err, 0, sizeof(int32_t), st) != cudaSuccess) return BEP_ERR_CUDA;
    return bep::launch_plan(d, ws, topk, cu_seqlens, slot_expert, dest, maxvio, st) == cudaSuccess
               ? BEP_OK
               : BEP_ERR_CUDA;
}
