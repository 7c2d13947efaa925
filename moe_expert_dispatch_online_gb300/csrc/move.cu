// HBM-bound stages of balanced expert-parallel dispatch (sm_103a):
// fused permute/dispatch, weighted combine, combine backward, prefetch_weight
// and reduce_grad.
//
// MoonEP pages (ai-maestro.online): "The core idea: dynamic redundant experts"
// (zero copy: permute/unpermute fused, tokens written straight into their
// expert-grouped positions; duplicated experts prefetched before expert
// compute; their gradients reduced back to the home ranks) and "The memory
// contract" (rows [E, E+B) are prefetch slots filled by prefetch_weight;
// reduce_grad reads each expert's slots from every rank, accumulates them into
// the home gradient and zeroes the consumed slots).
//
// Every row moves as 16-byte vectors. One warp owns one token: it reads the
// token's K destinations (lane k holds dest k), then streams the row with
// several independent 16-byte loads in flight per lane. Grids are a multiple
// of the SM count; warps stride over tokens. When there are fewer tokens than
// warps in the grid (small batches), each row is cut into `pieces` runs of
// 32*U vectors and a warp owns one (token, piece) item, so every warp of the
// grid has rows in flight.

#include <cuda_bf16.h>

#include "bep_internal.cuh"

namespace bep {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even, lo in the low half
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float* f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// Loads lane k's dest (k < K) and checks it. Returns the lane's dest; *okmask
// gets one bit per k whose dest lies inside the receive space.
__device__ __forceinline__ int load_dest(const int32_t* __restrict__ dest, int64_t tok, int K,
                                         int64_t nrows, unsigned* okmask, int32_t* status) {
    const int lane = threadIdx.x & 31;
    int dl = 0;
    bool ok = true;
    if (lane < K) {
        dl = dest[tok * K + lane];
        ok = dl >= 0 && (int64_t)dl < nrows;
    }
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (m != 0xffffffffu && lane == 0) set_status(status, BEP_DERR_BOUNDS);
    *okmask = m;
    return dl;
}

// The vectors [*v_lo, *v_hi) of item `item`'s row piece, for rows of nvec vectors cut
// into `pieces` runs of whole 32*U-vector steps; returns the item's token.
template <int U>
__device__ __forceinline__ int64_t piece_of(int64_t item, int pieces, int nvec, int* v_lo,
                                            int* v_hi) {
    if (pieces == 1) {
        *v_lo = 0;
        *v_hi = nvec;
        return item;
    }
    const int64_t tok = item / pieces;
    const int piece = (int)(item - tok * pieces);
    const int steps = (nvec + 32 * U - 1) / (32 * U);
    const int per = (steps + pieces - 1) / pieces;
    *v_lo = min(nvec, piece * per * 32 * U);
    *v_hi = min(nvec, (piece + 1) * per * 32 * U);
    return tok;
}

// ----------------------------------------------------------------------------- dispatch
// recv[dest[tok, k], :] = x[tok, :]
template <int U>
__global__ void __launch_bounds__(kThreads) dispatch_kernel(const uint4* __restrict__ x,
                                                            const int32_t* __restrict__ dest,
                                                            uint4* __restrict__ recv, int64_t ntok,
                                                            int K, int nvec, int64_t nrows,
                                                            int pieces, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t nitem = ntok * pieces;
    for (int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < nitem;
         item += nwarps) {
        int v_lo, v_hi;
        const int64_t tok = piece_of<U>(item, pieces, nvec, &v_lo, &v_hi);
        unsigned okmask;
        const int dl = load_dest(dest, tok, K, nrows, &okmask, status);
        const uint4* src = x + tok * nvec;
        for (int v0 = v_lo; v0 < v_hi; v0 += 32 * U) {
            uint4 val[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < v_hi) val[u] = ld_stream(src + v);
            }
            for (int k = 0; k < K; ++k) {
                const int dk = __shfl_sync(0xffffffffu, dl, k);
                if (!((okmask >> k) & 1u)) continue;
                uint4* dst = recv + (int64_t)dk * nvec;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + u * 32 + lane;
                    if (v < v_hi) dst[v] = val[u];
                }
            }
        }
    }
}

// ----------------------------------------------------------------------------- combine
// kWeighted:  out[tok, c] = bf16_rne(acc), acc = 0; for k in 0..K-1:
//             acc = fma(g[tok,k], y[dest[tok,k], c], acc)
// !kWeighted (backward of the dispatch): acc = acc + y[dest[tok,k], c] instead.
template <bool kWeighted>
__device__ __forceinline__ float combine_step(float g, float v, float acc) {
    return kWeighted ? __fmaf_rn(g, v, acc) : __fadd_rn(acc, v);
}

// kPieces: rows cut into pieces (small batches of long rows); without it a warp owns
// whole rows, which measured faster for this gather wherever rows are short or tokens
// many (the instance without pieces is the one combine always uses).
template <int U, bool kWeighted, bool kPieces>
__global__ void __launch_bounds__(kThreads) combine_kernel(const uint4* __restrict__ y,
                                                           const int32_t* __restrict__ dest,
                                                           const float* __restrict__ gates,
                                                           uint4* __restrict__ out, int64_t ntok,
                                                           int K, int nvec, int64_t nrows,
                                                           int pieces, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t nitem = kPieces ? ntok * pieces : ntok;
    for (int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < nitem;
         item += nwarps) {
        int v_lo = 0, v_hi = nvec;
        int64_t tok = item;
        if (kPieces) tok = piece_of<U>(item, pieces, nvec, &v_lo, &v_hi);
        unsigned okmask;
        const int dl = load_dest(dest, tok, K, nrows, &okmask, status);
        const float gl = (kWeighted && lane < K) ? gates[tok * K + lane] : 1.0f;
        for (int v0 = v_lo; v0 < v_hi; v0 += 32 * U) {
            float acc[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
            int k = 0;
            // two k at a time: both rows' loads are in flight before the (ordered) fmas
            for (; k + 1 < K; k += 2) {
                const int d0 = __shfl_sync(0xffffffffu, dl, k);
                const int d1 = __shfl_sync(0xffffffffu, dl, k + 1);
                const float g0 = __shfl_sync(0xffffffffu, gl, k);
                const float g1 = __shfl_sync(0xffffffffu, gl, k + 1);
                const bool ok0 = (okmask >> k) & 1u, ok1 = (okmask >> (k + 1)) & 1u;
                uint4 q0[U], q1[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + u * 32 + lane;
                    q0[u] = make_uint4(0, 0, 0, 0);
                    q1[u] = make_uint4(0, 0, 0, 0);
                    if (v < v_hi) {
                        if (ok0) q0[u] = ld_stream(y + (int64_t)d0 * nvec + v);
                        if (ok1) q1[u] = ld_stream(y + (int64_t)d1 * nvec + v);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float f[8];
                    bf16x8_to_f32(q0[u], f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[u][i] = combine_step<kWeighted>(g0, f[i], acc[u][i]);
                    bf16x8_to_f32(q1[u], f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[u][i] = combine_step<kWeighted>(g1, f[i], acc[u][i]);
                }
            }
            if (k < K) {
                const int d0 = __shfl_sync(0xffffffffu, dl, k);
                const float g0 = __shfl_sync(0xffffffffu, gl, k);
                const bool ok0 = (okmask >> k) & 1u;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + u * 32 + lane;
                    uint4 q = make_uint4(0, 0, 0, 0);
                    if (v < v_hi && ok0) q = ld_stream(y + (int64_t)d0 * nvec + v);
                    float f[8];
                    bf16x8_to_f32(q, f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[u][i] = combine_step<kWeighted>(g0, f[i], acc[u][i]);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < v_hi) out[tok * nvec + v] = f32x8_to_bf16(acc[u]);
            }
        }
    }
}

// ----------------------------------------------------------------------------- combine backward
// dy[dest[tok,k], c] = bf16_rne(g[tok,k] * dout[tok, c])
// kPieces as for combine_kernel: the instance with (token, piece) items measured faster at
// large batches and at every size for long rows; whole rows per warp (the other instance)
// measured faster for short rows in small batches (about 4,000-8,000 tokens of 2048).
template <int U, bool kPieces>
__global__ void __launch_bounds__(kThreads) combine_bwd_kernel(const uint4* __restrict__ dout,
                                                               const int32_t* __restrict__ dest,
                                                               const float* __restrict__ gates,
                                                               uint4* __restrict__ dy, int64_t ntok,
                                                               int K, int nvec, int64_t nrows,
                                                               int pieces, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t nitem = kPieces ? ntok * pieces : ntok;
    for (int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < nitem;
         item += nwarps) {
        int v_lo = 0, v_hi = nvec;
        int64_t tok = item;
        if (kPieces) tok = piece_of<U>(item, pieces, nvec, &v_lo, &v_hi);
        unsigned okmask;
        const int dl = load_dest(dest, tok, K, nrows, &okmask, status);
        const float gl = lane < K ? gates[tok * K + lane] : 0.0f;
        const uint4* src = dout + tok * nvec;
        for (int v0 = v_lo; v0 < v_hi; v0 += 32 * U) {
            float f[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * 32 + lane;
                uint4 q = make_uint4(0, 0, 0, 0);
                if (v < v_hi) q = ld_stream(src + v);
                bf16x8_to_f32(q, f[u]);
            }
            for (int k = 0; k < K; ++k) {
                const int dk = __shfl_sync(0xffffffffu, dl, k);
                const float gk = __shfl_sync(0xffffffffu, gl, k);
                if (!((okmask >> k) & 1u)) continue;
                uint4* dst = dy + (int64_t)dk * nvec;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + u * 32 + lane;
                    float p[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) p[i] = __fmul_rn(gk, f[u][i]);
                    if (v < v_hi) dst[v] = f32x8_to_bf16(p);
                }
            }
        }
    }
}

// ----------------------------------------------------------------------------- gate gradient
// dg[tok, k] = sum_c dout[tok, c] * y[dest[tok,k], c] in fp32: each lane sums its
// columns (16-byte vectors lane, lane+32, ...), then a butterfly reduces the warp.
__global__ void __launch_bounds__(kThreads) combine_dgates_kernel(const uint4* __restrict__ dout,
                                                                  const uint4* __restrict__ y,
                                                                  const int32_t* __restrict__ dest,
                                                                  float* __restrict__ dg,
                                                                  int64_t ntok, int K, int nvec,
                                                                  int64_t nrows, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t tok = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; tok < ntok;
         tok += nwarps) {
        unsigned okmask;
        const int dl = load_dest(dest, tok, K, nrows, &okmask, status);
        const uint4* src = dout + tok * nvec;
        for (int k = 0; k < K; ++k) {
            const int dk = __shfl_sync(0xffffffffu, dl, k);
            const bool ok = (okmask >> k) & 1u;
            float acc = 0.0f;
            if (ok) {
                const uint4* yr = y + (int64_t)dk * nvec;
                for (int v0 = 0; v0 < nvec; v0 += 128) {
                    uint4 a[4], b[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int v = v0 + u * 32 + lane;
                        a[u] = v < nvec ? src[v] : make_uint4(0, 0, 0, 0);
                        b[u] = v < nvec ? ld_stream(yr + v) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float fa[8], fb[8];
                        bf16x8_to_f32(a[u], fa);
                        bf16x8_to_f32(b[u], fb);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc = __fmaf_rn(fa[i], fb[i], acc);
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) dg[tok * K + k] = ok ? acc : 0.0f;
        }
    }
}

// ----------------------------------------------------------------------------- prefetch
// w_slots[s] = w_home[slot_expert[s]] for every used slot s = u*B + j. Each slot is
// one contiguous [H, H'] block of 32 KB tiles; the (used slot, tile) pairs are spread
// over the whole grid, slot by slot, so every CTA copies about the same number of tiles.
constexpr int kCopyU = 8;   // 16-byte vectors per thread per tile

__global__ void __launch_bounds__(kThreads) prefetch_kernel(const int32_t* __restrict__ slot_expert,
                                                            const uint4* __restrict__ w_home,
                                                            uint4* __restrict__ w_slots, int nslots,
                                                            int E, int64_t nvec, int32_t* status) {
    __shared__ int32_t s_slot[kMaxE];   // used slots in ascending order (nslots = R*B <= E <= kMaxE)
    __shared__ int32_t s_exp[kMaxE];    // their experts
    __shared__ int s_nused;
    if (threadIdx.x < 32) {
        // warp 0 lists the used slots: one ballot per 32 entries keeps their order
        const int lane = threadIdx.x;
        int n = 0;
        for (int b = 0; b < nslots; b += 32) {
            const int sl = b + lane;
            int e = sl < nslots ? slot_expert[sl] : -1;
            if (e >= E) {
                if (blockIdx.x == 0) set_status(status, BEP_DERR_BOUNDS);
                e = -1;
            }
            const unsigned m = __ballot_sync(0xffffffffu, e >= 0);
            if (e >= 0) {
                const int at = n + __popc(m & ((1u << lane) - 1u));
                s_slot[at] = sl;
                s_exp[at] = e;
            }
            n += __popc(m);
        }
        if (lane == 0) s_nused = n;
    }
    __syncthreads();
    const int64_t tile_vec = (int64_t)kThreads * kCopyU;
    const int64_t ntile = (nvec + tile_vec - 1) / tile_vec;
    const int64_t nwork = (int64_t)s_nused * ntile;
    for (int64_t w = blockIdx.x; w < nwork; w += gridDim.x) {
        const int k = (int)(w / ntile);
        const int64_t t = w - (int64_t)k * ntile;
        const uint4* src = w_home + (int64_t)s_exp[k] * nvec;
        uint4* dst = w_slots + (int64_t)s_slot[k] * nvec;
        const int64_t base = t * tile_vec + threadIdx.x;
        uint4 v[kCopyU];
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            const int64_t i = base + (int64_t)u * kThreads;
            if (i < nvec) v[u] = ld_stream(src + i);
        }
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            const int64_t i = base + (int64_t)u * kThreads;
            if (i < nvec) dst[i] = v[u];
        }
    }
}

// ----------------------------------------------------------------------------- reduce_grad
// One CTA lists, for every home expert e with replicas, its slots in ascending
// (rank, slot) order.
__global__ void __launch_bounds__(1024) reduce_grad_prep_kernel(const int32_t* __restrict__ slot_expert,
                                                                int nslots, int E, Workspace ws) {
    extern __shared__ int32_t sm[];
    int32_t* s_se = sm;            // [nslots]
    int32_t* s_n = sm + nslots;    // [E]
    int32_t* s_t = s_n + E;        // [E]
    __shared__ int s_tot[2];
    for (int s = threadIdx.x; s < nslots; s += blockDim.x) {
        int e = slot_expert[s];
        if (e < -1 || e >= E) {
            set_status(ws.status, BEP_DERR_BOUNDS);
            e = -1;
        }
        s_se[s] = e;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int n = 0;
        for (int s = 0; s < nslots; ++s) n += s_se[s] == e;
        s_n[e] = n;
        s_t[e] = n > 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {   // E <= 2048: two serial scans are cheap at this size
        int a = 0, b = 0;
        for (int e = 0; e < E; ++e) {
            const int n = s_n[e], t = s_t[e];
            s_n[e] = a;
            s_t[e] = b;
            a += n;
            b += t;
        }
        s_tot[0] = a;
        s_tot[1] = b;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int first = s_n[e];
        const int next = (e + 1 < E) ? s_n[e + 1] : s_tot[0];
        if (next == first) continue;
        const int idx = s_t[e];
        ws.rg_expert[idx] = e;
        ws.rg_first[idx] = first;
        int w = first;
        for (int s = 0; s < nslots; ++s)
            if (s_se[s] == e) ws.rg_slot[w++] = s;
    }
    if (threadIdx.x == 0) {
        ws.rg_first[s_tot[1]] = s_tot[0];
        *ws.rg_count = s_tot[1];
    }
}

// g_home[e] += red[slot] for its slots in order (fp32 adds), then the slots are zeroed.
// Work items are (touched expert, 32 KB tile of its gradient), strided over a
// persistent grid. Each thread owns kRedU float4 of the tile: it issues all of
// their gradient loads, then, slot by slot in ascending order, all of that
// slot's loads, before any add, so kRedU independent 16-byte loads are in
// flight per operand.
constexpr int kRedU = 8;

__global__ void __launch_bounds__(kThreads) reduce_grad_kernel(float4* __restrict__ g_home,
                                                               float4* __restrict__ red, int64_t nvec,
                                                               Workspace ws) {
    const int count = *ws.rg_count;
    const int64_t tile_vec = (int64_t)kThreads * kRedU;
    const int64_t ntile = (nvec + tile_vec - 1) / tile_vec;
    const int64_t nitems = (int64_t)count * ntile;
    for (int64_t item = blockIdx.x; item < nitems; item += gridDim.x) {
        const int it = (int)(item / ntile);
        const int64_t base = (item - (int64_t)it * ntile) * tile_vec + threadIdx.x;
        const int e = ws.rg_expert[it];
        const int s0 = ws.rg_first[it], s1 = ws.rg_first[it + 1];
        float4* g = g_home + (int64_t)e * nvec;
        float4 acc[kRedU];
#pragma unroll
        for (int u = 0; u < kRedU; ++u) {
            const int64_t i = base + (int64_t)u * kThreads;
            if (i < nvec) acc[u] = g[i];
        }
        for (int s = s0; s < s1; ++s) {
            float4* r = red + (int64_t)ws.rg_slot[s] * nvec;
            float4 v[kRedU];
#pragma unroll
            for (int u = 0; u < kRedU; ++u) {
                const int64_t i = base + (int64_t)u * kThreads;
                if (i < nvec) v[u] = r[i];
            }
#pragma unroll
            for (int u = 0; u < kRedU; ++u) {
                const int64_t i = base + (int64_t)u * kThreads;
                if (i >= nvec) continue;
                acc[u].x = __fadd_rn(acc[u].x, v[u].x);
                acc[u].y = __fadd_rn(acc[u].y, v[u].y);
                acc[u].z = __fadd_rn(acc[u].z, v[u].z);
                acc[u].w = __fadd_rn(acc[u].w, v[u].w);
                r[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < kRedU; ++u) {
            const int64_t i = base + (int64_t)u * kThreads;
            if (i < nvec) g[i] = acc[u];
        }
    }
}

int grid_for(int64_t work_warps, int num_sms) {
    const int64_t per_cta = kThreads / 32;
    int64_t g = (work_warps + per_cta - 1) / per_cta;
    const int64_t cap = (int64_t)num_sms * kCtasPerSm;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

// Row pieces per token: every 32*U-vector step of a row is an item of its own when the
// grid has more warps than there are tokens and rows are at least 4 steps long
// (4,096 tokens of 7168 bf16: dispatch 0.101 -> 0.091 ms, dispatch backward 0.105 ->
// 0.091 ms on one GB300); otherwise 1 (at 2 steps per row, pieces measured no better).
template <int U>
int pieces_for(int64_t ntok, int nvec, int num_sms) {
    const int64_t warps = (int64_t)num_sms * kCtasPerSm * (kThreads / 32);
    const int steps = (nvec + 32 * U - 1) / (32 * U);
    return (ntok < warps && steps >= 4) ? steps : 1;
}

}  // namespace

cudaError_t launch_dispatch(const Dims& d, const Workspace& ws, const uint16_t* x,
                            const int32_t* dest, uint16_t* recv, int num_sms, cudaStream_t st) {
    const int64_t ntok = (int64_t)d.R * d.S;
    if (ntok == 0) return cudaSuccess;
    const int pieces = pieces_for<4>(ntok, d.H / 8, num_sms);
    dispatch_kernel<4><<<grid_for(ntok * pieces, num_sms), kThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(x), dest, reinterpret_cast<uint4*>(recv), ntok, d.K,
        d.H / 8, (int64_t)d.R * d.C, pieces, ws.status);
    return cudaGetLastError();
}

cudaError_t launch_combine(const Dims& d, const Workspace& ws, const uint16_t* y,
                           const int32_t* dest, const float* gates, int D, uint16_t* out,
                           int num_sms, cudaStream_t st) {
    const int64_t ntok = (int64_t)d.R * d.S;
    if (ntok == 0) return cudaSuccess;
    // whole rows per warp: at 4,096 tokens and D = 2048, two pieces per row measured 7%
    // slower than one (each piece reloads the token's K destinations and gates)
    combine_kernel<4, true, false><<<grid_for(ntok, num_sms), kThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(y), dest, gates, reinterpret_cast<uint4*>(out), ntok, d.K,
        D / 8, (int64_t)d.R * d.C, 1, ws.status);
    return cudaGetLastError();
}

cudaError_t launch_combine_dgates(const Dims& d, const Workspace& ws, const uint16_t* dout,
                                  const uint16_t* y, const int32_t* dest, int D, float* dg,
                                  int num_sms, cudaStream_t st) {
    const int64_t ntok = (int64_t)d.R * d.S;
    if (ntok == 0) return cudaSuccess;
    combine_dgates_kernel<<<grid_for(ntok, num_sms), kThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(dout), reinterpret_cast<const uint4*>(y), dest, dg, ntok, d.K,
        D / 8, (int64_t)d.R * d.C, ws.status);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_bwd(const Dims& d, const Workspace& ws, const uint16_t* drecv,
                                const int32_t* dest, uint16_t* dx, int num_sms, cudaStream_t st) {
    const int64_t ntok = (int64_t)d.R * d.S;
    if (ntok == 0) return cudaSuccess;
    const int pieces = pieces_for<4>(ntok, d.H / 8, num_sms);
    if (pieces > 1)
        combine_kernel<4, false, true><<<grid_for(ntok * pieces, num_sms), kThreads, 0, st>>>(
            reinterpret_cast<const uint4*>(drecv), dest, nullptr, reinterpret_cast<uint4*>(dx), ntok,
            d.K, d.H / 8, (int64_t)d.R * d.C, pieces, ws.status);
    else
        combine_kernel<4, false, false><<<grid_for(ntok, num_sms), kThreads, 0, st>>>(
            reinterpret_cast<const uint4*>(drecv), dest, nullptr, reinterpret_cast<uint4*>(dx), ntok,
            d.K, d.H / 8, (int64_t)d.R * d.C, 1, ws.status);
    return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const Dims& d, const Workspace& ws, const uint16_t* dout,
                               const int32_t* dest, const float* gates, int D, uint16_t* dy,
                               int num_sms, cudaStream_t st) {
    const int64_t ntok = (int64_t)d.R * d.S;
    if (ntok == 0) return cudaSuccess;
    const int pieces = pieces_for<4>(ntok, D / 8, num_sms);
    const int64_t warps = (int64_t)num_sms * kCtasPerSm * (kThreads / 32);
    if (pieces > 1 || ntok >= warps)
        combine_bwd_kernel<4, true><<<grid_for(ntok * pieces, num_sms), kThreads, 0, st>>>(
            reinterpret_cast<const uint4*>(dout), dest, gates, reinterpret_cast<uint4*>(dy), ntok,
            d.K, D / 8, (int64_t)d.R * d.C, pieces, ws.status);
    else
        combine_bwd_kernel<4, false><<<grid_for(ntok, num_sms), kThreads, 0, st>>>(
            reinterpret_cast<const uint4*>(dout), dest, gates, reinterpret_cast<uint4*>(dy), ntok,
            d.K, D / 8, (int64_t)d.R * d.C, 1, ws.status);
    return cudaGetLastError();
}

cudaError_t launch_prefetch(const Dims& d, const Workspace& ws, const int32_t* slot_expert,
                            const uint16_t* w_home, uint16_t* w_slots, int num_sms,
                            cudaStream_t st) {
    if (d.R * d.B == 0) return cudaSuccess;
    const int64_t nvec = (int64_t)d.H * d.Hp / 8;
    prefetch_kernel<<<num_sms * kCtasPerSm / 2, kThreads, 0, st>>>(
        slot_expert, reinterpret_cast<const uint4*>(w_home), reinterpret_cast<uint4*>(w_slots),
        d.R * d.B, d.E, nvec, ws.status);
    return cudaGetLastError();
}

cudaError_t launch_reduce_grad(const Dims& d, const Workspace& ws, const int32_t* slot_expert,
                               float* g_home, float* red, int num_sms, cudaStream_t st) {
    const int nslots = d.R * d.B;
    if (nslots == 0) return cudaSuccess;
    reduce_grad_prep_kernel<<<1, 1024, (nslots + 2 * d.E) * 4, st>>>(slot_expert, nslots, d.E, ws);
    const int64_t nvec = (int64_t)d.H * d.Hp / 4;
    reduce_grad_kernel<<<num_sms * 4, kThreads, 0, st>>>(
        reinterpret_cast<float4*>(g_home), reinterpret_cast<float4*>(red), nvec, ws);
    return cudaGetLastError();
}

}  // namespace bep
