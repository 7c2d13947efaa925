// C ABI of libbep.so (declared in include/bep.h): argument checks, the
// context's workspace, and launches on the caller's stream.

#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

#include "bep_internal.cuh"

namespace {
// One NVTX range per call of a compute entry point, named after the call, so the
// kernels it queues show under that name in nsys / ncu --nvtx. Header-only NVTX:
// without an attached tool a range costs a pointer check.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace
#define BEP_RANGE(name) const NvtxRange bep_nvtx_range_(name)

struct bep_ctx {
    bep::Dims d;
    bep::Workspace ws;
    void* blob;
    int device;
    int num_sms;
    int comm_sms;   // SM budget of the token-moving kernels (0: every SM)
};

namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

int bep::make_dims(const bep_config* c, bep::Dims* d) {
    if (c->R < 1 || c->E < 1 || c->K < 1 || c->S < 0 || c->B < 0 || c->H < 1 || c->Hp < 1)
        return BEP_ERR_ARG;
    if (c->mode != BEP_TRAIN && c->mode != BEP_INFER) return BEP_ERR_ARG;
    if (c->R > bep::kMaxR || c->E > bep::kMaxE || c->K > bep::kMaxK || c->K > c->E)
        return BEP_ERR_SIZE;
    if (c->E % c->R != 0) return BEP_ERR_SIZE;
    if (c->H % 64 != 0 || c->Hp % 64 != 0) return BEP_ERR_SIZE;
    const int G = c->E / c->R;
    if (c->mode == BEP_TRAIN && c->B != G) return BEP_ERR_MODE;
    if (c->mode == BEP_INFER && !(c->B >= 1 && c->B < G)) return BEP_ERR_MODE;
    const int64_t rsk = (int64_t)c->R * c->S * c->K;
    if (rsk >= ((int64_t)1 << 31)) return BEP_ERR_SIZE;
    d->R = c->R;
    d->E = c->E;
    d->B = c->B;
    d->K = c->K;
    d->S = c->S;
    d->H = c->H;
    d->Hp = c->Hp;
    d->mode = c->mode;
    d->G = G;
    d->C = (int64_t)c->S * c->K;
    d->NCH = (c->S + bep::kChunkTokens - 1) / bep::kChunkTokens;
    d->NC = c->R * d->NCH;
    d->NROW = c->E + c->B;
    d->max_tiles = (int)(rsk / bep::kBM + (int64_t)c->R * d->NROW + 1);
    return BEP_OK;
}

namespace {

template <typename T>
T* carve(char*& p, size_t n) {
    T* out = reinterpret_cast<T*>(p);
    size_t bytes = (n * sizeof(T) + 255) & ~(size_t)255;
    p += bytes;
    return out;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? BEP_OK : BEP_ERR_CUDA; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// SMs that dispatch, combine and their backward kernels size their grids for.
int comm_sms(const bep_ctx* ctx) {
    return (ctx->comm_sms > 0 && ctx->comm_sms < ctx->num_sms) ? ctx->comm_sms : ctx->num_sms;
}

}  // namespace

extern "C" {

int bep_create(const bep_config* cfg, bep_ctx** out) {
    if (!cfg || !out) return BEP_ERR_ARG;
    *out = nullptr;
    bep::Dims d;
    int rc = bep::make_dims(cfg, &d);
    if (rc) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BEP_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BEP_ERR_CUDA;
    if (bep::plan_setup(dev) != cudaSuccess || bep::gemm_setup(dev) != cudaSuccess)
        return BEP_ERR_CUDA;

    const size_t E = d.E, R = d.R, NC = d.NC, NROW = d.NROW, NP = d.E + d.R;
    const size_t nslots = (size_t)d.R * d.B;
    size_t bytes = 0;
    auto add = [&](size_t n, size_t sz) { bytes += (n * sz + 255) & ~(size_t)255; };
    add(1, 4);                      // status
    add(1, 4);                      // plan_err
    add(E * (NC > 0 ? NC : 1), 4);  // off
    add(E, 4);                      // T
    add(R * NROW, 4);               // lens
    add(E + 1, 4);                  // pfirst
    for (int i = 0; i < 5; ++i) add(NP, 4);
    add((size_t)d.max_tiles, sizeof(bep::MTile));
    add(1, 4);                      // ntiles
    add(nslots + 1, 4);             // rg_expert
    add(nslots + 1, 4);             // rg_first
    add(nslots + 1, 4);             // rg_slot
    add(1, 4);                      // rg_count
    void* blob = nullptr;
    if (cudaMalloc(&blob, bytes) != cudaSuccess) return BEP_ERR_CUDA;
    if (cudaMemset(blob, 0, bytes) != cudaSuccess) {
        cudaFree(blob);
        return BEP_ERR_CUDA;
    }
    char* p = static_cast<char*>(blob);
    bep::Workspace ws;
    ws.status = carve<int32_t>(p, 1);
    ws.plan_err = carve<int32_t>(p, 1);
    ws.off = carve<int32_t>(p, E * (NC > 0 ? NC : 1));
    ws.T = carve<int32_t>(p, E);
    ws.lens = carve<int32_t>(p, R * NROW);
    ws.pfirst = carve<int32_t>(p, E + 1);
    ws.pstart = carve<int32_t>(p, NP);
    ws.plen = carve<int32_t>(p, NP);
    ws.prank = carve<int32_t>(p, NP);
    ws.prow = carve<int32_t>(p, NP);
    ws.pbase = carve<int32_t>(p, NP);
    ws.tiles = carve<bep::MTile>(p, (size_t)d.max_tiles);
    ws.ntiles = carve<int32_t>(p, 1);
    ws.rg_expert = carve<int32_t>(p, nslots + 1);
    ws.rg_first = carve<int32_t>(p, nslots + 1);
    ws.rg_slot = carve<int32_t>(p, nslots + 1);
    ws.rg_count = carve<int32_t>(p, 1);

    bep_ctx* ctx = static_cast<bep_ctx*>(malloc(sizeof(bep_ctx)));
    if (!ctx) {
        cudaFree(blob);
        return BEP_ERR_ARG;
    }
    ctx->d = d;
    ctx->ws = ws;
    ctx->blob = blob;
    ctx->device = dev;
    ctx->num_sms = sms;
    ctx->comm_sms = 0;
    *out = ctx;
    return BEP_OK;
}

void bep_destroy(bep_ctx* ctx) {
    if (!ctx) return;
    cudaFree(ctx->blob);
    free(ctx);
}

int bep_plan(bep_ctx* ctx, const int32_t* topk, int32_t* cu_seqlens, int32_t* slot_expert,
             int32_t* dest, double* maxvio, void* stream) {
    BEP_RANGE("bep_plan");
    if (!ctx || !cu_seqlens || !maxvio || (ctx->d.R * ctx->d.B > 0 && !slot_expert))
        return BEP_ERR_ARG;
    if (ctx->d.C > 0 && (!topk || !dest)) return BEP_ERR_ARG;
    if (!aligned(topk, 4) || !aligned(cu_seqlens, 4) || !aligned(slot_expert, 4) ||
        !aligned(dest, 4) || !aligned(maxvio, 8))
        return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_plan(ctx->d, ctx->ws, topk, cu_seqlens, slot_expert, dest, maxvio,
                                    as_stream(stream)));
}

int bep_prefetch_weight(bep_ctx* ctx, const int32_t* slot_expert, const uint16_t* w_home,
                        uint16_t* w_slots, void* stream) {
    BEP_RANGE("bep_prefetch_weight");
    if (!ctx) return BEP_ERR_ARG;
    if (ctx->d.R * ctx->d.B == 0) return BEP_OK;
    if (!slot_expert || !w_home || !w_slots) return BEP_ERR_ARG;
    if (!aligned(slot_expert, 4) || !aligned(w_home, 16) || !aligned(w_slots, 16))
        return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_prefetch(ctx->d, ctx->ws, slot_expert, w_home, w_slots,
                                        ctx->num_sms, as_stream(stream)));
}

int bep_dispatch(bep_ctx* ctx, const uint16_t* x, const int32_t* dest, uint16_t* recv,
                 void* stream) {
    BEP_RANGE("bep_dispatch");
    if (!ctx) return BEP_ERR_ARG;
    if (ctx->d.C == 0) return BEP_OK;
    if (!x || !dest || !recv) return BEP_ERR_ARG;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(dest, 4)) return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_dispatch(ctx->d, ctx->ws, x, dest, recv, comm_sms(ctx),
                                        as_stream(stream)));
}

int bep_grouped_gemm(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* recv,
                     const uint16_t* w_home, const uint16_t* w_slots, uint16_t* y, void* stream) {
    BEP_RANGE("bep_grouped_gemm");
    if (!ctx) return BEP_ERR_ARG;
    if (ctx->d.C == 0) return BEP_OK;
    if (!cu_seqlens || !recv || !w_home || !y) return BEP_ERR_ARG;
    if (ctx->d.R * ctx->d.B > 0 && !w_slots) return BEP_ERR_ARG;
    if (!aligned(cu_seqlens, 4) || !aligned(recv, 16) || !aligned(w_home, 16) ||
        !aligned(w_slots, 16) || !aligned(y, 16))
        return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_grouped_gemm(ctx->d, ctx->ws, cu_seqlens, recv, w_home, w_slots,
                                            y, ctx->num_sms, as_stream(stream)));
}

int bep_grouped_gemm_vm(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* recv,
                        const uint16_t* w_views, uint16_t* y, void* stream) {
    BEP_RANGE("bep_grouped_gemm_vm");
    if (!ctx) return BEP_ERR_ARG;
    if (ctx->d.C == 0) return BEP_OK;
    if (!cu_seqlens || !recv || !w_views || !y) return BEP_ERR_ARG;
    if (!aligned(cu_seqlens, 4) || !aligned(recv, 16) || !aligned(w_views, 16) || !aligned(y, 16))
        return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_grouped_gemm_vm(ctx->d, ctx->ws, cu_seqlens, recv, w_views, y,
                                               ctx->num_sms, as_stream(stream)));
}

int bep_combine(bep_ctx* ctx, const uint16_t* y, const int32_t* dest, const float* gates,
                int32_t D, uint16_t* out, void* stream) {
    BEP_RANGE("bep_combine");
    if (!ctx || D < 8 || D % 8 != 0) return BEP_ERR_ARG;
    if (ctx->d.C == 0) return BEP_OK;
    if (!y || !dest || !gates || !out) return BEP_ERR_ARG;
    if (!aligned(y, 16) || !aligned(out, 16) || !aligned(dest, 4) || !aligned(gates, 4))
        return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_combine(ctx->d, ctx->ws, y, dest, gates, D, out, comm_sms(ctx),
                                       as_stream(stream)));
}

int bep_combine_bwd(bep_ctx* ctx, const uint16_t* dout, const int32_t* dest, const float* gates,
                    int32_t D, uint16_t* dy, void* stream) {
    BEP_RANGE("bep_combine_bwd");
    if (!ctx || D < 8 || D % 8 != 0) return BEP_ERR_ARG;
    if (ctx->d.C == 0) return BEP_OK;
    if (!dout || !dest || !gates || !dy) return BEP_ERR_ARG;
    if (!aligned(dout, 16) || !aligned(dy, 16) || !aligned(dest, 4) || !aligned(gates, 4))
        return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_combine_bwd(ctx->d, ctx->ws, dout, dest, gates, D, dy,
                                           comm_sms(ctx), as_stream(stream)));
}

int bep_dispatch_bwd(bep_ctx* ctx, const uint16_t* drecv, const int32_t* dest, uint16_t* dx,
                     void* stream) {
    BEP_RANGE("bep_dispatch_bwd");
    if (!ctx) return BEP_ERR_ARG;
    if (ctx->d.C == 0) return BEP_OK;
    if (!drecv || !dest || !dx) return BEP_ERR_ARG;
    if (!aligned(drecv, 16) || !aligned(dx, 16) || !aligned(dest, 4)) return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_dispatch_bwd(ctx->d, ctx->ws, drecv, dest, dx, comm_sms(ctx),
                                            as_stream(stream)));
}

int bep_grouped_gemm_dx(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* dy,
                        const uint16_t* w_home, const uint16_t* w_slots, uint16_t* drecv,
                        void* stream) {
    BEP_RANGE("bep_grouped_gemm_dx");
    if (!ctx) return BEP_ERR_ARG;
    if (ctx->d.C == 0) return BEP_OK;
    if (!cu_seqlens || !dy || !w_home || !drecv) return BEP_ERR_ARG;
    if (ctx->d.R * ctx->d.B > 0 && !w_slots) return BEP_ERR_ARG;
    if (!aligned(cu_seqlens, 4) || !aligned(dy, 16) || !aligned(w_home, 16) ||
        !aligned(w_slots, 16) || !aligned(drecv, 16))
        return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_grouped_gemm_dx(ctx->d, ctx->ws, cu_seqlens, dy, w_home, w_slots,
                                               drecv, ctx->num_sms, as_stream(stream)));
}

static int grouped_gemm_dw(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* recv,
                           const uint16_t* dy, float* g_home, float* red, int accumulate,
                           void* stream) {
    if (!ctx) return BEP_ERR_ARG;
    if (ctx->d.mode != BEP_TRAIN) return BEP_ERR_MODE;
    if (ctx->d.H % bep::kBM != 0) return BEP_ERR_SIZE;
    if (ctx->d.C == 0 && accumulate) return BEP_OK;
    if (ctx->d.C == 0) {   // nothing to multiply: the overwrite zeroes the home rows
        if (!g_home) return BEP_ERR_ARG;
        if (!aligned(g_home, 16)) return BEP_ERR_ALIGN;
    } else {
        if (!cu_seqlens || !recv || !dy || !g_home || !red) return BEP_ERR_ARG;
        if (!aligned(cu_seqlens, 4) || !aligned(recv, 16) || !aligned(dy, 16) ||
            !aligned(g_home, 16) || !aligned(red, 16))
            return BEP_ERR_ALIGN;
    }
    return cuda_rc(bep::launch_grouped_gemm_dw(ctx->d, ctx->ws, cu_seqlens, recv, dy, g_home, red,
                                               accumulate, ctx->num_sms, as_stream(stream)));
}

int bep_grouped_gemm_dw(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* recv,
                        const uint16_t* dy, float* g_home, float* red, void* stream) {
    BEP_RANGE("bep_grouped_gemm_dw");
    return grouped_gemm_dw(ctx, cu_seqlens, recv, dy, g_home, red, 1, stream);
}

int bep_grouped_gemm_dw_overwrite(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* recv,
                                  const uint16_t* dy, float* g_home, float* red, void* stream) {
    BEP_RANGE("bep_grouped_gemm_dw_overwrite");
    return grouped_gemm_dw(ctx, cu_seqlens, recv, dy, g_home, red, 0, stream);
}

int bep_reduce_grad(bep_ctx* ctx, const int32_t* slot_expert, float* g_home, float* red,
                    void* stream) {
    BEP_RANGE("bep_reduce_grad");
    if (!ctx) return BEP_ERR_ARG;
    if (ctx->d.R * ctx->d.B == 0) return BEP_OK;
    if (!slot_expert || !g_home || !red) return BEP_ERR_ARG;
    if (!aligned(slot_expert, 4) || !aligned(g_home, 16) || !aligned(red, 16))
        return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_reduce_grad(ctx->d, ctx->ws, slot_expert, g_home, red,
                                           ctx->num_sms, as_stream(stream)));
}

int bep_combine_dgates(bep_ctx* ctx, const uint16_t* dout, const uint16_t* y, const int32_t* dest,
                       int32_t D, float* dgates, void* stream) {
    BEP_RANGE("bep_combine_dgates");
    if (!ctx || D < 8 || D % 8 != 0) return BEP_ERR_ARG;
    if (ctx->d.C == 0) return BEP_OK;
    if (!dout || !y || !dest || !dgates) return BEP_ERR_ARG;
    if (!aligned(dout, 16) || !aligned(y, 16) || !aligned(dest, 4) || !aligned(dgates, 4))
        return BEP_ERR_ALIGN;
    return cuda_rc(bep::launch_combine_dgates(ctx->d, ctx->ws, dout, y, dest, D, dgates,
                                              comm_sms(ctx), as_stream(stream)));
}

int bep_wait_selftest(bep_ctx* ctx, int32_t timeout_us, void* stream) {
    if (!ctx || timeout_us < 1 || timeout_us > 10000000) return BEP_ERR_ARG;
    return cuda_rc(bep::launch_wait_selftest(ctx->ws, (uint64_t)timeout_us * 1000ull,
                                             as_stream(stream)));
}

int bep_set_comm_sms(bep_ctx* ctx, int32_t sms) {
    if (!ctx || sms < 0) return BEP_ERR_ARG;
    ctx->comm_sms = sms;
    return BEP_OK;
}

int bep_status(bep_ctx* ctx, int32_t* device_err, void* stream) {
    if (!ctx || !device_err) return BEP_ERR_ARG;
    int32_t h = 0;
    cudaStream_t st = as_stream(stream);
    if (cudaMemcpyAsync(&h, ctx->ws.status, sizeof(int32_t), cudaMemcpyDeviceToHost, st) !=
        cudaSuccess)
        return BEP_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return BEP_ERR_CUDA;
    *device_err = h;
    return BEP_OK;
}

int bep_clear_status(bep_ctx* ctx, void* stream) {
    if (!ctx) return BEP_ERR_ARG;
    return cuda_rc(cudaMemsetAsync(ctx->ws.status, 0, sizeof(int32_t), as_stream(stream)));
}

const char* bep_strerror(int32_t code) {
    switch (code) {
        case BEP_OK: return "ok";
        case BEP_ERR_ARG: return "invalid argument";
        case BEP_ERR_ALIGN: return "misaligned pointer";
        case BEP_ERR_MODE: return "B inconsistent with mode (TRAIN: B == E/R; INFER: 1 <= B < E/R)";
        case BEP_ERR_SIZE: return "size outside the supported limits";
        case BEP_ERR_CUDA: return "CUDA runtime error";
        case BEP_DERR_EXPERT_ID: return "device: expert id out of range";
        case BEP_DERR_DUP_ID: return "device: duplicate expert id in one token";
        case BEP_DERR_INFEASIBLE: return "device: plan does not give every rank S*K slots";
        case BEP_DERR_BOUNDS: return "device: index out of range";
        case BEP_DERR_TIMEOUT: return "device: bounded wait timed out";
        default: return code > 0 ? "device: several error bits" : "unknown error";
    }
}

}  // extern "C"
