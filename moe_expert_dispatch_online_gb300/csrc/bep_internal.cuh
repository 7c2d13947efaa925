// Internal declarations shared by the translation units of libbep.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bep.h"

namespace bep {

constexpr int kChunkTokens = 256;   // planner chunk: tokens of one rank, never spanning ranks
constexpr int kMaxE = 2048;
constexpr int kMaxR = 64;
constexpr int kMaxK = 32;

// GEMM tiling (tcgen05, one CTA per tile, M = 128 rows of recv)
constexpr int kBM = 128;
constexpr int kBK = 64;

// One GEMM m-tile: 128 (or fewer, at a segment's end) receive rows that share a weight row.
struct MTile {
    int32_t row0;    // first global receive row
    int32_t rows;    // valid rows, 1..128
    int32_t wsel;    // >= 0: home row index into w_home; < 0: -(1 + u*B + j), slot of w_slots
    int32_t pad;
};

struct Workspace {
    int32_t* status;     // [1] sticky device error bits (bep_status)
    int32_t* plan_err;   // [1] error bits of the current bep_plan call only
    int32_t* off;        // [E][NC]: chunk counts, then exclusive offsets along chunks
    int32_t* T;          // [E]
    int32_t* lens;       // [R][E+B] segment lengths
    int32_t* pfirst;     // [E+1] first piece of each expert
    int32_t* pstart;     // [E+R] piece: first position inside the expert's (r,t)-ordered list
    int32_t* plen;       // [E+R]
    int32_t* prank;      // [E+R]
    int32_t* prow;       // [E+R]
    int32_t* pbase;      // [E+R] dest = pbase + position
    MTile* tiles;        // [max_tiles]
    int32_t* ntiles;     // [1]
    int32_t* rg_expert;  // [R*B] reduce_grad: home experts with replicas, ascending
    int32_t* rg_first;   // [R*B+1] first entry of each in rg_slot
    int32_t* rg_slot;    // [R*B] flat slot indices u*B + j, ascending per expert
    int32_t* rg_count;   // [1] number of such experts
};

struct Dims {
    int R, E, B, K, S, H, Hp, mode;
    int G;          // E / R
    int64_t C;      // S*K slots per rank
    int NCH;        // chunks per rank
    int NC;         // chunks in total
    int NROW;       // E + B
    int max_tiles;  // GEMM m-tiles upper bound
};

// configuration checks shared by the entry points (bep.cu)
int make_dims(const bep_config* c, Dims* d);

// planner (plan.cu)
cudaError_t plan_setup(int device);
cudaError_t launch_plan(const Dims& d, const Workspace& ws, const int32_t* topk, int32_t* cu,
                        int32_t* slot_expert, int32_t* dest, double* maxvio, cudaStream_t st);
// data movement (move.cu)
cudaError_t launch_prefetch(const Dims& d, const Workspace& ws, const int32_t* slot_expert,
                            const uint16_t* w_home, uint16_t* w_slots, int num_sms,
                            cudaStream_t st);
cudaError_t launch_dispatch(const Dims& d, const Workspace& ws, const uint16_t* x,
                            const int32_t* dest, uint16_t* recv, int num_sms, cudaStream_t st);
cudaError_t launch_combine(const Dims& d, const Workspace& ws, const uint16_t* y,
                           const int32_t* dest, const float* gates, int D, uint16_t* out,
                           int num_sms, cudaStream_t st);
cudaError_t launch_combine_bwd(const Dims& d, const Workspace& ws, const uint16_t* dout,
                               const int32_t* dest, const float* gates, int D, uint16_t* dy,
                               int num_sms, cudaStream_t st);
cudaError_t launch_combine_dgates(const Dims& d, const Workspace& ws, const uint16_t* dout,
                                  const uint16_t* y, const int32_t* dest, int D, float* dg,
                                  int num_sms, cudaStream_t st);
cudaError_t launch_dispatch_bwd(const Dims& d, const Workspace& ws, const uint16_t* drecv,
                                const int32_t* dest, uint16_t* dx, int num_sms, cudaStream_t st);
cudaError_t launch_reduce_grad(const Dims& d, const Workspace& ws, const int32_t* slot_expert,
                               float* g_home, float* red, int num_sms, cudaStream_t st);
// grouped GEMM (gemm.cu)
cudaError_t gemm_setup(int device);
cudaError_t launch_wait_selftest(const Workspace& ws, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_grouped_gemm(const Dims& d, const Workspace& ws, const int32_t* cu,
                                const uint16_t* recv, const uint16_t* w_home,
                                const uint16_t* w_slots, uint16_t* y, int num_sms,
                                cudaStream_t st);
cudaError_t launch_grouped_gemm_vm(const Dims& d, const Workspace& ws, const int32_t* cu,
                                   const uint16_t* recv, const uint16_t* w_views, uint16_t* y,
                                   int num_sms, cudaStream_t st);
cudaError_t launch_grouped_gemm_dx(const Dims& d, const Workspace& ws, const int32_t* cu,
                                   const uint16_t* dy, const uint16_t* w_home,
                                   const uint16_t* w_slots, uint16_t* drecv, int num_sms,
                                   cudaStream_t st);
cudaError_t launch_grouped_gemm_dw(const Dims& d, const Workspace& ws, const int32_t* cu,
                                   const uint16_t* recv, const uint16_t* dy, float* g_home,
                                   float* red, int accumulate, int num_sms, cudaStream_t st);

__device__ __forceinline__ int64_t i64max(int64_t a, int64_t b) { return a > b ? a : b; }
__device__ __forceinline__ int64_t i64min(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ void set_status(int32_t* status, int bits) {
    atomicOr(status, bits);
}

}  // namespace bep
