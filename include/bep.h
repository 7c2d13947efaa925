/*
 * bep.h -- balanced expert-parallel dispatch for one GB300 (sm_103a).
 *
 * C ABI of libbep.so. The hot path of MoonEP-style perfectly balanced expert
 * parallelism: an online planner, a fused permute/dispatch, a grouped expert
 * GEMM over one [E+B, H, H'] weight tensor addressed by row index, a weighted
 * combine, and the backward fold (combine backward, reduce_grad).
 *
 * Sources (page title / host, then section):
 *   [P1] "Moonshot AI libera MoonEP ..." (noticiai.com.br)
 *   [P2] "Moonshot AI Open-Sources MoonEP: A Perfectly Balanced Expert
 *        Parallelism Library for MoE Training" (spaxe.top)
 *   [P4] "Moonshot AI open-sources MoonEP" (ai-maestro.online): "The problem
 *        MoonEP targets", "The core idea: dynamic redundant experts",
 *        "The memory contract".
 *
 * The R ranks are virtual: R partitions of this GPU's HBM. A "remote" write
 * in the pages is an ordinary global store here.
 *
 * Conventions for every call below.
 *   - Device pointers are caller-owned (the library never frees them), must
 *     be 16-byte aligned, and must stay valid until the work queued on
 *     `stream` has finished. Arrays are dense and row-major in the shapes
 *     given. bf16 tensors are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All calls except bep_create/bep_destroy/bep_status are
 *     asynchronous: nothing synchronises with the host, so a whole step can
 *     be captured in a CUDA graph.
 *   - Return value: BEP_OK, or a negative BEP_ERR_* detected on the host
 *     before anything is queued (the call then has no effect).
 *   - Errors found on the device (bad expert ids, bounds, a plan that does
 *     not balance, a timed-out wait) are OR-ed into the context's status
 *     word; kernels that would read invalid indices skip the bad element.
 *     bep_status() reads and reports the word.
 *   - The context owns only its planning/scheduling workspace, allocated
 *     once in bep_create (static shapes: no allocation afterwards). Calls
 *     sharing one context must be ordered on one stream.
 */
#ifndef BEP_H_
#define BEP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* host-side return codes */
#define BEP_OK          0
#define BEP_ERR_ARG    -1   /* null pointer, bad dimension or mode value        */
#define BEP_ERR_ALIGN  -2   /* a pointer is not 16-byte aligned                 */
#define BEP_ERR_MODE   -3   /* TRAIN needs B == E/R; INFER needs 1 <= B < E/R   */
#define BEP_ERR_SIZE   -4   /* E % R != 0, R*S*K >= 2^31, or a size limit below */
#define BEP_ERR_CUDA   -5   /* a CUDA runtime call failed (no device, OOM, ...) */

/* device status word bits (bep_status) */
#define BEP_DERR_EXPERT_ID   1   /* a top-K id outside [0, E)                     */
#define BEP_DERR_DUP_ID      2   /* one token names the same expert twice         */
#define BEP_DERR_INFEASIBLE  4   /* a rank did not end with exactly S*K slots     */
#define BEP_DERR_BOUNDS      8   /* a dest / cu_seqlens / slot entry out of range */
#define BEP_DERR_TIMEOUT    16   /* a bounded device wait gave up                 */

/* modes ([P4] "The memory contract": how to set B) */
#define BEP_TRAIN 0   /* B == E/R: every expert the GEMM touches is local        */
#define BEP_INFER 1   /* B <  E/R: remote experts beyond B read from home rows   */

/* Size limits checked by bep_create: 1 <= R <= 64, 1 <= E <= 2048, E % R == 0,
 * 1 <= K <= 32, K <= E, S >= 0, R*S*K < 2^31, H % 64 == 0, H' % 64 == 0,
 * 64 <= H, 64 <= H'. */
typedef struct bep_config {
    int32_t R;     /* virtual ranks                                   */
    int32_t E;     /* routed experts; home group g owns [g*G, (g+1)*G), G = E/R */
    int32_t B;     /* prefetch slots per rank                         */
    int32_t K;     /* top-K experts per token                         */
    int32_t S;     /* tokens per rank                                 */
    int32_t H;     /* hidden size (GEMM reduction dim, dispatch row)  */
    int32_t Hp;    /* H', expert intermediate size (GEMM output dim)  */
    int32_t mode;  /* BEP_TRAIN or BEP_INFER                          */
} bep_config;

typedef struct bep_ctx bep_ctx;

/* Validates cfg, selects the current CUDA device, allocates the workspace
 * (plan tables, GEMM tile table, status word). *out receives the context.
 * Returns BEP_ERR_ARG/MODE/SIZE for a bad cfg (nothing allocated), or
 * BEP_ERR_CUDA. */
int bep_create(const bep_config* cfg, bep_ctx** out);

/* Frees the workspace. Waits for nothing: the caller synchronises first. */
void bep_destroy(bep_ctx* ctx);

/* The online planner ([P4] "The core idea": redundant experts planned on the
 * GPU from the current router output so that every rank receives exactly
 * S*K token-slots; "The problem MoonEP targets": maxvio).
 *   topk        [R, S, K] int32, expert ids of each token (rank-major tokens)
 *   cu_seqlens  [R, E+B+1] int32 out: per rank, offsets of the row segments
 *               0..E+B-1 inside that rank's S*K receive rows; cu[u][0] = 0,
 *               cu[u][E+B] = S*K. Rows [0,E) are home-expert rows, [E,E+B) are
 *               the rank's prefetch slots. (The pages' cu_seqlens[E+B] is the
 *               same data without the leading zero.)
 *   slot_expert [R, B] int32 out: expert held by each prefetch slot, -1 unused
 *   dest        [R, S, K] int32 out: flat row index into the [R*S*K] receive
 *               space for every (token, k); rank u owns rows [u*S*K, (u+1)*S*K)
 *   maxvio      [1] double out: max_e(T_e / Tbar) - 1, Tbar = R*S*K/E
 * Deterministic: the same topk always yields the same outputs. */
int bep_plan(bep_ctx* ctx, const int32_t* topk, int32_t* cu_seqlens, int32_t* slot_expert,
             int32_t* dest, double* maxvio, void* stream);

/* bep_plan without a context and without any allocation. The pages have no
 * counterpart: this is an addition for callers that cannot call cudaMalloc
 * when they plan -- services whose device memory is handed out once at
 * start-up and may not grow afterwards, and embedders (plug-ins inside a host
 * framework that owns the allocator, or code that cannot create and keep a
 * bep_ctx between calls).
 *   cfg, topk, cu_seqlens, slot_expert, dest, maxvio: as for bep_plan.
 *   device_err [1] int32, device memory (caller-owned): cleared, then receives
 *               this call's BEP_DERR_* bits (what bep_status reports for a
 *               context).
 * The planner's scratch tables live in a 2 MiB file-scope device array that
 * every GPU loading the library reserves until the process exits; a
 * configuration needing more than 2 MiB (about E * R * ceil(S/256) * 4 bytes
 * plus small tables: the S=8192, E=384, R=8 workload needs 0.4 MiB, and
 * S=43008 is the largest S that fits at R=8, E=384, B=48) returns
 * BEP_ERR_SIZE before anything is queued. No cudaMalloc, cudaFree or
 * allocating library routine is called. The first call in a CUDA context
 * looks up the array's device address and sets kernel attributes, so make
 * that first call before any stream capture; the lookup is repeated for a new
 * context (after a device reset, say). All calls share the array: calls whose
 * work overlaps on the GPU race, so the caller serialises them (one stream). */
int bep_plan_noalloc(const bep_config* cfg, const int32_t* topk, int32_t* cu_seqlens,
                     int32_t* slot_expert, int32_t* dest, double* maxvio, int32_t* device_err,
                     void* stream);

/* buffer.prefetch_weight ([P4] "The memory contract": rows [E, E+B) are local
 * prefetch slots): w_slots[u][j] = w_home[slot_expert[u][j]] for every used
 * slot; unused slots are left as they are.
 *   slot_expert [R, B] int32 (from bep_plan)
 *   w_home      [E, H, H'] bf16, the home rows [0, E)
 *   w_slots     [R, B, H, H'] bf16, every rank's slots */
int bep_prefetch_weight(bep_ctx* ctx, const int32_t* slot_expert, const uint16_t* w_home,
                        uint16_t* w_slots, void* stream);

/* Fused permute/dispatch ([P4] "The core idea", zero copy: tokens are written
 * directly into their expert-grouped positions): recv[dest[r,t,k], :] = x[r,t,:].
 *   x    [R, S, H] bf16
 *   dest [R, S, K] int32 (from bep_plan)
 *   recv [R*S*K, H] bf16 out, the static per-rank [S*K, H] buffers */
int bep_dispatch(bep_ctx* ctx, const uint16_t* x, const int32_t* dest, uint16_t* recv,
                 void* stream);

/* Grouped expert GEMM ([P4] "The memory contract": one [E+B, H, H'] weight
 * tensor addressed by row index, cu_seqlens selecting the active rows):
 * for rank u and row rho with a non-empty segment,
 *   y[u*S*K + seg, :] = recv[u*S*K + seg, :] @ W(u, rho),
 *   W(u, rho) = rho < E ? w_home[rho] : w_slots[u][rho - E]   ([H, H'] bf16),
 * bf16 inputs, fp32 accumulation, bf16 (round to nearest even) output.
 * Rows of y outside every segment are not written. A cu_seqlens table with any
 * segment outside [0, S*K] or ending before it starts is refused as a whole
 * (BEP_DERR_BOUNDS, nothing written); the same holds for the other GEMMs. */
int bep_grouped_gemm(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* recv,
                     const uint16_t* w_home, const uint16_t* w_slots, uint16_t* y,
                     void* stream);

/* The pages' "VM group GEMM" ([P4] "The memory contract": each rank's weights
 * are one contiguous [E+B, H, H'] tensor and the GEMM addresses experts by row
 * index only): the product of bep_grouped_gemm, with rank u's weight row rho
 * read from w_views[u][rho].
 *   w_views [R, E+B, H, H'] bf16: the R per-rank tensors back to back, e.g. the
 *           aliased views of bep_weights_create (no copy), or any buffer laid
 *           out that way. */
int bep_grouped_gemm_vm(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* recv,
                        const uint16_t* w_views, uint16_t* y, void* stream);

/* Weight store with the pages' memory contract ([P4] "The memory contract"):
 * per layer one physical block of home rows [E, H, H'], one slot pool
 * [R, B, H, H'] shared by every layer (the extra memory is B experts per
 * projection in total, not per layer), and per layer R views [E+B, H, H'],
 * back to back, in which rank u's rows [0, E) alias the layer's home rows and
 * rows [E, E+B) alias rank u's part of the pool (CUDA virtual memory
 * management; nothing is copied). E*H*H'*2 and B*H*H'*2 bytes must be
 * multiples of the mapping granularity (2 MiB), else BEP_ERR_SIZE. The store
 * allocates device memory; bep_weights_destroy frees it. */
typedef struct bep_weights bep_weights;
int bep_weights_create(const bep_config* cfg, int32_t layers, bep_weights** out);
/* Device pointers of layer `layer`: home [E, H, H'], the shared pool
 * [R, B, H, H'] (the w_slots of bep_prefetch_weight), views [R, E+B, H, H']
 * (the w_views of bep_grouped_gemm_vm). Any output pointer may be NULL. */
int bep_weights_get(bep_weights* w, int32_t layer, uint16_t** home, uint16_t** slots,
                    uint16_t** views);
void bep_weights_destroy(bep_weights* w);

/* Weighted unpermute/combine ([P4] "The core idea": fused permute/unpermute):
 *   out[r,t,c] = bf16_rne(acc), acc = 0; for k = 0..K-1:
 *                acc = fmaf(gates[r,t,k], float(y[dest[r,t,k], c]), acc)
 *   y [R*S*K, D] bf16; dest, gates [R, S, K] (int32, fp32); out [R, S, D] bf16.
 *   D % 8 == 0 (D = H' after the GEMM). */
int bep_combine(bep_ctx* ctx, const uint16_t* y, const int32_t* dest, const float* gates,
                int32_t D, uint16_t* out, void* stream);

/* Backward of the combine with respect to y:
 *   dy[dest[r,t,k], c] = bf16_rne(gates[r,t,k] * float(dout[r,t,c]))  (fp32 product)
 *   dout [R, S, D] bf16; dy [R*S*K, D] bf16 out. */
int bep_combine_bwd(bep_ctx* ctx, const uint16_t* dout, const int32_t* dest,
                    const float* gates, int32_t D, uint16_t* dy, void* stream);

/* Gradient of the combine with respect to the gates (the other half of the
 * combine's backward, [P4] "The core idea"):
 *   dgates[r,t,k] = sum_c float(dout[r,t,c]) * float(y[dest[r,t,k], c])   (fp32)
 *   dout [R, S, D] bf16; y [R*S*K, D] bf16 (the combine's input); dest [R, S, K];
 *   dgates [R, S, K] fp32 out. D % 8 == 0. The fp32 sum's order is the
 *   library's (per-lane partial sums, then a butterfly over 32 lanes). */
int bep_combine_dgates(bep_ctx* ctx, const uint16_t* dout, const uint16_t* y, const int32_t* dest,
                       int32_t D, float* dgates, void* stream);

/* Backward of the dispatch ([P4] "The core idea": in the backward pass the
 * gradients flow back to where the tokens came from): every token's gradient
 * is the sum of the gradients of its K receive rows,
 *   dx[r,t,c] = bf16_rne(acc), acc = 0; for k = 0..K-1: acc = acc + float(drecv[dest[r,t,k], c])
 *   drecv [R*S*K, H] bf16; dest [R, S, K] int32; dx [R, S, H] bf16 out. */
int bep_dispatch_bwd(bep_ctx* ctx, const uint16_t* drecv, const int32_t* dest, uint16_t* dx,
                     void* stream);

/* Input gradient of the grouped expert GEMM ([P4] "The memory contract": the
 * same [E+B, H, H'] rows serve the backward pass): for rank u and every
 * non-empty segment rho,
 *   drecv[u*S*K + seg, :] = dy[u*S*K + seg, :] @ W(u, rho)^T,
 * W(u, rho) as in bep_grouped_gemm; bf16 in, fp32 accumulate, bf16 out.
 *   dy [R*S*K, H'] bf16; drecv [R*S*K, H] bf16 out (rows outside every segment
 *   are not written). */
int bep_grouped_gemm_dx(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* dy,
                        const uint16_t* w_home, const uint16_t* w_slots, uint16_t* drecv,
                        void* stream);

/* Weight gradient of the grouped expert GEMM ([P2]; [P4] "The memory contract":
 * training mirrors the weight layout in an fp32 [E+B, H, H'] gradient whose
 * rows [E, E+B) are a separate reduce buffer, invisible to the framework's own
 * gradient reduce): for rank u and every non-empty segment rho,
 *   rho <  E: g_home[rho]            += recv[seg]^T @ dy[seg]
 *   rho >= E: red[u][rho - E]        += recv[seg]^T @ dy[seg]
 * bf16 in, fp32 accumulate; the fp32 products are added to the existing
 * contents (one fp32 add per element). Training mode only (BEP_ERR_MODE
 * otherwise: with overflow rows two segments would share a home row);
 * H % 128 == 0 (BEP_ERR_SIZE otherwise).
 *   recv [R*S*K, H] bf16; dy [R*S*K, H'] bf16; g_home [E, H, H'] fp32 in/out;
 *   red [R, B, H, H'] fp32 in/out. */
int bep_grouped_gemm_dw(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* recv,
                        const uint16_t* dy, float* g_home, float* red, void* stream);

/* The same weight gradient written instead of added (a GEMM with beta = 0), for
 * the first micro-batch of a step, whose gradient buffers would otherwise have
 * to be zeroed first:
 *   g_home[e]          = recv[seg]^T @ dy[seg]  for every expert e, seg = its
 *                        home segment (rank e / (E/R), row e); zeros when that
 *                        segment is empty (all of e's tokens went to replicas,
 *                        or none were routed to e)
 *   red[u][rho - E]    = recv[seg]^T @ dy[seg]  for every non-empty slot segment;
 *                        slots without tokens are not written
 * bf16 in, fp32 accumulate, the fp32 sums stored as they are. reduce_grad then
 * adds the replica slots into the home rows as after bep_grouped_gemm_dw.
 * Arguments, layouts, restrictions and errors as bep_grouped_gemm_dw, and one
 * more: the table must be a training plan's, with home row e used only on e's
 * home rank; a non-empty row e < E on any other rank is refused on the device
 * (BEP_DERR_BOUNDS latched, nothing written). With S*K == 0 only g_home is
 * touched (zeroed); cu_seqlens, recv, dy and red may then be NULL. */
int bep_grouped_gemm_dw_overwrite(bep_ctx* ctx, const int32_t* cu_seqlens, const uint16_t* recv,
                                  const uint16_t* dy, float* g_home, float* red, void* stream);

/* reduce_grad ([P2]; [P4] "The memory contract": each rank reads its own
 * experts' slots from every rank's reduce buffer, accumulates them into its
 * parameter gradient and zeroes the consumed slots):
 *   for e in [0,E): for r = 0..R-1 ascending: for j with slot_expert[r][j] == e:
 *       g_home[e] += red[r][j]   (fp32 adds, in this order);   red[r][j] = 0
 *   slot_expert [R, B] int32; g_home [E, H, H'] fp32 (in/out);
 *   red [R, B, H, H'] fp32 (in/out: consumed slots become zero). */
int bep_reduce_grad(bep_ctx* ctx, const int32_t* slot_expert, float* g_home, float* red,
                    void* stream);

/* SM budget of the token-moving kernels (dispatch, combine, combine_bwd,
 * combine_dgates, dispatch_bwd): their grids are sized for `sms` SMs, so
 * the rest of the GPU stays free for concurrent work, as a communication
 * library with a fixed SM budget runs ([P4] "Benchmarks against DeepEP v2":
 * the pages' comparison uses 32 SMs). 0 (the default) = every SM. Affects
 * only launches made after the call. */
int bep_set_comm_sms(bep_ctx* ctx, int32_t sms);

/* Failure-path self-test (the pages have no counterpart): one GPU thread waits,
 * through the same bounded-wait code the grouped GEMMs use, on a barrier that
 * nothing ever signals. After timeout_us (1 .. 10^7) the wait gives up, sets
 * BEP_DERR_TIMEOUT in the status word and the kernel returns, so the context
 * stays usable. Asynchronous on `stream`. */
int bep_wait_selftest(bep_ctx* ctx, int32_t timeout_us, void* stream);

/* Waits for `stream`, then reads the status word into *device_err (0 = no
 * device error). The only call that blocks the host. */
int bep_status(bep_ctx* ctx, int32_t* device_err, void* stream);

/* Clears the status word (asynchronous, on `stream`). */
int bep_clear_status(bep_ctx* ctx, void* stream);

/* Static description of a return code or status bit set. */
const char* bep_strerror(int32_t code);

#ifdef __cplusplus
}
#endif
#endif /* BEP_H_ */
