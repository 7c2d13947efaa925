// Grouped expert GEMMs over one [E+B, H, H'] weight tensor (sm_103a, tcgen05).
//
// MoonEP pages (ai-maestro.online), "The memory contract": the group GEMM
// consumes a single [E+B, H, H'] weight tensor and addresses experts purely by
// row index; cu_seqlens from the planner selects the active rows. Rows [0, E)
// are the home experts, rows [E, E+B) a rank's prefetch slots; overflow
// experts (inference) are read from their home rows. In training the fp32
// gradient mirrors the layout: rows [0, E) are the parameter gradient, rows
// [E, E+B) a separate reduce buffer that reduce_grad folds back.
//
// Three products share one kernel (template MODE):
//   FWD  Y[seg]     = recv[seg] @ W(u,rho)          A: recv, K-major  B: W, MN-major
//   DX   dRecv[seg] = dY[seg] @ W(u,rho)^T          A: dY, K-major    B: W^T, K-major
//   DW   dW(u,rho) += recv[seg]^T @ dY[seg] (fp32)  A: recv^T, MN-major  B: dY, MN-major
//        dW of a home row accumulates into g_home[rho], of slot j into red[u][j].
// FWD2 / DX2 are FWD / DX with two 128-row m-tiles per unit sharing each weight stage;
// they run the segments of 768 rows or more in a launch of their own before the
// FWD / DX launch that runs the others (large batches with K >= 2,048 and N tiles of 256).
// There both TMEM accumulators belong to one unit: the epilogue frees the first before it
// drains the second, and the MMA thread starts the next unit's first m-tile meanwhile.
//
// Design (one GB300):
//   * a one-CTA prep kernel turns cu_seqlens [R, E+B+1] into a work list on the
//     device (FWD/DX: m-tiles of 128 rows sharing a weight row, FWD2/DX2: 256 rows;
//     DW: one entry per non-empty segment), so the host never learns segment sizes;
//   * a persistent kernel, one CTA per SM, strides over work units with the n
//     tile fastest, so neighbouring CTAs share their A tile in L2;
//   * warp 0 issues TMA loads (128-byte swizzle) into a shared-memory ring guarded
//     by mbarriers (4 stages of 48 KB; FWD2/DX2: 3 stages of 64 KB);
//   * warp 1 (lane 0) issues tcgen05.mma.kind::f16 (M=128, N=BN<=256, K=16,
//     bf16 in, fp32 accumulate; M=64 for a FWD/DX m-tile of at most 64 rows) into
//     one of two TMEM accumulators; tcgen05.commit frees each stage and publishes
//     each finished tile;
//   * 4 (DW, FWD2, DX2: 8) epilogue warps drain the other accumulator with tcgen05.ld:
//     FWD/DX round to bf16 (nearest even) and store only the rows inside the
//     segment; DW adds the fp32 tile into the gradient rows;
//   * DW only: a segment's last K block usually extends past the segment, into
//     the next segment's rows; the 32 lanes of warp 1 zero those rows of both
//     operand tiles in shared memory before lane 0 issues the MMAs that read them.
// When 256 divides H and H', DW runs instead on clusters of two CTAs that share
// each 256 x 256 gradient tile (grouped_gemm_dw_pair_kernel, cta_group::2): half
// the operand bytes per SM and a six-stage ring; there a separate tail warp in
// each CTA zeroes its own tile's rows past a segment end.
// Every mbarrier wait is bounded (2 s on the global timer); on expiry the CTA
// records BEP_DERR_TIMEOUT, every role leaves its loop, and TMEM is freed.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "bep_internal.cuh"

namespace bep {
namespace {

constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBChunkBytes = 64 * kBK * 2;      // 8 KB: 64 rows x 64 columns of bf16
constexpr int kOutBox = 32 * 128;               // epilogue staging box: 32 rows x 128 B
                                                // (DW: 32 fp32 columns; FWD/DX: 64 bf16 columns)
constexpr uint64_t kTimeoutNs = 2000000000ull;

// kFwd2 / kDx2: the forward / input-gradient product with a unit of two 128-row m-tiles
// of one segment that share each weight stage (two accumulators, one per m-tile).
enum GemmMode : int { kFwd = 0, kDx = 1, kDw = 2, kFwd2 = 3, kDx2 = 4 };

template <int MODE>
struct ModeCfg {
    static constexpr bool kDual = MODE == kFwd2 || MODE == kDx2;   // two m-tiles per unit
    static constexpr bool kAmn = MODE == kDw;          // A operand MN-major (recv^T)
    static constexpr bool kBmn = MODE != kDx && MODE != kDx2;   // B operand MN-major
    static constexpr int kEpiWarps = (MODE == kDw || kDual) ? 8 : 4;
    static constexpr int kStages = kDual ? 3 : 4;
    static constexpr int kOutBufs = (MODE == kDw || kDual) ? 1 : 2;   // staging boxes per epilogue warp
    static constexpr int kATiles = kDual ? 2 : 1;  // A tiles (128 rows) per stage
    static constexpr int kWarps = 2 + kEpiWarps;
    static constexpr int kThreads = 32 * kWarps;
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity. false: gave up (timeout
// here, or another role of this CTA already gave up).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status, uint64_t timeout_ns = kTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            set_status(status, BEP_DERR_TIMEOUT);
            return false;
        }
    }
}

// After a bounded wait gave up: wait, again with a limit, for a phase this
// thread knows it started (TMA bytes it armed, MMAs it committed), ignoring
// the abort flag. Used only on the abort path, so that the kernel frees TMEM
// and leaves only once its own copies and MMAs have landed (or the limit ran out).
constexpr uint64_t kDrainNs = 20ull * 1000 * 1000;   // 20 ms
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kDrainNs) return false;
    return true;
}

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Element-wise fp32 add of a shared-memory box into global memory, performed by
// the memory system (one fp32 rounding per element); completion is tracked per
// issuing thread with bulk groups.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int c0,
                                                  int c1) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(c0), "r"(c1)
        : "memory");
}
// Plain copy of a shared-memory box into global memory (the box's rows must all lie
// inside the destination); completion is tracked per issuing thread with bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading / stride
// byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Operand descriptor for the 16-deep K step kk of a 64-deep stage.
//   K-major tile (rows x 64 K, 128-byte rows): 8-row groups 1024 B apart; a
//   K step advances 32 B inside the swizzled row.
//   MN-major tile (64 K-rows x 64-column chunks, 8 KB per chunk): chunks 8 KB
//   apart along M/N, 8-row K groups 1024 B apart; a K step is 16 rows = 2048 B.
template <bool kMN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
    return kMN ? sdesc_sw128(base + kk * 2048, kBChunkBytes, 1024)
               : sdesc_sw128(base + kk * 32, 16, 1024);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A/B major
// bits 15/16 (1 = MN-major), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ---- SM pairs (a cluster of two CTAs running one cta_group::2 MMA stream)
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}

// Arrive on the mbarrier at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ void mbar_arrive_rank(uint64_t* bar, uint32_t rank) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr(bar, rank))
                 : "memory");
}

// TMA tile load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (bar_cl: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap* map, uint32_t bar_cl, void* dst, int c0,
                                                 int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cl), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait (as mbar_wait) for a barrier that the other CTA of the pair arrives on,
// with cluster-scope acquire: what that CTA wrote before its release is visible after.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  int32_t* status) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kTimeoutNs) {
            *abort_flag = 1;
            set_status(status, BEP_DERR_TIMEOUT);
            return false;
        }
    }
}

// Zero the rows [tail, 16 * ceil(tail / 16)) of a stage's two 64-column A chunks and
// two B chunks in this CTA's shared memory (whole 128-byte rows, so the swizzle does
// not matter), then make the stores visible to the tensor core's async proxy. Warp-wide.
__device__ __forceinline__ void zero_tail_rows(uint8_t* a_stage, uint8_t* b_stage, int tail, int lane) {
    const int nrow = 16 - (tail & 15);
    const int n16 = nrow * 8 * 4;   // rows x 16-byte pieces x (2 A + 2 B chunks)
    for (int i = lane; i < n16; i += 32) {
        const int piece = i & 7;
        const int rc = i >> 3;
        const int r = tail + rc % nrow;
        const int c = rc / nrow;
        uint8_t* base = c < 2 ? a_stage + c * kBChunkBytes : b_stage + (c - 2) * kBChunkBytes;
        *reinterpret_cast<uint4*>(base + r * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
}

// One MMA of the pair: M = 256 rows, 128 from each CTA's A tile; N columns, N/2 from each
// CTA's B tile; each CTA's TMEM receives its own 128 rows. Issued by one thread of CTA 0.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at this offset in both CTAs of the pair when every MMA
// issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}

// The same commit, arriving on CTA 0's barrier only (drain after an abort).
__device__ __forceinline__ void mma_commit_pair_lead(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"((uint16_t)1)
        : "memory");
}

// Load 32 columns of this warp's 32 TMEM lanes; the wait sits in the same asm
// statement so no use of r[] can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- work list
// Exclusive scan of one int per thread over the block; *total gets the sum.
// Every thread of the block must call it (it synchronises).
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int incl = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();   // s_warp may still be read by a previous call
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nwarps ? s_warp[lane] : 0;
        int wi = w;
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        if (lane < nwarps) s_warp[lane] = wi - w;
        if (lane == 31) s_warp[32] = wi;
    }
    __syncthreads();
    *total = s_warp[32];
    return s_warp[warp] + incl - v;
}

// seg_mode == 0: m-tiles of <= 128 rows per non-empty segment (FWD, DX). The tiles
//   of segments with three or more m-tiles ("long": after their first tile the
//   weight row is in L2, so they are tensor-bound) and of shorter segments
//   ("short": their tiles mostly stream a whole weight row, HBM-bound) form two lists, each in
//   (rank, row) order, merged evenly so that both kinds run side by side, when the
//   short tiles are a fifth or more of all tiles (skewed inference batches). A long
//   segment's tiles keep their order, with at most a few short tiles between two
//   of them. Otherwise (training sizes: a few short segments among many long ones)
//   the order is plain (rank, row, m).
// seg_mode == 3: as 0 with tiles of <= 256 rows (two m-tiles: the kFwd2 units), for the
//   segments of kDualMinRows rows or more only; seg_mode == 4: as 0 for the other segments.
// seg_mode == 1: one entry per non-empty segment, rows = its length (DW).
// seg_mode == 2: as 1, plus an entry with rows = 0 for every expert whose home segment
//   (rank e / (E/R), row e) is empty, so that an overwriting DW writes its zeros; a
//   non-empty home row on any other rank refuses the table.
// DW entries are merged the same way, long against short: every unit of a segment adds
//   (or writes) a whole 256 KB gradient tile, but runs MMAs only over the segment's rows,
//   so a segment of a few hundred rows is all gradient traffic and a long one all MMAs.
//   Skewed routings have both (at maxvio 10 on the S=8192, E=384 workload, 136 of 372
//   segments hold fewer than 256 rows); merged evenly, CTAs on short segments move
//   gradients while the others keep the tensor pipes busy.
constexpr int kDwShortRows = 1024;
constexpr int kDualMinRows = 768;

__global__ void __launch_bounds__(1024) gemm_tiles_kernel(const int32_t* __restrict__ cu, Dims d,
                                                          Workspace ws, int seg_mode) {
    const bool dw = seg_mode == 1 || seg_mode == 2;
    // FWD/DX: rows per tile (kFwd2: two m-tiles)
    const int tile = seg_mode == 3 ? 2 * kBM : kBM;
    auto tile_of = [&](int) { return tile; };
    __shared__ int s_warp[33];
    const int n_items = d.R * d.NROW;
    const int per = (n_items + blockDim.x - 1) / blockDim.x;
    const int lo = min(n_items, (int)threadIdx.x * per), hi = min(n_items, lo + per);
    int bad = 0;
    auto tiles_of = [&](int i, int* start, int* len) -> int {
        const int u = i / d.NROW, rho = i % d.NROW;
        const int a = cu[u * (d.NROW + 1) + rho], b = cu[u * (d.NROW + 1) + rho + 1];
        if (a < 0 || b < a || (int64_t)b > d.C) {
            bad = 1;
            return 0;
        }
        *start = a;
        *len = b - a;
        if (seg_mode == 2 && rho < d.E) {
            // a training plan uses home row e only on e's home rank; another rank's rows
            // there would make two units write one gradient row
            if (u == rho / (d.E / d.R)) return 1;
            if (b > a) bad = 1;
            return 0;
        }
        if (dw) return b > a ? 1 : 0;
        // seg_mode 3 takes the segments of kDualMinRows rows or more, seg_mode 4 the others
        if ((seg_mode == 3 && b - a < kDualMinRows) || (seg_mode == 4 && b - a >= kDualMinRows))
            return 0;
        const int tl = tile_of(b - a);
        return (b - a + tl - 1) / tl;
    };
    // FWD/DX: a segment of three or more m-tiles is long; DW: one of kDwShortRows rows or more
    auto is_long = [&](int n, int l) { return dw ? l >= kDwShortRows : l > 2 * kBM; };
    // the merge is for the accumulating DW only: the overwriting one reads no gradient, its
    // short segments' units are light, and there merging measured no faster
    int nlong = 0, nshort = 0;
    for (int i = lo; i < hi; ++i) {
        int s = 0, l = 0;
        const int n = tiles_of(i, &s, &l);
        if (is_long(n, l)) nlong += n;
        else nshort += n;
    }
    int Nl = 0, Ns = 0;
    int run_l = block_exclusive_scan(nlong, s_warp, &Nl);
    int run_s = block_exclusive_scan(nshort, s_warp, &Ns);
    const int total = Nl + Ns;
    // FWD/DX: merge only where the short tiles are a fifth or more of the work (skewed
    // inference batches); with a few short tiles among many long ones (training) spreading
    // them only moved weight rows out of L2 early, so the order stays plain. DW: merge
    // whenever both kinds are present.
    const bool mix = Nl > 0 && Ns > 0 && seg_mode != 2 && (seg_mode == 1 || 4 * (int64_t)Ns >= Nl);
    // one inconsistent segment anywhere refuses the whole table: nothing is computed
    const bool ok = !__syncthreads_or(bad) && total <= d.max_tiles;
    // merged position of the k-th long tile / k-th short tile: order by the stamps
    // (2k+1)/(2 Nl) and (2k+1)/(2 Ns), a long tile first on a tie
    // (32-bit division when the products fit, as they do below ~46k tiles)
    const bool narrow = (int64_t)(2 * total + 1) * total < (int64_t)UINT32_MAX;
    auto div = [&](int64_t a, int b) -> int64_t {
        return narrow ? (int64_t)((uint32_t)a / (uint32_t)b) : a / b;
    };
    auto pos_long = [&](int k) -> int {
        const int64_t q = div((2 * (int64_t)k + 1) * Ns + Nl - 1, Nl);
        return k + (int)(q / 2 < Ns ? q / 2 : Ns);
    };
    auto pos_short = [&](int k) -> int {
        const int64_t y = div((2 * (int64_t)k + 1) * Nl, Ns);
        return k + (int)((y + 1) / 2 < Nl ? (y + 1) / 2 : Nl);
    };
    for (int i = lo; i < hi && ok; ++i) {
        int s = 0, l = 0;
        const int n = tiles_of(i, &s, &l);
        const int u = i / d.NROW, rho = i % d.NROW;
        const int wsel = rho < d.E ? rho : -(1 + u * d.B + (rho - d.E));
        for (int m = 0; m < n; ++m) {
            MTile t;
            const int tl = tile_of(l);
            t.row0 = (int32_t)(u * d.C + s + m * tl);
            t.rows = dw ? l : min(tl, l - m * tl);
            t.wsel = wsel;
            t.pad = u * d.NROW + rho;   // row of rank u's [E+B] view
            // plain (rank, row, m) order: the position among all tiles of this thread's range
            const int plain = run_l + run_s + m;
            const int at = !mix            ? plain
                           : is_long(n, l)   ? pos_long(run_l + m)
                                             : pos_short(run_s + m);
            ws.tiles[at] = t;
        }
        if (is_long(n, l)) run_l += n;
        else run_s += n;
    }
    if (threadIdx.x == 0) {
        if (!ok) set_status(ws.status, BEP_DERR_BOUNDS);
        *ws.ntiles = ok ? total : 0;
    }
}

struct GemmParams {
    const MTile* tiles;
    const int32_t* ntiles;
    uint16_t* out;       // FWD / DX: bf16 [R*C, N]
    float* g_home;       // DW: [E, H, H'] fp32
    float* red;          // DW: [R*B, H, H'] fp32
    int N;               // output columns
    int Kdim;            // FWD / DX: reduction length (H / H')
    int H;               // rows of one expert's weight block
    int BN;
    int tmem_cols;
    int mtd;             // DW: m-blocks per weight row (H / 128)
    int vm;              // FWD / DX: weights as R consecutive [E+B, H, H'] views (tmB0)
    int accumulate;      // DW: 1 = add the products to the gradient, 0 = write them
    int32_t* status;
};

// Units of work, identical for every role of a CTA.
struct Unit {
    MTile t;
    int nt;
    int mblk;   // DW: m-block inside the [H, H'] gradient
    int kb_n;   // K blocks of 64
    int tail;   // DW: valid rows of the last K block (64 = full)
};

template <int MODE>
__device__ __forceinline__ Unit unit_at(const GemmParams& p, int unit, int NT) {
    Unit u;
    if (MODE == kDw) {
        const int per = p.mtd * NT;
        const int seg = unit / per;
        const int rem = unit - seg * per;
        u.t = p.tiles[seg];
        u.mblk = rem / NT;
        u.nt = rem - u.mblk * NT;
        u.kb_n = (u.t.rows + kBK - 1) / kBK;
        u.tail = u.t.rows - (u.kb_n - 1) * kBK;
    } else {
        const int mt = unit / NT;
        u.t = p.tiles[mt];
        u.nt = unit - mt * NT;
        u.mblk = 0;
        u.kb_n = p.Kdim / kBK;
        u.tail = kBK;
    }
    return u;
}

// ---------------------------------------------------------------- the GEMM
template <int MODE>
__global__ void __launch_bounds__(ModeCfg<MODE>::kThreads, 1) grouped_gemm_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
    const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO0,
    const __grid_constant__ CUtensorMap tmO1, const GemmParams p) {
    using CF = ModeCfg<MODE>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned carve-up: A ring, B ring, barriers
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int BN = p.BN;
    const int b_bytes = BN * kBK * 2;
    uint8_t* smA = smem;
    constexpr int kStages = CF::kStages;
    constexpr int kAStage = CF::kATiles * kABytes;   // A bytes per stage
    uint8_t* smB = smem + kStages * kAStage;
    uint8_t* smO = smB + kStages * b_bytes;   // a 4 KB staging box per epilogue warp
    uint64_t* bars = reinterpret_cast<uint64_t*>(smO + CF::kEpiWarps * CF::kOutBufs * kOutBox);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* tfull = bars + 2 * kStages;
    uint64_t* tempty = bars + 2 * kStages + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    uint64_t* drain = bars + 2 * kStages + 5;   // the MMA thread's last commit after an abort
    int32_t* status = p.status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], CF::kEpiWarps);
        }
        mbar_init(drain, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(s_tmem)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    const int NT = p.N / BN;
    const int total = MODE == kDw ? *p.ntiles * p.mtd * NT : *p.ntiles * NT;
    const uint32_t stage_bytes = (uint32_t)(kAStage + b_bytes);
    const int acc_stride = p.tmem_cols / 2;   // two accumulators, power-of-two spaced columns
    uint32_t pr_s = 0, pr_ph = 0, pr_armed = 0;   // the producer's ring position and stages armed

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
            // The boxes of K block kb of unit u: op(map, piece, c0, c1), pieces 0-1
            // are the A tile's 8 KB chunks, pieces 2.. the B tile's.
            auto kblock = [&](const Unit& u, int kb, auto&& op) {
                const int n0 = u.nt * BN;
                const CUtensorMap* tmB = (MODE == kDw || p.vm || u.t.wsel >= 0) ? &tmB0 : &tmB1;
                const int brow0 = (p.vm ? u.t.pad : (u.t.wsel >= 0 ? u.t.wsel : (-1 - u.t.wsel))) * p.H;
                if (MODE == kFwd || MODE == kFwd2) {
                    op(&tmA, 0, kb * kBK, u.t.row0);
                    if (CF::kDual) op(&tmA, 1, kb * kBK, u.t.row0 + kBM);
                    for (int c = 0; c < BN / 64; ++c) op(tmB, 2 + c, n0 + c * 64, brow0 + kb * kBK);
                } else if (MODE == kDx || MODE == kDx2) {
                    op(&tmA, 0, kb * kBK, u.t.row0);
                    if (CF::kDual) op(&tmA, 1, kb * kBK, u.t.row0 + kBM);
                    op(tmB, 2, kb * kBK, brow0 + n0);
                } else {
                    const int r0 = u.t.row0 + kb * kBK;
                    for (int c = 0; c < 2; ++c) op(&tmA, c, u.mblk * kBM + c * 64, r0);
                    for (int c = 0; c < BN / 64; ++c) op(&tmB0, 2 + c, n0 + c * 64, r0);
                }
            };
            uint32_t& s = pr_s;
            uint32_t& ph = pr_ph;
            bool live = true;
            // FWD: a CTA's odd units walk K from the end. The CTAs stay close to lockstep
            // (every unit has the same K length), so successive waves of units alternate
            // direction, and the units of a segment that straddles two waves start where
            // the earlier wave ended: on the weight and row tiles most recently loaded,
            // which are still in L2, instead of on the first ones, long evicted. At the
            // S=8192, E=384 routings this took 1-2 GB (7-8%) off the DRAM traffic per launch
            // at the same time; for DX it measured 1.8% slower, so DX keeps one direction.
            int it = 0;
            for (int unit = blockIdx.x; unit < total && live; unit += gridDim.x, ++it) {
                const Unit u = unit_at<MODE>(p, unit, NT);
                const bool rev = (MODE == kFwd || MODE == kFwd2) && (it & 1);
                for (int kb = 0; kb < u.kb_n; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, s_abort, status)) {
                        live = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], stage_bytes);
                    ++pr_armed;
                    uint8_t* a_dst = smA + s * kAStage;
                    uint8_t* b_dst = smB + s * b_bytes;
                    kblock(u, rev ? u.kb_n - 1 - kb : kb, [&](const CUtensorMap* m, int piece, int c0, int c1) {
                        // A: DW's two 8 KB column chunks, or a dual unit's second 128-row tile
                        uint8_t* dst = piece < 2 ? a_dst + piece * (CF::kDual ? kABytes : kBChunkBytes)
                                                 : b_dst + (piece - 2) * kBChunkBytes;
                        tma_load_2d(m, &full[s], dst, c0, c1);
                    });
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer (lane 0)
        // DW: the last K block of a segment usually holds rows of the next
        // segment past `tail`. Only its first ceil(tail/16) K steps are issued;
        // the rows of the last issued step past `tail` (at most 15) are zeroed in
        // both operand tiles by all 32 lanes (whole 128-byte rows, so the
        // swizzle does not matter) before lane 0 issues the MMAs.
        // FWD/DX: an m-tile of at most 64 rows (a segment's last) runs M=64 MMAs, which
        // put row r of the accumulator in TMEM lane 32 * (r / 16) + r % 16.
        // FWD2/DX2: every unit runs both m-tiles at M=128, whatever its rows. A segment's
        // odd last m-tile is paired with the rows that follow it (the next segment's, or
        // the tensor's out-of-bounds zeros), whose results the epilogue never stores.
        // All units then take the same time, so the CTAs stay in lockstep, and the units
        // that share a receive-row or weight tile read each K block of it together, while
        // L2 holds it. With units of two lengths the CTAs drift apart over a launch, and
        // on the S=8192, E=384 workload at maxvio 0.2 (segments of ~1,400 rows) the launch
        // read 40 GB from DRAM instead of 21.
        const uint32_t idesc_full = idesc_bf16(kBM, BN, CF::kAmn, CF::kBmn);
        const uint32_t idesc_half = idesc_bf16(kBM / 2, BN, CF::kAmn, CF::kBmn);
        uint32_t s = 0, ph = 0;
        bool live = true;
        int it = 0;
        for (int unit = blockIdx.x; unit < total && live; unit += gridDim.x, ++it) {
            const Unit u = unit_at<MODE>(p, unit, NT);
            const uint32_t idesc =
                (MODE != kDw && !CF::kDual && u.t.rows <= kBM / 2) ? idesc_half : idesc_full;
            // dual modes: both accumulators belong to one unit (m-tile 0 in the first, m-tile
            // 1 in the second), so units alternate on one barrier pair
            const int acc = CF::kDual ? 0 : it & 1;
            const uint32_t aph = CF::kDual ? (uint32_t)(it & 1) : (uint32_t)((it >> 1) & 1);
            if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], aph ^ 1u, s_abort, status))) break;
            tc_fence_after();
            const uint32_t dt = tmem_base + (uint32_t)(acc * acc_stride);
            const uint32_t dt1 = tmem_base + (uint32_t)acc_stride;
            int kb = 0;
            if (CF::kDual) {
                // The epilogue frees the first accumulator before it drains the second:
                // run the first m-tile's MMAs over the stages already in the ring (up to all
                // of them) while the second accumulator is drained, then the second m-tile's
                // on the same stages, and only then release those stages.
                const int pre = min(kStages, u.kb_n);
                uint32_t s0 = s, ph0 = ph;
                for (int j = 0; j < pre && live; ++j) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&full[s0], ph0, s_abort, status))) {
                        live = false;
                        break;
                    }
                    if (lane == 0) {
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(smA + s0 * kAStage);
                        const uint32_t b0 = smem_u32(smB + s0 * b_bytes);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            mma_bf16(dt, operand_desc<CF::kAmn>(a0, kk), operand_desc<CF::kBmn>(b0, kk),
                                     idesc, (j | kk) != 0);
                    }
                    __syncwarp();
                    if (++s0 == kStages) {
                        s0 = 0;
                        ph0 ^= 1u;
                    }
                }
                if (!live) break;
                if (!__all_sync(0xffffffffu, mbar_wait(&tempty[1], aph ^ 1u, s_abort, status))) break;
                tc_fence_after();
                for (int j = 0; j < pre; ++j) {
                    if (lane == 0) {
                        const uint32_t a1 = smem_u32(smA + s * kAStage) + kABytes;
                        const uint32_t b0 = smem_u32(smB + s * b_bytes);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            mma_bf16(dt1, operand_desc<CF::kAmn>(a1, kk), operand_desc<CF::kBmn>(b0, kk),
                                     idesc_full, (j | kk) != 0);
                        mma_commit(&empty[s]);
                    }
                    __syncwarp();
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                kb = pre;
            }
            for (; kb < u.kb_n; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, s_abort, status))) {
                    live = false;
                    break;
                }
                const bool last = MODE == kDw && kb == u.kb_n - 1;
                const int ksteps = last ? (u.tail + 15) / 16 : kBK / 16;
                if (last && (u.tail & 15)) {
                    const int nrow = 16 - (u.tail & 15);
                    const int nchunk = 2 + BN / 64;            // A: 2 chunks, B: BN/64 chunks
                    const int n16 = nrow * 8 * nchunk;         // 16-byte pieces to clear
                    for (int i = lane; i < n16; i += 32) {
                        const int piece = i & 7;
                        const int rc = i >> 3;
                        const int r = u.tail + rc % nrow;
                        const int c = rc / nrow;
                        uint8_t* base = c < 2 ? smA + s * kABytes + c * kBChunkBytes
                                              : smB + s * b_bytes + (c - 2) * kBChunkBytes;
                        *reinterpret_cast<uint4*>(base + r * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
                    }
                    // generic-proxy stores become visible to the tensor core's async proxy
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                }
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smA + s * kAStage);
                    const uint32_t b0 = smem_u32(smB + s * b_bytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        if (kk < ksteps) {
                            mma_bf16(dt, operand_desc<CF::kAmn>(a0, kk), operand_desc<CF::kBmn>(b0, kk),
                                     idesc, (kb | kk) != 0);
                            if (CF::kDual)
                                mma_bf16(dt1, operand_desc<CF::kAmn>(a0 + kABytes, kk),
                                         operand_desc<CF::kBmn>(b0, kk), idesc_full, (kb | kk) != 0);
                        }
                    mma_commit(&empty[s]);
                }
                __syncwarp();
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (live && lane == 0) mma_commit(&tfull[acc]);
        }
    } else if (warp < 2 + CF::kEpiWarps) {
        // ---------------------------------------------------- epilogue
        const int e = warp - 2;
        const int q = warp & 3;                            // TMEM lanes 32q..32q+31 are this warp's
        const int halves = CF::kEpiWarps / 4;              // warps sharing one lane quadrant
        const int cspan = BN / halves;
        const int c_lo = (e / 4) * cspan;
        int it = 0;
        int obox = 0, last_store = -1;   // FWD/DX: next staging box; box of the newest TMA store
        for (int unit = blockIdx.x; unit < total; unit += gridDim.x, ++it) {
            const int acc = CF::kDual ? 0 : it & 1;
            const uint32_t aph = CF::kDual ? (uint32_t)(it & 1) : (uint32_t)((it >> 1) & 1);
            const bool got = mbar_wait(&tfull[acc], aph, s_abort, status);
            __syncwarp();
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const Unit u = unit_at<MODE>(p, unit, NT);
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * acc_stride);
            if (MODE == kDw) {
                // 32 rows x 32 columns at a time: stage the fp32 box in shared memory
                // (128-byte swizzle: 16-byte piece j of row r sits at j ^ (r & 7)), then
                // one lane has the memory system add it to the gradient rows (one fp32
                // rounding per element). Measured alternatives -- two staging boxes per
                // warp with a 3-stage operand ring, red.global.add.v4 per row or read back
                // coalesced, and a load/add/store on the LSU path with the next chunk in
                // flight -- were slower or no faster on the S=8192, E=384 workload.
                const CUtensorMap* tmO = u.t.wsel >= 0 ? &tmO0 : &tmO1;
                const int orow0 = (u.t.wsel >= 0 ? u.t.wsel : (-1 - u.t.wsel)) * p.H +
                                  u.mblk * kBM + q * 32;
                uint8_t* stg = smO + e * kOutBox;
                uint4* srow = reinterpret_cast<uint4*>(stg + lane * 128);
                for (int c0 = c_lo; c0 < c_lo + cspan; c0 += 32) {
                    uint32_t r[32];
                    if (u.t.rows > 0) {
                        tmem_ld_32x32b_x32(tbase + (uint32_t)c0, r);
                    } else {   // an empty home segment (overwrite only): its gradient is zero
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = 0u;
                    }
                    if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        srow[j ^ (lane & 7)] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        if (p.accumulate) tma_reduce_add_2d(tmO, stg, u.nt * BN + c0, orow0);
                        else tma_store_2d(tmO, stg, u.nt * BN + c0, orow0);
                        bulk_commit();
                    }
                }
            } else {
                // 64 columns at a time: round to bf16 (nearest even) and stage the warp's
                // 32 rows x 128 B in shared memory (16-byte piece j of row r sits at
                // j ^ (r & 7), the 128-byte swizzle). A box whose 32 rows all lie inside
                // the segment leaves by one TMA store; a segment's ragged last box is read
                // back a row per 8 lanes and stored by the threads (each instruction writes
                // four whole 128-byte lines), skipping the rows past the segment end, which
                // belong to the next segment's tile. Two boxes per warp alternate, so one
                // store can be in flight while the next box is filled.
                // this warp's rows: 32q..32q+31 of a full tile, or, of an M=64 tile (FWD/DX),
                // 16q..16q+15 in lanes 0-15 of its quadrant; a dual unit drains its first
                // m-tile from the first accumulator, then its second from the second (none of
                // whose rows may lie in the segment)
                for (int half = 0; half < (CF::kDual ? 2 : 1); ++half) {
                const int trows = CF::kDual ? min(u.t.rows - half * kBM, kBM) : u.t.rows;
                const int trow0 = u.t.row0 + half * kBM;
                const uint32_t tb = tbase + (uint32_t)(half * acc_stride);
                const int wrows = (!CF::kDual && trows <= kBM / 2) ? 16 : 32;
                const int nvalid = min(wrows, trows - q * wrows);   // of them inside the segment
                const int rsub = lane >> 3, piece = lane & 7;
                const int orow = trow0 + q * wrows;
                uint16_t* ybase = p.out + (int64_t)orow * p.N + (int64_t)u.nt * BN;
                if constexpr (CF::kDual) {
                    // Read the warp's 128 columns of this accumulator into registers (as bf16)
                    // and free the accumulator before staging and storing them: the next unit's
                    // MMAs into it wait only for these TMEM loads. Freed after the stores instead,
                    // the MMA thread waited 8% of its time for the first accumulator in the
                    // input-gradient GEMM (32 K blocks per unit) and 2.6% in the forward.
                    uint4 pk[2][8];
                    if (nvalid > 0) {
#pragma unroll
                        for (int ci = 0; ci < 2; ++ci)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                uint32_t r[32];
                                tmem_ld_32x32b_x32(tb + (uint32_t)(c_lo + 64 * ci + 32 * h), r);
#pragma unroll
                                for (int v = 0; v < 4; ++v) {
                                    uint4& o = pk[ci][4 * h + v];
                                    o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                                    o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                                    o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                                    o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                                }
                            }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[half]);   // this half's accumulator is free
#pragma unroll
                    for (int ci = 0; ci < 2; ++ci) {
                        if (nvalid <= 0) break;
                        const int c0 = c_lo + 64 * ci;
                        uint8_t* stg = smO + e * kOutBox;   // one staging box per warp
                        uint4* srow = reinterpret_cast<uint4*>(stg + lane * 128);
                        if (lane == 0) bulk_wait_read_all();   // the box's previous store has read it
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j) srow[j ^ (lane & 7)] = pk[ci][j];
                        if (nvalid == 32) {
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&tmO0, stg, u.nt * BN + c0, orow);
                                bulk_commit();
                            }
                        } else {
                            __syncwarp();
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const int rr = 4 * k + rsub;
                                const uint4 o =
                                    *reinterpret_cast<const uint4*>(stg + rr * 128 + ((piece ^ (rr & 7)) << 4));
                                if (rr < nvalid)
                                    *reinterpret_cast<uint4*>(ybase + (int64_t)rr * p.N + c0 + piece * 8) = o;
                            }
                            __syncwarp();   // the box is read back before it is filled again
                        }
                    }
                } else {
                    for (int c0 = c_lo; c0 < c_lo + cspan && nvalid > 0; c0 += 64) {
                        const int b = obox++ % CF::kOutBufs;
                        uint8_t* stg = smO + (e * CF::kOutBufs + b) * kOutBox;
                        uint4* srow = reinterpret_cast<uint4*>(stg + lane * 128);
                        // a store issued from this box earlier has read it: every bulk group but the
                        // newest is complete after wait_group.read 1; if the newest came from this box
                        // too, wait for it as well
                        if (lane == 0) {
                            if (last_store == b) bulk_wait_read_all();
                            else bulk_wait_read_1();
                        }
                        __syncwarp();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t r[32];
                            tmem_ld_32x32b_x32(tb + (uint32_t)(c0 + 32 * h), r);
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                uint4 o;
                                o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                                o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                                o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                                o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                                srow[(4 * h + v) ^ (lane & 7)] = o;
                            }
                        }
                        if (nvalid == 32) {
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&tmO0, stg, u.nt * BN + c0, orow);
                                bulk_commit();
                            }
                            last_store = b;
                        } else {
                            __syncwarp();
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const int rr = 4 * k + rsub;
                                const uint4 o =
                                    *reinterpret_cast<const uint4*>(stg + rr * 128 + ((piece ^ (rr & 7)) << 4));
                                if (rr < nvalid)
                                    *reinterpret_cast<uint4*>(ybase + (int64_t)rr * p.N + c0 + piece * 8) = o;
                            }
                            __syncwarp();   // the box is read back before it is filled again
                        }
                    }
                }
                }   // half
            }
            if (!CF::kDual) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[acc]);
            }
        }
        // every store or reduce this warp issued has completed before the CTA ends
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    __syncthreads();
    if (*s_abort) {
        // A wait gave up. Before TMEM and shared memory are released, what was started
        // lands: the producer waits (bounded) for the full phase of each stage it armed
        // last (at most the ring), the MMA thread commits once more and waits for that,
        // and the epilogue warps have already waited for their stores and reduces.
        if (warp == 0 && lane == 0) {
            for (uint32_t i = 0; i < pr_armed && i < (uint32_t)kStages; ++i) {
                if (pr_s == 0) {
                    pr_s = kStages;
                    pr_ph ^= 1u;
                }
                --pr_s;
                mbar_drain(&full[pr_s], pr_ph);
            }
        } else if (warp == 1 && lane == 0) {
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(p.tmem_cols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- DW on SM pairs
// The weight gradient with each 256 x 256 output tile shared by a cluster of two
// CTAs on neighbouring SMs (tcgen05 cta_group::2). CTA r of the pair loads, per
// 64-row K block, its 128 columns h of recv (A) and its 128 columns h' of dY (B):
// 32 KB per stage instead of the 48 KB one CTA needs for a 128 x 256 tile, so a
// six-stage ring fits where the single-CTA kernel holds four. One thread of CTA 0
// issues M=256, N=256 MMAs that read both CTAs' tiles; each CTA's TMEM receives
// its own 128 gradient rows, and each CTA's 8 epilogue warps add them into the
// gradient exactly as the single-CTA kernel does (same tiles of 32 x 32 fp32, same
// K order, so the sums are the same bit for bit).
//   barriers        owner   arrivals
//   full[s]         CTA 0   CTA 0's producer (expect_tx) + both CTAs' TMA bytes; in a tail
//                           stage only a plain arrive from CTA 0's producer
//   ptail[k % 8]    both    own producer (expect_tx) + own TMA bytes of the k-th tail stage
//   zpeer[k % 8]    CTA 0   each CTA's tail warp, once its rows of the k-th tail stage are zero
//   empty[s]        both    the MMA thread's multicast commit
//   tfull[a]        both    the MMA thread's multicast commit at the end of a unit
//   tempty[a]       CTA 0   the 8 epilogue warps of each CTA
// CTA 1's loads count on CTA 0's full barrier, so CTA 0 knows when the whole stage
// is in. A segment's last K block usually holds rows of the next segment: in that
// "tail stage" each CTA loads its tiles onto its own barrier, and a tail warp of each
// CTA zeroes the extra rows and tells CTA 0's MMA thread (CTA 1 with one remote
// arrive per unit), ahead of the MMAs that need it and off the MMA thread. The ring holds 6 stages, so at most 6 tail
// stages are loaded and not yet consumed; 8 ptail and 8 zpeer barriers therefore
// never see two unobserved phases, which a parity wait could not tell apart.
// Every wait is bounded; the CTAs meet at a cluster barrier before TMEM is freed
// and either exits.
constexpr int kPairStages = 6;
constexpr int kPairEpiWarps = 8;
constexpr int kPairTailWarp = 2 + kPairEpiWarps;   // warp that zeroes its CTA's tail rows
constexpr int kPairThreads = 32 * (3 + kPairEpiWarps);
constexpr int kPairHalf = 2 * kBChunkBytes;   // 16 KB: one CTA's A (or B) tile of a K block
constexpr int kPairTails = 8;                 // ptail / zpeer barriers (> stages in the ring)
constexpr int kPairBars = 2 * kPairStages + 4 + 2 * kPairTails;
constexpr int kPairBN = 256;
constexpr int kPairBM = 256;

__global__ void __launch_bounds__(kPairThreads, 1) grouped_gemm_dw_pair_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
    const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmR,
    const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* smA = smem;
    uint8_t* smB = smA + kPairStages * kPairHalf;
    uint8_t* smO = smB + kPairStages * kPairHalf;   // a 4 KB staging box per epilogue warp
    uint64_t* bars = reinterpret_cast<uint64_t*>(smO + kPairEpiWarps * kOutBox);
    uint64_t* full = bars;
    uint64_t* empty = bars + kPairStages;
    uint64_t* tfull = bars + 2 * kPairStages;
    uint64_t* tempty = bars + 2 * kPairStages + 2;
    uint64_t* ptail = bars + 2 * kPairStages + 4;
    uint64_t* zpeer = ptail + kPairTails;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + kPairBars);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    uint64_t* drain = bars + kPairBars + 1;   // CTA 0's MMA thread's last commit after an abort
    int32_t* status = p.status;
    const uint32_t rank = cluster_rank();
    const bool lead = rank == 0;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 2 * kPairEpiWarps);
        }
        for (int k = 0; k < kPairTails; ++k) {
            mbar_init(&ptail[k], 1);
            mbar_init(&zpeer[k], 2);
        }
        mbar_init(drain, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        // one warp of each CTA performs the pair's allocation together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(s_tmem)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers exist before any remote arrive or multicast commit
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    const int NT = p.N / kPairBN;
    const int per_seg = (p.H / kPairBM) * NT;
    const int total = *p.ntiles * per_seg;
    const int cl0 = (int)cluster_id(), ncl = (int)cluster_count();
    const int acc_stride = p.tmem_cols / 2;
    auto unit_of = [&](int unit, MTile* t, int* mp, int* nt, int* kb_n, int* tail) {
        const int seg = unit / per_seg;
        const int rem = unit - seg * per_seg;
        *t = p.tiles[seg];
        *mp = rem / NT;
        *nt = rem - *mp * NT;
        *kb_n = (t->rows + kBK - 1) / kBK;
        *tail = t->rows - (*kb_n - 1) * kBK;
    };
    // the producer's ring position, stages armed and tail stages armed (drain after an abort)
    uint32_t pr_s = 0, pr_ph = 0, pr_armed = 0, pr_tk = 0;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (each CTA its own half)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
            uint32_t& s = pr_s;
            uint32_t& ph = pr_ph;
            uint32_t& tk = pr_tk;
            bool live = true;
            for (int unit = cl0; unit < total && live; unit += ncl) {
                MTile t;
                int mp, nt, kb_n, tail;
                unit_of(unit, &t, &mp, &nt, &kb_n, &tail);
                const int h0 = mp * kPairBM + (int)rank * 128;
                const int n0 = nt * kPairBN + (int)rank * 128;
                for (int kb = 0; kb < kb_n; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, s_abort, status)) {
                        live = false;
                        break;
                    }
                    // CTA 0's barrier counts both CTAs' 32 KB, except in a tail stage, whose
                    // bytes each CTA counts on its own ptail barrier (its tail warp zeroes
                    // the extra rows); CTA 0 then completes the stage's full phase at once
                    const bool tstage = kb == kb_n - 1 && (tail & 15);
                    const int r0 = t.row0 + kb * kBK;
                    ++pr_armed;
                    if (tstage) {
                        uint64_t* tb = &ptail[tk++ % kPairTails];
                        mbar_arrive_expect_tx(tb, 2 * kPairHalf);
                        for (int c = 0; c < 2; ++c) {
                            tma_load_2d(&tmA, tb, smA + s * kPairHalf + c * kBChunkBytes, h0 + c * 64, r0);
                            tma_load_2d(&tmB, tb, smB + s * kPairHalf + c * kBChunkBytes, n0 + c * 64, r0);
                        }
                        if (lead) mbar_arrive(&full[s]);
                    } else {
                        if (lead) mbar_arrive_expect_tx(&full[s], 4 * kPairHalf);
                        const uint32_t bar = cluster_addr(&full[s], 0);
                        for (int c = 0; c < 2; ++c) {
                            tma_load_2d_pair(&tmA, bar, smA + s * kPairHalf + c * kBChunkBytes, h0 + c * 64, r0);
                            tma_load_2d_pair(&tmB, bar, smB + s * kPairHalf + c * kBChunkBytes, n0 + c * 64, r0);
                        }
                    }
                    if (++s == kPairStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer (CTA 0 only)
        // A segment's last K block usually holds rows of the next segment past
        // `tail`: only its first ceil(tail/16) K steps are issued, after the tail
        // warps of both CTAs have zeroed the rows of the last issued step past `tail`
        // (at most 15) in their A and B tiles.
        if (lead) {
            const uint32_t idesc = idesc_bf16(kPairBM, kPairBN, true, true);
            uint32_t s = 0, ph = 0, zc = 0;
            bool live = true;
            int it = 0;
            for (int unit = cl0; unit < total && live; unit += ncl, ++it) {
                MTile t;
                int mp, nt, kb_n, tail;
                unit_of(unit, &t, &mp, &nt, &kb_n, &tail);
                const int acc = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], aph ^ 1u, s_abort, status))) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(acc * acc_stride);
                for (int kb = 0; kb < kb_n; ++kb) {
                    const bool last = kb == kb_n - 1;
                    const bool tstage = last && (tail & 15);
                    bool ok = mbar_wait(&full[s], ph, s_abort, status);
                    if (ok && tstage)
                        ok = mbar_wait_cluster(&zpeer[zc % kPairTails], (zc / kPairTails) & 1u, s_abort, status);
                    if (!__all_sync(0xffffffffu, ok)) {
                        live = false;
                        break;
                    }
                    if (tstage) ++zc;
                    const int ksteps = last ? (tail + 15) / 16 : kBK / 16;
                    if (lane == 0) {
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(smA + s * kPairHalf);
                        const uint32_t b0 = smem_u32(smB + s * kPairHalf);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            if (kk < ksteps)
                                mma_bf16_pair(dt, operand_desc<true>(a0, kk), operand_desc<true>(b0, kk), idesc,
                                              (kb | kk) != 0);
                        mma_commit_pair(&empty[s]);
                    }
                    __syncwarp();
                    if (++s == kPairStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (live && lane == 0) mma_commit_pair(&tfull[acc]);
            }
        }
    } else if (warp == kPairTailWarp) {
        // ---------------------------------------------------- tail rows (both CTAs)
        // Follow the stage sequence; in each unit's tail stage wait for the CTA's own
        // bytes, zero the rows past the segment end and release the stage to CTA 0's MMA
        // thread (zpeer counts one arrival from each CTA).
        {
            uint32_t s = 0, tc = 0;
            for (int unit = cl0; unit < total; unit += ncl) {
                MTile t;
                int mp, nt, kb_n, tail;
                unit_of(unit, &t, &mp, &nt, &kb_n, &tail);
                const uint32_t st = (s + (uint32_t)kb_n - 1) % kPairStages;
                s = (s + (uint32_t)kb_n) % kPairStages;
                if (!(tail & 15)) continue;
                if (!__all_sync(0xffffffffu, mbar_wait(&ptail[tc % kPairTails], (tc / kPairTails) & 1u,
                                                       s_abort, status)))
                    break;
                zero_tail_rows(smA + st * kPairHalf, smB + st * kPairHalf, tail, lane);
                if (lane == 0) {
                    if (lead) mbar_arrive(&zpeer[tc % kPairTails]);
                    else mbar_arrive_rank(&zpeer[tc % kPairTails], 0);
                }
                ++tc;
                __syncwarp();
            }
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs: own 128 rows)
        const int e = warp - 2;
        const int q = warp & 3;
        const int c_lo = (e / 4) * (kPairBN / 2);
        int it = 0;
        for (int unit = cl0; unit < total; unit += ncl, ++it) {
            const int acc = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            const bool got = mbar_wait(&tfull[acc], aph, s_abort, status);
            __syncwarp();
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            MTile t;
            int mp, nt, kb_n, tail;
            unit_of(unit, &t, &mp, &nt, &kb_n, &tail);
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * acc_stride);
            const CUtensorMap* tmO = t.wsel >= 0 ? &tmG : &tmR;
            const int orow0 = (t.wsel >= 0 ? t.wsel : (-1 - t.wsel)) * p.H + mp * kPairBM +
                              (int)rank * 128 + q * 32;
            uint8_t* stg = smO + e * kOutBox;
            uint4* srow = reinterpret_cast<uint4*>(stg + lane * 128);
            for (int c0 = c_lo; c0 < c_lo + kPairBN / 2; c0 += 32) {
                uint32_t r[32];
                if (t.rows > 0) {
                    tmem_ld_32x32b_x32(tbase + (uint32_t)c0, r);
                } else {   // an empty home segment (overwrite only): its gradient is zero
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;
                }
                if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    srow[j ^ (lane & 7)] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    if (p.accumulate) tma_reduce_add_2d(tmO, stg, nt * kPairBN + c0, orow0);
                    else tma_store_2d(tmO, stg, nt * kPairBN + c0, orow0);
                    bulk_commit();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (lead) mbar_arrive(&tempty[acc]);
                else mbar_arrive_rank(&tempty[acc], 0);
            }
        }
        if (lane == 0) bulk_wait_all();   // every reduce this warp issued has been applied
        __syncwarp();
    }

    __syncthreads();
    if (*s_abort) {
        // A wait gave up. Before TMEM and shared memory are released, what was started
        // lands, each wait bounded: each CTA's producer waits for the tail-stage loads it
        // counted on its own barriers, CTA 0's producer for the full phase of each stage
        // it armed last (which also counts CTA 1's bytes of those stages), and CTA 0's MMA
        // thread commits once more and waits for that; the epilogue warps have already
        // waited for their reduces. CTA 1's loads of a stage CTA 0 never armed cannot be
        // observed (their bytes count on CTA 0's barrier): the short sleep after the drains
        // is the fallback bound for those.
        if (warp == 0 && lane == 0) {
            for (uint32_t n = pr_tk > kPairTails ? pr_tk - kPairTails : 0; n < pr_tk; ++n)
                mbar_drain(&ptail[n % kPairTails], (n / kPairTails) & 1u);
            if (lead) {
                for (uint32_t i = 0; i < pr_armed && i < (uint32_t)kPairStages; ++i) {
                    if (pr_s == 0) {
                        pr_s = kPairStages;
                        pr_ph ^= 1u;
                    }
                    --pr_s;
                    mbar_drain(&full[pr_s], pr_ph);
                }
            }
        } else if (warp == 1 && lane == 0 && lead) {
            mma_commit_pair_lead(drain);
            mbar_drain(drain, 0);
        }
        if (threadIdx.x == 0)
            for (int i = 0; i < 20; ++i) __nanosleep(10000);
        __syncthreads();
    }
    cluster_sync();   // neither CTA leaves while the other may still signal it or read its tiles
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(p.tmem_cols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- wait self-test
// One thread waits, through the GEMM's bounded-wait helper, on an mbarrier that
// nothing ever arrives on. The wait gives up after timeout_ns, records
// BEP_DERR_TIMEOUT and the kernel returns: the failure path is exercised without
// faulting or hanging anything.
__global__ void wait_selftest_kernel(int32_t* status, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(&bar, 0, &abort_flag, status, timeout_ns);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
    if (g_encode) return cudaSuccess;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                       cudaEnableDefault, &q);
    if (err != cudaSuccess) return err;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box [box_rows, box_cols], 128-byte swizzle.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
               uint32_t box_cols) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D fp32 tensor [rows, cols], 32 x 32 boxes (128-byte rows), 128-byte swizzle: the
// target of the DW epilogue's bulk reduce-add.
bool encode_2d_f32(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int pick_bn(int n) {
    for (int bn = 256; bn >= 64; bn -= 64)
        if (n % bn == 0) return bn;
    return 64;
}

template <int MODE>
size_t smem_bytes(int BN) {
    using CF = ModeCfg<MODE>;
    const size_t stage_out = (size_t)CF::kEpiWarps * CF::kOutBufs * kOutBox;
    return 1024 + (size_t)CF::kStages * (CF::kATiles * kABytes + BN * kBK * 2) + stage_out +
           (2 * CF::kStages + 4) * 8 + 16;
}

// The forward runs the segments of kDualMinRows rows or more with two m-tiles per unit
// (kFwd2: one weight stage feeds two 128-row m-tiles, both accumulators of TMEM, so
// BN = 256), in a launch of its own before the other segments, when the batch has on
// average at least kDualRows receive rows per expert and K is at least kDualMinK:
// elsewhere (inference batches, small K) the two launches and the per-unit hand-over
// between the two accumulators cost more than the halved weight reads save.
constexpr int kDualRows = 512;
constexpr int kDualMinK = 2048;
bool use_dual(const Dims& d, int K, int BN) {
    return BN == 256 && K >= kDualMinK && (int64_t)d.R * d.C >= (int64_t)kDualRows * d.E;
}

int tmem_cols_for(int BN) {
    int c = 32;
    while (c < 2 * BN) c <<= 1;
    return c;
}

size_t pair_smem_bytes() {
    return 1024 + (size_t)kPairStages * 2 * kPairHalf + (size_t)kPairEpiWarps * kOutBox + kPairBars * 8 + 16;
}

// Clusters of two that can be resident at once, per device (0: no pair launch).
constexpr int kMaxDevices = 64;
int g_pair_clusters[kMaxDevices] = {};

cudaLaunchConfig_t pair_config(int clusters, cudaStream_t st, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = pair_smem_bytes();
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                        const CUtensorMap& o0, const CUtensorMap& o1, const GemmParams& prm,
                        int num_sms, cudaStream_t st) {
    grouped_gemm_kernel<MODE><<<num_sms, ModeCfg<MODE>::kThreads, smem_bytes<MODE>(prm.BN), st>>>(
        a, b0, b1, o0, o1, prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_wait_selftest(const Workspace& ws, uint64_t timeout_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(ws.status, timeout_ns);
    return cudaGetLastError();
}

cudaError_t gemm_setup(int device) {
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(grouped_gemm_kernel<kFwd>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_bytes<kFwd>(256));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(grouped_gemm_kernel<kFwd2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_bytes<kFwd2>(256));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(grouped_gemm_kernel<kDx2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_bytes<kDx2>(256));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(grouped_gemm_kernel<kDx>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_bytes<kDx>(256));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(grouped_gemm_kernel<kDw>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_bytes<kDw>(256));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(grouped_gemm_dw_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)pair_smem_bytes());
    if (err != cudaSuccess) return err;
    // how many SM pairs can hold one pair kernel CTA each at once (0 keeps DW on single CTAs)
    int nsm = 0;
    err = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, device);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config(nsm / 2, nullptr, attr);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_dw_pair_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        clusters = 0;
    }
    if (device >= 0 && device < kMaxDevices) g_pair_clusters[device] = clusters;
    return cudaSuccess;
}

cudaError_t launch_grouped_gemm(const Dims& d, const Workspace& ws, const int32_t* cu,
                                const uint16_t* recv, const uint16_t* w_home,
                                const uint16_t* w_slots, uint16_t* y, int num_sms,
                                cudaStream_t st) {
    if (d.C == 0) return cudaSuccess;
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    const int BN = pick_bn(d.Hp);
    const bool dual = use_dual(d, d.H, BN);
    CUtensorMap tmA, tmBh, tmBs;
    if (!encode_2d(&tmA, recv, (uint64_t)d.R * d.C, d.H, kBM, kBK)) return cudaErrorInvalidValue;
    if (!encode_2d(&tmBh, w_home, (uint64_t)d.E * d.H, d.Hp, kBK, 64)) return cudaErrorInvalidValue;
    const uint64_t slot_rows = (uint64_t)(d.R * d.B > 0 ? d.R * d.B : 1) * d.H;
    if (!encode_2d(&tmBs, w_slots ? w_slots : w_home, slot_rows, d.Hp, kBK, 64))
        return cudaErrorInvalidValue;
    GemmParams prm = {};
    prm.tiles = ws.tiles;
    prm.ntiles = ws.ntiles;
    CUtensorMap tmY;   // Y [R*C, H'] in 32-row x 64-column boxes: the epilogue's stores
    if (!encode_2d(&tmY, y, (uint64_t)d.R * d.C, d.Hp, 32, 64)) return cudaErrorInvalidValue;
    prm.out = y;
    prm.N = d.Hp;
    prm.Kdim = d.H;
    prm.H = d.H;
    prm.BN = BN;
    prm.tmem_cols = tmem_cols_for(BN);   // two BN-column accumulators (kFwd2: one unit's two)
    prm.mtd = 1;
    prm.status = ws.status;
    if (!dual) {
        gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, 0);
        return launch_mode<kFwd>(tmA, tmBh, tmBs, tmY, tmY, prm, num_sms, st);
    }
    // long segments two m-tiles per unit, then the others one per unit
    gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, 3);
    err = launch_mode<kFwd2>(tmA, tmBh, tmBs, tmY, tmY, prm, num_sms, st);
    if (err != cudaSuccess) return err;
    gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, 4);
    return launch_mode<kFwd>(tmA, tmBh, tmBs, tmY, tmY, prm, num_sms, st);
}

// The pages' "VM group GEMM": every rank's weights are one contiguous [E+B, H, H']
// tensor and the GEMM addresses them by row index alone. w_views holds the R
// views back to back ([R, E+B, H, H']); with bep_weights_create they alias the
// home rows and the shared slot pool without copies.
cudaError_t launch_grouped_gemm_vm(const Dims& d, const Workspace& ws, const int32_t* cu,
                                   const uint16_t* recv, const uint16_t* w_views, uint16_t* y,
                                   int num_sms, cudaStream_t st) {
    if (d.C == 0) return cudaSuccess;
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    const int BN = pick_bn(d.Hp);
    const bool dual = use_dual(d, d.H, BN);
    CUtensorMap tmA, tmV;
    if (!encode_2d(&tmA, recv, (uint64_t)d.R * d.C, d.H, kBM, kBK)) return cudaErrorInvalidValue;
    if (!encode_2d(&tmV, w_views, (uint64_t)d.R * d.NROW * d.H, d.Hp, kBK, 64))
        return cudaErrorInvalidValue;
    GemmParams prm = {};
    prm.tiles = ws.tiles;
    prm.ntiles = ws.ntiles;
    prm.out = y;
    prm.N = d.Hp;
    prm.Kdim = d.H;
    prm.H = d.H;
    prm.BN = BN;
    prm.tmem_cols = tmem_cols_for(BN);   // two BN-column accumulators (kFwd2: one unit's two)
    prm.mtd = 1;
    prm.vm = 1;
    prm.status = ws.status;
    CUtensorMap tmY;
    if (!encode_2d(&tmY, y, (uint64_t)d.R * d.C, d.Hp, 32, 64)) return cudaErrorInvalidValue;
    if (!dual) {
        gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, 0);
        return launch_mode<kFwd>(tmA, tmV, tmV, tmY, tmY, prm, num_sms, st);
    }
    gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, 3);
    err = launch_mode<kFwd2>(tmA, tmV, tmV, tmY, tmY, prm, num_sms, st);
    if (err != cudaSuccess) return err;
    gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, 4);
    return launch_mode<kFwd>(tmA, tmV, tmV, tmY, tmY, prm, num_sms, st);
}

cudaError_t launch_grouped_gemm_dx(const Dims& d, const Workspace& ws, const int32_t* cu,
                                   const uint16_t* dy, const uint16_t* w_home,
                                   const uint16_t* w_slots, uint16_t* drecv, int num_sms,
                                   cudaStream_t st) {
    if (d.C == 0) return cudaSuccess;
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    const int BN = pick_bn(d.H);
    const bool dual = use_dual(d, d.Hp, BN);
    CUtensorMap tmA, tmBh, tmBs;
    // A: dY [R*C, H'] rows, 64-wide K boxes; B: W rows h (N) x 64 columns h' (K)
    if (!encode_2d(&tmA, dy, (uint64_t)d.R * d.C, d.Hp, kBM, kBK)) return cudaErrorInvalidValue;
    if (!encode_2d(&tmBh, w_home, (uint64_t)d.E * d.H, d.Hp, BN, kBK)) return cudaErrorInvalidValue;
    const uint64_t slot_rows = (uint64_t)(d.R * d.B > 0 ? d.R * d.B : 1) * d.H;
    if (!encode_2d(&tmBs, w_slots ? w_slots : w_home, slot_rows, d.Hp, BN, kBK))
        return cudaErrorInvalidValue;
    GemmParams prm = {};
    prm.tiles = ws.tiles;
    prm.ntiles = ws.ntiles;
    CUtensorMap tmY;   // dRecv [R*C, H] in 32-row x 64-column boxes
    if (!encode_2d(&tmY, drecv, (uint64_t)d.R * d.C, d.H, 32, 64)) return cudaErrorInvalidValue;
    prm.out = drecv;
    prm.N = d.H;
    prm.Kdim = d.Hp;
    prm.H = d.H;
    prm.BN = BN;
    prm.tmem_cols = tmem_cols_for(BN);   // two BN-column accumulators (kDx2: one unit's two)
    prm.mtd = 1;
    prm.status = ws.status;
    if (!dual) {
        gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, 0);
        return launch_mode<kDx>(tmA, tmBh, tmBs, tmY, tmY, prm, num_sms, st);
    }
    // as the forward: long segments two m-tiles per unit, then the others one per unit
    gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, 3);
    err = launch_mode<kDx2>(tmA, tmBh, tmBs, tmY, tmY, prm, num_sms, st);
    if (err != cudaSuccess) return err;
    gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, 4);
    return launch_mode<kDx>(tmA, tmBh, tmBs, tmY, tmY, prm, num_sms, st);
}

cudaError_t launch_grouped_gemm_dw(const Dims& d, const Workspace& ws, const int32_t* cu,
                                   const uint16_t* recv, const uint16_t* dy, float* g_home,
                                   float* red, int accumulate, int num_sms, cudaStream_t st) {
    if (d.C == 0)   // no rows: every home segment is empty
        return accumulate ? cudaSuccess
                          : cudaMemsetAsync(g_home, 0, (size_t)d.E * d.H * d.Hp * sizeof(float), st);
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws, accumulate ? 1 : 2);
    const int BN = pick_bn(d.Hp);
    CUtensorMap tmA, tmB;
    // A: recv^T in 64 (h) x 64 (row) boxes; B: dY in 64 (h') x 64 (row) boxes
    if (!encode_2d(&tmA, recv, (uint64_t)d.R * d.C, d.H, kBK, 64)) return cudaErrorInvalidValue;
    if (!encode_2d(&tmB, dy, (uint64_t)d.R * d.C, d.Hp, kBK, 64)) return cudaErrorInvalidValue;
    // outputs: g_home as [E*H, H'] and red as [R*B*H, H'] fp32 rows
    CUtensorMap tmG, tmR;
    if (!encode_2d_f32(&tmG, g_home, (uint64_t)d.E * d.H, d.Hp)) return cudaErrorInvalidValue;
    const uint64_t red_rows = (uint64_t)(d.R * d.B > 0 ? d.R * d.B : 1) * d.H;
    if (!encode_2d_f32(&tmR, red, red_rows, d.Hp)) return cudaErrorInvalidValue;
    GemmParams prm = {};
    prm.tiles = ws.tiles;
    prm.ntiles = ws.ntiles;
    prm.g_home = g_home;
    prm.red = red;
    prm.N = d.Hp;
    prm.Kdim = 0;
    prm.H = d.H;
    prm.BN = BN;
    prm.tmem_cols = tmem_cols_for(BN);
    prm.mtd = d.H / kBM;
    prm.accumulate = accumulate;
    prm.status = ws.status;
    // SM pairs when the tile divides the gradient: 256 x 256 tiles, six-stage rings
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const int pairs = (dev >= 0 && dev < kMaxDevices) ? g_pair_clusters[dev] : 0;
    if (pairs > 0 && num_sms >= 2 && d.H % kPairBM == 0 && d.Hp % kPairBN == 0) {
        prm.BN = kPairBN;
        prm.tmem_cols = 2 * kPairBN;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = pair_config(pairs < num_sms / 2 ? pairs : num_sms / 2, st, attr);
        return cudaLaunchKernelEx(&cfg, grouped_gemm_dw_pair_kernel, tmA, tmB, tmG, tmR, prm);
    }
    return launch_mode<kDw>(tmA, tmB, tmB, tmG, tmR, prm, num_sms, st);
}

}  // namespace bep
