// Grouped expert GEMM over one [E+B, H, H'] weight tensor (sm_103a, tcgen05).
//
// MoonEP pages (ai-maestro.online), "The memory contract": the group GEMM
// consumes a single [E+B, H, H'] weight tensor and addresses experts purely by
// row index; cu_seqlens from the planner selects the active rows. Rows [0, E)
// are the home experts, rows [E, E+B) a rank's prefetch slots; overflow
// experts (inference) are read from their home rows.
//
// Design (one GB300):
//   * a one-CTA prep kernel turns cu_seqlens [R, E+B+1] into a list of m-tiles
//     (128 receive rows sharing one weight row); the host never learns the
//     segment sizes (no host synchronisation);
//   * a persistent kernel, one CTA per SM, strides over (m-tile, n-tile) work
//     units, n fastest so that neighbouring CTAs share the A tile and a weight
//     row's column blocks stay in L2 while its m-tiles pass;
//   * warp 0 issues TMA loads (A: 128 x 64 bf16, K-major, 128-byte swizzle;
//     B: 64 x BN bf16 in 64-column chunks, N contiguous = MN-major, 128-byte
//     swizzle) into a 4-stage shared-memory ring guarded by mbarriers;
//   * warp 1 (one thread) issues tcgen05.mma.kind::f16 (M=128, N=BN, K=16,
//     bf16 in, fp32 accumulate) into one of two TMEM accumulators, and
//     tcgen05.commit frees each stage and publishes each finished tile;
//   * warps 2..5 drain the other accumulator (tcgen05.ld 32x32b), round to
//     bf16 (nearest even) and store only the rows inside the segment, so a
//     tile never writes into the next segment.
// Every mbarrier wait is bounded (2 s on the global timer); on expiry the CTA
// records BEP_DERR_TIMEOUT, every role leaves its loop, and TMEM is freed.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "bep_internal.cuh"

namespace bep {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBChunkBytes = 64 * kBK * 2;      // 8 KB: 64 K-rows x 64 N columns
constexpr uint64_t kTimeoutNs = 2000000000ull;

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
                                          int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kTimeoutNs) {
            *abort_flag = 1;
            set_status(status, BEP_DERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
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

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B MN-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
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

// ---------------------------------------------------------------- tile list
__global__ void __launch_bounds__(1024) gemm_tiles_kernel(const int32_t* __restrict__ cu, Dims d,
                                                          Workspace ws) {
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
        return (b - a + kBM - 1) / kBM;
    };
    int sum = 0;
    for (int i = lo; i < hi; ++i) {
        int s, l;
        sum += tiles_of(i, &s, &l);
    }
    // block exclusive scan
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
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
    int run = s_warp[warp] + incl - sum;
    const int total = s_warp[32];
    if (total > d.max_tiles) bad = 1;
    for (int i = lo; i < hi && total <= d.max_tiles; ++i) {
        int s = 0, l = 0;
        const int n = tiles_of(i, &s, &l);
        const int u = i / d.NROW, rho = i % d.NROW;
        const int wsel = rho < d.E ? rho : -(1 + u * d.B + (rho - d.E));
        for (int m = 0; m < n; ++m) {
            MTile t;
            t.row0 = (int32_t)(u * d.C + s + m * kBM);
            t.rows = min(kBM, l - m * kBM);
            t.wsel = wsel;
            t.pad = 0;
            ws.tiles[run + m] = t;
        }
        run += n;
    }
    if (bad) set_status(ws.status, BEP_DERR_BOUNDS);
    if (threadIdx.x == 0) *ws.ntiles = total <= d.max_tiles ? total : 0;
}

// ---------------------------------------------------------------- the GEMM
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmBh,
    const __grid_constant__ CUtensorMap tmBs, const MTile* __restrict__ tiles,
    const int32_t* __restrict__ ntiles_ptr, uint16_t* __restrict__ y, int H, int Hp, int BN,
    int tmem_cols, int32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned carve-up: A ring, B ring, barriers
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int b_bytes = BN * kBK * 2;
    uint8_t* smA = smem;
    uint8_t* smB = smem + kStages * kABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smB + kStages * b_bytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* tfull = bars + 2 * kStages;
    uint64_t* tempty = bars + 2 * kStages + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(s_tmem)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    const int ntiles = *ntiles_ptr;
    const int NT = Hp / BN;
    const int total = ntiles * NT;
    const int KB = H / kBK;
    const uint32_t stage_bytes = (uint32_t)(kABytes + b_bytes);
    const int acc_stride = tmem_cols / 2;   // two accumulators, power-of-two spaced columns

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
            uint32_t s = 0, ph = 0;
            bool live = true;
            for (int unit = blockIdx.x; unit < total && live; unit += gridDim.x) {
                const int mt = unit / NT, nt = unit - (unit / NT) * NT;
                const MTile t = tiles[mt];
                const CUtensorMap* tmB = t.wsel >= 0 ? &tmBh : &tmBs;
                const int brow0 = (t.wsel >= 0 ? t.wsel : (-1 - t.wsel)) * H;
                const int n0 = nt * BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, s_abort, status)) {
                        live = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], stage_bytes);
                    tma_load_2d(&tmA, &full[s], smA + s * kABytes, kb * kBK, t.row0);
                    for (int c = 0; c < BN / 64; ++c)
                        tma_load_2d(tmB, &full[s], smB + s * b_bytes + c * kBChunkBytes, n0 + c * 64,
                                    brow0 + kb * kBK);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_bf16(kBM, BN);
            uint32_t s = 0, ph = 0;
            bool live = true;
            int it = 0;
            for (int unit = blockIdx.x; unit < total && live; unit += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!mbar_wait(&tempty[acc], aph ^ 1u, s_abort, status)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(acc * acc_stride);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[s], ph, s_abort, status)) {
                        live = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smA + s * kABytes);
                    const uint32_t b0 = smem_u32(smB + s * b_bytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // A: K-major, advance 16 elements (32 B) inside the 128-byte swizzle row.
                        // B: MN-major, advance 16 K-rows = two 8-row groups of 1024 B.
                        const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(b0 + kk * 2048, kBChunkBytes, 1024);
                        mma_bf16(dt, ad, bd, idesc, (kb | kk) != 0);
                    }
                    mma_commit(&empty[s]);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (live) mma_commit(&tfull[acc]);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue (warps 2..5)
        const int q = warp & 3;   // TMEM lanes 32q..32q+31 are this warp's
        int it = 0;
        for (int unit = blockIdx.x; unit < total; unit += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            const bool got = mbar_wait(&tfull[acc], aph, s_abort, status);
            __syncwarp();
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const int mt = unit / NT, nt = unit - (unit / NT) * NT;
            const MTile t = tiles[mt];
            const int row = q * 32 + lane;
            const bool valid = row < t.rows;
            uint16_t* yrow = y + (int64_t)(t.row0 + row) * Hp + (int64_t)nt * BN;
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * acc_stride + c0), r);
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(yrow + c0);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                        o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                        o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                        o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                        dst[v] = o;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }

    __syncthreads();
    if (*s_abort) {
        // let copies and MMAs that were already issued land before the memory goes away
        for (int i = 0; i < 100; ++i) __nanosleep(10000);
    }
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(tmem_cols)
                     : "memory");
    }
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

int pick_bn(int Hp) {
    for (int bn = 256; bn >= 64; bn -= 64)
        if (Hp % bn == 0) return bn;
    return 64;
}

size_t smem_bytes(int BN) {
    return 1024 + (size_t)kStages * (kABytes + BN * kBK * 2) + (2 * kStages + 4) * 8 + 16;
}

}  // namespace

cudaError_t gemm_setup(int device) {
    (void)device;
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    return cudaFuncSetAttribute(grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes(256));
}

cudaError_t launch_grouped_gemm(const Dims& d, const Workspace& ws, const int32_t* cu,
                                const uint16_t* recv, const uint16_t* w_home,
                                const uint16_t* w_slots, uint16_t* y, int num_sms,
                                cudaStream_t st) {
    if (d.C == 0) return cudaSuccess;
    cudaError_t err = get_encoder();
    if (err != cudaSuccess) return err;
    gemm_tiles_kernel<<<1, 1024, 0, st>>>(cu, d, ws);
    const int BN = pick_bn(d.Hp);
    CUtensorMap tmA, tmBh, tmBs;
    if (!encode_2d(&tmA, recv, (uint64_t)d.R * d.C, d.H, kBM, kBK)) return cudaErrorInvalidValue;
    if (!encode_2d(&tmBh, w_home, (uint64_t)d.E * d.H, d.Hp, kBK, 64)) return cudaErrorInvalidValue;
    const uint64_t slot_rows = (uint64_t)(d.R * d.B > 0 ? d.R * d.B : 1) * d.H;
    if (!encode_2d(&tmBs, w_slots ? w_slots : w_home, slot_rows, d.Hp, kBK, 64))
        return cudaErrorInvalidValue;
    int tmem_cols = 32;
    while (tmem_cols < 2 * BN) tmem_cols <<= 1;
    grouped_gemm_kernel<<<num_sms, kThreads, smem_bytes(BN), st>>>(
        tmA, tmBh, tmBs, ws.tiles, ws.ntiles, y, d.H, d.Hp, BN, tmem_cols, ws.status);
    return cudaGetLastError();
}

}  // namespace bep
