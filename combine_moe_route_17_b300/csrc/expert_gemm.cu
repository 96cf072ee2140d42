// Expert GEMM on the expert-major recv rows, on the 5th-generation tensor
// cores: out[r] = bf16_RN( sum_h rows[r][h] * W[e(r)][n][h] ), fp32
// accumulation, where e(r) is the expert of row r.  The expert-major layout
// puts every expert's rows in one run (MoE survey, section 1.1, step 2:
// same-expert samples contiguous, then step 3: expert computation), so each
// 128-row tile of a run is one dense [128 x K] x [K x 128] product.
//
// Tiles are 128 rows of one expert's run x BN columns of N (BN = 256 when N
// allows it, else 128).  A persistent grid, one CTA per SM, walks them:
//  - warp 0 (one thread) copies 128x64 and BNx64 bf16 tiles of the rows and
//    of the expert's weights with TMA (cp.async.bulk.tensor, 128-byte
//    swizzle) into a 4-stage shared-memory ring (full / empty mbarriers);
//  - warp 1 (one thread) issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32,
//    M=128, N=BN, K=16 per instruction) into one of two BN-column TMEM
//    accumulators, frees each stage with tcgen05.commit and hands the
//    finished accumulator to the epilogue;
//  - warps 2..5 read that accumulator with tcgen05.ld (warp w owns TMEM lanes
//    32*(w%4).., i.e. rows), round to bf16, store the rows that belong to the
//    expert and hand the accumulator back, while the next tile's MMAs run.
// Every mbarrier wait is bounded; a wait that runs out sets
// MOE_ERR_TIMEOUT, the CTA drains its copies and MMAs in flight, skips the
// rest of its work and still frees TMEM.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is fetched at run time

#include <mutex>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kBM = 128, kBK = 64, kStages = 4;
constexpr uint32_t kTileABytes = kBM * kBK * 2;       // 16 KB
constexpr uint64_t kGemmWaitNs = 2000000000ull;       // 2 s

// Column tile BN (128 or 256): B tile BN x 64, fp32 accumulator in BN TMEM
// columns.
template <int BN>
struct Tile {
    static constexpr uint32_t kTileBBytes = BN * kBK * 2;
    static constexpr uint32_t kStageBytes = kTileABytes + kTileBBytes;
    // Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
    // A and B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
    // N >> 3 in bits 17-22, M >> 4 in bits 24-28.
    static constexpr uint32_t kInstrDesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                           ((uint32_t)(BN >> 3) << 17) |
                                           ((uint32_t)(kBM >> 4) << 24);
};

__device__ __forceinline__ uint32_t sa(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: start address >> 4 (bits 0-13), stride between 8-row
// groups 1024 B >> 4 (bits 32-45), descriptor version 1 (bits 46-47),
// swizzle mode 128 B (value 2 in bits 61-63).  The leading offset is unused
// for this layout.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(1024u >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(n) : "memory");
}

__device__ __forceinline__ void bar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(sa(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of parity `parity` to complete, for at most kGemmWaitNs
// or until another thread of the CTA has given up (*abort set).
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t parity, volatile int* abort) {
    if (bar_try(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!bar_try(b, parity)) {
        if (*abort || globaltimer_ns() - t0 > kGemmWaitNs) return false;
    }
    return true;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(sa(dst)),
        "l"(map), "r"(x), "r"(y), "r"(sa(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     sa(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct GemmArgs {
    const int32_t* counts;  // [E] rows of each expert
    int E, N, K;
    int e_lo, e_hi;         // the experts whose tiles this launch computes
    uint16_t* out;          // [nrows][N]
    uint32_t* err;          // may be NULL
};

// ---------------------------------------------------------------------------
// Persistent form: one CTA per SM walks the tiles t = blockIdx.x, +gridDim.x,
// ... (t = row tile * column tiles + column tile, so the CTAs working at one
// time share their row tiles through L2).  Warp 0 copies, warp 1 issues the
// MMAs into two BN-column TMEM accumulators in turn, warps 2..5 drain the
// other accumulator (warp w reads TMEM lanes 32*(w%4)..+32), so the epilogue
// of one tile runs under the MMAs of the next.  tfull[a] (MMA -> epilogue,
// by tcgen05.commit) and tempty[a] (epilogue -> MMA, one arrival per
// epilogue warp) hand the accumulators over; the shared-memory ring runs on
// across tiles.

constexpr int kPThreads = 192;

template <int BN>
struct PTile {
    static constexpr size_t kTables = 2 * (MOE_MAX_EXPERTS + 1) * sizeof(int);
    static constexpr size_t kSmem = 1024 + kStages * Tile<BN>::kStageBytes + 1024 + kTables;
};

// Largest e in [0, E) with toff[e] <= mt (the expert whose row tiles hold mt;
// empty experts share their successor's start and are skipped).
__device__ __forceinline__ int tile_expert(const int* toff, int E, int mt) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (toff[mid] <= mt) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void bar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}

// SiLU in fp32 (x * logistic(x)), for the gated epilogue.
__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

// EPI = 0: out[row][n0 + c] = bf16(acc[c]).  EPI = 1 (gated, BN = 256): the
// tile's columns are 128 gate columns then the 128 matching up columns, and
// out[row][n0/2 + c] = bf16(silu(acc[c]) * acc[128 + c]), out being N/2 wide.
template <int BN, int EPI>
__global__ void __launch_bounds__(kPThreads, 1)
    expert_gemm_persistent(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, GemmArgs a) {
    static_assert(EPI == 0 || BN == 256, "the gated epilogue pairs two 128-column halves");
    using TL = Tile<BN>;
    constexpr uint32_t kStageBytes = TL::kStageBytes;
    constexpr uint32_t kCols = 2 * BN;  // two accumulators
    grid_dependency_sync();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char* tilesA = smem;
    unsigned char* tilesB = smem + kStages * kTileABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* mdone = tempty + 2;  // every MMA of this CTA has completed
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mdone + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    int* s_total = const_cast<int*>(s_abort + 1);
    int* toff = reinterpret_cast<int*>(smem + kStages * kStageBytes + 1024);  // [E+1] row tiles
    int* roff = toff + MOE_MAX_EXPERTS + 1;                                     // [E+1] rows

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & (kWarp - 1);
    const int ntn = a.N / BN;
    if (warp == 0) {
        // rows of every expert (the layout's offsets), tiles of the experts
        // in [e_lo, e_hi) only: the others get no tile
        int c[8], ct[8], rsum = 0, tsum = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = lane * 8 + q;
            c[q] = e < a.E ? __ldg(a.counts + e) : 0;
            ct[q] = (e >= a.e_lo && e < a.e_hi) ? (c[q] + kBM - 1) / kBM : 0;
            rsum += c[q];
            tsum += ct[q];
        }
        int rinc = rsum, tinc = tsum;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int ru = __shfl_up_sync(kFull, rinc, o), tu = __shfl_up_sync(kFull, tinc, o);
            if (lane >= o) {
                rinc += ru;
                tinc += tu;
            }
        }
        int row = rinc - rsum, t = tinc - tsum;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = lane * 8 + q;
            if (e <= a.E) {
                toff[e] = t;
                roff[e] = row;
            }
            row += c[q];
            t += ct[q];
        }
        if (lane == kWarp - 1) {
            toff[a.E] = tinc;  // E <= 256 = 32 * 8, so entry E may lie past the last lane's 8
            roff[a.E] = rinc;
            *s_total = tinc * ntn;
        }
        if (lane == 0) {
            for (int i = 0; i < kStages; ++i) {
                bar_init(&full[i], 1);
                bar_init(&empty[i], 1);
            }
            for (int i = 0; i < 2; ++i) {
                bar_init(&tfull[i], 1);
                bar_init(&tempty[i], 4);
            }
            bar_init(mdone, 1);
            *s_abort = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    __syncthreads();
    const int total = *s_total;
    if ((int)blockIdx.x >= total) return;  // no tile for this CTA

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sa(s_tmem)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int nk = a.K / kBK;

    if (warp == 0 && lane == 0) {
        // copy thread: the ring runs on across tiles
        int kbg = 0;
        for (int t = blockIdx.x; t < total && !*s_abort; t += gridDim.x) {
            const int mt = t / ntn, n0 = (t % ntn) * BN;
            const int e = tile_expert(toff, a.E, mt);
            const int m0 = roff[e] + (mt - toff[e]) * kBM;
            for (int kb = 0; kb < nk; ++kb, ++kbg) {
                const int st = kbg % kStages;
                const uint32_t ph = (uint32_t)(kbg / kStages) & 1u;
                if (!bar_wait(&empty[st], ph ^ 1u, s_abort)) {
                    *s_abort = 1;
                    break;
                }
                bar_expect_tx(&full[st], kStageBytes);
                tma_load_2d(tilesA + st * kTileABytes, &tmA, kb * kBK, m0, &full[st]);
                tma_load_2d(tilesB + st * TL::kTileBBytes, &tmB, kb * kBK, e * a.N + n0,
                            &full[st]);
            }
        }
        if (*s_abort) {
            // let the copies still in flight (at most one per stage) land
            const int first = kbg > kStages ? kbg - kStages : 0;
            for (int i = first; i < kbg; ++i) {
                const uint64_t t0 = globaltimer_ns();
                while (!bar_try(&full[i % kStages], (uint32_t)(i / kStages) & 1u) &&
                       globaltimer_ns() - t0 < kGemmWaitNs) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // MMA thread
        int kbg = 0, i = 0;
        for (int t = blockIdx.x; t < total && !*s_abort; t += gridDim.x, ++i) {
            const int acc = i & 1;
            const uint32_t aph = (uint32_t)(i >> 1) & 1u;
            if (!bar_wait(&tempty[acc], aph ^ 1u, s_abort)) {
                *s_abort = 1;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * BN);
            for (int kb = 0; kb < nk; ++kb, ++kbg) {
                const int st = kbg % kStages;
                const uint32_t ph = (uint32_t)(kbg / kStages) & 1u;
                if (!bar_wait(&full[st], ph, s_abort)) {
                    *s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t sA = sa(tilesA + st * kTileABytes);
                const uint32_t sB = sa(tilesB + st * TL::kTileBBytes);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                    tc_mma(d, sw128_desc(sA + k * 32), sw128_desc(sB + k * 32), TL::kInstrDesc,
                           (kb > 0 || k > 0) ? 1u : 0u);
                tc_commit(&empty[st]);
            }
            tc_commit(&tfull[acc]);
        }
        // before TMEM is freed: every MMA issued here has completed (bounded)
        tc_commit(mdone);
        const uint64_t t0 = globaltimer_ns();
        while (!bar_try(mdone, 0u) && globaltimer_ns() - t0 < kGemmWaitNs) {
        }
    } else if (warp >= 2) {
        // epilogue warps: lanes 32*(warp%4).. of the accumulator are rows
        const int q = warp & 3;
        int i = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
            const int acc = i & 1;
            const uint32_t aph = (uint32_t)(i >> 1) & 1u;
            const bool ok = bar_wait(&tfull[acc], aph, s_abort);
            __syncwarp();
            if (!ok || *s_abort) {
                if (lane == 0) *s_abort = 1;
                break;
            }
            tc_fence_after();
            const int mt = t / ntn, n0 = (t % ntn) * BN;
            const int e = tile_expert(toff, a.E, mt);
            const int m0 = roff[e] + (mt - toff[e]) * kBM, m_end = roff[e + 1];
            const int row = m0 + q * 32 + lane;
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            if (EPI == 1) {
                uint16_t* orow = a.out + (int64_t)row * (a.N / 2) + n0 / 2;
#pragma unroll 1
                for (int cchunk = 0; cchunk < BN / 64; ++cchunk) {
                    uint32_t g[32], u[32];
                    tc_ld32(tbase + (uint32_t)(cchunk * 32), g);
                    tc_ld32(tbase + (uint32_t)(BN / 2 + cchunk * 32), u);
                    if (row < m_end) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + cchunk * 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            float h[8];
#pragma unroll
                            for (int z = 0; z < 8; ++z)
                                h[z] = silu(__uint_as_float(g[8 * v + z])) *
                                       __uint_as_float(u[8 * v + z]);
                            uint4 o;
                            o.x = pack_bf16x2(h[0], h[1]);
                            o.y = pack_bf16x2(h[2], h[3]);
                            o.z = pack_bf16x2(h[4], h[5]);
                            o.w = pack_bf16x2(h[6], h[7]);
                            dst[v] = o;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) bar_arrive(&tempty[acc]);
                continue;
            }
            uint16_t* orow = a.out + (int64_t)row * a.N + n0;
#pragma unroll 1
            for (int cchunk = 0; cchunk < BN / 32; ++cchunk) {
                uint32_t r[32];
                tc_ld32(tbase + (uint32_t)(cchunk * 32), r);
                if (row < m_end) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + cchunk * 32);
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
            if (lane == 0) bar_arrive(&tempty[acc]);
        }
    }
    __syncthreads();
    if (*s_abort && threadIdx.x == 0 && a.err) raise_error(a.err, MOE_ERR_TIMEOUT, blockIdx.x);
    tc_fence_after();
    __syncwarp();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols)
                     : "memory");
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// 2D map over a row-major bf16 matrix [rows][cols], boxes of box_rows rows x
// 64 columns with the 128-byte swizzle; reads past the last row give zeros.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
              uint32_t box_rows) {
    EncodeTiled fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace
}  // namespace moe

namespace moe {
namespace {

// One persistent launch: out = rows x W^T per expert run, EPI as in the kernel.
moe_status launch_gemm(const moe_shape& s, const uint16_t* rows, int K, const uint16_t* weights,
                       int N, const int32_t* counts, uint16_t* out, void* workspace, int epi,
                       int e_lo, int e_hi, cudaStream_t stream) {
    const int64_t nrows = (int64_t)s.T * s.k;
    const bool wide = epi == 1 || N % 256 == 0;  // 256-column tiles: half the row-tile loads
    const int BN = wide ? 256 : 128;
    CUtensorMap mA, mB;
    if (!make_map(&mA, rows, (uint64_t)nrows, (uint64_t)K, kBM) ||
        !make_map(&mB, weights, (uint64_t)s.E * N, (uint64_t)K, (uint32_t)BN))
        return MOE_ERR_CUDA;
    auto kern = epi == 1 ? expert_gemm_persistent<256, 1>
                         : (wide ? expert_gemm_persistent<256, 0> : expert_gemm_persistent<128, 0>);
    const size_t smem = wide ? PTile<256>::kSmem : PTile<128>::kSmem;
    const moe_status sst = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (sst != MOE_OK) return sst;
    GemmArgs ga;
    ga.counts = counts;
    ga.E = s.E;
    ga.N = N;
    ga.K = K;
    ga.e_lo = e_lo;
    ga.e_hi = e_hi;
    ga.out = out;
    ga.err = workspace ? &ws_ptr<WsHeader>(workspace, 0)->error : nullptr;
    return launch_k(kern, dim3(device_sm_count()), dim3(kPThreads), smem, stream, mA, mB, ga);
}

moe_status check_gemm_shape(const moe_shape& s, int K, int N) {
    if (N < 128 || N % 128 != 0 || K < kBK || K % kBK != 0) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)s.E * N >= ((int64_t)1 << 31) || N > (1 << 20)) return MOE_ERR_UNSUPPORTED;
    const int64_t nrows = (int64_t)s.T * s.k;
    if ((nrows + kBM - 1) / kBM + s.E > (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

namespace moe {
namespace {

// Expert range of wave w (-1: every expert); false if w is out of range.
bool wave_experts(const moe_shape& s, int wave, int& e_lo, int& e_hi) {
    if (wave < -1 || wave >= s.W) return false;
    e_lo = wave < 0 ? 0 : wave * (s.E / s.W);
    e_hi = wave < 0 ? s.E : (wave + 1) * (s.E / s.W);
    return true;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_expert_gemm_wave(const moe_shape* shape, const uint16_t* rows,
                                           const uint16_t* weights, int N,
                                           const int32_t* expert_counts, uint16_t* out, int wave,
                                           void* workspace, cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if ((st = check_gemm_shape(s, s.H, N)) != MOE_OK) return st;
    int e_lo = 0, e_hi = 0;
    if (!wave_experts(s, wave, e_lo, e_hi)) return MOE_ERR_INVALID_ARG;
    if (!weights || !aligned(weights, 16) || !expert_counts || !aligned(expert_counts, 4))
        return MOE_ERR_INVALID_ARG;
    if (!need(rows, s, 16) || !need(out, s, 16)) return MOE_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    return launch_gemm(s, rows, s.H, weights, N, expert_counts, out, workspace, 0, e_lo, e_hi,
                       stream);
}

extern "C" moe_status moe_expert_gemm(const moe_shape* shape, const uint16_t* rows,
                                      const uint16_t* weights, int N,
                                      const int32_t* expert_counts, uint16_t* out,
                                      void* workspace, cudaStream_t stream) {
    return moe_expert_gemm_wave(shape, rows, weights, N, expert_counts, out, -1, workspace,
                                stream);
}

extern "C" moe_status moe_expert_ffn_wave(const moe_shape* shape, const uint16_t* rows,
                                          const uint16_t* w13, const uint16_t* w2, int F,
                                          const int32_t* expert_counts, uint16_t* hidden,
                                          uint16_t* out, int wave, void* workspace,
                                          cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (F < 128 || F % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if ((st = check_gemm_shape(s, s.H, 2 * F)) != MOE_OK) return st;
    if ((st = check_gemm_shape(s, F, s.H)) != MOE_OK) return st;
    if (s.H % 128 != 0) return MOE_ERR_UNSUPPORTED;
    int e_lo = 0, e_hi = 0;
    if (!wave_experts(s, wave, e_lo, e_hi)) return MOE_ERR_INVALID_ARG;
    if (!w13 || !aligned(w13, 16) || !w2 || !aligned(w2, 16) || !expert_counts ||
        !aligned(expert_counts, 4))
        return MOE_ERR_INVALID_ARG;
    if (!need(rows, s, 16) || !need(hidden, s, 16) || !need(out, s, 16))
        return MOE_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    // hidden = silu(x W1^T) * (x W3^T): w13 holds, per expert, F/128 blocks of
    // 256 rows (128 rows of W1, then the same 128 rows of W3)
    st = launch_gemm(s, rows, s.H, w13, 2 * F, expert_counts, hidden, workspace, 1, e_lo, e_hi,
                     stream);
    if (st != MOE_OK) return st;
    // out = hidden W2^T
    return launch_gemm(s, hidden, F, w2, s.H, expert_counts, out, workspace, 0, e_lo, e_hi,
                       stream);
}

extern "C" moe_status moe_expert_ffn(const moe_shape* shape, const uint16_t* rows,
                                     const uint16_t* w13, const uint16_t* w2, int F,
                                     const int32_t* expert_counts, uint16_t* hidden,
                                     uint16_t* out, void* workspace, cudaStream_t stream) {
    return moe_expert_ffn_wave(shape, rows, w13, w2, F, expert_counts, hidden, out, -1,
                               workspace, stream);
}
