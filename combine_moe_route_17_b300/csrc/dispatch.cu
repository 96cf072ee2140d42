// Dispatch: permute token rows by destination and exchange them
// ("混合专家模型跨卡通信机制解析", section 四: permute_by_device, then
// all_to_all), with same-expert rows contiguous (MoE survey, section 1.1,
// step 2) and the exchange cut into W waves of E/W experts ("不规则与流水化
// AllToAll", section "Wave-Scheduled 流水化").
//
// With the R ranks living in one GPU's memory, the fused form writes every
// token row straight into its recv rows: one warp per token reads the row
// once (16-byte vectors, no L1 allocation) and stores it to each of its
// selected rows of the requested wave.  The staged form first writes the send
// layout (the local permute), then moves each (source, wave) run of send rows
// to the recv layout (the exchange), which is a data-dependent block
// transpose of contiguous row runs.
#include <math.h>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kRowWarps = 8;
constexpr int kVecUnroll = 8;  // 16-byte vectors in flight per lane

struct ScatterArgs {
    const uint4* x;
    const int32_t* idx;
    const int32_t* rank;
    const int32_t* table;  // first dst row of (source, expert): rstart or sstart
    const int32_t* rtable; // rstart, for the optional recv-row map of the permute
    int64_t T, Tr, nrows;
    int H8, E, k, Ew, wave;
    int reverse;        // walk tokens from the last one down
    int keep_x;         // x rows are read again by a later wave call: keep them in L2
    int expert_major;   // recv rows ordered (rank, expert, source, token, slot)
    const int32_t* eoff;  // first row of each expert (expert-major)
    const int32_t* cpre;  // slots of expert e in the sources before s
    uint4* dst;         // NULL: write the maps only
    int32_t* dst_map;   // slot_of (fused) or send_pos (permute)
    int32_t* src_row;   // token of each recv row (fused only), may be NULL
    int32_t* slot_of;   // permute only: recv row of (t, j), may be NULL
    uint32_t* err;
};

// Loads batch `base` of the x row: kVecUnroll 16-byte vectors per lane.
__device__ __forceinline__ void load_x_batch(const uint4* __restrict__ src, int H8, int base,
                                             int lane, uint64_t ld_pol, uint4 (&v)[kVecUnroll]) {
#pragma unroll
    for (int u = 0; u < kVecUnroll; ++u) {
        const int p = base + u * kWarp + lane;
        if (p < H8) v[u] = ld_nc_v4_hint(src + p, ld_pol);
    }
}

// Stores the x row to every row of `mask` (row of slot j in lane j); v holds
// its first batch, already loaded.
__device__ __forceinline__ void copy_row_to_many(const uint4* __restrict__ src, uint4* dst_base,
                                                 int H8, unsigned mask, int32_t row, int lane,
                                                 uint64_t ld_pol, uint64_t st_pol,
                                                 uint4 (&v)[kVecUnroll]) {
    for (int base = 0; base < H8; base += kWarp * kVecUnroll) {
        if (base > 0) load_x_batch(src, H8, base, lane, ld_pol, v);
        for (unsigned m = mask; m; m &= m - 1) {
            const int j = __ffs(m) - 1;
            const int32_t r = __shfl_sync(kFull, row, j);
            uint4* d = dst_base + (int64_t)r * H8;
#pragma unroll
            for (int u = 0; u < kVecUnroll; ++u) {
                const int p = base + u * kWarp + lane;
                if (p < H8) st_v4_hint(d + p, v[u], st_pol);
            }
        }
    }
}

// Slot (t, lane) of this call, first half: lanes j < k load token t's j-th
// expert and, for a slot of the call's wave, its rank inside (source,
// expert); returns whether the slot belongs to the wave.  A bad expert index
// sets the error word and the slot is skipped.
__device__ __forceinline__ bool slot_expert(const ScatterArgs& a, int64_t t, int lane, int& e,
                                            int32_t& r) {
    if (lane >= a.k) return false;
    const int64_t sl = t * a.k + lane;
    e = __ldg(a.idx + sl);
    if (e < 0 || e >= a.E) {
        raise_error(a.err, MOE_ERR_DEVICE_CHECK, (uint32_t)sl);
        return false;
    }
    if (a.wave >= 0 && e / a.Ew != a.wave) return false;
    r = __ldg(a.rank + sl);  // read in slot_row, after the caller's x loads are issued
    return true;
}

// Second half: the slot's row (first row of (source, expert) plus its rank),
// and its maps.  A row out of range sets the error word and the slot is
// skipped.
template <bool TO_SEND>
__device__ __forceinline__ bool slot_row(const ScatterArgs& a, int64_t t, int lane, int e,
                                         int32_t r, int32_t& row) {
    const int64_t s = t / a.Tr;
    const int64_t sl = t * a.k + lane;
    const int64_t rw = (!TO_SEND && a.expert_major)
                           ? (int64_t)__ldg(a.eoff + e) + __ldg(a.cpre + s * a.E + e) + r
                           : (int64_t)__ldg(a.table + s * a.E + e) + r;
    if (rw < 0 || rw >= a.nrows) {
        raise_error(a.err, MOE_ERR_DEVICE_CHECK, (uint32_t)sl);
        return false;
    }
    row = (int32_t)rw;
    a.dst_map[sl] = row;
    if (!TO_SEND && a.src_row) a.src_row[rw] = (int32_t)t;
    if (TO_SEND && a.slot_of) {
        const int64_t rr = a.expert_major
                               ? (int64_t)__ldg(a.eoff + e) + __ldg(a.cpre + s * a.E + e) + r
                               : (int64_t)__ldg(a.rtable + s * a.E + e) + r;
        if (rr >= 0 && rr < a.nrows) a.slot_of[sl] = (int32_t)rr;
    }
    return true;
}

// Both halves: whether slot (t, lane) belongs to the call's wave, and its row.
template <bool TO_SEND>
__device__ __forceinline__ bool resolve_slot(const ScatterArgs& a, int64_t t, int lane,
                                             int32_t& row) {
    int e = 0;
    int32_t r = 0;
    return slot_expert(a, t, lane, e, r) && slot_row<TO_SEND>(a, t, lane, e, r, row);
}

// Register path: one warp per token reads its x row once (16-byte vectors,
// kVecUnroll in flight per lane) and stores it to each of its rows of the wave.
// Once the wave's slots are known, the row's first batch is loaded while
// their ranks and first rows are looked up.
template <bool TO_SEND>
__global__ void __launch_bounds__(kRowWarps* kWarp) scatter_rows_kernel(ScatterArgs a) {
    grid_dependency_sync();
    const int lane = threadIdx.x & (kWarp - 1);
    const int64_t nw = (int64_t)gridDim.x * kRowWarps;
    const uint64_t ld_pol = a.keep_x ? l2_policy_evict_last() : l2_policy_evict_first();
    const uint64_t st_pol = l2_policy_evict_first();
    for (int64_t i = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5); i < a.T; i += nw) {
        const int64_t t = a.reverse ? a.T - 1 - i : i;
        int e = 0;
        int32_t r = 0;
        const bool in_wave = slot_expert(a, t, lane, e, r);
        if (!__ballot_sync(kFull, in_wave)) continue;
        const uint4* src = a.x + t * a.H8;
        uint4 v[kVecUnroll];
        if (a.dst) load_x_batch(src, a.H8, 0, lane, ld_pol, v);
        int32_t row = 0;
        const bool mine = in_wave && slot_row<TO_SEND>(a, t, lane, e, r, row);
        const unsigned mask = __ballot_sync(kFull, mine);
        if (mask && a.dst)
            copy_row_to_many(src, a.dst, a.H8, mask, row, lane, ld_pol, st_pol, v);
    }
}

// ---------------------------------------------------------------------------
// Bulk-copy path (MOE_BULK_COPY): the row copies staged through shared memory
// by the bulk-copy engine instead of registers.  One warp per token resolves
// the rows as above; its lane 0 then moves the x row global -> shared with one
// cp.async.bulk (completion on an mbarrier) and shared -> global to each row
// of the wave with bulk stores (one bulk group per token).  Three row buffers
// per warp keep the next token's load in flight while the two tokens before
// it store; a buffer is refilled only once the stores that read it have
// finished reading (cp.async.bulk.wait_group.read).  Every mbarrier wait is
// bounded; one that runs out raises MOE_ERR_TIMEOUT and the warp stops
// issuing copies, after giving the load in flight a second bounded wait.

constexpr int kBulkSlots = 3;                   // row buffers per warp
constexpr int kBulkMaxWarps = 8;                // warps per CTA at most
constexpr size_t kBulkSmemBudget = 200 * 1024;  // row buffers of one CTA
constexpr uint64_t kBulkWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits (bounded) for the phase of `parity` of barrier b to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try(b, parity))
        if (globaltimer_ns() - t0 > kBulkWaitNs) return false;
    return true;
}

__device__ __forceinline__ void bulk_load_row(void* sdst, const void* gsrc, uint32_t bytes,
                                              uint64_t* bar, uint64_t pol) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void bulk_store_row(void* gdst, const void* ssrc, uint32_t bytes,
                                               uint64_t pol) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::
                     "l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes), "l"(pol)
                 : "memory");
}

template <bool TO_SEND>
__global__ void __launch_bounds__(kBulkMaxWarps* kWarp) scatter_rows_bulk_kernel(ScatterArgs a) {
    grid_dependency_sync();
    extern __shared__ __align__(128) unsigned char bulk_smem[];
    __shared__ __align__(8) uint64_t bars[kBulkMaxWarps][kBulkSlots];
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t row_bytes = (uint32_t)a.H8 * 16u;
    unsigned char* buf = bulk_smem + (size_t)warp * kBulkSlots * row_bytes;
    if (lane == 0) {
        for (int q = 0; q < kBulkSlots; ++q)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[warp][q]))
                         : "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    const uint64_t ld_pol = a.keep_x ? l2_policy_evict_last() : l2_policy_evict_first();
    const uint64_t st_pol = l2_policy_evict_first();
    const int64_t nw = (int64_t)gridDim.x * nwarps;
    uint32_t phase = 0;       // parity bit of each slot's next completion (lane 0)
    int slot = 0;             // buffer of the next load
    int p_slot = -1;          // buffer of the token whose load is in flight
    unsigned p_mask = 0;      // its slots in the wave
    int32_t p_row = 0;        // its row, lane j holding slot j
    bool ok = true;           // no wait has run out
    for (int64_t i = (int64_t)blockIdx.x * nwarps + warp;; i += nw) {
        const bool have = i < a.T;
        unsigned mask = 0;
        int32_t row = 0;
        int64_t t = 0;
        if (have) {
            t = a.reverse ? a.T - 1 - i : i;
            const bool mine = resolve_slot<TO_SEND>(a, t, lane, row);
            mask = __ballot_sync(kFull, mine);
        }
        if (!a.dst) {
            if (!have) break;
            continue;
        }
        // start this token's load: its buffer was last read by the stores of
        // the token three loads back; of the groups committed so far only the
        // newest (two loads back) may still be reading
        if (have && mask) {
            if (lane == 0 && ok) {
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                bulk_load_row(buf + (size_t)slot * row_bytes, a.x + t * a.H8, row_bytes,
                              &bars[warp][slot], ld_pol);
            }
        }
        // finish the previous token: wait for its row, store it to its rows
        if (p_slot >= 0) {
            if (lane == 0 && ok) {
                ok = mbar_wait(&bars[warp][p_slot], (phase >> p_slot) & 1u);
                if (!ok) {
                    raise_error(a.err, MOE_ERR_TIMEOUT, (uint32_t)i);
                    // no more copies; the late load still has to land before
                    // the buffers can go
                    mbar_wait(&bars[warp][p_slot], (phase >> p_slot) & 1u);
                }
                phase ^= 1u << p_slot;
            }
            const bool go = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            for (unsigned m = p_mask; m; m &= m - 1) {
                const int32_t r = __shfl_sync(kFull, p_row, __ffs(m) - 1);
                if (lane == 0 && go)
                    bulk_store_row(a.dst + (int64_t)r * a.H8, buf + (size_t)p_slot * row_bytes,
                                   row_bytes, st_pol);
            }
            if (lane == 0 && go) asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            p_slot = -1;
        }
        if (have && mask) {
            p_slot = slot;
            p_mask = mask;
            p_row = row;
            slot = slot + 1 == kBulkSlots ? 0 : slot + 1;
        }
        if (!have) break;
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Capacity-factor dispatch (MoE survey, section 1.1, eq. 3 and step 2): a
// fixed [E][EC][H] buffer.  The slots of expert e are counted over all
// sources in (token, slot) order; a slot's position is the count of earlier
// sources (cpre) plus its rank inside its source; the first EC positions are
// kept at row e*EC + position, later slots are dropped (cap_slot = -1), and
// the rows an expert does not fill are zeroed.

struct CapArgs {
    const uint4* x;
    const int32_t* idx;
    const int32_t* rank;
    const int32_t* cpre;     // [R][E]
    const int32_t* cnt_se;   // [R][E]
    int64_t T, Tr, EC, ncap;  // ncap = E * EC rows
    int H8, E, k, R;
    uint4* rows;
    int32_t* cap_slot;
    int32_t* dropped;  // [E], may be NULL
    uint32_t* err;
};

__global__ void __launch_bounds__(kRowWarps* kWarp) capacity_scatter_kernel(CapArgs a) {
    grid_dependency_sync();
    const int lane = threadIdx.x & (kWarp - 1);
    const int64_t nw = (int64_t)gridDim.x * kRowWarps;
    const uint64_t pol = l2_policy_evict_first();
    for (int64_t t = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5); t < a.T; t += nw) {
        const int64_t s = t / a.Tr;
        int32_t row = 0;
        bool kept = false;
        if (lane < a.k) {
            const int64_t sl = t * a.k + lane;
            const int e = __ldg(a.idx + sl);
            int32_t slot = -1;
            if (e < 0 || e >= a.E) {
                raise_error(a.err, MOE_ERR_DEVICE_CHECK, (uint32_t)sl);
            } else {
                const int64_t pos = (int64_t)__ldg(a.cpre + s * a.E + e) + __ldg(a.rank + sl);
                if (pos < a.EC) {
                    const int64_t rw = (int64_t)e * a.EC + pos;
                    if (pos >= 0 && rw < a.ncap) {
                        row = (int32_t)rw;
                        slot = row;
                        kept = true;
                    } else {
                        raise_error(a.err, MOE_ERR_DEVICE_CHECK, (uint32_t)sl);
                    }
                }
            }
            a.cap_slot[sl] = slot;
        }
        const unsigned mask = __ballot_sync(kFull, kept);
        if (mask) {
            uint4 v[kVecUnroll];
            load_x_batch(a.x + t * a.H8, a.H8, 0, lane, pol, v);
            copy_row_to_many(a.x + t * a.H8, a.rows, a.H8, mask, row, lane, pol, pol, v);
        }
    }
}

// Zeroes the rows [c_e, EC) of every expert e (blockIdx.y) and writes the
// dropped count max(c_e - EC, 0).
__global__ void __launch_bounds__(kRowWarps* kWarp) capacity_pad_kernel(CapArgs a) {
    grid_dependency_sync();
    const int e = blockIdx.y;
    const int lane = threadIdx.x & (kWarp - 1);
    const int64_t last = (int64_t)(a.R - 1) * a.E + e;
    const int64_t ce = (int64_t)__ldg(a.cpre + last) + __ldg(a.cnt_se + last);
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.dropped)
        a.dropped[e] = (int32_t)(ce > a.EC ? ce - a.EC : 0);
    const int64_t nw = (int64_t)gridDim.x * kRowWarps;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const uint64_t pol = l2_policy_evict_first();
    for (int64_t p = ce + (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5); p < a.EC; p += nw) {
        uint4* d = a.rows + ((int64_t)e * a.EC + p) * a.H8;
        for (int q = lane; q < a.H8; q += kWarp) st_v4_hint(d + q, zero, pol);
    }
}

struct ExchangeArgs {
    const uint4* src;
    uint4* dst;
    const int32_t* cnt_se;
    const int32_t* sstart;
    const int32_t* rstart;
    int64_t nrows;
    int E, H8, e_lo, e_hi, direction;
    int expert_major;
    const int32_t* eoff;
    const int32_t* cpre;
    uint32_t* err;
};

// blockIdx.y = source rank s.  The send rows of the wave's experts form one
// contiguous run of source s; each row's expert is found by binary search in
// the run's per-expert start table and mapped to its recv row.
__global__ void __launch_bounds__(kRowWarps* kWarp) exchange_kernel(ExchangeArgs a) {
    grid_dependency_sync();
    __shared__ int32_t s_ss[MOE_MAX_EXPERTS];
    __shared__ int32_t s_rs[MOE_MAX_EXPERTS];
    const int s = blockIdx.y;
    const int ne = a.e_hi - a.e_lo;
    for (int i = threadIdx.x; i < ne; i += blockDim.x) {
        const int e = a.e_lo + i;
        s_ss[i] = a.sstart[s * a.E + e];
        s_rs[i] = a.expert_major ? a.eoff[e] + a.cpre[s * a.E + e] : a.rstart[s * a.E + e];
    }
    __syncthreads();
    const int64_t first = s_ss[0];
    const int64_t nrun = (int64_t)a.sstart[s * a.E + a.e_hi - 1] +
                         a.cnt_se[s * a.E + a.e_hi - 1] - first;
    const int lane = threadIdx.x & (kWarp - 1);
    const int64_t nw = (int64_t)gridDim.x * kRowWarps;
    for (int64_t i = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5); i < nrun; i += nw) {
        const int64_t sr = first + i;
        int lo = 0, hi = ne;  // largest q with s_ss[q] <= sr
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_ss[mid] <= sr) lo = mid;
            else hi = mid;
        }
        const int64_t rr = (int64_t)s_rs[lo] + (sr - s_ss[lo]);
        if (sr < 0 || sr >= a.nrows || rr < 0 || rr >= a.nrows) {
            if (lane == 0) raise_error(a.err, MOE_ERR_DEVICE_CHECK, (uint32_t)sr);
            continue;
        }
        const int64_t from = a.direction == 0 ? sr : rr;
        const int64_t to = a.direction == 0 ? rr : sr;
        const uint4* src = a.src + from * a.H8;
        uint4* dst = a.dst + to * a.H8;
        for (int base = 0; base < a.H8; base += kWarp * kVecUnroll) {
            uint4 v[kVecUnroll];
#pragma unroll
            for (int u = 0; u < kVecUnroll; ++u) {
                const int p = base + u * kWarp + lane;
                if (p < a.H8) v[u] = ld_nc_v4(src + p);
            }
#pragma unroll
            for (int u = 0; u < kVecUnroll; ++u) {
                const int p = base + u * kWarp + lane;
                if (p < a.H8) st_v4(dst + p, v[u]);
            }
        }
    }
}

moe_status check_ws(const moe_shape& s, const void* ws, size_t ws_bytes, WsLayout& L) {
    L = ws_layout(s);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// Geometry of the bulk-copy scatter for rows of row_bytes: warps per CTA (as
// many as kBulkSlots row buffers each fit in the shared-memory budget, at most
// kBulkMaxWarps; 0 if not even one warp's buffers fit) and its shared memory.
int bulk_warps(size_t row_bytes) {
    const size_t per_warp = (size_t)kBulkSlots * row_bytes;
    const size_t n = per_warp ? kBulkSmemBudget / per_warp : 0;
    return (int)(n > (size_t)kBulkMaxWarps ? kBulkMaxWarps : n);
}

moe_status launch_scatter_bulk(const ScatterArgs& a, bool to_send, int64_t T, cudaStream_t stream) {
    const size_t row_bytes = (size_t)a.H8 * 16;
    const int nwarps = bulk_warps(row_bytes);
    if (nwarps < 1) return MOE_ERR_UNSUPPORTED;
    const size_t smem = (size_t)nwarps * kBulkSlots * row_bytes;
    const void* kern = to_send ? reinterpret_cast<const void*>(scatter_rows_bulk_kernel<true>)
                               : reinterpret_cast<const void*>(scatter_rows_bulk_kernel<false>);
    moe_status st = ensure_dynamic_smem(kern, smem);
    if (st != MOE_OK) return st;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nwarps * kWarp, smem) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    // persistent: every resident CTA walks the tokens, a warp per token
    const int grid = grid_for(T, nwarps, (int64_t)per_sm * device_sm_count());
    const dim3 block(nwarps * kWarp);
    return to_send ? launch_k(scatter_rows_bulk_kernel<true>, dim3(grid), block, smem, stream, a)
                   : launch_k(scatter_rows_bulk_kernel<false>, dim3(grid), block, smem, stream, a);
}

moe_status launch_scatter(const moe_shape& s, const WsLayout& L, const void* ws, const uint16_t* x,
                          const int32_t* idx, int wave, bool to_send, uint16_t* dst,
                          int32_t* dst_map, int32_t* src_row, int32_t* slot_of,
                          cudaStream_t stream, bool expert_major = false, bool bulk = false) {
    ScatterArgs a;
    a.x = reinterpret_cast<const uint4*>(x);
    a.idx = idx;
    a.rank = ws_ptr<int32_t>(ws, L.rank);
    a.table = ws_ptr<int32_t>(ws, to_send ? L.sstart : L.rstart);
    a.rtable = ws_ptr<int32_t>(ws, L.rstart);
    a.T = s.T;
    a.Tr = s.T / s.R;
    a.nrows = (int64_t)s.T * s.k;
    a.H8 = s.H / 8;
    a.E = s.E;
    a.k = s.k;
    a.Ew = s.E / s.W;
    a.wave = wave;
    // Wave calls come in order 0..W-1 and each reads the x rows of its
    // tokens: odd waves walk the tokens backwards, so a wave starts on the
    // rows the previous one read last, and every wave but the last keeps the
    // rows it reads in L2 (evict_last) for the next.
    a.reverse = (wave > 0 && (wave & 1)) ? 1 : 0;
    a.keep_x = (wave >= 0 && wave < s.W - 1) ? 1 : 0;
    a.expert_major = expert_major ? 1 : 0;
    a.eoff = ws_ptr<int32_t>(ws, L.eoff);
    a.cpre = ws_ptr<int32_t>(ws, L.cpre);
    a.dst = reinterpret_cast<uint4*>(dst);
    a.dst_map = dst_map;
    a.src_row = src_row;
    a.slot_of = slot_of;
    a.err = &const_cast<WsHeader*>(ws_ptr<WsHeader>(ws, 0))->error;
    if (bulk && dst) return launch_scatter_bulk(a, to_send, s.T, stream);
    const dim3 grid(grid_for(s.T, kRowWarps)), block(kRowWarps * kWarp);
    return to_send ? launch_k(scatter_rows_kernel<true>, grid, block, 0, stream, a)
                   : launch_k(scatter_rows_kernel<false>, grid, block, 0, stream, a);
}

moe_status launch_exchange(const moe_shape& s, const WsLayout& L, const void* ws, int wave,
                           int direction, const uint16_t* src, uint16_t* dst,
                           cudaStream_t stream, bool expert_major = false) {
    ExchangeArgs a;
    a.src = reinterpret_cast<const uint4*>(src);
    a.dst = reinterpret_cast<uint4*>(dst);
    a.cnt_se = ws_ptr<int32_t>(ws, L.cnt_se);
    a.sstart = ws_ptr<int32_t>(ws, L.sstart);
    a.rstart = ws_ptr<int32_t>(ws, L.rstart);
    a.nrows = (int64_t)s.T * s.k;
    a.E = s.E;
    a.H8 = s.H / 8;
    const int Ew = s.E / s.W;
    a.e_lo = wave < 0 ? 0 : wave * Ew;
    a.e_hi = wave < 0 ? s.E : (wave + 1) * Ew;
    a.direction = direction;
    a.expert_major = expert_major ? 1 : 0;
    a.eoff = ws_ptr<int32_t>(ws, L.eoff);
    a.cpre = ws_ptr<int32_t>(ws, L.cpre);
    a.err = &const_cast<WsHeader*>(ws_ptr<WsHeader>(ws, 0))->error;
    int gx = (device_sm_count() * 8 + s.R - 1) / s.R;
    const int64_t per_src = ((int64_t)(s.T / s.R) * s.k + kRowWarps - 1) / kRowWarps;
    if (gx > per_src) gx = (int)(per_src > 0 ? per_src : 1);
    dim3 grid(gx, s.R);
    return launch_k(exchange_kernel, grid, dim3(kRowWarps * kWarp), 0, stream, a);
}

}  // namespace

moe_status exchange_rows(const moe_shape& s, const void* ws, size_t ws_bytes, int wave,
                         int direction, const uint16_t* src, uint16_t* dst, cudaStream_t stream,
                         bool expert_major) {
    WsLayout L;
    moe_status st = check_ws(s, ws, ws_bytes, L);
    if (st != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;
    return launch_exchange(s, L, ws, wave, direction, src, dst, stream, expert_major);
}

}  // namespace moe

extern "C" moe_status moe_permute_by_device(const moe_shape* shape, const uint16_t* x,
                                            const int32_t* idx, const void* workspace,
                                            size_t ws_bytes, int wave, uint16_t* send,
                                            int32_t* send_pos, int32_t* slot_of,
                                            cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    WsLayout L;
    if ((st = check_ws(s, workspace, ws_bytes, L)) != MOE_OK) return st;
    if (wave < -1 || wave >= s.W) return MOE_ERR_INVALID_ARG;
    if (!need(x, s, 16) || !need(idx, s, 4) || !need(send, s, 16) || !need(send_pos, s, 4))
        return MOE_ERR_INVALID_ARG;
    if (slot_of && !aligned(slot_of, 4)) return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    return launch_scatter(s, L, workspace, x, idx, wave, true, send, send_pos, nullptr, slot_of,
                          stream);
}

extern "C" moe_status moe_all_to_all(const moe_shape* shape, const void* workspace,
                                     size_t ws_bytes, int wave, int direction,
                                     const uint16_t* src, uint16_t* dst, cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (wave < -1 || wave >= s.W || (direction != 0 && direction != 1)) return MOE_ERR_INVALID_ARG;
    if (!need(src, s, 16) || !need(dst, s, 16)) return MOE_ERR_INVALID_ARG;
    if (s.T > 0 && src == dst) return MOE_ERR_INVALID_ARG;
    return exchange_rows(s, workspace, ws_bytes, wave, direction, src, dst, stream);
}

extern "C" moe_status moe_dispatch(const moe_shape* shape, const uint16_t* x, const int32_t* idx,
                                   const void* workspace, size_t ws_bytes, int wave,
                                   unsigned flags, uint16_t* send, uint16_t* recv,
                                   int32_t* slot_of, int32_t* src_row, int32_t* send_pos,
                                   cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    WsLayout L;
    if ((st = check_ws(s, workspace, ws_bytes, L)) != MOE_OK) return st;
    if (wave < -1 || wave >= s.W || (flags & ~(MOE_STAGED | MOE_EXPERT_MAJOR | MOE_BULK_COPY)))
        return MOE_ERR_INVALID_ARG;
    const bool em = (flags & MOE_EXPERT_MAJOR) != 0;
    const bool bulk = (flags & MOE_BULK_COPY) != 0;
    if (bulk && bulk_warps((size_t)s.H * 2) < 1) return MOE_ERR_UNSUPPORTED;
    if (!need(x, s, 16) || !need(idx, s, 4) || !need(recv, s, 16) || !need(slot_of, s, 4))
        return MOE_ERR_INVALID_ARG;
    if (src_row && !aligned(src_row, 4)) return MOE_ERR_INVALID_ARG;
    const bool staged = (flags & MOE_STAGED) != 0;
    if (staged && (!need(send, s, 16) || !need(send_pos, s, 4))) return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    if (!staged)
        return launch_scatter(s, L, workspace, x, idx, wave, false, recv, slot_of, src_row,
                              nullptr, stream, em, bulk);
    // staged: permute this wave's rows into the send layout, then exchange them
    st = launch_scatter(s, L, workspace, x, idx, wave, true, send, send_pos, nullptr, slot_of,
                        stream, em, bulk);
    if (st != MOE_OK) return st;
    if (src_row) {
        // the token of every recv row, through the fused map pass (no row copies)
        st = launch_scatter(s, L, workspace, x, idx, wave, false, nullptr, slot_of, src_row,
                            nullptr, stream, em);
        if (st != MOE_OK) return st;
    }
    return launch_exchange(s, L, workspace, wave, 0, send, recv, stream, em);
}

extern "C" moe_status moe_expert_capacity(const moe_shape* shape, double capacity_factor,
                                          int64_t* capacity) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    if (!capacity || !(capacity_factor >= 0.0) || capacity_factor > 1e6) return MOE_ERR_INVALID_ARG;
    const moe_shape& s = *shape;
    // EC = ceil(k * f * T / E), evaluated left to right in IEEE double
    const double ec = ceil((double)s.k * capacity_factor * (double)s.T / (double)s.E);
    if (ec * (double)s.E >= 2147483648.0) return MOE_ERR_UNSUPPORTED;
    *capacity = (int64_t)ec;
    return MOE_OK;
}

namespace moe {
namespace {

moe_status check_capacity(const moe_shape& s, int64_t EC) {
    if (EC < 0) return MOE_ERR_INVALID_ARG;
    if (EC * (int64_t)s.E >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    if (EC * (int64_t)s.E * s.H >= ((int64_t)1 << 46)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_dispatch_capacity(const moe_shape* shape, int64_t capacity,
                                            const uint16_t* x, const int32_t* idx,
                                            const void* workspace, size_t ws_bytes,
                                            uint16_t* cap_rows, int32_t* cap_slot,
                                            int32_t* dropped, cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if ((st = check_capacity(s, capacity)) != MOE_OK) return st;
    WsLayout L;
    if ((st = check_ws(s, workspace, ws_bytes, L)) != MOE_OK) return st;
    const bool any_rows = capacity > 0;
    if (!need(x, s, 16) || !need(idx, s, 4) || !need(cap_slot, s, 4)) return MOE_ERR_INVALID_ARG;
    if (any_rows && (!cap_rows || !aligned(cap_rows, 16))) return MOE_ERR_INVALID_ARG;
    if (dropped && !aligned(dropped, 4)) return MOE_ERR_INVALID_ARG;
    CapArgs a;
    a.x = reinterpret_cast<const uint4*>(x);
    a.idx = idx;
    a.rank = ws_ptr<int32_t>(workspace, L.rank);
    a.cpre = ws_ptr<int32_t>(workspace, L.cpre);
    a.cnt_se = ws_ptr<int32_t>(workspace, L.cnt_se);
    a.T = s.T;
    a.Tr = s.T / s.R;
    a.EC = capacity;
    a.ncap = capacity * s.E;
    a.H8 = s.H / 8;
    a.E = s.E;
    a.k = s.k;
    a.R = s.R;
    a.rows = reinterpret_cast<uint4*>(cap_rows);
    a.cap_slot = cap_slot;
    a.dropped = dropped;
    a.err = &const_cast<WsHeader*>(ws_ptr<WsHeader>(workspace, 0))->error;
    if (s.T > 0) {
        st = launch_k(capacity_scatter_kernel, dim3(grid_for(s.T, kRowWarps)),
                      dim3(kRowWarps * kWarp), 0, stream, a);
        if (st != MOE_OK) return st;
    }
    if (!any_rows && !dropped) return MOE_OK;
    int gx = (int)((capacity + kRowWarps - 1) / kRowWarps);
    const int cap_x = (device_sm_count() * 8 + s.E - 1) / s.E;
    if (gx > cap_x) gx = cap_x;
    if (gx < 1) gx = 1;
    return launch_k(capacity_pad_kernel, dim3(gx, s.E), dim3(kRowWarps * kWarp), 0, stream, a);
}
