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

#include <atomic>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kRowWarps = 8;
constexpr int kVecUnroll = 8;  // 16-byte vectors in flight per lane
// The row scatter runs 4-warp CTAs, so the launches of several waves that run
// at the same time can share every SM.
constexpr int kScatterThreads = 128;
constexpr int kScatterWarps = kScatterThreads / kWarp;

// x-row load policies of the row scatter
constexpr int kXEvictFirst = 0;   // read once
constexpr int kXEvictLast = 1;    // read again by a later wave call: keep in L2
constexpr int kXEvictNormal = 2;  // read by concurrent wave calls at about the same time

struct ScatterArgs {
    const uint4* x;
    const int32_t* idx;
    const int32_t* rank;
    const int32_t* table;  // first dst row of (source, expert): rstart or sstart
    const int32_t* rtable; // rstart, for the optional recv-row map of the permute
    int64_t T, Tr, nrows;
    int H8, E, k, W, Ew, wave;
    int reverse;        // hand the tickets out from the last tokens down
    int x_policy;       // kXEvict*
    int budget;         // > 0: concurrent waves; this wave takes a share of `budget` CTAs
    int expert_major;   // recv rows ordered (rank, expert, source, token, slot)
    const int32_t* eoff;  // first row of each expert (expert-major), also the wave sizes
    const int32_t* cpre;  // slots of expert e in the sources before s
    uint4* dst;         // NULL: write the maps only
    int32_t* dst_map;   // slot_of (fused) or send_pos (permute)
    int32_t* src_row;   // token of each recv row (fused only), may be NULL
    int32_t* slot_of;   // permute only: recv row of (t, j), may be NULL
    uint32_t* tick;     // this call's (ticket, done) pair in the workspace
    uint32_t* err;
};

// A ticket of the row scatter covers m batches of tb tokens; a batch's
// tb * k slots sit one per lane.  The ticket is sized to about kRowsPerTicket
// rows of the call (from its rows per token), so a dense call (every wave)
// takes one token per ticket and a sparse wave up to kMaxBatches batches,
// whose index loads are issued together.
constexpr int kMaxBatches = 4;
constexpr int kRowsPerTicket = 8;

__device__ __forceinline__ void ticket_shape(int64_t rows, int T, int k, int& tb, int& m) {
    const int tbmax = kWarp / k;
    int64_t g = rows > 0 ? ((int64_t)kRowsPerTicket * T + rows / 2) / rows
                         : (int64_t)tbmax * kMaxBatches;
    g = g < 1 ? 1 : (g > (int64_t)tbmax * kMaxBatches ? (int64_t)tbmax * kMaxBatches : g);
    tb = (int)(g < tbmax ? g : tbmax);
    m = (int)((g + tb / 2) / tb);
    m = m < 1 ? 1 : (m > kMaxBatches ? kMaxBatches : m);
}

__device__ __forceinline__ int64_t wave_rows(const ScatterArgs& a, int w) {
    return (int64_t)__ldg(a.eoff + (w + 1) * a.Ew) - __ldg(a.eoff + w * a.Ew);
}

// Copies one x row to the rows rows[j] (j in mask), 16-byte vectors, kVecUnroll
// in flight per lane.
__device__ __forceinline__ void copy_row_to_rows(const uint4* __restrict__ src, uint4* dst_base,
                                                 int H8, unsigned mask, const int32_t* rows,
                                                 int lane, uint64_t ld_pol, uint64_t st_pol) {
    for (int base = 0; base < H8; base += kWarp * kVecUnroll) {
        uint4 v[kVecUnroll];
#pragma unroll
        for (int u = 0; u < kVecUnroll; ++u) {
            const int p = base + u * kWarp + lane;
            if (p < H8) v[u] = ld_nc_v4_hint(src + p, ld_pol);
        }
        for (unsigned m = mask; m; m &= m - 1) {
            uint4* d = dst_base + (int64_t)rows[__ffs(m) - 1] * H8;
#pragma unroll
            for (int u = 0; u < kVecUnroll; ++u) {
                const int p = base + u * kWarp + lane;
                if (p < H8) st_v4_hint(d + p, v[u], st_pol);
            }
        }
    }
}

// Copies one x row to the rows held by lanes lane_base + j (j in mask).
__device__ __forceinline__ void copy_row_to_many(const uint4* __restrict__ src, uint4* dst_base,
                                                 int H8, unsigned mask, int32_t row, int lane,
                                                 uint64_t ld_pol, uint64_t st_pol) {
    for (int base = 0; base < H8; base += kWarp * kVecUnroll) {
        uint4 v[kVecUnroll];
#pragma unroll
        for (int u = 0; u < kVecUnroll; ++u) {
            const int p = base + u * kWarp + lane;
            if (p < H8) v[u] = ld_nc_v4_hint(src + p, ld_pol);
        }
        for (unsigned m = mask; m; m &= m - 1) {
            const int32_t r = __shfl_sync(kFull, row, __ffs(m) - 1);
            uint4* d = dst_base + (int64_t)r * H8;
#pragma unroll
            for (int u = 0; u < kVecUnroll; ++u) {
                const int p = base + u * kWarp + lane;
                if (p < H8) st_v4_hint(d + p, v[u], st_pol);
            }
        }
    }
}

// Row scatter of one wave (or all).  A warp takes a ticket, resolves the rows
// of its batches' slots (expert, then rank and row table: one chain of loads
// for the whole ticket, rows kept in shared memory) and copies each token's x
// row (16-byte vectors, read once per ticket) to its rows of the wave.
// Tickets come from an atomic counter in token order (the next one fetched
// while the current one is copied), so warps that drew light tickets take
// more of them; the last warp to finish resets the ticket pair for the next
// call.
//
// Concurrent waves (budget > 0): the W wave launches run at the same time,
// each launched with up to `budget` CTAs; a launch keeps the share of the
// budget that its wave's tickets are of all waves' tickets (the expert offsets
// give every wave's size, so every launch computes the same shares) and its
// other CTAs leave at once.  The waves then progress through the tokens at
// about the same pace, in the same order, so a token's x row is read from
// memory by the first wave to reach it and from L2 by the others.
template <bool TO_SEND>
__global__ void __launch_bounds__(kScatterThreads, 8) scatter_rows_kernel(ScatterArgs a) {
    grid_dependency_sync();
    __shared__ int32_t s_row[kScatterWarps][kMaxBatches][kWarp];
    __shared__ uint32_t s_ball[kScatterWarps][kMaxBatches];
    __shared__ int64_t s_part[kScatterWarps];
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    // T * k < 2^31 (checked on the host): token, slot and ticket indices fit
    // 32 bits; row offsets in elements are formed in 64 bits
    const int k = a.k, T = (int)a.T, Tr = (int)a.Tr;
    int tb, m;
    ticket_shape(a.wave < 0 ? (int64_t)T * k : wave_rows(a, a.wave), T, k, tb, m);
    const int per_ticket = tb * m;
    const int nticket = (T + per_ticket - 1) / per_ticket;
    int ncta = gridDim.x;
    if (a.budget > 0 && a.wave >= 0) {
        int64_t mine = 0;
        for (int w = threadIdx.x; w < a.W; w += kScatterThreads) {
            int tbw, mw;
            ticket_shape(wave_rows(a, w), T, k, tbw, mw);
            mine += (T + tbw * mw - 1) / (tbw * mw);
        }
#pragma unroll
        for (int o = kWarp / 2; o; o >>= 1) mine += __shfl_xor_sync(kFull, mine, o);
        if (lane == 0) s_part[warp] = mine;
        __syncthreads();
        int64_t all = 0;
#pragma unroll
        for (int q = 0; q < kScatterWarps; ++q) all += s_part[q];
        int64_t n = all > 0 ? (int64_t)a.budget * nticket / all : 1;
        n = n < 1 ? 1 : (n > ncta ? ncta : n);
        if ((int64_t)blockIdx.x >= n) return;
        ncta = (int)n;
    }
    const uint64_t ld_pol = a.x_policy == kXEvictLast    ? l2_policy_evict_last()
                            : a.x_policy == kXEvictFirst ? l2_policy_evict_first()
                                                         : l2_policy_evict_normal();
    const uint64_t st_pol = l2_policy_evict_first();
    const uint32_t nwarps = (uint32_t)ncta * kScatterWarps;  // warps taking tickets
    const int l = lane / k, j = lane - (lane / k) * k;  // token of a batch, slot of the token
    const unsigned kmask = (k >= 32) ? kFull : ((1u << k) - 1u);
    int32_t* rowbuf = &s_row[warp][0][0];
    uint32_t tk = 0;
    if (lane == 0) tk = atomicAdd(a.tick, 1u);
    uint32_t u = __shfl_sync(kFull, tk, 0);
    while (u < (uint32_t)nticket) {
        if (lane == 0) tk = atomicAdd(a.tick, 1u);  // the next ticket, fetched ahead
        const int tt = (a.reverse ? nticket - 1 - (int)u : (int)u) * per_ticket;
        // 1. the experts of every slot of the ticket, loads issued together
        int ev[kMaxBatches];
#pragma unroll
        for (int q = 0; q < kMaxBatches; ++q) {
            const int t = tt + q * tb + l;
            ev[q] = (q < m && l < tb && t < T) ? __ldg(a.idx + t * k + j) : -2;
        }
        // 2. rank and first row of the wave's slots, then their rows and maps
#pragma unroll
        for (int q = 0; q < kMaxBatches; ++q) {
            const int e = ev[q];
            const int t = tt + q * tb + l;
            const int sl = t * k + j;
            int32_t row = -1;
            if (e != -2) {
                if (e < 0 || e >= a.E) {
                    raise_error(a.err, MOE_ERR_DEVICE_CHECK, (uint32_t)sl);
                } else if (a.wave < 0 || e / a.Ew == a.wave) {
                    const int s = t / Tr;
                    const int32_t r = __ldg(a.rank + sl);
                    const int64_t rw =
                        (!TO_SEND && a.expert_major)
                            ? (int64_t)__ldg(a.eoff + e) + __ldg(a.cpre + s * a.E + e) + r
                            : (int64_t)__ldg(a.table + s * a.E + e) + r;
                    if (rw >= 0 && rw < a.nrows) {
                        row = (int32_t)rw;
                        a.dst_map[sl] = row;
                        if (!TO_SEND && a.src_row) a.src_row[rw] = (int32_t)t;
                        if (TO_SEND && a.slot_of) {
                            const int64_t rr =
                                a.expert_major
                                    ? (int64_t)__ldg(a.eoff + e) + __ldg(a.cpre + s * a.E + e) + r
                                    : (int64_t)__ldg(a.rtable + s * a.E + e) + r;
                            if (rr >= 0 && rr < a.nrows) a.slot_of[sl] = (int32_t)rr;
                        }
                    } else {
                        raise_error(a.err, MOE_ERR_DEVICE_CHECK, (uint32_t)sl);
                    }
                }
            }
            if (q < m) {
                rowbuf[q * kWarp + lane] = row;
                const unsigned ball = __ballot_sync(kFull, row >= 0);
                if (lane == 0) s_ball[warp][q] = ball;
            }
        }
        __syncwarp();
        // 3. copy each token's x row to its rows of the wave
        if (a.dst) {
            for (int q = 0; q < m; ++q) {
                const unsigned ball = s_ball[warp][q];
                if (!ball) continue;
                const int t0 = tt + q * tb;
                for (int p = 0; p < tb; ++p) {
                    const unsigned mm = (ball >> (p * k)) & kmask;
                    if (mm)
                        copy_row_to_rows(a.x + (int64_t)(t0 + p) * a.H8, a.dst, a.H8, mm,
                                         rowbuf + q * kWarp + p * k, lane, ld_pol, st_pol);
                }
            }
        }
        __syncwarp();  // the next ticket rewrites rowbuf
        u = __shfl_sync(kFull, tk, 0);
    }
    // every warp took one ticket past the end; the last one out resets the pair
    if (lane == 0) {
        __threadfence();
        if (atomicAdd(a.tick + 1, 1u) == nwarps - 1) {
            a.tick[0] = 0u;
            a.tick[1] = 0u;
            __threadfence();
        }
    }
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
        if (mask) copy_row_to_many(a.x + t * a.H8, a.rows, a.H8, mask, row, lane, pol, pol);
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

// CTAs of the row scatter that fit on the device at once (every SM full).
int scatter_capacity(const void* kern) {
    static std::atomic<int> cache[2][kMaxDevices];  // 0: not queried yet
    const int d = current_device();
    const int which = kern == reinterpret_cast<const void*>(scatter_rows_kernel<true>) ? 1 : 0;
    const bool cached = d >= 0 && d < kMaxDevices;
    int n = cached ? cache[which][d].load(std::memory_order_relaxed) : 0;
    if (n > 0) return n;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kScatterThreads, 0) !=
            cudaSuccess ||
        per_sm <= 0)
        per_sm = 4;
    n = per_sm * device_sm_count();
    if (cached) cache[which][d].store(n, std::memory_order_relaxed);
    return n;
}

moe_status launch_scatter(const moe_shape& s, const WsLayout& L, const void* ws, const uint16_t* x,
                          const int32_t* idx, int wave, bool to_send, uint16_t* dst,
                          int32_t* dst_map, int32_t* src_row, int32_t* slot_of,
                          cudaStream_t stream, bool expert_major = false,
                          bool concurrent = false) {
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
    a.W = s.W;
    a.wave = wave;
    a.expert_major = expert_major ? 1 : 0;
    a.eoff = ws_ptr<int32_t>(ws, L.eoff);
    a.cpre = ws_ptr<int32_t>(ws, L.cpre);
    a.dst = reinterpret_cast<uint4*>(dst);
    a.dst_map = dst_map;
    a.src_row = src_row;
    a.slot_of = slot_of;
    a.tick = const_cast<uint32_t*>(ws_ptr<uint32_t>(ws, L.tickets)) +
             2 * (wave < 0 ? kTicketSlots - 1 : wave);
    a.err = &const_cast<WsHeader*>(ws_ptr<WsHeader>(ws, 0))->error;
    const void* kern = to_send ? reinterpret_cast<const void*>(scatter_rows_kernel<true>)
                               : reinterpret_cast<const void*>(scatter_rows_kernel<false>);
    const int cap = scatter_capacity(kern);
    // at most one CTA per kScatterWarps tokens (a ticket holds at least one)
    const int need_ctas = grid_for(s.T, kScatterWarps);
    int grid = need_ctas < cap ? need_ctas : cap;
    if (concurrent && wave >= 0 && s.W > 1) {
        // All W launches are resident together: each keeps a share of the
        // device proportional to its rows (one CTA per wave held back, so the
        // shares never exceed what fits), walking the tokens forwards.
        a.budget = cap - s.W > s.W ? cap - s.W : s.W;
        a.reverse = 0;
        a.x_policy = kXEvictNormal;
    } else {
        // Wave calls one after the other, in order 0..W-1: each reads the x
        // rows of its tokens, so odd waves walk the tokens backwards (a wave
        // starts on the rows the previous one read last) and every wave but
        // the last keeps the rows it reads in L2 for the next.
        a.budget = 0;
        a.reverse = (wave > 0 && (wave & 1)) ? 1 : 0;
        a.x_policy = (wave >= 0 && wave < s.W - 1) ? kXEvictLast : kXEvictFirst;
    }
    const dim3 block(kScatterThreads);
    return to_send ? launch_k(scatter_rows_kernel<true>, dim3(grid), block, 0, stream, a)
                   : launch_k(scatter_rows_kernel<false>, dim3(grid), block, 0, stream, a);
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
    if (wave < -1 || wave >= s.W ||
        (flags & ~(MOE_STAGED | MOE_EXPERT_MAJOR | MOE_WAVES_CONCURRENT)))
        return MOE_ERR_INVALID_ARG;
    const bool em = (flags & MOE_EXPERT_MAJOR) != 0;
    const bool concurrent = (flags & MOE_WAVES_CONCURRENT) != 0;
    if (!need(x, s, 16) || !need(idx, s, 4) || !need(recv, s, 16) || !need(slot_of, s, 4))
        return MOE_ERR_INVALID_ARG;
    if (src_row && !aligned(src_row, 4)) return MOE_ERR_INVALID_ARG;
    const bool staged = (flags & MOE_STAGED) != 0;
    if (staged && (!need(send, s, 16) || !need(send_pos, s, 4))) return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    if (!staged)
        return launch_scatter(s, L, workspace, x, idx, wave, false, recv, slot_of, src_row,
                              nullptr, stream, em, concurrent);
    // staged: permute this wave's rows into the send layout, then exchange them
    st = launch_scatter(s, L, workspace, x, idx, wave, true, send, send_pos, nullptr, slot_of,
                        stream, em);
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
