// moe_build_send_counts: the send-count matrix S[src][dst], the per-expert
// counts and the alltoallv send/recv offsets ("不规则与流水化 AllToAll", table
// "经典 vs 不规则": Alltoallv needs the full send-count / recv-count
// matrices; section "与其他原语的衔接": the top-k index set is the send-count
// matrix), plus every (token, slot)'s rank among the slots of the same source
// rank and expert, which fixes its row in the send and recv layouts.
//
// One pass over idx.  Tiles are runs of up to kTileTokens tokens of ONE source
// rank; a tile's CTA takes a ticket (so every tile it waits on is already
// running or done), histograms its slots with __match_any_sync, scans the
// per-warp histograms inside the CTA, and gets each expert's count over the
// earlier tiles of its source from a decoupled look-back (single-pass
// prefix scan with per-bin look-back): tiles publish their own count first and
// their inclusive count once known; a successor adds aggregates until it meets
// an inclusive count.  Every wait is bounded by a time limit; a wait that runs
// out raises MOE_ERR_TIMEOUT and the pass finishes with what it has.
//
// The last tile of each source writes that source's row of C and its whole
// send side (S row, send offsets, first send rows).  The CTA that finishes
// last (ticketed completion counter, no waiting) builds what needs every
// source: c, the recv offsets and the recv and expert-major row tables.
//
// moe_route_and_count fuses the routing into the same pass: a tile's CTA
// routes its own tokens first (route_core.cuh), keeping the chosen experts in
// shared memory for the histogram, so the counts need no second launch and
// no re-read of idx, and one tile's routing overlaps the look-back of the
// tiles before it.
#include <mutex>

#include "route_core.cuh"

namespace moe {
namespace {

constexpr int kMaxTileSlots = kTileTokens * MOE_MAX_TOPK;  // 2048
constexpr int kLookWindow = 8;  // predecessor status words read per look-back round trip
constexpr int kSegRows = kMaxTileSlots / (kCountWarps * kWarp);  // 32-slot rows per warp
constexpr uint16_t kNoExpert = 0xFFFF;                     // > any expert index

struct CountArgs {
    const int32_t* idx;
    int T, E, k, R;
    int64_t nchunk, ntiles;
    uint64_t* status;   // [R][nchunk][E]
    int32_t* cnt_se;    // [R][E]
    int32_t* sstart;    // [R][E]
    int32_t* rstart;    // [R][E]
    int32_t* cpre;      // [R][E]  slots of expert e in sources before s
    int32_t* eoff;      // [E+1]   first row of expert e in the expert-major layout
    int32_t* rank;      // [T*k]
    WsHeader* hdr;
    int32_t* expert_counts;       // [E]
    int32_t* rank_expert_counts;  // [R][E]
    int32_t* send_counts;         // [R][R]
    int64_t* send_off;            // [R][R+1]
    int64_t* recv_off;            // [R][R+1]
    int64_t* recv_base;           // [R+1]
    int mark_failure;             // a raised error also sets recv_base[R] = -(status)
};

struct TileSmem {
    int32_t wcnt[kCountWarps][MOE_MAX_EXPERTS];  // per-warp histogram, then warp prefix
    int32_t excl[MOE_MAX_EXPERTS];               // count over earlier tiles of the source
    int32_t incl[MOE_MAX_EXPERTS];               // last tile of a source: C[s][e]
    int32_t pre[MOE_MAX_EXPERTS + 1];            // last tile: exclusive prefix of C[s][.]
    uint16_t lrank[kMaxTileSlots];               // rank inside the warp's segment
    uint16_t ex[kMaxTileSlots];                  // expert of the slot (kNoExpert: invalid)
};

// Shared memory of the finishing CTA, sized by R and E (dynamic shared
// memory; the tile phase uses the same bytes as a TileSmem).
struct FinishLayout {
    size_t C, S, rp, colsum, ecnt, rbase, bytes;
};

__host__ __device__ inline FinishLayout finish_layout(int R, int E) {
    FinishLayout f;
    size_t off = 0;
    f.C = off;       // int32 [R][E]  C[s][e]
    off += (size_t)R * E * 4;
    f.S = off;       // int32 [R][R]  S[s][d], then its exclusive row prefix
    off += (size_t)R * R * 4;
    f.rp = off;      // int32 [R][R]  rp[d][s], exclusive column prefix of S
    off += (size_t)R * R * 4;
    f.colsum = off;  // int32 [R]     rows received by d
    off += (size_t)R * 4;
    f.ecnt = off;    // int32 [E]     slots of expert e
    off += (size_t)E * 4;
    off = (off + 7) & ~(size_t)7;
    f.rbase = off;   // int64 [R+1]
    off += (size_t)(R + 1) * 8;
    f.bytes = off;
    return f;
}

__host__ __device__ inline size_t count_smem_bytes(int R, int E) {
    const size_t f = finish_layout(R, E).bytes;
    return f > sizeof(TileSmem) ? f : sizeof(TileSmem);
}

// Zeroes the per-warp histograms; callers run it before the barrier that
// precedes count_tile.
__device__ inline void zero_histograms(TileSmem& sm, int E) {
    for (int i = threadIdx.x; i < kCountWarps * E; i += kCountThreads) sm.wcnt[i / E][i % E] = 0;
}

// The last tile of source s knows the source's count of every expert,
// C[s][.]: it writes that row and the whole send side of the source (S[s][.],
// send_off[s][.] and the first send row of every (s, e)), which need no
// other source.  Warp 0 scans the E <= 256 counts, 8 per lane.
__device__ void source_tail(const CountArgs& a, int64_t s, TileSmem& sm) {
    const int tid = threadIdx.x, lane = tid & (kWarp - 1), warp = tid >> 5;
    const int E = a.E, R = a.R, Er = E / R;
    const int64_t base = s * (int64_t)E;
    for (int e = tid; e < E; e += kCountThreads) {
        const int32_t v = sm.incl[e];
        a.cnt_se[base + e] = v;
        a.rank_expert_counts[base + e] = v;
    }
    if (warp != 0) return;
    int32_t v[8], run = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int e = lane * 8 + q;
        v[q] = e < E ? sm.incl[e] : 0;
        run += v[q];
    }
    int32_t inc = run;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int32_t u = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += u;
    }
    int32_t ex = inc - run;
    const int32_t row0 = (int32_t)(s * (a.T / a.R) * a.k);  // first send row of source s
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int e = lane * 8 + q;
        if (e < E) {
            sm.pre[e] = ex;
            a.sstart[base + e] = row0 + ex;
        }
        ex += v[q];
    }
    if (lane == kWarp - 1) sm.pre[E] = inc;
    __syncwarp();
    int64_t* so = a.send_off + s * (R + 1);
    for (int d = lane; d < R; d += kWarp) {
        a.send_counts[s * R + d] = sm.pre[(d + 1) * Er] - sm.pre[d * Er];
        so[d] = sm.pre[d * Er];
    }
    if (lane == 0) so[R] = sm.pre[E];
    // rstart[s][e] gets its part from this source alone: the slots of source s
    // before e inside e's rank; the finishing CTA adds where (d, s) starts
    for (int e = lane; e < E; e += kWarp) a.rstart[base + e] = sm.pre[e] - sm.pre[(e / Er) * Er];
}

// FROM_SMEM: the tile's experts are already in sm.ex (the fused routing
// wrote them there before the caller's barrier) instead of in idx.
template <bool FROM_SMEM>
__device__ void count_tile(const CountArgs& a, int64_t tile, uint32_t tag, uint64_t wait_ns,
                           TileSmem& sm) {
    const int tid = threadIdx.x, lane = tid & (kWarp - 1), warp = tid >> 5;
    const int E = a.E, k = a.k;
    const int64_t Tr = a.T / a.R;
    const int64_t s = tile / a.nchunk, c = tile % a.nchunk;
    const int64_t tok_lo = s * Tr + c * kTileTokens;
    const int64_t tok_hi = min(tok_lo + kTileTokens, (s + 1) * Tr);
    const int64_t slot_lo = tok_lo * k;
    const int n = (int)((tok_hi - tok_lo) * k);
    uint32_t* err = &a.hdr->error;

    // 1. per-warp histogram over a contiguous segment; ranks inside the segment.
    // A warp's segment is at most kSegRows rows of 32 slots; their expert
    // indices are loaded together first.
    const int seg = ((n + kCountWarps * kWarp - 1) / (kCountWarps * kWarp)) * kWarp;
    const int w_lo = warp * seg, w_hi = min(n, w_lo + seg);
    int ev[kSegRows];
#pragma unroll
    for (int q = 0; q < kSegRows; ++q) {
        const int i = w_lo + q * kWarp + lane;
        if (FROM_SMEM)
            ev[q] = (i < w_hi) ? (int)sm.ex[i] : -1;
        else
            ev[q] = (i < w_hi) ? __ldg(a.idx + slot_lo + i) : -1;
    }
#pragma unroll
    for (int q = 0; q < kSegRows; ++q) {
        const int base = w_lo + q * kWarp;
        if (base >= w_hi) break;
        const int i = base + lane;
        int e = ev[q];
        if (i < w_hi && (e < 0 || e >= E)) {
            raise_error(err, MOE_ERR_DEVICE_CHECK, (uint32_t)(slot_lo + i));
            e = -1;
        }
        const unsigned peers = __match_any_sync(kFull, e);
        int r = 0;
        if (e >= 0) r = sm.wcnt[warp][e] + __popc(peers & lanemask_lt());
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) sm.wcnt[warp][e] += __popc(peers);
        __syncwarp();
        if (i < w_hi) {
            sm.ex[i] = (e >= 0) ? (uint16_t)e : kNoExpert;
            sm.lrank[i] = (uint16_t)r;
        }
    }
    __syncthreads();

    // 2. per expert: exclusive prefix over warps, tile total, look-back
    const bool publish = (a.hdr->fault_tile_p1 == 0) || ((int64_t)a.hdr->fault_tile_p1 - 1 != tile);
    for (int e = tid; e < E; e += kCountThreads) {
        int32_t run = 0;
#pragma unroll
        for (int w = 0; w < kCountWarps; ++w) {
            const int32_t v = sm.wcnt[w][e];
            sm.wcnt[w][e] = run;
            run += v;
        }
        const uint32_t agg = (uint32_t)run;
        uint64_t* my = a.status + ((size_t)tile * E + e);
        uint32_t excl = 0;
        if (c == 0) {
            if (publish) st_relaxed_u64(my, pack_status(tag, kFlagPrefix, agg));
        } else {
            if (publish) st_relaxed_u64(my, pack_status(tag, kFlagAggregate, agg));
            // Walk back over the same source's tiles s*nchunk .. tile-1, reading
            // a window of kLookWindow status words per round trip.
            int64_t p = tile - 1;
            const int64_t first = s * a.nchunk;
            const uint64_t t0 = globaltimer_ns();
            unsigned backoff = 32;
            bool done = false;
            while (!done) {
                uint64_t wd[kLookWindow];
#pragma unroll
                for (int q = 0; q < kLookWindow; ++q)
                    wd[q] = (p - q >= first) ? ld_relaxed_u64(a.status + ((size_t)(p - q) * E + e))
                                             : 0ull;
                int used = 0;
#pragma unroll
                for (int q = 0; q < kLookWindow; ++q) {
                    if (done || used != q || p - q < first) continue;
                    const uint64_t flag = status_flag(wd[q], tag);
                    if (flag == 0) continue;  // not published yet: poll again from here
                    excl += status_count(wd[q]);
                    used = q + 1;
                    if (flag == kFlagPrefix || p - q == first) done = true;
                }
                if (done) break;
                p -= used;
                if (used == 0) {
                    if (globaltimer_ns() - t0 > wait_ns) {
                        raise_error(err, MOE_ERR_TIMEOUT, (uint32_t)tile);
                        break;
                    }
                    __nanosleep(backoff);
                    if (backoff < 1024) backoff <<= 1;
                }
            }
            if (publish) st_relaxed_u64(my, pack_status(tag, kFlagPrefix, excl + agg));
        }
        sm.excl[e] = (int32_t)excl;
        sm.incl[e] = (int32_t)(excl + agg);
    }
    __syncthreads();
    if (c == a.nchunk - 1) source_tail(a, s, sm);

    // 3. rank of each slot within (source, expert)
    for (int i = tid; i < n; i += kCountThreads) {
        const int e = sm.ex[i];
        if (e != kNoExpert) a.rank[slot_lo + i] = sm.excl[e] + sm.wcnt[i / seg][e] + sm.lrank[i];
    }
}

// Exclusive prefix over n <= 64 int32 values v(i), lane l holding entries 2l
// and 2l+1; returns them in e0, e1 and the total.
__device__ __forceinline__ void warp_scan64(int32_t v0, int32_t v1, int lane, int32_t& e0,
                                            int32_t& e1, int32_t& total) {
    int32_t inc = v0 + v1;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int32_t u = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += u;
    }
    total = __shfl_sync(kFull, inc, kWarp - 1);
    e0 = inc - v0 - v1;
    e1 = e0 + v0;
}

// Builds what needs every source: c, cpre, the recv offsets, recv_base, the
// first row of every expert in the expert-major layout and the first recv row
// of every (source, expert).  One CTA.  C arrives from the sources' last tiles
// (source_tail) through L2 in one round of vector loads; rows and columns of S
// are scanned one warp each; rstart holds each entry's offset inside its rank,
// to which the start of (d, s) is added.  With no tiles (T = 0) it writes
// every table itself, all zeros.
__device__ void finish_counts(const CountArgs& a, uint32_t tag, unsigned char* dsm) {
    const int tid = threadIdx.x, lane = tid & (kWarp - 1), warp = tid >> 5;
    const int E = a.E, R = a.R, Er = E / R;
    const FinishLayout F = finish_layout(R, E);
    int32_t* C = reinterpret_cast<int32_t*>(dsm + F.C);
    int32_t* S = reinterpret_cast<int32_t*>(dsm + F.S);
    int32_t* rp = reinterpret_cast<int32_t*>(dsm + F.rp);
    int32_t* colsum = reinterpret_cast<int32_t*>(dsm + F.colsum);
    int64_t* rbase = reinterpret_cast<int64_t*>(dsm + F.rbase);
    int32_t* ecnt = reinterpret_cast<int32_t*>(dsm + F.ecnt);
    const bool tiles = a.nchunk > 0;
    const int RE = R * E;

    if (!tiles) {
        for (int i = tid; i < RE; i += kCountThreads) {
            C[i] = 0;
            a.cnt_se[i] = 0;
            a.rank_expert_counts[i] = 0;
            a.sstart[i] = 0;
            a.rstart[i] = 0;
        }
        for (int i = tid; i < R * R; i += kCountThreads) a.send_counts[i] = 0;
        for (int i = tid; i < R * (R + 1); i += kCountThreads) a.send_off[i] = 0;
    } else if ((E & 3) == 0) {  // cnt_se starts on 256 bytes, so its rows are int4-aligned
        const int4* src = reinterpret_cast<const int4*>(a.cnt_se);
        int4* dst = reinterpret_cast<int4*>(C);
        for (int i = tid; i < RE / 4; i += kCountThreads) dst[i] = __ldcg(src + i);
    } else {
        for (int i = tid; i < RE; i += kCountThreads) C[i] = __ldcg(a.cnt_se + i);
    }
    __syncthreads();
    for (int i = tid; i < R * R; i += kCountThreads) {
        const int s = i / R, d = i % R;
        int32_t sum = 0;
        for (int e = d * Er; e < (d + 1) * Er; ++e) sum += C[s * E + e];
        S[i] = sum;
    }
    // c and cpre[s][e] = slots of expert e in the sources before s
    for (int e = tid; e < E; e += kCountThreads) {
        int32_t tot = 0;
        for (int s = 0; s < R; ++s) {
            a.cpre[s * E + e] = tot;
            tot += C[s * E + e];
        }
        a.expert_counts[e] = tot;
        ecnt[e] = tot;
    }
    __syncthreads();
    // columns: recv_off[d][s] = sum over s' < s of S[s'][d]
    for (int d = warp; d < R; d += kCountWarps) {
        const int s0 = 2 * lane, s1 = 2 * lane + 1;
        const int32_t v0 = s0 < R ? S[s0 * R + d] : 0, v1 = s1 < R ? S[s1 * R + d] : 0;
        int32_t e0, e1, tot;
        warp_scan64(v0, v1, lane, e0, e1, tot);
        int64_t* ro = a.recv_off + (size_t)d * (R + 1);
        if (s0 < R) { ro[s0] = e0; rp[d * R + s0] = e0; }
        if (s1 < R) { ro[s1] = e1; rp[d * R + s1] = e1; }
        if (lane == 0) { ro[R] = tot; colsum[d] = tot; }
    }
    __syncthreads();
    // first row of every expert in the expert-major layout: exclusive scan of
    // the expert totals, 8 per lane (E <= 256)
    if (warp == 1) {
        int32_t v[8], run = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = lane * 8 + q;
            v[q] = e < E ? ecnt[e] : 0;
            run += v[q];
        }
        int32_t inc = run;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int32_t u = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += u;
        }
        int32_t ex = inc - run;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = lane * 8 + q;
            if (e < E) a.eoff[e] = ex;
            ex += v[q];
        }
        if (lane == kWarp - 1) a.eoff[E] = inc;
    }
    // recv_base[d] = rows received by the ranks before d
    if (warp == 0) {
        const int d0 = 2 * lane, d1 = 2 * lane + 1;
        const int32_t v0 = d0 < R ? colsum[d0] : 0, v1 = d1 < R ? colsum[d1] : 0;
        int32_t e0, e1, tot;
        warp_scan64(v0, v1, lane, e0, e1, tot);
        if (d0 < R) { a.recv_base[d0] = e0; rbase[d0] = e0; }
        if (d1 < R) { a.recv_base[d1] = e1; rbase[d1] = e1; }
        if (lane == 0) { a.recv_base[R] = tot; rbase[R] = tot; }
    }
    __syncthreads();
    // first recv row of (s, e) = where (d, s) starts + the part source_tail
    // left in rstart; an int4 never straddles two ranks when 4 divides E / R
    if (tiles && (Er & 3) == 0) {
        int4* rs = reinterpret_cast<int4*>(a.rstart);
        for (int i = tid; i < RE / 4; i += kCountThreads) {
            const int4 v = __ldcg(rs + i);
            const int s = (4 * i) / E, d = ((4 * i) % E) / Er;
            const int32_t add = (int32_t)rbase[d] + rp[d * R + s];
            rs[i] = make_int4(v.x + add, v.y + add, v.z + add, v.w + add);
        }
    } else if (tiles) {
        for (int i = tid; i < RE; i += kCountThreads) {
            const int s = i / E, d = (i % E) / Er;
            a.rstart[i] = __ldcg(a.rstart + i) + (int32_t)rbase[d] + rp[d * R + s];
        }
    }
    if (tid == 0) {
        if (a.mark_failure) {
            // every tile has raised its errors before counting itself done
            const uint32_t e = *(volatile uint32_t*)&a.hdr->error;
            if (e != 0) a.recv_base[R] = -(int64_t)e;
        }
        a.hdr->ticket = 0;
        a.hdr->done = 0;
        a.hdr->epoch = tag;
    }
}

__global__ void __launch_bounds__(kCountThreads) send_counts_kernel(CountArgs a) {
    grid_dependency_sync();
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ int64_t s_tile;
    __shared__ int s_last;
    __shared__ uint32_t s_tag;
    __shared__ uint64_t s_wait;
    if (threadIdx.x == 0) {
        s_tile = (int64_t)atomicAdd(&a.hdr->ticket, 1u);
        s_tag = next_tag(*(volatile uint32_t*)&a.hdr->epoch);
        const uint64_t wn = *(volatile uint64_t*)&a.hdr->wait_ns;
        s_wait = wn ? wn : kDefaultWaitNs;
    }
    zero_histograms(*reinterpret_cast<TileSmem*>(dsm), a.E);  // while the ticket is in flight
    __syncthreads();
    const int64_t tile = s_tile;
    const uint32_t tag = s_tag;
    if (tile < a.ntiles)
        count_tile<false>(a, tile, tag, s_wait, *reinterpret_cast<TileSmem*>(dsm));

    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&a.hdr->done, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    finish_counts(a, tag, dsm);
}

// Routes the tokens [tok_lo, tok_hi) of one tile, G lanes per token and
// kCountWarps * 32 / G tokens per pass; the next pass's logits are loaded
// before the current token is routed.  ex[(t - tok_lo) * k + j] receives the
// j-th expert of token t.
template <int EPL, int G, bool VEC>
__device__ __forceinline__ void route_tile(const float* __restrict__ logits,
                                           int32_t* __restrict__ idx, float* __restrict__ w,
                                           const RouteParams& p, int64_t tok_lo, int64_t tok_hi,
                                           uint16_t* ex) {
    constexpr int TPW = kWarp / G;
    constexpr int kPass = kCountWarps * TPW;
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    const int sub = lane / G, gl = lane % G;
    const unsigned smask = (G == kWarp) ? kFull : (((1u << G) - 1u) << (sub * G));
    int64_t t = tok_lo + warp * TPW + sub;
    float cur[EPL], nxt[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) nxt[i] = 0.f;
    if (t < tok_hi) load_token<EPL, VEC>(logits + t * p.E, gl * EPL, p.E, cur);
    for (; t < tok_hi; t += kPass) {  // a whole G-lane group shares t
        if (t + kPass < tok_hi) load_token<EPL, VEC>(logits + (t + kPass) * p.E, gl * EPL, p.E, nxt);
        route_token<EPL, G>(cur, t, gl, lane, sub, smask, p, idx, w, ex + (t - tok_lo) * p.k);
#pragma unroll
        for (int i = 0; i < EPL; ++i) cur[i] = nxt[i];
    }
}

template <int EPL, int G, bool VEC>
__global__ void __launch_bounds__(kCountThreads)
    route_count_kernel(const float* __restrict__ logits, int32_t* __restrict__ idx,
                       float* __restrict__ w, RouteParams rp, CountArgs a) {
    grid_dependency_sync();
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ int64_t s_tile;
    __shared__ int s_last;
    __shared__ uint32_t s_tag;
    __shared__ uint64_t s_wait;
    if (threadIdx.x == 0) {
        s_tile = (int64_t)atomicAdd(&a.hdr->ticket, 1u);
        s_tag = next_tag(*(volatile uint32_t*)&a.hdr->epoch);
        const uint64_t wn = *(volatile uint64_t*)&a.hdr->wait_ns;
        s_wait = wn ? wn : kDefaultWaitNs;
    }
    zero_histograms(*reinterpret_cast<TileSmem*>(dsm), a.E);
    __syncthreads();
    const int64_t tile = s_tile;
    const uint32_t tag = s_tag;
    if (tile < a.ntiles) {
        TileSmem& sm = *reinterpret_cast<TileSmem*>(dsm);
        const int64_t Tr = a.T / a.R;
        const int64_t s = tile / a.nchunk, c = tile % a.nchunk;
        const int64_t tok_lo = s * Tr + c * kTileTokens;
        const int64_t tok_hi = min(tok_lo + kTileTokens, (s + 1) * Tr);
        route_tile<EPL, G, VEC>(logits, idx, w, rp, tok_lo, tok_hi, sm.ex);
        __syncthreads();
        count_tile<true>(a, tile, tag, s_wait, sm);
    }

    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&a.hdr->done, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    finish_counts(a, tag, dsm);
}

template <int EPL, int G>
moe_status launch_route_count(const moe_shape& s, bool vec, const float* logits, int32_t* idx,
                              float* w, const CountArgs& a, cudaStream_t stream) {
    const size_t smem = count_smem_bytes(a.R, a.E);
    const auto kern = vec ? route_count_kernel<EPL, G, true> : route_count_kernel<EPL, G, false>;
    const moe_status sst = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (sst != MOE_OK) return sst;
    const RouteParams rp{s.E, s.k, s.n_groups, s.topk_groups, s.group_topn, &a.hdr->error};
    const int grid = (int)(a.ntiles > 0 ? a.ntiles : 1);
    return launch_k(kern, dim3(grid), dim3(kCountThreads), smem, stream, logits, idx, w, rp, a);
}

moe_status launch_counts(const CountArgs& a, cudaStream_t stream) {
    const size_t smem = count_smem_bytes(a.R, a.E);
    const moe_status sst =
        ensure_dynamic_smem(reinterpret_cast<const void*>(send_counts_kernel), smem);
    if (sst != MOE_OK) return sst;
    const int grid = (int)(a.ntiles > 0 ? a.ntiles : 1);
    return launch_k(send_counts_kernel, dim3(grid), dim3(kCountThreads), smem, stream, a);
}

CountArgs count_args(const moe_shape& s, const WsLayout& L, void* ws, const int32_t* idx,
                     int32_t* expert_counts, int32_t* rank_expert_counts, int32_t* send_counts,
                     int64_t* send_off, int64_t* recv_off, int64_t* recv_base) {
    CountArgs a;
    a.idx = idx;
    a.T = s.T;
    a.E = s.E;
    a.k = s.k;
    a.R = s.R;
    a.nchunk = L.nchunk;
    a.ntiles = L.ntiles;
    a.status = ws_ptr<uint64_t>(ws, L.status);
    a.cnt_se = ws_ptr<int32_t>(ws, L.cnt_se);
    a.sstart = ws_ptr<int32_t>(ws, L.sstart);
    a.rstart = ws_ptr<int32_t>(ws, L.rstart);
    a.cpre = ws_ptr<int32_t>(ws, L.cpre);
    a.eoff = ws_ptr<int32_t>(ws, L.eoff);
    a.rank = ws_ptr<int32_t>(ws, L.rank);
    a.hdr = ws_ptr<WsHeader>(ws, 0);
    a.expert_counts = expert_counts;
    a.rank_expert_counts = rank_expert_counts;
    a.send_counts = send_counts;
    a.send_off = send_off;
    a.recv_off = recv_off;
    a.recv_base = recv_base;
    a.mark_failure = 0;
    return a;
}

moe_status check_count_outputs(const int32_t* expert_counts, const int32_t* rank_expert_counts,
                               const int32_t* send_counts, const int64_t* send_off,
                               const int64_t* recv_off, const int64_t* recv_base) {
    if (!expert_counts || !rank_expert_counts || !send_counts || !send_off || !recv_off ||
        !recv_base)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(expert_counts, 4) || !aligned(rank_expert_counts, 4) ||
        !aligned(send_counts, 4) || !aligned(send_off, 8) || !aligned(recv_off, 8) ||
        !aligned(recv_base, 8))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_build_send_counts(const moe_shape* shape, const int32_t* idx,
                                            int32_t* expert_counts, int32_t* rank_expert_counts,
                                            int32_t* send_counts, int64_t* send_off,
                                            int64_t* recv_off, int64_t* recv_base,
                                            void* workspace, size_t ws_bytes,
                                            cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const WsLayout L = ws_layout(s);
    if (!workspace || !aligned(workspace, 256) || ws_bytes < L.total) return MOE_ERR_INVALID_ARG;
    if (!need(idx, s, 4)) return MOE_ERR_INVALID_ARG;
    if ((st = check_count_outputs(expert_counts, rank_expert_counts, send_counts, send_off,
                                  recv_off, recv_base)) != MOE_OK)
        return st;
    if (L.ntiles >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;

    return launch_counts(count_args(s, L, workspace, idx, expert_counts, rank_expert_counts,
                                    send_counts, send_off, recv_off, recv_base),
                         stream);
}

// ---------------------------------------------------------------------------
// Send counts for callers that cannot allocate device memory.
//
// The same count kernel, with its scratch (look-back status words, tile
// tickets, per-slot ranks, row tables) in a fixed file-scope device array
// instead of a caller-supplied workspace.  In host code the array's name is
// only a stand-in, not a device address, so the address is looked up with
// cudaGetSymbolAddress once per device and cached.

// 4 MiB on every device that loads the library, held until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace moe {
namespace {

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDeviceState {
    void* ptr = nullptr;  // device address of g_noalloc_scratch on that device
};
NoAllocDeviceState g_noalloc_state[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// First call on a device: resolve the array's device address and zero it on
// `stream` (stream-ordered, so the kernel that follows sees zeros).  That
// first call must not be captured into a graph: a captured zero-fill runs only
// when the graph does, while the cached address would already count as set up.
moe_status noalloc_scratch(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDeviceState& st = g_noalloc_state[dev];
    if (!st.ptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MOE_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return MOE_ERR_INVALID_ARG;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        if (cudaMemsetAsync(p, 0, kNoAllocScratchBytes, stream) != cudaSuccess) return MOE_ERR_CUDA;
        st.ptr = p;
    }
    *out = st.ptr;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_build_send_counts_noalloc(const moe_shape* shape, const int32_t* idx,
                                                    int32_t* expert_counts,
                                                    int32_t* rank_expert_counts,
                                                    int32_t* send_counts, int64_t* send_off,
                                                    int64_t* recv_off, int64_t* recv_base,
                                                    cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const WsLayout L = ws_layout(s);
    if (L.total > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
    if (!need(idx, s, 4)) return MOE_ERR_INVALID_ARG;
    if ((st = check_count_outputs(expert_counts, rank_expert_counts, send_counts, send_off,
                                  recv_off, recv_base)) != MOE_OK)
        return st;
    void* ws = nullptr;
    if ((st = noalloc_scratch(stream, &ws)) != MOE_OK) return st;
    // The array keeps the last call's contents: clear its error word (and the
    // detail beside it) so that only this call's device-side checks count.
    if (cudaMemsetAsync(ws, 0, 2 * sizeof(uint32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
    CountArgs a = count_args(s, L, ws, idx, expert_counts, rank_expert_counts, send_counts,
                             send_off, recv_off, recv_base);
    a.mark_failure = 1;  // no error word the caller can read: report in recv_base[R]
    return launch_counts(a, stream);
}

// Routing and counts in one launch (route_count_kernel) when the sub-warp
// routing handles the shape; otherwise the two launches one after the other.
// The results are those of moe_route_topk followed by moe_build_send_counts.
extern "C" moe_status moe_route_and_count(const moe_shape* shape, const float* logits, int32_t* idx,
                                          float* w, int32_t* expert_counts,
                                          int32_t* rank_expert_counts, int32_t* send_counts,
                                          int64_t* send_off, int64_t* recv_off, int64_t* recv_base,
                                          void* workspace, size_t ws_bytes, cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const WsLayout L = ws_layout(s);
    if (!workspace || !aligned(workspace, 256) || ws_bytes < L.total) return MOE_ERR_INVALID_ARG;
    if (!need(logits, s, 4) || !need(idx, s, 4) || !need(w, s, 4)) return MOE_ERR_INVALID_ARG;
    if ((st = check_count_outputs(expert_counts, rank_expert_counts, send_counts, send_off,
                                  recv_off, recv_base)) != MOE_OK)
        return st;
    if (L.ntiles >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
    int epl = 4, g = 1;
    fast_geometry(s.E, epl, g);
    if (!fast_groups_ok(s, epl)) {
        if ((st = moe_route_topk(shape, logits, idx, w, workspace, stream)) != MOE_OK) return st;
        return moe_build_send_counts(shape, idx, expert_counts, rank_expert_counts, send_counts,
                                     send_off, recv_off, recv_base, workspace, ws_bytes, stream);
    }
    const CountArgs a = count_args(s, L, workspace, idx, expert_counts, rank_expert_counts,
                                   send_counts, send_off, recv_off, recv_base);
    const bool vec = (s.E % 4 == 0) && aligned(logits, 16);
    if (epl == 4) {
        switch (g) {
            case 1: return launch_route_count<4, 1>(s, vec, logits, idx, w, a, stream);
            case 2: return launch_route_count<4, 2>(s, vec, logits, idx, w, a, stream);
            case 4: return launch_route_count<4, 4>(s, vec, logits, idx, w, a, stream);
            case 8: return launch_route_count<4, 8>(s, vec, logits, idx, w, a, stream);
            case 16: return launch_route_count<4, 16>(s, vec, logits, idx, w, a, stream);
            default: return launch_route_count<4, 32>(s, vec, logits, idx, w, a, stream);
        }
    }
    if (g <= 16) return launch_route_count<8, 16>(s, vec, logits, idx, w, a, stream);
    return launch_route_count<8, 32>(s, vec, logits, idx, w, a, stream);
}
