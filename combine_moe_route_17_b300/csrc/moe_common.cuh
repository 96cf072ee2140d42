// Shared definitions of the B300 MoE dispatch/combine library: workspace
// layout, host-side validation and small device helpers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <utility>

#include "moe_route.h"

namespace moe {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xFFFFFFFFu;

// Look-back scan tile: a tile is up to kTileTokens consecutive tokens of ONE
// source rank, i.e. up to kTileTokens * k (<= 2048) expert slots.
constexpr int kTileTokens = 128;
constexpr int kCountThreads = 256;
constexpr int kCountWarps = kCountThreads / kWarp;

constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // bounded wait: 1 s

// ------------------------------------------------------------ workspace ----

// Header at offset 0 of every workspace.
struct WsHeader {
    uint32_t error;          // first moe_status raised on the device (0 = none)
    uint32_t error_info;     // detail of that error (tile, token, ...)
    uint32_t epoch;          // tag of the last completed count pass
    uint32_t ticket;         // tile tickets handed out in the running count pass
    uint32_t done;           // tiles finished in the running count pass
    int32_t fault_tile_p1;   // test hook: 1 + tile that skips publishing (0 = off)
    uint64_t wait_ns;        // bounded-wait limit (0 = kDefaultWaitNs)
};

// Byte offsets of the workspace regions for one shape.  Every region starts
// on a 256-byte boundary.
struct WsLayout {
    int64_t nchunk;      // tiles per source rank
    int64_t ntiles;      // R * nchunk
    size_t status;       // uint64 [R][nchunk][E]   look-back status words
    size_t cnt_se;       // int32  [R][E]           C[s][e]
    size_t sstart;       // int32  [R][E]           first send row of (s, e)
    size_t rstart;       // int32  [R][E]           first recv row of (s, e)
    size_t cpre;         // int32  [R][E]           slots of expert e in sources before s
    size_t eoff;         // int32  [E+1]            first row of expert e, expert-major layout
    size_t rank;         // int32  [T*k]            rank of (t, j) within (s, e)
    size_t total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline WsLayout ws_layout(const moe_shape& s) {
    WsLayout L;
    const int64_t Tr = s.R > 0 ? (int64_t)s.T / s.R : 0;
    L.nchunk = (Tr + kTileTokens - 1) / kTileTokens;
    L.ntiles = (int64_t)s.R * L.nchunk;
    size_t off = align256(sizeof(WsHeader));
    L.status = off;
    off = align256(off + sizeof(uint64_t) * (size_t)L.ntiles * (size_t)s.E);
    L.cnt_se = off;
    off = align256(off + sizeof(int32_t) * (size_t)s.R * s.E);
    L.sstart = off;
    off = align256(off + sizeof(int32_t) * (size_t)s.R * s.E);
    L.rstart = off;
    off = align256(off + sizeof(int32_t) * (size_t)s.R * s.E);
    L.cpre = off;
    off = align256(off + sizeof(int32_t) * (size_t)s.R * s.E);
    L.eoff = off;
    off = align256(off + sizeof(int32_t) * ((size_t)s.E + 1));
    L.rank = off;
    off = align256(off + sizeof(int32_t) * (size_t)s.T * s.k);
    L.total = off;
    return L;
}

template <typename T>
__host__ __device__ inline T* ws_ptr(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}
template <typename T>
__host__ __device__ inline const T* ws_ptr(const void* ws, size_t off) {
    return reinterpret_cast<const T*>(static_cast<const char*>(ws) + off);
}

// Look-back status word:
//   [63] 1, [62:34] pass tag, [33:32] flag, [31] 1, [30:0] count.
// Every other workspace region holds non-negative int32 values, whose bit 31
// is 0, so no stale data of another shape's layout can pass for a published
// word; words of an earlier pass carry another tag; zero-filled words have
// bit 63 clear.
constexpr uint64_t kFlagAggregate = 1;  // this tile's own count
constexpr uint64_t kFlagPrefix = 2;     // inclusive count of this and all earlier tiles
constexpr uint32_t kTagMask = 0x1FFFFFFFu;
constexpr uint64_t kStatusMarks = (1ull << 63) | (1ull << 31);

__host__ __device__ inline uint32_t next_tag(uint32_t epoch) {
    // tags cycle through 1 .. 2^29-1
    return (epoch % kTagMask) + 1u;
}
__device__ inline uint64_t pack_status(uint32_t tag, uint64_t flag, uint32_t count) {
    return kStatusMarks | ((uint64_t)(tag & kTagMask) << 34) | (flag << 32) |
           (uint64_t)(count & 0x7FFFFFFFu);
}
// Flag of a word published in pass `tag` (0 if not published in that pass).
__device__ inline uint64_t status_flag(uint64_t w, uint32_t tag) {
    if ((w & kStatusMarks) != kStatusMarks || (uint32_t)((w >> 34) & kTagMask) != tag) return 0;
    return (w >> 32) & 3u;
}
__device__ inline uint32_t status_count(uint64_t w) { return (uint32_t)(w & 0x7FFFFFFFu); }

// ------------------------------------------------------------ host side ----

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

inline moe_status validate(const moe_shape* sp) {
    if (!sp) return MOE_ERR_INVALID_ARG;
    const moe_shape& s = *sp;
    if (s.T < 0 || s.H < 8 || s.E < 1 || s.k < 1 || s.R < 1 || s.W < 1) return MOE_ERR_INVALID_ARG;
    if (s.H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (s.T % s.R != 0 || s.E % s.R != 0 || s.E % s.W != 0) return MOE_ERR_INVALID_ARG;
    if (s.k > s.E) return MOE_ERR_INVALID_ARG;
    if (s.E > MOE_MAX_EXPERTS || s.k > MOE_MAX_TOPK || s.R > MOE_MAX_RANKS) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)s.T * s.k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)s.T * s.k * s.H >= ((int64_t)1 << 46)) return MOE_ERR_UNSUPPORTED;
    if (s.n_groups < 1) return MOE_ERR_INVALID_ARG;
    if (s.n_groups > 1) {
        if (s.E % s.n_groups != 0) return MOE_ERR_INVALID_ARG;
        const int gsz = s.E / s.n_groups;
        if (s.topk_groups < 1 || s.topk_groups > s.n_groups) return MOE_ERR_INVALID_ARG;
        if (s.group_topn < 1 || s.group_topn > gsz) return MOE_ERR_INVALID_ARG;
        if ((int64_t)s.topk_groups * gsz < s.k) return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

// Per-token / per-slot buffers may be NULL only for an empty batch.
inline bool need(const void* p, const moe_shape& s, size_t align) {
    if (s.T == 0) return p == nullptr || aligned(p, align);
    return p != nullptr && aligned(p, align);
}

// Launches `kern` with programmatic stream serialization: the kernel may be
// scheduled while the previous kernel of the stream drains, and waits for it
// (griddepcontrol.wait, the first thing every kernel of this library does)
// before touching memory.  After another kind of predecessor, or none, it
// runs as an ordinary launch.
template <typename... KArgs, typename... Args>
inline moe_status launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

// ---------------------------------------------------- per-device state ----
// A process may drive several GPUs from several threads: the SM count and the
// dynamic shared memory limit a kernel was opted into (cudaFuncSetAttribute
// acts on the current device) are kept per device, under a lock.

constexpr int kMaxDevices = 64;

inline int current_device() {
    int d = 0;
    return cudaGetDevice(&d) == cudaSuccess ? d : 0;
}

// Multiprocessor count of the current device (148 on B300 if the query fails).
inline int device_sm_count() {
    static std::atomic<int> cache[kMaxDevices];  // 0: not queried yet
    const int d = current_device();
    const bool cached = d >= 0 && d < kMaxDevices;
    int n = cached ? cache[d].load(std::memory_order_relaxed) : 0;
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0)
        n = 148;
    if (cached) cache[d].store(n, std::memory_order_relaxed);
    return n;
}

// Makes sure `func` may use `bytes` of dynamic shared memory on the current
// device (a no-op up to the default 48 KB); each (device, kernel) is raised
// once, to the largest size asked for so far, so a launch under stream
// capture finds it already done after one eager call.
inline moe_status ensure_dynamic_smem(const void* func, size_t bytes) {
    if (bytes <= 48 * 1024) return MOE_OK;
    struct Entry {
        int dev;
        const void* func;
        size_t bytes;
    };
    constexpr int kEntries = 256;
    static Entry table[kEntries];
    static int used = 0;
    static std::mutex mu;
    const int d = current_device();
    std::lock_guard<std::mutex> lock(mu);
    int slot = -1;
    for (int i = 0; i < used; ++i)
        if (table[i].dev == d && table[i].func == func) slot = i;
    if (slot >= 0 && table[slot].bytes >= bytes) return MOE_OK;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    if (slot < 0 && used < kEntries) slot = used++;
    if (slot >= 0) table[slot] = Entry{d, func, bytes};
    return MOE_OK;
}

inline int grid_for(int64_t items, int per_block, int64_t cap = 1 << 30) {
    int64_t g = (items + per_block - 1) / per_block;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (int)g;
}

// Moves the rows of one wave (-1 = all) between the send layout and the recv
// layout (direction 0: send -> recv, 1: recv -> send).  Defined in dispatch.cu.
moe_status exchange_rows(const moe_shape& s, const void* ws, size_t ws_bytes, int wave,
                         int direction, const uint16_t* src, uint16_t* dst, cudaStream_t stream,
                         bool expert_major = false);

// ----------------------------------------------------------- device side ----

// Start of every kernel: wait until the previous kernel of the stream has
// completed and its writes are visible (immediate without a programmatic
// predecessor), then let the next kernel be scheduled; it waits the same way.
__device__ inline void grid_dependency_sync() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ inline void raise_error(uint32_t* err, uint32_t code, uint32_t info) {
    if (err && atomicCAS(err, 0u, code) == 0u) err[1] = info;
}

__device__ inline uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ inline uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ inline void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ inline unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// 16-byte loads that bypass L1 (read-only data) and stores with an
// evict-first hint (data not re-read by this kernel).
__device__ inline uint4 ld_nc_v4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ inline uint4 ld_v4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ inline void st_cs_v4(uint4* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ inline void st_v4(uint4* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// L2 eviction-priority policies (createpolicy) and 16-byte accesses that
// carry one: rows that a later call reads again stay in L2 with evict_last;
// rows streamed once leave first.
__device__ inline uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ inline uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ inline uint4 ld_nc_v4_hint(const uint4* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ inline void st_v4_hint(uint4* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

__device__ inline float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ inline float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ inline uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

}  // namespace moe
