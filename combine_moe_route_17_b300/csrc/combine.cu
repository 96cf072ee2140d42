// Combine: y = sum_i G(x)_i E_i(x) (MoE survey, section 1.1, eq. 1; step 4
// "output combine" of its expert-parallel flow), the last step of the
// forward pass of "混合专家模型跨卡通信机制解析", section 四: expert outputs
// come back along the dispatch path and are weighted by the gates in the
// original token order.
//
// One warp per token gathers its k rows (K*U 16-byte loads in flight per
// lane, CombineUnroll), accumulates w_j * row_j in fp32 in j order with fmaf, rounds once to
// bf16 and writes the y row.  With the ranks in one GPU's memory the return
// all_to_all is fused into the gather; the staged form first moves the rows
// back to the send layout and gathers through send_pos, with the same result.
//
// Also here: the harness's scalar stand-in expert (not part of the timed path).
#include "moe_common.cuh"

namespace moe {
namespace {

// 4-warp CTAs: at k = 6 (54 registers) they pack 36 warps per SM against 32
// with 8-warp CTAs; c2's combine measured 79.7 -> 78.6 us, the others even.
constexpr int kCombWarps = 4;
constexpr int kMaxWaveId = MOE_MAX_EXPERTS;  // waves are < E <= 256

// Loads in flight per lane: K rows x U vector positions.  k = 7..8 takes two
// positions (16 loads, about 116 registers, 16 warps per SM) with plain
// L1-allocating loads: on B300 that gathers the c3 / c4 expert rows at 6.7-6.8
// TB/s where one position with L1::no_allocate loads gave 6.3.  k = 6 takes two
// positions with the L1::no_allocate loads (12 loads, 90 registers); plain
// loads made it slower.  The other k keep the form they had.
template <int K>
struct CombineUnroll {
    static constexpr int U = K <= 2 ? 4 : (K <= 4 ? 2 : (K >= 6 && K <= 8 ? 2 : 1));
    static constexpr bool kPlainLoads = K >= 7 && K <= 8;
};

// The last wave of token t: the largest wave among its k experts, or
// 0x7FFFFFFF (>= kMaxWaveId) if an expert index is out of range, which the
// caller reports.
template <int K>
__device__ __forceinline__ int last_wave(const int32_t* __restrict__ idx, int64_t t, int E, int Ew,
                                         int lane) {
    int wv = -1;
    if (lane < K) {
        const int e = __ldg(idx + t * K + lane);
        wv = (e >= 0 && e < E) ? e / Ew : 0x7FFFFFFF;
    }
    return (int)__reduce_max_sync(kFull, (unsigned)(wv + 1)) - 1;
}

// wave >= 0: only the tokens whose last wave is `wave` (their rows are all in
// once that wave's experts have run); wave < 0: every token.
template <int K>
__global__ void __launch_bounds__(kCombWarps* kWarp)
    combine_kernel(const uint4* __restrict__ rows, const int32_t* __restrict__ map,
                   const float* __restrict__ w, int64_t T, int H8, int64_t nrows,
                   uint4* __restrict__ y, uint32_t* err, const int32_t* __restrict__ idx, int E,
                   int Ew, int wave, int allow_dropped) {
    grid_dependency_sync();
    constexpr int U = CombineUnroll<K>::U;
    const int lane = threadIdx.x & (kWarp - 1);
    const int64_t nw = (int64_t)gridDim.x * kCombWarps;
    for (int64_t t = (int64_t)blockIdx.x * kCombWarps + (threadIdx.x >> 5); t < T; t += nw) {
        if (wave >= 0) {
            const int lw = last_wave<K>(idx, t, E, Ew, lane);
            if (lw >= kMaxWaveId) {  // an expert index out of range
                if (lane == 0 && err) raise_error(err, MOE_ERR_DEVICE_CHECK, (uint32_t)t);
                continue;
            }
            if (lw != wave) continue;
        }
        int32_t my_r = 0;
        float my_w = 0.0f;
        bool ok = false;
        if (lane < K) {
            const int32_t r = __ldg(map + t * K + lane);
            ok = (r >= 0 && (int64_t)r < nrows);
            if (ok) {
                my_r = r;
                my_w = __ldg(w + t * K + lane);
            } else if (err && !(allow_dropped && r == -1)) {
                raise_error(err, MOE_ERR_DEVICE_CHECK, (uint32_t)(t * K + lane));
            }
        }
        const unsigned okm = __ballot_sync(kFull, ok);
        const uint4* src[K];
        float wj[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            src[j] = rows + (int64_t)__shfl_sync(kFull, my_r, j) * H8;
            wj[j] = __shfl_sync(kFull, my_w, j);
        }
        uint4* yrow = y + t * H8;
        for (int base = 0; base < H8; base += kWarp * U) {
            uint4 v[K][U];
#pragma unroll
            for (int j = 0; j < K; ++j) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int p = base + u * kWarp + lane;
                    if (((okm >> j) & 1u) && p < H8)
                        v[j][u] = CombineUnroll<K>::kPlainLoads ? ld_v4(src[j] + p)
                                                                : ld_nc_v4(src[j] + p);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int p = base + u * kWarp + lane;
                float acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if ((okm >> j) & 1u) {
                        const uint4 a = v[j][u];
                        acc[0] = fmaf(wj[j], bf16_lo(a.x), acc[0]);
                        acc[1] = fmaf(wj[j], bf16_hi(a.x), acc[1]);
                        acc[2] = fmaf(wj[j], bf16_lo(a.y), acc[2]);
                        acc[3] = fmaf(wj[j], bf16_hi(a.y), acc[3]);
                        acc[4] = fmaf(wj[j], bf16_lo(a.z), acc[4]);
                        acc[5] = fmaf(wj[j], bf16_hi(a.z), acc[5]);
                        acc[6] = fmaf(wj[j], bf16_lo(a.w), acc[6]);
                        acc[7] = fmaf(wj[j], bf16_hi(a.w), acc[7]);
                    }
                }
                if (p < H8) {
                    uint4 o;
                    o.x = pack_bf16x2(acc[0], acc[1]);
                    o.y = pack_bf16x2(acc[2], acc[3]);
                    o.z = pack_bf16x2(acc[4], acc[5]);
                    o.w = pack_bf16x2(acc[6], acc[7]);
                    st_v4(yrow + p, o);
                }
            }
        }
    }
}

// nrows: rows of `rows` (T*k, or E*EC for the capacity layout, where a
// slot of -1 is a dropped slot, skipped without an error).
template <int K>
moe_status launch_combine_k(const moe_shape& s, const uint16_t* rows, const int32_t* map,
                            const float* w, uint16_t* y, uint32_t* err, const int32_t* idx,
                            int wave, int64_t nrows, int allow_dropped, cudaStream_t st) {
    const int grid = grid_for(s.T, kCombWarps);
    return launch_k(combine_kernel<K>, dim3(grid), dim3(kCombWarps * kWarp), 0, st,
                    reinterpret_cast<const uint4*>(rows), map, w, (int64_t)s.T, s.H / 8, nrows,
                    reinterpret_cast<uint4*>(y), err, idx, s.E, s.E / s.W, wave, allow_dropped);
}

using CombineLauncher = moe_status (*)(const moe_shape&, const uint16_t*, const int32_t*,
                                       const float*, uint16_t*, uint32_t*, const int32_t*, int,
                                       int64_t, int, cudaStream_t);

moe_status gather_combine(const moe_shape& s, const uint16_t* rows, const int32_t* map,
                          const float* w, uint16_t* y, uint32_t* err, cudaStream_t st,
                          const int32_t* idx = nullptr, int wave = -1, int64_t nrows = -1,
                          int allow_dropped = 0) {
    static constexpr CombineLauncher table[MOE_MAX_TOPK] = {
        &launch_combine_k<1>,  &launch_combine_k<2>,  &launch_combine_k<3>,
        &launch_combine_k<4>,  &launch_combine_k<5>,  &launch_combine_k<6>,
        &launch_combine_k<7>,  &launch_combine_k<8>,  &launch_combine_k<9>,
        &launch_combine_k<10>, &launch_combine_k<11>, &launch_combine_k<12>,
        &launch_combine_k<13>, &launch_combine_k<14>, &launch_combine_k<15>,
        &launch_combine_k<16>};
    if (nrows < 0) nrows = (int64_t)s.T * s.k;
    return table[s.k - 1](s, rows, map, w, y, err, idx, wave, nrows, allow_dropped, st);
}

// Stand-in expert: rows[r] = bf16_RN(scale_e * float(rows[r])), one fp32
// multiply per element, in place.  One warp per token, its k rows in turn
// (wave >= 0: only the rows of experts in that wave).
__global__ void __launch_bounds__(kCombWarps* kWarp)
    standin_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ slot_of,
                   const float* __restrict__ scale, int64_t T, int H8, int k, int E,
                   int64_t nrows, uint4* rows, int Ew, int wave) {
    grid_dependency_sync();
    const int lane = threadIdx.x & (kWarp - 1);
    const int64_t nw = (int64_t)gridDim.x * kCombWarps;
    for (int64_t t = (int64_t)blockIdx.x * kCombWarps + (threadIdx.x >> 5); t < T; t += nw) {
        for (int j = 0; j < k; ++j) {
            const int32_t r = __ldg(slot_of + t * k + j);
            const int e = __ldg(idx + t * k + j);
            if (r < 0 || (int64_t)r >= nrows || e < 0 || e >= E) continue;
            if (wave >= 0 && e / Ew != wave) continue;
            const float sc = __ldg(scale + e);
            uint4* row = rows + (int64_t)r * H8;
            for (int p = lane; p < H8; p += kWarp) {
                uint4 a = ld_v4(row + p);
                a.x = pack_bf16x2(__fmul_rn(sc, bf16_lo(a.x)), __fmul_rn(sc, bf16_hi(a.x)));
                a.y = pack_bf16x2(__fmul_rn(sc, bf16_lo(a.y)), __fmul_rn(sc, bf16_hi(a.y)));
                a.z = pack_bf16x2(__fmul_rn(sc, bf16_lo(a.z)), __fmul_rn(sc, bf16_hi(a.z)));
                a.w = pack_bf16x2(__fmul_rn(sc, bf16_lo(a.w)), __fmul_rn(sc, bf16_hi(a.w)));
                st_v4(row + p, a);
            }
        }
    }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_combine(const moe_shape* shape, const uint16_t* expert_out,
                                  const int32_t* slot_of, const float* w, void* workspace,
                                  size_t ws_bytes, unsigned flags, uint16_t* staging,
                                  const int32_t* send_pos, uint16_t* y, cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (flags & ~(MOE_STAGED | MOE_EXPERT_MAJOR)) return MOE_ERR_INVALID_ARG;
    const bool staged = (flags & MOE_STAGED) != 0;
    const bool em = (flags & MOE_EXPERT_MAJOR) != 0;
    if (!need(expert_out, s, 16) || !need(w, s, 4) || !need(y, s, 16)) return MOE_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (staged) {
        if (!workspace || !need(staging, s, 16) || !need(send_pos, s, 4)) return MOE_ERR_INVALID_ARG;
        if (ws_bytes < ws_layout(s).total) return MOE_ERR_INVALID_ARG;
    } else if (!need(slot_of, s, 4)) {
        return MOE_ERR_INVALID_ARG;
    }
    if (s.T == 0) return MOE_OK;
    uint32_t* err = workspace ? &ws_ptr<WsHeader>(workspace, 0)->error : nullptr;
    if (!staged) return gather_combine(s, expert_out, slot_of, w, y, err, stream);
    st = exchange_rows(s, workspace, ws_bytes, -1, 1, expert_out, staging, stream, em);
    if (st != MOE_OK) return st;
    return gather_combine(s, staging, send_pos, w, y, err, stream);
}

extern "C" moe_status moe_expert_standin(const moe_shape* shape, const int32_t* idx,
                                         const int32_t* slot_of, const float* scale,
                                         uint16_t* rows, cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (!need(idx, s, 4) || !need(slot_of, s, 4) || !need(rows, s, 16) || !scale ||
        !aligned(scale, 4))
        return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    return launch_k(standin_kernel, dim3(grid_for(s.T, kCombWarps)), dim3(kCombWarps * kWarp), 0,
                    stream, idx, slot_of, scale, (int64_t)s.T, s.H / 8, s.k, s.E,
                    (int64_t)s.T * s.k, reinterpret_cast<uint4*>(rows), s.E / s.W, -1);
}

extern "C" moe_status moe_expert_standin_wave(const moe_shape* shape, const int32_t* idx,
                                              const int32_t* slot_of, const float* scale,
                                              int wave, uint16_t* rows, cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (wave < -1 || wave >= s.W) return MOE_ERR_INVALID_ARG;
    if (!need(idx, s, 4) || !need(slot_of, s, 4) || !need(rows, s, 16) || !scale ||
        !aligned(scale, 4))
        return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    return launch_k(standin_kernel, dim3(grid_for(s.T, kCombWarps)), dim3(kCombWarps * kWarp), 0,
                    stream, idx, slot_of, scale, (int64_t)s.T, s.H / 8, s.k, s.E,
                    (int64_t)s.T * s.k, reinterpret_cast<uint4*>(rows), s.E / s.W, wave);
}

extern "C" moe_status moe_combine_wave(const moe_shape* shape, const uint16_t* expert_out,
                                       const int32_t* slot_of, const int32_t* idx, const float* w,
                                       void* workspace, int wave, uint16_t* y,
                                       cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (wave < -1 || wave >= s.W) return MOE_ERR_INVALID_ARG;
    if (!need(expert_out, s, 16) || !need(slot_of, s, 4) || !need(idx, s, 4) || !need(w, s, 4) ||
        !need(y, s, 16))
        return MOE_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    uint32_t* err = workspace ? &ws_ptr<WsHeader>(workspace, 0)->error : nullptr;
    return gather_combine(s, expert_out, slot_of, w, y, err, stream, idx, wave);
}

extern "C" moe_status moe_expert_standin_capacity(const moe_shape* shape, int64_t capacity,
                                                  const int32_t* idx, const int32_t* cap_slot,
                                                  const float* scale, uint16_t* cap_rows,
                                                  cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (capacity < 0) return MOE_ERR_INVALID_ARG;
    if (capacity * (int64_t)s.E >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    if (!need(idx, s, 4) || !need(cap_slot, s, 4) || !scale || !aligned(scale, 4))
        return MOE_ERR_INVALID_ARG;
    if (capacity > 0 && (!cap_rows || !aligned(cap_rows, 16))) return MOE_ERR_INVALID_ARG;
    if (s.T == 0 || capacity == 0) return MOE_OK;
    return launch_k(standin_kernel, dim3(grid_for(s.T, kCombWarps)), dim3(kCombWarps * kWarp), 0,
                    stream, idx, cap_slot, scale, (int64_t)s.T, s.H / 8, s.k, s.E,
                    capacity * s.E, reinterpret_cast<uint4*>(cap_rows), s.E / s.W, -1);
}

extern "C" moe_status moe_combine_capacity(const moe_shape* shape, int64_t capacity,
                                           const uint16_t* cap_out, const int32_t* cap_slot,
                                           const float* w, void* workspace, uint16_t* y,
                                           cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (capacity < 0) return MOE_ERR_INVALID_ARG;
    if (capacity * (int64_t)s.E >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    if (!need(cap_slot, s, 4) || !need(w, s, 4) || !need(y, s, 16)) return MOE_ERR_INVALID_ARG;
    if (capacity > 0 && (!cap_out || !aligned(cap_out, 16))) return MOE_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    uint32_t* err = workspace ? &ws_ptr<WsHeader>(workspace, 0)->error : nullptr;
    return gather_combine(s, cap_out, cap_slot, w, y, err, stream, nullptr, -1, capacity * s.E, 1);
}
