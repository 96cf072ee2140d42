// moe_route_topk: softmax-of-top-k gating, G(x) = softmax(TopK(l, k)) with
// the other experts at -inf (MoE system-optimisation survey, crad.ict.ac.cn,
// section 1.1, eq. 2), plus the constrained case of "不规则与流水化 AllToAll",
// section "EP 不规则 a2a 的来源", read as group-limited routing.
//
// Logits become order-preserving unsigned keys.  Each of the k selection
// rounds is a local max over a lane's registers plus two reductions
// (redux.sync): the maximum key, then the lowest expert index holding it,
// which is exactly "higher logit first, ties to the lower index".
//
// route_fast_kernel (every plain shape, and group shapes whose groups are
// whole lanes) gives each token G lanes of EPL contiguous experts;
// route_topk_kernel (the other group shapes) gives each token a warp, lane l
// holding experts l, l+32, l+64, ...
#include "route_core.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;

// Warp-wide best entry among keys[i] of expert lane + 32 i: returns the key
// and the expert index (lowest index among equal keys).
template <int EPL>
__device__ __forceinline__ void warp_best(const uint32_t (&key)[EPL], int lane, uint32_t& best_key,
                                          int& best_e) {
    uint32_t lk = 0;
    int li = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        if (key[i] > lk) {
            lk = key[i];
            li = i;
        }
    }
    best_key = __reduce_max_sync(kFull, lk);
    const uint32_t cand = (lk == best_key) ? (uint32_t)(lane + kWarp * li) : 0xFFFFFFFFu;
    best_e = (int)__reduce_min_sync(kFull, cand);
}

template <int EPL>
__device__ __forceinline__ void clear_entry(uint32_t (&key)[EPL], int lane, int e) {
    if ((e & (kWarp - 1)) == lane) {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (i == (e >> 5)) key[i] = 0u;
    }
}

template <int EPL>
__global__ void __launch_bounds__(kRouteWarps* kWarp)
    route_topk_kernel(const float* __restrict__ logits, int32_t* __restrict__ idx,
                      float* __restrict__ w, int T, int E, int k, int n_groups, int topk_groups,
                      int group_topn, uint32_t* err) {
    grid_dependency_sync();
    __shared__ float s_gscore[kRouteWarps][MOE_MAX_EXPERTS];
    __shared__ uint8_t s_gkept[kRouteWarps][MOE_MAX_EXPERTS];

    const int lane = threadIdx.x & (kWarp - 1);
    const int wib = threadIdx.x >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * kRouteWarps;

    for (int64_t t = (int64_t)blockIdx.x * kRouteWarps + wib; t < T; t += nwarps) {
        const float* row = logits + t * E;
        uint32_t key[EPL];
        bool bad = false;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + kWarp * i;
            if (e < E) {
                const float v = __ldg(row + e);
                bad |= !isfinite(v);
                key[i] = ordered_key(v);
            } else {
                key[i] = 0u;
            }
        }
        if (__any_sync(kFull, bad) && lane == 0) raise_error(err, MOE_ERR_DEVICE_CHECK, (uint32_t)t);

        if (n_groups > 1) {
            // Group score: fp32 sum of the group's group_topn best logits,
            // added in selection (descending) order.
            const int gsz = E / n_groups;
            uint32_t tmp[EPL];
#pragma unroll
            for (int i = 0; i < EPL; ++i) tmp[i] = key[i];
            for (int g = 0; g < n_groups; ++g) {
                float score = 0.0f;
                for (int n = 0; n < group_topn; ++n) {
                    uint32_t gk[EPL];
#pragma unroll
                    for (int i = 0; i < EPL; ++i) {
                        const int e = lane + kWarp * i;
                        gk[i] = (e < E && e / gsz == g) ? tmp[i] : 0u;
                    }
                    uint32_t bk;
                    int be;
                    warp_best<EPL>(gk, lane, bk, be);
                    const float v = key_value(bk);
                    score = (n == 0) ? v : __fadd_rn(score, v);
                    clear_entry<EPL>(tmp, lane, be);
                }
                if (lane == 0) s_gscore[wib][g] = score;
            }
            __syncwarp();
            // keep the topk_groups best groups: higher score, then lower index
            uint32_t gkey[MOE_MAX_EXPERTS / kWarp];
#pragma unroll
            for (int i = 0; i < MOE_MAX_EXPERTS / kWarp; ++i) {
                const int g = lane + kWarp * i;
                gkey[i] = (g < n_groups) ? ordered_key(s_gscore[wib][g]) : 0u;
                if (g < n_groups) s_gkept[wib][g] = 0;
            }
            __syncwarp();
            for (int n = 0; n < topk_groups; ++n) {
                uint32_t bk;
                int bg;
                warp_best<MOE_MAX_EXPERTS / kWarp>(gkey, lane, bk, bg);
                if (lane == 0) s_gkept[wib][bg] = 1;
                clear_entry<MOE_MAX_EXPERTS / kWarp>(gkey, lane, bg);
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + kWarp * i;
                if (e < E && !s_gkept[wib][e / gsz]) key[i] = 0u;
            }
            __syncwarp();
        }

        // k selection rounds; lane j keeps the j-th choice
        int my_e = 0;
        float my_v = 0.0f, top_v = 0.0f;
        for (int j = 0; j < k; ++j) {
            uint32_t bk;
            int be;
            warp_best<EPL>(key, lane, bk, be);
            const float v = key_value(bk);
            if (j == 0) top_v = v;
            if (lane == j) {
                my_e = be;
                my_v = v;
            }
            clear_entry<EPL>(key, lane, be);
        }

        // softmax over the k chosen (eq. 2), shifted by the largest logit
        const float ex = (lane < k) ? expf(my_v - top_v) : 0.0f;
        float sum = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
        if (lane < k) {
            idx[t * k + lane] = my_e;
            w[t * k + lane] = __fdiv_rn(ex, sum);
        }
    }
}

// ---------------------------------------------------------------------------
// Sub-warp routing (route_core.cuh): a warp routes 32/G tokens at once, the
// reductions of a token running on its own G-lane member mask.

constexpr int kFastThreads = 256;

template <int EPL, int G, bool VEC, int K>
__global__ void __launch_bounds__(kFastThreads)
    route_fast_kernel(const float* __restrict__ logits, int32_t* __restrict__ idx,
                      float* __restrict__ w, int64_t T, int E, int k, int n_groups,
                      int topk_groups, int group_topn, uint32_t* err) {
    grid_dependency_sync();
    constexpr int TPW = kWarp / G;  // tokens per warp
    const int lane = threadIdx.x & (kWarp - 1);
    const int sub = lane / G;
    const int gl = lane % G;
    const unsigned smask = (G == kWarp) ? kFull : (((1u << G) - 1u) << (sub * G));
    const int64_t warp_id = ((int64_t)blockIdx.x * kFastThreads + threadIdx.x) / kWarp;
    const int64_t nwarps = (int64_t)gridDim.x * (kFastThreads / kWarp);

    for (int64_t tb = warp_id * TPW; tb < T; tb += nwarps * TPW) {
        const int64_t t = tb + sub;
        if (t >= T) continue;  // a whole G-lane group leaves; masks never cross groups
        // keys straight from the loads (the conversion waits on them anyway)
        const float* row = logits + t * E;
        const int e0 = gl * EPL;
        uint32_t key[EPL];
        bool bad = false;
        if (VEC) {
#pragma unroll
            for (int q = 0; q < EPL / 4; ++q) {
                if (e0 + 4 * q < E) {
                    const float4 v = ld_nc_f4(row + e0 + 4 * q);
                    bad |= !isfinite(v.x) || !isfinite(v.y) || !isfinite(v.z) || !isfinite(v.w);
                    key[4 * q + 0] = ordered_key(v.x);
                    key[4 * q + 1] = ordered_key(v.y);
                    key[4 * q + 2] = ordered_key(v.z);
                    key[4 * q + 3] = ordered_key(v.w);
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u) key[4 * q + u] = 0u;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                if (e0 + i < E) {
                    const float v = __ldg(row + e0 + i);
                    bad |= !isfinite(v);
                    key[i] = ordered_key(v);
                } else {
                    key[i] = 0u;
                }
            }
        }
        if (bad) raise_error(err, MOE_ERR_DEVICE_CHECK, (uint32_t)t);
        route_keys<EPL, G, K>(key, t, gl, lane, sub, smask, E, k, n_groups, topk_groups,
                              group_topn, idx, w, nullptr);
    }
}

template <int EPL, int G>
moe_status launch_fast(const moe_shape& s, bool vec, const float* logits, int32_t* idx, float* w,
                 uint32_t* err, int sms, cudaStream_t st) {
    const int64_t per_block = (int64_t)(kFastThreads / kWarp) * (kWarp / G);
    int64_t grid = (s.T + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sms * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    // the common k of vector-loaded shapes get kernels with k fixed at
    // compile time (the selection rounds unroll)
    auto kern = route_fast_kernel<EPL, G, false, 0>;
    if (vec) {
        switch (s.k) {
            case 2: kern = route_fast_kernel<EPL, G, true, 2>; break;
            case 6: kern = route_fast_kernel<EPL, G, true, 6>; break;
            case 8: kern = route_fast_kernel<EPL, G, true, 8>; break;
            default: kern = route_fast_kernel<EPL, G, true, 0>; break;
        }
    }
    return launch_k(kern, dim3((unsigned)grid), dim3(kFastThreads), 0, st, logits, idx, w,
                    (int64_t)s.T, s.E, s.k, s.n_groups, s.topk_groups, s.group_topn, err);
}

template <int EPL>
moe_status launch_route(const moe_shape& s, const float* logits, int32_t* idx, float* w,
                        uint32_t* err, cudaStream_t st) {
    const int grid = grid_for(s.T, kRouteWarps);
    return launch_k(route_topk_kernel<EPL>, dim3(grid), dim3(kRouteWarps * kWarp), 0, st, logits,
                    idx, w, s.T, s.E, s.k, s.n_groups, s.topk_groups, s.group_topn, err);
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_topk(const moe_shape* shape, const float* logits, int32_t* idx,
                                     float* w, void* workspace, cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (!need(logits, s, 4) || !need(idx, s, 4) || !need(w, s, 4)) return MOE_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    uint32_t* err = workspace ? &ws_ptr<WsHeader>(workspace, 0)->error : nullptr;
    int fepl = 4, fg = 1;
    fast_geometry(s.E, fepl, fg);
    if (fast_groups_ok(s, fepl)) {
        const bool vec = (s.E % 4 == 0) && aligned(logits, 16);
        const int sms = device_sm_count();
        if (fepl == 4) {
            switch (fg) {
                case 1: return launch_fast<4, 1>(s, vec, logits, idx, w, err, sms, stream);
                case 2: return launch_fast<4, 2>(s, vec, logits, idx, w, err, sms, stream);
                case 4: return launch_fast<4, 4>(s, vec, logits, idx, w, err, sms, stream);
                case 8: return launch_fast<4, 8>(s, vec, logits, idx, w, err, sms, stream);
                case 16: return launch_fast<4, 16>(s, vec, logits, idx, w, err, sms, stream);
                default: return launch_fast<4, 32>(s, vec, logits, idx, w, err, sms, stream);
            }
        }
        if (fg <= 16) return launch_fast<8, 16>(s, vec, logits, idx, w, err, sms, stream);
        return launch_fast<8, 32>(s, vec, logits, idx, w, err, sms, stream);
    }
    const int epl = (s.E + kWarp - 1) / kWarp;
    if (epl <= 1) return launch_route<1>(s, logits, idx, w, err, stream);
    if (epl <= 2) return launch_route<2>(s, logits, idx, w, err, stream);
    if (epl <= 4) return launch_route<4>(s, logits, idx, w, err, stream);
    return launch_route<8>(s, logits, idx, w, err, stream);
}
