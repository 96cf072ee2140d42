// moe_route_topk: softmax-of-top-k gating, G(x) = softmax(TopK(l, k)) with
// the other experts at -inf (MoE system-optimisation survey, crad.ict.ac.cn,
// section 1.1, eq. 2), plus the constrained case of "不规则与流水化 AllToAll",
// section "EP 不规则 a2a 的来源", read as group-limited routing.
//
// One warp per token.  Lane l holds the logits of experts l, l+32, l+64, ...
// (EPL = ceil(E/32) registers), converted to order-preserving unsigned keys.
// Each of the k selection rounds is a local max over EPL registers plus two
// warp reductions (redux.sync): the maximum key, then the lowest expert index
// holding it, which is exactly "higher logit first, ties to the lower index".
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;

// Order-preserving map from finite floats to unsigned keys; -0 maps like +0.
// Key 0 is reserved for "not selectable" (removed, masked or padding).
__device__ __forceinline__ uint32_t ordered_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    const uint32_t k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return k == 0u ? 1u : k;
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

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

template <int EPL>
void launch_route(const moe_shape& s, const float* logits, int32_t* idx, float* w, uint32_t* err,
                  cudaStream_t st) {
    const int grid = grid_for(s.T, kRouteWarps);
    route_topk_kernel<EPL><<<grid, kRouteWarps * kWarp, 0, st>>>(
        logits, idx, w, s.T, s.E, s.k, s.n_groups, s.topk_groups, s.group_topn, err);
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
    const int epl = (s.E + kWarp - 1) / kWarp;
    if (epl <= 1) launch_route<1>(s, logits, idx, w, err, stream);
    else if (epl <= 2) launch_route<2>(s, logits, idx, w, err, stream);
    else if (epl <= 4) launch_route<4>(s, logits, idx, w, err, stream);
    else launch_route<8>(s, logits, idx, w, err, stream);
    return launch_status();
}
