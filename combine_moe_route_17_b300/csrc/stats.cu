// moe_imbalance_stats: the routing-imbalance summaries of the DODOCO summary
// (gist.science), section "方法论": per-expert max/mean token ratio (routing
// skew, independent of the expert-to-rank map) and a per-rank Gini
// coefficient, plus the hot/cold expert ratio of the Lina post, section "推理".
//
// Gini over the R rank loads L_d = sum_{rank(e)=d} c_e as the mean absolute
// difference over ordered pairs divided by twice the mean:
//   G = sum_i sum_j |L_i - L_j| / (2 R sum_d L_d).
// Numerator and denominator are exact int64; each ratio is one IEEE double
// division, so the result is bit-identical to any exact evaluation.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kStatsThreads = 256;

__global__ void __launch_bounds__(kStatsThreads)
    stats_kernel(const int32_t* __restrict__ c, int T, int E, int k, int R, moe_stats* out,
                 int64_t* rank_load) {
    grid_dependency_sync();
    __shared__ int64_t s_L[MOE_MAX_RANKS];
    __shared__ int32_t s_wmax[kStatsThreads / kWarp], s_wmin[kStatsThreads / kWarp];
    __shared__ long long s_part[kStatsThreads / kWarp];
    const int tid = threadIdx.x, lane = tid & (kWarp - 1), warp = tid >> 5;
    const int Er = E / R;

    int32_t mx = INT32_MIN, mn = INT32_MAX;
    for (int e = tid; e < E; e += kStatsThreads) {
        const int32_t v = c[e];
        mx = max(mx, v);
        mn = min(mn, v);
    }
    mx = __reduce_max_sync(kFull, mx);
    mn = __reduce_min_sync(kFull, mn);
    if (lane == 0) {
        s_wmax[warp] = mx;
        s_wmin[warp] = mn;
    }
    for (int d = tid; d < R; d += kStatsThreads) {
        int64_t L = 0;
        for (int e = d * Er; e < (d + 1) * Er; ++e) L += c[e];
        s_L[d] = L;
        if (rank_load) rank_load[d] = L;
    }
    __syncthreads();

    long long num = 0;
    for (int i = tid; i < R * R; i += kStatsThreads) {
        const int64_t a = s_L[i / R], b = s_L[i % R];
        num += a > b ? a - b : b - a;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) num += __shfl_xor_sync(kFull, num, o);
    if (lane == 0) s_part[warp] = num;
    __syncthreads();

    if (tid == 0) {
        int32_t gmax = s_wmax[0], gmin = s_wmin[0];
        long long gnum = 0;
        for (int w = 0; w < kStatsThreads / kWarp; ++w) {
            gmax = max(gmax, s_wmax[w]);
            gmin = min(gmin, s_wmin[w]);
            gnum += s_part[w];
        }
        int64_t total = 0;
        for (int d = 0; d < R; ++d) total += s_L[d];
        const int64_t den = 2 * (int64_t)R * total;
        const int64_t slots = (int64_t)T * k;
        moe_stats st;
        st.max_load = gmax;
        st.min_load = gmin;
        st.gini_num = gnum;
        st.gini_den = den;
        st.gini = den > 0 ? __ddiv_rn((double)gnum, (double)den) : 0.0;
        st.max_over_mean = slots > 0 ? __ddiv_rn((double)((int64_t)gmax * E), (double)slots) : 0.0;
        if (slots == 0) st.hot_over_cold = 0.0;
        else st.hot_over_cold = gmin > 0 ? __ddiv_rn((double)gmax, (double)gmin) : __longlong_as_double(0x7FF0000000000000ll);
        *out = st;
    }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_imbalance_stats(const moe_shape* shape, const int32_t* expert_counts,
                                          moe_stats* dev_stats, int64_t* rank_load,
                                          cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (!expert_counts || !dev_stats || !aligned(expert_counts, 4) || !aligned(dev_stats, 8))
        return MOE_ERR_INVALID_ARG;
    if (rank_load && !aligned(rank_load, 8)) return MOE_ERR_INVALID_ARG;
    return launch_k(stats_kernel, dim3(1), dim3(kStatsThreads), 0, stream, expert_counts, s.T, s.E,
                    s.k, s.R, dev_stats, rank_load);
}
