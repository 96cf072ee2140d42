// Placement and concentration summaries of the per-expert counts.
//
// Greedy expert placement: MoE system-optimisation survey (crad.ict.ac.cn),
// section 4.2.2 "设备负载均衡" -- experts taken in descending order of load,
// each assigned to the least-loaded device, every device holding the same
// number of experts.  Ties go to the lower expert index and, among equally
// loaded ranks, the lower rank.  The per-rank Gini before (contiguous blocks)
// and after the placement uses the DODOCO summary's per-rank Gini.
//
// Fitted symmetric-Dirichlet alpha: the DODOCO summary's third summary of
// the send-count matrix, read as the method of moments of a
// Dirichlet-multinomial of the N slots over E experts, which solves to
// alpha = (N^2 - S2) / (E S2 - N^2 - (E-1) N) with S2 = sum c_e^2.
//
// Both run as one CTA on the device, so no host round trip sits between the
// count pass and a placement decision.
#include <math.h>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kPlaceThreads = 256;

__device__ void gini_of(const int64_t* L, int R, int64_t* num_out, int64_t* tot_out,
                        unsigned long long* s_num, unsigned long long* s_tot) {
    // sum_i sum_j |L_i - L_j| and sum L, exact in 64-bit integers
    const int tid = threadIdx.x;
    if (tid == 0) {
        *s_num = 0ull;
        *s_tot = 0ull;
    }
    __syncthreads();
    unsigned long long part = 0ull;
    for (int p = tid; p < R * R; p += kPlaceThreads) {
        const int64_t a = L[p / R], b = L[p % R];
        part += (unsigned long long)(a > b ? a - b : b - a);
    }
    atomicAdd(s_num, part);
    if (tid < R) atomicAdd(s_tot, (unsigned long long)L[tid]);
    __syncthreads();
    *num_out = (int64_t)*s_num;
    *tot_out = (int64_t)*s_tot;
    __syncthreads();
}

__global__ void __launch_bounds__(kPlaceThreads)
    place_kernel(const int32_t* __restrict__ c, int E, int R, int32_t* placement,
                 int32_t* relabel, moe_placement* out) {
    grid_dependency_sync();
    __shared__ int32_t s_c[MOE_MAX_EXPERTS];
    __shared__ int32_t s_order[MOE_MAX_EXPERTS];
    __shared__ int64_t s_load[MOE_MAX_RANKS];
    __shared__ int64_t s_before[MOE_MAX_RANKS];
    __shared__ int32_t s_filled[MOE_MAX_RANKS];
    __shared__ unsigned long long s_num, s_tot;
    const int tid = threadIdx.x, lane = tid & (kWarp - 1);
    const int per = E / R;
    for (int e = tid; e < E; e += kPlaceThreads) s_c[e] = __ldg(c + e);
    for (int d = tid; d < R; d += kPlaceThreads) {
        s_load[d] = 0;
        s_filled[d] = 0;
    }
    __syncthreads();
    // position of e in the order (count descending, index ascending)
    for (int e = tid; e < E; e += kPlaceThreads) {
        const int32_t ce = s_c[e];
        int pos = 0;
        for (int f = 0; f < E; ++f) pos += (s_c[f] > ce) || (s_c[f] == ce && f < e);
        s_order[pos] = e;
    }
    for (int d = tid; d < R; d += kPlaceThreads) {
        int64_t L = 0;
        for (int e = d * per; e < (d + 1) * per; ++e) L += s_c[e];
        s_before[d] = L;
    }
    __syncthreads();
    if (tid < kWarp) {
        // lane holds ranks lane and lane + 32; loads are below 2^31 (T*k)
        for (int i = 0; i < E; ++i) {
            const int e = s_order[i];
            uint32_t key = 0xFFFFFFFFu;
            int dk = 0x7FFFFFFF;
            for (int d = lane; d < R; d += kWarp) {
                if (s_filled[d] < per && (uint32_t)s_load[d] < key) {
                    key = (uint32_t)s_load[d];
                    dk = d;
                }
            }
            const uint32_t m = __reduce_min_sync(kFull, key);
            const int best = (int)__reduce_min_sync(kFull, key == m ? (uint32_t)dk : 0x7FFFFFFFu);
            if (lane == 0) {
                placement[e] = best;
                relabel[e] = best * per + s_filled[best];
                s_filled[best] += 1;
                s_load[best] += s_c[e];
            }
            __syncwarp();
        }
    }
    __syncthreads();
    int64_t nb, tb, na, ta;
    gini_of(s_before, R, &nb, &tb, &s_num, &s_tot);
    gini_of(s_load, R, &na, &ta, &s_num, &s_tot);
    if (tid == 0) {
        int64_t mb = 0, ma = 0;
        for (int d = 0; d < R; ++d) {
            mb = s_before[d] > mb ? s_before[d] : mb;
            ma = s_load[d] > ma ? s_load[d] : ma;
        }
        const int64_t den = 2 * (int64_t)R * tb;
        out->gini_num_before = nb;
        out->gini_num_after = na;
        out->gini_den = den;
        out->max_rank_load_before = mb;
        out->max_rank_load_after = ma;
        out->gini_before = den > 0 ? (double)nb / (double)den : 0.0;
        out->gini_after = den > 0 ? (double)na / (double)den : 0.0;
    }
}

__global__ void __launch_bounds__(kPlaceThreads)
    alpha_kernel(const int32_t* __restrict__ c, int E, double* alpha) {
    grid_dependency_sync();
    __shared__ unsigned long long s_n, s_s2;
    if (threadIdx.x == 0) {
        s_n = 0ull;
        s_s2 = 0ull;
    }
    __syncthreads();
    unsigned long long n = 0ull, s2 = 0ull;
    for (int e = threadIdx.x; e < E; e += kPlaceThreads) {
        const int32_t v = __ldg(c + e);
        const unsigned long long u = v > 0 ? (unsigned long long)v : 0ull;
        n += u;
        s2 += u * u;
    }
    atomicAdd(&s_n, n);
    atomicAdd(&s_s2, s2);
    __syncthreads();
    if (threadIdx.x == 0) {
        const int64_t N = (int64_t)s_n, S2 = (int64_t)s_s2;
        const int64_t num = N * N - S2;
        const int64_t den = (int64_t)E * S2 - N * N - (int64_t)(E - 1) * N;
        *alpha = (N == 0 || den <= 0) ? (double)INFINITY : (double)num / (double)den;
    }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_place_experts_greedy(const moe_shape* shape,
                                               const int32_t* expert_counts, int32_t* placement,
                                               int32_t* relabel, moe_placement* dev_out,
                                               cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (!expert_counts || !placement || !relabel || !dev_out || !aligned(expert_counts, 4) ||
        !aligned(placement, 4) || !aligned(relabel, 4) || !aligned(dev_out, 8))
        return MOE_ERR_INVALID_ARG;
    return launch_k(place_kernel, dim3(1), dim3(kPlaceThreads), 0, stream, expert_counts, s.E, s.R,
                    placement, relabel, dev_out);
}

extern "C" moe_status moe_dirichlet_alpha(const moe_shape* shape, const int32_t* expert_counts,
                                          double* dev_alpha, cudaStream_t stream) {
    using namespace moe;
    moe_status st = validate(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if ((int64_t)s.T * s.k > ((int64_t)1 << 27)) return MOE_ERR_UNSUPPORTED;
    if (!expert_counts || !dev_alpha || !aligned(expert_counts, 4) || !aligned(dev_alpha, 8))
        return MOE_ERR_INVALID_ARG;
    return launch_k(alpha_kernel, dim3(1), dim3(kPlaceThreads), 0, stream, expert_counts, s.E,
                    dev_alpha);
}
