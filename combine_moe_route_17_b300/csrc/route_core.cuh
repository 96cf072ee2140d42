// Per-token routing core shared by the routing kernel and the fused
// routing-and-count kernel: softmax-of-top-k gating, G(x) = softmax(TopK(l,
// k)) with the other experts at -inf (MoE system-optimisation survey,
// crad.ict.ac.cn, section 1.1, eq. 2), and the constrained case of
// "不规则与流水化 AllToAll", section "EP 不规则 a2a 的来源", read as
// group-limited routing.
//
// G lanes (a power of two) route one token, lane q of the token's group
// holding the EPL contiguous experts [q*EPL, (q+1)*EPL).  route_keys routes
// a token from its lanes' ordered keys; load_token / route_token split the
// load from the key conversion, so a caller can issue the next token's loads
// before routing the current one.
//
// Group-limited routing is handled when a group is a whole number L of lanes
// (gsz % EPL == 0, L = gsz / EPL a power of two) and group_topn <= 4: each
// lane's 4 largest keys are merged over the L lanes of the group by a
// butterfly, and the group score is the fp32 sum of the group_topn largest
// values added in descending order.  Groups are then ranked by (score
// descending, group index ascending) and the topk_groups first kept.
//
// Each lane sorts its keys once; the k rounds then pick the largest head over
// the group's lanes and, among equal heads, the lowest lane (which holds the
// lowest expert index); lane (j mod G) of the token's group keeps the j-th
// choice and writes its idx / weight entries at the end.
#pragma once

#include "moe_common.cuh"

namespace moe {

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

// Compare-exchange for sort_lane: position a ends with the pair that comes
// first in (key descending, index ascending).
__device__ __forceinline__ void cmp_swap(uint32_t& ka, int& ia, uint32_t& kb, int& ib) {
    const bool sw = kb > ka || (kb == ka && ib < ia);
    const uint32_t k0 = sw ? kb : ka, k1 = sw ? ka : kb;
    const int i0 = sw ? ib : ia, i1 = sw ? ia : ib;
    ka = k0;
    kb = k1;
    ia = i0;
    ib = i1;
}

// Sorts EPL (4 or 8) (key, index) pairs by (key descending, index ascending)
// with Batcher's odd-even merge network (5 or 19 compare-exchanges).
template <int EPL>
__device__ __forceinline__ void sort_lane(uint32_t (&k)[EPL], int (&ix)[EPL]) {
    static_assert(EPL == 4 || EPL == 8, "sort_lane: 4 or 8 entries");
    constexpr int kNet4[5][2] = {{0, 1}, {2, 3}, {0, 2}, {1, 3}, {1, 2}};
    constexpr int kNet8[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6},
                                  {5, 7}, {1, 2}, {5, 6}, {0, 4}, {1, 5}, {2, 6}, {3, 7},
                                  {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
    if constexpr (EPL == 4) {
#pragma unroll
        for (int c = 0; c < 5; ++c) cmp_swap(k[kNet4[c][0]], ix[kNet4[c][0]], k[kNet4[c][1]], ix[kNet4[c][1]]);
    } else {
#pragma unroll
        for (int c = 0; c < 19; ++c) cmp_swap(k[kNet8[c][0]], ix[kNet8[c][0]], k[kNet8[c][1]], ix[kNet8[c][1]]);
    }
}

// Sorts four keys in descending order (the 4-input network of sort_lane,
// keys only).
__device__ __forceinline__ void sort4_keys(uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
    uint32_t h, l;
    h = max(a, b); l = min(a, b); a = h; b = l;
    h = max(c, d); l = min(c, d); c = h; d = l;
    h = max(a, c); l = min(a, c); a = h; c = l;
    h = max(b, d); l = min(b, d); b = h; d = l;
    h = max(b, c); l = min(b, c); b = h; c = l;
}

// a and b each hold four keys in descending order; a becomes the four
// largest of the eight, in descending order.  max(a[i], b[3 - i]) are those
// four (as a bitonic sequence), and two compare-exchange stages sort them.
__device__ __forceinline__ void merge_top4(uint32_t (&a)[4], const uint32_t (&b)[4]) {
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = max(a[i], b[3 - i]);
    const uint32_t h0 = max(c[0], c[2]), l0 = min(c[0], c[2]);
    const uint32_t h1 = max(c[1], c[3]), l1 = min(c[1], c[3]);
    a[0] = max(h0, h1);
    a[1] = min(h0, h1);
    a[2] = max(l0, l1);
    a[3] = min(l0, l1);
}

// The four largest of a lane's EPL (4 or 8) keys, in descending order.
template <int EPL>
__device__ __forceinline__ void lane_top4(const uint32_t (&key)[EPL], uint32_t (&tn)[4]) {
    tn[0] = key[0]; tn[1] = key[1]; tn[2] = key[2]; tn[3] = key[3];
    sort4_keys(tn[0], tn[1], tn[2], tn[3]);
    if constexpr (EPL == 8) {
        uint32_t hi[4] = {key[4], key[5], key[6], key[7]};
        sort4_keys(hi[0], hi[1], hi[2], hi[3]);
        merge_top4(tn, hi);
    }
}

__device__ __forceinline__ float4 ld_nc_f4(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// A token's EPL logits of lane gl (experts e0 = gl*EPL ..), raw: the key
// conversion and the finiteness check happen in route_token, so the loads
// stay in flight while the caller works on something else.
template <int EPL, bool VEC>
__device__ __forceinline__ void load_token(const float* row, int e0, int E, float (&v)[EPL]) {
    if (VEC) {
#pragma unroll
        for (int q = 0; q < EPL / 4; ++q) {
            float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e0 + 4 * q < E) f = ld_nc_f4(row + e0 + 4 * q);
            v[4 * q + 0] = f.x;
            v[4 * q + 1] = f.y;
            v[4 * q + 2] = f.z;
            v[4 * q + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) v[i] = (e0 + i < E) ? __ldg(row + e0 + i) : 0.f;
    }
}

struct RouteParams {
    int E, k, n_groups, topk_groups, group_topn;
    uint32_t* err;
};

// Routes token t from the ordered keys of lane gl's EPL experts (key 0 for
// padding) in its G-lane group (member mask smask); writes idx[t*k + j] and
// w[t*k + j] and, when ex_out is not null, ex_out[j] = the j-th expert.
// Every lane of the group must call it together.
// K > 0: k is the compile-time constant K (the rounds unroll); K = 0: k at
// run time.
template <int EPL, int G, int K = 0>
__device__ __forceinline__ void route_keys(uint32_t (&key)[EPL], int64_t t, int gl, int lane,
                                           int sub, unsigned smask, int E, int k, int n_groups,
                                           int topk_groups, int group_topn,
                                           int32_t* __restrict__ idx, float* __restrict__ w,
                                           uint16_t* ex_out) {
    const int kk = K > 0 ? K : k;
    if (n_groups > 1) {
        // The group's four largest keys: each lane's four largest, merged
        // over the group's L lanes (a bitonic merge of two sorted 4-lists per
        // step).
        const int L = E / n_groups / EPL;  // lanes per group
        uint32_t tn[4];
        lane_top4<EPL>(key, tn);
        for (int off = 1; off < L; off <<= 1) {
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = __shfl_xor_sync(smask, tn[q], off);
            merge_top4(tn, o);
        }
        float sc = key_value(tn[0]);
#pragma unroll
        for (int q = 1; q < 4; ++q)
            if (q < group_topn) sc = __fadd_rn(sc, key_value(tn[q]));
        const uint32_t gk = ordered_key(sc);
        const int g = gl / L;
        int rank = 0;
        for (int g2 = 0; g2 < n_groups; ++g2) {
            const uint32_t o = __shfl_sync(smask, gk, sub * G + g2 * L);
            rank += (o > gk) || (o == gk && g2 < g);
        }
        if (g >= n_groups || rank >= topk_groups) {
#pragma unroll
            for (int i = 0; i < EPL; ++i) key[i] = 0u;
        }
    }

    // Each lane sorts its keys (key descending, expert ascending); a round is
    // then one max over the lanes' heads, a ballot (the lowest lane whose head
    // equals it holds the lowest expert index: lanes hold ascending experts),
    // a shuffle for that expert, and a pop of the winner's head.
    constexpr int M = G >= 16 ? 1 : (G == 8 ? 2 : 4);  // choices per lane (k <= 16, k <= E)
    uint32_t sk[EPL];
    int si[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        sk[i] = key[i];
        si[i] = i;
    }
    sort_lane<EPL>(sk, si);
    uint32_t my_key[M];
    int my_e[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        my_key[m] = 0u;
        my_e[m] = 0;
    }
    uint32_t top_key = 0u;
    auto round = [&](int j) {
        const uint32_t bk = __reduce_max_sync(smask, sk[0]);
        const unsigned hit = __ballot_sync(smask, sk[0] == bk) & smask;
        const int wl = __ffs(hit) - 1;
        const int be = (wl - sub * G) * EPL + __shfl_sync(smask, si[0], wl);
        if (j == 0) top_key = bk;
        if (lane == wl) {
#pragma unroll
            for (int i = 0; i + 1 < EPL; ++i) {
                sk[i] = sk[i + 1];
                si[i] = si[i + 1];
            }
            sk[EPL - 1] = 0u;
        }
        if ((j & (G - 1)) == gl) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                if (m == j / G) {
                    my_key[m] = bk;
                    my_e[m] = be;
                }
            }
        }
    };
    if constexpr (K > 0) {
#pragma unroll
        for (int j = 0; j < K; ++j) round(j);
    } else {
        for (int j = 0; j < kk; ++j) round(j);
    }

    // softmax over the k chosen (eq. 2), shifted by the largest logit; the
    // butterfly gives every lane of the group the same sum
    const float top_v = key_value(top_key);
    float ex[M];
    float part = 0.0f;
#pragma unroll
    for (int m = 0; m < M; ++m) {
        ex[m] = 0.0f;
        if (gl + m * G < kk) {
            ex[m] = expf(key_value(my_key[m]) - top_v);
            part += ex[m];
        }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) part += __shfl_xor_sync(smask, part, off);
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const int j = gl + m * G;
        if (j < kk) {
            idx[t * kk + j] = my_e[m];
            w[t * kk + j] = __fdiv_rn(ex[m], part);
            if (ex_out) ex_out[j] = (uint16_t)my_e[m];
        }
    }
}

// route_keys from the raw logits v that load_token gave lane gl: the key
// conversion and the finiteness check, then the routing.
template <int EPL, int G>
__device__ __forceinline__ void route_token(const float (&v)[EPL], int64_t t, int gl, int lane,
                                            int sub, unsigned smask, const RouteParams& p,
                                            int32_t* __restrict__ idx, float* __restrict__ w,
                                            uint16_t* ex_out) {
    const int e0 = gl * EPL;
    uint32_t key[EPL];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        if (e0 + i < p.E) {
            bad |= !isfinite(v[i]);
            key[i] = ordered_key(v[i]);
        } else {
            key[i] = 0u;
        }
    }
    if (bad) raise_error(p.err, MOE_ERR_DEVICE_CHECK, (uint32_t)t);
    route_keys<EPL, G>(key, t, gl, lane, sub, smask, p.E, p.k, p.n_groups, p.topk_groups,
                       p.group_topn, idx, w, ex_out);
}

// Experts per lane and lanes per token of the sub-warp routing for E experts:
// four per lane up to E = 128 (a whole warp per token at 128: a 4-key lane
// sort and 4-deep pops cost less than two 8-key tokens per warp), eight above.
inline void fast_geometry(int E, int& epl, int& g) {
    epl = E > 128 ? 8 : 4;
    const int lanes = (E + epl - 1) / epl;
    g = 1;
    while (g < lanes) g <<= 1;
}

// Whether the sub-warp routing handles the shape's group-limited routing.
inline bool fast_groups_ok(const moe_shape& s, int epl) {
    if (s.n_groups <= 1) return true;
    const int gsz = s.E / s.n_groups;
    if (gsz % epl != 0 || s.group_topn > 4) return false;
    const int L = gsz / epl;
    return (L & (L - 1)) == 0;
}

}  // namespace moe
