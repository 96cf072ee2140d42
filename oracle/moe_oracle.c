/*
 * CPU ORACLE for MoE expert-parallel dispatch and combine -- TEST INFRASTRUCTURE.
 *
 * Only tests, the smoke check and the bench's CPU-baseline leg may load this.
 * Plain single-threaded C, written from the source pages:
 *
 *  - gating G(x) = softmax(TopK(x W_gate, k)) with the other experts at -inf:
 *    MoE system-optimisation survey (crad.ict.ac.cn), section 1.1, eq. (2);
 *  - MoE output y = sum_i G(x)_i E_i(x): same survey, section 1.1, eq. (1), and
 *    step (4) "output combine" of its expert-parallel flow;
 *  - constrained (node/group-limited) versus free top-k routing, the send-count
 *    matrix and Alltoallv-style send/recv counts: "不规则与流水化 AllToAll",
 *    section "EP 不规则 a2a 的来源" and table "经典 vs 不规则";
 *  - permute_by_device -> all_to_all -> local experts -> all_to_all -> combine:
 *    "混合专家模型跨卡通信机制解析", section 四 (forward-pass pseudo-code);
 *  - same-expert rows contiguous after dispatch: survey section 1.1, step (2);
 *  - waves of E/W experts each: "不规则与流水化 AllToAll", section
 *    "Wave-Scheduled 流水化";
 *  - per-expert max/mean and per-rank Gini of the send-count matrix: DODOCO
 *    summary (gist.science), section "方法论"; hot/cold expert ratio: Lina blog
 *    post, section "推理".
 *
 * Readings where the pages are silent (tie-break toward the lower expert
 * index, renormalised softmax over the k chosen, fp32 group scores, the
 * recv layout (dst, src, expert, token, slot), fp64 combine rounded once to
 * bf16, the mean-absolute-difference Gini) are the ones the design notes list.
 *
 * Compile without fast-math and without FP contraction: every float
 * expression here must round exactly as IEEE binary32 / binary64 says.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 ---- */

/* bfloat16: 1 sign bit, 8 exponent bits (binary32's range), 7 fraction bits.
 * A finite nonzero magnitude a = f * 2^ex with f in [0.5, 1) has 8 significant
 * bits in bf16, so its spacing is 2^(ex-8); below 2^-126 the spacing is fixed
 * at 2^-133 (subnormals).  nearbyint() under the default rounding mode rounds
 * to nearest with ties to even. */
uint16_t oracle_bf16_from_double(double v) {
    if (isnan(v)) return (uint16_t)0x7FC0;
    uint32_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    double r = 0.0;
    if (isinf(a)) {
        r = a;
    } else if (a != 0.0) {
        int ex;
        (void)frexp(a, &ex);
        int q = ex - 8;
        if (q < -133) q = -133;
        r = ldexp(nearbyint(ldexp(a, -q)), q);
    }
    /* r has at most 8 significant bits, so the binary32 conversion is exact
     * (or overflows to +inf beyond the largest bf16, as it must). */
    float f = (float)r;
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (bits >> 16));
}

static float bf16_to_float(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

double oracle_bf16_to_double(uint16_t b) { return (double)bf16_to_float(b); }

void oracle_bf16_round_array(const double* v, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_double(v[i]);
}

/* ------------------------------------------------------------- routing ---- */

/* Expert a comes before expert b iff its logit is larger, or the logits are
 * equal (IEEE ==, so -0 == +0) and a has the lower index. */
static int comes_before(float la, int a, float lb, int b) {
    return (la > lb) || (la == lb && a < b);
}

int oracle_route_topk(int T, int E, int k, int n_groups, int topk_groups, int group_topn,
                      const float* logits, int32_t* idx, float* w) {
    if (T < 0 || E < 1 || k < 1 || k > E) return -1;
    if (n_groups < 1 || E % n_groups != 0) return -1;
    const int gsz = E / n_groups;
    if (n_groups > 1) {
        if (topk_groups < 1 || topk_groups > n_groups) return -1;
        if (group_topn < 1 || group_topn > gsz) return -1;
        if ((int64_t)topk_groups * gsz < k) return -1;
    }
    char* allowed = (char*)malloc((size_t)E);
    char* taken = (char*)malloc((size_t)E);
    float* gscore = (float*)malloc(sizeof(float) * (size_t)n_groups);
    char* gkept = (char*)malloc((size_t)n_groups);
    double* ex = (double*)malloc(sizeof(double) * (size_t)k);
    if (!allowed || !taken || !gscore || !gkept || !ex) return -3;
    int rc = 0;

    for (int t = 0; t < T && rc == 0; ++t) {
        const float* l = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e) {
            if (!isfinite(l[e])) rc = -2;
        }
        if (rc) break;

        /* Group-limited routing: the constrained (V3-style) case of the
         * irregular-AllToAll page, read as expert groups. */
        if (n_groups > 1) {
            for (int g = 0; g < n_groups; ++g) {
                memset(taken, 0, (size_t)E);
                float score = 0.0f;
                for (int n = 0; n < group_topn; ++n) {
                    int best = -1;
                    for (int e = g * gsz; e < (g + 1) * gsz; ++e) {
                        if (taken[e]) continue;
                        if (best < 0 || comes_before(l[e], e, l[best], best)) best = e;
                    }
                    if (best < 0) return -1; /* unreachable: group_topn <= group size */
                    taken[best] = 1;
                    score = (n == 0) ? l[best] : (score + l[best]); /* fp32 adds */
                }
                gscore[g] = score;
                gkept[g] = 0;
            }
            for (int n = 0; n < topk_groups; ++n) {
                int best = -1;
                for (int g = 0; g < n_groups; ++g) {
                    if (gkept[g]) continue;
                    if (best < 0 || comes_before(gscore[g], g, gscore[best], best)) best = g;
                }
                if (best < 0) return -1; /* unreachable: topk_groups <= n_groups */
                gkept[best] = 1;
            }
            for (int e = 0; e < E; ++e) allowed[e] = gkept[e / gsz];
        } else {
            memset(allowed, 1, (size_t)E);
        }

        /* TopK: k linear passes, each taking the first remaining expert in
         * the order; idx lists them in that order. */
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (!allowed[e] || taken[e]) continue;
                if (best < 0 || comes_before(l[e], e, l[best], best)) best = e;
            }
            if (best < 0) return -1; /* unreachable: k <= allowed experts */
            taken[best] = 1;
            idx[(size_t)t * k + j] = best;
        }

        /* softmax over the k kept logits (eq. 2: the others are -inf). */
        const double m = (double)l[idx[(size_t)t * k]];
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            ex[j] = exp((double)l[idx[(size_t)t * k + j]] - m);
            sum += ex[j];
        }
        for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = (float)(ex[j] / sum);
    }
    free(allowed);
    free(taken);
    free(gscore);
    free(gkept);
    free(ex);
    return rc;
}

/* -------------------------------------------------------------- counts ---- */

static int shape_ok(int T, int E, int k, int R) {
    if (T < 0 || E < 1 || k < 1 || k > E || R < 1) return 0;
    if (T % R != 0 || E % R != 0) return 0;
    return 1;
}

int oracle_send_counts(int T, int E, int k, int R, const int32_t* idx, int32_t* C, int32_t* c,
                       int32_t* S, int64_t* send_off, int64_t* recv_off, int64_t* recv_base) {
    if (!shape_ok(T, E, k, R)) return -1;
    const int Tr = T / R, Er = E / R;
    memset(C, 0, sizeof(int32_t) * (size_t)R * E);
    for (int t = 0; t < T; ++t) {
        const int s = t / Tr;
        for (int j = 0; j < k; ++j) {
            const int e = idx[(size_t)t * k + j];
            if (e < 0 || e >= E) return -2;
            C[(size_t)s * E + e] += 1;
        }
    }
    for (int e = 0; e < E; ++e) {
        int32_t tot = 0;
        for (int s = 0; s < R; ++s) tot += C[(size_t)s * E + e];
        c[e] = tot;
    }
    for (int s = 0; s < R; ++s) {
        for (int d = 0; d < R; ++d) {
            int32_t v = 0;
            for (int e = d * Er; e < (d + 1) * Er; ++e) v += C[(size_t)s * E + e];
            S[(size_t)s * R + d] = v;
        }
    }
    /* send_off[s][d] = sum_{d' < d} S[s][d'];  row s has R+1 entries. */
    for (int s = 0; s < R; ++s) {
        send_off[(size_t)s * (R + 1)] = 0;
        for (int d = 0; d < R; ++d)
            send_off[(size_t)s * (R + 1) + d + 1] = send_off[(size_t)s * (R + 1) + d] + S[(size_t)s * R + d];
    }
    /* recv_off[d][s] = sum_{s' < s} S[s'][d];  row d has R+1 entries. */
    for (int d = 0; d < R; ++d) {
        recv_off[(size_t)d * (R + 1)] = 0;
        for (int s = 0; s < R; ++s)
            recv_off[(size_t)d * (R + 1) + s + 1] = recv_off[(size_t)d * (R + 1) + s] + S[(size_t)s * R + d];
    }
    /* recv_base[d] = rows received by ranks before d. */
    recv_base[0] = 0;
    for (int d = 0; d < R; ++d) recv_base[d + 1] = recv_base[d] + recv_off[(size_t)d * (R + 1) + R];
    return 0;
}

/* ------------------------------------------------------------ dispatch ---- */

int oracle_dispatch_maps(int T, int E, int k, int R, const int32_t* idx, int32_t* send_pos,
                         int32_t* slot_of, int32_t* src_row) {
    if (!shape_ok(T, E, k, R)) return -1;
    const int Tr = T / R, Er = E / R;
    const size_t RE = (size_t)R * E;
    int32_t* C = (int32_t*)malloc(sizeof(int32_t) * RE);
    int32_t* c = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    int32_t* S = (int32_t*)malloc(sizeof(int32_t) * (size_t)R * R);
    int64_t* so = (int64_t*)malloc(sizeof(int64_t) * (size_t)R * (R + 1));
    int64_t* ro = (int64_t*)malloc(sizeof(int64_t) * (size_t)R * (R + 1));
    int64_t* rb = (int64_t*)malloc(sizeof(int64_t) * (size_t)(R + 1));
    int64_t* sstart = (int64_t*)malloc(sizeof(int64_t) * RE);
    int64_t* rstart = (int64_t*)malloc(sizeof(int64_t) * RE);
    int64_t* seen = (int64_t*)calloc(RE, sizeof(int64_t));
    if (!C || !c || !S || !so || !ro || !rb || !sstart || !rstart || !seen) return -3;
    int rc = oracle_send_counts(T, E, k, R, idx, C, c, S, so, ro, rb);
    if (rc == 0) {
        for (int s = 0; s < R; ++s) {
            /* Send layout: source s owns rows [s*(T/R)*k, (s+1)*(T/R)*k), in
             * (destination rank, expert, token, slot) order; since rank(e) is
             * monotone in e this is (expert, token, slot) order. */
            int64_t run = (int64_t)s * Tr * k;
            for (int e = 0; e < E; ++e) {
                sstart[(size_t)s * E + e] = run;
                run += C[(size_t)s * E + e];
            }
            /* Recv layout: rank d's rows start at recv_base[d]; inside, one
             * block per source s at recv_off[d][s]; inside a block, (expert,
             * token, slot) order. */
            for (int d = 0; d < R; ++d) {
                int64_t r = rb[d] + ro[(size_t)d * (R + 1) + s];
                for (int e = d * Er; e < (d + 1) * Er; ++e) {
                    rstart[(size_t)s * E + e] = r;
                    r += C[(size_t)s * E + e];
                }
            }
        }
        for (int t = 0; t < T; ++t) {
            const int s = t / Tr;
            for (int j = 0; j < k; ++j) {
                const int e = idx[(size_t)t * k + j];
                const size_t se = (size_t)s * E + e;
                const int64_t within = seen[se]++;
                if (send_pos) send_pos[(size_t)t * k + j] = (int32_t)(sstart[se] + within);
                const int64_t rr = rstart[se] + within;
                if (slot_of) slot_of[(size_t)t * k + j] = (int32_t)rr;
                if (src_row) src_row[rr] = t;
            }
        }
    }
    free(C); free(c); free(S); free(so); free(ro); free(rb);
    free(sstart); free(rstart); free(seen);
    return rc;
}

int oracle_dispatch_rows(int T, int H, int E, int k, int W, int wave, const int32_t* idx,
                         const uint16_t* x, const int32_t* send_pos, const int32_t* slot_of,
                         uint16_t* send, uint16_t* recv) {
    if (T < 0 || H < 1 || E < 1 || k < 1 || W < 1 || E % W != 0 || wave >= W) return -1;
    const int Ew = E / W;
    const size_t row = sizeof(uint16_t) * (size_t)H;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const int e = idx[(size_t)t * k + j];
            if (wave >= 0 && e / Ew != wave) continue;
            if (send) memcpy(send + (size_t)send_pos[(size_t)t * k + j] * H, x + (size_t)t * H, row);
            if (recv) memcpy(recv + (size_t)slot_of[(size_t)t * k + j] * H, x + (size_t)t * H, row);
        }
    }
    return 0;
}

/* ---------------------------------------------------- stand-in expert ---- */

int oracle_expert_standin(int T, int H, int k, const int32_t* idx, const int32_t* slot_of,
                          const float* scale, const uint16_t* recv, uint16_t* out) {
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const size_t r = (size_t)slot_of[(size_t)t * k + j];
            const float s = scale[idx[(size_t)t * k + j]];
            for (int h = 0; h < H; ++h) {
                const float p = s * bf16_to_float(recv[r * H + h]); /* one fp32 multiply */
                out[r * H + h] = oracle_bf16_from_double((double)p);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------- combine ---- */

int oracle_combine(int T, int H, int k, int t0, int t1, const uint16_t* out,
                   const int32_t* slot_of, const float* w, uint16_t* y) {
    if (t0 < 0 || t1 > T || t0 > t1 || H < 1 || k < 1) return -1;
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    if (!acc) return -3;
    for (int t = t0; t < t1; ++t) {
        for (int h = 0; h < H; ++h) acc[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            const double wj = (double)w[(size_t)t * k + j];
            const uint16_t* o = out + (size_t)slot_of[(size_t)t * k + j] * H;
            for (int h = 0; h < H; ++h) acc[h] += wj * oracle_bf16_to_double(o[h]);
        }
        for (int h = 0; h < H; ++h) y[(size_t)t * H + h] = oracle_bf16_from_double(acc[h]);
    }
    free(acc);
    return 0;
}

/* --------------------------------------------------------------- stats ---- */

int oracle_imbalance_stats(int T, int E, int k, int R, const int32_t* c, oracle_stats* st,
                           int64_t* rank_load) {
    if (!shape_ok(T, E, k, R)) return -1;
    const int Er = E / R;
    int32_t mx = c[0], mn = c[0];
    for (int e = 1; e < E; ++e) {
        if (c[e] > mx) mx = c[e];
        if (c[e] < mn) mn = c[e];
    }
    int64_t* L = (int64_t*)calloc((size_t)R, sizeof(int64_t));
    if (!L) return -3;
    int64_t total = 0;
    for (int e = 0; e < E; ++e) {
        L[e / Er] += c[e];
        total += c[e];
    }
    /* Gini as the mean absolute difference over all ordered pairs of rank
     * loads, divided by twice the mean: sum_i sum_j |L_i - L_j| / (2 R sum L). */
    int64_t num = 0;
    for (int i = 0; i < R; ++i)
        for (int j = 0; j < R; ++j) num += (L[i] > L[j]) ? (L[i] - L[j]) : (L[j] - L[i]);
    const int64_t den = 2 * (int64_t)R * total;
    st->max_load = mx;
    st->min_load = mn;
    st->gini_num = num;
    st->gini_den = den;
    st->gini = den > 0 ? (double)num / (double)den : 0.0;
    const int64_t slots = (int64_t)T * k;
    st->max_over_mean = slots > 0 ? (double)((int64_t)mx * E) / (double)slots : 0.0;
    if (slots == 0) st->hot_over_cold = 0.0;
    else st->hot_over_cold = mn > 0 ? (double)mx / (double)mn : INFINITY;
    if (rank_load)
        for (int d = 0; d < R; ++d) rank_load[d] = L[d];
    free(L);
    return 0;
}

/* ------------------------------------------------------------ capacity ---- */
/* Expert capacity, MoE system-optimisation survey (crad.ict.ac.cn), section
 * 1.1 "专家容量", eq. (3): EC = k * f * T / E, rounded up to whole rows.
 * Step 2 of the same section: samples beyond an expert's capacity are dropped,
 * unused capacity is filled with zeros. */

int64_t oracle_expert_capacity(int T, int E, int k, double f) {
    if (T < 0 || E < 1 || k < 1 || !(f >= 0.0)) return -1;
    return (int64_t)ceil((double)k * f * (double)T / (double)E);
}

int oracle_capacity_maps(int T, int E, int k, int64_t EC, const int32_t* idx, int32_t* cap_slot,
                         int32_t* dropped) {
    if (T < 0 || E < 1 || k < 1 || EC < 0) return -1;
    int64_t* seen = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    if (!seen) return -3;
    for (int e = 0; e < E; ++e) dropped[e] = 0;
    /* slots of each expert are counted in (t, j) order: the first EC are kept */
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const int e = idx[(size_t)t * k + j];
            if (e < 0 || e >= E) { free(seen); return -2; }
            const int64_t pos = seen[e]++;
            if (pos < EC) {
                cap_slot[(size_t)t * k + j] = (int32_t)((int64_t)e * EC + pos);
            } else {
                cap_slot[(size_t)t * k + j] = -1;
                dropped[e] += 1;
            }
        }
    }
    free(seen);
    return 0;
}

int oracle_capacity_rows(int T, int H, int E, int k, int64_t EC, const uint16_t* x,
                         const int32_t* cap_slot, uint16_t* rows) {
    if (T < 0 || H < 1 || E < 1 || k < 1 || EC < 0) return -1;
    memset(rows, 0, sizeof(uint16_t) * (size_t)E * (size_t)EC * (size_t)H); /* zero padding */
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            const int32_t r = cap_slot[(size_t)t * k + j];
            if (r >= 0) memcpy(rows + (size_t)r * H, x + (size_t)t * H, sizeof(uint16_t) * (size_t)H);
        }
    return 0;
}

int oracle_capacity_standin(int H, int E, int64_t EC, const float* scale, const uint16_t* rows,
                            uint16_t* out) {
    if (H < 1 || E < 1 || EC < 0) return -1;
    for (int64_t r = 0; r < (int64_t)E * EC; ++r) {
        const float s = scale[r / EC];
        for (int h = 0; h < H; ++h) {
            const float p = s * bf16_to_float(rows[(size_t)r * H + h]); /* one fp32 multiply */
            out[(size_t)r * H + h] = oracle_bf16_from_double((double)p);
        }
    }
    return 0;
}

int oracle_capacity_combine(int T, int H, int k, const uint16_t* out, const int32_t* cap_slot,
                            const float* w, uint16_t* y) {
    if (T < 0 || H < 1 || k < 1) return -1;
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    if (!acc) return -3;
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) acc[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            const int32_t r = cap_slot[(size_t)t * k + j];
            if (r < 0) continue; /* dropped: no expert output */
            const double wj = (double)w[(size_t)t * k + j];
            for (int h = 0; h < H; ++h) acc[h] += wj * oracle_bf16_to_double(out[(size_t)r * H + h]);
        }
        for (int h = 0; h < H; ++h) y[(size_t)t * H + h] = oracle_bf16_from_double(acc[h]);
    }
    free(acc);
    return 0;
}

/* ------------------------------------------------- placement and alpha ---- */
/* Greedy expert placement, MoE survey (crad.ict.ac.cn) section 4.2.2
 * "设备负载均衡": experts taken in descending order of load, each assigned to
 * the device with the smallest load so far, every device holding the same
 * number of experts (E/R).  Ties: the lower expert index first, the lower
 * rank among equally loaded ranks.  relabel[e] = d*(E/R) + (order in which e
 * joined rank d): renaming the experts by relabel makes the contiguous
 * expert-to-rank map realise the placement. */
int oracle_place_greedy(int E, int R, const int32_t* c, int32_t* placement, int32_t* relabel) {
    if (E < 1 || R < 1 || E % R != 0) return -1;
    const int per = E / R;
    int* order = (int*)malloc(sizeof(int) * (size_t)E);
    int64_t* load = (int64_t*)calloc((size_t)R, sizeof(int64_t));
    int* filled = (int*)calloc((size_t)R, sizeof(int));
    if (!order || !load || !filled) { free(order); free(load); free(filled); return -3; }
    for (int e = 0; e < E; ++e) order[e] = e;
    /* insertion sort: count descending, index ascending */
    for (int i = 1; i < E; ++i) {
        const int v = order[i];
        int j = i - 1;
        while (j >= 0 && (c[order[j]] < c[v] || (c[order[j]] == c[v] && order[j] > v))) {
            order[j + 1] = order[j];
            --j;
        }
        order[j + 1] = v;
    }
    for (int i = 0; i < E; ++i) {
        const int e = order[i];
        int best = -1;
        for (int d = 0; d < R; ++d) {
            if (filled[d] >= per) continue;
            if (best < 0 || load[d] < load[best]) best = d;
        }
        placement[e] = best;
        relabel[e] = best * per + filled[best];
        filled[best] += 1;
        load[best] += c[e];
    }
    free(order); free(load); free(filled);
    return 0;
}

/* Gini of the rank loads under a placement (DODOCO's per-rank Gini):
 * G = sum_i sum_j |L_i - L_j| / (2 R sum L), numerator and denominator exact. */
int oracle_placement_gini(int E, int R, const int32_t* c, const int32_t* placement,
                          int64_t* num, int64_t* den, double* gini) {
    if (E < 1 || R < 1) return -1;
    int64_t* L = (int64_t*)calloc((size_t)R, sizeof(int64_t));
    if (!L) return -3;
    for (int e = 0; e < E; ++e) {
        if (placement[e] < 0 || placement[e] >= R) { free(L); return -2; }
        L[placement[e]] += c[e];
    }
    int64_t n = 0, tot = 0;
    for (int i = 0; i < R; ++i) {
        tot += L[i];
        for (int j = 0; j < R; ++j) n += L[i] > L[j] ? L[i] - L[j] : L[j] - L[i];
    }
    *num = n;
    *den = 2 * (int64_t)R * tot;
    *gini = *den > 0 ? (double)n / (double)*den : 0.0;
    free(L);
    return 0;
}

/* Fitted symmetric-Dirichlet alpha of the per-expert counts (DODOCO, section
 * "方法论": the third summary of the send-count matrix).  The pages do not give
 * the fit; reading: method of moments for a Dirichlet-multinomial of the
 * N = sum c_e slots over E experts, i.e. the variance of a share c_e / N,
 *   Var = (1/E)(1 - 1/E) (N + E alpha) / (N (1 + E alpha)),
 * equated to the observed (1/E) sum_e (c_e/N - 1/E)^2.  With S2 = sum c_e^2
 * this solves exactly to
 *   alpha = (N^2 - S2) / (E S2 - N^2 - (E-1) N),
 * exact integers, then one double division.  A denominator <= 0 (counts no
 * more spread than multinomial sampling) gives +inf; all slots on one expert
 * gives 0.  Requires N <= 2^27 so that E S2 fits in int64. */
int oracle_dirichlet_alpha(int E, const int32_t* c, double* alpha) {
    if (E < 1) return -1;
    int64_t N = 0, S2 = 0;
    for (int e = 0; e < E; ++e) {
        if (c[e] < 0) return -2;
        N += c[e];
        S2 += (int64_t)c[e] * c[e];
    }
    if (N > ((int64_t)1 << 27)) return -1;
    const int64_t num = N * N - S2;
    const int64_t den = (int64_t)E * S2 - N * N - (int64_t)(E - 1) * N;
    if (N == 0 || den <= 0) *alpha = INFINITY;
    else *alpha = (double)num / (double)den;
    return 0;
}

/* ------------------------------------------------ expert-major layout ---- */
/* Recv rows ordered (destination rank, expert, source, token, slot): every
 * expert's rows are one contiguous run, which a per-expert GEMM consumes
 * directly (MoE survey section 1.1, step 2: samples of the same expert in
 * contiguous memory).  With contiguous expert blocks per rank this is the
 * order (expert, token, slot): row(t, j) = sum of the counts of the experts
 * before e + the position of (t, j) among e's slots in (t, j) order. */
int oracle_dispatch_maps_expert_major(int T, int E, int k, const int32_t* idx, int32_t* slot_of,
                                      int32_t* src_row, int64_t* expert_off /*E+1*/) {
    if (T < 0 || E < 1 || k < 1) return -1;
    int64_t* cnt = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int64_t* seen = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    if (!cnt || !seen) { free(cnt); free(seen); return -3; }
    for (int64_t n = 0; n < (int64_t)T * k; ++n) {
        if (idx[n] < 0 || idx[n] >= E) { free(cnt); free(seen); return -2; }
        cnt[idx[n]] += 1;
    }
    expert_off[0] = 0;
    for (int e = 0; e < E; ++e) expert_off[e + 1] = expert_off[e] + cnt[e];
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            const int e = idx[(size_t)t * k + j];
            const int64_t row = expert_off[e] + seen[e]++;
            slot_of[(size_t)t * k + j] = (int32_t)row;
            if (src_row) src_row[row] = t;
        }
    free(cnt); free(seen);
    return 0;
}
