/*
 * CPU ORACLE for MoE expert-parallel dispatch and combine -- TEST INFRASTRUCTURE.
 *
 * Plain, slow, single-threaded C that computes what the dispatch/combine hot
 * path must produce, written from the definitions on the source pages.  Only
 * the test suite, the smoke check and the bench's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Conventions (all arrays row-major, caller-owned):
 *   T tokens, H hidden, E experts, k experts per token, R virtual ranks, W waves.
 *   src(t)  = t / (T/R)        tokens split into R equal contiguous sources
 *   rank(e) = e / (E/R)        experts split into R equal contiguous blocks
 *   wave(e) = e / (E/W)        experts split into W equal contiguous waves
 *   bf16 values are passed as their uint16 bit patterns.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Round a real number to bfloat16 (nearest, ties to even); returns the bits. */
uint16_t oracle_bf16_from_double(double v);
double oracle_bf16_to_double(uint16_t b);
void oracle_bf16_round_array(const double* v, uint16_t* out, int64_t n);

/* Gating: softmax(TopK(logits, k)) with ties toward the lower expert index.
 * n_groups > 1 selects group-limited routing: group score = fp32 sum of the
 * group's group_topn best logits; keep topk_groups groups; top-k inside them. */
int oracle_route_topk(int T, int E, int k, int n_groups, int topk_groups, int group_topn,
                      const float* logits, int32_t* idx, float* w);

/* Send-count matrix, per-expert counts and alltoallv offsets. */
int oracle_send_counts(int T, int E, int k, int R, const int32_t* idx,
                       int32_t* C /*R*E*/, int32_t* c /*E*/, int32_t* S /*R*R*/,
                       int64_t* send_off /*R*(R+1)*/, int64_t* recv_off /*R*(R+1)*/,
                       int64_t* recv_base /*R+1*/);

/* Row maps of the dispatch: send row and recv row of every (t, j), and the
 * token of every recv row.  Any output may be NULL. */
int oracle_dispatch_maps(int T, int E, int k, int R, const int32_t* idx,
                         int32_t* send_pos /*T*k*/, int32_t* slot_of /*T*k*/,
                         int32_t* src_row /*T*k*/);

/* Row copies of the dispatch (bit copies of bf16 rows).  wave < 0 writes every
 * row; wave = w writes only the rows of experts in wave w.  send/recv may be NULL. */
int oracle_dispatch_rows(int T, int H, int E, int k, int W, int wave, const int32_t* idx,
                         const uint16_t* x, const int32_t* send_pos, const int32_t* slot_of,
                         uint16_t* send, uint16_t* recv);

/* Stand-in expert: out[r] = bf16_RN(fp32(s_e * fp32(recv[r]))) for the expert e of row r. */
int oracle_expert_standin(int T, int H, int k, const int32_t* idx, const int32_t* slot_of,
                          const float* scale, const uint16_t* recv, uint16_t* out);

/* Combine: y[t] = bf16_RN( sum_j w[t][j] * out[slot_of[t][j]] ) summed in fp64.
 * Tokens [t0, t1) only (t1 <= T); y is indexed by absolute token. */
int oracle_combine(int T, int H, int k, int t0, int t1, const uint16_t* out,
                   const int32_t* slot_of, const float* w, uint16_t* y);

/* Imbalance statistics of the per-expert counts c[E] over R ranks. */
typedef struct {
    int32_t max_load, min_load;
    int64_t gini_num, gini_den;
    double max_over_mean, hot_over_cold, gini;
} oracle_stats;

int oracle_imbalance_stats(int T, int E, int k, int R, const int32_t* c,
                           oracle_stats* st, int64_t* rank_load /*R, may be NULL*/);

/* Capacity-factor variant (MoE survey section 1.1, eq. 3 and step 2).
 * EC = ceil(k * f * T / E) computed as ((double)k * f * T) / E in IEEE double.
 * Maps: the slots of each expert are counted in (t, j) row-major order; a slot
 * at position p < EC is kept at row e*EC + p, later ones are dropped (-1);
 * dropped[e] counts them.  Rows: rows[e*EC + p] = x[t] for kept slots, every
 * other row (padding) zero.  Stand-in: out[r] = bf16_RN(fp32(s_{r/EC} *
 * fp32(rows[r]))).  Combine: y[t] = bf16_RN(sum over kept j of w_j *
 * out[cap_slot]) in fp64. */
int64_t oracle_expert_capacity(int T, int E, int k, double f);
int oracle_capacity_maps(int T, int E, int k, int64_t EC, const int32_t* idx, int32_t* cap_slot,
                         int32_t* dropped /*E*/);
int oracle_capacity_rows(int T, int H, int E, int k, int64_t EC, const uint16_t* x,
                         const int32_t* cap_slot, uint16_t* rows /*E*EC*H*/);
int oracle_capacity_standin(int H, int E, int64_t EC, const float* scale, const uint16_t* rows,
                            uint16_t* out);
int oracle_capacity_combine(int T, int H, int k, const uint16_t* out, const int32_t* cap_slot,
                            const float* w, uint16_t* y);

/* Greedy expert placement (MoE survey section 4.2.2): experts in descending
 * load (ties: lower index) each to the least-loaded rank with room (E/R
 * experts per rank; ties: lower rank).  relabel[e] = rank*(E/R) + the order
 * in which e joined its rank. */
int oracle_place_greedy(int E, int R, const int32_t* c, int32_t* placement, int32_t* relabel);
/* Per-rank Gini of the loads under a placement (exact numerator, denominator). */
int oracle_placement_gini(int E, int R, const int32_t* c, const int32_t* placement,
                          int64_t* num, int64_t* den, double* gini);
/* Fitted symmetric-Dirichlet alpha: (N^2 - S2) / (E S2 - N^2 - (E-1) N), +inf if
 * the denominator is <= 0; N = sum c_e <= 2^27. */
int oracle_dirichlet_alpha(int E, const int32_t* c, double* alpha);

/* Expert-major recv layout: rows ordered (rank, expert, source, token, slot),
 * i.e. (expert, token, slot); expert_off[e] = first row of expert e. */
int oracle_dispatch_maps_expert_major(int T, int E, int k, const int32_t* idx, int32_t* slot_of,
                                      int32_t* src_row, int64_t* expert_off /*E+1*/);

#ifdef __cplusplus
}
#endif
#endif
