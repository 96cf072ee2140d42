/*
 * moe_route.h -- C ABI of the B300 MoE expert-parallel dispatch/combine path.
 *
 * The operations follow the forward pass of an expert-parallel MoE layer as
 * the source pages state it:
 *   gating -> permute_by_device -> all_to_all -> local experts -> all_to_all
 *   -> combine                        ("混合专家模型跨卡通信机制解析", section 四)
 * with G(x) = softmax(TopK(x W_gate, k)) (MoE system-optimisation survey,
 * crad.ict.ac.cn, section 1.1, eq. 2), y = sum_i G(x)_i E_i(x) (same section,
 * eq. 1), Alltoallv send/recv counts from the routing ("不规则与流水化
 * AllToAll", table "经典 vs 不规则" and section "与其他原语的衔接") and W waves
 * of E/W experts each (same page, section "Wave-Scheduled 流水化").
 *
 * The R expert-parallel ranks are partitions of ONE GPU's memory: source rank
 * s owns tokens [s*T/R, (s+1)*T/R); destination rank d owns experts
 * [d*E/R, (d+1)*E/R); wave w holds experts [w*E/W, (w+1)*E/W).  The alltoallv
 * is therefore a data-dependent device-memory transpose.
 *
 * Conventions for every entry point:
 *  - All buffer pointers are DEVICE pointers owned by the caller, 16-byte
 *    aligned, dense row-major.  bf16 tensors are passed as uint16_t bit
 *    patterns.  The library never allocates; all per-call state lives in the
 *    caller's workspace (moe_build_send_counts_noalloc alone uses a fixed
 *    array inside the library instead).
 *  - Calls are asynchronous on `stream`.  Shapes and pointers are validated on
 *    the host before any launch; a rejected call launches nothing and returns
 *    MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED.  A failed launch returns
 *    MOE_ERR_CUDA.  Conditions found on the device (a look-back wait that ran
 *    out, an index out of range, a non-finite logit) never trap: they set the
 *    workspace error word, the kernel skips the offending access, and
 *    moe_get_device_error() reports them.
 *  - One workspace must not be used by two calls that overlap on the GPU,
 *    with one exception: once moe_build_send_counts (or moe_route_and_count)
 *    has completed, the calls that follow it only read the workspace's tables
 *    and set its error word atomically (moe_dispatch, the combines, the
 *    experts), so those may overlap one another, as a wave pipeline does.
 *
 * Row layouts (R ranks, (t, j) = token t's j-th expert, e = idx[t][j]):
 *  - send (after permute_by_device): source s owns rows
 *    [s*(T/R)*k, (s+1)*(T/R)*k), ordered by (destination rank, expert,
 *    token, slot);
 *  - recv (after the exchange): destination d's rows start at recv_base[d];
 *    inside, one block per source s at recv_off[d][s]; inside a block rows
 *    are ordered by (expert, token, slot).  Same-expert rows are contiguous.
 *  The layout does not depend on W; a wave is a sub-range of every (s, d)
 *  block.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ROUTE_ABI_VERSION 1

#define MOE_MAX_EXPERTS 256 /* E <= 256                      */
#define MOE_MAX_TOPK 16     /* k <= 16                       */
#define MOE_MAX_RANKS 64    /* R <= 64                       */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* a shape, pointer or size the contract rejects */
    MOE_ERR_UNSUPPORTED = 2,  /* valid in principle, beyond this build's limits */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed            */
    MOE_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up              */
    MOE_ERR_DEVICE_CHECK = 5  /* a device-side check failed (index, non-finite)  */
} moe_status;

/* Problem shape.  Preconditions: T >= 0, T % R == 0, 1 <= E <= 256,
 * E % R == 0, 1 <= R <= 64, E % W == 0, 1 <= k <= min(E, 16), H >= 8,
 * H % 8 == 0 (16-byte rows), T*k < 2^31.  n_groups == 1 selects plain top-k;
 * n_groups > 1 selects group-limited routing, which needs E % n_groups == 0,
 * 1 <= topk_groups <= n_groups, 1 <= group_topn <= E/n_groups and
 * topk_groups * (E/n_groups) >= k. */
typedef struct {
    int32_t T, H, E, k, R, W;
    int32_t n_groups, topk_groups, group_topn;
} moe_shape;

/* Routing-imbalance summary (DODOCO summary, section "方法论": per-expert
 * max/mean and per-rank Gini of the send-count matrix; Lina post, section
 * "推理": hot/cold expert ratio). */
typedef struct {
    int32_t max_load, min_load;  /* max_e c_e, min_e c_e                        */
    int64_t gini_num, gini_den;  /* sum_i sum_j |L_i - L_j| and 2 R sum_d L_d    */
    double max_over_mean;        /* max_e c_e * E / (T k); 0 when T k == 0       */
    double hot_over_cold;        /* max/min; +inf if min == 0; 0 when T k == 0  */
    double gini;                 /* gini_num / gini_den; 0 when the sum is 0    */
} moe_stats;

/* Flags. */
#define MOE_STAGED 1u /* moe_dispatch / moe_combine: go through the send layout */
/* moe_dispatch / moe_combine: the expert-major recv layout.  Recv rows are
 * ordered (destination rank, expert, source, token, slot), so every expert's
 * rows form one run starting at expert_off[e] = sum of the counts of experts
 * before e (MoE survey section 1.1, step 2: same-expert samples contiguous),
 * which a per-expert GEMM consumes directly.  Rank d's rows still start at
 * recv_base[d]; only the order inside a rank changes.  Pass the same flag to
 * moe_combine in the staged form (the fused combine follows slot_of). */
#define MOE_EXPERT_MAJOR 2u
/* moe_dispatch: make the row copies with the bulk-copy engine, staged through
 * shared memory (cp.async.bulk global -> shared with mbarrier completion, then
 * shared -> global to each destination row), instead of through registers.
 * The results are identical.  Rows must fit three times in a warp's share of
 * a 200 KB shared-memory budget (H <= 34133); larger H returns
 * MOE_ERR_UNSUPPORTED.  On B300 the register path is the faster one for the
 * shapes measured; this form is kept for comparison. */
#define MOE_BULK_COPY 4u

/* Checks a shape against the preconditions above. */
moe_status moe_validate_shape(const moe_shape* shape);

/* Bytes of device workspace a shape needs (rank of every (t, j), look-back
 * status words, the per-(source, expert) row tables and a small header). */
moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes);

/* Zero-fills a workspace (stream-ordered).  Required once before first use;
 * afterwards every call leaves it ready for the next one, whatever shape the
 * next call has (the workspace must be large enough for that shape).  After
 * a call has reported MOE_ERR_TIMEOUT, zero-fill it again before reuse. */
moe_status moe_workspace_init(void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Top-k gating (survey section 1.1, eq. 2).  logits fp32 [T][E] -> idx int32
 * [T][k] listing the chosen experts by descending logit, ties toward the lower
 * expert index (IEEE compare, so -0 == +0), and w fp32 [T][k] =
 * exp(l_j - l_max) / sum_i exp(l_i - l_max) over the k chosen.  Group-limited
 * routing (n_groups > 1): a group's score is the fp32 sum of its group_topn
 * best logits in descending order; the topk_groups best groups (ties toward
 * the lower group) are kept and the k experts are chosen inside them.
 * workspace may be NULL; if given, non-finite logits set MOE_ERR_DEVICE_CHECK. */
moe_status moe_route_topk(const moe_shape* shape, const float* logits, int32_t* idx, float* w,
                          void* workspace, cudaStream_t stream);

/* Send-count matrix and alltoallv offsets ("不规则与流水化 AllToAll", table
 * "经典 vs 不规则": full send/recv-count matrices).  From idx int32 [T][k]:
 *   rank_expert_counts int32 [R][E]: C[s][e] = #{(t,j): src(t)=s, idx=e}
 *   expert_counts      int32 [E]   : c_e = sum_s C[s][e]
 *   send_counts        int32 [R][R]: S[s][d] = sum_{rank(e)=d} C[s][e]
 *   send_off  int64 [R][R+1]: send_off[s][d] = sum_{d'<d} S[s][d']
 *   recv_off  int64 [R][R+1]: recv_off[d][s] = sum_{s'<s} S[s'][d]
 *   recv_base int64 [R+1]   : recv_base[d] = sum_{d'<d} sum_s S[s][d']
 * and, in the workspace, every (t, j)'s rank among the pairs of the same
 * source and expert plus the row tables moe_dispatch needs.  One pass:
 * per-tile histograms then a decoupled look-back scan with a bounded wait. */
moe_status moe_build_send_counts(const moe_shape* shape, const int32_t* idx,
                                 int32_t* expert_counts, int32_t* rank_expert_counts,
                                 int32_t* send_counts, int64_t* send_off, int64_t* recv_off,
                                 int64_t* recv_base, void* workspace, size_t ws_bytes,
                                 cudaStream_t stream);

/* First row of every expert in the expert-major recv layout (MoE survey,
 * section 1.1, step 2: the samples of one expert are contiguous):
 * expert_off int32 [E+1] (device), expert_off[e] = sum of the counts c_e' of
 * the experts e' < e, expert_off[E] = T*k.  moe_build_send_counts computes
 * this table in its finishing CTA and keeps it in the workspace; this call
 * copies it out (stream-ordered, so call it after the count pass on the same
 * stream).  A per-expert GEMM reads expert e's rows as
 * [expert_off[e], expert_off[e+1]). */
moe_status moe_expert_offsets(const moe_shape* shape, const void* workspace, size_t ws_bytes,
                              int32_t* expert_off, cudaStream_t stream);

/* Dispatch: permute token rows by destination and exchange them
 * ("混合专家模型跨卡通信机制解析", section 四, steps 2-3).
 *   x bf16 [T][H] -> recv bf16 [T*k][H] (recv layout above), slot_of int32
 *   [T][k] (recv row of (t, j)), src_row int32 [T*k] (token of a recv row).
 * wave = -1 moves every row; wave = w in [0, W) moves only the rows of the
 * experts of wave w (and writes only their slot_of / src_row entries); calls
 * for w = 0..W-1 in stream order equal one call with wave = -1.  Since the
 * wave calls of one pass write disjoint rows and entries and only read the
 * workspace, they may also run at the same time, each on its own stream
 * after moe_build_send_counts (and joined before anything reads recv); on
 * B300 that is the faster form, the waves' launch ramps and tails
 * overlapping one another.
 * flags = 0: fused, x rows are written straight to their recv rows.
 * flags = MOE_STAGED: x -> send (send layout, send_pos int32 [T][k] = send
 *   row of (t, j)) then the send -> recv block transpose of the same wave.
 * send and send_pos may be NULL unless MOE_STAGED.  Needs the workspace
 * filled by moe_build_send_counts for the same idx. */
moe_status moe_dispatch(const moe_shape* shape, const uint16_t* x, const int32_t* idx,
                        const void* workspace, size_t ws_bytes, int wave, unsigned flags,
                        uint16_t* send, uint16_t* recv, int32_t* slot_of, int32_t* src_row,
                        int32_t* send_pos, cudaStream_t stream);

/* The local permute step alone (permute_by_device): x -> send rows of wave
 * `wave` (-1 = all) and send_pos; slot_of may be NULL. */
moe_status moe_permute_by_device(const moe_shape* shape, const uint16_t* x, const int32_t* idx,
                                 const void* workspace, size_t ws_bytes, int wave,
                                 uint16_t* send, int32_t* send_pos, int32_t* slot_of,
                                 cudaStream_t stream);

/* The exchange alone (all_to_all): copies the rows of wave `wave` (-1 = all)
 * between the send layout and the recv layout.  direction 0: src is in send
 * layout, dst in recv layout (dispatch); direction 1: the reverse (the
 * return trip of the expert outputs). */
moe_status moe_all_to_all(const moe_shape* shape, const void* workspace, size_t ws_bytes,
                          int wave, int direction, const uint16_t* src, uint16_t* dst,
                          cudaStream_t stream);

/* Combine (survey section 1.1, eq. 1 and step 4): y bf16 [T][H] with
 *   y[t] = bf16_RN( sum_{j=0..k-1} w[t][j] * float(expert_out[slot_of[t][j]]) )
 * accumulated in fp32 in j order (fused reverse exchange).
 * flags = MOE_STAGED: expert_out (recv layout) is first returned to the send
 * layout in `staging` bf16 [T*k][H] and gathered through send_pos; same y.
 * workspace may be NULL for the fused form; if given, a row index out of
 * range sets MOE_ERR_DEVICE_CHECK (the term is skipped). */
moe_status moe_combine(const moe_shape* shape, const uint16_t* expert_out,
                       const int32_t* slot_of, const float* w, void* workspace,
                       size_t ws_bytes, unsigned flags, uint16_t* staging,
                       const int32_t* send_pos, uint16_t* y, cudaStream_t stream);

/* Imbalance statistics of expert_counts int32 [E] (device): *dev_stats (a
 * device moe_stats) and, if rank_load is not NULL, the rank loads int64 [R]
 * L_d = sum_{rank(e)=d} c_e.  Integers are exact; each ratio is one IEEE
 * double division of exact integers. */
moe_status moe_imbalance_stats(const moe_shape* shape, const int32_t* expert_counts,
                               moe_stats* dev_stats, int64_t* rank_load, cudaStream_t stream);

/* Harness only, not part of the timed path: the per-expert scalar stand-in
 * expert, in place on recv rows: rows[slot_of[t][j]] =
 * bf16_RN(scale[idx[t][j]] * float(rows[slot_of[t][j]])) with one fp32
 * multiply ("混合专家模型跨卡通信机制解析", section 四, step 4, with a scalar
 * per expert standing in for local_experts). */
moe_status moe_expert_standin(const moe_shape* shape, const int32_t* idx, const int32_t* slot_of,
                              const float* scale, uint16_t* rows, cudaStream_t stream);

/* Wave-pipelined expert step (harness, like moe_expert_standin): the same
 * stand-in applied only to the rows whose expert is in wave `wave` (-1 = all
 * rows).  Calling it for wave w once moe_dispatch(wave=w) has completed lets
 * the experts of wave w run while wave w+1 is dispatched ("不规则与流水化
 * AllToAll", section "Wave-Scheduled 流水化": a wave's compute overlaps the
 * next wave's exchange). */
moe_status moe_expert_standin_wave(const moe_shape* shape, const int32_t* idx,
                                   const int32_t* slot_of, const float* scale, int wave,
                                   uint16_t* rows, cudaStream_t stream);

/* Combine of one wave of a wave-pipelined layer: y[t] as in moe_combine, for
 * exactly the tokens whose last wave -- the largest wave among their k
 * experts -- is `wave` (-1 = every token).  Waves are dispatched and run in
 * order, so all k rows of such a token are ready once wave `wave`'s experts
 * have run; each token's y is written once, accumulated in fp32 in j order,
 * and is bit-identical to moe_combine's.  Calling it for w = 0..W-1 writes
 * every y row; it lets the combine of wave w-1 overlap the experts of wave w
 * and the dispatch of wave w+1 (same page and section).  idx is the routing
 * int32 [T][k].  workspace may be NULL; if given, an expert index or row out
 * of range sets MOE_ERR_DEVICE_CHECK and the token or term is skipped. */
moe_status moe_combine_wave(const moe_shape* shape, const uint16_t* expert_out,
                            const int32_t* slot_of, const int32_t* idx, const float* w,
                            void* workspace, int wave, uint16_t* y, cudaStream_t stream);

/* ---- Capacity-factor variant (MoE survey section 1.1, "专家容量", eq. 3;
 * step 2 "样本分发": samples beyond an expert's capacity are dropped and
 * unused capacity is filled with zeros).  The rows live in a fixed
 * [E][capacity][H] buffer: expert e owns rows [e*capacity, (e+1)*capacity),
 * so rank d (experts [d*E/R, (d+1)*E/R)) owns a contiguous block of it. */

/* capacity = ceil(k * f * T / E), evaluated as ((double)k * f * T) / E in IEEE
 * double, then rounded up.  f >= 0; MOE_ERR_UNSUPPORTED if E * capacity
 * reaches 2^31.  Host only. */
moe_status moe_expert_capacity(const moe_shape* shape, double capacity_factor,
                               int64_t* capacity);

/* Capacity dispatch, after moe_build_send_counts on `workspace`.  The slots of
 * expert e are counted over all sources in (token, slot) order; the slot at
 * position p < capacity goes to row e*capacity + p of cap_rows (bf16
 * [E*capacity][H], a bit copy of x[t]) and cap_slot[t][j] = that row; later
 * slots are dropped: cap_slot = -1.  Rows p >= count_e of every expert are
 * zeroed.  dropped int32 [E] (may be NULL) receives max(count_e - capacity, 0).
 * cap_rows may be NULL when capacity == 0. */
moe_status moe_dispatch_capacity(const moe_shape* shape, int64_t capacity, const uint16_t* x,
                                 const int32_t* idx, const void* workspace, size_t ws_bytes,
                                 uint16_t* cap_rows, int32_t* cap_slot, int32_t* dropped,
                                 cudaStream_t stream);

/* Harness: the stand-in expert on the kept rows of the capacity buffer, in
 * place (padding rows stay zero, which is the stand-in of a zero row). */
moe_status moe_expert_standin_capacity(const moe_shape* shape, int64_t capacity,
                                       const int32_t* idx, const int32_t* cap_slot,
                                       const float* scale, uint16_t* cap_rows,
                                       cudaStream_t stream);

/* Capacity combine: y[t] = bf16_RN(sum over the kept j of w[t][j] *
 * float(cap_out[cap_slot[t][j]])), fp32 in j order; a dropped slot (-1)
 * contributes nothing (the gates are not renormalised); a token whose slots
 * were all dropped gets y = 0.  workspace may be NULL; if given, a row out of
 * range (other than -1) sets MOE_ERR_DEVICE_CHECK. */
moe_status moe_combine_capacity(const moe_shape* shape, int64_t capacity,
                                const uint16_t* cap_out, const int32_t* cap_slot,
                                const float* w, void* workspace, uint16_t* y,
                                cudaStream_t stream);

/* ---- Expert computation on the expert-major rows (MoE survey section 1.1,
 * step 3 "专家计算") ---- */

/* A linear expert on the 5th-generation tensor cores (tcgen05.mma, TMA, TMEM):
 *   out[r][n] = bf16_RN( sum_h rows[r][h] * weights[e(r)][n][h] ),
 * fp32 accumulation, where rows bf16 [T*k][H] are the expert-major recv rows
 * (moe_dispatch with MOE_EXPERT_MAJOR) and e(r) is the expert whose run holds
 * row r: expert e owns rows [sum_{e'<e} c_e', sum_{e'<=e} c_e') with c =
 * expert_counts int32 [E] (device, from moe_build_send_counts).  weights bf16
 * [E][N][H] (each output column a row of H values), out bf16 [T*k][N].
 * Requires H % 64 == 0 and N % 128 == 0; MOE_ERR_UNSUPPORTED otherwise or
 * if T*k/128 + E exceeds 65535 row tiles.  workspace may be NULL; if given, a
 * wait that runs out (2 s) sets MOE_ERR_TIMEOUT there.  With N == H, out
 * feeds moe_combine directly in place of the stand-in expert. */
moe_status moe_expert_gemm(const moe_shape* shape, const uint16_t* rows, const uint16_t* weights,
                           int N, const int32_t* expert_counts, uint16_t* out, void* workspace,
                           cudaStream_t stream);

/* A gated FFN expert on the same tensor-core kernel, two launches:
 *   hidden[r] = bf16_RN( silu(x W1_e^T) * (x W3_e^T) )      (fp32 throughout)
 *   out[r]    = bf16_RN( hidden[r] W2_e^T ),
 * silu(z) = z / (1 + exp(-z)).  w13 bf16 [E][2F][H] holds, per expert, F/128
 * blocks of 256 rows: 128 rows of W1 then the same 128 rows of W3 (so each
 * 256-column accumulator pairs gate and up columns); w2 bf16 [E][H][F];
 * hidden bf16 [T*k][F] is caller-owned scratch; out bf16 [T*k][H] feeds
 * moe_combine.  Requires H % 128 == 0 and F % 128 == 0. */
moe_status moe_expert_ffn(const moe_shape* shape, const uint16_t* rows, const uint16_t* w13,
                          const uint16_t* w2, int F, const int32_t* expert_counts,
                          uint16_t* hidden, uint16_t* out, void* workspace, cudaStream_t stream);

/* The tensor-core experts of one wave: moe_expert_gemm / moe_expert_ffn over
 * the experts [w*E/W, (w+1)*E/W) only (wave = -1: every expert).  In the
 * expert-major layout those experts' rows are one contiguous run, which is
 * all these calls read and write; other rows of out (and hidden) are left as
 * they are.  Each wave's rows come out bit-identical to the all-expert call's
 * (the same tiles, in the same order).  So moe_dispatch(wave=w), this call
 * and moe_combine_wave(w) pipeline the layer wave by wave ("不规则与流水化
 * AllToAll", section "Wave-Scheduled 流水化").  A wave outside [-1, W) is
 * MOE_ERR_INVALID_ARG. */
moe_status moe_expert_gemm_wave(const moe_shape* shape, const uint16_t* rows,
                                const uint16_t* weights, int N, const int32_t* expert_counts,
                                uint16_t* out, int wave, void* workspace, cudaStream_t stream);
moe_status moe_expert_ffn_wave(const moe_shape* shape, const uint16_t* rows, const uint16_t* w13,
                               const uint16_t* w2, int F, const int32_t* expert_counts,
                               uint16_t* hidden, uint16_t* out, int wave, void* workspace,
                               cudaStream_t stream);

/* ---- Placement and concentration summaries of the per-expert counts ---- */

/* Output of moe_place_experts_greedy (device memory).  Rank loads L_d are the
 * slots received by rank d; Gini = sum_i sum_j |L_i - L_j| / (2 R sum L) with
 * exact integer numerators and denominator and one double division each. */
typedef struct {
    int64_t gini_num_before;      /* contiguous blocks: rank(e) = e / (E/R) */
    int64_t gini_num_after;       /* the greedy placement */
    int64_t gini_den;
    int64_t max_rank_load_before;
    int64_t max_rank_load_after;
    double gini_before;
    double gini_after;
} moe_placement;

/* Greedy expert placement (MoE survey section 4.2.2, "设备负载均衡"):
 * experts taken in descending order of expert_counts int32 [E] (ties: lower
 * index first), each assigned to the least-loaded rank that still has room
 * for E/R experts (ties: lower rank).  placement int32 [E] receives each
 * expert's rank; relabel int32 [E] a new expert id, rank*(E/R) + the order in
 * which the expert joined its rank: mapping the routing indices through
 * relabel makes the contiguous expert-to-rank blocks of this library realise
 * the placement.  *dev_out receives the per-rank Gini and the largest rank
 * load before and after.  One CTA; all pointers are device pointers. */
moe_status moe_place_experts_greedy(const moe_shape* shape, const int32_t* expert_counts,
                                    int32_t* placement, int32_t* relabel,
                                    moe_placement* dev_out, cudaStream_t stream);

/* Fitted symmetric-Dirichlet alpha of expert_counts int32 [E] (the DODOCO
 * summary's third summary of the send-count matrix; the fit is not given on
 * the pages and is read as the method of moments of a Dirichlet-multinomial
 * of the N = sum c_e slots):
 *   alpha = (N^2 - S2) / (E S2 - N^2 - (E-1) N),  S2 = sum c_e^2,
 * exact integers and one double division; +inf when the denominator is <= 0
 * (counts no more spread than sampling noise) or N = 0; 0 when every slot is
 * on one expert.  *dev_alpha is device memory.  MOE_ERR_UNSUPPORTED if
 * T*k > 2^27. */
moe_status moe_dirichlet_alpha(const moe_shape* shape, const int32_t* expert_counts,
                               double* dev_alpha, cudaStream_t stream);

/* moe_build_send_counts for callers that cannot allocate device memory (the
 * source pages have no counterpart of this call).  Some callers cannot call
 * cudaMalloc: a memory planner that must learn the alltoallv counts before
 * any exchange buffer exists, a runtime whose device memory all belongs to
 * its own pool, or code that may not allocate at that point.  This entry
 * point takes only the inputs and outputs of moe_build_send_counts; its
 * scratch is a fixed 4 MiB device array inside the library, which every GPU
 * that loads the library holds until the process exits.
 *  - Shapes whose workspace (moe_workspace_size) exceeds 4 MiB are rejected
 *    with MOE_ERR_UNSUPPORTED; nothing is allocated, ever.
 *  - Runs on the current device.  The first call on a device looks up the
 *    array's address and zero-fills it on `stream`; make that first call
 *    before any stream capture (a first call on a capturing stream returns
 *    MOE_ERR_INVALID_ARG and launches nothing).  The address is kept for
 *    the life of the process: after cudaDeviceReset on a device, do not
 *    call this entry point again on that device in the same process.
 *  - Every call shares the one array, which keeps the last call's contents:
 *    calls that overlap on the GPU (concurrent streams, several host
 *    threads) race and must be serialised by the caller.  Each call clears
 *    the array's error word first (stream-ordered).
 *  - A failure found on the device (an expert index out of range, a
 *    look-back wait that ran out) cannot be returned by the call, which has
 *    already returned; it shows in the outputs instead: recv_base[R], the
 *    total row count, is set to -(moe_status), e.g. -MOE_ERR_DEVICE_CHECK,
 *    and the other outputs are then not meaningful.  A non-negative
 *    recv_base[R] (which equals T*k) means the pass found nothing wrong.
 *  - The per-slot ranks and row tables it computes stay in the array, so
 *    moe_dispatch still needs a workspace filled by moe_build_send_counts. */
moe_status moe_build_send_counts_noalloc(const moe_shape* shape, const int32_t* idx,
                                         int32_t* expert_counts, int32_t* rank_expert_counts,
                                         int32_t* send_counts, int64_t* send_off,
                                         int64_t* recv_off, int64_t* recv_base,
                                         cudaStream_t stream);

/* moe_route_topk followed by moe_build_send_counts, in one launch where the
 * sub-warp routing handles the shape (every plain shape, and group-limited
 * shapes whose groups are a power-of-two number of whole lanes with
 * group_topn <= 4); otherwise it makes the two launches.  Each look-back tile
 * routes its own tokens and keeps their experts in shared memory for the
 * histogram (the fused gating-and-counting kernel the MoE survey, section 4.5,
 * names among its kernel optimisations).  Arguments, outputs and workspace are
 * those of the two calls; the results are bit-identical to them.  On B300 the
 * two launches are the faster choice for the shapes measured: the routing is
 * issue-bound and wants every warp slot of the GPU, while the fused launch
 * runs it on one CTA per look-back tile. */
moe_status moe_route_and_count(const moe_shape* shape, const float* logits, int32_t* idx, float* w,
                               int32_t* expert_counts, int32_t* rank_expert_counts,
                               int32_t* send_counts, int64_t* send_off, int64_t* recv_off,
                               int64_t* recv_base, void* workspace, size_t ws_bytes,
                               cudaStream_t stream);

/* Synchronises `stream`, returns the workspace error word as a status
 * (MOE_OK if clear) and clears it. */
moe_status moe_get_device_error(void* workspace, cudaStream_t stream);

/* Test hook: makes the next moe_build_send_counts and moe_route_and_count
 * calls skip publishing the look-back status of tile `tile` (tile < 0 switches it off), and sets the
 * bounded wait to `wait_ns` nanoseconds (0 keeps the default of 1 s).  Used to
 * check that a wait which never ends gives up with MOE_ERR_TIMEOUT. */
moe_status moe_debug_set_fault(void* workspace, int tile, uint64_t wait_ns, cudaStream_t stream);

/* Short text for a status code. */
const char* moe_status_string(moe_status status);

/* ABI version this library was built with (MOE_ROUTE_ABI_VERSION). */
int moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ROUTE_H */
