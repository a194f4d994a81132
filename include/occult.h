/*
 * occult.h -- C ABI of the GB300 (sm_103a) Occult collaboration-aware MoE layer.
 *
 * Source of every operation: "Occult: Optimizing Collaborative Communication
 * across Experts for Accelerated Parallel MoE Training and Inference"
 * (arXiv 2505.13345), Appendix A.1 Algorithm 2 (the refactored pipeline) and
 * Appendix A.2 Algorithms 3-9; Sec. 2.1 Eq. 1-4; Sec. 3.2 Algorithm 1.
 *
 * The Nd expert-parallel devices of the paper are virtual partitions of one GPU:
 * virtual device d owns the experts of placement row d and a contiguous range
 * of the SFD (dispatched) tensor.  The two all-to-all exchanges of Algorithm 2
 * are therefore identities on the device-major SFD buffers (their byte counts,
 * N_sfd * d * sizeof(element) per direction, are what crosses devices in the
 * paper's setting).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory:    every pointer is a DEVICE pointer unless the comment says "host".
 *            All buffers belong to the caller; the library never allocates,
 *            frees or synchronises (except occult_device_error, which reads back
 *            one word).  Row-major, densely packed unless stated.  Buffers start
 *            on a 16-byte boundary (the kernels move 16-byte vectors); a bf16
 *            layer's expert-GEMM output that does not is refused with
 *            OCCULT_ERR_UNSUPPORTED.
 * Execution: calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *            default stream) and capture into CUDA graphs.
 * Sizing:    data-dependent sizes are bounded by their worst case so that no
 *            host synchronisation is needed: N_sfd <= T * min(k, Nd) SFD rows,
 *            N_epd = T * k EPD rows.  Actual counts are written to device memory.
 * Types:     x, the weights and the EPD intermediate h are in the layer dtype
 *            (OCCULT_F32 or OCCULT_BF16).  Everything after the second linear
 *            layer -- y_epd, y_sfd, the shared-expert output and the layer output
 *            y -- is fp32, as is all accumulation: the paper keeps its merged SFD
 *            tensor in fp32 as well, and rounding these to bf16 would alone use up
 *            most of the 2e-2 * rms(y) error budget of a bf16 layer.  Logits and
 *            gates are fp32.
 * Errors:    0 on success, a negative OCCULT_ERR_* code otherwise.  Arguments
 *            are checked on the host before anything is launched; a failed check
 *            launches nothing.  A bounded device-side wait that expires sets a
 *            device error word (read with occult_device_error) and the kernel
 *            returns early, leaving its outputs undefined.
 */
#ifndef OCCULT_H_
#define OCCULT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OCCULT_OK                   0
#define OCCULT_ERR_INVALID_ARG     -1  /* null pointer, bad size or option           */
#define OCCULT_ERR_UNSUPPORTED     -2  /* valid layer this build does not run         */
#define OCCULT_ERR_WORKSPACE       -3  /* workspace smaller than occult_workspace_size */
#define OCCULT_ERR_CUDA            -4  /* a CUDA runtime/driver call failed          */
#define OCCULT_ERR_DEVICE_TIMEOUT  -5  /* a bounded device wait expired               */

#define OCCULT_F32   0
#define OCCULT_BF16  1

#define OCCULT_ROUTE_EXACT           0  /* Eq. 2 top-k                                 */
#define OCCULT_ROUTE_DEVICE_LIMITED  1  /* keep `limit_devices` devices, then top-k   */
#define OCCULT_ROUTE_SCORE_PRUNED    2  /* Sec. 3.3 routing-score-based pruning       */
#define OCCULT_ROUTE_SIMILARITY_PRUNED 3 /* Sec. 3.3 expert-similarity-based pruning:
                                            occult_route_similarity only           */

/* Largest supported sizes. */
#define OCCULT_MAX_EXPERTS  256
#define OCCULT_MAX_VDEV     32
#define OCCULT_MAX_TOPK     16
/* Padded EPD copies of gathered rows (x_epd, dy_epd): the EPD rows
 * exp_off[s] .. exp_off[s+1]-1 of expert slot s sit at rows
 * exp_off[s] + OCCULT_EPD_PAD * s onwards, followed by zero rows up to a whole
 * number of OCCULT_EPD_PAD rows from that start; such a copy has
 * T*top_k + OCCULT_EPD_PAD * n_experts rows of d elements. */
#define OCCULT_EPD_PAD      128

typedef void* occult_stream_t;   /* cudaStream_t */

/* One MoE layer.  Shapes: T tokens (N_ori), hidden d, Ne experts, top-k,
 * SwiGLU intermediate `inter` (I), Nd virtual devices (Ne % Nd == 0),
 * n_loc = Ne / Nd experts per device. */
typedef struct occult_desc {
  int32_t T;
  int32_t d;
  int32_t n_experts;
  int32_t top_k;
  int32_t inter;
  int32_t n_vdev;
  int32_t dtype;          /* OCCULT_F32 | OCCULT_BF16                              */
  int32_t route_mode;     /* OCCULT_ROUTE_*                                        */
  int32_t limit_devices;  /* devices kept per token by the pruning modes (>= 1,
                             and they must hold at least top_k experts)            */
  int32_t renorm;         /* 1: renormalise the k gates to sum to one              */
  int32_t n_shared;       /* always-on shared experts (0 = none)                   */
  int32_t shared_inter;   /* intermediate size of each shared expert               */
  int32_t shared_gate;    /* 1: scale the shared output by sigmoid(w_sg . x)       */
} occult_desc_t;

/* Human-readable name of an OCCULT_* return code (static string). */
const char* occult_strerror(int code);

/* Checks a descriptor; returns 0 or OCCULT_ERR_INVALID_ARG / _UNSUPPORTED.
 * bf16 layers need d % 64 == 0, inter % 64 == 0, shared_inter % 64 == 0. */
int occult_check_desc(const occult_desc_t* desc);

/* Workspace selectors of occult_workspace_size. */
#define OCCULT_WS_BUILD_BRIM     0   /* occult_build_brim for desc->T tokens       */
#define OCCULT_WS_PROFILE_COACT  1   /* occult_profile_coact for n_tok tokens      */
#define OCCULT_WS_EXPERT_BWD     2   /* occult_expert_bwd for desc->T tokens       */

/* Host: bytes of device workspace `ws` the entry point selected by `op` needs
 * (n_tok: profiled tokens, used by OCCULT_WS_PROFILE_COACT only).  The other
 * entry points need no workspace.  Workspace contents need no initialisation
 * and are not meaningful after the call. */
int occult_workspace_size(const occult_desc_t* desc, int32_t op, int32_t n_tok, size_t* bytes);

/* Host: reads and clears the device error word of the current device (one
 * 4-byte device-to-host copy, synchronising).  *code receives 0 or a negative
 * OCCULT_ERR_* value latched by a kernel since the last call. */
int occult_device_error(int32_t* code);

/*
 * occult_selftest_wait -- exercises the library's failure detection; the paper
 * has no counterpart.  Every pipelined kernel waits on its barriers with a time
 * limit, after which it latches OCCULT_ERR_DEVICE_TIMEOUT (read with
 * occult_device_error) and returns, leaving the context usable.  This launches
 * one such wait on a barrier that nothing completes (complete = 0), which must
 * give up after limit_ns nanoseconds (0 < limit_ns <= 2e9) and latch the error,
 * or that the kernel completes itself (complete = 1), which must not.  It reads
 * and writes no caller memory.
 */
int occult_selftest_wait(int32_t complete, int64_t limit_ns, occult_stream_t stream);

/*
 * occult_place -- Algorithm 1 (Sec. 3.2), HOST function, run once offline.
 *   C               host int64 [Ne, Ne] co-activation counts (Eq. 3).
 *   placement       host int32 [Nd, Ne/Nd] out: device d's experts in the order
 *                   Algorithm 1 adds them (this order numbers the local experts).
 *   expert_to_vdev  host int32 [Ne] out: device of every expert.
 * Comparisons are made on integer sums of C (P = C / max C only rescales), ties
 * go to the lowest expert id, each device is filled to exactly Ne/Nd experts.
 */
int occult_place(const int64_t* C, int32_t n_experts, int32_t n_vdev,
                 int32_t* placement, int32_t* expert_to_vdev);

/*
 * occult_route -- router of Sec. 2.1 Eq. 2 (Algorithm 2 step 1).
 *   logits          fp32 [T, Ne] router logits g(x).
 *   expert_to_vdev  int32 [Ne] device of each expert (from the placement).
 *   ids      out    int32 [T, k] chosen experts, descending logit; equal logits
 *                   go to the lower id.  The choice is made on the fp32 logits.
 *   gates    out    fp32 [T, k] softmax probabilities of the chosen experts
 *                   (renormalised over the k if desc->renorm).
 *   vmask    out    uint32 [T] bit d set iff the token uses virtual device d.
 * Device-limited mode keeps the desc->limit_devices devices with the largest
 * summed softmax mass over all their experts (ties: lower device), takes the
 * top-k among their experts and renormalises the gates.
 * Score-pruned mode is Sec. 3.3's routing-score-based pruning: the kept devices
 * are those of the token's routed (top-k) experts taken in descending score
 * until desc->limit_devices are found; ids are then the top-k of all sorted
 * scores among the experts of the kept devices, gates their probabilities
 * (renormalised if desc->renorm).
 * OCCULT_ROUTE_SIMILARITY_PRUNED needs occult_route_similarity (INVALID_ARG).
 */
int occult_route(const occult_desc_t* desc, const float* logits, const int32_t* expert_to_vdev,
                 int32_t* ids, float* gates, uint32_t* vmask, occult_stream_t stream);

/*
 * occult_route_similarity -- Sec. 3.3 expert-similarity-based pruning
 * (desc->route_mode must be OCCULT_ROUTE_SIMILARITY_PRUNED).
 *   logits, expert_to_vdev  as occult_route.
 *   table           fp32 [Ne, Ne] similarity table T (row e: similarity of expert
 *                   e to every expert; occult_similarity_finish builds it).  A NaN
 *                   entry ranks below every number.
 *   ids      out    int32 [T, k]: slot j holds the token's j-th routed expert
 *                   (descending score) if it lies on a kept device, else the
 *                   expert of a kept device, not selected yet, with the largest
 *                   table[routed_j, .] (ties: lower id).  The kept devices are
 *                   found as in score-pruned mode; routed experts on them count
 *                   as selected before any replacement.
 *   gates    out    fp32 [T, k] the routed experts' probabilities (renormalised
 *                   over the k if desc->renorm): a replacement keeps its slot's
 *                   routing weight.
 *   routed   out    int32 [T, k] the routed experts (nullable): the experts whose
 *                   probabilities the gates are, for occult_router_grad.
 *   vmask    out    as occult_route, for the final ids.
 */
int occult_route_similarity(const occult_desc_t* desc, const float* logits,
                            const int32_t* expert_to_vdev, const float* table, int32_t* ids,
                            float* gates, int32_t* routed, uint32_t* vmask,
                            occult_stream_t stream);

/*
 * occult_similarity_accumulate -- App. A.3 Eq. 8 accumulator over one batch of
 * profiled router logits.
 *   logits    fp32 [n_tok, Ne] (Ne = desc->n_experts).
 *   G         fp64 [Ne, Ne] in/out: G += logits^T logits.  The caller zeroes G
 *             before the first batch; batches may be of any size (n_tok >= 0).
 * Deterministic: each entry adds its batch's products in token order.
 */
int occult_similarity_accumulate(const occult_desc_t* desc, const float* logits, int32_t n_tok,
                                 double* G, occult_stream_t stream);

/*
 * occult_similarity_finish -- the similarity table from the accumulated G:
 *   table[i, j] = sign(G_ij) G_ij^2 / (G_ii G_jj)  (fp32 [Ne, Ne]; 0 where G_ii G_jj = 0),
 * Eq. 8's squared cosine similarity with the sign of Eq. 6's cosine kept, so
 * that it orders experts as the cosine does.
 */
int occult_similarity_finish(const occult_desc_t* desc, const double* G, float* table,
                             occult_stream_t stream);

/*
 * occult_router_grad -- gradient of sum_tj dgates_tj * gates_tj with respect to
 * the router logits, through the softmax of Eq. 2 (the choice of experts is
 * piecewise constant: no gradient through it).
 *   logits     fp32 [T, Ne] the router logits the gates came from.
 *   gate_ids   int32 [T, k] the experts whose probabilities the gates are (the
 *              ids of occult_route; `routed` of occult_route_similarity).
 *   dgates     fp32 [T, k] upstream gradient of the gates (occult_gate_grad).
 *   dlogits    out fp32 [T, Ne].  With p = softmax(logits), A = sum_j dg_j g_j:
 *              plain gates  dz_e = p_e (sum_{j: id_j = e} dg_j - A);
 *              desc->renorm dz_e = sum_{j: id_j = e} g_j (dg_j - A).
 */
int occult_router_grad(const occult_desc_t* desc, const float* logits, const int32_t* gate_ids,
                       const float* dgates, float* dlogits, occult_stream_t stream);

/*
 * occult_build_brim -- BRIM0 (Algorithm 3) and BRIM1 (Algorithm 5).
 *   ids, gates, vmask  from occult_route.
 *   placement   int32 [Nd, n_loc] device-major expert lists; slot s = d*n_loc + j
 *               holds expert placement[s].  It must hold every expert exactly
 *               once (as occult_place writes it): device buffers are not
 *               checked, and any other content is undefined behaviour.  The
 *               same holds for ids and the other outputs of earlier steps.
 *   brim0    out int32 [Nd, T]: running counter over active (d, t) pairs taken
 *               device by device, token by token; -1 where token t uses no
 *               expert of device d.  Non-negative values are SFD row indices.
 *   seg_off  out int32 [Nd + 1]: device d received SFD rows [seg_off[d], seg_off[d+1]).
 *   brim1    out int32 [Ne, T]: row s = d*n_loc + j; entry [s, r] for
 *               r < n_d = seg_off[d+1]-seg_off[d] is device d's Algorithm 5
 *               counter (local EPD index) of (local expert j, received row r),
 *               or -1 if that row does not activate that expert.  Entries with
 *               r >= n_d are not written.
 *   exp_off  out int32 [Ne + 1]: EPD rows of slot s are [exp_off[s], exp_off[s+1]);
 *               device d's EPD tensor starts at exp_off[d*n_loc], so the global
 *               EPD row of brim1[s, r] >= 0 is exp_off[d*n_loc] + brim1[s, r].
 *   epd_src  out int32 [T*k]: SFD row feeding each EPD row (the condensed,
 *               non-negative BRIM1 entries' column coordinates).
 *   epd_gate out fp32 [T*k]: routing weight of each EPD row (Algorithm 7's w).
 *   counts   out int32 [4]: {N_sfd, N_epd, max C_T, reserved}.
 *   ws       device workspace of occult_workspace_size(OCCULT_WS_BUILD_BRIM)
 *            bytes (per-tile column counts); OCCULT_ERR_WORKSPACE if smaller.
 */
int occult_build_brim(const occult_desc_t* desc, const int32_t* ids, const float* gates,
                      const uint32_t* vmask, const int32_t* placement,
                      int32_t* brim0, int32_t* seg_off, int32_t* brim1, int32_t* exp_off,
                      int32_t* epd_src, float* epd_gate, int32_t* counts,
                      void* ws, size_t ws_bytes, occult_stream_t stream);

/*
 * occult_build_brim_noalloc -- occult_build_brim without a caller workspace.
 * The paper has no counterpart; this entry point exists for callers that cannot
 * allocate device memory: code whose device memory belongs to an allocator it
 * cannot reach from plain C, serving loops that forbid allocation after
 * start-up (cudaMalloc and cudaFree may synchronise the device), and processes
 * that must keep a fixed device footprint.  Same arguments and results as
 * occult_build_brim minus ws / ws_bytes; it allocates nothing.
 *   Scratch:  a static device array of OCCULT_STATIC_SCRATCH_BYTES inside the
 *             library, loaded on every GPU that uses the library and kept until
 *             the process exits.  A layer needing more scratch than that (more
 *             than 32768 tokens at 256 experts, 97600 at 64) gets
 *             OCCULT_ERR_WORKSPACE and no launch.  Nothing in the array has to start at zero, and each call
 *             leaves its contents behind.
 *   Sharing:  every call on a device uses the same array, so calls that overlap
 *             on the GPU (unordered streams) race and give wrong results; order
 *             them on one stream or with events.
 *   Set-up:   the first call on a device looks up the array's device address
 *             with that device current (a lookup that fails returns
 *             OCCULT_ERR_CUDA and is tried again by the next call); make that
 *             first call before any stream capture on the device.
 */
#define OCCULT_STATIC_SCRATCH_BYTES 1183744
int occult_build_brim_noalloc(const occult_desc_t* desc, const int32_t* ids, const float* gates,
                              const uint32_t* vmask, const int32_t* placement,
                              int32_t* brim0, int32_t* seg_off, int32_t* brim1,
                              int32_t* exp_off, int32_t* epd_src, float* epd_gate,
                              int32_t* counts, occult_stream_t stream);

/*
 * occult_dispatch -- Algorithm 4: x_sfd[brim0[d, t]] = x[t] for every
 * non-negative entry (stage one of scattering, ORI -> SFD).  The result is the
 * first all-to-all's send buffer, segment d going to virtual device d.
 *   x        [T, d] layer dtype, 16-byte aligned.
 *   x_sfd    out [T*min(k,Nd), d] layer dtype, 16-byte aligned; rows >= N_sfd
 *            untouched.
 *   sfd_tok  out int32 [T*min(k,Nd)] ORI token of each SFD row (nullable).
 */
int occult_dispatch(const occult_desc_t* desc, const void* x, const int32_t* brim0,
                    const uint32_t* vmask, void* x_sfd, int32_t* sfd_tok,
                    occult_stream_t stream);

/*
 * occult_dispatch_epd -- stage one of scattering, the (identity) exchange of a
 * single source and the device-local expansion in one pass: token t's row goes
 * to the EPD row of each of its experts (Algorithm 5's numbering: slot s of
 * expert ids[t, j] on device dv = s / n_loc, row exp_off[dv * n_loc] +
 * brim1[s][brim0[dv][t] - seg_off[dv]]), in the padded layout (OCCULT_EPD_PAD):
 *   x_epd[row + OCCULT_EPD_PAD * s] = x[t], and zeros in each slot's padding.
 * Used for the upstream gradient dy, whose only readers are the backward GEMMs.
 *   x       [T, d] bf16, 16-byte aligned;  ids int32 [T, k] from occult_route;
 *   x_epd   out bf16 [T*k + OCCULT_EPD_PAD*Ne, d], 16-byte aligned.
 * bf16 layers only.
 */
int occult_dispatch_epd(const occult_desc_t* desc, const void* x, const int32_t* ids,
                        const int32_t* placement, const int32_t* brim0, const int32_t* seg_off,
                        const int32_t* brim1, const int32_t* exp_off, void* x_epd,
                        occult_stream_t stream);

/*
 * occult_expert_up -- scattering sparse matmul (Algorithm 6, stage two of
 * scattering, SFD -> EPD) fused with the SwiGLU activation and the weight
 * modulation of Algorithm 7:
 *   h_epd[r, :] = epd_gate[r] * silu(A_r . W_g[e]^T) * (A_r . W_u[e]^T),
 *   A_r = x_sfd[epd_src[r]], e = placement[s] for the slot s whose segment holds r.
 *   w1     [Ne, 2*I, d]: rows [0, I) of expert e are W_g, rows [I, 2I) are W_u.
 *   h_epd  out [T*k, I] layer dtype.
 *   gu_epd out [T*k, 2*I] bf16, nullable: the pre-activations G | U of every EPD
 *          row, saved for occult_expert_bwd (bf16 layers only).
 *   x_epd  out bf16, nullable (requires gu_epd): the gathered rows A_r written
 *          to their padded EPD copy (OCCULT_EPD_PAD: T*k + OCCULT_EPD_PAD*Ne
 *          rows of d), which occult_expert_bwd reads for dw1 instead of
 *          gathering x_sfd again.
 * bf16 layers run on the tcgen05 tensor cores (fp32 accumulate in TMEM).
 */
int occult_expert_up(const occult_desc_t* desc, const void* x_sfd, const int32_t* epd_src,
                     const float* epd_gate, const int32_t* exp_off, const int32_t* placement,
                     const void* w1, void* h_epd, void* gu_epd, void* x_epd,
                     occult_stream_t stream);

/*
 * occult_expert_down -- the second linear layer of Algorithm 8 on the EPD rows:
 *   y_epd[r, :] = h_epd[r, :] . W_d[e]^T,   w2 [Ne, d, I],  y_epd out fp32 [T*k, d].
 * The merge of Algorithm 8 (summing a token's local experts) is done without
 * atomics by occult_combine.
 */
int occult_expert_down(const occult_desc_t* desc, const void* h_epd, const int32_t* exp_off,
                       const int32_t* placement, const void* w2, void* y_epd,
                       occult_stream_t stream);

/*
 * occult_expert_down_merge -- occult_expert_down with the merge folded into it
 * as fp32 atomic additions, which is how the paper's merging SMM aggregates
 * (Algorithm 8; Sec. 3.1 footnote 3: fp32 atomic adds, cast afterwards).  On one
 * GPU the second all-to-all is the identity and both merge stages are plain sums,
 * so every EPD row is added straight into its token's output row:
 *   y[sfd_tok[epd_src[r]]] += h_epd[r, :] . W_d[e]^T   for every EPD row r.
 *   epd_src  int32 [T*k] from occult_build_brim.
 *   sfd_tok  int32 [T*min(k,Nd)] from occult_dispatch (token of every SFD row).
 *   y        in/out fp32 [T, d].  zero_y = 1: the call zeroes y first; zero_y = 0:
 *            the rows are added to what y holds (e.g. the shared experts' output).
 * The additions land in no fixed order: y equals occult_combine's ordered merge
 * up to fp32 rounding of the k terms of each element, but is not bit-reproducible
 * from run to run (use occult_expert_down + occult_combine for that).
 */
int occult_expert_down_merge(const occult_desc_t* desc, const void* h_epd, const int32_t* exp_off,
                             const int32_t* placement, const void* w2, const int32_t* epd_src,
                             const int32_t* sfd_tok, void* y, int32_t zero_y,
                             occult_stream_t stream);

/* occult_expert_ffn -- occult_expert_up followed by occult_expert_down. */
int occult_expert_ffn(const occult_desc_t* desc, const void* x_sfd, const int32_t* epd_src,
                      const float* epd_gate, const int32_t* exp_off, const int32_t* placement,
                      const void* w1, const void* w2, void* h_epd, void* y_epd,
                      occult_stream_t stream);

/*
 * occult_shared_ffn -- always-on shared experts on the token's own device (no
 * all-to-all):  y_s[t] = s_t * W_d^s (silu(W_g^s x_t) * (W_u^s x_t)), with
 * s_t = sigmoid(w_sg . x_t) if desc->shared_gate else 1.  Several shared
 * experts are stacked on the intermediate axis, S = n_shared * shared_inter:
 *   ws1 [2*S, d] (gate rows then up rows), ws2 [d, S], w_sg [d] (nullable
 *   without a gate), h_s out [T, S], s_gate out fp32 [T], y_s out fp32 [T, d].
 */
int occult_shared_ffn(const occult_desc_t* desc, const void* x, const void* ws1,
                      const void* ws2, const void* w_sg, void* h_s, float* s_gate, void* y_s,
                      occult_stream_t stream);

/*
 * occult_combine -- the two-stage merge: stage one (EPD -> SFD, Algorithm 8's
 * aggregation over a row's local experts) and stage two (SFD -> ORI,
 * Algorithm 9, devices summed in order 0..Nd-1), in fp32:
 *   y_sfd[v] = sum_j y_epd[exp_off[d*n_loc] + brim1[d*n_loc + j, v - seg_off[d]]]
 *   y[t]     = sum_d y_sfd[brim0[d, t]]  (+ y_shared[t])
 *   y_epd     fp32 [T*k, d] from occult_expert_down.
 *   y_shared  fp32 [T, d] nullable: shared-expert output added to every token.
 *   y_sfd     out fp32 [T*min(k,Nd), d] nullable: when given, stage one is
 *             written out (the second all-to-all's send buffer) and stage two
 *             reads it back; when NULL both stages run fused per token.
 *   y         out fp32 [T, d].
 */
int occult_combine(const occult_desc_t* desc, const void* y_epd, const int32_t* brim0,
                   const int32_t* seg_off, const int32_t* brim1, const int32_t* exp_off,
                   const void* y_shared, void* y_sfd, void* y, occult_stream_t stream);

/*
 * occult_merge_sfd -- stage one of the merge alone (EPD -> SFD, the aggregation
 * of Algorithm 8): y_sfd[v] = sum_j y_epd[exp_off[d*n_loc] + brim1[d*n_loc + j,
 * v - seg_off[d]]] for every received row v of every device d, fp32, local
 * experts in placement order.  y_sfd out fp32 [T*min(k,Nd), d] in the receive
 * layout of brim0 (the second all-to-all's send buffer); rows >= N_sfd
 * untouched.  Other arguments as occult_combine.
 */
int occult_merge_sfd(const occult_desc_t* desc, const void* y_epd, const int32_t* brim0,
                     const int32_t* seg_off, const int32_t* brim1, const int32_t* exp_off,
                     void* y_sfd, occult_stream_t stream);

/*
 * occult_combine_sfd -- stage two alone (SFD -> ORI, Algorithm 9):
 *   y[t] = sum over d = 0..Nd-1 with row_map[d, t] >= 0 of y_sfd[row_map[d, t]]
 *          (+ y_shared[t]),   fp32, devices in ascending order.
 *   row_map   int32 [Nd, T]: brim0 of occult_build_brim when y_sfd is in the
 *             receive layout, brim0_send of occult_shard_plan when it is in the
 *             sources' send layout (after the second all-to-all).
 *   y_sfd     fp32 [T*min(k,Nd), d];  y_shared fp32 [T, d] nullable;  y out fp32 [T, d].
 */
int occult_combine_sfd(const occult_desc_t* desc, const void* y_sfd, const int32_t* row_map,
                       const void* y_shared, void* y, occult_stream_t stream);

/* Largest number of source shards of the sharded-source mode. */
#define OCCULT_MAX_SOURCES 32

/*
 * occult_shard_plan -- sharded-source expert parallelism (App. A.1: Algorithm 2
 * runs on every device; each source device builds BRIM0 over its own tokens with
 * Algorithm 3, dispatches them with Algorithm 4, and all_to_all_single sends SFD
 * segment d to device d with BRIM0 row d's non-zero counts as split sizes).  The
 * T tokens are split into contiguous source shards that stand for the source
 * devices.
 *   n_src      1 <= n_src <= OCCULT_MAX_SOURCES source shards.
 *   src_off    HOST int32 [n_src + 1]: shard s holds tokens [src_off[s],
 *              src_off[s+1]); src_off[0] = 0, src_off[n_src] = T, non-decreasing
 *              (empty shards allowed).  Copied at launch.
 *   vmask      uint32 [T] from occult_route.
 *   brim0      int32 [Nd, T] from occult_build_brim: the receive layout, which
 *              for contiguous shards is device-major, then source, then token.
 *   brim0_send out int32 [Nd, T]: each token's row in the send layout (the
 *              sources' SFD tensors end to end: source-major, then device, then
 *              token) -- Algorithm 3 over shard s, offset by the rows of shards
 *              0..s-1; -1 where brim0 is -1.  occult_dispatch with it as brim0
 *              fills the send buffers.
 *   counts     out int32 [n_src, Nd]: rows shard s sends to device d (split sizes).
 *   send_off   out int32 [n_src, Nd]: first row of block (s, d) in the send layout.
 *   recv_off   out int32 [n_src, Nd]: first row of block (s, d) in the receive layout.
 */
int occult_shard_plan(const occult_desc_t* desc, int32_t n_src, const int32_t* src_off,
                      const uint32_t* vmask, const int32_t* brim0, int32_t* brim0_send,
                      int32_t* counts, int32_t* send_off, int32_t* recv_off,
                      occult_stream_t stream);

/*
 * occult_all_to_all -- the exchange of the sharded-source mode as block copies
 * between the two layouts of occult_shard_plan: block (s, d) moves counts[s, d]
 * rows from send_off[s, d] to recv_off[s, d] (reverse = 0, the first all-to-all:
 * sources' SFD tensors -> devices) or back (reverse = 1, the second all-to-all:
 * stage-one sums -> their sources).
 *   src, dst   row buffers of at least T*min(k,Nd) rows of row_bytes bytes, not
 *              overlapping, 16-byte aligned; rows >= N_sfd of dst untouched.
 *   row_bytes  bytes per row, a positive multiple of 16 (d*2 for bf16 x, d*4 for
 *              the fp32 stage-one sums).
 */
int occult_all_to_all(const occult_desc_t* desc, int32_t n_src, const int32_t* counts,
                      const int32_t* send_off, const int32_t* recv_off, const void* src,
                      void* dst, int64_t row_bytes, int32_t reverse, occult_stream_t stream);

/*
 * occult_expert_bwd -- backward of the expert computation (bf16 layers).  The
 * paper states that its sparse kernels serve the backward pass too (Sec. 1) but
 * gives no backward pseudo-code; these are the derivatives of Eq. 1 run through
 * the same BRIM-indexed layout.  With dy_sfd = occult_dispatch(dy) (stage one of
 * scattering applied to the upstream gradient) and the forward's h_epd and gu_epd:
 *   dh'_r   = W_d[e]^T dy_sfd[src_r]            (dgrad through W_d, gathered rows)
 *   dg_r    = <dh'_r, silu(G_r) U_r>             -> dg_epd fp32 [T*k]
 *   dG, dU  = g_r dh'_r * U silu'(G), g_r dh'_r * silu(G) -> dgu_epd bf16 [T*k, 2I]
 *   dx_epd  = [dG | dU] . [W_g; W_u]           -> fp32 [T*k, d]; occult_combine merges
 *                                                 it to dx [T, d] (stage one + two)
 *   dw2[e]  = sum_r dy_sfd[src_r] h'_r^T        -> fp32 [Ne, d, I]
 *   dw1[e]  = sum_r [dG | dU]_r x_sfd[src_r]^T  -> fp32 [Ne, 2I, d]
 * Weight gradients are written, not accumulated; experts without rows get zeros.
 *   x_epd   nullable: the padded EPD copy of the x rows that occult_expert_up
 *           wrote; given, dw1 reads it as tiles (x_sfd may then be NULL); NULL:
 *           dw1 gathers x_sfd through epd_src.
 *   dy_epd  nullable, bf16 [T*k + OCCULT_EPD_PAD*Ne, d]: with dy_sfd given, a
 *           scratch copy that the dh' GEMM writes its gathered dy rows to and
 *           dw2 reads as tiles (NULL: dw2 gathers dy_sfd again); with dy_sfd
 *           NULL, the input: dy in the padded EPD layout (occult_dispatch_epd),
 *           read as tiles by dh' and dw2.
 *   Both choices give the same bits.
 *   ws  occult_workspace_size(OCCULT_WS_EXPERT_BWD) bytes.
 */
int occult_expert_bwd(const occult_desc_t* desc, const void* x_sfd, const void* dy_sfd,
                      const int32_t* epd_src, const float* epd_gate, const int32_t* exp_off,
                      const int32_t* placement, const void* w1, const void* w2,
                      const void* h_epd, const void* gu_epd, void* dgu_epd, float* dx_epd,
                      float* dw1, float* dw2, float* dg_epd, const void* x_epd, void* dy_epd,
                      void* ws, size_t ws_bytes, occult_stream_t stream);

/*
 * occult_expert_bwd_merge -- occult_expert_bwd with the merge of dx folded into
 * the dgrad through [W_g; W_u] as fp32 atomic additions (as occult_expert_down_merge
 * does for y): dx[sfd_tok[epd_src[r]]] += [dG | dU]_r . [W_g; W_u] for every EPD
 * row r, so dx_epd is never written.  Same arguments as occult_expert_bwd except
 *   sfd_tok  int32 [T*min(k,Nd)] from occult_dispatch (token of every SFD row);
 *   dx       out fp32 [T, d] (zeroed by the call, then accumulated; no fixed
 *            order of the additions, so not bit-reproducible).
 */
int occult_expert_bwd_merge(const occult_desc_t* desc, const void* x_sfd, const void* dy_sfd,
                            const int32_t* epd_src, const float* epd_gate, const int32_t* exp_off,
                            const int32_t* placement, const void* w1, const void* w2,
                            const void* h_epd, const void* gu_epd, void* dgu_epd,
                            const int32_t* sfd_tok, float* dx, float* dw1, float* dw2,
                            float* dg_epd, const void* x_epd, void* dy_epd, void* ws,
                            size_t ws_bytes, occult_stream_t stream);

/*
 * The four GEMMs of occult_expert_bwd as separate calls, for callers that time,
 * overlap or reorder them (same derivatives of Eq. 1, same layouts; the paper
 * gives no backward pseudo-code, Sec. 1).  Run in this order they equal
 * occult_expert_bwd / occult_expert_bwd_merge.  bf16 layers only.
 *
 * occult_expert_dgrad_down -- dh'_r = W_d[e]^T dy_sfd[src_r], then dg_r and
 *   dG | dU as in occult_expert_bwd.
 *   dgu_epd out bf16 [T*k, 2I];  dg_epd out fp32 [T*k];
 *   dy_epd  with dy_sfd given: out bf16, nullable, the gathered dy rows written
 *           to their padded EPD copy (OCCULT_EPD_PAD), for
 *           occult_expert_wgrad_down; with dy_sfd NULL: the input, dy in the
 *           padded EPD layout (occult_dispatch_epd), read as tiles.
 *   ws      occult_workspace_size(OCCULT_WS_EXPERT_BWD) bytes.
 */
int occult_expert_dgrad_down(const occult_desc_t* desc, const void* dy_sfd,
                             const int32_t* epd_src, const float* epd_gate,
                             const int32_t* exp_off, const int32_t* placement, const void* w2,
                             const void* gu_epd, void* dgu_epd, float* dg_epd, void* dy_epd,
                             void* ws, size_t ws_bytes, occult_stream_t stream);

/*
 * occult_expert_dgrad_up -- dx rows [dG | dU]_r . [W_g; W_u] (fp32).
 *   sfd_tok NULL: dx is dx_epd, out fp32 [T*k, d], one row per EPD row (merge it
 *            with occult_combine); zero_dx must be 0.
 *   sfd_tok given (int32 [T*min(k,Nd)], token of every SFD row): dx is fp32
 *            [T, d] and every row is added into its token's row with fp32 atomics
 *            (no fixed order); zero_dx = 1 zeroes dx first, 0 adds to it.
 */
int occult_expert_dgrad_up(const occult_desc_t* desc, const void* dgu_epd, const int32_t* epd_src,
                           const int32_t* exp_off, const int32_t* placement, const void* w1,
                           const int32_t* sfd_tok, float* dx, int32_t zero_dx,
                           occult_stream_t stream);

/*
 * occult_expert_wgrad_down -- dw2[e] = sum over e's EPD rows r of
 *   dy_sfd[src_r] h'_r^T, out fp32 [Ne, d, I] (written; zeros for experts
 *   without rows).
 *   dy_epd  nullable: the padded EPD copy of the dy rows that
 *           occult_expert_dgrad_down wrote; given, it is read as tiles and
 *           dy_sfd / epd_src are not read (may be NULL); NULL: the rows are
 *           gathered from dy_sfd through epd_src.  Both give the same bits.
 */
int occult_expert_wgrad_down(const occult_desc_t* desc, const void* dy_sfd,
                             const int32_t* epd_src, const void* dy_epd, const int32_t* exp_off,
                             const int32_t* placement, const void* h_epd, float* dw2,
                             occult_stream_t stream);

/*
 * occult_expert_wgrad_up -- dw1[e] = sum over e's EPD rows r of
 *   [dG | dU]_r x_sfd[src_r]^T, out fp32 [Ne, 2I, d] (written; zeros for experts
 *   without rows).
 *   x_epd  nullable: the padded EPD copy of the x rows (OCCULT_EPD_PAD), as
 *          occult_expert_up writes it; given, its rows are read as tiles and
 *          x_sfd / epd_src are not read (may be NULL); NULL: the rows are
 *          gathered from x_sfd through epd_src.  Both give the same bits.
 */
int occult_expert_wgrad_up(const occult_desc_t* desc, const void* x_sfd, const int32_t* epd_src,
                           const void* x_epd, const int32_t* exp_off, const int32_t* placement,
                           const void* dgu_epd, float* dw1, occult_stream_t stream);

/*
 * occult_zero_f32 -- buf[0..n) = 0 (fp32), asynchronously: the starting value of
 * a buffer that fp32 atomic merges add into (Sec. 3.1 footnote 3: the merging
 * SMM adds into an fp32 tensor), e.g. y before occult_expert_down_merge with
 * zero_y = 0, or dx before occult_expert_dgrad_up with zero_dx = 0.
 */
int occult_zero_f32(float* buf, int64_t n, occult_stream_t stream);

/*
 * occult_gate_grad -- gate gradients back in token order: dgates[t, j] =
 * dg_epd[EPD row of (t, ids[t, j])], the row found as in the combine (BRIM0 gives
 * the token's received row on the expert's device, BRIM1 its EPD row).
 *   dgates out fp32 [T, k].
 */
int occult_gate_grad(const occult_desc_t* desc, const int32_t* ids, const int32_t* placement,
                     const int32_t* brim0, const int32_t* seg_off, const int32_t* brim1,
                     const int32_t* exp_off, const float* dg_epd, float* dgates,
                     occult_stream_t stream);

/*
 * occult_profile_coact -- co-activation profiling (Sec. 2.1 Eq. 3-4, Sec. 2.2).
 *   ids      int32 [n_tok, k] routing of the profiling batch.
 *   vmask    uint32 [n_tok] (nullable) device masks under the current placement.
 *   C        out int64 [Ne, Ne]: tokens activating both i and j (diagonal = load).
 *   P        out fp32 [Ne, Ne] (nullable): C / max C.
 *   ct_hist  out int64 [min(k,Nd) + 1] (nullable, needs vmask): tokens per C_T value.
 *   ws       device workspace of occult_workspace_size(OCCULT_WS_PROFILE_COACT)
 *            bytes (per-expert token bitsets); OCCULT_ERR_WORKSPACE if smaller.
 * Counts are exact integers built from per-expert token bitsets (no atomics).
 */
int occult_profile_coact(const occult_desc_t* desc, const int32_t* ids, int32_t n_tok,
                         const uint32_t* vmask, int64_t* C, float* P, int64_t* ct_hist,
                         void* ws, size_t ws_bytes, occult_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* OCCULT_H_ */
