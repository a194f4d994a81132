// Host launchers of the Occult GB300 kernels (internal to the library; the
// public surface is include/occult.h).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace occult {

int launch_route(const LaunchCtx& ctx, const occult_desc_t& ds, const float* logits,
                 const int32_t* e2v, const float* table, int32_t* ids, float* gates,
                 int32_t* routed, uint32_t* vmask);
int launch_router_grad(const LaunchCtx& ctx, const occult_desc_t& ds, const float* logits,
                       const int32_t* gate_ids, const float* dgates, float* dlogits);

int launch_build_brim(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids,
                      const float* gates, const uint32_t* vmask, const int32_t* placement,
                      int32_t* brim0, int32_t* seg_off, int32_t* brim1, int32_t* exp_off,
                      int32_t* epd_src, float* epd_gate, int32_t* counts, void* ws);
size_t brim_ws_bytes(const occult_desc_t& ds);

int launch_dispatch(const LaunchCtx& ctx, const occult_desc_t& ds, const void* x,
                    const int32_t* brim0, const uint32_t* vmask, void* x_sfd, int32_t* sfd_tok);
// token rows (bf16) to the padded EPD layout (OCCULT_EPD_PAD), one pass
int launch_dispatch_epd(const LaunchCtx& ctx, const occult_desc_t& ds, const void* x,
                        const int32_t* ids, const int32_t* placement, const int32_t* brim0,
                        const int32_t* seg_off, const int32_t* brim1, const int32_t* exp_off,
                        void* x_epd);

int launch_combine(const LaunchCtx& ctx, const occult_desc_t& ds, const float* y_epd,
                   const int32_t* brim0, const int32_t* seg_off, const int32_t* brim1,
                   const int32_t* exp_off, const float* y_shared, float* y_sfd, float* y);

// p[0, n) = 0 (fp32)
int launch_zero_f32(const LaunchCtx& ctx, float* p, size_t n);

// stage one only (EPD -> SFD, y_sfd written) / stage two only (SFD -> ORI)
int launch_merge_sfd(const LaunchCtx& ctx, const occult_desc_t& ds, const float* y_epd,
                     const int32_t* brim0, const int32_t* seg_off, const int32_t* brim1,
                     const int32_t* exp_off, float* y_sfd);
int launch_combine_sfd(const LaunchCtx& ctx, const occult_desc_t& ds, const float* y_sfd,
                       const int32_t* brim0, const float* y_shared, float* y);

// Contiguous source shards of the sharded-source mode, passed by value.
struct ShardSplit {
  int n;                                 // shards (source devices)
  int off[OCCULT_MAX_SOURCES + 1];       // shard s holds tokens [off[s], off[s+1])
};
int launch_shard_plan(const LaunchCtx& ctx, const occult_desc_t& ds, const ShardSplit& split,
                      const uint32_t* vmask, const int32_t* brim0, int32_t* brim0_send,
                      int32_t* counts, int32_t* send_off, int32_t* recv_off);
int launch_all_to_all(const LaunchCtx& ctx, const occult_desc_t& ds, int n_src, const void* src,
                      void* dst, int64_t row_bytes, const int32_t* counts,
                      const int32_t* send_off, const int32_t* recv_off, int reverse);

int launch_similarity_accumulate(const LaunchCtx& ctx, int Ne, const float* logits, int n_tok,
                                 double* G);
int launch_similarity_finish(const LaunchCtx& ctx, int Ne, const double* G, float* table);

size_t profile_ws_bytes(const occult_desc_t& ds, int n_tok);
int launch_profile(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids, int n_tok,
                   const uint32_t* vmask, int64_t* C, float* P, int64_t* ct_hist, void* ws);

// Operand modes of the grouped GEMM: the operand is a row-major matrix whose rows
// run along K (K-major) or whose rows are K indices (MN-major: stored K x MN);
// loaded by TMA, or gathered row by row (rows picked by `gather`) with cp.async.
enum : int { OP_TMA_K = 0, OP_GATHER_K = 1, OP_TMA_MN = 2, OP_GATHER_MN = 3 };
// Epilogues: SwiGLU + gate -> layer dtype (optionally also G|U); plain fp32;
// SwiGLU backward -> dG|dU in the layer dtype plus partial gate gradients.
// EPI_F32_RED: fp32 rows added (red.global.add) into out[out_tok[out_src[r]]]
// instead of stored at row r (the merge of Algorithm 8 as fp32 atomic adds).
// EPI_SWIGLU_SAVE: EPI_SWIGLU with G|U saved (chosen by the launcher when gu_out
// is given; its stores go through shared memory).
enum : int { EPI_SWIGLU = 0, EPI_F32 = 1, EPI_SWIGLU_BWD = 2, EPI_F32_RED = 3, EPI_SWIGLU_SAVE = 4 };

// Grouped GEMM over segments.
//  rows mode (wgrad = false): output rows [seg_off[s], seg_off[s+1]) use weight
//    group seg_group[s] (s when NULL); out = A . B^T over K, A rows gathered by
//    `gather` (row r reads gather[r]) for OP_GATHER_K.  B's group g occupies rows
//    [g*b_group_rows, (g+1)*b_group_rows) of B (K-major), or K rows likewise
//    (MN-major).  With EPI_SWIGLU the group holds 2*N_out rows (gate then up) and
//    out = row_gate * silu(A.Bg^T) * (A.Bu^T).
//  wgrad mode: segment s reduces over EPD rows [seg_off[s], seg_off[s+1]) and
//    writes matrix seg_group[s] of out (out_group_stride apart, M_total x N_out):
//    out[m][n] = sum_r A[r][m] * B[r][n], both operands MN-major, the gathered one
//    read at row gather[r] and zero past the segment's end.
struct GroupedGemm {
  int a_mode = OP_TMA_K, b_mode = OP_TMA_K, epi = EPI_F32;
  bool wgrad = false;
  const void* A = nullptr;
  int64_t a_rows = 0, a_cols = 0;  // A as stored
  const void* B = nullptr;
  int64_t b_rows = 0, b_cols = 0;  // B as stored
  const int32_t* gather = nullptr;
  int a_pad = 0, b_pad = 0;           // operand rows that are EPD rows of segment s (wgrad:
                                      // its K rows; forward / dgrad: A's rows) are read at
                                      // row + pad * s (a padded EPD copy)
  void* a_copy = nullptr;             // gathered K-major A (training up-projection, dgrad
                                      // through W_d): padded EPD copy of its rows, or NULL
  int64_t b_group_rows = 0;
  int n_groups = 0;
  const int32_t* seg_off = nullptr;   // device; NULL: one segment of max_rows rows
  const int32_t* seg_group = nullptr; // device, nullable
  int n_seg = 0;
  int64_t max_rows = 0;               // upper bound of the rows (rows mode)
  int K = 0;                          // rows mode reduction length
  int M_total = 0;                    // wgrad: output rows per matrix
  int N_out = 0;
  const float* row_gate = nullptr;
  void* out = nullptr;
  int64_t ldo = 0;
  int64_t out_group_stride = 0;
  void* gu_out = nullptr;             // EPI_SWIGLU: optional G|U [rows, 2*N_out]
  const void* gu_in = nullptr;        // EPI_SWIGLU_BWD: G|U [rows, 2*N_out]
  float* dg_part = nullptr;           // EPI_SWIGLU_BWD: [rows, 2 * ceil(N_out/256)]
  const int32_t* out_src = nullptr;   // EPI_F32_RED: SFD row of every output row
  const int32_t* out_tok = nullptr;   // EPI_F32_RED: token of every SFD row
  int64_t out_rows = 0;               // EPI_F32_RED: rows of the merged output (tokens)
};

int launch_grouped_gemm_bf16(const LaunchCtx& ctx, const GroupedGemm& g);
int launch_grouped_gemm_f32(const LaunchCtx& ctx, const GroupedGemm& g);

size_t expert_bwd_ws_bytes(const occult_desc_t& ds);
int launch_dg_reduce(const LaunchCtx& ctx, const float* part, int rows, int n_part, float* dg);
int launch_gate_grad(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids,
                     const int32_t* placement, const int32_t* brim0, const int32_t* seg_off,
                     const int32_t* brim1, const int32_t* exp_off, const float* dg_epd,
                     float* dgates);

// one bounded wait that nothing completes (complete = 0) or that completes
int launch_selftest_wait(const LaunchCtx& ctx, int complete, uint64_t limit_ns);

// s[t] = sigmoid(w . x_t) for the shared-expert gate
int launch_shared_gate(const LaunchCtx& ctx, const occult_desc_t& ds, const void* x,
                       const void* w_sg, float* s_gate);

}  // namespace occult
