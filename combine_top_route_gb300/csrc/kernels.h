// Host launchers of the Occult GB300 kernels (internal to the library; the
// public surface is include/occult.h).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace occult {

int launch_route(const LaunchCtx& ctx, const occult_desc_t& ds, const float* logits,
                 const int32_t* e2v, int32_t* ids, float* gates, uint32_t* vmask);

int launch_build_brim(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids,
                      const float* gates, const uint32_t* vmask, const int32_t* placement,
                      int32_t* brim0, int32_t* seg_off, int32_t* brim1, int32_t* exp_off,
                      int32_t* epd_src, float* epd_gate, int32_t* counts, void* ws);
size_t brim_ws_bytes(const occult_desc_t& ds);

int launch_dispatch(const LaunchCtx& ctx, const occult_desc_t& ds, const void* x,
                    const int32_t* brim0, const uint32_t* vmask, void* x_sfd, int32_t* sfd_tok);

int launch_combine(const LaunchCtx& ctx, const occult_desc_t& ds, const float* y_epd,
                   const int32_t* brim0, const int32_t* seg_off, const int32_t* brim1,
                   const int32_t* exp_off, const float* y_shared, float* y_sfd, float* y);

size_t profile_ws_bytes(const occult_desc_t& ds, int n_tok);
int launch_profile(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids, int n_tok,
                   const uint32_t* vmask, int64_t* C, float* P, int64_t* ct_hist, void* ws);

// Grouped GEMM over row segments: output rows [seg_off[s], seg_off[s+1]) use
// weight group seg_group[s] (s when NULL).  Output row r reads A row gather[r]
// (r when NULL).  With swiglu, the group's B holds 2*N_out rows (gate rows then
// up rows) and out = row_gate * silu(A.Bg^T) * (A.Bu^T) in the layer dtype;
// otherwise out = A.B^T in fp32.
struct GroupedGemm {
  const void* A;
  int64_t a_rows;            // rows addressable in A
  const int32_t* gather;     // nullable
  const void* B;             // [n_groups * b_group_rows, K]
  int64_t b_group_rows;
  int n_groups;
  const int32_t* seg_off;    // [n_seg + 1] device; NULL: one segment of max_rows rows
  const int32_t* seg_group;  // [n_seg] device, nullable
  int n_seg;
  int64_t max_rows;          // upper bound of seg_off[n_seg]
  const float* row_gate;     // nullable, swiglu only
  void* out;
  int64_t ldo;
  int N_out;
  int K;
  bool swiglu;
};

int launch_grouped_gemm_bf16(const LaunchCtx& ctx, const GroupedGemm& g);
int launch_grouped_gemm_f32(const LaunchCtx& ctx, const GroupedGemm& g);

// s[t] = sigmoid(w . x_t) for the shared-expert gate
int launch_shared_gate(const LaunchCtx& ctx, const occult_desc_t& ds, const void* x,
                       const void* w_sg, float* s_gate);

}  // namespace occult
