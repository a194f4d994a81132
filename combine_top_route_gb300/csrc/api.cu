// C ABI of the Occult GB300 layer: argument checks, then launches.  See
// include/occult.h for the meaning, layout and ownership of every argument.
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace occult {

// device error word, latched by bounded waits that expire
__device__ int g_dev_err;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::once_flag once;
  int num_sms = 0;
  int* err = nullptr;
  cudaError_t status = cudaSuccess;
};
DeviceInfo g_devices[kMaxDevices];

}  // namespace

int launch_ctx(occult_stream_t stream, LaunchCtx* ctx) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OCCULT_ERR_CUDA;
  DeviceInfo& di = g_devices[dev];
  std::call_once(di.once, [&] {
    di.status = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (di.status == cudaSuccess)
      di.status = cudaGetSymbolAddress(reinterpret_cast<void**>(&di.err), g_dev_err);
  });
  if (di.status != cudaSuccess) return OCCULT_ERR_CUDA;
  ctx->stream = static_cast<cudaStream_t>(stream);
  ctx->dev_err = di.err;
  ctx->num_sms = di.num_sms;
  return OCCULT_OK;
}

}  // namespace occult

using namespace occult;

namespace {

int min_i(int a, int b) { return a < b ? a : b; }

#define OCCULT_REQUIRE(cond) \
  do {                       \
    if (!(cond)) return OCCULT_ERR_INVALID_ARG; \
  } while (0)

#define OCCULT_CTX(stream)                      \
  LaunchCtx ctx;                                \
  do {                                          \
    int rc_ = launch_ctx((stream), &ctx);       \
    if (rc_) return rc_;                        \
  } while (0)

int check(const occult_desc_t* ds) {
  if (!ds) return OCCULT_ERR_INVALID_ARG;
  if (ds->T < 0 || ds->d <= 0 || ds->n_experts <= 0 || ds->top_k <= 0 || ds->inter <= 0 ||
      ds->n_vdev <= 0)
    return OCCULT_ERR_INVALID_ARG;
  if (ds->n_experts % ds->n_vdev != 0) return OCCULT_ERR_INVALID_ARG;
  if (ds->top_k > ds->n_experts) return OCCULT_ERR_INVALID_ARG;
  if (ds->dtype != OCCULT_F32 && ds->dtype != OCCULT_BF16) return OCCULT_ERR_INVALID_ARG;
  if (ds->route_mode < OCCULT_ROUTE_EXACT || ds->route_mode > OCCULT_ROUTE_SIMILARITY_PRUNED)
    return OCCULT_ERR_INVALID_ARG;
  if (ds->n_experts > OCCULT_MAX_EXPERTS || ds->n_vdev > OCCULT_MAX_VDEV ||
      ds->top_k > OCCULT_MAX_TOPK)
    return OCCULT_ERR_UNSUPPORTED;
  const int n_loc = ds->n_experts / ds->n_vdev;
  if (ds->route_mode != OCCULT_ROUTE_EXACT) {
    if (ds->limit_devices < 1 || ds->limit_devices > ds->n_vdev) return OCCULT_ERR_INVALID_ARG;
    if (ds->limit_devices * n_loc < ds->top_k) return OCCULT_ERR_INVALID_ARG;
  }
  if (ds->n_shared < 0 || (ds->n_shared > 0 && ds->shared_inter <= 0)) return OCCULT_ERR_INVALID_ARG;
  // 16-byte row vectors
  const int vec = ds->dtype == OCCULT_BF16 ? 8 : 4;
  if (ds->d % vec != 0) return OCCULT_ERR_UNSUPPORTED;
  if (ds->dtype == OCCULT_BF16) {
    // tensor-core tiles step K by 64 and write 32-column chunks
    if (ds->d % 64 != 0 || ds->inter % 64 != 0) return OCCULT_ERR_UNSUPPORTED;
    if (ds->n_shared > 0 && (ds->n_shared * ds->shared_inter) % 64 != 0) return OCCULT_ERR_UNSUPPORTED;
  }
  // int32 indices
  if (static_cast<int64_t>(ds->T) * ds->top_k >= (1ll << 31) ||
      static_cast<int64_t>(ds->T) * ds->n_experts >= (1ll << 31))
    return OCCULT_ERR_UNSUPPORTED;
  return OCCULT_OK;
}

}  // namespace

extern "C" {

const char* occult_strerror(int code) {
  switch (code) {
    case OCCULT_OK: return "success";
    case OCCULT_ERR_INVALID_ARG: return "invalid argument";
    case OCCULT_ERR_UNSUPPORTED: return "unsupported layer shape or option";
    case OCCULT_ERR_WORKSPACE: return "workspace too small";
    case OCCULT_ERR_CUDA: return "CUDA call failed";
    case OCCULT_ERR_DEVICE_TIMEOUT: return "bounded device wait expired";
    default: return "unknown error";
  }
}

int occult_check_desc(const occult_desc_t* desc) { return check(desc); }

int occult_workspace_size(const occult_desc_t* desc, int32_t op, int32_t n_tok, size_t* bytes) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(bytes);
  if (op == OCCULT_WS_BUILD_BRIM) {
    *bytes = brim_ws_bytes(*desc);
    return OCCULT_OK;
  }
  if (op == OCCULT_WS_EXPERT_BWD) {
    *bytes = expert_bwd_ws_bytes(*desc);
    return OCCULT_OK;
  }
  OCCULT_REQUIRE(op == OCCULT_WS_PROFILE_COACT && n_tok >= 0);
  *bytes = profile_ws_bytes(*desc, n_tok);
  return OCCULT_OK;
}

int occult_device_error(int32_t* code) {
  OCCULT_REQUIRE(code);
  OCCULT_CTX(nullptr);
  int v = 0;
  if (cudaMemcpy(&v, ctx.dev_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return OCCULT_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(ctx.dev_err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return OCCULT_ERR_CUDA;
  *code = v;
  return OCCULT_OK;
}

int occult_selftest_wait(int32_t complete, int64_t limit_ns, occult_stream_t stream) {
  OCCULT_REQUIRE(complete == 0 || complete == 1);
  OCCULT_REQUIRE(limit_ns > 0 && limit_ns <= static_cast<int64_t>(kWaitLimitNs));
  OCCULT_CTX(stream);
  return launch_selftest_wait(ctx, complete, static_cast<uint64_t>(limit_ns));
}

int occult_route(const occult_desc_t* desc, const float* logits, const int32_t* expert_to_vdev,
                 int32_t* ids, float* gates, uint32_t* vmask, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->route_mode != OCCULT_ROUTE_SIMILARITY_PRUNED);
  OCCULT_REQUIRE(desc->T == 0 || (logits && expert_to_vdev && ids && gates && vmask));
  OCCULT_CTX(stream);
  return launch_route(ctx, *desc, logits, expert_to_vdev, nullptr, ids, gates, nullptr, vmask);
}

int occult_route_similarity(const occult_desc_t* desc, const float* logits,
                            const int32_t* expert_to_vdev, const float* table, int32_t* ids,
                            float* gates, int32_t* routed, uint32_t* vmask,
                            occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->route_mode == OCCULT_ROUTE_SIMILARITY_PRUNED);
  OCCULT_REQUIRE(desc->T == 0 || (logits && expert_to_vdev && table && ids && gates && vmask));
  OCCULT_CTX(stream);
  return launch_route(ctx, *desc, logits, expert_to_vdev, table, ids, gates, routed, vmask);
}

int occult_similarity_accumulate(const occult_desc_t* desc, const float* logits, int32_t n_tok,
                                 double* G, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(n_tok >= 0 && G && (n_tok == 0 || logits));
  OCCULT_REQUIRE(static_cast<int64_t>(n_tok) * desc->n_experts < (1ll << 31));
  OCCULT_CTX(stream);
  return launch_similarity_accumulate(ctx, desc->n_experts, logits, n_tok, G);
}

int occult_similarity_finish(const occult_desc_t* desc, const double* G, float* table,
                             occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(G && table);
  OCCULT_CTX(stream);
  return launch_similarity_finish(ctx, desc->n_experts, G, table);
}

int occult_router_grad(const occult_desc_t* desc, const float* logits, const int32_t* gate_ids,
                       const float* dgates, float* dlogits, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->T == 0 || (logits && gate_ids && dgates && dlogits));
  OCCULT_CTX(stream);
  return launch_router_grad(ctx, *desc, logits, gate_ids, dgates, dlogits);
}

int occult_build_brim(const occult_desc_t* desc, const int32_t* ids, const float* gates,
                      const uint32_t* vmask, const int32_t* placement, int32_t* brim0,
                      int32_t* seg_off, int32_t* brim1, int32_t* exp_off, int32_t* epd_src,
                      float* epd_gate, int32_t* counts, void* ws, size_t ws_bytes,
                      occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(placement && seg_off && exp_off && counts);
  OCCULT_REQUIRE(desc->T == 0 || (ids && gates && vmask && brim0 && brim1 && epd_src && epd_gate));
  const size_t need = brim_ws_bytes(*desc);
  if (ws_bytes < need || (need > 0 && !ws)) return OCCULT_ERR_WORKSPACE;
  OCCULT_CTX(stream);
  return launch_build_brim(ctx, *desc, ids, gates, vmask, placement, brim0, seg_off, brim1,
                           exp_off, epd_src, epd_gate, counts, ws);
}

int occult_dispatch(const occult_desc_t* desc, const void* x, const int32_t* brim0,
                    const uint32_t* vmask, void* x_sfd, int32_t* sfd_tok, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->T == 0 || (x && brim0 && vmask && x_sfd));
  // rows move as 16-byte vectors
  OCCULT_REQUIRE(reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(x_sfd) % 16 == 0);
  OCCULT_CTX(stream);
  return launch_dispatch(ctx, *desc, x, brim0, vmask, x_sfd, sfd_tok);
}

int occult_dispatch_epd(const occult_desc_t* desc, const void* x, const int32_t* ids,
                        const int32_t* placement, const int32_t* brim0, const int32_t* seg_off,
                        const int32_t* brim1, const int32_t* exp_off, void* x_epd,
                        occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  if (desc->dtype != OCCULT_BF16) return OCCULT_ERR_UNSUPPORTED;
  OCCULT_REQUIRE(placement && exp_off);
  OCCULT_REQUIRE(desc->T == 0 || (x && ids && brim0 && seg_off && brim1 && x_epd));
  OCCULT_REQUIRE(reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(x_epd) % 16 == 0);
  OCCULT_CTX(stream);
  return launch_dispatch_epd(ctx, *desc, x, ids, placement, brim0, seg_off, brim1, exp_off, x_epd);
}

static int expert_up(const LaunchCtx& ctx, const occult_desc_t* desc, const void* x_sfd,
                     const int32_t* epd_src, const float* epd_gate, const int32_t* exp_off,
                     const int32_t* placement, const void* w1, void* h_epd, void* gu_epd,
                     void* x_epd) {
  GroupedGemm g;
  g.a_mode = OP_GATHER_K;
  g.b_mode = OP_TMA_K;
  g.epi = EPI_SWIGLU;
  g.A = x_sfd;
  g.a_rows = static_cast<int64_t>(desc->T) * min_i(desc->top_k, desc->n_vdev);
  g.a_cols = desc->d;
  g.gather = epd_src;
  g.B = w1;
  g.b_rows = 2ll * desc->inter * desc->n_experts;
  g.b_cols = desc->d;
  g.b_group_rows = 2ll * desc->inter;
  g.n_groups = desc->n_experts;
  g.seg_off = exp_off;
  g.seg_group = placement;
  g.n_seg = desc->n_experts;
  g.max_rows = static_cast<int64_t>(desc->T) * desc->top_k;
  g.row_gate = epd_gate;
  g.out = h_epd;
  g.ldo = desc->inter;
  g.N_out = desc->inter;
  g.K = desc->d;
  g.gu_out = gu_epd;
  g.a_copy = x_epd;
  return desc->dtype == OCCULT_BF16 ? launch_grouped_gemm_bf16(ctx, g)
                                    : launch_grouped_gemm_f32(ctx, g);
}

static int expert_down(const LaunchCtx& ctx, const occult_desc_t* desc, const void* h_epd,
                       const int32_t* exp_off, const int32_t* placement, const void* w2,
                       void* y_epd, const int32_t* out_src = nullptr,
                       const int32_t* out_tok = nullptr) {
  GroupedGemm g;
  g.a_mode = OP_TMA_K;
  g.b_mode = OP_TMA_K;
  g.epi = EPI_F32;
  g.A = h_epd;
  g.a_rows = static_cast<int64_t>(desc->T) * desc->top_k;
  g.a_cols = desc->inter;
  g.gather = nullptr;
  g.B = w2;
  g.b_rows = static_cast<int64_t>(desc->d) * desc->n_experts;
  g.b_cols = desc->inter;
  g.b_group_rows = desc->d;
  g.n_groups = desc->n_experts;
  g.seg_off = exp_off;
  g.seg_group = placement;
  g.n_seg = desc->n_experts;
  g.max_rows = static_cast<int64_t>(desc->T) * desc->top_k;
  g.row_gate = nullptr;
  g.out = y_epd;
  g.ldo = desc->d;
  g.N_out = desc->d;
  g.K = desc->inter;
  g.out_src = out_src;
  g.out_tok = out_tok;
  g.out_rows = out_tok ? desc->T : 0;
  return desc->dtype == OCCULT_BF16 ? launch_grouped_gemm_bf16(ctx, g)
                                    : launch_grouped_gemm_f32(ctx, g);
}

int occult_expert_up(const occult_desc_t* desc, const void* x_sfd, const int32_t* epd_src,
                     const float* epd_gate, const int32_t* exp_off, const int32_t* placement,
                     const void* w1, void* h_epd, void* gu_epd, void* x_epd,
                     occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(exp_off && placement && w1);
  OCCULT_REQUIRE(desc->T == 0 || (x_sfd && epd_src && epd_gate && h_epd));
  OCCULT_REQUIRE(!(x_epd && !gu_epd));
  OCCULT_CTX(stream);
  if (desc->T == 0) return OCCULT_OK;
  if (gu_epd && desc->dtype != OCCULT_BF16) return OCCULT_ERR_UNSUPPORTED;
  return expert_up(ctx, desc, x_sfd, epd_src, epd_gate, exp_off, placement, w1, h_epd, gu_epd,
                   x_epd);
}

int occult_expert_down(const occult_desc_t* desc, const void* h_epd, const int32_t* exp_off,
                       const int32_t* placement, const void* w2, void* y_epd,
                       occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(exp_off && placement && w2);
  OCCULT_REQUIRE(desc->T == 0 || (h_epd && y_epd));
  OCCULT_CTX(stream);
  if (desc->T == 0) return OCCULT_OK;
  return expert_down(ctx, desc, h_epd, exp_off, placement, w2, y_epd);
}

int occult_expert_down_merge(const occult_desc_t* desc, const void* h_epd, const int32_t* exp_off,
                             const int32_t* placement, const void* w2, const int32_t* epd_src,
                             const int32_t* sfd_tok, void* y, int32_t zero_y,
                             occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(exp_off && placement && w2);
  OCCULT_REQUIRE(zero_y == 0 || zero_y == 1);
  OCCULT_REQUIRE(desc->T == 0 || (h_epd && epd_src && sfd_tok && y));
  OCCULT_CTX(stream);
  if (desc->T == 0) return OCCULT_OK;
  if (zero_y) {
    rc = launch_zero_f32(ctx, static_cast<float*>(y), static_cast<size_t>(desc->T) * desc->d);
    if (rc) return rc;
  }
  return expert_down(ctx, desc, h_epd, exp_off, placement, w2, y, epd_src, sfd_tok);
}

int occult_expert_ffn(const occult_desc_t* desc, const void* x_sfd, const int32_t* epd_src,
                      const float* epd_gate, const int32_t* exp_off, const int32_t* placement,
                      const void* w1, const void* w2, void* h_epd, void* y_epd,
                      occult_stream_t stream) {
  int rc = occult_expert_up(desc, x_sfd, epd_src, epd_gate, exp_off, placement, w1, h_epd,
                            nullptr, nullptr, stream);
  if (rc) return rc;
  return occult_expert_down(desc, h_epd, exp_off, placement, w2, y_epd, stream);
}

int occult_shared_ffn(const occult_desc_t* desc, const void* x, const void* ws1, const void* ws2,
                      const void* w_sg, void* h_s, float* s_gate, void* y_s,
                      occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->n_shared > 0);
  OCCULT_REQUIRE(!desc->shared_gate || (w_sg && s_gate));
  OCCULT_REQUIRE(desc->T == 0 || (x && ws1 && ws2 && h_s && y_s));
  OCCULT_CTX(stream);
  if (desc->T == 0) return OCCULT_OK;
  // one segment of T rows, identity gather, one weight group
  if (desc->shared_gate) {
    rc = launch_shared_gate(ctx, *desc, x, w_sg, s_gate);
    if (rc) return rc;
  }
  const int S = desc->n_shared * desc->shared_inter;
  GroupedGemm g;
  g.a_mode = OP_TMA_K;
  g.b_mode = OP_TMA_K;
  g.epi = EPI_SWIGLU;
  g.A = x;
  g.a_rows = desc->T;
  g.a_cols = desc->d;
  g.gather = nullptr;
  g.B = ws1;
  g.b_rows = 2ll * S;
  g.b_cols = desc->d;
  g.b_group_rows = 2ll * S;
  g.n_groups = 1;
  g.seg_off = nullptr;
  g.seg_group = nullptr;
  g.n_seg = 1;
  g.max_rows = desc->T;
  g.row_gate = desc->shared_gate ? s_gate : nullptr;
  g.out = h_s;
  g.ldo = S;
  g.N_out = S;
  g.K = desc->d;
  rc = desc->dtype == OCCULT_BF16 ? launch_grouped_gemm_bf16(ctx, g) : launch_grouped_gemm_f32(ctx, g);
  if (rc) return rc;
  g.epi = EPI_F32;
  g.A = h_s;
  g.a_rows = desc->T;
  g.a_cols = S;
  g.B = ws2;
  g.b_rows = desc->d;
  g.b_cols = S;
  g.b_group_rows = desc->d;
  g.row_gate = nullptr;
  g.out = y_s;
  g.ldo = desc->d;
  g.N_out = desc->d;
  g.K = S;
  return desc->dtype == OCCULT_BF16 ? launch_grouped_gemm_bf16(ctx, g) : launch_grouped_gemm_f32(ctx, g);
}

// The four GEMMs of the expert backward.  Argument checks are done by the public
// entry points; T > 0 here.

// dh' = dy_sfd[src] . W_d (W_d read MN-major), SwiGLU backward -> dG|dU, dg; with
// dy_epd given, the gathered dy rows are also written to that padded EPD copy.
// Without dy_sfd the dy rows are read as tiles from dy_epd (occult_dispatch_epd).
static int dgrad_down(const LaunchCtx& ctx, const occult_desc_t* desc, const void* dy_sfd,
                      const int32_t* epd_src, const float* epd_gate, const int32_t* exp_off,
                      const int32_t* placement, const void* w2, const void* gu_epd,
                      void* dgu_epd, float* dg_epd, void* dy_epd, void* ws) {
  const int64_t rows = static_cast<int64_t>(desc->T) * desc->top_k;
  const int64_t n_sfd_max = static_cast<int64_t>(desc->T) * min_i(desc->top_k, desc->n_vdev);
  const int Ne = desc->n_experts, d = desc->d, I = desc->inter;
  float* dg_part = static_cast<float*>(ws);
  GroupedGemm g;
  g.a_mode = OP_GATHER_K;
  g.b_mode = OP_TMA_MN;
  g.epi = EPI_SWIGLU_BWD;
  g.A = dy_sfd; g.a_rows = n_sfd_max; g.a_cols = d;
  g.gather = epd_src;
  g.B = w2; g.b_rows = static_cast<int64_t>(Ne) * d; g.b_cols = I;
  g.b_group_rows = d;
  g.n_groups = Ne;
  g.seg_off = exp_off; g.seg_group = placement; g.n_seg = Ne; g.max_rows = rows;
  g.K = d; g.N_out = I;
  g.row_gate = epd_gate;
  g.out = dgu_epd; g.ldo = 2ll * I;
  g.gu_in = gu_epd; g.dg_part = dg_part;
  g.a_copy = dy_epd;
  if (!dy_sfd) {
    g.a_mode = OP_TMA_K;
    g.A = dy_epd; g.a_rows = rows + static_cast<int64_t>(OCCULT_EPD_PAD) * Ne;
    g.a_pad = OCCULT_EPD_PAD;
    g.gather = nullptr;
    g.a_copy = nullptr;
  }
  int rc = launch_grouped_gemm_bf16(ctx, g);
  if (rc) return rc;
  return launch_dg_reduce(ctx, dg_part, static_cast<int>(rows), 2 * ((I + 255) / 256), dg_epd);
}

// dx_epd = [dG|dU] . [W_g; W_u] (W1 read MN-major), fp32; with sfd_tok given the
// rows are added into dx[token] (fp32 atomics) instead of written to dx_out's EPD rows
static int dgrad_up(const LaunchCtx& ctx, const occult_desc_t* desc, const void* dgu_epd,
                    const int32_t* epd_src, const int32_t* exp_off, const int32_t* placement,
                    const void* w1, const int32_t* sfd_tok, float* dx_out) {
  const int64_t rows = static_cast<int64_t>(desc->T) * desc->top_k;
  const int Ne = desc->n_experts, d = desc->d, I = desc->inter;
  GroupedGemm h;
  h.a_mode = OP_TMA_K;
  h.b_mode = OP_TMA_MN;
  h.epi = EPI_F32;
  h.A = dgu_epd; h.a_rows = rows; h.a_cols = 2ll * I;
  h.B = w1; h.b_rows = 2ll * I * Ne; h.b_cols = d;
  h.b_group_rows = 2ll * I;
  h.n_groups = Ne;
  h.seg_off = exp_off; h.seg_group = placement; h.n_seg = Ne; h.max_rows = rows;
  h.K = 2 * I; h.N_out = d;
  h.out = dx_out; h.ldo = d;
  if (sfd_tok) {
    h.out_src = epd_src;
    h.out_tok = sfd_tok;
    h.out_rows = desc->T;
  }
  return launch_grouped_gemm_bf16(ctx, h);
}

// dW_d[e] = sum over e's rows of dy_sfd[src] (x) h' : M = d, N = I; the dy rows
// gathered from dy_sfd, or read as tiles from their padded EPD copy dy_epd
static int wgrad_down(const LaunchCtx& ctx, const occult_desc_t* desc, const void* dy_sfd,
                      const int32_t* epd_src, const void* dy_epd, const int32_t* exp_off,
                      const int32_t* placement, const void* h_epd, float* dw2) {
  const int64_t rows = static_cast<int64_t>(desc->T) * desc->top_k;
  const int64_t n_sfd_max = static_cast<int64_t>(desc->T) * min_i(desc->top_k, desc->n_vdev);
  const int Ne = desc->n_experts, d = desc->d, I = desc->inter;
  GroupedGemm w;
  w.wgrad = true;
  w.a_mode = OP_GATHER_MN;
  w.b_mode = OP_TMA_MN;
  w.epi = EPI_F32;
  w.A = dy_sfd; w.a_rows = n_sfd_max; w.a_cols = d;
  w.gather = epd_src;
  if (dy_epd) {
    w.a_mode = OP_TMA_MN;
    w.A = dy_epd; w.a_rows = rows + static_cast<int64_t>(OCCULT_EPD_PAD) * Ne;
    w.a_pad = OCCULT_EPD_PAD;
    w.gather = nullptr;
  }
  w.B = h_epd; w.b_rows = rows; w.b_cols = I;
  w.seg_off = exp_off; w.seg_group = placement; w.n_seg = Ne;
  w.M_total = d; w.N_out = I;
  w.out = dw2; w.ldo = I; w.out_group_stride = static_cast<int64_t>(d) * I;
  return launch_grouped_gemm_bf16(ctx, w);
}

// [dW_g; dW_u][e] = sum over e's rows of [dG|dU] (x) x_sfd[src] : M = 2I, N = d; the x
// rows gathered from x_sfd, or read as tiles from their padded EPD copy x_epd
static int wgrad_up(const LaunchCtx& ctx, const occult_desc_t* desc, const void* x_sfd,
                    const int32_t* epd_src, const void* x_epd, const int32_t* exp_off,
                    const int32_t* placement, const void* dgu_epd, float* dw1) {
  const int64_t rows = static_cast<int64_t>(desc->T) * desc->top_k;
  const int64_t n_sfd_max = static_cast<int64_t>(desc->T) * min_i(desc->top_k, desc->n_vdev);
  const int Ne = desc->n_experts, d = desc->d, I = desc->inter;
  GroupedGemm v;
  v.wgrad = true;
  v.a_mode = OP_TMA_MN;
  v.b_mode = OP_GATHER_MN;
  v.epi = EPI_F32;
  v.A = dgu_epd; v.a_rows = rows; v.a_cols = 2ll * I;
  v.B = x_sfd; v.b_rows = n_sfd_max; v.b_cols = d;
  v.gather = epd_src;
  if (x_epd) {
    v.b_mode = OP_TMA_MN;
    v.B = x_epd; v.b_rows = rows + static_cast<int64_t>(OCCULT_EPD_PAD) * Ne;
    v.b_pad = OCCULT_EPD_PAD;
    v.gather = nullptr;
  }
  v.seg_off = exp_off; v.seg_group = placement; v.n_seg = Ne;
  v.M_total = 2 * I; v.N_out = d;
  v.out = dw1; v.ldo = d; v.out_group_stride = 2ll * I * d;
  return launch_grouped_gemm_bf16(ctx, v);
}

static int zero_weights(const LaunchCtx& ctx, float* w, size_t n) {
  return cudaMemsetAsync(w, 0, n * sizeof(float), ctx.stream) == cudaSuccess ? OCCULT_OK
                                                                             : OCCULT_ERR_CUDA;
}

static size_t w1_elems(const occult_desc_t* desc) {
  return static_cast<size_t>(desc->n_experts) * 2 * desc->inter * desc->d;
}
static size_t w2_elems(const occult_desc_t* desc) {
  return static_cast<size_t>(desc->n_experts) * desc->d * desc->inter;
}

// The expert backward; with sfd_tok given, the dgrad through [W_g; W_u] adds its
// rows into dx[token] (fp32 atomics) instead of writing the EPD rows to dx_out.
static int expert_bwd(const occult_desc_t* desc, const void* x_sfd, const void* dy_sfd,
                      const int32_t* epd_src, const float* epd_gate, const int32_t* exp_off,
                      const int32_t* placement, const void* w1, const void* w2,
                      const void* h_epd, const void* gu_epd, void* dgu_epd, float* dx_out,
                      const int32_t* sfd_tok, float* dw1, float* dw2, float* dg_epd,
                      const void* x_epd, void* dy_epd, void* ws, size_t ws_bytes,
                      occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  if (desc->dtype != OCCULT_BF16) return OCCULT_ERR_UNSUPPORTED;
  OCCULT_REQUIRE(exp_off && placement && w1 && w2 && dw1 && dw2);
  OCCULT_REQUIRE(desc->T == 0 || ((x_sfd || x_epd) && (dy_sfd || dy_epd) && epd_src && epd_gate &&
                                  h_epd && gu_epd && dgu_epd && dx_out && dg_epd));
  const size_t need = expert_bwd_ws_bytes(*desc);
  if (ws_bytes < need || (need > 0 && !ws)) return OCCULT_ERR_WORKSPACE;
  OCCULT_CTX(stream);
  if (desc->T == 0) {
    // no rows: every weight gradient is zero
    rc = zero_weights(ctx, dw1, w1_elems(desc));
    return rc ? rc : zero_weights(ctx, dw2, w2_elems(desc));
  }
  if (sfd_tok) {
    rc = launch_zero_f32(ctx, dx_out, static_cast<size_t>(desc->T) * desc->d);
    if (rc) return rc;
  }
  rc = dgrad_down(ctx, desc, dy_sfd, epd_src, epd_gate, exp_off, placement, w2, gu_epd, dgu_epd,
                  dg_epd, dy_epd, ws);
  if (rc) return rc;
  rc = dgrad_up(ctx, desc, dgu_epd, epd_src, exp_off, placement, w1, sfd_tok, dx_out);
  if (rc) return rc;
  rc = wgrad_down(ctx, desc, dy_sfd, epd_src, dy_epd, exp_off, placement, h_epd, dw2);
  if (rc) return rc;
  return wgrad_up(ctx, desc, x_sfd, epd_src, x_epd, exp_off, placement, dgu_epd, dw1);
}

int occult_expert_bwd(const occult_desc_t* desc, const void* x_sfd, const void* dy_sfd,
                      const int32_t* epd_src, const float* epd_gate, const int32_t* exp_off,
                      const int32_t* placement, const void* w1, const void* w2,
                      const void* h_epd, const void* gu_epd, void* dgu_epd, float* dx_epd,
                      float* dw1, float* dw2, float* dg_epd, const void* x_epd, void* dy_epd,
                      void* ws, size_t ws_bytes, occult_stream_t stream) {
  return expert_bwd(desc, x_sfd, dy_sfd, epd_src, epd_gate, exp_off, placement, w1, w2, h_epd,
                    gu_epd, dgu_epd, dx_epd, nullptr, dw1, dw2, dg_epd, x_epd, dy_epd, ws,
                    ws_bytes, stream);
}

int occult_expert_bwd_merge(const occult_desc_t* desc, const void* x_sfd, const void* dy_sfd,
                            const int32_t* epd_src, const float* epd_gate, const int32_t* exp_off,
                            const int32_t* placement, const void* w1, const void* w2,
                            const void* h_epd, const void* gu_epd, void* dgu_epd,
                            const int32_t* sfd_tok, float* dx, float* dw1, float* dw2,
                            float* dg_epd, const void* x_epd, void* dy_epd, void* ws,
                            size_t ws_bytes, occult_stream_t stream) {
  if (desc && desc->T > 0 && !sfd_tok) return OCCULT_ERR_INVALID_ARG;
  return expert_bwd(desc, x_sfd, dy_sfd, epd_src, epd_gate, exp_off, placement, w1, w2, h_epd,
                    gu_epd, dgu_epd, dx, sfd_tok, dw1, dw2, dg_epd, x_epd, dy_epd, ws, ws_bytes,
                    stream);
}

int occult_expert_dgrad_down(const occult_desc_t* desc, const void* dy_sfd,
                             const int32_t* epd_src, const float* epd_gate,
                             const int32_t* exp_off, const int32_t* placement, const void* w2,
                             const void* gu_epd, void* dgu_epd, float* dg_epd, void* dy_epd,
                             void* ws, size_t ws_bytes, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  if (desc->dtype != OCCULT_BF16) return OCCULT_ERR_UNSUPPORTED;
  OCCULT_REQUIRE(exp_off && placement && w2);
  OCCULT_REQUIRE(desc->T == 0 || ((dy_sfd || dy_epd) && epd_src && epd_gate && gu_epd && dgu_epd &&
                                  dg_epd));
  const size_t need = expert_bwd_ws_bytes(*desc);
  if (ws_bytes < need || (need > 0 && !ws)) return OCCULT_ERR_WORKSPACE;
  OCCULT_CTX(stream);
  if (desc->T == 0) return OCCULT_OK;
  return dgrad_down(ctx, desc, dy_sfd, epd_src, epd_gate, exp_off, placement, w2, gu_epd, dgu_epd,
                    dg_epd, dy_epd, ws);
}

int occult_expert_dgrad_up(const occult_desc_t* desc, const void* dgu_epd, const int32_t* epd_src,
                           const int32_t* exp_off, const int32_t* placement, const void* w1,
                           const int32_t* sfd_tok, float* dx, int32_t zero_dx,
                           occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  if (desc->dtype != OCCULT_BF16) return OCCULT_ERR_UNSUPPORTED;
  OCCULT_REQUIRE(exp_off && placement && w1);
  OCCULT_REQUIRE(zero_dx == 0 || zero_dx == 1);
  OCCULT_REQUIRE(!(zero_dx && !sfd_tok));
  OCCULT_REQUIRE(desc->T == 0 || (dgu_epd && epd_src && dx));
  OCCULT_CTX(stream);
  if (desc->T == 0) return OCCULT_OK;
  if (zero_dx) {
    rc = launch_zero_f32(ctx, dx, static_cast<size_t>(desc->T) * desc->d);
    if (rc) return rc;
  }
  return dgrad_up(ctx, desc, dgu_epd, epd_src, exp_off, placement, w1, sfd_tok, dx);
}

int occult_expert_wgrad_down(const occult_desc_t* desc, const void* dy_sfd,
                             const int32_t* epd_src, const void* dy_epd, const int32_t* exp_off,
                             const int32_t* placement, const void* h_epd, float* dw2,
                             occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  if (desc->dtype != OCCULT_BF16) return OCCULT_ERR_UNSUPPORTED;
  OCCULT_REQUIRE(exp_off && placement && dw2);
  OCCULT_REQUIRE(desc->T == 0 || ((dy_epd || (dy_sfd && epd_src)) && h_epd));
  OCCULT_CTX(stream);
  if (desc->T == 0) return zero_weights(ctx, dw2, w2_elems(desc));
  return wgrad_down(ctx, desc, dy_sfd, epd_src, dy_epd, exp_off, placement, h_epd, dw2);
}

int occult_expert_wgrad_up(const occult_desc_t* desc, const void* x_sfd, const int32_t* epd_src,
                           const void* x_epd, const int32_t* exp_off, const int32_t* placement,
                           const void* dgu_epd, float* dw1, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  if (desc->dtype != OCCULT_BF16) return OCCULT_ERR_UNSUPPORTED;
  OCCULT_REQUIRE(exp_off && placement && dw1);
  OCCULT_REQUIRE(desc->T == 0 || ((x_epd || (x_sfd && epd_src)) && dgu_epd));
  OCCULT_CTX(stream);
  if (desc->T == 0) return zero_weights(ctx, dw1, w1_elems(desc));
  return wgrad_up(ctx, desc, x_sfd, epd_src, x_epd, exp_off, placement, dgu_epd, dw1);
}

int occult_zero_f32(float* buf, int64_t n, occult_stream_t stream) {
  OCCULT_REQUIRE(n >= 0 && (n == 0 || buf));
  OCCULT_CTX(stream);
  if (n == 0) return OCCULT_OK;
  return launch_zero_f32(ctx, buf, static_cast<size_t>(n));
}

int occult_gate_grad(const occult_desc_t* desc, const int32_t* ids, const int32_t* placement,
                     const int32_t* brim0, const int32_t* seg_off, const int32_t* brim1,
                     const int32_t* exp_off, const float* dg_epd, float* dgates,
                     occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->T == 0 || (ids && placement && brim0 && seg_off && brim1 && exp_off &&
                                  dg_epd && dgates));
  OCCULT_CTX(stream);
  return launch_gate_grad(ctx, *desc, ids, placement, brim0, seg_off, brim1, exp_off, dg_epd,
                          dgates);
}

int occult_combine(const occult_desc_t* desc, const void* y_epd, const int32_t* brim0,
                   const int32_t* seg_off, const int32_t* brim1, const int32_t* exp_off,
                   const void* y_shared, void* y_sfd, void* y, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->T == 0 || (y_epd && brim0 && seg_off && brim1 && exp_off && y));
  OCCULT_CTX(stream);
  return launch_combine(ctx, *desc, static_cast<const float*>(y_epd), brim0, seg_off, brim1,
                        exp_off, static_cast<const float*>(y_shared), static_cast<float*>(y_sfd),
                        static_cast<float*>(y));
}

int occult_merge_sfd(const occult_desc_t* desc, const void* y_epd, const int32_t* brim0,
                     const int32_t* seg_off, const int32_t* brim1, const int32_t* exp_off,
                     void* y_sfd, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->T == 0 || (y_epd && brim0 && seg_off && brim1 && exp_off && y_sfd));
  OCCULT_CTX(stream);
  return launch_merge_sfd(ctx, *desc, static_cast<const float*>(y_epd), brim0, seg_off, brim1,
                          exp_off, static_cast<float*>(y_sfd));
}

int occult_combine_sfd(const occult_desc_t* desc, const void* y_sfd, const int32_t* row_map,
                       const void* y_shared, void* y, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->T == 0 || (y_sfd && row_map && y));
  OCCULT_CTX(stream);
  return launch_combine_sfd(ctx, *desc, static_cast<const float*>(y_sfd), row_map,
                            static_cast<const float*>(y_shared), static_cast<float*>(y));
}

int occult_shard_plan(const occult_desc_t* desc, int32_t n_src, const int32_t* src_off,
                      const uint32_t* vmask, const int32_t* brim0, int32_t* brim0_send,
                      int32_t* counts, int32_t* send_off, int32_t* recv_off,
                      occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(n_src >= 1 && n_src <= OCCULT_MAX_SOURCES && src_off);
  OCCULT_REQUIRE(counts && send_off && recv_off);
  OCCULT_REQUIRE(desc->T == 0 || (vmask && brim0 && brim0_send));
  ShardSplit split;
  split.n = n_src;
  OCCULT_REQUIRE(src_off[0] == 0 && src_off[n_src] == desc->T);
  for (int s = 0; s <= n_src; ++s) {
    OCCULT_REQUIRE(s == 0 || src_off[s] >= src_off[s - 1]);
    split.off[s] = src_off[s];
  }
  OCCULT_CTX(stream);
  return launch_shard_plan(ctx, *desc, split, vmask, brim0, brim0_send, counts, send_off,
                           recv_off);
}

int occult_all_to_all(const occult_desc_t* desc, int32_t n_src, const int32_t* counts,
                      const int32_t* send_off, const int32_t* recv_off, const void* src,
                      void* dst, int64_t row_bytes, int32_t reverse, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(n_src >= 1 && n_src <= OCCULT_MAX_SOURCES);
  OCCULT_REQUIRE(counts && send_off && recv_off);
  OCCULT_REQUIRE(row_bytes > 0 && row_bytes % 16 == 0);
  OCCULT_REQUIRE(reverse == 0 || reverse == 1);
  OCCULT_REQUIRE(desc->T == 0 || (src && dst));
  OCCULT_REQUIRE(reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(dst) % 16 == 0);
  if (desc->T > 0) {
    // the two buffers must not overlap
    const int64_t rows = static_cast<int64_t>(desc->T) * min_i(desc->top_k, desc->n_vdev);
    const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(dst);
    const uintptr_t n = static_cast<uintptr_t>(rows * row_bytes);
    OCCULT_REQUIRE(a + n <= b || b + n <= a);
  }
  OCCULT_CTX(stream);
  return launch_all_to_all(ctx, *desc, n_src, src, dst, row_bytes, counts, send_off, recv_off,
                           reverse);
}

int occult_profile_coact(const occult_desc_t* desc, const int32_t* ids, int32_t n_tok,
                         const uint32_t* vmask, int64_t* C, float* P, int64_t* ct_hist, void* ws,
                         size_t ws_bytes, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(n_tok >= 0 && C);
  OCCULT_REQUIRE(n_tok == 0 || ids);
  OCCULT_REQUIRE(!ct_hist || vmask);
  const size_t need = profile_ws_bytes(*desc, n_tok);
  if (ws_bytes < need || (need > 0 && !ws)) return OCCULT_ERR_WORKSPACE;
  OCCULT_CTX(stream);
  return launch_profile(ctx, *desc, ids, n_tok, vmask, C, P, ct_hist, ws);
}

}  // extern "C"
