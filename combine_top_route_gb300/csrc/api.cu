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
  if (ds->route_mode != OCCULT_ROUTE_EXACT && ds->route_mode != OCCULT_ROUTE_DEVICE_LIMITED)
    return OCCULT_ERR_INVALID_ARG;
  if (ds->n_experts > OCCULT_MAX_EXPERTS || ds->n_vdev > OCCULT_MAX_VDEV ||
      ds->top_k > OCCULT_MAX_TOPK)
    return OCCULT_ERR_UNSUPPORTED;
  const int n_loc = ds->n_experts / ds->n_vdev;
  if (ds->route_mode == OCCULT_ROUTE_DEVICE_LIMITED) {
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

int occult_route(const occult_desc_t* desc, const float* logits, const int32_t* expert_to_vdev,
                 int32_t* ids, float* gates, uint32_t* vmask, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(desc->T == 0 || (logits && expert_to_vdev && ids && gates && vmask));
  OCCULT_CTX(stream);
  return launch_route(ctx, *desc, logits, expert_to_vdev, ids, gates, vmask);
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
  OCCULT_CTX(stream);
  return launch_dispatch(ctx, *desc, x, brim0, vmask, x_sfd, sfd_tok);
}

static int expert_up(const LaunchCtx& ctx, const occult_desc_t* desc, const void* x_sfd,
                     const int32_t* epd_src, const float* epd_gate, const int32_t* exp_off,
                     const int32_t* placement, const void* w1, void* h_epd) {
  GroupedGemm g;
  g.A = x_sfd;
  g.a_rows = static_cast<int64_t>(desc->T) * min_i(desc->top_k, desc->n_vdev);
  g.gather = epd_src;
  g.B = w1;
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
  g.swiglu = true;
  return desc->dtype == OCCULT_BF16 ? launch_grouped_gemm_bf16(ctx, g)
                                    : launch_grouped_gemm_f32(ctx, g);
}

static int expert_down(const LaunchCtx& ctx, const occult_desc_t* desc, const void* h_epd,
                       const int32_t* exp_off, const int32_t* placement, const void* w2,
                       void* y_epd) {
  GroupedGemm g;
  g.A = h_epd;
  g.a_rows = static_cast<int64_t>(desc->T) * desc->top_k;
  g.gather = nullptr;
  g.B = w2;
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
  g.swiglu = false;
  return desc->dtype == OCCULT_BF16 ? launch_grouped_gemm_bf16(ctx, g)
                                    : launch_grouped_gemm_f32(ctx, g);
}

int occult_expert_up(const occult_desc_t* desc, const void* x_sfd, const int32_t* epd_src,
                     const float* epd_gate, const int32_t* exp_off, const int32_t* placement,
                     const void* w1, void* h_epd, occult_stream_t stream) {
  int rc = check(desc);
  if (rc) return rc;
  OCCULT_REQUIRE(exp_off && placement && w1);
  OCCULT_REQUIRE(desc->T == 0 || (x_sfd && epd_src && epd_gate && h_epd));
  OCCULT_CTX(stream);
  if (desc->T == 0) return OCCULT_OK;
  return expert_up(ctx, desc, x_sfd, epd_src, epd_gate, exp_off, placement, w1, h_epd);
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

int occult_expert_ffn(const occult_desc_t* desc, const void* x_sfd, const int32_t* epd_src,
                      const float* epd_gate, const int32_t* exp_off, const int32_t* placement,
                      const void* w1, const void* w2, void* h_epd, void* y_epd,
                      occult_stream_t stream) {
  int rc = occult_expert_up(desc, x_sfd, epd_src, epd_gate, exp_off, placement, w1, h_epd, stream);
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
  g.A = x;
  g.a_rows = desc->T;
  g.gather = nullptr;
  g.B = ws1;
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
  g.swiglu = true;
  rc = desc->dtype == OCCULT_BF16 ? launch_grouped_gemm_bf16(ctx, g) : launch_grouped_gemm_f32(ctx, g);
  if (rc) return rc;
  g.A = h_s;
  g.a_rows = desc->T;
  g.B = ws2;
  g.b_group_rows = desc->d;
  g.row_gate = nullptr;
  g.out = y_s;
  g.ldo = desc->d;
  g.N_out = desc->d;
  g.K = S;
  g.swiglu = false;
  return desc->dtype == OCCULT_BF16 ? launch_grouped_gemm_bf16(ctx, g) : launch_grouped_gemm_f32(ctx, g);
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
