// Backward helpers of the Occult layer: the gate gradient per EPD row (sum of the
// SwiGLU-backward epilogue's per-tile partials), and its transposed BRIM merge
// back to token order (the same BRIM0 -> BRIM1 walk the forward combine uses).
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

__global__ void __launch_bounds__(256)
dg_reduce_kernel(const float* __restrict__ part, int rows, int n_part, float* __restrict__ dg) {
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int i = 0; i < n_part; ++i) s += part[static_cast<size_t>(r) * n_part + i];
    dg[r] = s;
  }
}

// dgates[t, j] = dg_epd[EPD row of (t, ids[t, j])]: slot s of the expert, its
// device d, the token's received row BRIM0[d, t], then BRIM1[s, row].
__global__ void __launch_bounds__(256)
gate_grad_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ placement,
                 const int32_t* __restrict__ brim0, const int32_t* __restrict__ seg_off,
                 const int32_t* __restrict__ brim1, const int32_t* __restrict__ exp_off,
                 const float* __restrict__ dg_epd, int T, int k, int Ne, int n_loc,
                 float* __restrict__ dgates) {
  __shared__ int s_slot_of[OCCULT_MAX_EXPERTS];
  for (int s = threadIdx.x; s < Ne; s += blockDim.x) s_slot_of[placement[s]] = s;
  __syncthreads();
  const int n = T * k;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int t = i / k;
    const int s = s_slot_of[ids[i]];
    const int d = s / n_loc;
    const int r_local = brim0[static_cast<size_t>(d) * T + t] - seg_off[d];
    const int u = brim1[static_cast<size_t>(s) * T + r_local];
    dgates[i] = dg_epd[exp_off[d * n_loc] + u];
  }
}

int blocks_for(const LaunchCtx& ctx, int64_t n) {
  int64_t b = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(ctx.num_sms) * 8;
  return static_cast<int>(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

size_t expert_bwd_ws_bytes(const occult_desc_t& ds) {
  // one partial gate gradient per EPD row, 256-column tile of I and column half
  const size_t n_part = 2 * ((static_cast<size_t>(ds.inter) + 255) / 256);
  return static_cast<size_t>(ds.T) * ds.top_k * n_part * sizeof(float);
}

int launch_dg_reduce(const LaunchCtx& ctx, const float* part, int rows, int n_part, float* dg) {
  if (rows == 0) return OCCULT_OK;
  dg_reduce_kernel<<<blocks_for(ctx, rows), 256, 0, ctx.stream>>>(part, rows, n_part, dg);
  return cuda_status(cudaGetLastError());
}

int launch_gate_grad(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids,
                     const int32_t* placement, const int32_t* brim0, const int32_t* seg_off,
                     const int32_t* brim1, const int32_t* exp_off, const float* dg_epd,
                     float* dgates) {
  const int64_t n = static_cast<int64_t>(ds.T) * ds.top_k;
  if (n == 0) return OCCULT_OK;
  gate_grad_kernel<<<blocks_for(ctx, n), 256, 0, ctx.stream>>>(
      ids, placement, brim0, seg_off, brim1, exp_off, dg_epd, ds.T, ds.top_k, ds.n_experts,
      ds.n_experts / ds.n_vdev, dgates);
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
