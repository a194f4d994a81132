// Backward helpers of the Occult layer: the gate gradient per EPD row (sum of the
// SwiGLU-backward epilogue's per-tile partials), its transposed BRIM merge back
// to token order (the same BRIM0 -> BRIM1 walk the forward combine uses), and
// the gradient of the router logits through the softmax of Eq. 2.
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

__global__ void __launch_bounds__(256)
dg_reduce_kernel(const float* __restrict__ part, int rows, int n_part, float* __restrict__ dg) {
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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
  launch_pdl(dg_reduce_kernel, blocks_for(ctx, rows), 256, 0, ctx.stream, part, rows, n_part, dg);
  return cuda_status(cudaGetLastError());
}

int launch_gate_grad(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids,
                     const int32_t* placement, const int32_t* brim0, const int32_t* seg_off,
                     const int32_t* brim1, const int32_t* exp_off, const float* dg_epd,
                     float* dgates) {
  const int64_t n = static_cast<int64_t>(ds.T) * ds.top_k;
  if (n == 0) return OCCULT_OK;
  launch_pdl(gate_grad_kernel, blocks_for(ctx, n), 256, 0, ctx.stream,
      ids, placement, brim0, seg_off, brim1, exp_off, dg_epd, ds.T, ds.top_k, ds.n_experts,
      ds.n_experts / ds.n_vdev, dgates);
  return cuda_status(cudaGetLastError());
}

namespace {

// d-logits through Eq. 2's softmax: one warp per token, lane l holds experts
// l, l+32, ...  p = softmax(z) as the router computes it (fp32, max subtracted,
// fixed-order warp tree); the gates are g_j = p[gate_ids_j], renormalised over j
// when `renorm`.  With A = sum_j dg_j g_j:
//   plain:   dz_e = p_e (sum_{j: id_j = e} dg_j - A)
//   renorm:  dz_e = sum_{j: id_j = e} g_j (dg_j - A)   (0 for unselected experts)
template <int PER_LANE>
__global__ void __launch_bounds__(256)
router_grad_kernel(const float* __restrict__ logits, const int32_t* __restrict__ gate_ids,
                   const float* __restrict__ dgates, int T, int Ne, int k, int renorm,
                   float* __restrict__ dlogits) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const float NEG = -__int_as_float(0x7f800000);
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += gridDim.x * 8) {
    const float* row = logits + static_cast<size_t>(t) * Ne;
    float v[PER_LANE];
    float mx = NEG;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < Ne ? row[e] : NEG;
      mx = fmaxf(mx, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float p[PER_LANE];
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      p[i] = (lane + 32 * i < Ne) ? expf(v[i] - mx) : 0.f;
      part += p[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    const float Z = part;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) p[i] = p[i] / Z;
    // lane j < k: slot j's expert, upstream gradient and gate
    const int gid = lane < k ? gate_ids[static_cast<size_t>(t) * k + lane] : 0;
    const float dg = lane < k ? dgates[static_cast<size_t>(t) * k + lane] : 0.f;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const float pi = __shfl_sync(0xffffffffu, p[i], gid & 31);
      if ((gid >> 5) == i) q = pi;
    }
    if (lane >= k) q = 0.f;
    float S = q;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    const float g = renorm ? q / S : q;
    float A = dg * g;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) A += __shfl_xor_sync(0xffffffffu, A, o);
    float dz[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) dz[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e_j = __shfl_sync(0xffffffffu, gid, j);
      const float dg_j = __shfl_sync(0xffffffffu, dg, j);
      const float g_j = __shfl_sync(0xffffffffu, g, j);
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i)
        if (lane + 32 * i == e_j) dz[i] += renorm ? g_j * (dg_j - A) : dg_j;
    }
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (e < Ne) dlogits[static_cast<size_t>(t) * Ne + e] = renorm ? dz[i] : p[i] * (dz[i] - A);
    }
  }
}

}  // namespace

int launch_router_grad(const LaunchCtx& ctx, const occult_desc_t& ds, const float* logits,
                       const int32_t* gate_ids, const float* dgates, float* dlogits) {
  if (ds.T == 0) return OCCULT_OK;
  int blocks = (ds.T + 7) / 8;
  if (blocks > ctx.num_sms * 16) blocks = ctx.num_sms * 16;
#define OCCULT_RGRAD_LAUNCH(PL)                                                            \
  launch_pdl(router_grad_kernel<PL>, blocks, 256, 0, ctx.stream, logits, gate_ids, dgates, ds.T,   \
                                                          ds.n_experts, ds.top_k, ds.renorm, \
                                                          dlogits)
  if (ds.n_experts <= 32) OCCULT_RGRAD_LAUNCH(1);
  else if (ds.n_experts <= 64) OCCULT_RGRAD_LAUNCH(2);
  else if (ds.n_experts <= 128) OCCULT_RGRAD_LAUNCH(4);
  else OCCULT_RGRAD_LAUNCH(8);
#undef OCCULT_RGRAD_LAUNCH
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
