// Router kernel: Occult paper Sec. 2.1 Eq. 2 (top-k of the softmax of the
// router logits) and the device-limited pruning mode of Sec. 3.3 (keep a few
// devices, choose the top-k among their experts).
//
// One warp per token.  Lane l holds experts l, l+32, ... (up to 8 per lane for
// 256 experts).  The softmax denominator is a fixed-order warp tree, so the
// gates are deterministic; the top-k choice is made on the fp32 logits
// (descending value, lower id first) and never depends on exp rounding.
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

constexpr int kWarpsPerBlock = 8;

struct Cand {
  float v;
  int id;
};

// true if a ranks before b: larger logit, or equal logit and lower id
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v = __shfl_xor_sync(0xffffffffu, c.v, o);
    int id = __shfl_xor_sync(0xffffffffu, c.id, o);
    if (before(v, id, c.v, c.id)) { c.v = v; c.id = id; }
  }
  return c;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int PER_LANE>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_kernel(const float* __restrict__ logits, const int32_t* __restrict__ e2v, int T, int Ne,
             int k, int Nd, int renorm, int limited, int n_keep, int32_t* __restrict__ ids,
             float* __restrict__ gates, uint32_t* __restrict__ vmask) {
  __shared__ float s_ex[kWarpsPerBlock][PER_LANE * 32];
  __shared__ int s_dev[PER_LANE * 32];
  for (int e = threadIdx.x; e < PER_LANE * 32; e += blockDim.x) s_dev[e] = e < Ne ? e2v[e] : -1;
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float NEG = -__int_as_float(0x7f800000);  // -inf

  for (int t = blockIdx.x * kWarpsPerBlock + warp; t < T; t += gridDim.x * kWarpsPerBlock) {
    const float* row = logits + static_cast<size_t>(t) * Ne;
    float v[PER_LANE];
    int dev[PER_LANE];
    float mx = NEG;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < Ne ? row[e] : NEG;
      dev[i] = s_dev[e];
      mx = fmaxf(mx, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float ex[PER_LANE];
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      ex[i] = (lane + 32 * i < Ne) ? expf(v[i] - mx) : 0.f;
      part += ex[i];
    }
    const float Z = warp_sum(part);

    // device-limited mode: devices allowed for this token
    uint32_t allowed = 0xffffffffu;
    if (limited) {
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i) s_ex[warp][lane + 32 * i] = ex[i];
      __syncwarp();
      // lane d sums the (unnormalised) probabilities of its device's experts in
      // ascending expert order; the common 1/Z does not change the ranking
      float m = NEG;
      if (lane < Nd) {
        m = 0.f;
        for (int e = 0; e < Ne; ++e)
          if (s_dev[e] == lane) m += s_ex[warp][e];
      }
      allowed = 0u;
      Cand dc{m, lane};
      for (int r = 0; r < n_keep; ++r) {
        Cand b = warp_best(dc);
        allowed |= 1u << b.id;
        if (lane == b.id) dc.v = NEG, dc.id = 0x7fffffff;
      }
      __syncwarp();
    }

    // top-k by logit among allowed experts
    bool taken[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i)
      taken[i] = (lane + 32 * i >= Ne) || !((allowed >> (dev[i] & 31)) & 1u);
    uint32_t vm = 0;
    float gsum = 0.f;
    int my_id = 0;
    float my_g = 0.f;
    for (int j = 0; j < k; ++j) {
      Cand c{NEG, 0x7fffffff};
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i)
        if (!taken[i] && before(v[i], lane + 32 * i, c.v, c.id)) { c.v = v[i]; c.id = lane + 32 * i; }
      Cand b = warp_best(c);
      const int owner = b.id & 31, slot = b.id >> 5;
      float g = 0.f;
      int d = 0;
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i)
        if (lane == owner && slot == i) { taken[i] = true; g = ex[i]; d = dev[i]; }
      g = __shfl_sync(0xffffffffu, g, owner) / Z;
      d = __shfl_sync(0xffffffffu, d, owner);
      vm |= 1u << d;
      gsum += g;
      if (lane == j) { my_id = b.id; my_g = g; }
    }
    if (renorm) my_g = my_g / gsum;
    if (lane < k) {
      ids[static_cast<size_t>(t) * k + lane] = my_id;
      gates[static_cast<size_t>(t) * k + lane] = my_g;
    }
    if (lane == 0) vmask[t] = vm;
  }
}

}  // namespace

int launch_route(const LaunchCtx& ctx, const occult_desc_t& ds, const float* logits,
                 const int32_t* e2v, int32_t* ids, float* gates, uint32_t* vmask) {
  if (ds.T == 0) return OCCULT_OK;
  const int limited = ds.route_mode == OCCULT_ROUTE_DEVICE_LIMITED;
  int blocks = (ds.T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > ctx.num_sms * 16) blocks = ctx.num_sms * 16;
#define OCCULT_ROUTE_LAUNCH(PL)                                                              \
  route_kernel<PL><<<blocks, kWarpsPerBlock * 32, 0, ctx.stream>>>(                          \
      logits, e2v, ds.T, ds.n_experts, ds.top_k, ds.n_vdev, ds.renorm, limited,              \
      ds.limit_devices, ids, gates, vmask)
  if (ds.n_experts <= 32) OCCULT_ROUTE_LAUNCH(1);
  else if (ds.n_experts <= 64) OCCULT_ROUTE_LAUNCH(2);
  else if (ds.n_experts <= 128) OCCULT_ROUTE_LAUNCH(4);
  else OCCULT_ROUTE_LAUNCH(8);
#undef OCCULT_ROUTE_LAUNCH
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
