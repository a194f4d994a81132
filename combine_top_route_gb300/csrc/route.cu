// Router kernel: Occult paper Sec. 2.1 Eq. 2 (top-k of the softmax of the
// router logits) and the collaboration pruning of Sec. 3.3: the device-limited
// mode (keep the devices of largest gate mass, top-k among their experts) and
// the pages' own two rules, whose kept devices are those of the routed experts
// in descending score -- routing-score-based pruning (top-k of all sorted
// scores within them) and expert-similarity-based pruning (each routed expert
// outside them replaced by its most similar free expert inside, table T of
// App. A.3).
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

// One top-k pass over the experts whose device is in `allowed`: lane j < k
// receives slot j's expert and probability (exp / Z), `vm` the devices used,
// `gsum` the sum of the k probabilities.  With `walk`, the devices of the chosen
// experts are also collected in slot order into `kept` until `n_keep` are found
// (Sec. 3.3's device range).
template <int PER_LANE>
__device__ __forceinline__ void topk_pass(const float (&v)[PER_LANE], const float (&ex)[PER_LANE],
                                          const int (&dev)[PER_LANE], int Ne, int k, float Z,
                                          uint32_t allowed, bool walk, int n_keep, int& my_id,
                                          float& my_g, uint32_t& vm, float& gsum,
                                          uint32_t& kept) {
  const int lane = threadIdx.x & 31;
  const float NEG = -__int_as_float(0x7f800000);
  bool taken[PER_LANE];
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i)
    taken[i] = (lane + 32 * i >= Ne) || !((allowed >> (dev[i] & 31)) & 1u);
  vm = 0;
  gsum = 0.f;
  int n_kept = 0;
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
    if (walk && !((kept >> d) & 1u) && n_kept < n_keep) {
      kept |= 1u << d;
      ++n_kept;
    }
    if (lane == j) { my_id = b.id; my_g = g; }
  }
}

// mode: 0 top-k, 1 device-limited (gate mass), 2 routing-score-based pruning,
// 3 expert-similarity-based pruning with `table` [Ne, Ne]
template <int PER_LANE>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_kernel(const float* __restrict__ logits, const int32_t* __restrict__ e2v,
             const float* __restrict__ table, int T, int Ne, int k, int Nd, int renorm, int mode,
             int n_keep, int32_t* __restrict__ ids, float* __restrict__ gates,
             int32_t* __restrict__ routed, uint32_t* __restrict__ vmask) {
  __shared__ float s_ex[kWarpsPerBlock][PER_LANE * 32];
  __shared__ int s_dev[PER_LANE * 32];
  pdl_wait();
  pdl_trigger();
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
    if (mode == 1) {
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

    // top-k by logit among the allowed experts; for the pages' pruning rules this
    // is the routed set, whose devices (in descending score) give the kept range
    uint32_t vm = 0, kept = 0;
    float gsum = 0.f;
    int my_id = 0;
    float my_g = 0.f;
    topk_pass<PER_LANE>(v, ex, dev, Ne, k, Z, allowed, mode >= 2, n_keep, my_id, my_g, vm, gsum,
                        kept);
    if (mode == 3 && routed && lane < k) routed[static_cast<size_t>(t) * k + lane] = my_id;
    if (mode == 2) {
      // routing-score-based pruning: the top k of all sorted scores that lie on
      // the kept devices
      topk_pass<PER_LANE>(v, ex, dev, Ne, k, Z, kept, false, 0, my_id, my_g, vm, gsum, kept);
    } else if (mode == 3) {
      // expert-similarity-based pruning: routed experts on the kept devices stay
      // (and count as selected); each other slot, in descending score, takes the
      // most similar free expert of the kept devices and keeps its routing weight
      uint32_t sel = 0;  // bit i: expert lane + 32 i selected
      for (int j = 0; j < k; ++j) {
        const int rid = __shfl_sync(0xffffffffu, my_id, j);
        if ((kept >> s_dev[rid]) & 1u)
#pragma unroll
          for (int i = 0; i < PER_LANE; ++i)
            if (lane + 32 * i == rid) sel |= 1u << i;
      }
      for (int j = 0; j < k; ++j) {
        const int rid = __shfl_sync(0xffffffffu, my_id, j);
        if ((kept >> s_dev[rid]) & 1u) continue;
        const float* trow = table + static_cast<size_t>(rid) * Ne;
        Cand c{NEG, 0x7fffffff};
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
          const int e = lane + 32 * i;
          if (e < Ne && ((kept >> (dev[i] & 31)) & 1u) && !((sel >> i) & 1u)) {
            float s = trow[e];
            if (s != s) s = NEG;  // a NaN entry ranks last
            if (before(s, e, c.v, c.id)) { c.v = s; c.id = e; }
          }
        }
        const Cand b = warp_best(c);
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i)
          if (lane + 32 * i == b.id) sel |= 1u << i;
        if (lane == j) my_id = b.id;
      }
      // devices of the final experts
      const int my_dev = lane < k ? s_dev[my_id] : 0;
      vm = __reduce_or_sync(0xffffffffu, lane < k ? 1u << my_dev : 0u);
    }
    if (renorm) my_g = my_g / gsum;
    if (lane < k) {
      ids[static_cast<size_t>(t) * k + lane] = my_id;
      gates[static_cast<size_t>(t) * k + lane] = my_g;
    }
    if (lane == 0) vmask[t] = vm;
  }
}

// ---- plain top-k for up to 64 experts and k <= 8: eight lanes per token --------
// Lane s of a token's eight holds experts 8s .. 8s+7 and sorts them (a 19-step
// network on (logit, id) with the same order as above); three exchange rounds
// with the lanes 1, 2 and 4 apart each keep the best eight of two sorted lists
// (elementwise best of one list and the other reversed, then a bitonic clean), so
// every lane ends with the token's top eight in order.  Four tokens per warp.
__device__ __forceinline__ void cas8(float* v, int* id, int a, int b) {
  if (before(v[b], id[b], v[a], id[a])) {
    const float tv = v[a]; v[a] = v[b]; v[b] = tv;
    const int ti = id[a]; id[a] = id[b]; id[b] = ti;
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_top8_kernel(const float* __restrict__ logits, const int32_t* __restrict__ e2v, int T,
                  int Ne, int k, int renorm, int32_t* __restrict__ ids, float* __restrict__ gates,
                  uint32_t* __restrict__ vmask) {
  __shared__ int s_dev[64];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < 64; e += blockDim.x) s_dev[e] = e < Ne ? e2v[e] : 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const float NEG = -__int_as_float(0x7f800000);  // -inf
  for (int base = (blockIdx.x * kWarpsPerBlock + warp) * 4; base < T;
       base += gridDim.x * kWarpsPerBlock * 4) {
    const int t = base + (lane >> 3);
    const bool valid = t < T;
    const float* row = logits + static_cast<size_t>(valid ? t : 0) * Ne;
    float v[8];
    int id[8];
    float mx = NEG;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      id[i] = sub * 8 + i;
      v[i] = (valid && id[i] < Ne) ? row[id[i]] : NEG;
      mx = fmaxf(mx, v[i]);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) part += (valid && id[i] < Ne) ? expf(v[i] - mx) : 0.f;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    const float Z = part;
    // sort the lane's eight, best first
    cas8(v, id, 0, 1); cas8(v, id, 2, 3); cas8(v, id, 4, 5); cas8(v, id, 6, 7);
    cas8(v, id, 0, 2); cas8(v, id, 1, 3); cas8(v, id, 4, 6); cas8(v, id, 5, 7);
    cas8(v, id, 1, 2); cas8(v, id, 5, 6); cas8(v, id, 0, 4); cas8(v, id, 3, 7);
    cas8(v, id, 1, 5); cas8(v, id, 2, 6); cas8(v, id, 1, 4); cas8(v, id, 3, 6);
    cas8(v, id, 2, 4); cas8(v, id, 3, 5); cas8(v, id, 3, 4);
    // merge with the lanes 1, 2, 4 apart: best eight of the two lists
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      float pv[8];
      int pid[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        pv[i] = __shfl_xor_sync(0xffffffffu, v[7 - i], o);
        pid[i] = __shfl_xor_sync(0xffffffffu, id[7 - i], o);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (before(pv[i], pid[i], v[i], id[i])) { v[i] = pv[i]; id[i] = pid[i]; }
#pragma unroll
      for (int dd = 4; dd > 0; dd >>= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if ((i & dd) == 0) cas8(v, id, i, i + dd);
    }
    // every lane holds the token's top eight; lane j < k writes slot j
    uint32_t vm = 0;
    float gsum = 0.f, my_g = 0.f;
    int my_id = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        const float g = expf(v[j] - mx) / Z;
        vm |= 1u << s_dev[id[j]];
        gsum += g;
        if (j == sub) { my_g = g; my_id = id[j]; }
      }
    }
    if (renorm) my_g = my_g / gsum;
    if (valid && sub < k) {
      ids[static_cast<size_t>(t) * k + sub] = my_id;
      gates[static_cast<size_t>(t) * k + sub] = my_g;
    }
    if (valid && sub == 0) vmask[t] = vm;
  }
}

}  // namespace

int launch_route(const LaunchCtx& ctx, const occult_desc_t& ds, const float* logits,
                 const int32_t* e2v, const float* table, int32_t* ids, float* gates,
                 int32_t* routed, uint32_t* vmask) {
  if (ds.T == 0) return OCCULT_OK;
  if (ds.route_mode == OCCULT_ROUTE_EXACT && ds.n_experts <= 64 && ds.top_k <= 8) {
    int blocks = (ds.T + 4 * kWarpsPerBlock - 1) / (4 * kWarpsPerBlock);
    if (blocks > ctx.num_sms * 16) blocks = ctx.num_sms * 16;
    return cuda_status(launch_pdl(route_top8_kernel, blocks, kWarpsPerBlock * 32, 0, ctx.stream,
                                  logits, e2v, ds.T, ds.n_experts, ds.top_k, ds.renorm, ids,
                                  gates, vmask));
  }
  int blocks = (ds.T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > ctx.num_sms * 16) blocks = ctx.num_sms * 16;
#define OCCULT_ROUTE_LAUNCH(PL)                                                              \
  launch_pdl(route_kernel<PL>, blocks, kWarpsPerBlock * 32, 0, ctx.stream, logits, e2v, table,   \
             ds.T, ds.n_experts, ds.top_k, ds.n_vdev, ds.renorm, ds.route_mode,                  \
             ds.limit_devices, ids, gates, routed, vmask)
  if (ds.n_experts <= 32) OCCULT_ROUTE_LAUNCH(1);
  else if (ds.n_experts <= 64) OCCULT_ROUTE_LAUNCH(2);
  else if (ds.n_experts <= 128) OCCULT_ROUTE_LAUNCH(4);
  else OCCULT_ROUTE_LAUNCH(8);
#undef OCCULT_ROUTE_LAUNCH
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
