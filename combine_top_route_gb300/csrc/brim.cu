// BRIM builder: Occult paper Appendix A.2, Algorithm 3 (BRIM0) and Algorithm 5
// (BRIM1), plus the condensed EPD arrays the grouped GEMMs consume.
//
// Both algorithms are running counters over a flattened order: BRIM0 over
// (device, token) pairs, device-major; BRIM1 on device d over (local expert,
// received SFD row) pairs, expert-major.  Because a device's received rows are
// in token order, the BRIM1 counter of (expert slot s, token t) is
//     exp_off[s] - exp_off[d*n_loc] + #{tokens t' < t choosing expert slot s},
// and the BRIM0 entry of (d, t) is seg_off[d] + #{tokens t' < t using device d}.
// The kernel computes both with warp ballots and prefix popcounts: one CTA of 32
// warps, warp w owning a contiguous token range.  Pass 1 counts every column
// (devices and expert slots) per warp, a scan over warps and columns gives each
// warp its starting counters, and pass 2 writes every entry in token order.
// Everything is integer and deterministic.
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kDevCols = 32;

template <int W64>
__global__ void __launch_bounds__(kThreads, 1)
brim_kernel(const int32_t* __restrict__ ids, const float* __restrict__ gates,
            const uint32_t* __restrict__ vmask, const int32_t* __restrict__ placement, int T,
            int k, int Ne, int Nd, int n_loc, int32_t* __restrict__ brim0,
            int32_t* __restrict__ seg_off, int32_t* __restrict__ brim1,
            int32_t* __restrict__ exp_off, int32_t* __restrict__ epd_src,
            float* __restrict__ epd_gate, int32_t* __restrict__ counts) {
  constexpr int NSLOT = 64 * W64;
  constexpr int NCOL = kDevCols + NSLOT;
  constexpr int NW32 = 2 * W64;
  __shared__ int s_cnt[kWarps][NCOL];
  __shared__ int s_slot_of[NSLOT];
  __shared__ int s_expert[NSLOT];
  __shared__ int s_seg[kDevCols + 1];
  __shared__ int s_exp[NSLOT + 1];
  __shared__ int s_maxct;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int s = threadIdx.x; s < NSLOT; s += kThreads) {
    s_expert[s] = s < Ne ? placement[s] : -1;
  }
  if (threadIdx.x == 0) s_maxct = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < Ne; s += kThreads) s_slot_of[s_expert[s]] = s;
  __syncthreads();

  // contiguous token range of this warp, a whole number of 32-token chunks
  const int per_warp = ((T + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int t_begin = warp * per_warp;
  const int t_end = min(T, t_begin + per_warp);

  // slot mask of one token: bit s set iff the token chose expert s_expert[s]
  auto slot_mask = [&](int t, bool valid, uint64_t* sm) {
#pragma unroll
    for (int w = 0; w < W64; ++w) sm[w] = 0;
    if (valid) {
      for (int j = 0; j < k; ++j) {
        const int s = s_slot_of[ids[static_cast<size_t>(t) * k + j]];
#pragma unroll
        for (int w = 0; w < W64; ++w)
          if ((s >> 6) == w) sm[w] |= 1ull << (s & 63);
      }
    }
  };

  // ---- pass 1: per-warp column counts -------------------------------------
  int dev_acc = 0;              // lane d: tokens of this warp using device d
  int slot_acc[NW32];           // lane b: tokens choosing slot w32*32 + b
#pragma unroll
  for (int i = 0; i < NW32; ++i) slot_acc[i] = 0;
  int maxct = 0;
  for (int c = t_begin; c < t_end; c += 32) {
    const int t = c + lane;
    const bool valid = t < t_end;
    const uint32_t vm = valid ? vmask[t] : 0u;
    maxct = max(maxct, __popc(vm));
    uint64_t sm[W64];
    slot_mask(t, valid, sm);
    for (int d = 0; d < Nd; ++d) {
      const unsigned bal = __ballot_sync(0xffffffffu, (vm >> d) & 1u);
      if (lane == d) dev_acc += __popc(bal);
    }
#pragma unroll
    for (int w32 = 0; w32 < NW32; ++w32) {
      for (int b = 0; b < 32; ++b) {
        if (w32 * 32 + b >= Ne) break;
        const unsigned bit = static_cast<unsigned>(sm[w32 >> 1] >> ((w32 & 1) * 32 + b)) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, bit);
        if (lane == b) slot_acc[w32] += __popc(bal);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) maxct = max(maxct, __shfl_xor_sync(0xffffffffu, maxct, o));
  if (lane == 0) atomicMax(&s_maxct, maxct);
  s_cnt[warp][lane] = dev_acc;
#pragma unroll
  for (int w32 = 0; w32 < NW32; ++w32) s_cnt[warp][kDevCols + w32 * 32 + lane] = slot_acc[w32];
  __syncthreads();

  // ---- exclusive scan over warps, per column -------------------------------
  for (int col = threadIdx.x; col < NCOL; col += kThreads) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int v = s_cnt[w][col];
      s_cnt[w][col] = run;
      run += v;
    }
    // column totals parked in the scan arrays, turned into offsets below
    if (col < kDevCols) s_seg[col + 1] = run;
    else s_exp[col - kDevCols + 1] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    s_seg[0] = 0;
    for (int d = 0; d < Nd; ++d) s_seg[d + 1] += s_seg[d];
    s_exp[0] = 0;
    for (int s = 0; s < Ne; ++s) s_exp[s + 1] += s_exp[s];
    counts[0] = s_seg[Nd];
    counts[1] = s_exp[Ne];
    counts[2] = s_maxct;
    counts[3] = 0;
  }
  __syncthreads();
  for (int d = threadIdx.x; d <= Nd; d += kThreads) seg_off[d] = s_seg[d];
  for (int s = threadIdx.x; s <= Ne; s += kThreads) exp_off[s] = s_exp[s];

  // ---- pass 2: write BRIM0, BRIM1 and the EPD arrays in token order --------
  int dev_run = lane < Nd ? s_seg[lane] + s_cnt[warp][lane] : 0;
  int slot_run[NW32];
#pragma unroll
  for (int w32 = 0; w32 < NW32; ++w32) {
    const int s = w32 * 32 + lane;
    slot_run[w32] = s < Ne ? s_exp[s] + s_cnt[warp][kDevCols + s] : 0;
  }
  for (int c = t_begin; c < t_end; c += 32) {
    const int t = c + lane;
    const bool valid = t < t_end;
    const uint32_t vm = valid ? vmask[t] : 0u;
    uint64_t sm[W64];
    slot_mask(t, valid, sm);
    int my_ids[OCCULT_MAX_TOPK];
    float my_g[OCCULT_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < OCCULT_MAX_TOPK; ++j) {
      my_ids[j] = (valid && j < k) ? ids[static_cast<size_t>(t) * k + j] : -1;
      my_g[j] = (valid && j < k) ? gates[static_cast<size_t>(t) * k + j] : 0.f;
    }
    // BRIM0 (Algorithm 3)
    for (int d = 0; d < Nd; ++d) {
      const unsigned bit = (vm >> d) & 1u;
      const unsigned bal = __ballot_sync(0xffffffffu, bit);
      const int base = __shfl_sync(0xffffffffu, dev_run, d);
      if (valid)
        brim0[static_cast<size_t>(d) * T + t] = bit ? base + __popc(bal & lanemask_lt()) : -1;
      if (lane == d) dev_run += __popc(bal);
    }
    // BRIM1 (Algorithm 5) and the condensed EPD arrays
#pragma unroll
    for (int w32 = 0; w32 < NW32; ++w32) {
      for (int b = 0; b < 32; ++b) {
        const int s = w32 * 32 + b;
        if (s >= Ne) break;
        const unsigned bit = static_cast<unsigned>(sm[w32 >> 1] >> ((w32 & 1) * 32 + b)) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, bit);
        const int base = __shfl_sync(0xffffffffu, slot_run[w32], b);
        const int dv = s / n_loc;
        if (valid && ((vm >> dv) & 1u)) {
          // this thread wrote brim0[dv, t] above; same-thread reads see it
          const int sfd = brim0[static_cast<size_t>(dv) * T + t];
          const int r_local = sfd - s_seg[dv];
          int val = -1;
          if (bit) {
            const int row = base + __popc(bal & lanemask_lt());
            val = row - s_exp[dv * n_loc];
            const int e = s_expert[s];
            float g = 0.f;
#pragma unroll
            for (int j = 0; j < OCCULT_MAX_TOPK; ++j)
              if (my_ids[j] == e) g = my_g[j];
            epd_src[row] = sfd;
            epd_gate[row] = g;
          }
          brim1[static_cast<size_t>(s) * T + r_local] = val;
        }
        if (lane == b) slot_run[w32] += __popc(bal);
      }
    }
  }
}

}  // namespace

int launch_build_brim(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids,
                      const float* gates, const uint32_t* vmask, const int32_t* placement,
                      int32_t* brim0, int32_t* seg_off, int32_t* brim1, int32_t* exp_off,
                      int32_t* epd_src, float* epd_gate, int32_t* counts) {
  const int n_loc = ds.n_experts / ds.n_vdev;
#define OCCULT_BRIM_LAUNCH(W)                                                                 \
  brim_kernel<W><<<1, kThreads, 0, ctx.stream>>>(ids, gates, vmask, placement, ds.T, ds.top_k, \
                                                 ds.n_experts, ds.n_vdev, n_loc, brim0,        \
                                                 seg_off, brim1, exp_off, epd_src, epd_gate,   \
                                                 counts)
  if (ds.n_experts <= 64) OCCULT_BRIM_LAUNCH(1);
  else if (ds.n_experts <= 128) OCCULT_BRIM_LAUNCH(2);
  else OCCULT_BRIM_LAUNCH(4);
#undef OCCULT_BRIM_LAUNCH
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
