// BRIM builder: Occult paper Appendix A.2, Algorithm 3 (BRIM0) and Algorithm 5
// (BRIM1), plus the condensed EPD arrays the grouped GEMMs consume.
//
// Both algorithms are running counters over a flattened order: BRIM0 over
// (device, token) pairs, device-major; BRIM1 on device d over (local expert,
// received SFD row) pairs, expert-major.  Because a device's received rows are
// in token order, the BRIM1 counter of (expert slot s, token t) is
//     exp_off[s] - exp_off[d*n_loc] + #{tokens t' < t choosing expert slot s},
// and the BRIM0 entry of (d, t) is seg_off[d] + #{tokens t' < t using device d}.
// So both are exclusive prefix counts over tokens, one column per device and one
// per expert slot, computed with warp ballots and popcounts:
//   1. count  -- every CTA counts its 64-token tile per column;
//   2. scan   -- one CTA (a warp scan per column) turns the tile counts into per-tile
//                column offsets, and
//                the column totals into seg_off / exp_off;
//   3. fill   -- every CTA re-counts per warp, adds the warp prefix to its tile
//                offsets and writes BRIM0, BRIM1, epd_src and epd_gate.
// Integer and deterministic; the workspace holds the [tiles, columns] counts.
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

constexpr int kWarps = 2;
constexpr int kTile = kWarps * 32;  // tokens per CTA (small tiles: many CTAs in flight)
constexpr int kDevCols = 32;        // device columns (padded to the ballot width)

__host__ __device__ constexpr int ncols(int Ne) { return kDevCols + Ne + 1; }  // + max C_T

// bit s of a W64-word mask held in registers (unrolled select, no local memory)
template <int W64>
__device__ __forceinline__ unsigned mask_bit(const uint64_t* m, int s) {
  uint64_t w = m[0];
#pragma unroll
  for (int i = 1; i < W64; ++i)
    if ((s >> 6) == i) w = m[i];
  return static_cast<unsigned>(w >> (s & 63)) & 1u;
}

template <int W64>
__device__ __forceinline__ void slot_mask(const int32_t* __restrict__ ids, int t, int k, bool valid,
                                          const int* s_slot_of, uint64_t* m) {
#pragma unroll
  for (int i = 0; i < W64; ++i) m[i] = 0;
  if (!valid) return;
  for (int j = 0; j < k; ++j) {
    const int s = s_slot_of[ids[static_cast<size_t>(t) * k + j]];
#pragma unroll
    for (int i = 0; i < W64; ++i)
      if ((s >> 6) == i) m[i] |= 1ull << (s & 63);
  }
}

// Per-warp column counts of one 32-token chunk into s_wcnt[warp][col].
template <int W64>
__device__ __forceinline__ void warp_counts(const int32_t* __restrict__ ids,
                                           const uint32_t* __restrict__ vmask, int T, int k,
                                           int Ne, int Nd, const int* s_slot_of, int t0,
                                           int* wcnt, uint64_t* m, uint32_t* vm_out) {
  const int lane = threadIdx.x & 31;
  const int t = t0 + lane;
  const bool valid = t < T;
  const uint32_t vm = valid ? vmask[t] : 0u;
  slot_mask<W64>(ids, t, k, valid, s_slot_of, m);
  for (int d = lane; d < kDevCols; d += 32) wcnt[d] = 0;
  for (int d = 0; d < Nd; ++d) {
    const unsigned bal = __ballot_sync(0xffffffffu, (vm >> d) & 1u);
    if (lane == 0) wcnt[d] = __popc(bal);
  }
  for (int s = 0; s < Ne; ++s) {
    const unsigned bal = __ballot_sync(0xffffffffu, mask_bit<W64>(m, s));
    if (lane == 0) wcnt[kDevCols + s] = __popc(bal);
  }
  int ct = __popc(vm);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ct = max(ct, __shfl_xor_sync(0xffffffffu, ct, o));
  if (lane == 0) wcnt[kDevCols + Ne] = ct;
  *vm_out = vm;
}

template <int W64>
__global__ void __launch_bounds__(kTile)
brim_count_kernel(const int32_t* __restrict__ ids, const uint32_t* __restrict__ vmask,
                  const int32_t* __restrict__ placement, int T, int k, int Ne, int Nd,
                  int32_t* __restrict__ tile_cnt) {
  constexpr int NS = 64 * W64;
  __shared__ int s_slot_of[NS];
  __shared__ int s_wcnt[kWarps][kDevCols + NS + 1];
  const int warp = threadIdx.x >> 5;
  for (int s = threadIdx.x; s < Ne; s += kTile) s_slot_of[placement[s]] = s;
  __syncthreads();
  uint64_t m[W64];
  uint32_t vm;
  warp_counts<W64>(ids, vmask, T, k, Ne, Nd, s_slot_of, blockIdx.x * kTile + warp * 32,
                   s_wcnt[warp], m, &vm);
  __syncthreads();
  const int nc = ncols(Ne);
  for (int c = threadIdx.x; c < nc; c += kTile) {
    int v = 0;
    if (c == nc - 1) {
      for (int w = 0; w < kWarps; ++w) v = max(v, s_wcnt[w][c]);
    } else {
      for (int w = 0; w < kWarps; ++w) v += s_wcnt[w][c];
    }
    tile_cnt[static_cast<size_t>(blockIdx.x) * nc + c] = v;
  }
}

// One CTA: exclusive scan of every column over tiles (one warp per column, 32
// tiles per step), then the offsets.
__global__ void __launch_bounds__(1024)
brim_scan_kernel(int n_tiles, int Ne, int Nd, int32_t* __restrict__ tile_cnt,
                 int32_t* __restrict__ seg_off, int32_t* __restrict__ exp_off,
                 int32_t* __restrict__ counts) {
  __shared__ int s_tot[kDevCols + OCCULT_MAX_EXPERTS + 1];
  __shared__ int s_off[kDevCols + OCCULT_MAX_EXPERTS + 1];
  const int nc = ncols(Ne);
  const int lane = threadIdx.x & 31;
  for (int c = threadIdx.x >> 5; c < nc; c += blockDim.x >> 5) {
    int run = 0;
    for (int b0 = 0; b0 < n_tiles; b0 += 32) {
      const int b = b0 + lane;
      int32_t* pcell = tile_cnt + static_cast<size_t>(b) * nc + c;
      const int v = b < n_tiles ? *pcell : 0;
      if (c == nc - 1) {
        int m = v;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        run = max(run, m);
      } else {
        int inc = v;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, inc, sh);
          if (lane >= sh) inc += u;
        }
        if (b < n_tiles) *pcell = run + inc - v;
        run += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
    if (lane == 0) s_tot[c] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int a = 0;
    for (int d = 0; d < Nd; ++d) s_off[d] = a, a += s_tot[d];
    s_off[Nd] = a;
    counts[0] = a;
    int e = 0;
    for (int s = 0; s < Ne; ++s) s_off[kDevCols + s] = e, e += s_tot[kDevCols + s];
    s_off[kDevCols + Ne] = e;
    counts[1] = e;
    counts[2] = s_tot[nc - 1];
    counts[3] = 0;
  }
  __syncthreads();
  for (int d = threadIdx.x; d <= Nd; d += blockDim.x) seg_off[d] = s_off[d];
  for (int s = threadIdx.x; s <= Ne; s += blockDim.x) exp_off[s] = s_off[kDevCols + s];
  // tile offsets become absolute: tile prefix + column offset
  for (int i = threadIdx.x; i < n_tiles * nc; i += blockDim.x) {
    const int c = i % nc;
    if (c < Nd) tile_cnt[i] += s_off[c];
    else if (c >= kDevCols && c < kDevCols + Ne) tile_cnt[i] += s_off[c];
  }
}

template <int W64>
__global__ void __launch_bounds__(kTile)
brim_fill_kernel(const int32_t* __restrict__ ids, const float* __restrict__ gates,
                 const uint32_t* __restrict__ vmask, const int32_t* __restrict__ placement,
                 int T, int k, int Ne, int Nd, int n_loc, const int32_t* __restrict__ tile_off,
                 const int32_t* __restrict__ seg_off, const int32_t* __restrict__ exp_off,
                 int32_t* __restrict__ brim0, int32_t* __restrict__ brim1,
                 int32_t* __restrict__ epd_src, float* __restrict__ epd_gate) {
  constexpr int NS = 64 * W64;
  __shared__ int s_slot_of[NS];
  __shared__ int s_expert[NS];
  __shared__ int s_wcnt[kWarps][kDevCols + NS + 1];
  __shared__ int s_seg[kDevCols + 1];
  __shared__ int s_ebase[kDevCols];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nc = ncols(Ne);
  for (int s = threadIdx.x; s < Ne; s += kTile) {
    s_slot_of[placement[s]] = s;
    s_expert[s] = placement[s];
  }
  for (int d = threadIdx.x; d <= Nd; d += kTile) s_seg[d] = seg_off[d];
  for (int d = threadIdx.x; d < Nd; d += kTile) s_ebase[d] = exp_off[d * n_loc];
  __syncthreads();
  uint64_t m[W64];
  uint32_t vm;
  const int t0 = blockIdx.x * kTile + warp * 32;
  warp_counts<W64>(ids, vmask, T, k, Ne, Nd, s_slot_of, t0, s_wcnt[warp], m, &vm);
  __syncthreads();
  // exclusive prefix over the warps of this tile, plus the tile's offsets
  const int32_t* toff = tile_off + static_cast<size_t>(blockIdx.x) * nc;
  for (int c = threadIdx.x; c < nc - 1; c += kTile) {
    int run = (c < Nd || (c >= kDevCols && c < kDevCols + Ne)) ? toff[c] : 0;
    for (int w = 0; w < kWarps; ++w) {
      const int v = s_wcnt[w][c];
      s_wcnt[w][c] = run;
      run += v;
    }
  }
  __syncthreads();
  const int t = t0 + lane;
  const bool valid = t < T;
  if (t0 >= T) return;
  int my_ids[OCCULT_MAX_TOPK];
  float my_g[OCCULT_MAX_TOPK];
#pragma unroll
  for (int j = 0; j < OCCULT_MAX_TOPK; ++j) {
    my_ids[j] = (valid && j < k) ? ids[static_cast<size_t>(t) * k + j] : -1;
    my_g[j] = (valid && j < k) ? gates[static_cast<size_t>(t) * k + j] : 0.f;
  }
  const int* wb = s_wcnt[warp];
  const unsigned lt = lanemask_lt();
  for (int d = 0; d < Nd; ++d) {
    // BRIM0 (Algorithm 3)
    const unsigned bit = (vm >> d) & 1u;
    const unsigned bal = __ballot_sync(0xffffffffu, bit);
    const int sfd = bit ? wb[d] + __popc(bal & lt) : -1;
    if (valid) brim0[static_cast<size_t>(d) * T + t] = sfd;
    if (bal == 0) continue;
    // BRIM1 (Algorithm 5) of device d and the condensed EPD arrays
    const int r_local = sfd - s_seg[d];
    const int ebase = s_ebase[d];
    for (int j = 0; j < n_loc; ++j) {
      const int s = d * n_loc + j;
      const unsigned sbit = mask_bit<W64>(m, s);
      const unsigned sbal = __ballot_sync(0xffffffffu, sbit);
      if (bit) {
        int val = -1;
        if (sbit) {
          const int row = wb[kDevCols + s] + __popc(sbal & lt);
          val = row - ebase;
          const int e = s_expert[s];
          float g = 0.f;
#pragma unroll
          for (int q = 0; q < OCCULT_MAX_TOPK; ++q)
            if (my_ids[q] == e) g = my_g[q];
          epd_src[row] = sfd;
          epd_gate[row] = g;
        }
        brim1[static_cast<size_t>(s) * T + r_local] = val;
      }
    }
  }
}

}  // namespace

size_t brim_ws_bytes(const occult_desc_t& ds) {
  const size_t tiles = (static_cast<size_t>(ds.T) + kTile - 1) / kTile;
  return tiles * ncols(ds.n_experts) * sizeof(int32_t);
}

int launch_build_brim(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids,
                      const float* gates, const uint32_t* vmask, const int32_t* placement,
                      int32_t* brim0, int32_t* seg_off, int32_t* brim1, int32_t* exp_off,
                      int32_t* epd_src, float* epd_gate, int32_t* counts, void* ws) {
  const int n_loc = ds.n_experts / ds.n_vdev;
  const int tiles = (ds.T + kTile - 1) / kTile;
  int32_t* tile_cnt = static_cast<int32_t*>(ws);
  const int T = ds.T, k = ds.top_k, Ne = ds.n_experts, Nd = ds.n_vdev;
#define OCCULT_BRIM_COUNT(W)                                                                   \
  brim_count_kernel<W><<<tiles, kTile, 0, ctx.stream>>>(ids, vmask, placement, T, k, Ne, Nd,    \
                                                        tile_cnt)
#define OCCULT_BRIM_FILL(W)                                                                    \
  brim_fill_kernel<W><<<tiles, kTile, 0, ctx.stream>>>(ids, gates, vmask, placement, T, k, Ne,  \
                                                       Nd, n_loc, tile_cnt, seg_off, exp_off,   \
                                                       brim0, brim1, epd_src, epd_gate)
  if (tiles > 0) {
    if (Ne <= 64) OCCULT_BRIM_COUNT(1);
    else if (Ne <= 128) OCCULT_BRIM_COUNT(2);
    else OCCULT_BRIM_COUNT(4);
  }
  brim_scan_kernel<<<1, 1024, 0, ctx.stream>>>(tiles, Ne, Nd, tile_cnt, seg_off, exp_off, counts);
  if (tiles > 0) {
    if (Ne <= 64) OCCULT_BRIM_FILL(1);
    else if (Ne <= 128) OCCULT_BRIM_FILL(2);
    else OCCULT_BRIM_FILL(4);
  }
#undef OCCULT_BRIM_COUNT
#undef OCCULT_BRIM_FILL
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
