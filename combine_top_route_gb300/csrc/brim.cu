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
//   1. count  -- one warp per 32-token tile counts the tile per column;
//   2. scan   -- one warp per column turns the tile counts into inclusive prefixes
//                over tiles (in place; the last tile's is the column total);
//   3. fill   -- every CTA derives seg_off / exp_off from the column totals, re-counts
//                per warp (the ballots give each tile's own count, so its exclusive
//                offset is the inclusive prefix minus that count) and writes BRIM0,
//                BRIM1, epd_src and epd_gate; CTA 0 also writes seg_off, exp_off and
//                the counts.
// Integer and deterministic; the workspace holds the [tiles, columns] counts.
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

constexpr int kTile = 32;           // tokens per tile: one warp
constexpr int kWarpsPerCta = 4;
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

// slot mask of token t: bit s set iff the token chose the expert in slot s
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

// 1. count: one warp per 32-token tile writes its column counts, column-major
//    (cnt[c * n_tiles + tile]); the last column holds the tile's max C_T.
template <int W64>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
brim_count_kernel(const int32_t* __restrict__ ids, const uint32_t* __restrict__ vmask,
                  const int32_t* __restrict__ placement, int T, int k, int Ne, int Nd,
                  int n_tiles, int32_t* __restrict__ cnt) {
  constexpr int NS = 64 * W64;
  __shared__ int s_slot_of[NS];
  pdl_wait();
  pdl_trigger();
  for (int s = threadIdx.x; s < Ne; s += blockDim.x) s_slot_of[placement[s]] = s;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int tile = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (tile >= n_tiles) return;
  const int t = tile * kTile + lane;
  const bool valid = t < T;
  const uint32_t vm = valid ? vmask[t] : 0u;
  uint64_t m[W64];
  slot_mask<W64>(ids, t, k, valid, s_slot_of, m);
  for (int d = 0; d < kDevCols; ++d) {
    const unsigned bal = __ballot_sync(0xffffffffu, d < Nd && ((vm >> d) & 1u));
    if (lane == 0) cnt[static_cast<size_t>(d) * n_tiles + tile] = __popc(bal);
  }
  for (int s = 0; s < Ne; ++s) {
    const unsigned bal = __ballot_sync(0xffffffffu, mask_bit<W64>(m, s));
    if (lane == 0) cnt[static_cast<size_t>(kDevCols + s) * n_tiles + tile] = __popc(bal);
  }
  int ct = __popc(vm);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ct = max(ct, __shfl_xor_sync(0xffffffffu, ct, o));
  if (lane == 0) cnt[static_cast<size_t>(kDevCols + Ne) * n_tiles + tile] = ct;
}

// 2. scan: one warp per column: inclusive prefix over tiles, eight 32-tile chunks
//    loaded at a time so that their loads overlap; the last column (the tiles'
//    max C_T) is reduced to its maximum, left in its last tile's entry.
constexpr int kScanWarps = 4;
__global__ void __launch_bounds__(kScanWarps * 32)
brim_scan_kernel(int n_tiles, int Ne, int32_t* __restrict__ cnt) {
  const int nc = ncols(Ne);
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (c >= nc) return;
  int32_t* col = cnt + static_cast<size_t>(c) * n_tiles;
  const bool is_max = c == nc - 1;
  int run = 0;
  for (int b0 = 0; b0 < n_tiles; b0 += 8 * 32) {
    int v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int b = b0 + 32 * u + lane;
      v[u] = b < n_tiles ? col[b] : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int b = b0 + 32 * u + lane;
      if (is_max) {
        int m = v[u];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        run = max(run, m);
      } else {
        int inc = v[u];
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
          const int w = __shfl_up_sync(0xffffffffu, inc, sh);
          if (lane >= sh) inc += w;
        }
        if (b < n_tiles) col[b] = run + inc;
        run += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
  }
  if (is_max && lane == 0) col[n_tiles - 1] = run;
}

// Exclusive prefix of the column totals (the inclusive prefixes' last entries):
// out[i] = sum of the totals of columns first .. first+i-1 for i <= n (n <= 256).
// Every thread of the CTA must call it.
__device__ void column_offsets(const int32_t* __restrict__ cnt, int n_tiles, int first, int n,
                               int* out) {
  __shared__ int s_part[kWarpsPerCta];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int run = 0;  // each warp scans 64 consecutive columns, 32 at a time
  for (int h = 0; h < 2; ++h) {
    const int i = warp * 64 + h * 32 + lane;
    const int v = i < n ? cnt[static_cast<size_t>(first + i) * n_tiles + n_tiles - 1] : 0;
    int inc = v;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
      const int w = __shfl_up_sync(0xffffffffu, inc, sh);
      if (lane >= sh) inc += w;
    }
    if (i < n) out[i] = run + inc - v;
    run += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) s_part[warp] = run;
  __syncthreads();
  int base = 0, tot = 0;
  for (int w = 0; w < kWarpsPerCta; ++w) {
    if (w < warp) base += s_part[w];
    tot += s_part[w];
  }
  for (int h = 0; h < 2; ++h) {
    const int i = warp * 64 + h * 32 + lane;
    if (i < n) out[i] += base;
  }
  if (threadIdx.x == 0) out[n] = tot;
  __syncthreads();
}

// 3. fill: one warp per (tile, device): BRIM0 of device d for the tile's tokens,
//    then BRIM1 and the EPD arrays of d's expert slots.  Offsets are the tile's
//    exclusive prefix plus the column offset (seg_off / exp_off).
template <int W64>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
brim_fill_kernel(const int32_t* __restrict__ ids, const float* __restrict__ gates,
                 const uint32_t* __restrict__ vmask, const int32_t* __restrict__ placement,
                 int T, int k, int Ne, int Nd, int n_loc, int n_tiles,
                 const int32_t* __restrict__ pre, int32_t* __restrict__ seg_off,
                 int32_t* __restrict__ exp_off, int32_t* __restrict__ counts,
                 int32_t* __restrict__ brim0, int32_t* __restrict__ brim1,
                 int32_t* __restrict__ epd_src, float* __restrict__ epd_gate) {
  constexpr int NS = 64 * W64;
  __shared__ int s_slot_of[NS];
  __shared__ int s_expert[NS];
  __shared__ int s_seg[OCCULT_MAX_VDEV + 1];
  __shared__ int s_exp[OCCULT_MAX_EXPERTS + 1];
  pdl_wait();
  pdl_trigger();
  for (int s = threadIdx.x; s < Ne; s += blockDim.x) {
    s_slot_of[placement[s]] = s;
    s_expert[s] = placement[s];
  }
  // segment offsets of the devices and of the expert slots from the column totals
  column_offsets(pre, n_tiles, 0, Nd, s_seg);
  column_offsets(pre, n_tiles, kDevCols, Ne, s_exp);
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= Nd; i += blockDim.x) seg_off[i] = s_seg[i];
    for (int i = threadIdx.x; i <= Ne; i += blockDim.x) exp_off[i] = s_exp[i];
    if (threadIdx.x == 0) {
      counts[0] = s_seg[Nd];
      counts[1] = s_exp[Ne];
      counts[2] = pre[static_cast<size_t>(kDevCols + Ne) * n_tiles + n_tiles - 1];
      counts[3] = 0;
    }
  }
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (w >= n_tiles * Nd) return;
  const int tile = w / Nd, d = w - tile * Nd;
  const int t = tile * kTile + lane;
  const bool valid = t < T;
  const unsigned lt = lanemask_lt();
  // BRIM0 (Algorithm 3)
  const uint32_t vm = valid ? vmask[t] : 0u;
  const unsigned bit = (vm >> d) & 1u;
  const unsigned bal = __ballot_sync(0xffffffffu, bit);
  // the tile's exclusive offset: its inclusive prefix less its own count
  const int dbase = pre[static_cast<size_t>(d) * n_tiles + tile] - __popc(bal) + s_seg[d];
  const int sfd = bit ? dbase + __popc(bal & lt) : -1;
  if (valid) brim0[static_cast<size_t>(d) * T + t] = sfd;
  if (bal == 0) return;
  // BRIM1 (Algorithm 5) of device d and the condensed EPD arrays
  uint64_t m[W64];
  slot_mask<W64>(ids, t, k, valid, s_slot_of, m);
  int my_ids[OCCULT_MAX_TOPK];
  float my_g[OCCULT_MAX_TOPK];
#pragma unroll
  for (int j = 0; j < OCCULT_MAX_TOPK; ++j) {
    my_ids[j] = (bit && j < k) ? ids[static_cast<size_t>(t) * k + j] : -1;
    my_g[j] = (bit && j < k) ? gates[static_cast<size_t>(t) * k + j] : 0.f;
  }
  const int r_local = sfd - s_seg[d];
  const int ebase = s_exp[d * n_loc];
  for (int j0 = 0; j0 < n_loc; j0 += 32) {
    // lane i holds the row base of slot d*n_loc + j0 + i
    const int sl = d * n_loc + j0 + lane;
    const int sbase_l = (j0 + lane < n_loc)
        ? pre[static_cast<size_t>(kDevCols + sl) * n_tiles + tile] + s_exp[sl] : 0;
    const int jn = min(32, n_loc - j0);
    for (int j = 0; j < jn; ++j) {
      const int s = d * n_loc + j0 + j;
      const unsigned sbit = mask_bit<W64>(m, s);
      const unsigned sbal = __ballot_sync(0xffffffffu, sbit);
      const int sbase = __shfl_sync(0xffffffffu, sbase_l, j) - __popc(sbal);
      if (bit) {
        int val = -1;
        if (sbit) {
          const int row = sbase + __popc(sbal & lt);
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
  int32_t* cnt = static_cast<int32_t*>(ws);
  const int T = ds.T, k = ds.top_k, Ne = ds.n_experts, Nd = ds.n_vdev;
  const int cgrid = (tiles + kWarpsPerCta - 1) / kWarpsPerCta;
  const int fgrid = (tiles * Nd + kWarpsPerCta - 1) / kWarpsPerCta;
#define OCCULT_BRIM_COUNT(W)                                                                   \
  launch_pdl(brim_count_kernel<W>, cgrid, kWarpsPerCta * 32, 0, ctx.stream, ids, vmask,         \
             placement, T, k, Ne, Nd, tiles, cnt)
#define OCCULT_BRIM_FILL(W)                                                                    \
  launch_pdl(brim_fill_kernel<W>, fgrid, kWarpsPerCta * 32, 0, ctx.stream, ids, gates, vmask,  \
             placement, T, k, Ne, Nd, n_loc, tiles, cnt, seg_off, exp_off, counts, brim0,      \
             brim1, epd_src, epd_gate)
  if (tiles == 0) {
    // no tokens: every offset and count is zero
    if (cudaMemsetAsync(seg_off, 0, (Nd + 1) * sizeof(int32_t), ctx.stream) != cudaSuccess ||
        cudaMemsetAsync(exp_off, 0, (Ne + 1) * sizeof(int32_t), ctx.stream) != cudaSuccess ||
        cudaMemsetAsync(counts, 0, 4 * sizeof(int32_t), ctx.stream) != cudaSuccess)
      return OCCULT_ERR_CUDA;
    return OCCULT_OK;
  }
  if (Ne <= 64) OCCULT_BRIM_COUNT(1);
  else if (Ne <= 128) OCCULT_BRIM_COUNT(2);
  else OCCULT_BRIM_COUNT(4);
  launch_pdl(brim_scan_kernel, (ncols(Ne) + kScanWarps - 1) / kScanWarps, kScanWarps * 32, 0,
             ctx.stream, tiles, Ne, cnt);
  if (Ne <= 64) OCCULT_BRIM_FILL(1);
  else if (Ne <= 128) OCCULT_BRIM_FILL(2);
  else OCCULT_BRIM_FILL(4);
#undef OCCULT_BRIM_COUNT
#undef OCCULT_BRIM_FILL
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
