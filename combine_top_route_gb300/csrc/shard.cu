// Sharded-source expert parallelism: the first all-to-all as a real exchange of
// row blocks between source shards and virtual devices.
//
// Occult paper, App. A.1 Algorithm 2 runs on every device of the expert-
// parallel group: each source device builds BRIM0 over its own tokens
// (Algorithm 3), dispatches them into its SFD tensor (Algorithm 4) and sends
// segment d to device d with all_to_all_single, whose split sizes are the
// non-zero counts of BRIM0 row d (the text after Algorithm 4).  Here the T
// tokens of one batch are split into contiguous shards [src_off[s],
// src_off[s+1]) standing for the source devices.
//
// * plan   -- counts[s, d] = tokens of shard s using device d; the send layout
//             lays the sources' SFD tensors end to end (source-major, then
//             device, then token), the receive layout is device-major, then
//             source, then token -- for contiguous shards exactly the layout of
//             the single-source BRIM0 of occult_build_brim.  So a token's send
//             row is its receive row moved from its block's receive offset to
//             its block's send offset:
//                 brim0_send[d, t] = brim0[d, t] - recv_off[s, d] + send_off[s, d],
//             which is Algorithm 3 over shard s's tokens placed after shards
//             0..s-1 (a per-shard exclusive prefix count, offset by the rows of
//             earlier shards).
// * all_to_all -- row blocks copied between the two layouts (either way), one
//             warp per destination row in 16-byte vectors.
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

constexpr int kCountThreads = 256;
constexpr int kMapThreads = 256;
constexpr int kA2aWarps = 8;
constexpr int kMaxBlocks = OCCULT_MAX_SOURCES * OCCULT_MAX_VDEV;

// 1. counts: one CTA per shard; each warp ballots 32 tokens per device and the
//    warps' counts are summed in shared memory.
__global__ void __launch_bounds__(kCountThreads)
shard_count_kernel(const uint32_t* __restrict__ vmask, ShardSplit split, int Nd,
                   int32_t* __restrict__ counts) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_cnt[kCountThreads / 32][OCCULT_MAX_VDEV];
  const int s = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int a = split.off[s], b = split.off[s + 1];
  int my = 0;  // lane d counts device d
  for (int t0 = a + warp * 32; t0 < b; t0 += kCountThreads) {
    const int t = t0 + lane;
    const uint32_t vm = t < b ? vmask[t] : 0u;
    for (int d = 0; d < Nd; ++d) {
      const int c = __popc(__ballot_sync(0xffffffffu, (vm >> d) & 1u));
      if (lane == d) my += c;
    }
  }
  s_cnt[warp][lane] = my;
  __syncthreads();
  if (threadIdx.x < Nd) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kCountThreads / 32; ++w) c += s_cnt[w][threadIdx.x];
    counts[s * Nd + threadIdx.x] = c;
  }
}

// Block offsets of both layouts from the counts, in shared memory:
//   send_off[s, d] = sum over blocks (s', d') before (s, d) in source-major order,
//   recv_off[s, d] = sum over blocks (d', s') before (d, s) in device-major order.
// Warp 0 scans the source-major order, warp 1 the device-major one.
__device__ void block_offsets(const int32_t* __restrict__ counts, int n_src, int Nd, int* s_cnt,
                              int* s_send, int* s_recv) {
  const int nb = n_src * Nd;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) s_cnt[i] = counts[i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp < 2) {
    int run = 0;
    for (int i0 = 0; i0 < nb; i0 += 32) {
      const int i = i0 + lane;
      int b = i;
      if (warp == 1) {
        const int d = i / n_src;
        b = (i - d * n_src) * Nd + d;
      }
      const int v = i < nb ? s_cnt[b] : 0;
      int inc = v;
#pragma unroll
      for (int sh = 1; sh < 32; sh <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, sh);
        if (lane >= sh) inc += u;
      }
      if (i < nb) (warp == 0 ? s_send : s_recv)[b] = run + inc - v;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  __syncthreads();
}

// 2. send map: brim0_send over (d, t); CTA 0 also writes the block offsets.
__global__ void __launch_bounds__(kMapThreads)
shard_map_kernel(const int32_t* __restrict__ brim0, ShardSplit split, int T, int Nd,
                 const int32_t* __restrict__ counts, int32_t* __restrict__ send_off,
                 int32_t* __restrict__ recv_off, int32_t* __restrict__ brim0_send) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_cnt[kMaxBlocks], s_send[kMaxBlocks], s_recv[kMaxBlocks];
  const int n_src = split.n;
  block_offsets(counts, n_src, Nd, s_cnt, s_send, s_recv);
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int i = threadIdx.x; i < n_src * Nd; i += blockDim.x) {
      send_off[i] = s_send[i];
      recv_off[i] = s_recv[i];
    }
  }
  const int d = blockIdx.y;
  for (int t = blockIdx.x * kMapThreads + threadIdx.x; t < T; t += gridDim.x * kMapThreads) {
    // shard of token t: the last s with off[s] <= t (empty shards are skipped)
    int lo = 0, hi = n_src - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (split.off[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const size_t i = static_cast<size_t>(d) * T + t;
    const int v = brim0[i];
    brim0_send[i] = v >= 0 ? v - s_recv[lo * Nd + d] + s_send[lo * Nd + d] : -1;
  }
}

// 3. exchange: destination rows in the destination layout's block order; a
//    warp finds the block of its row by binary search over the block offsets
//    and copies the row from the same place in that block of the source layout.
__global__ void __launch_bounds__(kA2aWarps * 32)
all_to_all_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t row_bytes,
                  int64_t max_rows, const int32_t* __restrict__ counts,
                  const int32_t* __restrict__ send_off, const int32_t* __restrict__ recv_off,
                  int n_src, int Nd, int reverse) {
  pdl_wait();
  pdl_trigger();
  // blocks listed in destination order: dst offset, src offset
  __shared__ int s_dst[kMaxBlocks + 1], s_src[kMaxBlocks];
  const int nb = n_src * Nd;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    // i-th block in destination order -> (s, d)
    int s, d;
    if (reverse) s = i / Nd, d = i - s * Nd;           // send layout: source-major
    else d = i / n_src, s = i - d * n_src;             // receive layout: device-major
    const int b = s * Nd + d;
    s_dst[i] = reverse ? send_off[b] : recv_off[b];
    s_src[i] = reverse ? recv_off[b] : send_off[b];
    if (i == nb - 1) s_dst[nb] = s_dst[i] + counts[b];  // rows in all
  }
  __syncthreads();
  const int64_t total = min(static_cast<int64_t>(s_dst[nb]), max_rows);
  const int lane = threadIdx.x & 31;
  const int64_t nvec = row_bytes / 16;
  for (int64_t r = blockIdx.x * kA2aWarps + (threadIdx.x >> 5); r < total;
       r += static_cast<int64_t>(gridDim.x) * kA2aWarps) {
    // last block whose destination offset is <= r: non-empty and holding r
    int lo = 0, hi = nb - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_dst[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int64_t sr = s_src[lo] + (r - s_dst[lo]);
    if (sr < 0 || sr >= max_rows) continue;  // offsets that are not a plan: move nothing
    const uint4* sp = reinterpret_cast<const uint4*>(src + sr * row_bytes);
    uint4* dp = reinterpret_cast<uint4*>(dst + r * row_bytes);
    for (int64_t v0 = lane; v0 < nvec; v0 += 32 * 4) {
      uint4 buf[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < nvec) buf[u] = ld_nc_v4(sp + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < nvec) st_v4(dp + v0 + 32 * u, buf[u]);
    }
  }
}

}  // namespace

int launch_shard_plan(const LaunchCtx& ctx, const occult_desc_t& ds, const ShardSplit& split,
                      const uint32_t* vmask, const int32_t* brim0, int32_t* brim0_send,
                      int32_t* counts, int32_t* send_off, int32_t* recv_off) {
  const int Nd = ds.n_vdev;
  launch_pdl(shard_count_kernel, split.n, kCountThreads, 0, ctx.stream, vmask, split, Nd, counts);
  const int gx = ds.T > 0 ? (ds.T + kMapThreads - 1) / kMapThreads : 1;
  const dim3 grid(gx < 4 * ctx.num_sms ? gx : 4 * ctx.num_sms, Nd);
  launch_pdl(shard_map_kernel, grid, kMapThreads, 0, ctx.stream, brim0, split, ds.T, Nd, counts, send_off,
                                                         recv_off, brim0_send);
  return cuda_status(cudaGetLastError());
}

int launch_all_to_all(const LaunchCtx& ctx, const occult_desc_t& ds, int n_src, const void* src,
                      void* dst, int64_t row_bytes, const int32_t* counts,
                      const int32_t* send_off, const int32_t* recv_off, int reverse) {
  const int64_t max_rows = static_cast<int64_t>(ds.T) * (ds.top_k < ds.n_vdev ? ds.top_k : ds.n_vdev);
  if (max_rows == 0) return OCCULT_OK;
  int64_t blocks = (max_rows + kA2aWarps - 1) / kA2aWarps;
  const int64_t cap = static_cast<int64_t>(ctx.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  launch_pdl(all_to_all_kernel, static_cast<int>(blocks), kA2aWarps * 32, 0, ctx.stream,
      static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), row_bytes, max_rows, counts,
      send_off, recv_off, n_src, ds.n_vdev, reverse);
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
