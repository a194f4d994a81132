// Co-activation profiling: Occult paper Sec. 2.1 Eq. 3 (C[i, j] = tokens whose
// router output is non-zero for both i and j, diagonal = expert load) and Eq. 4
// (P = C / max C), plus the histogram of per-token replica counts C_T (Sec. 2.2).
//
// Atomics-free: one warp per 32-token chunk turns the routing into per-expert
// token bitsets (one ballot per expert), then C[i, j] is the popcount of the
// AND of two bitsets, summed by warp reductions (integers: exact in any order).
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

template <int W64>
__global__ void __launch_bounds__(256)
bitset_kernel(const int32_t* __restrict__ ids, const uint32_t* __restrict__ vmask, int n_tok,
              int k, int Ne, int max_ct, int nwords, uint32_t* __restrict__ bits,
              int32_t* __restrict__ chunk_hist) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int nchunks = (n_tok + 31) / 32;
  for (int ch = blockIdx.x * 8 + (threadIdx.x >> 5); ch < nchunks; ch += gridDim.x * 8) {
    const int t = ch * 32 + lane;
    const bool valid = t < n_tok;
    uint64_t m[W64];
#pragma unroll
    for (int w = 0; w < W64; ++w) m[w] = 0;
    if (valid) {
      for (int j = 0; j < k; ++j) {
        const int e = ids[static_cast<size_t>(t) * k + j];
#pragma unroll
        for (int w = 0; w < W64; ++w)
          if ((e >> 6) == w) m[w] |= 1ull << (e & 63);
      }
    }
#pragma unroll
    for (int w32 = 0; w32 < 2 * W64; ++w32) {
      for (int b = 0; b < 32; ++b) {
        const int e = w32 * 32 + b;
        if (e >= Ne) break;
        const unsigned bal =
            __ballot_sync(0xffffffffu, static_cast<unsigned>(m[w32 >> 1] >> ((w32 & 1) * 32 + b)) & 1u);
        if (lane == b) bits[static_cast<size_t>(e) * nwords + ch] = bal;
      }
    }
    if (chunk_hist) {
      const int ct = valid ? __popc(vmask[t]) : -1;
      for (int c = 0; c <= max_ct; ++c) {
        const unsigned bal = __ballot_sync(0xffffffffu, ct == c);
        if (lane == 0) chunk_hist[static_cast<size_t>(ch) * (max_ct + 1) + c] = __popc(bal);
      }
    }
  }
}

// C[i, j]: block i keeps expert i's token bitset in shared memory; warp w takes
// j = w, w + 8, ..., its lanes stride over the words and the popcounts are summed
// with a warp reduction (integers: exact in any order).
constexpr int kPairWarps = 8;
constexpr int kMaxSharedWords = 8192;  // 256K tokens; longer batches read global memory
__global__ void __launch_bounds__(kPairWarps * 32)
pair_count_kernel(const uint32_t* __restrict__ bits, int Ne, int nwords, int64_t* __restrict__ C) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t s_bi[kMaxSharedWords];
  const int i = blockIdx.x;
  const uint32_t* bi = bits + static_cast<size_t>(i) * nwords;
  const bool in_smem = nwords <= kMaxSharedWords;
  if (in_smem)
    for (int w = threadIdx.x; w < nwords; w += blockDim.x) s_bi[w] = bi[w];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int j = warp; j < Ne; j += kPairWarps) {
    const uint32_t* bj = bits + static_cast<size_t>(j) * nwords;
    long long acc = 0;
    for (int w = lane; w < nwords; w += 32) acc += __popc((in_smem ? s_bi[w] : bi[w]) & bj[w]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) C[static_cast<size_t>(i) * Ne + j] = acc;
  }
}

// P = C / max C and the C_T histogram (sum of the per-chunk counts): every thread
// sums a strided share of the chunks for all C_T values, then warp and block
// reductions (integers: exact in any order).
__global__ void __launch_bounds__(1024)
finish_kernel(const int64_t* __restrict__ C, int Ne, float* __restrict__ P,
              const int32_t* __restrict__ chunk_hist, int nchunks, int max_ct,
              int64_t* __restrict__ ct_hist) {
  pdl_wait();
  pdl_trigger();
  __shared__ long long s_max[32];
  __shared__ long long s_hist[32][OCCULT_MAX_TOPK + 1];  // per warp
  const int lane = threadIdx.x & 31;
  long long mx = 0;
  for (int i = threadIdx.x; i < Ne * Ne; i += blockDim.x) mx = max(mx, (long long)C[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) s_max[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    mx = threadIdx.x < (blockDim.x >> 5) ? s_max[threadIdx.x] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (threadIdx.x == 0) s_max[0] = mx;
  }
  __syncthreads();
  mx = s_max[0];
  if (P) {
    for (int i = threadIdx.x; i < Ne * Ne; i += blockDim.x)
      P[i] = mx > 0 ? static_cast<float>(static_cast<double>(C[i]) / static_cast<double>(mx)) : 0.f;
  }
  if (ct_hist) {
    long long loc[OCCULT_MAX_TOPK + 1];
#pragma unroll
    for (int c = 0; c <= OCCULT_MAX_TOPK; ++c) loc[c] = 0;
    for (int ch = threadIdx.x; ch < nchunks; ch += blockDim.x) {
      const int32_t* row = chunk_hist + static_cast<size_t>(ch) * (max_ct + 1);
#pragma unroll
      for (int c = 0; c <= OCCULT_MAX_TOPK; ++c)
        if (c <= max_ct) loc[c] += row[c];
    }
#pragma unroll
    for (int c = 0; c <= OCCULT_MAX_TOPK; ++c) {
      long long v = loc[c];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s_hist[threadIdx.x >> 5][c] = v;
    }
    __syncthreads();
    for (int c = threadIdx.x; c <= max_ct; c += blockDim.x) {
      long long v = 0;
      for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) v += s_hist[w][c];
      ct_hist[c] = v;
    }
  }
}

}  // namespace

size_t profile_ws_bytes(const occult_desc_t& ds, int n_tok) {
  const size_t nwords = (static_cast<size_t>(n_tok) + 31) / 32;
  const int max_ct = ds.top_k < ds.n_vdev ? ds.top_k : ds.n_vdev;
  size_t b = nwords * ds.n_experts * sizeof(uint32_t);
  b = (b + 255) & ~static_cast<size_t>(255);
  b += nwords * (max_ct + 1) * sizeof(int32_t);
  return b;
}

int launch_profile(const LaunchCtx& ctx, const occult_desc_t& ds, const int32_t* ids, int n_tok,
                   const uint32_t* vmask, int64_t* C, float* P, int64_t* ct_hist, void* ws) {
  const int nwords = (n_tok + 31) / 32;
  const int max_ct = ds.top_k < ds.n_vdev ? ds.top_k : ds.n_vdev;
  uint32_t* bits = static_cast<uint32_t*>(ws);
  size_t off = static_cast<size_t>(nwords) * ds.n_experts * sizeof(uint32_t);
  off = (off + 255) & ~static_cast<size_t>(255);
  int32_t* chunk_hist = (vmask && ct_hist)
      ? reinterpret_cast<int32_t*>(static_cast<char*>(ws) + off) : nullptr;
  if (nwords > 0) {
    int blocks = (nwords + 7) / 8;
    if (blocks > ctx.num_sms * 8) blocks = ctx.num_sms * 8;
#define OCCULT_BITSET_LAUNCH(W)                                                              \
    launch_pdl(bitset_kernel<W>, blocks, 256, 0, ctx.stream, ids, vmask, n_tok, ds.top_k,            \
                                                     ds.n_experts, max_ct, nwords, bits,     \
                                                     chunk_hist)
    if (ds.n_experts <= 64) OCCULT_BITSET_LAUNCH(1);
    else if (ds.n_experts <= 128) OCCULT_BITSET_LAUNCH(2);
    else OCCULT_BITSET_LAUNCH(4);
#undef OCCULT_BITSET_LAUNCH
  }
  launch_pdl(pair_count_kernel, ds.n_experts, kPairWarps * 32, 0, ctx.stream, bits, ds.n_experts, nwords,
                                                                       C);
  launch_pdl(finish_kernel, 1, 1024, 0, ctx.stream, C, ds.n_experts, P, chunk_hist, nwords, max_ct,
                                            chunk_hist ? ct_hist : nullptr);
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
