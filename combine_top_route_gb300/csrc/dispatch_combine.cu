// Row-movement kernels of the Occult pipeline (HBM-bound):
//  * dispatch -- Appendix A.2 Algorithm 4, stage one of scattering (ORI -> SFD):
//    each token row is read once and written to the SFD row BRIM0 gives it on
//    every device it uses.
//  * dispatch to EPD -- with a single source the first all-to-all is the
//    identity, so stage one, the exchange and the device-local expansion
//    (Algorithm 5's EPD rows) can be one pass: each token row is read once and
//    written to the EPD row of each of its experts, in the padded layout the
//    GEMMs read as tiles.
//  * combine  -- the two-stage merge: stage one (EPD -> SFD) sums a received
//    row's local experts (the aggregation of Algorithm 8, done without atomics),
//    stage two (SFD -> ORI, Algorithm 9) sums the token's devices in order
//    0..Nd-1.  Inputs, accumulation and outputs are fp32 (the paper keeps its
//    merged SFD tensor in fp32 too), in a fixed order, so results are
//    deterministic.  Fused by default (one warp per token walks BRIM0 then
//    BRIM1); a materialised mode writes the SFD stage-one result out (the second
//    all-to-all's send buffer) and reads it back.
// Rows move as 16-byte vectors (8 bf16 or 4 fp32); one warp per token row.
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

constexpr int kWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
dispatch_kernel(const T* __restrict__ x, const int32_t* __restrict__ brim0,
                const uint32_t* __restrict__ vmask, int ntok, int Nd, int D,
                T* __restrict__ x_sfd, int32_t* __restrict__ sfd_tok) {
  const int lane = threadIdx.x & 31;
  const int nvec = D / Vec16<T>::N;
  pdl_wait();
  pdl_trigger();
  for (int t = blockIdx.x * kWarps + (threadIdx.x >> 5); t < ntok; t += gridDim.x * kWarps) {
    const uint32_t vm = vmask[t];
    // SFD rows of this token, one per device it uses (at most 32)
    int my_row = -1;
    if (lane < Nd && ((vm >> lane) & 1u)) my_row = brim0[static_cast<size_t>(lane) * ntok + t];
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * D);
    for (int v0 = lane; v0 < nvec; v0 += 32 * 4) {
      uint4 buf[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < nvec) buf[u] = ld_nc_v4(src + v0 + 32 * u);
      uint32_t rest = vm;
      while (rest) {
        const int d = __ffs(rest) - 1;
        rest &= rest - 1;
        const int row = __shfl_sync(0xffffffffu, my_row, d);
        uint4* dst = reinterpret_cast<uint4*>(x_sfd + static_cast<size_t>(row) * D);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (v0 + 32 * u < nvec) st_v4(dst + v0 + 32 * u, buf[u]);
      }
    }
    if (sfd_tok && my_row >= 0) sfd_tok[my_row] = t;
  }
}

// Token t's row to the padded EPD row of each of its k experts: slot s =
// slot_of[ids[t, j]] on device dv = s / n_loc, EPD row exp_off[dv * n_loc] +
// BRIM1[s][BRIM0[dv][t] - seg_off[dv]] (the device's EPD rows are numbered in
// slot order, as Algorithm 5 counts them), stored at that row + OCCULT_EPD_PAD * s.
// The rows after each slot's rows, up to a whole number of OCCULT_EPD_PAD from the
// slot's start, are zeroed.
__global__ void __launch_bounds__(kWarps * 32)
dispatch_epd_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ ids,
                    const int32_t* __restrict__ placement, const int32_t* __restrict__ brim0,
                    const int32_t* __restrict__ seg_off, const int32_t* __restrict__ brim1,
                    const int32_t* __restrict__ exp_off, int ntok, int k, int Ne, int n_loc,
                    int D, __nv_bfloat16* __restrict__ x_epd) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_slot_of[OCCULT_MAX_EXPERTS];
  for (int s = threadIdx.x; s < Ne; s += blockDim.x) s_slot_of[placement[s]] = s;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int nvec = D / 8;
  const int warp0 = blockIdx.x * kWarps + (threadIdx.x >> 5), n_warps = gridDim.x * kWarps;
  for (int t = warp0; t < ntok; t += n_warps) {
    int my_row = 0;
    if (lane < k) {
      const int s = s_slot_of[ids[static_cast<size_t>(t) * k + lane]];
      const int dv = s / n_loc;
      const int r_local = brim0[static_cast<size_t>(dv) * ntok + t] - seg_off[dv];
      my_row = exp_off[dv * n_loc] + brim1[static_cast<size_t>(s) * ntok + r_local] +
               OCCULT_EPD_PAD * s;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * D);
    for (int v0 = lane; v0 < nvec; v0 += 32 * 4) {
      uint4 buf[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < nvec) buf[u] = ld_nc_v4(src + v0 + 32 * u);
      for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xffffffffu, my_row, j);
        uint4* dst = reinterpret_cast<uint4*>(x_epd + static_cast<size_t>(row) * D);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (v0 + 32 * u < nvec) st_v4(dst + v0 + 32 * u, buf[u]);
      }
    }
  }
  // padding: (slot, row after its rows) pairs, one warp each
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (int i = warp0; i < Ne * OCCULT_EPD_PAD; i += n_warps) {
    const int s = i / OCCULT_EPD_PAD, j = i - s * OCCULT_EPD_PAD;
    const int n = exp_off[s + 1] - exp_off[s];
    const int padded = (n + OCCULT_EPD_PAD - 1) / OCCULT_EPD_PAD * OCCULT_EPD_PAD;
    if (n + j >= padded) continue;
    uint4* dst = reinterpret_cast<uint4*>(
        x_epd + (static_cast<size_t>(exp_off[s]) + OCCULT_EPD_PAD * s + n + j) * D);
    for (int v = lane; v < nvec; v += 32) st_v4(dst + v, zero);
  }
}

// Fused stage one + stage two: y[t] = sum_d (sum_j y_epd[...]) (+ y_shared[t]).
// With y_sfd given, also writes each device's stage-one sum there (and does not
// write y: the stage-two kernel does, from y_sfd).  Everything is fp32.
template <bool WRITE_SFD>
__global__ void __launch_bounds__(kWarps * 32, 3)
combine_fused_kernel(const float* __restrict__ y_epd, const int32_t* __restrict__ brim0,
                     const int32_t* __restrict__ seg_off, const int32_t* __restrict__ brim1,
                     const int32_t* __restrict__ exp_off, const float* __restrict__ y_shared,
                     int ntok, int Nd, int n_loc, int D, float* __restrict__ y_sfd,
                     float* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  constexpr int VN = 4;
  constexpr int kChunk = 8;  // EPD rows loaded per pass (all of them for k <= 8)
  __shared__ int s_rows[kWarps][OCCULT_MAX_TOPK];
  __shared__ int s_devs[kWarps][OCCULT_MAX_TOPK];
  __shared__ int s_sfd[kWarps][OCCULT_MAX_VDEV];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nvec = D / VN;
  for (int t = blockIdx.x * kWarps + warp; t < ntok; t += gridDim.x * kWarps) {
    // Row list of the token in merge order (device ascending, then local
    // expert in placement order): lane d walks device d's BRIM1 column, a warp
    // scan of the per-device counts places every row.
    int* rows = s_rows[warp];
    int* devs = s_devs[warp];
    int* sfd = s_sfd[warp];
    int v0 = -1, c = 0;
    if (lane < Nd) {
      v0 = brim0[static_cast<size_t>(lane) * ntok + t];
      if (v0 >= 0) {
        const int r = v0 - seg_off[lane];
        for (int j = 0; j < n_loc; ++j)
          c += brim1[static_cast<size_t>(lane * n_loc + j) * ntok + r] >= 0;
      }
      sfd[lane] = v0;
    }
    int o = c;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, o, sh);
      if (lane >= sh) o += u;
    }
    const int n = min(__shfl_sync(0xffffffffu, o, 31), OCCULT_MAX_TOPK);
    o -= c;
    if (c > 0) {
      const int r = v0 - seg_off[lane];
      const int base = exp_off[lane * n_loc];
      for (int j = 0; j < n_loc; ++j) {
        const int u = brim1[static_cast<size_t>(lane * n_loc + j) * ntok + r];
        if (u >= 0 && o < OCCULT_MAX_TOPK) {
          rows[o] = base + u;
          devs[o] = lane;
          ++o;
        }
      }
    }
    __syncwarp();
    for (int v = lane; v < nvec; v += 32) {
      float acc[VN], part[VN];
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = 0.f, part[i] = 0.f;
      for (int j0 = 0; j0 < n; j0 += kChunk) {
        float4 buf[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
          if (j0 + j < n) {
            const uint4 u = ld_nc_v4(reinterpret_cast<const float4*>(y_epd + static_cast<size_t>(rows[j0 + j]) * D) + v);
            buf[j] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                 __uint_as_float(u.w));
          }
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          const int jj = j0 + j;
          if (jj < n) {
            part[0] += buf[j].x; part[1] += buf[j].y; part[2] += buf[j].z; part[3] += buf[j].w;
            // close the device's stage-one sum at its last expert
            if (jj + 1 == n || devs[jj + 1] != devs[jj]) {
              if (WRITE_SFD) {
                st_v4(reinterpret_cast<float4*>(y_sfd + static_cast<size_t>(sfd[devs[jj]]) * D) + v,
                      pack16(part, float()));
              }
#pragma unroll
              for (int i = 0; i < VN; ++i) acc[i] += part[i], part[i] = 0.f;
            }
          }
        }
      }
      if (!WRITE_SFD) {
        if (y_shared) {
          const uint4 u = ld_nc_v4(reinterpret_cast<const float4*>(y_shared + static_cast<size_t>(t) * D) + v);
          acc[0] += __uint_as_float(u.x); acc[1] += __uint_as_float(u.y);
          acc[2] += __uint_as_float(u.z); acc[3] += __uint_as_float(u.w);
        }
        st_v4(reinterpret_cast<float4*>(y + static_cast<size_t>(t) * D) + v, pack16(acc, float()));
      }
    }
    __syncwarp();
  }
}

// Stage two from a materialised SFD tensor: y[t] = sum_d y_sfd[brim0[d, t]] (+ shared).
// The token's rows are first listed in device order (ballot + popcount), then
// loaded eight at a time so that their loads are in flight together.
__global__ void __launch_bounds__(kWarps * 32, 3)
combine_sfd_kernel(const float* __restrict__ y_sfd, const int32_t* __restrict__ brim0,
                   const float* __restrict__ y_shared, int ntok, int Nd, int D,
                   float* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  constexpr int VN = 4;
  constexpr int kChunk = 8;
  __shared__ int s_rows[kWarps][OCCULT_MAX_VDEV];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nvec = D / VN;
  int* rows = s_rows[warp];
  for (int t = blockIdx.x * kWarps + warp; t < ntok; t += gridDim.x * kWarps) {
    const int my_row = lane < Nd ? brim0[static_cast<size_t>(lane) * ntok + t] : -1;
    const unsigned bal = __ballot_sync(0xffffffffu, my_row >= 0);
    if (my_row >= 0) rows[__popc(bal & lanemask_lt())] = my_row;
    const int n = __popc(bal);
    __syncwarp();
    for (int v = lane; v < nvec; v += 32) {
      float acc[VN];
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = 0.f;
      for (int j0 = 0; j0 < n; j0 += kChunk) {
        uint4 buf[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
          if (j0 + j < n)
            buf[j] = ld_nc_v4(reinterpret_cast<const float4*>(y_sfd + static_cast<size_t>(rows[j0 + j]) * D) + v);
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
          if (j0 + j < n) {
            float f[VN];
            unpack16(buf[j], f, float());
#pragma unroll
            for (int i = 0; i < VN; ++i) acc[i] += f[i];
          }
      }
      if (y_shared) {
        float f[VN];
        unpack16(ld_nc_v4(reinterpret_cast<const float4*>(y_shared + static_cast<size_t>(t) * D) + v), f, float());
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] += f[i];
      }
      st_v4(reinterpret_cast<float4*>(y + static_cast<size_t>(t) * D) + v, pack16(acc, float()));
    }
    __syncwarp();
  }
}

// y = 0 before a merge by atomic additions (a kernel rather than a memset, so
// that it joins the stream's chain of dependent launches).
__global__ void __launch_bounds__(256)
zero_f32_kernel(float4* __restrict__ p, size_t n4) {
  pdl_wait();
  pdl_trigger();
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = z;
}

int grid_for(const LaunchCtx& ctx, int ntok) {
  int blocks = (ntok + kWarps - 1) / kWarps;
  const int cap = ctx.num_sms * 16;
  return blocks < cap ? (blocks > 0 ? blocks : 1) : cap;
}

}  // namespace

int launch_dispatch(const LaunchCtx& ctx, const occult_desc_t& ds, const void* x,
                    const int32_t* brim0, const uint32_t* vmask, void* x_sfd, int32_t* sfd_tok) {
  if (ds.T == 0) return OCCULT_OK;
  const int g = grid_for(ctx, ds.T);
  if (ds.dtype == OCCULT_BF16)
    launch_pdl(dispatch_kernel<__nv_bfloat16>, g, kWarps * 32, 0, ctx.stream,
               static_cast<const __nv_bfloat16*>(x), brim0, vmask, ds.T, ds.n_vdev, ds.d,
               static_cast<__nv_bfloat16*>(x_sfd), sfd_tok);
  else
    launch_pdl(dispatch_kernel<float>, g, kWarps * 32, 0, ctx.stream, static_cast<const float*>(x),
               brim0, vmask, ds.T, ds.n_vdev, ds.d, static_cast<float*>(x_sfd), sfd_tok);
  return cuda_status(cudaGetLastError());
}

int launch_dispatch_epd(const LaunchCtx& ctx, const occult_desc_t& ds, const void* x,
                        const int32_t* ids, const int32_t* placement, const int32_t* brim0,
                        const int32_t* seg_off, const int32_t* brim1, const int32_t* exp_off,
                        void* x_epd) {
  if (ds.T == 0) return OCCULT_OK;
  const int g = grid_for(ctx, ds.T);
  launch_pdl(dispatch_epd_kernel, g, kWarps * 32, 0, ctx.stream,
             static_cast<const __nv_bfloat16*>(x), ids, placement, brim0, seg_off, brim1, exp_off,
             ds.T, ds.top_k, ds.n_experts, ds.n_experts / ds.n_vdev, ds.d,
             static_cast<__nv_bfloat16*>(x_epd));
  return cuda_status(cudaGetLastError());
}

int launch_zero_f32(const LaunchCtx& ctx, float* p, size_t n) {
  if (n == 0) return OCCULT_OK;
  if (n % 4 != 0 || reinterpret_cast<uintptr_t>(p) % 16 != 0) {
    // not a whole number of aligned vectors: the plain memset
    return cuda_status(cudaMemsetAsync(p, 0, n * sizeof(float), ctx.stream));
  }
  const size_t n4 = n / 4;
  size_t blocks = (n4 + 255) / 256;
  const size_t cap = static_cast<size_t>(ctx.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return cuda_status(launch_pdl(zero_f32_kernel, static_cast<unsigned>(blocks), 256, 0, ctx.stream,
                                reinterpret_cast<float4*>(p), n4));
}

int launch_merge_sfd(const LaunchCtx& ctx, const occult_desc_t& ds, const float* y_epd,
                     const int32_t* brim0, const int32_t* seg_off, const int32_t* brim1,
                     const int32_t* exp_off, float* y_sfd) {
  if (ds.T == 0) return OCCULT_OK;
  const int g = grid_for(ctx, ds.T);
  launch_pdl(combine_fused_kernel<true>, g, kWarps * 32, 0, ctx.stream,
      y_epd, brim0, seg_off, brim1, exp_off, nullptr, ds.T, ds.n_vdev, ds.n_experts / ds.n_vdev,
      ds.d, y_sfd, nullptr);
  return cuda_status(cudaGetLastError());
}

int launch_combine_sfd(const LaunchCtx& ctx, const occult_desc_t& ds, const float* y_sfd,
                       const int32_t* brim0, const float* y_shared, float* y) {
  if (ds.T == 0) return OCCULT_OK;
  const int g = grid_for(ctx, ds.T);
  launch_pdl(combine_sfd_kernel, g, kWarps * 32, 0, ctx.stream, y_sfd, brim0, y_shared, ds.T, ds.n_vdev,
                                                        ds.d, y);
  return cuda_status(cudaGetLastError());
}

int launch_combine(const LaunchCtx& ctx, const occult_desc_t& ds, const float* y_epd,
                   const int32_t* brim0, const int32_t* seg_off, const int32_t* brim1,
                   const int32_t* exp_off, const float* y_shared, float* y_sfd, float* y) {
  if (ds.T == 0) return OCCULT_OK;
  const int g = grid_for(ctx, ds.T);
  const int n_loc = ds.n_experts / ds.n_vdev;
  if (y_sfd) {
    launch_pdl(combine_fused_kernel<true>, g, kWarps * 32, 0, ctx.stream,
        y_epd, brim0, seg_off, brim1, exp_off, nullptr, ds.T, ds.n_vdev, n_loc, ds.d, y_sfd,
        nullptr);
    launch_pdl(combine_sfd_kernel, g, kWarps * 32, 0, ctx.stream, y_sfd, brim0, y_shared, ds.T,
                                                          ds.n_vdev, ds.d, y);
  } else {
    launch_pdl(combine_fused_kernel<false>, g, kWarps * 32, 0, ctx.stream,
        y_epd, brim0, seg_off, brim1, exp_off, y_shared, ds.T, ds.n_vdev, n_loc, ds.d, nullptr,
        y);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
