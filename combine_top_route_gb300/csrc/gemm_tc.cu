// Grouped expert GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// This is the only dense contraction of the Occult layer: the scattering
// sparse matmul (Appendix A.2 Algorithm 6, SFD -> EPD, fused with the SwiGLU
// activation and Algorithm 7's weight modulation) and the second linear layer
// of Algorithm 8 (EPD rows times W_d).  Algorithm 6 tiles each expert's BRIM1
// row; the paper condenses the non-empty parts of BRIM1 into fixed-length
// sub-vectors, one thread-block each, the expert given by the sub-vector's
// coordinate.  Here those sub-vectors are the 128-row M tiles of every expert's
// contiguous EPD segment, scheduled by a persistent kernel (one CTA per SM).
//
// CTA = 6 warps (contiguous A) or 10 warps (gathered A), warp-specialised:
//   warp 0      TMA producer: B (weights) as 2-D tiles, and A as 2-D tiles when
//               its rows are contiguous.
//   warps 6..9  (gathered A only) copy the tile's 128 A rows -- the SFD rows of
//               the condensed BRIM1 -- with 16-byte cp.async straight into the
//               128-byte-swizzled layout the tensor cores read; one warp
//               instruction moves four whole 128-byte row segments.  (TMA
//               tile::gather4 does the same in fewer instructions but measured
//               2.3x slower on this GEMM.)
//   warp 1      owns TMEM (512 columns = two 128x256 fp32 accumulators); lane 0
//               issues tcgen05.mma kind::f16 (bf16 in, fp32 accumulate).
//   warps 2..5  epilogue: tcgen05.ld the accumulator (one row per thread);
//               SwiGLU + gate -> bf16 (the EPD intermediate feeding the second
//               matmul), or plain -> fp32 (the merge input; every sum after the
//               second linear layer stays in fp32).
// Tile 128 x 256 x 64, 4 smem stages of 48 KB, both operands K-major with the
// 128-byte swizzle.  Accumulators are double-buffered so the epilogue of one
// tile overlaps the main loop of the next.  Every wait is bounded (2 s).
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int kStages = 4;
constexpr int kATileBytes = BM * BK * 2;   // 16 KB
constexpr int kBTileBytes = BN * BK * 2;   // 32 KB
constexpr int kStageBytes = kATileBytes + kBTileBytes;
constexpr int kGatherWarp0 = 6;   // first A-gather warp
__host__ __device__ constexpr int threads_for(bool gather) { return gather ? 320 : 192; }
constexpr int kMaxSeg = OCCULT_MAX_EXPERTS;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);

struct SmemTail {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem_base;
  int abort_flag;
  int mt_off[kMaxSeg + 1];
};
constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + sizeof(SmemTail);

struct Params {
  const __nv_bfloat16* a_ptr;  // A rows (gathered A only)
  int64_t a_ld;                // elements between A rows
  const int32_t* seg_off;
  const int32_t* seg_group;
  const int32_t* gather;
  const float* row_gate;
  void* out;       // bf16 with SwiGLU, fp32 otherwise
  int64_t ldo;
  int64_t b_group_rows;
  int n_seg;
  int N_out;
  int K;
  int single_rows; // rows of the only segment when seg_off is NULL
  int half_n;      // swiglu: rows from a group's gate rows to its up rows
  int n_tiles_n;
  int* dev_err;
};

__device__ __forceinline__ int seg_at(const Params& p, int s) {
  return p.seg_off ? p.seg_off[s] : (s ? p.single_rows : 0);
}

struct TileInfo {
  int seg, m0, rows, nt;
};

__device__ __forceinline__ TileInfo decode_tile(int tau, const Params& p, const int* mt_off) {
  TileInfo ti;
  const int mt = tau / p.n_tiles_n;
  ti.nt = tau - mt * p.n_tiles_n;
  // largest s with mt_off[s] <= mt (segments without tiles are skipped)
  int lo = 0, hi = p.n_seg;  // invariant: mt_off[lo] <= mt < mt_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (mt_off[mid] <= mt) lo = mid; else hi = mid;
  }
  ti.seg = lo;
  const int s0 = seg_at(p, lo);
  ti.m0 = s0 + (mt - mt_off[lo]) * BM;
  ti.rows = min(BM, seg_at(p, lo + 1) - ti.m0);
  return ti;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

template <bool GATHER, bool SWIGLU>
__global__ void __launch_bounds__(threads_for(GATHER), 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  SmemTail* tail = reinterpret_cast<SmemTail*>(smem + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- prologue ------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // TMA arrival (+ one per A-gather warp)
      mbar_init(&tail->full[s], GATHER ? 5 : 1);
      mbar_init(&tail->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tail->tfull[a], 1);
      mbar_init(&tail->tempty[a], 4);
    }
    tail->abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    // M-tile prefix over segments (one lane walks them; at most 256)
    if (lane == 0) {
      int acc = 0;
      for (int s = 0; s < p.n_seg; ++s) {
        tail->mt_off[s] = acc;
        acc += (seg_at(p, s + 1) - seg_at(p, s) + BM - 1) / BM;
      }
      tail->mt_off[p.n_seg] = acc;
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
    }
  } else if (warp == 1) {
    tmem_alloc(&tail->tmem_base, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int total = tail->mt_off[p.n_seg] * p.n_tiles_n;
  const uint32_t tbase = tail->tmem_base;
  volatile int* abort_flag = &tail->abort_flag;
  const int k_blocks = p.K / BK;

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tau = blockIdx.x; tau < total && ok; tau += gridDim.x) {
      const TileInfo ti = decode_tile(tau, p, tail->mt_off);
      const int grp = p.seg_group ? p.seg_group[ti.seg] : ti.seg;
      const int b_row0 = static_cast<int>(grp * p.b_group_rows) + ti.nt * (SWIGLU ? BN / 2 : BN);
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (!mbar_wait(&tail->empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + stage * kStageBytes;
        uint8_t* sb = sa + kATileBytes;
        if (lane == 0)
          mbar_arrive_expect_tx(&tail->full[stage], GATHER ? kBTileBytes : kStageBytes);
        __syncwarp();
        if (!GATHER && lane == 0) tma_load_2d(sa, &tmA, kb * BK, ti.m0, &tail->full[stage]);
        if (lane == 0) {
          if (SWIGLU) {
            tma_load_2d(sb, &tmB, kb * BK, b_row0, &tail->full[stage]);
            tma_load_2d(sb + kBTileBytes / 2, &tmB, kb * BK, b_row0 + p.half_n, &tail->full[stage]);
          } else {
            tma_load_2d(sb, &tmB, kb * BK, b_row0, &tail->full[stage]);
          }
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      if (lane == 0) latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  } else if (warp == 1) {
    // ---- MMA issuer --------------------------------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < total && ok; tau += gridDim.x, ++it) {
        const int a = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait(&tail->tempty[a], aph ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tbase + a * BN;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(&tail->full[stage], phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * kStageBytes);
          const uint32_t sb = sa + kATileBytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            tc_mma_f16(d_tmem, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32),
                       kIdesc, (kb | kk) != 0);
          }
          tc_commit(&tail->empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok) tc_commit(&tail->tfull[a]);
      }
      if (!ok) {
        latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
    }
    __syncwarp();
  } else if (warp < kGatherWarp0) {
    // ---- epilogue ----------------------------------------------------------
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    int it = 0;
    bool ok = true;
    for (int tau = blockIdx.x; tau < total; tau += gridDim.x, ++it) {
      const TileInfo ti = decode_tile(tau, p, tail->mt_off);
      const int a = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!mbar_wait(&tail->tfull[a], aph, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t t_row = tbase + a * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      const bool valid = row < ti.rows;
      const int64_t grow = ti.m0 + row;
      uint32_t v0[32], v1[32];
      if (SWIGLU) {
        const float g = (valid && p.row_gate) ? p.row_gate[grow] : 1.0f;
        const int col0 = ti.nt * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          tmem_ld32(t_row + c, v0);
          tmem_ld32(t_row + BN / 2 + c, v1);
          tmem_ld_wait();
          if (valid && col0 + c < p.N_out) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = g * silu_f(__uint_as_float(v0[2 * i])) * __uint_as_float(v1[2 * i]);
              const float h1 =
                  g * silu_f(__uint_as_float(v0[2 * i + 1])) * __uint_as_float(v1[2 * i + 1]);
              pk[i] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                  grow * p.ldo + col0 + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      } else {
        const int col0 = ti.nt * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          tmem_ld32(t_row + c, v0);
          tmem_ld_wait();
          if (valid && col0 + c < p.N_out) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.out) + grow * p.ldo +
                                                  col0 + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_uint4(v0[4 * i], v0[4 * i + 1], v0[4 * i + 2], v0[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->tempty[a]);
    }
    if (!ok) {
      if (lane == 0) latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  }

  if (GATHER && warp >= kGatherWarp0) {
    // ---- A gather (cp.async) -------------------------------------------------
    // Lane l copies 16-byte chunk (l % 8) of rows (l / 8) + 4 i, i < 8, of this
    // warp's 32 rows; chunk c of row r lands at r*128 + ((c ^ (r % 8)) * 16), the
    // 128-byte swizzle.  A stage is signalled full kInFlight stages late, once
    // this thread's copies for it have landed and been fenced for the async proxy.
    constexpr int kInFlight = kStages - 1;
    const int gw = warp - kGatherWarp0;
    const int chunk = lane & 7;
    const int rsub = lane >> 3;
    uint32_t dst_off[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = gw * 32 + rsub + 4 * i;
      dst_off[i] = static_cast<uint32_t>(r * 128 + ((chunk ^ (r & 7)) << 4));
    }
    int stage = 0, arr_stage = 0, inflight = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tau = blockIdx.x; tau < total && ok; tau += gridDim.x) {
      const TileInfo ti = decode_tile(tau, p, tail->mt_off);
      const __nv_bfloat16* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = min(gw * 32 + rsub + 4 * i, ti.rows - 1);
        src[i] = p.a_ptr + static_cast<int64_t>(p.gather[ti.m0 + r]) * p.a_ld + chunk * 8;
      }
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (!mbar_wait(&tail->empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + stage * kStageBytes;
#pragma unroll
        for (int i = 0; i < 8; ++i) cp_async_16(sa + dst_off[i], src[i] + kb * BK);
        cp_async_commit();
        if (++inflight > kInFlight) {
          cp_async_wait<kInFlight>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tail->full[arr_stage]);
          if (++arr_stage == kStages) arr_stage = 0;
          --inflight;
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    // every copy lands before the CTA may exit, also after an abort
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    if (ok) {
      for (; inflight > 0; --inflight) {
        if (lane == 0) mbar_arrive(&tail->full[arr_stage]);
        if (++arr_stage == kStages) arr_stage = 0;
      }
    } else {
      if (lane == 0) latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, kTmemCols);
}

// ---- host side ---------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, 128-byte swizzle.
int make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_cols,
             uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return OCCULT_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OCCULT_OK : OCCULT_ERR_CUDA;
}

template <bool GATHER, bool SWIGLU>
int launch_tc(const LaunchCtx& ctx, const CUtensorMap& ma, const CUtensorMap& mb, const Params& p) {
  auto kern = grouped_gemm_tc_kernel<GATHER, SWIGLU>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return OCCULT_ERR_CUDA;
  kern<<<ctx.num_sms, threads_for(GATHER), kSmemBytes, ctx.stream>>>(ma, mb, p);
  return cuda_status(cudaGetLastError());
}

}  // namespace

int launch_grouped_gemm_bf16(const LaunchCtx& ctx, const GroupedGemm& g) {
  if (g.n_seg > kMaxSeg || g.K % BK != 0 || g.N_out % 32 != 0) return OCCULT_ERR_UNSUPPORTED;
  if (g.max_rows == 0 || g.n_seg == 0) return OCCULT_OK;
  CUtensorMap ma, mb;
  int rc;
  // (gathered A is copied by cp.async; its map is made but unused)
  rc = make_map(&ma, g.A, g.a_rows, g.K, BK, BM);
  if (rc) return rc;
  rc = make_map(&mb, g.B, g.b_group_rows * g.n_groups, g.K, BK, g.swiglu ? BN / 2 : BN);
  if (rc) return rc;
  Params p;
  p.seg_off = g.seg_off;
  p.seg_group = g.seg_group;
  p.gather = g.gather;
  p.a_ptr = static_cast<const __nv_bfloat16*>(g.A);
  p.a_ld = g.K;
  p.row_gate = g.row_gate;
  p.out = g.out;
  p.ldo = g.ldo;
  p.b_group_rows = g.b_group_rows;
  p.n_seg = g.n_seg;
  p.N_out = g.N_out;
  p.K = g.K;
  p.single_rows = static_cast<int>(g.max_rows);
  p.half_n = g.swiglu ? g.N_out : 0;
  const int tile_n = g.swiglu ? BN / 2 : BN;
  p.n_tiles_n = (g.N_out + tile_n - 1) / tile_n;
  p.dev_err = ctx.dev_err;
  if (g.gather) {
    if (!g.swiglu) return OCCULT_ERR_UNSUPPORTED;
    return launch_tc<true, true>(ctx, ma, mb, p);
  }
  return g.swiglu ? launch_tc<false, true>(ctx, ma, mb, p) : launch_tc<false, false>(ctx, ma, mb, p);
}

}  // namespace occult
