// Grouped expert GEMMs on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// These are the only dense contractions of the Occult layer:
//  forward  -- the scattering sparse matmul (Appendix A.2 Algorithm 6, SFD -> EPD)
//              fused with the SwiGLU activation and Algorithm 7's weight
//              modulation, and the second linear layer of Algorithm 8;
//  backward -- their transposes (dgrad through W_d and through [W_g; W_u], with
//              the SwiGLU derivative fused into the first) and the per-expert
//              weight gradients, whose reduction runs over an expert's EPD rows.
// Algorithm 6 tiles each expert's BRIM1 row; the paper condenses the non-empty
// parts of BRIM1 into fixed-length sub-vectors, one thread block each.  Here those
// sub-vectors are the 128-row M tiles of every expert's contiguous EPD segment
// (or, for weight gradients, the 64-row K blocks of that segment), scheduled by a
// persistent kernel.
//
// The forward, dgrad and weight-gradient GEMMs run on CTA pairs (2-CTA
// clusters, one CTA per SM) when the segments are long enough:
// tcgen05.mma.cta_group::2 computes a 256 x 256 tile, rows 0..127 in the even
// CTA, 128..255 (the segment's next M tile) in the odd one; each CTA stages its
// own 128 A rows and half of the 256 B rows, so a 64-deep k block moves 32 KB into
// each SM instead of 48 KB and six stages fit.  The routed forward GEMMs swap the
// operands (weights on the MMA's M, the segment's rows on its N, a runtime N of
// the unit's rows rounded up to 16), so a segment's last unit carries at most 15
// padding rows instead of up to 255 (the merged down-projection on long segments
// keeps plain units, visited in token windows).  Short segments (decode) run one
// 128 x 256 tile per CTA with four 48 KB stages.
//
// Operands whose rows are EPD rows may also come from a padded EPD layout (each
// segment's rows followed by zero rows up to a multiple of 128), read as plain
// TMA tiles: the weight gradients' x and dy rows, and the dy rows of the dgrad
// through W_d.
//
// CTA = 10 warps, plus 4 when an operand is gathered (and 1 when the gathered A
// rows are also copied out to a padded EPD layout); warp-specialised:
//   warp 0       TMA producer for every operand held as a plain 2-D matrix.
//   warp 1       owns TMEM (512 columns = two 128x256 fp32 accumulators, double-
//                buffered so one tile's epilogue overlaps the next main loop);
//                lane 0 issues tcgen05.mma kind::f16 (bf16 in, fp32 accumulate)
//                -- in a pair only the even CTA's, for both; the odd CTA's lane 0
//                forwards the completion of its gathered stages to the even one.
//   warps 2..9   epilogue: tcgen05.ld of the accumulator, two warps per TMEM
//                lane quarter (half of the columns each).
//   warps 10..13 producers for a gathered operand (rows picked by the condensed
//                BRIM1): K-major rows (forward, dgrad) by cp.async, written
//                straight into the 128-byte swizzle the tensor cores read and
//                zero-filled past a unit's rows (TMA tile::gather4 measured 2.3x
//                slower there); MN-major rows (weight gradients without the
//                padded layouts) by TMA tile::gather4, four 128-byte rows an
//                instruction.
//   warp 14      (the training up-projection, and the dgrad through W_d when it
//                gathers) copies the gathered A rows of a stage to the padded
//                EPD copy before the stage is released.
// Operands are K-major (rows along K) or MN-major (rows along K of a matrix
// stored K x MN); both use the 128-byte swizzle.  Every wait is bounded (2 s).
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int kATileBytes = BM * BK * 2;   // 16 KB
constexpr int kBTileBytes = BN * BK * 2;   // 32 KB
constexpr int kMaxStages = 7;
constexpr int kMnAtomBytes = BK * 128;     // one 64-element MN atom over the 64 K rows
constexpr int kEpiWarp0 = 2;               // first epilogue warp
constexpr int kEpiWarps = 8;               // two per TMEM lane quarter, half the columns each
constexpr int kGatherWarp0 = kEpiWarp0 + kEpiWarps;  // first cp.async producer warp
constexpr int kCopyWarp = kGatherWarp0 + 4;           // stores the gathered A rows
constexpr int kMaxSeg = OCCULT_MAX_EXPERTS;
constexpr uint32_t kTmemCols = 512;

// A CTA pair keeps half of the B tile per CTA: 32 KB stages, six of them, in the
// shared memory that holds four 48 KB stages of a single CTA.
// The forward SwiGLU epilogue stores straight from registers and needs no
// staging buffer: a pair running it takes that 32 KB as a seventh stage.
__host__ __device__ constexpr bool epi_staged(int epi, bool swap = false) {
  return swap || epi != EPI_SWIGLU;
}
// The SwiGLU backward's epilogue keeps two 4 KB slots a warp (G | U of one 32 x 32
// chunk copied ahead of use, dG | dU written back in place): 64 KB, which a pair
// pays for with one operand stage.
__host__ __device__ constexpr int epi_bytes_for(int epi, bool swap = false) {
  return epi == EPI_SWIGLU_BWD && !swap ? 8 * 2 * 4096 : (epi_staged(epi, swap) ? 8 * 32 * 32 * 4 : 0);
}
__host__ __device__ constexpr int stages_for(bool pair, int epi = EPI_F32, bool swap = false) {
  return epi == EPI_SWIGLU_BWD && !swap ? (pair ? 5 : 3)
                                        : (pair ? (epi_staged(epi, swap) ? 6 : 7) : 4);
}
__host__ __device__ constexpr int b_stage_bytes(bool pair) { return pair ? kBTileBytes / 2 : kBTileBytes; }
__host__ __device__ constexpr int stage_bytes(bool pair) { return kATileBytes + b_stage_bytes(pair); }
__host__ __device__ constexpr bool op_gathered(int m) { return m == OP_GATHER_K || m == OP_GATHER_MN; }
__host__ __device__ constexpr bool op_mn(int m) { return m == OP_TMA_MN || m == OP_GATHER_MN; }
// The training GEMMs that gather K-major A rows (the up-projection with the G|U
// save, the dgrad through W_d) can also write those rows, as they stand in the
// stages, to a padded EPD copy that the weight gradients then read as tiles: one
// more warp copies them out.
__host__ __device__ constexpr bool copies_a(int am, int epi, bool wgrad, bool swap) {
  return am == OP_GATHER_K && !wgrad && !swap && (epi == EPI_SWIGLU_SAVE || epi == EPI_SWIGLU_BWD);
}
__host__ __device__ constexpr int threads_for(int am, int bm, bool copy_a = false) {
  return 32 * (kGatherWarp0 + ((op_gathered(am) || op_gathered(bm)) ? 4 : 0) + (copy_a ? 1 : 0));
}
// kind::f16 instruction descriptor, bf16 A/B, fp32 D, M = 128 (a CTA pair: 256),
// N = 256; bits 15 and 16 select MN-major A and B
__host__ __device__ constexpr uint32_t idesc_for(int am, int bm, bool pair) {
  return idesc_bf16_f32(pair ? 2 * BM : BM, BN) | (op_mn(am) ? (1u << 15) : 0u) |
         (op_mn(bm) ? (1u << 16) : 0u);
}

struct SmemTail {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t gfull[kMaxStages];        // a pair's odd CTA: its own cp.async arrivals
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t gu_full[2 * kEpiWarps];   // SwiGLU backward: a G|U slot's TMA load landed
  uint32_t tmem_base;
  int abort_flag;
  int mt_off[kMaxSeg + 1];
};
// per epilogue warp: 32 rows x 32 words, XOR-swizzled (the SwiGLU backward: two
// such 4 KB slots); after the tail (rounded up to 128 bytes so that the 16-byte
// accesses stay aligned), when staged
constexpr int kTailBytes = (static_cast<int>(sizeof(SmemTail)) + 127) & ~127;
constexpr int kEpiBytes = kEpiWarps * 32 * 32 * 4;
// Offset of the epilogue buffers from the tail: the SwiGLU backward's slots are
// TMA boxes with the 64-byte swizzle and start on 1024-byte boundaries.
__host__ __device__ constexpr int epi_off(int epi, bool swap = false) {
  return epi == EPI_SWIGLU_BWD && !swap ? (kTailBytes + 1023) & ~1023 : kTailBytes;
}
static_assert(epi_bytes_for(EPI_F32) == kEpiBytes && epi_bytes_for(EPI_SWIGLU_BWD) == 2 * kEpiBytes,
              "epilogue buffers: 4 KB a warp, 8 KB a warp for the SwiGLU backward");
__host__ __device__ constexpr int smem_bytes(bool pair, int epi, bool swap = false) {
  return 1024 /*alignment slack*/ + stages_for(pair, epi, swap) * stage_bytes(pair) +
         epi_off(epi, swap) + epi_bytes_for(epi, swap);
}
static_assert(smem_bytes(false, EPI_F32) <= 232448 && smem_bytes(true, EPI_F32) <= 232448 &&
              smem_bytes(false, EPI_SWIGLU) <= 232448 && smem_bytes(true, EPI_SWIGLU) <= 232448 &&
              smem_bytes(false, EPI_SWIGLU_BWD) <= 232448 &&
              smem_bytes(true, EPI_SWIGLU_BWD) <= 232448,
              "shared memory");

struct Params {
  // schedule
  const int32_t* seg_off;      // rows (forward / dgrad) or K rows (wgrad) of each segment
  const int32_t* seg_group;    // weight group or output matrix of each segment
  int n_seg;
  int single_rows;             // rows of the only segment when seg_off is NULL
  int K;                       // reduction length (forward / dgrad)
  int N_out;                   // output columns
  int M_total;                 // wgrad: output rows of each matrix
  int n_tiles_m;               // wgrad: M tiles per matrix
  int n_tiles_n;
  // operands
  const int32_t* gather;       // source row of every gathered operand row
  const __nv_bfloat16* g_ptr;  // gathered operand's matrix
  int64_t g_ld;                // its row length (elements)
  int g_rows;                  // its rows (an MN-major gather names row g_rows for a
                               // row past the segment: outside the map, zero-filled)
  int a_pad, b_pad;            // TMA operand rows that are EPD rows of segment s (wgrad:
                               // the K rows; forward / dgrad: A's rows) are read at
                               // row + pad * s (a padded EPD copy)
  __nv_bfloat16* a_copy;       // copies_a: padded EPD copy of the gathered A rows
                               // ([rows, K]; segment s's rows from seg_off[s] +
                               // OCCULT_EPD_PAD * s), or NULL
  int64_t b_group_rows;        // B rows per weight group (forward / dgrad)
  int half_n;                  // SwiGLU: up rows' offset in a B group; SwiGLU bwd: I
  // epilogue
  const float* row_gate;
  void* out;                   // bf16 h (SwiGLU), fp32 (plain), bf16 dG|dU (SwiGLU bwd)
  int64_t ldo;
  int64_t out_group_stride;    // wgrad: elements between output matrices
  __nv_bfloat16* gu_out;       // SwiGLU: optional copy of G|U for the backward
  const __nv_bfloat16* gu_in;  // SwiGLU bwd: G|U saved by the forward
  float* dg_part;              // SwiGLU bwd: [rows, 2 * n_tiles_n] partial gate gradients
  const int32_t* out_src;      // fp32 reduce: SFD row of every output row
  const int32_t* out_tok;      // fp32 reduce: token (output row) of every SFD row
  int* dev_err;
  int n_win;                   // forward / dgrad: each segment's units split into n_win
                               // windows, visited window-major (n_win * n_seg <= 256)
};

__device__ __forceinline__ int seg_at(const Params& p, int s) {
  return p.seg_off ? p.seg_off[s] : (s ? p.single_rows : 0);
}

// Units (a pair: two M tiles) of segment s, and the first unit of its window w
// of n_win: the windows split each segment's units evenly, in order.
template <bool PAIR>
__device__ __forceinline__ int seg_units(const Params& p, int s) {
  const int mt = (seg_at(p, s + 1) - seg_at(p, s) + BM - 1) / BM;
  return PAIR ? (mt + 1) / 2 : mt;
}
__device__ __forceinline__ int win_first(int units, int w, int n_win) {
  return static_cast<int>((static_cast<int64_t>(w) * units) / n_win);
}

// The i-th unit a CTA (pair) takes.  Forward and dgrad units cost the same
// (K is fixed), so they go round-robin.  Weight-gradient units reduce over their
// expert's rows, which vary several-fold between experts: they are ordered by
// decreasing rows and dealt out in a snake (even rounds left to right, odd
// rounds right to left), so that every CTA ends with about the same sum of K.
template <bool WGRAD>
__device__ __forceinline__ int unit_at(int i, int unit0, int n_units) {
  return i * n_units + ((WGRAD && (i & 1)) ? n_units - 1 - unit0 : unit0);
}

struct TileInfo {
  int seg;      // segment
  int grp;      // weight group / output matrix
  int m0;       // first output row (forward/dgrad: EPD row; wgrad: row of the matrix)
  int rows;     // valid output rows
  int nt;       // N tile
  int k0, k1;   // wgrad: EPD rows [k0, k1) reduced over
  int kb;       // k blocks
  int t0;       // swapped: the unit's first EPD row (its tokens are the MMA's N)
  int urows;    // swapped: the unit's rows (<= 256)
  int nmma;     // swapped: the MMA's N, urows rounded up to 16 (each CTA holds half)
};

// Tile tau of the schedule.  For a CTA pair tau is a unit of
// two consecutive M tiles of one segment and `rank` picks one; a segment with an
// odd number of M tiles ends with a unit whose second tile has no rows (it
// repeats the first tile's rows and stores nothing).
//
// Swapped (SWAP) units put the weights on the MMA's M side (256 weight rows, 128
// in each CTA) and the unit's EPD rows on its N side: N is the unit's row count
// rounded up to 16 (each CTA holds half of the rows), so a segment's last unit
// computes no more than 15 padding rows.  m0 / rows are then this CTA's half of
// the rows (m0 = t0 when that half is empty), nt the weight block.
template <bool WGRAD, bool PAIR, bool SWAP = false, bool WIN = false>
__device__ __forceinline__ TileInfo decode_tile(int tau, const Params& p, const int* mt_off,
                                                int rank) {
  TileInfo ti;
  ti.t0 = ti.urows = ti.nmma = 0;
  if (WGRAD) {
    // a pair's unit is two consecutive M tiles of the output matrix
    const int units_m = PAIR ? p.n_tiles_m / 2 : p.n_tiles_m;
    const int per = units_m * p.n_tiles_n;
    const int r = tau / per;   // rank of the segment by decreasing rows
    ti.seg = mt_off[r];
    const int rem = tau - r * per;
    const int mt = rem / p.n_tiles_n;
    ti.nt = rem - mt * p.n_tiles_n;
    ti.m0 = (PAIR ? 2 * mt + rank : mt) * BM;
    ti.rows = min(BM, p.M_total - ti.m0);
    ti.k0 = seg_at(p, ti.seg);
    ti.k1 = seg_at(p, ti.seg + 1);
    ti.kb = (ti.k1 - ti.k0 + BK - 1) / BK;
  } else {
    const int mt = tau / p.n_tiles_n;
    ti.nt = tau - mt * p.n_tiles_n;
    // largest window v with mt_off[v] <= mt (windows without tiles are skipped);
    // v = w * n_seg + s, whose units start at unit win_first(w) of segment s.
    // Without windows v is the segment and its units start at its first row.
    int lo = 0, hi = WIN ? p.n_win * p.n_seg : p.n_seg;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (mt_off[mid] <= mt) lo = mid; else hi = mid;
    }
    int seg = lo, u = mt - mt_off[lo];
    if constexpr (WIN) {
      if (p.n_win > 1) {
        seg = lo % p.n_seg;
        u += win_first(seg_units<PAIR>(p, seg), lo / p.n_seg, p.n_win);
      }
    }
    ti.seg = seg;
    if (SWAP) {
      ti.t0 = seg_at(p, seg) + u * (2 * BM);
      ti.urows = min(2 * BM, seg_at(p, seg + 1) - ti.t0);
      ti.nmma = (ti.urows + 15) & ~15;
      const int half = ti.nmma / 2;
      ti.rows = max(0, min(half, ti.urows - rank * half));
      ti.m0 = ti.rows > 0 ? ti.t0 + rank * half : ti.t0;
    } else {
      ti.m0 = seg_at(p, seg) + (PAIR ? 2 * u + rank : u) * BM;
      ti.rows = min(BM, seg_at(p, seg + 1) - ti.m0);
      if (PAIR && ti.rows <= 0) {
        ti.m0 -= BM;
        ti.rows = 0;
      }
    }
    ti.k0 = ti.k1 = 0;
    ti.kb = p.K / BK;
  }
  ti.grp = p.seg_group ? p.seg_group[ti.seg] : ti.seg;
  return ti;
}

// Writes a warp's 32 rows x W words (one row per lane, W = 16: 32 bf16, W = 32:
// 32 fp32) through shared memory so that the global stores cover whole row
// segments: W/4 lanes per row, 128/W rows per instruction.  16-byte chunk c of
// row r is kept at chunk c ^ (r % 8) of its 128-byte row (no bank conflicts on
// either side).  Rows >= valid are not written.  `out` is the address of the
// warp's first row at this column.
// The two halves are also callable alone: stage_v4 puts 16-byte chunk j of the
// lane's row in place, flush_rows stores the staged rows.
__device__ __forceinline__ void stage_v4(uint32_t* buf, int j, const uint4& v) {
  const int lane = threadIdx.x & 31;
  *reinterpret_cast<uint4*>(buf + lane * 32 + 4 * (j ^ (lane & 7))) = v;
}
template <int W>
__device__ __forceinline__ void flush_rows(uint32_t* buf, char* out, int64_t row_bytes, int valid);
template <int W>
__device__ __forceinline__ void store_rows(uint32_t* buf, const uint32_t* v, char* out,
                                           int64_t row_bytes, int valid) {
#pragma unroll
  for (int j = 0; j < W / 4; ++j)
    stage_v4(buf, j, make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
  flush_rows<W>(buf, out, row_bytes, valid);
}
template <int W>
__device__ __forceinline__ void flush_rows(uint32_t* buf, char* out, int64_t row_bytes, int valid) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  constexpr int LPR = W / 4;     // lanes per row
  constexpr int RPI = 32 / LPR;  // rows per instruction
#pragma unroll
  for (int it = 0; it < 32 / RPI; ++it) {
    const int r = it * RPI + lane / LPR;
    const int c4 = lane % LPR;
    if (r < valid)
      st_v4(out + r * row_bytes + c4 * 16,
            *reinterpret_cast<const uint4*>(buf + r * 32 + 4 * (c4 ^ (r & 7))));
  }
  __syncwarp();
}

// Like store_rows<32> (32 rows x 32 fp32 through shared memory, 8 lanes a row),
// but each 16-byte chunk is added to row dst_row(r) of `out` with a vector
// reduction; lane r of the warp holds dst_row(r) in `my_dst`.
__device__ __forceinline__ void red_rows32(uint32_t* buf, const uint32_t* v, float* out,
                                           int64_t ldo, int64_t my_dst, int valid) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint4*>(buf + lane * 32 + 4 * (j ^ (lane & 7))) =
        make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = it * 4 + lane / 8;
    const int c4 = lane % 8;
    const int64_t dst = __shfl_sync(0xffffffffu, my_dst, r);
    if (r < valid) {
      const uint4 u = *reinterpret_cast<const uint4*>(buf + r * 32 + 4 * (c4 ^ (r & 7)));
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                   :: "l"(out + dst * ldo + c4 * 4), "f"(__uint_as_float(u.x)),
                      "f"(__uint_as_float(u.y)), "f"(__uint_as_float(u.z)),
                      "f"(__uint_as_float(u.w)) : "memory");
    }
  }
  __syncwarp();
}

// silu and the logistic function with CUDA's fast exponential and division
// intrinsics (a few ulp; the IEEE division cost the SwiGLU backward 12 % of its
// time).  For g < -87 the denominator overflows and both give 0.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }
__device__ __forceinline__ float sigmoid_f(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }

// This thread's G and U segments of a SwiGLU-backward tile (BN / 2 columns of
// one row, fewer at the matrix's edge) fetched into L2.
__device__ __forceinline__ void gu_prefetch_l2(const __nv_bfloat16* g, int I, int cols) {
  const int n = min(BN / 2, cols);
  for (int c = 0; c < n; c += 64) {   // 128-byte lines
    prefetch_l2(g + c);
    prefetch_l2(g + I + c);
  }
}

// The SwiGLU backward's G and U for one warp's chunk of 32 rows x 32 columns sit
// in a 4 KB slot: G in [0, 2 KB), U in [2 KB, 4 KB), each a TMA box of 64-byte
// rows with the 64-byte swizzle: row r's 16-byte piece j (columns 8j..8j+7) at
// r * 64 + ((j ^ ((r >> 1) & 3)) << 4), so that lane r reading its own row's
// piece j touches every bank once per eight lanes.
__device__ __forceinline__ uint32_t gu_slot_off(int r, int j) {
  return static_cast<uint32_t>(r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
}
// Shared-memory descriptor of one K=16 slice of an operand tile.
//  K-major: rows along M/N at 128 B, 8-row groups every 1024 B; slice kk starts
//           32 bytes further inside the swizzle atom.
//  MN-major: 64-element MN atoms every kMnAtomBytes (leading byte offset), 8-row
//           K groups every 1024 B (stride byte offset); slice kk starts 2 groups on.
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
  if (MN) return smem_desc_sw128_mn(base + kk * 2048, kMnAtomBytes, 1024);
  return smem_desc_sw128(base + kk * 32);
}

}  // namespace

namespace {

template <int AM, int BMODE, int EPI, bool WGRAD, bool PAIR, bool SWAP>
__global__ void __launch_bounds__(threads_for(AM, BMODE, copies_a(AM, EPI, WGRAD, SWAP)), 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC,
                       const __grid_constant__ CUtensorMap tmD, const Params p) {
  pdl_wait();
  pdl_trigger();
  static_assert(!(PAIR && !WGRAD && (op_mn(AM) || op_gathered(BMODE))),
                "paired forward / dgrad GEMMs take A K-major and B a plain matrix");
  static_assert(!(WGRAD && (!op_mn(AM) || !op_mn(BMODE))), "weight gradients are MN-major");
  static_assert(!WGRAD || (epi_staged(EPI, SWAP) && kEpiBytes >= 4 * kMaxSeg),
                "weight gradients sort the segments in the epilogue buffers");
  static_assert(!SWAP || (PAIR && !WGRAD && !op_mn(AM) && BMODE == OP_TMA_K &&
                          (EPI == EPI_SWIGLU || EPI == EPI_F32 || EPI == EPI_F32_RED)),
                "swapped units: paired forward GEMMs with K-major rows and weights");
  // Swapped: the stage's first 16 KB hold this CTA's 128 weight rows (the MMA's
  // A), the next 16 KB its half of the unit's rows (the MMA's B).
  // the SwiGLU forward, with or without the G|U save
  constexpr bool kSwiGLU = EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_SAVE;
  constexpr int kStages = stages_for(PAIR, EPI, SWAP);
  constexpr int kStageBytes = stage_bytes(PAIR);
  constexpr int kBBytes = b_stage_bytes(PAIR);
  constexpr bool kGather = op_gathered(AM) || op_gathered(BMODE);
  // MN-major gathers (weight gradients) are TMA tile::gather4 loads counted in the
  // stage's transaction bytes; K-major gathers are cp.async copies counted as
  // arrivals (and, in a pair, forwarded by the odd CTA)
  constexpr bool kGatherMN = AM == OP_GATHER_MN || BMODE == OP_GATHER_MN;
  constexpr bool kGatherCp = kGather && !kGatherMN;
  constexpr bool kCopyA = copies_a(AM, EPI, WGRAD, SWAP);
  // the merges visit their units window-major (Params::n_win)
  constexpr bool kWin = EPI == EPI_F32_RED;
  const int n_win = kWin ? p.n_win : 1;
  // a stage is released by the MMAs' commit and, when the A rows are copied out,
  // by the copy warp once its store has read them
  const bool copy_a = kCopyA && p.a_copy != nullptr;
  constexpr uint32_t kIdesc = idesc_for(AM, BMODE, PAIR);
  // TMA bytes of one stage of one CTA; a pair's even CTA expects both CTAs' bytes
  constexpr uint32_t kTmaCta = (AM == OP_GATHER_K ? 0u : uint32_t(kATileBytes)) +
                               (BMODE == OP_GATHER_K ? 0u : uint32_t(kBBytes));
  constexpr uint32_t kTmaBytes = PAIR ? 2 * kTmaCta : kTmaCta;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  SmemTail* tail = reinterpret_cast<SmemTail*>(smem + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // A CTA pair (2-CTA cluster) walks the schedule as one unit; its even CTA
  // (rank 0) issues the MMAs for both and owns the full / accumulator-empty
  // barriers they wait on.
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;
  const int unit0 = PAIR ? blockIdx.x >> 1 : blockIdx.x;
  const int n_units = PAIR ? gridDim.x >> 1 : gridDim.x;

  // ---- prologue ------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // the TMA arrival, plus one per cp.async producer thread (and, in a pair,
      // one forwarded from the odd CTA for all of its producer threads)
      mbar_init(&tail->full[s], kGatherCp ? 1 + 128 + (PAIR ? 1 : 0) : 1);
      mbar_init(&tail->empty[s], copy_a ? 2 : 1);
      mbar_init(&tail->gfull[s], 128);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tail->tfull[a], 1);
      mbar_init(&tail->tempty[a], PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    for (int i = 0; i < 2 * kEpiWarps; ++i) mbar_init(&tail->gu_full[i], 1);
    tail->abort_flag = 0;
    mbar_fence_init();
  }
  if (WGRAD) {
    // the segments in order of decreasing rows (ties by index) into mt_off, the
    // rows staged in the epilogue buffers, which nothing else uses yet
    int* len = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(tail) + kTailBytes);
    for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) len[s] = seg_at(p, s + 1) - seg_at(p, s);
    __syncthreads();
    for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) {
      const int ls = len[s];
      int r = 0;
      for (int t = 0; t < p.n_seg; ++t) r += (len[t] > ls) || (len[t] == ls && t < s);
      tail->mt_off[r] = s;
    }
  }
  if (warp == 0) {
    if (!WGRAD) {
      // M-tile (pair: two-tile unit) prefix over the windows of the segments,
      // window-major (at most 256 windows in all): the lanes load 32 windows'
      // segment bounds at a time and scan their unit counts
      const int nv = n_win * p.n_seg;
      int carry = 0;
      for (int v0 = 0; v0 < nv; v0 += 32) {
        const int v = v0 + lane;
        int c = 0;
        if (v < nv) {
          const int sg = kWin ? v % p.n_seg : v;
          const int units = seg_units<PAIR>(p, sg);
          c = kWin ? win_first(units, v / p.n_seg + 1, n_win) - win_first(units, v / p.n_seg, n_win)
                   : units;
        }
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        if (v < nv) tail->mt_off[v] = carry + incl - c;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) tail->mt_off[nv] = carry;
    }
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      if (EPI == EPI_SWIGLU_BWD && !SWAP) {
        prefetch_tmap(&tmC);
        prefetch_tmap(&tmD);
      }
    }
  } else if (warp == 1) {
    if (PAIR) tmem_alloc_pair(&tail->tmem_base, kTmemCols);
    else tmem_alloc(&tail->tmem_base, kTmemCols);
  }
  tc_fence_before();
  // a pair: both CTAs' barriers exist before either signals the other's
  if (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();

  const int total = WGRAD ? p.n_seg * (PAIR ? p.n_tiles_m / 2 : p.n_tiles_m) * p.n_tiles_n
                          : tail->mt_off[n_win * p.n_seg] * p.n_tiles_n;
  const uint32_t tbase = tail->tmem_base;
  volatile int* abort_flag = &tail->abort_flag;
  // the even CTA's full and accumulator-empty barriers, as cluster addresses
  const uint32_t full_lead = PAIR ? smem_addr_in_rank(&tail->full[0], 0) : 0u;
  const uint32_t tempty_lead = PAIR ? smem_addr_in_rank(&tail->tempty[0], 0) : 0u;

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0, tau = unit0; tau < total && ok; tau = unit_at<WGRAD>(++i, unit0, n_units)) {
      const TileInfo ti = decode_tile<WGRAD, PAIR, SWAP, kWin>(tau, p, tail->mt_off, rank);
      const int n0 = ti.nt * (kSwiGLU ? BN / 2 : BN);
      for (int kb = 0; kb < ti.kb; ++kb) {
        if (!mbar_wait(&tail->empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + stage * kStageBytes;
        uint8_t* sb = sa + kATileBytes;
        uint64_t* bar = &tail->full[stage];
        if (lane == 0) {
          // K row of an MN-major operand: weight rows (dgrad) or EPD rows (wgrad)
          const int krow = WGRAD ? ti.k0 + kb * BK : static_cast<int>(ti.grp * p.b_group_rows) + kb * BK;
          const int krow_a = WGRAD ? krow + p.a_pad * ti.seg : krow;
          const int krow_b = WGRAD ? krow + p.b_pad * ti.seg : krow;
          // K-major A rows (forward / dgrad): EPD rows, padded or not
          const int arow = ti.m0 + (WGRAD ? 0 : p.a_pad * ti.seg);
          if (SWAP) {
            // this CTA's 128 weight rows of the unit's 256 (SwiGLU: 64 gate rows
            // and the 64 up rows of the same units) and 128 rows of its half of
            // the unit's rows (only the first nmma/2 are read by the MMA)
            if (leader) mbar_arrive_expect_tx(bar, kTmaBytes);
            const uint32_t lbar = full_lead + stage * 8;
            if (kSwiGLU) {
              // TMEM lane quarter q holds 16 gate rows and the 16 up rows of the
              // same intermediate units, so that one warp's epilogue sees both:
              // one 5-D box (K, 16 rows, gate/up, 4 groups of 16 units, expert)
              tma_load_5d_pair(sa, &tmB, kb * BK, 0, 0, (ti.nt * (BN / 2) + rank * 64) / 16, ti.grp,
                               lbar);
            } else {
              const int wrow = static_cast<int>(ti.grp * p.b_group_rows) + ti.nt * BN + rank * BM;
              tma_load_2d_pair(sa, &tmB, kb * BK, wrow, lbar);
            }
            if (AM == OP_TMA_K) tma_load_2d_pair(sb, &tmA, kb * BK, arow, lbar);
          } else if (PAIR) {
            // this CTA's A rows and its half of the B tile (SwiGLU: the gate rows
            // in the even CTA, the up rows in the odd one), all counted on the
            // even CTA's barrier
            if (leader) mbar_arrive_expect_tx(bar, kTmaBytes);
            const uint32_t lbar = full_lead + stage * 8;
            if (AM == OP_TMA_K) tma_load_2d_pair(sa, &tmA, kb * BK, arow, lbar);
            if (AM == OP_TMA_MN)
              for (int a = 0; a < BM / 64; ++a)
                tma_load_2d_pair(sa + a * kMnAtomBytes, &tmA, ti.m0 + 64 * a, krow_a, lbar);
            if (BMODE == OP_TMA_K) {
              const int brow = static_cast<int>(ti.grp * p.b_group_rows) + n0 +
                               rank * (kSwiGLU ? p.half_n : BN / 2);
              tma_load_2d_pair(sb, &tmB, kb * BK, brow, lbar);
            } else if (BMODE == OP_TMA_MN) {
              for (int a = 0; a < 2; ++a)
                tma_load_2d_pair(sb + a * kMnAtomBytes, &tmB, n0 + rank * (BN / 2) + 64 * a, krow_b, lbar);
            }
          } else {
            mbar_arrive_expect_tx(bar, kTmaBytes);
            if (AM == OP_TMA_K) {
              tma_load_2d(sa, &tmA, kb * BK, arow, bar);
            } else if (AM == OP_TMA_MN) {
              for (int a = 0; a < BM / 64; ++a) tma_load_2d(sa + a * kMnAtomBytes, &tmA, ti.m0 + 64 * a, krow_a, bar);
            }
            if (BMODE == OP_TMA_K) {
              const int brow = static_cast<int>(ti.grp * p.b_group_rows) + n0;
              if (kSwiGLU) {
                tma_load_2d(sb, &tmB, kb * BK, brow, bar);
                tma_load_2d(sb + kBTileBytes / 2, &tmB, kb * BK, brow + p.half_n, bar);
              } else {
                tma_load_2d(sb, &tmB, kb * BK, brow, bar);
              }
            } else if (BMODE == OP_TMA_MN) {
              for (int a = 0; a < BN / 64; ++a) tma_load_2d(sb + a * kMnAtomBytes, &tmB, n0 + 64 * a, krow_b, bar);
            }
          }
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (PAIR && ok) {
      // the even CTA's commits release this CTA's stages: wait for the release of
      // every stage, so that none lands after the CTA has exited
      for (int i = 0; i < kStages && ok; ++i) {
        if (!mbar_wait(&tail->empty[stage], phase ^ 1u, abort_flag)) ok = false;
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      if (lane == 0) latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---- MMA issuer --------------------------------------------------------
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tau = unit0; tau < total && ok; tau = unit_at<WGRAD>(++it, unit0, n_units)) {
        const TileInfo ti = decode_tile<WGRAD, PAIR, SWAP, kWin>(tau, p, tail->mt_off, rank);
        const int a = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!(PAIR ? mbar_wait_cluster(&tail->tempty[a], aph ^ 1u, abort_flag)
                   : mbar_wait(&tail->tempty[a], aph ^ 1u, abort_flag))) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tbase + a * BN;
        const uint32_t idesc = SWAP ? idesc_bf16_f32(2 * BM, ti.nmma) : kIdesc;
        for (int kb = 0; kb < ti.kb; ++kb) {
          if (!(PAIR ? mbar_wait_cluster(&tail->full[stage], phase, abort_flag)
                     : mbar_wait(&tail->full[stage], phase, abort_flag))) { ok = false; break; }
          // cp.async data arrived through the generic proxy: make it visible to
          // the tensor cores' (async proxy) operand reads
          if (kGatherCp) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * kStageBytes);
          const uint32_t sb = sa + kATileBytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (PAIR)
              tc_mma_f16_pair(d_tmem, operand_desc<op_mn(AM)>(sa, kk), operand_desc<op_mn(BMODE)>(sb, kk),
                              idesc, (kb | kk) != 0);
            else
              tc_mma_f16(d_tmem, operand_desc<op_mn(AM)>(sa, kk), operand_desc<op_mn(BMODE)>(sb, kk),
                         kIdesc, (kb | kk) != 0);
          }
          if (PAIR) tc_commit_pair(&tail->empty[stage], 0x3);
          else tc_commit(&tail->empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        // with no k block the commit arrives at once and the epilogue writes zeros
        if (ok) {
          if (PAIR) tc_commit_pair(&tail->tfull[a], 0x3);
          else tc_commit(&tail->tfull[a]);
        }
      }
      if (!ok) {
        latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
    } else if (PAIR && kGatherCp && lane == 0) {
      // ---- odd CTA: forwards its gathered stages to the even CTA -------------
      // Its cp.async copies complete on its own barrier; once a stage's have all
      // landed, they are made visible to the async proxy (the even CTA's MMAs
      // read them) and counted as one arrival on the even CTA's full barrier.
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0, tau = unit0; tau < total && ok; tau = unit_at<WGRAD>(++i, unit0, n_units)) {
        const TileInfo ti = decode_tile<WGRAD, PAIR, SWAP, kWin>(tau, p, tail->mt_off, rank);
        for (int kb = 0; kb < ti.kb; ++kb) {
          if (!mbar_wait(&tail->gfull[stage], phase, abort_flag)) { ok = false; break; }
          fence_proxy_async_smem();
          mbar_arrive_remote(full_lead + stage * 8);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
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
    const int half = (warp - kEpiWarp0) / 4;  // which half of the tile's columns
    const int row = quarter * 32 + lane;
    // SwiGLU backward: this warp's two G | U slots, the slot of the next chunk to
    // process, whether that chunk (the next tile's first) is already in flight,
    // the parity each slot's barrier completes with next, the slots with a load
    // in flight
    constexpr bool kGuStaged = EPI == EPI_SWIGLU_BWD && !SWAP;
    uint8_t* gbuf = reinterpret_cast<uint8_t*>(tail) + epi_off(EPI, SWAP) + (warp - kEpiWarp0) * 8192;
    uint64_t* gbar = &tail->gu_full[2 * (warp - kEpiWarp0)];
    int gslot = 0;
    bool gnext = false;
    uint32_t gpar = 0, gpend = 0;
    int it = 0;
    bool ok = true;
    for (int tau = unit0; tau < total; tau = unit_at<WGRAD>(++it, unit0, n_units)) {
      const TileInfo ti = decode_tile<WGRAD, PAIR, SWAP, kWin>(tau, p, tail->mt_off, rank);
      const int a = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      const bool valid = row < ti.rows;
      const int64_t grow = ti.m0 + row;
      // Loads that do not depend on the accumulator are issued before waiting
      // for it, so that their latency hides behind the tile's MMAs: the row
      // gates, the merge's destination rows.  The SwiGLU backward also fetches
      // the next tile's G|U rows into L2 while this one is processed (the first
      // tile's too).
      const __nv_bfloat16* gu_row = nullptr;
      if (EPI == EPI_SWIGLU_BWD && !SWAP) {
        const int64_t ld_gu = 2 * static_cast<int64_t>(p.half_n);
        const int c0 = ti.nt * BN + half * (BN / 2);
        gu_row = p.gu_in + (valid ? grow : ti.m0) * ld_gu + c0;
        if (it == 0 && valid && c0 < p.N_out) gu_prefetch_l2(gu_row, p.half_n, p.N_out - c0);
        const int tau_n = unit_at<WGRAD>(it + 1, unit0, n_units);
        if (tau_n < total) {
          const TileInfo tn = decode_tile<WGRAD, PAIR, SWAP, kWin>(tau_n, p, tail->mt_off, rank);
          const int cn = tn.nt * BN + half * (BN / 2);
          if (row < tn.rows && cn < p.N_out)
            gu_prefetch_l2(p.gu_in + (tn.m0 + row) * ld_gu + cn, p.half_n, p.N_out - cn);
        }
      }
      float g_pre = 0.f;
      if (EPI == EPI_SWIGLU_BWD && !SWAP && valid) g_pre = p.row_gate[grow];
      if (kSwiGLU && !SWAP) g_pre = (valid && p.row_gate) ? p.row_gate[grow] : 1.0f;
      int64_t dst_pre = 0;
      if (EPI == EPI_F32_RED && !SWAP && valid) dst_pre = p.out_tok[p.out_src[grow]];
      constexpr int kSwapChunks = 4;  // a swapped unit's columns: at most 4 chunks a warp
      int64_t dst_sw[kSwapChunks];
      float gate_sw[kSwapChunks];
      if (SWAP) {
#pragma unroll
        for (int j = 0; j < kSwapChunks; ++j) {
          const int col_l = half * 32 + 64 * j + lane;
          dst_sw[j] = 0;
          gate_sw[j] = 1.0f;
          if (col_l < ti.urows) {
            if (EPI == EPI_F32_RED) dst_sw[j] = p.out_tok[p.out_src[ti.t0 + col_l]];
            if (EPI == EPI_F32) dst_sw[j] = ti.t0 + col_l;
            if (EPI == EPI_SWIGLU && p.row_gate) gate_sw[j] = p.row_gate[ti.t0 + col_l];
          }
        }
      }
      // valid 32-column chunks of this warp's half of a SwiGLU-backward tile
      auto gu_chunks = [&](const TileInfo& t) {
        return max(0, min(4, (p.N_out - t.nt * BN - half * (BN / 2)) / 32));
      };
      // this warp's 32 x 32 chunk of G and of U (column c of its half of tile t)
      // into slot sl by two TMA boxes, issued by lane 0 once the slot's last TMA
      // store has read it (rows past the matrix arrive as zeros)
      auto gu_load = [&](int sl, const TileInfo& t, int c) {
        if (lane == 0) {
          bulk_wait_read<0>();
          mbar_arrive_expect_tx(gbar + sl, 4096);
          const int col = t.nt * BN + half * (BN / 2) + c;
          const int r0 = t.m0 + quarter * 32;
          tma_load_2d(gbuf + sl * 4096, &tmC, col, r0, gbar + sl);
          tma_load_2d(gbuf + sl * 4096 + 2048, &tmC, p.half_n + col, r0, gbar + sl);
        }
        gpend |= 1u << sl;
      };
      if (kGuStaged && !gnext && gu_chunks(ti) > 0) {
        // no chunk of this tile in flight yet: its first one now, while the MMAs run
        gu_load(gslot, ti, 0);
      }
      gnext = false;
      if (!mbar_wait(&tail->tfull[a], aph, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t t_row = tbase + a * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      const int wrows = max(0, min(32, ti.rows - quarter * 32));  // valid rows of this warp
      const int64_t wrow0 = ti.m0 + quarter * 32;
      uint32_t* ebuf = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(tail) + kTailBytes) +
                       (warp - kEpiWarp0) * 32 * 32;
      uint32_t v0[32], v1[32];
      if (SWAP) {
        // TMEM columns are the unit's rows t0 + c (nmma of them), lanes this CTA's
        // weight rows; each warp takes the 32-column chunks of its half
        if (EPI == EPI_SWIGLU) {
          // lanes 0..15: gate rows of intermediate units i0 .. i0+15, lanes 16..31:
          // their up rows; after one exchange each lane holds G and U of one unit
          // for 16 of the chunk's columns (lanes < 16 the first 16)
          const int i0 = ti.nt * (BN / 2) + rank * 64 + quarter * 16;
          const int li = lane & 15;
          const bool hi = lane >= 16;
          __nv_bfloat16* hout = static_cast<__nv_bfloat16*>(p.out);
          uint16_t* hb = reinterpret_cast<uint16_t*>(ebuf);  // [32 columns][16 units]
          // a last weight block past N_out (N_out % 128 != 0) leaves quarters idle
          const int c_end = i0 < p.N_out ? ti.nmma : 0;
#pragma unroll
          for (int j = 0; j < kSwapChunks; ++j) {
            const int c = half * 32 + 64 * j;
            if (c >= c_end) break;
            tmem_ld32(t_row + c, v0);
            tmem_ld_wait();
            const float gl = gate_sw[j];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const uint32_t send = hi ? v0[t] : v0[16 + t];
              const float recv = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 16));
              const int col = hi ? 16 + t : t;
              const float G = hi ? recv : __uint_as_float(v0[t]);
              const float U = hi ? __uint_as_float(v0[16 + t]) : recv;
              const float gj = __shfl_sync(0xffffffffu, gl, col);
              const float hv = gj * silu_f(G) * U;
              hb[col * 16 + li] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
            }
            __syncwarp();
            // 32 rows of 32 bytes: two 16-byte chunks a row
#pragma unroll
            for (int it2 = 0; it2 < 2; ++it2) {
              const int q = it2 * 32 + lane;
              const int r = q >> 1, c2 = q & 1;
              if (c + r < ti.urows)
                st_v4(hout + (ti.t0 + c + r) * p.ldo + i0 + c2 * 8,
                      *reinterpret_cast<const uint4*>(hb + r * 16 + c2 * 8));
            }
            __syncwarp();
          }
        } else {
          // fp32 rows: lanes are 32 output columns, transposed through shared
          // memory so that each row's 128 bytes leave as 16-byte vectors (8 lanes
          // a row), stored at row t0 + c (plain) or added into the token's row
          const int d0 = ti.nt * BN + rank * BM + quarter * 32;
          float* out = static_cast<float*>(p.out);
          const int c_end = d0 < p.N_out ? ti.nmma : 0;
#pragma unroll
          for (int j = 0; j < kSwapChunks; ++j) {
            const int c = half * 32 + 64 * j;
            if (c >= c_end) break;
            const int64_t dst_l = dst_sw[j];
            tmem_ld32(t_row + c, v0);
            tmem_ld_wait();
#pragma unroll
            for (int r = 0; r < 32; ++r)
              ebuf[r * 32 + ((((lane >> 2) ^ (r & 7)) << 2) | (lane & 3))] = v0[r];
            __syncwarp();
#pragma unroll
            for (int it2 = 0; it2 < 8; ++it2) {
              const int r = it2 * 4 + (lane >> 3), c4 = lane & 7;
              const int64_t dst = __shfl_sync(0xffffffffu, dst_l, r);
              if (c + r < ti.urows) {
                const uint4 u = *reinterpret_cast<const uint4*>(ebuf + r * 32 + ((c4 ^ (r & 7)) << 2));
                float* o = out + dst * p.ldo + d0 + c4 * 4;
                if (EPI == EPI_F32_RED)
                  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                               :: "l"(o), "f"(__uint_as_float(u.x)), "f"(__uint_as_float(u.y)),
                                  "f"(__uint_as_float(u.z)), "f"(__uint_as_float(u.w)) : "memory");
                else
                  st_v4(o, u);
              }
            }
            __syncwarp();
          }
        }
      } else if (EPI == EPI_SWIGLU_SAVE) {
        // h and the saved G | U leave through this warp's staging buffer, eight
        // rows of 64 bytes per store instruction (a row per lane would touch 32
        // rows per instruction, three times per chunk, and throttle the LSU)
        const float g = g_pre;
        const int col0 = ti.nt * (BN / 2);
        const int64_t ld_gu = 2 * static_cast<int64_t>(p.N_out);
        __nv_bfloat16* hout = static_cast<__nv_bfloat16*>(p.out) + wrow0 * p.ldo + col0;
        __nv_bfloat16* gout = p.gu_out + wrow0 * ld_gu + col0;
#pragma unroll 1
        for (int c = half * (BN / 4); c < (half + 1) * (BN / 4); c += 32) {
          tmem_ld32(t_row + c, v0);
          tmem_ld32(t_row + BN / 2 + c, v1);
          tmem_ld_wait();
          if (col0 + c < p.N_out) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = g * silu_f(__uint_as_float(v0[2 * i])) * __uint_as_float(v1[2 * i]);
              const float h1 =
                  g * silu_f(__uint_as_float(v0[2 * i + 1])) * __uint_as_float(v1[2 * i + 1]);
              pk[i] = pack_bf16x2(h0, h1);
            }
            store_rows<16>(ebuf, pk, reinterpret_cast<char*>(hout + c), p.ldo * 2, wrows);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
            store_rows<16>(ebuf, pk, reinterpret_cast<char*>(gout + c), ld_gu * 2, wrows);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
            store_rows<16>(ebuf, pk, reinterpret_cast<char*>(gout + p.N_out + c), ld_gu * 2, wrows);
          }
        }
      } else if (EPI == EPI_SWIGLU) {
        const float g = g_pre;
        const int col0 = ti.nt * (BN / 2);
#pragma unroll 1
        for (int c = half * (BN / 4); c < (half + 1) * (BN / 4); c += 32) {
          tmem_ld32(t_row + c, v0);
          tmem_ld32(t_row + BN / 2 + c, v1);
          tmem_ld_wait();
          if (col0 + c < p.N_out) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = g * silu_f(__uint_as_float(v0[2 * i])) * __uint_as_float(v1[2 * i]);
              const float h1 =
                  g * silu_f(__uint_as_float(v0[2 * i + 1])) * __uint_as_float(v1[2 * i + 1]);
              pk[i] = pack_bf16x2(h0, h1);
            }
            // one 64-byte row segment per thread (stores were measured not to limit
            // this kernel, and staging them costs more than it saves)
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                    grow * p.ldo + col0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
              if (p.gu_out) {
                // G and U for the backward, rows [G | U] of 2*N_out
                uint4* gu = reinterpret_cast<uint4*>(p.gu_out + grow * (2 * static_cast<int64_t>(p.N_out)) + col0 + c);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  gu[i] = make_uint4(pack_bf16x2(__uint_as_float(v0[8 * i]), __uint_as_float(v0[8 * i + 1])),
                                     pack_bf16x2(__uint_as_float(v0[8 * i + 2]), __uint_as_float(v0[8 * i + 3])),
                                     pack_bf16x2(__uint_as_float(v0[8 * i + 4]), __uint_as_float(v0[8 * i + 5])),
                                     pack_bf16x2(__uint_as_float(v0[8 * i + 6]), __uint_as_float(v0[8 * i + 7])));
                gu += p.N_out / 8;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  gu[i] = make_uint4(pack_bf16x2(__uint_as_float(v1[8 * i]), __uint_as_float(v1[8 * i + 1])),
                                     pack_bf16x2(__uint_as_float(v1[8 * i + 2]), __uint_as_float(v1[8 * i + 3])),
                                     pack_bf16x2(__uint_as_float(v1[8 * i + 4]), __uint_as_float(v1[8 * i + 5])),
                                     pack_bf16x2(__uint_as_float(v1[8 * i + 6]), __uint_as_float(v1[8 * i + 7])));
              }
            }
          }
        }
      } else if (EPI == EPI_SWIGLU_BWD) {
        // accumulator = dh' (gradient of the modulated intermediate) for the
        // tile's 256 columns of I.  G and U of the forward arrive chunk by chunk
        // in this warp's two slots by TMA, one chunk ahead (the next tile's first
        // chunk during this tile's last); dG and dU overwrite them in place and
        // leave by TMA stores (a warp with fewer than 32 rows of the segment
        // stores its rows itself, so that no store reaches past the segment).
        const float g = g_pre;
        const int col0 = ti.nt * BN + half * (BN / 2);
        const int I = p.half_n;
        const int nch = gu_chunks(ti);
        float dg = 0.f;
#pragma unroll 1
        for (int ch = 0; ch < nch; ++ch) {
          const int c = ch * 32;
          tmem_ld32(t_row + half * (BN / 2) + c, v0);
          // the chunk after this one: this tile's next, or the next tile's first
          if (ch + 1 < nch) {
            gu_load(gslot ^ 1, ti, c + 32);
          } else {
            const int tau_n = unit_at<WGRAD>(it + 1, unit0, n_units);
            if (tau_n < total) {
              const TileInfo tn = decode_tile<WGRAD, PAIR, SWAP, kWin>(tau_n, p, tail->mt_off, rank);
              if (gu_chunks(tn) > 0) {
                gu_load(gslot ^ 1, tn, 0);
                gnext = true;
              }
            }
          }
          if (!mbar_wait(gbar + gslot, (gpar >> gslot) & 1u, abort_flag)) {
            tmem_ld_wait();
            ok = false;
            break;
          }
          gpar ^= 1u << gslot;
          gpend &= ~(1u << gslot);
          uint8_t* slot = gbuf + gslot * 4096;
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4* gp = reinterpret_cast<uint4*>(slot + gu_slot_off(lane, j));
            uint4* up = reinterpret_cast<uint4*>(slot + 2048 + gu_slot_off(lane, j));
            const uint4 gq = *gp, uq = *up;
            const uint32_t pg[4] = {gq.x, gq.y, gq.z, gq.w};
            const uint32_t pu[4] = {uq.x, uq.y, uq.z, uq.w};
            uint32_t og[4], ou[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float dG[2], dU[2];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const float G = __uint_as_float(h ? (pg[i] & 0xffff0000u) : (pg[i] << 16));
                const float U = __uint_as_float(h ? (pu[i] & 0xffff0000u) : (pu[i] << 16));
                const float dhp = __uint_as_float(v0[8 * j + 2 * i + h]);
                const float sg = sigmoid_f(G);
                const float sv = G * sg;
                dg = fmaf(dhp, sv * U, dg);
                const float dh = g * dhp;
                dG[h] = dh * U * sg * (1.0f + G * (1.0f - sg));
                dU[h] = dh * sv;
              }
              og[i] = pack_bf16x2(dG[0], dG[1]);
              ou[i] = pack_bf16x2(dU[0], dU[1]);
            }
            *gp = make_uint4(og[0], og[1], og[2], og[3]);
            *up = make_uint4(ou[0], ou[1], ou[2], ou[3]);
          }
          // this lane's writes ordered before the TMA engine's accesses to the
          // slot (the store below, the load two chunks on)
          fence_proxy_async_smem();
          if (wrows == 32) {
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmD, slot, col0 + c, static_cast<int>(wrow0));
              tma_store_2d(&tmD, slot + 2048, I + col0 + c, static_cast<int>(wrow0));
              bulk_commit();
            }
          } else {
            __syncwarp();
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + wrow0 * p.ldo + col0 + c;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = (lane >> 2) + 8 * i, j = lane & 3;
              if (r < wrows) {
                st_v4(o + r * p.ldo + j * 8, *reinterpret_cast<const uint4*>(slot + gu_slot_off(r, j)));
                st_v4(o + r * p.ldo + I + j * 8,
                      *reinterpret_cast<const uint4*>(slot + 2048 + gu_slot_off(r, j)));
              }
            }
          }
          __syncwarp();        // the slot is refilled two chunks on
          gslot ^= 1;
        }
        if (!ok) break;
        // one partial per (row, N tile, column half)
        if (valid) p.dg_part[grow * (2 * p.n_tiles_n) + 2 * ti.nt + half] = dg;
      } else if (EPI == EPI_F32_RED) {
        // fp32 rows added into their tokens' output rows (the merge)
        const int col0 = ti.nt * BN;
        const int64_t my_dst = dst_pre;
#pragma unroll 1
        for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
          tmem_ld32(t_row + c, v0);
          tmem_ld_wait();
          if (col0 + c < p.N_out)
            red_rows32(ebuf, v0, static_cast<float*>(p.out) + col0 + c, p.ldo, my_dst, wrows);
        }
      } else {
        // plain fp32 tile; a weight-gradient tile without rows is zero
        const int col0 = ti.nt * BN;
        float* obase = static_cast<float*>(p.out) + (WGRAD ? ti.grp * p.out_group_stride : 0);
#pragma unroll 1
        for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
          tmem_ld32(t_row + c, v0);
          tmem_ld_wait();
          if (col0 + c < p.N_out) {
            if (WGRAD && ti.kb == 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v0[i] = 0u;
            }
            store_rows<32>(ebuf, v0, reinterpret_cast<char*>(obase + wrow0 * p.ldo + col0 + c),
                           p.ldo * 4, wrows);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // the accumulator may be overwritten: tell the CTA that issues the MMAs
        if (PAIR && !leader) mbar_arrive_cluster(tempty_lead + a * 8);
        else mbar_arrive(&tail->tempty[a]);
      }
    }
    if (kGuStaged) {
      // the TMA stores complete, and a load still in flight (after a timeout)
      // lands, before the CTA may exit
      if (lane == 0) bulk_wait<0>();
      volatile int no_abort = 0;
      for (int sl = 0; sl < 2; ++sl)
        if (gpend & (1u << sl)) mbar_wait(gbar + sl, (gpar >> sl) & 1u, &no_abort);
      __syncwarp();
    }
    if (!ok) {
      if (lane == 0) latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  }

  if (kGatherMN && warp >= kGatherWarp0 && warp < kCopyWarp) {
    // ---- TMA gathers of the MN-major operand (weight gradients) -----------------
    // K row k of a stage is EPD row k0 + kb*64 + k, whose source row the gather
    // array names (past the segment's end: row g_rows, outside the map, zeros).  Warp gw takes rows
    // 16 gw .. 16 gw + 15; lane j < 16 holds row 16 gw + j's source, loaded four
    // stages ahead.  Lane i < 4 * atoms issues one tile::gather4: rows
    // 16 gw + 4 (i % 4) .. + 3 of MN atom i / 4 (64 columns, 128 bytes a row),
    // landing in the 128-byte-swizzled MN-major layout the MMA reads, counted in
    // the stage's transaction bytes on the (even CTA's) full barrier.
    constexpr bool kOnA = AM == OP_GATHER_MN;
    constexpr int kAtoms = (kOnA ? BM : (PAIR ? BN / 2 : BN)) / 64;
    const CUtensorMap* gmap = kOnA ? &tmA : &tmB;
    const int gw = warp - kGatherWarp0;
    const int grp = lane & 3, atom = lane >> 2;
    const int k_first = 16 * gw + 4 * grp;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0, tau = unit0; tau < total && ok; tau = unit_at<WGRAD>(++i, unit0, n_units)) {
      const TileInfo ti = decode_tile<WGRAD, PAIR, SWAP, kWin>(tau, p, tail->mt_off, rank);
      auto load_idx = [&](int kb) -> int {
        const int r = ti.k0 + kb * BK + 16 * gw + (lane & 15);
        return r < ti.k1 ? p.gather[r] : p.g_rows;
      };
      int idx_cur = ti.kb > 0 ? load_idx(0) : p.g_rows;
      int idx_1 = ti.kb > 1 ? load_idx(1) : p.g_rows;
      int idx_2 = ti.kb > 2 ? load_idx(2) : p.g_rows;
      int idx_3 = ti.kb > 3 ? load_idx(3) : p.g_rows;
      const int mn0 = kOnA ? ti.m0 : ti.nt * BN + (PAIR ? rank * (BN / 2) : 0);
      for (int kb = 0; kb < ti.kb; ++kb) {
        const int idx_4 = kb + 4 < ti.kb ? load_idx(kb + 4) : p.g_rows;
        if (!mbar_wait(&tail->empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        const int y0 = __shfl_sync(0xffffffffu, idx_cur, 4 * grp);
        const int y1 = __shfl_sync(0xffffffffu, idx_cur, 4 * grp + 1);
        const int y2 = __shfl_sync(0xffffffffu, idx_cur, 4 * grp + 2);
        const int y3 = __shfl_sync(0xffffffffu, idx_cur, 4 * grp + 3);
        if (lane < 4 * kAtoms) {
          uint8_t* sa = smem + stage * kStageBytes;
          uint8_t* dst = (kOnA ? sa : sa + kATileBytes) + atom * kMnAtomBytes +
                         (k_first >> 3) * 1024 + (k_first & 7) * 128;
          if (PAIR)
            tma_gather4_pair(dst, gmap, mn0 + 64 * atom, y0, y1, y2, y3, full_lead + stage * 8);
          else
            tma_gather4(dst, gmap, mn0 + 64 * atom, y0, y1, y2, y3, &tail->full[stage]);
        }
        __syncwarp();
        idx_cur = idx_1;
        idx_1 = idx_2;
        idx_2 = idx_3;
        idx_3 = idx_4;
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      if (lane == 0) latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  }

  if (kGatherCp && warp >= kGatherWarp0 && warp < kCopyWarp) {
    // ---- cp.async producers for the gathered K-major operand --------------------
    // Every thread arrives on a stage's full barrier asynchronously, when its
    // copies for that stage have landed (cp.async.mbarrier.arrive); the MMA thread
    // fences them for the async proxy after its wait.
    static_assert(!kGatherCp || AM == OP_GATHER_K, "cp.async gathers are K-major A operands");
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0, tau = unit0; tau < total && ok; tau = unit_at<WGRAD>(++i, unit0, n_units)) {
      const TileInfo ti = decode_tile<WGRAD, PAIR, SWAP, kWin>(tau, p, tail->mt_off, rank);
      // K-major rows (forward / dgrad A): lane l copies 16-byte chunk (l % 8) of
      // rows (l / 8) + 4 i, i < 8, of this warp's 32 rows; chunk c of row r lands
      // at r*128 + ((c ^ (r % 8)) * 16)
      // Rows past the tile's valid rows are zero-filled (their source address
      // clamped to a valid row, from which nothing is read): the copy of the A
      // rows relies on it for the zeros after a segment's rows.
      const __nv_bfloat16* src_k[8];
      uint32_t dst_k[8];
      uint32_t live = 0;
      {
        const int gw = warp - kGatherWarp0, chunk = lane & 7, rsub = lane >> 3;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = gw * 32 + rsub + 4 * i;
          dst_k[i] = static_cast<uint32_t>(r * 128 + ((chunk ^ (r & 7)) << 4));
          const int rr = max(0, min(r, ti.rows - 1));  // a pair's empty half reads row 0
          src_k[i] = p.g_ptr + static_cast<int64_t>(p.gather[ti.m0 + rr]) * p.g_ld + chunk * 8;
          live |= (r < ti.rows ? 1u : 0u) << i;
        }
      }
      for (int kb = 0; kb < ti.kb; ++kb) {
        if (!mbar_wait(&tail->empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + stage * kStageBytes;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          cp_async_16_zfill((SWAP ? sa + kATileBytes : sa) + dst_k[i], src_k[i] + kb * BK,
                            ((live >> i) & 1u) ? 16u : 0u);
        cp_async_arrive_noinc(PAIR && !leader ? &tail->gfull[stage] : &tail->full[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    // every copy lands before the CTA may exit, also after an abort
    cp_async_wait_all();
    if (!ok) {
      if (lane == 0) latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
  }

  if (kCopyA && warp == kCopyWarp) {
    // ---- the gathered A rows out to their padded EPD copy -----------------------
    // Follows the stages as the MMAs do.  Once a stage's A rows have landed (in a
    // pair's odd CTA: its own cp.async barrier), this CTA's 128 rows of k block kb
    // are copied out in the unit of N tile kb % n_tiles_n, so that an M tile's
    // copies are spread over its N tiles' units: 16-byte pieces from shared
    // memory (undoing the 128-byte swizzle) to global stores, four 128-byte rows
    // an instruction; the stage is released once the pieces are in registers.
    // The zero-filled rows after a segment's end land in its padding.
    if (copy_a) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int chunk = lane & 7, rsub = lane >> 3;
      for (int i = 0, tau = unit0; tau < total && ok; tau = unit_at<WGRAD>(++i, unit0, n_units)) {
        const TileInfo ti = decode_tile<WGRAD, PAIR, SWAP, kWin>(tau, p, tail->mt_off, rank);
        __nv_bfloat16* dst = p.a_copy + (static_cast<int64_t>(ti.m0) + OCCULT_EPD_PAD * ti.seg) * p.K;
        for (int kb = 0; kb < ti.kb; ++kb) {
          uint64_t* landed = PAIR && !leader ? &tail->gfull[stage] : &tail->full[stage];
          if (!mbar_wait(landed, phase, abort_flag)) { ok = false; break; }
          if (ti.rows > 0 && kb % p.n_tiles_n == ti.nt) {
            const uint8_t* sa = smem + stage * kStageBytes;
            char* out = reinterpret_cast<char*>(dst + kb * BK) + chunk * 16;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint4 v[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int r = (g * 8 + j) * 4 + rsub;
                v[j] = *reinterpret_cast<const uint4*>(sa + r * 128 + ((chunk ^ (r & 7)) << 4));
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int r = (g * 8 + j) * 4 + rsub;
                st_v4(out + static_cast<int64_t>(r) * p.K * 2, v[j]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&tail->empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        if (lane == 0) latch_error(p.dev_err, OCCULT_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  // a pair: neither CTA exits (or frees its TMEM) while the other may still
  // signal it or run MMAs into it
  if (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if (PAIR) tmem_dealloc_pair(tbase, kTmemCols);
    else tmem_dealloc(tbase, kTmemCols);
  }
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

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, 128-byte swizzle
// (or the given one).
int make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_cols,
             uint32_t box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
             CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return OCCULT_ERR_CUDA;
  const int esize = dtype == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : 2;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dtype, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OCCULT_OK : OCCULT_ERR_CUDA;
}

// SwiGLU weights [Ne, 2I, K] (gate rows then up rows of every expert) as a 5-D
// tensor (K, 16 rows, gate/up, I/16 groups, expert); box (64, 16, 2, 4, 1):
// 4 groups of 16 gate rows each followed by the same units' up rows.
int make_map_swiglu5d(CUtensorMap* m, const void* base, int64_t n_exp, int64_t I, int64_t K) {
  auto fn = encode_fn();
  if (!fn || I % 64 != 0) return fn ? OCCULT_ERR_UNSUPPORTED : OCCULT_ERR_CUDA;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(K), 16, 2, static_cast<cuuint64_t>(I / 16),
                              static_cast<cuuint64_t>(n_exp)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(I * K) * 2,
                                 static_cast<cuuint64_t>(16 * K) * 2,
                                 static_cast<cuuint64_t>(2 * I * K) * 2};
  const cuuint32_t box[5] = {BK, 16, 2, 4, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OCCULT_OK : OCCULT_ERR_CUDA;
}

// Tensor map of one operand: K-major tiles are 64 K columns x 128 or 256 rows;
// MN-major tiles are loaded as 64 MN columns x 64 K rows.
int operand_map(CUtensorMap* m, int mode, const void* ptr, int64_t rows, int64_t cols,
                uint32_t k_major_rows) {
  if (mode == OP_TMA_K) return make_map(m, ptr, rows, cols, BK, k_major_rows);
  if (mode == OP_TMA_MN) return make_map(m, ptr, rows, cols, 64, BK);
  // MN-major gathers: tile::gather4 of 64-column rows (the box is one row high)
  if (mode == OP_GATHER_MN) return make_map(m, ptr, rows, cols, 64, 1);
  // K-major gathers are copied by cp.async: a valid placeholder map
  return make_map(m, ptr, rows, cols, BK, BK);
}

template <int AM, int BMODE, int EPI, bool WGRAD, bool PAIR, bool SWAP = false>
int launch_tc(const LaunchCtx& ctx, const CUtensorMap& ma, const CUtensorMap& mb,
              const CUtensorMap& mc, const CUtensorMap& md, const Params& p) {
  auto kern = grouped_gemm_tc_kernel<AM, BMODE, EPI, WGRAD, PAIR, SWAP>;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3(threads_for(AM, BMODE, copies_a(AM, EPI, WGRAD, SWAP)));
  cfg.dynamicSmemBytes = smem_bytes(PAIR, EPI, SWAP);
  cfg.stream = ctx.stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = PAIR ? attr : attr + 1;
  cfg.numAttrs = PAIR ? 2 : 1;
  // persistent grid: one CTA per SM, or as many co-resident CTA pairs as fit
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int n_pairs = 0;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    smem_bytes(PAIR, EPI, SWAP));
    if (PAIR && attr_err == cudaSuccess) {
      cfg.gridDim = dim3(2 * (ctx.num_sms / 2));
      attr_err = cudaOccupancyMaxActiveClusters(&n_pairs, kern, &cfg);
    }
  });
  if (attr_err != cudaSuccess || (PAIR && n_pairs < 1)) return OCCULT_ERR_CUDA;
  cfg.gridDim = dim3(PAIR ? 2 * n_pairs : ctx.num_sms);
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, md, p));
}

}  // namespace

// Largest part of the merged down-projection's output that one window of units
// adds into.  On the 32768-token training shape (y: 268 MB fp32) two windows
// took the plain units from 947 to 918-930 us (swapped units 1005 -> 988 us, and
// four windows were slower than two: each window reads W_d again).  The dgrad through [W_g; W_u]
// re-reads twice the weights and ran slower with windows (1455 us; 1484 with
// two, 1543 with four): it keeps one.
constexpr int64_t kMergeWindowBytes = int64_t(160) << 20;

int launch_grouped_gemm_bf16(const LaunchCtx& ctx, const GroupedGemm& g) {
  if (g.n_seg > kMaxSeg || g.N_out % 32 != 0) return OCCULT_ERR_UNSUPPORTED;
  if (!g.wgrad && g.K % BK != 0) return OCCULT_ERR_UNSUPPORTED;
  // the epilogues write (or add) 16-byte vectors along output rows
  if (reinterpret_cast<uintptr_t>(g.out) % 16 != 0 || g.ldo % 8 != 0) return OCCULT_ERR_UNSUPPORTED;
  if (g.n_seg == 0 || (!g.wgrad && g.max_rows == 0)) return OCCULT_OK;
  // Forward and dgrad GEMMs run on CTA pairs (one 256 x 256 tile per pair, each
  // CTA holding 128 rows of B), gathered A rows included: each CTA gathers its
  // own 128 rows with cp.async and the odd CTA forwards its stages' completion
  // to the even CTA's barrier with a CTA-scope release (a cluster-scope release
  // there cost ~1 us per stage and made the pair 2.5x slower than one CTA).  TMA
  // tile::gather4 (one instruction per four 128-byte rows) measured 2.6x slower
  // than cp.async on single CTAs.
  // A pair works on two M tiles of one segment at a time: segments shorter than
  // that (decode-sized batches, ~50 rows an expert) leave half of each pair idle
  // and run faster on single CTAs.
  const int am = g.a_mode;
  const int64_t avg_rows = g.seg_off ? g.max_rows / g.n_seg : g.max_rows;
  const bool pair = g.wgrad ? g.M_total % (2 * BM) == 0
                            : !op_gathered(g.b_mode) && avg_rows >= 2 * BM;
  // Paired routed forward GEMMs swap operands (weights on M, the segment's rows on
  // N) so that a segment's last unit computes its rows rounded up to 16, not to
  // 256 (decode-sized segments stay on single CTAs: a swapped pair measured
  // slower there, 164 vs 135 us for the DeepSeek decode up-projection).
  const int epi_eff = g.epi == EPI_F32 && g.out_tok ? EPI_F32_RED
                    : (g.epi == EPI_SWIGLU && g.gu_out ? EPI_SWIGLU_SAVE : g.epi);
  // The merged down-projection keeps plain units when segments are long (~4096
  // rows an expert on the 32768-token training shape: 947 us plain against
  // 1005 us swapped, one window each), where a unit's padding is small and the
  // merge epilogue needs no transpose.
  const bool swap = pair && !g.wgrad && g.seg_off && g.b_mode == OP_TMA_K &&
                    ((epi_eff == EPI_SWIGLU && g.a_mode == OP_GATHER_K && !g.gu_out) ||
                     ((epi_eff == EPI_F32 || (epi_eff == EPI_F32_RED && avg_rows < 2048)) &&
                      g.a_mode == OP_TMA_K));
  CUtensorMap ma, mb;
  int rc = operand_map(&ma, am, g.A, g.a_rows, g.a_cols, BM);
  if (rc) return rc;
  // B (weights) boxes: pairs and SwiGLU halves 128 rows, single CTAs 256;
  // swapped SwiGLU a 5-D view of [Ne, 2, I/16, 16, d] taking 4 groups of 16 gate
  // rows and their 16 up rows at once
  if (swap && g.epi == EPI_SWIGLU)
    rc = make_map_swiglu5d(&mb, g.B, g.n_groups, g.N_out, g.b_cols);
  else
    rc = operand_map(&mb, g.b_mode, g.B, g.b_rows, g.b_cols,
                     (pair || g.epi == EPI_SWIGLU) ? BN / 2 : BN);
  if (rc) return rc;
  // the SwiGLU backward's G|U (in) and dG|dU (out): [rows, 2 N_out] bf16, boxes of
  // 32 columns x 32 rows with the 64-byte swizzle; unused (zero) otherwise
  CUtensorMap mc{}, md{};
  if (epi_eff == EPI_SWIGLU_BWD) {
    if (reinterpret_cast<uintptr_t>(g.gu_in) % 16 != 0) return OCCULT_ERR_UNSUPPORTED;
    rc = make_map(&mc, g.gu_in, g.max_rows, 2ll * g.N_out, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!rc) rc = make_map(&md, g.out, g.max_rows, g.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc) return rc;
  }
  // the padded EPD copy of the gathered A rows ([rows + OCCULT_EPD_PAD * segments,
  // K] bf16) is written in 16-byte pieces
  if (g.a_copy && (!copies_a(g.a_mode, epi_eff, g.wgrad, swap) || !g.seg_off ||
                   reinterpret_cast<uintptr_t>(g.a_copy) % 16 != 0))
    return OCCULT_ERR_UNSUPPORTED;
  Params p{};
  p.seg_off = g.seg_off;
  p.seg_group = g.seg_group;
  p.n_seg = g.n_seg;
  // The merges add into an fp32 output of out_rows x N_out that need not fit in
  // L2: each segment's rows (token order) are split into windows visited
  // window-major, so that the rows being added to at a time span about
  // 1 / n_win of the tokens (at the price of reading the weights n_win times).
  // Only the down-projection's merge (weights K-major, W_d) takes windows.
  p.n_win = 1;
  if (epi_eff == EPI_F32_RED && g.seg_off && g.out_rows > 0 && g.b_mode == OP_TMA_K) {
    const int64_t out_bytes = g.out_rows * g.N_out * 4;
    const int64_t want = (out_bytes + kMergeWindowBytes - 1) / kMergeWindowBytes;
    p.n_win = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, kMaxSeg / g.n_seg)));
  }
  p.single_rows = static_cast<int>(g.max_rows);
  p.K = g.K;
  p.N_out = g.N_out;
  p.M_total = g.M_total;
  p.n_tiles_m = (g.M_total + BM - 1) / BM;
  const int tile_n = g.epi == EPI_SWIGLU ? BN / 2 : BN;
  p.n_tiles_n = (g.N_out + tile_n - 1) / tile_n;
  p.gather = g.gather;
  const bool a_gathered = op_gathered(g.a_mode);
  p.g_ptr = static_cast<const __nv_bfloat16*>(a_gathered ? g.A : g.B);
  p.g_ld = a_gathered ? g.a_cols : g.b_cols;
  p.g_rows = static_cast<int>(a_gathered ? g.a_rows : g.b_rows);
  p.b_group_rows = g.b_group_rows;
  p.a_pad = g.a_pad;
  p.b_pad = g.b_pad;
  p.a_copy = static_cast<__nv_bfloat16*>(g.a_copy);
  p.half_n = g.epi == EPI_SWIGLU ? g.N_out : (g.epi == EPI_SWIGLU_BWD ? g.N_out : 0);
  p.row_gate = g.row_gate;
  p.out = g.out;
  p.ldo = g.ldo;
  p.out_group_stride = g.out_group_stride;
  p.gu_out = static_cast<__nv_bfloat16*>(g.gu_out);
  p.gu_in = static_cast<const __nv_bfloat16*>(g.gu_in);
  p.dg_part = g.dg_part;
  p.out_src = g.out_src;
  p.out_tok = g.out_tok;
  p.dev_err = ctx.dev_err;
  const int bm = g.b_mode, ep = epi_eff;
  // the instantiations the layer uses
#define OCCULT_ROWS_GEMM(AM_, BM_, EP_)                                                 \
  if (am == AM_ && bm == BM_ && ep == EP_)                                             \
    return pair ? launch_tc<AM_, BM_, EP_, false, true>(ctx, ma, mb, mc, md, p)                \
                : launch_tc<AM_, BM_, EP_, false, false>(ctx, ma, mb, mc, md, p);
  if (swap) {
    if (am == OP_GATHER_K && ep == EPI_SWIGLU)
      return launch_tc<OP_GATHER_K, OP_TMA_K, EPI_SWIGLU, false, true, true>(ctx, ma, mb, mc, md, p);
    if (am == OP_TMA_K && ep == EPI_F32)
      return launch_tc<OP_TMA_K, OP_TMA_K, EPI_F32, false, true, true>(ctx, ma, mb, mc, md, p);
    if (am == OP_TMA_K && ep == EPI_F32_RED)
      return launch_tc<OP_TMA_K, OP_TMA_K, EPI_F32_RED, false, true, true>(ctx, ma, mb, mc, md, p);
  }
  if (!g.wgrad) {
    OCCULT_ROWS_GEMM(OP_GATHER_K, OP_TMA_K, EPI_SWIGLU)     // up-projection
    OCCULT_ROWS_GEMM(OP_GATHER_K, OP_TMA_K, EPI_SWIGLU_SAVE)  // the same, G|U saved
    OCCULT_ROWS_GEMM(OP_TMA_K, OP_TMA_K, EPI_SWIGLU)        // shared experts' up-projection
    OCCULT_ROWS_GEMM(OP_TMA_K, OP_TMA_K, EPI_F32)           // down-projections
    OCCULT_ROWS_GEMM(OP_TMA_K, OP_TMA_K, EPI_F32_RED)       // down-projection + merge
    OCCULT_ROWS_GEMM(OP_GATHER_K, OP_TMA_MN, EPI_SWIGLU_BWD)  // dgrad through W_d
    OCCULT_ROWS_GEMM(OP_TMA_K, OP_TMA_MN, EPI_SWIGLU_BWD)     // the same, dy rows in EPD order
    OCCULT_ROWS_GEMM(OP_TMA_K, OP_TMA_MN, EPI_F32)          // dgrad through [W_g; W_u]
    OCCULT_ROWS_GEMM(OP_TMA_K, OP_TMA_MN, EPI_F32_RED)      // the same + merge of dx
#undef OCCULT_ROWS_GEMM
  } else if (ep == EPI_F32) {
    if (am == OP_GATHER_MN && bm == OP_TMA_MN)
      return pair ? launch_tc<OP_GATHER_MN, OP_TMA_MN, EPI_F32, true, true>(ctx, ma, mb, mc, md, p)
                  : launch_tc<OP_GATHER_MN, OP_TMA_MN, EPI_F32, true, false>(ctx, ma, mb, mc, md, p);
    if (am == OP_TMA_MN && bm == OP_GATHER_MN)
      return pair ? launch_tc<OP_TMA_MN, OP_GATHER_MN, EPI_F32, true, true>(ctx, ma, mb, mc, md, p)
                  : launch_tc<OP_TMA_MN, OP_GATHER_MN, EPI_F32, true, false>(ctx, ma, mb, mc, md, p);
    // both operands as tiles: one of them the padded EPD copy of the rows
    if (am == OP_TMA_MN && bm == OP_TMA_MN)
      return pair ? launch_tc<OP_TMA_MN, OP_TMA_MN, EPI_F32, true, true>(ctx, ma, mb, mc, md, p)
                  : launch_tc<OP_TMA_MN, OP_TMA_MN, EPI_F32, true, false>(ctx, ma, mb, mc, md, p);
  }
  return OCCULT_ERR_UNSUPPORTED;
}

}  // namespace occult
