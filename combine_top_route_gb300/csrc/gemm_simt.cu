// fp32 grouped expert GEMM (CUDA cores, FFMA) for fp32 layers.
//
// Same contract as the tensor-core kernel (Algorithm 6 scattering matmul fused
// with SwiGLU and Algorithm 7 modulation, or the plain second linear layer of
// Algorithm 8), for layers whose parity bar is fp32: tcgen05 has no fp32-input
// kind, and tf32 would not meet it.  32 x 32 output tiles, K staged through
// shared memory 32 at a time, each thread owning four rows of one column.
// Also the shared-expert gate s_t = sigmoid(w_sg . x_t).
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

constexpr int TM = 32, TN = 32, TK = 32;

struct SimtParams {
  const float* A;
  const int32_t* gather;
  const float* B;
  int64_t b_group_rows;
  const int32_t* seg_off;
  const int32_t* seg_group;
  int n_seg;
  int single_rows;
  const float* row_gate;
  float* out;
  int64_t ldo;
  int N_out;
  int K;
  const int32_t* out_src;  // nullable: rows added into out[out_tok[out_src[r]]]
  const int32_t* out_tok;
};

template <bool SWIGLU>
__global__ void __launch_bounds__(256)
grouped_gemm_f32_kernel(const SimtParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sa[TM][TK + 1];
  __shared__ float sg[TN][TK + 1];
  __shared__ float su[TN][TK + 1];
  __shared__ int s_rows[TM];
  __shared__ int s_info[3];
  // locate this block's M tile among the segments
  if (threadIdx.x == 0) {
    int mt = blockIdx.x, seg = -1, m0 = 0, rows = 0;
    for (int s = 0; s < p.n_seg; ++s) {
      const int lo = p.seg_off ? p.seg_off[s] : 0;
      const int hi = p.seg_off ? p.seg_off[s + 1] : p.single_rows;
      const int tiles = (hi - lo + TM - 1) / TM;
      if (mt < tiles) {
        seg = s;
        m0 = lo + mt * TM;
        rows = min(TM, hi - m0);
        break;
      }
      mt -= tiles;
    }
    s_info[0] = seg;
    s_info[1] = m0;
    s_info[2] = rows;
  }
  __syncthreads();
  const int seg = s_info[0];
  if (seg < 0) return;
  const int m0 = s_info[1], rows = s_info[2];
  const int grp = p.seg_group ? p.seg_group[seg] : seg;
  const int n0 = blockIdx.y * TN;
  if (threadIdx.x < TM) {
    const int r = min(static_cast<int>(threadIdx.x), rows - 1);
    s_rows[threadIdx.x] = p.gather ? p.gather[m0 + r] : m0 + r;
  }
  __syncthreads();
  const int tx = threadIdx.x & 31;   // column
  const int ty = threadIdx.x >> 5;   // rows ty, ty+8, ty+16, ty+24
  const float* Bg = p.B + static_cast<int64_t>(grp) * p.b_group_rows * p.K;
  float accg[4] = {0, 0, 0, 0}, accu[4] = {0, 0, 0, 0};
  for (int k0 = 0; k0 < p.K; k0 += TK) {
    for (int i = threadIdx.x; i < TM * TK; i += 256) {
      const int r = i / TK, c = i % TK;
      sa[r][c] = (k0 + c < p.K) ? p.A[static_cast<int64_t>(s_rows[r]) * p.K + k0 + c] : 0.f;
      const int n = n0 + r;
      const bool in = n < p.N_out && k0 + c < p.K;
      sg[r][c] = in ? Bg[static_cast<int64_t>(n) * p.K + k0 + c] : 0.f;
      if (SWIGLU) su[r][c] = in ? Bg[static_cast<int64_t>(p.N_out + n) * p.K + k0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < TK; ++c) {
      const float bg = sg[tx][c];
      const float bu = SWIGLU ? su[tx][c] : 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = sa[ty + 8 * i][c];
        accg[i] = fmaf(a, bg, accg[i]);
        if (SWIGLU) accu[i] = fmaf(a, bu, accu[i]);
      }
    }
    __syncthreads();
  }
  const int n = n0 + tx;
  if (n >= p.N_out) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty + 8 * i;
    if (r >= rows) continue;
    const int64_t orow = m0 + r;
    float v = accg[i];
    if (SWIGLU) {
      const float g = p.row_gate ? p.row_gate[orow] : 1.0f;
      v = g * (v / (1.0f + expf(-v))) * accu[i];
    }
    if (p.out_tok) atomicAdd(&p.out[static_cast<int64_t>(p.out_tok[p.out_src[orow]]) * p.ldo + n], v);
    else p.out[orow * p.ldo + n] = v;
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
shared_gate_kernel(const T* __restrict__ x, const T* __restrict__ w, int ntok, int D,
                   float* __restrict__ s) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < ntok; t += gridDim.x * 8) {
    float acc = 0.f;
    for (int i = lane; i < D; i += 32) acc = fmaf(to_f32(x[static_cast<int64_t>(t) * D + i]), to_f32(w[i]), acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) s[t] = 1.0f / (1.0f + expf(-acc));
  }
}

}  // namespace

int launch_grouped_gemm_f32(const LaunchCtx& ctx, const GroupedGemm& g) {
  if (g.max_rows == 0 || g.n_seg == 0) return OCCULT_OK;
  SimtParams p;
  p.A = static_cast<const float*>(g.A);
  p.gather = g.gather;
  p.B = static_cast<const float*>(g.B);
  p.b_group_rows = g.b_group_rows;
  p.seg_off = g.seg_off;
  p.seg_group = g.seg_group;
  p.n_seg = g.n_seg;
  p.single_rows = static_cast<int>(g.max_rows);
  p.row_gate = g.row_gate;
  p.out = static_cast<float*>(g.out);
  p.ldo = g.ldo;
  p.N_out = g.N_out;
  p.K = g.K;
  p.out_src = g.out_src;
  p.out_tok = g.out_tok;
  const int64_t m_tiles = (g.max_rows + TM - 1) / TM + g.n_seg;
  dim3 grid(static_cast<unsigned>(m_tiles), (g.N_out + TN - 1) / TN);
  if (g.epi == EPI_SWIGLU) launch_pdl(grouped_gemm_f32_kernel<true>, grid, 256, 0, ctx.stream, p);
  else launch_pdl(grouped_gemm_f32_kernel<false>, grid, 256, 0, ctx.stream, p);
  return cuda_status(cudaGetLastError());
}

int launch_shared_gate(const LaunchCtx& ctx, const occult_desc_t& ds, const void* x,
                       const void* w_sg, float* s_gate) {
  if (ds.T == 0) return OCCULT_OK;
  int blocks = (ds.T + 7) / 8;
  if (blocks > ctx.num_sms * 8) blocks = ctx.num_sms * 8;
  if (ds.dtype == OCCULT_BF16)
    launch_pdl(shared_gate_kernel<__nv_bfloat16>, blocks, 256, 0, ctx.stream,
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_sg), ds.T,
        ds.d, s_gate);
  else
    launch_pdl(shared_gate_kernel<float>, blocks, 256, 0, ctx.stream,
        static_cast<const float*>(x), static_cast<const float*>(w_sg), ds.T, ds.d, s_gate);
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
