// Expert similarity table of the expert-similarity-based pruning: Occult paper
// App. A.3, Eq. 6-8.  The cosine similarity of two experts' columns of the
// profiled router logits H is computed, as Eq. 8 does, from inner products that
// add up over batches of profiled tokens: the accumulator is G = H^T H (fp64),
// and the table holds sign(G_ij) G_ij^2 / (G_ii G_jj), which orders experts as
// the cosine of Eq. 6 does.
//
// Deterministic: one thread per (i, j) entry sums its batch's products in token
// order (fp32 products are exact in fp64) and adds the sum to G.
#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

__global__ void __launch_bounds__(256)
similarity_accumulate_kernel(const float* __restrict__ H, int n_tok, int Ne, double* __restrict__ G) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= Ne * Ne) return;
  const int i = e / Ne, j = e - i * Ne;
  double acc = 0.0;
  for (int t = 0; t < n_tok; ++t) {
    const float* row = H + static_cast<size_t>(t) * Ne;
    acc = fma(static_cast<double>(row[i]), static_cast<double>(row[j]), acc);
  }
  G[e] += acc;
}

__global__ void __launch_bounds__(256)
similarity_finish_kernel(const double* __restrict__ G, int Ne, float* __restrict__ table) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= Ne * Ne) return;
  const int i = e / Ne, j = e - i * Ne;
  const double g = G[e];
  const double den = G[i * Ne + i] * G[j * Ne + j];
  table[e] = den > 0.0 ? static_cast<float>(copysign(g * g / den, g)) : 0.f;
}

}  // namespace

int launch_similarity_accumulate(const LaunchCtx& ctx, int Ne, const float* logits, int n_tok,
                                 double* G) {
  if (n_tok == 0) return OCCULT_OK;
  const int n = Ne * Ne;
  launch_pdl(similarity_accumulate_kernel, (n + 255) / 256, 256, 0, ctx.stream, logits, n_tok, Ne, G);
  return cuda_status(cudaGetLastError());
}

int launch_similarity_finish(const LaunchCtx& ctx, int Ne, const double* G, float* table) {
  const int n = Ne * Ne;
  launch_pdl(similarity_finish_kernel, (n + 255) / 256, 256, 0, ctx.stream, G, Ne, table);
  return cuda_status(cudaGetLastError());
}

}  // namespace occult
