// Expert placement rescheduling: Occult paper Sec. 3.2, Algorithm 1, on the host.
//
// A greedy, farthest-point-style split of the co-activation graph into Nd
// equal device lists.  Device 0 opens with the most collaborative pair
// (largest off-diagonal count, first in row-major order); every later device
// opens with the unused expert least collaborative with all experts placed so
// far; each device then keeps taking the unused expert most collaborative with
// its own experts until it holds Ne/Nd.  The paper compares means of the
// normalised graph P = C / max C; every candidate shares the denominator and P
// is C up to a positive factor, so comparing integer sums of C gives the same
// choices exactly.  Ties go to the lowest expert id.  With Ne/Nd = 1 device 0
// keeps only the first expert of the pair.
#include <stdint.h>

#include <vector>

#include "../../include/occult.h"

extern "C" int occult_place(const int64_t* C, int32_t n_experts, int32_t n_vdev,
                            int32_t* placement, int32_t* expert_to_vdev) {
  if (!C || !placement || !expert_to_vdev) return OCCULT_ERR_INVALID_ARG;
  if (n_experts <= 0 || n_vdev <= 0 || n_experts % n_vdev != 0) return OCCULT_ERR_INVALID_ARG;
  const int Ne = n_experts, Nd = n_vdev, n_loc = Ne / Nd;
  std::vector<char> used(Ne, 0);
  std::vector<int> placed;          // every expert placed so far, in order
  std::vector<std::vector<int>> L(Nd);
  auto take = [&](int d, int e) {
    L[d].push_back(e);
    placed.push_back(e);
    used[e] = 1;
  };
  for (int d = 0; d < Nd; ++d) {
    if (d == 0) {
      int bi = -1, bj = -1;
      for (int i = 0; i < Ne; ++i)
        for (int j = 0; j < Ne; ++j)
          if (i != j && (bi < 0 || C[(int64_t)i * Ne + j] > C[(int64_t)bi * Ne + bj])) bi = i, bj = j;
      if (bi < 0) bi = 0, bj = -1;  // single expert
      take(0, bi);
      if (n_loc >= 2 && bj >= 0) take(0, bj);
    } else {
      int best = -1;
      int64_t best_v = 0;
      for (int e = 0; e < Ne; ++e) {
        if (used[e]) continue;
        int64_t v = 0;
        for (int t : placed) v += C[(int64_t)t * Ne + e];
        if (best < 0 || v < best_v) best = e, best_v = v;
      }
      take(d, best);
    }
    while (static_cast<int>(L[d].size()) < n_loc) {
      int best = -1;
      int64_t best_v = 0;
      for (int e = 0; e < Ne; ++e) {
        if (used[e]) continue;
        int64_t v = 0;
        for (int t : L[d]) v += C[(int64_t)t * Ne + e];
        if (best < 0 || v > best_v) best = e, best_v = v;
      }
      take(d, best);
    }
  }
  for (int d = 0; d < Nd; ++d)
    for (int j = 0; j < n_loc; ++j) {
      placement[d * n_loc + j] = L[d][j];
      expert_to_vdev[L[d][j]] = d;
    }
  return OCCULT_OK;
}
