// Work split of the tensor-core product kernels (b_tc_kernel, q_tc_kernel)
// and of the split-K sum behind them.  Host and device share it: the host
// picks the grid, the kernels find their ranges and the owners of a row
// block.  Plain C++ apart from the __host__ __device__ marks, so that the
// host logic also builds (and is tested) without the CUDA compiler.
//
// The launch's T = row blocks x TK tile columns (row block major) go to its
// G CTAs in contiguous ranges, CTA c taking [c T / G, (c + 1) T / G) -- a
// "stream-K" cut: every CTA gets within one tile column of the same work,
// and a range may run on into the next row block.  A row block's partial
// sums come from the CTAs owning its tile columns, numbered from the first
// of them; the sum adds them in that order.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define LW_TC_HD __host__ __device__ __forceinline__
#else
#define LW_TC_HD inline
#endif

namespace lw {

// The CTA owning tile column x (0 <= x < T, 1 <= G <= T): the largest c with
// floor(c T / G) <= x.
LW_TC_HD int tc_owner(long long x, long long T, int G) {
  return (int)(((x + 1) * G + T - 1) / T) - 1;
}

// CTAs whose ranges hold tile columns of row block rb.
LW_TC_HD int tc_owners_of(int rb, int TK, long long T, int G) {
  const long long xb = (long long)rb * TK;
  return tc_owner(xb + TK - 1, T, G) - tc_owner(xb, T, G) + 1;
}

struct TcGrid {
  int G;        // CTAs
  int owners;   // most CTAs of one row block (1: no split-K sum)
};

// The grid of a launch over n_blocks row blocks of TK tile columns on
// `slots` resident CTAs: among the grids tried (every resident CTA; n_blocks
// x m; T / L; one CTA) the one with the fewest tile columns on its busiest
// CTA, counting half a tile column per row block a range touches
// (accumulator read-out), whose busiest row block has at most max_split
// owners (the workspace holds max_split partials per output).  Ties keep
// the grid tried first.
inline TcGrid tc_plan(int n_blocks, int TK, int max_split, int slots) {
  const long long T = (long long)n_blocks * TK;
  const int g0 = (int)(slots < T ? slots : T);
  TcGrid best{1, 1};
  double best_cost = 1e300;
  auto consider = [&](long long Gl) {
    if (Gl < 1 || Gl > g0) return;
    const int G = (int)Gl;
    int owners = 0;
    for (int rb = 0; rb < n_blocks; ++rb) {
      const int k = tc_owners_of(rb, TK, T, G);
      if (k > owners) owners = k;
    }
    if (owners > max_split) return;
    long long segs = 1;   // most row blocks one CTA's range touches
    for (int c = 0; c < G; ++c) {
      const long long x0 = T * c / G, x1 = T * (c + 1) / G;
      const long long k = (x1 - 1) / TK - x0 / TK + 1;
      if (k > segs) segs = k;
    }
    const double cost = (double)((T + G - 1) / G) + 0.5 * (double)segs;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = TcGrid{G, owners};
    }
  };
  consider(g0);
  for (int m = 1; m <= max_split && m <= TK; ++m) consider((long long)n_blocks * m);
  for (int L = 1; L <= TK; ++L) consider(T / L);
  consider(1);
  return best;
}

// Owners of row block rb in 32-bit arithmetic, for T x (G + 1) < 2^32 (the
// split-K sum's per-thread count; equal to tc_owners_of there).
LW_TC_HD int tc_owners_of32(int rb, int TK, uint32_t T, uint32_t G) {
  const uint32_t x = (uint32_t)rb * (uint32_t)TK;
  return (int)(((x + (uint32_t)TK) * G + T - 1u) / T - ((x + 1u) * G + T - 1u) / T) + 1;
}

}  // namespace lw
