// Shape of the compact decode table used by the table-driven 4-/6-bit
// product kernel (lw_qlut.cuh).  Shared by the host (to pick the kernel for
// a bundle) and the device (to build the table from the staged lw_table), so
// that both sides agree.  Not part of the ABI.
//
// The decode rule is the pages' canonical one ("LazyWeights: Decode-on-Demand
// Edge LLMs", "3 . Decode on demand"): an 11-bit peek p of the stream picks
// the codeword.  Canonical codes put every code of length <= L in the peek
// range [0, limit(L)).  Instead of comparing p against the per-length limits
// one by one, the kernel looks p up in a table.  A table of all 2048 peeks is
// too large to replicate once per lane in shared memory, so it is compacted:
// codes of length <= 11 - s fill aligned blocks of 2^s peeks below
// T = limit(11 - s), where the low s peek bits do not matter; the first
// longer code, of length L1, spans the B = 2^(11 - L1) < 2^s peeks
// [T, T + B), which can share the last coarse index.  So
//     index(p) = max(p >> s, p - C),   C = T + B - T / 2^s - 1,
// is p >> s up to T + B - 1 and p - C from T + B on, and maps the peeks onto
// n = T / 2^s + 1 + (2048 - T - B) entries without losing any code (T = 2048:
// n = 2048 / 2^s).  Every 32-bit window maps to an index in [0, n).  s is
// chosen per table to make n smallest.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define LW_HD __host__ __device__ __forceinline__
#else
#define LW_HD inline
#endif

namespace lw {

// entries the kernel's shared-memory table holds (each replicated once per
// lane: 128 bytes per entry)
constexpr int kLutCap = 512;

struct LutShape {
  int s;   // low peek bits ignored below T
  int C;   // index offset of the fine region
  int T;   // first peek of the codes longer than 11 - s (2048: none)
  int n;   // entries
};

// limit(L) in 11-bit peek space from a table's lim_m1 (lim_m1[L - lmin] =
// (limit(L) << 21) - 1 for lmin <= L < lmax; every code has length <= lmax,
// so limit(lmax) = 2048).  Needs 1 <= lmin <= lmax <= 11.
LW_HD int lut_limit(const uint32_t* lim_m1, int lmin, int lmax, int L) {
  if (L < lmin) return 0;
  if (L >= lmax) return 2048;
  return (int)((lim_m1[L - lmin] + 1u) >> 21);
}

// The shape for one choice of s (1 <= s <= 10).
LW_HD LutShape lut_shape_at(const uint32_t* lim_m1, int lmin, int lmax, int s) {
  const int T = lut_limit(lim_m1, lmin, lmax, 11 - s);
  if (T >= 2048) return LutShape{s, 2048, T, 2048 >> s};
  int L1 = 12 - s;   // length of the code starting at peek T
  while (L1 < 11 && lut_limit(lim_m1, lmin, lmax, L1) <= T) ++L1;
  const int B = 1 << (11 - L1);
  return LutShape{s, T + B - (T >> s) - 1, T, (T >> s) + 1 + (2048 - T - B)};
}
// The smallest shape; among equally small ones, the one of smallest s.
LW_HD LutShape lut_shape(const uint32_t* lim_m1, int lmin, int lmax) {
  LutShape best{0, 0, 2048, 2048};
  if (lmin < 1 || lmax > 11 || lmin > lmax) return best;   // not a valid table
  for (int s = 1; s <= 10; ++s) {
    const LutShape c = lut_shape_at(lim_m1, lmin, lmax, s);
    if (c.n < best.n) best = c;
  }
  return best;
}
#if defined(__CUDACC__)
// lut_shape by one warp, lane s - 1 trying s (every lane gets the result).
__device__ __forceinline__ LutShape lut_shape_warp(const uint32_t* lim_m1, int lmin, int lmax,
                                                   int lane) {
  if (lmin < 1 || lmax > 11 || lmin > lmax) return LutShape{0, 0, 2048, 2048};
  LutShape c{0, 0, 2048, 2048};
  if (lane < 10) c = lut_shape_at(lim_m1, lmin, lmax, lane + 1);
  // smallest n, then smallest s (n <= 2048 < 2^12, s <= 10 < 2^4)
  const unsigned key = __reduce_min_sync(0xFFFFFFFFu, ((unsigned)c.n << 4) | (unsigned)c.s);
  const int src = (int)(key & 15u) - 1;   // the lane that tried the winning s (>= 0: n < 2048)
  if (src < 0) return LutShape{0, 0, 2048, 2048};
  return LutShape{__shfl_sync(0xFFFFFFFFu, c.s, src), __shfl_sync(0xFFFFFFFFu, c.C, src),
                  __shfl_sync(0xFFFFFFFFu, c.T, src), __shfl_sync(0xFFFFFFFFu, c.n, src)};
}
#endif
// The peek that table index i stands for (any peek mapping to i decodes the
// same codeword).
LW_HD int lut_peek(const LutShape& sh, int i) {
  return i < (sh.T >> sh.s) ? (i << sh.s) : i + sh.C;
}

}  // namespace lw
