// Host check of the tensor-core products' work split (lw_tcplan.h), built
// with the plain C++ compiler by tests/test_tc_plan.py.  For a sweep of
// launch shapes it checks, from the definitions rather than the formulas:
//  * tc_plan's grid is within the resident CTAs and the tile columns;
//  * every CTA's range [c T / G, (c + 1) T / G) is non-empty;
//  * tc_owner(x) is the one CTA whose range holds x (brute force);
//  * every row block has tc_owners_of CTAs holding its tile columns, at most
//    the reported owners, which is at most max_split (the workspace's
//    partials per output); each such CTA's partial index c - owner(first
//    column) is below it;
//  * the 32-bit owner count equals the 64-bit one wherever it is used;
//  * the grid is no worse than every fixed split of the row blocks into
//    at most max_split equal parts (the previous scheme), under the cost
//    the plan minimises.
// Prints "ok <shapes>" or the first failure, and exits nonzero on failure.
#include <cstdio>
#include <vector>

#include "lw_tcplan.h"

static int fail(const char* what, int nb, int TK, int ms, int slots, long long x) {
  std::printf("FAIL %s: n_blocks %d TK %d max_split %d slots %d at %lld\n", what, nb, TK, ms,
              slots, x);
  return 1;
}

// the cost tc_plan minimises, recomputed from the ranges
static double cost_of(long long T, int TK, int G) {
  long long longest = 0, segs = 0;
  for (int c = 0; c < G; ++c) {
    const long long x0 = T * c / G, x1 = T * (c + 1) / G;
    if (x1 - x0 > longest) longest = x1 - x0;
    const long long k = (x1 - 1) / TK - x0 / TK + 1;
    if (k > segs) segs = k;
  }
  return (double)longest + 0.5 * (double)segs;
}

int main() {
  const int slot_list[] = {1, 2, 3, 76, 151, 152, 304, 456};
  int shapes = 0;
  for (int nb = 1; nb <= 60; nb += (nb < 8 ? 1 : 7)) {
    for (int TK = 1; TK <= 64; TK += (TK < 6 ? 1 : 5)) {
      const int ms = TK / 2 < 1 ? 1 : (TK / 2 > 32 ? 32 : TK / 2);   // the workspace's splits
      for (int slots : slot_list) {
        ++shapes;
        const long long T = (long long)nb * TK;
        const lw::TcGrid g = lw::tc_plan(nb, TK, ms, slots);
        const int G = g.G;
        if (G < 1 || G > slots || G > T) return fail("grid size", nb, TK, ms, slots, G);
        std::vector<int> owner_of(T, -1);
        for (int c = 0; c < G; ++c) {
          const long long x0 = T * c / G, x1 = T * (c + 1) / G;
          if (x1 <= x0) return fail("empty range", nb, TK, ms, slots, c);
          for (long long x = x0; x < x1; ++x) {
            if (owner_of[x] != -1) return fail("tile column in two ranges", nb, TK, ms, slots, x);
            owner_of[x] = c;
          }
        }
        for (long long x = 0; x < T; ++x) {
          if (owner_of[x] < 0) return fail("tile column in no range", nb, TK, ms, slots, x);
          if (lw::tc_owner(x, T, G) != owner_of[x]) return fail("tc_owner", nb, TK, ms, slots, x);
        }
        int most = 0;
        for (int rb = 0; rb < nb; ++rb) {
          const long long xb = (long long)rb * TK;
          const int first = owner_of[xb];
          const int count = owner_of[xb + TK - 1] - first + 1;   // ranges are in CTA order
          for (long long x = xb; x < xb + TK; ++x) {
            const int sp = owner_of[x] - first;
            if (sp < 0 || sp >= count) return fail("partial index", nb, TK, ms, slots, x);
          }
          if (lw::tc_owners_of(rb, TK, T, G) != count) return fail("tc_owners_of", nb, TK, ms, slots, rb);
          if (T * (long long)(G + 1) < (1LL << 32) &&
              lw::tc_owners_of32(rb, TK, (uint32_t)T, (uint32_t)G) != count)
            return fail("tc_owners_of32", nb, TK, ms, slots, rb);
          if (count > most) most = count;
        }
        if (most != g.owners) return fail("reported owners", nb, TK, ms, slots, most);
        if (most > ms) return fail("owners above the workspace's splits", nb, TK, ms, slots, most);
        // no worse than any fixed split into ns <= ms equal parts that fits
        // in one wave of the resident CTAs
        const double mine = cost_of(T, TK, G);
        for (int ns = 1; ns <= ms && ns <= TK; ++ns) {
          if ((long long)nb * ns > slots) break;
          const double fixed = (double)((TK + ns - 1) / ns) + 0.5;
          if (mine > fixed + 1e-9) return fail("worse than a fixed split", nb, TK, ms, slots, ns);
        }
      }
    }
  }
  std::printf("ok %d\n", shapes);
  return 0;
}
