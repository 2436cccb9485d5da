// Host launch of the fused 4-/6-bit product kernel (q_product_kernel), shared
// by the plain and grouped launches (lw_q.cu) and the strip-list launch
// (lw_strips.cu), which instantiate it with and without a strip list.
#pragma once

#include "lw_internal.h"
#include "lw_launch.h"
#include "lw_qkern.cuh"

namespace lw {

// Comparator-count bucket (kernel variant) for a table's code-length span.
inline int ncmp_bucket(int span) { return span <= 4 ? 4 : (span <= 7 ? 7 : (span <= 8 ? 8 : 10)); }

using QPKernel = void (*)(const dev::QLaunch);

template <int FMT, bool TWIN, int BP, bool STRIPS>
QPKernel pick_product(int ncmp) {
  if constexpr (TWIN) {
    return dev::q_product_kernel<FMT, true, BP, 0, STRIPS>;
  } else {
    switch (ncmp) {
      case 4: return dev::q_product_kernel<FMT, false, BP, 4, STRIPS>;
      case 7: return dev::q_product_kernel<FMT, false, BP, 7, STRIPS>;
      case 8: return dev::q_product_kernel<FMT, false, BP, 8, STRIPS>;
      default: return dev::q_product_kernel<FMT, false, BP, 10, STRIPS>;
    }
  }
}

template <int FMT, bool TWIN, bool STRIPS>
QPKernel pick_product_b(int bp, int ncmp) {
  switch (bp) {
    case 1: return pick_product<FMT, TWIN, 1, STRIPS>(ncmp);
    case 2: return pick_product<FMT, TWIN, 2, STRIPS>(ncmp);
    case 4: return pick_product<FMT, TWIN, 4, STRIPS>(ncmp);
    default: return pick_product<FMT, TWIN, 8, STRIPS>(ncmp);
  }
}

// One launch of the fused product over n matrices of one format (matrix i
// reads x[i], `batch` <= 8 rows, writes y[i], workspace ws[i]); with STRIPS
// a single matrix restricted to the n_strips 64-row strips listed in the
// device array `strips` (their tiles only: a smaller grid, no traffic for
// the other strips).
template <bool STRIPS>
lw_status q_products_impl(const lw_dev_bundle* const* bs, int n, const float* const* x, int batch,
                          float* const* y, void* const* ws, const int32_t* strips, int n_strips,
                          int32_t* status, cudaStream_t st) {
  const int fmt = bs[0]->fmt;
  const bool twin = bs[0]->twin != 0;
  int span = 0, max_rows = 0;
  for (int i = 0; i < n; ++i) {
    span = bs[i]->lmax - bs[i]->lmin > span ? bs[i]->lmax - bs[i]->lmin : span;
    max_rows = bs[i]->max_tile_rows > max_rows ? bs[i]->max_tile_rows : max_rows;
  }
  const int ncmp = twin ? 0 : ncmp_bucket(span);
  const int bp = batch <= 1 ? 1 : (batch <= 2 ? 2 : (batch <= 4 ? 4 : 8));
  QPKernel k;
  if constexpr (STRIPS) {
    k = fmt == LW_FMT_Q4_PAIR ? pick_product_b<dev::kQ4, false, true>(bp, ncmp)
                              : pick_product_b<dev::kQ6, false, true>(bp, ncmp);
  } else if (fmt == LW_FMT_Q4_PAIR) {
    k = twin ? pick_product_b<dev::kQ4, true, false>(bp, ncmp)
             : pick_product_b<dev::kQ4, false, false>(bp, ncmp);
  } else {
    k = twin ? pick_product_b<dev::kQ6, true, false>(bp, ncmp)
             : pick_product_b<dev::kQ6, false, false>(bp, ncmp);
  }
  dev::QLaunch g{};
  g.n = n;
  const int stage_rows = max_rows + dev::kLookahead;
  const int qpb = qparam_tile_bytes(fmt);
  const int mid_offset = stage_rows * 128 + qpb + bp * 1024;
  const int stage_bytes = (mid_offset + 64 + 127) / 128 * 128;
  long long total = 0;
  for (int i = 0; i < n; ++i) {
    const lw_dev_bundle* b = bs[i];
    dev::QArgs& a = g.m[i];
    a.words = b->words;
    a.tile_off = b->tile_off;
    a.lane_bits = b->lane_bits;
    a.lane_mid = twin ? nullptr : b->lane_mid;
    a.table = b->table;
    a.qparams = static_cast<const uint8_t*>(b->qparams);
    a.strips = STRIPS ? strips : nullptr;
    a.x = x[i];
    a.ws = workspace_partials(b, ws[i]);
    a.counters = workspace_counters(b, ws[i]);
    a.y = y[i];
    a.status = status;
    a.TK = (int)(b->cols / 256);
    a.N = (int)b->rows;
    a.K = (int)b->cols;
    a.n_tiles = STRIPS ? n_strips * a.TK : (int)tiles_of(b->rows, b->cols);
    a.batch = batch;
    a.stage_rows = stage_rows;
    a.mid_offset = mid_offset;
    a.stage_bytes = stage_bytes;
    g.first[i] = (int)total;
    total += a.n_tiles;
  }
  if (total > (1ll << 30)) return fail(LW_ERR_SHAPE, "group too large");
  g.first[n] = (int)total;
  // one stage per CTA (the most resident CTAs) unless the grid leaves each
  // CTA three or more tiles, where prefetching the next tile pays
  const size_t smem1 = (size_t)dev::kStageOff + (size_t)stage_bytes;
  const size_t smem2 = smem1 + (size_t)stage_bytes;
  const long long blocks1 = persistent_blocks((const void*)k, dev::kQThreads, smem1, (int)total);
  const int nstage = blocks1 > 0 && total >= 3 * blocks1 ? 2 : 1;
  for (int i = 0; i < n; ++i) g.m[i].nstage = nstage;
  const size_t smem = nstage == 2 ? smem2 : smem1;
  return launch_persistent((const void*)k, dev::kQThreads, smem, (int)total, st, [&](int blocks) {
    launch_pdl(k, blocks, dev::kQThreads, smem, st, g);
  });
}

}  // namespace lw
