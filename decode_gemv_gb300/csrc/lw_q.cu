// Launchers for the 4-/6-bit kernels (instantiations of lw_qkern.cuh).
#include <mutex>
#include <unordered_map>

#include "lw_internal.h"
#include "lw_launch.h"
#include "lw_qkern.cuh"
#include "lw_qtc.cuh"
#include "lw_qlaunch.h"

namespace lw {

static_assert(LW_MAX_GROUP == dev::kMaxGroup, "group size");

namespace {

using QKernel = void (*)(const dev::QArgs);

template <int FMT, bool TWIN>
QKernel pick_decode(int ncmp) {
  if (TWIN) return dev::q_decode_kernel<FMT, true, 0>;
  switch (ncmp) {
    case 4: return dev::q_decode_kernel<FMT, false, 4>;
    case 7: return dev::q_decode_kernel<FMT, false, 7>;
    case 8: return dev::q_decode_kernel<FMT, false, 8>;
    default: return dev::q_decode_kernel<FMT, false, 10>;
  }
}

template <int FMT>
QKernel pick_tc(int ncmp) {
  switch (ncmp) {
    case 4: return dev::q_tc_kernel<FMT, 4>;
    case 7: return dev::q_tc_kernel<FMT, 7>;
    case 8: return dev::q_tc_kernel<FMT, 8>;
    default: return dev::q_tc_kernel<FMT, 10>;
  }
}

}  // namespace

lw_status launch_q_tc_product(const lw_dev_bundle* b, const float* x, int batch, float* y, void* ws,
                              int32_t* status, cudaStream_t st) {
  const int fmt = b->fmt;
  const int ncmp = ncmp_bucket(b->lmax - b->lmin);
  QKernel k = fmt == LW_FMT_Q4_PAIR ? pick_tc<dev::kQ4>(ncmp) : pick_tc<dev::kQ6>(ncmp);
  dev::QArgs a{};
  a.words = b->words;
  a.tile_off = b->tile_off;
  a.lane_bits = b->lane_bits;
  a.lane_mid = b->lane_mid;
  a.table = b->table;
  a.qparams = static_cast<const uint8_t*>(b->qparams);
  a.x = x;
  a.ws = workspace_partials(b, ws);
  a.counters = workspace_counters(b, ws);
  a.y = y;
  a.status = status;
  a.TK = (int)(b->cols / 256);
  a.N = (int)b->rows;
  a.K = (int)b->cols;
  a.n_tiles = (int)tiles_of(b->rows, b->cols);
  a.batch = batch;
  a.stage_rows = b->max_tile_rows + dev::kLookahead;
  // stage: coded rows | scales (and mins) | lane_mid
  a.mid_offset = a.stage_rows * 128 + qparam_tile_bytes(fmt);
  a.stage_bytes = (a.mid_offset + 64 + 127) / 128 * 128;
  a.bpad = (batch + 15) / 16 * 16;
  const int need = dev::qt_tmem_need(a.bpad);
  a.tmem_cols = need <= 32 ? 32 : (need <= 64 ? 64 : (need <= 128 ? 128 : 256));
  // header | X^T halves (2 x 2 bpad x 256 B) | tile stages (4 strips x 1 or
  // 2): two stages per strip unless one stage lets more CTAs reside
  a.xs_off = dev::kQtXsOff;
  a.wstage_off = a.xs_off + 2 * a.bpad * 512;
  size_t smem2 = (size_t)a.wstage_off + 8 * (size_t)a.stage_bytes;
  size_t smem1 = (size_t)a.wstage_off + 4 * (size_t)a.stage_bytes;
  const int per_sm2 = tc_resident_blocks((const void*)k, dev::kQtThreads, smem2, a.tmem_cols);
  const int per_sm1 = tc_resident_blocks((const void*)k, dev::kQtThreads, smem1, a.tmem_cols);
  a.nstage = per_sm1 > per_sm2 ? 1 : 2;
  const int per_sm = a.nstage == 1 ? per_sm1 : per_sm2;
  const size_t smem = a.nstage == 1 ? smem1 : smem2;
  if (per_sm < 1) return fail(LW_ERR_UNSUPPORTED, "tensor-core kernel does not fit (%zu B smem)", smem);
  const int n_blocks = (int)((b->rows / 64 + 3) / 4);
  const TcGrid g = tc_pick_grid(n_blocks, a.TK, tc_max_split(b), per_sm * device_sm_count());
  launch_pdl(k, g.G, dev::kQtThreads, smem, st, a);
  lw_status s = check_launch("tensor-core product kernel");
  if (s == LW_OK && g.owners > 1) s = launch_tc_sum(a.ws, y, (int)b->rows, batch, a.TK, g.G, st);
  return s;
}

// Fused products of n matrices of one format (one launch): matrix i reads
// x[i] (`batch` rows), writes y[i] and uses workspace ws[i].
// The table-driven kernel when it takes the launch (lut_takes), else the
// comparator kernel (any table, any batch).
lw_status launch_q_products(const lw_dev_bundle* const* bs, int n, const float* const* x, int batch,
                            float* const* y, void* const* ws, int32_t* status, cudaStream_t st) {
  if (lut_takes(bs, n, batch)) return launch_q_lut(bs, n, x, batch, y, ws, status, st);
  return q_products_impl<false>(bs, n, x, batch, y, ws, nullptr, 0, status, st);
}

lw_status launch_q_product(const lw_dev_bundle* b, const float* x, int batch, float* y, void* ws,
                           int32_t* status, cudaStream_t st) {
  return launch_q_products(&b, 1, &x, batch, &y, &ws, status, st);
}

lw_status launch_q_decode(const lw_dev_bundle* b, void* out, int32_t* status, cudaStream_t st) {
  const int fmt = b->fmt;
  const bool twin = b->twin != 0;
  const int ncmp = twin ? 0 : ncmp_bucket(b->lmax - b->lmin);
  QKernel k;
  if (fmt == LW_FMT_Q4_PAIR)
    k = twin ? pick_decode<dev::kQ4, true>(ncmp) : pick_decode<dev::kQ4, false>(ncmp);
  else
    k = twin ? pick_decode<dev::kQ6, true>(ncmp) : pick_decode<dev::kQ6, false>(ncmp);
  dev::QArgs a{};
  a.words = b->words;
  a.tile_off = b->tile_off;
  a.lane_bits = b->lane_bits;
  a.lane_mid = twin ? nullptr : b->lane_mid;
  a.table = b->table;
  a.out = static_cast<uint8_t*>(out);
  a.status = status;
  a.TK = (int)(b->cols / 256);
  a.N = (int)b->rows;
  a.K = (int)b->cols;
  a.n_tiles = (int)tiles_of(b->rows, b->cols);
  a.stage_rows = b->max_tile_rows + dev::kLookahead;
  a.mid_offset = a.stage_rows * 128;
  a.stage_bytes = (a.mid_offset + 64 + 127) / 128 * 128;
  const size_t smem = (size_t)dev::kStageOff + 2 * (size_t)a.stage_bytes;
  return launch_persistent((const void*)k, dev::kQThreads, smem, a.n_tiles, st, [&](int blocks) {
    launch_pdl(k, blocks, dev::kQThreads, smem, st, a);
  });
}

}  // namespace lw
