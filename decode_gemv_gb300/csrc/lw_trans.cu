// lw_transcode_twin: launcher of the load-time transcode (lw_trans.cuh).
#include "lw_internal.h"
#include "lw_launch.h"
#include "lw_trans.cuh"

namespace lw {
namespace {

using TKernel = void (*)(const dev::TArgs);

template <int FMT>
TKernel pick(int span) {
  if (span <= 4) return dev::t_transcode_kernel<FMT, 4>;
  if (span <= 8) return dev::t_transcode_kernel<FMT, 8>;
  return dev::t_transcode_kernel<FMT, 10>;
}

int twin_width(int fmt) { return fmt == LW_FMT_Q6 ? 6 : 4; }

}  // namespace
}  // namespace lw

using namespace lw;

extern "C" int32_t lw_twin_tile_rows(int32_t fmt) {
  if (fmt != LW_FMT_Q4_PAIR && fmt != LW_FMT_Q6 && fmt != LW_FMT_BF16_EXP) return 0;
  return 512 * twin_width(fmt) / 32;
}

extern "C" lw_status lw_transcode_twin(const lw_dev_bundle* coded, const lw_dev_bundle* twin,
                                       int32_t* d_status, void* stream) {
  clear_error();
  lw_status s = check_dev_bundle(coded, false, false);
  if (s != LW_OK) return s;
  if (coded->twin) return fail(LW_ERR_INVALID_ARG, "source must be a coded bundle");
  if (!twin) return fail(LW_ERR_INVALID_ARG, "NULL twin view");
  if (!twin->twin || twin->fmt != coded->fmt || twin->rows != coded->rows || twin->cols != coded->cols)
    return fail(LW_ERR_INVALID_ARG, "twin view must be a twin of the same format and shape");
  if (twin->max_tile_rows != lw_twin_tile_rows(coded->fmt))
    return fail(LW_ERR_INVALID_ARG, "twin max_tile_rows must be %d", lw_twin_tile_rows(coded->fmt));
  if (!twin->words || !twin->tile_off || !twin->lane_bits ||
      (reinterpret_cast<uintptr_t>(twin->words) & 15u) || (reinterpret_cast<uintptr_t>(twin->tile_off) & 3u) ||
      (reinterpret_cast<uintptr_t>(twin->lane_bits) & 1u))
    return fail(LW_ERR_INVALID_ARG, "twin words (16-byte aligned), tile_off and lane_bits required");
  if (coded->fmt == LW_FMT_BF16_EXP && !coded->vflags)
    return fail(LW_ERR_INVALID_ARG, "BF16 bundle without verbatim flags");
  const int64_t n_tiles = tiles_of(coded->rows, coded->cols);
  const int R2 = lw_twin_tile_rows(coded->fmt);
  // the twin's words must not overlap the coded sections the kernel reads
  const char* w0 = reinterpret_cast<const char*>(twin->words);
  const char* w1 = w0 + (size_t)n_tiles * R2 * 128;
  auto overlaps = [&](const void* p, size_t n) {
    const char* a = static_cast<const char*>(p);
    return p && a < w1 && w0 < a + n;
  };
  if (overlaps(coded->words, 1) || overlaps(coded->lane_mid, (size_t)n_tiles * 64) ||
      overlaps(coded->table, sizeof(lw_table)) || overlaps(coded->tile_off, (size_t)(n_tiles + 1) * 4))
    return fail(LW_ERR_INVALID_ARG, "twin words overlap the coded bundle");

  dev::TArgs a{};
  a.words = coded->words;
  a.tile_off = coded->tile_off;
  a.lane_bits = coded->lane_bits;
  a.lane_mid = coded->lane_mid;
  a.table = coded->table;
  a.vflags = coded->vflags;
  a.tw_words = const_cast<uint32_t*>(twin->words);
  a.tw_tile_off = const_cast<uint32_t*>(twin->tile_off);
  a.tw_lane_bits = const_cast<uint16_t*>(twin->lane_bits);
  a.status = d_status;
  a.n_tiles = (int)n_tiles;
  a.TK = (int)(coded->cols / 256);
  a.GW = (int)((coded->cols / 64 + 31) / 32);
  a.stage_rows = coded->max_tile_rows + dev::kLookahead;
  a.mid_offset = a.stage_rows * 128;
  a.stage_bytes = (a.mid_offset + 64 + 127) / 128 * 128;
  const int span = coded->lmax - coded->lmin;
  TKernel k = coded->fmt == LW_FMT_Q4_PAIR ? pick<LW_FMT_Q4_PAIR>(span)
              : coded->fmt == LW_FMT_Q6    ? pick<LW_FMT_Q6>(span)
                                           : pick<LW_FMT_BF16_EXP>(span);
  const size_t smem = (size_t)dev::kStageOff + 2 * (size_t)a.stage_bytes;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // plain stream order (no programmatic serialisation): the twin buffers may
  // still be read by the previous kernel
  lw_status r = launch_persistent((const void*)k, dev::kQThreads, smem, a.n_tiles, st,
                                  [&](int blocks) { k<<<blocks, dev::kQThreads, smem, st>>>(a); });
  if (r != LW_OK) return r;
  // and a plain-order kernel after it: the next call's kernels read bundle
  // sections before their programmatic wait, so they must not start before
  // the twin is complete
  dev::t_order_kernel<<<1, 1, 0, st>>>();
  return check_launch("transcode order kernel");
}
