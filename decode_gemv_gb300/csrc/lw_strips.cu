// lw_decode_gemm_strips: the fused 4-/6-bit product over a list of 64-row
// strips (tile-skip launch list): the table-driven kernel when the bundle's
// table fits it, else the strip-list instantiations of q_product_kernel,
// which live in this translation unit.
#include "lw_qlaunch.h"

using namespace lw;

extern "C" lw_status lw_decode_gemm_strips(const lw_dev_bundle* b, const int32_t* strips,
                                           int32_t n_strips, const void* X, int32_t batch, float* Y,
                                           void* ws, size_t ws_bytes, int32_t* d_status,
                                           void* stream) {
  clear_error();
  lw_status s = check_dev_bundle(b, false, true);
  if (s != LW_OK) return s;
  if (b->fmt == LW_FMT_BF16_EXP) return fail(LW_ERR_UNSUPPORTED, "strip lists take 4-/6-bit bundles");
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!X || !Y || !ws || !a16(X) || !a16(ws) || (reinterpret_cast<uintptr_t>(Y) & 7u))
    return fail(LW_ERR_INVALID_ARG, "X, Y, workspace missing or misaligned");
  if (batch < 1 || batch > 256) return fail(LW_ERR_INVALID_ARG, "batch %d outside 1..256", batch);
  if (n_strips < 0 || n_strips > b->rows / 64 || (n_strips > 0 && !strips) ||
      (reinterpret_cast<uintptr_t>(strips) & 3u))
    return fail(LW_ERR_INVALID_ARG, "strip list of %d entries (at most %lld)", n_strips,
                (long long)(b->rows / 64));
  const int pass = batch < 8 ? batch : 8;
  if (ws_bytes < workspace_counter_bytes(b) + workspace_partials_bytes(b, pass))
    return fail(LW_ERR_INVALID_ARG, "workspace of %zu bytes too small", ws_bytes);
  if ((long long)n_strips * (b->cols / 256) > (1ll << 30)) return fail(LW_ERR_SHAPE, "too many tiles");
  if (n_strips == 0) return LW_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* xf = static_cast<const float*>(X);
  for (int b0 = 0; b0 < batch; b0 += 8) {
    const int nb = batch - b0 < 8 ? batch - b0 : 8;
    const float* xp = xf + (size_t)b0 * b->cols;
    float* yp = Y + (size_t)b0 * b->rows;
    void* wp = ws;
    s = lut_takes(&b, 1, nb) ? launch_q_lut(&b, 1, &xp, nb, &yp, &wp, d_status, st, strips, n_strips)
                    : q_products_impl<true>(&b, 1, &xp, nb, &yp, &wp, strips, n_strips, d_status, st);
    if (s != LW_OK) return s;
  }
  return LW_OK;
}
