// Device-facing C-ABI calls of liblw: argument checks, then the launchers.
#include <cstdint>
#include <mutex>
#include <new>
#include <unordered_map>

#include "lw_internal.h"
#include "lw_launch.h"

namespace lw {

int device_sm_count() {
  static std::mutex mu;
  static int cache[128] = {0};
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 128) return 1;
  std::lock_guard<std::mutex> g(mu);
  if (!cache[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    cache[d] = n > 0 ? n : 1;
  }
  return cache[d];
}

int resident_blocks(const void* kernel, int threads, size_t smem) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> occ;           // (kernel, smem, device) -> blocks
  static std::unordered_map<uint64_t, size_t> smem_set;   // (kernel, device) -> limit set
  int d = 0;
  cudaGetDevice(&d);
  const uint64_t kd = (reinterpret_cast<uint64_t>(kernel) << 7) ^ (uint64_t)d;
  const uint64_t key = kd * 1315423911ull ^ (uint64_t)smem;
  std::lock_guard<std::mutex> g(mu);
  // the dynamic shared-memory limit of a kernel only ever grows, so a cached
  // occupancy answer stays valid for every size at or below it
  size_t& cur = smem_set[kd];
  if (smem > 48 * 1024 && smem > cur) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cur = smem;
  }
  auto it = occ.find(key);
  if (it != occ.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  occ[key] = n;
  return n;
}

int tc_resident_blocks(const void* kernel, int threads, size_t& smem, int tmem_cols) {
  int d = 0, per_sm_smem = 0, regs_sm = 65536, reserved = 1024;
  cudaGetDevice(&d);
  cudaDeviceGetAttribute(&per_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d);
  cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, d);
  cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, d);
  const int max_ctas = 512 / tmem_cols;
  const size_t floor_smem = (size_t)per_sm_smem / (size_t)(max_ctas + 1) + 1;
  if (smem < floor_smem) smem = floor_smem;
  if (resident_blocks(kernel, threads, smem) < 1) return 0;   // also raises the smem limit
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int warp_regs = ((fa.numRegs + 7) / 8 * 8 * 32 + 255) / 256 * 256;
  int per_sm = max_ctas;
  const int by_regs = regs_sm / (warp_regs * (threads / 32));
  const int by_smem = (int)((size_t)per_sm_smem / (smem + (size_t)reserved));
  per_sm = by_regs < per_sm ? by_regs : per_sm;
  per_sm = by_smem < per_sm ? by_smem : per_sm;
  return per_sm < 1 ? 1 : per_sm;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lw_status check_dev_bundle(const lw_dev_bundle* b, bool want_twin, bool product) {
  if (!b) return fail(LW_ERR_INVALID_ARG, "NULL bundle");
  if (b->fmt != LW_FMT_Q4_PAIR && b->fmt != LW_FMT_Q6 && b->fmt != LW_FMT_BF16_EXP)
    return fail(LW_ERR_UNSUPPORTED, "unknown format %d", b->fmt);
  if (b->rows <= 0 || b->cols <= 0 || b->rows % 64 || b->cols % 256)
    return fail(LW_ERR_SHAPE, "shape %lldx%lld is not a positive multiple of 64x256",
                (long long)b->rows, (long long)b->cols);
  if (b->rows > (1ll << 30) || b->cols > (1ll << 30) || tiles_of(b->rows, b->cols) > (1ll << 30))
    return fail(LW_ERR_SHAPE, "matrix too large");
  if (want_twin && !b->twin) return fail(LW_ERR_INVALID_ARG, "expected a twin bundle");
  if (!want_twin && product && b->twin) return fail(LW_ERR_INVALID_ARG, "expected a coded bundle, got a twin");
  // words may be absent only when no tile has a coded row (all verbatim)
  if ((!b->words && b->max_tile_rows > 0) || !b->tile_off || !b->lane_bits || !b->table)
    return fail(LW_ERR_INVALID_ARG, "missing words/tile_off/lane_bits/table");
  if (!b->twin && !b->lane_mid) return fail(LW_ERR_INVALID_ARG, "missing lane_mid");
  if (!aligned16(b->words) || !aligned16(b->table) || !aligned16(b->lane_mid) ||
      !aligned16(b->lane_bits))
    return fail(LW_ERR_INVALID_ARG, "words, lane_bits, table and lane_mid must be 16-byte aligned");
  if (b->max_tile_rows < 0 || b->max_tile_rows > 1024)
    return fail(LW_ERR_INVALID_ARG, "max_tile_rows %d out of range", b->max_tile_rows);
  if (!b->twin && (b->lmin < 1 || b->lmax > LW_MAX_CODE_LEN || b->lmin > b->lmax))
    return fail(LW_ERR_INVALID_ARG, "lmin/lmax %d/%d out of range", b->lmin, b->lmax);
  if (b->fmt != LW_FMT_BF16_EXP) {
    if (product && (!b->qparams || !aligned16(b->qparams)))
      return fail(LW_ERR_INVALID_ARG, "qparams missing or not 16-byte aligned");
  } else if (!b->signman || !b->vflags || !b->vrow_off || !aligned16(b->signman)) {
    // vexp may be NULL: a matrix without verbatim groups has no such section
    return fail(LW_ERR_INVALID_ARG, "BF16 side sections missing or misaligned");
  }
  return LW_OK;
}

}  // namespace lw

using namespace lw;

// Whether `rows` activation rows of a 4-/6-bit matrix go to the tensor-core
// kernel.  It gives each CTA 256 rows x a range of tile columns, so it pays
// from kQtMinRows rows on when the matrix has enough of those units to fill
// the device (about 1.5 per SM); a smaller matrix stays on the CUDA-core
// kernel (a CTA per tile) while one pass of 8 rows covers the batch.
static bool q_use_tc(const lw_dev_bundle* b, int rows) {
  if (b->twin || rows < kQtMinRows) return false;
  const long long units = ((b->rows / 64 + 3) / 4) * (long long)tc_max_split(b);
  return rows > 8 || 2 * units >= 3LL * device_sm_count();
}

extern "C" size_t lw_workspace_bytes(const lw_dev_bundle* b, int32_t batch) {
  if (!b || batch < 1 || b->rows <= 0 || b->cols <= 0) return 0;
  size_t part = workspace_partials_bytes(b, 8);
  const bool tc = b->fmt == LW_FMT_BF16_EXP ? batch >= 16 : q_use_tc(b, batch);
  if (tc && workspace_tc_bytes(b) > part) part = workspace_tc_bytes(b);
  return workspace_counter_bytes(b) + part;
}

static lw_status product(const lw_dev_bundle* b, const void* X, int32_t batch, float* Y, void* ws,
                         size_t ws_bytes, int32_t* d_status, void* stream, bool twin) {
  clear_error();
  lw_status s = check_dev_bundle(b, twin, true);
  if (s != LW_OK) return s;
  if (!X || !Y || !ws) return fail(LW_ERR_INVALID_ARG, "NULL x/y/workspace");
  if (batch < 1 || batch > 256) return fail(LW_ERR_INVALID_ARG, "batch %d outside 1..256", batch);
  if (!aligned16(X) || (reinterpret_cast<uintptr_t>(Y) & 7u) || !aligned16(ws))
    return fail(LW_ERR_INVALID_ARG, "x/workspace must be 16-byte aligned, y 8-byte aligned");
  if (ws_bytes < lw_workspace_bytes(b, batch))
    return fail(LW_ERR_INVALID_ARG, "workspace of %zu bytes < %zu", ws_bytes, lw_workspace_bytes(b, batch));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (b->fmt == LW_FMT_BF16_EXP) {
    if ((reinterpret_cast<uintptr_t>(X) & 15u) != 0)
      return fail(LW_ERR_INVALID_ARG, "x must be 16-byte aligned");
    const uint16_t* xb = static_cast<const uint16_t*>(X);
    if (batch >= 16) {   // coded and direct-palette twin alike
      // tensor cores (tcgen05) for up to 64 activation rows per launch
      for (int b0 = 0; b0 < batch; b0 += 64) {
        const int nb = batch - b0 < 64 ? batch - b0 : 64;
        s = nb >= 16 ? launch_bf16_tc_product(b, xb + (size_t)b0 * b->cols, nb,
                                              Y + (size_t)b0 * b->rows, ws, d_status, st)
                     : launch_bf16_product(b, xb + (size_t)b0 * b->cols, nb,
                                           Y + (size_t)b0 * b->rows, ws, d_status, st);
        if (s != LW_OK) return s;
      }
      return LW_OK;
    }
    return launch_bf16_product(b, xb, batch, Y, ws, d_status, st);
  }
  // tensor cores for passes of kQtMinRows..32 activation rows, CUDA cores
  // for passes of up to 8 (each pass decodes the matrix once)
  const float* xf = static_cast<const float*>(X);
  for (int b0 = 0; b0 < batch;) {
    const int left = batch - b0;
    const bool tc = q_use_tc(b, left);
    const int nb = tc ? (left < 32 ? left : 32) : (left < 8 ? left : 8);
    s = tc ? launch_q_tc_product(b, xf + (size_t)b0 * b->cols, nb, Y + (size_t)b0 * b->rows, ws,
                                 d_status, st)
           : launch_q_product(b, xf + (size_t)b0 * b->cols, nb, Y + (size_t)b0 * b->rows, ws,
                              d_status, st);
    if (s != LW_OK) return s;
    b0 += nb;
  }
  return LW_OK;
}

extern "C" lw_status lw_decode_gemv(const lw_dev_bundle* b, const void* x, float* y, void* ws,
                                    size_t ws_bytes, int32_t* d_status, void* stream) {
  return product(b, x, 1, y, ws, ws_bytes, d_status, stream, false);
}

extern "C" lw_status lw_decode_gemm(const lw_dev_bundle* b, const void* X, int32_t batch, float* Y,
                                    void* ws, size_t ws_bytes, int32_t* d_status, void* stream) {
  return product(b, X, batch, Y, ws, ws_bytes, d_status, stream, false);
}

static size_t group_slice(const lw_dev_bundle* b) {
  return (lw_workspace_bytes(b, 1) + 255) / 256 * 256;
}

extern "C" size_t lw_workspace_bytes_group(const lw_dev_bundle* const* b, int32_t n) {
  if (!b || n < 1 || n > LW_MAX_GROUP) return 0;
  size_t total = 0;
  for (int i = 0; i < n; ++i) {
    if (!b[i]) return 0;
    total += group_slice(b[i]);
  }
  return total;
}

static lw_status gemm_group(const lw_dev_bundle* const* b, int32_t n, const void* const* x,
                            int32_t batch, float* const* y, void* ws, size_t ws_bytes,
                            int32_t* d_status, void* stream, bool twin) {
  clear_error();
  if (!b || !x || !y || n < 1 || n > LW_MAX_GROUP)
    return fail(LW_ERR_INVALID_ARG, "group of %d matrices (1..%d) or NULL arrays", n, LW_MAX_GROUP);
  if (batch < 1 || batch > 8) return fail(LW_ERR_INVALID_ARG, "group batch %d outside 1..8", batch);
  if (!ws || !aligned16(ws)) return fail(LW_ERR_INVALID_ARG, "workspace NULL or not 16-byte aligned");
  const float* xs[LW_MAX_GROUP];
  float* ys[LW_MAX_GROUP];
  void* wss[LW_MAX_GROUP];
  size_t off = 0;
  for (int i = 0; i < n; ++i) {
    lw_status s = check_dev_bundle(b[i], twin, true);
    if (s != LW_OK) return s;
    if (b[i]->fmt == LW_FMT_BF16_EXP)
      return fail(LW_ERR_UNSUPPORTED, "groups take 4-/6-bit bundles");
    if (b[i]->fmt != b[0]->fmt) return fail(LW_ERR_INVALID_ARG, "mixed formats in a group");
    if (!x[i] || !y[i] || !aligned16(x[i]) || (reinterpret_cast<uintptr_t>(y[i]) & 7u))
      return fail(LW_ERR_INVALID_ARG, "matrix %d: x must be 16-byte aligned, y 8-byte aligned", i);
    xs[i] = static_cast<const float*>(x[i]);
    ys[i] = y[i];
    wss[i] = static_cast<char*>(ws) + off;
    off += group_slice(b[i]);
  }
  if (ws_bytes < off) return fail(LW_ERR_INVALID_ARG, "workspace of %zu bytes < %zu", ws_bytes, off);
  return launch_q_products(b, n, xs, batch, ys, wss, d_status, static_cast<cudaStream_t>(stream));
}

extern "C" lw_status lw_decode_gemv_group(const lw_dev_bundle* const* b, int32_t n,
                                          const void* const* x, float* const* y, void* ws,
                                          size_t ws_bytes, int32_t* d_status, void* stream) {
  return gemm_group(b, n, x, 1, y, ws, ws_bytes, d_status, stream, false);
}

extern "C" lw_status lw_twin_gemv_group(const lw_dev_bundle* const* b, int32_t n,
                                        const void* const* x, float* const* y, void* ws,
                                        size_t ws_bytes, int32_t* d_status, void* stream) {
  return gemm_group(b, n, x, 1, y, ws, ws_bytes, d_status, stream, true);
}

extern "C" lw_status lw_decode_gemm_group(const lw_dev_bundle* const* b, int32_t n,
                                          const void* const* X, int32_t batch, float* const* Y,
                                          void* ws, size_t ws_bytes, int32_t* d_status,
                                          void* stream) {
  return gemm_group(b, n, X, batch, Y, ws, ws_bytes, d_status, stream, false);
}

extern "C" lw_status lw_twin_gemm_group(const lw_dev_bundle* const* b, int32_t n,
                                        const void* const* X, int32_t batch, float* const* Y,
                                        void* ws, size_t ws_bytes, int32_t* d_status,
                                        void* stream) {
  return gemm_group(b, n, X, batch, Y, ws, ws_bytes, d_status, stream, true);
}

extern "C" lw_status lw_twin_gemv(const lw_dev_bundle* b, const void* x, float* y, void* ws,
                                  size_t ws_bytes, int32_t* d_status, void* stream) {
  return product(b, x, 1, y, ws, ws_bytes, d_status, stream, true);
}

extern "C" lw_status lw_twin_gemm(const lw_dev_bundle* b, const void* X, int32_t batch, float* Y,
                                  void* ws, size_t ws_bytes, int32_t* d_status, void* stream) {
  return product(b, X, batch, Y, ws, ws_bytes, d_status, stream, true);
}

extern "C" lw_status lw_decode(const lw_dev_bundle* b, void* out, int32_t* d_status, void* stream) {
  clear_error();
  lw_status s = check_dev_bundle(b, b ? b->twin != 0 : false, false);
  if (s != LW_OK) return s;
  if (!out || !aligned16(out)) return fail(LW_ERR_INVALID_ARG, "out must be non-NULL and 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (b->fmt == LW_FMT_BF16_EXP) return launch_bf16_decode(b, out, d_status, st);
  return launch_q_decode(b, out, d_status, st);
}

// ---------------------------------------------------------------------------
// Step graphs: a decode step's calls captured once on a stream and replayed
// (CUDA graphs; the programmatic launch dependencies become graph edges).
// ---------------------------------------------------------------------------
struct lw_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

extern "C" lw_status lw_graph_begin(void* stream) {
  clear_error();
  if (!stream) return fail(LW_ERR_INVALID_ARG, "capture needs a created stream, not the default one");
  const cudaError_t e = cudaStreamBeginCapture(static_cast<cudaStream_t>(stream),
                                               cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return fail(LW_ERR_CUDA, "begin capture: %s", cudaGetErrorString(e));
  return LW_OK;
}

extern "C" lw_status lw_graph_end(void* stream, lw_graph** out) {
  clear_error();
  if (!stream || !out) return fail(LW_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  lw_graph* g = new (std::nothrow) lw_graph;
  if (!g) return fail(LW_ERR_ALLOC, "graph");
  cudaError_t e = cudaStreamEndCapture(static_cast<cudaStream_t>(stream), &g->graph);
  if (e == cudaSuccess) e = cudaGraphInstantiate(&g->exec, g->graph, 0);
  if (e != cudaSuccess) {
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
    cudaGetLastError();
    return fail(LW_ERR_CUDA, "end capture / instantiate: %s", cudaGetErrorString(e));
  }
  *out = g;
  return LW_OK;
}

extern "C" lw_status lw_graph_launch(const lw_graph* g, void* stream) {
  clear_error();
  if (!g || !g->exec) return fail(LW_ERR_INVALID_ARG, "NULL graph");
  const cudaError_t e = cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(LW_ERR_CUDA, "graph launch: %s", cudaGetErrorString(e));
  return LW_OK;
}

extern "C" void lw_graph_free(lw_graph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}
