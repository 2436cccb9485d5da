// Host-side launch helpers shared by liblw's .cu files.
#pragma once

#include <cuda_runtime.h>

#include "lw_internal.h"
#include "lw_lut.h"
#include "lw_tcplan.h"

namespace lw {

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Resident blocks per SM for `kernel` with `threads` threads and `smem` bytes of
// dynamic shared memory; raises the kernel's dynamic shared-memory limit first.
// Cached per (kernel, smem).  0 if it cannot run.
int resident_blocks(const void* kernel, int threads, size_t smem);

// Launch kernel `k` with programmatic stream serialisation allowed: it may
// be scheduled while the previous kernel of the stream drains, and waits
// for it in-kernel (pdl_wait) before touching data that kernel may write.
// Errors surface through cudaGetLastError (check_launch).
template <class Arg>
inline void launch_pdl(void (*k)(Arg), int grid, int block, size_t smem, cudaStream_t st,
                       const Arg& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  (void)cudaLaunchKernelEx(&cfg, k, a);
}

inline lw_status check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(LW_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return LW_OK;
}

// Blocks of a persistent grid of `threads`-thread blocks that each own one
// tile at a time: every resident block, but no more blocks than tiles (more
// resident warps hide more of the decoder's dependency latency than an
// even tile count per block would gain).
inline long long persistent_blocks(const void* kernel, int threads, size_t smem, int n_tiles) {
  const int per_sm = resident_blocks(kernel, threads, smem);
  if (per_sm < 1) return 0;
  const long long resident = (long long)per_sm * device_sm_count();
  return resident < n_tiles ? resident : (n_tiles > 0 ? n_tiles : 1);
}

template <class Launch>
lw_status launch_persistent(const void* kernel, int threads, size_t smem, int n_tiles,
                            cudaStream_t st, Launch&& launch) {
  (void)st;
  const long long blocks = persistent_blocks(kernel, threads, smem, n_tiles);
  if (blocks < 1)
    return fail(LW_ERR_UNSUPPORTED, "kernel does not fit on an SM (%zu bytes of shared memory)",
                smem);
  launch((int)blocks);
  return check_launch("product kernel");
}

// Resident CTAs per SM of a tensor-core kernel with `threads` threads and
// `tmem_cols` tensor-memory columns per CTA, from its own budgets (registers,
// shared memory, tensor memory): the runtime's occupancy query answers 1 for
// these kernels whatever their shared memory.  Raises `smem` so that at most
// 512 / tmem_cols CTAs fit on an SM (a tensor-memory allocation then never
// waits) and the kernel's shared-memory limit to it.  0 if it cannot run.
int tc_resident_blocks(const void* kernel, int threads, size_t& smem, int tmem_cols);

// Workspace layout: one uint32 split-K counter per 64-row strip (padded to
// 256 bytes), then fp32 partial sums -- [K/256][min(batch, 8)][N] for the
// CUDA-core products, [split <= tc_max_split][64][N] for the tensor-core BF16
// product.  The counters sit first so that every path finds them at the same
// place; every call that completes leaves them at zero.
// K splits of the tensor-core product: at most one per two tile columns,
// and 32
inline int tc_max_split(const lw_dev_bundle* b) {
  const int half_tk = (int)(b->cols / 512);
  return half_tk < 1 ? 1 : (half_tk > 32 ? 32 : half_tk);
}
// Grid of a tensor-core launch over n_blocks 256-row blocks of TK tile
// columns on `slots` resident CTAs (tc_plan of lw_tcplan.h, remembered for a
// few recent shapes per host thread).
TcGrid tc_pick_grid(int n_blocks, int TK, int max_split, int slots);
// The split-K sum behind a tensor-core launch of grid G (owners > 1):
// y[b][n] = sum of ws[j][b][n] over the owners j of n's row block in
// ascending order; row blocks of one owner were written by the product and
// are skipped (one launch, programmatic dependent launch on `st`).
lw_status launch_tc_sum(const float* ws, float* y, int N, int batch, int TK, int G, cudaStream_t st);
inline size_t workspace_counter_bytes(const lw_dev_bundle* b) {
  return ((size_t)(b->rows / 64) * sizeof(uint32_t) + 255) / 256 * 256;
}
inline size_t workspace_partials_bytes(const lw_dev_bundle* b, int batch) {
  const size_t chunk = batch > 8 ? 8 : (size_t)batch;
  return (size_t)(b->cols / 256) * chunk * (size_t)b->rows * sizeof(float);
}
inline size_t workspace_tc_bytes(const lw_dev_bundle* b) {
  return (size_t)tc_max_split(b) * 64 * (size_t)b->rows * sizeof(float);
}
inline uint32_t* workspace_counters(const lw_dev_bundle* b, void* ws) {
  (void)b;
  return static_cast<uint32_t*>(ws);
}
inline float* workspace_partials(const lw_dev_bundle* b, void* ws) {
  return reinterpret_cast<float*>(static_cast<char*>(ws) + workspace_counter_bytes(b));
}

// Table-driven 4-/6-bit product kernel (and the fixed-width twins on the same
// skeleton): usable for a coded bundle whose lut_entries hint is 1..kLutCap.
// The pending one-shot request of lw_test_stall_next (microseconds; 0:
// none), cleared by the call.
int take_test_stall();
// The table-driven kernel takes a launch when every matrix's table fits it
// and the pass has at most kLutMaxRowsQ4 (4-bit) or kLutMaxRowsQ6 (6-bit)
// activation rows.  Beyond those the staged activation slices leave the ring
// 8 stages or fewer next to the table, too few for the decoding warps, and
// the comparator kernel is faster (measured: 6-bit at 4 and 8 rows, 4-bit at
// 8).  Both kernels execute the same floating-point operations in the same
// order, so the choice never changes a result bit.
constexpr int kLutMaxRowsQ4 = 4;
constexpr int kLutMaxRowsQ6 = 2;
constexpr int kLutMaxRowsB16 = 4;   // BF16 exponent: coded single matrices
bool lut_takes(const lw_dev_bundle* const* bs, int n, int batch);
bool lut_fits(const lw_dev_bundle* b);
// With a strip list (device array of n_strips 64-row strips), n must be 1.
lw_status launch_q_lut(const lw_dev_bundle* const* bs, int n, const float* const* x, int batch,
                       float* const* y, void* const* ws, int32_t* status, cudaStream_t st,
                       const int32_t* strips = nullptr, int n_strips = 0);

// ws: the caller's whole workspace (counters, then partial sums)
lw_status launch_q_product(const lw_dev_bundle* b, const float* x, int batch, float* y, void* ws,
                           int32_t* status, cudaStream_t st);
lw_status launch_q_products(const lw_dev_bundle* const* bs, int n, const float* const* x, int batch,
                            float* const* y, void* const* ws, int32_t* status, cudaStream_t st);
lw_status launch_q_decode(const lw_dev_bundle* b, void* out, int32_t* status, cudaStream_t st);
lw_status launch_bf16_product(const lw_dev_bundle* b, const uint16_t* x, int batch, float* y,
                              void* ws, int32_t* status, cudaStream_t st);
lw_status launch_bf16_decode(const lw_dev_bundle* b, void* out, int32_t* status, cudaStream_t st);
lw_status launch_bf16_tc_product(const lw_dev_bundle* b, const uint16_t* x, int batch, float* y,
                                 void* ws, int32_t* status, cudaStream_t st);
// 4-/6-bit tensor-core product, kQtMinRows..32 activation rows per launch
// (below kQtMinRows the CUDA-core kernel, whose cost grows with the rows, is
// still faster)
constexpr int kQtMinRows = 6;
lw_status launch_q_tc_product(const lw_dev_bundle* b, const float* x, int batch, float* y, void* ws,
                              int32_t* status, cudaStream_t st);

}  // namespace lw
