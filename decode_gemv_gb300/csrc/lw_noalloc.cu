// lw_decode_gemv_noalloc: the fused decode + GEMV for callers that cannot
// allocate device memory.
//
// Who needs it: code running while a CUDA graph is being captured (an
// allocation there is illegal or breaks the capture), engines whose device
// memory is owned by their own pool allocator and which do not hand out
// scratch buffers to libraries, real-time paths that must not pay for the
// implicit synchronisation of cudaMalloc/cudaFree, and bindings from other
// languages that have no device allocator at hand.  They pass inputs and
// outputs only; the scratch that lw_decode_gemv takes as `ws` comes from a
// fixed array in this library instead.
//
// The array lives in device memory for as long as the library is loaded, on
// every GPU that loads it.  All calls share it: two calls whose kernels
// overlap on the GPU (different streams, or different host threads) race on
// it and give wrong results -- serialise them.  The array keeps the last
// call's contents; the parts that must start at zero (the per-strip counters
// of the ordered split-K reduction) are cleared on the caller's stream at the
// start of every call.
#include <cstdint>
#include <mutex>

#include "lw_internal.h"
#include "lw_launch.h"

namespace {

// Maximum scratch: 16 MiB per GPU.  A matrix fits if lw_workspace_bytes(b, 1)
// <= 16 MiB.  That figure counts the partial sums reserved for a pass of 8
// activation rows, (K/256) * 8 * N * 4 bytes, plus N/64 counters -- about
// (K/256) * N <= 512 Ki -- although a batch-1 call writes an eighth of the
// partials: the limit is the workspace lw_decode_gemv would demand, so that
// the two entry points accept the same matrices.  Every matrix of the 7-8B
// layers used here fits (e.g. 14336 x 4096 and 4096 x 14336 need 7.3 MB);
// larger ones are rejected with LW_ERR_UNSUPPORTED.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the array on the current device.  Outside stream capture
// it is looked up on every call (after a device reset the module may load at
// another address); under capture, where the lookup is not made, the address
// the last call outside capture found on this device is used, so a first
// call must come before any capture.
lw_status scratch_on_current_device(cudaStream_t st, void** out) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
    cudaGetLastError();
    return lw::fail(LW_ERR_CUDA, "lw_decode_gemv_noalloc: no current device");
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    const cudaError_t e = cudaGetLastError();
    return lw::fail(LW_ERR_CUDA, "lw_decode_gemv_noalloc: stream: %s", cudaGetErrorString(e));
  }
  std::lock_guard<std::mutex> g(g_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return lw::fail(LW_ERR_CUDA, "lw_decode_gemv_noalloc: cudaGetSymbolAddress: %s",
                      cudaGetErrorString(e));
    }
    g_scratch_ptr[d] = p;
  } else if (!g_scratch_ptr[d]) {
    return lw::fail(LW_ERR_CUDA,
                    "lw_decode_gemv_noalloc: first call on device %d made under stream capture; "
                    "make one call outside capture first", d);
  }
  *out = g_scratch_ptr[d];
  return LW_OK;
}

}  // namespace

extern "C" size_t lw_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" lw_status lw_decode_gemv_noalloc(const lw_dev_bundle* b, const void* x, float* y,
                                            int32_t* d_status, void* stream) {
  lw::clear_error();
  lw_status s = lw::check_dev_bundle(b, false, true);
  if (s != LW_OK) return s;
  // the argument checks of lw_decode_gemv, before anything is queued
  if (!x || !y) return lw::fail(LW_ERR_INVALID_ARG, "lw_decode_gemv_noalloc: NULL x/y");
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(y) & 7u))
    return lw::fail(LW_ERR_INVALID_ARG,
                    "lw_decode_gemv_noalloc: x must be 16-byte aligned, y 8-byte aligned");
  const size_t need = lw_workspace_bytes(b, 1);
  if (need > kNoAllocScratchBytes)
    return lw::fail(LW_ERR_UNSUPPORTED,
                    "lw_decode_gemv_noalloc: a %lldx%lld matrix needs %zu bytes of scratch, more "
                    "than the fixed %zu; use lw_decode_gemv with a caller workspace",
                    (long long)b->rows, (long long)b->cols, need, kNoAllocScratchBytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  s = scratch_on_current_device(st, &ws);
  if (s != LW_OK) return s;
  // the strip counters must start at zero; nothing else needs clearing
  uint32_t* counters = lw::workspace_counters(b, ws);
  if (cudaMemsetAsync(counters, 0, (size_t)(b->rows / 64) * sizeof(uint32_t), st) != cudaSuccess)
    return lw::check_launch("lw_decode_gemv_noalloc: clearing counters");
  return lw_decode_gemv(b, x, y, ws, need, d_status, stream);
}
