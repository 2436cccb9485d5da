// Library-internal declarations shared by the host builder and the CUDA
// launchers of liblw.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <string>

#include "lw.h"

namespace lw {

// Thread-local text for lw_last_error(); returns `s` for convenient returns.
lw_status fail(lw_status s, const char* fmt, ...);
void clear_error();

inline int64_t tiles_of(int64_t rows, int64_t cols) { return (rows / 64) * (cols / 256); }

// Q4 tiles carry 256 pair symbols per lane, Q6 and BF16 up to 512.
inline int lane_symbols(int fmt) { return fmt == LW_FMT_Q4_PAIR ? 256 : 512; }

// Bytes of one tile's quantisation parameters (scales/mins) in LW_SEC_QPARAMS.
inline int qparam_tile_bytes(int fmt) {
  return fmt == LW_FMT_Q4_PAIR ? 64 * 2 * 2 : (fmt == LW_FMT_Q6 ? 4 * 32 * 16 : 0);
}

// Host-side checks of a device view shared by every launcher.
lw_status check_dev_bundle(const lw_dev_bundle* b, bool want_twin, bool product);

}  // namespace lw
