// The host bundle behind the opaque lw_bundle handle of lw.h: the sections
// of one matrix's bundle as owned arrays.  Shared by the builder
// (lw_host.cpp) and the serialiser (lw_file.cpp).  Not part of the ABI.
#pragma once

#include <cstdint>
#include <vector>

#include "lw.h"

struct lw_bundle {
  lw_desc desc{};
  std::vector<uint32_t> words, tile_off;
  std::vector<uint16_t> lane_bits, lane_mid, qparams;
  lw_table table{};
  std::vector<uint8_t> signman, vexp;
  std::vector<uint32_t> vflags, vrow_off;
  int32_t max_tile_rows = 0;
  int64_t n_verbatim = 0;
};
