// Bundle files: one matrix's bundle as a single byte string, for shipping a
// coded model and loading it back ("Unweight: Compressing LLM Weights for
// Faster Inference", "One Format, Two Purposes": the Huffman bundle is the
// distribution format; at load time the runtime may transcode it).
//
// Layout (little-endian; every offset from the start of the string):
//   0    char[8]  "LWBUNDLE"
//   8    uint32   format version (1)
//   12   uint32   header bytes (192)
//   16   int32    fmt            20  int32  twin
//   24   int64    rows           32  int64  cols
//   40   int32    max_tile_rows  44  int32  sections (LW_NUM_SECTIONS)
//   48   int64    n_verbatim
//   56   uint64   bytes of section i, i = 0..15 (0 = absent; the order of
//                 lw_sections.ptr[])
//   184  uint32   section alignment (64)   188  uint32  0
//   192  the sections in order, each starting at a multiple of 64 (zero
//        padding between them)
//   end  uint64   FNV-1a (64-bit) of every byte before it, at the first
//        multiple of 64 after the last section; the string ends there.
// Loading checks the header, the checksum, every section's size against the
// shape and format, and then the full consistency checks of
// lw_validate_sections (tile offsets, lane lengths, the decoder table against
// its code lengths, the BF16 verbatim bookkeeping), so a loaded bundle is as
// trustworthy as a freshly encoded one.
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "lw_bundle.h"
#include "lw_internal.h"

using namespace lw;

namespace {

constexpr char kMagic[8] = {'L', 'W', 'B', 'U', 'N', 'D', 'L', 'E'};
constexpr uint32_t kVersion = 1;
constexpr uint64_t kHeader = 192;
constexpr uint64_t kAlign = 64;
constexpr int kSlots = 16;
static_assert(LW_NUM_SECTIONS <= kSlots, "header section slots");
static_assert(sizeof(lw_table) == 1024, "table bytes");

bool little_endian() {
  const uint16_t probe = 1;
  uint8_t b;
  std::memcpy(&b, &probe, 1);
  return b == 1;
}

uint64_t align_up(uint64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

uint64_t fnv1a64(const uint8_t* p, uint64_t n) {
  uint64_t h = 0xcbf29ce484222325ull;
  for (uint64_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 0x100000001b3ull;
  }
  return h;
}

template <class T>
void put(uint8_t* base, uint64_t at, T v) { std::memcpy(base + at, &v, sizeof v); }
template <class T>
T get(const uint8_t* base, uint64_t at) {
  T v;
  std::memcpy(&v, base + at, sizeof v);
  return v;
}

// total bytes of the serialised form of a bundle with these section sizes
uint64_t total_bytes(const uint64_t* sec) {
  uint64_t off = kHeader;
  for (int i = 0; i < LW_NUM_SECTIONS; ++i) off = align_up(off) + sec[i];
  return align_up(off) + 8;
}

template <class T>
bool take(std::vector<T>& v, const uint8_t* p, uint64_t n) {
  if (n % sizeof(T)) return false;
  v.resize(n / sizeof(T));
  if (n) std::memcpy(v.data(), p, n);
  return true;
}

}  // namespace

extern "C" size_t lw_bundle_serialized_bytes(const lw_bundle* b) {
  if (!b) return 0;
  lw_sections s;
  if (lw_bundle_sections(b, &s) != LW_OK) return 0;
  return (size_t)total_bytes(s.bytes);
}

extern "C" lw_status lw_bundle_serialize(const lw_bundle* b, void* buf, size_t cap) {
  clear_error();
  if (!b || !buf) return fail(LW_ERR_INVALID_ARG, "NULL argument");
  if (!little_endian()) return fail(LW_ERR_UNSUPPORTED, "bundle files are little-endian");
  lw_sections s;
  lw_status st = lw_bundle_sections(b, &s);
  if (st != LW_OK) return st;
  const uint64_t total = total_bytes(s.bytes);
  if (cap < total) return fail(LW_ERR_INVALID_ARG, "buffer of %zu bytes < %llu", cap,
                               (unsigned long long)total);
  uint8_t* o = static_cast<uint8_t*>(buf);
  std::memset(o, 0, (size_t)total);
  std::memcpy(o, kMagic, 8);
  put<uint32_t>(o, 8, kVersion);
  put<uint32_t>(o, 12, (uint32_t)kHeader);
  put<int32_t>(o, 16, b->desc.fmt);
  put<int32_t>(o, 20, b->desc.twin);
  put<int64_t>(o, 24, b->desc.rows);
  put<int64_t>(o, 32, b->desc.cols);
  put<int32_t>(o, 40, b->max_tile_rows);
  put<int32_t>(o, 44, LW_NUM_SECTIONS);
  put<int64_t>(o, 48, b->n_verbatim);
  for (int i = 0; i < LW_NUM_SECTIONS; ++i) put<uint64_t>(o, 56 + 8 * i, s.bytes[i]);
  put<uint32_t>(o, 184, (uint32_t)kAlign);
  uint64_t off = kHeader;
  for (int i = 0; i < LW_NUM_SECTIONS; ++i) {
    off = align_up(off);
    if (s.bytes[i]) std::memcpy(o + off, s.ptr[i], (size_t)s.bytes[i]);
    off += s.bytes[i];
  }
  off = align_up(off);
  put<uint64_t>(o, off, fnv1a64(o, off));
  return LW_OK;
}

extern "C" lw_status lw_bundle_deserialize(const void* buf, size_t n, lw_bundle** out) {
  clear_error();
  if (!buf || !out) return fail(LW_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  if (!little_endian()) return fail(LW_ERR_UNSUPPORTED, "bundle files are little-endian");
  const uint8_t* p = static_cast<const uint8_t*>(buf);
  if (n < kHeader + 8 || std::memcmp(p, kMagic, 8) != 0)
    return fail(LW_ERR_CORRUPT, "not a bundle (magic)");
  if (get<uint32_t>(p, 8) != kVersion) return fail(LW_ERR_UNSUPPORTED, "bundle version %u", get<uint32_t>(p, 8));
  if (get<uint32_t>(p, 12) != kHeader || get<int32_t>(p, 44) != LW_NUM_SECTIONS ||
      get<uint32_t>(p, 184) != kAlign)
    return fail(LW_ERR_CORRUPT, "bundle header fields");
  uint64_t sec[kSlots];
  for (int i = 0; i < kSlots; ++i) sec[i] = get<uint64_t>(p, 56 + 8 * i);
  for (int i = LW_NUM_SECTIONS; i < kSlots; ++i)
    if (sec[i]) return fail(LW_ERR_CORRUPT, "unknown section %d", i);
  // sizes first (no overflow: each is checked against the string's length)
  uint64_t off = kHeader;
  for (int i = 0; i < LW_NUM_SECTIONS; ++i) {
    if (sec[i] > (uint64_t)n) return fail(LW_ERR_CORRUPT, "section %d larger than the file", i);
    off = align_up(off) + sec[i];
    if (off > (uint64_t)n) return fail(LW_ERR_CORRUPT, "section %d runs past the end", i);
  }
  const uint64_t end = align_up(off);
  if (end + 8 != (uint64_t)n) return fail(LW_ERR_CORRUPT, "bundle length %zu, expected %llu", n,
                                          (unsigned long long)(end + 8));
  if (fnv1a64(p, end) != get<uint64_t>(p, end)) return fail(LW_ERR_CORRUPT, "checksum mismatch");

  lw_desc d{};
  d.fmt = get<int32_t>(p, 16);
  d.twin = get<int32_t>(p, 20);
  d.rows = get<int64_t>(p, 24);
  d.cols = get<int64_t>(p, 32);
  if (d.fmt != LW_FMT_Q4_PAIR && d.fmt != LW_FMT_Q6 && d.fmt != LW_FMT_BF16_EXP)
    return fail(LW_ERR_CORRUPT, "format %d", d.fmt);
  if (d.twin != 0 && d.twin != 1) return fail(LW_ERR_CORRUPT, "twin flag %d", d.twin);
  if (d.rows <= 0 || d.cols <= 0 || d.rows % 64 || d.cols % 256 || d.rows > (1ll << 31) ||
      d.cols > (1ll << 31))
    return fail(LW_ERR_CORRUPT, "shape %lldx%lld", (long long)d.rows, (long long)d.cols);
  const bool bf16 = d.fmt == LW_FMT_BF16_EXP;
  // sections a bundle of this kind never has
  if (bf16 ? sec[LW_SEC_QPARAMS] != 0
           : (sec[LW_SEC_SIGNMAN] | sec[LW_SEC_VFLAGS] | sec[LW_SEC_VROW_OFF] | sec[LW_SEC_VEXP]) != 0)
    return fail(LW_ERR_CORRUPT, "section present that format %d does not use", d.fmt);
  if (d.twin && sec[LW_SEC_LANE_MID]) return fail(LW_ERR_CORRUPT, "twin bundle with lane mids");
  if (sec[LW_SEC_TABLE] != sizeof(lw_table)) return fail(LW_ERR_CORRUPT, "table section size");

  lw_bundle* B = new (std::nothrow) lw_bundle;
  if (!B) return fail(LW_ERR_ALLOC, "bundle");
  bool ok = true;
  try {
    B->desc = d;
    const uint8_t* at[LW_NUM_SECTIONS];
    off = kHeader;
    for (int i = 0; i < LW_NUM_SECTIONS; ++i) {
      off = align_up(off);
      at[i] = p + off;
      off += sec[i];
    }
    ok = take(B->words, at[LW_SEC_WORDS], sec[LW_SEC_WORDS]) &&
         take(B->tile_off, at[LW_SEC_TILE_OFF], sec[LW_SEC_TILE_OFF]) &&
         take(B->lane_bits, at[LW_SEC_LANE_BITS], sec[LW_SEC_LANE_BITS]) &&
         take(B->qparams, at[LW_SEC_QPARAMS], sec[LW_SEC_QPARAMS]) &&
         take(B->signman, at[LW_SEC_SIGNMAN], sec[LW_SEC_SIGNMAN]) &&
         take(B->vflags, at[LW_SEC_VFLAGS], sec[LW_SEC_VFLAGS]) &&
         take(B->vrow_off, at[LW_SEC_VROW_OFF], sec[LW_SEC_VROW_OFF]) &&
         take(B->vexp, at[LW_SEC_VEXP], sec[LW_SEC_VEXP]) &&
         take(B->lane_mid, at[LW_SEC_LANE_MID], sec[LW_SEC_LANE_MID]);
    if (ok) std::memcpy(&B->table, at[LW_SEC_TABLE], sizeof(lw_table));
  } catch (const std::bad_alloc&) {
    delete B;
    return fail(LW_ERR_ALLOC, "bundle sections");
  }
  if (!ok) {
    delete B;
    return fail(LW_ERR_CORRUPT, "section size not a multiple of its element size");
  }
  // derived fields: recomputed, and the header must agree with them
  const int64_t n_tiles = tiles_of(d.rows, d.cols);
  if ((int64_t)B->tile_off.size() != n_tiles + 1) {
    delete B;
    return fail(LW_ERR_CORRUPT, "tile offsets do not match the shape");
  }
  int32_t wmax = 0;
  for (int64_t t = 0; t < n_tiles; ++t) {
    const int64_t w = (int64_t)B->tile_off[t + 1] - (int64_t)B->tile_off[t];
    if (w > wmax) wmax = (int32_t)(w > (1 << 30) ? (1 << 30) : w);
  }
  B->max_tile_rows = wmax;
  B->n_verbatim = bf16 ? (int64_t)(B->vexp.size() / 64) : 0;
  if (get<int32_t>(p, 40) != B->max_tile_rows || get<int64_t>(p, 48) != B->n_verbatim) {
    delete B;
    return fail(LW_ERR_CORRUPT, "header statistics disagree with the sections");
  }
  lw_sections s;
  lw_status st = lw_bundle_sections(B, &s);
  if (st == LW_OK) st = lw_validate_sections(&d, &s);
  if (st != LW_OK) {
    delete B;
    return st;
  }
  *out = B;
  return LW_OK;
}

extern "C" lw_status lw_bundle_save(const lw_bundle* b, const char* path) {
  clear_error();
  if (!b || !path) return fail(LW_ERR_INVALID_ARG, "NULL argument");
  const size_t n = lw_bundle_serialized_bytes(b);
  if (!n) return fail(LW_ERR_INVALID_ARG, "bundle has no sections");
  std::vector<uint8_t> buf;
  try {
    buf.resize(n);
  } catch (const std::bad_alloc&) {
    return fail(LW_ERR_ALLOC, "%zu bytes", n);
  }
  lw_status st = lw_bundle_serialize(b, buf.data(), n);
  if (st != LW_OK) return st;
  FILE* f = std::fopen(path, "wb");
  if (!f) return fail(LW_ERR_IO, "cannot open %s for writing", path);
  const size_t w = std::fwrite(buf.data(), 1, n, f);
  const int c = std::fclose(f);
  if (w != n || c != 0) return fail(LW_ERR_IO, "short write to %s", path);
  return LW_OK;
}

extern "C" lw_status lw_bundle_load(const char* path, lw_bundle** out) {
  clear_error();
  if (!path || !out) return fail(LW_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  FILE* f = std::fopen(path, "rb");
  if (!f) return fail(LW_ERR_IO, "cannot open %s", path);
  std::vector<uint8_t> buf;
  bool ok = std::fseek(f, 0, SEEK_END) == 0;
  const long len = ok ? std::ftell(f) : -1;
  ok = ok && len >= 0 && std::fseek(f, 0, SEEK_SET) == 0;
  if (ok) {
    try {
      buf.resize((size_t)len);
    } catch (const std::bad_alloc&) {
      std::fclose(f);
      return fail(LW_ERR_ALLOC, "%ld bytes", len);
    }
    ok = std::fread(buf.data(), 1, (size_t)len, f) == (size_t)len;
  }
  std::fclose(f);
  if (!ok) return fail(LW_ERR_IO, "cannot read %s", path);
  return lw_bundle_deserialize(buf.data(), buf.size(), out);
}

extern "C" lw_status lw_bundle_desc(const lw_bundle* b, lw_desc* out) {
  if (!b || !out) return fail(LW_ERR_INVALID_ARG, "NULL argument");
  *out = b->desc;
  return LW_OK;
}
