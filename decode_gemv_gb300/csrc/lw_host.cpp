// Host side of liblw: the bundle builder and the non-device C-ABI calls.
//
// Builds, per weight matrix, the coded layout of "LazyWeights: Decode-on-
// Demand Edge LLMs" ("2 . Code them", Fig. 3(a)): one optimal length-limited
// (11-bit) canonical Huffman table, 4-bit codes paired into byte symbols,
// 64x256 tiles split into 32 lanes of two rows, each lane a stream of 32-bit
// words, the lanes' words interleaved, per-tile offsets; and the BF16 layout
// of "Unweight" ("The exponent's exploitable redundancy"): exponent bytes
// coded over the matrix's top-16 palette, sign+mantissa bytes raw, 64-column
// groups holding an out-of-palette exponent stored verbatim.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <numeric>
#include <thread>
#include <vector>

#include "lw_bundle.h"
#include "lw_lut.h"
#include "lw_internal.h"

namespace lw {

static thread_local std::string g_err;

lw_status fail(lw_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

void clear_error() { g_err.clear(); }

// ---------------------------------------------------------------------------
// Optimal length-limited code lengths: package-merge in its "counts only"
// form.  Level d (d = lmax deepest .. 1) holds the sorted merge of the
// leaves with the packages formed from pairs of level d+1.  Selecting the
// first 2n-2 items of level 1 and walking down, the first m items of a level
// contain some prefix of the (sorted) leaves -- each such leaf gains one bit
// -- and p packages, which stand for the first 2p items of the next level.
// ---------------------------------------------------------------------------
static bool limited_lengths(const std::vector<uint64_t>& cnt, int lmax,
                            std::vector<uint8_t>& len) {
  const int alpha = (int)cnt.size();
  len.assign(alpha, 0);
  std::vector<int> leaf;
  for (int s = 0; s < alpha; ++s)
    if (cnt[s]) leaf.push_back(s);
  const int n = (int)leaf.size();
  if (n == 0) return true;
  if (n == 1) { len[leaf[0]] = 1; return true; }
  if ((int64_t)n > ((int64_t)1 << lmax)) return false;
  std::stable_sort(leaf.begin(), leaf.end(),
                   [&](int a, int b) { return cnt[a] < cnt[b]; });

  // is_leaf[d][i]: item i of level d is a leaf (else a package); weight[d][i]
  std::vector<std::vector<uint8_t>> is_leaf(lmax + 1);
  std::vector<std::vector<uint64_t>> weight(lmax + 1);
  weight[lmax].resize(n);
  is_leaf[lmax].assign(n, 1);
  for (int i = 0; i < n; ++i) weight[lmax][i] = cnt[leaf[i]];
  for (int d = lmax - 1; d >= 1; --d) {
    const std::vector<uint64_t>& below = weight[d + 1];
    const size_t npk = below.size() / 2;
    std::vector<uint64_t>& w = weight[d];
    std::vector<uint8_t>& f = is_leaf[d];
    w.reserve(n + npk);
    f.reserve(n + npk);
    size_t i = 0, j = 0;
    while (i < (size_t)n || j < npk) {
      const bool take_leaf =
          j >= npk || (i < (size_t)n && cnt[leaf[i]] <= below[2 * j] + below[2 * j + 1]);
      if (take_leaf) { w.push_back(cnt[leaf[i]]); f.push_back(1); ++i; }
      else { w.push_back(below[2 * j] + below[2 * j + 1]); f.push_back(0); ++j; }
    }
  }
  size_t m = 2 * (size_t)n - 2;
  for (int d = 1; d <= lmax && m > 0; ++d) {
    size_t leaves_here = 0;
    for (size_t i = 0; i < m; ++i) leaves_here += is_leaf[d][i];
    for (size_t k = 0; k < leaves_here; ++k) len[leaf[k]]++;
    m = 2 * (m - leaves_here);
  }
  return true;
}

// Canonical codes from lengths (shortest first, ties by symbol value).
static void canonical(const std::vector<uint8_t>& len, std::vector<uint32_t>& code) {
  uint32_t nl[LW_MAX_CODE_LEN + 2] = {0}, next[LW_MAX_CODE_LEN + 2] = {0};
  for (uint8_t l : len) if (l) nl[l]++;
  uint32_t c = 0;
  for (int L = 1; L <= LW_MAX_CODE_LEN; ++L) {
    c = (c + nl[L - 1]) << 1;
    next[L] = c;
  }
  code.assign(len.size(), 0);
  for (size_t s = 0; s < len.size(); ++s)
    if (len[s]) code[s] = next[len[s]]++;
}

}  // namespace lw

using namespace lw;

// ---------------------------------------------------------------------------
// Decoder table
// ---------------------------------------------------------------------------
extern "C" lw_status lw_table_from_lengths(int32_t fmt, const uint8_t* code_len, int32_t alpha,
                                           const uint8_t* palette, int32_t n_palette,
                                           lw_table* out) {
  if (!code_len || !out || alpha <= 0 || alpha > 256)
    return fail(LW_ERR_INVALID_ARG, "lw_table_from_lengths: bad arguments");
  if (fmt == LW_FMT_BF16_EXP && (!palette || n_palette < 1 || n_palette > 16))
    return fail(LW_ERR_INVALID_ARG, "lw_table_from_lengths: BF16 needs a palette of 1..16");
  std::memset(out, 0, sizeof *out);
  out->fmt = fmt;
  out->alpha = alpha;
  uint32_t count[LW_MAX_CODE_LEN + 2] = {0};
  int n = 0, lmin = 99, lmax = 0;
  for (int s = 0; s < alpha; ++s) {
    const int L = code_len[s];
    if (L > LW_MAX_CODE_LEN) return fail(LW_ERR_CORRUPT, "code length %d > 11", L);
    if (!L) continue;
    count[L]++;
    n++;
    lmin = std::min(lmin, L);
    lmax = std::max(lmax, L);
  }
  if (n == 0) return fail(LW_ERR_CORRUPT, "table has no symbol");
  // Kraft sum in units of 2^-11
  uint64_t kraft = 0;
  for (int L = 1; L <= LW_MAX_CODE_LEN; ++L) kraft += (uint64_t)count[L] << (LW_MAX_CODE_LEN - L);
  const bool lone = (n == 1);
  if (lone) {
    if (lmin != 1) return fail(LW_ERR_CORRUPT, "a lone symbol must have length 1");
  } else if (kraft != (1u << LW_MAX_CODE_LEN)) {
    return fail(LW_ERR_CORRUPT, "code is not complete (Kraft sum %llu/2048)",
                (unsigned long long)kraft);
  }
  uint32_t first[LW_MAX_CODE_LEN + 2] = {0}, base[LW_MAX_CODE_LEN + 2] = {0};
  uint32_t c = 0, b = 0;
  for (int L = 1; L <= LW_MAX_CODE_LEN; ++L) {
    c = (c + count[L - 1]) << 1;
    first[L] = c;
    base[L] = b;
    b += count[L];
  }
  int k = 0;
  for (int L = 1; L <= LW_MAX_CODE_LEN; ++L)
    for (int s = 0; s < alpha; ++s)
      if (code_len[s] == L) out->sym[k++] = (uint16_t)s;
  out->n_sym = n;
  if (lone) {  // the second length-1 code ("1") decodes to the same symbol
    out->sym[1] = out->sym[0];
    out->phantom = 1;
  }
  out->lmin = lmin;
  out->lmax = lmax;
  for (int j = 0; j < 12; ++j) { out->lim_m1[j] = 0xFFFFFFFFu; out->off[j] = 0; }
  for (int L = lmin; L <= lmax; ++L) {
    out->off[L - lmin] = (int32_t)base[L] - (int32_t)first[L];
    if (L < lmax) {
      const uint64_t limit = (uint64_t)(first[L] + count[L]) << (LW_MAX_CODE_LEN - L);
      out->lim_m1[L - lmin] = (uint32_t)((limit << 21) - 1);
    }
  }
  for (int s = 0; s < alpha; ++s) out->code_len[s] = code_len[s];
  if (fmt == LW_FMT_BF16_EXP) {
    out->n_palette = n_palette;
    for (int i = 0; i < n_palette; ++i) out->palette[i] = palette[i];
  }
  return LW_OK;
}

// ---------------------------------------------------------------------------
// Bundle
// ---------------------------------------------------------------------------

namespace {

// Run fn(t) for t in [0, n) on up to hardware_concurrency threads.
template <class F>
void parallel_for(int64_t n, F fn) {
  unsigned nt = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
  if (n < 64 || nt == 1) {
    for (int64_t t = 0; t < n; ++t) fn(t);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> th;
  for (unsigned i = 0; i < nt; ++i)
    th.emplace_back([&] {
      for (int64_t t; (t = next.fetch_add(16)) < n;)
        for (int64_t u = t; u < std::min(n, t + 16); ++u) fn(u);
    });
  for (auto& x : th) x.join();
}

// Symbols of one lane in lane order.  Returns the count.
struct LaneSource {
  int fmt;
  int64_t N, K, TK;
  const uint8_t* codes = nullptr;        // Q4 / Q6
  const uint8_t* palidx = nullptr;       // BF16: palette index per weight
  const uint8_t* verb = nullptr;         // BF16: [N][K/64] 0/1
  // Symbols of lane l of tile t in lane order; *first = how many belong to
  // the lane's first row.
  int operator()(int64_t t, int l, uint16_t* out, int* first = nullptr) const {
    const int64_t s = t / TK, kt = t % TK;
    int n = 0;
    for (int half = 0; half < 2; ++half) {
      if (half == 1 && first) *first = n;
      const int64_t r = 64 * s + 2 * l + half;
      if (fmt == LW_FMT_Q4_PAIR) {
        const uint8_t* row = codes + r * K + 256 * kt;
        for (int j = 0; j < 256; j += 2) out[n++] = (uint16_t)(row[j] | (row[j + 1] << 4));
      } else if (fmt == LW_FMT_Q6) {
        const uint8_t* row = codes + r * K + 256 * kt;
        for (int j = 0; j < 256; ++j) out[n++] = row[j];
      } else {
        for (int g = 0; g < 4; ++g) {
          if (verb[r * (K / 64) + 4 * kt + g]) continue;
          const uint8_t* p = palidx + r * K + 256 * kt + 64 * g;
          for (int j = 0; j < 64; ++j) out[n++] = p[j];
        }
      }
    }
    return n;
  }
};

// MSB-first bit writer into one lane's words (stride 32 in the interleave).
struct BitWriter {
  uint32_t* base;   // word 0 of the lane
  uint64_t acc = 0;
  int nacc = 0;
  int64_t j = 0;
  void put(uint32_t code, int len) {
    acc = (acc << len) | code;
    nacc += len;
    while (nacc >= 32) {
      base[32 * j++] = (uint32_t)(acc >> (nacc - 32));
      nacc -= 32;
    }
  }
  void flush() {
    if (nacc > 0) base[32 * j++] = (uint32_t)(acc << (32 - nacc));
    nacc = 0;
  }
};

lw_status pack_huffman(lw_bundle* B, const LaneSource& src, int alpha) {
  const int64_t n_tiles = tiles_of(B->desc.rows, B->desc.cols);
  const int maxsym = lane_symbols(B->desc.fmt);
  // histogram of the coded symbols, per thread then summed
  std::vector<uint64_t> hist(alpha, 0);
  {
    const unsigned nt = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
    std::vector<std::vector<uint64_t>> part(nt, std::vector<uint64_t>(alpha, 0));
    std::atomic<int64_t> next{0};
    std::vector<std::thread> th;
    for (unsigned i = 0; i < nt; ++i)
      th.emplace_back([&, i] {
        std::vector<uint16_t> buf(maxsym);
        for (int64_t t; (t = next.fetch_add(1)) < n_tiles;)
          for (int l = 0; l < 32; ++l) {
            const int n = src(t, l, buf.data());
            for (int k = 0; k < n; ++k) part[i][buf[k]]++;
          }
      });
    for (auto& x : th) x.join();
    for (auto& p : part)
      for (int s = 0; s < alpha; ++s) hist[s] += p[s];
  }
  std::vector<uint8_t> len;
  bool any = false;
  for (auto h : hist) any |= (h != 0);
  if (any) {
    if (!limited_lengths(hist, LW_MAX_CODE_LEN, len))
      return fail(LW_ERR_UNSUPPORTED, "alphabet too large for 11-bit codes");
  } else {
    // nothing is coded (every BF16 group verbatim): a one-symbol table keeps
    // the device table well formed
    len.assign(alpha, 0);
    len[0] = 1;
  }
  uint8_t palette[16];
  std::memcpy(palette, B->table.palette, sizeof palette);
  const int32_t n_palette = B->table.n_palette;
  lw_status st = lw_table_from_lengths(B->desc.fmt, len.data(), alpha, palette, n_palette,
                                       &B->table);
  if (st != LW_OK) return st;
  std::vector<uint32_t> code;
  canonical(len, code);

  // pass 1: lane bit counts and W_t
  B->lane_bits.assign(n_tiles * 32, 0);
  B->lane_mid.assign(n_tiles * 32, 0);
  std::vector<uint32_t> wt(n_tiles, 0);
  std::atomic<bool> overflow{false};
  parallel_for(n_tiles, [&](int64_t t) {
    std::vector<uint16_t> buf(maxsym);
    uint32_t w = 0;
    for (int l = 0; l < 32; ++l) {
      int first = 0;
      const int n = src(t, l, buf.data(), &first);
      uint64_t bits = 0, mid = 0;
      for (int k = 0; k < n; ++k) {
        if (k == first) mid = bits;
        bits += len[buf[k]];
      }
      if (first >= n) mid = bits;
      if (bits > 0xFFFF) overflow = true;
      B->lane_bits[t * 32 + l] = (uint16_t)bits;
      B->lane_mid[t * 32 + l] = (uint16_t)mid;
      w = std::max<uint32_t>(w, (uint32_t)((bits + 31) / 32));
    }
    wt[t] = w;
  });
  if (overflow) return fail(LW_ERR_UNSUPPORTED, "lane longer than 65535 bits");
  B->tile_off.assign(n_tiles + 1, 0);
  uint64_t rows = 0;
  for (int64_t t = 0; t < n_tiles; ++t) {
    B->tile_off[t] = (uint32_t)rows;
    rows += wt[t];
    B->max_tile_rows = std::max<int32_t>(B->max_tile_rows, (int32_t)wt[t]);
  }
  if (rows > 0xFFFFFFFFull) return fail(LW_ERR_UNSUPPORTED, "matrix too large");
  B->tile_off[n_tiles] = (uint32_t)rows;
  // pass 2: words
  try {
    B->words.assign(rows * 32, 0);
  } catch (const std::bad_alloc&) {
    return fail(LW_ERR_ALLOC, "words");
  }
  parallel_for(n_tiles, [&](int64_t t) {
    std::vector<uint16_t> buf(maxsym);
    for (int l = 0; l < 32; ++l) {
      const int n = src(t, l, buf.data());
      BitWriter bw{B->words.data() + (uint64_t)B->tile_off[t] * 32 + l};
      for (int k = 0; k < n; ++k) bw.put(code[buf[k]], len[buf[k]]);
      bw.flush();
    }
  });
  return LW_OK;
}

// Fixed-width twin: each lane's 512 values at `width` bits, MSB-first.
void pack_twin(lw_bundle* B, const uint8_t* vals /* [N][K] */, int width) {
  const int64_t N = B->desc.rows, K = B->desc.cols, TK = K / 256;
  const int64_t n_tiles = tiles_of(N, K);
  const uint32_t wt = (uint32_t)(512 * width / 32);
  B->max_tile_rows = (int32_t)wt;
  B->tile_off.resize(n_tiles + 1);
  for (int64_t t = 0; t <= n_tiles; ++t) B->tile_off[t] = (uint32_t)(t * wt);
  B->lane_bits.assign(n_tiles * 32, (uint16_t)(512 * width));
  B->words.assign((uint64_t)n_tiles * wt * 32, 0);
  parallel_for(n_tiles, [&](int64_t t) {
    const int64_t s = t / TK, kt = t % TK;
    for (int l = 0; l < 32; ++l) {
      BitWriter bw{B->words.data() + (uint64_t)t * wt * 32 + l};
      for (int half = 0; half < 2; ++half) {
        const uint8_t* row = vals + (64 * s + 2 * l + half) * K + 256 * kt;
        for (int j = 0; j < 256; ++j) bw.put(row[j], width);
      }
      bw.flush();
    }
  });
}

void arrange_qparams(lw_bundle* B, const uint16_t* scales, const uint16_t* mins) {
  const int64_t N = B->desc.rows, K = B->desc.cols, TK = K / 256;
  const int64_t n_tiles = tiles_of(N, K);
  if (B->desc.fmt == LW_FMT_Q4_PAIR) {
    B->qparams.resize(n_tiles * 128);
    for (int64_t t = 0; t < n_tiles; ++t) {
      const int64_t s = t / TK, kt = t % TK;
      for (int i = 0; i < 64; ++i) {
        B->qparams[(t * 64 + i) * 2 + 0] = scales[(64 * s + i) * TK + kt];
        B->qparams[(t * 64 + i) * 2 + 1] = mins[(64 * s + i) * TK + kt];
      }
    }
  } else if (B->desc.fmt == LW_FMT_Q6) {
    const int64_t G = K / 16;
    B->qparams.resize(n_tiles * 4 * 32 * 8);
    for (int64_t t = 0; t < n_tiles; ++t) {
      const int64_t s = t / TK, kt = t % TK;
      for (int l = 0; l < 32; ++l)
        for (int i = 0; i < 32; ++i) {
          const int64_t r = 64 * s + 2 * l + i / 16;
          const int q = i / 8;
          B->qparams[((t * 4 + q) * 32 + l) * 8 + i % 8] = scales[r * G + 16 * kt + i % 16];
        }
    }
  }
}

// BF16 side data: palette, verbatim groups, sign+mantissa bytes.
struct Bf16Split {
  std::vector<uint8_t> palidx;   // [N][K], 0xFF outside the palette
  std::vector<uint8_t> verb;     // [N][K/64]
};

void split_bf16(lw_bundle* B, const uint16_t* bits, Bf16Split& sp) {
  const int64_t N = B->desc.rows, K = B->desc.cols, TK = K / 256, G = K / 64;
  uint64_t hist[256] = {0};
  for (int64_t i = 0; i < N * K; ++i) hist[(bits[i] >> 7) & 0xFF]++;
  std::vector<int> order;
  for (int e = 0; e < 256; ++e) if (hist[e]) order.push_back(e);
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return hist[a] > hist[b]; });   // ties: smaller value first
  if (order.size() > 16) order.resize(16);
  std::sort(order.begin(), order.end());
  uint8_t map[256];
  std::memset(map, 0xFF, sizeof map);
  B->table.n_palette = (int32_t)order.size();
  for (size_t i = 0; i < order.size(); ++i) {
    B->table.palette[i] = (uint8_t)order[i];
    map[order[i]] = (uint8_t)i;
  }
  sp.palidx.resize(N * K);
  sp.verb.assign(N * G, 0);
  for (int64_t i = 0; i < N * K; ++i) {
    sp.palidx[i] = map[(bits[i] >> 7) & 0xFF];
    if (sp.palidx[i] == 0xFF) sp.verb[i / 64] = 1;
  }
  const int64_t GW = (G + 31) / 32;
  B->vflags.assign(N * GW, 0);
  B->vrow_off.assign(N + 1, 0);
  int64_t nv = 0;
  for (int64_t r = 0; r < N; ++r) {
    B->vrow_off[r] = (uint32_t)nv;
    for (int64_t g = 0; g < G; ++g)
      if (sp.verb[r * G + g]) {
        B->vflags[r * GW + g / 32] |= 1u << (g % 32);
        nv++;
      }
  }
  B->vrow_off[N] = (uint32_t)nv;
  B->n_verbatim = nv;
  B->vexp.resize(nv * 64);
  int64_t v = 0;
  for (int64_t r = 0; r < N; ++r)
    for (int64_t g = 0; g < G; ++g)
      if (sp.verb[r * G + g]) {
        for (int j = 0; j < 64; ++j)
          B->vexp[v * 64 + j] = (uint8_t)((bits[r * K + 64 * g + j] >> 7) & 0xFF);
        v++;
      }
  // sign+mantissa bytes, tile-major, 16-byte chunks interleaved over lanes
  const int64_t n_tiles = tiles_of(N, K);
  B->signman.resize(n_tiles * 16384);
  parallel_for(n_tiles, [&](int64_t t) {
    const int64_t s = t / TK, kt = t % TK;
    uint8_t* dst = B->signman.data() + t * 16384;
    for (int l = 0; l < 32; ++l)
      for (int q = 0; q < 512; ++q) {
        const int64_t r = 64 * s + 2 * l + q / 256;
        const uint16_t w = bits[r * K + 256 * kt + q % 256];
        dst[((q / 16) * 32 + l) * 16 + q % 16] = (uint8_t)(((w >> 8) & 0x80) | (w & 0x7F));
      }
  });
}

}  // namespace

extern "C" lw_status lw_encode_bundle(const lw_desc* desc, const void* payload,
                                      const uint16_t* scales, const uint16_t* mins,
                                      lw_bundle** out) {
  clear_error();
  if (!desc || !payload || !out) return fail(LW_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  const int fmt = desc->fmt;
  if (fmt != LW_FMT_Q4_PAIR && fmt != LW_FMT_Q6 && fmt != LW_FMT_BF16_EXP)
    return fail(LW_ERR_UNSUPPORTED, "unknown format %d", fmt);
  if (desc->rows <= 0 || desc->cols <= 0 || desc->rows % 64 || desc->cols % 256)
    return fail(LW_ERR_SHAPE, "shape %lldx%lld is not a positive multiple of 64x256",
                (long long)desc->rows, (long long)desc->cols);
  if ((fmt == LW_FMT_Q4_PAIR && (!scales || !mins)) || (fmt == LW_FMT_Q6 && !scales))
    return fail(LW_ERR_INVALID_ARG, "missing scales/mins");
  const int64_t N = desc->rows, K = desc->cols;
  if (fmt != LW_FMT_BF16_EXP) {
    const uint8_t* c = (const uint8_t*)payload;
    const uint8_t top = fmt == LW_FMT_Q4_PAIR ? 16 : 64;
    for (int64_t i = 0; i < N * K; ++i)
      if (c[i] >= top) return fail(LW_ERR_INVALID_ARG, "code %d out of range at %lld", c[i], (long long)i);
  }
  lw_bundle* B = new (std::nothrow) lw_bundle;
  if (!B) return fail(LW_ERR_ALLOC, "bundle");
  B->desc = *desc;
  lw_status st = LW_OK;
  try {
    if (fmt != LW_FMT_BF16_EXP) {
      arrange_qparams(B, scales, mins);
      if (desc->twin) {
        pack_twin(B, (const uint8_t*)payload, fmt == LW_FMT_Q4_PAIR ? 4 : 6);
        B->table.fmt = fmt;
        B->table.alpha = fmt == LW_FMT_Q4_PAIR ? 256 : 64;
      } else {
        LaneSource src{fmt, N, K, K / 256, (const uint8_t*)payload};
        st = pack_huffman(B, src, fmt == LW_FMT_Q4_PAIR ? 256 : 64);
      }
    } else {
      Bf16Split sp;
      split_bf16(B, (const uint16_t*)payload, sp);
      if (desc->twin) {
        // direct palette: 4-bit index per weight, 0 in verbatim groups
        std::vector<uint8_t> idx(N * K);
        for (int64_t i = 0; i < N * K; ++i)
          idx[i] = sp.verb[i / 64] ? 0 : sp.palidx[i];
        pack_twin(B, idx.data(), 4);
        B->table.fmt = fmt;
        B->table.alpha = 16;
      } else {
        LaneSource src{fmt, N, K, K / 256, nullptr, sp.palidx.data(), sp.verb.data()};
        st = pack_huffman(B, src, 16);
      }
    }
  } catch (const std::bad_alloc&) {
    st = fail(LW_ERR_ALLOC, "host allocation");
  }
  if (st != LW_OK) { delete B; return st; }
  *out = B;
  return LW_OK;
}

extern "C" lw_status lw_bundle_sections(const lw_bundle* B, lw_sections* s) {
  if (!B || !s) return fail(LW_ERR_INVALID_ARG, "NULL argument");
  std::memset(s, 0, sizeof *s);
  auto put = [&](int id, const void* p, size_t n) { s->ptr[id] = n ? p : nullptr; s->bytes[id] = n; };
  put(LW_SEC_WORDS, B->words.data(), B->words.size() * 4);
  put(LW_SEC_TILE_OFF, B->tile_off.data(), B->tile_off.size() * 4);
  put(LW_SEC_LANE_BITS, B->lane_bits.data(), B->lane_bits.size() * 2);
  put(LW_SEC_TABLE, &B->table, sizeof(lw_table));
  put(LW_SEC_QPARAMS, B->qparams.data(), B->qparams.size() * 2);
  put(LW_SEC_SIGNMAN, B->signman.data(), B->signman.size());
  put(LW_SEC_VFLAGS, B->vflags.data(), B->vflags.size() * 4);
  put(LW_SEC_VROW_OFF, B->vrow_off.data(), B->vrow_off.size() * 4);
  put(LW_SEC_VEXP, B->vexp.data(), B->vexp.size());
  put(LW_SEC_LANE_MID, B->lane_mid.data(), B->lane_mid.size() * 2);
  uint64_t tot = 0;
  for (int i = 0; i < LW_NUM_SECTIONS; ++i) tot += s->bytes[i];
  s->coded_bytes = tot;
  s->n_tiles = (uint64_t)tiles_of(B->desc.rows, B->desc.cols);
  s->n_verbatim = B->n_verbatim;
  s->max_tile_rows = B->max_tile_rows;
  s->max_len = B->table.lmax;
  s->min_len = B->table.lmin;
  s->palette_size = B->table.n_palette;
  s->bits_per_weight = 8.0 * (double)tot / ((double)B->desc.rows * (double)B->desc.cols);
  if (!B->desc.twin)
    s->lut_entries = lw::lut_shape(B->table.lim_m1, B->table.lmin, B->table.lmax).n;
  return LW_OK;
}

extern "C" void lw_bundle_free(lw_bundle* b) { delete b; }

extern "C" lw_status lw_validate_sections(const lw_desc* d, const lw_sections* s) {
  if (!d || !s) return fail(LW_ERR_INVALID_ARG, "NULL argument");
  if (d->rows <= 0 || d->cols <= 0 || d->rows % 64 || d->cols % 256)
    return fail(LW_ERR_SHAPE, "bad shape");
  const int64_t n_tiles = tiles_of(d->rows, d->cols);
  if (s->bytes[LW_SEC_TILE_OFF] != (uint64_t)(n_tiles + 1) * 4 ||
      s->bytes[LW_SEC_LANE_BITS] != (uint64_t)n_tiles * 64 ||
      s->bytes[LW_SEC_TABLE] != sizeof(lw_table))
    return fail(LW_ERR_CORRUPT, "section sizes do not match the shape");
  const uint32_t* off = (const uint32_t*)s->ptr[LW_SEC_TILE_OFF];
  const uint16_t* lb = (const uint16_t*)s->ptr[LW_SEC_LANE_BITS];
  if (off[0] != 0) return fail(LW_ERR_CORRUPT, "tile_off[0] != 0");
  for (int64_t t = 0; t < n_tiles; ++t) {
    if (off[t + 1] < off[t]) return fail(LW_ERR_CORRUPT, "tile_off decreases at %lld", (long long)t);
    const uint32_t wt = off[t + 1] - off[t];
    if ((int64_t)wt > s->max_tile_rows) return fail(LW_ERR_CORRUPT, "tile %lld longer than max_tile_rows", (long long)t);
    for (int l = 0; l < 32; ++l)
      if (lb[t * 32 + l] > wt * 32) return fail(LW_ERR_CORRUPT, "lane bits exceed W_t at tile %lld", (long long)t);
  }
  if (!d->twin) {
    if (s->bytes[LW_SEC_LANE_MID] != (uint64_t)n_tiles * 64)
      return fail(LW_ERR_CORRUPT, "lane_mid size does not match the shape");
    const uint16_t* mid = (const uint16_t*)s->ptr[LW_SEC_LANE_MID];
    for (int64_t i = 0; i < n_tiles * 32; ++i)
      if (mid[i] > lb[i]) return fail(LW_ERR_CORRUPT, "lane_mid beyond lane_bits at lane %lld", (long long)i);
  }
  if ((uint64_t)off[n_tiles] * 128 != s->bytes[LW_SEC_WORDS])
    return fail(LW_ERR_CORRUPT, "word count does not match tile_off");
  const lw_table* tb = (const lw_table*)s->ptr[LW_SEC_TABLE];
  if (tb->fmt != d->fmt) return fail(LW_ERR_CORRUPT, "table format mismatch");
  if (d->twin) {
    // a twin reads no code from its table: only the alphabet and, for BF16,
    // the palette that maps its 4-bit indices back to exponent bytes
    const int alpha = d->fmt == LW_FMT_Q4_PAIR ? 256 : (d->fmt == LW_FMT_Q6 ? 64 : 16);
    if (tb->alpha != alpha) return fail(LW_ERR_CORRUPT, "twin table alphabet %d", tb->alpha);
    if (d->fmt == LW_FMT_BF16_EXP) {
      if (tb->n_palette < 1 || tb->n_palette > 16)
        return fail(LW_ERR_CORRUPT, "twin palette size %d", tb->n_palette);
      for (int i = 1; i < tb->n_palette; ++i)
        if (tb->palette[i] <= tb->palette[i - 1])
          return fail(LW_ERR_CORRUPT, "twin palette not ascending");
    }
  }
  if (!d->twin) {
    lw_table chk;
    lw_status st = lw_table_from_lengths(tb->fmt, tb->code_len, tb->alpha, tb->palette,
                                         tb->n_palette, &chk);
    if (st != LW_OK) return st;
    if (std::memcmp(&chk, tb, offsetof(lw_table, reserved1)) != 0)
      return fail(LW_ERR_CORRUPT, "decoder table does not match its code lengths");
  }
  if (d->fmt == LW_FMT_BF16_EXP) {
    const int64_t G = d->cols / 64, GW = (G + 31) / 32;
    if (s->bytes[LW_SEC_VFLAGS] != (uint64_t)(d->rows * GW * 4) ||
        s->bytes[LW_SEC_VROW_OFF] != (uint64_t)(d->rows + 1) * 4 ||
        s->bytes[LW_SEC_SIGNMAN] != (uint64_t)n_tiles * 16384)
      return fail(LW_ERR_CORRUPT, "BF16 section sizes do not match the shape");
    const uint32_t* vf = (const uint32_t*)s->ptr[LW_SEC_VFLAGS];
    const uint32_t* vo = (const uint32_t*)s->ptr[LW_SEC_VROW_OFF];
    uint64_t nv = 0;
    for (int64_t r = 0; r < d->rows; ++r) {
      if (vo[r] != nv) return fail(LW_ERR_CORRUPT, "vrow_off wrong at row %lld", (long long)r);
      for (int64_t w = 0; w < GW; ++w) nv += (uint64_t)__builtin_popcount(vf[r * GW + w]);
    }
    if (vo[d->rows] != nv || s->bytes[LW_SEC_VEXP] != nv * 64)
      return fail(LW_ERR_CORRUPT, "verbatim count mismatch");
  } else if (s->bytes[LW_SEC_QPARAMS] != (uint64_t)n_tiles * qparam_tile_bytes(d->fmt)) {
    return fail(LW_ERR_CORRUPT, "qparams size does not match the shape");
  }
  return LW_OK;
}

extern "C" const char* lw_status_string(lw_status s) {
  switch (s) {
    case LW_OK: return "LW_OK";
    case LW_ERR_INVALID_ARG: return "LW_ERR_INVALID_ARG";
    case LW_ERR_SHAPE: return "LW_ERR_SHAPE";
    case LW_ERR_UNSUPPORTED: return "LW_ERR_UNSUPPORTED";
    case LW_ERR_ALLOC: return "LW_ERR_ALLOC";
    case LW_ERR_CORRUPT: return "LW_ERR_CORRUPT";
    case LW_ERR_CUDA: return "LW_ERR_CUDA";
    case LW_ERR_IO: return "LW_ERR_IO";
  }
  return "unknown lw_status";
}

extern "C" const char* lw_last_error(void) { return g_err.c_str(); }

extern "C" int32_t lw_table_lut_entries(const lw_table* t) {
  if (!t || t->lmin < 1 || t->lmax > LW_MAX_CODE_LEN || t->lmin > t->lmax) return 0;
  return lw::lut_shape(t->lim_m1, t->lmin, t->lmax).n;
}

extern "C" int32_t lw_version(void) { return 4; }
