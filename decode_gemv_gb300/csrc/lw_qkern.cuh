// Kernels for 4-bit (pair-coded) and 6-bit Huffman-coded weights and their
// fixed-width twins: fused decode + GEMV/small-batch GEMM, and decode only.
//
// Method: "LazyWeights: Decode-on-Demand Edge LLMs" -- "2 . Code them" and
// Fig. 3(a) (64x256 tiles of 32 interleaved lanes of two rows), "3 . Decode on
// demand" and Fig. 3(b) (per lane: an 11-bit peek compared against per-length
// limits, the length's offset added to index the symbol table, the buffer
// shifted by the length), and the runtime paragraph after Fig. 3 (software
// decode fused into the GEMV; the fixed-width twin).
//
// GB300 mapping (ours, not the pages'):
//  * a persistent grid of two-warp CTAs; a CTA owns one tile at a time and
//    lane l of warp h decodes row 2l + h of the tile: lane l's first row
//    from the start of its stream, its second from the recorded mid offset,
//    so the tile's 64 rows run as 64 independent streams;
//  * each CTA stages its tiles in shared memory (one or two buffers), filled
//    by bulk asynchronous copies (TMA engine, no multicast) completed on an
//    mbarrier: the tile's coded rows, its scales/mins, the lanes' mid offsets
//    and the matching 256-column slice of every activation row; the decoder
//    table arrives the same way, once per CTA, and is checked lane-parallel;
//  * the interleave puts word j of lane l at shared word 32j + l, so every
//    lane's refill hits bank l: conflict-free however far lanes drift apart;
//  * a lane keeps three stream words in registers; one 32-bit window serves
//    two symbols (a code is at most 11 bits, so after the first code at
//    least 21 valid bits remain), and the words advance at most once per
//    symbol pair;
//  * comparator limits live in registers, two per word, tested by integer
//    multiply-adds on the FMA pipe (the integer ALU pipe, as busy, takes
//    the merges); per-length offsets (pre-scaled to shared addresses) and
//    the symbol table (pre-converted to fp32) in shared memory, read with
//    explicit ld.shared;
//  * dot products use packed fp32 FMA (FFMA2): even and odd columns in the
//    two halves;
//  * codes enter the FMA as the exact fp32 values 16 + c (4-bit) and 64 + c
//    (6-bit), which the twin builds from bits with one shift and one logic
//    op; the bias is removed once per row (4-bit: - 16 * sum x) or per group
//    (6-bit: - 96 * sum x, folding the code offset 32 in), so the twin and
//    the coded kernel execute the same floating-point operations and give
//    bitwise-equal results;
//  * split-K: each tile writes its partial sums to the workspace; the last
//    tile of a row strip to finish (an atomicInc counter that wraps back to
//    zero) adds the strip's partials in ascending tile order -- one launch,
//    deterministic.
#pragma once

#include "lw_dev.cuh"

namespace lw {
namespace dev {

struct QArgs {
  const uint32_t* words;
  const uint32_t* tile_off;
  const uint16_t* lane_bits;
  const uint16_t* lane_mid;  // coded bundles: bit where each lane's second row starts
  const lw_table* table;
  const uint8_t* qparams;
  const int32_t* strips; // products: 64-row strips to compute (n_tiles = entries x TK), or
                         // nullptr for every strip
  const float* x;        // [batch][K] (products)
  float* ws;             // partials [TK][batch][N] (products)
  uint32_t* counters;    // [N/64] strip counters (products), zero between calls
  float* y;              // [batch][N] (products)
  uint8_t* out;          // decode-only output
  int32_t* status;
  int n_tiles, TK, N, K, batch;
  int stage_rows;        // rows of 128 B per stage buffer = max_tile_rows + 3
  int stage_bytes;       // bytes per stage buffer (multiple of 128)
  int nstage;            // stage buffers per CTA: 2 (prefetch the next tile
                         // while decoding) or 1 (more resident CTAs)
  int mid_offset;        // byte offset of the tile's lane_mid copy in a stage
  // tensor-core product only
  int nsplit, bpad, tmem_cols, xs_off, wstage_off;
  // BF16 exponent bundles in the table-driven kernel (x then holds bf16)
  const uint8_t* signman;   // [n_tiles][32 chunks][32 lanes][16 B]
  const uint32_t* vflags;   // [N][GW]
  const uint32_t* vrow_off; // [N + 1]
  const uint8_t* vexp;      // [n_verbatim][64]
  int GW;
};

// The product kernel's launch: one matrix, or a group of independent
// matrices of one format decoded in one grid (their tiles concatenated, in
// order).  Passed as a grid constant: per-matrix fields are read from the
// constant bank by index.
constexpr int kMaxGroup = 8;
struct QLaunch {
  QArgs m[kMaxGroup];          // stage_rows, stage_bytes, nstage, mid_offset, batch
                               // and status agree across the group
  int first[kMaxGroup + 1];    // first global tile of each matrix; first[n] = total
  int n;
};

// Tile of the bundle behind list tile lt: with a strip list (a.strips not
// NULL), entry lt / TK names the strip and lt % TK the tile column; without
// one, lt itself.  An entry outside the
// matrix, or not above the previous entry, is invalid (ok = false): it maps
// to a tile of strip 0, which is read but whose results are dropped.
template <bool STRIPS>
__device__ __forceinline__ int list_tile(const QArgs& a, int lt, bool& ok) {
  if (!STRIPS || !a.strips) {
    ok = true;
    return lt;
  }
  const int si = lt / a.TK, kt = lt - si * a.TK;
  const int st = __ldg(a.strips + si);
  const int prev = si > 0 ? __ldg(a.strips + si - 1) : -1;
  ok = st >= 0 && st < a.N / 64 && st > prev;
  return ok ? st * a.TK + kt : kt;
}

// Advance `m` to the matrix holding global tile t (t never decreases).
__device__ __forceinline__ int group_seek(const QLaunch& g, int t, int m) {
  while (m + 1 < g.n && t >= g.first[m + 1]) ++m;
  return m;
}

constexpr int kQ4 = LW_FMT_Q4_PAIR, kQ6 = LW_FMT_Q6, kB16 = LW_FMT_BF16_EXP;

template <int FMT> struct QFmt;
template <> struct QFmt<LW_FMT_Q4_PAIR> {
  static constexpr int alpha = 256, qp_bytes = 256;
};
template <> struct QFmt<LW_FMT_Q6> {
  static constexpr int alpha = 64, qp_bytes = 2048;
};
template <> struct QFmt<LW_FMT_BF16_EXP> {
  static constexpr int alpha = 16, qp_bytes = 0;
};

// shared-memory map (bytes)
constexpr int kOffOff = 0;        // 64 B: offset table (BF16 kernels; the 4-/6-bit kernels keep it in static shared memory)
constexpr int kFlagOff = 64;      // int: "this CTA adds the strip's partials" broadcast
constexpr int kTabOff = 128;      // symbol values: float2[256] (4-bit) / float[64]; decode: uint32[256]
constexpr int kBarOff = 2176;     // uint64 mbarriers: stage 0, stage 1, table
constexpr int kRawTabOff = 2304;  // the bundle's lw_table, bulk-copied once per CTA
constexpr int kStageOff = 3328;   // one or two stage buffers
constexpr int kLookahead = 3;     // stream words a lane holds in registers
constexpr int kQThreads = 64;     // two warps per CTA, one per row of each lane
static_assert(kRawTabOff + (int)sizeof(lw_table) <= kStageOff, "shared-memory map");

__host__ __device__ constexpr int q_x_offset(int stage_rows, int qp_bytes) {
  return stage_rows * 128 + qp_bytes;
}

// Issue the copies of tile t, whose coded rows are [r0, r1), into one stage
// (thread `lead` issues; every caller gets the result).  Activation slices
// (products): xmode 1 = expected and copied now, 2 = expected, copied later
// by q_issue_x, 0 = none (the tensor-core path stages them itself).  Returns
// false if the tile is longer than the stage allows (the other copies are
// still issued, so the barrier completes).
// Copies of tile t's activation slices (products), on a barrier whose
// expected bytes already include them (thread `lead`).
template <int FMT>
__device__ __forceinline__ void q_issue_x(const QArgs& a, int t, uint8_t* stage, uint64_t* bar,
                                          bool lead) {
  if (!lead) return;
  const int kt = t % a.TK;
  uint8_t* xs = stage + q_x_offset(a.stage_rows, QFmt<FMT>::qp_bytes);
  for (int b = 0; b < a.batch; ++b)
    bulk_g2s(xs + b * 1024, a.x + (size_t)b * a.K + (size_t)kt * 256, 1024, bar);
}

template <int FMT, bool PRODUCT>
__device__ __forceinline__ bool q_issue(const QArgs& a, int t, uint32_t r0, uint32_t r1,
                                        uint8_t* stage, uint64_t* bar, bool lead,
                                        int xmode = 1) {
  const bool fits = r1 >= r0 && r1 - r0 <= (uint32_t)(a.stage_rows - kLookahead);
  if (lead) {
    const uint32_t wbytes = fits ? (r1 - r0) * 128u : 0u;
    constexpr uint32_t qpb = PRODUCT ? QFmt<FMT>::qp_bytes : 0u;
    const uint32_t xbytes = PRODUCT && xmode ? (uint32_t)a.batch * 1024u : 0u;
    const uint32_t mbytes = a.lane_mid ? 64u : 0u;
    mbar_arrive_expect_tx(bar, wbytes + qpb + xbytes + mbytes);
    if (wbytes) bulk_g2s(stage, a.words + (size_t)r0 * 32, wbytes, bar);
    if (PRODUCT) bulk_g2s(stage + a.stage_rows * 128, a.qparams + (size_t)t * qpb, qpb, bar);
    if (mbytes) bulk_g2s(stage + a.mid_offset, a.lane_mid + (size_t)t * 32, 64, bar);
  }
  if (PRODUCT && xmode == 1) q_issue_x<FMT>(a, t, stage, bar, lead);
  return fits;
}

// Start the bulk copy of the decoder table into shared memory at `dst`
// (one thread).
__device__ __forceinline__ void table_issue(uint8_t* dst, const lw_table* tb, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, (uint32_t)sizeof(lw_table));
  bulk_g2s(dst, tb, (uint32_t)sizeof(lw_table), bar);
}

// Checks of a staged table by one warp (every warp of a CTA may run them;
// they agree): the format, the length span fits the launch's comparator
// count, limits ascend, every limit below the longest length is even in
// 11-bit peek space (the comparator tests 10-bit peeks against limit / 2),
// and every window maps to an index inside the symbol table.  Lane j checks
// length index j.  True if the table is good.
__device__ __forceinline__ bool table_ok_warp(const lw_table* tb, int want_fmt, int want_alpha,
                                              int ncmp, int lane) {
  const int lmin = tb->lmin, lmax = tb->lmax;
  const int n_entries = tb->n_sym + (tb->phantom ? 1 : 0);
  bool ok = tb->fmt == want_fmt && tb->alpha == want_alpha && lmin >= 1 &&
            lmax <= LW_MAX_CODE_LEN && lmin <= lmax && lmax - lmin <= ncmp &&
            n_entries >= 1 && n_entries <= want_alpha;
  if (ok && lane < 12) {
    const int nl = lmax - lmin, j = lane;
    const uint32_t hi = tb->lim_m1[j];
    if (j >= nl) ok = ok && hi == 0xFFFFFFFFu;
    if (j < nl) ok = ok && ((((hi + 1u) >> 21) & 1u) == 0u);
    if (j <= nl) {
      const int L = lmin + j;
      const uint32_t prev_hi = j > 0 ? tb->lim_m1[j - 1] : 0u;
      if (j > 0) ok = ok && hi >= prev_hi && prev_hi != 0xFFFFFFFFu;
      const uint32_t cmax = hi >> (32 - L);
      const uint32_t cmin = j == 0 ? 0u : (prev_hi + 1u) >> (32 - L);
      const long long lo_idx = (long long)tb->off[j] + cmin;
      const long long hi_idx = (long long)tb->off[j] + cmax;
      ok = ok && lo_idx >= 0 && hi_idx < n_entries;
    }
  }
  return __all_sync(0xFFFFFFFFu, ok);
}

// Lane bit reader over a staged tile.  Registers cur:nxt:nx2 hold stream
// words j, j+1, j+2 where j = consumed / 32; pos = consumed % 32.
struct LaneBits {
  uint32_t cur, nxt, nx2;
  uint32_t wp;      // shared address of word j + 3 of this lane (may run past the stage)
  uint32_t w0;      // shared address of word 0 of this lane
  uint32_t wlast;   // last row this lane may read (clamp for corrupt streams)
  int pos;
  __device__ __forceinline__ void init(uint32_t wb, int lane, int stage_rows) {
    init_at(wb, lane, stage_rows, 0u);
  }
  // start at stream bit `bit` (clamped so that every read stays inside the
  // stage; a lane whose start was clamped fails its length check)
  __device__ __forceinline__ void init_at(uint32_t wb, int lane, int stage_rows, uint32_t bit) {
    uint32_t j0 = bit >> 5;
    if (j0 > (uint32_t)(stage_rows - kLookahead)) j0 = (uint32_t)(stage_rows - kLookahead);
    w0 = wb + 4u * (uint32_t)lane;
    cur = lds_u32(w0 + 128u * j0);
    nxt = lds_u32(w0 + 128u * (j0 + 1));
    nx2 = lds_u32(w0 + 128u * (j0 + 2));
    wp = w0 + 128u * (j0 + 3);
    wlast = w0 + (uint32_t)(stage_rows - 1) * 128u;
    pos = (int)(bit & 31u);
  }
  __device__ __forceinline__ uint32_t window() const { return __funnelshift_l(nxt, cur, pos); }
  // consume n (< 32) bits
  __device__ __forceinline__ void advance(int n) {
    pos += n;
    if (pos >= 32) {
      pos -= 32;
      cur = nxt;
      nxt = nx2;
      nx2 = lds_u32(min(wp, wlast));
      wp += 128u;
    }
  }
  __device__ __forceinline__ uint32_t consumed() const {
    return ((wp - w0) >> 7) * 32u + (uint32_t)pos - 96u;
  }
};

// The comparator: the number of per-length limits a window's code reaches.
// Every limit below the longest length is even in the 11-bit peek space, so
// the first 10 window bits p decide each test exactly: p reaches limit q
// when p >= t_q, t_q = limit_q / 2 (unused slots hold t = 1024, which no
// 10-bit peek reaches).  Two limits are tested by one integer multiply-add
// (the FMA pipe): word k holds two 11-bit fields, at bits k and 16 + k,
// each p + 1024 - t; such a field never exceeds 2047, so no field carries
// into the next, and its top bit (bit 10 + k, resp. 26 + k) is set exactly
// when p >= t.  The words' result bits sit at distinct positions; bit
// selects merge them into one word, a mask clears the rest (each field's
// low bits), and one population count gives the number of limits reached:
// the length is lmin + that count, and kScale = 4 times it is the byte
// offset of the length's entry in the offset table (32-bit entries).
template <int NP>
struct Cmp {
  static constexpr int kScale = 4;
  static_assert(NP <= 5, "at most 10 limits");
  uint32_t c[NP > 0 ? NP : 1];   // word k: (1024 - t_2k) << k | (1024 - t_2k+1) << (16 + k)
  __device__ __forceinline__ void load(const lw_table* tb, int ncmp) {
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      // lim_m1 = (limit << 21) - 1  ->  limit / 2 = (lim_m1 + 1) >> 22
      const uint32_t tl = 2 * k < ncmp ? ((tb->lim_m1[2 * k] + 1u) >> 22) : 1024u;
      const uint32_t th = 2 * k + 1 < ncmp ? ((tb->lim_m1[2 * k + 1] + 1u) >> 22) : 1024u;
      c[k] = ((1024u - tl) << k) | ((1024u - th) << (16 + k));
    }
  }
  static __device__ __forceinline__ uint32_t sel(uint32_t a, uint32_t b, uint32_t k) {
    return (a & k) | (b & ~k);
  }
  // a * B + c as one integer multiply-add
  template <uint32_t B>
  static __device__ __forceinline__ uint32_t imad(uint32_t a, uint32_t c) {
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "n"(B), "r"(c));
    return d;
  }
  // number of limits the window's code reaches
  __device__ __forceinline__ uint32_t count(uint32_t w) const {
    const uint32_t p = w >> 22;
    constexpr uint32_t R0 = (1u << 10) | (1u << 26);   // result bits of word 0
    uint32_t r[NP > 0 ? NP : 1];
    r[0] = imad<0x00010001u>(p, c[0]);
    if constexpr (NP > 1) r[1] = imad<0x00020002u>(p, c[1]);
    if constexpr (NP > 2) r[2] = imad<0x00040004u>(p, c[2]);
    if constexpr (NP > 3) r[3] = imad<0x00080008u>(p, c[3]);
    if constexpr (NP > 4) r[4] = imad<0x00100010u>(p, c[4]);
    uint32_t z;
    if constexpr (NP <= 1) {
      z = r[0] & R0;
    } else if constexpr (NP == 2) {
      z = sel(r[1], r[0], R0 << 1) & (R0 * 3u);
    } else if constexpr (NP == 3) {
      z = sel(r[2], sel(r[1], r[0], R0 << 1), R0 << 2) & (R0 * 7u);
    } else {
      z = sel(sel(r[1], r[0], R0 << 1), sel(r[3], r[2], R0 << 3), R0 * 3u);
      if constexpr (NP == 5) z = sel(r[4], z, R0 << 4) & (R0 * 31u);
      else z &= R0 * 15u;
    }
    return __popc(z);
  }
};

// Write the offset-table entry of length index c (count() returns its byte
// offset from the table start; the table spans 64 bytes).
template <int NP>
__device__ __forceinline__ void put_off(uint32_t* tab, int c, uint32_t v) {
  constexpr int S = Cmp<NP>::kScale;
  if (c * S < 64) tab[c * S / 4] = v;
}

// Decode two symbols from one window.  Returns the shared addresses of their
// symbol-table entries (entry size ESZ bytes).
// With `hold` set the reader does not advance (the lane's symbols come from
// elsewhere this step); the entries returned are then meaningless but valid
// shared addresses, so a warp decodes without branching on `hold`.
template <int NP, int ESZ>
__device__ __forceinline__ void q_decode2(LaneBits& lb, const Cmp<NP>& cmp, int lmin, uint32_t s_off,
                                          uint32_t& e0, uint32_t& e1, bool hold = false) {
  // on the dependency chain: count -> length (one add) -> next window;
  // the offset-table address is scaled off the chain
  const uint32_t w = lb.window();
  const uint32_t z0 = cmp.count(w);
  const int L0 = (int)z0 + lmin;
  const uint32_t w1 = w << L0;
  const uint32_t z1 = cmp.count(w1);
  const int L1 = (int)z1 + lmin;
  e0 = lds_u32(s_off + (uint32_t)Cmp<NP>::kScale * z0) + __funnelshift_l(w, 0u, L0) * ESZ;
  e1 = lds_u32(s_off + (uint32_t)Cmp<NP>::kScale * z1) + __funnelshift_l(w1, 0u, L1) * ESZ;
  lb.advance(hold ? 0 : L0 + L1);
}

// fp32 value 16 + c of a 4-bit code: shift the code to bits 19..22 (SH > 0:
// right shift, SH < 0: left shift) -- exact, one shift + one logic op.
template <int SH>
__device__ __forceinline__ float q4_twin_val(uint32_t w) {
  const uint32_t t = SH >= 0 ? (w >> SH) : (w << (-SH));
  return __uint_as_float(0x41800000u | (t & 0x00780000u));
}

// fp32 value 64 + c of the 6-bit code at bit offset O of (w0:w1:w2).
template <int O>
__device__ __forceinline__ float q6_twin_val(uint32_t w0, uint32_t w1, uint32_t w2) {
  constexpr int A = O / 32, B = O % 32;
  const uint32_t wa = A == 0 ? w0 : (A == 1 ? w1 : w2);
  const uint32_t wn = A == 0 ? w1 : w2;
  uint32_t t;
  if (B <= 26) t = B <= 9 ? (wa >> (9 - B)) : (wa << (B - 9));
  else t = __funnelshift_l(wn, wa, B) >> 9;
  return __uint_as_float(0x42800000u | (t & 0x007E0000u));
}

// Sum of the tile's 256 activations of one row (fixed order: 8 sequential
// per lane, then a butterfly; every lane takes lane 0's value).
__device__ __forceinline__ float tile_sum256(uint32_t sx, int lane) {
  const float4 u = lds_f4(sx + 32u * (uint32_t)lane);
  const float4 v = lds_f4(sx + 32u * (uint32_t)lane + 16u);
  float s = ((((((u.x + u.y) + u.z) + u.w) + v.x) + v.y) + v.z) + v.w;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, m);
  return __shfl_sync(0xFFFFFFFFu, s, 0);
}

// Sum of the 16 activations of group (lane & 15), sequential.
__device__ __forceinline__ float group_sum16(uint32_t sx, int lane) {
  const uint32_t p = sx + 64u * (uint32_t)(lane & 15);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 u = lds_f4(p + 16u * i);
    s = (((s + u.x) + u.y) + u.z) + u.w;
  }
  return s;
}

__device__ __forceinline__ uint32_t atom_inc_acq_rel(uint32_t* p, uint32_t wrap) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(wrap)
               : "memory");
  return old;
}

// One-warp version (a warp owns a tile; lane l holds rows 2l and 2l+1):
// partial sums of rows (row0, row0+1) for tile (strip, kt) -> workspace; the
// last tile of the strip to arrive adds all partials of the strip in
// ascending tile order and writes y.
template <int BP>
__device__ __forceinline__ void warp_commit(const QArgs& a, int strip, int kt, int lane,
                                         const float (&p0)[BP], const float (&p1)[BP]) {
  const int row0 = strip * 64 + 2 * lane;
#pragma unroll
  for (int b = 0; b < BP; ++b)
    if (b < a.batch)
      *reinterpret_cast<float2*>(a.ws + ((size_t)kt * a.batch + b) * a.N + row0) =
          make_float2(p0[b], p1[b]);
  // the warp barrier orders every lane's partials before lane 0's release;
  // the last arriver's acquire (then the barrier) orders the reads after it
  __syncwarp();
  uint32_t old = 0;
  if (lane == 0) old = atom_inc_acq_rel(a.counters + strip, (unsigned)(a.TK - 1));
  old = __shfl_sync(0xFFFFFFFFu, old, 0);
  if (old != (uint32_t)(a.TK - 1)) return;
  __syncwarp();
  for (int b = 0; b < a.batch; ++b) {
    const float* base = a.ws + (size_t)b * a.N + row0;
    const size_t step = (size_t)a.batch * a.N;
    float2 s = __ldcg(reinterpret_cast<const float2*>(base));
    for (int k0 = 1; k0 < a.TK; k0 += 8) {
      float2 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (k0 + i < a.TK) v[i] = __ldcg(reinterpret_cast<const float2*>(base + (size_t)(k0 + i) * step));
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (k0 + i < a.TK) { s.x += v[i].x; s.y += v[i].y; }
    }
    *reinterpret_cast<float2*>(a.y + (size_t)b * a.N + row0) = s;
  }
}

// Partial sums of row `row` (row 2l + h of strip `strip`) for tile column kt
// -> workspace; then the CTA's thread 0 counts the tile in, and the CTA that
// completes the strip adds all of its partials in ascending tile order and
// writes y.  Ends with the stage released (the barrier follows every read of
// it).
template <int BP>
__device__ __forceinline__ void q_commit(const QArgs& a, uint8_t* smem, int strip, int kt, int row,
                                         const float (&part)[BP], bool valid = true) {
  if (!valid) {   // an invalid strip-list entry: nothing to add (CTA-uniform)
    __syncthreads();
    return;
  }
#pragma unroll
  for (int b = 0; b < BP; ++b)
    if (b < a.batch) a.ws[((size_t)kt * a.batch + b) * a.N + row] = part[b];
  // the barrier orders both warps' partials before thread 0's release; the
  // last arriver's acquire (then the barrier) orders the reads after it
  __syncthreads();
  volatile int* flag = reinterpret_cast<volatile int*>(smem + kFlagOff);
  if (threadIdx.x == 0)
    *flag = atom_inc_acq_rel(a.counters + strip, (unsigned)(a.TK - 1)) == (uint32_t)(a.TK - 1);
  __syncthreads();
  if (!*flag) return;
  const size_t step = (size_t)a.batch * a.N;
  for (int b = 0; b < a.batch; ++b) {
    const float* base = a.ws + (size_t)b * a.N + row;
    float s = __ldcg(base);
    for (int k0 = 1; k0 < a.TK; k0 += 8) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (k0 + i < a.TK) v[i] = __ldcg(base + (size_t)(k0 + i) * step);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (k0 + i < a.TK) s += v[i];
    }
    a.y[(size_t)b * a.N + row] = s;
  }
}

// Stage the symbol table and the offsets of a checked table (whole CTA).
// ESZ = bytes per symbol entry; VAL converts a symbol to its entry.
template <int NP, int ESZ, class Val>
__device__ __forceinline__ void table_stage(uint8_t* smem, uint32_t* offtab, const lw_table* tb,
                                            int alpha, Val val) {
  const uint32_t s_tab = smem_addr(smem) + kTabOff;
  if (threadIdx.x < 16)
    put_off<NP>(offtab, threadIdx.x,
                s_tab + (uint32_t)(ESZ * (threadIdx.x < 12 ? tb->off[threadIdx.x] : 0)));
  for (int i = threadIdx.x; i < alpha; i += blockDim.x) val(i, (uint32_t)tb->sym[i]);
}

// ---------------------------------------------------------------------------
// Fused product kernel: one persistent grid of two-warp CTAs.
// ---------------------------------------------------------------------------
// resident CTAs per SM the register budget is sized for (more activation
// rows need more accumulator registers)
__host__ __device__ constexpr int q_min_ctas(int bp) { return bp <= 4 ? 16 : 12; }

template <int FMT, bool TWIN, int BP, int NCMP, bool STRIPS = false>
__global__ void __launch_bounds__(kQThreads, q_min_ctas(BP))
    q_product_kernel(const __grid_constant__ QLaunch g) {
  extern __shared__ __align__(128) uint8_t smem[];
  using F = QFmt<FMT>;
  constexpr int NP = (NCMP + 1) / 2;
  constexpr int ESZ = FMT == kQ4 ? 8 : 4;
  // unrolling of the decode loops: deeper for one activation row (more
  // steps in flight), shallower for more rows (their accumulators need the
  // registers)
  constexpr int kUnrollQ4 = BP == 1 ? 16 : 8;
  constexpr int kUnrollQ6 = BP == 1 ? 2 : 1;
  // offsets in static shared memory: their address is a link-time constant
  __shared__ __align__(16) uint32_t offtab[16];
  const uint32_t s_off = smem_addr(offtab);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const lw_table* tb = reinterpret_cast<const lw_table*>(smem + kRawTabOff);
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool lead = threadIdx.x == 0;
  const QArgs& u = g.m[0];   // fields shared by the group
  const int xoff = q_x_offset(u.stage_rows, F::qp_bytes);
  const int total = g.first[g.n];

  const bool two = u.nstage == 2;
  uint8_t* stage0 = smem + kStageOff;
  uint8_t* stage1 = two ? stage0 + u.stage_bytes : stage0;
  const int nw = gridDim.x;
  int t = blockIdx.x;
  // activation rows beyond `batch` stay zero in every stage
  for (int i = u.batch * 256 + threadIdx.x; i < BP * 256; i += kQThreads) {
    reinterpret_cast<float*>(stage0 + xoff)[i] = 0.f;
    reinterpret_cast<float*>(stage1 + xoff)[i] = 0.f;
  }
  if (lead) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar[2], 1);
    fence_barrier_init();
  }
  __syncthreads();
  // a strip list is written by earlier work on the stream: read it only
  // after that work is complete
  if (STRIPS) pdl_wait();
  // matrices of tiles t, t + nw, t + 2 nw
  int cm = group_seek(g, t, 0);
  int cn = group_seek(g, t + nw, cm);
  // the table and the first tile are copied at once
  if (!TWIN && lead) table_issue(smem + kRawTabOff, g.m[cm].table, &bar[2]);
  uint32_t par0 = 0u, par1 = 0u, tpar = 0u;
  bool fit0 = true, fit1 = true;
  if (t < total) {   // the bundle part now, the activations after the wait below
    const QArgs& a = g.m[cm];
    bool ok;
    const int rt = list_tile<STRIPS>(a, t - g.first[cm], ok);
    fit0 = q_issue<FMT, true>(a, rt, __ldg(a.tile_off + rt), __ldg(a.tile_off + rt + 1), stage0,
                              &bar[0], lead, 2);
  }
  // row range of the next tile to issue (t + nw), loaded one tile ahead
  uint32_t nr0 = 0, nr1 = 0;
  if (t + nw < total) {
    const QArgs& a = g.m[cn];
    bool ok;
    const int rt = list_tile<STRIPS>(a, t + nw - g.first[cn], ok);
    nr0 = __ldg(a.tile_off + rt);
    nr1 = __ldg(a.tile_off + rt + 1);
  }

  Cmp<NP> cmp;
  int lmin = 1;
  int tab_m = -1;   // matrix whose table is staged
  pdl_wait();
  if (t < total) q_issue_x<FMT>(g.m[cm], t - g.first[cm], stage0, &bar[0], lead);

  for (int it = 0; t < total; ++it, t += nw) {
    const QArgs& a = g.m[cm];
    const QArgs& an = g.m[cn];                 // matrix of tile t + nw
    bool valid, okn;
    const int lt = list_tile<STRIPS>(a, t - g.first[cm], valid);   // tile t within its matrix
    const int ltn = list_tile<STRIPS>(an, t + nw - g.first[cn], okn);
    const bool odd = two && (it & 1);
    const bool more = t + nw < total;
    const uint32_t ir0 = nr0, ir1 = nr1;     // rows of tile t + nw
    const int c2 = group_seek(g, t + 2 * nw, cn);
    if (t + 2 * nw < total) {
      const QArgs& a2 = g.m[c2];
      bool ok2;
      const int lt2 = list_tile<STRIPS>(a2, t + 2 * nw - g.first[c2], ok2);
      nr0 = __ldg(a2.tile_off + lt2);
      nr1 = __ldg(a2.tile_off + lt2 + 1);
    }
    if (!TWIN && cm != tab_m) {
      // this matrix's decoder table (copied now unless the prologue already
      // did); every reader of the previous one is past the commit's barriers
      if (tab_m >= 0 && lead) table_issue(smem + kRawTabOff, a.table, &bar[2]);
      const bool got = __syncthreads_and(mbar_wait(&bar[2], tpar));
      tpar ^= 1u;
      const bool ok = got && __syncthreads_and(table_ok_warp(tb, FMT, F::alpha, NCMP, lane));
      if (!ok) {
        if (lead) report(a.status, got ? LW_DEV_BAD_TABLE : LW_DEV_TIMEOUT);
        if (!got) mbar_wait(&bar[2], tpar ^ 1u);   // let the copies in flight land
        if (odd) mbar_wait(&bar[1], par1);
        else mbar_wait(&bar[0], par0);
        return;
      }
      table_stage<NP, ESZ>(smem, offtab, tb, F::alpha, [&](int i, uint32_t sy) {
        if (FMT == kQ4)
          reinterpret_cast<float2*>(smem + kTabOff)[i] =
              make_float2(16.f + (float)(sy & 15u), 16.f + (float)((sy >> 4) & 15u));
        else
          reinterpret_cast<float*>(smem + kTabOff)[i] = 64.f + (float)(sy & 63u);
      });
      cmp.load(tb, tb->lmax - tb->lmin);
      lmin = tb->lmin;
      __syncthreads();
      tab_m = cm;
    }
    // two stages: the other one was released by the barrier that closed the
    // previous tile
    if (two && more) {
      if (odd) fit0 = q_issue<FMT, true>(an, ltn, ir0, ir1, stage0, &bar[0], lead);
      else fit1 = q_issue<FMT, true>(an, ltn, ir0, ir1, stage1, &bar[1], lead);
    }
    uint8_t* st = odd ? stage1 : stage0;
    const bool got = odd ? mbar_wait(&bar[1], par1) : mbar_wait(&bar[0], par0);
    if (!__syncthreads_and(got)) {
      if (lead) report(a.status, LW_DEV_TIMEOUT);
      if (two && more) {   // let the copy in flight land before leaving
        if (odd) mbar_wait(&bar[0], par0);
        else mbar_wait(&bar[1], par1);
      }
      return;
    }
    if (odd) par1 ^= 1u; else par0 ^= 1u;
    const bool fit = odd ? fit1 : fit0;
    const int strip = lt / a.TK, kt = lt % a.TK;
    float part[BP];
#pragma unroll
    for (int b = 0; b < BP; ++b) part[b] = 0.f;
    const uint32_t wb = smem_addr(st);
    const uint32_t qp = wb + (uint32_t)a.stage_rows * 128u;
    const uint32_t sx = wb + (uint32_t)xoff;
    if (!fit) {
      if (lead) report(a.status, LW_DEV_TILE_SIZE);
    } else if (FMT == kQ4) {
      float S[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) S[b] = tile_sum256(sx + 1024u * b, lane);
      const uint32_t q2 = lds_u32(qp + 4u * (uint32_t)(2 * lane + h));   // scale | min << 16
      float2 acc[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) acc[b] = make_float2(0.f, 0.f);
      if (!TWIN) {
        // this lane's row as one stream: 128 pair symbols decoded two at a
        // time (the unrolled steps overlap: a step's decode does not wait for
        // the previous step's table reads)
        const uint32_t mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        LaneBits lb;
        lb.init_at(wb, lane, a.stage_rows, h ? mid : 0u);
#pragma unroll kUnrollQ4
        for (int j = 0; j < 64; ++j) {
          uint32_t e0, e1;
          q_decode2<NP, 8>(lb, cmp, lmin, s_off, e0, e1);
          const float2 v0 = lds_f2(e0), v1 = lds_f2(e1);
#pragma unroll
          for (int b = 0; b < BP; ++b) {
            const float4 xv = lds_f4(sx + 1024u * b + 16u * (uint32_t)j);
            acc[b] = __ffma2_rn(v0, make_float2(xv.x, xv.y), acc[b]);
            acc[b] = __ffma2_rn(v1, make_float2(xv.z, xv.w), acc[b]);
          }
        }
        const uint32_t end = h ? (uint32_t)__ldg(a.lane_bits + (size_t)lt * 32 + lane) : mid;
        if (lb.consumed() != end) report(a.status, LW_DEV_LANE_LENGTH);
      } else {
#pragma unroll 2
        for (int jj = 0; jj < 32; ++jj) {
          const uint32_t w = lds_u32(wb + (uint32_t)((32 * h + jj) * 128 + 4 * lane));
          const float2 v0 = make_float2(q4_twin_val<9>(w), q4_twin_val<5>(w));
          const float2 v1 = make_float2(q4_twin_val<1>(w), q4_twin_val<-3>(w));
          const float2 v2 = make_float2(q4_twin_val<-7>(w), q4_twin_val<-11>(w));
          const float2 v3 = make_float2(q4_twin_val<-15>(w), q4_twin_val<-19>(w));
#pragma unroll
          for (int b = 0; b < BP; ++b) {
            const float4 xa = lds_f4(sx + 1024u * b + 32u * jj);
            const float4 xb = lds_f4(sx + 1024u * b + 32u * jj + 16u);
            acc[b] = __ffma2_rn(v0, make_float2(xa.x, xa.y), acc[b]);
            acc[b] = __ffma2_rn(v1, make_float2(xa.z, xa.w), acc[b]);
            acc[b] = __ffma2_rn(v2, make_float2(xb.x, xb.y), acc[b]);
            acc[b] = __ffma2_rn(v3, make_float2(xb.z, xb.w), acc[b]);
          }
        }
      }
      const float sc = __half2float(__ushort_as_half((unsigned short)(q2 & 0xFFFFu)));
      const float mn = __half2float(__ushort_as_half((unsigned short)(q2 >> 16)));
#pragma unroll
      for (int b = 0; b < BP; ++b) part[b] = fmaf(sc, (acc[b].x + acc[b].y) - 16.f * S[b], mn * S[b]);
    } else {  // 6-bit
      float X[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) X[b] = group_sum16(sx + 1024u * b, lane);
      if (!TWIN) {
        const uint32_t mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        LaneBits lb;
        lb.init_at(wb, lane, a.stage_rows, h ? mid : 0u);
#pragma unroll kUnrollQ6
        for (int g = 0; g < 16; ++g) {
          float2 acc[BP];
#pragma unroll
          for (int b = 0; b < BP; ++b) acc[b] = make_float2(0.f, 0.f);
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            uint32_t e0, e1;
            q_decode2<NP, 4>(lb, cmp, lmin, s_off, e0, e1);
            const float2 v = make_float2(lds_f32(e0), lds_f32(e1));
#pragma unroll
            for (int b = 0; b < BP; ++b)
              acc[b] = __ffma2_rn(v, lds_f2(sx + 1024u * b + 64u * g + 8u * m), acc[b]);
          }
          // scale of group g of row 2l + h: chunk 2h + g/8, position g%8
          const uint32_t sa = qp + (uint32_t)((((2 * h + (g >> 3)) * 32) + lane) * 16 + 2 * (g & 7));
          const float sc = __half2float(__ushort_as_half((unsigned short)lds_u16(sa)));
#pragma unroll
          for (int b = 0; b < BP; ++b) {
            const float Xg = __shfl_sync(0xFFFFFFFFu, X[b], g);
            part[b] = fmaf(sc, (acc[b].x + acc[b].y) - 96.f * Xg, part[b]);
          }
        }
        const uint32_t end = h ? (uint32_t)__ldg(a.lane_bits + (size_t)lt * 32 + lane) : mid;
        if (lb.consumed() != end) report(a.status, LW_DEV_LANE_LENGTH);
      } else {
#pragma unroll 1
        for (int g = 0; g < 16; ++g) {
          float2 acc[BP];
#pragma unroll
          for (int b = 0; b < BP; ++b) acc[b] = make_float2(0.f, 0.f);
          const uint32_t r = (uint32_t)(48 * h + 3 * g);
          const uint32_t a0 = wb + r * 128u + 4u * lane;
          const uint32_t w0 = lds_u32(a0), w1 = lds_u32(a0 + 128u), w2 = lds_u32(a0 + 256u);
          float v[16];
          v[0] = q6_twin_val<0>(w0, w1, w2);    v[1] = q6_twin_val<6>(w0, w1, w2);
          v[2] = q6_twin_val<12>(w0, w1, w2);   v[3] = q6_twin_val<18>(w0, w1, w2);
          v[4] = q6_twin_val<24>(w0, w1, w2);   v[5] = q6_twin_val<30>(w0, w1, w2);
          v[6] = q6_twin_val<36>(w0, w1, w2);   v[7] = q6_twin_val<42>(w0, w1, w2);
          v[8] = q6_twin_val<48>(w0, w1, w2);   v[9] = q6_twin_val<54>(w0, w1, w2);
          v[10] = q6_twin_val<60>(w0, w1, w2);  v[11] = q6_twin_val<66>(w0, w1, w2);
          v[12] = q6_twin_val<72>(w0, w1, w2);  v[13] = q6_twin_val<78>(w0, w1, w2);
          v[14] = q6_twin_val<84>(w0, w1, w2);  v[15] = q6_twin_val<90>(w0, w1, w2);
#pragma unroll
          for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int b = 0; b < BP; ++b)
              acc[b] = __ffma2_rn(make_float2(v[2 * m], v[2 * m + 1]),
                                  lds_f2(sx + 1024u * b + 64u * g + 8u * m), acc[b]);
          const uint32_t sa = qp + (uint32_t)((((2 * h + (g >> 3)) * 32) + lane) * 16 + 2 * (g & 7));
          const float sc = __half2float(__ushort_as_half((unsigned short)lds_u16(sa)));
#pragma unroll
          for (int b = 0; b < BP; ++b) {
            const float Xg = __shfl_sync(0xFFFFFFFFu, X[b], g);
            part[b] = fmaf(sc, (acc[b].x + acc[b].y) - 96.f * Xg, part[b]);
          }
        }
      }
    }
    // the next kernel may start its prologue once every CTA has decoded its
    // last tile (earlier, its CTAs would crowd into the slots this grid leaves)
    if (!more) pdl_trigger();
    // this thread's reads of the stage come before the next bulk copy into it
    fence_proxy_async();
    q_commit<BP>(a, smem, strip, kt, strip * 64 + 2 * lane + h, part, valid);
    if (STRIPS && !valid && lead) report(a.status, LW_DEV_BAD_STRIPS);
    if (!two && more)   // single stage: refill it now (released by the commit's barrier)
      fit0 = q_issue<FMT, true>(an, ltn, ir0, ir1, stage0, &bar[0], lead);
    cm = cn;
    cn = c2;
  }
}

// ---------------------------------------------------------------------------
// Decode only: restore fixed-width codes to HBM.
//  Q4 -> packed bytes [N][K/2] (low nibble = even column); Q6 -> uint8 [N][K].
//  Two-warp CTAs; lane l of warp h restores row 2l + h of each tile.
// ---------------------------------------------------------------------------
template <int FMT, bool TWIN, int NCMP>
__global__ void __launch_bounds__(kQThreads) q_decode_kernel(const QArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  using F = QFmt<FMT>;
  constexpr int NP = (NCMP + 1) / 2;
  // offsets in static shared memory: their address is a link-time constant
  __shared__ __align__(16) uint32_t offtab[16];
  const uint32_t s_off = smem_addr(offtab);
  const uint32_t s_sym = smem_addr(smem) + kTabOff;   // uint32 per canonical index
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const lw_table* tb = reinterpret_cast<const lw_table*>(smem + kRawTabOff);
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool lead = threadIdx.x == 0;
  uint8_t* stage0 = smem + kStageOff;
  uint8_t* stage1 = stage0 + a.stage_bytes;
  const int nw = gridDim.x;
  int t = blockIdx.x;
  if (lead) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar[2], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (!TWIN && lead) table_issue(smem + kRawTabOff, a.table, &bar[2]);
  uint32_t par0 = 0u, par1 = 0u;
  bool fit0 = true, fit1 = true;
  if (t < a.n_tiles)
    fit0 = q_issue<FMT, false>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1), stage0,
                               &bar[0], lead);
  Cmp<NP> cmp;
  int lmin = 1;
  uint32_t first_bad = 0u;   // table entries at or past it are phantom
  if (!TWIN) {
    const bool got = __syncthreads_and(mbar_wait(&bar[2], 0u));
    const bool ok = got && __syncthreads_and(table_ok_warp(tb, FMT, F::alpha, NCMP, lane));
    if (!ok) {
      if (lead) report(a.status, got ? LW_DEV_BAD_TABLE : LW_DEV_TIMEOUT);
      if (!got) mbar_wait(&bar[2], 0u);        // let the copies in flight land
      if (t < a.n_tiles) mbar_wait(&bar[0], 0u);
      return;
    }
    table_stage<NP, 4>(smem, offtab, tb, 256, [&](int i, uint32_t sy) {
      reinterpret_cast<uint32_t*>(smem + kTabOff)[i] = sy;
    });
    cmp.load(tb, tb->lmax - tb->lmin);
    lmin = tb->lmin;
    first_bad = s_sym + 4u * (uint32_t)tb->n_sym;
    __syncthreads();
  }
  pdl_wait();
  if (t >= a.n_tiles) pdl_trigger();
  for (int it = 0; t < a.n_tiles; ++it, t += nw) {
    const bool odd = it & 1;
    const bool more = t + nw < a.n_tiles;
    if (more) {   // the other stage was released by the barrier closing the previous tile
      const uint32_t ir0 = __ldg(a.tile_off + t + nw), ir1 = __ldg(a.tile_off + t + nw + 1);
      if (odd) fit0 = q_issue<FMT, false>(a, t + nw, ir0, ir1, stage0, &bar[0], lead);
      else fit1 = q_issue<FMT, false>(a, t + nw, ir0, ir1, stage1, &bar[1], lead);
    }
    uint8_t* st = odd ? stage1 : stage0;
    const bool got = odd ? mbar_wait(&bar[1], par1) : mbar_wait(&bar[0], par0);
    if (!__syncthreads_and(got)) {
      if (lead) report(a.status, LW_DEV_TIMEOUT);
      if (more) {
        if (odd) mbar_wait(&bar[0], par0);
        else mbar_wait(&bar[1], par1);
      }
      return;
    }
    if (odd) par1 ^= 1u; else par0 ^= 1u;
    if (!(odd ? fit1 : fit0)) {
      if (lead) report(a.status, LW_DEV_TILE_SIZE);
    } else {
      const uint32_t wb = smem_addr(st);
      const int strip = t / a.TK, kt = t % a.TK;
      const size_t r = (size_t)strip * 64 + 2 * lane + h;
      LaneBits lb;
      uint32_t mid = 0;
      if (!TWIN) {
        mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        lb.init_at(wb, lane, a.stage_rows, h ? mid : 0u);
      }
      bool bad = false;
      // each lane writes its row in 16-byte stores (four packed words)
      uint32_t pw[4];
      if (FMT == kQ4) {
        uint4* o = reinterpret_cast<uint4*>(a.out + r * (a.K / 2) + (size_t)kt * 128);
#pragma unroll 4
        for (int q = 0; q < 32; ++q) {
          uint32_t packed = 0;
          if (!TWIN) {
#pragma unroll
            for (int i = 0; i < 4; i += 2) {
              uint32_t e0, e1;
              q_decode2<NP, 4>(lb, cmp, lmin, s_off, e0, e1);
              bad |= (e0 >= first_bad) | (e1 >= first_bad);
              packed |= (lds_u32(e0) & 0xFFu) << (8 * i);
              packed |= (lds_u32(e1) & 0xFFu) << (8 * i + 8);
            }
          } else {
            const uint32_t w = lds_u32(wb + (uint32_t)((32 * h + q) * 128 + 4 * lane));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t ce = (w >> (28 - 8 * i)) & 15u, co = (w >> (24 - 8 * i)) & 15u;
              packed |= (ce | (co << 4)) << (8 * i);
            }
          }
          pw[q & 3] = packed;
          if ((q & 3) == 3) o[q >> 2] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
      } else {
        uint4* o = reinterpret_cast<uint4*>(a.out + r * a.K + (size_t)kt * 256);
#pragma unroll 4
        for (int q = 0; q < 64; ++q) {
          uint32_t packed = 0;
          if (!TWIN) {
#pragma unroll
            for (int i = 0; i < 4; i += 2) {
              uint32_t e0, e1;
              q_decode2<NP, 4>(lb, cmp, lmin, s_off, e0, e1);
              bad |= (e0 >= first_bad) | (e1 >= first_bad);
              packed |= (lds_u32(e0) & 0x3Fu) << (8 * i);
              packed |= (lds_u32(e1) & 0x3Fu) << (8 * i + 8);
            }
          } else {
            // codes 256h + 4q .. +3 at stream bits 6*(256h + 4q): 24 bits
            const uint32_t bit = 6u * (256u * h + 4u * q);
            const uint32_t w0 = lds_u32(wb + (bit / 32) * 128u + 4u * lane);
            const uint32_t w1 = (bit / 32 + 1 < 96u) ? lds_u32(wb + (bit / 32 + 1) * 128u + 4u * lane) : 0u;
            const uint32_t win = __funnelshift_l(w1, w0, bit % 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) packed |= ((win >> (26 - 6 * i)) & 63u) << (8 * i);
          }
          pw[q & 3] = packed;
          if ((q & 3) == 3) o[q >> 2] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
      }
      if (!TWIN) {
        if (bad) report(a.status, LW_DEV_BAD_CODE);
        const uint32_t end = h ? (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane) : mid;
        if (lb.consumed() != end) report(a.status, LW_DEV_LANE_LENGTH);
      }
    }
    if (!more) pdl_trigger();   // last tile decoded (see q_product_kernel)
    fence_proxy_async();
    __syncthreads();   // both warps are done with this stage
  }
}

}  // namespace dev
}  // namespace lw
