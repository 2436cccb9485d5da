// Table-driven canonical-code decoding on the GPU, shared by the
// table-driven product kernel (lw_qlut.cuh) and the BF16 tensor-core kernel
// (lw_btc.cuh).
//
// Method: "LazyWeights: Decode-on-Demand Edge LLMs", "3 . Decode on demand":
// an 11-bit peek of a lane's stream selects its codeword, the lane then
// shifts by the code's length.  Here the peek indexes a compact table
// (lw_lut.h) in shared memory, replicated once per lane (lane l's copy of
// entry i at table + 128 i + 4 l: a warp's 32 lookups are one conflict-free
// wavefront); an entry holds the length (bits 0..4) and the symbol in the
// form its kernel consumes.  One 32-bit window serves two symbols.
#pragma once

#include <cuda_fp16.h>

#include "lw_dev.cuh"
#include "lw_lut.h"

namespace lw {
namespace dev {

// a * b + c as one integer multiply-add (FMA pipe; the compiler would
// otherwise often use shift-and-add forms on the integer ALU pipe)
__device__ __forceinline__ uint32_t imad(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t shf_l_wrap(uint32_t lo, uint32_t hi, uint32_t n) {
  uint32_t d;
  asm("shf.l.wrap.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(lo), "r"(hi), "r"(n));
  return d;
}
__device__ __forceinline__ uint32_t shf_r_clamp(uint32_t lo, uint32_t hi, uint32_t n) {
  uint32_t d;
  asm("shf.r.clamp.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(lo), "r"(hi), "r"(n));
  return d;
}
// fp16 bit pattern of a small integer c (0..15), exactly.
__device__ __forceinline__ uint32_t f16_bits(uint32_t c) {
  return (uint32_t)__half_as_ushort(__uint2half_rn(c));
}

// Table entry of a 4-bit pair symbol / a 6-bit code of length L.
//  4-bit: low half = fp16(c_even) with L in its bits 0..4 (an fp16 of an
//  integer below 16 has its lowest 7 mantissa bits zero, so the junk is below
//  half an ulp of 1024 and the rounding add of 1024 in q4_vals removes it);
//  high half = fp16(c_odd).  Bits 0..4 of the entry are L and bit 5 is zero,
//  as the stream advance needs.
//  6-bit: high half = fp16(1024 + c), low half = L.
//  BF16 exponent: the palette's exponent byte at bits 23..30 (its place in
//  an fp32), L at bits 0..4.
__device__ __forceinline__ uint32_t lut_entry(const lw_table* tb, uint32_t sym, int L) {
  if (tb->fmt == LW_FMT_Q4_PAIR)
    return (f16_bits((sym >> 4) & 15u) << 16) | f16_bits(sym & 15u) | (uint32_t)L;
  if (tb->fmt == LW_FMT_BF16_EXP) return ((uint32_t)tb->palette[sym & 15u] << 23) | (uint32_t)L;
  return ((0x6400u | (sym & 63u)) << 16) | (uint32_t)L;
}

// Build the replicated table of a checked, staged lw_table: consumer warp w
// takes entries 32 w .. 32 w + 31, then 32 (w + NW) .., ...; lane j decodes
// entry i0 + j and stores its 32 copies (lane l's copy of entry i at
// table + 128 i + 4 l).
__device__ __forceinline__ void lut_build(const lw_table* tb, const LutShape& sh, uint32_t lut,
                                          int warp, int nw, int lane) {
  const int lmin = tb->lmin, lmax = tb->lmax;
  // the limits in registers (lim_m1[j] = all ones from lmax - lmin on)
  uint32_t lim[10];
#pragma unroll
  for (int j = 0; j < 10; ++j) lim[j] = tb->lim_m1[j];
  for (int i0 = warp * 32; i0 < sh.n; i0 += nw * 32) {
    // lane j decodes entry i0 + j
    uint32_t e = 0;
    const int i = i0 + lane;
    if (i < sh.n) {
      const uint32_t win = (uint32_t)lut_peek(sh, i) << 21;
      // the code's length: lmin plus the limits below the window
      int L = lmin;
#pragma unroll
      for (int j = 0; j < 10; ++j) L += (j < lmax - lmin && win > lim[j]) ? 1 : 0;
      const int idx = (int)(win >> (32 - L)) + tb->off[L - lmin];
      e = lut_entry(tb, tb->sym[idx], L);
      // the lane writes its entry's 32 copies, copy (lane + r) mod 32 at
      // step r: the warp's 32 stores of a step hit 32 different banks
      const uint32_t row = lut + (uint32_t)i * 128u;
#pragma unroll 8
      for (int r = 0; r < 32; ++r)
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(row + 4u * (uint32_t)((lane + r) & 31)), "r"(e)
                     : "memory");
    }
  }
}

// A lane's row stream: stream words cur (j), nxt (j + 1) and nx2 (j + 2),
// bit position pos (bits 0..4; bits 8 and up collect the table entries'
// other fields and are never read), wp = shared address of nx2.  The window
// of a step needs only cur and nxt; nx2, loaded a step ahead, keeps the
// shared-memory load off the decode's dependency chain.
struct LStream {
  uint32_t cur, nxt, nx2, pos, wp, w0, wlast;
  __device__ __forceinline__ void init(uint32_t wb, int lane, int stage_rows, uint32_t bit) {
    uint32_t j0 = bit >> 5;
    if (j0 > (uint32_t)(stage_rows - 3)) j0 = (uint32_t)(stage_rows - 3);   // corrupt start
    w0 = wb + 4u * (uint32_t)lane;
    wlast = w0 + (uint32_t)(stage_rows - 1) * 128u;
    cur = lds_u32(w0 + 128u * j0);
    nxt = lds_u32(w0 + 128u * (j0 + 1));
    wp = w0 + 128u * (j0 + 2);
    nx2 = lds_u32(wp);
    pos = bit & 31u;
  }
  __device__ __forceinline__ uint32_t consumed() const {
    return ((wp - w0) >> 7) * 32u - 64u + (pos & 31u);
  }
};

// Per-table decode constants (registers).
// Word q (compile-time after unrolling) of a 16-byte value.
__device__ __forceinline__ uint32_t l_word(const uint4& v, int q) {
  return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
}

// fp32 bits of a BF16 weight from its sign+mantissa byte K of word w and
// its exponent field E (exp << 23 in bits 23..30; other bits of E are
// ignored): the byte permute puts the byte's mantissa at bits 16..22 and its
// sign at bit 31; one logic op takes bits 23..30 from E.
template <int K>
__device__ __forceinline__ float b16_value(uint32_t w, uint32_t E) {
  constexpr uint32_t sel = 0x44u | ((uint32_t)K << 8) | (((uint32_t)K | 8u) << 12);
  uint32_t t;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(w), "r"(0u), "r"(sel));
  return __uint_as_float((t & 0x807FFFFFu) | (E & 0x7F800000u));
}

struct LDec {
  uint32_t lutl;   // shared address of entry 0, lane's copy
  int negC;
  uint32_t sh;     // 21 + s
};

// Decode the next two symbols of a stream: their table entries.  go = 0
// holds the stream where it is (the entries' lengths do not count: a BF16
// verbatim group has no symbols), go = 1 advances it -- a multiplier of the
// multiply-add that advances the position anyway (FMA pipe, no extra op).
//
// CLAMP keeps the next word's address inside the stage (for kernels whose
// stages are not followed by a guard; a corrupt stream then fails its
// length check without reading elsewhere).
template <bool CLAMP = false>
__device__ __forceinline__ void l_decode2(LStream& st, const LDec& d, uint32_t& e0, uint32_t& e1,
                                          uint32_t go = 1u) {
  const uint32_t w = shf_l_wrap(st.nxt, st.cur, st.pos);
  const int i0 = __viaddmax_s32((int)(w >> 21), d.negC, (int)(w >> d.sh));
  e0 = lds_u32(imad((uint32_t)i0, 128u, d.lutl));
  const uint32_t w1 = shf_l_wrap(0u, w, e0);
  const int i1 = __viaddmax_s32((int)(w1 >> 21), d.negC, (int)(w1 >> d.sh));
  e1 = lds_u32(imad((uint32_t)i1, 128u, d.lutl));
  const uint32_t p2 = imad(imad(e1, 1u, e0), go, st.pos);
  const uint32_t hb = p2 & 32u;   // 32 when the window moves on by a word
  st.pos = imad(hb, 0xFFFFFFFFu, p2);   // p2 - hb
  st.cur = shf_r_clamp(st.cur, st.nxt, hb);
  st.nxt = shf_r_clamp(st.nxt, st.nx2, hb);
  st.wp = imad(hb, 4u, st.wp);
  if (CLAMP) st.wp = st.wp < st.wlast ? st.wp : st.wlast;
  st.nx2 = lds_u32(st.wp);
}




}  // namespace dev
}  // namespace lw
