// Load-time transcode of a Huffman-coded bundle into its fixed-width twin,
// on the device.
//
// "Unweight: Compressing LLM Weights for Faster Inference", "Four approaches
// to using compressed weights" (the palette pipelines: Huffman-coded
// exponents transcoded to 4-bit palette indices) and "One Format, Two
// Purposes" (the coded bundle is shipped; the runtime transcodes it at load
// time); the twin layout of "LazyWeights: Decode-on-Demand Edge LLMs" (the
// decode-free fixed-width layout of the same tiles and lanes, runtime
// paragraph after Fig. 3).
//
// The twin of a tile keeps the coded tile's lanes and interleave with every
// value at a fixed width w (4-bit codes: 4, 6-bit codes: 6, BF16 palette
// index: 4, zero in verbatim groups): lane l holds row 2l's 256 values then
// row 2l+1's, MSB-first, so row h of lane l fills words [h R, (h+1) R),
// R = 256 w / 32, of the tile's 2R word rows.  Lane l of warp h decodes row
// 2l + h of the staged coded tile (the comparator decoder of the product
// kernels) and writes its R words; the warp's 32 lanes write one 128-byte
// row per store.  The twin's tile offsets (t * 2R) and lane bit counts
// (512 w) are written too.  Every other twin section equals the coded
// bundle's.
#pragma once

#include "lw_qkern.cuh"

namespace lw {
namespace dev {

struct TArgs {
  const uint32_t* words;       // coded bundle
  const uint32_t* tile_off;
  const uint16_t* lane_bits;
  const uint16_t* lane_mid;
  const lw_table* table;
  const uint32_t* vflags;      // BF16
  uint32_t* tw_words;          // twin (written)
  uint32_t* tw_tile_off;
  uint16_t* tw_lane_bits;
  int32_t* status;
  int n_tiles, TK, GW;
  int stage_rows, stage_bytes, mid_offset;
};

template <int FMT> struct TFmt;
template <> struct TFmt<LW_FMT_Q4_PAIR> { static constexpr int alpha = 256, width = 4; };
template <> struct TFmt<LW_FMT_Q6> { static constexpr int alpha = 64, width = 6; };
template <> struct TFmt<LW_FMT_BF16_EXP> { static constexpr int alpha = 16, width = 4; };

// Copies of coded tile t (rows [r0, r1)) and its lane mids into one stage.
__device__ __forceinline__ bool t_issue(const TArgs& a, int t, uint32_t r0, uint32_t r1,
                                        uint8_t* stage, uint64_t* bar, bool lead) {
  const bool fits = r1 >= r0 && r1 - r0 <= (uint32_t)(a.stage_rows - kLookahead);
  if (lead) {
    const uint32_t wbytes = fits ? (r1 - r0) * 128u : 0u;
    mbar_arrive_expect_tx(bar, wbytes + 64u);
    if (wbytes) bulk_g2s(stage, a.words + (size_t)r0 * 32, wbytes, bar);
    bulk_g2s(stage + a.mid_offset, a.lane_mid + (size_t)t * 32, 64, bar);
  }
  return fits;
}

// byte with its two nibbles swapped: pair symbol (c_even | c_odd << 4) ->
// the two 4-bit codes in stream order (c_even first, MSB-first)
__device__ __forceinline__ uint32_t nib_swap(uint32_t s) { return ((s & 15u) << 4) | ((s >> 4) & 15u); }

template <int FMT, int NCMP>
__global__ void __launch_bounds__(kQThreads) t_transcode_kernel(const TArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NP = (NCMP + 1) / 2;
  constexpr int W = TFmt<FMT>::width;
  constexpr int R = 256 * W / 32;          // twin words per row
  __shared__ __align__(16) uint32_t offtab[16];
  const uint32_t s_off = smem_addr(offtab);
  const uint32_t s_sym = smem_addr(smem) + kTabOff;   // symbol per canonical index
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
  if (lead) table_issue(smem + kRawTabOff, a.table, &bar[2]);
  uint32_t par0 = 0u, par1 = 0u;
  bool fit0 = true, fit1 = true;
  if (t < a.n_tiles)
    fit0 = t_issue(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1), stage0, &bar[0], lead);
  const bool got = __syncthreads_and(mbar_wait(&bar[2], 0u));
  const bool ok = got && __syncthreads_and(table_ok_warp(tb, FMT, TFmt<FMT>::alpha, NCMP, lane));
  if (!ok) {
    if (lead) report(a.status, got ? LW_DEV_BAD_TABLE : LW_DEV_TIMEOUT);
    if (!got) mbar_wait(&bar[2], 0u);        // let the copies in flight land
    if (t < a.n_tiles) mbar_wait(&bar[0], 0u);
    return;
  }
  table_stage<NP, 4>(smem, offtab, tb, TFmt<FMT>::alpha, [&](int i, uint32_t sy) {
    reinterpret_cast<uint32_t*>(smem + kTabOff)[i] = sy;
  });
  Cmp<NP> cmp;
  cmp.load(tb, tb->lmax - tb->lmin);
  const int lmin = tb->lmin;
  const uint32_t first_bad = s_sym + 4u * (uint32_t)tb->n_sym;   // phantom entries
  __syncthreads();
  // the twin's tile offsets and lane bit counts
  for (int i = blockIdx.x * kQThreads + threadIdx.x; i <= a.n_tiles; i += nw * kQThreads)
    a.tw_tile_off[i] = (uint32_t)i * (uint32_t)(2 * R);
  for (int i = blockIdx.x * kQThreads + threadIdx.x; i < a.n_tiles * 32; i += nw * kQThreads)
    a.tw_lane_bits[i] = (uint16_t)(512 * W);

  for (int it = 0; t < a.n_tiles; ++it, t += nw) {
    const bool odd = it & 1;
    const bool more = t + nw < a.n_tiles;
    if (more) {   // the other stage was released by the barrier closing the previous tile
      const uint32_t ir0 = __ldg(a.tile_off + t + nw), ir1 = __ldg(a.tile_off + t + nw + 1);
      if (odd) fit0 = t_issue(a, t + nw, ir0, ir1, stage0, &bar[0], lead);
      else fit1 = t_issue(a, t + nw, ir0, ir1, stage1, &bar[1], lead);
    }
    // BF16: verbatim flags of this row's 4 groups in the tile
    uint32_t fw = 0;
    if (FMT == LW_FMT_BF16_EXP) {
      const size_t r = (size_t)(t / a.TK) * 64 + 2 * lane + h;
      const int g0 = 4 * (t % a.TK);
      fw = (__ldg(a.vflags + r * (size_t)a.GW + g0 / 32) >> (g0 % 32)) & 15u;
    }
    uint8_t* st = odd ? stage1 : stage0;
    const bool got_t = odd ? mbar_wait(&bar[1], par1) : mbar_wait(&bar[0], par0);
    if (!__syncthreads_and(got_t)) {
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
      const uint32_t mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
      LaneBits lb;
      lb.init_at(wb, lane, a.stage_rows, h ? mid : 0u);
      uint32_t* o = a.tw_words + ((size_t)t * (2 * R) + (size_t)h * R) * 32 + lane;
      bool bad = false;
      if (FMT == LW_FMT_Q4_PAIR) {
        // 128 pair symbols -> 32 words of 8 codes
#pragma unroll 2
        for (int q = 0; q < 32; ++q) {
          uint32_t e0, e1, e2, e3;
          q_decode2<NP, 4>(lb, cmp, lmin, s_off, e0, e1);
          q_decode2<NP, 4>(lb, cmp, lmin, s_off, e2, e3);
          bad |= (e0 >= first_bad) | (e1 >= first_bad) | (e2 >= first_bad) | (e3 >= first_bad);
          o[32 * q] = (nib_swap(lds_u32(e0)) << 24) | (nib_swap(lds_u32(e1)) << 16) |
                      (nib_swap(lds_u32(e2)) << 8) | nib_swap(lds_u32(e3));
        }
      } else if (FMT == LW_FMT_Q6) {
        // 256 codes of 6 bits -> 48 words; four codes (24 bits) per step
        uint64_t acc = 0;
        int nacc = 0, j = 0;
#pragma unroll 1
        for (int q = 0; q < 64; ++q) {
          uint32_t e0, e1, e2, e3;
          q_decode2<NP, 4>(lb, cmp, lmin, s_off, e0, e1);
          q_decode2<NP, 4>(lb, cmp, lmin, s_off, e2, e3);
          bad |= (e0 >= first_bad) | (e1 >= first_bad) | (e2 >= first_bad) | (e3 >= first_bad);
          const uint32_t v = ((lds_u32(e0) & 63u) << 18) | ((lds_u32(e1) & 63u) << 12) |
                             ((lds_u32(e2) & 63u) << 6) | (lds_u32(e3) & 63u);
          acc = (acc << 24) | v;
          nacc += 24;
          if (nacc >= 32) {
            nacc -= 32;
            o[32 * j++] = (uint32_t)(acc >> nacc);
          }
        }
      } else {
        // BF16: 4 groups of 64 weights; palette index per weight, 0 in a
        // verbatim group (the reader holds there: its symbols are not in
        // the stream)
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          const bool v = (fw >> g) & 1u;
#pragma unroll 1
          for (int q = 0; q < 8; ++q) {
            uint32_t word = 0;
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
              uint32_t e0, e1;
              q_decode2<NP, 4>(lb, cmp, lmin, s_off, e0, e1, v);
              bad |= !v && ((e0 >= first_bad) | (e1 >= first_bad));
              const uint32_t i0 = v ? 0u : (lds_u32(e0) & 15u), i1 = v ? 0u : (lds_u32(e1) & 15u);
              word |= (i0 << (28 - 4 * i)) | (i1 << (24 - 4 * i));
            }
            o[32 * (8 * g + q)] = word;
          }
        }
      }
      if (bad) report(a.status, LW_DEV_BAD_CODE);
      const uint32_t end = h ? (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane) : mid;
      if (lb.consumed() != end) report(a.status, LW_DEV_LANE_LENGTH);
    }
    fence_proxy_async();
    __syncthreads();   // both warps are done with this stage
  }
}

// An empty one-thread kernel, launched in plain stream order after the
// transcode: a kernel launched next with programmatic serialisation may run
// its prologue (which reads bundle sections) once this one has started, so
// only after the transcode has completed and its writes are visible.
__global__ void t_order_kernel() {}

}  // namespace dev
}  // namespace lw
