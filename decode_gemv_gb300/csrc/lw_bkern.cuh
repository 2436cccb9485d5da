// Kernels for BF16 weights whose exponent byte is Huffman-coded over the
// matrix's top-16 palette ("Unweight: Compressing LLM Weights for Faster
// Inference", "The exponent's exploitable redundancy"; reconstruction in fast
// on-chip memory, "How reconstructive matmul works"), laid out in the tiles
// and lanes of "LazyWeights" ("2 . Code them", Fig. 3(a)).
//
// Per tile (64 rows x 256 columns) and lane (rows 2l, 2l+1): the coded
// palette indices of the lane's non-verbatim 64-column groups, row 2l first;
// verbatim groups' raw exponent bytes come from a side array; every weight's
// sign+mantissa byte is stored raw (16-byte chunks interleaved over lanes).
// The fp32 value of a weight is built in registers from its exponent and
// its sign+mantissa byte:  f32 = (sm & 0x80) << 24 | exp << 23 | (sm & 0x7F) << 16
// -- one byte permute and one three-input logic op.
//
// Same machinery as the 4-/6-bit kernels: two-warp CTAs (warp h decodes row
// 2l + h of lane l), the tile's coded rows, activations and second-row
// offsets staged in shared memory by bulk asynchronous copies, the table
// bulk-copied and checked lane-parallel, the multiply-add comparator, FFMA2
// accumulation (even / odd columns), ordered split-K through the last tile
// of each strip.  The twin reads a
// fixed 4-bit palette index per weight ([UW] "direct palette").
#pragma once

#include "lw_qkern.cuh"

namespace lw {
namespace dev {

struct BArgs {
  const uint32_t* words;
  const uint32_t* tile_off;
  const uint16_t* lane_bits;
  const uint16_t* lane_mid;
  const lw_table* table;
  const uint8_t* signman;   // [n_tiles][32 chunks][32 lanes][16 B]
  const uint32_t* vflags;   // [N][GW]
  const uint32_t* vrow_off; // [N + 1]
  const uint8_t* vexp;      // [n_verbatim][64]
  const uint16_t* x;        // bf16 [batch][K]
  float* ws;
  uint32_t* counters;
  float* y;
  uint16_t* out;            // decode only: bf16 bits [N][K]
  int32_t* status;
  int n_tiles, TK, N, K, GW, batch;
  int stage_rows, stage_bytes;
  int x_offset, mid_offset, xf_offset;   // byte offsets inside a stage
  // tensor-core product only
  int bpad, tmem_cols, slab_off, xs_off, wstage_off;
  int lut_off, lut_cap;   // table-driven decode: replicated table (bytes, entries)
};

// shared-memory map (bytes) for the CUDA-core BF16 kernels: the 4-/6-bit
// map (offsets, flag, barriers, raw table, stage), with the exponent table
// in place of the symbol values
constexpr int kBTabOff = 128;     // uint32 exp << 23 per canonical index (16) / palette index

// Copies of tile t (coded rows [r0, r1)): its words, activations (bf16) and
// second-row offsets.
// Copies of tile t's activation rows (bf16) on a barrier whose expected
// bytes already include them (lane 0).
__device__ __forceinline__ void b_issue_x(const BArgs& a, int t, uint8_t* stage, uint64_t* bar,
                                          int lane) {
  if (lane != 0) return;
  const int kt = t % a.TK;
  for (int b = 0; b < a.batch; ++b)
    bulk_g2s(stage + a.x_offset + b * 512, a.x + (size_t)b * a.K + (size_t)kt * 256, 512, bar);
}

template <bool PRODUCT, bool TWIN>
__device__ __forceinline__ bool b_issue(const BArgs& a, int t, uint32_t r0, uint32_t r1,
                                        uint8_t* stage, uint64_t* bar, int lane,
                                        bool with_x = true) {
  const bool fits = r1 >= r0 && r1 - r0 <= (uint32_t)(a.stage_rows - kLookahead);
  if (lane == 0) {
    const uint32_t wbytes = fits ? (r1 - r0) * 128u : 0u;
    const uint32_t xbytes = PRODUCT ? (uint32_t)a.batch * 512u : 0u;
    const uint32_t mbytes = TWIN ? 0u : 64u;
    mbar_arrive_expect_tx(bar, wbytes + xbytes + mbytes);
    if (wbytes) bulk_g2s(stage, a.words + (size_t)r0 * 32, wbytes, bar);
    if (mbytes) bulk_g2s(stage + a.mid_offset, a.lane_mid + (size_t)t * 32, 64, bar);
  }
  if (PRODUCT && with_x) b_issue_x(a, t, stage, bar, lane);
  return fits;
}

// fp32 bits of a weight from its exponent field (e23 = exp << 23) and the
// sign+mantissa byte K of word w.
template <int K>
__device__ __forceinline__ float b_value(uint32_t w, uint32_t e23) {
  // bytes of t: [0, 0, b, b's sign replicated] (prmt selector bit 3 = sign)
  constexpr uint32_t sel = 0x44u | ((uint32_t)K << 8) | (((uint32_t)K | 8u) << 12);
  uint32_t t;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(w), "r"(0u), "r"(sel));
  return __uint_as_float((t & 0x807F0000u) | e23);
}

// Per-row verbatim information of a lane for tile column kt: 4 flag bits
// (groups 4kt .. 4kt+3) and the index of the row's first verbatim group at
// or after group 4kt.
__device__ __forceinline__ void b_row_flags(const BArgs& a, size_t r, int kt, uint32_t& fw,
                                            uint32_t& vbase) {
  const int g0 = 4 * kt;
  const uint32_t* f = a.vflags + r * (size_t)a.GW;
  uint32_t before = 0;
  for (int w = 0; w < g0 / 32; ++w) before += __popc(__ldg(f + w));
  const uint32_t cur = __ldg(f + g0 / 32);
  before += __popc(cur & ((1u << (g0 % 32)) - 1u));
  fw = (cur >> (g0 % 32)) & 15u;
  vbase = __ldg(a.vrow_off + r) + before;
}

// Chunk c (16 weights) of group g of row h: this lane's 16 sign+mantissa bytes.
__device__ __forceinline__ uint4 b_load_sm(const BArgs& a, int t, int lane, int h, int k) {
  const uint4* base = reinterpret_cast<const uint4*>(a.signman + (size_t)t * 16384);
  return __ldg(base + (16 * h + k) * 32 + lane);
}

// Chunk c of verbatim group idx: its 16 raw exponent bytes.
__device__ __forceinline__ uint4 b_load_vexp(const BArgs& a, uint32_t idx, int c) {
  return __ldg(reinterpret_cast<const uint4*>(a.vexp + (size_t)idx * 64) + c);
}

__device__ __forceinline__ uint32_t u4w(const uint4& v, int q) {
  return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
}

// exponent field (exp << 23) of byte K of word w (verbatim groups)
template <int K>
__device__ __forceinline__ uint32_t b_vexp23(uint32_t w) {
  return ((w >> (8 * K)) & 0xFFu) << 23;
}

// Exponent fields (exp << 23) of weights 2p, 2p+1 of chunk k of this lane's
// row h: from the verbatim bytes `ve` in a verbatim group (v), else decoded
// (coded) or read as a palette index (twin).  Branch-free in v: the coded
// stream is read in every lane and advances only in coded groups.  Returns
// the larger of the two table addresses used (phantom-entry check).
template <bool TWIN, int NP>
__device__ __forceinline__ uint32_t b_exponents(LaneBits& lb, const Cmp<NP>& cmp, int lmin,
                                                uint32_t s_off, uint32_t s_tab, uint32_t wb, int h,
                                                int lane, int k, int p, bool v, const uint4& ve,
                                                uint32_t& E0, uint32_t& E1) {
  uint32_t e0, e1;
  if (!TWIN) {
    q_decode2<NP, 4>(lb, cmp, lmin, s_off, e0, e1, v);
  } else {
    // direct palette: word j of the lane holds indices 8j..8j+7 (MSB first)
    const int q0 = 16 * k + 2 * p;               // index within the row
    const uint32_t wa = lds_u32(wb + (uint32_t)((32 * h + (q0 >> 3)) * 128 + 4 * lane));
    const int sh = 28 - 4 * (q0 & 7);
    e0 = s_tab + 4u * ((wa >> sh) & 15u);
    e1 = s_tab + 4u * ((wa >> (sh - 4)) & 15u);
  }
  const uint32_t t0 = lds_u32(e0), t1 = lds_u32(e1);
  const uint32_t wv = u4w(ve, p >> 1);
  E0 = v ? ((p & 1) ? b_vexp23<2>(wv) : b_vexp23<0>(wv)) : t0;
  E1 = v ? ((p & 1) ? b_vexp23<3>(wv) : b_vexp23<1>(wv)) : t1;
  return e0 > e1 ? e0 : e1;
}

// ---------------------------------------------------------------------------
// Shared prologue of the CUDA-core BF16 kernels (two-warp CTAs): barriers,
// the table copy and check, the exponent table.  Returns false (after
// reporting) if the CTA must stop; the first tile's copy is issued here.
// ---------------------------------------------------------------------------
template <bool TWIN, int NCMP, bool PRODUCT>
__device__ __forceinline__ bool b_prologue(const BArgs& a, uint8_t* smem, uint64_t* bar, int t,
                                           bool& fit, int lane) {
  const bool lead = threadIdx.x == 0;
  const lw_table* tb = reinterpret_cast<const lw_table*>(smem + kRawTabOff);
  if (lead) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[2], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (lead) table_issue(smem + kRawTabOff, a.table, &bar[2]);
  fit = true;
  if (t < a.n_tiles)   // the bundle part now, the activations after the wait below
    fit = b_issue<PRODUCT, TWIN>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1),
                                 smem + kStageOff, &bar[0], lead ? 0 : 1, false);
  const bool got = __syncthreads_and(mbar_wait(&bar[2], 0u));
  const bool ok = got && (TWIN || __syncthreads_and(table_ok_warp(tb, LW_FMT_BF16_EXP, 16, NCMP, lane)));
  if (!ok) {
    if (lead) report(a.status, got ? LW_DEV_BAD_TABLE : LW_DEV_TIMEOUT);
    if (!got) mbar_wait(&bar[2], 0u);
    if (t < a.n_tiles) {   // (the first tile's barrier expects the activations too)
      pdl_wait();
      if (PRODUCT) b_issue_x(a, t, smem + kStageOff, &bar[0], lead ? 0 : 1);
      mbar_wait(&bar[0], 0u);
    }
    return false;
  }
  // coded: offsets and exp << 23 per canonical index; twin: per palette index
  const uint32_t s_tab = smem_addr(smem) + kBTabOff;
  if (threadIdx.x < 16) {
    if (!TWIN) {
      put_off<(NCMP + 1) / 2>(reinterpret_cast<uint32_t*>(smem + kOffOff), threadIdx.x,
                              s_tab + (uint32_t)(4 * (threadIdx.x < 12 ? tb->off[threadIdx.x] : 0)));
      const uint32_t sy = tb->sym[threadIdx.x] & 15u;
      reinterpret_cast<uint32_t*>(smem + kBTabOff)[threadIdx.x] = (uint32_t)tb->palette[sy] << 23;
    } else {
      reinterpret_cast<uint32_t*>(smem + kBTabOff)[threadIdx.x] =
          (uint32_t)tb->palette[threadIdx.x] << 23;
    }
  }
  __syncthreads();
  pdl_wait();
  if (PRODUCT && t < a.n_tiles) b_issue_x(a, t, smem + kStageOff, &bar[0], lead ? 0 : 1);
  return true;
}

// ---------------------------------------------------------------------------
// Fused product (CUDA cores), persistent grid of two-warp CTAs: lane l of
// warp h handles row 2l + h of each tile.
// ---------------------------------------------------------------------------
template <bool TWIN, int BP, int NCMP>
__global__ void __launch_bounds__(64, 12) b_product_kernel(const BArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  const uint32_t s_off = sbase + kOffOff;
  const uint32_t s_tab = sbase + kBTabOff;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const lw_table* tb = reinterpret_cast<const lw_table*>(smem + kRawTabOff);
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool lead = threadIdx.x == 0;
  uint8_t* stage = smem + kStageOff;
  const int nw = gridDim.x;
  int t = blockIdx.x;
  uint32_t par = 0u;
  bool fit = true;
  if (!b_prologue<TWIN, NCMP, true>(a, smem, bar, t, fit, lane)) return;
  constexpr int NP = (NCMP + 1) / 2;
  Cmp<NP> cmp;
  int lmin = 1;
  if (!TWIN) {
    cmp.load(tb, tb->lmax - tb->lmin);
    lmin = tb->lmin;
  }
  QArgs qa{};
  qa.ws = a.ws;
  qa.counters = a.counters;
  qa.y = a.y;
  qa.N = a.N;
  qa.TK = a.TK;
  qa.batch = a.batch;

  for (; t < a.n_tiles; t += nw) {
    const bool more = t + nw < a.n_tiles;
    uint32_t nr0 = 0, nr1 = 0;
    if (more) {
      nr0 = __ldg(a.tile_off + t + nw);
      nr1 = __ldg(a.tile_off + t + nw + 1);
    }
    const int strip = t / a.TK, kt = t % a.TK;
    const size_t r = (size_t)strip * 64 + 2 * lane + h;
    // this row's verbatim flags and first sign+mantissa chunk (global loads
    // overlap the copy in flight)
    uint32_t fw, vb;
    b_row_flags(a, r, kt, fw, vb);
    uint4 n_sm = b_load_sm(a, t, lane, h, 0);
    uint4 n_ve = (fw & 1u) ? b_load_vexp(a, vb, 0) : make_uint4(0, 0, 0, 0);
    if (!__syncthreads_and(mbar_wait(&bar[0], par))) {
      if (lead) report(a.status, LW_DEV_TIMEOUT);
      return;
    }
    par ^= 1u;
    float part[BP];
#pragma unroll
    for (int b = 0; b < BP; ++b) part[b] = 0.f;
    const uint32_t wb = smem_addr(stage);
    if (fit) {
      // activations bf16 -> fp32 (both warps), rows >= batch are zero
      const uint32_t xs = wb + (uint32_t)a.x_offset;
      float* xf = reinterpret_cast<float*>(stage + a.xf_offset);
#pragma unroll
      for (int b = 0; b < BP; ++b) {
        for (int i = threadIdx.x; i < 128; i += 64) {
          const uint32_t two = b < a.batch ? lds_u32(xs + 512u * b + 4u * i) : 0u;
          xf[256 * b + 2 * i] = __uint_as_float(two << 16);
          xf[256 * b + 2 * i + 1] = __uint_as_float(two & 0xFFFF0000u);
        }
      }
    }
    __syncthreads();
    if (fit) {
      const uint32_t sx = wb + (uint32_t)a.xf_offset;
      LaneBits lb;
      uint32_t mid = 0;
      if (!TWIN) {
        mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        lb.init_at(wb, lane, a.stage_rows, h ? mid : 0u);
      }
      float2 acc[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) acc[b] = make_float2(0.f, 0.f);
      // 16 chunks of 16 weights (chunk k: group k/4, part k%4); the next
      // chunk's bytes are loaded while this one is processed
#pragma unroll 2
      for (int k = 0; k < 16; ++k) {
        const bool v = (fw >> (k >> 2)) & 1u;
        const uint4 sm = n_sm, ve = n_ve;
        if (k < 15) {
          const int k1 = k + 1, g1 = k1 >> 2;
          n_sm = b_load_sm(a, t, lane, h, k1);
          if ((fw >> g1) & 1u) n_ve = b_load_vexp(a, vb + __popc(fw & ((1u << g1) - 1u)), k1 & 3);
        }
#pragma unroll
        for (int p = 0; p < 8; ++p) {       // weights 2p, 2p+1 of the chunk
          uint32_t E0, E1;                   // exp << 23
          b_exponents<TWIN, NP>(lb, cmp, lmin, s_off, s_tab, wb, h, lane, k, p, v, ve, E0, E1);
          const uint32_t sw = u4w(sm, p >> 1);
          const float2 f = (p & 1) ? make_float2(b_value<2>(sw, E0), b_value<3>(sw, E1))
                                   : make_float2(b_value<0>(sw, E0), b_value<1>(sw, E1));
#pragma unroll
          for (int b = 0; b < BP; ++b)
            acc[b] = __ffma2_rn(f, lds_f2(sx + 1024u * b + 4u * (uint32_t)(16 * k + 2 * p)), acc[b]);
        }
      }
#pragma unroll
      for (int b = 0; b < BP; ++b) part[b] = acc[b].x + acc[b].y;
      if (!TWIN) {
        const uint32_t end = h ? (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane) : mid;
        if (lb.consumed() != end) report(a.status, LW_DEV_LANE_LENGTH);
      }
    } else if (lead) {
      report(a.status, LW_DEV_TILE_SIZE);
    }
    if (!more) pdl_trigger();   // last tile decoded (see q_product_kernel)
    fence_proxy_async();
    q_commit<BP>(qa, smem, strip, kt, (int)r, part);
    if (more)   // refill the stage (released by the commit's barrier)
      fit = b_issue<true, TWIN>(a, t + nw, nr0, nr1, stage, &bar[0], lead ? 0 : 1);
  }
}

// ---------------------------------------------------------------------------
// Decode only: bf16 bits [N][K]; two-warp CTAs, lane l of warp h restores
// row 2l + h of each tile.
// ---------------------------------------------------------------------------
template <bool TWIN, int NCMP>
__global__ void __launch_bounds__(64) b_decode_kernel(const BArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  const uint32_t s_off = sbase + kOffOff;
  const uint32_t s_tab = sbase + kBTabOff;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const lw_table* tb = reinterpret_cast<const lw_table*>(smem + kRawTabOff);
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool lead = threadIdx.x == 0;
  uint8_t* stage = smem + kStageOff;
  const int nw = gridDim.x;
  int t = blockIdx.x;
  uint32_t par = 0u;
  bool fit = true;
  if (!b_prologue<TWIN, NCMP, false>(a, smem, bar, t, fit, lane)) return;
  constexpr int NP = (NCMP + 1) / 2;
  Cmp<NP> cmp;
  int lmin = 1;
  uint32_t first_bad = 0u;   // table entries at or past it are phantom
  if (!TWIN) {
    cmp.load(tb, tb->lmax - tb->lmin);
    lmin = tb->lmin;
    first_bad = s_tab + 4u * (uint32_t)tb->n_sym;
  }
  for (; t < a.n_tiles; t += nw) {
    const bool more = t + nw < a.n_tiles;
    uint32_t nr0 = 0, nr1 = 0;
    if (more) {
      nr0 = __ldg(a.tile_off + t + nw);
      nr1 = __ldg(a.tile_off + t + nw + 1);
    }
    const int strip = t / a.TK, kt = t % a.TK;
    const size_t r = (size_t)strip * 64 + 2 * lane + h;
    uint32_t fw, vb;
    b_row_flags(a, r, kt, fw, vb);
    if (!__syncthreads_and(mbar_wait(&bar[0], par))) {
      if (lead) report(a.status, LW_DEV_TIMEOUT);
      return;
    }
    par ^= 1u;
    if (fit) {
      const uint32_t wb = smem_addr(stage);
      LaneBits lb;
      uint32_t mid = 0;
      if (!TWIN) {
        mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        lb.init_at(wb, lane, a.stage_rows, h ? mid : 0u);
      }
      bool bad = false;
      // each lane writes its row's 16 weights of a chunk as two 16-byte stores
      uint4* o = reinterpret_cast<uint4*>(a.out + r * a.K + (size_t)kt * 256);
      for (int k = 0; k < 16; ++k) {
        const int g = k >> 2;
        const bool v = (fw >> g) & 1u;
        const uint4 sm = b_load_sm(a, t, lane, h, k);
        const uint4 ve = v ? b_load_vexp(a, vb + __popc(fw & ((1u << g) - 1u)), k & 3)
                           : make_uint4(0, 0, 0, 0);
        uint32_t pw[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          uint32_t E0, E1;
          const uint32_t e = b_exponents<TWIN, NP>(lb, cmp, lmin, s_off, s_tab, wb, h, lane, k, p, v, ve,
                                                   E0, E1);
          if (!TWIN) bad |= !v && e >= first_bad;
          const uint32_t sw = u4w(sm, p >> 1);
          const uint32_t f0 = (p & 1) ? __float_as_uint(b_value<2>(sw, E0)) : __float_as_uint(b_value<0>(sw, E0));
          const uint32_t f1 = (p & 1) ? __float_as_uint(b_value<3>(sw, E1)) : __float_as_uint(b_value<1>(sw, E1));
          pw[p] = (f0 >> 16) | (f1 & 0xFFFF0000u);
        }
        o[2 * k] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        o[2 * k + 1] = make_uint4(pw[4], pw[5], pw[6], pw[7]);
      }
      if (!TWIN) {
        if (bad) report(a.status, LW_DEV_BAD_CODE);
        const uint32_t end = h ? (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane) : mid;
        if (lb.consumed() != end) report(a.status, LW_DEV_LANE_LENGTH);
      }
    } else if (lead) {
      report(a.status, LW_DEV_TILE_SIZE);
    }
    if (!more) pdl_trigger();
    fence_proxy_async();
    __syncthreads();   // both warps are done with the stage
    if (more) fit = b_issue<false, TWIN>(a, t + nw, nr0, nr1, stage, &bar[0], lead ? 0 : 1);
  }
}

}  // namespace dev
}  // namespace lw
