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
// Same machinery as the 4-/6-bit kernels: one warp per tile, the tile's
// coded rows, activations and second-row offsets staged in shared memory by
// bulk asynchronous copies, the lane's two rows decoded as independent
// streams, an fp16x2 comparator, FFMA2 accumulation (even / odd columns),
// ordered split-K through the last tile of each strip.  The twin reads a
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
  int nsplit, bpad, tmem_cols, slab_off, xs_off, wstage_off;
};

// shared-memory map (bytes) for the BF16 kernels
constexpr int kBTabOff = 128;     // uint32 exp << 23 per canonical index (16) / palette index
constexpr int kBStageOff = 2304;  // per warp: one stage buffer

// Copies of tile t (coded rows [r0, r1)): its words, activations (bf16) and
// second-row offsets.
template <bool PRODUCT, bool TWIN>
__device__ __forceinline__ bool b_issue(const BArgs& a, int t, uint32_t r0, uint32_t r1,
                                        uint8_t* stage, uint64_t* bar, int lane) {
  const bool fits = r1 >= r0 && r1 - r0 <= (uint32_t)(a.stage_rows - kLookahead);
  if (lane == 0) {
    const uint32_t wbytes = fits ? (r1 - r0) * 128u : 0u;
    const uint32_t xbytes = PRODUCT ? (uint32_t)a.batch * 512u : 0u;
    const uint32_t mbytes = TWIN ? 0u : 64u;
    mbar_arrive_expect_tx(bar, wbytes + xbytes + mbytes);
    if (wbytes) bulk_g2s(stage, a.words + (size_t)r0 * 32, wbytes, bar);
    if (PRODUCT) {
      const int kt = t % a.TK;
      for (int b = 0; b < a.batch; ++b)
        bulk_g2s(stage + a.x_offset + b * 512, a.x + (size_t)b * a.K + (size_t)kt * 256, 512, bar);
    }
    if (mbytes) bulk_g2s(stage + a.mid_offset, a.lane_mid + (size_t)t * 32, 64, bar);
  }
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

// ---------------------------------------------------------------------------
// Fused product (CUDA cores), persistent grid of one-warp CTAs.
// ---------------------------------------------------------------------------
template <bool TWIN, int BP, int NCMP>
__global__ void __launch_bounds__(32, 12) b_product_kernel(const BArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  const uint32_t s_off = sbase + kOffOff;
  const uint32_t s_tab = sbase + kBTabOff;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const int lane = threadIdx.x & 31;
  uint8_t* stage = smem + kBStageOff;
  const int nw = gridDim.x;
  int t = blockIdx.x;

  if (lane == 0) {
    mbar_init(&bar[0], 1);
    fence_barrier_init();
  }
  __syncwarp();
  uint32_t par = 0u;
  bool fit = true;
  if (t < a.n_tiles)
    fit = b_issue<true, TWIN>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1), stage, bar,
                              lane);
  // table: coded -> exp << 23 per canonical index; twin -> per palette index
  if (!TWIN) {
    if (lane == 0) *reinterpret_cast<int*>(smem + kFlagOff) = table_ok(a.table, LW_FMT_BF16_EXP, 16, NCMP) ? 0 : 1;
    if (lane < 16) {
      put_off<(NCMP + 1) / 2>(reinterpret_cast<uint32_t*>(smem + kOffOff), lane,
          s_tab + (uint32_t)(4 * (lane < 12 ? a.table->off[lane] : 0)));
      const uint32_t sy = a.table->sym[lane] & 15u;
      reinterpret_cast<uint32_t*>(smem + kBTabOff)[lane] = (uint32_t)a.table->palette[sy] << 23;
    }
  } else if (lane < 16) {
    reinterpret_cast<uint32_t*>(smem + kBTabOff)[lane] = (uint32_t)a.table->palette[lane] << 23;
  }
  __syncwarp();
  if (!TWIN && *reinterpret_cast<volatile int*>(smem + kFlagOff)) {
    if (lane == 0) report(a.status, LW_DEV_BAD_TABLE);
    if (t < a.n_tiles) mbar_wait(&bar[0], 0u);
    return;
  }
  constexpr int NP = (NCMP + 1) / 2;
  Cmp<NP> cmp;
  int lmin = 1;
  if (!TWIN) {
    cmp.load(a.table, a.table->lmax - a.table->lmin);
    lmin = a.table->lmin;
  }

  for (; t < a.n_tiles; t += nw) {
    const bool more = t + nw < a.n_tiles;
    uint32_t nr0 = 0, nr1 = 0;
    if (more) {
      nr0 = __ldg(a.tile_off + t + nw);
      nr1 = __ldg(a.tile_off + t + nw + 1);
    }
    const int strip = t / a.TK, kt = t % a.TK;
    const size_t r0 = (size_t)strip * 64 + 2 * lane;
    // per-row verbatim flags (global loads overlap the copy in flight)
    uint32_t fw0, vb0, fw1, vb1;
    b_row_flags(a, r0, kt, fw0, vb0);
    b_row_flags(a, r0 + 1, kt, fw1, vb1);
    if (!mbar_wait(&bar[0], par)) {
      if (lane == 0) report(a.status, LW_DEV_TIMEOUT);
      return;
    }
    par ^= 1u;
    float part0[BP], part1[BP];
#pragma unroll
    for (int b = 0; b < BP; ++b) part0[b] = part1[b] = 0.f;
    if (fit) {
      const uint32_t wb = smem_addr(stage);
      // activations bf16 -> fp32 (this warp's copy), rows >= batch are zero
      __syncwarp();
      const uint32_t xs = wb + (uint32_t)a.x_offset;
      float* xf = reinterpret_cast<float*>(stage + a.xf_offset);
#pragma unroll
      for (int b = 0; b < BP; ++b) {
        for (int i = lane; i < 128; i += 32) {
          const uint32_t two = b < a.batch ? lds_u32(xs + 512u * b + 4u * i) : 0u;
          xf[256 * b + 2 * i] = __uint_as_float(two << 16);
          xf[256 * b + 2 * i + 1] = __uint_as_float(two & 0xFFFF0000u);
        }
      }
      __syncwarp();
      const uint32_t sx = wb + (uint32_t)a.xf_offset;
      LaneBits la, lr;
      uint32_t mid = 0;
      if (!TWIN) {
        mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        la.init(wb, lane, a.stage_rows);
        lr.init_at(wb, lane, a.stage_rows, mid);
      }
      float2 acc0[BP], acc1[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) acc0[b] = acc1[b] = make_float2(0.f, 0.f);
      // 16 chunks of 16 weights per row (chunk k: group k/4, part k%4); the
      // next chunk's bytes are loaded while this one is processed
      uint4 n_sm0 = b_load_sm(a, t, lane, 0, 0), n_sm1 = b_load_sm(a, t, lane, 1, 0);
      uint4 n_ve0 = (fw0 & 1u) ? b_load_vexp(a, vb0, 0) : make_uint4(0, 0, 0, 0);
      uint4 n_ve1 = (fw1 & 1u) ? b_load_vexp(a, vb1, 0) : make_uint4(0, 0, 0, 0);
#pragma unroll 1
      for (int k = 0; k < 16; ++k) {
        const int g = k >> 2;
        const bool v0 = (fw0 >> g) & 1u, v1 = (fw1 >> g) & 1u;
        const uint4 sm0 = n_sm0, sm1 = n_sm1, ve0 = n_ve0, ve1 = n_ve1;
        if (k < 15) {
          const int k1 = k + 1, g1 = k1 >> 2;
          n_sm0 = b_load_sm(a, t, lane, 0, k1);
          n_sm1 = b_load_sm(a, t, lane, 1, k1);
          if ((fw0 >> g1) & 1u) n_ve0 = b_load_vexp(a, vb0 + __popc(fw0 & ((1u << g1) - 1u)), k1 & 3);
          if ((fw1 >> g1) & 1u) n_ve1 = b_load_vexp(a, vb1 + __popc(fw1 & ((1u << g1) - 1u)), k1 & 3);
        }
#pragma unroll
        for (int p = 0; p < 8; ++p) {       // weights 2p, 2p+1 of the chunk
          uint32_t E[4];                     // exp << 23: row0 (2p, 2p+1), row1 (2p, 2p+1)
          const uint32_t wv0 = u4w(ve0, p >> 1), wv1 = u4w(ve1, p >> 1);
          if (!TWIN) {
            if (!v0) {
              uint32_t e0, e1;
              q_decode2<NP, 4>(la, cmp, lmin, s_off, e0, e1);
              E[0] = lds_u32(e0);
              E[1] = lds_u32(e1);
            } else {
              E[0] = (p & 1) ? b_vexp23<2>(wv0) : b_vexp23<0>(wv0);
              E[1] = (p & 1) ? b_vexp23<3>(wv0) : b_vexp23<1>(wv0);
            }
            if (!v1) {
              uint32_t e0, e1;
              q_decode2<NP, 4>(lr, cmp, lmin, s_off, e0, e1);
              E[2] = lds_u32(e0);
              E[3] = lds_u32(e1);
            } else {
              E[2] = (p & 1) ? b_vexp23<2>(wv1) : b_vexp23<0>(wv1);
              E[3] = (p & 1) ? b_vexp23<3>(wv1) : b_vexp23<1>(wv1);
            }
          } else {
            // direct palette: word j of the lane holds indices 8j..8j+7 (MSB first)
            const int q0 = 16 * k + 2 * p;               // index within the row
            const uint32_t wa = lds_u32(wb + (uint32_t)((q0 >> 3) * 128 + 4 * lane));
            const uint32_t wc = lds_u32(wb + (uint32_t)((32 + (q0 >> 3)) * 128 + 4 * lane));
            const int sh = 28 - 4 * (q0 & 7);
            E[0] = v0 ? ((p & 1) ? b_vexp23<2>(wv0) : b_vexp23<0>(wv0)) : lds_u32(s_tab + 4u * ((wa >> sh) & 15u));
            E[1] = v0 ? ((p & 1) ? b_vexp23<3>(wv0) : b_vexp23<1>(wv0)) : lds_u32(s_tab + 4u * ((wa >> (sh - 4)) & 15u));
            E[2] = v1 ? ((p & 1) ? b_vexp23<2>(wv1) : b_vexp23<0>(wv1)) : lds_u32(s_tab + 4u * ((wc >> sh) & 15u));
            E[3] = v1 ? ((p & 1) ? b_vexp23<3>(wv1) : b_vexp23<1>(wv1)) : lds_u32(s_tab + 4u * ((wc >> (sh - 4)) & 15u));
          }
          const uint32_t s0 = u4w(sm0, p >> 1), s1 = u4w(sm1, p >> 1);
          float2 f0, f1;
          if (p & 1) {
            f0 = make_float2(b_value<2>(s0, E[0]), b_value<3>(s0, E[1]));
            f1 = make_float2(b_value<2>(s1, E[2]), b_value<3>(s1, E[3]));
          } else {
            f0 = make_float2(b_value<0>(s0, E[0]), b_value<1>(s0, E[1]));
            f1 = make_float2(b_value<0>(s1, E[2]), b_value<1>(s1, E[3]));
          }
#pragma unroll
          for (int b = 0; b < BP; ++b) {
            const float2 xv = lds_f2(sx + 1024u * b + 4u * (uint32_t)(16 * k + 2 * p));
            acc0[b] = __ffma2_rn(f0, xv, acc0[b]);
            acc1[b] = __ffma2_rn(f1, xv, acc1[b]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < BP; ++b) {
        part0[b] = acc0[b].x + acc0[b].y;
        part1[b] = acc1[b].x + acc1[b].y;
      }
      if (!TWIN && (la.consumed() != mid ||
                    lr.consumed() != (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane)))
        report(a.status, LW_DEV_LANE_LENGTH);
    } else if (lane == 0) {
      report(a.status, LW_DEV_TILE_SIZE);
    }
    if (more) {   // refill the stage now, overlapping the commit
      __syncwarp();
      fence_proxy_async();
      fit = b_issue<true, TWIN>(a, t + nw, nr0, nr1, stage, bar, lane);
    }
    QArgs qa{};
    qa.ws = a.ws;
    qa.counters = a.counters;
    qa.y = a.y;
    qa.N = a.N;
    qa.TK = a.TK;
    qa.batch = a.batch;
    warp_commit<BP>(qa, strip, kt, lane, part0, part1);
  }
}

// ---------------------------------------------------------------------------
// Decode only: bf16 bits [N][K].
// ---------------------------------------------------------------------------
template <bool TWIN, int NCMP>
__global__ void __launch_bounds__(32) b_decode_kernel(const BArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  const uint32_t s_off = sbase + kOffOff;
  const uint32_t s_tab = sbase + kBTabOff;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const int lane = threadIdx.x & 31;
  uint8_t* stage = smem + kBStageOff;
  const int nw = gridDim.x;
  int t = blockIdx.x;
  if (lane == 0) {
    mbar_init(&bar[0], 1);
    fence_barrier_init();
  }
  __syncwarp();
  uint32_t par = 0u;
  bool fit = true;
  if (t < a.n_tiles)
    fit = b_issue<false, TWIN>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1), stage, bar,
                               lane);
  int n_sym = 16;
  if (!TWIN) {
    if (lane == 0) *reinterpret_cast<int*>(smem + kFlagOff) = table_ok(a.table, LW_FMT_BF16_EXP, 16, NCMP) ? 0 : 1;
    if (lane < 16) {
      put_off<(NCMP + 1) / 2>(reinterpret_cast<uint32_t*>(smem + kOffOff), lane,
          s_tab + (uint32_t)(4 * (lane < 12 ? a.table->off[lane] : 0)));
      const uint32_t sy = a.table->sym[lane] & 15u;
      reinterpret_cast<uint32_t*>(smem + kBTabOff)[lane] = (uint32_t)a.table->palette[sy] << 23;
    }
    n_sym = a.table->n_sym;
  } else if (lane < 16) {
    reinterpret_cast<uint32_t*>(smem + kBTabOff)[lane] = (uint32_t)a.table->palette[lane] << 23;
  }
  __syncwarp();
  if (!TWIN && *reinterpret_cast<volatile int*>(smem + kFlagOff)) {
    if (lane == 0) report(a.status, LW_DEV_BAD_TABLE);
    if (t < a.n_tiles) mbar_wait(&bar[0], 0u);
    return;
  }
  constexpr int NP = (NCMP + 1) / 2;
  Cmp<NP> cmp;
  int lmin = 1;
  if (!TWIN) {
    cmp.load(a.table, a.table->lmax - a.table->lmin);
    lmin = a.table->lmin;
  }
  const uint32_t first_bad = s_tab + 4u * (uint32_t)n_sym;
  for (; t < a.n_tiles; t += nw) {
    const bool more = t + nw < a.n_tiles;
    uint32_t nr0 = 0, nr1 = 0;
    if (more) {
      nr0 = __ldg(a.tile_off + t + nw);
      nr1 = __ldg(a.tile_off + t + nw + 1);
    }
    const int strip = t / a.TK, kt = t % a.TK;
    if (!mbar_wait(&bar[0], par)) {
      if (lane == 0) report(a.status, LW_DEV_TIMEOUT);
      return;
    }
    par ^= 1u;
    if (fit) {
      const uint32_t wb = smem_addr(stage);
      LaneBits la;
      if (!TWIN) la.init(wb, lane, a.stage_rows);
      bool bad = false, bad_len = false;
      for (int h = 0; h < 2; ++h) {
        const size_t r = (size_t)strip * 64 + 2 * lane + h;
        if (!TWIN && h == 1 && la.consumed() != lds_u16(wb + (uint32_t)a.mid_offset + 2u * lane))
          bad_len = true;
        uint32_t fw, vb;
        b_row_flags(a, r, kt, fw, vb);
        uint32_t* o = reinterpret_cast<uint32_t*>(a.out + r * a.K + (size_t)kt * 256);
        for (int k = 0; k < 16; ++k) {
          const int g = k >> 2;
          const bool v = (fw >> g) & 1u;
          const uint4 sm = b_load_sm(a, t, lane, h, k);
          const uint4 ve = v ? b_load_vexp(a, vb + __popc(fw & ((1u << g) - 1u)), k & 3)
                             : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            uint32_t E0, E1;
            const uint32_t wv = u4w(ve, p >> 1);
            if (v) {
              E0 = (p & 1) ? b_vexp23<2>(wv) : b_vexp23<0>(wv);
              E1 = (p & 1) ? b_vexp23<3>(wv) : b_vexp23<1>(wv);
            } else if (!TWIN) {
              uint32_t e0, e1;
              q_decode2<NP, 4>(la, cmp, lmin, s_off, e0, e1);
              bad |= (e0 >= first_bad) | (e1 >= first_bad);
              E0 = lds_u32(e0);
              E1 = lds_u32(e1);
            } else {
              const int q0 = 16 * k + 2 * p;
              const uint32_t wa = lds_u32(wb + (uint32_t)((32 * h + (q0 >> 3)) * 128 + 4 * lane));
              const int sh = 28 - 4 * (q0 & 7);
              E0 = lds_u32(s_tab + 4u * ((wa >> sh) & 15u));
              E1 = lds_u32(s_tab + 4u * ((wa >> (sh - 4)) & 15u));
            }
            const uint32_t s = u4w(sm, p >> 1);
            const uint32_t f0 = (p & 1) ? __float_as_uint(b_value<2>(s, E0)) : __float_as_uint(b_value<0>(s, E0));
            const uint32_t f1 = (p & 1) ? __float_as_uint(b_value<3>(s, E1)) : __float_as_uint(b_value<1>(s, E1));
            o[8 * k + p] = (f0 >> 16) | (f1 & 0xFFFF0000u);
          }
        }
      }
      if (!TWIN) {
        if (bad) report(a.status, LW_DEV_BAD_CODE);
        if (bad_len || la.consumed() != (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane))
          report(a.status, LW_DEV_LANE_LENGTH);
      }
    } else if (lane == 0) {
      report(a.status, LW_DEV_TILE_SIZE);
    }
    if (more) {
      __syncwarp();
      fence_proxy_async();
      fit = b_issue<false, TWIN>(a, t + nw, nr0, nr1, stage, bar, lane);
    }
  }
}

}  // namespace dev
}  // namespace lw
