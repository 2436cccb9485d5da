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
//  * one warp owns one tile at a time; lane l decodes lane stream l;
//  * a persistent grid; each warp double-buffers its tiles in shared memory,
//    filled by bulk asynchronous copies (TMA engine, no multicast) completed
//    on an mbarrier: the tile's coded rows, its scales/mins and the matching
//    256-column slice of every activation row;
//  * the interleave puts word j of lane l at shared word 32j + l, so every
//    lane's refill hits bank l: conflict-free however far lanes drift apart;
//  * comparator limits live in registers, the per-length offsets and the
//    symbol table (pre-converted to fp32) in shared memory;
//  * dot products use packed fp32 FMA (FFMA2): even and odd columns in the
//    two halves;
//  * codes enter the FMA as the exact fp32 values 16 + c (4-bit) and 64 + c
//    (6-bit), which the twin builds from bits with one shift and one logic
//    op; the bias is removed once per row (4-bit: - 16 * sum x) or per group
//    (6-bit: - 96 * sum x, folding the code offset 32 in), so the twin and
//    the coded kernel execute the same floating-point operations and give
//    bitwise-equal results.
//  * per-tile partial sums go to a workspace; a second kernel adds them in
//    ascending tile order (deterministic split-K).
#pragma once

#include "lw_dev.cuh"

namespace lw {
namespace dev {

struct QArgs {
  const uint32_t* words;
  const uint32_t* tile_off;
  const uint16_t* lane_bits;
  const lw_table* table;
  const uint8_t* qparams;
  const float* x;        // [batch][K] (products)
  float* ws;             // [TK][batch][N] (products)
  uint8_t* out;          // decode-only output
  int32_t* status;
  int n_tiles, TK, N, K, batch;
  int stage_rows;        // rows of 128 B per stage buffer = max_tile_rows + 2
  int stage_bytes;       // bytes per stage buffer (multiple of 128)
};

constexpr int kQ4 = LW_FMT_Q4_PAIR, kQ6 = LW_FMT_Q6;

template <int FMT> struct QFmt;
template <> struct QFmt<LW_FMT_Q4_PAIR> {
  static constexpr int alpha = 256, nsym = 256, qp_bytes = 256, twin_rows = 64;
};
template <> struct QFmt<LW_FMT_Q6> {
  static constexpr int alpha = 64, nsym = 512, qp_bytes = 2048, twin_rows = 96;
};

// shared-memory map (bytes)
constexpr int kOffOff = 0;       // int[16]: per-length symbol offsets
constexpr int kFlagOff = 64;     // int: table rejected
constexpr int kTabOff = 128;     // symbol values: float2[256] (4-bit) / float[64]
constexpr int kBarOff = 2176;    // uint64 mbarriers, 2 per warp (<= 8 warps)
constexpr int kStageOff = 2304;  // per warp: two stage buffers

__host__ __device__ constexpr int q_x_offset(int stage_rows, int qp_bytes) {
  return stage_rows * 128 + qp_bytes;
}

// Issue the copies of tile t into one stage (called by the whole warp; lane 0
// issues).  Returns false if the tile is longer than the stage allows (the
// copies of everything else are still issued, so the barrier completes).
template <int FMT, bool PRODUCT>
__device__ __forceinline__ bool q_issue(const QArgs& a, int t, uint8_t* stage, uint64_t* bar,
                                        int lane) {
  const uint32_t r0 = __ldg(a.tile_off + t), r1 = __ldg(a.tile_off + t + 1);
  const bool fits = r1 >= r0 && r1 - r0 <= (uint32_t)(a.stage_rows - 2);
  if (lane == 0) {
    const uint32_t wbytes = fits ? (r1 - r0) * 128u : 0u;
    constexpr uint32_t qpb = PRODUCT ? QFmt<FMT>::qp_bytes : 0u;
    const uint32_t xbytes = PRODUCT ? (uint32_t)a.batch * 1024u : 0u;
    mbar_arrive_expect_tx(bar, wbytes + qpb + xbytes);
    if (wbytes) bulk_g2s(stage, a.words + (size_t)r0 * 32, wbytes, bar);
    if (PRODUCT) {
      bulk_g2s(stage + a.stage_rows * 128, a.qparams + (size_t)t * qpb, qpb, bar);
      const int kt = t % a.TK;
      uint8_t* xs = stage + q_x_offset(a.stage_rows, qpb);
      for (int b = 0; b < a.batch; ++b)
        bulk_g2s(xs + b * 1024, a.x + (size_t)b * a.K + (size_t)kt * 256, 1024, bar);
    }
  }
  return fits;
}

// Lane bit reader over a staged tile: cur:nxt hold the 64 stream bits
// starting at word (consumed/32); pos = consumed % 32.
struct LaneBits {
  uint32_t cur, nxt;
  const uint32_t* wp;      // next word to load (this lane's column)
  const uint32_t* wlast;   // last row this lane may read
  int pos, nref;
  __device__ __forceinline__ void init(const uint32_t* wb, int lane, int stage_rows) {
    cur = wb[lane];
    nxt = wb[32 + lane];
    wp = wb + 64 + lane;
    wlast = wb + (stage_rows - 1) * 32 + lane;
    pos = 0;
    nref = 0;
  }
  __device__ __forceinline__ uint32_t window() const { return __funnelshift_l(nxt, cur, pos); }
  __device__ __forceinline__ void advance(int L) {
    pos += L;
    if (pos >= 32) {
      pos -= 32;
      cur = nxt;
      nxt = *wp;
      wp = wp < wlast ? wp + 32 : wp;
      ++nref;
    }
  }
  __device__ __forceinline__ uint32_t consumed() const { return (uint32_t)nref * 32u + (uint32_t)pos; }
};

// Comparator decode of one symbol: returns the symbol-table index.
template <int NCMP>
__device__ __forceinline__ int q_decode_index(LaneBits& lb, const uint32_t (&lim)[NCMP > 0 ? NCMP : 1],
                                              int lmin, const int* s_off) {
  const uint32_t w = lb.window();
  int cnt = 0;
#pragma unroll
  for (int q = 0; q < NCMP; ++q) cnt += (w > lim[q]) ? 1 : 0;
  const int L = lmin + cnt;
  const int idx = (int)(w >> (32 - L)) + s_off[cnt];
  lb.advance(L);
  return idx;
}

// fp32 value 16 + c of the 4-bit code whose bits start at `shift_to_19`
// (positive: right shift, negative: left shift) -- exact, one shift + one op.
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

// Sum of the tile's 256 activations of row b (fixed order: 8 sequential per
// lane, then a butterfly; every lane takes lane 0's value).
__device__ __forceinline__ float tile_sum256(const float* sx, int lane) {
  const float4 u = reinterpret_cast<const float4*>(sx)[2 * lane];
  const float4 v = reinterpret_cast<const float4*>(sx)[2 * lane + 1];
  float s = ((((((u.x + u.y) + u.z) + u.w) + v.x) + v.y) + v.z) + v.w;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, m);
  return __shfl_sync(0xFFFFFFFFu, s, 0);
}

// Sum of 16 activations starting at sx[16*g] for g = lane (< 16), sequential.
__device__ __forceinline__ float group_sum16(const float* sx, int lane) {
  const float4* p = reinterpret_cast<const float4*>(sx + 16 * (lane & 15));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 u = p[i];
    s = (((s + u.x) + u.y) + u.z) + u.w;
  }
  return s;
}

// ---------------------------------------------------------------------------
// Fused product kernel: one persistent grid of WARPS-warp CTAs.
// ---------------------------------------------------------------------------
template <int FMT, bool TWIN, int BP, int NCMP, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) q_product_kernel(const QArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  using F = QFmt<FMT>;
  int* s_off = reinterpret_cast<int*>(smem + kOffOff);
  int* s_flag = reinterpret_cast<int*>(smem + kFlagOff);
  float* s_tab = reinterpret_cast<float*>(smem + kTabOff);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int xoff = q_x_offset(a.stage_rows, F::qp_bytes);

  if (!TWIN) {
    if (threadIdx.x == 0) *s_flag = table_ok(a.table, FMT, F::alpha, NCMP) ? 0 : 1;
    if (threadIdx.x < 16) s_off[threadIdx.x] = threadIdx.x < 12 ? a.table->off[threadIdx.x] : 0;
    for (int i = threadIdx.x; i < F::alpha; i += blockDim.x) {
      const uint32_t sy = a.table->sym[i];
      if (FMT == kQ4)
        reinterpret_cast<float2*>(s_tab)[i] = make_float2(16.f + (float)(sy & 15u), 16.f + (float)((sy >> 4) & 15u));
      else
        s_tab[i] = 64.f + (float)(sy & 63u);
    }
  }
  uint8_t* stage[2] = {smem + kStageOff + (2 * warp) * a.stage_bytes,
                       smem + kStageOff + (2 * warp + 1) * a.stage_bytes};
  uint64_t* bar = s_bar + 2 * warp;
  // activation rows beyond `batch` stay zero in both stages
  for (int s = 0; s < 2; ++s)
    for (int i = a.batch * 256 + lane; i < BP * 256; i += 32)
      reinterpret_cast<float*>(stage[s] + xoff)[i] = 0.f;
  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (!TWIN && *s_flag) {
    if (threadIdx.x == 0) report(a.status, LW_DEV_BAD_TABLE);
    return;
  }
  uint32_t lim[NCMP > 0 ? NCMP : 1];
  int lmin = 1;
  if (!TWIN) {
#pragma unroll
    for (int q = 0; q < NCMP; ++q) lim[q] = a.table->lim_m1[q];
    lmin = a.table->lmin;
  }

  const int nw = gridDim.x * WARPS;
  int t = blockIdx.x * WARPS + warp;
  // stage / barrier of the current tile ("c") and of the prefetched one ("n")
  uint8_t* st_c = stage[0];
  uint8_t* st_n = stage[1];
  uint64_t* bar_c = &bar[0];
  uint64_t* bar_n = &bar[1];
  uint32_t par_c = 0u, par_n = 0u;
  bool fit_c = true, fit_n = true;
  if (t < a.n_tiles) fit_c = q_issue<FMT, true>(a, t, st_c, bar_c, lane);

  for (; t < a.n_tiles; t += nw) {
    if (t + nw < a.n_tiles) {
      __syncwarp();
      fence_proxy_async();
      fit_n = q_issue<FMT, true>(a, t + nw, st_n, bar_n, lane);
    }
    if (!mbar_wait(bar_c, par_c)) {
      if (lane == 0) report(a.status, LW_DEV_TIMEOUT);
      if (t + nw < a.n_tiles) mbar_wait(bar_n, par_n);   // let any copy in flight land
      return;
    }
    par_c ^= 1u;
    const uint8_t* cur_stage = st_c;
    const bool fit = fit_c;
    {  // rotate: the prefetched tile becomes current for the next iteration
      uint8_t* ts = st_c; st_c = st_n; st_n = ts;
      uint64_t* tb = bar_c; bar_c = bar_n; bar_n = tb;
      const uint32_t tp = par_c; par_c = par_n; par_n = tp;
      fit_c = fit_n;
    }
    if (!fit) {
      if (lane == 0) report(a.status, LW_DEV_TILE_SIZE);
      continue;
    }
    const uint32_t* wb = reinterpret_cast<const uint32_t*>(cur_stage);
    const uint8_t* qp = cur_stage + a.stage_rows * 128;
    const float* sx = reinterpret_cast<const float*>(cur_stage + xoff);
    const int strip = t / a.TK, kt = t % a.TK;
    const int row0 = strip * 64 + 2 * lane;

    LaneBits lb;
    if (!TWIN) lb.init(wb, lane, a.stage_rows);
    float part0[BP], part1[BP];   // rows 2l and 2l+1

    if (FMT == kQ4) {
      float S[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) S[b] = tile_sum256(sx + 256 * b, lane);
      const uint2 q2 = reinterpret_cast<const uint2*>(qp)[lane];   // rows 2l, 2l+1: (scale | min<<16)
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float2 acc[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b) acc[b] = make_float2(0.f, 0.f);
        if (!TWIN) {
#pragma unroll 4
          for (int j = 0; j < 128; ++j) {
            const int idx = q_decode_index<NCMP>(lb, lim, lmin, s_off);
            const float2 v = reinterpret_cast<const float2*>(s_tab)[idx];
#pragma unroll
            for (int b = 0; b < BP; ++b)
              acc[b] = __ffma2_rn(v, reinterpret_cast<const float2*>(sx + 256 * b)[j], acc[b]);
          }
        } else {
#pragma unroll 2
          for (int jj = 0; jj < 32; ++jj) {
            const uint32_t w = wb[(32 * h + jj) * 32 + lane];
            const float2 v0 = make_float2(q4_twin_val<9>(w), q4_twin_val<5>(w));
            const float2 v1 = make_float2(q4_twin_val<1>(w), q4_twin_val<-3>(w));
            const float2 v2 = make_float2(q4_twin_val<-7>(w), q4_twin_val<-11>(w));
            const float2 v3 = make_float2(q4_twin_val<-15>(w), q4_twin_val<-19>(w));
#pragma unroll
            for (int b = 0; b < BP; ++b) {
              const float4 xa = reinterpret_cast<const float4*>(sx + 256 * b)[2 * jj];
              const float4 xb = reinterpret_cast<const float4*>(sx + 256 * b)[2 * jj + 1];
              acc[b] = __ffma2_rn(v0, make_float2(xa.x, xa.y), acc[b]);
              acc[b] = __ffma2_rn(v1, make_float2(xa.z, xa.w), acc[b]);
              acc[b] = __ffma2_rn(v2, make_float2(xb.x, xb.y), acc[b]);
              acc[b] = __ffma2_rn(v3, make_float2(xb.z, xb.w), acc[b]);
            }
          }
        }
        const uint32_t qv = h ? q2.y : q2.x;
        const float sc = __half2float(__ushort_as_half((unsigned short)(qv & 0xFFFFu)));
        const float mn = __half2float(__ushort_as_half((unsigned short)(qv >> 16)));
#pragma unroll
        for (int b = 0; b < BP; ++b) {
          const float A = (acc[b].x + acc[b].y) - 16.f * S[b];
          const float v = fmaf(sc, A, mn * S[b]);
          if (h) part1[b] = v; else part0[b] = v;
        }
      }
    } else {  // 6-bit
      float X[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) X[b] = group_sum16(sx + 256 * b, lane);
      const uint16_t* sc16 = reinterpret_cast<const uint16_t*>(qp);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float rowp[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b) rowp[b] = 0.f;
#pragma unroll 1
        for (int g = 0; g < 16; ++g) {
          float2 acc[BP];
#pragma unroll
          for (int b = 0; b < BP; ++b) acc[b] = make_float2(0.f, 0.f);
          if (!TWIN) {
#pragma unroll 2
            for (int m = 0; m < 8; ++m) {
              const int i0 = q_decode_index<NCMP>(lb, lim, lmin, s_off);
              const int i1 = q_decode_index<NCMP>(lb, lim, lmin, s_off);
              const float2 v = make_float2(s_tab[i0], s_tab[i1]);
#pragma unroll
              for (int b = 0; b < BP; ++b)
                acc[b] = __ffma2_rn(v, reinterpret_cast<const float2*>(sx + 256 * b + 16 * g)[m], acc[b]);
            }
          } else {
            const int r = 48 * h + 3 * g;
            const uint32_t w0 = wb[r * 32 + lane], w1 = wb[(r + 1) * 32 + lane],
                           w2 = wb[(r + 2) * 32 + lane];
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
                                    reinterpret_cast<const float2*>(sx + 256 * b + 16 * g)[m], acc[b]);
          }
          // scale of group g of row h: chunk (2h + g/8), position g%8
          const float sc = __half2float(__ushort_as_half(sc16[(((2 * h + (g >> 3)) * 32) + lane) * 8 + (g & 7)]));
#pragma unroll
          for (int b = 0; b < BP; ++b) {
            const float Xg = __shfl_sync(0xFFFFFFFFu, X[b], g);
            rowp[b] = fmaf(sc, (acc[b].x + acc[b].y) - 96.f * Xg, rowp[b]);
          }
        }
#pragma unroll
        for (int b = 0; b < BP; ++b) {
          if (h) part1[b] = rowp[b]; else part0[b] = rowp[b];
        }
      }
    }
    if (!TWIN && lb.consumed() != (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane))
      report(a.status, LW_DEV_LANE_LENGTH);
#pragma unroll
    for (int b = 0; b < BP; ++b)
      if (b < a.batch)
        *reinterpret_cast<float2*>(a.ws + ((size_t)kt * a.batch + b) * a.N + row0) =
            make_float2(part0[b], part1[b]);
  }
}

// ---------------------------------------------------------------------------
// Decode only: restore fixed-width codes to HBM.
//  Q4 -> packed bytes [N][K/2] (low nibble = even column); Q6 -> uint8 [N][K].
// ---------------------------------------------------------------------------
template <int FMT, bool TWIN, int NCMP, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) q_decode_kernel(const QArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  using F = QFmt<FMT>;
  int* s_off = reinterpret_cast<int*>(smem + kOffOff);
  int* s_flag = reinterpret_cast<int*>(smem + kFlagOff);
  uint16_t* s_sym = reinterpret_cast<uint16_t*>(smem + kTabOff);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n_sym = 0;
  if (!TWIN) {
    if (threadIdx.x == 0) *s_flag = table_ok(a.table, FMT, F::alpha, NCMP) ? 0 : 1;
    if (threadIdx.x < 16) s_off[threadIdx.x] = threadIdx.x < 12 ? a.table->off[threadIdx.x] : 0;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s_sym[i] = a.table->sym[i];
    n_sym = a.table->n_sym;
  }
  uint8_t* stage[2] = {smem + kStageOff + (2 * warp) * a.stage_bytes,
                       smem + kStageOff + (2 * warp + 1) * a.stage_bytes};
  uint64_t* bar = s_bar + 2 * warp;
  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (!TWIN && *s_flag) {
    if (threadIdx.x == 0) report(a.status, LW_DEV_BAD_TABLE);
    return;
  }
  uint32_t lim[NCMP > 0 ? NCMP : 1];
  int lmin = 1;
  if (!TWIN) {
#pragma unroll
    for (int q = 0; q < NCMP; ++q) lim[q] = a.table->lim_m1[q];
    lmin = a.table->lmin;
  }
  const int nw = gridDim.x * WARPS;
  int t = blockIdx.x * WARPS + warp;
  uint8_t* st_c = stage[0];
  uint8_t* st_n = stage[1];
  uint64_t* bar_c = &bar[0];
  uint64_t* bar_n = &bar[1];
  uint32_t par_c = 0u, par_n = 0u;
  bool fit_c = true, fit_n = true;
  if (t < a.n_tiles) fit_c = q_issue<FMT, false>(a, t, st_c, bar_c, lane);
  for (; t < a.n_tiles; t += nw) {
    if (t + nw < a.n_tiles) {
      __syncwarp();
      fence_proxy_async();
      fit_n = q_issue<FMT, false>(a, t + nw, st_n, bar_n, lane);
    }
    if (!mbar_wait(bar_c, par_c)) {
      if (lane == 0) report(a.status, LW_DEV_TIMEOUT);
      if (t + nw < a.n_tiles) mbar_wait(bar_n, par_n);
      return;
    }
    par_c ^= 1u;
    const uint8_t* cur_stage = st_c;
    const bool fit = fit_c;
    {
      uint8_t* ts = st_c; st_c = st_n; st_n = ts;
      uint64_t* tb = bar_c; bar_c = bar_n; bar_n = tb;
      const uint32_t tp = par_c; par_c = par_n; par_n = tp;
      fit_c = fit_n;
    }
    if (!fit) {
      if (lane == 0) report(a.status, LW_DEV_TILE_SIZE);
      continue;
    }
    const uint32_t* wb = reinterpret_cast<const uint32_t*>(cur_stage);
    const int strip = t / a.TK, kt = t % a.TK;
    LaneBits lb;
    if (!TWIN) lb.init(wb, lane, a.stage_rows);
    bool bad = false;
    for (int h = 0; h < 2; ++h) {
      const size_t r = (size_t)strip * 64 + 2 * lane + h;
      if (FMT == kQ4) {
        uint32_t* o = reinterpret_cast<uint32_t*>(a.out + r * (a.K / 2) + (size_t)kt * 128);
        for (int q = 0; q < 32; ++q) {
          uint32_t packed = 0;
          if (!TWIN) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int idx = q_decode_index<NCMP>(lb, lim, lmin, s_off);
              bad |= idx >= n_sym;
              packed |= (uint32_t)(s_sym[idx] & 0xFFu) << (8 * i);
            }
          } else {
            const uint32_t w = wb[(32 * h + q) * 32 + lane];   // codes 8q..8q+7, MSB first
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t ce = (w >> (28 - 8 * i)) & 15u, co = (w >> (24 - 8 * i)) & 15u;
              packed |= (ce | (co << 4)) << (8 * i);
            }
          }
          o[q] = packed;
        }
      } else {
        uint32_t* o = reinterpret_cast<uint32_t*>(a.out + r * a.K + (size_t)kt * 256);
        for (int q = 0; q < 64; ++q) {
          uint32_t packed = 0;
          if (!TWIN) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int idx = q_decode_index<NCMP>(lb, lim, lmin, s_off);
              bad |= idx >= n_sym;
              packed |= (uint32_t)(s_sym[idx] & 0x3Fu) << (8 * i);
            }
          } else {
            // codes 256h + 4q .. +3 at stream bits 6*(256h + 4q): 24 bits
            const uint32_t bit = 6u * (256u * h + 4u * q);
            const uint32_t w0 = wb[(bit / 32) * 32 + lane];
            const uint32_t w1 = (bit / 32 + 1 < 96u) ? wb[(bit / 32 + 1) * 32 + lane] : 0u;
            const uint32_t win = __funnelshift_l(w1, w0, bit % 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) packed |= ((win >> (26 - 6 * i)) & 63u) << (8 * i);
          }
          o[q] = packed;
        }
      }
    }
    if (!TWIN) {
      if (bad) report(a.status, LW_DEV_BAD_CODE);
      if (lb.consumed() != (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane))
        report(a.status, LW_DEV_LANE_LENGTH);
    }
  }
}

// y[b][r] = sum over tiles kt of ws[kt][b][r], kt ascending.
__global__ void reduce_tiles_kernel(const float* __restrict__ ws, float* __restrict__ y, int TK,
                                    int BN) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BN) return;
  float s = ws[i];
  for (int kt = 1; kt < TK; ++kt) s += ws[(size_t)kt * BN + i];
  y[i] = s;
}

}  // namespace dev
}  // namespace lw
