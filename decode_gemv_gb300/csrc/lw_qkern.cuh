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
//  * a lane keeps three stream words in registers; one 32-bit window serves
//    two symbols (a code is at most 11 bits, so after the first code at
//    least 21 valid bits remain), and the words advance at most once per
//    symbol pair;
//  * comparator limits live in registers; per-length offsets (pre-scaled to
//    shared addresses) and the symbol table (pre-converted to fp32) in shared
//    memory, read with explicit ld.shared;
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
  const float* x;        // [batch][K] (products)
  float* ws;             // partials [TK][batch][N] (products)
  uint32_t* counters;    // [N/64] strip counters (products), zero between calls
  float* y;              // [batch][N] (products)
  uint8_t* out;          // decode-only output
  int32_t* status;
  int n_tiles, TK, N, K, batch;
  int stage_rows;        // rows of 128 B per stage buffer = max_tile_rows + 3
  int stage_bytes;       // bytes per stage buffer (multiple of 128)
  int nstage;            // stage buffers per warp: 2 (prefetch the next tile
                         // while decoding) or 1 (more resident warps)
  int mid_offset;        // byte offset of the tile's lane_mid copy in a stage
};

constexpr int kQ4 = LW_FMT_Q4_PAIR, kQ6 = LW_FMT_Q6;

template <int FMT> struct QFmt;
template <> struct QFmt<LW_FMT_Q4_PAIR> {
  static constexpr int alpha = 256, qp_bytes = 256;
};
template <> struct QFmt<LW_FMT_Q6> {
  static constexpr int alpha = 64, qp_bytes = 2048;
};

// shared-memory map (bytes)
constexpr int kOffOff = 0;       // uint32[16]: symbol-table base address per length index
constexpr int kFlagOff = 64;     // int: table rejected
constexpr int kTabOff = 128;     // symbol values: float2[256] (4-bit) / float[64]
constexpr int kBarOff = 2176;    // uint64 mbarriers, 2 per warp (<= 8 warps)
constexpr int kStageOff = 2304;  // per warp: one or two stage buffers
constexpr int kLookahead = 3;    // stream words a lane holds in registers

__host__ __device__ constexpr int q_x_offset(int stage_rows, int qp_bytes) {
  return stage_rows * 128 + qp_bytes;
}

// Issue the copies of tile t, whose coded rows are [r0, r1), into one stage
// (whole warp; lane 0 issues).  Returns false if the tile is longer than the stage allows (the other copies
// are still issued, so the barrier completes).
template <int FMT, bool PRODUCT>
__device__ __forceinline__ bool q_issue(const QArgs& a, int t, uint32_t r0, uint32_t r1,
                                        uint8_t* stage, uint64_t* bar, int lane) {
  const bool fits = r1 >= r0 && r1 - r0 <= (uint32_t)(a.stage_rows - kLookahead);
  if (lane == 0) {
    const uint32_t wbytes = fits ? (r1 - r0) * 128u : 0u;
    constexpr uint32_t qpb = PRODUCT ? QFmt<FMT>::qp_bytes : 0u;
    const uint32_t xbytes = PRODUCT ? (uint32_t)a.batch * 1024u : 0u;
    const uint32_t mbytes = (PRODUCT && a.lane_mid) ? 64u : 0u;
    mbar_arrive_expect_tx(bar, wbytes + qpb + xbytes + mbytes);
    if (wbytes) bulk_g2s(stage, a.words + (size_t)r0 * 32, wbytes, bar);
    if (PRODUCT) {
      bulk_g2s(stage + a.stage_rows * 128, a.qparams + (size_t)t * qpb, qpb, bar);
      const int kt = t % a.TK;
      uint8_t* xs = stage + q_x_offset(a.stage_rows, qpb);
      for (int b = 0; b < a.batch; ++b)
        bulk_g2s(xs + b * 1024, a.x + (size_t)b * a.K + (size_t)kt * 256, 1024, bar);
      if (mbytes) bulk_g2s(stage + a.mid_offset, a.lane_mid + (size_t)t * 32, 64, bar);
    }
  }
  return fits;
}

// Lane bit reader over a staged tile.  Registers cur:nxt:nx2 hold stream
// words j, j+1, j+2 where j = consumed / 32; pos = consumed % 32.
struct LaneBits {
  uint32_t cur, nxt, nx2;
  uint32_t wp;      // shared address of word j + 3 of this lane
  uint32_t wlast;   // last row this lane may read (clamp for corrupt streams)
  int pos, nref;
  __device__ __forceinline__ void init(uint32_t wb, int lane, int stage_rows) {
    const uint32_t base = wb + 4u * (uint32_t)lane;
    cur = lds_u32(base);
    nxt = lds_u32(base + 128u);
    nx2 = lds_u32(base + 256u);
    wp = base + 384u;
    wlast = base + (uint32_t)(stage_rows - 1) * 128u;
    pos = 0;
    nref = 0;
  }
  // start at stream bit `bit` (clamped so that every read stays inside the
  // stage; a lane whose start was clamped fails its length check)
  __device__ __forceinline__ void init_at(uint32_t wb, int lane, int stage_rows, uint32_t bit) {
    uint32_t j0 = bit >> 5;
    if (j0 > (uint32_t)(stage_rows - kLookahead)) j0 = (uint32_t)(stage_rows - kLookahead);
    const uint32_t base = wb + 4u * (uint32_t)lane;
    cur = lds_u32(base + 128u * j0);
    nxt = lds_u32(base + 128u * (j0 + 1));
    nx2 = lds_u32(base + 128u * (j0 + 2));
    wp = base + 128u * (j0 + 3);
    wlast = base + (uint32_t)(stage_rows - 1) * 128u;
    if (wp > wlast) wp = wlast;
    pos = (int)(bit & 31u);
    nref = (int)j0;
  }
  __device__ __forceinline__ uint32_t window() const { return __funnelshift_l(nxt, cur, pos); }
  // consume n (< 32) bits
  __device__ __forceinline__ void advance(int n) {
    pos += n;
    if (pos >= 32) {
      pos -= 32;
      cur = nxt;
      nxt = nx2;
      nx2 = lds_u32(wp);
      wp = min(wp + 128u, wlast);
      ++nref;
    }
  }
  __device__ __forceinline__ uint32_t consumed() const { return (uint32_t)nref * 32u + (uint32_t)pos; }
};

__device__ __forceinline__ __half2 as_h2(uint32_t b) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = b;
  return h;
}
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// The comparator thresholds of a table as fp16 pairs.  Every limit below the
// longest length is even in the 11-bit peek space, so the first 10 window
// bits p decide each test exactly: with v = 1024 + p and T = 1024 + limit/2
// (both exact in fp16), the saturating sum v + (1 - T) = p - limit/2 + 1,
// clamped to [0, 1], is 1 exactly when the peek reaches the limit.  One
// fp16x2 add tests two limits; unused slots hold a limit no peek reaches.
template <int NP>
struct Cmp {
  uint32_t c[NP > 0 ? NP : 1];   // fp16x2: (1 - T_2k, 1 - T_2k+1)
  __device__ __forceinline__ void load(const lw_table* tb, int ncmp) {
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      uint32_t lohi[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = 2 * k + h;
        // lim_m1 = (limit << 21) - 1  ->  limit / 2 = (lim_m1 + 1) >> 22
        const uint32_t half_lim = q < ncmp ? ((tb->lim_m1[q] + 1u) >> 22) : 1024u;
        lohi[h] = __half_as_ushort(__float2half_rn(1.f - (1024.f + (float)half_lim)));
      }
      c[k] = lohi[0] | (lohi[1] << 16);
    }
  }
  // number of limits the window's code reaches (0 .. 2*NP)
  __device__ __forceinline__ int count(uint32_t w) const {
    const __half2 v = as_h2((w >> 22) * 0x00010001u + 0x64006400u);
    __half2 s[NP > 0 ? NP : 1];
#pragma unroll
    for (int k = 0; k < NP; ++k) s[k] = __hadd2_sat(v, as_h2(c[k]));
#pragma unroll
    for (int step = 1; step < NP; step *= 2)
#pragma unroll
      for (int k = 0; k + step < NP; k += 2 * step) s[k] = __hadd2(s[k], s[k + step]);
    // low half: 1024 + s.lo + s.hi  ->  bits 0x6400 + count
    const __half2 r = __hadd2(__hadd2(s[0], as_h2(0x00006400u)), __lowhigh2highlow(s[0]));
    return (int)(h2_bits(r) & 0xFFFFu) - 0x6400;
  }
};

// Decode two symbols from one window.  Returns the shared addresses of their
// symbol-table entries (entry size ESZ bytes).
template <int NP, int ESZ>
__device__ __forceinline__ void q_decode2(LaneBits& lb, const Cmp<NP>& cmp, int lmin, uint32_t s_off,
                                          uint32_t& e0, uint32_t& e1) {
  const uint32_t w = lb.window();
  const int c0 = cmp.count(w);
  const int L0 = lmin + c0;
  const uint32_t w1 = w << L0;
  const int c1 = cmp.count(w1);
  const int L1 = lmin + c1;
  e0 = lds_u32(s_off + 4u * (uint32_t)c0) + __funnelshift_l(w, 0u, L0) * ESZ;
  e1 = lds_u32(s_off + 4u * (uint32_t)c1) + __funnelshift_l(w1, 0u, L1) * ESZ;
  lb.advance(L0 + L1);
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

// Partial sums of rows (row0, row0+1) for tile (strip, kt) -> workspace; the
// last tile of the strip to arrive adds all partials of the strip in
// ascending tile order and writes y.
template <int BP>
__device__ __forceinline__ void q_commit(const QArgs& a, int strip, int kt, int lane,
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

// ---------------------------------------------------------------------------
// Fused product kernel: one persistent grid of WARPS-warp CTAs.
// ---------------------------------------------------------------------------
// resident warps per SM the register budget is sized for (more activation
// rows need more accumulator registers)
__host__ __device__ constexpr int q_target_warps(int bp) { return bp <= 4 ? 16 : 12; }

template <int FMT, bool TWIN, int BP, int NCMP, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, q_target_warps(BP) / WARPS)
    q_product_kernel(const QArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  using F = QFmt<FMT>;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t s_off = sbase + kOffOff;
  const uint32_t s_tab = sbase + kTabOff;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int xoff = q_x_offset(a.stage_rows, F::qp_bytes);
  constexpr int ESZ = FMT == kQ4 ? 8 : 4;

  const bool two = a.nstage == 2;
  uint8_t* stage0 = smem + kStageOff + (a.nstage * warp) * a.stage_bytes;
  uint8_t* stage1 = two ? stage0 + a.stage_bytes : stage0;
  uint64_t* bar = s_bar + 2 * warp;
  const int nw = gridDim.x * WARPS;
  int t = blockIdx.x * WARPS + warp;
  // activation rows beyond `batch` stay zero in every stage
  for (int i = a.batch * 256 + lane; i < BP * 256; i += 32) {
    reinterpret_cast<float*>(stage0 + xoff)[i] = 0.f;
    reinterpret_cast<float*>(stage1 + xoff)[i] = 0.f;
  }
  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  __syncwarp();
  // the first tile's copy starts before the table is staged
  uint32_t par0 = 0u, par1 = 0u;
  bool fit0 = true, fit1 = true;
  if (t < a.n_tiles)
    fit0 = q_issue<FMT, true>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1), stage0,
                              &bar[0], lane);
  // row range of the next tile to issue (t + nw), loaded one tile ahead
  uint32_t nr0 = 0, nr1 = 0;
  if (t + nw < a.n_tiles) {
    nr0 = __ldg(a.tile_off + t + nw);
    nr1 = __ldg(a.tile_off + t + nw + 1);
  }

  if (!TWIN) {
    if (threadIdx.x == 0)
      *reinterpret_cast<int*>(smem + kFlagOff) = table_ok(a.table, FMT, F::alpha, NCMP) ? 0 : 1;
    if (threadIdx.x < 16)
      reinterpret_cast<uint32_t*>(smem + kOffOff)[threadIdx.x] =
          s_tab + (uint32_t)(ESZ * (threadIdx.x < 12 ? a.table->off[threadIdx.x] : 0));
    for (int i = threadIdx.x; i < F::alpha; i += blockDim.x) {
      const uint32_t sy = a.table->sym[i];
      if (FMT == kQ4)
        reinterpret_cast<float2*>(smem + kTabOff)[i] =
            make_float2(16.f + (float)(sy & 15u), 16.f + (float)((sy >> 4) & 15u));
      else
        reinterpret_cast<float*>(smem + kTabOff)[i] = 64.f + (float)(sy & 63u);
    }
  }
  __syncthreads();
  if (!TWIN && *reinterpret_cast<volatile int*>(smem + kFlagOff)) {
    if (threadIdx.x == 0) report(a.status, LW_DEV_BAD_TABLE);
    if (t < a.n_tiles) mbar_wait(&bar[0], 0u);   // let the first copy land
    return;
  }
  constexpr int NP = (NCMP + 1) / 2;
  Cmp<NP> cmp;
  int lmin = 1;
  if (!TWIN) {
    cmp.load(a.table, a.table->lmax - a.table->lmin);
    lmin = a.table->lmin;
  }

  for (int it = 0; t < a.n_tiles; ++it, t += nw) {
    const bool odd = two && (it & 1);
    const bool more = t + nw < a.n_tiles;
    const uint32_t ir0 = nr0, ir1 = nr1;     // rows of tile t + nw
    if (t + 2 * nw < a.n_tiles) {
      nr0 = __ldg(a.tile_off + t + 2 * nw);
      nr1 = __ldg(a.tile_off + t + 2 * nw + 1);
    }
    if (two && more) {
      __syncwarp();
      fence_proxy_async();
      if (odd) fit0 = q_issue<FMT, true>(a, t + nw, ir0, ir1, stage0, &bar[0], lane);
      else fit1 = q_issue<FMT, true>(a, t + nw, ir0, ir1, stage1, &bar[1], lane);
    }
    uint8_t* st = odd ? stage1 : stage0;
    const bool ok = odd ? mbar_wait(&bar[1], par1) : mbar_wait(&bar[0], par0);
    if (!ok) {
      if (lane == 0) report(a.status, LW_DEV_TIMEOUT);
      if (two && more) {   // let the copy in flight land before leaving
        if (odd) mbar_wait(&bar[0], par0);
        else mbar_wait(&bar[1], par1);
      }
      return;
    }
    if (odd) par1 ^= 1u; else par0 ^= 1u;
    const bool fit = odd ? fit1 : fit0;
    const int strip = t / a.TK, kt = t % a.TK;
    float part0[BP], part1[BP];   // rows 2l and 2l+1
#pragma unroll
    for (int b = 0; b < BP; ++b) part0[b] = part1[b] = 0.f;
    if (!fit) {
      if (lane == 0) report(a.status, LW_DEV_TILE_SIZE);
      if (!two && more) {
        __syncwarp();
        fit0 = q_issue<FMT, true>(a, t + nw, ir0, ir1, stage0, &bar[0], lane);
      }
      q_commit<BP>(a, strip, kt, lane, part0, part1);
      continue;
    }
    const uint32_t wb = smem_addr(st);
    const uint32_t qp = wb + (uint32_t)a.stage_rows * 128u;
    const uint32_t sx = wb + (uint32_t)xoff;

    LaneBits lb;
    if (!TWIN) lb.init(wb, lane, a.stage_rows);

    if (FMT == kQ4) {
      float S[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) S[b] = tile_sum256(sx + 1024u * b, lane);
      const uint2 q2 = lds_u2(qp + 8u * (uint32_t)lane);   // rows 2l, 2l+1: (scale | min<<16)
      if (!TWIN) {
        // rows 2l and 2l+1 are decoded as two independent streams (the second
        // starts at the lane's recorded mid offset); 64 symbol pairs each,
        // the table entries of pair j read while pair j+1 is decoded
        const uint32_t mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        LaneBits lr;
        lr.init_at(wb, lane, a.stage_rows, mid);
        float2 acc0[BP], acc1[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b) acc0[b] = acc1[b] = make_float2(0.f, 0.f);
        uint32_t a0, a1, c0, c1;
        q_decode2<NP, 8>(lb, cmp, lmin, s_off, a0, a1);
        q_decode2<NP, 8>(lr, cmp, lmin, s_off, c0, c1);
#pragma unroll 2
        for (int j = 0; j < 64; ++j) {
          const float2 va0 = lds_f2(a0), va1 = lds_f2(a1), vc0 = lds_f2(c0), vc1 = lds_f2(c1);
          if (j < 63) {
            q_decode2<NP, 8>(lb, cmp, lmin, s_off, a0, a1);
            q_decode2<NP, 8>(lr, cmp, lmin, s_off, c0, c1);
          }
#pragma unroll
          for (int b = 0; b < BP; ++b) {
            const float4 xv = lds_f4(sx + 1024u * b + 16u * (uint32_t)j);
            acc0[b] = __ffma2_rn(va0, make_float2(xv.x, xv.y), acc0[b]);
            acc0[b] = __ffma2_rn(va1, make_float2(xv.z, xv.w), acc0[b]);
            acc1[b] = __ffma2_rn(vc0, make_float2(xv.x, xv.y), acc1[b]);
            acc1[b] = __ffma2_rn(vc1, make_float2(xv.z, xv.w), acc1[b]);
          }
        }
        const float sc0 = __half2float(__ushort_as_half((unsigned short)(q2.x & 0xFFFFu)));
        const float mn0 = __half2float(__ushort_as_half((unsigned short)(q2.x >> 16)));
        const float sc1 = __half2float(__ushort_as_half((unsigned short)(q2.y & 0xFFFFu)));
        const float mn1 = __half2float(__ushort_as_half((unsigned short)(q2.y >> 16)));
#pragma unroll
        for (int b = 0; b < BP; ++b) {
          part0[b] = fmaf(sc0, (acc0[b].x + acc0[b].y) - 16.f * S[b], mn0 * S[b]);
          part1[b] = fmaf(sc1, (acc1[b].x + acc1[b].y) - 16.f * S[b], mn1 * S[b]);
        }
        if (lb.consumed() != mid || lr.consumed() != (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane))
          report(a.status, LW_DEV_LANE_LENGTH);
      } else {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          float2 acc[BP];
#pragma unroll
          for (int b = 0; b < BP; ++b) acc[b] = make_float2(0.f, 0.f);
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
      }
    } else {  // 6-bit
      float X[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) X[b] = group_sum16(sx + 1024u * b, lane);
      if (!TWIN) {
        // both rows as independent streams, group by group
        const uint32_t mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        LaneBits lr;
        lr.init_at(wb, lane, a.stage_rows, mid);
        float rowp0[BP], rowp1[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b) rowp0[b] = rowp1[b] = 0.f;
        uint32_t a0, a1, c0, c1;
        q_decode2<NP, 4>(lb, cmp, lmin, s_off, a0, a1);
        q_decode2<NP, 4>(lr, cmp, lmin, s_off, c0, c1);
#pragma unroll 1
        for (int g = 0; g < 16; ++g) {
          float2 acc0[BP], acc1[BP];
#pragma unroll
          for (int b = 0; b < BP; ++b) acc0[b] = acc1[b] = make_float2(0.f, 0.f);
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const float2 v0 = make_float2(lds_f32(a0), lds_f32(a1));
            const float2 v1 = make_float2(lds_f32(c0), lds_f32(c1));
            if (g < 15 || m < 7) {
              q_decode2<NP, 4>(lb, cmp, lmin, s_off, a0, a1);
              q_decode2<NP, 4>(lr, cmp, lmin, s_off, c0, c1);
            }
#pragma unroll
            for (int b = 0; b < BP; ++b) {
              const float2 xv = lds_f2(sx + 1024u * b + 64u * g + 8u * m);
              acc0[b] = __ffma2_rn(v0, xv, acc0[b]);
              acc1[b] = __ffma2_rn(v1, xv, acc1[b]);
            }
          }
          const uint32_t sa0 = qp + (uint32_t)((((g >> 3) * 32) + lane) * 16 + 2 * (g & 7));
          const uint32_t sa1 = qp + (uint32_t)((((2 + (g >> 3)) * 32) + lane) * 16 + 2 * (g & 7));
          const float s0 = __half2float(__ushort_as_half((unsigned short)lds_u16(sa0)));
          const float s1 = __half2float(__ushort_as_half((unsigned short)lds_u16(sa1)));
#pragma unroll
          for (int b = 0; b < BP; ++b) {
            const float Xg = __shfl_sync(0xFFFFFFFFu, X[b], g);
            rowp0[b] = fmaf(s0, (acc0[b].x + acc0[b].y) - 96.f * Xg, rowp0[b]);
            rowp1[b] = fmaf(s1, (acc1[b].x + acc1[b].y) - 96.f * Xg, rowp1[b]);
          }
        }
#pragma unroll
        for (int b = 0; b < BP; ++b) {
          part0[b] = rowp0[b];
          part1[b] = rowp1[b];
        }
        if (lb.consumed() != mid || lr.consumed() != (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane))
          report(a.status, LW_DEV_LANE_LENGTH);
      } else {
        float rowp[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b) rowp[b] = 0.f;
#pragma unroll 1
        for (int G = 0; G < 32; ++G) {          // group g = G % 16 of row h = G / 16
          const int h = G >> 4, g = G & 15;
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
          // scale of group g of row h: chunk (2h + g/8), position g%8
          const uint32_t sa = qp + (uint32_t)((((2 * h + (g >> 3)) * 32) + lane) * 16 + 2 * (g & 7));
          const float sc = __half2float(__ushort_as_half((unsigned short)lds_u16(sa)));
#pragma unroll
          for (int b = 0; b < BP; ++b) {
            const float Xg = __shfl_sync(0xFFFFFFFFu, X[b], g);
            rowp[b] = fmaf(sc, (acc[b].x + acc[b].y) - 96.f * Xg, rowp[b]);
          }
          if (g == 15) {
#pragma unroll
            for (int b = 0; b < BP; ++b) {
              if (h) part1[b] = rowp[b]; else part0[b] = rowp[b];
              rowp[b] = 0.f;
            }
          }
        }
      }
    }
    if (!two && more) {   // single stage: refill it now, overlapping the commit
      __syncwarp();
      fence_proxy_async();
      fit0 = q_issue<FMT, true>(a, t + nw, ir0, ir1, stage0, &bar[0], lane);
    }
    q_commit<BP>(a, strip, kt, lane, part0, part1);
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
  const uint32_t sbase = smem_addr(smem);
  const uint32_t s_off = sbase + kOffOff;
  const uint32_t s_sym = sbase + kTabOff;   // uint32 per canonical index
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n_sym = 0;
  if (!TWIN) {
    if (threadIdx.x == 0)
      *reinterpret_cast<int*>(smem + kFlagOff) = table_ok(a.table, FMT, F::alpha, NCMP) ? 0 : 1;
    if (threadIdx.x < 16)
      reinterpret_cast<uint32_t*>(smem + kOffOff)[threadIdx.x] =
          s_sym + (uint32_t)(4 * (threadIdx.x < 12 ? a.table->off[threadIdx.x] : 0));
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
      reinterpret_cast<uint32_t*>(smem + kTabOff)[i] = a.table->sym[i];
    n_sym = a.table->n_sym;
  }
  uint8_t* stage0 = smem + kStageOff + (2 * warp) * a.stage_bytes;
  uint8_t* stage1 = stage0 + a.stage_bytes;
  uint64_t* bar = s_bar + 2 * warp;
  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (!TWIN && *reinterpret_cast<volatile int*>(smem + kFlagOff)) {
    if (threadIdx.x == 0) report(a.status, LW_DEV_BAD_TABLE);
    return;
  }
  constexpr int NP = (NCMP + 1) / 2;
  Cmp<NP> cmp;
  int lmin = 1;
  if (!TWIN) {
    cmp.load(a.table, a.table->lmax - a.table->lmin);
    lmin = a.table->lmin;
  }
  const uint32_t first_bad = s_sym + 4u * (uint32_t)n_sym;   // entries at or past it are phantom
  const int nw = gridDim.x * WARPS;
  int t = blockIdx.x * WARPS + warp;
  uint32_t par0 = 0u, par1 = 0u;
  bool fit0 = true, fit1 = true;
  if (t < a.n_tiles)
    fit0 = q_issue<FMT, false>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1), stage0,
                               &bar[0], lane);
  for (int it = 0; t < a.n_tiles; ++it, t += nw) {
    const bool odd = it & 1;
    if (t + nw < a.n_tiles) {
      __syncwarp();
      fence_proxy_async();
      const uint32_t ir0 = __ldg(a.tile_off + t + nw), ir1 = __ldg(a.tile_off + t + nw + 1);
      if (odd) fit0 = q_issue<FMT, false>(a, t + nw, ir0, ir1, stage0, &bar[0], lane);
      else fit1 = q_issue<FMT, false>(a, t + nw, ir0, ir1, stage1, &bar[1], lane);
    }
    uint8_t* st = odd ? stage1 : stage0;
    const bool ok = odd ? mbar_wait(&bar[1], par1) : mbar_wait(&bar[0], par0);
    if (!ok) {
      if (lane == 0) report(a.status, LW_DEV_TIMEOUT);
      if (t + nw < a.n_tiles) {
        if (odd) mbar_wait(&bar[0], par0);
        else mbar_wait(&bar[1], par1);
      }
      return;
    }
    if (odd) par1 ^= 1u; else par0 ^= 1u;
    if (!(odd ? fit1 : fit0)) {
      if (lane == 0) report(a.status, LW_DEV_TILE_SIZE);
      continue;
    }
    const uint32_t wb = smem_addr(st);
    const int strip = t / a.TK, kt = t % a.TK;
    LaneBits lb;
    if (!TWIN) lb.init(wb, lane, a.stage_rows);
    bool bad_len = false;
    bool bad = false;
    for (int h = 0; h < 2; ++h) {
      if (!TWIN && h == 1 && lb.consumed() != (uint32_t)__ldg(a.lane_mid + (size_t)t * 32 + lane))
        bad_len = true;
      const size_t r = (size_t)strip * 64 + 2 * lane + h;
      if (FMT == kQ4) {
        uint32_t* o = reinterpret_cast<uint32_t*>(a.out + r * (a.K / 2) + (size_t)kt * 128);
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
          o[q] = packed;
        }
      } else {
        uint32_t* o = reinterpret_cast<uint32_t*>(a.out + r * a.K + (size_t)kt * 256);
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
          o[q] = packed;
        }
      }
    }
    if (!TWIN) {
      if (bad) report(a.status, LW_DEV_BAD_CODE);
      if (bad_len || lb.consumed() != (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane))
        report(a.status, LW_DEV_LANE_LENGTH);
    }
  }
}

}  // namespace dev
}  // namespace lw
