// 4-bit (pair-coded) and 6-bit Huffman-coded weights times a batch of 6..32
// fp32 activation rows on the 5th-generation tensor cores.
//
// The codes and their tiles follow "LazyWeights: Decode-on-Demand Edge
// LLMs" ("2 . Code them", Fig. 3(a); comparator decode, "3 . Decode on
// demand"); reconstruction on chip feeding the tensor cores follows
// "Unweight: Compressing LLM Weights for Faster Inference" ("How
// reconstructive matmul works").  Exactness (ours): the tensor cores take
// BF16, the products must stay within 1e-3 of fp32/fp64 results, so
//  * each weight is dequantised in fp32 (4-bit: scale * c + min; 6-bit:
//    scale * (c - 32)) and split exactly into w = hi + lo, hi = w with its low
//    16 bits cleared (a BF16 value), lo = the remainder rounded to BF16
//    (|error| <= 2^-17 |w|);
//  * each activation likewise into x_hi + x_lo;
//  * per chunk of K = 16 two MMAs accumulate hi * [x_hi | x_lo] (N = 2 bpad)
//    and lo * x_hi (N = bpad) in FP32 tensor memory; y = D[:, b] +
//    D[:, bpad + b].  The dropped lo * x_lo term is below 2^-16 relative.
// Layout and pipeline as the BF16 tensor-core kernel: 8-warp CTAs own 256
// rows x a range of tile columns; warp w decodes row 2l + h (h = w / 4) of
// strip w % 4 and stores the split weights into tensor memory (lanes 32 s +
// l of operand tile h; hi and lo rings of kQtSlots chunks); X^T (hi and lo
// rows) is staged in 128-column halves one half ahead, loaded from global
// memory two chunks before it is converted and stored; with K split over
// CTAs each writes its partial sums and tc_sum_kernel (lw_bf16.cu) adds them
// in ascending split order.
// Every wait is bounded; on a timeout the CTA reports LW_DEV_TIMEOUT, waits
// (bounded) for its own MMAs and copies, frees its tensor memory and returns.
#pragma once

#include <cuda_bf16.h>

#include "lw_btc.cuh"

namespace lw {
namespace dev {

constexpr int kQtSlots = 2;         // operand ring depth per tile and hi/lo
constexpr int kQtThreads = 256;
constexpr int kQtMaxRows = 32;      // activation rows per pass
// dynamic shared-memory map (bytes)
constexpr int kQtTabOff = 0;        // symbol values: float2[256] (c0, c1) / float[64] (c - 32)
constexpr int kQtBarOff = 2048;     // wbar[4 strips][2], sbar[kQtSlots], xbar[2], tbar
constexpr int kQtSlotOff = 2176;    // tensor-memory address, broadcast word, abort flag,
                                    // chunk-slot arrival counters [kQtSlots]
constexpr int kQtRawTabOff = 2304;  // the bundle's lw_table
constexpr int kQtXsOff = 3328;      // X^T halves: 2 x [2 bpad rows][128 columns] bf16
static_assert(kQtRawTabOff + (int)sizeof(lw_table) <= kQtXsOff, "shared-memory map");

// tensor-memory columns: D0, D1 (2 bpad each), then the hi and lo rings
__host__ __device__ constexpr int qt_tmem_need(int bpad) {
  return 4 * bpad + 2 * 2 * kQtSlots * kACols;
}

// Split two fp32 values into packed BF16 hi parts (truncated) and lo parts
// (the exact remainders, rounded to nearest).
__device__ __forceinline__ void split_bf16x2(float2 w, uint32_t& hi, uint32_t& lo) {
  const uint32_t u0 = __float_as_uint(w.x), u1 = __float_as_uint(w.y);
  hi = __byte_perm(u0, u1, 0x7632);
  const float2 t = make_float2(__uint_as_float(u0 & 0xFFFF0000u), __uint_as_float(u1 & 0xFFFF0000u));
  const float2 r = __fadd2_rn(w, make_float2(-t.x, -t.y));   // exact
  const __nv_bfloat162 b = __floats2bfloat162_rn(r.x, r.y);
  lo = *reinterpret_cast<const uint32_t*>(&b);
}

// Activations of half hf of tile column kt: this thread's float4 items
// (item i: row n = i / 32, columns 4 (i % 32) .. +3 of the half).
__device__ __forceinline__ void qt_x_load(const QArgs& a, int kt, int hf, float4 (&v)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = (int)threadIdx.x + q * kQtThreads;
    v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < a.bpad * 32) {
      const int n = i >> 5, c = i & 31;
      if (n < a.batch)
        v[q] = __ldg(reinterpret_cast<const float4*>(a.x + (size_t)n * a.K + (size_t)kt * 256 +
                                                     128 * hf) + c);
    }
  }
}

// ... split and stored into buffer `xs`: x_hi in rows [0, bpad), x_lo in rows
// [bpad, 2 bpad), K-major core-matrix layout (element (n, k) at
// (n / 8) * 2048 + (k / 8) * 128 + (n % 8) * 16 + (k % 8) * 2).
__device__ __forceinline__ void qt_x_store(const QArgs& a, uint8_t* xs, const float4 (&v)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = (int)threadIdx.x + q * kQtThreads;
    if (i < a.bpad * 32) {
      const int n = i >> 5, k = 4 * (i & 31);
      uint32_t h0, l0, h1, l1;
      split_bf16x2(make_float2(v[q].x, v[q].y), h0, l0);
      split_bf16x2(make_float2(v[q].z, v[q].w), h1, l1);
      const int off = (k >> 3) * 128 + (k & 7) * 2;
      *reinterpret_cast<uint2*>(xs + (n >> 3) * 2048 + (n & 7) * 16 + off) = make_uint2(h0, h1);
      const int nl = n + a.bpad;
      *reinterpret_cast<uint2*>(xs + (nl >> 3) * 2048 + (nl & 7) * 16 + off) = make_uint2(l0, l1);
    }
  }
}

template <int FMT, int NCMP>
__global__ void __launch_bounds__(kQtThreads, 3) q_tc_kernel(const QArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(16) uint32_t offtab[16];
  using F = QFmt<FMT>;
  constexpr int NP = (NCMP + 1) / 2;
  constexpr int ESZ = FMT == kQ4 ? 8 : 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sq = warp & 3, h = warp >> 2;   // strip of the block, row of the lane
  const uint32_t s_off = smem_addr(offtab);
  const uint32_t s_tab = smem_addr(smem) + kQtTabOff;
  uint64_t* wbar = reinterpret_cast<uint64_t*>(smem + kQtBarOff) + 2 * sq;   // this strip's stages
  uint64_t* sbar = reinterpret_cast<uint64_t*>(smem + kQtBarOff) + 8;        // [kQtSlots] rings
  uint64_t* xbar = sbar + kQtSlots;                                          // [2] X^T buffers
  uint64_t* tbar = xbar + 2;                                                 // table copy
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(smem + kQtSlotOff);
  volatile uint32_t* abort_flag = tslot + 2;   // a wait ran out: stop at the next tile column
  uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + kQtSlotOff + 16);   // [kQtSlots]
  const lw_table* tb = reinterpret_cast<const lw_table*>(smem + kQtRawTabOff);
  uint8_t* xs0 = smem + a.xs_off;                        // [2][2 bpad x 128] bf16
  const int xs_bytes = a.bpad * 512;
  // this strip's stages: two (the next tile prefetched) or one (more CTAs fit)
  uint8_t* wst0 = smem + a.wstage_off + (a.nstage * sq) * a.stage_bytes;
  const bool two = a.nstage == 2;
  const bool lead = h == 0 && lane == 0;                 // issues this strip's tile copies

  if (warp < 4 && lane == 0) {
    mbar_init(&wbar[0], 1);
    mbar_init(&wbar[1], 1);
  }
  if (tid == 0) {
    for (int q = 0; q < kQtSlots; ++q) {
      mbar_init(&sbar[q], 1);
      cnt[q] = 0u;
    }
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    mbar_init(tbar, 1);
    *abort_flag = 0u;
  }
  if (lane == 0) fence_barrier_init();
  if (warp == 0) {
    tmem_alloc(smem_addr(const_cast<uint32_t*>(tslot)), (uint32_t)a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t t_lane = (uint32_t)(32 * sq) << 16;      // this warp's lane quarter
  const uint32_t col_hi = (uint32_t)(4 * a.bpad);         // first hi-ring column
  const uint32_t col_lo = col_hi + (uint32_t)(2 * kQtSlots * kACols);
  if (tid == 0) table_issue(smem + kQtRawTabOff, a.table, tbar);
  bool failed = false;
  bool timed_out = false;
  bool infl0 = false, infl1 = false;
  uint32_t wpar0 = 0u, wpar1 = 0u;
  const bool got = __syncthreads_and(mbar_wait(tbar, 0u));
  if (!got || !__syncthreads_and(table_ok_warp(tb, FMT, F::alpha, NCMP, lane))) {
    if (tid == 0) report(a.status, got ? LW_DEV_BAD_TABLE : LW_DEV_TIMEOUT);
    if (!got) mbar_wait(tbar, 0u);
    failed = true;
  } else {
    // symbol values: 4-bit (c0, c1), 6-bit c - 32; offsets as shared addresses
    if (tid < 16)
      put_off<NP>(offtab, tid, s_tab + (uint32_t)(ESZ * (tid < 12 ? tb->off[tid] : 0)));
    for (int i = tid; i < F::alpha; i += kQtThreads) {
      const uint32_t sy = tb->sym[i];
      if (FMT == kQ4)
        reinterpret_cast<float2*>(smem + kQtTabOff)[i] =
            make_float2((float)(sy & 15u), (float)((sy >> 4) & 15u));
      else
        reinterpret_cast<float*>(smem + kQtTabOff)[i] = (float)(int)(sy & 63u) - 32.f;
    }
  }
  Cmp<NP> cmp;
  int lmin = 1;
  if (!failed) {
    cmp.load(tb, tb->lmax - tb->lmin);
    lmin = tb->lmin;
  }
  __syncthreads();
  pdl_wait();
  const uint32_t idesc2 = idesc_bf16((uint32_t)(2 * a.bpad));   // hi x [x_hi | x_lo]
  const uint32_t idesc1 = idesc_bf16((uint32_t)a.bpad);         // lo x x_hi
  const int n_strips = a.N / 64;
  const int n_blocks = (n_strips + 3) / 4;
  const long long T = (long long)n_blocks * a.TK;   // tile columns of the launch (tc_owner)
  const int G = (int)gridDim.x;
  long long x = T * blockIdx.x / G;                 // this CTA's range [x, xe)
  const long long xe = T * (blockIdx.x + 1) / G;
  uint32_t gchunk = 0;   // ring commits issued by this CTA so far (uniform)
  uint32_t xk = 0;       // X^T halves consumed so far (uniform); current in buffer xk & 1
  uint32_t ts = 0;       // tile columns started (uniform)
  float4 xv[4];          // activations of the next X^T half, loaded ahead

  while (x < xe && !failed) {   // one segment: the range's part in one row block
    const int rb = (int)(x / a.TK);
    const long long xb = (long long)rb * a.TK;   // the row block's first tile column
    const long long xs = xe < xb + a.TK ? xe : xb + a.TK;
    const int kt0 = (int)(x - xb), kt1 = (int)(xs - xb);
    const int owner0 = tc_owner(xb, T, G);
    const int sp = (int)blockIdx.x - owner0;     // this CTA's partial of the row block
    const bool alone = tc_owner(xb + a.TK - 1, T, G) == owner0;   // y directly
    x = xs;
    const int strip = rb * 4 + sq;
    const bool has = strip < n_strips;
    const size_t r = (size_t)strip * 64 + 2 * lane + h;
    bool fit_cur = true, fit_nxt = true;
    if (has && two) {
      const int t = strip * a.TK + kt0;
      fit_cur = q_issue<FMT, true>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1),
                                   wst0 + (ts & 1) * a.stage_bytes, &wbar[ts & 1], lead, 0);
      if (ts & 1) infl1 = true; else infl0 = true;
    }
    // the segment's first X^T half (its buffer's last reader, half xk - 2, done)
    if (xk >= 2 && !mbar_wait(&xbar[xk & 1], ((xk - 2) >> 1) & 1u)) timed_out = true;
    if (__syncthreads_or(timed_out)) { failed = true; break; }
    qt_x_load(a, kt0, 0, xv);
    qt_x_store(a, xs0 + (xk & 1) * xs_bytes, xv);
    fence_proxy_async();
    bool first = true;
    for (int kt = kt0; kt < kt1; ++kt) {
      // one CTA barrier per tile column: every warp is done with the previous
      // column (its stage may be refilled), and a wait that ran out anywhere
      // stops all warps here
      if (__syncthreads_or(*abort_flag != 0u)) { failed = timed_out = true; break; }
      const int t = strip * a.TK + kt;
      const bool more = kt + 1 < kt1;
      const uint32_t cur = two ? ts & 1 : 0u;
      uint8_t* wstage = wst0 + cur * a.stage_bytes;
      if (has && !two) {   // one stage: this tile now (its last readers are past the barrier)
        fit_cur = q_issue<FMT, true>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1), wstage,
                                     &wbar[0], lead, 0);
        infl0 = true;
      }
      if (has && two && more) {   // the next tile into the other stage
        fit_nxt = q_issue<FMT, true>(a, t + 1, __ldg(a.tile_off + t + 1), __ldg(a.tile_off + t + 2),
                                     wst0 + (cur ^ 1u) * a.stage_bytes, &wbar[cur ^ 1u], lead, 0);
        if (cur) infl0 = true; else infl1 = true;
      }
      bool to = false;
      if (has) {
        to = !mbar_wait(&wbar[cur], cur ? wpar1 : wpar0);
        if (!to) {
          if (cur) { wpar1 ^= 1u; infl1 = false; } else { wpar0 ^= 1u; infl0 = false; }
        }
      }
      const uint32_t wb = smem_addr(wstage);
      const uint32_t qp = wb + (uint32_t)a.stage_rows * 128u;
      LaneBits lb;
      uint32_t mid = 0;
      const bool dec = has && fit_cur && !to;
      float sc = 0.f, mn = 0.f;   // 4-bit: this row's scale and min in this tile
      if (dec) {
        mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        lb.init_at(wb, lane, a.stage_rows, h ? mid : 0u);
        if (FMT == kQ4) {
          const uint32_t q2 = lds_u32(qp + 4u * (uint32_t)(2 * lane + h));
          sc = __half2float(__ushort_as_half((unsigned short)(q2 & 0xFFFFu)));
          mn = __half2float(__ushort_as_half((unsigned short)(q2 >> 16)));
        }
      }
      if (has && !fit_cur && lead) report(a.status, LW_DEV_TILE_SIZE);
      if (to) *abort_flag = 1u;
      for (int k = 0; k < 16; ++k) {
        const uint32_t slot = gchunk % kQtSlots;
        const bool next_half = k < 8 || more;
        // after an abort every wait is skipped and nothing is arrived on; the
        // warps run to the barrier at the next tile column.  `live` is kept
        // warp-uniform (the tensor-memory stores and the hand-off are warp-wide)
        bool live = *abort_flag == 0u;
        if (live && gchunk >= (uint32_t)kQtSlots)
          live = mbar_wait(&sbar[slot], ((gchunk - kQtSlots) / kQtSlots) & 1u);
        if (live && (k & 7) == 4 && next_half && xk >= 1)
          // the next X^T half goes into the other buffer once the MMAs that
          // last read it (the previous half) are done
          live = mbar_wait(&xbar[(xk + 1) & 1], ((xk - 1) >> 1) & 1u);
        live = __all_sync(0xFFFFFFFFu, live);
        if (!live) *abort_flag = 1u;
        if ((k & 7) == 2 && next_half) qt_x_load(a, k < 8 ? kt : kt + 1, k < 8 ? 1 : 0, xv);
        if (live && (k & 7) == 4 && next_half) {
          qt_x_store(a, xs0 + ((xk + 1) & 1) * xs_bytes, xv);
          fence_proxy_async();
        }
        uint32_t WH[8], WL[8];   // this lane's row, columns 16k .. 16k+15: hi and lo halves
        if (dec) {
          float s6 = 0.f;
          if (FMT == kQ6) {
            const uint32_t sa = qp + (uint32_t)((((2 * h + (k >> 3)) * 32) + lane) * 16 + 2 * (k & 7));
            s6 = __half2float(__ushort_as_half((unsigned short)lds_u16(sa)));
          }
#pragma unroll
          for (int p = 0; p < (FMT == kQ4 ? 4 : 8); ++p) {
            uint32_t e0, e1;
            q_decode2<NP, ESZ>(lb, cmp, lmin, s_off, e0, e1);
            if (FMT == kQ4) {   // two pair symbols: columns 4p .. 4p+3
              const float2 c0 = lds_f2(e0), c1 = lds_f2(e1);
              split_bf16x2(__ffma2_rn(make_float2(sc, sc), c0, make_float2(mn, mn)), WH[2 * p], WL[2 * p]);
              split_bf16x2(__ffma2_rn(make_float2(sc, sc), c1, make_float2(mn, mn)), WH[2 * p + 1],
                           WL[2 * p + 1]);
            } else {            // two single symbols: columns 2p, 2p+1
              split_bf16x2(__fmul2_rn(make_float2(s6, s6), make_float2(lds_f32(e0), lds_f32(e1))),
                           WH[p], WL[p]);
            }
          }
        } else {
#pragma unroll
          for (int p = 0; p < 8; ++p) WH[p] = WL[p] = 0u;
        }
        if (live) {
          const uint32_t rs = (uint32_t)((h * kQtSlots + (int)slot) * kACols);
          tmem_st8(tmem + t_lane + col_hi + rs, WH);
          tmem_st8(tmem + t_lane + col_lo + rs, WL);
          tmem_st_wait();
          fence_proxy_async();
          // the last of the 8 warps issues this chunk's MMAs
          const bool fst = first;
          chunk_arrive(&cnt[slot], 8u, lane, [&] {
            const uint64_t bd = sdesc(smem_addr(xs0) + (xk & 1) * (uint32_t)xs_bytes +
                                          256u * (uint32_t)(k & 7), 128u, 2048u);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t d = tmem + (uint32_t)(hh * 2 * a.bpad);
              const uint32_t ra = (uint32_t)((hh * kQtSlots + (int)slot) * kACols);
              umma_bf16_ta(d, tmem + col_hi + ra, bd, idesc2, fst ? 0u : 1u);
              umma_bf16_ta(d, tmem + col_lo + ra, bd, idesc1, 1u);
            }
            umma_commit(&sbar[slot]);
            if ((k & 7) == 7) umma_commit(&xbar[xk & 1]);   // X^T half free after these
          });
        }
        first = false;
        ++gchunk;
        if ((k & 7) == 7) ++xk;
      }
      if (dec) {
        const uint32_t end = h ? (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane) : mid;
        if (lb.consumed() != end) report(a.status, LW_DEV_LANE_LENGTH);
      }
      ++ts;
      if (two) fit_cur = fit_nxt;
    }
    if (failed || __syncthreads_or(*abort_flag != 0u)) { failed = timed_out = true; break; }
    if (x >= xe) pdl_trigger();   // last segment decoded
    // all MMAs of this segment done -> read the accumulators (warp w: tile h,
    // lanes of strip sq); y = hi-part columns + lo-part columns
    bool to3 = !mbar_wait(&sbar[(gchunk - 1) % kQtSlots], ((gchunk - 1) / kQtSlots) & 1u);
    if (__syncthreads_or(to3)) { failed = timed_out = true; break; }
    tc_fence_after();
    const size_t step = (size_t)a.batch * a.N;
    for (int j = 0; j < a.bpad; j += 16) {
      uint32_t rh[16], rl[16];
      tmem_ld16(tmem + t_lane + (uint32_t)(h * 2 * a.bpad + j), rh);
      tmem_ld16(tmem + t_lane + (uint32_t)(h * 2 * a.bpad + a.bpad + j), rl);
      tmem_ld_wait();
      if (has) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int b = j + i;
          if (b < a.batch) {
            const float v = __uint_as_float(rh[i]) + __uint_as_float(rl[i]);
            if (alone) a.y[(size_t)b * a.N + r] = v;
            else a.ws[(size_t)sp * step + (size_t)b * a.N + r] = v;
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();   // accumulators read before the next segment overwrites them
  }
  if (timed_out) {
    if (tid == 0) report(a.status, LW_DEV_TIMEOUT);
    // let this CTA's own MMAs and copies finish (bounded) before leaving
    if (gchunk > 0) mbar_wait(&sbar[(gchunk - 1) % kQtSlots], ((gchunk - 1) / kQtSlots) & 1u);
    if (infl0) mbar_wait(&wbar[0], wpar0);
    if (infl1) mbar_wait(&wbar[1], wpar1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
}

}  // namespace dev
}  // namespace lw
