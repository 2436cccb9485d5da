// BF16 exponent-coded weights times a batch of 16..64 activation rows on the
// 5th-generation tensor cores: decode, rebuild BF16 on chip, feed
// tcgen05.mma (BF16 x BF16 -> FP32 in tensor memory).
//
// "Unweight: Compressing LLM Weights for Faster Inference", "How
// reconstructive matmul works": compressed data is loaded, BF16 values are
// reconstructed on chip and fed to the tensor cores without a trip through
// main memory.  The Hopper producer/consumer/WGMMA design of the page
// becomes, on sm_103a:
//  * a CTA of 8 warps owns 256 output rows (4 row strips) and a range of
//    256-column tile columns; warp w decodes row 2l + h (h = w / 4) of lane l
//    of the tile of strip w % 4, one stream per lane (the lane's second row
//    starts at its recorded mid offset);
//  * the rebuilt BF16 weights go straight into tensor memory (tcgen05.st):
//    the CTA's rows form two M = 128 operand tiles, tile h holding row
//    2l + h of strip s in tensor-memory lane 32 s + l -- exactly the lanes
//    warp w may write; 16 columns (K = 16) per chunk, a ring of kSlots
//    chunks per tile;
//  * after each chunk one thread issues two tcgen05.mma (A from tensor
//    memory, X^T from shared memory, N = the padded batch) accumulating in
//    tensor memory, and a tcgen05.commit on the chunk's ring slot tells the
//    decoders when the slot may be rewritten;
//  * X^T is staged in 128-column halves, one half ahead (cp.async, two
//    buffers, each released by a commit after the last MMA that reads it);
//    each strip's
//    next tile, the rows' verbatim flags and first sign+mantissa chunk are
//    fetched while the current tile is decoded;
//  * the accumulators are read back with tcgen05.ld by the warp that owns
//    their lanes; with K split over CTAs each writes its partial sums and
//    a sum kernel launched right behind (tc_sum_kernel, lw_bf16.cu) adds
//    them in ascending split order;
//  * the decoder table is bulk-copied into shared memory and checked
//    lane-parallel.
// Every wait is bounded; on a timeout the CTA reports LW_DEV_TIMEOUT, waits
// (bounded) for its own MMAs and copies, frees its tensor memory and returns.
#pragma once

#include "lw_bkern.cuh"
#include "lw_lutdec.cuh"
#include "lw_tcplan.h"

namespace lw {
namespace dev {

constexpr int kSlots = 4;      // operand ring depth (chunks of K = 16)
constexpr int kACols = 8;      // tensor-memory columns of one chunk: 16 bf16 per lane

// ---- tcgen05 / tensor memory helpers (inline PTX) ---------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (here BF16 inputs, FP32 accumulate)
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on `bar` once every tcgen05.mma this thread issued so far has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (BF16 inputs, FP32 accumulate)
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// this thread's 8 consecutive 32-bit columns of its tensor-memory lane
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Chunk hand-off without a CTA barrier: each of the `nwarps` decoding warps,
// once its tensor-memory stores for the chunk are done (tcgen05.wait::st),
// arrives on the chunk slot's counter, and the warp completing a group of
// `nwarps` arrivals runs issue() on its lane 0.  The counter only grows: a
// warp arrives on a slot again only after the MMAs of the slot's previous
// chunk completed, i.e. after that chunk's group was full.  Ordering:
// tcgen05 stores -> fence before thread sync -> (syncwarp, fence, atomic)
// ... (atomic, fence) -> fence after thread sync -> tcgen05.mma.
template <class Issue>
__device__ __forceinline__ void chunk_arrive(uint32_t* cnt, uint32_t nwarps, int lane, Issue issue) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    if ((atomicAdd(cnt, 1u) + 1u) % nwarps == 0u) {
      __threadfence_block();
      tc_fence_after();
      issue();
    }
  }
  __syncwarp();
}

// Shared-memory matrix descriptor, K-major, no swizzle: 8x8 core matrices of
// 16-byte rows; lbo = byte distance between core matrices adjacent along K,
// sbo = along M/N; descriptor version 1 (sm_100 family), base offset 0.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: FP32 accumulator, BF16 A and B, both
// K-major, M = 128, N = n (multiple of 16, <= 256).
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// 16-byte asynchronous copy global -> shared; zero-filled when src_bytes is 0
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Half hf of X^T of tile column kt (bpad rows x 128 columns of bf16, rows
// >= batch zero) into `xs` in the K-major core-matrix layout: element (n, k)
// at (n / 8) * 2048 + (k / 8) * 128 + (n % 8) * 16 + (k % 8) * 2.  Whole
// CTA; one cp.async group per thread.
__device__ __forceinline__ void stage_xt(const BArgs& a, uint32_t xs, int kt, int hf) {
  for (int i = threadIdx.x; i < a.bpad * 16; i += blockDim.x) {
    const int n = i >> 4, kb = i & 15;
    const bool live = n < a.batch;
    const uint16_t* src = a.x + (size_t)(live ? n : 0) * a.K + (size_t)kt * 256 + 128 * hf + 8 * kb;
    cp_async16(xs + (uint32_t)((n >> 3) * 2048 + kb * 128 + (n & 7) * 16), src, live ? 16u : 0u);
  }
  cp_async_commit();
}

// shared-memory map of the tensor-core kernel (bytes; the X^T buffers and
// tile stages follow at the launch's offsets)
constexpr int kTcBarOff = 256;      // wbar[4 strips][2], sbar[kSlots], xbar[2], tbar
constexpr int kTcSlotOff = 384;     // tensor-memory address, broadcast word, abort flag,
                                    // chunk-slot arrival counters [kSlots]
constexpr int kTcRawTabOff = 1024;  // the bundle's lw_table
constexpr int kTcXsOff = 2048;
constexpr int kTcThreads = 256;

// tensor-memory columns: D0, D1 (bpad each), then the two operand rings
__host__ __device__ constexpr int tc_tmem_need(int bpad) { return 2 * bpad + 2 * kSlots * kACols; }


// LUT: exponents decoded through the compact table replicated per lane
// (lw_lutdec.cuh; a.lut_off, a.lut_cap) instead of the comparator -- the
// same operand values, so the same results.  TWIN: the fixed-width twin
// ("Unweight", "Four different execution pipelines": direct palette): each
// weight's exponent is its 4-bit palette index looked up in the palette, a
// verbatim group's raw byte as in the coded bundle -- again the same
// operands, so twin and coded results are bitwise equal.
template <int NCMP, bool LUT, bool TWIN>
__global__ void __launch_bounds__(kTcThreads, 3) b_tc_kernel(const BArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sq = warp & 3, h = warp >> 2;   // strip of the block, row of the lane
  const uint32_t sbase = smem_addr(smem);
  const uint32_t s_off = sbase + kOffOff;
  const uint32_t s_tab = sbase + kBTabOff;
  uint64_t* wbar = reinterpret_cast<uint64_t*>(smem + kTcBarOff) + 2 * sq;    // this strip's stages
  uint64_t* sbar = reinterpret_cast<uint64_t*>(smem + kTcBarOff) + 8;         // [kSlots] ring
  uint64_t* xbar = sbar + kSlots;                                             // [2] X^T buffers
  uint64_t* tbar = xbar + 2;                                                  // table copy
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(smem + kTcSlotOff);
  volatile uint32_t* abort_flag = tslot + 2;   // a wait ran out: stop at the next tile column
  uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + kTcSlotOff + 16);   // [kSlots]
  const lw_table* tb = reinterpret_cast<const lw_table*>(smem + kTcRawTabOff);
  const uint32_t xs0 = sbase + (uint32_t)a.xs_off;       // [2][bpad * 256]: X^T halves
  const uint32_t xs_bytes = (uint32_t)a.bpad * 256u;
  uint8_t* wst0 = smem + a.wstage_off + (2 * sq) * a.stage_bytes;   // this strip's two stages
  const bool lead = h == 0 && lane == 0;                 // issues this strip's tile copies

  if (warp < 4 && lane == 0) {
    mbar_init(&wbar[0], 1);
    mbar_init(&wbar[1], 1);
  }
  if (tid == 0) {
    for (int q = 0; q < kSlots; ++q) {
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
  const uint32_t col_a = (uint32_t)(2 * a.bpad);          // first operand-ring column
  if (tid == 0) table_issue(smem + kTcRawTabOff, a.table, tbar);
  bool failed = false;        // stop: rejected table or a wait that ran out
  bool timed_out = false;     // a wait ran out (reported as LW_DEV_TIMEOUT)
  // this strip's stages: copy not yet waited for / parity of the next wait
  bool infl0 = false, infl1 = false;
  uint32_t wpar0 = 0u, wpar1 = 0u;
  const bool got = __syncthreads_and(mbar_wait(tbar, 0u));
  if (!got || !(TWIN || __syncthreads_and(table_ok_warp(tb, LW_FMT_BF16_EXP, 16, NCMP, lane)))) {
    if (tid == 0) report(a.status, got ? LW_DEV_BAD_TABLE : LW_DEV_TIMEOUT);
    if (!got) mbar_wait(tbar, 0u);
    failed = true;
  } else if (TWIN) {
    if (warp == 0 && lane < 16)   // exp << 23 per palette index
      reinterpret_cast<uint32_t*>(smem + kBTabOff)[lane] = (uint32_t)tb->palette[lane] << 23;
  } else if (warp == 0 && lane < 16) {
    put_off<(NCMP + 1) / 2>(reinterpret_cast<uint32_t*>(smem + kOffOff), lane,
                            s_tab + (uint32_t)(4 * (lane < 12 ? tb->off[lane] : 0)));
    const uint32_t sy = tb->sym[lane] & 15u;
    reinterpret_cast<uint32_t*>(smem + kBTabOff)[lane] = (uint32_t)tb->palette[sy] << 23;
  }
  constexpr int NP = (NCMP + 1) / 2;
  Cmp<NP> cmp;
  Cmp<1> cmp1;   // (unused by the twin's lookup)
  int lmin = 1;
  if (!TWIN && !failed) {
    cmp.load(tb, tb->lmax - tb->lmin);
    lmin = tb->lmin;
  }
  LDec ldec{0u, 0, 21u};
  if (LUT && !failed) {
    // every warp finds the table's shape and builds an eighth of its entries
    const LutShape sh = lut_shape_warp(tb->lim_m1, tb->lmin, tb->lmax, lane);
    if (sh.n > a.lut_cap) {
      if (tid == 0) report(a.status, LW_DEV_BAD_TABLE);
      failed = true;
    } else {
      lut_build(tb, sh, sbase + (uint32_t)a.lut_off, warp, kTcThreads / 32, lane);
    }
    ldec.lutl = sbase + (uint32_t)a.lut_off + 4u * (uint32_t)lane;
    ldec.negC = -sh.C;
    ldec.sh = 21u + (uint32_t)sh.s;
  }
  __syncthreads();
  pdl_wait();
  const uint32_t idesc = idesc_bf16((uint32_t)a.bpad);
  const int n_strips = a.N / 64;
  const int n_blocks = (n_strips + 3) / 4;
  const long long T = (long long)n_blocks * a.TK;   // tile columns of the launch
  const int G = (int)gridDim.x;
  long long x = T * blockIdx.x / G;                 // this CTA's range [x, xe)
  const long long xe = T * (blockIdx.x + 1) / G;
  uint32_t gchunk = 0;   // ring commits issued by this CTA so far (uniform)
  uint32_t xk = 0;       // X^T halves consumed by this CTA so far (uniform): the
                         // current half sits in buffer xk & 1
  uint32_t ts = 0;       // tile columns this CTA has started (uniform)

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
    // prologue: the segment's first tile, X^T and flags
    bool fit_cur = true, fit_nxt = true;
    if (has) {
      const int t = strip * a.TK + kt0;
      fit_cur = b_issue<false, TWIN>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1),
                                      wst0 + (ts & 1) * a.stage_bytes, &wbar[ts & 1],
                                      lead ? 0 : 1);
      if (ts & 1) infl1 = true; else infl0 = true;
    }
    if (xk >= 2 && !mbar_wait(&xbar[xk & 1], ((xk - 2) >> 1) & 1u)) timed_out = true;
    if (__syncthreads_or(timed_out)) { failed = true; break; }
    stage_xt(a, xs0 + (xk & 1) * xs_bytes, kt0, 0);
    uint32_t fw = 0, vb = 0;
    if (has) b_row_flags(a, r, kt0, fw, vb);
    uint4 n_sm = make_uint4(0, 0, 0, 0), n_ve = n_sm;
    if (has) {
      n_sm = b_load_sm(a, strip * a.TK + kt0, lane, h, 0);
      if (fw & 1u) n_ve = b_load_vexp(a, vb, 0);
    }
    bool first = true;
    for (int kt = kt0; kt < kt1; ++kt) {
      // one CTA barrier per tile column: every warp is done with the previous
      // column (its stage may be refilled), and a wait that ran out anywhere
      // stops all warps here
      if (__syncthreads_or(*abort_flag != 0u)) { failed = timed_out = true; break; }
      const int t = strip * a.TK + kt;
      const bool more = kt + 1 < kt1;
      const uint32_t cur = ts & 1;
      uint8_t* wstage = wst0 + cur * a.stage_bytes;
      // next tile into the other stage (both of its readers finished the
      // previous tile before the barrier above)
      if (has && more) {
        fit_nxt = b_issue<false, TWIN>(a, t + 1, __ldg(a.tile_off + t + 1), __ldg(a.tile_off + t + 2),
                                        wst0 + (cur ^ 1u) * a.stage_bytes, &wbar[cur ^ 1u],
                                        lead ? 0 : 1);
        if (cur) infl0 = true; else infl1 = true;
      }
      // flags of the next tile column: its flag word now (used at its start),
      // its first verbatim index = this column's plus this column's count
      uint32_t nword = 0;
      if (has && more) nword = __ldg(a.vflags + r * (size_t)a.GW + (4 * (kt + 1)) / 32);
      const uint32_t nvb = vb + __popc(fw);
      uint4 p_sm = make_uint4(0, 0, 0, 0);   // the next column's first chunk
      uint32_t nfw = 0;
      bool to = false;
      if (has) {
        to = !mbar_wait(&wbar[cur], cur ? wpar1 : wpar0);
        if (!to) {
          if (cur) { wpar1 ^= 1u; infl1 = false; } else { wpar0 ^= 1u; infl0 = false; }
        }
      }
      const uint32_t wb = smem_addr(wstage);
      LaneBits lb;
      LStream ls;
      uint32_t mid = 0;
      const bool dec = has && fit_cur && !to;
      if (dec && !TWIN) {
        mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        if (LUT) ls.init(wb, lane, a.stage_rows, h ? mid : 0u);
        else lb.init_at(wb, lane, a.stage_rows, h ? mid : 0u);
      }
      if (has && !fit_cur && lead) report(a.status, LW_DEV_TILE_SIZE);
      if (to) *abort_flag = 1u;
      for (int k = 0; k < 16; ++k) {
        const uint32_t slot = gchunk % kSlots;
        // after an abort every wait is skipped and nothing is arrived on; the
        // warps run to the barrier at the next tile column
        // (`live` is kept warp-uniform: the tensor-memory stores and the
        // hand-off below are warp-wide)
        bool live = *abort_flag == 0u;
        if (live && gchunk >= (uint32_t)kSlots)
          live = mbar_wait(&sbar[slot], ((gchunk - kSlots) / kSlots) & 1u);
        if (live && (k & 7) == 4 && (k < 8 || more) && xk >= 1)
          // the next X^T half goes into the other buffer once the MMAs that
          // last read it (the previous half) are done
          live = mbar_wait(&xbar[(xk + 1) & 1], ((xk - 1) >> 1) & 1u);
        live = __all_sync(0xFFFFFFFFu, live);
        if (!live) *abort_flag = 1u;
        if ((k & 7) == 0) {   // this thread's part of the current X^T half
          cp_async_wait_all();
          fence_proxy_async();
        }
        if (live && (k & 7) == 4 && (k < 8 || more))
          stage_xt(a, xs0 + ((xk + 1) & 1) * xs_bytes, k < 8 ? kt : kt + 1, k < 8 ? 1 : 0);
        if (k == 8 && more && has) {
          p_sm = b_load_sm(a, t + 1, lane, h, 0);
          nfw = (nword >> ((4 * (kt + 1)) % 32)) & 15u;
        }
        uint32_t W[8];   // bf16x2 of this lane's row, columns 16k .. 16k+15
        if (dec) {
          const bool v = (fw >> (k >> 2)) & 1u;
          const uint4 sm = n_sm, ve = n_ve;
          if (k < 15) {
            const int k1 = k + 1, g1 = k1 >> 2;
            n_sm = b_load_sm(a, t, lane, h, k1);
            if ((fw >> g1) & 1u) n_ve = b_load_vexp(a, vb + __popc(fw & ((1u << g1) - 1u)), k1 & 3);
          } else if (more) {   // first chunk of the next tile column
            n_sm = p_sm;
            if (nfw & 1u) n_ve = b_load_vexp(a, nvb, 0);
          }

          if (TWIN) {
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              uint32_t E0, E1;
              b_exponents<true, 1>(lb, cmp1, 0, s_off, s_tab, wb, h, lane, k, p, v, ve, E0, E1);
              const uint32_t sw = u4w(sm, p >> 1);
              const uint32_t f0 = __float_as_uint((p & 1) ? b_value<2>(sw, E0) : b_value<0>(sw, E0));
              const uint32_t f1 = __float_as_uint((p & 1) ? b_value<3>(sw, E1) : b_value<1>(sw, E1));
              W[p] = __byte_perm(f0, f1, 0x7632);   // (bf16 of f1) << 16 | bf16 of f0
            }
          } else if (LUT) {
            // a verbatim group holds the stream (multiplier 0) and takes its
            // raw exponent bytes, moved to bits 23..30 (b16_value reads no more)
            const uint32_t go = v ? 0u : 1u, vm = v ? 0xFFFFFFFFu : 0u;
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              uint32_t e0, e1;
              l_decode2<true>(ls, ldec, e0, e1, go);
              const uint32_t sw = u4w(sm, p >> 1), vw = u4w(ve, p >> 1);
              const uint32_t ve0 = (p & 1) ? imad(vw, 1u << 7, 0u) : imad(vw, 1u << 23, 0u);
              const uint32_t ve1 = (p & 1) ? vw >> 1 : imad(vw, 1u << 15, 0u);
              const uint32_t E0 = (e0 & ~vm) | (ve0 & vm), E1 = (e1 & ~vm) | (ve1 & vm);
              const uint32_t f0 = __float_as_uint((p & 1) ? b16_value<2>(sw, E0) : b16_value<0>(sw, E0));
              const uint32_t f1 = __float_as_uint((p & 1) ? b16_value<3>(sw, E1) : b16_value<1>(sw, E1));
              W[p] = __byte_perm(f0, f1, 0x7632);   // (bf16 of f1) << 16 | bf16 of f0
            }
          } else {
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              uint32_t E0, E1;
              b_exponents<false, NP>(lb, cmp, lmin, s_off, s_tab, wb, h, lane, k, p, v, ve, E0, E1);
              const uint32_t sw = u4w(sm, p >> 1);
              const uint32_t f0 = __float_as_uint((p & 1) ? b_value<2>(sw, E0) : b_value<0>(sw, E0));
              const uint32_t f1 = __float_as_uint((p & 1) ? b_value<3>(sw, E1) : b_value<1>(sw, E1));
              W[p] = __byte_perm(f0, f1, 0x7632);   // (bf16 of f1) << 16 | bf16 of f0
            }
          }
        } else {
#pragma unroll
          for (int p = 0; p < 8; ++p) W[p] = 0u;
        }
        if (live) {
          tmem_st8(tmem + t_lane + col_a + (uint32_t)((h * kSlots + (int)slot) * kACols), W);
          tmem_st_wait();
          fence_proxy_async();
          // the last of the 8 warps issues this chunk's MMAs
          const bool fst = first;
          chunk_arrive(&cnt[slot], 8u, lane, [&] {
            const uint64_t bd = sdesc(xs0 + (xk & 1) * xs_bytes + 256u * (uint32_t)(k & 7), 128u, 2048u);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              umma_bf16_ta(tmem + (uint32_t)(hh * a.bpad),
                           tmem + col_a + (uint32_t)((hh * kSlots + (int)slot) * kACols), bd, idesc,
                           fst ? 0u : 1u);
            umma_commit(&sbar[slot]);
            if ((k & 7) == 7) umma_commit(&xbar[xk & 1]);   // X^T half free after these
          });
        }
        first = false;
        ++gchunk;
        if ((k & 7) == 7) ++xk;
      }
      if (dec && !TWIN) {
        const uint32_t end = h ? (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane) : mid;
        if ((LUT ? ls.consumed() : (uint32_t)lb.consumed()) != end) report(a.status, LW_DEV_LANE_LENGTH);
      }
      ++ts;
      fit_cur = fit_nxt;
      fw = nfw;
      vb = nvb;
    }
    if (failed || __syncthreads_or(*abort_flag != 0u)) { failed = timed_out = true; break; }
    if (x >= xe) pdl_trigger();   // last segment decoded
    // all MMAs of this segment done -> read the accumulators (warp w: tile h,
    // lanes of strip sq)
    bool to3 = !mbar_wait(&sbar[(gchunk - 1) % kSlots], ((gchunk - 1) / kSlots) & 1u);
    if (__syncthreads_or(to3)) { failed = timed_out = true; break; }
    tc_fence_after();
    const size_t step = (size_t)a.batch * a.N;
    for (int j = 0; j < a.bpad; j += 16) {
      uint32_t rr[16];
      tmem_ld16(tmem + t_lane + (uint32_t)(h * a.bpad + j), rr);
      tmem_ld_wait();
      if (has) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int b = j + i;
          if (b < a.batch) {
            if (alone) a.y[(size_t)b * a.N + r] = __uint_as_float(rr[i]);
            else a.ws[(size_t)sp * step + (size_t)b * a.N + r] = __uint_as_float(rr[i]);
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
    if (gchunk > 0) mbar_wait(&sbar[(gchunk - 1) % kSlots], ((gchunk - 1) / kSlots) & 1u);
    if (infl0) mbar_wait(&wbar[0], wpar0);
    if (infl1) mbar_wait(&wbar[1], wpar1);
  }
  cp_async_wait_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
}

}  // namespace dev
}  // namespace lw
