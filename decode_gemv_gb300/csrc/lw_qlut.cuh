// Table-driven fused decode + GEMV / small-batch GEMM for 4-bit (pair-coded)
// and 6-bit Huffman-coded weights and for BF16 weights whose exponents are
// Huffman-coded ("Unweight: Compressing LLM Weights for Faster Inference",
// "The exponent's exploitable redundancy"), and the same skeleton for the
// 4-/6-bit fixed-width twins.
//
// Method: "LazyWeights: Decode-on-Demand Edge LLMs" -- "2 . Code them" and
// Fig. 3(a) (64x256 tiles of 32 interleaved lanes of two rows), "3 . Decode on
// demand" (per lane: an 11-bit peek of the stream selects the codeword; the
// lane then shifts by its length) and the runtime paragraph after Fig. 3
// (software decode fused into the GEMV; the fixed-width twin as the
// decode-free comparator).
//
// GB300 mapping (ours):
//  * one persistent CTA per SM: four producer warps and NW consumer warps.
//    The producers fill a ring of S tile stages in shared memory with bulk
//    asynchronous copies (TMA engine, no multicast) -- a tile's coded rows,
//    its scales/mins, its lanes' mid offsets and bit counts and its slices of
//    the activations -- each stage completing on a "full" mbarrier (four
//    issuers: one thread's bulk copies alone reach about half of HBM's
//    bandwidth); a consumer warp takes the next tile (a shared counter),
//    waits for the stage to be announced for that tile and then for its
//    barrier, decodes it and releases the stage on its "empty" mbarrier.
//    Every wait is bounded.
//  * a consumer warp decodes a unit of a tile: with R = 2, a whole tile,
//    lane l running its two rows (2l from the start of its stream, 2l + 1
//    from its mid offset) as two interleaved streams that share the
//    activation loads; with R = 1, one row of every lane, so a tile's two
//    units run on two warps -- the scheduler then hides one warp's lookup
//    latency with another's work (a warp issues in order), and the
//    half-tile units balance better over the warps; the launcher takes
//    R = 1 for CTAs with few tiles;
//  * decoding is a lookup: the peek indexes a compact table (lw_lut.h) in
//    shared memory that is replicated once per lane -- lane l's copy of an
//    entry sits in bank l, so a warp's 32 lookups are one conflict-free
//    shared-memory wavefront whatever symbols the lanes decode.  An entry
//    holds the code length (bits 0..4) and the symbol's weights in a form
//    that only FMA-pipe instructions turn into fp32 (the integer ALU pipe,
//    the decoder's bottleneck, keeps the bit work): 4-bit pairs as two fp16
//    codes (the length sits in the low mantissa bits of one, where a
//    rounding fp16 add of 1024 drops it), 6-bit codes as the fp16 1024 + c,
//    BF16 exponent symbols as the palette's exponent at its fp32 position;
//  * one 32-bit window serves two symbols (an 11-bit code leaves at least 21
//    valid bits): window = funnel shift of two stream words by the bit
//    position; the second peek comes from the window shifted by the first
//    length; the position advances by both lengths and the words by at most
//    one per step, branch-free (the next word is reloaded every step);
//  * products in packed fp32 FMA (FFMA2) on the exact values 16 + c (4-bit)
//    and 64 + c (6-bit): even and odd columns in the two halves, then per
//    row and tile part = scale * (acc.x + acc.y - 16 X) + min * X (4-bit)
//    or, per 16-weight group, scale * (acc.x + acc.y - 96 X_group) (6-bit),
//    in a fixed order -- the operations of the comparator kernel, whose
//    results this kernel's equal bit for bit, as do the twin's;
//  * BF16: each weight's fp32 value is its sign+mantissa byte (read from
//    global memory a 16-weight chunk ahead) joined with the decoded exponent
//    by a byte permute and one logic op; a verbatim 64-column group holds
//    the stream (its lengths masked to zero) and takes its raw exponent
//    bytes; the activations are widened from bf16 once per tile; the
//    per-row sum is the comparator BF16 kernel's (bit for bit);
//  * split-K: each tile's partial sums go to the workspace; the last tile of
//    a 64-row strip to finish (an atomicInc counter that wraps back to zero)
//    adds them in ascending tile order -- one launch, deterministic;
//  * stream reads never leave shared memory: a stream starts inside its
//    stage and advances at most one 128-byte row per two symbols, and the
//    stages are followed by the table (or, without a table, by a guard), so
//    even a corrupt stream reads only this CTA's shared memory; it then
//    fails its length check.
#pragma once

#include "lw_dev.cuh"
#include "lw_lut.h"
#include "lw_lutdec.cuh"
#include "lw_qkern.cuh"

namespace lw {
namespace dev {

// One launch: up to kMaxGroup matrices of one format; the CTAs are
// partitioned among them (CTA c serves matrix m when cfirst[m] <= c <
// cfirst[m + 1]), each CTA walking its matrix's tiles c', c' + cnt, ...
struct LLaunch {
  QArgs m[kMaxGroup];
  int cfirst[kMaxGroup + 1];
  int n;
  int nstage;       // S: stages in the ring
  int stage_bytes;  // bytes per stage (multiple of 128)
  int stage_rows;   // rows of 128 B of coded words a stage holds
  int qp_off;       // offsets inside a stage: scales/mins, mid offsets, activations
  int mid_off;
  int lb_off;       // lane bit counts (coded bundles)
  int x_off;
  int ring_off;     // shared-memory offset of stage 0
  int xb_off;       // where a stage's activation copies land (BF16: bf16
                    // rows, widened into x_off by the consumer; else x_off)
  int vi_off;       // BF16: per row of the tile, first verbatim group << 4 | 4 flags
  long long wait_cycles;   // limit of every wait on a stage (SM clock cycles)
  int stall_tile;   // testing: local tile of CTA 0 whose stage is armed without copies (-1: none)
  int lut_off;      // shared-memory offset of the decode table (coded bundles)
  int lut_cap;      // entries it holds (>= every member's table)
};

// Shared-memory header (bytes).
constexpr int kLHdrNext = 0;     // int: next local tile to hand out
constexpr int kLHdrErr = 4;      // int: set when any warp gives up
constexpr int kLHdrTab = 8;      // uint64 mbarrier: table copy
constexpr int kLHdrBar = 64;     // uint64 mbarriers: full[S], then empty[S]
constexpr int kLMaxStages = 32;
constexpr int kLRawTab = kLHdrBar + 16 * kLMaxStages;   // 576: the staged lw_table
constexpr int kLHdrTiles = kLRawTab + (int)sizeof(lw_table);   // int[S]: tile each stage is armed for
constexpr int kLHdrBytes = kLHdrTiles + 4 * kLMaxStages;
constexpr int kLGuardRows = 132;  // rows a corrupt 6-bit stream may read past its stage
constexpr int kLProducers = 4;    // producer warps (each issues its own stages' copies)
constexpr int kLMaxConsumers = 24;  // consumer warps at most
// consumer warps a launch of R rows per unit may use (R = 2: 16, so that
// the kernel may keep more registers per thread)
template <int R>
constexpr int kLMaxConsumersR = R == 2 ? 16 : kLMaxConsumers;
// BF16 exponent bundles: 12 (more registers for the sign+mantissa and
// verbatim bytes in flight)
constexpr int kLMaxConsumersB16 = 12;
template <int FMT, int R>
constexpr int kLMaxConsumersOf = FMT == LW_FMT_BF16_EXP ? kLMaxConsumersB16 : kLMaxConsumersR<R>;

// exact fp32 value of the fp16 in the high half of e, plus c
__device__ __forceinline__ float f16hi_plus(uint32_t e, float c) {
  float f;
  asm("{.reg .b16 h; mov.b32 {_, h}, %1; add.rn.f32.f16 %0, h, %2;}" : "=f"(f) : "r"(e), "f"(c));
  return f;
}
__device__ __forceinline__ float f16lo_plus(uint32_t e, float c) {
  float f;
  asm("{.reg .b16 h; mov.b32 {h, _}, %1; add.rn.f32.f16 %0, h, %2;}" : "=f"(f) : "r"(e), "f"(c));
  return f;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// The codes enter the products as the exact fp32 values 16 + c (4-bit) and
// 64 + c (6-bit), the bias removed once per tile row (4-bit: 16 * sum x) or
// per 16-weight group (6-bit: 96 * sum x, folding in the code offset 32):
// the comparator kernel's operands and epilogue, so both kernels execute
// the same floating-point operations and give bitwise-equal results.
constexpr float kQ4Unbias = -1008.f;   // 1024 + c -> 16 + c
constexpr float kQ6Unbias = -960.f;    // 1024 + c -> 64 + c

// The exact fp32 values (16 + c_even, 16 + c_odd) of a 4-bit entry: one
// fp16x2 add of 1024 (rounding to the integer grid of [1024, 2048) drops the
// length bits), then two mixed-precision adds of -1008 -- all on the FMA
// pipes.
__device__ __forceinline__ float2 q4_vals(uint32_t e) {
  uint32_t h;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(e), "r"(0x64006400u));
  float lo, hi;
  asm("{.reg .b16 a, b; mov.b32 {a, b}, %2; add.rn.f32.f16 %0, a, %3; add.rn.f32.f16 %1, b, %3;}"
      : "=f"(lo), "=f"(hi) : "r"(h), "f"(kQ4Unbias));
  return make_float2(lo, hi);
}

// The exact fp32 values 16 + c of the four pairs of a 4-bit twin word (codes
// MSB-first in stream order: code k at bits 28 - 4k .. 31 - 4k; even columns
// are codes 0, 2, 4, 6): each logic op builds two fp16 1024 + c, each mixed-
// precision add subtracts 1008 -- the coded entries' values, so the twin's
// products are the coded kernel's.
__device__ __forceinline__ void q4_twin_word(uint32_t w, float2 (&v)[4]) {
  const uint32_t A = (w & 0x000F000Fu) | 0x64006400u;           // codes 3 | 7
  const uint32_t B = ((w >> 4) & 0x000F000Fu) | 0x64006400u;    // codes 2 | 6
  const uint32_t C = ((w >> 8) & 0x000F000Fu) | 0x64006400u;    // codes 1 | 5
  const uint32_t D = ((w >> 12) & 0x000F000Fu) | 0x64006400u;   // codes 0 | 4
  v[0] = make_float2(f16hi_plus(D, kQ4Unbias), f16hi_plus(C, kQ4Unbias));
  v[1] = make_float2(f16hi_plus(B, kQ4Unbias), f16hi_plus(A, kQ4Unbias));
  v[2] = make_float2(f16lo_plus(D, kQ4Unbias), f16lo_plus(C, kQ4Unbias));
  v[3] = make_float2(f16lo_plus(B, kQ4Unbias), f16lo_plus(A, kQ4Unbias));
}

// fp32 value 64 + c of the 6-bit code at stream bit B of the lane's twin
// words (row base address rb = stage + 4 lane; word j at rb + 128 j).
template <int B>
__device__ __forceinline__ float q6_twin_c(uint32_t w0, uint32_t w1) {
  constexpr int o = B % 32;
  uint32_t t;
  if constexpr (o <= 26) t = w0 >> (26 - o);   // the code is bits 31-o..26-o of w0
  else t = __funnelshift_l(w1, w0, o - 26);     // it continues into w1
  return f16lo_plus((t & 63u) | 0x6400u, kQ6Unbias);
}

// Split-K commit of a warp's unit (one row of every lane of a tile), in
// three parts that the consumer loop spreads over three units so that no
// warp waits for a round trip to L2: l_store writes the partial sum of each
// lane's row of tile (strip, kt); a unit later, l_count counts it in (lane
// 0: an acq_rel atomicInc that wraps to zero -- its release covers every
// lane's stores, ordered by the warp barrier, which by then have long
// landed); another unit later, l_finish reads the count, and the warp that
// brought it to 2 TK adds the strip's partials in ascending tile order and
// writes y.
template <int R, int BP>
__device__ __forceinline__ void l_store(const QArgs& a, int strip, int kt, int row,
                                        const float (&p)[R][BP]) {
#pragma unroll
  for (int b = 0; b < BP; ++b)
    if (b < a.batch) {
      float* q = a.ws + ((size_t)kt * a.batch + b) * a.N + strip * 64 + row;
      if (R == 2) *reinterpret_cast<float2*>(q) = make_float2(p[0][b], p[R - 1][b]);
      else *q = p[0][b];
    }
}
// UPT units per tile: the strip completes after UPT * TK of them
template <int UPT>
__device__ __forceinline__ uint32_t l_count(const QArgs& a, int strip, int lane) {
  __syncwarp();
  return lane == 0 ? atom_inc_acq_rel(a.counters + strip, (unsigned)(UPT * a.TK - 1)) : 0u;
}
// The strip's reduction (the last arriver's warp), G partials per round
// trip to L2 (G = 16: two groups of 8 loaded before either is added).
template <int G>
__device__ __forceinline__ void l_reduce(const QArgs& a, int strip, int lane) {
  const int row0 = strip * 64 + 2 * lane;
  const size_t step = (size_t)a.batch * a.N;
  for (int b = 0; b < a.batch; ++b) {
    const float2* base = reinterpret_cast<const float2*>(a.ws + (size_t)b * a.N + row0);
    const size_t st2 = step / 2;   // float2 stride between tiles of the strip
    // the sum runs in ascending tile order
    float2 s = make_float2(0.f, 0.f);
    for (int k0 = 0; k0 < a.TK; k0 += G) {
      float2 v[8], w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (k0 + i < a.TK) v[i] = __ldcg(base + (size_t)(k0 + i) * st2);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (G == 16 && k0 + 8 + i < a.TK) w[i] = __ldcg(base + (size_t)(k0 + 8 + i) * st2);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (k0 + i < a.TK) {
          if (k0 + i == 0) s = v[0];
          else { s.x += v[i].x; s.y += v[i].y; }
        }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (G == 16 && k0 + 8 + i < a.TK) { s.x += w[i].x; s.y += w[i].y; }
    }
    *reinterpret_cast<float2*>(a.y + (size_t)b * a.N + row0) = s;
  }
}
template <int UPT>
__device__ __forceinline__ void l_finish(const QArgs& a, int strip, int lane, uint32_t old) {
  if (__shfl_sync(0xFFFFFFFFu, old, 0) != (uint32_t)(UPT * a.TK - 1)) return;
  __syncwarp();   // the last arriver's acquire (lane 0) orders the reads below
  l_reduce<UPT == 1 ? 16 : 8>(a, strip, lane);
}

// Row range [r0, r1) and bundle tile t of local tile i of a CTA (zeros past
// its last tile).
__device__ __forceinline__ void l_rows(const QArgs& a, int c0, int cnt, int n_local, int i,
                                       uint32_t& r0, uint32_t& r1, int& t) {
  r0 = r1 = 0u;
  t = 0;
  if (i < n_local) {
    bool v;
    t = list_tile<true>(a, c0 + i * cnt, v);
    r0 = __ldg(a.tile_off + t);
    r1 = __ldg(a.tile_off + t + 1);
  }
}

template <int FMT, bool TWIN, int BP, int R>
__global__ void __launch_bounds__((kLMaxConsumersOf<FMT, R> + kLProducers) * 32, 1) q_lut_kernel(const __grid_constant__ LLaunch g) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int nthreads = blockDim.x;
  const int nw = nthreads / 32 - kLProducers;   // consumer warps; warps nw.. produce
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool producer = warp >= nw;
  int mi = 0;
  while (mi + 1 < g.n && (int)blockIdx.x >= g.cfirst[mi + 1]) ++mi;
  const QArgs& a = g.m[mi];
  const int cnt = g.cfirst[mi + 1] - g.cfirst[mi];
  const int c0 = (int)blockIdx.x - g.cfirst[mi];
  const int n_local = c0 < a.n_tiles ? (a.n_tiles - c0 + cnt - 1) / cnt : 0;
  const int S = g.nstage;
  uint64_t* tbar = reinterpret_cast<uint64_t*>(smem + kLHdrTab);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kLHdrBar);
  uint64_t* empty = full + kLMaxStages;
  volatile int* err = reinterpret_cast<volatile int*>(smem + kLHdrErr);
  const lw_table* tb = reinterpret_cast<const lw_table*>(smem + kLRawTab);
  const uint32_t sbase = smem_addr(smem);
  // Let the stream's next kernel be scheduled at once: its CTAs take each SM
  // as this kernel's CTA there exits, and run their prologue (barriers,
  // decode table, first weight copies) while the other SMs still drain.
  pdl_trigger();
  // the decoder table's copy goes out first (its barrier initialised just
  // before it; the CTA barrier below publishes the initialisation)
  if (!TWIN && threadIdx.x == 0) {
    mbar_init(tbar, 1);
    fence_barrier_init();
    table_issue(smem + kLRawTab, a.table, tbar);
  }
  // a producer's first loads (the row ranges of its first 32 tiles) go out
  // before anything else
  uint32_t cr0 = 0u, cr1 = 0u;
  int ct = 0;
  if (producer) l_rows(a, c0, cnt, n_local, (warp - nw) + lane * kLProducers, cr0, cr1, ct);

  // activation rows beyond `batch` stay zero in every stage
  if (BP > 1) {
    for (int s = 0; s < S; ++s)
      for (int i = a.batch * 256 + threadIdx.x; i < BP * 256; i += nthreads)
        reinterpret_cast<float*>(smem + g.ring_off + s * g.stage_bytes + g.x_off)[i] = 0.f;
  }
  int* stage_tile = reinterpret_cast<int*>(smem + kLHdrTiles);
  if (threadIdx.x == 0) {
    *reinterpret_cast<int*>(smem + kLHdrNext) = 0;
    *err = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2 / R);   // every unit of the tile releases it
      stage_tile[s] = -1;
    }
    fence_barrier_init();
  }
  __syncthreads();

  // ---- producers: fill the ring ----
  // kLProducers warps; producer p owns the stages s = p mod kLProducers and
  // fills local tiles i = p, p + kLProducers, ... in order (one warp issuing
  // bulk copies cannot keep HBM busy: each copy holds the issuing thread for
  // a few hundred ns).  Lane j loads the row ranges of the warp's tiles
  // 32 c + j of the current chunk c and the next (in flight a chunk ahead);
  // lane 0 issues each tile's copies once its stage is free.
  if (producer) {
    constexpr uint32_t qpb = QFmt<FMT>::qp_bytes;
    const int pw = warp - nw;                  // producer index
    auto rows_of = [&](int k, uint32_t& r0, uint32_t& r1, int& t) {
      l_rows(a, c0, cnt, n_local, pw + k * kLProducers, r0, r1, t);
    };
    uint32_t nr0, nr1;
    int nt, cb = 0;
    rows_of(32 + lane, nr0, nr1, nt);
    int issued = -1;   // last local tile this warp issued
    // A warp's first tile needs no free stage and its weight copies read the
    // bundle only: they go out before the wait for the previous kernel, its
    // activation copies after it.  Only one tile per warp: the CTA that
    // enters last (after the previous kernel's last CTA left its SM, so the
    // wait returns at once) must reach its activation copies quickly -- it
    // is the one that finishes last -- while the others have slack.
    // an activation row of a tile: 256 fp32 (4-/6-bit) or bf16 (BF16)
    constexpr uint32_t XROW = FMT == kB16 ? 512u : 1024u;
    const uint32_t xbytes = (uint32_t)a.batch * XROW;
    auto copy_xrows = [&](uint8_t* st, int kt, uint64_t* bar) {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(a.x) + (size_t)kt * XROW;
      for (int b = 0; b < a.batch; ++b)
        bulk_g2s(st + g.xb_off + b * XROW, src + (size_t)b * a.K * (XROW / 256), XROW, bar);
    };
    auto copy_x = [&](int k) {
      const int t = __shfl_sync(0xFFFFFFFFu, ct, k);
      if (lane == 0 && !(blockIdx.x == 0 && pw + k * kLProducers == g.stall_tile)) {
        const int i = pw + k * kLProducers, s = i % S;
        copy_xrows(smem + g.ring_off + s * g.stage_bytes, t % a.TK, &full[s]);
      }
    };
    bool waited = false;
    for (int k = 0; pw + k * kLProducers < n_local; ++k) {
      const int i = pw + k * kLProducers;
      if (!waited && (i >= S || k >= 1)) {
        pdl_wait();
        waited = true;
        for (int kk = 0; kk < k; ++kk) copy_x(kk);
      }
      if (k == cb + 32) {   // move to the next chunk; start loading the one after
        cr0 = nr0; cr1 = nr1; ct = nt;
        cb += 32;
        rows_of(cb + 32 + lane, nr0, nr1, nt);
      }
      const int s = i % S;
      int ok = 1;
      if (lane == 0 && i >= S) {   // stage s is free once tile i - S has been consumed
        bool got = mbar_try_wait(&empty[s], ((i / S) - 1) & 1);
        if (!got) {
          const long long t0 = clock64();
          while (!(got = mbar_try_wait(&empty[s], ((i / S) - 1) & 1)))
            if (*err || clock64() - t0 > g.wait_cycles) break;
        }
        if (!got && !*err) report(a.status, LW_DEV_TIMEOUT);
        ok = got && !*err;
      }
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
        if (lane == 0) *err = 1;
        break;
      }
      const int j = k - cb;   // 0..31: lane j of the current chunk
      const uint32_t r0 = __shfl_sync(0xFFFFFFFFu, cr0, j), r1 = __shfl_sync(0xFFFFFFFFu, cr1, j);
      const int t = __shfl_sync(0xFFFFFFFFu, ct, j);
      if (FMT == kB16) {
        // the verbatim information of the tile's rows (lane l: rows 2l and
        // 2l + 1): the 4 flags of the tile's 64-column groups and the index
        // of the row's first verbatim group from there (bundle data only)
        const int strip = t / a.TK, g0 = 4 * (t % a.TK);
        uint8_t* st = smem + g.ring_off + s * g.stage_bytes;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const size_t r = (size_t)strip * 64 + 2 * lane + h;
          const uint32_t* f = a.vflags + r * (size_t)a.GW;
          uint32_t before = 0;
          for (int w = 0; w < g0 / 32; ++w) before += __popc(__ldg(f + w));
          const uint32_t cur = __ldg(f + g0 / 32);
          before += __popc(cur & ((1u << (g0 % 32)) - 1u));
          const uint32_t vb = __ldg(a.vrow_off + r) + before;   // < 2^28 (at most N K / 64)
          *reinterpret_cast<uint32_t*>(st + g.vi_off + 4 * (2 * lane + h)) =
              (vb << 4) | ((cur >> (g0 % 32)) & 15u);
        }
        __syncwarp();   // every lane's stores before lane 0's arrival (a release)
      }
      if (lane == 0) {
        uint8_t* st = smem + g.ring_off + s * g.stage_bytes;
        const bool fits = r1 >= r0 && r1 - r0 <= (uint32_t)(g.stage_rows - 2);
        const uint32_t wbytes = fits ? (r1 - r0) * 128u : 0u;
        const uint32_t mbytes = TWIN ? 0u : 128u;   // mid offsets + lane bit counts
        // the stage records whether the tile fits (read by the consumer after
        // the barrier completes, which orders this store before it)
        *reinterpret_cast<volatile int*>(st + g.x_off + BP * 1024) = fits ? 1 : 0;
        // announce which tile stage s now carries: its consumer waits for this
        // before waiting on the barrier, so it never mistakes the stage's
        // previous phase (same parity, two phases back) for its own
        st_release(&stage_tile[s], i);
        mbar_arrive_expect_tx(&full[s], wbytes + qpb + mbytes + xbytes);
        // testing: a stage armed for copies that are never issued (nothing in
        // flight; its consumer's wait runs out)
        const bool stall = blockIdx.x == 0 && i == g.stall_tile;
        if (!stall) {
          if (wbytes) bulk_g2s(st, a.words + (size_t)r0 * 32, wbytes, &full[s]);
          if (qpb) bulk_g2s(st + g.qp_off, a.qparams + (size_t)t * qpb, qpb, &full[s]);
          if (!TWIN) {
            bulk_g2s(st + g.mid_off, a.lane_mid + (size_t)t * 32, 64, &full[s]);
            bulk_g2s(st + g.lb_off, a.lane_bits + (size_t)t * 32, 64, &full[s]);
          }
          if (waited) copy_xrows(st, t % a.TK, &full[s]);
        }
      }
      issued = i;
    }
    if (!waited) {   // every tile of this warp was in the first pass
      pdl_wait();
      for (int kk = 0; pw + kk * kLProducers <= issued; ++kk) copy_x(kk);
    }
    // after an error: let this warp's copies still in flight land before leaving
    if (lane == 0 && *err)
      for (int i = issued; i >= 0 && i > issued - S; i -= kLProducers) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&full[i % S], (i / S) & 1) && clock64() - t0 <= g.wait_cycles) {
        }
      }
    return;
  }

  // ---- consumers ----
  LDec dec{0u, 0, 21u};
  if (!TWIN) {
    const bool got = mbar_wait(tbar, 0u);
    bool ok = got && table_ok_warp(tb, FMT, QFmt<FMT>::alpha, 10, lane);
    LutShape sh{0, 0, 2048, 2048};
    if (ok) {
      sh = lut_shape_warp(tb->lim_m1, tb->lmin, tb->lmax, lane);
      ok = sh.n <= g.lut_cap;
    }
    if (!ok) {
      if (lane == 0 && warp == 0) report(a.status, got ? LW_DEV_BAD_TABLE : LW_DEV_TIMEOUT);
      *err = 1;
    } else {
      lut_build(tb, sh, sbase + (uint32_t)g.lut_off, warp, nw, lane);
    }
    dec.lutl = sbase + (uint32_t)g.lut_off + 4u * (uint32_t)lane;
    dec.negC = -sh.C;
    dec.sh = 21u + (uint32_t)sh.s;
    // the table is complete before any warp decodes (consumer warps only)
    asm volatile("bar.sync 1, %0;" ::"r"(nw * 32) : "memory");
  }
  pdl_wait();
  int* next = reinterpret_cast<int*>(smem + kLHdrNext);
  // commit pipeline: strip of the unit stored last (not yet counted), and
  // the strip counted last with its pending count (-1: none)
  int ps1 = -1, ps2 = -1;
  uint32_t old2 = 0u;
  constexpr int UPT = 2 / R;            // units per tile
  const int n_units = UPT * n_local;    // unit u: rows 2l + h0 .. 2l + h0 + R - 1 of tile u / UPT
  while (true) {
    int u = 0, e = 0;
    if (lane == 0) {
      u = atomicAdd(next, 1);
      e = *err;
    }
    u = __shfl_sync(0xFFFFFFFFu, u, 0);
    if (u >= n_units) break;
    // after an error in this CTA the remaining units are only counted (see
    // below): no wait, no decode
    bool ghost = __shfl_sync(0xFFFFFFFFu, e, 0) != 0;
    const int i = u / UPT, h0 = R == 1 ? (u & 1) : 0;
    const int s = i % S;
    if (!ghost) {
      // first the producer's announcement that stage s carries tile i (then
      // the barrier's phase i / S is the one in progress), then the barrier
      bool got = ld_acquire(&stage_tile[s]) == i && mbar_try_wait(&full[s], (i / S) & 1);
      if (!got) {
        const long long t0 = clock64();
        bool announced;
        while (!(announced = ld_acquire(&stage_tile[s]) == i)) {
          if (*err || clock64() - t0 > g.wait_cycles) break;
          __nanosleep(64);   // leave the issue slots to the warps that decode
        }
        if (announced)
          while (!(got = mbar_try_wait(&full[s], (i / S) & 1)))
            if (*err || clock64() - t0 > g.wait_cycles) break;
      }
      got = __all_sync(0xFFFFFFFFu, got);
      if (!got) {
        if (lane == 0 && !*err) report(a.status, LW_DEV_TIMEOUT);
        *err = 1;
        ghost = true;
      }
    }
    bool valid;
    const int t = list_tile<true>(a, c0 + i * cnt, valid);   // a tile of the bundle
    const int strip = t / a.TK, kt = t % a.TK;
    float p[R][BP];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < BP; ++b) p[r][b] = 0.f;
    // A ghost unit is counted without a partial sum: every unit of the launch
    // is counted exactly once whatever happens, so each strip counter wraps
    // back to zero and the workspace serves the next call (this launch's
    // outputs are void: *d_status holds the error).
    if (!ghost) {
      const uint32_t wb = sbase + (uint32_t)(g.ring_off + s * g.stage_bytes);
      const uint32_t qp = wb + (uint32_t)g.qp_off;
      const uint32_t sx = wb + (uint32_t)g.x_off;
      const bool fits = lds_s32(sx + BP * 1024) != 0;
      // the unit's row streams: row 2l from the lane's start, row 2l + 1 from its mid offset
      uint32_t start[R], end[R];
      if (!TWIN) {
        const uint32_t mid = lds_u16(wb + (uint32_t)g.mid_off + 2u * (uint32_t)lane);
        const uint32_t last = lds_u16(wb + (uint32_t)g.lb_off + 2u * (uint32_t)lane);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int h = h0 + r;
          start[r] = h ? mid : 0u;
          end[r] = h ? last : mid;
        }
      }
      if (!fits) {
        if (lane == 0) report(a.status, LW_DEV_TILE_SIZE);
      } else if (FMT == kQ4) {
        float xa[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b) xa[b] = tile_sum256(sx + 1024u * b, lane);
        float2 acc[R][BP];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int b = 0; b < BP; ++b) acc[r][b] = make_float2(0.f, 0.f);
        if (!TWIN) {
          LStream st[R];
#pragma unroll
          for (int r = 0; r < R; ++r) st[r].init(wb, lane, g.stage_rows, start[r]);
#pragma unroll 8
          for (int j = 0; j < 64; ++j) {
            float2 v[R][2];
#pragma unroll
            for (int r = 0; r < R; ++r) {
              uint32_t e0, e1;
              l_decode2(st[r], dec, e0, e1);
              v[r][0] = q4_vals(e0);
              v[r][1] = q4_vals(e1);
            }
#pragma unroll
            for (int b = 0; b < BP; ++b) {
              const float4 xv = lds_f4(sx + 1024u * b + 16u * (uint32_t)j);
#pragma unroll
              for (int r = 0; r < R; ++r) {
                acc[r][b] = __ffma2_rn(v[r][0], make_float2(xv.x, xv.y), acc[r][b]);
                acc[r][b] = __ffma2_rn(v[r][1], make_float2(xv.z, xv.w), acc[r][b]);
              }
            }
          }
#pragma unroll
          for (int r = 0; r < R; ++r)
            if (st[r].consumed() != end[r]) report(a.status, LW_DEV_LANE_LENGTH);
        } else {
          // twin: row 2l in words 0..31 of lane l, row 2l + 1 in words 32..63
          const uint32_t la = wb + 4u * (uint32_t)lane + 4096u * (uint32_t)h0;
#pragma unroll 4 / R
          for (int jj = 0; jj < 32; ++jj) {
            float2 v[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) q4_twin_word(lds_u32(la + 4096u * r + 128u * (uint32_t)jj), v[r]);
#pragma unroll
            for (int b = 0; b < BP; ++b) {
              const float4 xa4 = lds_f4(sx + 1024u * b + 32u * (uint32_t)jj);
              const float4 xb4 = lds_f4(sx + 1024u * b + 32u * (uint32_t)jj + 16u);
#pragma unroll
              for (int r = 0; r < R; ++r) {
                acc[r][b] = __ffma2_rn(v[r][0], make_float2(xa4.x, xa4.y), acc[r][b]);
                acc[r][b] = __ffma2_rn(v[r][1], make_float2(xa4.z, xa4.w), acc[r][b]);
                acc[r][b] = __ffma2_rn(v[r][2], make_float2(xb4.x, xb4.y), acc[r][b]);
                acc[r][b] = __ffma2_rn(v[r][3], make_float2(xb4.z, xb4.w), acc[r][b]);
              }
            }
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          // scale | min << 16 of row 2l + h0 + r
          const uint32_t q = lds_u32(qp + 4u * (uint32_t)(2 * lane + h0 + r));
          const float sc = __half2float(__ushort_as_half((unsigned short)(q & 0xFFFFu)));
          const float mn = __half2float(__ushort_as_half((unsigned short)(q >> 16)));
#pragma unroll
          for (int b = 0; b < BP; ++b)
            p[r][b] = fmaf(sc, (acc[r][b].x + acc[r][b].y) - 16.f * xa[b], mn * xa[b]);
        }
      } else if (FMT == kQ6) {  // 6-bit: 16 groups of 16 weights per row
        float X[BP];
#pragma unroll
        for (int b = 0; b < BP; ++b) X[b] = group_sum16(sx + 1024u * b, lane);
        LStream st[R];
        if (!TWIN)
#pragma unroll
          for (int r = 0; r < R; ++r) st[r].init(wb, lane, g.stage_rows, start[r]);
        // twin: row 2l in words 0..47, row 2l + 1 in words 48..95
        const uint32_t la = wb + 4u * (uint32_t)lane + 6144u * (uint32_t)h0;
#pragma unroll 1
        for (int gi = 0; gi < 16; ++gi) {
          float2 acc[R][BP];
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < BP; ++b) acc[r][b] = make_float2(0.f, 0.f);
          if (!TWIN) {
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              float2 v[R];
#pragma unroll
              for (int r = 0; r < R; ++r) {
                uint32_t e0, e1;
                l_decode2(st[r], dec, e0, e1);
                v[r] = make_float2(f16hi_plus(e0, kQ6Unbias), f16hi_plus(e1, kQ6Unbias));
              }
#pragma unroll
              for (int b = 0; b < BP; ++b) {
                const float2 xv = lds_f2(sx + 1024u * b + 64u * (uint32_t)gi + 8u * (uint32_t)m);
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r][b] = __ffma2_rn(v[r], xv, acc[r][b]);
              }
            }
          } else {
#pragma unroll
            for (int r = 0; r < R; ++r) {
              // group gi: codes 16 gi .. 16 gi + 15 at bits 96 gi .. of the row's words
              const uint32_t wa = la + 6144u * r + 128u * (uint32_t)(3 * gi);
              const uint32_t w0 = lds_u32(wa), w1 = lds_u32(wa + 128u), w2 = lds_u32(wa + 256u);
              float v[16];
              v[0] = q6_twin_c<0>(w0, w1);   v[1] = q6_twin_c<6>(w0, w1);
              v[2] = q6_twin_c<12>(w0, w1);  v[3] = q6_twin_c<18>(w0, w1);
              v[4] = q6_twin_c<24>(w0, w1);  v[5] = q6_twin_c<30>(w0, w1);
              v[6] = q6_twin_c<4>(w1, w2);   v[7] = q6_twin_c<10>(w1, w2);
              v[8] = q6_twin_c<16>(w1, w2);  v[9] = q6_twin_c<22>(w1, w2);
              v[10] = q6_twin_c<28>(w1, w2); v[11] = q6_twin_c<2>(w2, 0u);
              v[12] = q6_twin_c<8>(w2, 0u);  v[13] = q6_twin_c<14>(w2, 0u);
              v[14] = q6_twin_c<20>(w2, 0u); v[15] = q6_twin_c<26>(w2, 0u);
#pragma unroll
              for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int b = 0; b < BP; ++b)
                  acc[r][b] = __ffma2_rn(make_float2(v[2 * m], v[2 * m + 1]),
                                         lds_f2(sx + 1024u * b + 64u * (uint32_t)gi + 8u * (uint32_t)m),
                                         acc[r][b]);
            }
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            // scale of group gi of row 2l + h: chunk 2h + gi/8, position gi % 8
            const int h = h0 + r;
            const uint32_t sa = qp + (uint32_t)((((2 * h + (gi >> 3)) * 32) + lane) * 16 + 2 * (gi & 7));
            const float sc = __half2float(__ushort_as_half((unsigned short)lds_u16(sa)));
#pragma unroll
            for (int b = 0; b < BP; ++b) {
              const float Xg = __shfl_sync(0xFFFFFFFFu, X[b], gi);
              p[r][b] = fmaf(sc, (acc[r][b].x + acc[r][b].y) - 96.f * Xg, p[r][b]);
            }
          }
        }
        if (!TWIN)
#pragma unroll
          for (int r = 0; r < R; ++r)
            if (st[r].consumed() != end[r]) report(a.status, LW_DEV_LANE_LENGTH);
      } else {  // BF16 exponent (coded, R = 2): both rows of every lane
        static_assert(FMT != kB16 || (R == 2 && !TWIN), "BF16: coded, whole-tile units");
        // the tile's activations bf16 -> fp32, once, by this warp (rows
        // beyond the batch stay zero)
#pragma unroll
        for (int b = 0; b < BP; ++b)
          if (b < a.batch) {
            const uint4 w8 = lds_u4(wb + (uint32_t)g.xb_off + 512u * b + 16u * (uint32_t)lane);
            float4 lo, hi;
            lo.x = __uint_as_float(w8.x << 16); lo.y = __uint_as_float(w8.x & 0xFFFF0000u);
            lo.z = __uint_as_float(w8.y << 16); lo.w = __uint_as_float(w8.y & 0xFFFF0000u);
            hi.x = __uint_as_float(w8.z << 16); hi.y = __uint_as_float(w8.z & 0xFFFF0000u);
            hi.z = __uint_as_float(w8.w << 16); hi.w = __uint_as_float(w8.w & 0xFFFF0000u);
            float4* xf = reinterpret_cast<float4*>(smem + g.ring_off + s * g.stage_bytes + g.x_off +
                                                   1024 * b + 32 * lane);
            xf[0] = lo;
            xf[1] = hi;
          }
        __syncwarp();
        // per row: the flags of its 4 groups, its first verbatim group from here
        uint32_t fw[2], vb[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t vi = lds_u32(wb + (uint32_t)g.vi_off + 4u * (uint32_t)(2 * lane + h));
          fw[h] = vi & 15u;
          vb[h] = vi >> 4;
        }
        LStream st[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) st[h].init(wb, lane, g.stage_rows, start[h]);
        // sign+mantissa bytes of row h's 16-weight chunk k: one 16-byte load
        // per lane, a chunk ahead; a verbatim group's raw exponents likewise
        const uint4* smb = reinterpret_cast<const uint4*>(a.signman + (size_t)t * 16384) + lane;
        const uint4* veb = reinterpret_cast<const uint4*>(a.vexp);
        uint4 nsm[2], nve[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          nsm[h] = __ldg(smb + (16 * h) * 32);
          nve[h] = (fw[h] & 1u) ? __ldg(veb + (size_t)vb[h] * 4) : make_uint4(0u, 0u, 0u, 0u);
        }
        float2 acc[2][BP];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int b = 0; b < BP; ++b) acc[h][b] = make_float2(0.f, 0.f);
#pragma unroll 1
        for (int k = 0; k < 16; ++k) {
          uint4 sm[2], ve[2];
          uint32_t go[2], vm[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            sm[h] = nsm[h];
            ve[h] = nve[h];
            const bool v = (fw[h] >> (k >> 2)) & 1u;
            go[h] = v ? 0u : 1u;   // a verbatim group holds the stream
            vm[h] = v ? 0xFFFFFFFFu : 0u;
            if (k < 15) {
              const int g1 = (k + 1) >> 2;
              nsm[h] = __ldg(smb + (16 * h + k + 1) * 32);
              nve[h] = ((fw[h] >> g1) & 1u)
                           ? __ldg(veb + (size_t)(vb[h] + __popc(fw[h] & ((1u << g1) - 1u))) * 4 +
                                   ((k + 1) & 3))
                           : make_uint4(0u, 0u, 0u, 0u);
            }
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {   // weights 2q, 2q + 1 of the chunk
            float2 f[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t e0, e1;
              l_decode2(st[h], dec, e0, e1, go[h]);
              const uint32_t sw = l_word(sm[h], q >> 1), vw = l_word(ve[h], q >> 1);
              // exponent fields: the entry's, or the verbatim byte j (2 (q & 1) and
              // 2 (q & 1) + 1 of word vw) moved to bits 23..30 (b16_value reads
              // nothing else of it) -- by a multiply where a left shift does
              const uint32_t ve0 = (q & 1) ? imad(vw, 1u << 7, 0u) : imad(vw, 1u << 23, 0u);
              const uint32_t ve1 = (q & 1) ? vw >> 1 : imad(vw, 1u << 15, 0u);
              const uint32_t E0 = (e0 & ~vm[h]) | (ve0 & vm[h]);
              const uint32_t E1 = (e1 & ~vm[h]) | (ve1 & vm[h]);
              f[h] = (q & 1) ? make_float2(b16_value<2>(sw, E0), b16_value<3>(sw, E1))
                             : make_float2(b16_value<0>(sw, E0), b16_value<1>(sw, E1));
            }
#pragma unroll
            for (int b = 0; b < BP; ++b) {
              const float2 xv = lds_f2(sx + 1024u * b + 4u * (uint32_t)(16 * k + 2 * q));
#pragma unroll
              for (int h = 0; h < 2; ++h) acc[h][b] = __ffma2_rn(f[h], xv, acc[h][b]);
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int b = 0; b < BP; ++b) p[h][b] = acc[h][b].x + acc[h][b].y;
          if (st[h].consumed() != end[h]) report(a.status, LW_DEV_LANE_LENGTH);
        }
      }
      // release the stage (UPT units per stage): this warp's reads of it are
      // done (their values are in the partial sums), ordered before the
      // producer's next bulk copy into it
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      // a tile too long for its stage commits zeros, so that its strip still
      // completes; a tile behind an invalid strip-list entry commits nothing
      if (!valid && lane == 0 && h0 == 0) report(a.status, LW_DEV_BAD_STRIPS);
    }
    if (ps2 >= 0) l_finish<UPT>(a, ps2, lane, old2);
    ps2 = ps1;
    if (ps1 >= 0) old2 = l_count<UPT>(a, ps1, lane);
    if (valid && !ghost) l_store<R, BP>(a, strip, kt, 2 * lane + h0, p);
    ps1 = valid ? strip : -1;
  }
  // drain: the last count's round trip overlaps the pending finish
  const uint32_t old1 = ps1 >= 0 ? l_count<UPT>(a, ps1, lane) : 0u;
  if (ps2 >= 0) l_finish<UPT>(a, ps2, lane, old2);
  if (ps1 >= 0) l_finish<UPT>(a, ps1, lane, old1);
}

}  // namespace dev
}  // namespace lw
