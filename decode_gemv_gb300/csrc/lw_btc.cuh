// BF16 exponent-coded weights times a batch of 16..64 activation rows on the
// 5th-generation tensor cores: decode, rebuild BF16 in shared memory, feed
// tcgen05.mma (BF16 x BF16 -> FP32 in tensor memory).
//
// "Unweight: Compressing LLM Weights for Faster Inference", "How
// reconstructive matmul works": compressed data is loaded, BF16 values are
// reconstructed in shared memory and fed to the tensor cores without a trip
// through main memory.  The Hopper producer/consumer/WGMMA design of the page
// becomes, on sm_103a:
//  * a CTA of 4 warps owns 256 output rows (4 row strips) and a range of
//    256-column tile columns; warp w decodes the tile of strip w;
//  * the lane's two rows are decoded in 16-column chunks; after each chunk
//    the 4 warps have written a 256 x 16 slab of BF16 weights into shared
//    memory in the tensor core's K-major, no-swizzle layout (8x8 core
//    matrices); one thread then issues two tcgen05.mma (M = 128 each, N =
//    the padded batch, K = 16) against the matching slice of X^T, staged per
//    tile column in the same layout, accumulating in tensor memory;
//  * tcgen05.commit on a per-slot mbarrier tells the decoders when a slab
//    buffer may be rewritten (a ring of kSlots slabs);
//  * the accumulators are read back with tcgen05.ld (warp w reads tensor
//    memory lanes 32w..32w+31); split-K partials are added in ascending
//    split order by the last CTA of each 256-row block.
// Every wait is bounded; on a timeout the CTA reports LW_DEV_TIMEOUT, waits
// (bounded) for its own MMAs, frees its tensor memory and returns.
#pragma once

#include "lw_bkern.cuh"

namespace lw {
namespace dev {

constexpr int kSlots = 4;            // slab ring depth
constexpr int kSlabBytes = 128 * 16 * 2;   // M = 128 rows x K = 16 bf16

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

// ---- the kernel -----------------------------------------------------------
template <int NCMP>
__global__ void __launch_bounds__(128, 1) b_tc_kernel(const BArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t s_off = sbase + kOffOff;
  const uint32_t s_tab = sbase + kBTabOff;
  uint64_t* wbar = reinterpret_cast<uint64_t*>(smem + 256) + warp;   // this warp's tile copy
  uint64_t* sbar = reinterpret_cast<uint64_t*>(smem + 288);          // [kSlots] slab ring
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(smem + 320);
  volatile uint32_t* shared_word = reinterpret_cast<volatile uint32_t*>(smem + 324);
  const uint32_t slab0 = sbase + (uint32_t)a.slab_off;   // [pair 2][slot][4 KB]
  const uint32_t xs = sbase + (uint32_t)a.xs_off;        // X^T for one tile column
  uint8_t* wstage = smem + a.wstage_off + warp * a.stage_bytes;

  if (lane == 0) mbar_init(wbar, 1);
  if (tid == 0)
    for (int s = 0; s < kSlots; ++s) mbar_init(&sbar[s], 1);
  if (lane == 0) fence_barrier_init();
  if (warp == 0) {
    tmem_alloc(smem_addr(const_cast<uint32_t*>(tslot)), (uint32_t)a.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 0) {
    if (lane == 0)
      *reinterpret_cast<volatile int*>(smem + kFlagOff) =
          table_ok(a.table, LW_FMT_BF16_EXP, 16, NCMP) ? 0 : 1;
    if (lane < 16) {
      put_off<(NCMP + 1) / 2>(smem, lane,
          s_tab + (uint32_t)(4 * (lane < 12 ? a.table->off[lane] : 0)));
      const uint32_t sy = a.table->sym[lane] & 15u;
      reinterpret_cast<uint32_t*>(smem + kBTabOff)[lane] = (uint32_t)a.table->palette[sy] << 23;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool failed = false;      // stop: rejected table or a wait that ran out
  bool timed_out = false;   // a wait ran out (reported as LW_DEV_TIMEOUT)
  bool copy_pending = false;  // this warp's tile copy may still be in flight
  uint32_t pending_par = 0;   // ... on this phase of wbar
  uint32_t gchunk = 0;   // slab commits issued by this CTA so far (uniform)
  if (*reinterpret_cast<volatile int*>(smem + kFlagOff)) {
    if (tid == 0) report(a.status, LW_DEV_BAD_TABLE);
    failed = true;
  }
  constexpr int NP = (NCMP + 1) / 2;
  Cmp<NP> cmp;
  int lmin = 1;
  if (!failed) {
    cmp.load(a.table, a.table->lmax - a.table->lmin);
    lmin = a.table->lmin;
  }
  const uint32_t idesc = idesc_bf16((uint32_t)a.bpad);
  const int n_strips = a.N / 64;
  const int n_blocks = (n_strips + 3) / 4;
  const int units = n_blocks * a.nsplit;
  uint32_t wpar = 0;

  for (int u = blockIdx.x; u < units && !failed; u += gridDim.x) {
    const int rb = u / a.nsplit, sp = u % a.nsplit;
    const int kt0 = (int)((long long)a.TK * sp / a.nsplit);
    const int kt1 = (int)((long long)a.TK * (sp + 1) / a.nsplit);
    const int strip = rb * 4 + warp;
    const bool has = strip < n_strips;
    const size_t r0 = (size_t)strip * 64 + 2 * lane;
    bool first = true;
    for (int kt = kt0; kt < kt1 && !failed; ++kt) {
      const int t = strip * a.TK + kt;
      bool fit = true;
      if (has)
        fit = b_issue<false, false>(a, t, __ldg(a.tile_off + t), __ldg(a.tile_off + t + 1), wstage,
                                    wbar, lane);
      uint32_t fw0 = 0, vb0 = 0, fw1 = 0, vb1 = 0;
      if (has) {
        b_row_flags(a, r0, kt, fw0, vb0);
        b_row_flags(a, r0 + 1, kt, fw1, vb1);
      }
      // the X^T stage is rewritten only after the MMAs reading it are done
      bool to = false;
      if (gchunk > 0) to = !mbar_wait(&sbar[(gchunk - 1) % kSlots], ((gchunk - 1) / kSlots) & 1u);
      if (__syncthreads_or(to)) {
        failed = timed_out = true;
        copy_pending = has;
        pending_par = wpar;
        break;
      }
      for (int i = tid; i < a.bpad * 32; i += 128) {
        const int n = i >> 5, kb = i & 31;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (n < a.batch)
          v = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)n * a.K + (size_t)kt * 256 + 8 * kb));
        *reinterpret_cast<uint4*>(smem + a.xs_off + (n >> 3) * 4096 + kb * 128 + (n & 7) * 16) = v;
      }
      fence_proxy_async();
      if (has) {
        to = !mbar_wait(wbar, wpar);
        copy_pending = to;
        pending_par = wpar;
        wpar ^= 1u;
      }
      const uint32_t wb = smem_addr(wstage);
      LaneBits la, lr;
      uint32_t mid = 0;
      const bool dec = has && fit && !to;
      if (dec) {
        mid = lds_u16(wb + (uint32_t)a.mid_offset + 2u * (uint32_t)lane);
        la.init(wb, lane, a.stage_rows);
        lr.init_at(wb, lane, a.stage_rows, mid);
      }
      if (has && !fit && lane == 0) report(a.status, LW_DEV_TILE_SIZE);
      uint4 n_sm0 = make_uint4(0, 0, 0, 0), n_sm1 = n_sm0, n_ve0 = n_sm0, n_ve1 = n_sm0;
      if (dec) {
        n_sm0 = b_load_sm(a, t, lane, 0, 0);
        n_sm1 = b_load_sm(a, t, lane, 1, 0);
        if (fw0 & 1u) n_ve0 = b_load_vexp(a, vb0, 0);
        if (fw1 & 1u) n_ve1 = b_load_vexp(a, vb1, 0);
      }
      for (int k = 0; k < 16; ++k) {
        const uint32_t s = gchunk % kSlots;
        bool to2 = to;
        if (gchunk >= (uint32_t)kSlots)
          to2 |= !mbar_wait(&sbar[s], ((gchunk - kSlots) / kSlots) & 1u);
        uint32_t W0[8], W1[8];   // bf16x2 of rows 2l and 2l+1, columns 16k .. 16k+15
        if (dec) {
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
          for (int p = 0; p < 8; ++p) {
            uint32_t E[4];
            const uint32_t wv0 = u4w(ve0, p >> 1), wv1 = u4w(ve1, p >> 1);
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
            const uint32_t s0 = u4w(sm0, p >> 1), s1 = u4w(sm1, p >> 1);
            uint32_t f[4];
            if (p & 1) {
              f[0] = __float_as_uint(b_value<2>(s0, E[0]));
              f[1] = __float_as_uint(b_value<3>(s0, E[1]));
              f[2] = __float_as_uint(b_value<2>(s1, E[2]));
              f[3] = __float_as_uint(b_value<3>(s1, E[3]));
            } else {
              f[0] = __float_as_uint(b_value<0>(s0, E[0]));
              f[1] = __float_as_uint(b_value<1>(s0, E[1]));
              f[2] = __float_as_uint(b_value<0>(s1, E[2]));
              f[3] = __float_as_uint(b_value<1>(s1, E[3]));
            }
            W0[p] = __byte_perm(f[0], f[1], 0x7632);   // (bf16 of f1) << 16 | bf16 of f0
            W1[p] = __byte_perm(f[2], f[3], 0x7632);
          }
        } else {
#pragma unroll
          for (int p = 0; p < 8; ++p) W0[p] = W1[p] = 0u;
        }
        // rows m = 64 (warp & 1) + 2 lane + h of pair (warp >> 1)'s slab
        const uint32_t slab = slab0 + (uint32_t)(((warp >> 1) * kSlots + (int)s) * kSlabBytes);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t* W = h ? W1 : W0;
          const uint32_t m = (uint32_t)(64 * (warp & 1) + 2 * lane + h);
          uint8_t* row = smem + (slab - sbase) + (m >> 3) * 256 + (m & 7) * 16;
          *reinterpret_cast<uint4*>(row) = make_uint4(W[0], W[1], W[2], W[3]);
          *reinterpret_cast<uint4*>(row + 128) = make_uint4(W[4], W[5], W[6], W[7]);
        }
        fence_proxy_async();
        if (__syncthreads_or(to2)) { failed = timed_out = true; break; }
        if (tid == 0) {
          tc_fence_after();
          const uint64_t bd = sdesc(xs + 256u * (uint32_t)k, 128u, 4096u);
          umma_bf16(tmem, sdesc(slab0 + s * kSlabBytes, 128u, 256u), bd, idesc, first ? 0u : 1u);
          umma_bf16(tmem + (uint32_t)a.bpad, sdesc(slab0 + (kSlots + s) * kSlabBytes, 128u, 256u), bd,
                    idesc, first ? 0u : 1u);
          umma_commit(&sbar[s]);
        }
        first = false;
        ++gchunk;
      }
      if (dec && (la.consumed() != mid ||
                  lr.consumed() != (uint32_t)__ldg(a.lane_bits + (size_t)t * 32 + lane)))
        report(a.status, LW_DEV_LANE_LENGTH);
    }
    if (failed) break;
    // all MMAs of this unit done -> read the accumulators
    bool to3 = !mbar_wait(&sbar[(gchunk - 1) % kSlots], ((gchunk - 1) / kSlots) & 1u);
    if (__syncthreads_or(to3)) { failed = timed_out = true; break; }
    tc_fence_after();
    const size_t rows0 = (size_t)rb * 256 + 32 * warp + lane;   // D0 row; D1 row = +128
    const size_t step = (size_t)a.batch * a.N;
    for (int p = 0; p < 2; ++p) {
      const size_t row = rows0 + 128 * p;
      for (int j = 0; j < a.bpad; j += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(p * a.bpad + j), r);
        tmem_ld_wait();
        if (row < (size_t)a.N) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int b = j + i;
            if (b < a.batch) {
              if (a.nsplit == 1) a.y[(size_t)b * a.N + row] = __uint_as_float(r[i]);
              else a.ws[(size_t)sp * step + (size_t)b * a.N + row] = __uint_as_float(r[i]);
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();   // accumulators read before the next unit overwrites them
    if (a.nsplit > 1) {
      // the last split of this row block to finish adds the splits in order
      if (tid == 0) *shared_word = atom_inc_acq_rel(a.counters + rb, (unsigned)(a.nsplit - 1));
      __syncthreads();
      const bool last = *shared_word == (uint32_t)(a.nsplit - 1);
      __syncthreads();
      if (last) {
        for (int i = tid; i < 256 * a.batch; i += 128) {
          const int b = i >> 8;
          const size_t row = (size_t)rb * 256 + (i & 255);
          if (row >= (size_t)a.N) continue;
          const float* p = a.ws + (size_t)b * a.N + row;
          float acc = __ldcg(p);
          for (int q = 1; q < a.nsplit; ++q) acc += __ldcg(p + (size_t)q * step);
          a.y[(size_t)b * a.N + row] = acc;
        }
      }
    }
  }
  if (timed_out) {
    if (tid == 0) report(a.status, LW_DEV_TIMEOUT);
    // let this CTA's own MMAs and tile copy finish (bounded) before leaving
    if (gchunk > 0) mbar_wait(&sbar[(gchunk - 1) % kSlots], ((gchunk - 1) / kSlots) & 1u);
    if (copy_pending) mbar_wait(wbar, pending_par);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
}

}  // namespace dev
}  // namespace lw
