// Launchers for the BF16 exponent-coded kernels (lw_bkern.cuh, lw_btc.cuh),
// and the split-K sum and grid choice that both tensor-core products (BF16
// and 4-/6-bit) share.
#include "lw_btc.cuh"
#include "lw_internal.h"
#include "lw_launch.h"

namespace lw {

namespace {

using BKernel = void (*)(const dev::BArgs);

int ncmp_bucket_b(int span) { return span <= 4 ? 4 : (span <= 8 ? 8 : 10); }

template <bool TWIN, int BP>
BKernel pick_b_product(int ncmp) {
  if (TWIN) return dev::b_product_kernel<true, BP, 0>;
  switch (ncmp) {
    case 4: return dev::b_product_kernel<false, BP, 4>;
    case 8: return dev::b_product_kernel<false, BP, 8>;
    default: return dev::b_product_kernel<false, BP, 10>;
  }
}

template <bool TWIN>
BKernel pick_b_product_bp(int bp, int ncmp) {
  switch (bp) {
    case 1: return pick_b_product<TWIN, 1>(ncmp);
    case 2: return pick_b_product<TWIN, 2>(ncmp);
    case 4: return pick_b_product<TWIN, 4>(ncmp);
    default: return pick_b_product<TWIN, 8>(ncmp);
  }
}

BKernel pick_b_decode(bool twin, int ncmp) {
  if (twin) return dev::b_decode_kernel<true, 0>;
  switch (ncmp) {
    case 4: return dev::b_decode_kernel<false, 4>;
    case 8: return dev::b_decode_kernel<false, 8>;
    default: return dev::b_decode_kernel<false, 10>;
  }
}

dev::BArgs common_args(const lw_dev_bundle* b) {
  dev::BArgs a{};
  a.words = b->words;
  a.tile_off = b->tile_off;
  a.lane_bits = b->lane_bits;
  a.lane_mid = b->twin ? nullptr : b->lane_mid;
  a.table = b->table;
  a.signman = b->signman;
  a.vflags = b->vflags;
  a.vrow_off = b->vrow_off;
  a.vexp = b->vexp;
  a.TK = (int)(b->cols / 256);
  a.N = (int)b->rows;
  a.K = (int)b->cols;
  a.GW = (int)((b->cols / 64 + 31) / 32);
  a.n_tiles = (int)tiles_of(b->rows, b->cols);
  a.stage_rows = b->max_tile_rows + dev::kLookahead;
  return a;
}

BKernel pick_b_tc(int ncmp, bool lut, bool twin) {
  if (twin) return dev::b_tc_kernel<2, false, true>;
  if (lut) return dev::b_tc_kernel<10, true, false>;
  switch (ncmp) {
    case 4: return dev::b_tc_kernel<4, false, false>;
    case 8: return dev::b_tc_kernel<8, false, false>;
    default: return dev::b_tc_kernel<10, false, false>;
  }
}

// entries of a replicated decode table the tensor-core kernel takes (128 B
// each; larger tables decode by the comparator)
constexpr int kTcLutCap = 256;

}  // namespace

// Tensor-core product for 16..64 activation rows: the product kernel, and
// the split-K sum behind it when a row block's K range is split over CTAs;
// coded bundles and their direct-palette twins.
lw_status launch_bf16_tc_product(const lw_dev_bundle* b, const uint16_t* x, int batch, float* y,
                                 void* ws, int32_t* status, cudaStream_t st) {
  const bool twin = b->twin != 0;
  const bool lut = !twin && b->lut_entries >= 1 && b->lut_entries <= kTcLutCap;
  BKernel k = pick_b_tc(twin ? 0 : ncmp_bucket_b(b->lmax - b->lmin), lut, twin);
  dev::BArgs a = common_args(b);
  a.x = x;
  a.y = y;
  a.ws = workspace_partials(b, ws);
  a.counters = workspace_counters(b, ws);
  a.status = status;
  a.batch = batch;
  a.bpad = (batch + 15) / 16 * 16;
  const int need = dev::tc_tmem_need(a.bpad);
  a.tmem_cols = need <= 32 ? 32 : (need <= 64 ? 64 : (need <= 128 ? 128 : 256));
  a.mid_offset = a.stage_rows * 128;
  a.stage_bytes = (a.mid_offset + 128 + 127) / 128 * 128;
  // header | X^T halves (2 x bpad x 256 B) | tile stages (4 strips x 2)
  a.xs_off = dev::kTcXsOff;
  a.wstage_off = a.xs_off + 2 * a.bpad * 256;
  size_t smem = (size_t)a.wstage_off + 8 * (size_t)a.stage_bytes;
  if (lut) {   // the replicated decode table after the stages
    a.lut_off = (int)((smem + 127) / 128 * 128);
    a.lut_cap = b->lut_entries;
    smem = (size_t)a.lut_off + (size_t)a.lut_cap * 128;
  }
  const int per_sm = tc_resident_blocks((const void*)k, dev::kTcThreads, smem, a.tmem_cols);
  if (per_sm < 1) return fail(LW_ERR_UNSUPPORTED, "tensor-core kernel does not fit (%zu B smem)", smem);
  const int n_blocks = (int)((b->rows / 64 + 3) / 4);
  const TcGrid g = tc_pick_grid(n_blocks, a.TK, tc_max_split(b), per_sm * device_sm_count());
  launch_pdl(k, g.G, dev::kTcThreads, smem, st, a);
  lw_status s = check_launch("tensor-core product kernel");
  if (s == LW_OK && g.owners > 1) s = launch_tc_sum(a.ws, y, (int)b->rows, batch, a.TK, g.G, st);
  return s;
}

namespace dev {

// The split-K sum of a tensor-core product whose row blocks were split over
// CTAs (tc_owner): y[b][n] = partial 0 + partial 1 + ... of n's row block,
// in ascending order (partial j at ws[j][b][n]).  A kernel of its own,
// launched right behind the product with programmatic dependent launch, so
// that every SM takes part in the sum (a sum by one CTA per row block would
// be held to that SM's share of the L2 bandwidth).  One thread per 4
// consecutive outputs (N is a multiple of 64), kSumDepth loads in flight.
struct TcSumArgs {
  const float* ws;   // [owners][batch][N] fp32, 16-byte aligned
  float* y;          // [batch][N] fp32, 8-byte aligned
  int N, batch, TK, G;
};
constexpr int kSumThreads = 256;
constexpr int kSumDepth = 8;

// WIDE: T x (G + 1) does not fit 32 bits (the owners in 64-bit arithmetic)
template <bool WIDE>
__global__ void __launch_bounds__(kSumThreads) tc_sum_kernel(const TcSumArgs a) {
  pdl_trigger();
  pdl_wait();   // the product's partials are complete and visible
  const int n4 = a.N / 4;
  const size_t groups = (size_t)a.batch * n4;
  const size_t g = (size_t)blockIdx.x * kSumThreads + threadIdx.x;
  if (g >= groups) return;
  const int n = 4 * (int)(g % (size_t)n4);
  const long long T = (long long)((a.N / 64 + 3) / 4) * a.TK;
  const int rb = n >> 8;
  const int owners = WIDE ? tc_owners_of(rb, a.TK, T, a.G)
                          : tc_owners_of32(rb, a.TK, (uint32_t)T, (uint32_t)a.G);
  if (owners == 1) return;   // written by the product
  const float4* p = reinterpret_cast<const float4*>(a.ws) + g;
  const size_t step4 = groups;   // one partial, in float4
  float4 acc = __ldcg(p);
  for (int q0 = 1; q0 < owners; q0 += kSumDepth) {
    float4 v[kSumDepth];
#pragma unroll
    for (int j = 0; j < kSumDepth; ++j)
      if (q0 + j < owners) v[j] = __ldcg(p + (size_t)(q0 + j) * step4);
#pragma unroll
    for (int j = 0; j < kSumDepth; ++j) {
      if (q0 + j < owners) {
        acc.x += v[j].x;
        acc.y += v[j].y;
        acc.z += v[j].z;
        acc.w += v[j].w;
      }
    }
  }
  float2* yp = reinterpret_cast<float2*>(a.y + 4 * g);
  yp[0] = make_float2(acc.x, acc.y);
  yp[1] = make_float2(acc.z, acc.w);
}

}  // namespace dev

lw_status launch_tc_sum(const float* ws, float* y, int N, int batch, int TK, int G, cudaStream_t st) {
  dev::TcSumArgs a{ws, y, N, batch, TK, G};
  const long long groups = (long long)batch * N / 4;
  const int grid = (int)((groups + dev::kSumThreads - 1) / dev::kSumThreads);
  const unsigned long long T = (unsigned long long)((N / 64 + 3) / 4) * (unsigned long long)TK;
  if (T * (unsigned long long)(G + 1) >= (1ull << 32))
    launch_pdl(dev::tc_sum_kernel<true>, grid, dev::kSumThreads, 0, st, a);
  else
    launch_pdl(dev::tc_sum_kernel<false>, grid, dev::kSumThreads, 0, st, a);
  return check_launch("split-K sum kernel");
}

TcGrid tc_pick_grid(int n_blocks, int TK, int max_split, int slots) {
  // a few recent shapes per host thread (the pick is pure host arithmetic)
  struct Entry {
    int key[4];
    TcGrid g;
  };
  thread_local Entry cache[8];
  thread_local int used = 0, next = 0;
  const int key[4] = {n_blocks, TK, max_split, slots};
  for (int i = 0; i < used; ++i)
    if (cache[i].key[0] == key[0] && cache[i].key[1] == key[1] && cache[i].key[2] == key[2] &&
        cache[i].key[3] == key[3])
      return cache[i].g;
  const TcGrid g = tc_plan(n_blocks, TK, max_split, slots);
  Entry& e = cache[next];
  for (int i = 0; i < 4; ++i) e.key[i] = key[i];
  e.g = g;
  next = (next + 1) % 8;
  if (used < 8) ++used;
  return g;
}

lw_status launch_bf16_product(const lw_dev_bundle* b, const uint16_t* x, int batch, float* y,
                              void* ws, int32_t* status, cudaStream_t st) {
  const bool twin = b->twin != 0;
  const int ncmp = twin ? 0 : ncmp_bucket_b(b->lmax - b->lmin);
  for (int b0 = 0; b0 < batch; b0 += 8) {
    const int nb = batch - b0 < 8 ? batch - b0 : 8;
    if (lut_takes(&b, 1, nb)) {   // the table-driven kernel (same result bits)
      const float* xp = reinterpret_cast<const float*>(x + (size_t)b0 * b->cols);
      float* yp = y + (size_t)b0 * b->rows;
      void* wp = ws;
      const lw_status s = launch_q_lut(&b, 1, &xp, nb, &yp, &wp, status, st);
      if (s != LW_OK) return s;
      continue;
    }
    const int bp = nb <= 1 ? 1 : (nb <= 2 ? 2 : (nb <= 4 ? 4 : 8));
    BKernel k = twin ? pick_b_product_bp<true>(bp, ncmp) : pick_b_product_bp<false>(bp, ncmp);
    dev::BArgs a = common_args(b);
    a.x = x + (size_t)b0 * b->cols;
    a.ws = workspace_partials(b, ws);
    a.counters = workspace_counters(b, ws);
    a.y = y + (size_t)b0 * b->rows;
    a.status = status;
    a.batch = nb;
    // stage: coded rows | activations bf16 (bp x 512 B) | lane_mid (64 B) |
    // activations fp32 (bp x 1 KB)
    a.x_offset = a.stage_rows * 128;
    a.mid_offset = a.x_offset + bp * 512;
    a.xf_offset = a.mid_offset + 128;
    a.stage_bytes = (a.xf_offset + bp * 1024 + 127) / 128 * 128;
    const size_t smem = (size_t)dev::kStageOff + (size_t)a.stage_bytes;
    lw_status s = launch_persistent((const void*)k, 64, smem, a.n_tiles, st, [&](int blocks) {
      launch_pdl(k, blocks, 64, smem, st, a);
    });
    if (s != LW_OK) return s;
  }
  return LW_OK;
}

lw_status launch_bf16_decode(const lw_dev_bundle* b, void* out, int32_t* status, cudaStream_t st) {
  const bool twin = b->twin != 0;
  BKernel k = pick_b_decode(twin, twin ? 0 : ncmp_bucket_b(b->lmax - b->lmin));
  dev::BArgs a = common_args(b);
  a.out = static_cast<uint16_t*>(out);
  a.status = status;
  a.mid_offset = a.stage_rows * 128;
  a.stage_bytes = (a.mid_offset + 64 + 127) / 128 * 128;
  const size_t smem = (size_t)dev::kStageOff + (size_t)a.stage_bytes;
  return launch_persistent((const void*)k, 64, smem, a.n_tiles, st, [&](int blocks) {
    launch_pdl(k, blocks, 64, smem, st, a);
  });
}

}  // namespace lw
