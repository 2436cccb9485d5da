// Launcher of the table-driven 4-/6-bit product kernel (lw_qlut.cuh) and of
// its fixed-width-twin instantiations.
#include <mutex>

#include "lw_internal.h"
#include <atomic>

#include "lw_launch.h"
#include "lw_qlut.cuh"

namespace lw {

namespace {

using LKernel = void (*)(const dev::LLaunch);

template <int FMT, bool TWIN, int R>
LKernel pick_lut_r(int bp) {
  switch (bp) {
    case 1: return dev::q_lut_kernel<FMT, TWIN, 1, R>;
    case 2: return dev::q_lut_kernel<FMT, TWIN, 2, R>;
    case 4: return dev::q_lut_kernel<FMT, TWIN, 4, R>;
    default: return dev::q_lut_kernel<FMT, TWIN, 8, R>;
  }
}
template <int FMT, bool TWIN>
LKernel pick_lut(int bp, int r) {
  return r == 2 ? pick_lut_r<FMT, TWIN, 2>(bp) : pick_lut_r<FMT, TWIN, 1>(bp);
}
// BF16 exponent bundles: coded, whole-tile units, up to 4 rows per pass
LKernel pick_lut_b16(int bp) {
  switch (bp) {
    case 1: return dev::q_lut_kernel<dev::kB16, false, 1, 2>;
    case 2: return dev::q_lut_kernel<dev::kB16, false, 2, 2>;
    default: return dev::q_lut_kernel<dev::kB16, false, 4, 2>;
  }
}

// Largest dynamic shared memory a CTA may use on the current device.
int max_dyn_smem() {
  static std::mutex mu;
  static int cache[128] = {0};
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 128) return 0;
  std::lock_guard<std::mutex> g(mu);
  if (!cache[d]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    cache[d] = v > 0 ? v : 1;
  }
  return cache[d];
}

// The ring of a launch of n matrices of one format at `batch` activation
// rows: stage layout, table capacity and stage count S (capped at
// kLMaxStages, a multiple of the producer count).
struct LRing {
  int bp, stage_rows, qp_off, mid_off, lb_off, vi_off, xb_off, x_off, stage_bytes, ring_off, lut_cap,
      lut_bytes, S;
};
LRing lut_ring(const lw_dev_bundle* const* bs, int n, int batch) {
  LRing r{};
  const int fmt = bs[0]->fmt;
  const bool twin = bs[0]->twin != 0;
  r.bp = batch <= 1 ? 1 : (batch <= 2 ? 2 : (batch <= 4 ? 4 : 8));
  int max_rows = 0;
  for (int i = 0; i < n; ++i) max_rows = bs[i]->max_tile_rows > max_rows ? bs[i]->max_tile_rows : max_rows;
  // stage: coded rows (a stream reads up to two rows past its last word) |
  // scales/mins | mid offsets | lane bit counts | [BF16: verbatim
  // information (4 B per row), bf16 activation rows] | fp32 activation rows
  // | "fits" flag
  r.stage_rows = max_rows + 2;
  r.qp_off = r.stage_rows * 128;
  r.mid_off = r.qp_off + qparam_tile_bytes(fmt);
  r.lb_off = r.mid_off + 64;
  if (fmt == LW_FMT_BF16_EXP) {
    r.vi_off = r.mid_off + 128;
    r.xb_off = r.vi_off + 256;
    r.x_off = r.xb_off + r.bp * 512;
  } else {
    r.vi_off = 0;
    r.x_off = r.xb_off = r.mid_off + (twin ? 0 : 128);
  }
  r.stage_bytes = (r.x_off + r.bp * 1024 + 16 + 127) / 128 * 128;
  r.ring_off = (dev::kLHdrBytes + 127) / 128 * 128;
  // the decode table: the largest member's entries (the device checks each
  // table against it), and at least the rows a corrupt stream of the last
  // stage could read past it
  int lut_cap = 0;
  for (int i = 0; i < n; ++i) lut_cap = bs[i]->lut_entries > lut_cap ? bs[i]->lut_entries : lut_cap;
  if (lut_cap < dev::kLGuardRows) lut_cap = dev::kLGuardRows;
  r.lut_cap = lut_cap;
  r.lut_bytes = twin ? 0 : lut_cap * 128;
  int S = (max_dyn_smem() - r.ring_off - r.lut_bytes) / r.stage_bytes;
  if (S > dev::kLMaxStages) S = dev::kLMaxStages;
  S -= S % dev::kLProducers;   // every stage has one producer: stage s, producer s mod 4
  r.S = S;
  return r;
}

}  // namespace

bool lut_fits(const lw_dev_bundle* b) {
  return b->twin || (b->lut_entries >= 1 && b->lut_entries <= kLutCap);
}

bool lut_takes(const lw_dev_bundle* const* bs, int n, int batch) {
  const int fmt = bs[0]->fmt;
  if (fmt == LW_FMT_BF16_EXP && (n != 1 || bs[0]->twin)) return false;
  const int max_rows = fmt == LW_FMT_Q6 ? kLutMaxRowsQ6 : (fmt == LW_FMT_Q4_PAIR ? kLutMaxRowsQ4
                                                                               : kLutMaxRowsB16);
  if (batch > max_rows) return false;
  for (int i = 0; i < n; ++i)
    if (!lut_fits(bs[i])) return false;
  return true;
}

lw_status launch_q_lut(const lw_dev_bundle* const* bs, int n, const float* const* x, int batch,
                       float* const* y, void* const* ws, int32_t* status, cudaStream_t st,
                       const int32_t* strips, int n_strips) {
  const int fmt = bs[0]->fmt;
  const bool twin = bs[0]->twin != 0;
  const LRing ring = lut_ring(bs, n, batch);
  const int bp = ring.bp;
  long long total = 0;
  // tiles of each matrix (with a strip list, a single matrix: its listed strips')
  auto n_tiles = [&](int i) -> long long {
    return strips ? (long long)n_strips * (bs[i]->cols / 256) : tiles_of(bs[i]->rows, bs[i]->cols);
  };
  for (int i = 0; i < n; ++i) total += n_tiles(i);
  if (total < 1) return LW_OK;
  if (total > (1ll << 30)) return fail(LW_ERR_SHAPE, "group too large");
  dev::LLaunch g{};
  g.n = n;
  g.stage_rows = ring.stage_rows;
  g.qp_off = ring.qp_off;
  g.mid_off = ring.mid_off;
  g.lb_off = ring.lb_off;
  g.x_off = ring.x_off;
  g.xb_off = ring.xb_off;
  g.vi_off = ring.vi_off;
  g.stage_bytes = ring.stage_bytes;
  g.ring_off = ring.ring_off;
  g.lut_cap = ring.lut_cap;
  const int lut_bytes = ring.lut_bytes;
  const int S = ring.S;
  if (S < 2 * dev::kLProducers)
    return fail(LW_ERR_UNSUPPORTED, "tiles of %d rows do not fit the table-driven kernel",
                ring.stage_rows - 2);
  g.nstage = S;
  g.lut_off = g.ring_off + S * g.stage_bytes;
  g.wait_cycles = dev::kWaitCycles;
  g.stall_tile = -1;
  // testing (lw_test_stall_next): one launch whose first stage of CTA 0 is
  // never filled, and every wait of it limited to the requested time (SM
  // cycles at most 2.1 GHz)
  const int stall_us = take_test_stall();
  if (stall_us > 0) {
    g.wait_cycles = 2100LL * stall_us;
    g.stall_tile = 0;
  }
  const size_t smem = (size_t)g.lut_off + (size_t)lut_bytes;
  // CTAs: one per SM but one, shared among the matrices in proportion to
  // their tiles.  A CTA fills its SM's shared memory, so the next launch's
  // CTAs can only enter SMs this launch leaves; with one SM always spare, the
  // next launch's last CTA enters when this launch's second-to-last CTA
  // exits, and every CTA has its prologue (decode table, first copies) done
  // when the dependency wait returns.  With every SM in use, the CTA that
  // enters last began its prologue only then, and it set the call's end.
  const int sms = device_sm_count();
  const int G = sms > 1 ? sms - 1 : 1;
  int left = G;
  int max_per_cta = 1;
  g.cfirst[0] = 0;
  for (int i = 0; i < n; ++i) {
    const long long t = n_tiles(i);
    int c;
    if (i == n - 1) {
      c = left;
    } else {
      c = (int)((t * G + total / 2) / total);
      const int reserve = n - 1 - i;   // at least one CTA for each later matrix
      if (c > left - reserve) c = left - reserve;
    }
    if (c < 1) c = 1;
    if (c > t) c = (int)t;   // no idle CTAs beyond one per tile
    left -= c;
    g.cfirst[i + 1] = g.cfirst[i] + c;
    const int per = (int)((t + c - 1) / c);
    max_per_cta = per > max_per_cta ? per : max_per_cta;
  }
  const int grid = g.cfirst[n];
  // rows per unit: a whole tile per warp (R = 2: two interleaved streams per
  // lane sharing the activation loads) when a CTA has tiles for more than a
  // wave of 16 warps; half a tile per warp (R = 1: twice the warps, better
  // latency hiding and balance) for CTAs with fewer tiles
  const int R = max_per_cta > 16 || fmt == LW_FMT_BF16_EXP ? 2 : 1;
  LKernel k = fmt == LW_FMT_BF16_EXP ? pick_lut_b16(bp)
              : fmt == LW_FMT_Q4_PAIR
                  ? (twin ? pick_lut<dev::kQ4, true>(bp, R) : pick_lut<dev::kQ4, false>(bp, R))
                  : (twin ? pick_lut<dev::kQ6, true>(bp, R) : pick_lut<dev::kQ6, false>(bp, R));
  // consumer warps: at most 16 (R = 2) or kLMaxConsumers (R = 1), and
  // (2 / R) x four fewer than stages (copies in flight while every warp
  // decodes), spread so that a CTA's units come in whole waves, and at
  // least 8 (they build the decode table)
  int nw_max = (2 / R) * (S - 4);
  const int cap = fmt == LW_FMT_BF16_EXP ? dev::kLMaxConsumersB16
                  : (R == 2 ? dev::kLMaxConsumersR<2> : dev::kLMaxConsumersR<1>);
  if (nw_max > cap) nw_max = cap;
  const int units = (2 / R) * max_per_cta;
  const int waves = (units + nw_max - 1) / nw_max;
  int nw = (units + waves - 1) / waves;
  if (nw < 8) nw = 8 < nw_max ? 8 : nw_max;
  for (int i = 0; i < n; ++i) {
    const lw_dev_bundle* b = bs[i];
    dev::QArgs& a = g.m[i];
    a.words = b->words;
    a.tile_off = b->tile_off;
    a.lane_bits = b->lane_bits;
    a.lane_mid = twin ? nullptr : b->lane_mid;
    a.table = b->table;
    a.qparams = static_cast<const uint8_t*>(b->qparams);
    a.strips = strips;
    a.x = x[i];
    a.ws = workspace_partials(b, ws[i]);
    a.counters = workspace_counters(b, ws[i]);
    a.y = y[i];
    a.status = status;
    a.TK = (int)(b->cols / 256);
    a.N = (int)b->rows;
    a.K = (int)b->cols;
    a.n_tiles = (int)n_tiles(i);
    a.batch = batch;
    if (fmt == LW_FMT_BF16_EXP) {
      a.signman = b->signman;
      a.vflags = b->vflags;
      a.vrow_off = b->vrow_off;
      a.vexp = b->vexp;
      a.GW = (int)((b->cols / 64 + 31) / 32);
    }
  }
  const int threads = (nw + dev::kLProducers) * 32;
  if (resident_blocks((const void*)k, threads, smem) < 1)
    return fail(LW_ERR_UNSUPPORTED, "table-driven kernel does not fit on an SM (%zu bytes)", smem);
  launch_pdl(k, grid, threads, smem, st, g);
  return check_launch("table-driven product kernel");
}

std::atomic<int> g_test_stall_us{0};
int take_test_stall() { return g_test_stall_us.exchange(0); }

}  // namespace lw

extern "C" lw_status lw_test_stall_next(int32_t wait_us) {
  if (wait_us < 0 || wait_us > 1000000)
    return lw::fail(LW_ERR_INVALID_ARG, "wait_us %d outside 0..1000000", (int)wait_us);
  lw::g_test_stall_us.store(wait_us);
  return LW_OK;
}
