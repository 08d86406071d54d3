// libflce host side: the launch plans (forward vocabulary splits, backward
// row blocks x vocabulary slabs with its cost model, the one-call row
// blocks) and the workspace layouts that follow from them.
#pragma once

#include <algorithm>
#include <cmath>
#include <cstdlib>

#include "host_common.cuh"
#include "options.cuh"

namespace {

using namespace flce;

struct FwdPlan {
  int m_tiles = 0, n_tiles = 0, k_blocks = 0, S = 1, tps = 1, units = 0, grid = 0, nblk = 0;
};

// Split the vocabulary tiles of every row tile (tm rows) into S contiguous
// ranges so that (row tiles x S) units fill the persistent workers in
// near-whole waves.
constexpr size_t kFwdPartialsCap = size_t(256) << 20;

// Rows per forward GEMM launch: one raster group of 16 row tiles (4,096 rows
// on SM pairs).  Measured on 16,384 x 4,096 x 151,936: 11.3 ms per forward
// in four such launches against 11.8 ms in one launch over all rows (whose
// DRAM reads of W are twice as high).  FLCE_OPT_FWD_BLOCK_ROWS overrides it
// (rounded up to a tile; 0: all rows in one launch).
long long fwd_block_rows(long long N, int tm) {
  N = std::max(1LL, N);
  long long b = 16LL * tm;
  const int64_t o = opt(FLCE_OPT_FWD_BLOCK_ROWS);
  if (o == 0) return N;
  if (o > 0) b = o;
  return std::min(N, round_up(b, tm));
}

FwdPlan plan_forward(long long N, long long H, long long V, int workers, int tm,
                     size_t partials_cap = kFwdPartialsCap, long long part_rows = 0) {
  FwdPlan f;
  f.m_tiles = static_cast<int>(ceil_div(N, tm));
  f.n_tiles = static_cast<int>(ceil_div(V, BN));
  f.k_blocks = static_cast<int>(ceil_div(H, BK));
  f.nblk = static_cast<int>(ceil_div(N, SMALL_THREADS));
  long long best = LLONG_MAX;
  // at most 256 splits, and split partials (8 bytes per row and split) of
  // at most partials_cap bytes
  // part_rows: rows the partials array holds (all rows of a blocked forward)
  const long long s_mem = std::max(
      1LL, static_cast<long long>(partials_cap) / (8 * std::max(1LL, part_rows > 0 ? part_rows : N)));
  const int smax = static_cast<int>(std::min<long long>(std::min(f.n_tiles, 256), s_mem));
  for (int s = 1; s <= smax; ++s) {
    const int tps = static_cast<int>(ceil_div(f.n_tiles, s));
    const int se = static_cast<int>(ceil_div(f.n_tiles, tps));
    const long long units = static_cast<long long>(f.m_tiles) * se;
    const long long cost = ceil_div(std::max(units, 1LL), workers) * tps;
    if (cost < best) {
      best = cost;
      f.S = se;
      f.tps = tps;
    }
  }
  // FLCE_OPT_FWD_SPLITS = s pins the number of vocabulary splits (tests
  // compare split counts; results must not depend on them beyond fp32
  // rounding)
  if (const int64_t fs = opt(FLCE_OPT_FWD_SPLITS); fs > 0) {
    const int want = std::max(1, std::min(std::min(static_cast<int>(fs), f.n_tiles), smax));
    f.tps = static_cast<int>(ceil_div(f.n_tiles, want));
    f.S = static_cast<int>(ceil_div(f.n_tiles, f.tps));
  }
  f.units = f.m_tiles * f.S;
  f.grid = std::min(f.units, workers);
  return f;
}

// The plan of one cross-entropy forward call: splits chosen for a launch of
// fwd_block_rows rows, partials and block sums for all N rows.
FwdPlan plan_forward_call(long long N, long long H, long long V, int workers, int tm,
                          size_t partials_cap = kFwdPartialsCap) {
  FwdPlan f = plan_forward(fwd_block_rows(N, tm), H, V, workers, tm, partials_cap, N);
  f.nblk = static_cast<int>(ceil_div(std::max(1LL, N), SMALL_THREADS));
  return f;
}

// Backward tiling.  The dlogits buffer D holds R rows x ldD columns: the
// caller's chunk_rows x V bound (rows rounded up to 128).  D need not span the
// whole vocabulary: the backward walks blocks of R rows and, inside each, slabs
// of Vs vocabulary columns, so R can exceed chunk_rows while R x Vs stays inside
// the same bound.  dW is then read-modified-written once per row block instead
// of once per chunk_rows rows, and dH is summed over the slabs in fp32 partials
// (one per k-split) that are rounded to bf16 once per row block.
struct BwdPlan {
  long long R = 0;      // rows per block: the row capacity of D
  long long Vs = 0;     // vocabulary columns per slab (V when one slab)
  int n_slabs = 1;
  long long ldD = 0;    // row pitch of D in elements
  int dh_splits = 1;    // k-splits of the dH GEMM (fp32 partial sets)
  int dh_kb_per_split = 1;
  bool dh_f32 = false;  // dH through fp32 partials (several slabs or k-splits)
  double est_s = 0.0;   // modelled time of the backward GEMMs
  int buffers = 1;      // D buffers: 2 when the row blocks run pipelined (MODE_PIPE)
  bool dh_wide = false; // dH GEMM over 256 x 512 tiles (MODE_DH2; one slab, SM pairs)
};

// The dH GEMM of a one-slab plan with at least two waves of 256 x 256 tiles
// runs 256 x 512 tiles on SM pairs (default; FLCE_OPT_DH_WIDE = 0 keeps 256 x
// 256): its K walk (the whole vocabulary, over a few k-splits) leaves the
// non-overlapped epilogue small.  16,384 x 4,096 x 151,936: dH 11.7 -> 11.0
// ms per step; with fewer tiles (256 rows) it would only cut the parallelism.
bool dh_wide_for(int n_slabs, int tm, long long tiles, int workers) {
  return n_slabs == 1 && tm == 2 * BM && tiles >= 2LL * workers && opt_on(FLCE_OPT_DH_WIDE);
}

constexpr double kPlanFlops = 1.6e15;  // sustained bf16 tensor rate of the GPU (model)
constexpr double kPlanBytes = 6.0e12;  // sustained HBM bandwidth (model)
// per launch: prologue, last-wave imbalance, drain and the gap to the next
// (about 25 us measured inside a short launch; programmatic launch hides some)
constexpr double kPlanLaunch = 15e-6;
// share of the read-modify-write traffic of the fp32 outputs (dW, dH
// partials) that the MMAs do not hide: measured at the 2,816-row slab shape,
// the dW output added its full DRAM time
constexpr double kPlanRmwExposed = 0.7;

// Best dH k-split count for `tiles` output tiles and `kb` K blocks: the
// fewest splits whose last wave is at least 90% full (splits keep >= 8 K
// blocks each).  FLCE_OPT_DH_SPLITS overrides it.
int dh_split_count(long long tiles, long long kb, int workers) {
  if (const long long s = opt(FLCE_OPT_DH_SPLITS); s >= 1)
    return static_cast<int>(std::min<long long>({s, 16, std::max(1LL, kb / 8)}));
  int best_s = 1;
  double best_eff = -1.0;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && kb / s < 8) break;
    const double waves = static_cast<double>(tiles * s) / workers;
    const double eff = waves / std::ceil(waves);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best_s = s;
    }
    if (eff >= 0.9) break;
  }
  return best_s;
}

// Completes plan b for row block size R (D budget in elements): slab width,
// dH splits, memory check and modelled time.  False when R does not fit.
// pipelined: the row block runs as one launch (MODE_PIPE), so its slabs pay
// no launch cost of their own.
bool plan_candidate(BwdPlan& b, long long N, long long H, long long V, long long R,
                    long long budget, int workers, int tm, bool pipelined = false) {
  const long long ldV = round_up(V, 8);
  b.R = R;
  if (R * ldV <= budget) {
    b.n_slabs = 1;
    b.Vs = V;
    b.ldD = ldV;
  } else {
    const long long vs_max = (budget / R) / BN * BN;
    if (vs_max < BN) return false;
    b.n_slabs = static_cast<int>(ceil_div(V, vs_max));
    b.Vs = round_up(ceil_div(V, b.n_slabs), BN);
    b.ldD = b.Vs;
  }
  b.dh_wide = dh_wide_for(b.n_slabs, tm, ceil_div(R, tm) * ceil_div(H, BN), workers);
  const long long dh_tiles = ceil_div(R, tm) * ceil_div(H, b.dh_wide ? 2 * BN : BN);
  const long long kb = ceil_div(b.Vs, BK);
  int s = dh_split_count(dh_tiles, kb, workers);
  b.dh_kb_per_split = static_cast<int>(ceil_div(kb, s));
  s = static_cast<int>(ceil_div(kb, b.dh_kb_per_split));
  // dH partials and the gathered rows stay within the size of D
  auto aux = [&](int splits, bool f32) {
    return (f32 ? static_cast<double>(splits) * R * H * 4 : 0.0) + static_cast<double>(R) * H * 2;
  };
  // (a pipelined plan's budget is one of two buffers: the bound is the whole)
  const double aux_cap = 2.0 * budget * (pipelined ? 2 : 1);
  while (s > 1 && aux(s, true) > aux_cap) {
    --s;
    b.dh_kb_per_split = static_cast<int>(ceil_div(kb, s));
    s = static_cast<int>(ceil_div(kb, b.dh_kb_per_split));
  }
  b.dh_splits = s;
  b.dh_f32 = b.n_slabs > 1 || s > 1;
  if (b.n_slabs > 1 && aux(s, b.dh_f32) > aux_cap) return false;

  // modelled time: per launch max(tensor time, HBM operand time) + the
  // exposed share of the fp32 output traffic + launch cost
  const double t_kb = 2.0 * tm * BN * BK * workers / kPlanFlops;  // one tile x one 64-deep K block
  auto waves = [&](long long u) { return static_cast<double>(ceil_div(u, workers)); };
  auto slab_cost = [&](long long rows, long long w, bool first_block, bool first_slab) {
    const long long mt = ceil_div(rows, tm);
    const double d_bytes = 2.0 * rows * w;
    double t = 0.0;
    // dlogits: W slab read once per 16 row tiles
    t += std::max(waves(mt * ceil_div(w, BN)) * ceil_div(H, BK) * t_kb,
                  (d_bytes + 2.0 * w * H * ceil_div(mt, 16) + 2.0 * rows * H) / kPlanBytes);
    // dH
    const long long kbw = ceil_div(w, BK);
    const long long sw = ceil_div(kbw, b.dh_kb_per_split);
    const double dh_out = b.dh_f32 ? 4.0 * rows * H * sw * (first_slab ? 1 : 2) : 2.0 * rows * H;
    t += std::max(waves(mt * ceil_div(H, BN) * sw) * b.dh_kb_per_split * t_kb,
                  (d_bytes + 2.0 * w * H) / kPlanBytes) +
         kPlanRmwExposed * dh_out / kPlanBytes;
    // dW: a store on the first row block, a read-modify-write afterwards
    const long long vt = ceil_div(w, tm);
    t += std::max(waves(vt * ceil_div(H, BN)) * ceil_div(rows, BK) * t_kb,
                  (d_bytes + 2.0 * rows * H * ceil_div(vt, 8)) / kPlanBytes) +
         kPlanRmwExposed * 4.0 * w * H * (first_block ? 1 : 2) / kPlanBytes;
    return t + (pipelined ? 0.0 : 3 * kPlanLaunch);
  };
  auto block_cost = [&](long long rows, bool first_block) {
    const long long w_last = V - (b.n_slabs - 1) * b.Vs;
    double t = slab_cost(rows, b.n_slabs == 1 ? V : b.Vs, first_block, true);
    if (b.n_slabs > 2) t += (b.n_slabs - 2) * slab_cost(rows, b.Vs, first_block, false);
    if (b.n_slabs > 1) t += slab_cost(rows, w_last, first_block, false);
    if (b.dh_f32) t += rows * H * (4.0 * b.dh_splits + 2.0) / kPlanBytes + kPlanLaunch;
    return t;
  };
  const long long nb = ceil_div(N, R);
  const long long rows_last = N - (nb - 1) * R;
  if (nb == 1)
    b.est_s = block_cost(rows_last, true);
  else
    b.est_s = block_cost(R, true) + (nb - 2) * block_cost(R, false) + block_cost(rows_last, false);
  return true;
}

// FLCE_OPT_BWD_ROWS = rows fixes the row block (clamped to the budget)
// instead of the modelled choice.
long long bwd_rows_forced() { return opt(FLCE_OPT_BWD_ROWS); }

// buffers = 2: the plan of one of two D buffers that share the budget (the
// pipelined row blocks); R = 0 when no row block fits.
BwdPlan plan_backward(long long N, long long H, long long V, long long chunk_rows, int workers,
                      int tm, int buffers = 1) {
  N = std::max(1LL, N);
  const long long nr = round_up(N, BM);
  const long long R0 = std::min(round_up(std::max(1LL, chunk_rows), BM), nr);
  const long long budget = R0 * round_up(V, 8) / buffers;
  workers = std::max(1, workers);
  // the last plan, reused while the sizes and the options it reads are the same
  struct Key {
    long long N, H, V, R0, forced, splits, wide;
    int workers, tm, buffers;
  };
  thread_local Key last{-1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
  thread_local BwdPlan last_plan;
  const long long forced = bwd_rows_forced();
  const long long splits_opt = opt(FLCE_OPT_DH_SPLITS), wide_opt = opt(FLCE_OPT_DH_WIDE);
  if (last.N == N && last.H == H && last.V == V && last.R0 == R0 && last.forced == forced &&
      last.splits == splits_opt && last.wide == wide_opt && last.workers == workers && last.tm == tm &&
      last.buffers == buffers)
    return last_plan;

  BwdPlan best;
  // the caller's chunk: always fits one buffer; half of it may not
  const bool piped = buffers == 2;
  if (!plan_candidate(best, N, H, V, R0, budget, workers, tm, piped)) best = BwdPlan{};
  if (forced > 0) {
    BwdPlan b;
    const long long R = std::min(nr, std::max(R0, round_up(forced, BM)));
    if (plan_candidate(b, N, H, V, R, budget, workers, tm, piped)) best = b;
  } else {
    // larger row blocks in steps of one tile; a plan with vocabulary slabs
    // must beat the single-slab chunk plan by 5 % (the model misses some of
    // the slabs' extra traffic: on 16,384 x 4,096 x 151,936 at 4,096-row
    // chunks, 8,192- and 16,384-row blocks measured no faster), and each
    // later candidate the best so far by 2 %
    const bool single = best.n_slabs == 1;
    for (long long R = round_up(R0 + 1, tm); R <= round_up(nr, tm); R += tm) {
      BwdPlan b;
      if (!plan_candidate(b, N, H, V, std::min(R, nr), budget, workers, tm, piped)) break;
      const double margin = (single && best.R == R0) ? 0.95 : 0.98;
      if (best.R == 0 || b.est_s < best.est_s * margin) best = b;
      if (R >= nr) break;
    }
  }
  last = Key{N, H, V, R0, forced, splits_opt, wide_opt, workers, tm, buffers};
  last_plan = best;
  return best;
}

// The plan a backward call runs.  With several vocabulary slabs, both
// gradients wanted and pipelining on (FLCE_OPT_PIPELINE, dlogits written
// through TMA), the row blocks run pipelined (MODE_PIPE) over two D buffers
// that together stay within the dlogits budget, so that slab s + 1's
// dlogits are formed while slab s's dH and dW run: the plan of half the
// budget.  Otherwise the plain plan.
BwdPlan plan_backward_call(long long N, long long H, long long V, long long chunk_rows, int workers, int tm,
                           bool both) {
  const BwdPlan b = plan_backward(N, H, V, chunk_rows, workers, tm);
  if (!both || b.n_slabs <= 1 || !opt_on(FLCE_OPT_PIPELINE) || !opt_on(FLCE_OPT_D_TMA)) return b;
  BwdPlan q = plan_backward(N, H, V, chunk_rows, workers, tm, 2);
  if (q.R == 0 || q.n_slabs <= 1 || !q.dh_f32) return b;
  q.buffers = 2;
  return q;
}

// Forward scratch.  fb_skip > 0 adds what a forward that skips the ignored
// rows needs: the non-ignored row indices and count, and a gathered [fb_skip,
// H] block of h rows per launch.
struct FwdLayout {
  size_t zt = 0, part = 0, bsum = 0, bcnt = 0, bad = 0, idx = 0, blk = 0, count = 0, hc = 0, total = 0;
};
FwdLayout fwd_layout(long long N, const FwdPlan& f, long long H = 0, long long fb_skip = 0) {
  FwdLayout L;
  size_t o = 0;
  L.zt = o;
  o += align256(static_cast<size_t>(N) * 4);
  L.part = o;
  o += align256(static_cast<size_t>(f.S) * N * 8);
  L.bsum = o;
  o += align256(static_cast<size_t>(f.nblk) * 8);
  L.bcnt = o;
  o += align256(static_cast<size_t>(f.nblk) * 8);
  L.bad = o;
  o += 256;
  if (fb_skip > 0) {
    L.idx = o;
    o += align256(static_cast<size_t>(N) * 4);
    L.blk = o;
    o += align256(static_cast<size_t>(ceil_div(std::max(1LL, N), COMPACT_ROWS_PER_BLOCK)) * 4);
    L.count = o;
    o += 256;
    L.hc = o;
    o += align256(static_cast<size_t>(fb_skip) * H * 2);
  }
  L.total = o;
  return L;
}

// Distillation forward scratch: student and teacher split partials, the
// cross term, block sums.
struct KdFwdLayout {
  size_t ps = 0, pt = 0, pc = 0, bsum = 0, bcnt = 0, total = 0;
};
KdFwdLayout kd_fwd_layout(long long N, const FwdPlan& f) {
  KdFwdLayout L;
  size_t o = 0;
  L.ps = o;
  o += align256(static_cast<size_t>(f.S) * N * 8);
  L.pt = o;
  o += align256(static_cast<size_t>(f.S) * N * 8);
  L.pc = o;
  o += align256(static_cast<size_t>(f.S) * N * 4);
  L.bsum = o;
  o += align256(static_cast<size_t>(f.nblk) * 8);
  L.bcnt = o;
  o += align256(static_cast<size_t>(f.nblk) * 8);
  L.total = o;
  return L;
}

// Jensen-Shannon forward scratch: the distillation forward's (pass 1, both
// heads' log-sum-exp) plus the mixture-term partials of pass 2 and the two lse
// vectors when the caller does not ask for them.  The mixture-term partials
// hold kJsdColParts slots per vocabulary split: with 8 epilogue warps, each
// half of a tile's columns writes its own.
// With fb_skip > 0, also what a forward that skips the ignored rows needs:
// the non-ignored row indices and count, and one launch's gathered rows of
// both heads ([fb_skip, H_s] and [fb_skip, H_t] bf16).
constexpr int kJsdColParts = 2;
struct JsdFwdLayout {
  KdFwdLayout kd;
  size_t pj = 0, lse_s = 0, lse_t = 0, idx = 0, blk = 0, count = 0, hs = 0, ht = 0, total = 0;
};
JsdFwdLayout jsd_fwd_layout(long long N, const FwdPlan& f, long long H_s = 0, long long H_t = 0,
                            long long fb_skip = 0) {
  JsdFwdLayout L;
  L.kd = kd_fwd_layout(N, f);
  size_t o = L.kd.total;
  L.pj = o;
  o += align256(static_cast<size_t>(f.S) * kJsdColParts * N * 8);
  L.lse_s = o;
  o += align256(static_cast<size_t>(N) * 4);
  L.lse_t = o;
  o += align256(static_cast<size_t>(N) * 4);
  if (fb_skip > 0) {
    L.idx = o;
    o += align256(static_cast<size_t>(N) * 4);
    L.blk = o;
    o += align256(static_cast<size_t>(ceil_div(std::max(1LL, N), COMPACT_ROWS_PER_BLOCK)) * 4);
    L.count = o;
    o += 256;
    L.hs = o;
    o += align256(static_cast<size_t>(fb_skip) * H_s * 2);
    L.ht = o;
    o += align256(static_cast<size_t>(fb_skip) * H_t * 2);
  }
  L.total = o;
  return L;
}

// Dependency counters of one pipelined row-block launch (MODE_PIPE): per
// slab, two per row tile (at most R / 128 of them) and two per BN-wide
// vocabulary tile of the slab; the last word counts the units drawn.
long long pipe_dep_words(const BwdPlan& b) {
  return 2LL * b.n_slabs * (ceil_div(b.R, BM) + ceil_div(b.Vs, BN)) + 1;
}

// dW over at most this many K blocks (64 rows each) runs 8 epilogue warps:
// at 256 rows (4 blocks) its output epilogue, not the MMAs, set the pace
// (8 warps: 410 us against 443 us for the 248,320 x 2,048 fp32 gradient); at
// 4,096 rows 4 warps were 1-2 % faster
constexpr int kDwWideEpilogueMaxKBlocks = 16;

// Pipelined row blocks: how many units an SM pair may hold drawn but not
// finished.  Two keep the next unit's loads behind the current unit's MMAs;
// on the 131,072 x 2,560 x 151,936 step (256-row chunks) three took as long
// and six 6 % longer (the drawn units run further ahead of the finished
// ones); on 8,192 rows of the same shape one took 30 % longer.
constexpr int kPipeLookahead = 2;

// Row tiles per dH raster group: 8 (FLCE_OPT_DH_GROUP overrides).  A wave of 76
// units then covers 8 row tiles x ~9.5 column tiles, the fewest D and W
// slices per wave.  On 16,384 x 4,096 x 151,936, interleaved runs timed the
// step 1.3% faster than with all 16 row tiles (the dH launch itself took the
// same time); a dH launch's DRAM bytes vary more between GPUs than between
// the two groups.
int dh_group_rows(int m_tiles) {
  const int64_t g = opt(FLCE_OPT_DH_GROUP);
  return g > 0 ? static_cast<int>(std::min<int64_t>(g, m_tiles)) : m_tiles;
}

// dW raster: one vocabulary tile's column tiles after one another, so that a
// wave covers few D slices, each read once.  16,384 x 4,096 x 151,936: a dW
// launch read 2.25 / 4.34 GB (store / reduce-add) from DRAM against 3.67 /
// 5.75 GB with groups of 8 vocabulary tiles and 4.2 / 6.3 GB with 16, in the
// same time.  At short K the launch is bound by its fp32 write stream, which
// groups of 8 vocabulary tiles write faster: 256 x 2,048 x 248,320 took 381
// against 407 us with groups of 1.
int dw_group(int k_blocks, int m_tiles) {
  return k_blocks <= kDwWideEpilogueMaxKBlocks ? std::min(8, std::max(1, m_tiles)) : 1;
}

// Parameters of the pipelined launch (MODE_PIPE) of one row block: base
// carries the call's fields (V, rows_cap, the row count or the compaction's
// device-side count); rows is the block's row capacity (compacted) or its
// rows, block its index (block 0 stores dW, later blocks add to it).
GemmParams pipe_params(const BwdPlan& b, const GemmParams& base, long long H, int tm, int rows, int block) {
  GemmParams q = base;
  q.m_tiles = static_cast<int>(ceil_div(rows, tm));  // row tiles at most (compacted: fewer)
  q.n_tiles = static_cast<int>(ceil_div(H, BN));
  q.cols = q.n_tiles;
  q.n_per_unit = 1;
  q.pp_slabs = b.n_slabs;
  q.pp_vs = static_cast<int>(b.Vs);
  q.pp_kh = static_cast<int>(ceil_div(H, BK));
  q.pp_dh_kbps = b.dh_kb_per_split;
  q.pp_dl_group = std::min(16, q.m_tiles);
  q.group_m = dh_group_rows(q.m_tiles);
  q.dw_k_blocks = static_cast<int>(ceil_div(rows, BK));
  q.dw_group_m = dw_group(q.dw_k_blocks, static_cast<int>(ceil_div(b.Vs, tm)));
  q.dW_accumulate = block > 0 ? 1 : 0;
  q.pp_dep_words = static_cast<int>(pipe_dep_words(b));
  q.pp_lookahead = kPipeLookahead;
  return q;
}

struct BwdLayout {
  size_t D = 0, dh_part = 0, bad = 0, idx = 0, blk = 0, count = 0, hc = 0, dep = 0, total = 0;
};
// dlogits block, dH fp32 partials, validation counter, the row compaction
// buffers (valid-row indices, per-block counts, their total, the gathered h
// rows of one chunk), and for a pipelined plan two sets of dependency
// counters (used by alternate row blocks).
BwdLayout bwd_layout(long long N, long long H, const BwdPlan& b) {
  BwdLayout L;
  size_t o = 0;
  L.D = o;
  o += align256(static_cast<size_t>(b.buffers) * b.R * b.ldD * 2);
  L.dh_part = o;
  if (b.dh_f32) o += align256(static_cast<size_t>(b.dh_splits) * b.R * H * 4);
  L.bad = o;
  o += 256;
  L.idx = o;
  o += align256(static_cast<size_t>(N) * 4);
  L.blk = o;
  o += align256(static_cast<size_t>(ceil_div(N, COMPACT_ROWS_PER_BLOCK)) * 4);
  L.count = o;
  o += 256;
  L.hc = o;
  o += align256(static_cast<size_t>(b.R) * H * 2);
  L.dep = o;
  if (b.buffers == 2) o += align256(static_cast<size_t>(2 * pipe_dep_words(b)) * 4);
  L.total = o;
  return L;
}

// Workspace a backward call may need for these sizes: the larger of the
// plain plan's and the pipelined plan's (the call takes one of them).
size_t bwd_workspace(long long N, long long H, long long V, long long chunk_rows, int workers, int tm) {
  return std::max(bwd_layout(N, H, plan_backward(N, H, V, chunk_rows, workers, tm)).total,
                  bwd_layout(N, H, plan_backward_call(N, H, V, chunk_rows, workers, tm, true)).total);
}

// The distillation backward: the backward's buffers (student width) and one
// chunk's gathered teacher rows for the row compaction.
struct DistillBwdLayout {
  BwdLayout b;
  size_t hc_t = 0, total = 0;
};
DistillBwdLayout distill_bwd_layout(long long N, long long H_s, long long H_t, const BwdPlan& b) {
  DistillBwdLayout L;
  L.b = bwd_layout(N, H_s, b);
  L.hc_t = L.b.total;
  L.total = L.hc_t + align256(static_cast<size_t>(b.R) * H_t * 2);
  return L;
}

// ---- forward + backward in one call without the logits recompute

// Row blocks of R rows over the whole vocabulary: the forward GEMM keeps the
// block's exponentials (bf16, R x ldD, within the dlogits budget) and chunk
// maxima (fp32, R x ldD / 32), so the backward needs no second logits GEMM.  Taken
// when the budget holds at least 2,048 rows (or every row) of the full
// vocabulary; otherwise the call runs the forward and the tiled backward.
struct FusedPlan {
  bool fused = false;
  long long R = 0, ldD = 0;
  FwdPlan f;
  BwdPlan b;  // dH / dW stages over one slab of V columns
};

FusedPlan plan_fused(long long N, long long H, long long V, long long chunk_rows, int workers, int tm) {
  FusedPlan fp;
  N = std::max(1LL, N);
  const long long nr = round_up(N, BM);
  // the block is the caller's chunk (rounded up to 128 rows): exponentials in
  // its dlogits budget, the chunk maxima (1/16 of it) on top
  // (at most 32,768 rows: the dlogits pass puts one row per grid row)
  fp.R = std::min(std::min(round_up(std::max(1LL, chunk_rows), BM), nr), 32768LL);
  fp.ldD = round_up(V, 32);
  fp.fused = fp.R >= std::min<long long>(2048, nr);
  if (!fp.fused) return fp;
  fp.f = plan_forward(fp.R, H, V, workers, tm, kFwdPartialsCap, N);
  fp.b.R = fp.R;
  fp.b.Vs = V;
  fp.b.n_slabs = 1;
  fp.b.ldD = fp.ldD;
  const long long kb = ceil_div(V, BK);
  fp.b.dh_wide = dh_wide_for(1, tm, ceil_div(fp.R, tm) * ceil_div(H, BN), workers);
  int sp = dh_split_count(ceil_div(fp.R, tm) * ceil_div(H, fp.b.dh_wide ? 2 * BN : BN), kb, workers);
  fp.b.dh_kb_per_split = static_cast<int>(ceil_div(kb, sp));
  fp.b.dh_splits = static_cast<int>(ceil_div(kb, fp.b.dh_kb_per_split));
  fp.b.dh_f32 = fp.b.dh_splits > 1;
  return fp;
}

struct FusedLayout {
  size_t zt = 0, part = 0, bsum = 0, bcnt = 0, bad = 0, E = 0, mx = 0, lse = 0, dh_part = 0, idx = 0,
         blk = 0, count = 0, hc = 0, lp = 0, wg = 0, total = 0;
};
FusedLayout fused_layout(long long N, long long H, const FusedPlan& fp) {
  FusedLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  L.zt = take(static_cast<size_t>(N) * 4);
  L.part = take(static_cast<size_t>(fp.f.S) * N * 8);
  // loss block sums: one segment of ceil(R / 256) per row block
  const size_t nblk = static_cast<size_t>(ceil_div(std::max(1LL, N), fp.R) * ceil_div(fp.R, SMALL_THREADS));
  L.bsum = take(nblk * 8);
  L.bcnt = take(nblk * 8);
  L.bad = take(256);
  L.E = take(static_cast<size_t>(fp.R) * fp.ldD * 2);
  L.mx = take(static_cast<size_t>(fp.R) * (fp.ldD / 32) * 4);
  L.lse = take(static_cast<size_t>(N) * 4);
  L.dh_part = take(fp.b.dh_f32 ? static_cast<size_t>(fp.b.dh_splits) * fp.R * H * 4 : 0);
  L.idx = take(static_cast<size_t>(N) * 4);
  L.blk = take(static_cast<size_t>(ceil_div(std::max(1LL, N), COMPACT_ROWS_PER_BLOCK)) * 4);
  L.count = take(256);
  L.hc = take(static_cast<size_t>(fp.R) * H * 2);  // the block's rows of h (row compaction)
  L.lp = take(static_cast<size_t>(N) * 4);          // GRPO: log-probs and backward weights
  L.wg = take(static_cast<size_t>(N) * 4);
  L.total = o;
  return L;
}

}  // namespace
