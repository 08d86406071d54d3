// Host-side check of the pipelined backward's unit schedule (MODE_PIPE).
//
// A pipelined row block runs as one launch whose SM pairs draw unit indices
// from a counter in increasing order; a unit waits until some dependency
// counters reach their targets.  The launch finishes, whichever of its pairs
// are resident, when every unit that adds to a counter a unit waits on comes
// earlier in the order; and the unit reads complete data when each target
// equals the number of units that add to that counter.  This program decodes
// every unit of many launches with the library's own decoding and counter
// helpers (compiled for the host) and checks, per launch:
//   - every counter a unit waits on or adds to lies inside the launch's
//     counter words (the last word, the draw counter, excluded);
//   - every wait's target equals the number of units that add to its counter,
//     and all of those units come before the waiting unit;
//   - each slab's dlogits, dH and dW units are decoded exactly once, within
//     their tile ranges, and the launch's unit count is their sum;
//   - independently of how the counters are laid out, from the data each
//     unit touches: a dH or dW unit waits for every dlogits unit of its slab
//     that wrote a tile of the dlogits it reads; a dlogits unit of slab s
//     waits for every dH and dW unit of slab s - 2 that read a tile it
//     overwrites (the same buffer); a dH unit waits for the dH unit of the
//     previous slab that added to the same fp32 partial tile -- each such
//     unit earlier in the order and adding to a counter the waiting unit
//     waits on.
// The launches are those the planner makes for the library's workloads (with
// and without row compaction, both CTA-group tile heights) and a seeded sweep
// of plans.  For the planner's plans it checks the backward's workspace: the
// regions (dlogits buffers, dH partials, compaction buffers, dependency
// counters) 256-byte aligned and disjoint, inside the size the library
// reports, the dlogits inside the O(chunk_rows x V) budget, and room in the
// dH partials for every k-split a slab's units write; and the forward's
// vocabulary splits and workspace.  It also checks that
// the raster decoding every GEMM launch uses
// (decode_grid) maps its unit indices one to one onto (k-split, row tile,
// column unit), over a sweep of grid shapes and raster groups.  Exit status
// 0 and "ok" when every check passes.
#include <cstdint>
#include <cstdio>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "plan.cuh"

namespace {

int g_fails = 0;
long long g_launches = 0, g_units = 0;

#define EXPECT(cond, ...)                      \
  do {                                         \
    if (!(cond)) {                             \
      if (g_fails++ < 20) {                    \
        std::fprintf(stderr, "FAIL: ");        \
        std::fprintf(stderr, __VA_ARGS__);     \
        std::fprintf(stderr, "\n");            \
      }                                        \
    }                                          \
  } while (0)

uint64_t unit_key(int kind, int slab, int m, int n, int kb0) {
  return (static_cast<uint64_t>(kind) << 60) | (static_cast<uint64_t>(slab) << 44) |
         (static_cast<uint64_t>(m) << 28) | (static_cast<uint64_t>(n) << 16) | static_cast<uint64_t>(kb0);
}

// Unit `later` must not start before unit `earlier` has finished (a data
// hazard between them): `earlier` comes first in the order and adds to a
// counter that `later` waits on (whose target counts all its adders).
template <int TM>
void expect_ordered(const GemmParams& q, const DynShape& d, const std::vector<Unit>& units, int earlier, int later,
                    const char* why, const char* what) {
  EXPECT(earlier < later, "%s: unit %d must follow unit %d (%s) but comes first", what, later, earlier, why);
  PipeWait w[2];
  const int nw = pipe_unit_waits<TM, 1>(q, d, units[later], w);
  int idx[2];
  const int ns = pipe_unit_signals<TM>(q, units[earlier], idx);
  bool covered = false;
  for (int i = 0; i < nw; ++i)
    for (int j = 0; j < ns; ++j) covered = covered || (w[i].idx == idx[j] && w[i].target > 0);
  EXPECT(covered, "%s: unit %d (kind %d, slab %d) does not wait for unit %d (kind %d, slab %d): %s", what, later,
         units[later].kind, units[later].slab, earlier, units[earlier].kind, units[earlier].slab, why);
}

// The hazards on the two dlogits buffers (slab s in buffer s % 2) and on the
// fp32 dH partials, enumerated from the tiles each unit reads or writes:
//   dlogits unit (s, m, vt): writes rows of row tile m, columns [vt*BN, +BN)
//     of slab s's buffer;
//   dH unit (s, m, ht, K blocks kb0..kb1): reads rows of row tile m, columns
//     [kb0*BK, kb1*BK) of that buffer; adds to partial tile (split, m, ht);
//   dW unit (s, dvt, ht): reads every row, columns [dvt*TM, +TM).
template <int TM>
void check_hazards(const GemmParams& q, const DynShape& d, const std::vector<Unit>& units, const char* what) {
  std::unordered_map<uint64_t, int> at;
  at.reserve(units.size() * 2);
  for (int u = 0; u < static_cast<int>(units.size()); ++u) {
    const Unit& t = units[u];
    at[unit_key(t.kind, t.slab, t.m, t.n0, t.kb0)] = u;
  }
  auto find = [&](int kind, int slab, int m, int n, int kb0) -> int {
    const auto it = at.find(unit_key(kind, slab, m, n, kb0));
    return it == at.end() ? -1 : it->second;
  };
  for (int u = 0; u < static_cast<int>(units.size()); ++u) {
    const Unit& t = units[u];
    const PipeSlab ps = pipe_slab<TM>(q, d, t.slab);
    if (t.kind == KIND_DH) {
      // read after write: the dlogits tiles of its row tile that its K range covers
      const int c0 = t.kb0 * BK, c1 = std::min(t.kb1 * BK, ps.width);
      for (int vt = c0 / BN; vt * BN < c1; ++vt) {
        const int w = find(KIND_DL, t.slab, t.m, vt, 0);
        EXPECT(w >= 0, "%s: no dlogits unit (slab %d, %d, %d) for dH unit %d", what, t.slab, t.m, vt, u);
        if (w >= 0) expect_ordered<TM>(q, d, units, w, u, "dH reads the dlogits it wrote", what);
      }
      // the fp32 partial tile: the previous slab's unit of the same tile and split
      if (t.slab > 0) {
        const PipeSlab pp = pipe_slab<TM>(q, d, t.slab - 1);
        if (t.split < pp.splits) {
          const int w = find(KIND_DH, t.slab - 1, t.m, t.n0, t.split * q.pp_dh_kbps);
          EXPECT(w >= 0, "%s: no dH unit of slab %d for partial tile (%d, %d, %d)", what, t.slab - 1, t.split,
                 t.m, t.n0);
          if (w >= 0) expect_ordered<TM>(q, d, units, w, u, "dH adds to the partial the previous slab left", what);
        }
      }
    } else if (t.kind == KIND_DW) {
      // read after write: the dlogits tile (every row tile) holding its columns
      const int vt = t.m * TM / BN;
      for (int m = 0; m < d.m_tiles; ++m) {
        const int w = find(KIND_DL, t.slab, m, vt, 0);
        EXPECT(w >= 0, "%s: no dlogits unit (slab %d, %d, %d) for dW unit %d", what, t.slab, m, vt, u);
        if (w >= 0) expect_ordered<TM>(q, d, units, w, u, "dW reads the dlogits it wrote", what);
      }
    } else if (t.slab >= 2) {
      // write after read: slab s - 2's readers of this tile of the same buffer
      const PipeSlab po = pipe_slab<TM>(q, d, t.slab - 2);
      const int c0 = t.n0 * BN, c1 = std::min(c0 + BN, po.width);
      for (int split = 0; split < po.splits; ++split) {
        const int k0 = split * q.pp_dh_kbps * BK, k1 = std::min((split + 1) * q.pp_dh_kbps * BK, po.width);
        if (k1 <= c0 || k0 >= c1) continue;
        for (int ht = 0; ht < q.n_tiles; ++ht) {
          const int r = find(KIND_DH, t.slab - 2, t.m, ht, split * q.pp_dh_kbps);
          EXPECT(r >= 0, "%s: no dH unit (slab %d, %d, %d, split %d)", what, t.slab - 2, t.m, ht, split);
          if (r >= 0) expect_ordered<TM>(q, d, units, r, u, "dlogits overwrites what dH read", what);
        }
      }
      if (po.n_dw > 0)
        for (int dvt = c0 / TM; dvt * TM < c1 && dvt < po.dwt; ++dvt)
          for (int ht = 0; ht < q.n_tiles; ++ht) {
            const int r = find(KIND_DW, t.slab - 2, dvt, ht, 0);
            EXPECT(r >= 0, "%s: no dW unit (slab %d, %d, %d)", what, t.slab - 2, dvt, ht);
            if (r >= 0) expect_ordered<TM>(q, d, units, r, u, "dlogits overwrites what dW read", what);
          }
    }
  }
}

template <int TM>
void check_launch(const GemmParams& q, const char* what) {
  const DynShape d = dyn_shape<MODE_PIPE, TM>(q);
  const int words = q.pp_dep_words - 1;  // the last word counts the units drawn
  const int S = q.pp_slabs;
  std::vector<Unit> units(d.num_units > 0 ? d.num_units : 0);
  std::vector<long long> total(words, 0), seen(words, 0);
  for (int u = 0; u < d.num_units; ++u) {
    units[u] = decode_unit<MODE_PIPE, TM>(q, d, u);
    int idx[2];
    const int n = pipe_unit_signals<TM>(q, units[u], idx);
    for (int i = 0; i < n; ++i) {
      EXPECT(idx[i] >= 0 && idx[i] < words, "%s: unit %d adds to counter %d of %d", what, u, idx[i], words);
      if (idx[i] >= 0 && idx[i] < words) ++total[idx[i]];
    }
  }
  for (int u = 0; u < d.num_units; ++u) {
    PipeWait w[2];
    const int n = pipe_unit_waits<TM, 1>(q, d, units[u], w);
    for (int i = 0; i < n; ++i) {
      const int c = w[i].idx;
      EXPECT(c >= 0 && c < words, "%s: unit %d waits on counter %d of %d", what, u, c, words);
      if (c < 0 || c >= words) continue;
      EXPECT(w[i].target == total[c], "%s: unit %d (kind %d, slab %d) waits for %u arrivals on counter %d, which %lld units add to",
             what, u, units[u].kind, units[u].slab, w[i].target, c, total[c]);
      EXPECT(seen[c] >= static_cast<long long>(w[i].target),
             "%s: unit %d (kind %d, slab %d) waits on counter %d, of whose %u arrivals only %lld come from earlier units",
             what, u, units[u].kind, units[u].slab, c, w[i].target, seen[c]);
    }
    int idx[2];
    const int m = pipe_unit_signals<TM>(q, units[u], idx);
    for (int i = 0; i < m; ++i)
      if (idx[i] >= 0 && idx[i] < words) ++seen[idx[i]];
  }
  // every unit of every slab and kind exactly once
  std::set<std::tuple<int, int, int, int, int>> keys;
  std::vector<long long> count(3 * (S + 1), 0);
  for (int u = 0; u < d.num_units; ++u) {
    const Unit& t = units[u];
    EXPECT(t.slab >= 0 && t.slab < S, "%s: unit %d in slab %d of %d", what, u, t.slab, S);
    if (t.slab < 0 || t.slab >= S) continue;
    const PipeSlab ps = pipe_slab<TM>(q, d, t.slab);
    const int m_hi = t.kind == KIND_DW ? ps.dwt : d.m_tiles;
    const int n_hi = t.kind == KIND_DL ? ps.vt : q.n_tiles;
    const int k_hi = t.kind == KIND_DL ? q.pp_kh : t.kind == KIND_DH ? ps.kb : d.dw_k_blocks;
    EXPECT(t.m >= 0 && t.m < m_hi && t.n0 >= 0 && t.n0 < n_hi && t.n1 == t.n0 + 1,
           "%s: unit %d (kind %d) tile (%d, %d..%d) outside (%d, %d)", what, u, t.kind, t.m, t.n0, t.n1, m_hi, n_hi);
    // an empty K range only for the dW units of a block without rows (their
    // epilogue writes the zero product)
    const bool k_ok = t.kb0 >= 0 && t.kb1 <= k_hi &&
                      (t.kb0 < t.kb1 || (t.kind == KIND_DW && k_hi == 0 && t.kb0 == 0 && t.kb1 == 0));
    EXPECT(k_ok, "%s: unit %d (kind %d) K blocks %d..%d of %d", what, u, t.kind, t.kb0, t.kb1, k_hi);
    EXPECT(keys.insert(std::make_tuple(t.kind, t.slab, t.m, t.n0, t.kb0)).second, "%s: unit %d decoded twice",
           what, u);
    ++count[3 * t.slab + t.kind];
  }
  long long sum = 0;
  for (int s = 0; s < S; ++s) {
    const PipeSlab ps = pipe_slab<TM>(q, d, s);
    EXPECT(count[3 * s + KIND_DL] == ps.n_dl && count[3 * s + KIND_DH] == ps.n_dh &&
               count[3 * s + KIND_DW] == ps.n_dw,
           "%s: slab %d has %lld / %lld / %lld units, expected %d / %d / %d", what, s, count[3 * s],
           count[3 * s + 1], count[3 * s + 2], ps.n_dl, ps.n_dh, ps.n_dw);
    sum += ps.n_dl + ps.n_dh + ps.n_dw;
  }
  EXPECT(sum == d.num_units, "%s: %d units, expected %lld", what, d.num_units, sum);
  check_hazards<TM>(q, d, units, what);
  ++g_launches;
  g_units += d.num_units;
}

// Every row block of one backward call, as the library launches them.
// valid < 0: no row compaction (each block has its own rows); else the
// number of non-ignored rows, which the compacted blocks take in turn.
void check_call(const BwdPlan& b, long long N, long long H, long long V, int tm, long long valid,
                const char* name) {
  if (b.buffers != 2 || b.n_slabs < 2) {
    EXPECT(false, "%s: the plan is not pipelined (buffers %d, slabs %d)", name, b.buffers, b.n_slabs);
    return;
  }
  int count_dev = static_cast<int>(valid);
  GemmParams base{};
  base.N = static_cast<int>(N);
  base.H = static_cast<int>(H);
  base.V = static_cast<int>(V);
  base.ldD = static_cast<int>(b.ldD);
  base.rows_cap = static_cast<int>(b.R);
  int block = 0;
  for (long long row0 = 0; row0 < N; row0 += b.R, ++block) {
    GemmParams p = base;
    int rows;
    if (valid >= 0) {
      rows = static_cast<int>(b.R);
      p.row0 = 0;
      p.rows = rows;
      p.dyn_count = &count_dev;
      p.chunk_first = static_cast<int>(row0);
    } else {
      rows = static_cast<int>(std::min(b.R, N - row0));
      p.row0 = static_cast<int>(row0);
      p.rows = rows;
    }
    const GemmParams q = pipe_params(b, p, H, tm, rows, block);
    char what[160];
    std::snprintf(what, sizeof(what), "%s block %d", name, block);
    if (tm == 2 * BM)
      check_launch<2 * BM>(q, what);
    else
      check_launch<BM>(q, what);
  }
}

// decode_grid over one grid: every (k-split, row tile, column unit) once, in
// range, with its K blocks and output columns.
void check_grid(int m_tiles, int cols, int n_per_unit, int group_m, int k_splits, int kb_per_split, bool col_split) {
  const int n_tiles = cols * n_per_unit - (n_per_unit > 1 ? 1 : 0);  // a ragged last column unit
  const int k_blocks = col_split ? kb_per_split : k_splits * kb_per_split - (kb_per_split > 1 ? 1 : 0);
  const int splits = col_split ? 1 : k_splits;
  std::vector<char> hit(static_cast<size_t>(splits) * m_tiles * cols, 0);
  const int units = splits * m_tiles * cols;
  for (int u = 0; u < units; ++u) {
    const Unit t = decode_grid(u, m_tiles, cols, n_tiles, n_per_unit, group_m, kb_per_split, k_blocks, col_split);
    const int c = t.n0 / n_per_unit;
    const int ks = col_split ? 0 : t.kb0 / kb_per_split;
    const bool in = t.m >= 0 && t.m < m_tiles && c >= 0 && c < cols && ks >= 0 && ks < splits &&
                    t.n0 == c * n_per_unit && t.n1 == std::min(n_tiles, t.n0 + n_per_unit) && t.n1 > t.n0 &&
                    t.kb1 == std::min(k_blocks, t.kb0 + kb_per_split) && t.kb1 > t.kb0 &&
                    t.split == (col_split ? c : ks);
    EXPECT(in, "grid %dx%d (n/unit %d, group %d, splits %d): unit %d decodes to (%d, %d..%d, K %d..%d, split %d)",
           m_tiles, cols, n_per_unit, group_m, k_splits, u, t.m, t.n0, t.n1, t.kb0, t.kb1, t.split);
    if (!in) continue;
    char& h = hit[(static_cast<size_t>(ks) * m_tiles + t.m) * cols + c];
    EXPECT(!h, "grid %dx%d (group %d, splits %d): (%d, %d, %d) decoded twice", m_tiles, cols, group_m, k_splits, ks,
           t.m, c);
    h = 1;
  }
  // a row tile's column units stay inside one raster group of group_m rows
  // (units of a group list its row tiles first, then move to the next column)
  const int g = std::min(group_m, std::max(m_tiles, 1));
  if (m_tiles > 0 && cols > 1) {
    const Unit a = decode_grid(0, m_tiles, cols, n_tiles, n_per_unit, group_m, kb_per_split, k_blocks, col_split);
    const Unit b = decode_grid(std::min(g, m_tiles), m_tiles, cols, n_tiles, n_per_unit, group_m, kb_per_split,
                               k_blocks, col_split);
    EXPECT(a.m == 0 && a.n0 == 0 && b.m == 0 && b.n0 == n_per_unit,
           "grid %dx%d (group %d): unit %d is not the first row tile's second column unit", m_tiles, cols, group_m,
           std::min(g, m_tiles));
  }
}

// The backward's workspace for plan b: regions aligned, disjoint, inside
// what flce_workspace_bytes reports (bwd_workspace), the dlogits inside the
// caller's budget, and a dH partial set for each k-split of any slab.
void check_layout(long long N, long long H, long long V, long long chunk, int workers, int tm, const BwdPlan& b,
                  const char* name) {
  if (b.R <= 0) {
    EXPECT(false, "%s: no row block fits", name);
    return;
  }
  const BwdLayout L = bwd_layout(N, H, b);
  struct Region {
    const char* what;
    size_t off, bytes;
  };
  const Region regs[] = {
      {"dlogits", L.D, static_cast<size_t>(b.buffers) * b.R * b.ldD * 2},
      {"dH partials", L.dh_part, b.dh_f32 ? static_cast<size_t>(b.dh_splits) * b.R * H * 4 : 0},
      {"validation word", L.bad, 4},
      {"row indices", L.idx, static_cast<size_t>(N) * 4},
      {"block counts", L.blk, static_cast<size_t>(ceil_div(N, COMPACT_ROWS_PER_BLOCK)) * 4},
      {"row count", L.count, 4},
      {"gathered rows", L.hc, static_cast<size_t>(b.R) * H * 2},
      {"dependency counters", L.dep, b.buffers == 2 ? static_cast<size_t>(2 * pipe_dep_words(b)) * 4 : 0},
  };
  const int n = static_cast<int>(sizeof(regs) / sizeof(regs[0]));
  for (int i = 0; i < n; ++i) {
    EXPECT(regs[i].off % 256 == 0, "%s: %s at offset %zu", name, regs[i].what, regs[i].off);
    EXPECT(regs[i].off + regs[i].bytes <= L.total, "%s: %s ends past the layout", name, regs[i].what);
    for (int j = 0; j < n; ++j)
      if (i != j && regs[i].bytes > 0 && regs[j].bytes > 0)
        EXPECT(regs[i].off + regs[i].bytes <= regs[j].off || regs[j].off + regs[j].bytes <= regs[i].off,
               "%s: %s and %s overlap", name, regs[i].what, regs[j].what);
  }
  EXPECT(L.total <= bwd_workspace(N, H, V, chunk, workers, tm), "%s: layout of %zu bytes above the reported %zu",
         name, L.total, bwd_workspace(N, H, V, chunk, workers, tm));
  const long long r0 = std::min(round_up(std::max(1LL, chunk), BM), round_up(std::max(1LL, N), BM));
  EXPECT(static_cast<long long>(b.buffers) * b.R * b.ldD <= r0 * round_up(V, 8),
         "%s: dlogits %d x %lld x %lld above the budget %lld x %lld", name, b.buffers, b.R, b.ldD, r0,
         round_up(V, 8));
  if (b.dh_f32) {
    for (int s = 0; s < b.n_slabs; ++s) {
      const long long width = std::min(b.Vs, V - s * b.Vs);
      const long long splits = ceil_div(ceil_div(width, BK), b.dh_kb_per_split);
      EXPECT(splits <= b.dh_splits, "%s: slab %d needs %lld dH partial sets, the workspace holds %d", name, s,
             splits, b.dh_splits);
    }
  }
}

// The forward's plan and workspace for one call: the vocabulary splits cover
// every vocabulary tile once (S ranges of tps tiles, the last one partial),
// the split partials fit their cap, and the regions (target logits, split
// partials, block sums, validation word, and the row-skipping buffers) are
// 256-byte aligned, disjoint and inside the layout.
void check_forward(long long N, long long H, long long V, int workers, int tm, const char* name) {
  const FwdPlan f = plan_forward_call(N, H, V, workers, tm);
  EXPECT(f.S >= 1 && f.S <= 256 && f.tps >= 1 && static_cast<long long>(f.S - 1) * f.tps < f.n_tiles &&
             static_cast<long long>(f.S) * f.tps >= f.n_tiles,
         "%s: %d splits of %d tiles for %d vocabulary tiles", name, f.S, f.tps, f.n_tiles);
  EXPECT(static_cast<size_t>(f.S) * N * 8 <= std::max(kFwdPartialsCap, static_cast<size_t>(N) * 8),
         "%s: split partials %d x %lld rows above their cap", name, f.S, N);
  const long long fb = fwd_block_rows(N, tm);
  const FwdLayout L = fwd_layout(N, f, H, fb);
  struct Region {
    const char* what;
    size_t off, bytes;
  };
  const Region regs[] = {
      {"target logits", L.zt, static_cast<size_t>(N) * 4},
      {"split partials", L.part, static_cast<size_t>(f.S) * N * 8},
      {"block sums", L.bsum, static_cast<size_t>(f.nblk) * 8},
      {"block counts", L.bcnt, static_cast<size_t>(f.nblk) * 8},
      {"validation word", L.bad, 4},
      {"row indices", L.idx, static_cast<size_t>(N) * 4},
      {"index block counts", L.blk, static_cast<size_t>(ceil_div(std::max(1LL, N), COMPACT_ROWS_PER_BLOCK)) * 4},
      {"row count", L.count, 4},
      {"gathered rows", L.hc, static_cast<size_t>(fb) * H * 2},
  };
  const int n = static_cast<int>(sizeof(regs) / sizeof(regs[0]));
  for (int i = 0; i < n; ++i) {
    EXPECT(regs[i].off % 256 == 0, "%s: forward %s at offset %zu", name, regs[i].what, regs[i].off);
    EXPECT(regs[i].off + regs[i].bytes <= L.total, "%s: forward %s ends past the layout", name, regs[i].what);
    for (int j = 0; j < n; ++j)
      if (i != j && regs[i].bytes > 0 && regs[j].bytes > 0)
        EXPECT(regs[i].off + regs[i].bytes <= regs[j].off || regs[j].off + regs[j].bytes <= regs[i].off,
               "%s: forward %s and %s overlap", name, regs[i].what, regs[j].what);
  }
}

void set_rows(long long r) {
  init_options();
  g_options[FLCE_OPT_BWD_ROWS].store(r);
}

void planned(long long N, long long H, long long V, long long chunk, int cg, long long rows, long long valid,
             const char* name) {
  set_rows(rows);
  const int tm = cg * BM;
  const int workers = cg == 2 ? 76 : 152;
  const BwdPlan b = plan_backward_call(N, H, V, chunk, workers, tm, true);
  check_layout(N, H, V, chunk, workers, tm, b, name);
  check_call(b, N, H, V, tm, valid, name);
}

// splitmix64 (Steele, Lea, Flood: "Fast splittable pseudorandom number
// generators"), for the seeded sweep
uint64_t g_state = 0x5eed;
uint64_t next_u64() {
  uint64_t z = (g_state += 0x9e3779b97f4a7c15ULL);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}
long long uniform(long long lo, long long hi) {  // [lo, hi]
  return lo + static_cast<long long>(next_u64() % static_cast<uint64_t>(hi - lo + 1));
}

}  // namespace

int main() {
  // the planner's launches for the library's workloads and the GPU tests'
  // pipelined cases, with and without row compaction, both tile heights
  planned(131072, 2560, 151936, 256, 2, 0, -1, "131072x2560x151936");
  planned(131072, 2560, 151936, 256, 2, 0, 131072 - 1000, "131072x2560x151936 compacted");
  planned(131072, 2560, 151936, 256, 1, 0, -1, "131072x2560x151936 cg1");
  for (int cg = 1; cg <= 2; ++cg) {
    planned(3000, 512, 20000, 256, cg, 768, -1, "3000x512x20000");
    planned(3000, 512, 20000, 256, cg, 768, 2760, "3000x512x20000 compacted");
    planned(1000, 264, 7777, 128, cg, 512, -1, "1000x264x7777");
    planned(1000, 264, 7777, 128, cg, 512, 920, "1000x264x7777 compacted");
    planned(1000, 128, 4000, 128, cg, 256, 0, "1000x128x4000 all rows ignored");
    planned(8192, 2560, 151936, 256, cg, 3328, -1, "8192x2560x151936");
  }
  set_rows(0);
  // the planner's plans over a seeded sweep of problem sizes: the workspace
  // layout of the plain and the pipelined plan, and the schedule of the
  // pipelined one
  long long plans = 0;
  for (int i = 0; i < 300; ++i) {
    const int cg = (i & 1) ? 2 : 1;
    const int tm = cg * BM, workers = cg == 2 ? 76 : 152;
    const long long N = uniform(1, 140000), H = 8 * uniform(8, 1024), V = uniform(1000, 260000);
    const long long chunks[] = {128, 256, 1024, 4096};
    const long long chunk = chunks[uniform(0, 3)];
    char name[96];
    std::snprintf(name, sizeof(name), "planned %d (N %lld, H %lld, V %lld, chunk %lld, cg %d)", i, N, H, V, chunk,
                  cg);
    check_forward(N, H, V, workers, tm, name);
    const BwdPlan plain = plan_backward(N, H, V, chunk, workers, tm);
    check_layout(N, H, V, chunk, workers, tm, plain, name);
    const BwdPlan b = plan_backward_call(N, H, V, chunk, workers, tm, true);
    check_layout(N, H, V, chunk, workers, tm, b, name);
    if (b.buffers == 2 && N <= 20000) check_call(b, N, H, V, tm, (i % 3 == 0) ? -1 : uniform(0, N), name);
    ++plans;
  }
  // a seeded sweep of plans: row capacity, slab width, vocabulary, width,
  // dH k-split depth, tile height, live rows (some blocks empty)
  for (int i = 0; i < 400; ++i) {
    const int tm = (i & 1) ? 2 * BM : BM;
    BwdPlan b;
    b.R = 64 * uniform(1, 48);
    b.Vs = BN * uniform(1, 24);
    const long long V = uniform(b.Vs + 1, 7 * b.Vs);
    b.n_slabs = static_cast<int>(ceil_div(V, b.Vs));
    b.ldD = b.Vs;
    b.dh_kb_per_split = static_cast<int>(uniform(1, ceil_div(b.Vs, BK)));
    b.dh_f32 = true;
    b.buffers = 2;
    const long long H = 8 * uniform(1, 512);
    const long long N = uniform(1, 4 * b.R);
    const long long valid = (i % 3 == 0) ? -1 : uniform(0, N);
    char name[96];
    std::snprintf(name, sizeof(name), "sweep %d (R %lld, Vs %lld, V %lld, H %lld, N %lld)", i, b.R, b.Vs, V, H, N);
    check_call(b, N, H, V, tm, valid, name);
  }
  // the raster decoding of every GEMM launch
  long long grids = 0;
  for (int i = 0; i < 3000; ++i) {
    const int m_tiles = static_cast<int>(uniform(1, 40));
    const int cols = static_cast<int>(uniform(1, 40));
    const int n_per_unit = static_cast<int>(uniform(1, 3));
    const int group_m = static_cast<int>(uniform(1, 48));
    const int k_splits = static_cast<int>(uniform(1, 6));
    const int kb = static_cast<int>(uniform(1, 9));
    check_grid(m_tiles, cols, n_per_unit, group_m, k_splits, kb, (i % 4) == 0);
    ++grids;
  }
  if (g_fails) {
    std::printf("FAILED: %d checks in %lld launches\n", g_fails, g_launches);
    return 1;
  }
  std::printf("ok: %lld launches, %lld units; %lld planned layouts; %lld raster grids\n", g_launches, g_units,
              plans, grids);
  return 0;
}
