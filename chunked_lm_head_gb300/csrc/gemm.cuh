// Persistent tcgen05 GEMM engine of libflce and its epilogues.
//
// One CTA per SM, running alone (CG = 1) or as one half of an SM pair
// (CG = 2, tcgen05 cta_group::2 with 256 x 256 tiles).  Warp 0 (one lane)
// streams operand tiles with TMA into a shared-memory ring; warp 1 (one lane
// of the pair's first CTA) issues tcgen05.mma into fp32 TMEM accumulators;
// warps 2-5 drain an accumulator with tcgen05.ld and run the mode's epilogue,
// overlapping the MMAs of the next tile where two accumulators fit in TMEM.
//
// Modes (the contractions of the chunked LM-head losses):
//   FWD         Z = h W^T over a split of the vocabulary; epilogue keeps an
//               online row max / sum of exp in registers (each thread owns one
//               row of the accumulator, so no cross-thread reduction is
//               needed) and gathers the target logit.  Emits per-(row, split)
//               partials.  bf16 or (kF8) e4m3 operands with row scales.
//   DLOGITS     the same Z recomputed for one row chunk; epilogue forms
//               D = (exp(Z - lse) - onehot(t)) * m * w * g in bf16.
//   DH          dH[chunk rows] = D W         (K = vocabulary; W read MN-major)
//   DW          dW (+)= D^T h[chunk rows]    (K = chunk rows; D and h MN-major;
//               TMA store / fp32 reduce-add epilogue)
//   KD_FWD      distillation: student and teacher logits of a tile side by
//               side in TMEM; online log-sum-exp of both heads and the
//               teacher-weighted logit difference
//   KD_DLOGITS  distillation: D = (p_s - p_t) * m * w * g
//   DHDW        the DH and DW units of one vocabulary slab in one launch (dH
//               units first, then dW units): one launch's fixed cost per
//               slab instead of two, and the dH and dW streams overlap
//
// Sources: Unsloth, "Reinforcement Learning GRPO with 7x longer context",
// sections "Flattened sequence-length chunking" (chunk logits are
// hidden @ lm_head, upcast to fp32, log-softmaxed, target gathered) and
// "Offloading activations for log-softmax" (backward recomputes the chunk);
// TRL v1.13 article, speed & memory section (keep both GEMM operands bf16 on
// the tensor cores instead of the fp32 SIMT path; the distillation trainer
// computes each chunk with both heads).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace flce {

constexpr int BM = 128;  // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;  // accumulator columns (fp32 TMEM columns)
constexpr int BK = 64;   // one 128-byte swizzle row of bf16 per stage
constexpr int UMMA_K = 16;
constexpr int MN_BOX_BYTES = 64 * BK * 2;  // one 64(MN) x 64(K) swizzled box
constexpr int EPI_WARPS = 4;
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
// dW epilogue staging: per epilogue warp two 32x32 fp32 boxes (128B-swizzled)
// handed to TMA store / reduce-add.
constexpr int OUT_BOX_BYTES = 32 * 32 * 4;
constexpr int OUT_STAGE_BYTES = EPI_WARPS * 2 * OUT_BOX_BYTES;
constexpr int SMEM_BAR_BYTES = 512;
// PIPE: unit indices in flight between the fetching thread and the CTA's
// roles (a ring of this many slots, each with a full and an empty mbarrier)
constexpr int kUnitRing = 6;

// Tile geometry of one CTA (CG = 1) or of an SM pair running 2-CTA MMAs
// (CG = 2: a 256 x 256 tile, A rows and B columns split across the pair).
template <int CG>
struct TileCfg {
  static constexpr int TM = BM * CG;         // tile rows of the CTA group
  static constexpr int B_ROWS = BN / CG;     // B rows (output columns) held by each CTA
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;  // 48 KiB (CG 1) / 32 KiB (CG 2)
  static constexpr int NSTAGE = CG == 1 ? 4 : 6;
  static constexpr int SMEM = 1024 + NSTAGE * STAGE + OUT_STAGE_BYTES + SMEM_BAR_BYTES;
  static_assert(SMEM <= 232448, "exceeds the 227 KiB shared memory of one CTA");
};
constexpr long long WAIT_LIMIT_CYCLES = 2000000000LL;  // ~1 s at 2 GHz
constexpr long long DRAIN_LIMIT_CYCLES = 400000000LL;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2f = 0.6931471805599453f;

enum Mode : int {
  MODE_FWD = 0,
  MODE_DLOGITS = 1,
  MODE_DH = 2,
  MODE_DW = 3,
  // distillation (student and teacher heads in one tile pipeline): K runs
  // over the student's hidden blocks into TMEM columns [0, BN), then over the
  // teacher's into [BN, 2 BN)
  MODE_KD_FWD = 4,
  MODE_KD_DLOGITS = 5,
  // Jensen-Shannon distillation, same two-head pipeline: the per-row mixture
  // terms given both heads' log-sum-exp, and the student's dlogits
  MODE_JSD_FWD = 6,
  MODE_JSD_DLOGITS = 7,
  // forward that also keeps each row block's exp(logit - chunk max) in bf16
  // (and the chunk maxima) for a backward without the logits recompute
  MODE_FUSED_FWD = 8,
  // DH and DW of one slab in one launch: units [0, dH units) are DH units
  // (operands tmA / tmB, output tmC), the rest DW units (tmA2 / tmB2, tmC2)
  MODE_DHDW = 9,
  // the whole backward of one row block in one launch: for each vocabulary
  // slab its DLOGITS units (tmA3 / tmB3, D out through tmC3), then its DH
  // units (tmA / tmB, tmC) and DW units (tmA2 / tmB2, tmC2).  Units wait on
  // device-side counters for the units whose output they read or overwrite.
  MODE_PIPE = 10,
  // DH over 256 x 512 tiles (SM pairs only): each stage holds one A block and
  // the B blocks of two adjacent 256-column tiles, whose two accumulators fill
  // TMEM; a quarter fewer operand bytes per FLOP than two separate tiles.  For
  // K walks long enough that the epilogue's lack of overlap does not count
  MODE_DH2 = 11
};
// unit kinds of MODE_PIPE
constexpr int KIND_DL = 0, KIND_DH = 1, KIND_DW = 2;
// Shared-memory layout of one kernel instantiation: the operand ring and the
// output staging boxes.  dW at short K with 16 epilogue warps (four per TMEM
// lane quarter, each on a quarter of the tile's columns) trades two operand
// stages for one staging box per warp: its units are a few K blocks long and
// their fp32 output, not the MMAs, sets the pace.
template <int MODE, int CG, int EW>
struct KernelCfg {
  static constexpr bool kWideN = MODE == MODE_DH2;  // two B tiles per stage
  static constexpr int STAGE = TileCfg<CG>::A_BYTES + (kWideN ? 2 : 1) * TileCfg<CG>::B_BYTES;
  static constexpr int TILE_N = (kWideN ? 2 : 1) * BN;  // accumulator columns of a unit's tile
  static constexpr bool kDeepOut = MODE == MODE_DW && EW == 16;
  static constexpr int NSTAGE = kWideN ? 4 : kDeepOut ? (CG == 1 ? 3 : 4) : TileCfg<CG>::NSTAGE;
  static constexpr int OUT_BYTES = kDeepOut ? EW * OUT_BOX_BYTES : OUT_STAGE_BYTES;
  static constexpr int BOXES_PER_WARP = OUT_BYTES / OUT_BOX_BYTES / EW > 0 ? OUT_BYTES / OUT_BOX_BYTES / EW : 1;
  static constexpr int SMEM = 1024 + NSTAGE * STAGE + OUT_BYTES + SMEM_BAR_BYTES;
  static_assert(SMEM <= 232448, "exceeds the 227 KiB shared memory of one CTA");
  static_assert(!kWideN || CG == 2, "256 x 512 dH tiles run on SM pairs");
  static_assert(BOXES_PER_WARP * EW * OUT_BOX_BYTES <= OUT_BYTES, "staging boxes exceed the staging area");
};
template <int MODE>
__host__ __device__ constexpr bool is_kd() {
  return MODE == MODE_KD_FWD || MODE == MODE_KD_DLOGITS || MODE == MODE_JSD_FWD ||
         MODE == MODE_JSD_DLOGITS;
}
// modes that may run 8 epilogue warps, two per TMEM lane quarter, each
// taking half of the tile's columns: dW, and the two-head modes whose
// epilogue does not overlap the next tile's MMAs (the Jensen-Shannon
// forward's per-row partials of each half go to a slot of their own)
template <int MODE>
__host__ __device__ constexpr bool wide_epilogue_mode() {
  return MODE == MODE_DW || MODE == MODE_DHDW || MODE == MODE_KD_DLOGITS || MODE == MODE_JSD_DLOGITS ||
         MODE == MODE_JSD_FWD;
}
// modes whose accumulator rows are rows of h (all but dW, whose accumulator
// rows are vocabulary rows): under row compaction they map through row_idx
// and take their row count from the device (DHDW, PIPE: their DH and DLOGITS
// units only)
template <int MODE>
__host__ __device__ constexpr bool rows_are_tokens() {
  return MODE != MODE_DW && MODE != MODE_DHDW && MODE != MODE_PIPE;
}
// modes whose units are (row tile, vocabulary split) with per-row partials
template <int MODE>
__host__ __device__ constexpr bool is_split_fwd() {
  return MODE == MODE_FWD || MODE == MODE_KD_FWD || MODE == MODE_JSD_FWD || MODE == MODE_FUSED_FWD;
}

// Threads of a GEMM CTA with `ew` epilogue warps: 4, one per TMEM lane
// quarter; or 8 / 16 (the dW mode at short K), two / four per quarter, each
// on a share of the tile's columns, so that the fp32 output epilogue keeps
// up with MMAs over only a few K blocks.
__host__ __device__ constexpr int gemm_threads(int ew) { return 64 + 32 * ew; }
// PIPE adds one warp that waits on the units' dependency counters ahead of
// the producer (see pipe_wait_deps).
template <int MODE>
__host__ __device__ constexpr int kernel_threads(int ew) {
  return gemm_threads(ew) + (MODE == MODE_PIPE ? 32 : 0);
}

// bit 0 of the device error word: a bounded wait ran out.
constexpr int DEVERR_TIMEOUT = 1;

struct GemmParams {
  int m_tiles, n_tiles, k_blocks;
  int cols;           // column units per k-split: FWD vocabulary splits, else n_tiles
  int n_per_unit;     // FWD: vocabulary tiles per split; else 1
  int kb_per_split;   // DH split-K: k-blocks per split; else k_blocks
  int num_units;      // = k_splits * m_tiles * cols
  int group_m;        // rasterisation: row tiles that share column units
  int row0, rows;     // first global row of this pass, rows in this pass
  int rows_cap;       // row capacity of the chunk buffers (DH split partials)
  int N, H, V, ldD;
  const int64_t* targets;
  const float* weights;
  const float* lse;
  float grad_scale;
  long long ignore_index;
  // logit transform y = f(z) before the log-softmax: linear y = tf_a * z
  // (tf_softcap == 0), or soft-capped y = tf_b * tanh(tf_a * z) with
  // dy/dz = tf_d * (1 - tanh^2)
  int tf_softcap;
  float tf_a, tf_b, tf_d;
  float2* partials;   // FWD: [splits][N] (max*log2e, sum exp2)
  float* zt;          // FWD: [N] target logit
  uint16_t* D;        // DLOGITS out [rows_cap][ldD] bf16
  uint16_t* dH;       // DH out [N][H] bf16 (single split)
  float* dH_part;     // DH out [k_splits][rows_cap][H] fp32 (split-K)
  float* dW;          // DW out [V][H] fp32
  int dW_accumulate;
  int* err;           // device error word
  // Row compaction (backwards on non-ignored rows only): row_idx maps a
  // compacted row to its original row; this pass holds compacted rows
  // [chunk_first, chunk_first + rows) with rows = min(*dyn_count - chunk_first,
  // rows_cap) read on the device.  row_idx == nullptr: rows are row0 + i.
  // The forward modes read row_idx too.  The fused forward's rows are a
  // block of a permutation that puts the non-ignored rows first (with
  // dyn_count, only those are computed); the forward's and the distillation
  // forwards', with dyn_count, a block of the non-ignored rows.
  const int* row_idx;
  const int* dyn_count;
  int chunk_first;
  int k_splits;
  // distillation: student K blocks (the rest of k_blocks are the teacher's),
  // teacher log-sum-exp and the extra forward partials
  int k_blocks_s;
  const float* lse_t;
  float2* partials_t;  // [splits][N] (teacher max*log2e, sum exp2)
  float* partials_c;   // [splits][N] sum exp2(u_t - m_t) * (z_t - z_s)
  // Jensen-Shannon forward terms: 2 = each tile's columns are split between
  // two epilogue warps, which write their per-row partials to slots 2 split
  // and 2 split + 1 (the partial array then holds 2 x splits slots); else 1
  int col_parts;
  // e4m3 forward: logits = acc * a_scale[row] * b_scale[vocabulary row]
  const float* a_scale;
  const float* b_scale;
  // Vocabulary slab of a backward pass: logit columns [v0, v0 + width) held
  // in D at local columns [0, width).  0 in the forward modes.
  int v0;
  // DH into fp32 partials (through tmC): reduce-add onto the previous slabs'
  // sums, else a plain store
  int dh_accumulate;
  // Jensen-Shannon distillation: mixture weight of the teacher, and (dlogits)
  // each row's KL(p_student || mixture) in natural-log units
  float jsd_beta;
  const float* kl_sm;
  // FUSED_FWD: per row and 32-column chunk, the chunk's maximum transformed
  // logit x log2(e), [rows_cap][ldD / 32]; the exponentials go to D
  float* mx;
  // dlogits modes: divide grad_scale by max(*count_scale, 1) (a count on the
  // device) and multiply it by *scale_dev (a scale on the device), when set
  const long long* count_scale;
  const float* scale_dev;
  // DLOGITS: write D through tmC (bf16 [rows_cap][ldD], 64 x 32 boxes) from
  // shared memory instead of per-thread global stores
  int d_tma;
  // DHDW: the DW units' grid (vocabulary tiles of the slab x hidden tiles,
  // K = the block's rows, one split); the DH units use the fields above
  int dw_m_tiles, dw_n_tiles, dw_k_blocks, dw_group_m;
  // PIPE: slabs of pp_vs vocabulary columns (the last one narrower) over the
  // whole vocabulary; pp_kh K blocks of H per DLOGITS tile; row tiles at most
  // m_tiles (the capacity); dH k-splits of dh_kbps K blocks.  D holds two
  // buffers of rows_cap rows, slab s in buffer s % 2.  Dependency counters:
  // pp_dep (this launch's, zero at its start) and pp_dep_zero (the next
  // launch's, zeroed here), pp_dep_words each.
  // pp_lookahead: units a pair may hold drawn but not finished (1..kUnitRing)
  int pp_slabs, pp_vs, pp_kh, pp_dh_kbps, pp_dl_group, pp_dep_words, pp_lookahead;
  unsigned* pp_dep;
  unsigned* pp_dep_zero;
};

// grad_scale of the dlogits modes with its device-side factors: / max(count, 1)
// and * scale, each when given.
__device__ __forceinline__ float device_grad_scale(const GemmParams& p) {
  float g = p.grad_scale;
  if (p.count_scale != nullptr) g *= 1.f / fmaxf(1.f, static_cast<float>(*p.count_scale));
  if (p.scale_dev != nullptr) g *= *p.scale_dev;
  return g;
}

// Problem extents that depend on the device-side row count of a compacted pass.
// DHDW: m_tiles / k_blocks / kb_per_split are its DH units', dh_units of them,
// followed by dw_units DW units of dw_k_blocks K blocks.
// PIPE: dh_units = the units of one full slab.
struct DynShape {
  int rows, m_tiles, k_blocks, kb_per_split, num_units;
  int dh_units, dw_units, dw_k_blocks;
};

// PIPE: one vocabulary slab of the row block -- its columns, its tiles for
// DLOGITS (BN wide), DW (TM wide) and DH (BK-deep K blocks, dh_kbps per
// split), and its unit counts.
struct PipeSlab {
  int v0, width, vt, dwt, kb, splits, n_dl, n_dh, n_dw;
};

template <int TM>
__host__ __device__ __forceinline__ PipeSlab pipe_slab(const GemmParams& p, const DynShape& d, int s) {
  PipeSlab q;
  q.v0 = s * p.pp_vs;
  q.width = min(p.pp_vs, p.V - q.v0);
  q.vt = (q.width + BN - 1) / BN;
  q.dwt = (q.width + TM - 1) / TM;
  q.kb = (q.width + BK - 1) / BK;
  q.splits = (q.kb + p.pp_dh_kbps - 1) / p.pp_dh_kbps;
  q.n_dl = d.m_tiles * q.vt;
  q.n_dh = q.splits * d.m_tiles * p.n_tiles;
  // an empty first row block still writes zeros to dW, an empty later one
  // has nothing to add
  q.n_dw = (d.rows == 0 && p.dW_accumulate) ? 0 : q.dwt * p.n_tiles;
  return q;
}

template <int MODE, int TM>
__host__ __device__ __forceinline__ DynShape dyn_shape(const GemmParams& p) {
  DynShape d{p.rows, p.m_tiles, p.k_blocks, p.kb_per_split, p.num_units, 0, 0, 0};
  if constexpr (MODE == MODE_PIPE) {
    if (p.dyn_count != nullptr) {
      d.rows = max(0, min(*p.dyn_count - p.chunk_first, p.rows_cap));
      d.m_tiles = (d.rows + TM - 1) / TM;
      d.dw_k_blocks = (d.rows + BK - 1) / BK;
    } else {
      d.dw_k_blocks = p.dw_k_blocks;
    }
    // units of phase p: slab p's DLOGITS units, then slab p - 1's DH and DW
    // units (phases 0 .. slabs); dh_units = the units of a middle phase
    const PipeSlab q0 = pipe_slab<TM>(p, d, 0);
    const PipeSlab ql = pipe_slab<TM>(p, d, p.pp_slabs - 1);
    d.dh_units = q0.n_dl + q0.n_dh + q0.n_dw;
    d.num_units = (p.pp_slabs - 1) * d.dh_units + ql.n_dl + ql.n_dh + ql.n_dw;  // every slab's units
    return d;
  }
  if constexpr (MODE == MODE_DHDW) {
    if (p.dyn_count != nullptr) {
      d.rows = max(0, min(*p.dyn_count - p.chunk_first, p.rows_cap));
      d.m_tiles = (d.rows + TM - 1) / TM;
      d.dw_k_blocks = (d.rows + BK - 1) / BK;
    } else {
      d.dw_k_blocks = p.dw_k_blocks;
    }
    d.dh_units = p.k_splits * d.m_tiles * p.cols;
    // an empty first pass still writes zeros to dW, an empty later pass has
    // nothing to add
    d.dw_units = (d.rows == 0 && p.dW_accumulate) ? 0 : p.dw_m_tiles * p.dw_n_tiles;
    d.num_units = d.dh_units + d.dw_units;
    return d;
  }
  if (p.dyn_count != nullptr) {
    d.rows = max(0, min(*p.dyn_count - p.chunk_first, p.rows_cap));
    if constexpr (rows_are_tokens<MODE>()) {
      d.m_tiles = (d.rows + TM - 1) / TM;
      d.num_units = p.k_splits * d.m_tiles * p.cols;
    } else if constexpr (MODE == MODE_DW) {
      // K = the pass's rows; an empty first pass still writes zeros to dW,
      // an empty later pass has nothing to add
      d.k_blocks = (d.rows + BK - 1) / BK;
      d.kb_per_split = max(d.k_blocks, 1);
      d.num_units = (d.rows == 0 && p.dW_accumulate) ? 0 : p.m_tiles * p.cols;
    }
  }
  return d;
}

struct Unit {
  int m, n0, n1, kb0, kb1, split;
  bool dw;   // DHDW, PIPE: a DW unit
  int kind;  // PIPE: KIND_DL / KIND_DH / KIND_DW
  int slab;  // PIPE: its vocabulary slab
};

// Unit u of a grid of (k-splits x m_tiles x cols) units, rasterised in
// groups of group_m row tiles that share their column units.
__host__ __device__ __forceinline__ Unit decode_grid(int u, int m_tiles, int cols, int n_tiles, int n_per_unit,
                                            int group_m_req, int kb_per_split, int k_blocks,
                                            bool col_split) {
  const int group_m = min(group_m_req, max(m_tiles, 1));
  const int per_split = m_tiles * cols;
  const int ks = u / per_split;
  const int r = u - ks * per_split;
  const int full_groups = m_tiles / group_m;
  int first_m, gsize, local;
  if (r < full_groups * group_m * cols) {
    const int g = r / (group_m * cols);
    first_m = g * group_m;
    gsize = group_m;
    local = r - g * group_m * cols;
  } else {
    first_m = full_groups * group_m;
    gsize = m_tiles - first_m;
    local = r - full_groups * group_m * cols;
  }
  Unit t;
  t.m = first_m + local % gsize;
  const int c = local / gsize;
  t.n0 = c * n_per_unit;
  t.n1 = min(n_tiles, t.n0 + n_per_unit);
  t.kb0 = ks * kb_per_split;
  t.kb1 = min(k_blocks, t.kb0 + kb_per_split);
  t.split = col_split ? c : ks;
  t.dw = false;
  t.kind = 0;
  t.slab = 0;
  return t;
}

template <int MODE, int TM = BM>
__host__ __device__ __forceinline__ Unit decode_unit(const GemmParams& p, const DynShape& d, int u) {
  if constexpr (MODE == MODE_PIPE) {
    // phase by phase: phase p holds slab p's DLOGITS units (p < slabs), then
    // slab p - 1's DH units and DW units (p > 0).  Phase 0 has the first
    // slab's DLOGITS units; every middle phase a full slab's DLOGITS, DH and
    // DW units (F of them); phase slabs - 1 the last slab's DLOGITS units and
    // a full slab's DH and DW; phase slabs the last slab's DH and DW.
    const int S = p.pp_slabs;
    const PipeSlab qf = pipe_slab<TM>(p, d, 0);
    const PipeSlab ql = pipe_slab<TM>(p, d, S - 1);
    const int F = d.dh_units;
    int ph, local;
    if (u < qf.n_dl) {
      ph = 0;
      local = u;
    } else if (u < qf.n_dl + (S - 2) * F) {
      ph = 1 + (u - qf.n_dl) / F;
      local = u - qf.n_dl - (ph - 1) * F;
    } else if (u < qf.n_dl + (S - 2) * F + ql.n_dl + qf.n_dh + qf.n_dw) {
      ph = S - 1;
      local = u - qf.n_dl - (S - 2) * F;
    } else {
      ph = S;
      local = u - qf.n_dl - (S - 2) * F - ql.n_dl - qf.n_dh - qf.n_dw;
    }
    Unit t;
    const PipeSlab qd = ph < S ? pipe_slab<TM>(p, d, ph) : ql;  // DLOGITS slab of the phase
    const int n_dl = ph < S ? qd.n_dl : 0;
    if (local < n_dl) {
      t = decode_grid(local, d.m_tiles, qd.vt, qd.vt, 1, p.pp_dl_group, p.pp_kh, p.pp_kh, false);
      t.kind = KIND_DL;
      t.slab = ph;
      return t;
    }
    local -= n_dl;
    const PipeSlab q = ph == S ? ql : qf;  // slab ph - 1: full unless the last
    if (local < q.n_dh) {
      t = decode_grid(local, d.m_tiles, p.n_tiles, p.n_tiles, 1, p.group_m, p.pp_dh_kbps, q.kb, false);
      t.kind = KIND_DH;
    } else {
      t = decode_grid(local - q.n_dh, q.dwt, p.n_tiles, p.n_tiles, 1, p.dw_group_m, max(d.dw_k_blocks, 1),
                      d.dw_k_blocks, false);
      t.kind = KIND_DW;
      t.dw = true;
    }
    t.slab = ph - 1;
    return t;
  }
  if constexpr (MODE == MODE_DHDW) {
    if (u >= d.dh_units) {
      Unit t = decode_grid(u - d.dh_units, p.dw_m_tiles, p.dw_n_tiles, p.dw_n_tiles, 1, p.dw_group_m,
                           max(d.dw_k_blocks, 1), d.dw_k_blocks, false);
      t.dw = true;
      return t;
    }
  }
  return decode_grid(u, d.m_tiles, p.cols, p.n_tiles, p.n_per_unit, p.group_m, d.kb_per_split, d.k_blocks,
                     is_split_fwd<MODE>());
}

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA's
// abort flag and the device error word) when the limit runs out, or when
// another role of the CTA has already aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* err, long long limit = WAIT_LIMIT_CYCLES) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(err, DEVERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// ---- PIPE: dependency counters between the units of one launch
//
// Four arrays of counters, each epilogue warp of a unit adding one when its
// share of the unit's output is in global memory: per slab and row tile, the
// DLOGITS units done (dl_row) and the DH units done (dh_row); per slab and
// BN-wide vocabulary tile, the DLOGITS units done (dl_col) and the DW units
// done (dw_col).  D holds two slabs (slab s in buffer s % 2), so
//   - a DH unit of slab s reads D rows of its row tile over the slab: it waits
//     for dl_row[s][m], and, so that the dH partials are summed slab after
//     slab, for dh_row[s - 1][m];
//   - a DW unit reads D columns of its vocabulary tile over all rows: it
//     waits for dl_col[s][vt];
//   - a DLOGITS unit of slab s overwrites a tile of the buffer that slab
//     s - 2's DH units of its row tile and DW units of its vocabulary tile
//     read: it waits for dh_row[s - 2][m] and dw_col[s - 2][vt].
// Units run in phases (phase p: slab p's DLOGITS units, then slab p - 1's DH
// and DW units), so every wait is on units of an earlier phase, i.e. earlier
// in the unit order.  Workers draw units from a counter in that order, so
// every unit a wait names has been drawn by a running worker and the lowest
// unfinished unit can always run, however many CTAs of the grid are
// resident.  Slab s + 1's dlogits are formed while slab s's dH and dW run.
struct PipeDeps {
  int mt_cap, vt_cap, slabs;
  __host__ __device__ int dl_row(int s, int m) const { return s * mt_cap + m; }
  __host__ __device__ int dh_row(int s, int m) const { return (slabs + s) * mt_cap + m; }
  __host__ __device__ int dl_col(int s, int vt) const { return 2 * slabs * mt_cap + s * vt_cap + vt; }
  __host__ __device__ int dw_col(int s, int vt) const {
    return 2 * slabs * mt_cap + (slabs + s) * vt_cap + vt;
  }
};

__host__ __device__ __forceinline__ PipeDeps pipe_deps(const GemmParams& p) {
  return PipeDeps{p.m_tiles, (p.pp_vs + BN - 1) / BN, p.pp_slabs};
}

// A dependency counter of a pipelined launch and the count it must reach.
struct PipeWait {
  int idx;
  unsigned target;
};

// The counters unit t waits on before its operands are loaded (at most 2,
// into w; returns how many), with ARR arrivals per finished unit.
template <int TM, int ARR>
__host__ __device__ __forceinline__ int pipe_unit_waits(const GemmParams& p, const DynShape& d, const Unit& t,
                                                        PipeWait* w) {
  const PipeDeps g = pipe_deps(p);
  int n = 0;
  if (t.kind == KIND_DH) {
    const PipeSlab q = pipe_slab<TM>(p, d, t.slab);
    w[n++] = PipeWait{g.dl_row(t.slab, t.m), static_cast<unsigned>(q.vt * ARR)};
    if (t.slab > 0) {
      const PipeSlab qp = pipe_slab<TM>(p, d, t.slab - 1);
      w[n++] = PipeWait{g.dh_row(t.slab - 1, t.m), static_cast<unsigned>(qp.splits * p.n_tiles * ARR)};
    }
  } else if (t.kind == KIND_DW) {
    w[n++] = PipeWait{g.dl_col(t.slab, t.m * TM / BN), static_cast<unsigned>(d.m_tiles * ARR)};
  } else if (t.slab > 1) {
    // DLOGITS over a tile of the buffer that slab s - 2 read
    const PipeSlab q = pipe_slab<TM>(p, d, t.slab - 2);
    const int vt = t.n0;
    const int dw_in = min(BN / TM, q.dwt - vt * (BN / TM));  // DW vocabulary tiles inside it
    w[n++] = PipeWait{g.dh_row(t.slab - 2, t.m), static_cast<unsigned>(q.splits * p.n_tiles * ARR)};
    w[n++] = PipeWait{g.dw_col(t.slab - 2, vt), static_cast<unsigned>(q.n_dw > 0 ? dw_in * p.n_tiles * ARR : 0)};
  }
  return n;
}

// The counters that each epilogue warp of unit t adds one arrival to once
// its share of the unit is in global memory (at most 2, into idx).
template <int TM>
__host__ __device__ __forceinline__ int pipe_unit_signals(const GemmParams& p, const Unit& t, int* idx) {
  const PipeDeps g = pipe_deps(p);
  if (t.kind == KIND_DL) {
    idx[0] = g.dl_row(t.slab, t.m);
    idx[1] = g.dl_col(t.slab, t.n0);
    return 2;
  }
  idx[0] = t.kind == KIND_DH ? g.dh_row(t.slab, t.m) : g.dw_col(t.slab, t.m * TM / BN);
  return 1;
}

// Bounded wait until counter c reaches target.  Gives up (raising the CTA's
// abort flag) when another role of the CTA has aborted, when another CTA has
// raised the device error word, or when the limit runs out (raising it).
__device__ __forceinline__ bool pipe_wait(const unsigned* c, unsigned target, volatile int* abort_flag,
                                          int* err) {
  if (target == 0 || ld_acquire_gpu(c) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_gpu(c) < target) {
    if (*abort_flag) return false;
    if (*reinterpret_cast<volatile int*>(err) & DEVERR_TIMEOUT) {
      *abort_flag = 1;
      return false;
    }
    if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
      *abort_flag = 1;
      atomicOr(err, DEVERR_TIMEOUT);
      return false;
    }
    __nanosleep(100);
  }
  return true;
}

// The waits of unit t before its operands are loaded (ARR arrivals per
// unit: one per epilogue warp of each CTA).  Run by the fetching thread; the
// producer then orders its bulk loads after them (fence.proxy.async).
template <int TM, int ARR>
__device__ __forceinline__ bool pipe_wait_deps(const GemmParams& p, const DynShape& d, const Unit& t,
                                               volatile int* abort_flag) {
  PipeWait w[2];
  const int n = pipe_unit_waits<TM, ARR>(p, d, t, w);
  for (int i = 0; i < n; ++i)
    if (!pipe_wait(p.pp_dep + w[i].idx, w[i].target, abort_flag, p.err)) return false;
  return true;
}

// Bounded wait on an mbarrier phase completed by a release-arrive of a peer
// CTA (cluster-scope acquire); as wait_bar otherwise.
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                 int* err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
      *abort_flag = 1;
      atomicOr(err, DEVERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// This epilogue warp's share of unit t is complete in global memory: count it.
template <int TM>
__device__ __forceinline__ void pipe_signal(const GemmParams& p, const Unit& t) {
  int idx[2];
  const int n = pipe_unit_signals<TM>(p, t, idx);
  for (int i = 0; i < n; ++i) red_release_gpu_add(p.pp_dep + idx[i], 1u);
}

// Bounded wait used only while shutting down (copies or MMAs in flight).
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, int* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > DRAIN_LIMIT_CYCLES) {
      atomicOr(err, DEVERR_TIMEOUT);
      return;
    }
  }
}

template <int MODE, int CG>
__device__ __forceinline__ void tma_ld(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                                       int32_t c1) {
  if constexpr (CG == 1)
    tma_load_2d(dst, map, bar, c0, c1);
  else
    tma_load_2d_pair(dst, map, bar, c0, c1);
}

// One pipeline stage of this CTA: its BM rows of A and its B_ROWS rows of B.
// `bar` is the full barrier of the MMA-issuing CTA (cluster address for CG 2);
// v0 is the first vocabulary column of the unit's slab, doff the first row of
// its D buffer (DH, DW).
template <int MODE, int CG, bool kF8 = false>
__device__ __forceinline__ void load_stage(const CUtensorMap* tA, const CUtensorMap* tB,
                                           const CUtensorMap* tA2, const CUtensorMap* tB2,
                                           uint32_t sA, uint32_t sB, uint32_t bar,
                                           const GemmParams& p, int m, int n, int kb, int rank, int v0,
                                           int doff = 0) {
  using C = TileCfg<CG>;
  // one stage row is 128 bytes of K: 64 bf16 or 128 e4m3 elements
  constexpr int BK = kF8 ? 128 : flce::BK;
  const int a0 = m * C::TM + rank * BM;         // first A row (M) of this CTA
  const int b0 = n * BN + rank * C::B_ROWS;     // first B row (N) of this CTA
  if constexpr (is_kd<MODE>()) {
    // student (h_s, W_s) blocks first, then the teacher's (h_t, W_t)
    const bool teacher = kb >= p.k_blocks_s;
    const int kk = teacher ? kb - p.k_blocks_s : kb;
    tma_ld<MODE, CG>(sA, teacher ? tA2 : tA, bar, kk * BK, p.row0 + a0);
    tma_ld<MODE, CG>(sB, teacher ? tB2 : tB, bar, kk * BK, v0 + b0);
  } else if constexpr (MODE == MODE_FWD || MODE == MODE_FUSED_FWD || MODE == MODE_DLOGITS) {
    // A = h rows (K-major, box 64 x 128), B = W vocabulary rows (K-major, box 64 x B_ROWS)
    tma_ld<MODE, CG>(sA, tA, bar, kb * BK, p.row0 + a0);
    tma_ld<MODE, CG>(sB, tB, bar, kb * BK, v0 + b0);
  } else if constexpr (MODE == MODE_DH) {
    // A = D rows of this chunk (K-major over the slab's vocabulary), B = W
    // with the hidden dimension contiguous (MN-major): 64-wide boxes
    tma_ld<MODE, CG>(sA, tA, bar, kb * BK, doff + a0);
#pragma unroll
    for (int j = 0; j < C::B_ROWS / 64; ++j)
      tma_ld<MODE, CG>(sB + j * MN_BOX_BYTES, tB, bar, b0 + 64 * j, v0 + kb * BK);
  } else if constexpr (MODE == MODE_DH2) {
    // as DH, with the B blocks of tiles 2n and 2n + 1 one after the other
    tma_ld<MODE, CG>(sA, tA, bar, kb * BK, doff + a0);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < C::B_ROWS / 64; ++j)
        tma_ld<MODE, CG>(sB + h * C::B_BYTES + j * MN_BOX_BYTES, tB, bar,
                         (2 * n + h) * BN + rank * C::B_ROWS + 64 * j, v0 + kb * BK);
  } else {
    static_assert(MODE == MODE_DW, "every mode needs its operand loads");
    // A = D^T (vocabulary contiguous: MN-major), B = h (hidden contiguous:
    // MN-major); K runs over the chunk's rows
#pragma unroll
    for (int j = 0; j < 2; ++j) tma_ld<MODE, CG>(sA + j * MN_BOX_BYTES, tA, bar, a0 + 64 * j, doff + kb * BK);
#pragma unroll
    for (int j = 0; j < C::B_ROWS / 64; ++j)
      tma_ld<MODE, CG>(sB + j * MN_BOX_BYTES, tB, bar, b0 + 64 * j, p.row0 + kb * BK);
  }
}

template <int MODE, int CG, bool kF8 = false>
__device__ __forceinline__ void mma_stage(uint32_t d_tmem, uint32_t sA, uint32_t sB, bool first) {
  if constexpr (MODE == MODE_DH2) {
    // the two 256-column tiles of the stage into accumulators d_tmem and d_tmem + BN
    mma_stage<MODE_DH, CG>(d_tmem, sA, sB, first);
    mma_stage<MODE_DH, CG>(d_tmem + BN, sA, sB + TileCfg<CG>::B_BYTES, first);
    return;
  }
  constexpr bool A_MN = (MODE == MODE_DW);
  constexpr bool B_MN = (MODE == MODE_DH || MODE == MODE_DW);
  constexpr uint32_t IDESC = kF8 ? idesc_e4m3_f32(TileCfg<CG>::TM, BN)
                                 : idesc_bf16_f32(TileCfg<CG>::TM, BN, A_MN, B_MN);
  // each instruction consumes 32 bytes of K (16 bf16 or 32 e4m3 elements)
#pragma unroll
  for (int k = 0; k < BK / UMMA_K; ++k) {
    // K-major: 8-row core groups 1024 B apart, K advances 32 B inside the
    // swizzle row.  MN-major: 64-wide MN boxes MN_BOX_BYTES apart, 8-row K
    // groups 1024 B apart, K advances 16 rows = 2048 B.
    const uint64_t ad = A_MN ? smem_desc_sw128(sA + k * 2048, MN_BOX_BYTES, 1024)
                             : smem_desc_sw128(sA + k * 32, 16, 1024);
    const uint64_t bd = B_MN ? smem_desc_sw128(sB + k * 2048, MN_BOX_BYTES, 1024)
                             : smem_desc_sw128(sB + k * 32, 16, 1024);
    const uint32_t acc = (first && k == 0) ? 0u : 1u;
    if constexpr (kF8) {
      if constexpr (CG == 1)
        umma_e4m3(d_tmem, ad, bd, IDESC, acc);
      else
        umma_e4m3_pair(d_tmem, ad, bd, IDESC, acc);
    } else {
      if constexpr (CG == 1)
        umma_bf16(d_tmem, ad, bd, IDESC, acc);
      else
        umma_bf16_pair(d_tmem, ad, bd, IDESC, acc);
    }
  }
}

template <int CG>
__device__ __forceinline__ void mma_commit_all(uint32_t bar) {
  if constexpr (CG == 1)
    umma_commit(bar);
  else
    umma_commit_pair_mc(bar, 0x3);  // the barrier at this offset in both CTAs
}

// v[j] for a run-time j in [0, 32) without dynamic register indexing (which
// would move v to local memory): a 5-level select tree on the bits of j.
__device__ __forceinline__ float select32(const float (&v)[32], int j) {
  float a[16], b[8], c[4], d[2];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = (j & 16) ? v[i + 16] : v[i];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = (j & 8) ? a[i + 8] : a[i];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = (j & 4) ? b[i + 4] : b[i];
#pragma unroll
  for (int i = 0; i < 2; ++i) d[i] = (j & 2) ? c[i + 2] : c[i];
  return (j & 1) ? d[1] : d[0];
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One 32-column chunk of this thread's row (32 bf16 = 64 bytes) into half
// `half` of a 32-row x 64-column bf16 box in 128B-swizzled shared memory
// (row = lane): 16-byte granule g of the row lands at g ^ (row & 7).
__device__ __forceinline__ void stage_bf16_half(uint32_t box, int lane, int half, const uint32_t (&pk)[16]) {
  const uint32_t row_addr = box + lane * 128;
#pragma unroll
  for (int g = 0; g < 4; ++g)
    st_shared_v4_u32(row_addr + (((half * 4 + g) ^ (lane & 7)) << 4), pk[4 * g], pk[4 * g + 1],
                     pk[4 * g + 2], pk[4 * g + 3]);
}

template <int MODE, bool kLong, int CG, bool kF8 = false, int EW = EPI_WARPS>
__global__ void __launch_bounds__(kernel_threads<MODE>(EW), 1)
    flce_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmA2,
                     const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmC2,
                     const __grid_constant__ CUtensorMap tmA3, const __grid_constant__ CUtensorMap tmB3,
                     const __grid_constant__ CUtensorMap tmC3, const __grid_constant__ GemmParams p) {
  using idx_t = typename std::conditional<kLong, long long, int>::type;
  using C = TileCfg<CG>;
  using K = KernelCfg<MODE, CG, EW>;
  constexpr int NST = K::NSTAGE;
  // accumulator buffers in TMEM: two (double-buffered) tiles, or one tile of
  // two accumulators (student, teacher) in the distillation modes
  constexpr int NACC = (is_kd<MODE>() || MODE == MODE_DH2) ? 1 : 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t out_stage = sbase + NST * K::STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NST * K::STAGE + K::OUT_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  // barrier layout: full[NST], empty[NST], tfull[2], tempty[2], drain
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (NST + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * NST + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * NST + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * NST + 4);
  // PIPE: unit ring (full: published by the pair's fetching thread in both
  // CTAs; empty: in the first CTA, one arrival per epilogue warp of the pair)
  auto ufull_bar = [&](int s) { return bar0 + 8u * (2 * NST + 5 + s); };
  auto uempty_bar = [&](int s) { return bar0 + 8u * (2 * NST + 5 + kUnitRing + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * NST + 5 + 2 * kUnitRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* unit_ring = abort_flag + 1;  // kUnitRing unit indices (-1: no more units)
  static_assert((2 * NST + 5 + 2 * kUnitRing) * 8 + 8 + 4 * kUnitRing <= SMEM_BAR_BYTES,
                "barriers exceed their shared-memory area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CG 2: the pair's first CTA (rank 0) issues the MMAs; both CTAs load their
  // half of the operands and drain their half of the accumulator rows.
  const int rank = CG == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  const bool issuer = rank == 0;
  const int worker = blockIdx.x / CG;
  const int nworkers = gridDim.x / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), EW * CG);
    }
    mbar_init(drain, 1);
    if constexpr (MODE == MODE_PIPE) {
      for (int r = 0; r < kUnitRing; ++r) {
        mbar_init(ufull_bar(r), 1);
        mbar_init(uempty_bar(r), EW * CG);
      }
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (is_kd<MODE>() || MODE == MODE_DHDW || MODE == MODE_PIPE) {
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
    }
    if constexpr (MODE == MODE_PIPE) {
      tma_prefetch_desc(&tmA3);
      tma_prefetch_desc(&tmB3);
    }
  }
  if constexpr (CG == 2) cluster_sync();  // peer barriers exist before any remote signal
  if (warp == 1) {
    if constexpr (CG == 1) {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    } else {
      tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above touches only this CTA's shared memory and TMEM, so it
  // may overlap the previous kernel's tail; nothing below reads or writes
  // global memory before that kernel has completed.
  grid_dependency_wait();
  grid_launch_dependents();
  const DynShape dsh = dyn_shape<MODE, C::TM>(p);
  if constexpr (MODE == MODE_PIPE) {
    // the next launch's counters start at zero (the previous launch, which
    // used them, has completed)
    if (p.pp_dep_zero != nullptr)
      for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.pp_dep_words; i += gridDim.x * blockDim.x)
        p.pp_dep_zero[i] = 0u;
  }
  // The k-th unit of this worker, or -1 when it has none left: round-robin
  // over the grid, or (PIPE) taken from the unit ring, whose indices the
  // pair's fetching thread draws from a counter in increasing order.
  auto unit_at = [&](int k) -> int {
    if constexpr (MODE == MODE_PIPE) {
      const int sl = k % kUnitRing;
      if (!wait_bar_cluster(ufull_bar(sl), static_cast<uint32_t>((k / kUnitRing) & 1), abort_flag, p.err))
        return -1;
      return unit_ring[sl];
    } else {
      const int u = worker + k * nworkers;
      return u < dsh.num_units ? u : -1;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int k_unit = 0; ok; ++k_unit) {
        const int u = unit_at(k_unit);
        if (u < 0) break;
        const Unit t = decode_unit<MODE, C::TM>(p, dsh, u);
        if constexpr (MODE == MODE_PIPE) {
          // the fetching thread saw this unit's inputs published; the bulk
          // loads below read them
          fence_proxy_async_global();
        }
        const int uv0 = MODE == MODE_PIPE ? t.slab * p.pp_vs : p.v0;  // the unit's first vocabulary column
        const int udoff = MODE == MODE_PIPE ? (t.slab & 1) * p.rows_cap : 0;  // its D buffer
        for (int n = t.n0; n < t.n1 && ok; ++n) {
          for (int kb = t.kb0; kb < t.kb1; ++kb) {
            if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
              ok = false;
              break;
            }
            const uint32_t sA = sbase + stage * K::STAGE;
            uint32_t fb = full_bar(stage);
            if constexpr (CG == 2) fb = mapa_shared(fb, 0);
            if (issuer) mbar_arrive_expect_tx(full_bar(stage), K::STAGE * CG);
            if constexpr (MODE == MODE_DHDW || MODE == MODE_PIPE) {
              if (t.dw)
                load_stage<MODE_DW, CG>(&tmA2, &tmB2, &tmA2, &tmB2, sA, sA + C::A_BYTES, fb, p, t.m, n, kb,
                                        rank, uv0, udoff);
              else if (MODE == MODE_PIPE && t.kind == KIND_DL)
                load_stage<MODE_DLOGITS, CG>(&tmA3, &tmB3, &tmA3, &tmB3, sA, sA + C::A_BYTES, fb, p, t.m, n,
                                             kb, rank, uv0);
              else
                load_stage<MODE_DH, CG>(&tmA, &tmB, &tmA, &tmB, sA, sA + C::A_BYTES, fb, p, t.m, n, kb, rank,
                                        uv0, udoff);
            } else {
              load_stage<MODE, CG, kF8>(&tmA, &tmB, &tmA2, &tmB2, sA, sA + C::A_BYTES, fb, p, t.m, n, kb,
                                        rank, uv0);
            }
            ++issued;
            if (++stage == NST) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // no copy into shared memory may still be in flight when the CTA
      // retires: the issuing CTA's full barriers count both CTAs' bytes
      if (issuer)
        for (long long i = (issued > NST ? issued - NST : 0); i < issued; ++i)
          drain_bar(full_bar(static_cast<int>(i % NST)), static_cast<uint32_t>((i / NST) & 1), p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && issuer) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int k_unit = 0; ok; ++k_unit) {
        const int u = unit_at(k_unit);
        if (u < 0) break;
        const Unit t = decode_unit<MODE, C::TM>(p, dsh, u);
        for (int n = t.n0; n < t.n1 && ok; ++n) {
          if (!wait_bar(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          for (int kb = t.kb0; kb < t.kb1; ++kb) {
            if (!wait_bar(full_bar(stage), phase, abort_flag, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sA = sbase + stage * K::STAGE;
            if constexpr (is_kd<MODE>()) {
              const bool teacher = kb >= p.k_blocks_s;
              mma_stage<MODE, CG>(d_tmem + (teacher ? BN : 0), sA, sA + C::A_BYTES,
                                  kb == t.kb0 || kb == p.k_blocks_s);
            } else if constexpr (MODE == MODE_DHDW || MODE == MODE_PIPE) {
              if (t.dw)
                mma_stage<MODE_DW, CG>(d_tmem, sA, sA + C::A_BYTES, kb == t.kb0);
              else if (MODE == MODE_PIPE && t.kind == KIND_DL)
                mma_stage<MODE_DLOGITS, CG>(d_tmem, sA, sA + C::A_BYTES, kb == t.kb0);
              else
                mma_stage<MODE_DH, CG>(d_tmem, sA, sA + C::A_BYTES, kb == t.kb0);
            } else {
              mma_stage<MODE, CG, kF8>(d_tmem, sA, sA + C::A_BYTES, kb == t.kb0);
            }
            mma_commit_all<CG>(empty_bar(stage));
            if (++stage == NST) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_all<CG>(tfull_bar(acc));
          if (++acc == NACC) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
      }
      // every MMA issued by this thread has finished before TMEM is freed
      if constexpr (CG == 1)
        umma_commit(drain);
      else
        umma_commit_pair(drain);
      drain_bar(drain, 0, p.err);
    }
    __syncwarp();
  } else if (MODE == MODE_PIPE && warp == 2 + EW) {
    // ------------------------------------------------------------ fetching
    // (PIPE; the pair's first CTA) draws unit indices in increasing order
    // from the launch's counter, waits until the units whose output each one
    // reads or overwrites are counted, and publishes it in both CTAs' unit
    // rings; -1 ends the loops.  Every unit waits only on lower indices,
    // which running workers have drawn, so the launch completes whichever of
    // its CTAs are resident.
    if constexpr (MODE == MODE_PIPE) {
      if (lane == 0 && issuer) {
        unsigned* counter = p.pp_dep + p.pp_dep_words - 1;
        const int ahead = min(max(p.pp_lookahead, 1), kUnitRing);
        for (int k = 0;; ++k) {
          const int sl = k % kUnitRing;
          // unit k - ahead finished (so its slot, and unit k - kUnitRing's, is free)
          const int j = k - ahead;
          if (j >= 0 && !wait_bar_cluster(uempty_bar(j % kUnitRing), static_cast<uint32_t>((j / kUnitRing) & 1),
                                          abort_flag, p.err))
            break;
          int u = static_cast<int>(atomicAdd(counter, 1u));
          if (u >= dsh.num_units) u = -1;
          if (u >= 0 && !pipe_wait_deps<C::TM, EW * CG>(p, dsh, decode_unit<MODE, C::TM>(p, dsh, u), abort_flag))
            u = -1;
          for (int r = 0; r < CG; ++r) {
            const uint32_t ring_r = CG == 2 ? mapa_shared(smem_u32(const_cast<int*>(unit_ring + sl)), r)
                                            : smem_u32(const_cast<int*>(unit_ring + sl));
            const uint32_t full_r = CG == 2 ? mapa_shared(ufull_bar(sl), r) : ufull_bar(sl);
            st_shared_cluster_u32(ring_r, static_cast<uint32_t>(u));
            mbar_arrive_cluster(full_r);
          }
          if (u < 0) break;
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;       // accumulator row owned by this thread
    // columns of the tile this warp takes: all, or one half (8 epilogue warps)
    static_assert(EW == EPI_WARPS || (EW == 2 * EPI_WARPS && wide_epilogue_mode<MODE>()) ||
                      (EW == 4 * EPI_WARPS && MODE == MODE_DW),
                  "8 epilogue warps: dW, DHDW, the two-head dlogits and the Jensen-Shannon terms; "
                  "16: dW only");
    constexpr int kColParts = EW / 4;
    constexpr int kChunks = K::TILE_N / 32 / kColParts;
    const int c_lo = ((warp - 2) / 4) * kChunks;
    // TMA staging boxes of this warp (KernelCfg: 8 boxes shared by 4 or 8
    // warps, or one per warp of 16)
    constexpr int kBoxes = K::BOXES_PER_WARP;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t tempty_target0 = CG == 2 ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
    const uint32_t tempty_target1 = CG == 2 ? mapa_shared(tempty_bar(1), 0) : tempty_bar(1);
    uint32_t acc = 0, acc_phase = 0;
    bool ok = true;
    for (int k_unit = 0; ok; ++k_unit) {
      int u = 0;
      if (lane == 0) u = unit_at(k_unit);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u < 0) break;
      const Unit t = decode_unit<MODE, C::TM>(p, dsh, u);
      // PIPE: the unit's kind (else the mode's) and its slab's first column
      const bool unit_dl = MODE == MODE_DLOGITS || (MODE == MODE_PIPE && t.kind == KIND_DL);
      const int uv0 = MODE == MODE_PIPE ? t.slab * p.pp_vs : p.v0;
      const int udoff = MODE == MODE_PIPE ? (t.slab & 1) * p.rows_cap : 0;  // D buffer of the slab
      // per-unit row state
      const int lr = t.m * C::TM + rank * BM + r;  // row inside this pass (original row: grow)
      bool row_ok;
      long long tgt = -1;
      float run_m = -INFINITY, run_s = 0.f;  // FWD: log2-domain max and sum
      float run_mt = -INFINITY, run_st = 0.f, run_c = 0.f;  // KD_FWD teacher state
      float jsd_t = 0.f, jsd_s = 0.f, klsm = 0.f;            // JSD: mixture terms (log2 units)
      float scale = 0.f, nl2 = 0.f, nlt = 0.f;              // DLOGITS / KD_DLOGITS
      // linear transform folded into the exp2 prescale, the gathered target
      // logit and the dlogits scale (soft-capped logits are formed explicitly)
      const float lin_a = p.tf_softcap ? 1.f : p.tf_a;
      const float l2a = kLog2e * lin_a;
      // DHDW: this unit's kind (a DW unit's accumulator rows are vocabulary rows)
      const bool unit_dw = MODE == MODE_DW || ((MODE == MODE_DHDW || MODE == MODE_PIPE) && t.dw);
      if (unit_dw) {
        row_ok = lr < p.V;  // rows of the accumulator are vocabulary rows here
      } else {
        row_ok = lr < dsh.rows;
      }
      // original row of this accumulator row (targets, weights, lse, dH;
      // the forward modes' partials and target logit)
      int grow = p.row0 + lr;
      if constexpr (rows_are_tokens<MODE>() || MODE == MODE_DHDW || MODE == MODE_PIPE) {
        if (!unit_dw && p.row_idx != nullptr) grow = row_ok ? p.row_idx[p.chunk_first + lr] : 0;
      }
      // DLOGITS also writes zero rows up to the next 64-row K block so that
      // the dW pass over this chunk reads zeros past its last row
      const bool row_store = lr < min((dsh.rows + BK - 1) / BK * BK, p.rows_cap);
      float a_sc = 1.f;  // e4m3 forward: this row's dequantisation scale
      if constexpr (MODE == MODE_FWD || MODE == MODE_FUSED_FWD) {
        if (row_ok) tgt = p.targets[grow];
        if constexpr (kF8) {
          if (row_ok) a_sc = p.a_scale[grow];
        }
      }
      if (unit_dl) {
        if (row_ok) {
          tgt = p.targets[grow];
          const bool valid = tgt != p.ignore_index;
          const float w = p.weights ? p.weights[grow] : 1.f;
          scale = valid ? w * device_grad_scale(p) : 0.f;
          nl2 = -p.lse[grow] * kLog2e;
        }
      }
      if constexpr (MODE == MODE_KD_DLOGITS || MODE == MODE_JSD_DLOGITS) {
        if (row_ok) {
          const bool valid = p.targets == nullptr || p.targets[grow] != p.ignore_index;
          const float w = p.weights ? p.weights[grow] : 1.f;
          scale = valid ? w * device_grad_scale(p) : 0.f;
          nl2 = -p.lse[grow] * kLog2e;
          nlt = -p.lse_t[grow] * kLog2e;
          if constexpr (MODE == MODE_JSD_DLOGITS) klsm = p.kl_sm[grow];
        }
      }
      if constexpr (MODE == MODE_JSD_FWD) {
        if (row_ok) {
          nl2 = -p.lse[grow] * kLog2e;
          nlt = -p.lse_t[grow] * kLog2e;
        }
      }
      const float scale_a = scale * lin_a;
      for (int n = t.n0; n < t.n1; ++n) {
        int got = 0;
        if (lane == 0) got = wait_bar(tfull_bar(acc), acc_phase, abort_flag, p.err) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem_base + lane_addr + acc * BN;
#pragma unroll 1
        for (int c = c_lo; c < c_lo + kChunks; ++c) {
          float v[32];
          if (t.kb1 > t.kb0) {
            tmem_ld32(tbase + c * 32, v);
          } else {  // empty K range (a compacted pass without rows): the product is zero
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
          }
          const int col0 = n * K::TILE_N + c * 32;
          if constexpr (MODE == MODE_FWD || MODE == MODE_FUSED_FWD) {
            if constexpr (kF8) {  // dequantise: row scale x per-vocabulary-row scale
              if (col0 + 32 <= p.V) {
                const float4* bs = reinterpret_cast<const float4*>(p.b_scale + col0);
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {
                  const float4 s4 = __ldg(bs + g4);
                  v[4 * g4] *= a_sc * s4.x;
                  v[4 * g4 + 1] *= a_sc * s4.y;
                  v[4 * g4 + 2] *= a_sc * s4.z;
                  v[4 * g4 + 3] *= a_sc * s4.w;
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  v[j] *= (col0 + j < p.V) ? a_sc * __ldg(p.b_scale + col0 + j) : 0.f;
              }
            }
            if (p.tf_softcap) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = p.tf_b * tanhf(p.tf_a * v[j]);
            }
            if (col0 + 32 > p.V) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j >= p.V) v[j] = -INFINITY;
            }
            float cm = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) cm = fmaxf(cm, v[j]);
            const float nm = fmaxf(run_m, cm * l2a);
            if (nm != -INFINITY) {
              float a = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) a += ex2_approx(fmaf(v[j], l2a, -nm));
              run_s = run_s * ex2_approx(run_m - nm) + a;
              run_m = nm;
            }
            if constexpr (MODE == MODE_FUSED_FWD) {
              // 2^(u log2e - chunk max) in [0, 1] as bf16, and the chunk max,
              // for the dlogits pass once the row's lse is known (an ignored
              // row's dlogits are zero: the pass does not read them)
              if (row_ok && tgt != p.ignore_index) {
                const float cmL = cm * l2a;
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                  const float e0 = cm == -INFINITY ? 0.f : ex2_approx(fmaf(v[j], l2a, -cmL));
                  const float e1 = cm == -INFINITY ? 0.f : ex2_approx(fmaf(v[j + 1], l2a, -cmL));
                  pk[j / 2] = pack_bf16x2(e0, e1);
                }
                uint16_t* dst = p.D + static_cast<idx_t>(lr) * p.ldD + col0;
#pragma unroll
                for (int g = 0; g < 4; ++g)
                  if (col0 + 8 * g < p.ldD)
                    *reinterpret_cast<uint4*>(dst + 8 * g) =
                        make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
                if (col0 < p.ldD) p.mx[static_cast<idx_t>(lr) * (p.ldD / 32) + col0 / 32] = cmL;
              }
            }
            const long long tj = tgt - col0;
            if (tj >= 0 && tj < 32 && tgt < p.V) {
              const float z = select32(v, static_cast<int>(tj)) * lin_a;
              if (row_ok) p.zt[grow] = z;
            }
          } else if (unit_dl) {
            uint32_t pk[16];
            const int gcol0 = uv0 + col0;  // vocabulary column of D's local column col0
            const long long tjl = tgt - gcol0;
            const int tj = (tjl >= 0 && tjl < 32) ? static_cast<int>(tjl) : -1;
            if (!p.tf_softcap && tj < 0 && gcol0 + 32 <= p.V) {
              // the common chunk: no target column, inside the vocabulary
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                float d0 = 0.f, d1 = 0.f;
                if (scale != 0.f) {
                  d0 = ex2_approx(fmaf(v[j], l2a, nl2)) * scale_a;
                  d1 = ex2_approx(fmaf(v[j + 1], l2a, nl2)) * scale_a;
                }
                pk[j / 2] = pack_bf16x2(d0, d1);
              }
            } else if (!p.tf_softcap) {
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                float d0 = 0.f, d1 = 0.f;
                if (scale != 0.f) {
                  float p0 = ex2_approx(fmaf(v[j], l2a, nl2));
                  float p1 = ex2_approx(fmaf(v[j + 1], l2a, nl2));
                  if (j == tj) p0 -= 1.f;
                  if (j + 1 == tj) p1 -= 1.f;
                  d0 = (gcol0 + j < p.V) ? p0 * scale_a : 0.f;
                  d1 = (gcol0 + j + 1 < p.V) ? p1 * scale_a : 0.f;
                }
                pk[j / 2] = pack_bf16x2(d0, d1);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                float d0 = 0.f, d1 = 0.f;
                if (scale != 0.f) {
                  const float t0 = tanhf(p.tf_a * v[j]);
                  const float t1 = tanhf(p.tf_a * v[j + 1]);
                  float p0 = ex2_approx(fmaf(p.tf_b * t0, kLog2e, nl2));
                  float p1 = ex2_approx(fmaf(p.tf_b * t1, kLog2e, nl2));
                  if (j == tj) p0 -= 1.f;
                  if (j + 1 == tj) p1 -= 1.f;
                  d0 = (gcol0 + j < p.V) ? p0 * scale * p.tf_d * (1.f - t0 * t0) : 0.f;
                  d1 = (gcol0 + j + 1 < p.V) ? p1 * scale * p.tf_d * (1.f - t1 * t1) : 0.f;
                }
                pk[j / 2] = pack_bf16x2(d0, d1);
              }
            }
            if (p.d_tma) {
              // two chunks fill one 32 x 64 box; TMA writes it (rows of the
              // box past the live rows hold zeros: their scale is 0)
              const int half = c & 1;
              const uint32_t box = out_stage + (warp - 2) * (2 * OUT_BOX_BYTES) + ((c >> 1) & 1) * OUT_BOX_BYTES;
              if (half == 0) {
                if (lane == 0) bulk_wait_read<1>();  // the copy that last used this box has read it
                __syncwarp();
              }
              stage_bf16_half(box, lane, half, pk);
              if (half == 1) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  const int lrow0 = t.m * C::TM + rank * BM + q * 32;
                  const int x = col0 - 32;  // first column of the box
                  if (x < p.ldD && lrow0 < p.rows_cap)
                    tma_store_2d(MODE == MODE_PIPE ? &tmC3 : &tmC, box, x, udoff + lrow0);
                  bulk_commit();
                }
              }
            } else if (row_store) {
              uint16_t* dst = p.D + static_cast<idx_t>(lr) * p.ldD + col0;
#pragma unroll
              for (int g = 0; g < 4; ++g)
                if (col0 + 8 * g < p.ldD)
                  *reinterpret_cast<uint4*>(dst + 8 * g) =
                      make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
            }
          } else if constexpr (MODE == MODE_KD_FWD) {
            float vt[32];
            tmem_ld32(tbase + BN + c * 32, vt);
            if (p.tf_softcap) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                v[j] = p.tf_b * tanhf(p.tf_a * v[j]);
                vt[j] = p.tf_b * tanhf(p.tf_a * vt[j]);
              }
            }
            const bool partial = col0 + 32 > p.V;
            if (partial) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j >= p.V) {
                  v[j] = -INFINITY;
                  vt[j] = -INFINITY;
                }
            }
            // student: online log-sum-exp (log2 domain)
            float cm = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) cm = fmaxf(cm, v[j]);
            const float nm = fmaxf(run_m, cm * l2a);
            if (nm != -INFINITY) {
              float a = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) a += ex2_approx(fmaf(v[j], l2a, -nm));
              run_s = run_s * ex2_approx(run_m - nm) + a;
              run_m = nm;
            }
            // teacher: online log-sum-exp and sum of 2^(u_t - m_t) (z_t - z_s)
            float ct = vt[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) ct = fmaxf(ct, vt[j]);
            const float nt = fmaxf(run_mt, ct * l2a);
            if (nt != -INFINITY) {
              float a = 0.f, cc = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float e = ex2_approx(fmaf(vt[j], l2a, -nt));
                a += e;
                if (!partial || col0 + j < p.V) cc += e * (vt[j] - v[j]);
              }
              const float rs = ex2_approx(run_mt - nt);
              run_st = run_st * rs + a;
              run_c = run_c * rs + cc * lin_a;
              run_mt = nt;
            }
          } else if constexpr (MODE == MODE_KD_DLOGITS) {
            float vt[32];
            tmem_ld32(tbase + BN + c * 32, vt);
            uint32_t pk[16];
            const int gcol0 = p.v0 + col0;
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float d[2] = {0.f, 0.f};
              if (scale != 0.f) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  float de;
                  if (!p.tf_softcap) {
                    const float ps = ex2_approx(fmaf(v[j + e], l2a, nl2));
                    const float pt = ex2_approx(fmaf(vt[j + e], l2a, nlt));
                    de = (ps - pt) * scale_a;
                  } else {
                    const float ts = tanhf(p.tf_a * v[j + e]);
                    const float ps = ex2_approx(fmaf(p.tf_b * ts, kLog2e, nl2));
                    const float pt = ex2_approx(fmaf(p.tf_b * tanhf(p.tf_a * vt[j + e]), kLog2e, nlt));
                    de = (ps - pt) * scale * p.tf_d * (1.f - ts * ts);
                  }
                  d[e] = (gcol0 + j + e < p.V) ? de : 0.f;
                }
              }
              pk[j / 2] = pack_bf16x2(d[0], d[1]);
            }
            if (row_store) {
              uint16_t* dst = p.D + static_cast<idx_t>(lr) * p.ldD + col0;
#pragma unroll
              for (int g = 0; g < 4; ++g)
                if (col0 + 8 * g < p.ldD)
                  *reinterpret_cast<uint4*>(dst + 8 * g) =
                      make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
            }
          } else if constexpr (MODE == MODE_JSD_FWD) {
            // per row: sum p_t (log2 p_t - log2 M) and sum p_s (log2 p_s - log2 M)
            // with M = beta p_t + (1 - beta) p_s, given both heads' lse
            float vt[32];
            tmem_ld32(tbase + BN + c * 32, vt);
            if (p.tf_softcap) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                v[j] = p.tf_b * tanhf(p.tf_a * v[j]);
                vt[j] = p.tf_b * tanhf(p.tf_a * vt[j]);
              }
            }
            if (row_ok) {
              const int gcol0 = p.v0 + col0;
              float at = 0.f, as = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float ls2 = fmaf(v[j], l2a, nl2);
                const float lt2 = fmaf(vt[j], l2a, nlt);
                const float ps = ex2_approx(ls2);
                const float pt = ex2_approx(lt2);
                const float mix = fmaf(p.jsd_beta, pt - ps, ps);
                // below 1e-37 both probabilities are negligible (each is at
                // most M / min(beta, 1 - beta)); past V there is no column
                if (mix > 1e-37f && gcol0 + j < p.V) {
                  const float lm2 = __log2f(mix);
                  at = fmaf(pt, lt2 - lm2, at);
                  as = fmaf(ps, ls2 - lm2, as);
                }
              }
              jsd_t += at;
              jsd_s += as;
            }
          } else if constexpr (MODE == MODE_JSD_DLOGITS) {
            // D = (1 - beta) p_s (ln(p_s / M) - KL(p_s || M)) m w g f'(z_s)
            float vt[32];
            tmem_ld32(tbase + BN + c * 32, vt);
            uint32_t pk[16];
            const int gcol0 = p.v0 + col0;
            const float omb = 1.f - p.jsd_beta;
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float d[2] = {0.f, 0.f};
              if (scale != 0.f) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  float ls2, lt2, fd;
                  if (!p.tf_softcap) {
                    ls2 = fmaf(v[j + e], l2a, nl2);
                    lt2 = fmaf(vt[j + e], l2a, nlt);
                    fd = scale_a;
                  } else {
                    const float ts = tanhf(p.tf_a * v[j + e]);
                    ls2 = fmaf(p.tf_b * ts, kLog2e, nl2);
                    lt2 = fmaf(p.tf_b * tanhf(p.tf_a * vt[j + e]), kLog2e, nlt);
                    fd = scale * p.tf_d * (1.f - ts * ts);
                  }
                  const float ps = ex2_approx(ls2);
                  const float pt = ex2_approx(lt2);
                  const float mix = fmaf(p.jsd_beta, pt - ps, ps);
                  float de = 0.f;
                  if (mix > 1e-37f && ps > 0.f)
                    de = omb * ps * (fmaf(ls2 - __log2f(mix), kLn2f, -klsm)) * fd;
                  d[e] = (gcol0 + j + e < p.V) ? de : 0.f;
                }
              }
              pk[j / 2] = pack_bf16x2(d[0], d[1]);
            }
            if (row_store) {
              uint16_t* dst = p.D + static_cast<idx_t>(lr) * p.ldD + col0;
#pragma unroll
              for (int g = 0; g < 4; ++g)
                if (col0 + 8 * g < p.ldD)
                  *reinterpret_cast<uint4*>(dst + 8 * g) =
                      make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
            }
          } else if ((MODE == MODE_DH || MODE == MODE_DH2 || (MODE == MODE_DHDW && !unit_dw)) &&
                     p.dH_part == nullptr) {
            if (row_ok) {  // the only pass over this row: bf16 dH directly
              uint16_t* dst = p.dH + static_cast<idx_t>(grow) * p.H + col0;
#pragma unroll
              for (int g = 0; g < 4; ++g)
                if (col0 + 8 * g < p.H)
                  *reinterpret_cast<uint4*>(dst + 8 * g) = make_uint4(
                      pack_bf16x2(v[8 * g], v[8 * g + 1]), pack_bf16x2(v[8 * g + 2], v[8 * g + 3]),
                      pack_bf16x2(v[8 * g + 4], v[8 * g + 5]), pack_bf16x2(v[8 * g + 6], v[8 * g + 7]));
            }
          } else {  // MODE_DW, or MODE_DH into fp32 partials (DHDW: either unit kind)
            // stage this warp's 32 x 32 box (row = lane) in 128B-swizzled
            // shared memory, then one lane hands it to TMA: a plain store on
            // the first pass over the output, an fp32 reduce-add in L2
            // afterwards.  Columns past H and dW rows past V are clipped by
            // TMA; boxes wholly outside the output are skipped.
            const uint32_t box = out_stage + (warp - 2) * (kBoxes * OUT_BOX_BYTES) + (c % kBoxes) * OUT_BOX_BYTES;
            if (lane == 0) bulk_wait_read<kBoxes - 1>();  // the copy that last used this box has read it
            __syncwarp();
            const uint32_t row_addr = box + lane * 128;
#pragma unroll
            for (int g = 0; g < 8; ++g)
              st_shared_v4(row_addr + ((g ^ (lane & 7)) << 4), v[4 * g], v[4 * g + 1], v[4 * g + 2],
                           v[4 * g + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int lrow0 = t.m * C::TM + rank * BM + q * 32;  // first accumulator row of the box
              int oy;
              bool inside, accumulate;
              if (unit_dw) {
                oy = uv0 + lrow0;  // vocabulary row of dW
                inside = oy < p.V;
                accumulate = p.dW_accumulate != 0;
              } else {
                // partial sums of k-split t.split: rows [split * rows_cap, +rows_cap)
                oy = t.split * p.rows_cap + lrow0;
                inside = lrow0 < p.rows_cap;
                // PIPE: a plain store on the block's first slab
                accumulate = MODE == MODE_PIPE ? t.slab > 0 : p.dh_accumulate != 0;
              }
              // DHDW: dW goes through tmC2, the dH partials through tmC
              const CUtensorMap* omap = ((MODE == MODE_DHDW || MODE == MODE_PIPE) && unit_dw) ? &tmC2 : &tmC;
              if (col0 < p.H && inside) {
                if (accumulate)
                  tma_reduce_add_2d(omap, box, col0, oy);
                else
                  tma_store_2d(omap, box, col0, oy);
              }
              bulk_commit();
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CG == 1)
            mbar_arrive(acc ? tempty_target1 : tempty_target0);
          else
            mbar_arrive_cluster(acc ? tempty_target1 : tempty_target0);
        }
        if (++acc == NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if constexpr (MODE == MODE_PIPE) {
        // this warp's boxes of the unit are in global memory before it
        // counts them (each epilogue warp of each CTA counts once)
        if (ok && lane == 0) {
          bulk_wait_all();
          fence_proxy_async_global();
          pipe_signal<C::TM>(p, t);
          // the unit's ring slot may take the next unit (the first CTA counts)
          const uint32_t ue = uempty_bar(k_unit % kUnitRing);
          if constexpr (CG == 1)
            mbar_arrive(ue);
          else
            mbar_arrive_cluster(mapa_shared(ue, 0));
        }
        __syncwarp();
      }
      if constexpr (MODE == MODE_FWD || MODE == MODE_FUSED_FWD) {
        if (ok && row_ok)
          p.partials[static_cast<idx_t>(t.split) * p.N + grow] = make_float2(run_m, run_s);
      }
      // the two-head forwards: the partial slot of this split and column part
      // (8 epilogue warps: the Jensen-Shannon terms only)
      const int slot = t.split * kColParts + (warp - 2) / 4;
      if constexpr (MODE == MODE_JSD_FWD) {
        if (ok && row_ok) p.partials[static_cast<idx_t>(slot) * p.N + grow] = make_float2(jsd_t, jsd_s);
      }
      if constexpr (MODE == MODE_KD_FWD) {
        if (ok && row_ok) {
          const idx_t o = static_cast<idx_t>(slot) * p.N + grow;
          p.partials[o] = make_float2(run_m, run_s);
          p.partials_t[o] = make_float2(run_mt, run_st);
          p.partials_c[o] = run_c;
        }
      }
    }
  }

  if constexpr (MODE == MODE_DW || MODE == MODE_DH || MODE == MODE_DH2 || MODE == MODE_DHDW || MODE == MODE_DLOGITS ||
                MODE == MODE_PIPE) {
    if (warp >= 2 && lane == 0) bulk_wait_all();  // output boxes written before the CTA retires
  }
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // neither CTA retires while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 1)
      tmem_dealloc(tmem_base, TMEM_COLS);
    else
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace flce
