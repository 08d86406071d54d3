// libflce host side: argument checks, TMA tensor maps, persistent GEMM
// launches (clusters, programmatic dependent launch), run-time switches,
// workspaces, and the stages the entry points share (dH / dW of a slab, the
// split-K dH reduction, the forward's combine and loss).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cstdlib>

#include "flce.h"
#include "plan.cuh"

namespace {

using namespace flce;

bool sizes_ok(long long N, long long H, long long V) {
  return N >= 0 && H > 0 && V > 0 && N < INT_MAX && H < INT_MAX && V < INT_MAX;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// --------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map: `inner` contiguous elements per row, `outer` rows of `ld_elems`
// elements; box box_inner x box_outer with 128-byte swizzle; out-of-range
// elements read as zero (loads) or are skipped (stores).
bool make_map_t(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, long long inner,
                long long outer, long long ld_elems, int box_inner, int box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_elems) * esize};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* m, const void* base, long long inner, long long outer, long long ld_elems,
              int box_inner, int box_outer) {
  return make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, ld_elems, box_inner,
                    box_outer);
}

// Programmatic dependent launch of the GEMMs (default; FLCE_OPT_PDL = 0 turns
// it off): a GEMM may be scheduled while the previous kernel of the stream
// drains, runs its prologue (barriers, TMEM, descriptor prefetch) and then
// waits in griddepcontrol.wait until that kernel has completed.  Each GEMM
// grid fits on the GPU at once, so the waiting CTAs never hold SMs that the
// kernel they wait for still needs.
bool pdl_on() { return opt_on(FLCE_OPT_PDL); }

// The two-head dlogits GEMMs and the Jensen-Shannon forward terms
// (distillation) run 8 epilogue warps (default; FLCE_OPT_WIDE_EPILOGUE = 0
// keeps 4): their tile fills TMEM, so the epilogue does not overlap the next tile's
// MMAs and its length adds to each tile's.
bool wide_epilogue_on() { return opt_on(FLCE_OPT_WIDE_EPILOGUE); }

// Launch on `grid` CTAs in clusters of `cluster` with the GEMMs' attributes.
template <class Kern, class... Args>
cudaError_t launch_persistent(Kern k, int grid, int cluster, int threads, int smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl_on()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The operand / output maps of one launch: (a, b, c) for every mode, (a2, b2,
// c2) for the second operand set of the two-head and DHDW modes, (a3, b3, c3)
// for the DLOGITS units of PIPE.  Unused ones repeat (a, b, c).
struct Maps {
  const CUtensorMap *a, *b, *c, *a2, *b2, *c2, *a3, *b3, *c3;
};

// Workers a GEMM launch starts: `workers`, or FLCE_OPT_GRID_WORKERS when set.
// Units are dealt round-robin or drawn from a counter, never tied to a
// particular worker, so any count computes the same result.
int grid_workers(int workers) {
  const int64_t g = opt(FLCE_OPT_GRID_WORKERS);
  return g > 0 ? static_cast<int>(g) : workers;
}

template <int MODE, bool kLong, int CG, int EW = EPI_WARPS>
cudaError_t launch_gemm_t(const Maps& m, const GemmParams& p, int workers, cudaStream_t st) {
  auto k = flce_gemm_kernel<MODE, kLong, CG, false, EW>;
  constexpr int smem = KernelCfg<MODE, CG, EW>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_persistent(k, CG * grid_workers(workers), CG, kernel_threads<MODE>(EW), smem, st, *m.a, *m.b, *m.c,
                           *m.a2, *m.b2, *m.c2, *m.a3, *m.b3, *m.c3, p);
}


// The epilogue width (4, 8 or 16 warps) and CTA group of one launch of MODE.
template <int MODE>
cudaError_t launch_gemm_maps(int cg, bool kLong, const Maps& mp, const GemmParams& p, int workers,
                             cudaStream_t st) {
  if constexpr (MODE == MODE_DH2) {  // SM pairs only
    (void)cg;
    return kLong ? launch_gemm_t<MODE, true, 2>(mp, p, workers, st)
                 : launch_gemm_t<MODE, false, 2>(mp, p, workers, st);
  }
  if constexpr (wide_epilogue_mode<MODE>()) {
    // the Jensen-Shannon forward's caller sized the partials for the column
    // parts it chose
    const bool wide = MODE == MODE_DW         ? p.k_blocks <= kDwWideEpilogueMaxKBlocks
                      : MODE == MODE_DHDW    ? p.dw_k_blocks <= kDwWideEpilogueMaxKBlocks
                      : MODE == MODE_JSD_FWD ? p.col_parts == 2
                                             : wide_epilogue_on();
    if constexpr (MODE == MODE_DW) {
      // short K: 16 epilogue warps (default; FLCE_OPT_DW_EPILOGUE_WARPS = 8
      // keeps 8)
      if (wide && opt(FLCE_OPT_DW_EPILOGUE_WARPS) == 16) {
        constexpr int EW = 4 * EPI_WARPS;
        if (cg == 2)
          return kLong ? launch_gemm_t<MODE, true, 2, EW>(mp, p, workers, st)
                       : launch_gemm_t<MODE, false, 2, EW>(mp, p, workers, st);
        return kLong ? launch_gemm_t<MODE, true, 1, EW>(mp, p, workers, st)
                     : launch_gemm_t<MODE, false, 1, EW>(mp, p, workers, st);
      }
    }
    if (wide) {
      constexpr int EW = 2 * EPI_WARPS;
      if (cg == 2)
        return kLong ? launch_gemm_t<MODE, true, 2, EW>(mp, p, workers, st)
                     : launch_gemm_t<MODE, false, 2, EW>(mp, p, workers, st);
      return kLong ? launch_gemm_t<MODE, true, 1, EW>(mp, p, workers, st)
                   : launch_gemm_t<MODE, false, 1, EW>(mp, p, workers, st);
    }
  }
  if constexpr (MODE != MODE_DH2) {
    if (cg == 2)
      return kLong ? launch_gemm_t<MODE, true, 2>(mp, p, workers, st)
                   : launch_gemm_t<MODE, false, 2>(mp, p, workers, st);
    return kLong ? launch_gemm_t<MODE, true, 1>(mp, p, workers, st)
                 : launch_gemm_t<MODE, false, 1>(mp, p, workers, st);
  }
}

// `workers`: CTAs (cg 1) or CTA pairs (cg 2), each running one persistent
// tile loop.  `c` is the output map of the modes that write through TMA (dW,
// dH partials, dlogits); the other modes ignore it.
template <int MODE>
cudaError_t launch_gemm(int cg, bool kLong, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const GemmParams& p, int workers, cudaStream_t st,
                        const CUtensorMap* a2 = nullptr, const CUtensorMap* b2 = nullptr,
                        const CUtensorMap* c2 = nullptr, const CUtensorMap* a3 = nullptr,
                        const CUtensorMap* b3 = nullptr, const CUtensorMap* c3 = nullptr) {
  // a2 / b2: the teacher's operands of the distillation modes, or the DW
  // units' operands of DHDW and PIPE, whose dW output map is c2; a3 / b3 /
  // c3: the DLOGITS units' operands and D output of PIPE (else unused)
  const Maps mp{&a, &b, &c, a2 ? a2 : &a, b2 ? b2 : &b, c2 ? c2 : &c, a3 ? a3 : &a, b3 ? b3 : &b,
                c3 ? c3 : &c};
  return launch_gemm_maps<MODE>(cg, kLong, mp, p, workers, st);
}

// The e4m3 forward: MODE_FWD with 8-bit operands.
cudaError_t launch_fwd_e4m3(int cg, bool kLong, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int workers, cudaStream_t st) {
  auto go = [&](auto kern, int smem, int grid_mult) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_persistent(kern, grid_mult * grid_workers(workers), grid_mult, gemm_threads(EPI_WARPS), smem, st,
                             a, b, b, a, b, b, a, b, b, p);
  };
  if (cg == 2)
    return kLong ? go(flce_gemm_kernel<MODE_FWD, true, 2, true>, TileCfg<2>::SMEM, 2)
                 : go(flce_gemm_kernel<MODE_FWD, false, 2, true>, TileCfg<2>::SMEM, 2);
  return kLong ? go(flce_gemm_kernel<MODE_FWD, true, 1, true>, TileCfg<1>::SMEM, 1)
               : go(flce_gemm_kernel<MODE_FWD, false, 1, true>, TileCfg<1>::SMEM, 1);
}

// CTA group of the GEMMs: 2 (SM pairs, 256-row tiles) unless
// FLCE_OPT_CTA_GROUP = 1.
int cta_group() { return opt(FLCE_OPT_CTA_GROUP) == 1 ? 1 : 2; }

// Persistent workers the GPU holds at once: CTAs, or co-resident CTA pairs.
int device_workers(int cg) {
  const int sms = device_sms();
  if (cg == 1) return sms;
  static int cached_dev = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return sms / 2;
  }
  if (dev == cached_dev && cached > 0) return cached;
  int n = 0;
  auto k = flce_gemm_kernel<MODE_FWD, false, 2>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(gemm_threads(EPI_WARPS), 1, 1);
  cfg.dynamicSmemBytes = TileCfg<2>::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, TileCfg<2>::SMEM) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  cached_dev = dev;
  cached = n;
  return n;
}

// A slab's dH and dW GEMMs in one launch when the plan has several slabs
// (default); FLCE_OPT_FUSE_DH_DW = 0 always launches them one after the other.
bool fuse_dh_dw_on() { return opt_on(FLCE_OPT_FUSE_DH_DW); }

// A backward of several vocabulary slabs runs each row block as one
// MODE_PIPE launch (default); FLCE_OPT_PIPELINE = 0 launches a slab's
// dlogits GEMM and its dH / dW GEMMs one after the other.
bool pipeline_on() { return opt_on(FLCE_OPT_PIPELINE); }

// Backward on non-ignored rows only (default); FLCE_OPT_COMPACT = 0 runs
// every row.
bool compact_on() { return opt_on(FLCE_OPT_COMPACT); }

// DLOGITS writes D through TMA boxes (default) or per-thread stores
// (FLCE_OPT_D_TMA = 0).
bool d_tma_on() { return opt_on(FLCE_OPT_D_TMA); }

bool validate_on() { return opt_on(FLCE_OPT_VALIDATE); }

// Stream-ordered workspace: the caller's, or one allocated here and freed on
// the same stream when the call ends.
struct Workspace {
  void* ptr = nullptr;
  bool owned = false;
  cudaStream_t st = nullptr;
  ~Workspace() {
    if (owned && ptr != nullptr) cudaFreeAsync(ptr, st);
  }
};

flce_status get_workspace(Workspace& ws, void* user, size_t user_bytes, size_t need, cudaStream_t st) {
  ws.st = st;
  if (user != nullptr) {
    if (user_bytes < need || !aligned(user, 256)) return FLCE_ERR_INVALID_ARG;
    ws.ptr = user;
    return FLCE_OK;
  }
  if (cudaMallocAsync(&ws.ptr, std::max<size_t>(need, 256), st) != cudaSuccess) {
    cudaGetLastError();
    ws.ptr = nullptr;
    return FLCE_ERR_OOM;
  }
  ws.owned = true;
  return FLCE_OK;
}

// Kernel form of a logit transform (see flce_logit_transform): y = a * z, or
// y = b * tanh(a * z) with dy/dz = d * (1 - tanh^2).  False on invalid values.
bool transform_params(const flce_logit_transform* tf, GemmParams& p) {
  p.tf_softcap = 0;
  p.tf_a = 1.f;
  p.tf_b = 1.f;
  p.tf_d = 1.f;
  if (tf == nullptr) return true;
  const float mul = tf->scale_multiply, div = tf->scale_divide, cap = tf->softcap, T = tf->temperature;
  if (!(std::isfinite(mul) && std::isfinite(div) && std::isfinite(cap) && std::isfinite(T))) return false;
  if (mul < 0.f || div < 0.f || cap < 0.f || !(T > 0.f)) return false;
  const float s1 = (mul != 0.f ? mul : 1.f) / (div != 0.f ? div : 1.f);
  if (!(s1 > 0.f) || !std::isfinite(s1)) return false;
  if (cap != 0.f) {
    p.tf_softcap = 1;
    p.tf_a = s1 / cap;
    p.tf_b = cap / T;
    p.tf_d = s1 / T;
  } else {
    p.tf_a = s1 / T;
  }
  return std::isfinite(p.tf_a) && std::isfinite(p.tf_b) && std::isfinite(p.tf_d) && p.tf_a > 0.f;
}

#define FLCE_CUDA_TRY(x)                 \
  do {                                   \
    if ((x) != cudaSuccess) {            \
      cudaGetLastError();                \
      return FLCE_ERR_CUDA;              \
    }                                    \
  } while (0)

// ---- row listing and gathering (row compaction)

// The non-ignored rows of targets[N], listed on the device: their indices in
// order into idx (followed by the ignored rows' when tail), their count into
// *count.  blk: scratch of ceil(N / COMPACT_ROWS_PER_BLOCK) ints.
flce_status list_valid_rows(const int64_t* targets, int N, long long ignore_index, int* blk, int* idx,
                            int* count, bool tail, cudaStream_t st) {
  const int nblk = static_cast<int>(ceil_div(std::max(N, 1), COMPACT_ROWS_PER_BLOCK));
  {
    ProfScope ps(K_COMPACT, st);
    compact_count_kernel<<<nblk, SMALL_THREADS, 0, st>>>(targets, N, ignore_index, blk);
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  ProfScope ps(K_COMPACT, st);
  compact_write_kernel<<<nblk, SMALL_THREADS, 0, st>>>(targets, N, ignore_index, blk, nblk, idx, count,
                                                       tail ? 1 : 0);
  FLCE_CUDA_TRY(cudaGetLastError());
  return FLCE_OK;
}

// Listed rows [first, first + cap) (idx; at most *count - first of them, or
// all when count is null) gathered from h[N][H] into hc[cap][H], with zero
// rows after the last up to the next 64.
flce_status gather_rows(const flce_bf16* h, long long H, const int* idx, const int* count, int N,
                        long long first, long long cap, uint16_t* hc, cudaStream_t st) {
  const int grid = static_cast<int>(
      std::max<long long>(1, std::min<long long>(ceil_div(cap * (H / 8), SMALL_THREADS), 8LL * device_sms())));
  ProfScope ps(K_GATHER, st);
  gather_rows_kernel<<<grid, SMALL_THREADS, 0, st>>>(h, static_cast<int>(H), idx, count, N,
                                                      static_cast<int>(first), static_cast<int>(cap), hc);
  FLCE_CUDA_TRY(cudaGetLastError());
  return FLCE_OK;
}

// Final deterministic reduction of the block partials into loss and count.
flce_status loss_tail(const FwdPlan& f, float* out_loss, int64_t* out_n_valid, const double* bsum,
                      const long long* bcnt, cudaStream_t st) {
  if (out_loss || out_n_valid) {
    ProfScope ps(K_FINAL, st);
    final_kernel<<<1, SMALL_THREADS, 0, st>>>(bsum, bcnt, f.nblk, out_loss,
                                              reinterpret_cast<long long*>(out_n_valid));
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  return FLCE_OK;
}

// ---- stages shared by the entry points


// dH and dW stages of the backward, shared by the cross-entropy and the
// distillation backwards.  For one row block and one vocabulary slab, the
// slab's bf16 dlogits sit in D (maps D_k / D_mn, local columns); B_dw maps the
// block's rows of h (the gathered rows when compacted).  ri / dc / first:
// compaction (original row of each compacted row, device-side row count, first
// compacted row of the block), or null.
struct DhDwStage {
  int cg, workers, tm;
  bool kLong;
  const BwdPlan* plan;
  long long H, V;
  float* dh_part;
  flce_bf16* dH;
  float* dW;
  const CUtensorMap* W_mn;
  const CUtensorMap* dW_map;
  const CUtensorMap* dhp_map;  // fp32 dH partials [dh_splits * R][H]
};

flce_status slab_dh_dw(const DhDwStage& a, const GemmParams& p, int rows, int block, int slab, int v0,
                       int width, const CUtensorMap& D_k, const CUtensorMap& D_mn,
                       const CUtensorMap& B_dw, cudaStream_t st) {
  const BwdPlan& b = *a.plan;
  if (a.dH && a.dW && fuse_dh_dw_on() && b.n_slabs > 1) {
    // both in one launch: the DH units (as below), then the DW units.  Only
    // for plans of several vocabulary slabs, whose short launches pay their
    // fixed cost twice per slab otherwise (131,072 x 2,560 x 151,936 at
    // 256-row chunks: 460 against 468 ms x GHz per step).  With one slab the
    // two long launches ran 3 % faster apart (16,384 x 4,096 x 151,936: 50.6
    // against 52.0 ms per step, same clocks).
    GemmParams q = p;
    q.v0 = v0;
    q.m_tiles = static_cast<int>(ceil_div(rows, a.tm));
    q.n_tiles = static_cast<int>(ceil_div(a.H, BN));
    q.k_blocks = static_cast<int>(ceil_div(width, BK));
    q.cols = q.n_tiles;
    q.n_per_unit = 1;
    q.kb_per_split = b.dh_kb_per_split;
    const int splits = static_cast<int>(ceil_div(q.k_blocks, q.kb_per_split));
    q.k_splits = splits;
    q.group_m = dh_group_rows(q.m_tiles);
    q.dH_part = b.dh_f32 ? a.dh_part : nullptr;
    q.dh_accumulate = slab > 0 ? 1 : 0;
    q.dw_m_tiles = static_cast<int>(ceil_div(width, a.tm));
    q.dw_n_tiles = static_cast<int>(ceil_div(a.H, BN));
    q.dw_k_blocks = static_cast<int>(ceil_div(rows, BK));
    q.dw_group_m = dw_group(q.dw_k_blocks, q.dw_m_tiles);
    q.dW_accumulate = block > 0 ? 1 : 0;
    q.num_units = splits * q.m_tiles * q.n_tiles + q.dw_m_tiles * q.dw_n_tiles;
    ProfScope ps(K_DHDW, st);
    FLCE_CUDA_TRY(launch_gemm<MODE_DHDW>(a.cg, a.kLong, D_k, *a.W_mn, b.dh_f32 ? *a.dhp_map : *a.W_mn, q,
                                         std::min(q.num_units, a.workers), st, &D_mn, &B_dw, a.dW_map));
    return FLCE_OK;
  }
  if (a.dH) {  // dH[rows] (+)= D[:, slab] W[slab]
    GemmParams q = p;
    q.v0 = v0;
    q.m_tiles = static_cast<int>(ceil_div(rows, a.tm));
    // 256 x 512 tiles: n_tiles counts pairs of 256-column tiles
    q.n_tiles = static_cast<int>(ceil_div(a.H, b.dh_wide ? 2 * BN : BN));
    q.k_blocks = static_cast<int>(ceil_div(width, BK));
    q.cols = q.n_tiles;
    q.n_per_unit = 1;
    q.kb_per_split = b.dh_kb_per_split;
    const int splits = static_cast<int>(ceil_div(q.k_blocks, q.kb_per_split));
    q.k_splits = splits;
    q.num_units = splits * q.m_tiles * q.n_tiles;
    q.group_m = b.dh_wide ? q.m_tiles : dh_group_rows(q.m_tiles);
    q.dH_part = b.dh_f32 ? a.dh_part : nullptr;
    q.dh_accumulate = slab > 0 ? 1 : 0;
    ProfScope ps(K_DH, st);
    if (b.dh_wide && a.cg == 2)
      FLCE_CUDA_TRY(launch_gemm<MODE_DH2>(a.cg, a.kLong, D_k, *a.W_mn, b.dh_f32 ? *a.dhp_map : *a.W_mn, q,
                                          std::min(q.num_units, a.workers), st));
    else
      FLCE_CUDA_TRY(launch_gemm<MODE_DH>(a.cg, a.kLong, D_k, *a.W_mn, b.dh_f32 ? *a.dhp_map : *a.W_mn, q,
                                         std::min(q.num_units, a.workers), st));
  }
  if (a.dW) {  // dW[slab] (+)= D[:, slab]^T h[rows]
    GemmParams q = p;
    q.v0 = v0;
    q.m_tiles = static_cast<int>(ceil_div(width, a.tm));
    q.n_tiles = static_cast<int>(ceil_div(a.H, BN));
    q.k_blocks = static_cast<int>(ceil_div(rows, BK));
    q.cols = q.n_tiles;
    q.n_per_unit = 1;
    q.kb_per_split = q.k_blocks;
    q.k_splits = 1;
    q.num_units = q.m_tiles * q.n_tiles;
    q.group_m = dw_group(q.k_blocks, q.m_tiles);
    q.dW_accumulate = block > 0 ? 1 : 0;
    ProfScope ps(K_DW, st);
    FLCE_CUDA_TRY(launch_gemm<MODE_DW>(a.cg, a.kLong, D_mn, B_dw, *a.dW_map, q,
                                       std::min(q.num_units, a.workers), st));
  }
  return FLCE_OK;
}

// The whole backward of one row block in one MODE_PIPE launch: for each
// vocabulary slab its dlogits units (A_dl x W_k into D through D_st), then its
// dH and dW units as slab_dh_dw runs them.  dep: this launch's dependency
// counters (zero at its start); dep_zero: the next launch's, which this one
// zeroes.  The grid is every co-resident SM pair; the pairs draw units in
// order, so the launch also completes on fewer.
flce_status pipe_block(const DhDwStage& a, const GemmParams& p, int rows, int block, const CUtensorMap& A_dl,
                       const CUtensorMap& W_k, const CUtensorMap& D_st, const CUtensorMap& D_k,
                       const CUtensorMap& D_mn, const CUtensorMap& B_dw, unsigned* dep, unsigned* dep_zero,
                       cudaStream_t st) {
  GemmParams q = pipe_params(*a.plan, p, a.H, a.tm, rows, block);
  q.dH_part = a.dh_part;
  q.pp_dep = dep;
  q.pp_dep_zero = dep_zero;
  ProfScope ps(K_PIPE, st);
  FLCE_CUDA_TRY(launch_gemm<MODE_PIPE>(a.cg, a.kLong, D_k, *a.W_mn, *a.dhp_map, q, a.workers, st, &D_mn, &B_dw,
                                       a.dW_map, &A_dl, &W_k, &D_st));
  return FLCE_OK;
}

// After the last slab of a row block: the block's fp32 dH partials, summed
// over the k-splits and rounded to bf16, into its rows of dH.
flce_status block_dh_finish(const DhDwStage& a, int row0, int rows, const int* ri, const int* dc,
                            int first, cudaStream_t st) {
  const BwdPlan& b = *a.plan;
  if (!a.dH || !b.dh_f32) return FLCE_OK;
  ProfScope ps(K_DH_REDUCE, st);
  const long long total = static_cast<long long>(rows) * (a.H / 4);
  const int grid = static_cast<int>(std::max<long long>(
      1, std::min<long long>(ceil_div(total, SMALL_THREADS), 8LL * device_sms())));
  if (a.kLong)
    dh_reduce_kernel<true><<<grid, SMALL_THREADS, 0, st>>>(a.dh_part, b.dh_splits, rows, static_cast<int>(b.R),
                                                           static_cast<int>(a.H), row0, a.dH, ri, dc, first);
  else
    dh_reduce_kernel<false><<<grid, SMALL_THREADS, 0, st>>>(a.dh_part, b.dh_splits, rows, static_cast<int>(b.R),
                                                            static_cast<int>(a.H), row0, a.dH, ri, dc, first);
  FLCE_CUDA_TRY(cudaGetLastError());
  return FLCE_OK;
}

// Cross-entropy forward tail: per-row combine of the split partials, then
// the deterministic loss / count reduction.
flce_status ce_forward_tail(bool kLong, const FwdPlan& f, int N, const float2* part, const float* zt,
                            const int64_t* targets, const float* weights, long long ignore,
                            float* out_logp, float* out_lse, float* out_loss, int64_t* out_n_valid,
                            double* bsum, long long* bcnt, cudaStream_t st, bool skip_ignored = false) {
  if (N > 0) {
    ProfScope ps(K_COMBINE, st);
    const int sk = skip_ignored ? 1 : 0;
    if (kLong)
      combine_kernel<true><<<f.nblk, SMALL_THREADS, 0, st>>>(part, f.S, N, N, zt, targets, weights, ignore,
                                                             out_logp, out_lse, bsum, bcnt, nullptr, sk);
    else
      combine_kernel<false><<<f.nblk, SMALL_THREADS, 0, st>>>(part, f.S, N, N, zt, targets, weights, ignore,
                                                              out_logp, out_lse, bsum, bcnt, nullptr, sk);
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  return loss_tail(f, out_loss, out_n_valid, bsum, bcnt, st);
}

}  // namespace
