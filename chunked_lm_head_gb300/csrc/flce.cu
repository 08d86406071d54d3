// libflce: the C-ABI entry points.  The tensor-core GEMM engine lives in
// gemm.cuh, the CUDA-core kernels in small_kernels.cuh, the launch plans and
// workspace layouts in plan.cuh, tensor maps, launches and shared stages in
// launch.cuh.  include/flce.h states the contract of every entry point.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

#include "flce.h"
#include "gemm.cuh"
#include "small_kernels.cuh"
#include "host_common.cuh"
#include "plan.cuh"
#include "launch.cuh"

namespace {
using namespace flce;
}  // namespace

extern "C" {

const char* flce_status_string(flce_status s) {
  switch (s) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARG: return "FLCE_ERR_INVALID_ARG";
    case FLCE_ERR_BAD_TARGET: return "FLCE_ERR_BAD_TARGET";
    case FLCE_ERR_UNSUPPORTED: return "FLCE_ERR_UNSUPPORTED";
    case FLCE_ERR_OOM: return "FLCE_ERR_OOM";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA";
    case FLCE_ERR_TIMEOUT: return "FLCE_ERR_TIMEOUT";
  }
  return "FLCE_ERR_UNKNOWN";
}

size_t flce_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t chunk_rows) {
  if (!sizes_ok(N, H, V)) return 0;
  const int cg = cta_group();
  const int workers = device_workers(cg);
  // the forward's layout with the buffers of flce_forward_ex2's row skipping
  const FwdLayout fl =
      fwd_layout(N, plan_forward_call(N, H, V, workers, BM * cg), H, fwd_block_rows(N, BM * cg));
  return std::max(fl.total, bwd_workspace(N, H, V, chunk_rows, workers, BM * cg));
}

flce_status flce_backward_plan(int64_t N, int64_t H, int64_t V, int64_t chunk_rows, int32_t workers,
                               int32_t cta_group_, flce_backward_plan_info* out) {
  if (out == nullptr || !sizes_ok(N, H, V)) return FLCE_ERR_INVALID_ARG;
  const int cg = cta_group_ == 1 || cta_group_ == 2 ? cta_group_ : cta_group();
  const int w = workers > 0 ? workers : device_workers(cg);
  const BwdPlan b = plan_backward_call(N, H, V, chunk_rows, w, BM * cg, true);
  out->rows_per_block = b.R;
  out->vocab_per_slab = b.Vs;
  out->row_blocks = ceil_div(std::max<int64_t>(N, 1), b.R);
  out->vocab_slabs = b.n_slabs;
  out->dh_splits = b.dh_splits;
  out->dlogits_bytes = b.buffers * b.R * b.ldD * 2;
  out->workspace_bytes = static_cast<int64_t>(bwd_workspace(N, H, V, chunk_rows, w, BM * cg));
  out->dlogits_buffers = b.buffers;
  out->dh_wide = b.dh_wide ? 1 : 0;
  return FLCE_OK;
}

// The forward; partials_cap bounds the vocabulary-split partials (8 bytes per
// row and split) so that a fixed scratch can hold them.
static flce_status forward_impl(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                                const float* weights, int64_t N, int64_t H, int64_t V,
                                int64_t ignore_index, const flce_logit_transform* transform,
                                float* out_logp, float* out_lse, float* out_loss,
                                int64_t* out_n_valid, void* workspace, size_t workspace_bytes,
                                void* stream, size_t partials_cap, bool skip_ignored = false) {
  if (!sizes_ok(N, H, V)) return FLCE_ERR_INVALID_ARG;
  GemmParams tfp{};
  if (!transform_params(transform, tfp)) return FLCE_ERR_INVALID_ARG;
  if (!out_logp && !out_lse && !out_loss && !out_n_valid) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!h || !W || !targets)) return FLCE_ERR_INVALID_ARG;
  if (H % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(h, 16) || !aligned(W, 16) || !aligned(targets, 8) || !aligned(weights, 4) ||
      !aligned(out_logp, 4) || !aligned(out_lse, 4) || !aligned(out_loss, 4) || !aligned(out_n_valid, 8))
    return FLCE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int cg = cta_group();
  const int workers = device_workers(cg);
  // rows per forward launch (FLCE_OPT_FWD_BLOCK_ROWS; 0: all rows in one launch)
  const long long fb = fwd_block_rows(N, BM * cg);
  const FwdPlan f = plan_forward_call(N, H, V, workers, BM * cg, partials_cap);
  const FwdLayout L = fwd_layout(N, f, H, skip_ignored ? fb : 0);
  Workspace ws;
  flce_status s = get_workspace(ws, workspace, workspace_bytes, L.total, st);
  if (s != FLCE_OK) return s;
  uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
  float* zt = reinterpret_cast<float*>(wb + L.zt);
  float2* part = reinterpret_cast<float2*>(wb + L.part);
  double* bsum = reinterpret_cast<double*>(wb + L.bsum);
  long long* bcnt = reinterpret_cast<long long*>(wb + L.bcnt);
  int* bad = reinterpret_cast<int*>(wb + L.bad);
  const bool validate = validate_on();
  const int Ni = static_cast<int>(N);

  if (N > 0) {
    if (validate) FLCE_CUDA_TRY(cudaMemsetAsync(bad, 0, sizeof(int), st));
    {
      ProfScope ps(K_PREP, st);
      prep_kernel<<<static_cast<int>(ceil_div(N, SMALL_THREADS)), SMALL_THREADS, 0, st>>>(
          targets, Ni, static_cast<int>(V), ignore_index, zt, validate ? bad : nullptr);
      FLCE_CUDA_TRY(cudaGetLastError());
    }
    if (validate) {
      int nbad = 0;
      FLCE_CUDA_TRY(cudaMemcpyAsync(&nbad, bad, sizeof(int), cudaMemcpyDeviceToHost, st));
      FLCE_CUDA_TRY(cudaStreamSynchronize(st));
      if (nbad != 0) return FLCE_ERR_BAD_TARGET;
    }
    // skip_ignored: the launches run over the non-ignored rows only, each
    // over a gathered block of fb of them (the count stays on the device)
    int* cidx = reinterpret_cast<int*>(wb + L.idx);
    int* ccount = reinterpret_cast<int*>(wb + L.count);
    uint16_t* hc = reinterpret_cast<uint16_t*>(wb + L.hc);
    if (skip_ignored) {
      const flce_status sl =
          list_valid_rows(targets, Ni, ignore_index, reinterpret_cast<int*>(wb + L.blk), cidx, ccount, false, st);
      if (sl != FLCE_OK) return sl;
    }
    CUtensorMap tA, tB;
    if (!make_map(&tA, skip_ignored ? hc : h, H, skip_ignored ? fb : N, H, BK, BM) ||
        !make_map(&tB, W, H, V, H, BK, BN / cg))
      return FLCE_ERR_CUDA;
    GemmParams p{};
    p.m_tiles = f.m_tiles;
    p.n_tiles = f.n_tiles;
    p.k_blocks = f.k_blocks;
    p.cols = f.S;
    p.n_per_unit = f.tps;
    p.kb_per_split = f.k_blocks;
    p.k_splits = 1;
    p.num_units = f.units;
    // 16 row tiles share each run of vocabulary tiles in L2: one launch's
    // rows (measured with one launch over all 16K rows of 16K x 4096 x
    // 151,936: DRAM reads 17.9 GB in groups of 16 against 36.6 GB of 8 and
    // 23.6 GB of 32, and the fastest launch)
    p.group_m = std::min(16, f.m_tiles);
    p.row0 = 0;
    p.rows = Ni;
    p.rows_cap = Ni;
    p.N = Ni;
    p.H = static_cast<int>(H);
    p.V = static_cast<int>(V);
    p.ldD = 0;
    p.targets = targets;
    p.weights = weights;
    p.ignore_index = ignore_index;
    p.partials = part;
    p.zt = zt;
    p.tf_softcap = tfp.tf_softcap;
    p.tf_a = tfp.tf_a;
    p.tf_b = tfp.tf_b;
    p.tf_d = tfp.tf_d;
    int* err = nullptr;
    FLCE_CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_device_error));
    p.err = err;
    const bool kLong = static_cast<long long>(N) * V >= INT_MAX ||
                       static_cast<long long>(f.S) * N >= INT_MAX;
    for (long long row0 = 0; row0 < N; row0 += fb) {
      GemmParams q = p;
      q.row0 = static_cast<int>(row0);
      q.rows = static_cast<int>(std::min(fb, N - row0));
      q.rows_cap = q.rows;
      q.m_tiles = static_cast<int>(ceil_div(q.rows, BM * cg));
      q.num_units = q.m_tiles * f.S;
      q.group_m = std::min(16, q.m_tiles);
      if (skip_ignored) {  // non-ignored rows [row0, row0 + fb), gathered
        q.row0 = 0;
        q.row_idx = cidx;
        q.dyn_count = ccount;
        q.chunk_first = static_cast<int>(row0);
        const flce_status sg = gather_rows(h, H, cidx, ccount, Ni, row0, fb, hc, st);
        if (sg != FLCE_OK) return sg;
      }
      ProfScope ps(K_FWD, st);
      FLCE_CUDA_TRY(launch_gemm<MODE_FWD>(cg, kLong, tA, tB, tB, q, std::min(q.num_units, workers), st));
    }
    return ce_forward_tail(kLong, f, Ni, part, zt, targets, weights, ignore_index, out_logp, out_lse,
                           out_loss, out_n_valid, bsum, bcnt, st, skip_ignored);
  }
  return loss_tail(f, out_loss, out_n_valid, bsum, bcnt, st);
}

flce_status flce_forward_ex(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                            const float* weights, int64_t N, int64_t H, int64_t V,
                            int64_t chunk_rows, int64_t ignore_index,
                            const flce_logit_transform* transform, float* out_logp, float* out_lse,
                            float* out_loss, int64_t* out_n_valid, void* workspace,
                            size_t workspace_bytes, void* stream) {
  (void)chunk_rows;
  return forward_impl(h, W, targets, weights, N, H, V, ignore_index, transform, out_logp, out_lse,
                      out_loss, out_n_valid, workspace, workspace_bytes, stream, kFwdPartialsCap);
}

}  // extern "C"

namespace {
// fewest rows for which flce_forward_ex2 skips ignored rows (2,048;
// FLCE_OPT_SKIP_MIN_ROWS overrides): below it the three extra launches cost
// more than the rows save
int64_t skip_min_rows() { return opt(FLCE_OPT_SKIP_MIN_ROWS); }
}  // namespace

extern "C" {

flce_status flce_forward_ex2(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                             const float* weights, int64_t N, int64_t H, int64_t V,
                             int64_t chunk_rows, int64_t ignore_index,
                             const flce_logit_transform* transform, uint32_t flags, float* out_logp,
                             float* out_lse, float* out_loss, int64_t* out_n_valid, void* workspace,
                             size_t workspace_bytes, void* stream) {
  (void)chunk_rows;
  if ((flags & ~static_cast<uint32_t>(FLCE_FORWARD_SKIP_IGNORED)) != 0) return FLCE_ERR_INVALID_ARG;
  const bool skip = (flags & FLCE_FORWARD_SKIP_IGNORED) != 0 && compact_on() && N >= skip_min_rows();
  return forward_impl(h, W, targets, weights, N, H, V, ignore_index, transform, out_logp, out_lse,
                      out_loss, out_n_valid, workspace, workspace_bytes, stream, kFwdPartialsCap, skip);
}

// The backward; count_scale (device int64, or NULL) divides grad_scale by
// max(*count_scale, 1) on the device, and scale_dev (device fp32, or NULL)
// multiplies it.
static flce_status backward_impl(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                                 const float* weights, const float* lse, float grad_scale,
                                 flce_bf16* dH, float* dW, int64_t N, int64_t H, int64_t V,
                                 int64_t chunk_rows, int64_t ignore_index,
                                 const flce_logit_transform* transform, void* workspace,
                                 size_t workspace_bytes, void* stream,
                                 const long long* count_scale, const float* scale_dev = nullptr) {
  if (!sizes_ok(N, H, V)) return FLCE_ERR_INVALID_ARG;
  GemmParams tfp{};
  if (!transform_params(transform, tfp)) return FLCE_ERR_INVALID_ARG;
  if (!dH && !dW) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!h || !W || !targets || !lse)) return FLCE_ERR_INVALID_ARG;
  if (H % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(h, 16) || !aligned(W, 16) || !aligned(dH, 16) || !aligned(dW, 16) ||
      !aligned(targets, 8) || !aligned(weights, 4) || !aligned(lse, 4) || !aligned(count_scale, 8) ||
      !aligned(scale_dev, 4))
    return FLCE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    if (dW) FLCE_CUDA_TRY(cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * H * 4, st));
    return FLCE_OK;
  }
  const int cg = cta_group();
  const int workers = device_workers(cg);
  const int tm = BM * cg;
  const BwdPlan b = plan_backward_call(N, H, V, chunk_rows, workers, tm, dH != nullptr && dW != nullptr);
  const BwdLayout L = bwd_layout(N, H, b);
  Workspace ws;
  flce_status s = get_workspace(ws, workspace, workspace_bytes, L.total, st);
  if (s != FLCE_OK) return s;
  uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
  uint16_t* Dbuf = reinterpret_cast<uint16_t*>(wb + L.D);
  float* dh_part = b.dh_f32 ? reinterpret_cast<float*>(wb + L.dh_part) : nullptr;

  if (validate_on()) {
    int* bad = reinterpret_cast<int*>(wb + L.bad);
    FLCE_CUDA_TRY(cudaMemsetAsync(bad, 0, sizeof(int), st));
    prep_kernel<<<static_cast<int>(ceil_div(N, SMALL_THREADS)), SMALL_THREADS, 0, st>>>(
        targets, static_cast<int>(N), static_cast<int>(V), ignore_index, nullptr, bad);
    FLCE_CUDA_TRY(cudaGetLastError());
    int nbad = 0;
    FLCE_CUDA_TRY(cudaMemcpyAsync(&nbad, bad, sizeof(int), cudaMemcpyDeviceToHost, st));
    FLCE_CUDA_TRY(cudaStreamSynchronize(st));
    if (nbad != 0) return FLCE_ERR_BAD_TARGET;
  }

  int* err = nullptr;
  FLCE_CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_device_error));
  CUtensorMap h_k, W_k, W_mn, h_mn, dW_map;
  if (!make_map(&h_k, h, H, N, H, BK, BM) || !make_map(&W_k, W, H, V, H, BK, BN / cg) ||
      !make_map(&W_mn, W, H, V, H, 64, BK) || !make_map(&h_mn, h, H, N, H, 64, BK))
    return FLCE_ERR_CUDA;
  if (dW && !make_map_t(&dW_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dW, H, V, H, 32, 32))
    return FLCE_ERR_CUDA;
  const bool kLong = static_cast<long long>(N) * V >= INT_MAX ||
                     b.R * b.ldD >= INT_MAX || static_cast<long long>(N) * H >= INT_MAX ||
                     static_cast<long long>(V) * H >= INT_MAX ||
                     static_cast<long long>(b.dh_splits) * b.R * H >= INT_MAX;

  GemmParams base{};
  base.N = static_cast<int>(N);
  base.H = static_cast<int>(H);
  base.V = static_cast<int>(V);
  base.ldD = static_cast<int>(b.ldD);
  base.targets = targets;
  base.weights = weights;
  base.lse = lse;
  base.grad_scale = grad_scale;
  base.count_scale = count_scale;
  base.scale_dev = scale_dev;
  CUtensorMap D_st;  // D as a TMA store target: [buffers * R][ldD] bf16, 64 x 32 boxes
  base.d_tma = d_tma_on() && make_map(&D_st, Dbuf, b.ldD, b.buffers * b.R, b.ldD, 64, 32) ? 1 : 0;
  base.ignore_index = ignore_index;
  base.D = Dbuf;
  base.dH = dH;
  base.dH_part = dh_part;
  base.dW = dW;
  base.err = err;
  base.rows_cap = static_cast<int>(b.R);
  base.tf_softcap = tfp.tf_softcap;
  base.tf_a = tfp.tf_a;
  base.tf_b = tfp.tf_b;
  base.tf_d = tfp.tf_d;

  // Row compaction: the chunks run over the non-ignored rows (count and
  // indices stay on the device; the kernels read each chunk's row count), so
  // ignored rows cost nothing in the three backward GEMMs.  Their dH rows are
  // zeroed up front.  A problem of one row tile gains nothing from it (its
  // GEMMs cover one tile of rows whatever the count), so it skips the listing
  // and gathering launches.
  const bool compact = compact_on() && N > tm;
  int* cidx = reinterpret_cast<int*>(wb + L.idx);
  int* cblk = reinterpret_cast<int*>(wb + L.blk);
  int* ccount = reinterpret_cast<int*>(wb + L.count);
  uint16_t* hc = reinterpret_cast<uint16_t*>(wb + L.hc);
  CUtensorMap hc_k, hc_mn, Dfix_k, Dfix_mn;
  if (compact) {
    const flce_status sl =
        list_valid_rows(targets, static_cast<int>(N), ignore_index, cblk, cidx, ccount, false, st);
    if (sl != FLCE_OK) return sl;
    if (dH) FLCE_CUDA_TRY(cudaMemsetAsync(dH, 0, static_cast<size_t>(N) * H * 2, st));
    if (!make_map(&hc_k, hc, H, b.R, H, BK, BM) || !make_map(&hc_mn, hc, H, b.R, H, 64, BK) ||
        !make_map(&Dfix_k, Dbuf, b.ldD, b.R, b.ldD, BK, BM) ||
        !make_map(&Dfix_mn, Dbuf, b.ldD, b.R, b.ldD, 64, BK))
      return FLCE_ERR_CUDA;
  }

  CUtensorMap dhp_map;
  if (dH && b.dh_f32 &&
      !make_map_t(&dhp_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dh_part, H, b.dh_splits * b.R, H, 32, 32))
    return FLCE_ERR_CUDA;
  const DhDwStage dhdw{cg, workers, tm, kLong, &b, H, V, dh_part, dH, dW, &W_mn, &dW_map, &dhp_map};
  // a pipelined plan: each row block in one launch whose units wait on one
  // another through counters in the workspace (two sets, alternate blocks),
  // D in two buffers of R rows (maps over both)
  const bool pipe = b.buffers == 2 && dH && dW && base.d_tma && b.dh_f32 && b.n_slabs > 1;
  if (b.buffers == 2 && !pipe) return FLCE_ERR_CUDA;  // the planner and this call disagree
  unsigned* dep = reinterpret_cast<unsigned*>(wb + L.dep);
  const long long dep_words = pipe_dep_words(b);
  CUtensorMap Dpipe_k, Dpipe_mn;
  if (pipe) {
    if (!make_map(&Dpipe_k, Dbuf, b.ldD, 2 * b.R, b.ldD, BK, BM) ||
        !make_map(&Dpipe_mn, Dbuf, b.ldD, 2 * b.R, b.ldD, 64, BK))
      return FLCE_ERR_CUDA;
    FLCE_CUDA_TRY(cudaMemsetAsync(dep, 0, static_cast<size_t>(2 * dep_words) * 4, st));
  }
  int block = 0;
  for (long long row0 = 0; row0 < N; row0 += b.R, ++block) {
    // rows: exact (plain) or the capacity whose live part the kernels read (compacted)
    const int rows = compact ? static_cast<int>(b.R) : static_cast<int>(std::min(b.R, N - row0));
    GemmParams p = base;
    p.row0 = compact ? 0 : static_cast<int>(row0);
    p.rows = rows;
    if (compact) {
      p.row_idx = cidx;
      p.dyn_count = ccount;
      p.chunk_first = static_cast<int>(row0);
      const flce_status sg = gather_rows(h, H, cidx, ccount, static_cast<int>(N), row0, b.R, hc, st);
      if (sg != FLCE_OK) return sg;
    }
    const CUtensorMap& A_dl = compact ? hc_k : h_k;
    const CUtensorMap& B_dw = compact ? hc_mn : h_mn;
    CUtensorMap D_k, D_mn;
    if (compact) {
      D_k = Dfix_k;
      D_mn = Dfix_mn;
    } else if (!make_map(&D_k, Dbuf, b.ldD, rows, b.ldD, BK, BM) ||
               !make_map(&D_mn, Dbuf, b.ldD, rows, b.ldD, 64, BK)) {
      return FLCE_ERR_CUDA;
    }
    if (pipe) {
      const flce_status s2 = pipe_block(dhdw, p, rows, block, A_dl, W_k, D_st, Dpipe_k, Dpipe_mn, B_dw,
                                        dep + (block % 2) * dep_words, dep + ((block + 1) % 2) * dep_words, st);
      if (s2 != FLCE_OK) return s2;
    }
    for (int slab = 0; slab < (pipe ? 0 : b.n_slabs); ++slab) {
      const int v0 = static_cast<int>(slab * b.Vs);
      const int width = static_cast<int>(std::min<long long>(b.Vs, V - v0));
      {  // (1) recompute the slab's logits, dlogits -> D[rows, 0:width] bf16
        GemmParams q = p;
        q.v0 = v0;
        q.m_tiles = static_cast<int>(ceil_div(rows, tm));
        q.n_tiles = static_cast<int>(ceil_div(width, BN));
        q.k_blocks = static_cast<int>(ceil_div(H, BK));
        q.cols = q.n_tiles;
        q.n_per_unit = 1;
        q.kb_per_split = q.k_blocks;
        q.k_splits = 1;
        q.num_units = q.m_tiles * q.n_tiles;
        // 16 row tiles per W run in L2 (16K x 4096 x 151,936: DRAM reads 1.9 GB
        // per 4096-row block at 16 against 3.5 GB at 8)
        q.group_m = std::min(16, q.m_tiles);
        ProfScope ps(K_DLOGITS, st);
        FLCE_CUDA_TRY(launch_gemm<MODE_DLOGITS>(cg, kLong, A_dl, W_k, q.d_tma ? D_st : W_k, q,
                                                std::min(q.num_units, workers), st));
      }
      // (2) dH[rows] (+)= D W[slab], (3) dW[slab] (+)= D^T h[rows]
      const flce_status s2 = slab_dh_dw(dhdw, p, rows, block, slab, v0, width, D_k, D_mn, B_dw, st);
      if (s2 != FLCE_OK) return s2;
    }
    const flce_status s3 = block_dh_finish(dhdw, p.row0, rows, compact ? cidx : nullptr,
                                           compact ? ccount : nullptr, static_cast<int>(row0), st);
    if (s3 != FLCE_OK) return s3;
  }
  return FLCE_OK;
}

flce_status flce_backward_ex(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                             const float* weights, const float* lse, float grad_scale,
                             flce_bf16* dH, float* dW, int64_t N, int64_t H, int64_t V,
                             int64_t chunk_rows, int64_t ignore_index,
                             const flce_logit_transform* transform, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return backward_impl(h, W, targets, weights, lse, grad_scale, dH, dW, N, H, V, chunk_rows,
                       ignore_index, transform, workspace, workspace_bytes, stream, nullptr);
}

flce_status flce_backward_ex2(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                              const float* weights, const float* lse, float grad_scale,
                              const flce_device_scale* device_scale, flce_bf16* dH, float* dW,
                              int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                              int64_t ignore_index, const flce_logit_transform* transform,
                              void* workspace, size_t workspace_bytes, void* stream) {
  const long long* count = device_scale ? reinterpret_cast<const long long*>(device_scale->count) : nullptr;
  const float* scale = device_scale ? device_scale->scale : nullptr;
  return backward_impl(h, W, targets, weights, lse, grad_scale, dH, dW, N, H, V, chunk_rows,
                       ignore_index, transform, workspace, workspace_bytes, stream, count, scale);
}

flce_status flce_forward(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                         const float* weights, int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                         int64_t ignore_index, float* out_logp, float* out_lse, float* out_loss,
                         int64_t* out_n_valid, void* workspace, size_t workspace_bytes,
                         void* stream) {
  return flce_forward_ex(h, W, targets, weights, N, H, V, chunk_rows, ignore_index, nullptr, out_logp,
                         out_lse, out_loss, out_n_valid, workspace, workspace_bytes, stream);
}

flce_status flce_backward(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                          const float* weights, const float* lse, float grad_scale, flce_bf16* dH,
                          float* dW, int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                          int64_t ignore_index, void* workspace, size_t workspace_bytes,
                          void* stream) {
  return flce_backward_ex(h, W, targets, weights, lse, grad_scale, dH, dW, N, H, V, chunk_rows,
                          ignore_index, nullptr, workspace, workspace_bytes, stream);
}

// Workspace of the fallback (forward, then the tiled backward with the count
// on the device): the larger of the two, plus lse and n_valid scratch.
struct FallbackLayout {
  size_t inner = 0, lse = 0, nv = 0, lp = 0, wg = 0, gsum = 0, gcnt = 0, total = 0;
};
static FallbackLayout fallback_layout(int64_t N, int64_t H, int64_t V, int64_t chunk_rows, int workers,
                                      int tm) {
  FallbackLayout L;
  const size_t fwd = fwd_layout(N, plan_forward_call(N, H, V, workers, tm)).total;
  const size_t bwd = bwd_workspace(N, H, V, chunk_rows, workers, tm);
  const size_t n4 = align256(static_cast<size_t>(std::max<int64_t>(N, 1)) * 4);
  const size_t nb8 = align256(static_cast<size_t>(ceil_div(std::max<int64_t>(N, 1), SMALL_THREADS)) * 8);
  L.inner = std::max(fwd, bwd);
  L.lse = L.inner;
  L.nv = L.lse + n4;
  L.lp = L.nv + 256;  // the GRPO call: log-probs, backward weights, loss block sums
  L.wg = L.lp + n4;
  L.gsum = L.wg + n4;
  L.gcnt = L.gsum + nb8;
  L.total = L.gcnt + nb8;
  return L;
}
static size_t fallback_workspace(int64_t N, int64_t H, int64_t V, int64_t chunk_rows, int workers,
                                 int tm) {
  return fallback_layout(N, H, V, chunk_rows, workers, tm).total;
}

// The GRPO objective of flce_grpo_forward_backward (NULL: the cross-entropy).
struct GrpoArgs {
  const float* adv;
  const float* old_logp;
  const float* ref_logp;
  float eps_low, eps_high, beta;
  float* out_token_loss;
};

size_t flce_forward_backward_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t chunk_rows) {
  if (!sizes_ok(N, H, V)) return 0;
  const int cg = cta_group();
  const int workers = device_workers(cg);
  const FusedPlan fp = plan_fused(N, H, V, chunk_rows, workers, BM * cg);
  if (fp.fused) return fused_layout(N, H, fp).total;
  return fallback_workspace(N, H, V, chunk_rows, workers, BM * cg);
}

static flce_status forward_backward_impl(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                                         const float* weights, int64_t N, int64_t H, int64_t V,
                                         int64_t chunk_rows, int64_t ignore_index,
                                         const flce_logit_transform* transform, float grad_scale,
                                         float* out_logp, float* out_lse, float* out_loss,
                                         int64_t* out_n_valid, flce_bf16* dH, float* dW, void* workspace,
                                         size_t workspace_bytes, void* stream, const GrpoArgs* grpo) {
  if (!sizes_ok(N, H, V)) return FLCE_ERR_INVALID_ARG;
  GemmParams tfp{};
  if (!transform_params(transform, tfp)) return FLCE_ERR_INVALID_ARG;
  if (!dH && !dW) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!h || !W || !targets)) return FLCE_ERR_INVALID_ARG;
  if (!std::isfinite(grad_scale)) return FLCE_ERR_INVALID_ARG;
  if (H % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(h, 16) || !aligned(W, 16) || !aligned(dH, 16) || !aligned(dW, 16) ||
      !aligned(targets, 8) || !aligned(weights, 4) || !aligned(out_logp, 4) || !aligned(out_lse, 4) ||
      !aligned(out_loss, 4) || !aligned(out_n_valid, 8))
    return FLCE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int cg = cta_group();
  const int workers = device_workers(cg);
  const int tm = BM * cg;
  const FusedPlan fp = plan_fused(N, H, V, chunk_rows, workers, tm);
  if (!fp.fused || N == 0) {
    // forward (lse and n_valid into scratch when the caller wants neither),
    // then the tiled backward with grad_scale / n_valid on the device
    Workspace ws;
    const FallbackLayout FL = fallback_layout(N, H, V, chunk_rows, workers, tm);
    flce_status s = get_workspace(ws, workspace, workspace_bytes, FL.total, st);
    if (s != FLCE_OK) return s;
    uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
    float* lse = out_lse ? out_lse : reinterpret_cast<float*>(wb + FL.lse);
    int64_t* nv = out_n_valid ? out_n_valid : reinterpret_cast<int64_t*>(wb + FL.nv);
    if (grpo == nullptr) {
      s = forward_impl(h, W, targets, weights, N, H, V, ignore_index, transform, out_logp, lse, out_loss, nv,
                       wb, FL.inner, stream, kFwdPartialsCap);
      if (s != FLCE_OK) return s;
      return backward_impl(h, W, targets, weights, lse, grad_scale, dH, dW, N, H, V, chunk_rows, ignore_index,
                           transform, wb, FL.inner, stream, reinterpret_cast<const long long*>(nv));
    }
    // GRPO: the forward's log-probs give each row's token loss and backward
    // weight, then the tiled backward runs with those weights
    float* lp = out_logp ? out_logp : reinterpret_cast<float*>(wb + FL.lp);
    float* wg = reinterpret_cast<float*>(wb + FL.wg);
    double* gsum = reinterpret_cast<double*>(wb + FL.gsum);
    long long* gcnt = reinterpret_cast<long long*>(wb + FL.gcnt);
    s = forward_impl(h, W, targets, nullptr, N, H, V, ignore_index, transform, lp, lse, nullptr, nv, wb,
                     FL.inner, stream, kFwdPartialsCap);
    if (s != FLCE_OK) return s;
    if (N > 0) {
      const int nblk = static_cast<int>(ceil_div(N, SMALL_THREADS));
      {
        ProfScope ps(K_GRPO, st);
        grpo_token_kernel<<<nblk, SMALL_THREADS, 0, st>>>(lp, grpo->old_logp, grpo->ref_logp, grpo->adv, targets,
                                                         static_cast<int>(N), ignore_index, grpo->eps_low,
                                                         grpo->eps_high, grpo->beta, grpo->out_token_loss, wg,
                                                         gsum, gcnt);
        FLCE_CUDA_TRY(cudaGetLastError());
      }
      if (out_loss) {
        ProfScope ps(K_FINAL, st);
        final_kernel<<<1, SMALL_THREADS, 0, st>>>(gsum, gcnt, nblk, out_loss, nullptr);
        FLCE_CUDA_TRY(cudaGetLastError());
      }
    } else if (out_loss) {
      FLCE_CUDA_TRY(cudaMemsetAsync(out_loss, 0, sizeof(float), st));
    }
    return backward_impl(h, W, targets, N > 0 ? wg : nullptr, lse, grad_scale, dH, dW, N, H, V, chunk_rows,
                         ignore_index, transform, wb, FL.inner, stream, reinterpret_cast<const long long*>(nv));
  }
  const FusedLayout L = fused_layout(N, H, fp);
  Workspace ws;
  flce_status s = get_workspace(ws, workspace, workspace_bytes, L.total, st);
  if (s != FLCE_OK) return s;
  uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
  float* zt = reinterpret_cast<float*>(wb + L.zt);
  float2* part = reinterpret_cast<float2*>(wb + L.part);
  double* bsum = reinterpret_cast<double*>(wb + L.bsum);
  long long* bcnt = reinterpret_cast<long long*>(wb + L.bcnt);
  int* bad = reinterpret_cast<int*>(wb + L.bad);
  uint16_t* E = reinterpret_cast<uint16_t*>(wb + L.E);
  float* mx = reinterpret_cast<float*>(wb + L.mx);
  float* lse = out_lse ? out_lse : reinterpret_cast<float*>(wb + L.lse);
  float* dh_part = fp.b.dh_f32 ? reinterpret_cast<float*>(wb + L.dh_part) : nullptr;
  int* cidx = reinterpret_cast<int*>(wb + L.idx);
  int* cblk = reinterpret_cast<int*>(wb + L.blk);
  int* ccount = reinterpret_cast<int*>(wb + L.count);
  uint16_t* hc = reinterpret_cast<uint16_t*>(wb + L.hc);
  // GRPO: the block's log-probs feed its token losses and backward weights
  float* lp = out_logp ? out_logp : (grpo ? reinterpret_cast<float*>(wb + L.lp) : nullptr);
  float* wg = reinterpret_cast<float*>(wb + L.wg);
  const float* dl_weights = grpo ? wg : weights;
  const int Ni = static_cast<int>(N);
  const bool validate = validate_on();
  // Row compaction: the blocks run over a permutation of the rows with the
  // non-ignored ones first.  A block's forward covers all its rows when the
  // caller asks for lse (defined for ignored rows too), else only the
  // non-ignored ones; its dH / dW GEMMs read the device-side count and cover
  // only the non-ignored rows.
  // (one row tile gains nothing from compaction: see backward_impl)
  const bool compact = compact_on() && N > tm;
  const bool fwd_valid_only = compact && out_lse == nullptr;

  if (validate) FLCE_CUDA_TRY(cudaMemsetAsync(bad, 0, sizeof(int), st));
  {
    ProfScope ps(K_PREP, st);
    prep_kernel<<<static_cast<int>(ceil_div(N, SMALL_THREADS)), SMALL_THREADS, 0, st>>>(
        targets, Ni, static_cast<int>(V), ignore_index, zt, validate ? bad : nullptr);
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  if (validate) {
    int nbad = 0;
    FLCE_CUDA_TRY(cudaMemcpyAsync(&nbad, bad, sizeof(int), cudaMemcpyDeviceToHost, st));
    FLCE_CUDA_TRY(cudaStreamSynchronize(st));
    if (nbad != 0) return FLCE_ERR_BAD_TARGET;
  }
  {  // n_valid on the device, before any dlogits
    const flce_status sl = list_valid_rows(targets, Ni, ignore_index, cblk, cidx, ccount, compact, st);
    if (sl != FLCE_OK) return sl;
  }
  if (compact && dH) {  // the dH GEMM writes the non-ignored rows only
    ProfScope ps(K_COMPACT, st);
    const int grid = static_cast<int>(
        std::max<long long>(1, std::min<long long>(ceil_div(N * (H / 8), SMALL_THREADS), 4LL * device_sms())));
    zero_tail_rows_kernel<<<grid, SMALL_THREADS, 0, st>>>(dH, static_cast<int>(H), cidx, ccount, Ni);
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  int* err = nullptr;
  FLCE_CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_device_error));
  CUtensorMap h_k, W_k, W_mn, h_mn, dW_map, dhp_map;
  if (!make_map(&h_k, h, H, N, H, BK, BM) || !make_map(&W_k, W, H, V, H, BK, BN / cg) ||
      !make_map(&W_mn, W, H, V, H, 64, BK) || !make_map(&h_mn, h, H, N, H, 64, BK))
    return FLCE_ERR_CUDA;
  if (dW && !make_map_t(&dW_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dW, H, V, H, 32, 32))
    return FLCE_ERR_CUDA;
  if (dH && fp.b.dh_f32 &&
      !make_map_t(&dhp_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dh_part, H, fp.b.dh_splits * fp.R, H, 32, 32))
    return FLCE_ERR_CUDA;
  CUtensorMap hc_k, hc_mn;
  if (compact && (!make_map(&hc_k, hc, H, fp.R, H, BK, BM) || !make_map(&hc_mn, hc, H, fp.R, H, 64, BK)))
    return FLCE_ERR_CUDA;
  const bool kLong = static_cast<long long>(N) * V >= INT_MAX || fp.R * fp.ldD >= INT_MAX ||
                     static_cast<long long>(N) * H >= INT_MAX || static_cast<long long>(V) * H >= INT_MAX ||
                     static_cast<long long>(fp.b.dh_splits) * fp.R * H >= INT_MAX ||
                     static_cast<long long>(fp.f.S) * N >= INT_MAX;

  GemmParams base{};
  base.N = Ni;
  base.H = static_cast<int>(H);
  base.V = static_cast<int>(V);
  base.ldD = static_cast<int>(fp.ldD);
  base.targets = targets;
  base.weights = weights;
  base.lse = lse;
  base.ignore_index = ignore_index;
  base.D = E;
  base.dH = dH;
  base.dH_part = dh_part;
  base.dW = dW;
  base.err = err;
  base.rows_cap = static_cast<int>(fp.R);
  base.tf_softcap = tfp.tf_softcap;
  base.tf_a = tfp.tf_a;
  base.tf_b = tfp.tf_b;
  base.tf_d = tfp.tf_d;
  const DhDwStage dhdw{cg, workers, tm, kLong, &fp.b, H, V, dh_part, dH, dW, &W_mn, &dW_map, &dhp_map};
  {  // the last block's segment may be shorter than the others: zero it whole
    const long long per = ceil_div(fp.R, SMALL_THREADS);
    const long long last = (ceil_div(N, fp.R) - 1) * per;
    FLCE_CUDA_TRY(cudaMemsetAsync(bsum + last, 0, per * 8, st));
    FLCE_CUDA_TRY(cudaMemsetAsync(bcnt + last, 0, per * 8, st));
  }
  int block = 0;
  for (long long row0 = 0; row0 < N; row0 += fp.R, ++block) {
    const int rows = static_cast<int>(std::min(fp.R, N - row0));
    GemmParams p = base;
    p.row0 = compact ? 0 : static_cast<int>(row0);
    p.rows = rows;
    if (compact) {  // the block's rows of h, in permutation order
      p.row_idx = cidx;
      p.chunk_first = static_cast<int>(row0);
      const flce_status sg = gather_rows(h, H, cidx, fwd_valid_only ? ccount : nullptr, Ni, row0, fp.R, hc, st);
      if (sg != FLCE_OK) return sg;
    }
    {  // (1) logits of the block: online lse partials, target logits, exponentials
      GemmParams q = p;
      q.m_tiles = static_cast<int>(ceil_div(rows, tm));
      q.n_tiles = fp.f.n_tiles;
      q.k_blocks = fp.f.k_blocks;
      q.cols = fp.f.S;
      q.n_per_unit = fp.f.tps;
      q.kb_per_split = fp.f.k_blocks;
      q.k_splits = 1;
      q.num_units = q.m_tiles * fp.f.S;
      q.group_m = std::min(16, q.m_tiles);
      q.partials = part;
      q.zt = zt;
      q.mx = mx;
      // without out_lse, the ignored rows' lse is never observed: skip them
      // (their partials stay unwritten; the combine gives them logp 0)
      if (fwd_valid_only) q.dyn_count = ccount;
      ProfScope ps(K_FWD, st);
      FLCE_CUDA_TRY(launch_gemm<MODE_FUSED_FWD>(cg, kLong, compact ? hc_k : h_k, W_k, W_k, q,
                                                std::min(q.num_units, workers), st));
    }
    {  // (2) the block's lse, logp and loss partials
      ProfScope ps(K_COMBINE, st);
      const int nb = static_cast<int>(ceil_div(rows, SMALL_THREADS));
      const long long b0 = block * ceil_div(fp.R, SMALL_THREADS);  // this block's segment
      // the block's rows: row0 + j, or cidx[row0 + j] (arrays not offset)
      const long long off = compact ? 0 : row0;
      const int* ri = compact ? cidx + row0 : nullptr;
      if (kLong)
        combine_kernel<true><<<nb, SMALL_THREADS, 0, st>>>(part + off, fp.f.S, Ni, rows, zt + off, targets + off,
                                                           weights ? weights + off : nullptr, ignore_index,
                                                           lp ? lp + off : nullptr, lse + off,
                                                           bsum + b0, bcnt + b0, ri);
      else
        combine_kernel<false><<<nb, SMALL_THREADS, 0, st>>>(part + off, fp.f.S, Ni, rows, zt + off, targets + off,
                                                            weights ? weights + off : nullptr, ignore_index,
                                                            lp ? lp + off : nullptr, lse + off,
                                                            bsum + b0, bcnt + b0, ri);
      FLCE_CUDA_TRY(cudaGetLastError());
      if (grpo) {  // token losses and weights of the block's rows; its loss sums replace the NLL's
        ProfScope pg(K_GRPO, st);
        auto at = [&](const float* a) { return a ? a + off : nullptr; };
        grpo_token_kernel<<<nb, SMALL_THREADS, 0, st>>>(
            lp + off, at(grpo->old_logp), at(grpo->ref_logp), grpo->adv + off, targets + off, rows, ignore_index,
            grpo->eps_low, grpo->eps_high, grpo->beta, grpo->out_token_loss ? grpo->out_token_loss + off : nullptr,
            wg + off, bsum + b0, bcnt + b0, ri);
        FLCE_CUDA_TRY(cudaGetLastError());
      }
    }
    {  // (3) exponentials -> dlogits, in place
      ProfScope ps(K_DLOGITS, st);
      const dim3 grid(static_cast<unsigned>(ceil_div(fp.ldD, SMALL_THREADS * FUSED_COLS_PER_THREAD)),
                      static_cast<unsigned>(rows));
      const int* ri = compact ? cidx + row0 : nullptr;
      if (kLong)
        fused_dlogits_kernel<true><<<grid, SMALL_THREADS, 0, st>>>(
            E, mx, static_cast<int>(fp.ldD), static_cast<int>(V), static_cast<int>(row0), ri, targets,
            dl_weights, lse, zt, ignore_index, ccount, grad_scale, tfp.tf_softcap, tfp.tf_a, tfp.tf_b, tfp.tf_d);
      else
        fused_dlogits_kernel<false><<<grid, SMALL_THREADS, 0, st>>>(
            E, mx, static_cast<int>(fp.ldD), static_cast<int>(V), static_cast<int>(row0), ri, targets,
            dl_weights, lse, zt, ignore_index, ccount, grad_scale, tfp.tf_softcap, tfp.tf_a, tfp.tf_b, tfp.tf_d);
      FLCE_CUDA_TRY(cudaGetLastError());
    }
    // (4) dH[rows] = D W, dW (+)= D^T h[rows]; compacted: the block's
    // non-ignored rows, min(n_valid - row0, rows) read on the device
    if (compact) p.dyn_count = ccount;
    CUtensorMap D_k, D_mn;
    if (!make_map(&D_k, E, fp.ldD, rows, fp.ldD, BK, BM) || !make_map(&D_mn, E, fp.ldD, rows, fp.ldD, 64, BK))
      return FLCE_ERR_CUDA;
    s = slab_dh_dw(dhdw, p, rows, block, 0, 0, static_cast<int>(V), D_k, D_mn, compact ? hc_mn : h_mn, st);
    if (s != FLCE_OK) return s;
    s = block_dh_finish(dhdw, p.row0, rows, compact ? cidx : nullptr, compact ? ccount : nullptr,
                        static_cast<int>(row0), st);
    if (s != FLCE_OK) return s;
  }
  if (out_loss || out_n_valid) {
    ProfScope ps(K_FINAL, st);
    // every segment entry was written: full blocks fill theirs, and the last
    // block's unused entries were zeroed before the loop
    final_kernel<<<1, SMALL_THREADS, 0, st>>>(bsum, bcnt,
                                              static_cast<int>(ceil_div(N, fp.R) * ceil_div(fp.R, SMALL_THREADS)),
                                              out_loss, reinterpret_cast<long long*>(out_n_valid));
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  return FLCE_OK;
}

flce_status flce_forward_backward(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                                  const float* weights, int64_t N, int64_t H, int64_t V,
                                  int64_t chunk_rows, int64_t ignore_index,
                                  const flce_logit_transform* transform, float grad_scale,
                                  float* out_logp, float* out_lse, float* out_loss,
                                  int64_t* out_n_valid, flce_bf16* dH, float* dW, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return forward_backward_impl(h, W, targets, weights, N, H, V, chunk_rows, ignore_index, transform, grad_scale,
                               out_logp, out_lse, out_loss, out_n_valid, dH, dW, workspace, workspace_bytes,
                               stream, nullptr);
}

flce_status flce_grpo_forward_backward(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                                       const float* advantages, const float* old_logp,
                                       const float* ref_logp, float eps_low, float eps_high, float beta,
                                       int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                                       int64_t ignore_index, const flce_logit_transform* transform,
                                       float grad_scale, float* out_logp, float* out_token_loss,
                                       float* out_loss, int64_t* out_n_valid, flce_bf16* dH, float* dW,
                                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!(std::isfinite(eps_low) && std::isfinite(eps_high) && std::isfinite(beta)) || eps_low < 0.f ||
      eps_low >= 1.f || eps_high < 0.f || beta < 0.f)
    return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!advantages || (beta > 0.f && !ref_logp))) return FLCE_ERR_INVALID_ARG;
  if (!aligned(advantages, 4) || !aligned(old_logp, 4) || !aligned(ref_logp, 4) || !aligned(out_token_loss, 4))
    return FLCE_ERR_UNSUPPORTED;
  const GrpoArgs g{advantages, old_logp, ref_logp, eps_low, eps_high, beta, out_token_loss};
  return forward_backward_impl(h, W, targets, nullptr, N, H, V, chunk_rows, ignore_index, transform, grad_scale,
                               out_logp, nullptr, out_loss, out_n_valid, dH, dW, workspace, workspace_bytes,
                               stream, &g);
}

flce_status flce_quantize_e4m3_rows(const flce_bf16* x, int64_t rows, int64_t cols, uint8_t* q,
                                    float* scale, void* stream) {
  if (rows < 0 || cols <= 0 || cols >= INT_MAX || (rows > 0 && (!x || !q || !scale)))
    return FLCE_ERR_INVALID_ARG;
  if (cols % 16 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4)) return FLCE_ERR_UNSUPPORTED;
  if (rows == 0) return FLCE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long threads = rows * 32;
  ProfScope ps(K_QUANT, st);
  quantize_e4m3_rows_kernel<<<static_cast<unsigned>(ceil_div(threads, SMALL_THREADS)), SMALL_THREADS, 0,
                              st>>>(x, rows, static_cast<int>(cols), q, scale);
  FLCE_CUDA_TRY(cudaGetLastError());
  return FLCE_OK;
}

flce_status flce_forward_e4m3(const uint8_t* h8, const float* h_scale, const uint8_t* W8,
                              const float* W_scale, const int64_t* targets, const float* weights,
                              int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                              int64_t ignore_index, const flce_logit_transform* transform,
                              float* out_logp, float* out_lse, float* out_loss,
                              int64_t* out_n_valid, void* workspace, size_t workspace_bytes,
                              void* stream) {
  (void)chunk_rows;
  if (!sizes_ok(N, H, V)) return FLCE_ERR_INVALID_ARG;
  GemmParams tfp{};
  if (!transform_params(transform, tfp)) return FLCE_ERR_INVALID_ARG;
  if (!out_logp && !out_lse && !out_loss && !out_n_valid) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!h8 || !h_scale || !W8 || !W_scale || !targets)) return FLCE_ERR_INVALID_ARG;
  if (H % 16 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(h8, 16) || !aligned(W8, 16) || !aligned(W_scale, 16) || !aligned(h_scale, 4) ||
      !aligned(targets, 8) || !aligned(weights, 4) || !aligned(out_logp, 4) || !aligned(out_lse, 4) ||
      !aligned(out_loss, 4) || !aligned(out_n_valid, 8))
    return FLCE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int cg = cta_group();
  const int workers = device_workers(cg);
  // launches of one raster group of rows each (as the bf16 forward)
  const long long fb = fwd_block_rows(N, BM * cg);
  const FwdPlan f = plan_forward_call(N, H, V, workers, BM * cg);
  const FwdLayout L = fwd_layout(N, f);
  Workspace ws;
  flce_status s = get_workspace(ws, workspace, workspace_bytes, L.total, st);
  if (s != FLCE_OK) return s;
  uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
  float* zt = reinterpret_cast<float*>(wb + L.zt);
  float2* part = reinterpret_cast<float2*>(wb + L.part);
  double* bsum = reinterpret_cast<double*>(wb + L.bsum);
  long long* bcnt = reinterpret_cast<long long*>(wb + L.bcnt);
  const int Ni = static_cast<int>(N);
  if (N > 0) {
    {
      ProfScope ps(K_PREP, st);
      prep_kernel<<<static_cast<int>(ceil_div(N, SMALL_THREADS)), SMALL_THREADS, 0, st>>>(
          targets, Ni, static_cast<int>(V), ignore_index, zt, nullptr);
      FLCE_CUDA_TRY(cudaGetLastError());
    }
    CUtensorMap tA, tB;
    if (!make_map_t(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, h8, H, N, H, 128, BM) ||
        !make_map_t(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W8, H, V, H, 128, BN / cg))
      return FLCE_ERR_CUDA;
    int* err = nullptr;
    FLCE_CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_device_error));
    GemmParams p{};
    p.m_tiles = f.m_tiles;
    p.n_tiles = f.n_tiles;
    p.k_blocks = static_cast<int>(ceil_div(H, 128));
    p.cols = f.S;
    p.n_per_unit = f.tps;
    p.kb_per_split = p.k_blocks;
    p.k_splits = 1;
    p.num_units = f.units;
    p.group_m = std::min(16, f.m_tiles);
    p.rows = Ni;
    p.rows_cap = Ni;
    p.N = Ni;
    p.H = static_cast<int>(H);
    p.V = static_cast<int>(V);
    p.targets = targets;
    p.weights = weights;
    p.ignore_index = ignore_index;
    p.partials = part;
    p.zt = zt;
    p.err = err;
    p.a_scale = h_scale;
    p.b_scale = W_scale;
    p.tf_softcap = tfp.tf_softcap;
    p.tf_a = tfp.tf_a;
    p.tf_b = tfp.tf_b;
    p.tf_d = tfp.tf_d;
    const bool kLong = static_cast<long long>(N) * V >= INT_MAX ||
                       static_cast<long long>(f.S) * N >= INT_MAX;
    for (long long row0 = 0; row0 < N; row0 += fb) {
      GemmParams q = p;
      q.row0 = static_cast<int>(row0);
      q.rows = static_cast<int>(std::min(fb, N - row0));
      q.rows_cap = q.rows;
      q.m_tiles = static_cast<int>(ceil_div(q.rows, BM * cg));
      q.num_units = q.m_tiles * f.S;
      q.group_m = std::min(16, q.m_tiles);
      ProfScope ps(K_FWD, st);
      FLCE_CUDA_TRY(launch_fwd_e4m3(cg, kLong, tA, tB, q, std::min(q.num_units, workers), st));
    }
    return ce_forward_tail(kLong, f, Ni, part, zt, targets, weights, ignore_index, out_logp, out_lse,
                           out_loss, out_n_valid, bsum, bcnt, st);
  }
  return loss_tail(f, out_loss, out_n_valid, bsum, bcnt, st);
}

size_t flce_kd_workspace_bytes(int64_t N, int64_t H_s, int64_t H_t, int64_t V, int64_t chunk_rows) {
  if (!sizes_ok(N, H_s, V) || !sizes_ok(N, H_t, V)) return 0;
  const int cg = cta_group();
  const int workers = device_workers(cg);
  // the forward's layout with the buffers of the row-skipping forwards
  const JsdFwdLayout fl = jsd_fwd_layout(N, plan_forward_call(N, H_s + H_t, V, workers, BM * cg), H_s, H_t,
                                         fwd_block_rows(N, BM * cg));
  const DistillBwdLayout bl =
      distill_bwd_layout(N, H_s, H_t, plan_backward(N, H_s, V, chunk_rows, workers, BM * cg));
  return std::max(fl.total, bl.total);
}

// Distillation forward, KL (jsd == false) or Jensen-Shannon with mixture
// weight beta.  Pass 1 runs both heads for their online log-sum-exp (and the
// KL cross term); the Jensen-Shannon terms need both final lse values, so a
// second pass over both heads forms them.
static flce_status distill_forward(bool jsd, float beta, const flce_bf16* h_s, const flce_bf16* W_s,
                                   int64_t H_s, const flce_bf16* h_t, const flce_bf16* W_t,
                                   int64_t H_t, const int64_t* targets, const float* weights,
                                   int64_t N, int64_t V, int64_t ignore_index,
                                   const flce_logit_transform* transform, float* out_kl,
                                   float* out_lse_s, float* out_lse_t, float* out_kl_sm,
                                   float* out_loss, int64_t* out_n_valid, void* workspace,
                                   size_t workspace_bytes, void* stream, bool skip_ignored = false) {
  if (!sizes_ok(N, H_s, V) || !sizes_ok(N, H_t, V)) return FLCE_ERR_INVALID_ARG;
  if (jsd && !(beta > 0.f && beta < 1.f)) return FLCE_ERR_INVALID_ARG;
  // ignored rows are skipped only where targets mark them
  skip_ignored = skip_ignored && targets != nullptr;
  GemmParams tfp{};
  if (!transform_params(transform, tfp)) return FLCE_ERR_INVALID_ARG;
  if (!out_kl && !out_lse_s && !out_lse_t && !out_kl_sm && !out_loss && !out_n_valid)
    return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!h_s || !W_s || !h_t || !W_t)) return FLCE_ERR_INVALID_ARG;
  if (H_s % 8 != 0 || H_t % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(h_s, 16) || !aligned(W_s, 16) || !aligned(h_t, 16) || !aligned(W_t, 16) ||
      !aligned(targets, 8) || !aligned(weights, 4) || !aligned(out_kl, 4) || !aligned(out_lse_s, 4) ||
      !aligned(out_lse_t, 4) || !aligned(out_kl_sm, 4) || !aligned(out_loss, 4) ||
      !aligned(out_n_valid, 8))
    return FLCE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int cg = cta_group();
  const int workers = device_workers(cg);
  const int kbs = static_cast<int>(ceil_div(H_s, BK));
  const int kbt = static_cast<int>(ceil_div(H_t, BK));
  // launches of one raster group of rows each (as the cross-entropy forward)
  const long long fb = fwd_block_rows(N, BM * cg);
  const FwdPlan f = plan_forward_call(N, H_s + H_t, V, workers, BM * cg);
  const JsdFwdLayout J = jsd_fwd_layout(N, f, H_s, H_t, skip_ignored ? fb : 0);
  const KdFwdLayout& L = J.kd;
  Workspace ws;
  flce_status s = get_workspace(ws, workspace, workspace_bytes, (jsd || skip_ignored) ? J.total : L.total, st);
  if (s != FLCE_OK) return s;
  uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
  float2* ps = reinterpret_cast<float2*>(wb + L.ps);
  float2* pt = reinterpret_cast<float2*>(wb + L.pt);
  float* pc = reinterpret_cast<float*>(wb + L.pc);
  double* bsum = reinterpret_cast<double*>(wb + L.bsum);
  long long* bcnt = reinterpret_cast<long long*>(wb + L.bcnt);
  // the Jensen-Shannon pass reads both lse vectors: the caller's, or scratch
  float* lse_s = out_lse_s;
  float* lse_t = out_lse_t;
  if (jsd) {
    if (!lse_s) lse_s = reinterpret_cast<float*>(wb + J.lse_s);
    if (!lse_t) lse_t = reinterpret_cast<float*>(wb + J.lse_t);
  }
  const int Ni = static_cast<int>(N);
  if (N > 0) {
    // skip_ignored: every launch runs over a gathered block of the
    // non-ignored rows (listed on the device, count read by the kernels)
    int* cidx = reinterpret_cast<int*>(wb + J.idx);
    int* ccount = reinterpret_cast<int*>(wb + J.count);
    uint16_t* hs_c = reinterpret_cast<uint16_t*>(wb + J.hs);
    uint16_t* ht_c = reinterpret_cast<uint16_t*>(wb + J.ht);
    if (skip_ignored) {
      const flce_status sl = list_valid_rows(targets, static_cast<int>(N), ignore_index,
                                             reinterpret_cast<int*>(wb + J.blk), cidx, ccount, false, st);
      if (sl != FLCE_OK) return sl;
    }
    CUtensorMap hs_k, Ws_k, ht_k, Wt_k;
    if (!make_map(&hs_k, skip_ignored ? hs_c : h_s, H_s, skip_ignored ? fb : N, H_s, BK, BM) ||
        !make_map(&Ws_k, W_s, H_s, V, H_s, BK, BN / cg) ||
        !make_map(&ht_k, skip_ignored ? ht_c : h_t, H_t, skip_ignored ? fb : N, H_t, BK, BM) ||
        !make_map(&Wt_k, W_t, H_t, V, H_t, BK, BN / cg))
      return FLCE_ERR_CUDA;
    // the block's rows of both heads, gathered (skip_ignored)
    auto gather_block = [&](long long row0) -> flce_status {
      const flce_status sg = gather_rows(h_s, H_s, cidx, ccount, static_cast<int>(N), row0, fb, hs_c, st);
      return sg != FLCE_OK ? sg : gather_rows(h_t, H_t, cidx, ccount, static_cast<int>(N), row0, fb, ht_c, st);
    };
    int* err = nullptr;
    FLCE_CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_device_error));
    GemmParams p{};
    p.m_tiles = f.m_tiles;
    p.n_tiles = f.n_tiles;
    p.k_blocks = kbs + kbt;
    p.k_blocks_s = kbs;
    p.cols = f.S;
    p.n_per_unit = f.tps;
    p.kb_per_split = kbs + kbt;
    p.k_splits = 1;
    p.num_units = f.units;
    p.group_m = std::min(16, f.m_tiles);
    p.rows = Ni;
    p.rows_cap = Ni;
    p.N = Ni;
    p.H = static_cast<int>(H_s);
    p.V = static_cast<int>(V);
    p.targets = targets;
    p.weights = weights;
    p.ignore_index = ignore_index;
    p.partials = ps;
    p.partials_t = pt;
    p.partials_c = pc;
    // the Jensen-Shannon pass: per-row partials of each column half of a
    // tile in a slot of their own (8 epilogue warps); pass 1 keeps 4 warps,
    // which timed as fast for its cheaper epilogue
    const int jsd_parts = wide_epilogue_on() ? kJsdColParts : 1;
    const int jsd_slots = f.S * jsd_parts;
    p.col_parts = 1;
    p.err = err;
    p.tf_softcap = tfp.tf_softcap;
    p.tf_a = tfp.tf_a;
    p.tf_b = tfp.tf_b;
    p.tf_d = tfp.tf_d;
    const bool kLong = static_cast<long long>(N) * V >= INT_MAX ||
                       static_cast<long long>(jsd_slots) * N >= INT_MAX;
    // one launch per block of fb rows: every unit of a launch shares its
    // rows' h tiles, and the 16 row tiles of a block share each W tile in L2
    auto block_params = [&](const GemmParams& base, long long row0) {
      GemmParams q = base;
      q.row0 = static_cast<int>(row0);
      q.rows = static_cast<int>(std::min(fb, N - row0));
      q.rows_cap = q.rows;
      q.m_tiles = static_cast<int>(ceil_div(q.rows, BM * cg));
      q.num_units = q.m_tiles * f.S;
      q.group_m = std::min(16, q.m_tiles);
      if (skip_ignored) {  // non-ignored rows [row0, row0 + fb), gathered
        q.row0 = 0;
        q.row_idx = cidx;
        q.chunk_first = static_cast<int>(row0);
        q.dyn_count = ccount;
      }
      return q;
    };
    for (long long row0 = 0; row0 < N; row0 += fb) {
      if (skip_ignored) {
        const flce_status sg = gather_block(row0);
        if (sg != FLCE_OK) return sg;
      }
      const GemmParams q = block_params(p, row0);
      ProfScope prof(K_KD_FWD, st);
      FLCE_CUDA_TRY(launch_gemm<MODE_KD_FWD>(cg, kLong, hs_k, Ws_k, Ws_k, q, std::min(q.num_units, workers), st,
                                             &ht_k, &Wt_k));
    }
    {
      ProfScope prof(K_COMBINE, st);
      float* kl = jsd ? nullptr : out_kl;
      const int sk = skip_ignored ? 1 : 0;
      if (kLong)
        kd_combine_kernel<true><<<f.nblk, SMALL_THREADS, 0, st>>>(ps, pt, pc, f.S, Ni, targets, weights,
                                                                  ignore_index, kl, lse_s, lse_t, bsum, bcnt, sk);
      else
        kd_combine_kernel<false><<<f.nblk, SMALL_THREADS, 0, st>>>(ps, pt, pc, f.S, Ni, targets, weights,
                                                                   ignore_index, kl, lse_s, lse_t, bsum, bcnt, sk);
      FLCE_CUDA_TRY(cudaGetLastError());
    }
    if (jsd) {
      float2* pj = reinterpret_cast<float2*>(wb + J.pj);
      GemmParams q = p;
      q.lse = lse_s;
      q.lse_t = lse_t;
      q.partials = pj;
      q.jsd_beta = beta;
      q.col_parts = jsd_parts;
      for (long long row0 = 0; row0 < N; row0 += fb) {
        if (skip_ignored) {
          const flce_status sg = gather_block(row0);
          if (sg != FLCE_OK) return sg;
        }
        const GemmParams qb = block_params(q, row0);
        ProfScope prof(K_JSD_FWD, st);
        FLCE_CUDA_TRY(launch_gemm<MODE_JSD_FWD>(cg, kLong, hs_k, Ws_k, Ws_k, qb, std::min(qb.num_units, workers),
                                                st, &ht_k, &Wt_k));
      }
      ProfScope prof(K_COMBINE, st);
      const int skj = skip_ignored ? 1 : 0;
      if (kLong)
        jsd_combine_kernel<true><<<f.nblk, SMALL_THREADS, 0, st>>>(pj, jsd_slots, Ni, targets, weights, ignore_index,
                                                                   beta, out_kl, out_kl_sm, bsum, bcnt, skj);
      else
        jsd_combine_kernel<false><<<f.nblk, SMALL_THREADS, 0, st>>>(pj, jsd_slots, Ni, targets, weights, ignore_index,
                                                                    beta, out_kl, out_kl_sm, bsum, bcnt, skj);
      FLCE_CUDA_TRY(cudaGetLastError());
    }
  }
  return loss_tail(f, out_loss, out_n_valid, bsum, bcnt, st);
}

flce_status flce_kd_forward(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                            const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                            const int64_t* targets, const float* weights, int64_t N, int64_t V,
                            int64_t chunk_rows, int64_t ignore_index,
                            const flce_logit_transform* transform, float* out_kl, float* out_lse_s,
                            float* out_lse_t, float* out_loss, int64_t* out_n_valid,
                            void* workspace, size_t workspace_bytes, void* stream) {
  (void)chunk_rows;
  return distill_forward(false, 0.f, h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, ignore_index,
                         transform, out_kl, out_lse_s, out_lse_t, nullptr, out_loss, out_n_valid,
                         workspace, workspace_bytes, stream);
}

flce_status flce_jsd_forward(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                             const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                             const int64_t* targets, const float* weights, int64_t N, int64_t V,
                             int64_t chunk_rows, int64_t ignore_index, float beta,
                             const flce_logit_transform* transform, float* out_jsd,
                             float* out_lse_s, float* out_lse_t, float* out_kl_sm, float* out_loss,
                             int64_t* out_n_valid, void* workspace, size_t workspace_bytes,
                             void* stream) {
  (void)chunk_rows;
  return distill_forward(true, beta, h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, ignore_index,
                         transform, out_jsd, out_lse_s, out_lse_t, out_kl_sm, out_loss, out_n_valid,
                         workspace, workspace_bytes, stream);
}

static bool distill_skip(uint32_t flags, int64_t N) {
  return (flags & FLCE_FORWARD_SKIP_IGNORED) != 0 && compact_on() && N >= skip_min_rows();
}

flce_status flce_kd_forward_ex2(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                const int64_t* targets, const float* weights, int64_t N, int64_t V,
                                int64_t chunk_rows, int64_t ignore_index,
                                const flce_logit_transform* transform, uint32_t flags, float* out_kl,
                                float* out_lse_s, float* out_lse_t, float* out_loss, int64_t* out_n_valid,
                                void* workspace, size_t workspace_bytes, void* stream) {
  (void)chunk_rows;
  if ((flags & ~static_cast<uint32_t>(FLCE_FORWARD_SKIP_IGNORED)) != 0) return FLCE_ERR_INVALID_ARG;
  return distill_forward(false, 0.f, h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, ignore_index,
                         transform, out_kl, out_lse_s, out_lse_t, nullptr, out_loss, out_n_valid,
                         workspace, workspace_bytes, stream, distill_skip(flags, N));
}

flce_status flce_jsd_forward_ex2(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                 const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                 const int64_t* targets, const float* weights, int64_t N, int64_t V,
                                 int64_t chunk_rows, int64_t ignore_index, float beta,
                                 const flce_logit_transform* transform, uint32_t flags, float* out_jsd,
                                 float* out_lse_s, float* out_lse_t, float* out_kl_sm, float* out_loss,
                                 int64_t* out_n_valid, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  (void)chunk_rows;
  if ((flags & ~static_cast<uint32_t>(FLCE_FORWARD_SKIP_IGNORED)) != 0) return FLCE_ERR_INVALID_ARG;
  return distill_forward(true, beta, h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, ignore_index,
                         transform, out_jsd, out_lse_s, out_lse_t, out_kl_sm, out_loss, out_n_valid,
                         workspace, workspace_bytes, stream, distill_skip(flags, N));
}

// Distillation backward (student gradients, teacher frozen): KL dlogits
// (jsd == false) or Jensen-Shannon dlogits with mixture weight beta and the
// forward's per-row KL(p_s || M); then the shared dH / dW stages.
static flce_status distill_backward(bool jsd, float beta, const float* kl_sm, const flce_bf16* h_s,
                                    const flce_bf16* W_s, int64_t H_s, const flce_bf16* h_t,
                                    const flce_bf16* W_t, int64_t H_t, const int64_t* targets,
                                    const float* weights, const float* lse_s, const float* lse_t,
                                    float grad_scale, flce_bf16* dH_s, float* dW_s, int64_t N,
                                    int64_t V, int64_t chunk_rows, int64_t ignore_index,
                                    const flce_logit_transform* transform, void* workspace,
                                    size_t workspace_bytes, void* stream,
                                    const flce_device_scale* device_scale = nullptr) {
  const long long* count_scale =
      device_scale ? reinterpret_cast<const long long*>(device_scale->count) : nullptr;
  const float* scale_dev = device_scale ? device_scale->scale : nullptr;
  if (!aligned(count_scale, 8) || !aligned(scale_dev, 4)) return FLCE_ERR_UNSUPPORTED;
  if (!sizes_ok(N, H_s, V) || !sizes_ok(N, H_t, V)) return FLCE_ERR_INVALID_ARG;
  if (jsd && !(beta > 0.f && beta < 1.f)) return FLCE_ERR_INVALID_ARG;
  GemmParams tfp{};
  if (!transform_params(transform, tfp)) return FLCE_ERR_INVALID_ARG;
  if (!dH_s && !dW_s) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!h_s || !W_s || !h_t || !W_t || !lse_s || !lse_t)) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && jsd && !kl_sm) return FLCE_ERR_INVALID_ARG;
  if (H_s % 8 != 0 || H_t % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(h_s, 16) || !aligned(W_s, 16) || !aligned(h_t, 16) || !aligned(W_t, 16) ||
      !aligned(dH_s, 16) || !aligned(dW_s, 16) || !aligned(targets, 8) || !aligned(weights, 4) ||
      !aligned(lse_s, 4) || !aligned(lse_t, 4) || !aligned(kl_sm, 4))
    return FLCE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    if (dW_s) FLCE_CUDA_TRY(cudaMemsetAsync(dW_s, 0, static_cast<size_t>(V) * H_s * 4, st));
    return FLCE_OK;
  }
  const int cg = cta_group();
  const int workers = device_workers(cg);
  const int tm = BM * cg;
  const BwdPlan b = plan_backward(N, H_s, V, chunk_rows, workers, tm);
  const DistillBwdLayout DL = distill_bwd_layout(N, H_s, H_t, b);
  const BwdLayout& L = DL.b;
  Workspace ws;
  flce_status s = get_workspace(ws, workspace, workspace_bytes, DL.total, st);
  if (s != FLCE_OK) return s;
  uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
  uint16_t* Dbuf = reinterpret_cast<uint16_t*>(wb + L.D);
  float* dh_part = b.dh_f32 ? reinterpret_cast<float*>(wb + L.dh_part) : nullptr;
  int* err = nullptr;
  FLCE_CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_device_error));
  CUtensorMap hs_k, Ws_k, ht_k, Wt_k, Ws_mn, hs_mn, dW_map;
  if (!make_map(&hs_k, h_s, H_s, N, H_s, BK, BM) || !make_map(&Ws_k, W_s, H_s, V, H_s, BK, BN / cg) ||
      !make_map(&ht_k, h_t, H_t, N, H_t, BK, BM) || !make_map(&Wt_k, W_t, H_t, V, H_t, BK, BN / cg) ||
      !make_map(&Ws_mn, W_s, H_s, V, H_s, 64, BK) || !make_map(&hs_mn, h_s, H_s, N, H_s, 64, BK))
    return FLCE_ERR_CUDA;
  if (dW_s && !make_map_t(&dW_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dW_s, H_s, V, H_s, 32, 32))
    return FLCE_ERR_CUDA;
  const long long H = H_s;
  const bool kLong = static_cast<long long>(N) * V >= INT_MAX || b.R * b.ldD >= INT_MAX ||
                     static_cast<long long>(N) * H >= INT_MAX ||
                     static_cast<long long>(V) * H >= INT_MAX ||
                     static_cast<long long>(b.dh_splits) * b.R * H >= INT_MAX;
  const int kbs = static_cast<int>(ceil_div(H_s, BK));
  const int kbt = static_cast<int>(ceil_div(H_t, BK));

  GemmParams base{};
  base.N = static_cast<int>(N);
  base.H = static_cast<int>(H_s);
  base.V = static_cast<int>(V);
  base.ldD = static_cast<int>(b.ldD);
  base.targets = targets;
  base.weights = weights;
  base.lse = lse_s;
  base.lse_t = lse_t;
  base.grad_scale = grad_scale;
  base.count_scale = count_scale;
  base.scale_dev = scale_dev;
  base.ignore_index = ignore_index;
  base.D = Dbuf;
  base.dH = dH_s;
  base.dH_part = dh_part;
  base.dW = dW_s;
  base.err = err;
  base.rows_cap = static_cast<int>(b.R);
  base.k_blocks_s = kbs;
  base.jsd_beta = beta;
  base.kl_sm = kl_sm;
  base.tf_softcap = tfp.tf_softcap;
  base.tf_a = tfp.tf_a;
  base.tf_b = tfp.tf_b;
  base.tf_d = tfp.tf_d;

  // Row compaction, as in the cross-entropy backward: where targets mark
  // ignored rows, the chunks run over the non-ignored rows of both heads
  // (gathered per chunk), and the ignored rows' dH is zeroed up front.
  const bool compact = targets != nullptr && compact_on();
  int* cidx = reinterpret_cast<int*>(wb + L.idx);
  int* cblk = reinterpret_cast<int*>(wb + L.blk);
  int* ccount = reinterpret_cast<int*>(wb + L.count);
  uint16_t* hcs = reinterpret_cast<uint16_t*>(wb + L.hc);
  uint16_t* hct = reinterpret_cast<uint16_t*>(wb + DL.hc_t);
  CUtensorMap hcs_k, hcs_mn, hct_k, Dfix_k, Dfix_mn;
  if (compact) {
    const flce_status sl =
        list_valid_rows(targets, static_cast<int>(N), ignore_index, cblk, cidx, ccount, false, st);
    if (sl != FLCE_OK) return sl;
    if (dH_s) FLCE_CUDA_TRY(cudaMemsetAsync(dH_s, 0, static_cast<size_t>(N) * H_s * 2, st));
    if (!make_map(&hcs_k, hcs, H_s, b.R, H_s, BK, BM) || !make_map(&hcs_mn, hcs, H_s, b.R, H_s, 64, BK) ||
        !make_map(&hct_k, hct, H_t, b.R, H_t, BK, BM) ||
        !make_map(&Dfix_k, Dbuf, b.ldD, b.R, b.ldD, BK, BM) ||
        !make_map(&Dfix_mn, Dbuf, b.ldD, b.R, b.ldD, 64, BK))
      return FLCE_ERR_CUDA;
  }

  CUtensorMap dhp_map;
  if (dH_s && b.dh_f32 &&
      !make_map_t(&dhp_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dh_part, H, b.dh_splits * b.R, H, 32, 32))
    return FLCE_ERR_CUDA;
  const DhDwStage dhdw{cg, workers, tm, kLong, &b, H, V, dh_part, dH_s, dW_s, &Ws_mn, &dW_map, &dhp_map};
  int block = 0;
  for (long long row0 = 0; row0 < N; row0 += b.R, ++block) {
    // rows: exact (plain) or the capacity whose live part the kernels read (compacted)
    const int rows = compact ? static_cast<int>(b.R) : static_cast<int>(std::min(b.R, N - row0));
    GemmParams p = base;
    p.row0 = compact ? 0 : static_cast<int>(row0);
    p.rows = rows;
    if (compact) {
      p.row_idx = cidx;
      p.dyn_count = ccount;
      p.chunk_first = static_cast<int>(row0);
      for (int head = 0; head < 2; ++head) {
        const flce_status sg = gather_rows(head == 0 ? h_s : h_t, head == 0 ? H_s : H_t, cidx, ccount,
                                           static_cast<int>(N), row0, b.R, head == 0 ? hcs : hct, st);
        if (sg != FLCE_OK) return sg;
      }
    }
    const CUtensorMap& As_k = compact ? hcs_k : hs_k;
    const CUtensorMap& At_k = compact ? hct_k : ht_k;
    const CUtensorMap& B_dw = compact ? hcs_mn : hs_mn;
    CUtensorMap D_k, D_mn;
    if (compact) {
      D_k = Dfix_k;
      D_mn = Dfix_mn;
    } else if (!make_map(&D_k, Dbuf, b.ldD, rows, b.ldD, BK, BM) ||
               !make_map(&D_mn, Dbuf, b.ldD, rows, b.ldD, 64, BK)) {
      return FLCE_ERR_CUDA;
    }
    for (int slab = 0; slab < b.n_slabs; ++slab) {
      const int v0 = static_cast<int>(slab * b.Vs);
      const int width = static_cast<int>(std::min<long long>(b.Vs, V - v0));
      {  // (1) student and teacher logits of the slab, distillation dlogits -> D
        GemmParams q = p;
        q.v0 = v0;
        q.m_tiles = static_cast<int>(ceil_div(rows, tm));
        q.n_tiles = static_cast<int>(ceil_div(width, BN));
        q.k_blocks = kbs + kbt;
        q.cols = q.n_tiles;
        q.n_per_unit = 1;
        q.kb_per_split = kbs + kbt;
        q.k_splits = 1;
        q.num_units = q.m_tiles * q.n_tiles;
        q.group_m = std::min(16, q.m_tiles);
        ProfScope prof(jsd ? K_JSD_DLOGITS : K_KD_DLOGITS, st);
        if (jsd)
          FLCE_CUDA_TRY(launch_gemm<MODE_JSD_DLOGITS>(cg, kLong, As_k, Ws_k, Ws_k, q,
                                                      std::min(q.num_units, workers), st, &At_k, &Wt_k));
        else
          FLCE_CUDA_TRY(launch_gemm<MODE_KD_DLOGITS>(cg, kLong, As_k, Ws_k, Ws_k, q,
                                                     std::min(q.num_units, workers), st, &At_k, &Wt_k));
      }
      const flce_status s2 = slab_dh_dw(dhdw, p, rows, block, slab, v0, width, D_k, D_mn, B_dw, st);
      if (s2 != FLCE_OK) return s2;
    }
    const flce_status s3 = block_dh_finish(dhdw, p.row0, rows, compact ? cidx : nullptr,
                                           compact ? ccount : nullptr, static_cast<int>(row0), st);
    if (s3 != FLCE_OK) return s3;
  }
  return FLCE_OK;
}

flce_status flce_kd_backward(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                             const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                             const int64_t* targets, const float* weights, const float* lse_s,
                             const float* lse_t, float grad_scale, flce_bf16* dH_s, float* dW_s,
                             int64_t N, int64_t V, int64_t chunk_rows, int64_t ignore_index,
                             const flce_logit_transform* transform, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return distill_backward(false, 0.f, nullptr, h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s,
                          lse_t, grad_scale, dH_s, dW_s, N, V, chunk_rows, ignore_index, transform,
                          workspace, workspace_bytes, stream);
}

flce_status flce_jsd_backward(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                              const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                              const int64_t* targets, const float* weights, const float* lse_s,
                              const float* lse_t, const float* kl_sm, float beta, float grad_scale,
                              flce_bf16* dH_s, float* dW_s, int64_t N, int64_t V, int64_t chunk_rows,
                              int64_t ignore_index, const flce_logit_transform* transform,
                              void* workspace, size_t workspace_bytes, void* stream) {
  return distill_backward(true, beta, kl_sm, h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s,
                          lse_t, grad_scale, dH_s, dW_s, N, V, chunk_rows, ignore_index, transform,
                          workspace, workspace_bytes, stream);
}

flce_status flce_kd_backward_ex2(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                 const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                 const int64_t* targets, const float* weights, const float* lse_s,
                                 const float* lse_t, float grad_scale,
                                 const flce_device_scale* device_scale, flce_bf16* dH_s, float* dW_s,
                                 int64_t N, int64_t V, int64_t chunk_rows, int64_t ignore_index,
                                 const flce_logit_transform* transform, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return distill_backward(false, 0.f, nullptr, h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s,
                          lse_t, grad_scale, dH_s, dW_s, N, V, chunk_rows, ignore_index, transform,
                          workspace, workspace_bytes, stream, device_scale);
}

flce_status flce_jsd_backward_ex2(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                  const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                  const int64_t* targets, const float* weights, const float* lse_s,
                                  const float* lse_t, const float* kl_sm, float beta, float grad_scale,
                                  const flce_device_scale* device_scale, flce_bf16* dH_s, float* dW_s,
                                  int64_t N, int64_t V, int64_t chunk_rows, int64_t ignore_index,
                                  const flce_logit_transform* transform, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return distill_backward(true, beta, kl_sm, h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s,
                          lse_t, grad_scale, dH_s, dW_s, N, V, chunk_rows, ignore_index, transform,
                          workspace, workspace_bytes, stream, device_scale);
}

flce_status flce_scale_grads(flce_bf16* dH, int64_t n_dH, float* dW, int64_t n_dW, const float* scale,
                             void* stream) {
  if (n_dH < 0 || n_dW < 0 || scale == nullptr || (n_dH > 0 && dH == nullptr) ||
      (n_dW > 0 && dW == nullptr))
    return FLCE_ERR_INVALID_ARG;
  if (!aligned(dH, 16) || !aligned(dW, 16) || !aligned(scale, 4)) return FLCE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = 8 * device_sms();
  if (n_dH > 0) {
    scale_bf16_kernel<<<grid, SMALL_THREADS, 0, st>>>(reinterpret_cast<__nv_bfloat16*>(dH), n_dH, scale);
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  if (n_dW > 0) {
    scale_f32_kernel<<<grid, SMALL_THREADS, 0, st>>>(dW, n_dW, scale);
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  return FLCE_OK;
}

size_t flce_grpo_workspace_bytes(int64_t N) {
  if (N < 0 || N >= INT_MAX) return 0;
  return 2 * align256(static_cast<size_t>(ceil_div(std::max<int64_t>(N, 1), SMALL_THREADS)) * 8);
}

flce_status flce_grpo_token_loss(const float* logp, const float* old_logp, const float* ref_logp,
                                 const float* advantages, const int64_t* targets, int64_t N,
                                 int64_t ignore_index, float eps_low, float eps_high, float beta,
                                 float* out_token_loss, float* out_weights, float* out_loss,
                                 int64_t* out_n_valid, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (N < 0 || N >= INT_MAX) return FLCE_ERR_INVALID_ARG;
  if (!(std::isfinite(eps_low) && std::isfinite(eps_high) && std::isfinite(beta)) || eps_low < 0.f ||
      eps_low >= 1.f || eps_high < 0.f || beta < 0.f)
    return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!logp || !advantages || (beta > 0.f && !ref_logp))) return FLCE_ERR_INVALID_ARG;
  if (!out_token_loss && !out_weights && !out_loss && !out_n_valid) return FLCE_ERR_INVALID_ARG;
  if (!aligned(logp, 4) || !aligned(old_logp, 4) || !aligned(ref_logp, 4) || !aligned(advantages, 4) ||
      !aligned(targets, 8) || !aligned(out_token_loss, 4) || !aligned(out_weights, 4) ||
      !aligned(out_loss, 4) || !aligned(out_n_valid, 8))
    return FLCE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nblk = static_cast<int>(ceil_div(std::max<int64_t>(N, 1), SMALL_THREADS));
  Workspace ws;
  const flce_status s = get_workspace(ws, workspace, workspace_bytes, flce_grpo_workspace_bytes(N), st);
  if (s != FLCE_OK) return s;
  uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
  double* bsum = reinterpret_cast<double*>(wb);
  long long* bcnt = reinterpret_cast<long long*>(wb + align256(static_cast<size_t>(nblk) * 8));
  {
    ProfScope ps(K_GRPO, st);
    grpo_token_kernel<<<nblk, SMALL_THREADS, 0, st>>>(logp, old_logp, ref_logp, advantages, targets,
                                                     static_cast<int>(N), ignore_index, eps_low, eps_high,
                                                     beta, out_token_loss, out_weights, bsum, bcnt);
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  if (out_loss || out_n_valid) {
    ProfScope ps(K_FINAL, st);
    final_kernel<<<1, SMALL_THREADS, 0, st>>>(bsum, bcnt, nblk, out_loss,
                                              reinterpret_cast<long long*>(out_n_valid));
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  return FLCE_OK;
}

flce_status flce_device_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return FLCE_ERR_CUDA;
  }
  int e = 0;
  if (cudaMemcpyFromSymbol(&e, g_device_error, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return FLCE_ERR_CUDA;
  }
  if (e != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    return FLCE_ERR_TIMEOUT;
  }
  return FLCE_OK;
}

flce_status flce_selftest_wait_timeout(int64_t limit_cycles, void* stream) {
  if (limit_cycles <= 0 || limit_cycles > WAIT_LIMIT_CYCLES) return FLCE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* err = nullptr;
  FLCE_CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_device_error));
  int* gave_up = nullptr;
  FLCE_CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&gave_up), g_selftest_flag));
  wait_selftest_kernel<<<1, 32, 0, st>>>(static_cast<long long>(limit_cycles), err, gave_up);
  FLCE_CUDA_TRY(cudaGetLastError());
  int h_gave_up = 0;
  FLCE_CUDA_TRY(cudaMemcpyAsync(&h_gave_up, gave_up, sizeof(int), cudaMemcpyDeviceToHost, st));
  FLCE_CUDA_TRY(cudaStreamSynchronize(st));
  return h_gave_up ? FLCE_OK : FLCE_ERR_CUDA;
}

flce_status flce_set_option(flce_option o, int64_t value) {
  const int i = static_cast<int>(o);
  if (i < 0 || i >= FLCE_OPT_COUNT) return FLCE_ERR_INVALID_ARG;
  if (value < kOptionDefs[i].lo || value > kOptionDefs[i].hi) return FLCE_ERR_INVALID_ARG;
  init_options();
  g_options[i].store(value);
  return FLCE_OK;
}

flce_status flce_get_option(flce_option o, int64_t* value) {
  const int i = static_cast<int>(o);
  if (i < 0 || i >= FLCE_OPT_COUNT || value == nullptr) return FLCE_ERR_INVALID_ARG;
  *value = opt(o);
  return FLCE_OK;
}

flce_status flce_profile_enable(int enable) {
  for (auto& r : g_prof_pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_prof_pending.clear();
  for (int k = 0; k < K_COUNT; ++k) {
    g_prof_ms[k] = 0.0;
    g_prof_n[k] = 0;
  }
  g_prof_on = enable != 0;
  return FLCE_OK;
}

int flce_profile_num_kinds(void) { return K_COUNT; }

const char* flce_profile_kind_name(int kind) {
  return (kind >= 0 && kind < K_COUNT) ? kKindNames[kind] : nullptr;
}

flce_status flce_profile_read(int kind, double* total_ms, int64_t* launches) {
  if (kind < 0 || kind >= K_COUNT || !total_ms || !launches) return FLCE_ERR_INVALID_ARG;
  flce_status s = FLCE_OK;
  for (auto& r : g_prof_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      cudaGetLastError();
      s = FLCE_ERR_CUDA;
    } else {
      g_prof_ms[r.kind] += ms;
      g_prof_n[r.kind] += 1;
    }
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_prof_pending.clear();
  *total_ms = g_prof_ms[kind];
  *launches = g_prof_n[kind];
  return s;
}

}  // extern "C"

// ===========================================================================
// Forward for callers that cannot allocate device memory.
//
// Some callers are not allowed to allocate at all: inference runtimes that
// own every byte of device memory through a fixed pool of their own (any other
// allocation breaks their accounting or fails outright), and services that
// must keep a constant memory footprint from start-up on (an allocation on
// the hot path could fail under memory pressure, or stall on the allocator).
// This entry point serves them: it takes the same inputs and outputs as
// flce_forward, but its scratch lives in one file-scope device array that the
// library owns, so nothing is allocated or freed by any call.
//
// The array is a fixed 16 MiB, resident on every device that loads this
// library until the process exits.  On the host its name is only a stand-in
// for the device copy, never a device address: the address is looked up with
// cudaGetSymbolAddress once per device and context (device code could name
// the array directly, host code must not).
namespace {
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
}  // namespace

static __device__ __align__(256) unsigned char g_flce_static_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxStaticScratchDevices = 128;
struct StaticScratchSlot {
  unsigned long long ctx_id = 0;  // context the address belongs to (0: none yet)
  void* addr = nullptr;
};
std::mutex g_static_scratch_mu;
StaticScratchSlot g_static_scratch[kMaxStaticScratchDevices];

// Unique id of the calling thread's current context (cuCtxGetId), or 0 when
// there is none yet.  A context rebuilt after a reset gets a new id, and a
// module reload in it may put the array at another address.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  return ctx == nullptr || get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_flce_static_scratch in the current device's context.
// Set-up runs once per device and context: on the first call with that
// device current, and again only if the context was rebuilt since (a device
// reset), since the array may then sit at another address.
flce_status static_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FLCE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxStaticScratchDevices) return FLCE_ERR_UNSUPPORTED;
  unsigned long long id = 0;
  if (!current_context_id(&id)) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  StaticScratchSlot& slot = g_static_scratch[dev];
  if (id == 0 || slot.addr == nullptr || slot.ctx_id != id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_flce_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FLCE_ERR_CUDA;
    }
    // the lookup creates the device's primary context if there was none
    if (id == 0 && (!current_context_id(&id) || id == 0)) return FLCE_ERR_CUDA;
    slot.ctx_id = id;
    slot.addr = p;
  }
  *out = slot.addr;
  return FLCE_OK;
}
}  // namespace

extern "C" flce_status flce_forward_static_scratch(const flce_bf16* h, const flce_bf16* W,
                                                   const int64_t* targets, const float* weights,
                                                   int64_t N, int64_t H, int64_t V,
                                                   int64_t chunk_rows, int64_t ignore_index,
                                                   float* out_logp, float* out_lse, float* out_loss,
                                                   int64_t* out_n_valid, void* stream) {
  (void)chunk_rows;
  if (!sizes_ok(N, H, V)) return FLCE_ERR_INVALID_ARG;
  const int cg = cta_group();
  // the vocabulary-split partials get what the array leaves after the
  // per-row target logits and block sums (fewer splits, same results up to
  // fp32 rounding of the combine)
  const FwdPlan f1 = plan_forward_call(N, H, V, device_workers(cg), BM * cg, 0);  // one split
  const size_t fixed = fwd_layout(N, f1).total - align256(static_cast<size_t>(std::max<int64_t>(N, 0)) * 8);
  if (fixed + align256(static_cast<size_t>(std::max<int64_t>(N, 0)) * 8) > kStaticScratchBytes)
    return FLCE_ERR_UNSUPPORTED;
  const size_t cap = kStaticScratchBytes - fixed - 256;  // 256: alignment of the partials block
  if (fwd_layout(N, plan_forward_call(N, H, V, device_workers(cg), BM * cg, cap)).total > kStaticScratchBytes)
    return FLCE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const flce_status s = static_scratch_address(&scratch);
  if (s != FLCE_OK) return s;
  // Every scratch word is written by this call before it is read (target
  // slots by the prep kernel, partials by the GEMM, block sums by the
  // combine, the validation counter by a memset), so stale contents of an
  // earlier call never leak into the result.
  return forward_impl(h, W, targets, weights, N, H, V, ignore_index, nullptr, out_logp, out_lse,
                      out_loss, out_n_valid, scratch, kStaticScratchBytes, stream, cap);
}
