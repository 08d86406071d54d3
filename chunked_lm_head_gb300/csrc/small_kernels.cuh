// libflce: the CUDA-core kernels around the GEMMs (target prep, split-
// vocabulary combine, deterministic loss reduction, split-K reduction of dH,
// row compaction, the one-call dlogits pass, distillation and GRPO
// reductions, e4m3 quantisation) and the device error word.
#pragma once

#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "gemm.cuh"

namespace flce {

__device__ int g_device_error;  // bit DEVERR_TIMEOUT: a bounded wait ran out
__device__ int g_selftest_flag;  // verdict of wait_selftest_kernel

constexpr float kLn2 = 0.6931471805599453f;
constexpr int SMALL_THREADS = 256;

// ------------------------------------------------------------ small kernels

// Target prep (mask step): the target-logit slots start as NaN so that a row
// whose target is never met in any vocabulary tile (out of range) yields NaN;
// optionally counts targets outside [0, V) that are not ignore_index.
__global__ void prep_kernel(const int64_t* __restrict__ targets, int N, int V, long long ignore,
                            float* __restrict__ zt, int* bad) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < N) {
    if (zt != nullptr) zt[i] = __int_as_float(0x7fc00000);
    if (bad != nullptr) {
      const long long t = targets[i];
      if (t != ignore && (t < 0 || t >= V)) atomicAdd(bad, 1);
    }
  }
}

// This block's sum of `contrib` and of `cnt` over its SMALL_THREADS threads,
// in a fixed order (warp shuffles, then the warps in turn), stored at
// blk_sum / blk_cnt[blockIdx.x].  Every thread of the block must call it.
__device__ __forceinline__ void block_sum_store(double contrib, long long cnt, double* blk_sum,
                                                long long* blk_cnt) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    contrib += __shfl_down_sync(0xffffffffu, contrib, off);
    cnt += __shfl_down_sync(0xffffffffu, cnt, off);
  }
  __shared__ double ssum[SMALL_THREADS / 32];
  __shared__ long long scnt[SMALL_THREADS / 32];
  if ((threadIdx.x & 31) == 0) {
    ssum[threadIdx.x >> 5] = contrib;
    scnt[threadIdx.x >> 5] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double a = 0.0;
    long long c = 0;
    for (int w = 0; w < SMALL_THREADS / 32; ++w) {
      a += ssum[w];
      c += scnt[w];
    }
    blk_sum[blockIdx.x] = a;
    blk_cnt[blockIdx.x] = c;
  }
}

// Split-vocabulary combine: lse = M + log sum_s s_s 2^(m_s - M) (log2 domain,
// converted to natural log), logp = z_t - lse on non-ignored rows, and this
// block's share of sum(w * logp) and of the valid-row count.
// Rows [0, N) of the arrays passed (callers offset them for a row range),
// or with `ri` the rows ri[0..N) of the whole arrays; `stride` is the
// distance between two splits' partials of one row.  skip_ignored: the
// forward skipped the ignored rows, whose lse becomes NaN.
template <bool kLong>
__global__ void combine_kernel(const float2* __restrict__ part, int S, int stride, int N,
                               const float* __restrict__ zt, const int64_t* __restrict__ targets,
                               const float* __restrict__ weights, long long ignore,
                               float* __restrict__ out_logp, float* __restrict__ out_lse,
                               double* __restrict__ blk_sum, long long* __restrict__ blk_cnt,
                               const int* __restrict__ ri, int skip_ignored = 0) {
  using idx_t = typename std::conditional<kLong, long long, int>::type;
  const int j = blockIdx.x * SMALL_THREADS + threadIdx.x;
  double contrib = 0.0;
  long long cnt = 0;
  const int i = j < N ? (ri ? ri[j] : j) : 0;  // the j-th row of this range
  if (j < N && skip_ignored && targets[i] == ignore) {  // forward skipped: lse not computed
    if (out_lse) out_lse[i] = __int_as_float(0x7fc00000);
    if (out_logp) out_logp[i] = 0.f;
  } else if (j < N) {
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, part[static_cast<idx_t>(s) * stride + i].x);
    float sum = 0.f;
    for (int s = 0; s < S; ++s) {
      const float2 q = part[static_cast<idx_t>(s) * stride + i];
      sum += q.y * exp2f(q.x - M);
    }
    const float lse = (M + log2f(sum)) * kLn2;
    const long long t = targets[i];
    const bool valid = t != ignore;
    const float logp = valid ? zt[i] - lse : 0.f;
    if (out_lse) out_lse[i] = lse;
    if (out_logp) out_logp[i] = logp;
    if (valid) {
      cnt = 1;
      contrib = static_cast<double>(weights ? weights[i] : 1.f) * static_cast<double>(logp);
    }
  }
  block_sum_store(contrib, cnt, blk_sum, blk_cnt);
}

// Loss = -sum(w logp) / n_valid over the block partials, in a fixed order
// (deterministic run to run); 0 when n_valid == 0.
__global__ void final_kernel(const double* __restrict__ blk_sum, const long long* __restrict__ blk_cnt,
                             int nblk, float* out_loss, long long* out_n_valid) {
  double a = 0.0;
  long long c = 0;
  for (int b = threadIdx.x; b < nblk; b += SMALL_THREADS) {
    a += blk_sum[b];
    c += blk_cnt[b];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_down_sync(0xffffffffu, a, off);
    c += __shfl_down_sync(0xffffffffu, c, off);
  }
  __shared__ double ssum[SMALL_THREADS / 32];
  __shared__ long long scnt[SMALL_THREADS / 32];
  if ((threadIdx.x & 31) == 0) {
    ssum[threadIdx.x >> 5] = a;
    scnt[threadIdx.x >> 5] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    long long n = 0;
    for (int w = 0; w < SMALL_THREADS / 32; ++w) {
      s += ssum[w];
      n += scnt[w];
    }
    if (out_n_valid) *out_n_valid = n;
    if (out_loss) *out_loss = n > 0 ? static_cast<float>(-s / static_cast<double>(n)) : 0.f;
  }
}

// dH[row, :] = bf16(sum over k-splits of the fp32 partials), split order
// fixed; row = row_idx[first + r] for a compacted pass (row count read from
// dyn_count), else row0 + r.
template <bool kLong>
__global__ void dh_reduce_kernel(const float* __restrict__ part, int splits, int rows, int rows_cap,
                                 int H, int row0, uint16_t* __restrict__ dH,
                                 const int* __restrict__ row_idx, const int* __restrict__ dyn_count,
                                 int first) {
  using idx_t = typename std::conditional<kLong, long long, int>::type;
  if (dyn_count != nullptr) rows = max(0, min(*dyn_count - first, rows_cap));
  const int h4 = H / 4;
  const idx_t total = static_cast<idx_t>(rows) * h4;
  for (idx_t e = static_cast<idx_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<idx_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(e / h4);
    const int c = static_cast<int>(e - static_cast<idx_t>(r) * h4) * 4;
    float4 s = *reinterpret_cast<const float4*>(part + static_cast<idx_t>(r) * H + c);
    for (int k = 1; k < splits; ++k) {
      const float4 q =
          *reinterpret_cast<const float4*>(part + (static_cast<idx_t>(k) * rows_cap + r) * H + c);
      s.x += q.x;
      s.y += q.y;
      s.z += q.z;
      s.w += q.w;
    }
    const int out_row = row_idx != nullptr ? row_idx[first + r] : row0 + r;
    *reinterpret_cast<uint2*>(dH + static_cast<idx_t>(out_row) * H + c) =
        make_uint2(pack_bf16x2(s.x, s.y), pack_bf16x2(s.z, s.w));
  }
}

// ---- row compaction: the indices of the non-ignored rows, in row order
constexpr int COMPACT_ROWS_PER_THREAD = 4;
constexpr int COMPACT_ROWS_PER_BLOCK = SMALL_THREADS * COMPACT_ROWS_PER_THREAD;

__global__ void compact_count_kernel(const int64_t* __restrict__ targets, int N, long long ignore,
                                     int* __restrict__ blk_cnt) {
  const int base = blockIdx.x * COMPACT_ROWS_PER_BLOCK + threadIdx.x * COMPACT_ROWS_PER_THREAD;
  int c = 0;
#pragma unroll
  for (int k = 0; k < COMPACT_ROWS_PER_THREAD; ++k)
    if (base + k < N && targets[base + k] != ignore) ++c;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_down_sync(0xffffffffu, c, off);
  __shared__ int wsum[SMALL_THREADS / 32];
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int w = 0; w < SMALL_THREADS / 32; ++w) s += wsum[w];
    blk_cnt[blockIdx.x] = s;
  }
}

// tail != 0: idx is a permutation of all N rows, the ignored rows (in row
// order) after the non-ignored ones.
__global__ void compact_write_kernel(const int64_t* __restrict__ targets, int N, long long ignore,
                                     const int* __restrict__ blk_cnt, int nblk, int* __restrict__ idx,
                                     int* __restrict__ total, int tail) {
  __shared__ int s_off, s_total;
  __shared__ int wtot[SMALL_THREADS / 32];
  if (threadIdx.x == 0) {
    int o = 0, all = 0;
    for (int b = 0; b < nblk; ++b) {
      if (b < static_cast<int>(blockIdx.x)) o += blk_cnt[b];
      all += blk_cnt[b];
    }
    s_off = o;
    s_total = all;
    if (static_cast<int>(blockIdx.x) == nblk - 1) *total = all;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int base = blockIdx.x * COMPACT_ROWS_PER_BLOCK + threadIdx.x * COMPACT_ROWS_PER_THREAD;
  bool keep[COMPACT_ROWS_PER_THREAD];
  int c = 0;
#pragma unroll
  for (int k = 0; k < COMPACT_ROWS_PER_THREAD; ++k) {
    keep[k] = base + k < N && targets[base + k] != ignore;
    c += keep[k] ? 1 : 0;
  }
  int x = c;  // inclusive scan over the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) wtot[warp] = x;
  __syncthreads();
  int pos = s_off + x - c;
  for (int w = 0; w < warp; ++w) pos += wtot[w];
#pragma unroll
  for (int k = 0; k < COMPACT_ROWS_PER_THREAD; ++k) {
    if (keep[k])
      idx[pos++] = base + k;
    else if (tail && base + k < N)  // pos = non-ignored rows before this one
      idx[s_total + base + k - pos] = base + k;
  }
}

// hc[r, :] = h[idx[first + r], :] for the pass's rows (min(*count - first,
// cap), or min(N - first, cap) without a count); zero rows up to the next
// 64-row boundary (the dW pass reads whole 64-row K blocks).
__global__ void gather_rows_kernel(const uint16_t* __restrict__ h, int H, const int* __restrict__ idx,
                                   const int* __restrict__ count, int N, int first, int cap,
                                   uint16_t* __restrict__ hc) {
  const int rows = max(0, min((count ? *count : N) - first, cap));
  const int pad = min((rows + 63) / 64 * 64, cap);
  const int h8 = H / 8;
  const long long total = static_cast<long long>(pad) * h8;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(e / h8);
    const int c = static_cast<int>(e - static_cast<long long>(r) * h8) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) v = *reinterpret_cast<const uint4*>(h + static_cast<long long>(idx[first + r]) * H + c);
    *reinterpret_cast<uint4*>(hc + static_cast<long long>(r) * H + c) = v;
  }
}

// dH rows of the ignored rows, idx[*count .. N) of a permutation that puts
// the non-ignored rows first, set to zero.
__global__ void zero_tail_rows_kernel(uint16_t* __restrict__ dH, int H, const int* __restrict__ idx,
                                      const int* __restrict__ count, int N) {
  const int first = *count;
  const int h8 = H / 8;
  const long long total = static_cast<long long>(N - first) * h8;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int j = first + static_cast<int>(e / h8);
    const int c = static_cast<int>(e % h8) * 8;
    *reinterpret_cast<uint4*>(dH + static_cast<long long>(idx[j]) * H + c) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Distillation combine: student and teacher log-sum-exps from the split
// partials, KL(p_t || p_s) = C / S_t - lse_t + lse_s per row, and the block's
// share of sum(m w kl) and of the counted rows (targets == NULL: all rows).
// skip_ignored: the forward skipped the ignored rows (lse NaN, kl 0).
template <bool kLong>
__global__ void kd_combine_kernel(const float2* __restrict__ ps, const float2* __restrict__ pt,
                                  const float* __restrict__ pc, int S, int N,
                                  const int64_t* __restrict__ targets,
                                  const float* __restrict__ weights, long long ignore,
                                  float* __restrict__ out_kl, float* __restrict__ out_lse_s,
                                  float* __restrict__ out_lse_t, double* __restrict__ blk_sum,
                                  long long* __restrict__ blk_cnt, int skip_ignored = 0) {
  using idx_t = typename std::conditional<kLong, long long, int>::type;
  const int i = blockIdx.x * SMALL_THREADS + threadIdx.x;
  double contrib = 0.0;
  long long cnt = 0;
  if (i < N && skip_ignored && targets != nullptr && targets[i] == ignore) {
    // the forward skipped this row: its log-sum-exps were not computed
    if (out_kl) out_kl[i] = 0.f;
    if (out_lse_s) out_lse_s[i] = __int_as_float(0x7fc00000);
    if (out_lse_t) out_lse_t[i] = __int_as_float(0x7fc00000);
  } else if (i < N) {
    float Ms = -INFINITY, Mt = -INFINITY;
    for (int s = 0; s < S; ++s) {
      Ms = fmaxf(Ms, ps[static_cast<idx_t>(s) * N + i].x);
      Mt = fmaxf(Mt, pt[static_cast<idx_t>(s) * N + i].x);
    }
    float Ss = 0.f, St = 0.f, Cc = 0.f;
    for (int s = 0; s < S; ++s) {
      const idx_t o = static_cast<idx_t>(s) * N + i;
      Ss += ps[o].y * exp2f(ps[o].x - Ms);
      const float r = exp2f(pt[o].x - Mt);
      St += pt[o].y * r;
      Cc += pc[o] * r;
    }
    const float lse_s = (Ms + log2f(Ss)) * kLn2;
    const float lse_t = (Mt + log2f(St)) * kLn2;
    const bool valid = targets == nullptr || targets[i] != ignore;
    const float kl = valid ? Cc / St - lse_t + lse_s : 0.f;
    if (out_kl) out_kl[i] = kl;
    if (out_lse_s) out_lse_s[i] = lse_s;
    if (out_lse_t) out_lse_t[i] = lse_t;
    if (valid) {
      cnt = 1;
      // the final kernel negates the sum (it serves -sum(w logp) for the
      // cross-entropy), so the KL enters with a minus sign
      contrib = -static_cast<double>(weights ? weights[i] : 1.f) * static_cast<double>(kl);
    }
  }
  block_sum_store(contrib, cnt, blk_sum, blk_cnt);
}

// Jensen-Shannon combine: per row, the split partials (log2 units) summed in
// split order -> jsd = ln2 (beta A_t + (1 - beta) A_s) (0 on masked rows) and
// kl_sm = ln2 A_s = KL(p_s || M); block sums of -w jsd and of the row count
// for the deterministic loss.  skip_ignored: the forward skipped the
// ignored rows (jsd 0, kl_sm NaN).
template <bool kLong>
__global__ void jsd_combine_kernel(const float2* __restrict__ pj, int S, int N,
                                   const int64_t* __restrict__ targets,
                                   const float* __restrict__ weights, long long ignore, float beta,
                                   float* __restrict__ out_jsd, float* __restrict__ out_kl_sm,
                                   double* __restrict__ blk_sum, long long* __restrict__ blk_cnt,
                                   int skip_ignored = 0) {
  using idx_t = typename std::conditional<kLong, long long, int>::type;
  const int i = blockIdx.x * SMALL_THREADS + threadIdx.x;
  double contrib = 0.0;
  long long cnt = 0;
  if (i < N && skip_ignored && targets != nullptr && targets[i] == ignore) {
    if (out_jsd) out_jsd[i] = 0.f;  // the forward skipped this row
    if (out_kl_sm) out_kl_sm[i] = __int_as_float(0x7fc00000);
  } else if (i < N) {
    float at = 0.f, as = 0.f;
    for (int s = 0; s < S; ++s) {
      const float2 q = pj[static_cast<idx_t>(s) * N + i];
      at += q.x;
      as += q.y;
    }
    const bool valid = targets == nullptr || targets[i] != ignore;
    const float jsd = valid ? kLn2 * (beta * at + (1.f - beta) * as) : 0.f;
    if (out_jsd) out_jsd[i] = jsd;
    if (out_kl_sm) out_kl_sm[i] = kLn2 * as;
    if (valid) {
      cnt = 1;
      contrib = -static_cast<double>(weights ? weights[i] : 1.f) * static_cast<double>(jsd);
    }
  }
  block_sum_store(contrib, cnt, blk_sum, blk_cnt);
}

// GRPO per-token objective on the sampled tokens' log-probs (one thread per
// row; flce_grpo_token_loss states the formula): the masked token loss, the
// weights -d(token loss)/d(logp) for the backward, and this block's sums of
// -(token loss) and of the mask (the final kernel negates the sum).  Rows
// [0, N) of the arrays passed, or with `ri` the rows ri[0..N) of the whole
// arrays.
__global__ void grpo_token_kernel(const float* __restrict__ logp, const float* __restrict__ old_logp,
                                  const float* __restrict__ ref_logp, const float* __restrict__ adv,
                                  const int64_t* __restrict__ targets, int N, long long ignore,
                                  float eps_low, float eps_high, float beta,
                                  float* __restrict__ out_tok, float* __restrict__ out_w,
                                  double* __restrict__ blk_sum, long long* __restrict__ blk_cnt,
                                  const int* __restrict__ ri = nullptr) {
  const int j = blockIdx.x * SMALL_THREADS + threadIdx.x;
  double contrib = 0.0;
  long long cnt = 0;
  if (j < N) {
    const int i = ri ? ri[j] : j;  // the j-th row of this range (arrays not offset with ri)
    const bool valid = targets == nullptr || targets[i] != ignore;
    float tok = 0.f, wt = 0.f;
    if (valid) {
      const float lp = logp[i];
      const float A = adv[i];
      const float r = old_logp != nullptr ? expf(lp - old_logp[i]) : 1.f;
      const float un = r * A;
      const float cl = fminf(fmaxf(r, 1.f - eps_low), 1.f + eps_high) * A;
      const float obj = fminf(un, cl);
      const float dobj = un <= cl ? un : 0.f;  // the clipped branch is constant in logp
      float kl = 0.f, dkl = 0.f;
      if (ref_logp != nullptr && beta != 0.f) {
        const float d = ref_logp[i] - lp;
        const float em1 = expm1f(d);
        kl = em1 - d;  // exp(d) - d - 1 without cancellation near d = 0
        dkl = -em1;    // d kl / d logp = 1 - exp(d)
      }
      tok = beta * kl - obj;
      wt = dobj - beta * dkl;
      cnt = 1;
      contrib = -static_cast<double>(tok);
    }
    if (out_tok) out_tok[i] = tok;
    if (out_w) out_w[i] = wt;
  }
  block_sum_store(contrib, cnt, blk_sum, blk_cnt);
}

// dlogits of one row block from the forward's stored exponentials, in place:
// E[r][v] = 2^(u log2e - mx[r][v / 32]) (bf16) becomes
//   D[r][v] = (E 2^(mx - lse log2e) - [v == t]) * m * w * g * f'(z),
// g = grad_scale / max(n_valid, 1) with n_valid read on the device.  The
// target column is formed from the exact fp32 target logit instead (so that
// p_t - 1 keeps its precision when p_t is near 1).  Grid: (column blocks of
// 256 threads x 32 columns, rows); a thread's 32 columns are one chunk.
// Local row r is row row0 + r, or with `ri` row ri[r] of a block whose
// non-ignored rows come first: rows from the next 64-row boundary past them
// are read by neither the dH nor the dW GEMM and are skipped.
constexpr int FUSED_COLS_PER_THREAD = 32;

template <bool kLong>
__global__ void fused_dlogits_kernel(uint16_t* __restrict__ E, const float* __restrict__ mx, int ldD,
                                     int V, int row0, const int* __restrict__ ri,
                                     const int64_t* __restrict__ targets,
                                     const float* __restrict__ weights, const float* __restrict__ lse,
                                     const float* __restrict__ zt, long long ignore,
                                     const int* __restrict__ n_valid, float grad_scale, int tf_softcap,
                                     float tf_a, float tf_b, float tf_d) {
  using idx_t = typename std::conditional<kLong, long long, int>::type;
  const int r = blockIdx.y;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * FUSED_COLS_PER_THREAD;
  if (c >= ldD) return;
  if (ri != nullptr && r >= (*n_valid - row0 + 63) / 64 * 64) return;  // row0: the block's first position
  const int row = ri ? ri[r] : row0 + r;
  const long long t = targets[row];
  const bool valid = t != ignore;
  const float g = grad_scale / fmaxf(1.f, static_cast<float>(*n_valid));
  const float scale = valid ? (weights ? weights[row] : 1.f) * g : 0.f;
  uint4* slot = reinterpret_cast<uint4*>(E + static_cast<idx_t>(r) * ldD + c);
  if (scale == 0.f) {  // ignored row (its exponentials may never have been written) or zero weight
#pragma unroll
    for (int h = 0; h < 4; ++h) slot[h] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  uint4 q[4] = {slot[0], slot[1], slot[2], slot[3]};
  const float cmL = mx[static_cast<idx_t>(r) * (ldD / 32) + c / 32];
  const float nlse2 = -lse[row] * kLog2e;
  const float base = ex2_approx(cmL + nlse2);  // 2^(chunk max - lse), both x log2(e)
  const float lin = tf_softcap ? 1.f : tf_a;    // linear transforms: du/dz = tf_a
  const long long tj = t - c;                   // target column inside this thread's 32, if any
  if (!tf_softcap && c + 32 <= V && (tj < 0 || tj >= 32)) {
    // the common chunk: inside the vocabulary, no target column, linear
    // transform: D = E * 2^(max - lse) * scale * a, two columns per step
    const float kf = base * scale * lin;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t w4[4] = {q[h].x, q[h].y, q[h].z, q[h].w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        o[k] = pack_bf16x2(__uint_as_float(w4[k] << 16) * kf, __uint_as_float(w4[k] & 0xffff0000u) * kf);
      slot[h] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    return;
  }
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    uint32_t w4[4] = {q[h].x, q[h].y, q[h].z, q[h].w};
    float d[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t bits = (k & 1) ? (w4[k >> 1] & 0xffff0000u) : (w4[k >> 1] << 16);
      const float ev = __uint_as_float(bits);
      const int j = 8 * h + k;
      float dk = 0.f;
      if (scale != 0.f && c + j < V) {
        if (tj == j) {
          const float ut = zt[row];
          const float pt = ex2_approx(fmaf(ut, kLog2e, nlse2));
          const float fd = tf_softcap ? tf_d * (1.f - (ut / tf_b) * (ut / tf_b)) : lin;
          dk = (pt - 1.f) * scale * fd;
        } else if (ev > 0.f) {
          float fd = lin;
          if (tf_softcap) {  // u = ln(E) + chunk max, tanh(a z) = u / b
            const float u = (__log2f(ev) + cmL) * kLn2;
            fd = tf_d * (1.f - (u / tf_b) * (u / tf_b));
          }
          dk = ev * base * scale * fd;
        }
      }
      d[k] = dk;
    }
    q[h].x = pack_bf16x2(d[0], d[1]);
    q[h].y = pack_bf16x2(d[2], d[3]);
    q[h].z = pack_bf16x2(d[4], d[5]);
    q[h].w = pack_bf16x2(d[6], d[7]);
  }
#pragma unroll
  for (int h = 0; h < 4; ++h) slot[h] = q[h];
}

// Per-row e4m3 quantisation (one warp per row): scale = max|x| / 448 (1 for
// an all-zero row), q = e4m3(x / scale), round to nearest even, saturating.
__global__ void quantize_e4m3_rows_kernel(const uint16_t* __restrict__ x, long long rows, int cols,
                                          uint8_t* __restrict__ q, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  const uint16_t* xr = x + row * cols;
  float amax = 0.f;
  for (int c = lane * 8; c < cols; c += 256) {
    const uint4 u = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[k] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[k] & 0xffff0000u)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (lane == 0) scale[row] = s;
  uint8_t* qr = q + row * cols;
  for (int c = lane * 8; c < cols; c += 256) {
    const uint4 u = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = __nv_cvt_float_to_fp8(__fdiv_rn(__uint_as_float(w[k] << 16), s), __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float_to_fp8(__fdiv_rn(__uint_as_float(w[k] & 0xffff0000u), s), __NV_SATFINITE, __NV_E4M3);
      o[k >> 1] |= (lo | (hi << 8)) << (16 * (k & 1));
    }
    *reinterpret_cast<uint2*>(qr + c) = make_uint2(o[0], o[1]);
  }
}

// Self-test of the bounded wait: one warp waits on an mbarrier that nothing
// arrives on, through the same wait routine the GEMM pipelines use, with a
// short limit; it must give up, raise the device error word and return.
// In-place scale of gradients by a scalar held in device memory (the
// incoming gradient of a loss, without a host synchronisation).  A scale of
// exactly 1 leaves the data untouched and moves no bytes.  Grid-stride over
// 16-byte vectors, then a scalar tail.
__global__ void scale_bf16_kernel(__nv_bfloat16* __restrict__ x, long long n, const float* __restrict__ scale) {
  const float s = *scale;
  if (s == 1.f) return;
  const long long nv = n / 8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  uint4* xv = reinterpret_cast<uint4*>(x);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nv; i += stride) {
    uint4 u = xv[i];
    __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      b[j] = __floats2bfloat162_rn(f.x * s, f.y * s);
    }
    xv[i] = u;
  }
  for (long long i = nv * 8 + blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n; i += stride)
    x[i] = __float2bfloat16_rn(__bfloat162float(x[i]) * s);
}

__global__ void scale_f32_kernel(float* __restrict__ x, long long n, const float* __restrict__ scale) {
  const float s = *scale;
  if (s == 1.f) return;
  const long long nv = n / 4;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  float4* xv = reinterpret_cast<float4*>(x);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nv; i += stride) {
    float4 v = xv[i];
    v.x *= s;
    v.y *= s;
    v.z *= s;
    v.w *= s;
    xv[i] = v;
  }
  for (long long i = nv * 4 + blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n; i += stride)
    x[i] *= s;
}

__global__ void wait_selftest_kernel(long long limit_cycles, int* err, int* gave_up) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = wait_bar(smem_u32(&bar), 0, &abort_flag, err, limit_cycles);
    *gave_up = ok ? 0 : 1;
  }
}

}  // namespace flce
