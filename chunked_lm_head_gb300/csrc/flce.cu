// libflce: C-ABI entry points, host-side planning, tensor maps and the small
// CUDA-core kernels (target prep, split-vocabulary combine, deterministic loss
// reduction, split-K reduction of dH).  The tensor-core work lives in
// gemm.cuh.  See include/flce.h for the contract of every entry point.
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
template <bool kLong>
__global__ void kd_combine_kernel(const float2* __restrict__ ps, const float2* __restrict__ pt,
                                  const float* __restrict__ pc, int S, int N,
                                  const int64_t* __restrict__ targets,
                                  const float* __restrict__ weights, long long ignore,
                                  float* __restrict__ out_kl, float* __restrict__ out_lse_s,
                                  float* __restrict__ out_lse_t, double* __restrict__ blk_sum,
                                  long long* __restrict__ blk_cnt) {
  using idx_t = typename std::conditional<kLong, long long, int>::type;
  const int i = blockIdx.x * SMALL_THREADS + threadIdx.x;
  double contrib = 0.0;
  long long cnt = 0;
  if (i < N) {
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
// for the deterministic loss.
template <bool kLong>
__global__ void jsd_combine_kernel(const float2* __restrict__ pj, int S, int N,
                                   const int64_t* __restrict__ targets,
                                   const float* __restrict__ weights, long long ignore, float beta,
                                   float* __restrict__ out_jsd, float* __restrict__ out_kl_sm,
                                   double* __restrict__ blk_sum, long long* __restrict__ blk_cnt) {
  using idx_t = typename std::conditional<kLong, long long, int>::type;
  const int i = blockIdx.x * SMALL_THREADS + threadIdx.x;
  double contrib = 0.0;
  long long cnt = 0;
  if (i < N) {
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
// -(token loss) and of the mask (the final kernel negates the sum).
__global__ void grpo_token_kernel(const float* __restrict__ logp, const float* __restrict__ old_logp,
                                  const float* __restrict__ ref_logp, const float* __restrict__ adv,
                                  const int64_t* __restrict__ targets, int N, long long ignore,
                                  float eps_low, float eps_high, float beta,
                                  float* __restrict__ out_tok, float* __restrict__ out_w,
                                  double* __restrict__ blk_sum, long long* __restrict__ blk_cnt) {
  const int i = blockIdx.x * SMALL_THREADS + threadIdx.x;
  double contrib = 0.0;
  long long cnt = 0;
  if (i < N) {
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
  uint4 q[4] = {slot[0], slot[1], slot[2], slot[3]};
  const float cmL = mx[static_cast<idx_t>(r) * (ldD / 32) + c / 32];
  const float nlse2 = -lse[row] * kLog2e;
  const float base = ex2_approx(cmL + nlse2);  // 2^(chunk max - lse), both x log2(e)
  const float lin = tf_softcap ? 1.f : tf_a;    // linear transforms: du/dz = tf_a
  const long long tj = t - c;                   // target column inside this thread's 32, if any
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

// ====================================================================== host
namespace {

using namespace flce;

constexpr int kDefaultSms = 152;

enum Kind {
  K_PREP, K_FWD, K_COMBINE, K_FINAL, K_DLOGITS, K_DH, K_DH_REDUCE, K_DW, K_COMPACT, K_GATHER,
  K_KD_FWD, K_KD_DLOGITS, K_QUANT, K_JSD_FWD, K_JSD_DLOGITS, K_GRPO, K_COUNT
};
const char* const kKindNames[K_COUNT] = {"prep_targets",  "fwd_logits_lse", "fwd_combine",
                                         "fwd_loss",      "bwd_dlogits",    "bwd_dH",
                                         "bwd_dH_reduce", "bwd_dW",         "bwd_compact_rows",
                                         "bwd_gather_rows", "kd_fwd_logits",  "kd_bwd_dlogits",
                                         "quantize_e4m3", "jsd_fwd_terms",  "jsd_bwd_dlogits",
                                         "grpo_token_loss"};

struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};
bool g_prof_on = false;
std::vector<ProfRec> g_prof_pending;
double g_prof_ms[K_COUNT];
long long g_prof_n[K_COUNT];

struct ProfScope {
  int kind;
  cudaStream_t st;
  cudaEvent_t a = nullptr, b = nullptr;
  ProfScope(int k, cudaStream_t s) : kind(k), st(s) {
    if (g_prof_on && cudaEventCreate(&a) == cudaSuccess && cudaEventCreate(&b) == cudaSuccess)
      cudaEventRecord(a, st);
  }
  ~ProfScope() {
    if (b != nullptr) {
      cudaEventRecord(b, st);
      g_prof_pending.push_back({kind, a, b});
    }
  }
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
inline long long round_up(long long a, long long b) { return ceil_div(a, b) * b; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return kDefaultSms;
  }
  return n;
}

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
// DRAM reads of W are twice as high).  FLCE_FWD_BLOCK_ROWS overrides it
// (rounded up to a tile; 0: all rows in one launch).
long long fwd_block_rows(long long N, int tm) {
  N = std::max(1LL, N);
  long long b = 16LL * tm;
  if (const char* e = std::getenv("FLCE_FWD_BLOCK_ROWS")) {
    b = std::atoll(e);
    if (b <= 0) return N;
  }
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
  // FLCE_FWD_SPLITS=s pins the number of vocabulary splits (tests compare
  // split counts; results must not depend on them beyond fp32 rounding)
  if (const char* e = std::getenv("FLCE_FWD_SPLITS")) {
    const int want = std::max(1, std::min(std::min(std::atoi(e), f.n_tiles), smax));
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
};

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
// blocks each).  FLCE_DH_SPLITS overrides it in plans made after it is set.
int dh_split_count(long long tiles, long long kb, int workers) {
  if (const char* e = std::getenv("FLCE_DH_SPLITS")) {
    const long long s = std::atoll(e);
    if (s >= 1) return static_cast<int>(std::min<long long>({s, 16, std::max(1LL, kb / 8)}));
  }
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
bool plan_candidate(BwdPlan& b, long long N, long long H, long long V, long long R,
                    long long budget, int workers, int tm) {
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
  const long long dh_tiles = ceil_div(R, tm) * ceil_div(H, BN);
  const long long kb = ceil_div(b.Vs, BK);
  int s = dh_split_count(dh_tiles, kb, workers);
  b.dh_kb_per_split = static_cast<int>(ceil_div(kb, s));
  s = static_cast<int>(ceil_div(kb, b.dh_kb_per_split));
  // dH partials and the gathered rows stay within the size of D
  auto aux = [&](int splits, bool f32) {
    return (f32 ? static_cast<double>(splits) * R * H * 4 : 0.0) + static_cast<double>(R) * H * 2;
  };
  while (s > 1 && aux(s, true) > 2.0 * budget) {
    --s;
    b.dh_kb_per_split = static_cast<int>(ceil_div(kb, s));
    s = static_cast<int>(ceil_div(kb, b.dh_kb_per_split));
  }
  b.dh_splits = s;
  b.dh_f32 = b.n_slabs > 1 || s > 1;
  if (b.n_slabs > 1 && aux(s, b.dh_f32) > 2.0 * budget) return false;

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
    return t + 3 * kPlanLaunch;
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

// FLCE_BWD_ROWS=<rows> fixes the row block (clamped to the budget) instead of
// the modelled choice.
long long bwd_rows_env() {
  const char* e = std::getenv("FLCE_BWD_ROWS");
  return e != nullptr ? std::atoll(e) : 0;
}

BwdPlan plan_backward(long long N, long long H, long long V, long long chunk_rows, int workers,
                      int tm) {
  N = std::max(1LL, N);
  const long long nr = round_up(N, BM);
  const long long R0 = std::min(round_up(std::max(1LL, chunk_rows), BM), nr);
  const long long budget = R0 * round_up(V, 8);
  workers = std::max(1, workers);
  struct Key {
    long long N, H, V, R0, forced;
    int workers, tm;
  };
  thread_local Key last{-1, -1, -1, -1, -1, -1, -1};
  thread_local BwdPlan last_plan;
  const long long forced = bwd_rows_env();
  if (last.N == N && last.H == H && last.V == V && last.R0 == R0 && last.forced == forced &&
      last.workers == workers && last.tm == tm)
    return last_plan;

  BwdPlan best;
  plan_candidate(best, N, H, V, R0, budget, workers, tm);  // the caller's chunk: always fits
  if (forced > 0) {
    BwdPlan b;
    const long long R = std::min(nr, std::max(R0, round_up(forced, BM)));
    if (plan_candidate(b, N, H, V, R, budget, workers, tm)) best = b;
  } else {
    // larger row blocks in steps of one tile; a plan with vocabulary slabs
    // must beat the single-slab chunk plan by 5 % (the model misses some of
    // the slabs' extra traffic: on 16,384 x 4,096 x 151,936 at 4,096-row
    // chunks, 8,192- and 16,384-row blocks measured no faster), and each
    // later candidate the best so far by 2 %
    const bool single = best.n_slabs == 1;
    for (long long R = round_up(R0 + 1, tm); R <= round_up(nr, tm); R += tm) {
      BwdPlan b;
      if (!plan_candidate(b, N, H, V, std::min(R, nr), budget, workers, tm)) break;
      const double margin = (single && best.R == R0) ? 0.95 : 0.98;
      if (b.est_s < best.est_s * margin) best = b;
      if (R >= nr) break;
    }
  }
  last = Key{N, H, V, R0, forced, workers, tm};
  last_plan = best;
  return best;
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
// vectors when the caller does not ask for them.
struct JsdFwdLayout {
  KdFwdLayout kd;
  size_t pj = 0, lse_s = 0, lse_t = 0, total = 0;
};
JsdFwdLayout jsd_fwd_layout(long long N, const FwdPlan& f) {
  JsdFwdLayout L;
  L.kd = kd_fwd_layout(N, f);
  size_t o = L.kd.total;
  L.pj = o;
  o += align256(static_cast<size_t>(f.S) * N * 8);
  L.lse_s = o;
  o += align256(static_cast<size_t>(N) * 4);
  L.lse_t = o;
  o += align256(static_cast<size_t>(N) * 4);
  L.total = o;
  return L;
}

struct BwdLayout {
  size_t D = 0, dh_part = 0, bad = 0, idx = 0, blk = 0, count = 0, hc = 0, total = 0;
};
// dlogits block, dH fp32 partials, validation counter, and the row
// compaction buffers (valid-row indices, per-block counts, their total, the
// gathered h rows of one chunk).
BwdLayout bwd_layout(long long N, long long H, const BwdPlan& b) {
  BwdLayout L;
  size_t o = 0;
  L.D = o;
  o += align256(static_cast<size_t>(b.R) * b.ldD * 2);
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
  L.total = o;
  return L;
}

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

// Programmatic dependent launch of the GEMMs (default; FLCE_PDL=0 turns it
// off): a GEMM may be scheduled while the previous kernel of the stream
// drains, runs its prologue (barriers, TMEM, descriptor prefetch) and then
// waits in griddepcontrol.wait until that kernel has completed.  Each GEMM
// grid fits on the GPU at once, so the waiting CTAs never hold SMs that the
// kernel they wait for still needs.
bool pdl_env() {
  const char* s = std::getenv("FLCE_PDL");
  return !(s != nullptr && s[0] == '0');
}

// Launch on `grid` CTAs in clusters of `cluster` with the GEMMs' attributes.
template <class Kern, class... Args>
cudaError_t launch_persistent(Kern k, int grid, int cluster, int smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
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
  if (pdl_env()) {
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

template <int MODE, bool kLong, int CG>
cudaError_t launch_gemm_t(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                          const CUtensorMap& a2, const CUtensorMap& b2, const GemmParams& p,
                          int workers, cudaStream_t st) {
  auto k = flce_gemm_kernel<MODE, kLong, CG>;
  constexpr int smem = TileCfg<CG>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_persistent(k, CG * workers, CG, smem, st, a, b, c, a2, b2, p);
}

// `workers`: CTAs (cg 1) or CTA pairs (cg 2), each running one persistent
// tile loop.  `c` is the output map of the modes that write through TMA (dW);
// the other modes ignore it.
template <int MODE>
cudaError_t launch_gemm(int cg, bool kLong, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const GemmParams& p, int workers, cudaStream_t st,
                        const CUtensorMap* a2 = nullptr, const CUtensorMap* b2 = nullptr) {
  // a2 / b2: the teacher's operands of the distillation modes (else unused)
  const CUtensorMap& A2 = a2 ? *a2 : a;
  const CUtensorMap& B2 = b2 ? *b2 : b;
  if (cg == 2)
    return kLong ? launch_gemm_t<MODE, true, 2>(a, b, c, A2, B2, p, workers, st)
                 : launch_gemm_t<MODE, false, 2>(a, b, c, A2, B2, p, workers, st);
  return kLong ? launch_gemm_t<MODE, true, 1>(a, b, c, A2, B2, p, workers, st)
               : launch_gemm_t<MODE, false, 1>(a, b, c, A2, B2, p, workers, st);
}

// The e4m3 forward: MODE_FWD with 8-bit operands.
cudaError_t launch_fwd_e4m3(int cg, bool kLong, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int workers, cudaStream_t st) {
  auto go = [&](auto kern, int smem, int grid_mult) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_persistent(kern, grid_mult * workers, grid_mult, smem, st, a, b, b, a, b, p);
  };
  if (cg == 2)
    return kLong ? go(flce_gemm_kernel<MODE_FWD, true, 2, true>, TileCfg<2>::SMEM, 2)
                 : go(flce_gemm_kernel<MODE_FWD, false, 2, true>, TileCfg<2>::SMEM, 2);
  return kLong ? go(flce_gemm_kernel<MODE_FWD, true, 1, true>, TileCfg<1>::SMEM, 1)
               : go(flce_gemm_kernel<MODE_FWD, false, 1, true>, TileCfg<1>::SMEM, 1);
}

// CTA group of the GEMMs: 2 (SM pairs, 256-row tiles) unless FLCE_CTA_GROUP=1.
int cta_group() {
  const char* s = std::getenv("FLCE_CTA_GROUP");
  return (s != nullptr && s[0] == '1') ? 1 : 2;
}

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
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
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

// Backward on non-ignored rows only (default); FLCE_COMPACT=0 runs every row.
bool compact_env() {
  const char* s = std::getenv("FLCE_COMPACT");
  return !(s != nullptr && s[0] == '0');
}

// DLOGITS writes D through TMA boxes (default) or per-thread stores
// (FLCE_D_TMA=0).
bool d_tma_env() {
  const char* s = std::getenv("FLCE_D_TMA");
  return !(s != nullptr && s[0] == '0');
}

bool validate_env() {
  const char* s = std::getenv("FLCE_VALIDATE");
  return s != nullptr && s[0] != '\0' && s[0] != '0';
}

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

// Row tiles per dH raster group: 8 (FLCE_DH_GROUP overrides).  A wave of 76
// units then covers 8 row tiles x ~9.5 column tiles, the fewest D and W
// slices per wave.  On 16,384 x 4,096 x 151,936, interleaved runs timed the
// step 1.3% faster than with all 16 row tiles (the dH launch itself took the
// same time); a dH launch's DRAM bytes vary more between GPUs than between
// the two groups.
int dh_group_rows(int m_tiles) {
  int g = 8;
  if (const char* e = std::getenv("FLCE_DH_GROUP")) g = std::atoi(e);
  return g > 0 ? std::min(g, m_tiles) : m_tiles;
}

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
  if (a.dH) {  // dH[rows] (+)= D[:, slab] W[slab]
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
    q.num_units = splits * q.m_tiles * q.n_tiles;
    q.group_m = dh_group_rows(q.m_tiles);
    q.dH_part = b.dh_f32 ? a.dh_part : nullptr;
    q.dh_accumulate = slab > 0 ? 1 : 0;
    ProfScope ps(K_DH, st);
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
    q.group_m = std::min(8, q.m_tiles);
    q.dW_accumulate = block > 0 ? 1 : 0;
    ProfScope ps(K_DW, st);
    FLCE_CUDA_TRY(launch_gemm<MODE_DW>(a.cg, a.kLong, D_mn, B_dw, *a.dW_map, q,
                                       std::min(q.num_units, a.workers), st));
  }
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
  int sp = dh_split_count(ceil_div(fp.R, tm) * ceil_div(H, BN), kb, workers);
  fp.b.dh_kb_per_split = static_cast<int>(ceil_div(kb, sp));
  fp.b.dh_splits = static_cast<int>(ceil_div(kb, fp.b.dh_kb_per_split));
  fp.b.dh_f32 = fp.b.dh_splits > 1;
  return fp;
}

struct FusedLayout {
  size_t zt = 0, part = 0, bsum = 0, bcnt = 0, bad = 0, E = 0, mx = 0, lse = 0, dh_part = 0, idx = 0,
         blk = 0, count = 0, hc = 0, total = 0;
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
  L.total = o;
  return L;
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
  const BwdLayout bl = bwd_layout(N, H, plan_backward(N, H, V, chunk_rows, workers, BM * cg));
  return std::max(fl.total, bl.total);
}

flce_status flce_backward_plan(int64_t N, int64_t H, int64_t V, int64_t chunk_rows, int32_t workers,
                               int32_t cta_group_, flce_backward_plan_info* out) {
  if (out == nullptr || !sizes_ok(N, H, V)) return FLCE_ERR_INVALID_ARG;
  const int cg = cta_group_ == 1 || cta_group_ == 2 ? cta_group_ : cta_group();
  const int w = workers > 0 ? workers : device_workers(cg);
  const BwdPlan b = plan_backward(N, H, V, chunk_rows, w, BM * cg);
  out->rows_per_block = b.R;
  out->vocab_per_slab = b.Vs;
  out->row_blocks = ceil_div(std::max<int64_t>(N, 1), b.R);
  out->vocab_slabs = b.n_slabs;
  out->dh_splits = b.dh_splits;
  out->dlogits_bytes = b.R * b.ldD * 2;
  out->workspace_bytes = static_cast<int64_t>(bwd_layout(N, H, b).total);
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
  // rows per forward launch (FLCE_FWD_BLOCK_ROWS; 0: all rows in one launch)
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
  const bool validate = validate_env();
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
      const int nblk = static_cast<int>(ceil_div(N, COMPACT_ROWS_PER_BLOCK));
      int* cblk = reinterpret_cast<int*>(wb + L.blk);
      ProfScope ps(K_COMPACT, st);
      compact_count_kernel<<<nblk, SMALL_THREADS, 0, st>>>(targets, Ni, ignore_index, cblk);
      FLCE_CUDA_TRY(cudaGetLastError());
      compact_write_kernel<<<nblk, SMALL_THREADS, 0, st>>>(targets, Ni, ignore_index, cblk, nblk, cidx, ccount,
                                                           0);
      FLCE_CUDA_TRY(cudaGetLastError());
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
    // 16 row tiles share each run of vocabulary tiles in L2 (measured on the
    // 16K x 4096 x 151,936 case: DRAM reads 17.9 GB at 16 against 36.6 GB at
    // 8 and 23.6 GB at 32, and the fastest launch)
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
        const long long total = fb * (H / 8);
        const int grid = static_cast<int>(std::min<long long>(ceil_div(total, SMALL_THREADS), 8LL * device_sms()));
        ProfScope ps(K_GATHER, st);
        gather_rows_kernel<<<grid, SMALL_THREADS, 0, st>>>(h, static_cast<int>(H), cidx, ccount, Ni,
                                                            static_cast<int>(row0), static_cast<int>(fb), hc);
        FLCE_CUDA_TRY(cudaGetLastError());
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

flce_status flce_forward_ex2(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                             const float* weights, int64_t N, int64_t H, int64_t V,
                             int64_t chunk_rows, int64_t ignore_index,
                             const flce_logit_transform* transform, uint32_t flags, float* out_logp,
                             float* out_lse, float* out_loss, int64_t* out_n_valid, void* workspace,
                             size_t workspace_bytes, void* stream) {
  (void)chunk_rows;
  if ((flags & ~static_cast<uint32_t>(FLCE_FORWARD_SKIP_IGNORED)) != 0) return FLCE_ERR_INVALID_ARG;
  const bool skip = (flags & FLCE_FORWARD_SKIP_IGNORED) != 0 && compact_env();
  return forward_impl(h, W, targets, weights, N, H, V, ignore_index, transform, out_logp, out_lse,
                      out_loss, out_n_valid, workspace, workspace_bytes, stream, kFwdPartialsCap, skip);
}

// The backward; count_scale (device int64, or NULL) divides grad_scale by
// max(*count_scale, 1) on the device.
static flce_status backward_impl(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                                 const float* weights, const float* lse, float grad_scale,
                                 flce_bf16* dH, float* dW, int64_t N, int64_t H, int64_t V,
                                 int64_t chunk_rows, int64_t ignore_index,
                                 const flce_logit_transform* transform, void* workspace,
                                 size_t workspace_bytes, void* stream,
                                 const long long* count_scale) {
  if (!sizes_ok(N, H, V)) return FLCE_ERR_INVALID_ARG;
  GemmParams tfp{};
  if (!transform_params(transform, tfp)) return FLCE_ERR_INVALID_ARG;
  if (!dH && !dW) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && (!h || !W || !targets || !lse)) return FLCE_ERR_INVALID_ARG;
  if (H % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(h, 16) || !aligned(W, 16) || !aligned(dH, 16) || !aligned(dW, 16) ||
      !aligned(targets, 8) || !aligned(weights, 4) || !aligned(lse, 4))
    return FLCE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    if (dW) FLCE_CUDA_TRY(cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * H * 4, st));
    return FLCE_OK;
  }
  const int cg = cta_group();
  const int workers = device_workers(cg);
  const int tm = BM * cg;
  const BwdPlan b = plan_backward(N, H, V, chunk_rows, workers, tm);
  const BwdLayout L = bwd_layout(N, H, b);
  Workspace ws;
  flce_status s = get_workspace(ws, workspace, workspace_bytes, L.total, st);
  if (s != FLCE_OK) return s;
  uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
  uint16_t* Dbuf = reinterpret_cast<uint16_t*>(wb + L.D);
  float* dh_part = b.dh_f32 ? reinterpret_cast<float*>(wb + L.dh_part) : nullptr;

  if (validate_env()) {
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
  CUtensorMap D_st;  // D as a TMA store target: [R][ldD] bf16, 64 x 32 boxes
  base.d_tma = d_tma_env() && make_map(&D_st, Dbuf, b.ldD, b.R, b.ldD, 64, 32) ? 1 : 0;
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
  // zeroed up front.
  const bool compact = compact_env();
  int* cidx = reinterpret_cast<int*>(wb + L.idx);
  int* cblk = reinterpret_cast<int*>(wb + L.blk);
  int* ccount = reinterpret_cast<int*>(wb + L.count);
  uint16_t* hc = reinterpret_cast<uint16_t*>(wb + L.hc);
  CUtensorMap hc_k, hc_mn, Dfix_k, Dfix_mn;
  if (compact) {
    const int nblk = static_cast<int>(ceil_div(N, COMPACT_ROWS_PER_BLOCK));
    {
      ProfScope ps(K_COMPACT, st);
      compact_count_kernel<<<nblk, SMALL_THREADS, 0, st>>>(targets, static_cast<int>(N), ignore_index,
                                                           cblk);
      FLCE_CUDA_TRY(cudaGetLastError());
    }
    {
      ProfScope ps(K_COMPACT, st);
      compact_write_kernel<<<nblk, SMALL_THREADS, 0, st>>>(targets, static_cast<int>(N), ignore_index,
                                                           cblk, nblk, cidx, ccount, 0);
      FLCE_CUDA_TRY(cudaGetLastError());
    }
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
      const long long total = b.R * (H / 8);
      const int grid = static_cast<int>(std::min<long long>(ceil_div(total, SMALL_THREADS), 8LL * device_sms()));
      ProfScope ps(K_GATHER, st);
      gather_rows_kernel<<<grid, SMALL_THREADS, 0, st>>>(h, static_cast<int>(H), cidx, ccount,
                                                          static_cast<int>(N), static_cast<int>(row0),
                                                          static_cast<int>(b.R), hc);
      FLCE_CUDA_TRY(cudaGetLastError());
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
    for (int slab = 0; slab < b.n_slabs; ++slab) {
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
static size_t fallback_workspace(int64_t N, int64_t H, int64_t V, int64_t chunk_rows, int workers,
                                 int tm) {
  const size_t fwd = fwd_layout(N, plan_forward_call(N, H, V, workers, tm)).total;
  const size_t bwd = bwd_layout(N, H, plan_backward(N, H, V, chunk_rows, workers, tm)).total;
  return std::max(fwd, bwd) + align256(static_cast<size_t>(std::max<int64_t>(N, 1)) * 4) + 256;
}

size_t flce_forward_backward_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t chunk_rows) {
  if (!sizes_ok(N, H, V)) return 0;
  const int cg = cta_group();
  const int workers = device_workers(cg);
  const FusedPlan fp = plan_fused(N, H, V, chunk_rows, workers, BM * cg);
  if (fp.fused) return fused_layout(N, H, fp).total;
  return fallback_workspace(N, H, V, chunk_rows, workers, BM * cg);
}

flce_status flce_forward_backward(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                                  const float* weights, int64_t N, int64_t H, int64_t V,
                                  int64_t chunk_rows, int64_t ignore_index,
                                  const flce_logit_transform* transform, float grad_scale,
                                  float* out_logp, float* out_lse, float* out_loss,
                                  int64_t* out_n_valid, flce_bf16* dH, float* dW, void* workspace,
                                  size_t workspace_bytes, void* stream) {
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
    const size_t need = fallback_workspace(N, H, V, chunk_rows, workers, tm);
    flce_status s = get_workspace(ws, workspace, workspace_bytes, need, st);
    if (s != FLCE_OK) return s;
    uint8_t* wb = static_cast<uint8_t*>(ws.ptr);
    const size_t inner = need - align256(static_cast<size_t>(std::max<int64_t>(N, 1)) * 4) - 256;
    float* lse = out_lse ? out_lse : reinterpret_cast<float*>(wb + inner);
    int64_t* nv = out_n_valid ? out_n_valid
                              : reinterpret_cast<int64_t*>(wb + inner + align256(static_cast<size_t>(std::max<int64_t>(N, 1)) * 4));
    s = forward_impl(h, W, targets, weights, N, H, V, ignore_index, transform, out_logp, lse, out_loss, nv,
                     wb, inner, stream, kFwdPartialsCap);
    if (s != FLCE_OK) return s;
    return backward_impl(h, W, targets, weights, lse, grad_scale, dH, dW, N, H, V, chunk_rows, ignore_index,
                         transform, wb, inner, stream, reinterpret_cast<const long long*>(nv));
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
  const int Ni = static_cast<int>(N);
  const bool validate = validate_env();
  // Row compaction: the blocks run over a permutation of the rows with the
  // non-ignored ones first.  A block's forward covers all its rows when the
  // caller asks for lse (defined for ignored rows too), else only the
  // non-ignored ones; its dH / dW GEMMs read the device-side count and cover
  // only the non-ignored rows.
  const bool compact = compact_env();
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
    const int nblk = static_cast<int>(ceil_div(N, COMPACT_ROWS_PER_BLOCK));
    ProfScope ps(K_COMPACT, st);
    compact_count_kernel<<<nblk, SMALL_THREADS, 0, st>>>(targets, Ni, ignore_index, cblk);
    FLCE_CUDA_TRY(cudaGetLastError());
    compact_write_kernel<<<nblk, SMALL_THREADS, 0, st>>>(targets, Ni, ignore_index, cblk, nblk, cidx, ccount,
                                                         compact ? 1 : 0);
    FLCE_CUDA_TRY(cudaGetLastError());
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
      const long long total = fp.R * (H / 8);
      const int grid = static_cast<int>(std::min<long long>(ceil_div(total, SMALL_THREADS), 8LL * device_sms()));
      ProfScope ps(K_GATHER, st);
      gather_rows_kernel<<<grid, SMALL_THREADS, 0, st>>>(h, static_cast<int>(H), cidx,
                                                          fwd_valid_only ? ccount : nullptr, Ni,
                                                          static_cast<int>(row0), static_cast<int>(fp.R), hc);
      FLCE_CUDA_TRY(cudaGetLastError());
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
                                                           out_logp ? out_logp + off : nullptr, lse + off,
                                                           bsum + b0, bcnt + b0, ri);
      else
        combine_kernel<false><<<nb, SMALL_THREADS, 0, st>>>(part + off, fp.f.S, Ni, rows, zt + off, targets + off,
                                                            weights ? weights + off : nullptr, ignore_index,
                                                            out_logp ? out_logp + off : nullptr, lse + off,
                                                            bsum + b0, bcnt + b0, ri);
      FLCE_CUDA_TRY(cudaGetLastError());
    }
    {  // (3) exponentials -> dlogits, in place
      ProfScope ps(K_DLOGITS, st);
      const dim3 grid(static_cast<unsigned>(ceil_div(fp.ldD, SMALL_THREADS * FUSED_COLS_PER_THREAD)),
                      static_cast<unsigned>(rows));
      const int* ri = compact ? cidx + row0 : nullptr;
      if (kLong)
        fused_dlogits_kernel<true><<<grid, SMALL_THREADS, 0, st>>>(
            E, mx, static_cast<int>(fp.ldD), static_cast<int>(V), static_cast<int>(row0), ri, targets, weights,
            lse, zt, ignore_index, ccount, grad_scale, tfp.tf_softcap, tfp.tf_a, tfp.tf_b, tfp.tf_d);
      else
        fused_dlogits_kernel<false><<<grid, SMALL_THREADS, 0, st>>>(
            E, mx, static_cast<int>(fp.ldD), static_cast<int>(V), static_cast<int>(row0), ri, targets, weights,
            lse, zt, ignore_index, ccount, grad_scale, tfp.tf_softcap, tfp.tf_a, tfp.tf_b, tfp.tf_d);
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
    // block's unused entries are zeroed below before the loop
    final_kernel<<<1, SMALL_THREADS, 0, st>>>(bsum, bcnt,
                                              static_cast<int>(ceil_div(N, fp.R) * ceil_div(fp.R, SMALL_THREADS)),
                                              out_loss, reinterpret_cast<long long*>(out_n_valid));
    FLCE_CUDA_TRY(cudaGetLastError());
  }
  return FLCE_OK;
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
  const FwdPlan f = plan_forward(N, H, V, workers, BM * cg);
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
    {
      ProfScope ps(K_FWD, st);
      FLCE_CUDA_TRY(launch_fwd_e4m3(cg, kLong, tA, tB, p, f.grid, st));
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
  const JsdFwdLayout fl = jsd_fwd_layout(N, plan_forward(N, H_s + H_t, V, workers, BM * cg));
  const BwdLayout bl = bwd_layout(N, H_s, plan_backward(N, H_s, V, chunk_rows, workers, BM * cg));
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
                                   size_t workspace_bytes, void* stream) {
  if (!sizes_ok(N, H_s, V) || !sizes_ok(N, H_t, V)) return FLCE_ERR_INVALID_ARG;
  if (jsd && !(beta > 0.f && beta < 1.f)) return FLCE_ERR_INVALID_ARG;
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
  const FwdPlan f = plan_forward(N, H_s + H_t, V, workers, BM * cg);
  const JsdFwdLayout J = jsd_fwd_layout(N, f);
  const KdFwdLayout& L = J.kd;
  Workspace ws;
  flce_status s = get_workspace(ws, workspace, workspace_bytes, jsd ? J.total : L.total, st);
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
    CUtensorMap hs_k, Ws_k, ht_k, Wt_k;
    if (!make_map(&hs_k, h_s, H_s, N, H_s, BK, BM) || !make_map(&Ws_k, W_s, H_s, V, H_s, BK, BN / cg) ||
        !make_map(&ht_k, h_t, H_t, N, H_t, BK, BM) || !make_map(&Wt_k, W_t, H_t, V, H_t, BK, BN / cg))
      return FLCE_ERR_CUDA;
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
    p.err = err;
    p.tf_softcap = tfp.tf_softcap;
    p.tf_a = tfp.tf_a;
    p.tf_b = tfp.tf_b;
    p.tf_d = tfp.tf_d;
    const bool kLong = static_cast<long long>(N) * V >= INT_MAX ||
                       static_cast<long long>(f.S) * N >= INT_MAX;
    {
      ProfScope prof(K_KD_FWD, st);
      FLCE_CUDA_TRY(launch_gemm<MODE_KD_FWD>(cg, kLong, hs_k, Ws_k, Ws_k, p, f.grid, st, &ht_k, &Wt_k));
    }
    {
      ProfScope prof(K_COMBINE, st);
      float* kl = jsd ? nullptr : out_kl;
      if (kLong)
        kd_combine_kernel<true><<<f.nblk, SMALL_THREADS, 0, st>>>(ps, pt, pc, f.S, Ni, targets, weights,
                                                                  ignore_index, kl, lse_s, lse_t, bsum, bcnt);
      else
        kd_combine_kernel<false><<<f.nblk, SMALL_THREADS, 0, st>>>(ps, pt, pc, f.S, Ni, targets, weights,
                                                                   ignore_index, kl, lse_s, lse_t, bsum, bcnt);
      FLCE_CUDA_TRY(cudaGetLastError());
    }
    if (jsd) {
      float2* pj = reinterpret_cast<float2*>(wb + J.pj);
      GemmParams q = p;
      q.lse = lse_s;
      q.lse_t = lse_t;
      q.partials = pj;
      q.jsd_beta = beta;
      {
        ProfScope prof(K_JSD_FWD, st);
        FLCE_CUDA_TRY(launch_gemm<MODE_JSD_FWD>(cg, kLong, hs_k, Ws_k, Ws_k, q, f.grid, st, &ht_k, &Wt_k));
      }
      ProfScope prof(K_COMBINE, st);
      if (kLong)
        jsd_combine_kernel<true><<<f.nblk, SMALL_THREADS, 0, st>>>(pj, f.S, Ni, targets, weights, ignore_index,
                                                                   beta, out_kl, out_kl_sm, bsum, bcnt);
      else
        jsd_combine_kernel<false><<<f.nblk, SMALL_THREADS, 0, st>>>(pj, f.S, Ni, targets, weights, ignore_index,
                                                                    beta, out_kl, out_kl_sm, bsum, bcnt);
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
                                    size_t workspace_bytes, void* stream) {
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
  const BwdLayout L = bwd_layout(N, H_s, b);
  Workspace ws;
  flce_status s = get_workspace(ws, workspace, workspace_bytes, L.total, st);
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

  CUtensorMap dhp_map;
  if (dH_s && b.dh_f32 &&
      !make_map_t(&dhp_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dh_part, H, b.dh_splits * b.R, H, 32, 32))
    return FLCE_ERR_CUDA;
  const DhDwStage dhdw{cg, workers, tm, kLong, &b, H, V, dh_part, dH_s, dW_s, &Ws_mn, &dW_map, &dhp_map};
  int block = 0;
  for (long long row0 = 0; row0 < N; row0 += b.R, ++block) {
    const int rows = static_cast<int>(std::min(b.R, N - row0));
    GemmParams p = base;
    p.row0 = static_cast<int>(row0);
    p.rows = rows;
    CUtensorMap D_k, D_mn;
    if (!make_map(&D_k, Dbuf, b.ldD, rows, b.ldD, BK, BM) ||
        !make_map(&D_mn, Dbuf, b.ldD, rows, b.ldD, 64, BK))
      return FLCE_ERR_CUDA;
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
          FLCE_CUDA_TRY(launch_gemm<MODE_JSD_DLOGITS>(cg, kLong, hs_k, Ws_k, Ws_k, q,
                                                      std::min(q.num_units, workers), st, &ht_k, &Wt_k));
        else
          FLCE_CUDA_TRY(launch_gemm<MODE_KD_DLOGITS>(cg, kLong, hs_k, Ws_k, Ws_k, q,
                                                     std::min(q.num_units, workers), st, &ht_k, &Wt_k));
      }
      const flce_status s2 = slab_dh_dw(dhdw, p, rows, block, slab, v0, width, D_k, D_mn, hs_mn, st);
      if (s2 != FLCE_OK) return s2;
    }
    const flce_status s3 = block_dh_finish(dhdw, p.row0, rows, nullptr, nullptr, 0, st);
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
// Some callers are not allowed to allocate at all: code that runs while a
// CUDA graph is being captured (an allocation there would be recorded or is
// forbidden), inference runtimes that own every byte of device memory through
// a fixed pool, and callers that must keep a constant memory footprint.  This
// entry point serves them: it takes the same inputs and outputs as
// flce_forward, but its scratch lives in one file-scope device array that the
// library owns, so nothing is allocated or freed by any call.
//
// The array is a fixed 16 MiB, resident on every device that loads this
// library until the process exits.  On the host its name is only a stand-in
// for the device copy, never a device address: the address is looked up once
// per device with cudaGetSymbolAddress (device code could name the array
// directly, host code must not).
namespace {
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
}  // namespace

static __device__ __align__(256) unsigned char g_flce_static_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxStaticScratchDevices = 128;
std::mutex g_static_scratch_mu;
void* g_static_scratch_addr[kMaxStaticScratchDevices];

// Device address of g_flce_static_scratch on the current device (looked up on
// the first call per device, with that device current).
flce_status static_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FLCE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxStaticScratchDevices) return FLCE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (g_static_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_flce_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FLCE_ERR_CUDA;
    }
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
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
