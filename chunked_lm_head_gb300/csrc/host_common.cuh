// libflce host side: launch-kind profiling (CUDA events around each launch)
// and the integer helpers shared by the planners and the entry points.
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "small_kernels.cuh"

namespace {

using namespace flce;

using namespace flce;

constexpr int kDefaultSms = 152;

enum Kind {
  K_PREP, K_FWD, K_COMBINE, K_FINAL, K_DLOGITS, K_DH, K_DH_REDUCE, K_DW, K_COMPACT, K_GATHER,
  K_KD_FWD, K_KD_DLOGITS, K_QUANT, K_JSD_FWD, K_JSD_DLOGITS, K_GRPO, K_DHDW, K_PIPE, K_COUNT
};
const char* const kKindNames[K_COUNT] = {"prep_targets",  "fwd_logits_lse", "fwd_combine",
                                         "fwd_loss",      "bwd_dlogits",    "bwd_dH",
                                         "bwd_dH_reduce", "bwd_dW",         "bwd_compact_rows",
                                         "bwd_gather_rows", "kd_fwd_logits",  "kd_bwd_dlogits",
                                         "quantize_e4m3", "jsd_fwd_terms",  "jsd_bwd_dlogits",
                                         "grpo_token_loss", "bwd_dH_dW",
                                         "bwd_pipeline"};

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

}  // namespace
