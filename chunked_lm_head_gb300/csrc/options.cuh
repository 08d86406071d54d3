// libflce run-time options: one process-wide table, read by every entry point.
//
// Each option starts from its FLCE_* environment variable, read once when the
// library first consults an option, else from its built-in default; after that
// only flce_set_option changes it.  Entry points read the table, never the
// environment, so a plan cannot change behind a caller's back between calls.
#pragma once

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "flce.h"

namespace {

struct OptionDef {
  const char* env;  // environment variable giving the initial value
  int64_t dflt;     // built-in default
  int64_t lo, hi;   // accepted range
};

// Indexed by flce_option.
constexpr OptionDef kOptionDefs[FLCE_OPT_COUNT] = {
    {"FLCE_CTA_GROUP", 2, 1, 2},              // FLCE_OPT_CTA_GROUP
    {"FLCE_COMPACT", 1, 0, 1},                // FLCE_OPT_COMPACT
    {"FLCE_VALIDATE", 0, 0, 1},               // FLCE_OPT_VALIDATE
    {"FLCE_PDL", 1, 0, 1},                    // FLCE_OPT_PDL
    {"FLCE_D_TMA", 1, 0, 1},                  // FLCE_OPT_D_TMA
    {"FLCE_WIDE_EPILOGUE", 1, 0, 1},          // FLCE_OPT_WIDE_EPILOGUE
    {"FLCE_BWD_ROWS", 0, 0, INT_MAX},         // FLCE_OPT_BWD_ROWS
    {"FLCE_FWD_SPLITS", 0, 0, 256},           // FLCE_OPT_FWD_SPLITS
    {"FLCE_DH_SPLITS", 0, 0, 16},             // FLCE_OPT_DH_SPLITS
    {"FLCE_DH_GROUP", 8, 0, 1 << 20},         // FLCE_OPT_DH_GROUP
    {"FLCE_FWD_BLOCK_ROWS", -1, -1, INT_MAX},  // FLCE_OPT_FWD_BLOCK_ROWS
    {"FLCE_SKIP_MIN_ROWS", 2048, 0, INT_MAX},  // FLCE_OPT_SKIP_MIN_ROWS
    {"FLCE_FUSE_DH_DW", 1, 0, 1},             // FLCE_OPT_FUSE_DH_DW
    {"FLCE_DW_EPILOGUE_WARPS", 16, 8, 16},    // FLCE_OPT_DW_EPILOGUE_WARPS
    {"FLCE_PIPELINE", 1, 0, 1},               // FLCE_OPT_PIPELINE
    {"FLCE_DH_WIDE", 1, 0, 1},                // FLCE_OPT_DH_WIDE
    {"FLCE_GRID_WORKERS", 0, 0, 4096},        // FLCE_OPT_GRID_WORKERS
};

std::atomic<int64_t> g_options[FLCE_OPT_COUNT];
std::once_flag g_options_once;

int64_t clamp_option(int o, int64_t v) {
  const OptionDef& d = kOptionDefs[o];
  return v < d.lo ? d.lo : (v > d.hi ? d.hi : v);
}

// The initial value of option o from its environment variable.  The on/off
// switches read "0" as off and anything else as on, except FLCE_VALIDATE,
// which is on for any value but empty or "0"; FLCE_CTA_GROUP is 1 only for
// "1".  The others are integers (FLCE_FWD_BLOCK_ROWS <= 0: one launch over
// all rows).
int64_t option_from_env(int o) {
  const OptionDef& d = kOptionDefs[o];
  const char* s = std::getenv(d.env);
  if (s == nullptr) return d.dflt;
  switch (o) {
    case FLCE_OPT_CTA_GROUP:
      return s[0] == '1' ? 1 : 2;
    case FLCE_OPT_COMPACT:
    case FLCE_OPT_FUSE_DH_DW:
    case FLCE_OPT_PIPELINE:
    case FLCE_OPT_DH_WIDE:
    case FLCE_OPT_PDL:
    case FLCE_OPT_D_TMA:
    case FLCE_OPT_WIDE_EPILOGUE:
      return s[0] == '0' ? 0 : 1;
    case FLCE_OPT_VALIDATE:
      return (s[0] != '\0' && s[0] != '0') ? 1 : 0;
    case FLCE_OPT_FWD_BLOCK_ROWS: {
      const long long v = std::atoll(s);
      return v <= 0 ? 0 : clamp_option(o, v);
    }
    default:
      return clamp_option(o, std::atoll(s));
  }
}

void init_options() {
  std::call_once(g_options_once, [] {
    for (int o = 0; o < FLCE_OPT_COUNT; ++o) g_options[o].store(option_from_env(o));
  });
}

int64_t opt(flce_option o) {
  init_options();
  return g_options[o].load(std::memory_order_relaxed);
}

bool opt_on(flce_option o) { return opt(o) != 0; }

}  // namespace
