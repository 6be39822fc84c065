// Launch-choice table per (format class, size bucket): which GEMM kernel, which token tile, Stream-K or not, and
// CTAs per SM.  The rows live in hq_tune_table.h, written by the package's tune.py from a timing sweep of every
// valid choice per bucket on the target GPU ("Tuning and JIT compilation per workload": device heuristics per range
// of input sizes; "Future plans": autotune).  The host planner takes its built-in rule where no row matches.
#pragma once
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

namespace hq {

// Format classes: the choices open to each differ (only INT4 has both GEMM kernels).
enum TuneClass {
  TC_INT4 = 0,    // INT4_SYM / UINT4_ZP weights, bf16 activations: UMMA or register-decode kernel
  TC_REGDEC = 1,  // INT8 / UINT2 / MXINT4 / E4M3 weights: register-decode kernel only
  TC_NVFP4 = 2,   // NVFP4 x NVFP4
  TC_MXFP4 = 3,   // MXFP4 x per-token FP8
  TC_MXFP4A = 4,  // MXFP4 x MXFP8
  TC_MXFP4X = 5,  // MXFP4 x MXFP4
};

// One choice.  -1 / 0 in a field leave it to the built-in rule.
struct TuneChoice {
  int kernel = -1;   // 0 UMMA, 1 register-decode
  int bt = 0;        // token tile
  int sk = -1;       // Stream-K split of K over CTAs: 0 off, 1 on
  int slots = 0;     // CTAs per SM in the persistent grid
  int grouped = -1;  // MoE activations: 0 indexed rows (gather), 1 expert-grouped copy
  int cpb = 0;       // with Stream-K: at least this many K blocks per CTA (fewer, longer pieces)
};

// A table row (the table ends with a row of class -1): applies to calls of class `cls` and kind `moe` (0 dense, 1 MoE,
// 2 MoE with the top-k combine: the Down GEMM, whose short K and reducing epilogue favour other tiles) whose key
// (dense: M; MoE: routed rows per expert, rounded up) is at most key_max and above the previous matching row's key_max.
struct TuneRow {
  int cls;
  int moe;
  int64_t key_max;
  TuneChoice c;
};

}  // namespace hq

#include "hq_tune_table.h"

namespace hq {

inline TuneChoice tune_lookup(int cls, int kind, int64_t key) {
  for (const TuneRow& r : kTuneRows)
    if (r.cls == cls && r.moe == kind && key <= r.key_max) return r.c;
  return TuneChoice{};
}

// HQ_TUNE="kernel=1,bt=16,sk=0,slots=2,grouped=0,cpb=2" replaces the table's choice for every call (the sweep times
// each candidate this way); fields left out keep the table's value.
inline void tune_env_override(TuneChoice& c) {
  const char* v = getenv("HQ_TUNE");
  if (!v) return;
  const char* names[6] = {"kernel=", "bt=", "sk=", "slots=", "grouped=", "cpb="};
  int* fields[6] = {&c.kernel, &c.bt, &c.sk, &c.slots, &c.grouped, &c.cpb};
  for (int i = 0; i < 6; ++i) {
    const char* p = strstr(v, names[i]);
    if (p && (p == v || p[-1] == ',')) *fields[i] = atoi(p + strlen(names[i]));
  }
}

}  // namespace hq
