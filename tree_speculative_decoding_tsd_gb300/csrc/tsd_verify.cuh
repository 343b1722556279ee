// Shared declarations of the tree-verify attention paths.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "tsd.h"

namespace tsd {

// Kernel arguments of every verify path (passed by value).
struct VerifyArgs {
  const void* q;
  const void* kc;
  const void* vc;
  const int32_t* plen;
  const void* kt;
  const void* vt;
  const uint64_t* mask;
  void* out;
  float* lse;
  float* ws_o;    // [B][Hq][R][nsplit][dv] normalised partial outputs
  float* ws_lse;  // [B][Hq][R][nsplit] log2-sum-exp of each partial
  int32_t* err;
  int B, R, Hq, Hkv, g, M, cap;
  int nsplit, split_len, nrg;
  float qscale;   // softmax scale * log2(e): scores are kept in the log2 domain
};

enum VerifyPathId { kPathGeneric = 0, kPathMma = 1 };

struct VerifyPlan {
  int path;
  int rb;         // packed rows per CTA
  int nrg;        // row groups per KV head
  int nsplit;     // prefix splits (grid x); a request uses ceil(P / split_len)
  int split_len;
  size_t ws_bytes;
};

VerifyPlan plan_verify(const tsd_attn_desc& d);

}  // namespace tsd
