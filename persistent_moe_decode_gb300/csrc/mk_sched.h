// Host task scheduler and descriptor encoder (no CUDA dependency).
#pragma once
#include <stdint.h>

#include <vector>

#include "../../include/mk.h"
#include "mk_layout.h"

namespace mk {

struct Plan {
  std::vector<int32_t> tasks;   // [n][32], SM-major
  std::vector<int32_t> off;     // [n_sm + 1]
  int n_bars = 0;               // counter words the step uses (layers 0..L-1)
};

// Checks everything the kernel relies on; returns MK_OK or MK_ERR_BAD_CONFIG.
int validate_config(const mk_config& c);

// Per-SM task lists of one step for `batch` sequences: for every layer one
// task of each phase per SM, in the configured wave order, then the FINAL
// task.  `bump_layer` / `bump` make the P1 task of that layer wait for a
// counter value that is never reached (testing aid for the timeout path).
int build_plan(const mk_config& c, int n_sm, int batch, Plan* out, int bump_layer = -1,
               int bump = 0);

// [s * total / n, (s + 1) * total / n): the share of SM s in an even split
inline void share(long long total, int n, int s, int* lo, int* hi) {
  *lo = (int)(total * s / n);
  *hi = (int)(total * (s + 1) / n);
}

// SMs that take attention items / UP slices (0 in the config = all)
inline int attn_sms(const mk_config& c, int n_sm) {
  return c.n_attn_claimers > 0 && c.n_attn_claimers < n_sm ? c.n_attn_claimers : n_sm;
}
inline int moe_sms(const mk_config& c, int n_sm) {
  return c.n_moe_claimers > 0 && c.n_moe_claimers < n_sm ? c.n_moe_claimers : n_sm;
}

// Split-KV items of one step: each sequence's keys cut into page ranges,
// spread over the attention SMs.  items: [n][8] (AI_* words), sm_off: [n_sm+1],
// meta: [batch][2] (first item, split count).  Returns the split size used
// (tokens; 0 = balanced page split), or -1 if more than max_items are needed.
int split_kv(const mk_config& c, int n_sm, int batch, const int32_t* seq_lens,
             std::vector<int32_t>* items, std::vector<int32_t>* sm_off,
             std::vector<int32_t>* meta);

}  // namespace mk
