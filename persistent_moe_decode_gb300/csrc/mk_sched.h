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
  int n_bars = 0;               // counter words the step uses (layers 0..L)
};

// Checks everything the kernel relies on; returns MK_OK or MK_ERR_BAD_CONFIG.
int validate_config(const mk_config& c);

// Named waves per layer in the configured order, flattened, task k dealt to
// SM k mod n_sm (§The task scheduler, the static part).  `bump_layer` /
// `bump` add to the norm task's first wait target (testing aid).
int build_plan(const mk_config& c, int n_sm, int batch, Plan* out, int bump_layer = -1,
               int bump = 0);

// counter targets shared by the scheduler and the kernel's own bookkeeping
inline int qkv_tiles_per_group(const mk_config& c) {
  return (c.n_q_heads / c.n_kv_heads + 2) * (c.head_dim / 32);
}
inline int oproj_tiles(const mk_config& c) { return c.n_kv_heads * c.hidden / kRowsOProj; }
inline int moe_target(const mk_config& c, int batch) {
  return batch * c.top_k * (c.hidden / kRowsDown);
}

}  // namespace mk
