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
inline bool wide_path(int batch) { return batch > kNarrowMaxBatch; }
inline int oproj_tiles(const mk_config& c, int batch) {
  return (wide_path(batch) ? c.n_kv_heads : 1) * c.hidden / kRowsOProj;
}
inline int rows_down(int batch) { return wide_path(batch) ? kRowsDownW : kRowsDownN; }
inline int rows_lm(int batch) { return wide_path(batch) ? kRowsLMW : kRowsLMN; }
// ATTN_COMBINE tasks per (sequence, KV group): 2 query heads each at batch <= 2,
// up to 4 above
inline int combine_split(const mk_config& c, int batch) {
  const int grp = c.n_q_heads / c.n_kv_heads;
  const int hp = batch <= 2 ? (grp < 2 ? grp : 2) : (grp < 4 ? grp : 4);
  return grp / hp;
}
inline int moe_target(const mk_config& c, int batch) {
  return batch * c.top_k * (c.hidden / rows_down(batch));
}

}  // namespace mk
