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
  int n_comb_sms = 0;           // SMs with a COMBINE task per layer
  int n_up_sms = 0;             // SMs with an UP task per layer
  int n_down_sms = 0;           // SMs with a DOWN task per layer
  int n_rtr_sms = 0;            // SMs whose P1 share holds router rows
};

// Checks everything the kernel relies on; returns MK_OK or MK_ERR_BAD_CONFIG.
int validate_config(const mk_config& c);

// Per-SM task lists of one step for `batch` sequences: for every layer one
// task of each phase per SM, then the FINAL task.  With n_attn < n_sm the SMs
// take roles: n_attn SMs spread over the blocks run the attention branch of the parallel layer
// (P1, ATTN, COMBINE, OUT), the others the expert branch (P1, ROUTE, UP,
// DOWN, OUT), so the two branches run side by side and only the O-proj (OUT,
// on every SM) follows the attention; with n_attn == n_sm every SM runs every
// phase in the configured wave order.  With one token the UP slices also
// produce the down projection's per-group partials and DOWN sums them.  `bump_layer` / `bump`
// make the P1 task of that layer wait for a counter value that is never
// reached (testing aid for the timeout path).
int build_plan(const mk_config& c, int n_sm, int batch, int n_attn, Plan* out, int bump_layer = -1,
               int bump = 0);

// [s * total / n, (s + 1) * total / n): the share of SM s in an even split
inline void share(long long total, int n, int s, int* lo, int* hi) {
  *lo = (int)(total * s / n);
  *hi = (int)(total * (s + 1) / n);
}

// SM roles: the na attention SMs of a role split are spread evenly over the
// n_sm blocks (so the attention branch's KV streams do not crowd one part of
// the chip).  SM s is an attention SM if the running count floor(s na / n_sm)
// steps at s; attention SMs before s: floor(s na / n_sm).
inline int attn_before(int s, int n_sm, int na) { return (int)((long long)s * na / n_sm); }
inline bool is_attn_sm(int s, int n_sm, int na) {
  return na >= n_sm || attn_before(s + 1, n_sm, na) > attn_before(s, n_sm, na);
}
// index among the expert-branch SMs (for an SM that is not an attention SM)
inline int moe_rank(int s, int n_sm, int na) { return s - attn_before(s, n_sm, na); }

// SMs that take UP slices when every SM runs every phase (0 in the config = all)
inline int moe_sms(const mk_config& c, int n_sm) {
  return c.n_moe_claimers > 0 && c.n_moe_claimers < n_sm ? c.n_moe_claimers : n_sm;
}

// Attention SMs of a step: config.n_attn_claimers if set, else a share of the
// SMs proportional to the attention's KV bytes (weighted by 1.6) against the
// routed experts' gate/up/down bytes of a layer (the two branches that run
// side by side).
// n_sm means no roles.
int attention_sms(const mk_config& c, int n_sm, int batch, const int32_t* seq_lens);

// Split-KV items of one step: each sequence's keys cut into page ranges,
// spread over the n_attn attention SMs.  items: [n][8] (AI_* words), sm_off: [n_sm+1],
// meta: [batch][2] (first item, split count).  Returns the split size used
// (tokens; 0 = balanced page split), or -1 if more than max_items are needed.
int split_kv(const mk_config& c, int n_sm, int n_attn, int batch, const int32_t* seq_lens,
             std::vector<int32_t>* items, std::vector<int32_t>* sm_off,
             std::vector<int32_t>* meta);

}  // namespace mk
