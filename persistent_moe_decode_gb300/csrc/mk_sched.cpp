// Host task scheduler: builds the per-SM task lists of one decode step.
//
// "Inside the megakernel serving engine for North Mini Code", §The task
// scheduler: the host builds named waves for each layer, chooses an order,
// flattens them into one task list and deals task k to SM k mod nSM
// (round-robin).  Any order without a circular wait is correct; the default
// puts the router and route setup ahead of attention.  Attention and expert
// tiles are not listed one by one: a fixed number of claimer tasks per wave
// drain shared queues whose length is known only during the step.
#include "mk_sched.h"

#include <algorithm>
#include <array>

namespace mk {

// contraction lengths of the wide (tensor-core) GEMV path
static bool supported_k(int k) {
  return k == 128 || k == 256 || k == 512 || k == 768 || k == 1024 || k == 2048;
}

// contraction lengths of the narrow (CUDA-core, whole-row) GEMV path
static bool narrow_k(int k) { return k == 128 || (k % 256 == 0 && k <= 4096); }

int validate_config(const mk_config& c) {
  if (c.n_layers < 1 || c.hidden < 32 || c.n_q_heads < 1 || c.n_kv_heads < 1) return MK_ERR_BAD_CONFIG;
  if (c.n_q_heads % c.n_kv_heads) return MK_ERR_BAD_CONFIG;
  const int grp = c.n_q_heads / c.n_kv_heads;
  if (grp > 8 || kConsumerWarps % c.n_kv_heads) return MK_ERR_BAD_CONFIG;
  if (c.head_dim != 64 && c.head_dim != 128) return MK_ERR_BAD_CONFIG;
  // both GEMV paths must be able to run every matrix of the model
  if (!supported_k(c.hidden) || !supported_k(c.moe_inter) || !supported_k(grp * c.head_dim))
    return MK_ERR_BAD_CONFIG;
  if (!narrow_k(c.hidden) || !narrow_k(c.moe_inter) || !narrow_k(c.n_q_heads * c.head_dim))
    return MK_ERR_BAD_CONFIG;
  if (c.hidden % kRowsOProj || c.hidden % kRowsDownN || c.hidden % kRowsDownW ||
      c.moe_inter % kRowsUp)
    return MK_ERR_BAD_CONFIG;
  if (c.n_experts < 1 || c.n_experts > 256 || c.top_k < 1 || c.top_k > 8 || c.top_k > c.n_experts)
    return MK_ERR_BAD_CONFIG;
  if (c.vocab < 1 || c.page_size != 16) return MK_ERR_BAD_CONFIG;
  // one 16-token page of every KV head (K or V) must fit half a stage
  if (c.n_kv_heads * c.page_size * c.head_dim * 2 > kStageData / 2) return MK_ERR_BAD_CONFIG;
  if (c.max_batch < 1 || c.max_batch > kMaxBatch) return MK_ERR_BAD_CONFIG;
  if (c.max_pages_per_seq < 1 || c.num_kv_pages < 1) return MK_ERR_BAD_CONFIG;
  if (!(c.rope_theta > 0.0) || !(c.rms_eps >= 0.f)) return MK_ERR_BAD_CONFIG;
  if (c.max_attn_items < 0 || c.n_attn_claimers < 0 || c.n_moe_claimers < 0 || c.sm_cap < 0 ||
      c.timeout_ms < 0 || c.trace_records < 0)
    return MK_ERR_BAD_CONFIG;
  if (c.kv_split_tokens < 0 || c.kv_split_tokens % 64) return MK_ERR_BAD_CONFIG;
  if (c.wave_order < MK_WAVES_DEFAULT || c.wave_order > MK_WAVES_INTERLEAVED) return MK_ERR_BAD_CONFIG;
  return MK_OK;
}

namespace {

using Desc = std::array<int32_t, kDescWords>;

Desc blank(int op, int layer, int tile) {
  Desc d;
  d.fill(0);
  d[F_OP] = op;
  d[F_LAYER] = layer;
  d[F_TILE] = tile;
  d[F_W0] = d[F_W1] = d[F_SIG] = d[F_PW] = -1;
  d[F_T0] = d[F_T1] = d[F_INC] = d[F_PT] = 0;
  return d;
}

enum Wave { W_NORM, W_QKV, W_ROUTER, W_ATTN, W_COMBINE, W_UP, W_DOWN, W_OPROJ };

}  // namespace

int build_plan(const mk_config& c, int n_sm, int batch, Plan* out, int bump_layer, int bump) {
  if (validate_config(c) != MK_OK || n_sm < 1 || batch < 1 || batch > c.max_batch)
    return MK_ERR_BAD_CONFIG;
  const BarLayout bl = bar_layout(c.n_kv_heads, c.n_experts, c.max_batch);
  const int L = c.n_layers, d = c.head_dim, hkv = c.n_kv_heads;
  auto bar = [&](int layer, int off) { return layer * bl.per_layer + off; };
  const int n_attn_c = c.n_attn_claimers > 0 ? c.n_attn_claimers : n_sm;
  const int n_moe_c = c.n_moe_claimers > 0 ? c.n_moe_claimers : n_sm;
  const int cpg = combine_split(c, batch);

  std::vector<Desc> flat;
  auto norm_task = [&](int l) {
    Desc t = blank(OP_NORM, l, 0);
    if (l > 0) {
      t[F_W0] = bar(l - 1, bl.o);
      t[F_T0] = oproj_tiles(c, batch) + (l == bump_layer ? bump : 0);
      t[F_W1] = bar(l - 1, bl.moe);
      t[F_T1] = moe_target(c, batch);
    }
    t[F_SIG] = bar(l, bl.x);
    t[F_INC] = 1;
    flat.push_back(t);
  };
  auto wave = [&](Wave w, int l) {
    switch (w) {
      case W_NORM:
        norm_task(l);
        break;
      case W_QKV: {
        const int tph = d / 32, heads = c.n_q_heads + 2 * hkv;
        for (int i = 0; i < heads * tph; i++) {
          Desc t = blank(OP_QKV, l, i);
          t[F_W0] = bar(l, bl.x);
          t[F_T0] = 1;
          flat.push_back(t);     // the signalled counter depends on the head: set by the kernel
        }
        break;
      }
      case W_ROUTER: {
        const int n = (c.n_experts + kRowsRouter - 1) / kRowsRouter;
        for (int i = 0; i < n; i++) {
          Desc t = blank(OP_ROUTER, l, i);
          t[F_W0] = bar(l, bl.x);
          t[F_T0] = 1;
          flat.push_back(t);
        }
        break;
      }
      case W_ATTN:
        for (int i = 0; i < n_attn_c; i++) flat.push_back(blank(OP_ATTN, l, i));
        break;
      case W_COMBINE:
        // ATTN_COMBINE tasks per (sequence, KV head); the wait target is the
        // sequence's split count of the step, read by the kernel
        for (int b = 0; b < batch; b++)
          for (int g = 0; g < hkv; g++)
            for (int cc = 0; cc < cpg; cc++) {
              Desc t = blank(OP_COMBINE, l, (b * hkv + g) * cpg + cc);
              t[F_W0] = bar(l, bl.items + b);
              t[F_T0] = -1;
              t[F_SIG] = bar(l, bl.attn);
              t[F_INC] = 1;
              t[F_ARG] = cpg;
              flat.push_back(t);
            }
        break;
      case W_UP:
      case W_DOWN:
        for (int i = 0; i < n_moe_c; i++) {
          Desc t = blank(w == W_UP ? OP_MOE_UP : OP_MOE_DOWN, l, i);
          t[F_PW] = bar(l, bl.route);
          t[F_PT] = 1;
          flat.push_back(t);
        }
        break;
      case W_OPROJ: {
        const int n = oproj_tiles(c, batch);
        for (int i = 0; i < n; i++) {
          Desc t = blank(OP_OPROJ, l, i);
          t[F_W0] = bar(l, bl.attn);
          t[F_T0] = batch * hkv * cpg;
          t[F_SIG] = bar(l, bl.o);
          t[F_INC] = 1;
          flat.push_back(t);
        }
        break;
      }
    }
  };

  static const Wave orders[3][8] = {
      {W_NORM, W_QKV, W_ROUTER, W_ATTN, W_COMBINE, W_UP, W_DOWN, W_OPROJ},
      {W_NORM, W_QKV, W_ROUTER, W_ATTN, W_COMBINE, W_OPROJ, W_UP, W_DOWN},
      {W_NORM, W_QKV, W_ROUTER, W_UP, W_ATTN, W_DOWN, W_COMBINE, W_OPROJ}};
  for (int l = 0; l < L; l++)
    for (Wave w : orders[c.wave_order]) wave(w, l);
  // final norm and LM head
  norm_task(L);
  {
    const int n = (c.vocab + rows_lm(batch) - 1) / rows_lm(batch);
    for (int i = 0; i < n; i++) {
      Desc u = blank(OP_LMHEAD, L, i);
      u[F_W0] = bar(L, bl.x);
      u[F_T0] = 1;
      flat.push_back(u);
    }
  }

  // deal round-robin
  std::vector<std::vector<int>> per_sm(n_sm);
  for (size_t k = 0; k < flat.size(); k++) {
    flat[k][F_SEQ] = (int32_t)k;
    per_sm[k % n_sm].push_back((int)k);
  }
  out->tasks.clear();
  out->tasks.reserve(flat.size() * kDescWords);
  out->off.assign(n_sm + 1, 0);
  for (int s = 0; s < n_sm; s++) {
    out->off[s] = (int32_t)(out->tasks.size() / kDescWords);
    for (int k : per_sm[s]) out->tasks.insert(out->tasks.end(), flat[k].begin(), flat[k].end());
  }
  out->off[n_sm] = (int32_t)(out->tasks.size() / kDescWords);
  out->n_bars = (L + 1) * bl.per_layer;
  return MK_OK;
}

}  // namespace mk
