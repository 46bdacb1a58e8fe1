// Host task scheduler: builds the per-SM task lists of one decode step.
//
// "Inside the megakernel serving engine for North Mini Code", §The task
// scheduler: the host builds named waves for each layer, chooses an order and
// gives each SM its list.  Here every wave is cut into equal shares (rows of
// a weight matrix, query heads to merge, hidden rows to produce) over the SMs
// that run it: all of them, or the SMs of one branch of the parallel layer.
// An SM's list holds one task per wave and layer; the shares whose size
// depends on routing (the experts' rows) are fixed as "slice s of n" and
// resolved on the device once the routing is known; with several tokens the
// SMs that hold such a slice claim fixed-size tiles of those rows from
// per-layer counters instead (the slice then only says that the SM takes
// part).  Any order of the waves
// in which ROUTE precedes UP precedes DOWN and ATTN precedes COMBINE precedes
// OUT (and, with several tokens, DOWN precedes OUT, whose expert sums wait for
// every DOWN task) has no circular wait (every wait points at an earlier wave
// of the same layer, or at the previous layer).
#include "mk_sched.h"

#include <math.h>

#include <algorithm>
#include <array>

namespace mk {

// contraction lengths the GEMV supports: whole 256-column segments (at most
// 16, the one-token path holds a lane's share of a row in registers), or one
// partial segment of a multiple of 8 columns
static bool gemv_k(int k) { return (k >= 8 && k < 256 && k % 8 == 0) || (k % 256 == 0 && k <= 4096); }

int validate_config(const mk_config& c) {
  if (c.n_layers < 1 || c.hidden < 8 || c.n_q_heads < 1 || c.n_kv_heads < 1) return MK_ERR_BAD_CONFIG;
  if (c.n_q_heads % c.n_kv_heads) return MK_ERR_BAD_CONFIG;
  const int grp = c.n_q_heads / c.n_kv_heads;
  if (grp > 8 || kConsumerWarps % c.n_kv_heads) return MK_ERR_BAD_CONFIG;
  if (c.head_dim != 64 && c.head_dim != 128) return MK_ERR_BAD_CONFIG;
  if (!gemv_k(c.hidden) || !gemv_k(c.moe_inter) || !gemv_k(c.n_q_heads * c.head_dim))
    return MK_ERR_BAD_CONFIG;
  // the attention keeps every query head's BF16 high and low halves in the
  // 16 KB reduction buffer
  if (c.n_q_heads * c.head_dim > 4096) return MK_ERR_BAD_CONFIG;
  // one token: the hidden vectors of all routed experts are staged together
  if (c.top_k * c.moe_inter > kXsFloats) return MK_ERR_BAD_CONFIG;
  if (c.n_experts < 1 || c.n_experts > 256 || c.top_k < 1 || c.top_k > 8 || c.top_k > c.n_experts)
    return MK_ERR_BAD_CONFIG;
  if (c.vocab < 1 || c.page_size != 16) return MK_ERR_BAD_CONFIG;
  // one 16-token page of every KV head (K or V) must fit half a stage
  if (c.n_kv_heads * c.page_size * c.head_dim * 2 > kStageBytes / 2) return MK_ERR_BAD_CONFIG;
  if (c.max_batch < 1 || c.max_batch > kMaxBatch || c.max_batch * c.top_k > kMaxActive)
    return MK_ERR_BAD_CONFIG;
  if (c.max_pages_per_seq < 1 || c.num_kv_pages < 1) return MK_ERR_BAD_CONFIG;
  if (!(c.rope_theta > 0.0) || !(c.rms_eps >= 0.f)) return MK_ERR_BAD_CONFIG;
  if (c.max_attn_items < 0 || c.n_attn_claimers < 0 || c.n_moe_claimers < 0 || c.sm_cap < 0 ||
      c.timeout_ms < 0 || c.trace_records < 0)
    return MK_ERR_BAD_CONFIG;
  if (c.kv_split_tokens < 0 || c.kv_split_tokens % 16) return MK_ERR_BAD_CONFIG;
  if (c.moe_stage_depth < 0 || c.moe_stage_depth > kStages) return MK_ERR_BAD_CONFIG;
  if (c.wave_order < MK_WAVES_DEFAULT || c.wave_order > MK_WAVES_INTERLEAVED) return MK_ERR_BAD_CONFIG;
  if (c.expert_format != MK_EXPERTS_BF16 && c.expert_format != MK_EXPERTS_FP8_E4M3) return MK_ERR_BAD_CONFIG;
  if (c.moe_claim_rows < -1 || (c.moe_claim_rows > 0 && c.moe_claim_rows % 16)) return MK_ERR_BAD_CONFIG;
  // 8-bit experts: the one-token path (tensor-core rows of 2048 bytes, or
  // CUDA-core rows of 256, 512 or 1024 bytes in 16-byte lane chunks; a whole
  // number of hidden rows in every 4096-row stage of the down projection)
  if (c.expert_format == MK_EXPERTS_FP8_E4M3 &&
      (c.max_batch != 1 || !(c.hidden == 2048 || c.hidden == 1024 || c.hidden == 512 || c.hidden == 256) ||
       c.moe_inter % 16))
    return MK_ERR_BAD_CONFIG;
  return MK_OK;
}

namespace {

using Desc = std::array<int32_t, kDescWords>;

Desc task(int op, int layer, int a0, int a1) {
  Desc d;
  d.fill(0);
  d[F_OP] = op;
  d[F_LAYER] = layer;
  d[F_A0] = a0;
  d[F_A1] = a1;
  return d;
}

}  // namespace

int attention_sms(const mk_config& c, int n_sm, int batch, const int32_t* seq_lens) {
  if (n_sm < 2) return n_sm;
  if (c.n_attn_claimers > 0) return c.n_attn_claimers < n_sm ? c.n_attn_claimers : n_sm;
  double keys = 0.0;
  for (int b = 0; b < batch; b++) keys += (double)(seq_lens[b] + 1);
  const double kv = keys * 2.0 * c.n_kv_heads * c.head_dim * 2.0;
  const double experts = (double)std::min(c.n_experts, batch * c.top_k);
  // gate, up and down: 2 bytes a weight.  8-bit experts move 1 byte a
  // weight but their pieces cost more than their bytes (the activations' term
  // split, the partial rows): weighted as 1.5 (48 attention SMs at 8K, the
  // measured best of 40 / 44 / 48 / 56 / 64 / 72)
  const double moe = experts * 3.0 * c.moe_inter * c.hidden * (c.expert_format == MK_EXPERTS_FP8_E4M3 ? 1.5 : 2.0);
  // The branches split the SMs in proportion to their bytes, a KV byte
  // weighted by w against an expert byte.  w folds in what the bytes do not
  // say: at short contexts the attention's fixed work per layer (query
  // staging, the merges, the combine) weighs more, and with several tokens
  // the expert GEMVs cost more per byte.  Fitted to the measured best splits
  // on the 30B/3.3B model: 40 attention SMs at batch 1 with 8K context
  // (w = 1.6), 128 at 256K, 20-24 at batch 4 with 8K, 22-26 at batch 16 with
  // contexts of 1K-32K.
  const double mean_ctx = keys / batch;
  const double w = 1.6 * pow(8192.0 / mean_ctx, 0.22) / pow((double)batch, 0.45);
  double ideal = n_sm * w * kv / (w * kv + moe);
  // several tokens: at least 16 % of the SMs on the attention branch, 23 %
  // from 8 tokens up.  As the contexts of a continuous batch shrink (short
  // sequences joining), the byte share would drop to 8 % and the expert
  // branch's per-byte cost (its multi-token GEMVs) does not follow; with the
  // expert tiles claimed, 36 of 152 SMs (32 within 0.5 %) were the best
  // fixed split over whole batch-16 runs and 24 over batch-4 runs.
  if (batch > 1) ideal = std::max(ideal, (batch >= 8 ? 0.23 : 0.16) * n_sm);
  // in steps of 4 SMs on a large GPU: each split has its own task lists,
  // built and uploaded the first time it is used, and the contexts of a
  // continuous batch move the ideal split by a few SMs every step
  const int q = n_sm >= 64 ? 4 : 1;
  const int na = q * (int)(ideal / q + 0.5);
  return std::max(1, std::min(n_sm - 1, na));
}

int build_plan(const mk_config& c, int n_sm, int batch, int n_attn, Plan* out, int bump_layer, int bump) {
  if (validate_config(c) != MK_OK || n_sm < 1 || batch < 1 || batch > c.max_batch || n_attn < 1 ||
      n_attn > n_sm)
    return MK_ERR_BAD_CONFIG;
  const BarLayout bl = bar_layout(c.max_batch);
  const int L = c.n_layers;
  const long long qrows = (long long)(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  const long long units = (long long)batch * c.n_q_heads;
  const bool roles = n_attn < n_sm;
  const int nmoe = roles ? n_sm - n_attn : moe_sms(c, n_sm);
  const int ncomb = roles ? n_attn : n_sm;
  // (one token: the UP slices also produce the down projection's per-group
  // partials and the DOWN wave adds them up, row by row)
  const int ndown = roles ? n_sm - n_attn : n_sm;

  static const int orders[3][7] = {
      {OP_P1, OP_ROUTE, OP_ATTN, OP_UP, OP_COMBINE, OP_DOWN, OP_OUT},
      {OP_P1, OP_ROUTE, OP_ATTN, OP_COMBINE, OP_UP, OP_DOWN, OP_OUT},
      {OP_P1, OP_ROUTE, OP_UP, OP_ATTN, OP_DOWN, OP_COMBINE, OP_OUT}};
  // the attention branch needs no routing; several tokens: the expert
  // branch's down rows only wait for its own UP wave, so they run while
  // attention is under way; one token: the expert branch takes its (few)
  // O-proj rows as soon as the attention is combined, before the sums of the
  // experts' partials, which nothing on the SM waits for
  static const int attn_role[4] = {OP_P1, OP_ATTN, OP_COMBINE, OP_OUT};
  static const int moe_role[5] = {OP_P1, OP_ROUTE, OP_UP, OP_DOWN, OP_OUT};
  static const int moe_role1[5] = {OP_P1, OP_ROUTE, OP_UP, OP_OUT, OP_DOWN};

  // P1 rows.  The router rows go, 8 rows (one stage) per SM or more if there
  // are few of them, to the first expert-branch SMs (all SMs when there are
  // no roles); they run first and
  // release the router counter on their own, so the routing can start soon
  // after the norm; they take no W_qkv rows.  The W_qkv rows are split over
  // the other SMs in proportion to their even share of all P1 rows.
  const long long total1 = c.n_experts + qrows;
  std::vector<int> r_lo(n_sm, 0), r_hi(n_sm, 0), q_lo(n_sm, 0), q_hi(n_sm, 0);
  {
    const int cand = roles ? n_sm - n_attn : n_sm;               // >= 1
    const int per = (std::max(8, (c.n_experts + cand - 1) / cand) + 7) / 8 * 8;
    int next = 0;
    for (int s = 0; s < n_sm && next < c.n_experts; s++) {
      if (roles && is_attn_sm(s, n_sm, n_attn)) continue;
      r_lo[s] = next;
      r_hi[s] = std::min(c.n_experts, next + per);
      next = r_hi[s];
    }
    std::vector<long long> wq(n_sm + 1, 0);
    for (int pass = 0; pass < 2 && wq[n_sm] == 0; pass++)
      for (int s = 0; s < n_sm; s++) {
        int lo, hi;
        share(total1, n_sm, s, &lo, &hi);
        // router SMs take no W_qkv rows, unless every SM holds router rows
        wq[s + 1] = wq[s] + ((pass == 0 && r_hi[s] > r_lo[s]) ? 0 : (hi - lo));
      }
    // in whole groups of 8 rows (one tensor-core stage of 2048-column rows)
    // where the row count allows it
    const long long qg = qrows % 8 == 0 ? 8 : 1;
    for (int s = 0; s < n_sm; s++) {
      q_lo[s] = wq[n_sm] > 0 ? (int)(qg * (qrows / qg * wq[s] / wq[n_sm])) : 0;
      q_hi[s] = wq[n_sm] > 0 ? (int)(qg * (qrows / qg * wq[s + 1] / wq[n_sm])) : 0;
    }
  }

  // O-proj rows.  One token: an attention-branch SM, idle from its COMBINE
  // until the layer ends, takes kOutAttnWeight times an expert-branch SM's
  // share.
  std::vector<int> o_lo(n_sm, 0), o_hi(n_sm, 0);
  {
    constexpr long long kOutAttnWeight = 4;
    std::vector<long long> wo(n_sm + 1, 0);
    for (int s = 0; s < n_sm; s++)
      wo[s + 1] = wo[s] + ((roles && batch == 1 && is_attn_sm(s, n_sm, n_attn)) ? kOutAttnWeight : 1);
    const long long og = c.hidden % 8 == 0 ? 8 : 1;   // whole groups of 8 rows
    for (int s = 0; s < n_sm; s++) {
      o_lo[s] = (int)(og * (c.hidden / og * wo[s] / wo[n_sm]));
      o_hi[s] = (int)(og * (c.hidden / og * wo[s + 1] / wo[n_sm]));
    }
  }

  out->tasks.clear();
  out->off.assign(n_sm + 1, 0);
  for (int s = 0; s < n_sm; s++) {
    out->off[s] = (int32_t)(out->tasks.size() / kDescWords);
    const int* ops;
    int nops;
    if (!roles) {
      ops = orders[c.wave_order];
      nops = 7;
    } else if (is_attn_sm(s, n_sm, n_attn)) {
      ops = attn_role;
      nops = 4;
    } else {
      ops = batch == 1 ? moe_role1 : moe_role;
      nops = 5;
    }
    std::vector<Desc> list;
    for (int l = 0; l < L; l++) {
      for (int k = 0; k < nops; k++) {
        const int op = ops[k];
        int lo = 0, hi = 0;
        switch (op) {
          case OP_P1: lo = r_lo[s]; hi = r_hi[s]; break;   // router rows; W_qkv rows below
          case OP_COMBINE: share(units, ncomb, roles ? attn_before(s, n_sm, n_attn) : s, &lo, &hi); break;
          case OP_OUT: lo = o_lo[s]; hi = o_hi[s]; break;
          case OP_DOWN: {
            // one token: hidden rows (sums of the experts' partials); several:
            // slice s of n over the routed experts' rows (like UP)
            const int slice = roles ? moe_rank(s, n_sm, n_attn) : s;
            if (batch == 1) {
              share(c.hidden, ndown, slice, &lo, &hi);
            } else {
              lo = slice < ndown ? slice : -1;
              hi = ndown;
            }
            break;
          }
          case OP_UP: {
            const int slice = roles ? moe_rank(s, n_sm, n_attn) : s;
            lo = slice < nmoe ? slice : -1;
            hi = nmoe;
            break;
          }
          default: break;
        }
        Desc t = task(op, l, lo, hi);
        if (op == OP_P1) {
          t[F_B0] = q_lo[s];
          t[F_B1] = q_hi[s];
          if (l == bump_layer) t[F_BUMP] = bump;
        }
        list.push_back(t);
      }
    }
    {
      // LM-head rows in whole groups of 8 (the last SM also takes the vocabulary's tail)
      int lo, hi;
      share(c.vocab / 8, n_sm, s, &lo, &hi);
      lo *= 8;
      hi = s == n_sm - 1 ? c.vocab : hi * 8;
      Desc t = task(OP_FINAL, L, lo, hi);
      if (L == bump_layer) t[F_BUMP] = bump;
      list.push_back(t);
    }
    for (size_t k = 0; k < list.size(); k++) {
      list[k][F_SEQ] = (int32_t)k;
      out->tasks.insert(out->tasks.end(), list[k].begin(), list[k].end());
    }
  }
  out->off[n_sm] = (int32_t)(out->tasks.size() / kDescWords);
  out->n_bars = L * bl.per_layer;
  out->n_comb_sms = ncomb;
  out->n_up_sms = roles ? nmoe : n_sm;
  out->n_down_sms = ndown;
  // P1 shares that hold router rows (each such SM signals the router counter
  // as soon as its router rows are done)
  int nr = 0;
  for (int s = 0; s < n_sm; s++) nr += r_hi[s] > r_lo[s];
  out->n_rtr_sms = nr;
  return MK_OK;
}

int split_kv(const mk_config& c, int n_sm, int n_attn, int batch, const int32_t* seq_lens,
             std::vector<int32_t>* items, std::vector<int32_t>* sm_off, std::vector<int32_t>* meta) {
  const int P = c.page_size;
  const int na = n_attn;
  items->clear();
  sm_off->assign(n_sm + 1, 0);
  meta->assign((size_t)batch * 2, 0);
  auto add = [&](int b, int t0, int t1) {
    const int32_t it[8] = {b, 0, 0, t0, t1, 0, seq_lens[b], 0};
    items->insert(items->end(), it, it + 8);
  };
  int split = c.kv_split_tokens;
  if (split > 0) {
    // fixed split size: items in sequence order, dealt out in contiguous runs
    long long n_items = 0;
    for (;;) {
      n_items = 0;
      for (int b = 0; b < batch; b++) n_items += (seq_lens[b] + 1 + split - 1) / split;
      if (n_items <= c.max_attn_items || split >= (1 << 24)) break;
      split *= 2;
    }
    if (n_items > c.max_attn_items) return -1;
    for (int b = 0; b < batch; b++) {
      const int keys = seq_lens[b] + 1;
      for (int t0 = 0; t0 < keys; t0 += split) add(b, t0, std::min(keys, t0 + split));
    }
    for (int s = 0; s <= n_sm; s++)
      (*sm_off)[s] = (int32_t)(n_items * attn_before(s, n_sm, na) / na);
  } else {
    // balanced: the concatenated pages of all sequences cut into na equal runs
    std::vector<long long> first(batch + 1, 0);
    for (int b = 0; b < batch; b++) first[b + 1] = first[b] + (seq_lens[b] + 1 + P - 1) / P;
    const long long T = first[batch];
    int b = 0;
    for (int s = 0; s < n_sm; s++) {
      (*sm_off)[s] = (int32_t)(items->size() / 8);
      if (!is_attn_sm(s, n_sm, na)) continue;
      const int r = attn_before(s, n_sm, na);
      const long long g0 = T * r / na, g1 = T * (r + 1) / na;
      while (b < batch && first[b + 1] <= g0) b++;
      for (int bb = b; bb < batch && first[bb] < g1; bb++) {
        const long long p0 = std::max(g0, first[bb]) - first[bb];
        const long long p1 = std::min(g1, first[bb + 1]) - first[bb];
        if (p1 <= p0) continue;
        const int keys = seq_lens[bb] + 1;
        add(bb, (int)(p0 * P), (int)std::min<long long>(keys, p1 * P));
      }
    }
    (*sm_off)[n_sm] = (int32_t)(items->size() / 8);
    if ((long long)(items->size() / 8) > c.max_attn_items) return -1;
    split = 0;
  }
  // split index, count and first item of every sequence (items of a sequence are contiguous)
  const int n = (int)(items->size() / 8);
  for (int k = 0; k < n; k++) {
    int32_t* it = items->data() + (size_t)k * 8;
    const int b = it[AI_B];
    if ((*meta)[b * 2 + 1] == 0) (*meta)[b * 2 + 0] = k;
    it[AI_S] = (*meta)[b * 2 + 1]++;
  }
  for (int k = 0; k < n; k++) {
    int32_t* it = items->data() + (size_t)k * 8;
    it[AI_NSPLIT] = (*meta)[it[AI_B] * 2 + 1];
    it[AI_BASE] = (*meta)[it[AI_B] * 2 + 0];
  }
  return split;
}

}  // namespace mk
