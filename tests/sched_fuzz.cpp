// The host scheduler over random configurations, built with AddressSanitizer
// and UndefinedBehaviorSanitizer by tests/test_sched_fuzz.py: every valid
// config (validate_config) with random SM counts, batches and lengths goes
// through attention_sms, split_kv and build_plan, and the shapes of what they
// return are checked.  Any out-of-bounds access or undefined behaviour aborts
// the run.
#include <stdio.h>
#include <stdlib.h>
#include <random>
#include <vector>
#include "mk_sched.h"
using namespace mk;
int main(int argc, char** argv) {
  std::mt19937 rng(argc > 1 ? atoi(argv[1]) : 1);
  auto pick = [&](std::initializer_list<int> v) { auto it = v.begin(); std::advance(it, rng() % v.size()); return *it; };
  long n_ok = 0, n_plans = 0;
  for (int iter = 0; iter < 4000; iter++) {
    mk_config c{};
    c.n_layers = 1 + rng() % 3;
    c.hidden = pick({64, 128, 256, 512, 1024, 2048, 4096});
    c.n_kv_heads = pick({1, 2, 4, 8});
    c.n_q_heads = c.n_kv_heads * pick({1, 2, 3, 4, 8});
    c.head_dim = pick({64, 128});
    c.n_experts = pick({1, 2, 8, 64, 128, 256});
    c.top_k = std::min(c.n_experts, pick({1, 2, 4, 8}));
    c.moe_inter = pick({64, 128, 256, 768, 1024});
    c.vocab = pick({1, 100, 1024, 32768});
    c.page_size = 16;
    c.rope_theta = 1e4; c.rms_eps = 1e-6f;
    c.max_batch = pick({1, 2, 4, 16});
    c.max_pages_per_seq = pick({1, 4, 64, 2048, 16384});
    c.num_kv_pages = 100000;
    c.max_attn_items = pick({0, 64, 8192});
    c.wave_order = rng() % 3;
    c.n_attn_claimers = pick({0, 0, 1, 7, 40, 152, 1000});
    c.n_moe_claimers = pick({0, 0, 3, 100});
    c.kv_split_tokens = pick({0, 0, 16, 64, 256});
    c.sm_cap = 0;
    c.moe_stage_depth = pick({0, 1, 3, 5});
    c.expert_format = pick({0, 0, 1});
    c.moe_claim_rows = pick({0, -1, 16, 128});
    if (validate_config(c) != MK_OK) continue;
    n_ok++;
    const int n_sm = pick({1, 2, 7, 36, 152});
    const int batch = 1 + rng() % c.max_batch;
    std::vector<int32_t> lens(batch);
    const int cap = c.max_pages_per_seq * 16 - 1;
    for (auto& l : lens) l = pick({0, 1, 15, 16, 17, 1000, 8192, 262144}) % (cap + 1);
    if (rng() % 4 == 0) for (auto& l : lens) l = cap;
    const int na = attention_sms(c, n_sm, batch, lens.data());
    if (na < 1 || na > n_sm) { printf("bad na %d (n_sm %d)\n", na, n_sm); return 1; }
    mk_config c2 = c;
    if (c2.max_attn_items == 0) c2.max_attn_items = 8192;
    std::vector<int32_t> it, so, me;
    const int split = split_kv(c2, n_sm, na, batch, lens.data(), &it, &so, &me);
    if (split >= 0) {
      if ((int)so.size() != n_sm + 1 || so.back() * 8 != (int)it.size()) { printf("bad sm_off\n"); return 1; }
      if ((int)me.size() != batch * 2) { printf("bad meta\n"); return 1; }
    }
    Plan plan;
    const int rc = build_plan(c, n_sm, batch, na, &plan);
    if (rc == MK_OK) {
      n_plans++;
      if ((int)plan.off.size() != n_sm + 1 || plan.off.back() * kDescWords != (int)plan.tasks.size()) {
        printf("bad plan off\n"); return 1;
      }
    }
  }
  printf("configs %ld plans %ld\n", n_ok, n_plans);
  return 0;
}
