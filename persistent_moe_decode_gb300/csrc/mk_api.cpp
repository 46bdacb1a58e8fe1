// C ABI of the persistent decode step (declared in include/mk.h).
//
// Mirrors the host loop of "Inside the megakernel serving engine for North
// Mini Code", §The serving engine around the kernel: the page tables and
// per-sequence state are snapshot into device memory (update_kv_page_tables),
// the counters are zeroed (clear_scratch_and_barriers), the split-KV schedule
// follows the live contexts (select_schedule(max_live_context)) and the
// persistent kernel is launched (launch_megakernel).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <new>
#include <vector>

#include "../../include/mk.h"
#include "mk_layout.h"
#include "mk_sched.h"

namespace mk {
cudaError_t launch_step(const Params& p, int n_sm, cudaStream_t stream);
cudaError_t relayout_down(const uint16_t* src, uint16_t* dst, int E, int H, int I);
cudaError_t relayout_down_e4m3(const uint8_t* src, uint8_t* dst, int E, int H, int I);
size_t step_smem_bytes();
int step_kernel_regs();
int static_counters(int device, uint32_t** out);
}  // namespace mk

using namespace mk;

namespace {

struct DevPlan {
  int32_t* tasks = nullptr;
  int32_t* off = nullptr;
  size_t n_tasks = 0;
  int n_comb_sms = 0, n_up_sms = 0, n_down_sms = 0, n_rtr_sms = 0;
};

// plans are cached per (batch, attention SMs)
inline int plan_key(int batch, int n_attn) { return batch * 4096 + n_attn; }

struct Staging {
  uint8_t* host = nullptr;   // pinned
  cudaEvent_t done = nullptr;
  bool pending = false;
};

}  // namespace

struct mk_handle {
  mk_config cfg;
  int device = 0;
  int n_sm = 0;
  Params base;                // everything but the per-step fields
  std::vector<void*> allocs;  // device allocations owned here
  size_t dev_bytes = 0;
  std::map<int, DevPlan> plans;   // per batch size
  int bump_layer = -1, bump = 0;
  // per-step device inputs
  int32_t* d_tokens = nullptr;
  int32_t* d_pos = nullptr;
  int32_t* d_pt = nullptr;
  float* d_rope = nullptr;
  int32_t* d_items = nullptr;
  int32_t* d_smoff = nullptr;
  int32_t* d_meta = nullptr;
  size_t step_bytes_cap = 0;
  Staging stage[2];
  int stage_idx = 0;
  // scheduled step
  bool scheduled = false;
  int batch = 0;
  int n_items = 0;
  int split = 0;
  int n_attn = 0;
  std::vector<int32_t> items, smoff, meta;
  int last_batch = 0;
  uint32_t* d_bars = nullptr;   // err words live at the start
  size_t bar_words = 0;
  int32_t* d_trace = nullptr;
  size_t trace_words = 0;
  int32_t* d_dbg = nullptr;
  size_t dbg_words = 0;
};

namespace {

constexpr int kErrWords = 32;

template <class T>
int dalloc(mk_handle* h, T** p, size_t count) {
  void* q = nullptr;
  const size_t bytes = std::max<size_t>(count * sizeof(T), 16);
  if (cudaMalloc(&q, bytes) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_OOM;
  }
  h->allocs.push_back(q);
  h->dev_bytes += bytes;
  *p = (T*)q;
  return MK_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int upload_ptrs(mk_handle* h, const void* const* src, int L, const void* const** dst) {
  if (!src) return MK_ERR_BAD_ARG;
  for (int l = 0; l < L; l++)
    if (!src[l] || !aligned16(src[l])) return MK_ERR_BAD_ARG;
  void** d = nullptr;
  int rc = dalloc(h, &d, (size_t)L);
  if (rc) return rc;
  if (cudaMemcpy(d, src, sizeof(void*) * L, cudaMemcpyHostToDevice) != cudaSuccess) return MK_ERR_CUDA;
  *dst = (const void* const*)d;
  return MK_OK;
}

// cuTensorMapEncodeTiled from the driver (through the runtime's entry-point
// lookup, so the library needs no link against libcuda)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    else
      cudaGetLastError();
  }
  return fn;
}

// tensor maps of every layer's K and V pool: 2-D [pages * hkv * page_size][d]
// BF16, boxes of 64 dims x (hkv * page_size) rows (one page of every KV head,
// half or all of its dims), 128-byte swizzle
int make_kv_maps(mk_handle* h, const mk_weights* w, const uint8_t** out) {
  static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
  const mk_config& c = h->cfg;
  const int L = c.n_layers;
  auto enc = tensor_map_encoder();
  if (!enc) return MK_ERR_CUDA;
  std::vector<CUtensorMap> maps((size_t)2 * L);
  const cuuint64_t dims[2] = {(cuuint64_t)c.head_dim,
                              (cuuint64_t)c.num_kv_pages * c.n_kv_heads * c.page_size};
  const cuuint64_t strides[1] = {(cuuint64_t)c.head_dim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)(c.n_kv_heads * c.page_size)};
  const cuuint32_t es[2] = {1, 1};
  if (dims[1] >= (1ull << 32)) return MK_ERR_BAD_CONFIG;
  for (int l = 0; l < L; l++)
    for (int kv = 0; kv < 2; kv++) {
      void* base = kv ? w->v_pool[l] : w->k_pool[l];
      if (enc(&maps[(size_t)2 * l + kv], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MK_ERR_BAD_ARG;
    }
  uint8_t* d = nullptr;
  int rc = dalloc(h, &d, maps.size() * sizeof(CUtensorMap));
  if (rc) return rc;
  if (cudaMemcpy(d, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) != cudaSuccess)
    return MK_ERR_CUDA;
  *out = d;
  return MK_OK;
}

// a 2-D tiled tensor map without swizzle: [outer][inner] elements of `esize`
// bytes, boxes of box_in x box_out
int make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
                uint64_t outer, uint32_t box_in, uint32_t box_out) {
  auto enc = tensor_map_encoder();
  if (!enc) return MK_ERR_CUDA;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * (uint64_t)esize};
  const cuuint32_t box[2] = {box_in, box_out};
  const cuuint32_t es[2] = {1, 1};
  if (outer >= (1ull << 32)) return MK_ERR_BAD_CONFIG;
  if (enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MK_ERR_BAD_ARG;
  return MK_OK;
}

// One token: a weight matrix [rows][K] (K = 2048 or 4096) viewed as 3-D
// [K / 64][rows][64] BF16 (strides: K * 2 bytes per row, 128 bytes per column
// block), boxes of every column block x (32768 / (2 K)) rows x 64 columns,
// 128-byte swizzle: one stage of whole rows per copy.
int make_row_map(CUtensorMap* m, const void* base, uint64_t rows, int K, int box_rows = 0) {
  auto enc = tensor_map_encoder();
  if (!enc) return MK_ERR_CUDA;
  const cuuint64_t dims[3] = {64, rows, (cuuint64_t)(K / 64)};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)(box_rows > 0 ? box_rows : 32768 / (2 * K)), (cuuint32_t)(K / 64)};
  const cuuint32_t es[3] = {1, 1, 1};
  if (rows >= (1ull << 32) || !aligned16(base)) return MK_ERR_BAD_ARG;
  if (enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MK_ERR_BAD_ARG;
  return MK_OK;
}

// the tensor maps of every layer's router, W_qkv, W_o, gate and up
// matrices and of the LM head (W_MAP_* order); none when the hidden size does
// not take the tensor-core path
int make_weight_maps(mk_handle* h, const mk_weights* w, const uint8_t** out) {
  const mk_config& c = h->cfg;
  *out = nullptr;
  const int H = c.hidden, KO = c.n_q_heads * c.head_dim, L = c.n_layers;
  if (!rotated_rows(H)) return MK_OK;
  if (!rotated_rows(KO)) return MK_ERR_BAD_CONFIG;   // both GEMV paths in one layer are not built
  std::vector<CUtensorMap> maps((size_t)W_MAPS_PER_LAYER * L + 1);
  const uint64_t qrows = (uint64_t)(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  const uint64_t erows = (uint64_t)c.n_experts * c.moe_inter;
  for (int l = 0; l < L; l++) {
    CUtensorMap* m = &maps[(size_t)W_MAPS_PER_LAYER * l];
    int rc = make_row_map(&m[W_MAP_ROUTER], w->w_router[l], (uint64_t)c.n_experts, H);
    if (!rc) rc = make_row_map(&m[W_MAP_QKV], w->w_qkv[l], qrows, H);
    if (!rc) rc = make_row_map(&m[W_MAP_O], w->w_o[l], (uint64_t)H, KO);
    // 8-bit experts: rows of H bytes, mapped as H / 2 two-byte columns (16
    // rows per box instead of 8; the copy moves bytes, the kernel reads E4M3)
    const int KE = c.expert_format == MK_EXPERTS_FP8_E4M3 ? H / 2 : H;
    if (!rc) rc = make_row_map(&m[W_MAP_GATE], w->w_gate[l], erows, KE);
    if (!rc) rc = make_row_map(&m[W_MAP_UP], w->w_up[l], erows, KE);
    if (rc) return rc;
  }
  int rc = make_row_map(&maps.back(), w->lm_head, (uint64_t)c.vocab, H);
  if (rc) return rc;
  uint8_t* d = nullptr;
  rc = dalloc(h, &d, maps.size() * sizeof(CUtensorMap));
  if (rc) return rc;
  if (cudaMemcpy(d, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) != cudaSuccess)
    return MK_ERR_CUDA;
  *out = d;
  return MK_OK;
}

// several tokens: the maps of every layer's W_down as [E H rows][I], boxes of
// 16 rows x all of I (the tensor-core down projection of the routed entries)
int make_down_maps(mk_handle* h, const mk_weights* w, const uint8_t** out) {
  const mk_config& c = h->cfg;
  *out = nullptr;
  if (!rotated_rows(c.hidden) || !mma_multi_down(c.moe_inter) || c.max_batch < 2) return MK_OK;
  std::vector<CUtensorMap> maps((size_t)c.n_layers);
  for (int l = 0; l < c.n_layers; l++) {
    const int rc = make_row_map(&maps[l], w->w_down[l], (uint64_t)c.n_experts * c.hidden, c.moe_inter,
                                kDownBoxRows);
    if (rc) return rc;
  }
  uint8_t* d = nullptr;
  int rc = dalloc(h, &d, maps.size() * sizeof(CUtensorMap));
  if (rc) return rc;
  if (cudaMemcpy(d, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) != cudaSuccess)
    return MK_ERR_CUDA;
  *out = d;
  return MK_OK;
}

// one token: the tensor map of the per-group partial buffer (24 x 256 fp32)
int make_moe_map(mk_handle* h, float* mpart, const uint8_t** mp) {
  const mk_config& c = h->cfg;
  CUtensorMap map;
  int rc = make_map_2d(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, mpart, (uint64_t)c.hidden,
                       (uint64_t)c.top_k * (c.moe_inter / 8), 24, 256);   // kMredCols
  if (rc) return rc;
  uint8_t* d = nullptr;
  rc = dalloc(h, &d, sizeof(CUtensorMap));
  if (rc) return rc;
  if (cudaMemcpy(d, &map, sizeof(CUtensorMap), cudaMemcpyHostToDevice) != cudaSuccess) return MK_ERR_CUDA;
  *mp = d;
  return MK_OK;
}

// the blocked copy of every layer's down projection ([E][I/8][H][8] per layer)
int make_down_blocks(mk_handle* h, const mk_weights* w, const uint16_t** out) {
  const mk_config& c = h->cfg;
  const size_t per_layer = (size_t)c.n_experts * c.moe_inter * c.hidden;
  const bool fp8 = c.expert_format == MK_EXPERTS_FP8_E4M3;
  uint16_t* d = nullptr;
  // elements of 2 bytes (BF16), or bytes (E4M3: half as many 2-byte words)
  int rc = dalloc(h, &d, fp8 ? per_layer * c.n_layers / 2 : per_layer * c.n_layers);
  if (rc) return rc;
  for (int l = 0; l < c.n_layers; l++) {
    const cudaError_t e =
        fp8 ? relayout_down_e4m3((const uint8_t*)w->w_down[l], (uint8_t*)d + per_layer * l, c.n_experts, c.hidden,
                                 c.moe_inter)
            : relayout_down((const uint16_t*)w->w_down[l], d + per_layer * l, c.n_experts, c.hidden, c.moe_inter);
    if (e != cudaSuccess) return MK_ERR_CUDA;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return MK_ERR_CUDA;
  *out = d;
  return MK_OK;
}

void free_plans(mk_handle* h) {
  for (auto& kv : h->plans) {
    cudaFree(kv.second.tasks);
    cudaFree(kv.second.off);
  }
  h->plans.clear();
}

int ensure_plan(mk_handle* h, int batch, int n_attn, DevPlan** out) {
  auto it = h->plans.find(plan_key(batch, n_attn));
  if (it == h->plans.end()) {
    Plan plan;
    int rc = build_plan(h->cfg, h->n_sm, batch, n_attn, &plan, h->bump_layer, h->bump);
    if (rc) return rc;
    DevPlan dp;
    dp.n_tasks = plan.tasks.size() / kDescWords;
    dp.n_comb_sms = plan.n_comb_sms;
    dp.n_up_sms = plan.n_up_sms;
    dp.n_down_sms = plan.n_down_sms;
    dp.n_rtr_sms = plan.n_rtr_sms;
    if (cudaMalloc(&dp.tasks, std::max<size_t>(plan.tasks.size() * 4, 16)) != cudaSuccess ||
        cudaMalloc(&dp.off, plan.off.size() * 4) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(dp.tasks);
      return MK_ERR_OOM;
    }
    if (cudaMemcpy(dp.tasks, plan.tasks.data(), plan.tasks.size() * 4, cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(dp.off, plan.off.data(), plan.off.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
      return MK_ERR_CUDA;
    it = h->plans.emplace(plan_key(batch, n_attn), dp).first;
  }
  *out = &it->second;
  return MK_OK;
}

size_t step_upload_bytes(const mk_config& c, int n_sm, int batch, int n_items) {
  return (size_t)batch * 4 * 2 + (size_t)batch * c.max_pages_per_seq * 4 +
         (size_t)batch * (c.head_dim / 2) * 2 * 4 + (size_t)n_items * 8 * 4 + (size_t)batch * 2 * 4 +
         (size_t)(n_sm + 1) * 4;
}

}  // namespace

extern "C" {

int mk_abi_version(void) { return MK_ABI_VERSION; }

const char* mk_strerror(int code) {
  switch (code) {
    case MK_OK: return "ok";
    case MK_ERR_BAD_CONFIG: return "unsupported or inconsistent config";
    case MK_ERR_OOM: return "allocation failed";
    case MK_ERR_BAD_PAGE: return "page index out of range";
    case MK_ERR_BATCH_TOO_LARGE: return "batch outside 1..max_batch";
    case MK_ERR_NOT_SCHEDULED: return "decode step without a scheduled batch";
    case MK_ERR_TIMEOUT: return "device wait timed out";
    case MK_ERR_CUDA: return "CUDA runtime error";
    case MK_ERR_BAD_ARG: return "bad argument";
    case MK_ERR_DEVICE: return "kernel reported an inconsistent task or queue";
  }
  return "unknown error";
}

int mk_plan(const mk_config* cfg, int n_sm, int batch, int32_t* tasks, int32_t* offsets,
            int* n_tasks_out, int* n_barriers_out) {
  if (!cfg) return MK_ERR_BAD_ARG;
  Plan plan;
  const int n_attn = cfg->n_attn_claimers > 0 && cfg->n_attn_claimers < n_sm ? cfg->n_attn_claimers : n_sm;
  int rc = build_plan(*cfg, n_sm, batch, n_attn, &plan);
  if (rc) return rc;
  if (n_tasks_out) *n_tasks_out = (int)(plan.tasks.size() / kDescWords);
  if (n_barriers_out) *n_barriers_out = plan.n_bars;
  if (tasks) memcpy(tasks, plan.tasks.data(), plan.tasks.size() * 4);
  if (offsets) memcpy(offsets, plan.off.data(), plan.off.size() * 4);
  return MK_OK;
}

int mk_plan_step(const mk_config* cfg, int n_sm, int batch, const int32_t* seq_lens, int32_t* info,
                 int32_t* tasks, int32_t* task_off, int32_t* items, int32_t* item_off, int32_t* meta) {
  if (!cfg || !seq_lens || !info || n_sm < 1) return MK_ERR_BAD_ARG;
  if (batch < 1 || batch > cfg->max_batch) return MK_ERR_BATCH_TOO_LARGE;
  mk_config c = *cfg;
  if (c.max_attn_items == 0) c.max_attn_items = 8192;
  for (int b = 0; b < batch; b++)
    if (seq_lens[b] < 0) return MK_ERR_BAD_ARG;
  // the same three calls mk_schedule_step makes
  const int na = attention_sms(c, n_sm, batch, seq_lens);
  std::vector<int32_t> it, so, me;
  const int split = split_kv(c, n_sm, na, batch, seq_lens, &it, &so, &me);
  if (split < 0) return MK_ERR_BAD_CONFIG;
  Plan plan;
  int rc = build_plan(c, n_sm, batch, na, &plan);
  if (rc) return rc;
  info[0] = (int32_t)(plan.tasks.size() / kDescWords);
  info[1] = (int32_t)(it.size() / 8);
  info[2] = na;
  info[3] = plan.n_comb_sms;
  info[4] = plan.n_up_sms;
  info[5] = plan.n_down_sms;
  info[6] = plan.n_rtr_sms;
  info[7] = split;
  info[8] = plan.n_bars;
  if (tasks) memcpy(tasks, plan.tasks.data(), plan.tasks.size() * 4);
  if (task_off) memcpy(task_off, plan.off.data(), plan.off.size() * 4);
  if (items) memcpy(items, it.data(), it.size() * 4);
  if (item_off) memcpy(item_off, so.data(), so.size() * 4);
  if (meta) memcpy(meta, me.data(), me.size() * 4);
  return MK_OK;
}

void mk_destroy(mk_handle* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_plans(h);
  for (void* p : h->allocs) cudaFree(p);
  for (auto& s : h->stage) {
    if (s.host) cudaFreeHost(s.host);
    if (s.done) cudaEventDestroy(s.done);
  }
  delete h;
}

int mk_create(const mk_config* cfg, const mk_weights* w, mk_handle** out) {
  if (!cfg || !w || !out) return MK_ERR_BAD_ARG;
  *out = nullptr;
  int rc = validate_config(*cfg);
  if (rc) return rc;
  if (!w->embed || !w->lm_head || !w->final_norm || !aligned16(w->embed) || !aligned16(w->lm_head) ||
      !aligned16(w->final_norm))
    return MK_ERR_BAD_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev < 1) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  mk_handle* h = new (std::nothrow) mk_handle();
  if (!h) return MK_ERR_OOM;
  h->cfg = *cfg;
  mk_config& c = h->cfg;
  if (c.max_attn_items == 0) c.max_attn_items = 8192;
  if (c.timeout_ms == 0) c.timeout_ms = 2000;
  cudaGetDevice(&h->device);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, h->device) != cudaSuccess) { delete h; return MK_ERR_CUDA; }
  int coop = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device);
  if (!coop || prop.sharedMemPerBlockOptin < step_smem_bytes()) { delete h; return MK_ERR_CUDA; }
  // the kernel's warpgroups re-split the block's registers; the split adds up
  // only for the launch allocation it was designed for
  if (step_kernel_regs() != kLaunchRegs) { delete h; return MK_ERR_CUDA; }
  h->n_sm = prop.multiProcessorCount;
  if (c.sm_cap > 0) h->n_sm = std::min(h->n_sm, c.sm_cap);

  const int L = c.n_layers, H = c.hidden, hq = c.n_q_heads, hkv = c.n_kv_heads, d = c.head_dim;
  const int E = c.n_experts, K = c.top_k, I = c.moe_inter, Bm = c.max_batch;
  const int grp = hq / hkv;
  Params& p = h->base;
  memset(&p, 0, sizeof(p));
  p.L = L; p.H = H; p.hq = hq; p.hkv = hkv; p.d = d; p.E = E; p.topk = K; p.I = I;
  p.V = c.vocab; p.P = c.page_size; p.grp = grp; p.qkv_rows = (hq + 2 * hkv) * d;
  p.max_pages = c.max_pages_per_seq; p.num_pages = c.num_kv_pages; p.Bmax = Bm;
  p.n_sm = h->n_sm;
  p.rms_eps = c.rms_eps;
  p.attn_scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
  p.embed = (const uint16_t*)w->embed;
  p.lm_head = (const uint16_t*)w->lm_head;
  p.final_norm = (const uint16_t*)w->final_norm;
  p.timeout_ns = (unsigned long long)c.timeout_ms * 1000000ull;
  p.bl = bar_layout(Bm);
  p.bar_per_layer = p.bl.per_layer;

#define TRY(x) do { int _r = (x); if (_r) { mk_destroy(h); return _r; } } while (0)
  TRY(upload_ptrs(h, (const void* const*)w->attn_norm, L, (const void* const**)&p.attn_norm));
  TRY(upload_ptrs(h, (const void* const*)w->w_qkv, L, (const void* const**)&p.w_qkv));
  TRY(upload_ptrs(h, (const void* const*)w->w_o, L, (const void* const**)&p.w_o));
  TRY(upload_ptrs(h, (const void* const*)w->w_router, L, (const void* const**)&p.w_router));
  TRY(upload_ptrs(h, (const void* const*)w->w_gate, L, (const void* const**)&p.w_gate));
  TRY(upload_ptrs(h, (const void* const*)w->w_up, L, (const void* const**)&p.w_up));
  TRY(upload_ptrs(h, (const void* const*)w->w_down, L, (const void* const**)&p.w_down));
  p.fp8 = c.expert_format == MK_EXPERTS_FP8_E4M3;
  if (p.fp8) {
    if (!w->s_gate || !w->s_up || !w->s_down) { mk_destroy(h); return MK_ERR_BAD_ARG; }
    TRY(upload_ptrs(h, (const void* const*)w->s_gate, L, (const void* const**)&p.s_gate));
    TRY(upload_ptrs(h, (const void* const*)w->s_up, L, (const void* const**)&p.s_up));
    TRY(upload_ptrs(h, (const void* const*)w->s_down, L, (const void* const**)&p.s_down));
  }
  TRY(upload_ptrs(h, (const void* const*)w->k_pool, L, (const void* const**)&p.k_pool));
  TRY(upload_ptrs(h, (const void* const*)w->v_pool, L, (const void* const**)&p.v_pool));
  TRY(make_kv_maps(h, w, &p.kv_maps));
  TRY(make_weight_maps(h, w, &p.w_maps));
  TRY(make_down_maps(h, w, &p.wd_maps));

  const size_t Ls = (size_t)L, Bs = (size_t)Bm, Ns = (size_t)h->n_sm;
  p.max_attn_items = c.max_attn_items;
  TRY(dalloc(h, &p.hloc, Ns * Bs * H));
  TRY(dalloc(h, &p.xloc, Ns * Bs * H));
  TRY(dalloc(h, &p.hdbg, (Ls + 1) * Bs * H));
  TRY(dalloc(h, &p.xdbg, (Ls + 1) * Bs * H));
  TRY(dalloc(h, &p.qkv, Ls * Bs * p.qkv_rows));
  TRY(dalloc(h, &p.rlog, Ls * Bs * E));
  TRY(dalloc(h, &p.ridx, Ls * Bs * K));
  TRY(dalloc(h, &p.rw, Ls * Bs * K));
  TRY(dalloc(h, &p.attn_part, (size_t)c.max_attn_items * hkv * grp * d));
  TRY(dalloc(h, &p.attn_ml, (size_t)c.max_attn_items * hkv * grp * 2));
  TRY(dalloc(h, &p.attn_out, Ls * Bs * hq * d));
  TRY(dalloc(h, &p.abuf, Ls * Bs * K * I));
  TRY(dalloc(h, &p.oproj, Ls * Bs * H));
  TRY(dalloc(h, &p.moe, Ls * Bs * H));
  TRY(dalloc(h, &p.mpart, (size_t)K * (I / 8) * H));
  TRY(dalloc(h, &p.mdown, Bs * K * H));
  TRY(make_moe_map(h, p.mpart, &p.mp_map));
  TRY(make_down_blocks(h, w, &p.wd_blk));
  h->bar_words = kErrWords + (size_t)L * p.bl.per_layer;
  TRY(dalloc(h, &h->d_bars, h->bar_words));
  p.err = h->d_bars;
  p.bars = h->d_bars + kErrWords;
  TRY(dalloc(h, &h->d_tokens, Bs));
  TRY(dalloc(h, &h->d_pos, Bs));
  TRY(dalloc(h, &h->d_pt, Bs * c.max_pages_per_seq));
  TRY(dalloc(h, &h->d_rope, Bs * (d / 2) * 2));
  TRY(dalloc(h, &h->d_items, (size_t)c.max_attn_items * 8));
  TRY(dalloc(h, &h->d_smoff, Ns + 1));
  TRY(dalloc(h, &h->d_meta, Bs * 2));
  if (c.trace_records > 0) {
    h->trace_words = (size_t)h->n_sm * c.trace_records * kTraceWords;
    TRY(dalloc(h, &h->d_trace, h->trace_words));
    p.trace = h->d_trace;
    p.trace_cap = c.trace_records;
    h->dbg_words = (size_t)L * kDbgRouteWords + Bs * c.max_pages_per_seq + Bs;
    TRY(dalloc(h, &h->d_dbg, h->dbg_words));
    p.dbg = h->d_dbg;
  }
  if (cudaMemset(h->d_bars, 0, h->bar_words * 4) != cudaSuccess) { mk_destroy(h); return MK_ERR_CUDA; }
  h->step_bytes_cap = step_upload_bytes(c, h->n_sm, Bm, c.max_attn_items);
  for (auto& s : h->stage) {
    if (cudaMallocHost(&s.host, h->step_bytes_cap) != cudaSuccess) { cudaGetLastError(); mk_destroy(h); return MK_ERR_OOM; }
    if (cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess) { mk_destroy(h); return MK_ERR_CUDA; }
  }
#undef TRY
  *out = h;
  return MK_OK;
}

int mk_schedule_step(mk_handle* h, int batch, const int32_t* seq_ids, const int32_t* tokens,
                     const int32_t* page_tables, const int32_t* seq_lens, void* stream) {
  (void)seq_ids;
  if (!h) return MK_ERR_BAD_ARG;
  const mk_config& c = h->cfg;
  h->scheduled = false;
  if (batch < 1 || batch > c.max_batch) return MK_ERR_BATCH_TOO_LARGE;
  if (!tokens || !page_tables || !seq_lens) return MK_ERR_BAD_ARG;
  const int P = c.page_size, MP = c.max_pages_per_seq, d = c.head_dim;
  long long total_keys = 0;
  for (int b = 0; b < batch; b++) {
    if (tokens[b] < 0 || tokens[b] >= c.vocab) return MK_ERR_BAD_ARG;
    if (seq_lens[b] < 0) return MK_ERR_BAD_ARG;
    if ((long long)seq_lens[b] + 1 > (long long)MP * P) return MK_ERR_BAD_PAGE;
    const int need = (seq_lens[b] + 1 + P - 1) / P;
    for (int i = 0; i < need; i++) {
      const int32_t pg = page_tables[(size_t)b * MP + i];
      if (pg < 0 || pg >= c.num_kv_pages) return MK_ERR_BAD_PAGE;
    }
    total_keys += seq_lens[b] + 1;
  }
  // select_schedule: the live contexts' pages cut into one run per SM
  const int na = attention_sms(c, h->n_sm, batch, seq_lens);
  const int S = split_kv(c, h->n_sm, na, batch, seq_lens, &h->items, &h->smoff, &h->meta);
  if (S < 0) return MK_ERR_BAD_CONFIG;
  const int n_items = (int)(h->items.size() / 8);

  DevPlan* plan = nullptr;
  int rc = ensure_plan(h, batch, na, &plan);
  if (rc) return rc;

  // stage the step state in pinned memory, then one upload per array
  Staging& st = h->stage[h->stage_idx];
  h->stage_idx ^= 1;
  if (st.pending) {
    cudaEventSynchronize(st.done);
    st.pending = false;
  }
  uint8_t* cur = st.host;
  int32_t* s_tok = (int32_t*)cur; cur += (size_t)batch * 4;
  int32_t* s_pos = (int32_t*)cur; cur += (size_t)batch * 4;
  int32_t* s_pt = (int32_t*)cur; cur += (size_t)batch * MP * 4;
  float* s_rope = (float*)cur; cur += (size_t)batch * (d / 2) * 2 * 4;
  int32_t* s_meta = (int32_t*)cur; cur += (size_t)batch * 2 * 4;
  int32_t* s_smoff = (int32_t*)cur; cur += (size_t)(h->n_sm + 1) * 4;
  int32_t* s_items = (int32_t*)cur;
  memcpy(s_tok, tokens, (size_t)batch * 4);
  memcpy(s_pos, seq_lens, (size_t)batch * 4);
  memcpy(s_pt, page_tables, (size_t)batch * MP * 4);
  for (int b = 0; b < batch; b++) {
    const double pos = (double)seq_lens[b];
    for (int i = 0; i < d / 2; i++) {
      const double ang = pos * pow(c.rope_theta, -2.0 * i / (double)d);
      s_rope[((size_t)b * (d / 2) + i) * 2 + 0] = (float)cos(ang);
      s_rope[((size_t)b * (d / 2) + i) * 2 + 1] = (float)sin(ang);
    }
  }
  memcpy(s_meta, h->meta.data(), (size_t)batch * 2 * 4);
  memcpy(s_smoff, h->smoff.data(), (size_t)(h->n_sm + 1) * 4);
  memcpy(s_items, h->items.data(), (size_t)n_items * 8 * 4);
  cudaStream_t sm = (cudaStream_t)stream;
  bool ok = cudaMemcpyAsync(h->d_tokens, s_tok, (size_t)batch * 4, cudaMemcpyHostToDevice, sm) == cudaSuccess &&
            cudaMemcpyAsync(h->d_pos, s_pos, (size_t)batch * 4, cudaMemcpyHostToDevice, sm) == cudaSuccess &&
            cudaMemcpyAsync(h->d_pt, s_pt, (size_t)batch * MP * 4, cudaMemcpyHostToDevice, sm) == cudaSuccess &&
            cudaMemcpyAsync(h->d_rope, s_rope, (size_t)batch * (d / 2) * 2 * 4, cudaMemcpyHostToDevice, sm) == cudaSuccess &&
            cudaMemcpyAsync(h->d_meta, s_meta, (size_t)batch * 2 * 4, cudaMemcpyHostToDevice, sm) == cudaSuccess &&
            cudaMemcpyAsync(h->d_smoff, s_smoff, (size_t)(h->n_sm + 1) * 4, cudaMemcpyHostToDevice, sm) == cudaSuccess &&
            cudaMemcpyAsync(h->d_items, s_items, (size_t)n_items * 8 * 4, cudaMemcpyHostToDevice, sm) == cudaSuccess &&
            cudaEventRecord(st.done, sm) == cudaSuccess;
  if (!ok) return MK_ERR_CUDA;
  st.pending = true;
  h->scheduled = true;
  h->batch = batch;
  h->n_items = n_items;
  h->split = S;
  h->n_attn = na;
  return MK_OK;
}

}  // extern "C"

namespace {

// kernel parameters of the scheduled step
Params step_params(const mk_handle* h, const DevPlan& plan, float* logits) {
  Params p = h->base;
  p.B = h->batch;
  p.n_attn_items = h->n_items;
  p.attn_meta = h->d_meta;
  p.attn_sm_off = h->d_smoff;
  p.tokens = h->d_tokens;
  p.pos = h->d_pos;
  p.page_tables = h->d_pt;
  p.rope = h->d_rope;
  p.attn_items = h->d_items;
  p.logits = logits;
  p.tasks = plan.tasks;
  p.task_off = plan.off;
  p.n_comb_sms = plan.n_comb_sms;
  p.n_up_sms = plan.n_up_sms;
  p.n_down_sms = plan.n_down_sms;
  p.n_rtr_sms = plan.n_rtr_sms;
  // expert-branch stage depth: measured on the 30B/3.3B model at 8K context
  // (112 expert SMs against 40 attention SMs: 3 stages in flight gave the
  // shortest step) and at 256K (12 expert SMs: the full ring)
  const int n_moe = h->n_attn < h->n_sm ? h->n_sm - h->n_attn : 0;
  p.moe_depth = h->cfg.moe_stage_depth > 0 ? h->cfg.moe_stage_depth : (n_moe > h->n_attn ? 3 : kStages);
  // expert tiles: claimed, 128 rows, from 4 tokens up, unless the config
  // fixes them (measured on the 30B/3.3B model: at batch 16 128-row tiles
  // ahead of 64, 192 and 256 and of static shares by 14 % at the same role
  // split; at batch 4 ahead of static shares by 4 %; at batch 2 behind by 5 %,
  // its few tiles cost about the same)
  p.claim_rows = h->cfg.moe_claim_rows > 0 ? h->cfg.moe_claim_rows
                 : h->cfg.moe_claim_rows == 0 && h->batch >= 4 ? 128 : 0;
  return p;
}

}  // namespace

extern "C" {

int mk_decode_step(mk_handle* h, float* logits, void* stream) {
  if (!h || !logits) return MK_ERR_BAD_ARG;
  if (!h->scheduled) return MK_ERR_NOT_SCHEDULED;
  DevPlan* plan = nullptr;
  int rc = ensure_plan(h, h->batch, h->n_attn, &plan);
  if (rc) return rc;
  cudaStream_t sm = (cudaStream_t)stream;
  if (cudaMemsetAsync(h->d_bars, 0, h->bar_words * 4, sm) != cudaSuccess) return MK_ERR_CUDA;
  if (h->d_trace && (cudaMemsetAsync(h->d_trace, 0xff, h->trace_words * 4, sm) != cudaSuccess ||
                     cudaMemsetAsync(h->d_dbg, 0xff, h->dbg_words * 4, sm) != cudaSuccess))
    return MK_ERR_CUDA;
  const Params p = step_params(h, *plan, logits);
  if (launch_step(p, h->n_sm, sm) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  h->last_batch = h->batch;
  return MK_OK;
}

int mk_decode_step_static(mk_handle* h, float* logits, void* stream) {
  if (!h || !logits) return MK_ERR_BAD_ARG;
  if (h->bar_words > (size_t)MK_STATIC_COUNTER_WORDS) return MK_ERR_BAD_CONFIG;
  if (!h->scheduled) return MK_ERR_NOT_SCHEDULED;
  auto it = h->plans.find(plan_key(h->batch, h->n_attn));
  if (it == h->plans.end()) return MK_ERR_NOT_SCHEDULED;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) {
    cudaGetLastError();
    return MK_ERR_BAD_ARG;
  }
  uint32_t* ctr = nullptr;
  int rc = static_counters(dev, &ctr);
  if (rc) return rc;
  cudaStream_t sm = (cudaStream_t)stream;
  if (cudaMemsetAsync(ctr, 0, h->bar_words * 4, sm) != cudaSuccess) return MK_ERR_CUDA;
  if (h->d_trace && (cudaMemsetAsync(h->d_trace, 0xff, h->trace_words * 4, sm) != cudaSuccess ||
                     cudaMemsetAsync(h->d_dbg, 0xff, h->dbg_words * 4, sm) != cudaSuccess))
    return MK_ERR_CUDA;
  Params p = step_params(h, it->second, logits);
  p.err = ctr;
  p.bars = ctr + kErrWords;
  if (launch_step(p, h->n_sm, sm) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  if (cudaMemcpyAsync(h->d_bars, ctr, kErrWords * 4, cudaMemcpyDeviceToDevice, sm) != cudaSuccess)
    return MK_ERR_CUDA;
  h->last_batch = h->batch;
  return MK_OK;
}

int mk_step_status(mk_handle* h, mk_error* out) {
  if (!h) return MK_ERR_BAD_ARG;
  uint32_t e[kErrWords];
  if (cudaMemcpy(e, h->d_bars, sizeof(e), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  int code = MK_OK;
  if (e[E_CODE] == DEV_TIMEOUT || e[E_CODE] == DEV_SMEM_TIMEOUT) code = MK_ERR_TIMEOUT;
  else if (e[E_CODE] != 0) code = MK_ERR_DEVICE;
  if (out) {
    out->code = code;
    out->sm = (int)e[E_SM];
    out->task = (int)e[E_TASK];
    out->op = (int)e[E_OP];
    out->barrier = (int)e[E_BAR];
    out->value = e[E_VAL];
    out->target = e[E_TGT];
  }
  return code;
}

int mk_get_routing(mk_handle* h, int32_t* idx, float* w) {
  if (!h) return MK_ERR_BAD_ARG;
  if (h->last_batch < 1) return MK_ERR_NOT_SCHEDULED;
  const mk_config& c = h->cfg;
  const int B = h->last_batch, K = c.top_k, Bm = c.max_batch;
  std::vector<int32_t> ti((size_t)c.n_layers * Bm * K);
  std::vector<float> tw((size_t)c.n_layers * Bm * K);
  if (cudaMemcpy(ti.data(), h->base.ridx, ti.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(tw.data(), h->base.rw, tw.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  for (int l = 0; l < c.n_layers; l++)
    for (int b = 0; b < B; b++)
      for (int j = 0; j < K; j++) {
        const size_t src = ((size_t)l * Bm + b) * K + j, dst = ((size_t)l * B + b) * K + j;
        if (idx) idx[dst] = ti[src];
        if (w) w[dst] = tw[src];
      }
  return MK_OK;
}

int mk_read_scratch(mk_handle* h, int which, int layer, void* dst, size_t bytes, size_t* size_out) {
  if (!h) return MK_ERR_BAD_ARG;
  const mk_config& c = h->cfg;
  const Params& p = h->base;
  const int B = h->last_batch > 0 ? h->last_batch : 1, Bm = c.max_batch, L = c.n_layers;
  const int H = c.hidden;
  const int maxl = (which == MK_SCRATCH_H || which == MK_SCRATCH_X) ? L : L - 1;
  if (layer < 0 || layer > maxl) return MK_ERR_BAD_ARG;
  const float* base = nullptr;
  size_t row = 0;   // floats per sequence
  switch (which) {
    case MK_SCRATCH_H: row = H; base = p.hdbg + (size_t)layer * Bm * H; break;
    case MK_SCRATCH_X: row = H; base = p.xdbg + (size_t)layer * Bm * H; break;
    case MK_SCRATCH_QKV: row = p.qkv_rows; base = p.qkv + (size_t)layer * Bm * p.qkv_rows; break;
    case MK_SCRATCH_ATTN: row = (size_t)p.hq * p.d; base = p.attn_out + (size_t)layer * Bm * row; break;
    case MK_SCRATCH_ROUTER: row = c.n_experts; base = p.rlog + (size_t)layer * Bm * row; break;
    case MK_SCRATCH_OPROJ: row = H; base = p.oproj + (size_t)layer * Bm * H; break;
    case MK_SCRATCH_MOE: row = H; base = p.moe + (size_t)layer * Bm * H; break;
    default: return MK_ERR_BAD_ARG;
  }
  const size_t full = row * 4 * (size_t)B;
  if (size_out) *size_out = full;
  if (dst && cudaMemcpy(dst, base, std::min(bytes, full), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  return MK_OK;
}

int mk_read_trace(mk_handle* h, void* dst, size_t bytes, size_t* size_out) {
  if (!h) return MK_ERR_BAD_ARG;
  const size_t full = h->trace_words * 4;
  if (size_out) *size_out = full;
  if (dst && full && cudaMemcpy(dst, h->d_trace, std::min(bytes, full), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  return MK_OK;
}

int mk_read_debug(mk_handle* h, int which, void* dst, size_t bytes, size_t* size_out) {
  if (!h) return MK_ERR_BAD_ARG;
  if (!h->d_dbg) return MK_ERR_BAD_CONFIG;
  if (h->last_batch < 1) return MK_ERR_NOT_SCHEDULED;
  const mk_config& c = h->cfg;
  const size_t route = (size_t)c.n_layers * kDbgRouteWords, pages = (size_t)c.max_batch * c.max_pages_per_seq;
  size_t off = 0, words = 0;
  switch (which) {
    case MK_DEBUG_ROUTE_GROUPS: off = 0; words = route; break;
    case MK_DEBUG_PAGE_GATHER: off = route; words = (size_t)h->last_batch * c.max_pages_per_seq; break;
    case MK_DEBUG_NEW_SLOT: off = route + pages; words = (size_t)h->last_batch; break;
    default: return MK_ERR_BAD_ARG;
  }
  if (size_out) *size_out = words * 4;
  if (dst && cudaMemcpy(dst, h->d_dbg + off, std::min(bytes, words * 4), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  return MK_OK;
}

int mk_debug_bump_wait(mk_handle* h, int layer, int delta) {
  if (!h || layer < 0 || layer > h->cfg.n_layers) return MK_ERR_BAD_ARG;
  cudaDeviceSynchronize();
  h->bump_layer = delta ? layer : -1;
  h->bump = delta;
  free_plans(h);
  return MK_OK;
}

}  // extern "C"

namespace mk {
// for the decode service (same library): the step's device token buffer and
// the handle's config and device
int32_t* handle_tokens(mk_handle* h) { return h->d_tokens; }
const mk_config* handle_config(const mk_handle* h) { return &h->cfg; }
int handle_device(const mk_handle* h) { return h->device; }
}  // namespace mk

extern "C" {

size_t mk_device_bytes(const mk_handle* h) { return h ? h->dev_bytes : 0; }
int mk_num_sms(const mk_handle* h) { return h ? h->n_sm : 0; }
size_t mk_step_upload_bytes(const mk_handle* h, int batch) {
  if (!h) return 0;
  return step_upload_bytes(h->cfg, h->n_sm, batch, h->scheduled ? h->n_items : 0);
}

}  // extern "C"
