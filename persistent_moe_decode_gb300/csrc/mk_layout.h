// Layout contract between the host scheduler and the persistent kernel:
// opcodes, the 32-word task descriptor, counter indices and targets, tile
// geometry and the kernel's parameter block.
//
// "Inside the megakernel serving engine for North Mini Code", §The task
// descriptor: a task is 32 int32 words, word 0 the opcode, the rest naming the
// layer, the output tile, the counter to wait on with its target count and the
// counter to signal.  §Barriers: counters are plain integers in global memory,
// zeroed before every step.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define MK_HD __host__ __device__
#else
#define MK_HD
#endif

namespace mk {

constexpr int kDescWords = 32;

enum Op : int32_t {
  OP_END = 0,
  OP_NORM = 1,       // fused residual add + RMSNorm of one layer (or the final norm)
  OP_QKV = 2,        // QKV GEMV tile with RoPE in the epilogue, appends K/V
  OP_ROUTER = 3,     // router GEMV tile; the last tile runs top-k + route setup
  OP_ATTN = 4,       // claimer on the split-KV attention queue
  OP_MOE_UP = 5,     // claimer on the expert gate/up queue (SiLU * up epilogue)
  OP_MOE_DOWN = 6,   // claimer on the expert down queue (routing weight epilogue)
  OP_OPROJ = 7,      // O-proj tile (full contraction, or one KV-head group on the wide path)
  OP_LMHEAD = 8,     // LM-head GEMV tile
  OP_COMBINE = 9     // merge the split-KV partials of one (sequence, KV head)
};

// descriptor words (host-built, read by the producer warp)
enum : int {
  F_OP = 0, F_LAYER = 1, F_TILE = 2,
  F_W0 = 3, F_T0 = 4,      // consumer-side wait: counter index, target (-1: none)
  F_W1 = 5, F_T1 = 6,
  F_SIG = 7, F_INC = 8,    // counter signalled on completion, increment (-1: none)
  F_PW = 9, F_PT = 10,     // producer-side wait before loading (MoE claimers: routing)
  F_SEQ = 11,              // position in the flattened step order (error reports)
  F_ARG = 12               // op-specific argument (ATTN_COMBINE: tasks per KV group)
};

// Tile geometry.  Two GEMV paths share the task structure:
//  narrow (batch <= 8): CUDA-core FMA on whole contiguous weight rows, one bulk
//    copy of up to 32 KB per stage;
//  wide (batch 9..16): warp-level tensor-core MMA on 16-row stages padded for
//    conflict-free fragment loads.
constexpr int kRowsQKVHalf = 16;  // a QKV tile: 16 rows + their RoPE partners d/2 further
constexpr int kRowsRouter = 16;
constexpr int kRowsUp = 16;       // 16 gate rows + the same 16 up rows
constexpr int kRowsDownN = 64, kRowsDownW = 32;
constexpr int kRowsLMN = 64, kRowsLMW = 32;
constexpr int kRowsOProj = 32;    // narrow: full contraction; wide: one KV group's columns
constexpr int kNarrowMaxBatch = 8;

// persistent block shape: 8 consumer warps + 1 producer warp
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 6;              // weight / KV stage ring depth
constexpr int kStageData = 32768;       // narrow stages: up to 32 KB of whole rows
constexpr int kStageRows = 16;          // wide stages: 16 rows x up to 1024 columns, padded
constexpr int kStageKcMax = 1024;
constexpr int kStageBytes = kStageRows * (kStageKcMax * 2 + 64);   // 33,792
constexpr int kTaskSlots = 8;           // resolved-task ring depth
constexpr int kMaxBatch = 16;
constexpr int kTraceWords = 16;         // words per timeline record

// rows of a [rows][K] BF16 matrix that one narrow stage carries
MK_HD inline int narrow_rows_per_stage(int K) {
  int r = 1;
  while (r * 2 * 2 * K <= kStageData && r < 128) r *= 2;
  return r;
}

// Counter block of one layer.  Index = layer * per_layer + offset.
struct BarLayout {
  int per_layer;
  int x;          // norm done: x[l] ready                      (target 1)
  int qkv;        // + g: QKV tiles of KV group g done          (target (grp + 2) * d / 32)
  int route;      // routing + queues written                   (target 1)
  int up;         // + e: gate/up tiles of expert e done        (target I / kRowsUp)
  int items;      // + b: split-KV items of sequence b done     (target: its split count)
  int attn;       // combines done                              (target B * hkv * tasks per group)
  int o;          // O-proj tiles done                          (target: O-proj tile count)
  int moe;        // down tiles done, weighted by token count   (target B * k * H / rows)
  int tk_router;  // ticket: last router tile runs top-k
  int claim;      // + q: claim counters of the three queues
};

inline BarLayout bar_layout(int hkv, int n_experts, int max_batch) {
  BarLayout b;
  int o = 0;
  b.x = o; o += 1;
  b.qkv = o; o += hkv;
  b.route = o; o += 1;
  b.up = o; o += n_experts;
  b.items = o; o += max_batch;
  b.attn = o; o += 1;
  b.o = o; o += 1;
  b.moe = o; o += 1;
  b.tk_router = o; o += 1;
  b.claim = o; o += 3;
  b.per_layer = (o + 31) & ~31;
  return b;
}

enum : int { Q_ATTN = 0, Q_UP = 1, Q_DOWN = 2 };

// device error word layout (mirrors mk_error)
enum : int { E_CODE = 0, E_SM = 1, E_TASK = 2, E_OP = 3, E_BAR = 4, E_VAL = 5, E_TGT = 6 };
enum : uint32_t { DEV_TIMEOUT = 1, DEV_BAD_PAGE = 2, DEV_BAD_ITEM = 3, DEV_BAD_OP = 4,
                  DEV_SMEM_TIMEOUT = 5 };

// attention queue item: 8 int32 words (one sequence, all KV heads, keys [t0, t1))
enum : int { AI_B = 0, AI_S = 1, AI_NSPLIT = 2, AI_T0 = 3, AI_T1 = 4, AI_BASE = 5, AI_POS = 6 };

struct Params {
  // model
  int L, H, hq, hkv, d, E, topk, I, V, P, grp, qkv_rows;
  int max_pages, num_pages, Bmax;
  float rms_eps, attn_scale_log2;
  // caller weights (device pointers; per-layer arrays are device arrays of L pointers)
  const uint16_t* embed;
  const uint16_t* lm_head;
  const uint16_t* final_norm;
  const uint16_t* const* attn_norm;
  const uint16_t* const* w_qkv;
  const uint16_t* const* w_o;
  const uint16_t* const* w_router;
  const uint16_t* const* w_gate;
  const uint16_t* const* w_up;
  const uint16_t* const* w_down;
  uint16_t* const* k_pool;
  uint16_t* const* v_pool;
  // this step
  int B;
  int wide;                    // 1: tensor-core GEMV path (batch > 8)
  int n_attn_items;
  const int32_t* tokens;       // [B]
  const int32_t* pos;          // [B] position of the new token (= cached length)
  const int32_t* page_tables;  // [B][max_pages]
  const float* rope;           // [B][d/2][2] cos, sin
  const int32_t* attn_items;   // [n_attn_items][8]
  const int32_t* attn_meta;    // [B][2]: first item of the sequence, its split count
  float* logits;               // [B][V] caller buffer
  // task lists
  const int32_t* tasks;        // [n][32]
  const int32_t* task_off;     // [n_sm + 1]
  // counters
  uint32_t* bars;
  int bar_per_layer;
  BarLayout bl;
  uint32_t* err;
  unsigned long long timeout_ns;
  int32_t* trace;      // [n_sm][trace_cap][kTraceWords] task timeline (nullptr: off)
  int trace_cap;
  // scratch (per-layer strides use Bmax); activations are fp32
  float* h;          // [L+1][Bmax][H]  residual entering the layer
  float* x;          // [L+1][Bmax][H]  normalised layer input
  float* q;          // [L][Bmax][hq d] query after RoPE
  uint16_t* knew;    // [L][Bmax][hkv d] new key after RoPE (BF16, as cached)
  uint16_t* vnew;    // [L][Bmax][hkv d]
  float* rlog;       // [L][Bmax][E]
  int32_t* ridx;     // [L][Bmax][k]
  float* rw;         // [L][Bmax][k]
  int32_t* ecnt;     // [L][E]
  int32_t* eoff;     // [L][E + 1]
  int32_t* elist;    // [L][Bmax * k]  entry = b * k + j, grouped by expert, b ascending
  int32_t* upq;      // [L][max_up]   e << 16 | tile
  int32_t* downq;    // [L][max_down]
  int32_t* qmeta;    // [L][4]        n_up, n_down, n_active
  int max_up, max_down;
  float* attn_part;  // [max_attn_items][hkv][grp][d] unnormalised split outputs
  float* attn_ml;    // [max_attn_items][hkv][grp][2] (max, sum) in the log2 domain
  int max_attn_items;
  float* attn_out;   // [L][Bmax][hq d]
  float* oproj;      // [L][hkv][Bmax][H] (narrow path: slot 0 holds the full product)
  float* abuf;       // [L][Bmax * k][I]
  float* ybuf;       // [L][Bmax][k][H]
};

}  // namespace mk
