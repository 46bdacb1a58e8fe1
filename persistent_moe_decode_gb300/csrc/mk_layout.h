// Layout contract between the host scheduler and the persistent kernel:
// opcodes, the 32-word task descriptor, counter indices and targets, stage
// geometry and the kernel's parameter block.
//
// "Inside the megakernel serving engine for North Mini Code", §The task
// descriptor: a task is 32 int32 words, word 0 the opcode, the rest naming the
// layer and the work.  §Barriers: counters are plain integers in global
// memory, zeroed before every step.
//
// GB300 task structure: every SM takes an equal share of every phase of a
// layer (one task per phase per SM), so that all 152 SMs stream weights for
// the whole layer and no phase waits on a few stragglers.  Per SM and layer:
//   P1      local residual add + RMSNorm, then its rows of [W_router; W_qkv]
//   ROUTE   top-k of every token and the per-expert grouping (shared memory)
//   ATTN    its split-KV attention items (pages of one sequence, all KV heads)
//   UP      its share of the routed experts' (gate, up) row pairs
//   COMBINE its (sequence, query head) merges of the split-KV partials
//   DOWN    its hidden rows of every routed expert's down projection, weighted
//           by the routing: the expert branch's share of the residual update
//   OUT     its hidden rows of the O-proj: the attention branch's share
// With one token each UP slice (whole groups of 8 intermediate columns) also
// multiplies its columns of the down projection, giving one partial hidden
// vector per group, and DOWN adds the groups' partials of its rows in group
// order.
// and after the last layer FINAL: local final norm and its LM-head rows.  The
// next layer adds both shares to the residual.
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
  OP_P1 = 1,
  OP_ROUTE = 2,
  OP_ATTN = 3,
  OP_UP = 4,
  OP_COMBINE = 5,
  OP_OUT = 6,
  OP_FINAL = 7,
  OP_DOWN = 8
};

// descriptor words (host-built, read by the producer warp)
enum : int {
  F_OP = 0, F_LAYER = 1,
  F_A0 = 2, F_A1 = 3,      // op-specific range: P1 rows of W_router, COMBINE
                           // units, OUT and DOWN hidden rows, FINAL vocabulary rows;
                           // UP: slice index and slice count
  F_SEQ = 4,               // position in the SM's list (error reports)
  F_BUMP = 5,              // P1 / FINAL: added to the wait target (testing aid)
  F_B0 = 6, F_B1 = 7       // P1: rows of W_qkv (F_A0 / F_A1: rows of W_router)
};

// persistent block shape: two consumer warpgroups (8 warps) + one producer
// warpgroup (one active warp).  At launch every thread holds kLaunchRegs
// registers; the producer warpgroup gives some back (setmaxnreg) and the
// consumers take them: 128 * kProducerRegs + 256 * kConsumerRegs must equal
// 384 * kLaunchRegs exactly.
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr int kProducerRegs = 72;
constexpr int kConsumerRegs = 216;
static_assert(128 * kProducerRegs + 256 * kConsumerRegs == kThreads * kLaunchRegs,
              "register split must add up to the launch allocation");
constexpr int kStages = 5;              // weight / KV stage ring depth
constexpr int kXsFloats = 8192;         // one-token activations staged in shared memory
constexpr int kStageBytes = 32768;      // one stage: whole weight rows or one KV page group
constexpr int kTaskSlots = 8;           // resolved-task ring depth
constexpr int kMaxBatch = 16;
constexpr int kTraceWords = 16;         // words per timeline record
constexpr int kPartFloats = 2048;       // one of the two GEMV partial-sum buffers
constexpr int kTokPass = 8;             // tokens per GEMV pass (activations in registers)
constexpr int kMaxActive = 128;         // routed experts of one step (B * k <= 128)
constexpr int kDbgRouteWords = 1 + kMaxActive + (kMaxActive + 1) + kMaxActive;   // 386

// whole rows of a [rows][K] BF16 matrix that one stage carries
MK_HD inline int rows_per_stage(int K) {
  const int r = kStageBytes / (2 * K);
  return r > 0 ? r : 1;
}

// One token: weight rows of 2048 or 4096 columns are multiplied on the tensor
// cores.  A stage of such rows arrives as ONE 3-D tensor copy of the matrix
// viewed as [K / 64 column blocks][rows][64 columns] (box: all column blocks x
// R = 32768 / (2 K) rows x 64 columns) with 128-byte swizzle: column block cb
// of row r is the 128-byte line cb R + r of the stage, its 16-byte chunk c
// stored at chunk c ^ (line & 7), so the eight rows an ldmatrix reads at one
// column fall in distinct banks.  Row shares of such matrices are multiples
// of 8 rows where the host chooses them, so a stage copies no row it does not
// use.
MK_HD inline bool rotated_rows(int K) { return K == 2048 || K == 4096; }
constexpr int kMmaRows = 128;           // rows of one tensor-core GEMV chunk (one partial buffer)
// Several tokens: rows of 2048 columns with at most 8 tokens, or of 4096
// columns with at most 4 (dense rows, an expert's gate / up rows) go to the
// tensor cores through the same maps; an expert's down rows (I columns, I a
// multiple of 128 up to 1024) through maps of W_down viewed as [E H rows][I]
// with boxes of 16 rows x all of I, 128-byte swizzle (row r of column block
// cb is the 128-byte line 16 cb + r).
MK_HD inline bool mma_multi_rows(int K, int nt) {
  return nt >= 1 && ((K == 2048 && nt <= 8) || (K == 4096 && nt <= 4));
}
MK_HD inline bool mma_multi_down(int K) { return K % 128 == 0 && K <= 1024; }
constexpr int kDownBoxRows = 16;
// tensor maps of the weight matrices bound for the tensor cores, per layer (W_MAP_* + 5 l), then the LM head
enum : int { W_MAP_ROUTER = 0, W_MAP_QKV = 1, W_MAP_O = 2, W_MAP_GATE = 3, W_MAP_UP = 4, W_MAPS_PER_LAYER = 5 };

// GEMV contraction segments: 256 columns (32 lanes x 8), or all of K below that
MK_HD inline int gemv_nseg(int K) { return K < 256 ? 1 : K / 256; }

// rows of one GEMV chunk (one fixed-order reduction): bounded by the partial
// buffer, rows * segments * tokens <= kPartFloats
MK_HD inline int gemv_chunk_rows(int K, int nt) {
  const int r = kPartFloats / (gemv_nseg(K) * (nt > 0 ? nt : 1));
  return r > 512 ? 512 : r;
}

// Counter block of one layer.  Index = layer * per_layer + offset.
struct BarLayout {
  int per_layer;
  int p1;      // P1 tasks done                                   (target n_sm)
  int up;      // UP tasks done                                   (target n_up_sms)
  int comb;    // COMBINE tasks done                              (target n_comb_sms)
  int out;     // OUT tasks done, and one-token DOWN tasks        (target n_sm [+ n_down_sms])
  int rtr;     // P1 tasks holding router rows done               (target n_rtr_sms)
  int down;    // several tokens: DOWN tasks done                 (target n_down_sms)
  int items;   // + b: split-KV items of sequence b done          (target: its split count)
  int claim_up;    // several tokens, claimed tiles: next UP tile of the layer (not waited on)
  int claim_down;  // several tokens, claimed tiles: next DOWN tile of the layer
};

inline BarLayout bar_layout(int max_batch) {
  BarLayout b;
  b.p1 = 0;
  b.up = 1;
  b.comb = 2;
  b.out = 3;
  b.rtr = 4;
  b.down = 5;
  b.items = 6;
  b.claim_up = 6 + max_batch;
  b.claim_down = 7 + max_batch;
  b.per_layer = (8 + max_batch + 31) & ~31;
  return b;
}

// device error word layout (mirrors mk_error)
enum : int { E_CODE = 0, E_SM = 1, E_TASK = 2, E_OP = 3, E_BAR = 4, E_VAL = 5, E_TGT = 6 };
enum : uint32_t { DEV_TIMEOUT = 1, DEV_BAD_PAGE = 2, DEV_BAD_ITEM = 3, DEV_BAD_OP = 4,
                  DEV_SMEM_TIMEOUT = 5 };

// attention item: 8 int32 words (one sequence, all KV heads, keys [t0, t1))
enum : int { AI_B = 0, AI_S = 1, AI_NSPLIT = 2, AI_T0 = 3, AI_T1 = 4, AI_BASE = 5, AI_POS = 6 };

struct Params {
  // model
  int L, H, hq, hkv, d, E, topk, I, V, P, grp, qkv_rows;
  int max_pages, num_pages, Bmax, n_sm;
  int n_comb_sms, n_up_sms;    // SMs that signal the COMBINE / UP counters of a layer
  int n_down_sms, n_rtr_sms;   // SMs with a DOWN task / with router rows in their P1 share
  int moe_depth;               // one token: stages an SM without attention items keeps in flight
  int claim_rows;              // several tokens: 0 = static expert shares; > 0 = the expert
                               // branch claims tiles of this many rows from per-layer counters
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
  // 8-bit experts (E4M3): w_gate / w_up / w_down hold bytes (same layouts),
  // weight = scale[row] * e4m3(byte); fp32 per-row scales [E][I], [E][I], [E][H]
  int fp8;
  const float* const* s_gate;
  const float* const* s_up;
  const float* const* s_down;
  const uint16_t* wd_blk;      // w_down re-laid out as [L][E][I / 8][H][8]: each 8-column group
                               // of an expert one contiguous [H][8] block (one token: the
                               // UP pieces' column slices stream as whole blocks)
  const uint8_t* mp_map;       // tensor map of mpart: 2-D [groups][H] fp32, boxes 24 x 256
  const uint8_t* wd_maps;      // several tokens: [L] tensor maps of W_down (16-row boxes;
                               // nullptr when not used)
  const uint8_t* w_maps;       // rows of 2048 / 4096 columns: [5 L + 1] tensor maps
                               // (W_MAP_*; the last the LM head), 3-D views described above
                               // (nullptr when the model's rows take the other GEMV path)
  const uint8_t* kv_maps;      // [L][2] tensor maps (128 bytes each) of the K and V pools:
                               // 2-D [rows = pages * hkv * page_size][d], boxes of
                               // 64 dims x (hkv * page_size) rows, 128-byte swizzle
  // this step
  int B;
  int n_attn_items;
  const int32_t* tokens;       // [B]
  const int32_t* pos;          // [B] position of the new token (= cached length)
  const int32_t* page_tables;  // [B][max_pages]
  const float* rope;           // [B][d/2][2] cos, sin
  const int32_t* attn_items;   // [n_attn_items][8]
  const int32_t* attn_sm_off;  // [n_sm + 1] items of SM s: [off[s], off[s+1])
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
  int32_t* dbg;        // with the timeline: integer results for exact checks (nullptr: off)
                       //   [L][kDbgRouteWords] block 0's grouping of each layer's routing:
                       //     n_act, act[128], off[129], ent[128];
                       //   then [Bmax][max_pages] the physical pages layer 0 streamed;
                       //   then [Bmax] the cache slot (page * P + row) of each new token
  // scratch; per-layer strides use Bmax; activations are fp32
  float* hloc;       // [n_sm][Bmax][H]  each SM's own copy of the residual stream
  float* xloc;       // [n_sm][Bmax][H]  each SM's own normalised layer input
  float* hdbg;       // [L+1][Bmax][H]   residual entering each layer (SM 0's copy)
  float* xdbg;       // [L+1][Bmax][H]   normalised input of each layer (SM 0's copy)
  float* qkv;        // [L][Bmax][qkv_rows] q, k, v before RoPE
  float* rlog;       // [L][Bmax][E]
  int32_t* ridx;     // [L][Bmax][k]     routing written by SM 0
  float* rw;         // [L][Bmax][k]
  float* attn_part;  // [max_attn_items][hkv][grp][d] unnormalised split outputs
  float* attn_ml;    // [max_attn_items][hkv][grp][2] (max, sum) in the log2 domain
  int max_attn_items;
  float* attn_out;   // [L][Bmax][hq d]
  float* abuf;       // [L][Bmax * k][I] expert hidden, by grouped slot
  float* oproj;      // [L][Bmax][H] O-proj output
  float* moe;        // [L][Bmax][H] weighted sum of the routed experts' outputs
  float* mpart;      // one token: [k * I / 8][H] the down projection of each 8-column
                     // group of the routed experts' hidden vectors, weighted
  float* mdown;      // several tokens: [Bmax * k][H] the weighted down projection of each
                     // (token, pick) entry, summed over the picks by OUT
};

}  // namespace mk
