// The persistent decode-step kernel for GB300 (sm_103a).
//
// "Inside the megakernel serving engine for North Mini Code":
//  - §What is a Megakernel / Fig 2: one thread block per SM stays resident for
//    the whole step and walks a host-built per-SM task list in global memory;
//  - §The threadblock shape / Listing 1: one fixed block shape for every
//    opcode, a warp that fetches descriptors ahead of the workers, worker
//    warps that never use __syncthreads (their own barrier excludes the
//    fetcher), weight tiles prefetched before the cross-SM wait on activations;
//  - §Barriers / Listing 2: counters in global memory, spun on, released
//    after a fence, O(1) in fan-in and fan-out;
//  - §Tasks: ATTN_DECODE over a partial KV slice, ATTN_COMBINE merging the
//    partial results; the MoE tiles indexed by the routing result.
//
// GB300 design (not the pages' H100 one):
//  - block = 8 consumer warps + 1 producer warp (setmaxnreg 216 / 72).  The
//    producer resolves the task list (attention items, the routed experts'
//    rows) and streams every weight / KV byte HBM -> shared memory into a
//    5-stage ring of 32 KB stages guarded by mbarriers: 3-D tensor copies of
//    whole weight rows laid out with the 128-byte swizzle (rows of 2048 or
//    4096 columns; 1-D bulk copies where no tensor map applies), 2-D tensor
//    copies of KV pages, all with an evict-first L2 policy (each of those
//    bytes is read once a step; the kernel's code and activations stay in
//    L2).  The ring runs ahead across task boundaries, so a task that waits
//    for its activations already has its weights in flight.
//  - roles: per step the SMs split into an attention branch (P1, ATTN,
//    COMBINE, OUT) and an expert branch (P1, ROUTE, UP, DOWN, OUT) of the
//    parallel layer; every SM of a branch takes an equal share of each of
//    its waves (one token: an attention SM takes 4 times an expert SM's
//    O-proj rows), except the routed experts' rows with 4 tokens or more,
//    which the expert SMs claim as 128-row tiles from per-layer counters.
//  - GEMV: mma.sync m16n8k16 on the tensor cores, BF16 weights against the
//    fp32 activations split into BF16 high and low halves, fp32 accumulate;
//    the stage's rows and column parts on the M side, the tokens (and the
//    halves) on the N side; one token for rows of 2048 / 4096 columns, up to
//    8 / 4 tokens for several, and an expert's down rows for up to 16 tokens.
//    The other shapes (the 16-token dense rows among them) run on the CUDA
//    cores with fp32 FMAs, 256-column segments per warp.  Every reduction
//    adds the warps' partial sums in a fixed order.  One token: an UP piece
//    also multiplies its columns of the down projection, one fp32 partial per
//    8-column group, summed by the DOWN wave.
//  - 8-bit experts (OCP E4M3, one fp32 scale per output row; batch 1): the
//    activations as four E4M3 terms against the E4M3 weights in mma.sync
//    m16n8k32, fp32 accumulate, in kernel instances of their own.
//  - the residual add + RMSNorm is computed by every SM for itself at the
//    start of each layer (its own copy of the residual stream), so no SM waits
//    for a norm task; the routing likewise (one token: by each expert SM's
//    producer warp).
//  - attention: one item = one sequence, all KV heads, a run of 16-token
//    pages.  S^T = K Q^T and O^T += V^T P^T on the tensor cores (mma.sync,
//    BF16 high + low halves of the fp32 query and probabilities), online
//    softmax in fp32.  The item holding the new token applies RoPE to its
//    key, patches K/V into the staged page and writes them to the cache.
//  - bounded waits: counter waits have a %globaltimer limit; shared-memory
//    waits (the consumer warps' own barrier is an mbarrier, not bar.sync) a
//    poll count and the stop word.  On expiry the block records the error,
//    sets a global stop word that every other wait checks, drains its own
//    in-flight copies and returns.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "mk_layout.h"
#include "mk_ptx.cuh"

namespace mk {

// ------------------------------------------------------------ shared memory
// Routing of the current layer, computed by every SM for itself.
struct RouteTab {
  int32_t idx[kMaxBatch][8];        // top-k experts of each token, best first
  float w[kMaxBatch][8];            // renormalised weights
  int32_t n_act;                    // routed (active) experts
  int32_t act[kMaxActive];          // active experts, ascending
  int32_t off[kMaxActive + 1];      // first grouped slot of each active expert
  int32_t ent[kMaxActive];          // grouped slots: b * k + j, tokens ascending per expert
  int32_t ecount[256];              // scratch: tokens per expert
  int32_t eslot[256];               // scratch: active index of an expert
};

struct __align__(128) Smem {
  uint8_t stage[kStages][kStageBytes];
  float xs[kXsFloats];                      // one token: the GEMV's activations (x of the
                                            // layer, the attention output, the experts' hidden)
  float red[2 * kPartFloats];               // GEMV partial sums (two buffers) / attention
                                            // query fragments and merge / combine sums
  float spart[128][kConsumerWarps];         // one token, split GEMV: the warps' sums of each row
  float actp[64];                           // one token: weighted hidden values of an UP piece
  float nred[kConsumerWarps][kMaxBatch];    // norm / combine reductions
  float rinv[kMaxBatch];
  RouteTab rt;
  int32_t task[kTaskSlots][kDescWords];     // resolved task ring
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[kTaskSlots];
  uint64_t tempty[kTaskSlots];
  uint64_t cbar;                            // bounded barrier of the 8 consumer warps
  uint64_t route_bar;                       // consumers -> producer: routing of a layer ready
  uint32_t cstage[kConsumerWarps];          // per consumer warp: stages consumed
  uint32_t cphase[kConsumerWarps];          // per consumer warp: barrier phases passed
  uint32_t cchunk[kConsumerWarps];          // per consumer warp: GEMV chunks reduced
  int32_t seen_bar[kConsumerWarps];         // per consumer warp: last counter waited on...
  int32_t seen_tgt[kConsumerWarps];         // ...and the target it reached
  unsigned long long t_ready;               // timeline: when the task's inputs were ready
  unsigned long long t_mark[4];             // timeline: first stage, stages done, reduced
  unsigned long long t_swait;               // timeline: time warp 0 waited for stages
  volatile int32_t abort_flag;
  int32_t xq_layer;                         // 8-bit experts: layer whose x terms are staged (-1: none)
  float xq_s0, aq_s0;                       // first-term scales of the staged x / hidden terms
};
// the dynamic shared memory is rounded up to a 1024-byte boundary (the
// swizzled tensor copies of KV pages need it), hence the extra 1 KB
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory of one block exceeds the sm_103a limit");

// resolved task words (written by the producer into the task ring)
enum : int {
  R_OP = 0, R_LAYER, R_TASK, R_KIND, R_FLAGS, R_ROW0, R_NROWS, R_K, R_NT, R_NBLK, R_A, R_E,
  R_REL0, R_ITEM, R_B, R_TT0, R_TT1, R_POS, R_NST, R_U0, R_U1, R_BUMP, R_ROW1, R_NROWS1, R_NGRP,
  R_PCOMMIT, R_PISSUE    // timeline only: %globaltimer (low word) when the producer handed the
                         // task over and when it issued the task's first copy (0: none)
};
// GEMV chunk kinds; K_P1 (router rows, then QKV rows) and K_MRED (the sum of
// the experts' per-group partials of OUT's rows) are one-token forms, and a
// one-token K_UP chunk also multiplies its columns of the down projection.
// K_MSUM (several tokens) adds each token's k weighted expert outputs of
// OUT's rows; it streams nothing.
enum : int { K_ROUTER = 0, K_QKV = 1, K_UP = 2, K_OPROJ = 3, K_DOWN = 4, K_LM = 5, K_P1 = 6,
             K_MRED = 7, K_MSUM = 8 };
// rows of one single-token GEMV chunk (one result per row in a 2048-float buffer)
constexpr int kRowChunk = kPartFloats;
// rows of an [H][8] down-projection block per stage (2048 x 16 bytes = one stage)
constexpr int kDownRows = kStageBytes / 16;
// hidden rows per window of the one-token partial sums (a tensor box of
// kMredCols x 256 fp32; 16-byte multiple; a DOWN share of up to kMredCols - 3
// rows takes one window)
constexpr int kMredCols = 24;
// chunk flags: first chunk of its task (P1 / FINAL run the norm first), last
// chunk of its task (signals completion)
enum : int { FL_FIRST = 1, FL_LAST = 2, FL_RTR = 8 };   // FL_RTR: the chunk ends its router rows

// ---------------------------------------------------------------- errors
__device__ __forceinline__ bool stopped(const Params& p) {
  return *(volatile uint32_t*)&p.err[E_CODE] != 0;
}

__device__ __noinline__ void report(const Params& p, uint32_t code, int task, int op, int bar, uint32_t val,
                       uint32_t tgt) {
  if (atomicCAS(&p.err[E_CODE], 0u, code) == 0u) {
    p.err[E_SM] = blockIdx.x;
    p.err[E_TASK] = (uint32_t)task;
    p.err[E_OP] = (uint32_t)op;
    p.err[E_BAR] = (uint32_t)bar;
    p.err[E_VAL] = val;
    p.err[E_TGT] = tgt;
    __threadfence();
  }
}

// Bounded wait on a shared-memory mbarrier phase, called by a whole warp:
// false = give up.  The phases come from this block's own warps and copies,
// so the wait is bounded by a poll count (several seconds of polling: past
// any real wait and past the counter waits' time limit, so a block waiting
// here on a thread that waits for a counter learns of that counter's
// time-out first) and by the stop word (another block has reported an error),
// read every 4096 polls by all lanes at once (one broadcast load, so the warp
// decides together).  The block's exit path reports a time-out
// (DEV_SMEM_TIMEOUT) once.  Every wait site inlines this loop, so it is kept
// to a few instructions: code that runs once per layer is fetched anew each
// time, and a call from these paths saves many registers.
constexpr uint32_t kWaitPolls = 1u << 28;

__device__ __forceinline__ bool wait_phase_slow(const Params& p, uint64_t* bar, uint32_t parity) {
  bool done = false;
  for (uint32_t it = 1;; ++it) {
    done = done || mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((it & 4095u) == 0 && (it >= kWaitPolls || stopped(p))) return false;
  }
}

__device__ __forceinline__ bool wait_phase(const Params& p, uint64_t* bar, uint32_t parity) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  return wait_phase_slow(p, bar, parity);
}

// bounded spin on a global counter (Listing 2's wait, with a time limit)
__device__ __forceinline__ bool spin_counter(const Params& p, int bar, uint32_t target, int task, int op) {
  const uint32_t* c = p.bars + bar;
  uint32_t v = ld_acquire_u32(c);
  if (v >= target) return true;
  const unsigned long long t0 = gtime_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(20);
    v = ld_acquire_u32(c);
    if (v >= target) return true;
    if ((it & 15u) == 0) {
      if (stopped(p)) return false;
      if (gtime_ns() - t0 > p.timeout_ns) {
        report(p, DEV_TIMEOUT, task, op, bar, v, target);
        return false;
      }
    }
  }
}

__device__ __forceinline__ int bar_index(const Params& p, int layer, int off) {
  return layer * p.bar_per_layer + off;
}

// split-KV stage geometry: pages of all KV heads per stage (K half, V half)
__device__ __forceinline__ int attn_page_bytes(const Params& p) { return p.hkv * p.P * p.d * 2; }
__device__ __forceinline__ int attn_pps(const Params& p) {
  const int pb = attn_page_bytes(p);
  return pb >= kStageBytes / 2 ? 1 : (kStageBytes / 2) / pb;
}

// share of slice s of n in [0, total); total * n < 2^32 for every device-side
// share (rows or groups of the routed experts over at most a few hundred
// slices), so 32-bit arithmetic suffices (a 64-bit division is a long
// software sequence on the critical path)
__device__ __forceinline__ void dshare(int total, int n, int s, int& lo, int& hi) {
  lo = (int)((uint32_t)total * (uint32_t)s / (uint32_t)n);
  hi = (int)((uint32_t)total * (uint32_t)(s + 1) / (uint32_t)n);
}

// one token: rows of a GEMV chunk.  Rows of 2048 or 4096 columns go to the
// tensor cores, whose per-warp partial sums of a chunk fill one kMmaRows x 8
// buffer; other row lengths go whole to one warp each.
__device__ __forceinline__ int one_rows(int K) { return rotated_rows(K) ? kMmaRows : kRowChunk; }

// One token: top-k of the router logits of layer l, softmax weights over the
// picks (the top-k of the softmax = the top-k of the logits; ties to the lower
// expert id) and the grouping, by one warp.  Lane j < k keeps the j-th pick;
// its rank among the picks (ascending expert id) is its active slot, and with
// one token every active expert has one entry.  keep: also store the routing
// in global memory (for inspection).
__device__ __forceinline__ void route_one(const Params& p, RouteTab& rt, int l, int lane, bool keep) {
  const int E = p.E, K = p.topk;
  float v[8];
  const float* rl = p.rlog + (size_t)l * p.Bmax * E;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldcg(rl + e) : -INFINITY;
  }
  // each pick: the lane's best remaining value (ties to its lower expert id),
  // then two warp reductions on an order-preserving integer key: the largest
  // key, and the lowest expert id holding it (-0 is taken as +0, so equal
  // values tie exactly as in a float comparison)
  uint32_t taken = 0;
  float my_v = -INFINITY;
  int my_e = 0x7fffffff;
#pragma unroll 1
  for (int j = 0; j < K; j++) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > bv || bi == 0x7fffffff)) {
        bv = v[i];
        bi = e;
      }
    }
    const uint32_t u = __float_as_uint(bv == 0.f ? 0.f : bv);
    const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const uint32_t emin = __reduce_min_sync(0xffffffffu, key == kmax ? (uint32_t)bi : 0xffffffffu);
    if ((int)(emin & 31u) == lane) taken |= 1u << (emin >> 5);
    if (lane == j) {
      my_v = __uint_as_float((kmax & 0x80000000u) ? (kmax & 0x7fffffffu) : ~kmax);
      my_e = (int)emin;
    }
  }
  const float top = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < K ? expf(my_v - top) : 0.f;
  float den = 0.f;
  for (int j = 0; j < K; j++) den += __shfl_sync(0xffffffffu, ex, j);   // fixed order
  const float w = ex / den;
  int rank = 0;
  for (int j = 0; j < K; j++) rank += __shfl_sync(0xffffffffu, my_e, j) < my_e;
  if (lane < K) {
    rt.idx[0][lane] = my_e;
    rt.w[0][lane] = w;
    rt.act[rank] = my_e;
    rt.off[rank] = rank;
    rt.ent[rank] = lane;
    if (keep) {
      p.ridx[(size_t)l * p.Bmax * K + lane] = my_e;
      p.rw[(size_t)l * p.Bmax * K + lane] = w;
    }
  }
  if (lane == 0) {
    rt.n_act = K;
    rt.off[K] = K;
  }
  __syncwarp();
}

// ===================================================================== producer
// One warp.  Resolves each descriptor into GEMV chunks / attention items,
// writes them straight into the task ring (lane 0 writes the words; no
// per-thread arrays, which would live in local memory) and streams their
// weight / KV stages.
// ONE: the batch has one token; TR: the task timeline is recorded (kernel
// instance); F8: the routed experts are 8-bit (E4M3)
template <bool ONE, bool TR, bool F8 = false>
struct Prod {
  const Params& p;
  Smem& S;
  int lane;
  uint32_t stage_seq = 0, task_seq = 0, route_seen = 0;
  bool ok = true;
  // header of the descriptor being resolved
  int op = 0, l = 0, ti = 0, bump = 0;
  // weight pointers of layer ptr_layer (cur) and of the next layer (nxt), lane
  // i holding matrix i (router, qkv, o, gate, up, down): the pointer tables
  // are read a layer ahead, so no stream waits on one
  const uint16_t* cur = nullptr;
  const uint16_t* nxt = nullptr;
  int ptr_layer = -1;
  // stages this SM keeps in flight: the whole ring, or moe_depth on an SM
  // without attention items (the expert branch)
  uint32_t depth = kStages;

  __device__ __forceinline__ Prod(const Params& pp, Smem& ss) : p(pp), S(ss), lane(threadIdx.x & 31) {
    if (ONE && p.attn_sm_off[blockIdx.x] == p.attn_sm_off[blockIdx.x + 1] && p.moe_depth > 0)
      depth = (uint32_t)min(p.moe_depth, kStages);
  }

  __device__ __forceinline__ const uint16_t* load_ptr(int layer) const {
    if (layer >= p.L || lane >= 6) return nullptr;
    const uint16_t* const* tab = lane == 0 ? p.w_router : lane == 1 ? p.w_qkv : lane == 2 ? p.w_o
                                 : lane == 3 ? p.w_gate : lane == 4 ? p.w_up : p.w_down;
    return tab[layer];
  }
  __device__ __forceinline__ void set_layer(int layer) {
    if (layer == ptr_layer || layer >= p.L) return;
    cur = (ptr_layer >= 0 && layer == ptr_layer + 1) ? nxt : load_ptr(layer);
    nxt = load_ptr(layer + 1);
    ptr_layer = layer;
  }
  // matrix i of the current layer
  __device__ __forceinline__ const uint16_t* wptr(int i) const {
    return (const uint16_t*)__shfl_sync(0xffffffffu, (unsigned long long)cur, i);
  }

  // reserve the next task slot, zero it and write the header; nullptr on give-up
  __device__ __forceinline__ int32_t* begin() {
    const uint32_t slot = task_seq % kTaskSlots;
    if (!wait_phase(p, &S.tempty[slot], ((task_seq / kTaskSlots) & 1u) ^ 1u)) return nullptr;
    int32_t* w = S.task[slot];
    w[lane] = 0;
    __syncwarp();
    if (lane == 0) {
      w[R_OP] = op;
      w[R_LAYER] = l;
      w[R_TASK] = ti;
      w[R_BUMP] = bump;
    }
    return w;
  }

  __device__ __forceinline__ void commit() {
    __syncwarp();
    if (lane == 0) {
      if (TR) S.task[task_seq % kTaskSlots][R_PCOMMIT] = (int32_t)(uint32_t)gtime_ns();
      mbar_arrive(&S.tfull[task_seq % kTaskSlots]);
    }
    task_seq++;
  }

  __device__ __forceinline__ bool acquire_stage(uint32_t& slot) {
    slot = stage_seq % kStages;
    bool ok = wait_phase(p, &S.empty[slot], ((stage_seq / kStages) & 1u) ^ 1u);
    // an expert-branch SM keeps at most moe_depth stages in flight: stage
    // stage_seq - moe_depth must have been consumed (its slot's phase of that
    // round has completed)
    if (ONE && ok && depth < (uint32_t)kStages && stage_seq >= depth) {
      const uint32_t n = stage_seq - depth;
      ok = wait_phase(p, &S.empty[n % kStages], (n / kStages) & 1u);
    }
    if (TR && lane == 0 && task_seq > 0) {
      // the copy is issued next (after the mbarrier's release, which orders this word)
      int32_t* w = S.task[(task_seq - 1) % kTaskSlots];
      if (w[R_PISSUE] == 0) w[R_PISSUE] = (int32_t)((uint32_t)gtime_ns() | 1u);
    }
    return ok;
  }

  // rows [row0, row0 + nrows) of a row-major [*, K] matrix, whole rows, one
  // copy per stage: a 1-D bulk copy, or (rows of 2048 or 4096 columns bound
  // for the tensor cores) a 3-D tensor copy through the matrix's map, which lands the
  // stage swizzled for the tensor-core GEMV (a whole box: rows past a short
  // last stage are copied too, or zero-filled past the matrix)
  // (map_row0: the first row's index in the map, when it differs from row0;
  // box_rows: rows of one box, 0 = a full 32 KB stage of rows)
  __device__ __forceinline__ bool stream_rows(const uint16_t* w, int row0, int nrows, int K,
                                              const uint8_t* map = nullptr, int map_row0 = -1,
                                              int box_rows = 0) {
    const bool rot = map != nullptr;
    const int rps = rot && box_rows > 0 ? box_rows : rows_per_stage(K);
    const int mrow0 = map_row0 >= 0 ? map_row0 : row0;
    for (int done = 0; done < nrows; done += rps) {
      const int rows = min(rps, nrows - done);
      uint32_t slot;
      if (!acquire_stage(slot)) return false;
      if (lane == 0) {
        if (rot) {
          mbar_arrive_expect_tx(&S.full[slot], (uint32_t)(rps * K * 2));
          tma_load_3d_hint(&S.stage[slot][0], map, 0, mrow0 + done, 0, &S.full[slot], policy_evict_first());
        } else {
          const uint32_t bytes = (uint32_t)(rows * K * 2);
          mbar_arrive_expect_tx(&S.full[slot], bytes);
          bulk_g2s_hint(&S.stage[slot][0], w + (size_t)(row0 + done) * K, bytes, &S.full[slot],
                        policy_evict_first());
        }
      }
      __syncwarp();
      stage_seq++;
    }
    return true;
  }

  // the tensor map of matrix `which` (W_MAP_*) of the current layer
  __device__ __forceinline__ const uint8_t* wmap(int which) const {
    return p.w_maps + ((size_t)W_MAPS_PER_LAYER * l + which) * 128;
  }

  // pages [pg0, pg0 + npages) of sequence b, all KV heads: K pages then V
  // pages, each as d / 64 swizzled boxes of (hkv * P rows) x 128 bytes.  The
  // page ids are read 32 at a time (lane k holds page c0 + k), the next 32
  // requested while the current ones stream, so no stage waits on a
  // page-table read.
  __device__ __forceinline__ bool stream_attn(int b, int pg0, int npages) {
    const int pb = attn_page_bytes(p);
    const int pps = attn_pps(p);                 // a power of two <= 8: divides 32
    const int rows = p.hkv * p.P;
    const int nbox = p.d / 64;
    const uint8_t* km = p.kv_maps + (size_t)l * 2 * 128;
    const uint8_t* vm = km + 128;
    const int32_t* ptab = p.page_tables + (size_t)b * p.max_pages + pg0;
    int id_next = lane < npages ? ptab[lane] : 0;
    for (int c0 = 0; c0 < npages; c0 += 32) {
      const int id = id_next;
      if (c0 + 32 + lane < npages) id_next = ptab[c0 + 32 + lane];
      const int cn = min(32, npages - c0);
      for (int q = 0; q < cn; q += pps) {
        const int n = min(pps, cn - q);
        const int pg = __shfl_sync(0xffffffffu, id, q + (lane % n));
        if (TR && p.dbg && l == 0 && lane < n)
          p.dbg[(size_t)p.L * kDbgRouteWords + (size_t)b * p.max_pages + pg0 + c0 + q + lane] = pg;
        const bool bad = (lane < 2 * n) && (pg < 0 || pg >= p.num_pages);
        if (__any_sync(0xffffffffu, bad)) {
          if (bad) report(p, DEV_BAD_PAGE, ti, OP_ATTN, -1, (uint32_t)pg, (uint32_t)p.num_pages);
          return false;
        }
        uint32_t slot;
        if (!acquire_stage(slot)) return false;
        if (lane == 0) mbar_arrive_expect_tx(&S.full[slot], (uint32_t)(2 * n * pb));
        __syncwarp();
        if (lane < 2 * n) {
          const bool is_k = lane < n;
          uint8_t* dst = &S.stage[slot][(is_k ? lane : pps + lane - n) * pb];
          for (int bx = 0; bx < nbox; bx++)
            tma_load_2d_hint(dst + bx * rows * 128, is_k ? km : vm, bx * 64, pg * rows, &S.full[slot],
                             policy_evict_first());
        }
        stage_seq++;
      }
    }
    return true;
  }

  // one GEMV chunk of nblk blocks x nrows rows: publish, then stream each block
  __device__ __forceinline__ bool chunk(int kind, int flags, int row0, int nrows, int nblk, int K, int nt,
                                        int a, int e, int rel0, const uint16_t* w0, const uint16_t* w1,
                                        const uint8_t* m0 = nullptr, const uint8_t* m1 = nullptr,
                                        int map_row0 = -1, int box_rows = 0) {
    int32_t* w = begin();
    if (!w) return false;
    if (lane == 0) {
      w[R_KIND] = kind;
      w[R_FLAGS] = flags;
      w[R_ROW0] = row0;
      w[R_NROWS] = nrows;
      w[R_NBLK] = nblk;
      w[R_K] = K;
      w[R_NT] = nt;
      w[R_A] = a;
      w[R_E] = e;
      w[R_REL0] = rel0;
    }
    commit();
    if (nrows > 0 && !stream_rows(w0, row0, nrows, K, m0, map_row0, box_rows)) return false;
    if (nblk > 1 && nrows > 0 && !stream_rows(w1, row0, nrows, K, m1, map_row0, box_rows)) return false;
    return true;
  }

  // rows [lo, hi) of w in chunks of cr; `first` / `last` mark the task's ends;
  // map: the matrix's tensor map when the chunks go to the tensor cores
  __device__ __forceinline__ bool rows_task(int kind, const uint16_t* w, int lo, int hi, int cr, int K,
                                            int nt, bool first, bool last, int last_extra = 0,
                                            const uint8_t* map = nullptr) {
    for (int c0 = lo; c0 < hi; c0 += cr) {
      const int flags = (first && c0 == lo ? FL_FIRST : 0) | (last && c0 + cr >= hi ? FL_LAST : 0) |
                        (c0 + cr >= hi ? last_extra : 0);
      if (!chunk(kind, flags, c0, min(cr, hi - c0), 1, K, nt, 0, 0, 0, w, nullptr, map)) return false;
    }
    return true;
  }

  // several tokens: the tensor map of matrix `which` when its rows go to the tensor cores
  __device__ __forceinline__ const uint8_t* mmap(int which, int K) const {
    return (p.w_maps && mma_multi_rows(K, p.B)) ? wmap(which) : nullptr;
  }

  // bounded spin of the whole warp on a global counter; every lane's load is
  // an acquire, so each lane's later reads see what was released with it
  __device__ __forceinline__ bool warp_spin(int bar, uint32_t target) {
    const uint32_t* c = p.bars + bar;
    const unsigned long long t0 = gtime_ns();
    for (uint32_t it = 0;; ++it) {
      const uint32_t v = ld_acquire_u32(c);
      if (__all_sync(0xffffffffu, v >= target)) return true;
      __nanosleep(32);
      if ((it & 15u) == 15u) {
        int give = 0;
        if (lane == 0) {
          if (stopped(p)) {
            give = 1;
          } else if (gtime_ns() - t0 > p.timeout_ns) {
            report(p, DEV_TIMEOUT, ti, op, bar, v, target);
            give = 1;
          }
        }
        if (__shfl_sync(0xffffffffu, give, 0)) return false;
      }
    }
  }

  // one token: the producer routes layer l itself as soon as the router
  // logits are complete, so the experts' weights stream while the consumers
  // still work on P1
  __device__ __forceinline__ bool route_here() {
    if (!warp_spin(bar_index(p, l, p.bl.rtr), (uint32_t)p.n_rtr_sms)) return false;
    route_one(p, S.rt, l, lane, blockIdx.x == 0);
    route_seen = l + 1;
    if (TR && p.dbg && blockIdx.x == 0) {
      int32_t* d = p.dbg + (size_t)l * kDbgRouteWords;
      const int n = S.rt.n_act;
      if (lane == 0) d[0] = n;
      for (int i = lane; i < n; i += 32) {
        d[1 + i] = S.rt.act[i];
        d[1 + kMaxActive + 1 + kMaxActive + i] = S.rt.ent[i];
      }
      for (int i = lane; i <= n; i += 32) d[1 + kMaxActive + i] = S.rt.off[i];
    }
    return true;
  }

  // the routing of layer l is in shared memory (written by this block's consumers)
  __device__ __forceinline__ bool wait_route() {
    if ((int)route_seen > l) return true;
    if (!wait_phase(p, &S.route_bar, (uint32_t)l & 1u)) return false;
    route_seen = l + 1;
    return true;
  }

  // one-token P1 / FINAL: chunks of up to kRowChunk rows; a P1 chunk holds its
  // router rows and its QKV rows as two groups
  // one token, P1: the router rows [a0, a1) first, in chunks of their own
  // (the last one releases the router counter), then the W_qkv rows [b0, b1);
  // FINAL: LM-head rows [a0, a1); OUT: O-proj rows [a0, a1).  One loop emits
  // every chunk (one copy of the hand-over and stream code): phase 0 walks
  // [a0, a1), phase 1 [b0, b1).
  __device__ __forceinline__ bool do_rows1(int a0, int a1, int b0, int b1) {
    const bool fin = op == OP_FINAL, out = op == OP_OUT;
    const int H = out ? p.hq * p.d : p.H;         // row length
    if (fin || out) b1 = b0;
    const int cr = one_rows(H);
    const uint16_t* m0 = fin ? p.lm_head : wptr(out ? 2 : 0);
    const bool rot = rotated_rows(H);
    const uint8_t* map0 = !rot ? nullptr : fin ? p.w_maps + (size_t)W_MAPS_PER_LAYER * p.L * 128
                                             : wmap(out ? W_MAP_O : W_MAP_ROUTER);
    const uint8_t* map1 = rot ? wmap(W_MAP_QKV) : nullptr;
    int ph = a1 > a0 ? 0 : 1, c0 = ph == 0 ? a0 : b0;
    bool first = true;
    do {
      const int hi = ph == 0 ? a1 : b1;
      const int c1 = min(hi, c0 + cr);
      const bool end_ph = c1 >= hi;
      const bool last = end_ph && (ph == 1 || b1 <= b0);
      int32_t* w = begin();
      if (!w) return false;
      if (lane == 0) {
        w[R_KIND] = fin ? K_LM : out ? K_OPROJ : K_P1;
        w[R_FLAGS] = (first ? FL_FIRST : 0) | (last ? FL_LAST : 0) | (op == OP_P1 && ph == 0 && end_ph ? FL_RTR : 0);
        w[R_ROW0] = ph == 0 ? c0 : 0;
        w[R_NROWS] = ph == 0 ? max(c1 - c0, 0) : 0;
        w[R_ROW1] = ph == 1 ? c0 : 0;
        w[R_NROWS1] = ph == 1 ? max(c1 - c0, 0) : 0;
        w[R_NBLK] = 1;
        w[R_K] = H;
        w[R_NT] = 1;
      }
      commit();
      if (c1 > c0 && !stream_rows(ph == 0 ? m0 : wptr(1), c0, c1 - c0, H, ph == 0 ? map0 : map1)) return false;
      first = false;
      c0 = c1;
      if (end_ph && ph == 0) {
        ph = 1;
        c0 = b0;
      }
    } while (c0 < (ph == 0 ? a1 : b1));
    return true;
  }

  __device__ __forceinline__ bool do_p1_final(int a0, int a1, int b0, int b1) {
    const int H = p.H, B = p.B;
    if (ONE) return do_rows1(a0, a1, b0, b1);
    const int cr = gemv_chunk_rows(H, B);
    if (op == OP_FINAL) {
      if (a1 <= a0) return chunk(K_LM, FL_FIRST | FL_LAST, 0, 0, 1, H, B, 0, 0, 0, nullptr, nullptr);
      const uint8_t* lm = (p.w_maps && mma_multi_rows(H, B)) ? p.w_maps + (size_t)W_MAPS_PER_LAYER * p.L * 128
                                                              : nullptr;
      return rows_task(K_LM, p.lm_head, a0, a1, cr, H, B, true, true, 0, lm);
    }
    // P1: router rows [a0, a1) (the last of their chunks releases the router
    // counter), then W_qkv rows [b0, b1)
    const int r0 = a0, r1 = a1, q0 = b0, q1 = b1;
    if (r1 <= r0 && q1 <= q0) return chunk(K_ROUTER, FL_FIRST | FL_LAST, 0, 0, 1, H, B, 0, 0, 0, nullptr, nullptr);
    if (r1 > r0 && !rows_task(K_ROUTER, wptr(0), r0, r1, cr, H, B, true, q1 <= q0, FL_RTR, mmap(W_MAP_ROUTER, H)))
      return false;
    if (q1 > q0 && !rows_task(K_QKV, wptr(1), q0, q1, cr, H, B, r1 <= r0, true, 0, mmap(W_MAP_QKV, H))) return false;
    return true;
  }

  __device__ __forceinline__ bool do_attn() {
    const int pps = attn_pps(p);
    const int sm = blockIdx.x;
    const int i0 = p.attn_sm_off[sm], i1 = p.attn_sm_off[sm + 1];
    for (int item = i0; item < i1; item++) {
      const int32_t iw = lane < 8 ? p.attn_items[(size_t)item * 8 + lane] : 0;
      const int b = __shfl_sync(0xffffffffu, iw, AI_B);
      const int t0 = __shfl_sync(0xffffffffu, iw, AI_T0);
      const int t1 = __shfl_sync(0xffffffffu, iw, AI_T1);
      const int pos = __shfl_sync(0xffffffffu, iw, AI_POS);
      const int pg0 = t0 / p.P, npages = (t1 + p.P - 1) / p.P - pg0;
      int32_t* w = begin();
      if (!w) return false;
      if (lane == 0) {
        w[R_B] = b;
        w[R_TT0] = t0;
        w[R_TT1] = t1;
        w[R_POS] = pos;
        w[R_ITEM] = item;
        w[R_NST] = (npages + pps - 1) / pps;
      }
      commit();
      if (!stream_attn(b, pg0, npages)) return false;
    }
    return true;
  }

  // one token: slice a0 of a1 over the routed experts' groups of 8
  // intermediate columns.  Each piece (one expert, n <= 8 groups) streams its
  // gate rows, its up rows and then its n groups of the down projection from
  // the blocked copy ([H][8] per group, contiguous): up to 2048 rows per
  // stage, one bulk copy each.
  __device__ __forceinline__ bool do_up1(int a0, int a1) {
    const int H = p.H, G = p.I / 8, n_act = S.rt.n_act;
    int g0 = 0, g1 = 0;
    if (a0 >= 0) {
      if (a1 >= n_act) {
        // at least one slice per expert: expert a takes slices
        // [a * a1 / n_act, (a + 1) * a1 / n_act), so no slice spans two
        // experts; slice a0's expert is the largest a with a * a1 / n_act <= a0
        const int a = ((a0 + 1) * n_act - 1) / a1;
        const int s0 = a * a1 / n_act, s1 = (a + 1) * a1 / n_act;
        dshare(G, s1 - s0, a0 - s0, g0, g1);
        g0 += a * G;
        g1 += a * G;
      } else {
        dshare(n_act * G, a1, a0, g0, g1);
      }
    }
    if (g1 <= g0) return chunk(K_UP, FL_LAST, 0, 0, 2, H, 0, 0, 0, 0, nullptr, nullptr);
    for (int g = g0; g < g1;) {
      const int a = g / G;
      const int ge = min(min(g1, (a + 1) * G), g + 8);
      const int e = S.rt.act[a];
      const int i0 = (g - a * G) * 8, i1 = (ge - a * G) * 8;
      const int ncb = ge - g;
      int32_t* w = begin();
      if (!w) return false;
      if (lane == 0) {
        w[R_KIND] = K_UP;
        w[R_FLAGS] = (g == g0 ? FL_FIRST : 0) | (ge == g1 ? FL_LAST : 0);
        w[R_ROW0] = i0;
        w[R_NROWS] = i1 - i0;
        w[R_NBLK] = 2;
        w[R_K] = H;
        w[R_NT] = 1;
        w[R_A] = a;
        w[R_E] = e;
        w[R_REL0] = g;
      }
      commit();
      // the piece's gate rows, its up rows, then each of its groups of the
      // down projection (an [H][8] block, streamed as H rows of 8): one
      // stream loop for all of them keeps the code short
      // (8-bit experts: the same rows and blocks in bytes, streamed as rows
      // of half as many two-byte words)
      const int es = F8 ? 2 : 1;
      const size_t eo = (size_t)e * p.I * H / es;
      const uint16_t* blk = p.wd_blk + (((size_t)l * p.E + e) * G + i0 / 8) * H * 8 / es;
      for (int sg = 0; sg < 2 + (F8 ? 0 : ncb); sg++) {
        const bool dn = sg >= 2;
        const uint16_t* src = dn ? blk + (size_t)(sg - 2) * H * 8 : wptr(3 + sg) + eo;
        // gate / up rows through their maps: rows of the [E I][H] matrix
        if (!stream_rows(src, dn ? 0 : (rotated_rows(H) ? e * p.I : 0) + i0, dn ? H : i1 - i0,
                         (dn ? 8 : H) / es,
                         dn || !rotated_rows(H) ? nullptr : wmap(sg == 0 ? W_MAP_GATE : W_MAP_UP)))
          return false;
      }
      // 8-bit down projection: quads of up to four groups, a stage holding
      // the quad's rows [h0, h0 + rd) (one 1-D copy per group)
      if constexpr (F8) {
        const int rd = min(H, 1024);
        const uint8_t* b8 = (const uint8_t*)blk;
        for (int q0 = 0; q0 < ncb; q0 += 4) {
          const int nq = min(4, ncb - q0);
          for (int h0 = 0; h0 < H; h0 += rd) {
            uint32_t slot;
            if (!acquire_stage(slot)) return false;
            if (lane == 0) mbar_arrive_expect_tx(&S.full[slot], (uint32_t)(nq * rd * 8));
            __syncwarp();
            if (lane < nq)
              bulk_g2s_hint(&S.stage[slot][lane * rd * 8], b8 + ((size_t)(q0 + lane) * H + h0) * 8,
                            (uint32_t)(rd * 8), &S.full[slot], policy_evict_first());
            stage_seq++;
          }
        }
      }
      g = ge;
    }
    return true;
  }

  // several tokens, claimed tiles: the next tile index of claim counter
  // `off` of this layer (lane 0's atomic add, broadcast).  The claim orders
  // nothing: a tile's inputs are ordered by the routing wait and the UP
  // counter, as with static shares.
  __device__ __forceinline__ int claim(int off) {
    int c = 0;
    if (lane == 0) c = (int)atomicAdd(p.bars + bar_index(p, l, off), 1u);
    return __shfl_sync(0xffffffffu, c, 0);
  }

  // several tokens: the chunks of an expert's gate / up pair rows [i0, i1)
  __device__ __forceinline__ bool up_rows(int a, int i0, int i1, bool last) {
    const int H = p.H;
    const int e = S.rt.act[a];
    const int cnt = S.rt.off[a + 1] - S.rt.off[a];
    const int cp = max(1, gemv_chunk_rows(H, cnt) / 2);
    const size_t eo = (size_t)e * p.I * H;
    const bool mma = p.w_maps && mma_multi_rows(H, cnt);
    const uint8_t* mg = mma ? wmap(W_MAP_GATE) : nullptr;
    const uint8_t* mu = mma ? wmap(W_MAP_UP) : nullptr;
    for (int c0 = i0; c0 < i1; c0 += cp)
      if (!chunk(K_UP, (last && c0 + cp >= i1) ? FL_LAST : 0, c0, min(cp, i1 - c0), 2, H, cnt, a, e, 0,
                 wptr(3) + eo, wptr(4) + eo, mg, mu, e * p.I + c0))
        return false;
    return true;
  }

  __device__ __forceinline__ bool do_up(int a0, int a1) {
    const int H = p.H;
    if (!wait_route()) return false;
    if (ONE) return do_up1(a0, a1);
    const int n_act = S.rt.n_act;
    // claimed tiles of claim_rows / 2 pair rows; the next tile is claimed
    // before this one streams, so the SM knows which chunk is its last
    if (p.claim_rows > 0) {
      const int T = max(1, p.claim_rows / 2), tpe = (p.I + T - 1) / T, ntiles = n_act * tpe;
      int c = a0 >= 0 ? claim(p.bl.claim_up) : ntiles;
      if (c >= ntiles) return chunk(K_UP, FL_LAST, 0, 0, 2, H, 0, 0, 0, 0, nullptr, nullptr);
      while (c < ntiles) {
        const int nx = claim(p.bl.claim_up);
        const int a = c / tpe, i0 = (c % tpe) * T;
        if (!up_rows(a, i0, min(i0 + T, p.I), nx >= ntiles)) return false;
        c = nx;
      }
      return true;
    }
    // static share: slice a0 of a1 over the routed experts' pair rows, as
    // (active expert, pair range) pieces of [p0, p1)
    int p0 = 0, p1 = 0;
    if (a0 >= 0) dshare(n_act * p.I, a1, a0, p0, p1);
    if (p1 <= p0) return chunk(K_UP, FL_LAST, 0, 0, 2, H, 0, 0, 0, 0, nullptr, nullptr);
    for (int a = p0 / p.I; a < n_act && a * p.I < p1; a++) {
      const int i0 = max(p0 - a * p.I, 0), i1 = min(p1 - a * p.I, p.I);
      if (!up_rows(a, i0, i1, a * p.I + i1 == p1)) return false;
    }
    return true;
  }

  // OUT: O-proj rows [a0, a1) (needs no routing).  Several tokens: then the
  // sum of each token's weighted expert outputs of the same rows (K_MSUM,
  // after every DOWN task)
  __device__ __forceinline__ bool do_out(int a0, int a1) {
    const int B = p.B;
    const int KO = p.hq * p.d;
    const int last = ONE ? FL_LAST : 0;
    if (a1 <= a0) return chunk(K_OPROJ, FL_LAST, 0, 0, 1, KO, B, 0, 0, 0, nullptr, nullptr);
    // (several tokens through the tensor cores: one partial per (row, warp,
    // token), at most kPartFloats of them per chunk)
    const uint8_t* mo = ONE ? nullptr : mmap(W_MAP_O, KO);
    const int co = ONE ? one_rows(KO) : mo ? kPartFloats / (kConsumerWarps * B) : gemv_chunk_rows(KO, B);
    for (int c0 = a0; c0 < a1; c0 += co)
      if (!chunk(K_OPROJ, c0 + co >= a1 ? last : 0, c0, min(co, a1 - c0), 1, KO, B, 0, 0, 0, wptr(2),
                 nullptr, mo))
        return false;
    if (ONE) return true;
    int32_t* w = begin();     // streams nothing
    if (!w) return false;
    if (lane == 0) {
      w[R_KIND] = K_MSUM;
      w[R_FLAGS] = FL_LAST;
      w[R_ROW0] = a0;
      w[R_NROWS] = a1 - a0;
      w[R_NT] = B;
    }
    commit();
    return true;
  }

  // DOWN: hidden rows [a0, a1) of every routed expert's down projection.
  // One token: the sum of the UP slices' per-group partials of those rows
  // (K_MRED), streamed once every UP slice has written them: 256 groups x 32
  // rows per stage.
  __device__ __forceinline__ bool do_down(int a0, int a1) {
    const int H = p.H, B = p.B;
    if (ONE) {
      int32_t* w = begin();
      if (!w) return false;
      if (lane == 0) {
        w[R_KIND] = K_MRED;
        w[R_FLAGS] = FL_LAST;
        w[R_ROW0] = a0;
        w[R_NROWS] = max(a1 - a0, 0);
        w[R_NT] = 1;
      }
      commit();
      if (a1 <= a0) return true;
      // the partials are written by other SMs (generic stores, released with
      // the counter): acquire, then order the async-proxy reads after it
      int good = 1;
      if (lane == 0) {
        good = spin_counter(p, bar_index(p, l, p.bl.up), (uint32_t)p.n_up_sms, ti, op);
        if (good) fence_proxy_async_global();
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) return false;
      const int ng = p.topk * (p.I / 8);
      for (int x0 = a0 & ~3; x0 < a1; x0 += kMredCols)
        for (int y0 = 0; y0 < ng; y0 += 256) {
          uint32_t slot;
          if (!acquire_stage(slot)) return false;
          if (lane == 0) {
            mbar_arrive_expect_tx(&S.full[slot], (uint32_t)kMredCols * 256u * 4u);
            tma_load_2d(&S.stage[slot][0], p.mp_map, x0, y0, &S.full[slot]);
          }
          __syncwarp();
          stage_seq++;
        }
      return true;
    }
    // several tokens: slice a0 of a1 over the routed experts' rows of the
    // down projection (expert-major: an expert's H rows, then the next
    // expert's); each chunk's epilogue writes its rows of every routed entry's
    // weighted output, summed by OUT
    if (!wait_route()) return false;
    const int n_act = S.rt.n_act;
    // claimed tiles of claim_rows down rows (expert-major), as in do_up
    if (p.claim_rows > 0) {
      const int T = p.claim_rows, tpe = (H + T - 1) / T, ntiles = n_act * tpe;
      int c = a0 >= 0 ? claim(p.bl.claim_down) : ntiles;
      if (c >= ntiles) return chunk(K_DOWN, FL_LAST, 0, 0, 1, p.I, 0, 0, 0, 0, nullptr, nullptr);
      while (c < ntiles) {
        const int nx = claim(p.bl.claim_down);
        const int a = c / tpe, h0 = (c % tpe) * T;
        if (!down_rows(a, h0, min(h0 + T, H), nx >= ntiles)) return false;
        c = nx;
      }
      return true;
    }
    int r0 = 0, r1 = 0;
    if (a0 >= 0) dshare(n_act * H, a1, a0, r0, r1);
    if (r1 <= r0) return chunk(K_DOWN, FL_LAST, 0, 0, 1, p.I, 0, 0, 0, 0, nullptr, nullptr);
    for (int a = r0 / H; a < n_act && a * H < r1; a++) {
      const int h0 = max(r0 - a * H, 0), h1 = min(r1 - a * H, H);
      if (!down_rows(a, h0, h1, a * H + h1 == r1)) return false;
    }
    return true;
  }

  // several tokens: the chunks of an expert's down rows [h0, h1)
  __device__ __forceinline__ bool down_rows(int a, int h0, int h1, bool last) {
    const int H = p.H;
    const int e = S.rt.act[a];
    const int cnt = S.rt.off[a + 1] - S.rt.off[a];
    // tensor cores: one fp32 partial per (row, warp, token) in the chunk's buffer
    const bool mma = p.wd_maps != nullptr;
    const int cd = mma ? max(kDownBoxRows, min(512, kPartFloats / (kConsumerWarps * cnt)) / kDownBoxRows *
                                               kDownBoxRows)
                       : gemv_chunk_rows(p.I, cnt);
    const uint16_t* wd = wptr(5) + (size_t)e * H * p.I;
    const uint8_t* md = mma ? p.wd_maps + (size_t)l * 128 : nullptr;
    for (int c0 = h0; c0 < h1; c0 += cd)
      if (!chunk(K_DOWN, (last && c0 + cd >= h1) ? FL_LAST : 0, c0, min(cd, h1 - c0), 1, p.I, cnt, a, e, 0, wd,
                 nullptr, md, nullptr, e * H + c0, kDownBoxRows))
        return false;
    return true;
  }

  __device__ __forceinline__ void run() {
    const int sm = blockIdx.x;
    const int t_begin = p.task_off[sm], t_end = p.task_off[sm + 1];
    for (ti = t_begin; ti < t_end && ok; ti++) {
      const int32_t word = p.tasks[(size_t)ti * kDescWords + lane];
      op = __shfl_sync(0xffffffffu, word, F_OP);
      l = __shfl_sync(0xffffffffu, word, F_LAYER);
      const int a0 = __shfl_sync(0xffffffffu, word, F_A0);
      const int a1 = __shfl_sync(0xffffffffu, word, F_A1);
      bump = __shfl_sync(0xffffffffu, word, F_BUMP);
      set_layer(l);
      switch (op) {
        case OP_P1:
        case OP_FINAL: {
          const int b0 = __shfl_sync(0xffffffffu, word, F_B0);
          const int b1 = __shfl_sync(0xffffffffu, word, F_B1);
          ok = do_p1_final(a0, a1, b0, b1);
          break;
        }
        case OP_ROUTE:
        case OP_COMBINE: {
          if (op == OP_ROUTE && ONE && !route_here()) {
            ok = false;
            break;
          }
          int32_t* w = begin();
          ok = w != nullptr;
          if (ok) {
            if (lane == 0) {
              w[R_U0] = a0;
              w[R_U1] = a1;
            }
            commit();
          }
          break;
        }
        case OP_ATTN: ok = do_attn(); break;
        case OP_UP: ok = do_up(a0, a1); break;
        case OP_OUT: ok = ONE ? do_rows1(a0, a1, 0, 0) : do_out(a0, a1); break;
        case OP_DOWN: ok = do_down(a0, a1); break;
        default:
          if (lane == 0) report(p, DEV_BAD_OP, ti, op, -1, 0, 0);
          ok = false;
      }
    }
    if (ok) {
      op = OP_END;
      ti = -1;
      ok = begin() != nullptr;
      if (ok) commit();
    }
    if (!ok) {
      // a wait gave up: a time-out, unless another block had already stopped
      // the step (the first report wins)
      if (lane == 0) report(p, DEV_SMEM_TIMEOUT, ti, op, -1, 0, 0);
      // stop: make sure no bulk copy of ours is still writing into shared memory
      const uint32_t n = stage_seq;
      const uint32_t first = n > (uint32_t)kStages ? n - kStages : 0u;
      if (lane == 0) {
        for (uint32_t s = first; s < n; s++) {
          const unsigned long long t0 = gtime_ns();
          while (!mbar_try_wait(&S.full[s % kStages], (s / kStages) & 1u)) {
            if (gtime_ns() - t0 > p.timeout_ns) break;
          }
        }
      }
      __syncwarp();
    }
  }
};

// ===================================================================== consumers
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// ONE: the batch has one token; TR: the task timeline is recorded (kernel instance)
template <bool ONE, bool TR>
struct Cons {
  const Params& p;
  Smem& S;
  const int tid, warp, lane, gl, cq;   // gl = lane / 4 (MMA group), cq = lane % 4
  const int32_t* t;                    // resolved task words, in its shared-memory slot
  uint32_t stage_seq;                  // stages this warp has consumed
  uint32_t cphase;                     // consumer-barrier phases this warp has passed

  __device__ __forceinline__ Cons(const Params& pp, Smem& ss, const int32_t* tt)
      : p(pp), S(ss), tid(threadIdx.x), warp(threadIdx.x >> 5), lane(threadIdx.x & 31),
        gl((threadIdx.x & 31) >> 2), cq(threadIdx.x & 3), t(tt),
        stage_seq(ss.cstage[threadIdx.x >> 5]), cphase(ss.cphase[threadIdx.x >> 5]) {}

  __device__ __forceinline__ void save() {
    __syncwarp();
    if (lane == 0) {
      S.cstage[warp] = stage_seq;
      S.cphase[warp] = cphase;
    }
    __syncwarp();
  }

  __device__ __forceinline__ bool aborted() { return S.abort_flag != 0; }

  // Barrier of the 8 consumer warps (the producer never joins).  It is an
  // mbarrier with a bounded wait rather than bar.sync, so a warp that has
  // already left after an error cannot leave the others waiting forever.
  __device__ __forceinline__ bool csync() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.cbar);
    const bool ok = wait_phase(p, &S.cbar, cphase & 1u);
    cphase++;
    if (!ok) S.abort_flag = 1;
    return ok && !aborted();
  }

  // cross-SM wait (thread 0 spins, the other consumers wait at the barrier).
  // Counters only grow, so a wait on the counter and target this block last
  // passed (or a lower target) needs no new wait.  Every warp keeps its own
  // copy of that (counter, target) pair, written only by itself after the
  // barrier: the copies agree because every warp makes the same sequence of
  // calls, and no warp can observe another's update half-way.
  __device__ __forceinline__ bool wait_counter(int bar, int target) {
    if (bar < 0) return true;
    if (bar == S.seen_bar[warp] && target <= S.seen_tgt[warp]) return true;
    if (tid == 0 && !spin_counter(p, bar, (uint32_t)target, t[R_TASK], t[R_OP])) S.abort_flag = 1;
    const bool ok = csync();
    if (ok && lane == 0) {
      S.seen_bar[warp] = bar;
      S.seen_tgt[warp] = target;
    }
    __syncwarp();
    if (TR && tid == 0) S.t_ready = gtime_ns();
    return ok;
  }

  // publish: every consumer's global stores are done; one thread releases the counter
  __device__ __forceinline__ bool signal(int bar, int inc) {
    if (!csync()) return false;
    if (tid == 0) red_release_add(p.bars + bar, (uint32_t)inc);
    return true;
  }

  // end of a chunk that finishes the SM's router rows (FL_RTR: release the
  // routing wait early) and / or its task (FL_LAST: bump the phase counter):
  // one barrier, then the releases (the block's stores, ordered before this
  // thread by the barrier, are visible before a counter moves)
  __device__ __forceinline__ bool finish(int flags) {
    const int op = t[R_OP], l = t[R_LAYER];
    int bar = -1;
    if (flags & FL_LAST) {
      if (op == OP_P1) bar = p.bl.p1;
      else if (op == OP_UP) bar = p.bl.up;
      else if (op == OP_OUT || (op == OP_DOWN && ONE)) bar = p.bl.out;
      else if (op == OP_DOWN) bar = p.bl.down;
    }
    if (!csync()) return false;
    if (tid == 0) {
      if (flags & FL_RTR) red_release_add(p.bars + bar_index(p, l, p.bl.rtr), 1u);
      if (bar >= 0) red_release_add(p.bars + bar_index(p, l, bar), 1u);
    }
    return true;
  }

  __device__ __forceinline__ bool stage_full(uint32_t& slot) {
    slot = stage_seq % kStages;
    const unsigned long long w0 = (TR && tid == 0) ? gtime_ns() : 0ull;
    if (!wait_phase(p, &S.full[slot], (stage_seq / kStages) & 1u)) {
      S.abort_flag = 1;
      return false;
    }
    if (TR && tid == 0) S.t_swait += gtime_ns() - w0;
    return true;
  }

  __device__ __forceinline__ void stage_release(uint32_t slot) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
    stage_seq++;
  }

  // fp32 activation row of token slot n of this GEMV chunk
  __device__ __forceinline__ const float* xrow(int n) const {
    const size_t Bm = (size_t)p.Bmax;
    switch (t[R_KIND]) {
      case K_ROUTER:
      case K_QKV:
      case K_LM:
        return p.xloc + ((size_t)blockIdx.x * Bm + n) * p.H;
      case K_UP:
        return p.xloc + ((size_t)blockIdx.x * Bm + S.rt.ent[S.rt.off[t[R_A]] + n] / p.topk) * p.H;
      case K_OPROJ:
        return p.attn_out + ((size_t)t[R_LAYER] * Bm + n) * p.hq * p.d;
      default:   // K_DOWN
        return p.abuf + ((size_t)t[R_LAYER] * Bm * p.topk + S.rt.off[t[R_A]] + n) * p.I;
    }
  }

  // OUT tasks of a layer (and, one token, its DOWN tasks): the next layer's
  // residual is complete
  __device__ __forceinline__ int out_target() const { return ONE ? p.n_sm + p.n_down_sms : p.n_sm; }

  // residual update of layer l, token n, float4 i4: O-proj + experts
  __device__ __forceinline__ float4 delta4(int l, int n, int i4) const {
    const size_t at = ((size_t)l * p.Bmax + n) * p.H;
    const float4 o = __ldcg((const float4*)(p.oproj + at) + i4);
    const float4 m = __ldcg((const float4*)(p.moe + at) + i4);
    return make_float4(o.x + m.x, o.y + m.y, o.z + m.z, o.w + m.w);
  }

  // ------------------------------------------------------------ RMSNorm
  // h_l = h_{l-1} + (oproj_{l-1} + moe_{l-1}) (the embedding row at l = 0),
  // this SM's own copy; x_l = h_l / sqrt(mean(h_l^2) + eps) * gain.  Thread t
  // owns columns 4 t + 1024 i.  SM 0 also keeps every layer's h and x for
  // inspection.
  // one token: every load (own residual copy, the previous layer's update,
  // the gain) issued together, each thread sums the eight warp partials
  // itself (same order in every thread), x goes to the staging buffer
  // NI: float4s per thread (H <= 1024 NI): the instance for the model's H
  // runs, and its code is no longer than it needs to be
  template <int NI>
  __device__ __forceinline__ bool norm1(int l, bool final_norm) {
    const int H = p.H, H4 = H / 4;
    const size_t Bm = (size_t)p.Bmax;
    float* hl = p.hloc + (size_t)blockIdx.x * Bm * H;
    float* xl = p.xloc + (size_t)blockIdx.x * Bm * H;
    const uint16_t* gain = final_norm ? p.final_norm : p.attn_norm[l];
    float4 h[NI];
    uint2 g[NI];
#pragma unroll
    for (int k = 0; k < NI; k++) {              // loads that do not wait for the previous layer
      const int i4 = tid + 256 * k;
      h[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      g[k] = make_uint2(0, 0);
      if (i4 < H4) {
        g[k] = *(const uint2*)(gain + i4 * 4);
        if (l == 0) {
          const uint2 e = *(const uint2*)(p.embed + (size_t)p.tokens[0] * H + i4 * 4);
          h[k] = make_float4(bf16lo(e.x), bf16hi(e.x), bf16lo(e.y), bf16hi(e.y));
        } else {
          h[k] = __ldcg((const float4*)hl + i4);
        }
      }
    }
    if (l > 0) {
      if (!wait_counter(bar_index(p, l - 1, p.bl.out), out_target() + t[R_BUMP])) return false;
      const float4* ol = (const float4*)(p.oproj + (size_t)(l - 1) * Bm * H);
      const float4* ml = (const float4*)(p.moe + (size_t)(l - 1) * Bm * H);
      float4 o[NI], m[NI];
#pragma unroll
      for (int k = 0; k < NI; k++) {
        const int i4 = tid + 256 * k;
        o[k] = i4 < H4 ? __ldcg(ol + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
        m[k] = i4 < H4 ? __ldcg(ml + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < NI; k++) {
        h[k].x += o[k].x + m[k].x;
        h[k].y += o[k].y + m[k].y;
        h[k].z += o[k].z + m[k].z;
        h[k].w += o[k].w + m[k].w;
      }
    }
    // the GEMVs of this layer take h * gain (in xs) and their epilogues scale
    // by 1 / rms (S.rinv[0]): W (h g / rms) = (W (h g)) / rms, so the sum of
    // squares is reduced while the GEMV already runs (one barrier)
    const bool keep = blockIdx.x == 0;
    float ssl = 0.f;
    float4 hg[NI];
#pragma unroll
    for (int k = 0; k < NI; k++) {
      const int i4 = tid + 256 * k;
      hg[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i4 < H4) {
        if (!final_norm) __stcg((float4*)hl + i4, h[k]);
        if (keep) __stcg((float4*)(p.hdbg + (size_t)l * Bm * H) + i4, h[k]);
        ssl += h[k].x * h[k].x + h[k].y * h[k].y + h[k].z * h[k].z + h[k].w * h[k].w;
        hg[k] = make_float4(h[k].x * bf16lo(g[k].x), h[k].y * bf16hi(g[k].x), h[k].z * bf16lo(g[k].y),
                            h[k].w * bf16hi(g[k].y));
        *(float4*)&S.xs[i4 * 4] = hg[k];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssl += __shfl_xor_sync(0xffffffffu, ssl, o);
    if (lane == 0) S.nred[warp][0] = ssl;
    if (!csync()) return false;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; w++) sum += S.nred[w][0];
    const float r = 1.0f / sqrtf(sum / (float)H + p.rms_eps);
    if (tid == 0) S.rinv[0] = r;     // read by the epilogues, after their barriers
    if (keep) {
#pragma unroll
      for (int k = 0; k < NI; k++) {
        const int i4 = tid + 256 * k;
        if (i4 < H4)
          __stcg((float4*)(p.xdbg + (size_t)l * Bm * H) + i4,
                 make_float4(hg[k].x * r, hg[k].y * r, hg[k].z * r, hg[k].w * r));
      }
    }
    (void)xl;
    return true;
  }

  __device__ __forceinline__ bool norm(int l, bool final_norm) {
    if (ONE) {
      const int H4 = p.H / 4;
      return H4 <= 256 ? norm1<1>(l, final_norm) : H4 <= 512 ? norm1<2>(l, final_norm) : norm1<4>(l, final_norm);
    }
    const int H4 = p.H / 4;
    return H4 <= 256 ? norm_multi<1>(l, final_norm) : H4 <= 512 ? norm_multi<2>(l, final_norm)
                     : norm_multi<4>(l, final_norm);
  }

  // several tokens: the same per token, with the loads of TB = 8 / NI tokens
  // in flight together (each thread holds columns 4 t + 1024 k, NI float4s of a
  // token), so a layer's norm waits for a few L2 round trips, not one per token
  template <int NI>
  __device__ __forceinline__ bool norm_multi(int l, bool final_norm) {
    constexpr int TB = 8 / NI;
    const int H = p.H, B = p.B, H4 = H / 4;
    const size_t Bm = (size_t)p.Bmax;
    if (l > 0 && !wait_counter(bar_index(p, l - 1, p.bl.out), out_target() + t[R_BUMP])) return false;
    float* hl = p.hloc + (size_t)blockIdx.x * Bm * H;
    float* xl = p.xloc + (size_t)blockIdx.x * Bm * H;
    const bool keep = blockIdx.x == 0;
    const uint16_t* gain = final_norm ? p.final_norm : p.attn_norm[l];
    // h = the residual + the previous layer's update (the embedding row at l = 0)
    for (int n0 = 0; n0 < B; n0 += TB) {
      float4 h[TB][NI];
#pragma unroll
      for (int b = 0; b < TB; b++)
#pragma unroll
        for (int k = 0; k < NI; k++) {
          const int n = n0 + b, i4 = tid + 256 * k;
          h[b][k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (n < B && i4 < H4) {
            if (l == 0) {
              const uint2 e = *(const uint2*)(p.embed + (size_t)p.tokens[n] * H + i4 * 4);
              h[b][k] = make_float4(bf16lo(e.x), bf16hi(e.x), bf16lo(e.y), bf16hi(e.y));
            } else {
              const float4 a = __ldcg((const float4*)(hl + n * H) + i4);
              const float4 d = delta4(l - 1, n, i4);
              h[b][k] = make_float4(a.x + d.x, a.y + d.y, a.z + d.z, a.w + d.w);
            }
          }
        }
#pragma unroll
      for (int b = 0; b < TB; b++) {
        const int n = n0 + b;
        if (n >= B) break;
        float ssl = 0.f;
#pragma unroll
        for (int k = 0; k < NI; k++) {
          const int i4 = tid + 256 * k;
          if (i4 < H4) {
            if (!final_norm) __stcg((float4*)(hl + n * H) + i4, h[b][k]);
            if (keep) __stcg((float4*)(p.hdbg + ((size_t)l * Bm + n) * H) + i4, h[b][k]);
            ssl += h[b][k].x * h[b][k].x + h[b][k].y * h[b][k].y + h[b][k].z * h[b][k].z + h[b][k].w * h[b][k].w;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ssl += __shfl_xor_sync(0xffffffffu, ssl, o);
        if (lane == 0) S.nred[warp][n] = ssl;
      }
    }
    if (!csync()) return false;
    if (tid < B) {
      float sum = 0.f;
      for (int w = 0; w < kConsumerWarps; w++) sum += S.nred[w][tid];
      S.rinv[tid] = 1.0f / sqrtf(sum / (float)H + p.rms_eps);
    }
    if (!csync()) return false;
    // x = h / rms * gain (the final norm has not stored its h: it adds the update again)
    float4 g[NI];
#pragma unroll
    for (int k = 0; k < NI; k++) {
      const int i4 = tid + 256 * k;
      g[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i4 < H4) {
        const uint2 gv = *(const uint2*)(gain + i4 * 4);
        g[k] = make_float4(bf16lo(gv.x), bf16hi(gv.x), bf16lo(gv.y), bf16hi(gv.y));
      }
    }
    for (int n0 = 0; n0 < B; n0 += TB) {
      float4 h[TB][NI];
#pragma unroll
      for (int b = 0; b < TB; b++)
#pragma unroll
        for (int k = 0; k < NI; k++) {
          const int n = n0 + b, i4 = tid + 256 * k;
          h[b][k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (n < B && i4 < H4) {
            if (final_norm) {
              const float4 a = __ldcg((const float4*)(hl + n * H) + i4);
              const float4 d = delta4(l - 1, n, i4);
              h[b][k] = make_float4(a.x + d.x, a.y + d.y, a.z + d.z, a.w + d.w);
            } else {
              h[b][k] = __ldcg((const float4*)(hl + n * H) + i4);
            }
          }
        }
#pragma unroll
      for (int b = 0; b < TB; b++) {
        const int n = n0 + b;
        if (n >= B) break;
        const float r = S.rinv[n];
#pragma unroll
        for (int k = 0; k < NI; k++) {
          const int i4 = tid + 256 * k;
          if (i4 < H4) {
            const float4 x = make_float4(h[b][k].x * r * g[k].x, h[b][k].y * r * g[k].y, h[b][k].z * r * g[k].z,
                                         h[b][k].w * r * g[k].w);
            __stcg((float4*)(xl + n * H) + i4, x);
            if (keep) __stcg((float4*)(p.xdbg + ((size_t)l * Bm + n) * H) + i4, x);
          }
        }
      }
    }
    return csync();
  }

  // one token: stage the O-proj's input (the attention output) in shared
  // memory, one coalesced global read per block instead of one per warp
  __device__ __forceinline__ bool stage_x() {
    const int l = t[R_LAYER];
    const size_t Bm = (size_t)p.Bmax;
    {
      const int n4 = p.hq * p.d / 4;
      const float4* src = (const float4*)(p.attn_out + (size_t)l * Bm * p.hq * p.d);
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = tid + 256 * k;
        v[k] = i < n4 ? __ldcg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = tid + 256 * k;
        if (i < n4) *(float4*)&S.xs[i * 4] = v[k];
      }
    }
    return csync();
  }

  // ------------------------------------------------------ GEMV chunk
  // y[row][n] = sum_k W[row][k] x[n][k] over whole rows streamed a stage at a
  // time.  The contraction is cut into 256-column segments; warp w serves
  // segment w % nsegp (+ nsegp, ...) of rows w / nsegp, + wps, ...; lane l
  // multiplies columns seg * 256 + 8 l .. + 8 against fp32 activations held in
  // registers.  RB rows x NB tokens run as independent FMA chains and are
  // reduced across the warp together (transposed butterfly: 9 shuffles for 8
  // sums).  Tokens beyond NB take further passes over the staged rows.
  template <int NB>
  __device__ __forceinline__ bool gemv(float* part) {
    constexpr int NSG = NB <= 4 ? 2 : 1;           // segments per warp held in registers
    constexpr int RB = 8 / NB;                     // rows per independent group (RB * NB = 8)
    const int K = t[R_K];
    const int nt = t[R_NT];
    const int nrows = t[R_NROWS], nblk = t[R_NBLK];
    const int rps = rows_per_stage(K);
    const int ksg = K < 256 ? K : 256;
    const int nseg = K / ksg;
    const int nsegp = nseg < 8 ? nseg : 8;         // warps sharing one row's segments
    const int wps = 8 / nsegp;                     // warps per segment slot
    const bool active = warp < nsegp * wps;
    const int nsg = (nseg + nsegp - 1) / nsegp;    // segments per warp
    const bool lane_on = lane * 8 < ksg;
    const int seg0 = warp % nsegp;
    const int rwarp = warp / nsegp;
    const int npass = (nt + NB - 1) / NB;

    float xr[NSG][NB][8];
    auto load_x = [&](int sg_first, int pass) {
#pragma unroll
      for (int q = 0; q < NSG; q++) {
        const int seg = seg0 + (sg_first + q) * nsegp;
#pragma unroll
        for (int b = 0; b < NB; b++) {
          const int n = pass * NB + b;
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
          if (active && seg < nseg && lane_on && n < nt) {
            const float* row = xrow(n);
            a = __ldcg((const float4*)(row + seg * ksg + lane * 8));
            c = __ldcg((const float4*)(row + seg * ksg + lane * 8 + 4));
          }
          xr[q][b][0] = a.x; xr[q][b][1] = a.y; xr[q][b][2] = a.z; xr[q][b][3] = a.w;
          xr[q][b][4] = c.x; xr[q][b][5] = c.y; xr[q][b][6] = c.z; xr[q][b][7] = c.w;
        }
      }
    };
    const bool keep = npass == 1 && nsg <= NSG;    // activations loaded once per chunk
    if (keep) load_x(0, 0);

    int tile_row0 = 0;
    for (int blk = 0; blk < nblk; blk++) {
      for (int done = 0; done < nrows; done += rps) {
        const int rows = min(rps, nrows - done);
        uint32_t slot;
        if (!stage_full(slot)) return false;
        if (TR && tid == 0 && blk == 0 && done == 0) S.t_mark[0] = gtime_ns();
        const uint8_t* base = S.stage[slot];
        for (int pass = 0; pass < npass; pass++) {
          for (int sg0 = 0; sg0 < nsg; sg0 += NSG) {
            if (!keep) load_x(sg0, pass);
#pragma unroll
            for (int q = 0; q < NSG; q++) {
              const int seg = seg0 + (sg0 + q) * nsegp;
              if (!(active && seg < nseg)) continue;
              for (int r0 = rwarp; r0 < rows; r0 += RB * wps) {
                float v[8];
                {
                  uint4 wv[RB];
#pragma unroll
                  for (int rr = 0; rr < RB; rr++) {
                    const int r = r0 + rr * wps;
                    wv[rr] = (lane_on && r < rows) ? lds128(base + ((size_t)r * K + seg * ksg + lane * 8) * 2)
                                                   : make_uint4(0, 0, 0, 0);
                  }
#pragma unroll
                  for (int rr = 0; rr < RB; rr++) {
                    const float w8[8] = {bf16lo(wv[rr].x), bf16hi(wv[rr].x), bf16lo(wv[rr].y),
                                         bf16hi(wv[rr].y), bf16lo(wv[rr].z), bf16hi(wv[rr].z),
                                         bf16lo(wv[rr].w), bf16hi(wv[rr].w)};
#pragma unroll
                    for (int b = 0; b < NB; b++) {
                      float a = 0.f;
#pragma unroll
                      for (int j = 0; j < 8; j++) a = fmaf(w8[j], xr[q][b][j], a);
                      v[rr * NB + b] = a;
                    }
                  }
                }
                // transposed butterfly over the 8 sums v[i] = (row i / NB, token i % NB)
#pragma unroll
                for (int i = 0; i < 4; i++) {
                  const bool up = lane & 16;
                  const float send = up ? v[i] : v[i + 4];
                  const float keepv = up ? v[i + 4] : v[i];
                  v[i] = keepv + __shfl_xor_sync(0xffffffffu, send, 16);
                }
#pragma unroll
                for (int i = 0; i < 2; i++) {
                  const bool up = lane & 8;
                  const float send = up ? v[i] : v[i + 2];
                  const float keepv = up ? v[i + 2] : v[i];
                  v[i] = keepv + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                {
                  const bool up = lane & 4;
                  const float send = up ? v[0] : v[1];
                  const float keepv = up ? v[1] : v[0];
                  v[0] = keepv + __shfl_xor_sync(0xffffffffu, send, 4);
                }
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
                if ((lane & 3) == 0) {
                  const int i = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
                  const int rr = i / NB, n = pass * NB + i % NB;
                  const int r = r0 + rr * wps;
                  if (r < rows && n < nt) part[((tile_row0 + done + r) * nseg + seg) * nt + n] = v[0];
                }
              }
            }
          }
        }
        stage_release(slot);
      }
      tile_row0 += nrows;
    }
    if (TR && tid == 0) S.t_mark[1] = gtime_ns();
    return true;
  }

  // -------------------------------- several tokens, expert chunks, tensor cores
  // Both write one fp32 partial per (row, warp, token) to part[(row * 8 +
  // warp) * nt + token]: the epilogue adds a row's eight warp partials in warp
  // order (as it adds the CUDA-core path's segment partials).
  //
  // Rows of K = 2048 NH columns with nt <= 8 / NH tokens (dense rows, or an
  // expert's gate and up rows: R_NBLK groups), stages as in the one-token
  // GEMV (R = 8 / NH rows x every column block, swizzled): the M side is
  // (row m % R, part m / R) of the warp's 256 NH columns in P = 2 NH parts,
  // the N side column n = 8 q + g of n-tile q holds token q (8 / (4 NH))
  // + g / (4 NH), part (g / 2) % P, high or low half g % 2 of x.  C[m][n] is
  // kept where the parts match; the lanes holding a token's parts of a row
  // are added (quad shuffles; with R = 4 also the two quads of a row).
  // (NQ: n-tiles in use, 1..4, fixed at compile time so that the unrolled
  // loops carry no per-tile predicates)
  template <int NH, int NQ>
  __device__ __forceinline__ bool gemv_mma_multi(float* part) {
    constexpr int R = 8 / NH, TPT = 2 / NH;       // rows per stage, tokens per n-tile
    const int nt = t[R_NT], nr = t[R_NROWS], nblk = t[R_NBLK];
    constexpr int nq = NQ;
    uint32_t xb[4][8][2];
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const int tk = q * TPT + gl / (4 * NH), j = (gl >> 1) & (2 * NH - 1), lo = gl & 1;
      const bool on = q < nq && tk < nt;
      const float* xr = on ? xrow(tk) : nullptr;
#pragma unroll
      for (int s = 0; s < 8; s++)
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
          float2 v = make_float2(0.f, 0.f);
          if (on) v = __ldcg((const float2*)(xr + mma_block<NH>(j, s >> 2) * 64 + (s & 3) * 16 + hf * 8 + 2 * cq));
          if (lo) v = make_float2(v.x - bf16f(f2bf(v.x)), v.y - bf16f(f2bf(v.y)));
          xb[q][s][hf] = pack_bf2(v.x, v.y);
        }
    }
    uint32_t aoff[8];
    {
      const int m = ((lane >> 3) & 1) * 8 + (lane & 7), kh = lane >> 4;
#pragma unroll
      for (int s = 0; s < 8; s++) {
        const int line = mma_block<NH>(m / R, s >> 2) * R + (m % R);
        aoff[s] = (uint32_t)(line * 128 + ((((s & 3) * 2 + kh) ^ (line & 7)) << 4));
      }
    }
    // this lane's part of the n-tile's columns 2 cq, 2 cq + 1, and the parts of
    // its M rows g (part g / R) and g + 8 (part (g + 8) / R)
    const int pc = cq & (2 * NH - 1), j0 = gl / R, j1 = (gl + 8) / R;
    for (int blk = 0; blk < nblk; blk++) {
      for (int done = 0; done < nr; done += R) {
        const int rows = min(R, nr - done);
        uint32_t slot;
        if (!stage_full(slot)) return false;
        if (TR && tid == 0 && blk == 0 && done == 0) S.t_mark[0] = gtime_ns();
        const uint8_t* base = S.stage[slot];
        float c[4][4];
#pragma unroll
        for (int q = 0; q < 4; q++) c[q][0] = c[q][1] = c[q][2] = c[q][3] = 0.f;
#pragma unroll
        for (int s = 0; s < 8; s++) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(a0, a1, a2, a3, base + aoff[s]);
#pragma unroll
          for (int q = 0; q < 4; q++)
            if (q < nq) mma_bf16(c[q], a0, a1, a2, a3, xb[q][s][0], xb[q][s][1]);
        }
        stage_release(slot);
#pragma unroll
        for (int q = 0; q < 4; q++) {
          if (q >= nq) break;
          float v = (pc == j0 ? c[q][0] + c[q][1] : 0.f) + (pc == j1 ? c[q][2] + c[q][3] : 0.f);
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          if (NH == 2) {
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
          }
          // NH = 1: lanes cq = 0, 2 hold tokens 2 q, 2 q + 1 of row g; NH = 2:
          // lane cq = 0 of quads g < 4 holds token q of row g
          const int tk = q * TPT + (NH == 1 ? (cq >> 1) : 0);
          const bool writer = NH == 1 ? !(cq & 1) : (cq == 0 && gl < R);
          if (writer && gl < rows && tk < nt)
            part[((blk * nr + done + gl) * kConsumerWarps + warp) * nt + tk] = v;
        }
      }
    }
    if (TR && tid == 0) S.t_mark[1] = gtime_ns();
    return true;
  }

  // Down rows of an expert (K = I, a multiple of 128 up to 1024), stages of 16
  // rows x every column block (swizzled, line 16 cb + r): the M side is the 16
  // rows, the K side the warp's I / 8 columns, the N side column n = 8 q + g
  // holds token 4 q + g / 2, high or low half g % 2 of its hidden vector.
  template <int NQ>
  __device__ __forceinline__ bool gemv_mma_down(float* part) {
    const int K = t[R_K], nt = t[R_NT], nr = t[R_NROWS];
    const int ks = K >> 7;                        // k-steps per warp (<= 8)
    constexpr int nq = NQ;                        // n-tiles: four tokens each
    const int col0 = warp * (K >> 3);
    uint32_t xb[4][8][2];
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const int tk = 4 * q + (gl >> 1), lo = gl & 1;
      const bool on = q < nq && tk < nt;
      const float* xr = on ? xrow(tk) : nullptr;
#pragma unroll
      for (int s = 0; s < 8; s++)
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
          float2 v = make_float2(0.f, 0.f);
          if (on && s < ks) v = __ldcg((const float2*)(xr + col0 + 16 * s + 8 * hf + 2 * cq));
          if (lo) v = make_float2(v.x - bf16f(f2bf(v.x)), v.y - bf16f(f2bf(v.y)));
          xb[q][s][hf] = pack_bf2(v.x, v.y);
        }
    }
    uint32_t aoff[8];
    {
      const int m = ((lane >> 3) & 1) * 8 + (lane & 7), kh = lane >> 4;
#pragma unroll
      for (int s = 0; s < 8; s++) {
        const int col = col0 + 16 * s + 8 * kh;
        const int line = (col >> 6) * kDownBoxRows + m;
        aoff[s] = (uint32_t)(line * 128 + ((((col & 63) >> 3) ^ (line & 7)) << 4));
      }
    }
    for (int done = 0; done < nr; done += kDownBoxRows) {
      uint32_t slot;
      if (!stage_full(slot)) return false;
      if (TR && tid == 0 && done == 0) S.t_mark[0] = gtime_ns();
      const uint8_t* base = S.stage[slot];
      float c[4][4];
#pragma unroll
      for (int q = 0; q < 4; q++) c[q][0] = c[q][1] = c[q][2] = c[q][3] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; s++) {
        if (s >= ks) break;
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a0, a1, a2, a3, base + aoff[s]);
#pragma unroll
        for (int q = 0; q < 4; q++)
          if (q < nq) mma_bf16(c[q], a0, a1, a2, a3, xb[q][s][0], xb[q][s][1]);
      }
      stage_release(slot);
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const int tk = 4 * q + cq;
        if (q < nq && tk < nt) {
          if (done + gl < nr) part[((done + gl) * kConsumerWarps + warp) * nt + tk] = c[q][0] + c[q][1];
          if (done + gl + 8 < nr) part[((done + gl + 8) * kConsumerWarps + warp) * nt + tk] = c[q][2] + c[q][3];
        }
      }
    }
    if (TR && tid == 0) S.t_mark[1] = gtime_ns();
    return true;
  }

  // ------------------------------------------------ one-token GEMV chunk
  // Row r of the chunk (rows numbered across its groups) belongs to warp
  // r % 8, which computes the whole row: lane l multiplies the 8-column
  // chunks l, l + 32, ... (consecutive 16-byte shared-memory reads across the
  // warp) against x in registers, then one warp reduction gives res[r].  No
  // cross-warp partial sums.  The activations are in shared memory (xs).
  __device__ __forceinline__ int row_groups() const {
    const int kind = t[R_KIND];
    return (kind == K_P1 || kind == K_UP) ? 2 : 1;
  }
  __device__ __forceinline__ int group_rows(int g) const {
    return (t[R_KIND] == K_P1 && g == 1) ? t[R_NROWS1] : t[R_NROWS];
  }
  template <int NCK>
  __device__ __forceinline__ void row_load_x(float (&x)[NCK][8], const float* src, int K) const {
#pragma unroll
    for (int c = 0; c < NCK; c++) {
      const int col = (lane + 32 * c) * 8;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (col < K) {
        a = *(const float4*)(src + col);
        b = *(const float4*)(src + col + 4);
      }
      x[c][0] = a.x; x[c][1] = a.y; x[c][2] = a.z; x[c][3] = a.w;
      x[c][4] = b.x; x[c][5] = b.y; x[c][6] = b.z; x[c][7] = b.w;
    }
  }
  template <int NCK>
  __device__ __forceinline__ bool gemv_row(float* res) {
    const int K = t[R_K];
    const int ngrp = row_groups();
    const int rps = rows_per_stage(K);
    // K is below 256 (one partial chunk per lane) or a multiple of 256 (whole
    // chunks): the chunk test is warp-uniform except in the first case
    const int nch = K >= 256 ? K / 256 : 1;
    const bool lane_on = K >= 256 || lane * 8 < K;
    float xa[NCK][8];
    row_load_x<NCK>(xa, S.xs, K);
    int rbase = 0;
    for (int g = 0; g < ngrp; g++) {
      const int nr = group_rows(g);
      for (int done = 0; done < nr; done += rps) {
        const int rows = min(rps, nr - done);
        uint32_t slot;
        if (!stage_full(slot)) return false;
        if (TR && tid == 0 && rbase + done == 0) S.t_mark[0] = gtime_ns();
        const uint8_t* base = S.stage[slot];
        for (int rr = (warp - (rbase + done) % 8 + 8) % 8; rr < rows; rr += 8) {
          const uint8_t* wrow = base + (size_t)rr * K * 2;
          float2 a = make_float2(0.f, 0.f);     // even / odd columns
#pragma unroll
          for (int c = 0; c < NCK; c++) {
            if (c < nch && lane_on) {
              const uint4 w = lds128(wrow + (lane + 32 * c) * 16);
              a = fma_bf2(w.x, make_float2(xa[c][0], xa[c][1]), a);
              a = fma_bf2(w.y, make_float2(xa[c][2], xa[c][3]), a);
              a = fma_bf2(w.z, make_float2(xa[c][4], xa[c][5]), a);
              a = fma_bf2(w.w, make_float2(xa[c][6], xa[c][7]), a);
            }
          }
          float v = a.x + a.y;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) res[rbase + done + rr] = v;
        }
        stage_release(slot);
      }
      rbase += nr;
    }
    if (TR && tid == 0) S.t_mark[1] = gtime_ns();
    return true;
  }

  // one token, rows of K = 2048 NH columns on the tensor cores (mma.sync
  // m16n8k16, BF16 in, fp32 accumulate).  A stage holds R = 8 / NH rows as
  // [K / 64 column blocks][R rows][64 columns], swizzled (rotated_rows).  Warp
  // w takes column blocks [4 NH w, 4 NH w + 4 NH) of every row, cut into
  // P = 2 NH parts of two blocks: the MMA's M side is (row m % R, part m / R),
  // its K side 16 columns of that part, its N side the activation: column
  // n = 2 j + t holds the BF16 high (t = 0) or low (t = 1) half of x over part
  // j, so every product keeps about 16 bits of x.  C[m][n] is the part's dot
  // product where n matches m's part; the lanes holding a row's parts are
  // added (quad shuffles; with R = 4 also the two quads of a row), and the
  // eight warp sums of a row meet in shared memory (spart, [row][warp]),
  // added in warp order after the barrier.  With R = 4 the parts take every
  // other block (parts 2 q and 2 q + 1 differ in block parity) so that the
  // eight rows of an ldmatrix tile lie in distinct 128-byte lines mod 8.
  template <int NH>
  __device__ __forceinline__ int mma_block(int j, int t) const {
    return NH == 1 ? 4 * warp + 2 * j + t : 8 * warp + 4 * (j >> 1) + 2 * t + (j & 1);
  }

  template <int NH>
  __device__ __forceinline__ bool gemv_mma(float* res) {
    constexpr int R = 8 / NH;                     // rows per stage
    const int ngrp = row_groups();
    // B fragments (x as k x n) for the 8 k-steps of the warp's parts: lane
    // (gl, cq) holds column n = gl, rows 2 cq, 2 cq + 1 and 8 + 2 cq, 9 + 2 cq
    uint32_t xb[8][2];
    {
      const int j = gl >> 1, lo = gl & 1;
      const bool on = j < 2 * NH;
#pragma unroll
      for (int s = 0; s < 8; s++) {
        const float* xs = S.xs + mma_block<NH>(j, s >> 2) * 64 + (s & 3) * 16 + 2 * cq;
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
          float2 v = on ? *(const float2*)(xs + hf * 8) : make_float2(0.f, 0.f);
          if (lo) v = make_float2(v.x - bf16f(f2bf(v.x)), v.y - bf16f(f2bf(v.y)));
          xb[s][hf] = pack_bf2(v.x, v.y);
        }
      }
    }
    // ldmatrix rows of this lane: tile i = lane / 8 holds M rows (i & 1) * 8 +
    // 0..7, columns 8 (i >> 1) .. + 7 of the k-step; lane & 7 is the M row
    uint32_t aoff[8];
    {
      const int m = ((lane >> 3) & 1) * 8 + (lane & 7), r = m % R, j = m / R, kh = lane >> 4;
#pragma unroll
      for (int s = 0; s < 8; s++) {
        const int line = mma_block<NH>(j, s >> 2) * R + r;
        aoff[s] = (uint32_t)(line * 128 + ((((s & 3) * 2 + kh) ^ (line & 7)) << 4));
      }
    }
    // C entries this lane keeps: M row gl is part gl / R, row gl + 8 part (gl + 8) / R
    const int j0 = gl / R, j1 = (gl + 8) / R;
    float* part = &S.spart[0][0];
    int rbase = 0;
    for (int g = 0; g < ngrp; g++) {
      const int nr = group_rows(g);
      for (int done = 0; done < nr; done += R) {
        const int rows = min(R, nr - done);
        uint32_t slot;
        if (!stage_full(slot)) return false;
        if (TR && tid == 0 && rbase + done == 0) S.t_mark[0] = gtime_ns();
        const uint8_t* base = S.stage[slot];
        float ca[4] = {0.f, 0.f, 0.f, 0.f}, cc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 8; s++) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(a0, a1, a2, a3, base + aoff[s]);
          mma_bf16((s & 1) ? cc : ca, a0, a1, a2, a3, xb[s][0], xb[s][1]);
        }
        stage_release(slot);
        float v = (cq == j0 ? (ca[0] + cc[0]) + (ca[1] + cc[1]) : 0.f) +
                  (cq == j1 ? (ca[2] + cc[2]) + (ca[3] + cc[3]) : 0.f);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (R == 4) v += __shfl_xor_sync(0xffffffffu, v, 16);
        if (cq == 0 && gl < rows) part[(rbase + done + gl) * kConsumerWarps + warp] = v;
      }
      rbase += nr;
    }
    if (TR && tid == 0) S.t_mark[1] = gtime_ns();
    if (!csync()) return false;
    if (tid < rbase) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; w++) v += part[tid * kConsumerWarps + w];
      res[tid] = v;
    }
    return true;
  }

  // 8-bit experts: a vector v as four E4M3 terms, v ~ sum_t s_t q_t with
  // s_t = s_0 16^-t and s_0 the power of two with max|v| / s_0 <= 448: term t
  // rounds the remainder r_t / s_t to nearest (r_0 = v, r_{t+1} = r_t -
  // s_t q_t), so each term adds about four bits (the remainder of a term
  // is at most half its largest step, 16 s_t) and four terms keep x to about
  // 16 bits of its largest element, as BF16 high + low halves would.  The
  // terms are the N columns of E4M3 tensor-core products.
  __device__ __forceinline__ static float e4m3_scale0(float mx) {
    const float y = mx / 448.f;
    if (!(y > 0.f)) return 1.f;
    int e = ((__float_as_int(y) >> 23) & 0xff) - 127;
    if (__float_as_int(y) & 0x7fffff) e++;           // round the exponent up unless a power of two
    e = max(-126, min(127, e));
    return __int_as_float((e + 127) << 23);
  }
  __device__ __forceinline__ static void e4m3_terms(float v, float s0, uint8_t (&q)[4]) {
#pragma unroll
    for (int t = 0; t < 4; t++) {
      const float st = s0 * __int_as_float((127 - 4 * t) << 23);     // s_0 16^-t
      const float inv = 1.f / st;                                     // a power of two: exact
      q[t] = f2e4m3(v * inv);
      v -= st * e4m3f(q[t]);
    }
  }

  // the layer's x / rms as E4M3 terms in the top quarter of xs ([4][H] bytes),
  // once per layer on this SM (every UP piece of the layer reads them); s0:
  // their first scale (every thread computes it from the same maximum; a
  // later piece reads the copy the first one left, ordered by the barriers
  // between the tasks)
  __device__ __forceinline__ bool stage_xq(float& s0) {
    const int l = t[R_LAYER], H = p.H;
    if (S.xq_layer == l) {
      s0 = S.xq_s0;
      return true;
    }
    const float rinv = S.rinv[0];
    float mx = 0.f;
    for (int k = tid; k < H; k += 256) mx = fmaxf(mx, fabsf(S.xs[k] * rinv));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) S.nred[warp][0] = mx;
    if (!csync()) return false;
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; w++) mx = fmaxf(mx, S.nred[w][0]);
    s0 = e4m3_scale0(mx);
    uint8_t* xq = (uint8_t*)(S.xs + kXsFloats * 3 / 4);
    for (int k = tid; k < H; k += 256) {
      uint8_t q[4];
      e4m3_terms(S.xs[k] * rinv, s0, q);
#pragma unroll
      for (int tt = 0; tt < 4; tt++) xq[tt * H + k] = q[tt];
    }
    if (!csync()) return false;
    if (tid == 0) {
      S.xq_s0 = s0;
      S.xq_layer = l;
    }
    return true;
  }

  // one token, 8-bit expert rows (E4M3) of K = 2048 columns on the tensor
  // cores: mma.sync m16n8k32 with both operands E4M3 and fp32 accumulation.
  // A stage holds 16 rows, copied as rows of 1024 two-byte words: column
  // block cb (128 bytes) of row r is the 128-byte line 16 cb + r, its 16-byte
  // chunk c stored at chunk c ^ (r & 7).  Warp w takes blocks 2 w and 2 w + 1
  // (columns [256 w, 256 w + 256)): eight k-steps of 32 columns, each one
  // ldmatrix of four 8 x 16-byte tiles (rows 0-7 / 8-15 x two chunks), which
  // are exactly the A fragment, and one MMA.  N side: column t < 4 holds the
  // x term t (stage_xq), so C[m][t] s_t summed over t is row m's dot product
  // with x / rms.  The eight warps' sums of a row meet in shared memory
  // (spart) and are added in warp order; the row scales are applied by the
  // epilogue.
  __device__ __forceinline__ bool gemv_mma_e4m3(float* res) {
    const int ngrp = row_groups(), H = p.H;
    float s0;
    if (!stage_xq(s0)) return false;
    const uint8_t* xq = (const uint8_t*)(S.xs + kXsFloats * 3 / 4);
    // this lane's term scales (columns 2 cq, 2 cq + 1; terms 4.. are absent)
    const float sa = cq < 2 ? s0 * __int_as_float((127 - 8 * cq) << 23) : 0.f;
    const float sb = cq < 2 ? s0 * __int_as_float((127 - 8 * cq - 4) << 23) : 0.f;
    uint32_t xb[8][2];
#pragma unroll
    for (int st = 0; st < 8; st++) {
      const int k0 = 256 * warp + 32 * st + 4 * cq;
      xb[st][0] = gl < 4 ? *(const uint32_t*)(xq + gl * H + k0) : 0u;
      xb[st][1] = gl < 4 ? *(const uint32_t*)(xq + gl * H + k0 + 16) : 0u;
    }
    uint32_t aoff[8];
    {
      const int r = ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
      for (int st = 0; st < 8; st++) {
        const int ch = 2 * st + (lane >> 4);
        const int line = (2 * warp + (ch >> 3)) * 16 + r;
        aoff[st] = (uint32_t)(line * 128 + (((ch & 7) ^ (r & 7)) << 4));
      }
    }
    float* part = &S.spart[0][0];
    int rbase = 0;
    for (int g = 0; g < ngrp; g++) {
      const int nr = group_rows(g);
      for (int done = 0; done < nr; done += 16) {
        const int rows = min(16, nr - done);
        uint32_t slot;
        if (!stage_full(slot)) return false;
        if (TR && tid == 0 && rbase + done == 0) S.t_mark[0] = gtime_ns();
        const uint8_t* base = S.stage[slot];
        float ca[4] = {0.f, 0.f, 0.f, 0.f}, cc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int st = 0; st < 8; st++) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(r0, r1, r2, r3, base + aoff[st]);
          mma_e4m3((st & 1) ? cc : ca, r0, r1, r2, r3, xb[st][0], xb[st][1]);
        }
        stage_release(slot);
        float v0 = sa * (ca[0] + cc[0]) + sb * (ca[1] + cc[1]);      // row gl
        float v8 = sa * (ca[2] + cc[2]) + sb * (ca[3] + cc[3]);      // row gl + 8
        v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
        v8 += __shfl_xor_sync(0xffffffffu, v8, 1);
        if (cq == 0) {
          if (gl < rows) part[(rbase + done + gl) * kConsumerWarps + warp] = v0;
          if (gl + 8 < rows) part[(rbase + done + gl + 8) * kConsumerWarps + warp] = v8;
        }
      }
      rbase += nr;
    }
    if (TR && tid == 0) S.t_mark[1] = gtime_ns();
    if (!csync()) return false;
    if (tid < rbase) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; w++) v += part[tid * kConsumerWarps + w];
      res[tid] = v;
    }
    return true;
  }

  // one token, 8-bit expert rows of K <= 1024 columns on the CUDA cores: row r
  // of the chunk belongs to warp r % 8; lane l multiplies the 16-column chunks
  // l, l + 32, ... (16 bytes each) against x / rms in registers, then one warp
  // reduction.  NCK: 16-byte chunks per lane (K <= 512 NCK).
  template <int NCK>
  __device__ __forceinline__ bool gemv_row_e4m3(float* res) {
    const int K = t[R_K];
    const int ngrp = row_groups();
    const int rps = rows_per_stage(K / 2);
    const float rinv = S.rinv[0];
    float xa[NCK][16];
#pragma unroll
    for (int c = 0; c < NCK; c++) {
      const int col = (lane + 32 * c) * 16;
#pragma unroll
      for (int j = 0; j < 16; j++) xa[c][j] = col < K ? S.xs[col + j] * rinv : 0.f;
    }
    int rbase = 0;
    for (int g = 0; g < ngrp; g++) {
      const int nr = group_rows(g);
      for (int done = 0; done < nr; done += rps) {
        const int rows = min(rps, nr - done);
        uint32_t slot;
        if (!stage_full(slot)) return false;
        if (TR && tid == 0 && rbase + done == 0) S.t_mark[0] = gtime_ns();
        const uint8_t* base = S.stage[slot];
        for (int rr = (warp - (rbase + done) % 8 + 8) % 8; rr < rows; rr += 8) {
          const uint8_t* wrow = base + (size_t)rr * K;
          float2 a = make_float2(0.f, 0.f);     // even / odd columns
#pragma unroll
          for (int c = 0; c < NCK; c++) {
            if ((lane + 32 * c) * 16 < K) {
              const uint4 w = lds128(wrow + (lane + 32 * c) * 16);
              const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int q = 0; q < 4; q++) {
                const float2 f0 = f16x2_to_float2(e4m3x2_to_f16x2(wd[q]));
                const float2 f1 = f16x2_to_float2(e4m3x2_to_f16x2(wd[q] >> 16));
                a = __ffma2_rn(f0, make_float2(xa[c][4 * q], xa[c][4 * q + 1]), a);
                a = __ffma2_rn(f1, make_float2(xa[c][4 * q + 2], xa[c][4 * q + 3]), a);
              }
            }
          }
          float v = a.x + a.y;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) res[rbase + done + rr] = v;
        }
        stage_release(slot);
      }
      rbase += nr;
    }
    if (TR && tid == 0) S.t_mark[1] = gtime_ns();
    return true;
  }

  // epilogue of a one-token chunk (after the barrier); token 0 throughout
  // (8-bit experts, K_UP: sg_t, su_t = the gate / up scales of row tid)
  template <bool F8 = false>
  __device__ __forceinline__ void epilogue_row(const float* res, float sg_t = 0.f, float su_t = 0.f) {
    const int l = t[R_LAYER], kind = t[R_KIND];
    const int nr = t[R_NROWS], row0 = t[R_ROW0];
    const size_t Bm = (size_t)p.Bmax;
    switch (kind) {
      case K_P1: {   // GEMV of h * gain: scale by 1 / rms
        const int nq = t[R_NROWS1], q0 = t[R_ROW1];
        const float r = S.rinv[0];
        for (int i = tid; i < nr + nq; i += 256) {
          if (i < nr) __stcg(p.rlog + (size_t)l * Bm * p.E + row0 + i, res[i] * r);
          else __stcg(p.qkv + (size_t)l * Bm * p.qkv_rows + q0 + i - nr, res[i] * r);
        }
        break;
      }
      case K_UP: {
        // the hidden values of the piece; times the routing weight, they are
        // the input of the piece's down-projection columns
        const int slot = S.rt.off[t[R_A]];
        const float wa = S.rt.w[0][S.rt.ent[slot] % p.topk];
        const float r = S.rinv[0];   // GEMV of h * gain: scale by 1 / rms
        // 8-bit experts: the GEMV took x / rms; each row times its scale
        // (a piece has at most 64 rows: row i is thread i's)
        for (int i = tid; i < nr; i += 256) {
          const float a = F8 ? silu_mul(res[i] * sg_t, res[nr + i] * su_t)
                                : silu_mul(res[i] * r, res[nr + i] * r);
          __stcg(p.abuf + ((size_t)l * Bm * p.topk + slot) * p.I + row0 + i, a);
          S.actp[i] = wa * a;
        }
        break;
      }
      case K_OPROJ:
        for (int i = tid; i < nr; i += 256) __stcg(p.oproj + (size_t)l * Bm * p.H + row0 + i, res[i]);
        break;
      default: {   // K_LM: GEMV of h * gain, scale by 1 / rms
        const float r = S.rinv[0];
        for (int i = tid; i < nr; i += 256) p.logits[row0 + i] = res[i] * r;
        break;
      }
    }
  }

  // one token, after the gate/up rows of an UP piece: its n = ncb groups of
  // the down projection, each group's [H][8] block in stages of up to 2048
  // rows.  Thread t takes rows t, t + 256, ... of the stage (consecutive
  // 16-byte reads) and writes the group's partial of each:
  //   mpart[g][h] = sum_{c < 8} W_down[e][h][8 g' + c] * w_e * act[8 g' + c]
  // (even and odd c summed apart, then added)
  __device__ __forceinline__ bool down_part() {
    const int H = p.H, ncb = t[R_NROWS] / 8, g0 = t[R_REL0];
    for (int c = 0; c < ncb; c++) {
      float xa[8];
#pragma unroll
      for (int j = 0; j < 8; j++) xa[j] = S.actp[8 * c + j];
      for (int r0 = 0; r0 < H; r0 += kDownRows) {
        const int rows = min(kDownRows, H - r0);
        uint32_t slot;
        if (!stage_full(slot)) return false;
        const uint8_t* st = S.stage[slot];
        for (int r = tid; r < rows; r += 256) {
          const uint4 w = lds128(st + r * 16);
          float2 a = __fmul2_rn(make_float2(bf16lo(w.x), bf16hi(w.x)), make_float2(xa[0], xa[1]));
          a = fma_bf2(w.y, make_float2(xa[2], xa[3]), a);
          a = fma_bf2(w.z, make_float2(xa[4], xa[5]), a);
          a = fma_bf2(w.w, make_float2(xa[6], xa[7]), a);
          __stcg(p.mpart + (size_t)(g0 + c) * H + r0 + r, a.x + a.y);
        }
        stage_release(slot);
      }
    }
    return true;
  }

  // The 8-bit down projection of an UP piece on the tensor cores (mma.sync
  // m16n8k32, E4M3 x E4M3, fp32 accumulate).  The piece's weighted hidden
  // values (S.actp, 8 per group) are first cut into four E4M3 terms (as x is
  // by stage_xq; kept in spart).  Its groups arrive as quads of up to four
  // groups, a stage holding the quad's rows [hb, hb + rd) (group slot j at
  // j rd 8 bytes, 8 bytes a row).  One MMA takes 16 rows (M) and the quad's 32
  // columns (K): lane (gl, cq) gives the 4 bytes of columns 4 (cq & 1) .. + 3
  // of group slot cq >> 1 (k 4 cq .. 4 cq + 3) and of slot 2 + (cq >> 1) (k 16
  // + 4 cq ..) in rows h0 + gl and h0 + gl + 8; the B fragment holds the
  // hidden terms of the same columns (N column t = term t).  (Each pair of
  // row loads swaps rows between the two groups' lanes, so the 32 lanes'
  // words fall in distinct banks.)  Warp w keeps its 16-row blocks h0 =
  // 16 (w + 8 i) over the piece's stages; the piece's total, times the row's
  // scale s_down[e][h] (staged in xs by op_row), goes to its first group's
  // partial row, zeros to its other groups' rows.
  __device__ __forceinline__ bool down_mma_e4m3() {
    constexpr int kMaxBlk = 16;                   // 16-row blocks a warp (H <= 2048)
    const int H = p.H, ncb = t[R_NROWS] / 8, g0 = t[R_REL0], nr = t[R_NROWS];
    const int nb = H / 128, rd = min(H, 1024);
    const float* scl = S.xs + kXsFloats / 2;
    uint8_t* aq = (uint8_t*)&S.spart[0][0];       // [4][64] hidden terms
    // the hidden values' terms (threads < nr: one value each)
    {
      const float v = tid < nr ? S.actp[tid] : 0.f;
      float mx = fabsf(v);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0 && warp < 2) S.nred[warp][1] = mx;
      if (!csync()) return false;
      const float s0 = e4m3_scale0(fmaxf(S.nred[0][1], S.nred[1][1]));
      if (tid < 64) {
        uint8_t q[4];
        e4m3_terms(v, s0, q);                     // v = 0 past nr: zero terms
#pragma unroll
        for (int tt = 0; tt < 4; tt++) aq[tt * 64 + tid] = q[tt];
      }
      if (tid == 0) S.aq_s0 = s0;
      if (!csync()) return false;
    }
    const float s0 = S.aq_s0;
    const float sa = cq < 2 ? s0 * __int_as_float((127 - 8 * cq) << 23) : 0.f;
    const float sb = cq < 2 ? s0 * __int_as_float((127 - 8 * cq - 4) << 23) : 0.f;
    const int g1 = cq >> 1, wsel = 4 * (cq & 1);
    float acc[kMaxBlk][4];
#pragma unroll
    for (int i = 0; i < kMaxBlk; i++) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    for (int q0 = 0; q0 < ncb; q0 += 4) {
      const int nq = min(4, ncb - q0);
      const bool onl = g1 < nq, onh = 2 + g1 < nq;    // this lane's two group slots are present
      // B: hidden terms of columns (slot g1, 4 (cq & 1) ..) and (slot 2 + g1, ..)
      const uint32_t b0 = gl < 4 && onl ? *(const uint32_t*)(aq + gl * 64 + (q0 + g1) * 8 + wsel) : 0u;
      const uint32_t b1 = gl < 4 && onh ? *(const uint32_t*)(aq + gl * 64 + (q0 + 2 + g1) * 8 + wsel) : 0u;
      // one 16-row block: its four row words and the MMA
      auto block = [&](const uint8_t* sl, const uint8_t* sh, int r, float* a) {
        const int ra = 8 * (r + gl + 8 * g1), rb = 8 * (r + gl + 8 - 8 * g1);
        const uint32_t la = onl ? *(const uint32_t*)(sl + ra) : 0u, lb = onl ? *(const uint32_t*)(sl + rb) : 0u;
        const uint32_t ha = onh ? *(const uint32_t*)(sh + ra) : 0u, hb2 = onh ? *(const uint32_t*)(sh + rb) : 0u;
        // rows r + gl (a0, a2) and r + gl + 8 (a1, a3) of the stage
        mma_e4m3(a, g1 ? lb : la, g1 ? la : lb, g1 ? hb2 : ha, g1 ? ha : hb2, b0, b1);
      };
      if (H == 2048) {
        // two stages of 1024 rows: blocks 0-7 of the warp in the first, 8-15
        // in the second (h0 = 16 w + 128 i), every index known at compile time
#pragma unroll
        for (int half = 0; half < 2; half++) {
          uint32_t slot;
          if (!stage_full(slot)) return false;
          const uint8_t* sl = S.stage[slot] + (size_t)g1 * 1024 * 8 + wsel;
#pragma unroll
          for (int j = 0; j < 8; j++) block(sl, sl + 2 * 1024 * 8, 16 * warp + 128 * j, acc[8 * half + j]);
          stage_release(slot);
        }
      } else {
        for (int hb = 0; hb < H; hb += rd) {
          uint32_t slot;
          if (!stage_full(slot)) return false;
          const uint8_t* sl = S.stage[slot] + (size_t)g1 * rd * 8 + wsel;          // slot g1
#pragma unroll
          for (int i = 0; i < kMaxBlk; i++) {
            const int h0 = 16 * (warp + 8 * i);
            if (i < nb && h0 >= hb && h0 < hb + rd) block(sl, sl + (size_t)2 * rd * 8, h0 - hb, acc[i]);
          }
          stage_release(slot);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxBlk; i++) {
      if (i < nb) {
        float v0 = sa * acc[i][0] + sb * acc[i][1], v8 = sa * acc[i][2] + sb * acc[i][3];
        v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
        v8 += __shfl_xor_sync(0xffffffffu, v8, 1);
        if (cq == 0) {
          const int h = 16 * (warp + 8 * i) + gl;
          __stcg(p.mpart + (size_t)g0 * H + h, v0 * scl[h]);
          __stcg(p.mpart + (size_t)g0 * H + h + 8, v8 * scl[h + 8]);
        }
      }
    }
    // the other groups' rows: one contiguous run of (ncb - 1) H floats
    float4* z = (float4*)(p.mpart + (size_t)(g0 + 1) * H);
    for (int k = tid; k < (ncb - 1) * H / 4; k += 256) __stcg(z + k, make_float4(0.f, 0.f, 0.f, 0.f));
    return true;
  }

  // one token, DOWN: rows [a0, a1) of the experts' share of the residual
  // update = the sum of every group's partial, in group order.  The partials
  // arrive as stages of 256 groups x kMredCols rows (from row a0 rounded down
  // to a multiple of 4); warp w adds groups w, w + 8, ... and the warps' sums
  // meet in shared memory in warp order.  red: 256 floats of scratch (the
  // task's completion barrier orders its last use).
  __device__ __forceinline__ bool moe_reduce(float* red) {
    const int a0 = t[R_ROW0], a1 = a0 + t[R_NROWS], l = t[R_LAYER];
    const int ng = p.topk * (p.I / 8);
    for (int x0 = a0 & ~3; x0 < a1; x0 += kMredCols) {
      float s = 0.f;
      for (int y0 = 0; y0 < ng; y0 += 256) {
        uint32_t slot;
        if (!stage_full(slot)) return false;
        const float* st = (const float*)S.stage[slot];
        const int n = min(256, ng - y0);
        if (lane < kMredCols)
          for (int g = warp; g < n; g += kConsumerWarps) s += st[g * kMredCols + lane];
        stage_release(slot);
      }
      red[warp * 32 + lane] = s;
      if (!csync()) return false;
      if (tid < kMredCols) {
        const int h = x0 + tid;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; w++) v += red[w * 32 + tid];
        if (h >= a0 && h < a1) __stcg(p.moe + (size_t)l * p.Bmax * p.H + h, v);
      }
      if (x0 + kMredCols < a1 && !csync()) return false;
    }
    return true;
  }

  // fixed-order sum over the contraction segments of element (row, n)
  __device__ __forceinline__ float seg_sum(const float* part, int row, int n, int nseg, int nt) const {
    float s = 0.f;
    for (int sg = 0; sg < nseg; sg++) s += part[(row * nseg + sg) * nt + n];
    return s;
  }

  // reduction + epilogue of a GEMV chunk (after the barrier)
  __device__ __forceinline__ void epilogue(const float* part, int nseg) {
    const int l = t[R_LAYER], kind = t[R_KIND];
    const int nt = t[R_NT], nrows = t[R_NROWS], row0 = t[R_ROW0];
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < nrows * nt; i += 256) {
      const int n = i / nrows, r = i % nrows;
      const float v = seg_sum(part, r, n, nseg, nt);
      switch (kind) {
        case K_ROUTER:
          __stcg(p.rlog + ((size_t)l * Bm + n) * p.E + row0 + r, v);
          break;
        case K_QKV:
          __stcg(p.qkv + ((size_t)l * Bm + n) * p.qkv_rows + row0 + r, v);
          break;
        case K_LM:
          p.logits[(size_t)n * p.V + row0 + r] = v;
          break;
        case K_UP: {
          const float u = seg_sum(part, nrows + r, n, nseg, nt);
          const int slot = S.rt.off[t[R_A]] + n;
          __stcg(p.abuf + ((size_t)l * Bm * p.topk + slot) * p.I + row0 + r, silu_mul(v, u));
          break;
        }
        case K_OPROJ:
          __stcg(p.oproj + ((size_t)l * Bm + n) * p.H + row0 + r, v);
          break;
        default: {   // K_DOWN: entry (token b, pick j), weighted by its routing weight
          const int ent = S.rt.ent[S.rt.off[t[R_A]] + n];
          const int b = ent / p.topk, j = ent % p.topk;
          __stcg(p.mdown + (size_t)ent * p.H + row0 + r, S.rt.w[b][j] * v);
          break;
        }
      }
    }
  }

  // several tokens, OUT: rows [row0, row0 + n) of each token's expert output,
  // the sum of its k weighted entries in pick order (every DOWN task has
  // written them)
  __device__ __forceinline__ void moe_sum() {
    const int l = t[R_LAYER], n = t[R_NROWS], row0 = t[R_ROW0], K = p.topk;
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < n * p.B; i += 256) {
      const int b = i / n, r = i % n;
      float s = 0.f;
      for (int j = 0; j < K; j++) s += __ldcg(p.mdown + (size_t)(b * K + j) * p.H + row0 + r);
      __stcg(p.moe + ((size_t)l * Bm + b) * p.H + row0 + r, s);
    }
  }

  // ------------------------------------------------------------ routing
  __device__ __forceinline__ bool route() {
    const int l = t[R_LAYER];
    const int E = p.E, K = p.topk, B = p.B;
    const size_t Bm = (size_t)p.Bmax;
    // one token: the producer warp has routed (the routing is in shared
    // memory before this task was handed over)
    if (ONE) return true;
    if (!wait_counter(bar_index(p, l, p.bl.rtr), p.n_rtr_sms)) return false;
    RouteTab& rt = S.rt;
    for (int n = warp; n < B; n += kConsumerWarps) {
      float v[8];
      const float* rl = p.rlog + ((size_t)l * Bm + n) * E;
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldcg(rl + e) : -INFINITY;
      }
      uint32_t taken = 0;
#pragma unroll 1
      for (int j = 0; j < K; j++) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const int e = lane + 32 * i;
          if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
            bv = v[i];
            bi = e;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == 0) {
          rt.idx[n][j] = bi;
          rt.w[n][j] = bv;     // the logit; replaced by the weight below
        }
      }
      __syncwarp();
      if (lane == 0) {
        const float top = rt.w[n][0];
        float den = 0.f;
#pragma unroll 1
        for (int j = 0; j < K; j++) den += expf(rt.w[n][j] - top);
#pragma unroll 1
        for (int j = 0; j < K; j++) {
          const float w = expf(rt.w[n][j] - top) / den;
          rt.w[n][j] = w;
          if (blockIdx.x == 0) {   // block 0 routes in every schedule
            p.ridx[((size_t)l * Bm + n) * K + j] = rt.idx[n][j];
            p.rw[((size_t)l * Bm + n) * K + j] = w;
          }
        }
      }
    }
    if (TR && tid == 0) S.t_mark[0] = gtime_ns();
    if (!csync()) return false;
    for (int e = tid; e < E; e += 256) {
      int c = 0;
      for (int n = 0; n < B; n++)
        for (int j = 0; j < K; j++) c += rt.idx[n][j] == e;
      rt.ecount[e] = c;
    }
    if (!csync()) return false;
    if (TR && tid == 0) S.t_mark[1] = gtime_ns();
    if (warp == 0) {
      // warp-wide exclusive scans over E <= 256 experts, 8 per lane
      int cnt[8], act[8], sc = 0, sa = 0;
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const int e = lane * 8 + i;
        cnt[i] = e < E ? rt.ecount[e] : 0;
        act[i] = cnt[i] > 0;
        sc += cnt[i];
        sa += act[i];
      }
      int ic = sc, ia = sa;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yc = __shfl_up_sync(0xffffffffu, ic, o), ya = __shfl_up_sync(0xffffffffu, ia, o);
        if (lane >= o) { ic += yc; ia += ya; }
      }
      int oc = ic - sc, oa = ia - sa;
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const int e = lane * 8 + i;
        if (e < E) {
          rt.eslot[e] = act[i] ? oa : -1;
          if (act[i]) {
            rt.act[oa] = e;
            rt.off[oa] = oc;
          }
        }
        oc += cnt[i];
        oa += act[i];
      }
      if (lane == 31) {
        rt.n_act = ia;
        rt.off[ia] = ic;
      }
    }
    if (!csync()) return false;
    if (TR && tid == 0) S.t_mark[2] = gtime_ns();
    for (int e = tid; e < E; e += 256) {
      const int a = rt.eslot[e];
      if (a < 0) continue;
      int i = rt.off[a];
      for (int n = 0; n < B; n++)
        for (int j = 0; j < K; j++)
          if (rt.idx[n][j] == e) rt.ent[i++] = n * K + j;
    }
    if (!csync()) return false;
    if (TR && p.dbg && blockIdx.x == 0) {
      int32_t* d = p.dbg + (size_t)l * kDbgRouteWords;
      const int n = rt.n_act;
      if (tid == 0) d[0] = n;
      for (int i = tid; i < n; i += 256) d[1 + i] = rt.act[i];
      for (int i = tid; i <= n; i += 256) d[1 + kMaxActive + i] = rt.off[i];
      for (int i = tid; i < rt.off[n]; i += 256) d[1 + kMaxActive + 1 + kMaxActive + i] = rt.ent[i];
    }
    if (tid == 0) mbar_arrive(&S.route_bar);   // the producer may now resolve the experts
    return true;
  }

  // -------------------------------------------------------- attention
  // byte offset of 16-byte chunk c (dims 8c .. 8c + 7) of row r in a page
  // image of `rows` rows stored as 128-byte swizzled boxes of 64 dims
  __device__ __forceinline__ static int kv_off(int r, int c, int rows) {
    return (c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
  }

  // One split-KV item: sequence b, keys [tt0, tt1), every KV head.  Warp w
  // serves KV group g = w % hkv and takes every NWG-th page of the item (NWG =
  // 8 / hkv warps per group), keeping its own online-softmax state; the NWG
  // states of a group are merged at the end.  Both products run on the tensor
  // cores (m16n8k16, BF16 in, fp32 out) with the page's 16 tokens as the M
  // side and the group's (up to 8) query heads as N, so no row is padding:
  //   S^T[token][head] = K Q^T:  A = the K rows (ldmatrix), B = Q^T held in
  //                              registers for the whole item;
  //   O^T[dim][head] += V^T P^T: A = V^T (ldmatrix.trans of the V rows),
  //                              B = P^T, the score accumulators converted to
  //                              BF16 and transposed in registers (movmatrix).
  // The fp32 query and probabilities are split into BF16 high + low halves
  // (two products each), so the contractions keep about 16 bits of their
  // mantissa.  Softmax per head in fp32 (log2 domain): the running maximum is
  // shared by the lanes of a head, the running sum is kept per lane and added
  // up at the end.  The query (RoPE applied here) is staged in shared memory
  // once per item, 16-byte chunks swizzled by row.  The KV pages arrive as
  // 128-byte swizzled boxes (kv_off): the eight rows an ldmatrix reads fall in
  // distinct banks.
  template <int D>
  __device__ __forceinline__ bool attn() {
    constexpr int KS = D / 16;            // QK k-steps = PV m-tiles
    const int hkv = p.hkv, grp = p.grp, P = p.P, hq = p.hq;
    const int NWG = kConsumerWarps / hkv;
    const int g = warp % hkv, jw = warp / hkv;
    const int l = t[R_LAYER], b = t[R_B];
    const int tt0 = t[R_TT0], tt1 = t[R_TT1], pos = t[R_POS];
    const size_t Bm = (size_t)p.Bmax;
    const int pb = hkv * P * D * 2;       // bytes of one page, all heads
    const int rows = hkv * P;             // rows of a page image (head-major)
    const int pps = attn_pps(p);
    if (!wait_counter(bar_index(p, l, p.bl.p1), p.n_sm)) return false;

    // query with RoPE -> BF16 hi / lo planes: [head][D] in 16-byte chunks, chunk c
    // of row h stored at chunk position c ^ (h & 7)
    uint8_t* qhi = (uint8_t*)S.red;
    uint8_t* qlo = qhi + hq * D * 2;
    const float* qraw = p.qkv + ((size_t)l * Bm + b) * p.qkv_rows;
    const float* rope = p.rope + (size_t)b * (D / 2) * 2;
    {
      // hq * D / 2 <= 2048 rotation pairs: at most 8 per thread, all loads first
      constexpr int NQ = 8;
      float x1[NQ], x2[NQ], cs[NQ], sn[NQ];
#pragma unroll
      for (int q = 0; q < NQ; q++) {
        const int i = tid + 256 * q;
        x1[q] = x2[q] = cs[q] = sn[q] = 0.f;
        if (i < hq * (D / 2)) {
          const int h = i / (D / 2), k = i % (D / 2);
          x1[q] = __ldcg(qraw + h * D + k);
          x2[q] = __ldcg(qraw + h * D + k + D / 2);
          cs[q] = rope[k * 2];
          sn[q] = rope[k * 2 + 1];
        }
      }
#pragma unroll
      for (int q = 0; q < NQ; q++) {
        const int i = tid + 256 * q;
        if (i < hq * (D / 2)) {
          const int h = i / (D / 2), k = i % (D / 2);
          const float y1 = x1[q] * cs[q] - x2[q] * sn[q], y2 = x2[q] * cs[q] + x1[q] * sn[q];
          const uint16_t h1 = f2bf(y1), h2 = f2bf(y2);
          const uint16_t l1 = f2bf(y1 - bf16f(h1)), l2 = f2bf(y2 - bf16f(h2));
          const int k2 = k + D / 2;
          const int o1 = h * D * 2 + (((k >> 3) ^ (h & 7)) << 4) + (k & 7) * 2;
          const int o2 = h * D * 2 + (((k2 >> 3) ^ (h & 7)) << 4) + (k2 & 7) * 2;
          *(uint16_t*)(qhi + o1) = h1;
          *(uint16_t*)(qhi + o2) = h2;
          *(uint16_t*)(qlo + o1) = l1;
          *(uint16_t*)(qlo + o2) = l2;
        }
      }
    }
    if (!csync()) return false;

    // B fragments of Q^T (k = dims, n = heads) for the whole item: lane (gl, cq)
    // holds head gl of the group, dims 16 s + 2 cq, +1 and 16 s + 8 + 2 cq, +1
    const int qrow = g * grp + gl;
    const bool qon = gl < grp;
    uint32_t qbh[KS][2], qbl[KS][2];
#pragma unroll
    for (int s = 0; s < KS; s++)
#pragma unroll
      for (int hf = 0; hf < 2; hf++) {
        const int off = qrow * D * 2 + (((2 * s + hf) ^ (qrow & 7)) << 4) + 4 * cq;
        qbh[s][hf] = qon ? *(const uint32_t*)(qhi + off) : 0u;
        qbl[s][hf] = qon ? *(const uint32_t*)(qlo + off) : 0u;
      }

    // this lane's softmax state: heads 2 cq, 2 cq + 1
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    // O^T accumulators: tile t, dims 16 t + gl (c0: head 2cq, c1: 2cq + 1) and
    // 16 t + 8 + gl (c2, c3)
    float o[KS][4];
#pragma unroll
    for (int s = 0; s < KS; s++) o[s][0] = o[s][1] = o[s][2] = o[s][3] = 0.f;

    // ldmatrix rows of this lane: K (A of S^T): tile i = lane / 8 holds tokens
    // (i & 1) * 8 + 0..7, dims chunk 2 s + (i >> 1); V (A of O^T, transposed):
    // tokens (i >> 1) * 8 + 0..7, dims chunk 2 t + (i & 1)
    const int kr = g * P + ((lane >> 3) & 1) * 8 + (lane & 7), kc = lane >> 4;
    const int vr = g * P + (lane >> 4) * 8 + (lane & 7), vc = (lane >> 3) & 1;

    const int pg0 = tt0 / P;
    const int npages = (tt1 + P - 1) / P - pg0;
    const int nst = t[R_NST];
    const float sc = p.attn_scale_log2;
    for (int st = 0; st < nst; st++) {
      uint32_t slot;
      if (!stage_full(slot)) return false;
      if (TR && tid == 0 && st == 0) S.t_mark[0] = gtime_ns();
      for (int qi = 0; qi < pps; qi++) {
        const int page = st * pps + qi;
        if (page >= npages) break;
        if (page % NWG != jw) continue;
        uint8_t* kp = S.stage[slot] + qi * pb;
        uint8_t* vp = S.stage[slot] + (pps + qi) * pb;
        const int tk0 = (pg0 + page) * P;
        const bool has_new = pos >= tk0 && pos < tk0 + P;
        // the new token's K (RoPE applied here) and V come from this step's QKV
        // output: patched into the staged page (group g's row) before it is
        // read, and written to the cache
        if (has_new) {
          const int row = pos - tk0;
          const float* krw = qraw + (size_t)(hq + g) * D;
          const float* vrw = qraw + (size_t)(hq + hkv + g) * D;
          const int pg = p.page_tables[(size_t)b * p.max_pages + pos / P];
          if (TR && p.dbg && l == 0 && g == 0 && lane == 0)
            p.dbg[(size_t)p.L * kDbgRouteWords + (size_t)p.Bmax * p.max_pages + b] = pg * P + row;
          uint16_t* kcache = p.k_pool[l] + (((size_t)pg * hkv + g) * P + row) * D;
          uint16_t* vcache = p.v_pool[l] + (((size_t)pg * hkv + g) * P + row) * D;
          const int r = g * P + row;
          for (int k = lane; k < D / 2; k += 32) {
            const float x1 = __ldcg(krw + k), x2 = __ldcg(krw + k + D / 2);
            const float c = rope[k * 2], s = rope[k * 2 + 1];
            const uint16_t k1 = f2bf(x1 * c - x2 * s), k2 = f2bf(x2 * c + x1 * s);
            const uint16_t v1 = f2bf(__ldcg(vrw + k)), v2 = f2bf(__ldcg(vrw + k + D / 2));
            const int o1 = kv_off(r, k >> 3, rows) + (k & 7) * 2;
            const int o2 = kv_off(r, (k + D / 2) >> 3, rows) + (k & 7) * 2;
            *(uint16_t*)(kp + o1) = k1;
            *(uint16_t*)(kp + o2) = k2;
            *(uint16_t*)(vp + o1) = v1;
            *(uint16_t*)(vp + o2) = v2;
            kcache[k] = k1;
            kcache[k + D / 2] = k2;
            vcache[k] = v1;
            vcache[k + D / 2] = v2;
          }
          __syncwarp();
        }
        // S^T = K Q^T, four independent accumulators (k-step parity x hi / lo)
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        float ta[4] = {0.f, 0.f, 0.f, 0.f}, tb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < KS; s++) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(a0, a1, a2, a3, kp + kv_off(kr, 2 * s + kc, rows));
          if (s & 1) {
            mma_bf16(sb, a0, a1, a2, a3, qbh[s][0], qbh[s][1]);
            mma_bf16(tb, a0, a1, a2, a3, qbl[s][0], qbl[s][1]);
          } else {
            mma_bf16(sa, a0, a1, a2, a3, qbh[s][0], qbh[s][1]);
            mma_bf16(ta, a0, a1, a2, a3, qbl[s][0], qbl[s][1]);
          }
        }
        // this lane: tokens gl (v0: head 2cq, v1: 2cq + 1) and gl + 8 (v2, v3)
        const int lo_t = max(tt0 - tk0, 0), hi_t = min(tt1 - tk0, P);   // valid rows [lo_t, hi_t)
        const bool ok0 = gl >= lo_t && gl < hi_t, ok1 = gl + 8 >= lo_t && gl + 8 < hi_t;
        const float v0 = ok0 ? ((sa[0] + ta[0]) + (sb[0] + tb[0])) * sc : -INFINITY;
        const float v1 = ok0 ? ((sa[1] + ta[1]) + (sb[1] + tb[1])) * sc : -INFINITY;
        const float v2 = ok1 ? ((sa[2] + ta[2]) + (sb[2] + tb[2])) * sc : -INFINITY;
        const float v3 = ok1 ? ((sa[3] + ta[3]) + (sb[3] + tb[3])) * sc : -INFINITY;
        // per head maximum over the page's 16 tokens (the 8 lanes of equal cq)
        float x0 = fmaxf(v0, v2), x1 = fmaxf(v1, v3);
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
          x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, sh));
          x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, sh));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float al0 = (n0 == -INFINITY) ? 1.f : exp2f(m0 - n0);
        const float al1 = (n1 == -INFINITY) ? 1.f : exp2f(m1 - n1);
        const float p0 = (n0 == -INFINITY) ? 0.f : exp2f(v0 - n0);
        const float p1 = (n1 == -INFINITY) ? 0.f : exp2f(v1 - n1);
        const float p2 = (n0 == -INFINITY) ? 0.f : exp2f(v2 - n0);
        const float p3 = (n1 == -INFINITY) ? 0.f : exp2f(v3 - n1);
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
        m0 = n0;
        m1 = n1;
        // P^T as the B operand: each 8 x 8 block [token][head] of the score
        // accumulators, transposed to [head][token]; high and low halves
        const uint32_t h01 = pack_bf2(p0, p1), h23 = pack_bf2(p2, p3);
        const uint32_t e01 = pack_bf2(p0 - bf16lo(h01), p1 - bf16hi(h01));
        const uint32_t e23 = pack_bf2(p2 - bf16lo(h23), p3 - bf16hi(h23));
        const uint32_t bh0 = movm_trans(h01), bh1 = movm_trans(h23);
        const uint32_t bl0 = movm_trans(e01), bl1 = movm_trans(e23);
        // O^T += V^T P^T
#pragma unroll
        for (int s = 0; s < KS; s++) {
          o[s][0] *= al0;
          o[s][1] *= al1;
          o[s][2] *= al0;
          o[s][3] *= al1;
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(a0, a1, a2, a3, vp + kv_off(vr, 2 * s + vc, rows));
          mma_bf16(o[s], a0, a1, a2, a3, bh0, bh1);
          mma_bf16(o[s], a0, a1, a2, a3, bl0, bl1);
        }
        if (has_new) fence_proxy_async_smem();
        __syncwarp();
      }
      stage_release(slot);
    }

    if (TR && tid == 0) S.t_mark[1] = gtime_ns();
    // running sums: add up the lanes of each head
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
      l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
    }
    // merge the NWG warps of each group: in round r the warps jw == r put
    // (max, sum, O) in shared memory and the warps jw == 0 fold them in
    // (the staged query is no longer needed: its fragments are in registers)
    float* mo = S.red;   // [hkv][D][8]
    if (!csync()) return false;
    for (int r = 1; r < NWG; r++) {
      if (jw == r) {
#pragma unroll
        for (int s = 0; s < KS; s++) {
          float* row0 = mo + ((size_t)g * D + 16 * s + gl) * 8 + 2 * cq;
          float* row1 = row0 + 8 * 8;
          *(float2*)row0 = make_float2(o[s][0], o[s][1]);
          *(float2*)row1 = make_float2(o[s][2], o[s][3]);
        }
        if (gl == 0) {
          S.nred[warp][2 * cq] = m0;
          S.nred[warp][2 * cq + 1] = m1;
          S.nred[warp][8 + 2 * cq] = l0;
          S.nred[warp][8 + 2 * cq + 1] = l1;
        }
      }
      if (!csync()) return false;
      if (jw == 0) {
        const int src = r * hkv + g;
        const float pm0 = S.nred[src][2 * cq], pm1 = S.nred[src][2 * cq + 1];
        const float pl0 = S.nred[src][8 + 2 * cq], pl1 = S.nred[src][8 + 2 * cq + 1];
        const float M0 = fmaxf(m0, pm0), M1 = fmaxf(m1, pm1);
        const float a0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - M0), b0 = (pm0 == -INFINITY) ? 0.f : exp2f(pm0 - M0);
        const float a1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - M1), b1 = (pm1 == -INFINITY) ? 0.f : exp2f(pm1 - M1);
        l0 = l0 * a0 + pl0 * b0;
        l1 = l1 * a1 + pl1 * b1;
        m0 = M0;
        m1 = M1;
#pragma unroll
        for (int s = 0; s < KS; s++) {
          const float* row0 = mo + ((size_t)g * D + 16 * s + gl) * 8 + 2 * cq;
          const float2 u = *(const float2*)row0, v = *(const float2*)(row0 + 8 * 8);
          o[s][0] = o[s][0] * a0 + u.x * b0;
          o[s][1] = o[s][1] * a1 + u.y * b1;
          o[s][2] = o[s][2] * a0 + v.x * b0;
          o[s][3] = o[s][3] * a1 + v.y * b1;
        }
      }
      if (!csync()) return false;
    }
    // the group's partials: heads 2cq, 2cq + 1 (those below grp), dims 16 t + gl, + 8
    const int item = t[R_ITEM];
    if (jw == 0) {
#pragma unroll
      for (int e = 0; e < 2; e++) {
        const int hh = 2 * cq + e;
        if (hh < grp) {
          const size_t it = ((size_t)item * hkv + g) * grp + hh;
          float* dst = p.attn_part + it * D;
#pragma unroll
          for (int s = 0; s < KS; s++) {
            __stcg(dst + 16 * s + gl, o[s][e]);
            __stcg(dst + 16 * s + 8 + gl, o[s][2 + e]);
          }
          if (gl == 0) {
            __stcg(p.attn_ml + it * 2 + 0, e ? m1 : m0);
            __stcg(p.attn_ml + it * 2 + 1, e ? l1 : l0);
          }
        }
      }
    }
    if (TR && tid == 0) S.t_mark[2] = gtime_ns();
    return signal(bar_index(p, l, p.bl.items + b), 1);
  }

  // ATTN_COMBINE of units [u0, u1) (unit = sequence b, query head h): merge the
  // sequence's split-KV partials in one pass.  Warp w takes splits w, w + 8,
  // ... (four loads in flight), lane l dims DPL l .. DPL l + DPL - 1, and keeps
  // a running maximum: each split rescales the warp's sums to the larger
  // maximum.  The warps' (maximum, sum, numerator) meet in shared memory and
  // are merged in warp order.
  template <int D>
  __device__ __forceinline__ bool combine() {
    constexpr int DPL = D / 32;
    const int l = t[R_LAYER], hkv = p.hkv, grp = p.grp;
    const size_t Bm = (size_t)p.Bmax;
    for (int u = t[R_U0]; u < t[R_U1]; u++) {
      const int b = u / p.hq, h = u % p.hq;
      const int g = h / grp, hh = h % grp;
      const int base = p.attn_meta[b * 2], nsplit = p.attn_meta[b * 2 + 1];
      if (!wait_counter(bar_index(p, l, p.bl.items + b), nsplit)) return false;
      float m = -INFINITY, den = 0.f, num[DPL];
#pragma unroll
      for (int j = 0; j < DPL; j++) num[j] = 0.f;
      for (int s0 = warp; s0 < nsplit; s0 += 4 * kConsumerWarps) {
        float2 ml[4];
        float ov[4][DPL];
#pragma unroll
        for (int q = 0; q < 4; q++) {
          const int s = s0 + q * kConsumerWarps;
          const size_t it = ((size_t)(base + min(s, nsplit - 1)) * hkv + g) * grp + hh;
          ml[q] = s < nsplit ? __ldcg((const float2*)(p.attn_ml + it * 2)) : make_float2(-INFINITY, 0.f);
          if constexpr (DPL == 4) {
            const float4 v = __ldcg((const float4*)(p.attn_part + it * D) + lane);
            ov[q][0] = v.x; ov[q][1 % DPL] = v.y; ov[q][2 % DPL] = v.z; ov[q][3 % DPL] = v.w;
          } else {
            const float2 v = __ldcg((const float2*)(p.attn_part + it * D) + lane);
            ov[q][0] = v.x; ov[q][1 % DPL] = v.y;
          }
        }
#pragma unroll
        for (int q = 0; q < 4; q++) {
          const float mn = fmaxf(m, ml[q].x);
          const float a = m == -INFINITY ? 0.f : exp2f(m - mn);
          const float w = ml[q].x == -INFINITY ? 0.f : exp2f(ml[q].x - mn);
          den = den * a + w * ml[q].y;
#pragma unroll
          for (int j = 0; j < DPL; j++) num[j] = num[j] * a + w * ov[q][j];
          m = mn;
        }
      }
      float* red = S.red;   // [warp][D]
#pragma unroll
      for (int j = 0; j < DPL; j++) red[warp * D + lane * DPL + j] = num[j];
      if (lane == 0) {
        S.nred[warp][0] = m;
        S.nred[warp][1] = den;
      }
      if (!csync()) return false;
      if (tid < D) {
        float M = -INFINITY;
        for (int w = 0; w < kConsumerWarps; w++) M = fmaxf(M, S.nred[w][0]);
        float sn = 0.f, sd = 0.f;
        for (int w = 0; w < kConsumerWarps; w++) {
          const float mw = S.nred[w][0];
          const float a = mw == -INFINITY ? 0.f : exp2f(mw - M);
          sn += a * red[w * D + tid];
          sd += a * S.nred[w][1];
        }
        __stcg(p.attn_out + ((size_t)l * Bm + b) * p.hq * D + (size_t)h * D + tid, sn / sd);
      }
      if (u + 1 < t[R_U1] && !csync()) return false;
    }
    return signal(bar_index(p, l, p.bl.comb), 1);
  }
};

// Every consumer path is inlined into the consumer loop: an out-of-line call
// saves the callee's registers to the stack, and the stacks of the block's
// threads do not fit the L1 left beside 227 KB of shared memory, so each call
// would cost L2 round trips.  With 216 registers per consumer thread (see
// the register split) the union of the paths needs no spill.  The per-warp
// pipeline counters travel through shared memory between paths.
template <bool ONE, bool TR>
__device__ __forceinline__ bool op_chunk(const Params& p, Smem& S, const int32_t* t) {
  Cons<ONE, TR> c(p, S, t);
  const int op = t[R_OP], kind = t[R_KIND], flags = t[R_FLAGS], l = t[R_LAYER];
  bool ok = true;
  if ((op == OP_P1 || op == OP_FINAL) && (flags & FL_FIRST)) ok = c.norm(l, op == OP_FINAL);
  const bool run = t[R_NROWS] > 0 && t[R_NT] > 0;
  if (ok && run && kind == K_OPROJ) ok = c.wait_counter(bar_index(p, l, p.bl.comb), p.n_comb_sms);
  if (ok && run && kind == K_DOWN) ok = c.wait_counter(bar_index(p, l, p.bl.up), p.n_up_sms);
  float* part = S.red + (S.cchunk[c.warp] & 1u) * kPartFloats;
  if (kind == K_MSUM) {
    if (ok && run) ok = c.wait_counter(bar_index(p, l, p.bl.down), p.n_down_sms);
    if (ok && run) c.moe_sum();
  } else {
    // dense rows and an expert's gate / up rows (up to 8 tokens at 2048
    // columns, 4 at 4096) and an expert's down rows on the tensor cores: one
    // partial per warp instead of one per 256-column segment
    const int nt = t[R_NT];
    const int K = t[R_K];
    const bool mma = run && ((kind != K_DOWN && p.w_maps && mma_multi_rows(K, nt)) ||
                             (kind == K_DOWN && p.wd_maps));
    if (ok && run) {
      // tokens per pass matched to the chunk (an expert's few routed tokens do
      // not pay for eight)
      if (mma && kind == K_DOWN) {
        const int nq = (nt + 3) >> 2;
        ok = nq <= 1 ? c.template gemv_mma_down<1>(part) : nq == 2 ? c.template gemv_mma_down<2>(part)
           : nq == 3 ? c.template gemv_mma_down<3>(part) : c.template gemv_mma_down<4>(part);
      } else if (mma && K == 2048) {
        const int nq = (nt + 1) >> 1;
        ok = nq <= 1 ? c.template gemv_mma_multi<1, 1>(part) : nq == 2 ? c.template gemv_mma_multi<1, 2>(part)
           : nq == 3 ? c.template gemv_mma_multi<1, 3>(part) : c.template gemv_mma_multi<1, 4>(part);
      } else if (mma) {
        ok = nt <= 1 ? c.template gemv_mma_multi<2, 1>(part) : nt == 2 ? c.template gemv_mma_multi<2, 2>(part)
           : nt == 3 ? c.template gemv_mma_multi<2, 3>(part) : c.template gemv_mma_multi<2, 4>(part);
      } else {
        ok = nt <= 1 ? c.template gemv<1>(part) : c.template gemv<8>(part);
      }
      ok = ok && c.csync();
    }
    if (ok && run) {
      c.epilogue(part, mma ? kConsumerWarps : gemv_nseg(t[R_K]));
      if (TR && c.tid == 0) S.t_mark[2] = gtime_ns();
      if (c.lane == 0) S.cchunk[c.warp]++;
    }
  }
  if (ok && (flags & (FL_RTR | FL_LAST))) ok = c.finish(flags);
  c.save();
  return ok;
}

// one-token chunk: one copy of the wrapper (norm, waits, epilogue,
// completion) around the GEMV shape for the row length
template <bool ONE, bool TR, bool F8>
__device__ __forceinline__ bool op_row(const Params& p, Smem& S, const int32_t* t) {
  Cons<ONE, TR> c(p, S, t);
  const int op = t[R_OP], kind = t[R_KIND], flags = t[R_FLAGS], l = t[R_LAYER];
  bool ok = true;
  if ((op == OP_P1 || op == OP_FINAL) && (flags & FL_FIRST)) ok = c.norm(l, op == OP_FINAL);
  int rows = t[R_NROWS];
  if (kind == K_P1) rows += t[R_NROWS1];
  const bool run = rows > 0;
  float* res = S.red + (S.cchunk[c.warp] & 1u) * kPartFloats;
  if (kind == K_MRED) {
    if (ok && run) ok = c.moe_reduce(res);
  } else {
    if (ok && run && kind == K_OPROJ) ok = c.wait_counter(bar_index(p, l, p.bl.comb), p.n_comb_sms) && c.stage_x();
    // 8-bit expert piece: its row scales, loaded now so that they arrive
    // while the gate / up rows stream (gate / up: row tid; down: rows
    // h = tid + 256 j, staged in shared memory before the down projection)
    float sg_t = 0.f, su_t = 0.f, sdv[8];
    if (F8 && kind == K_UP && run) {
      const size_t eo = (size_t)t[R_E];
      if (c.tid < t[R_NROWS]) {
        sg_t = __ldg(p.s_gate[l] + eo * p.I + t[R_ROW0] + c.tid);
        su_t = __ldg(p.s_up[l] + eo * p.I + t[R_ROW0] + c.tid);
      }
#pragma unroll
      for (int j = 0; j < 8; j++) sdv[j] = c.tid + 256 * j < p.H ? __ldg(p.s_down[l] + eo * p.H + c.tid + 256 * j) : 0.f;
    }
    if (ok && run) {
      const int K = t[R_K];
      // rows of 2048 or 4096 columns (every chunk kind: P1, O-proj, an UP
      // piece's gate and up rows, LM head) on the tensor cores: one code path
      // for the layer's GEMVs
      const bool split = rotated_rows(K);
      bool done8 = false;
      if constexpr (F8) {
        if (kind == K_UP) {        // 8-bit expert rows (K = 2048, or <= 1024)
          ok = split ? c.gemv_mma_e4m3(res)
                     : K <= 512 ? c.template gemv_row_e4m3<1>(res) : c.template gemv_row_e4m3<2>(res);
          done8 = true;
        }
      }
      if (done8) {
      } else if (split) ok = K == 2048 ? c.template gemv_mma<1>(res) : c.template gemv_mma<2>(res);
      else ok = K <= 256 ? c.template gemv_row<1>(res) : K <= 768 ? c.template gemv_row<3>(res)
              : K <= 2048 ? c.template gemv_row<8>(res) : c.template gemv_row<16>(res);
      // the tensor-core path's sums are written by the threads that run the
      // epilogue (except UP's, whose epilogue pairs row i with row nr + i);
      // its partial buffer is reused by the next chunk, which the
      // completion barrier below also orders when the task ends here
      if (ok && !(split && (flags & FL_LAST) && kind != K_UP)) ok = c.csync();
    }
    if (ok && run) {
      c.template epilogue_row<F8>(res, sg_t, su_t);
      if (TR && c.tid == 0) S.t_mark[2] = gtime_ns();
    }
    // an UP piece goes on with its columns of the down projection (8-bit:
    // the rows' scales staged in the upper half of xs first)
    if (F8 && ok && run && kind == K_UP) {
#pragma unroll
      for (int j = 0; j < 8; j++)
        if (c.tid + 256 * j < p.H) S.xs[kXsFloats / 2 + c.tid + 256 * j] = sdv[j];
    }
    if (ok && run && kind == K_UP) {
      if constexpr (F8) ok = c.csync() && c.down_mma_e4m3();
      else ok = c.csync() && c.down_part();
    }
  }
  if (ok && run && c.lane == 0) S.cchunk[c.warp]++;
  if (ok && (flags & (FL_RTR | FL_LAST))) ok = c.finish(flags);
  c.save();
  return ok;
}

template <bool ONE, bool TR>
__device__ __forceinline__ bool op_route(const Params& p, Smem& S, const int32_t* t) {
  Cons<ONE, TR> c(p, S, t);
  const bool ok = c.route();
  c.save();
  return ok;
}

template <bool ONE, bool TR, int D>
__device__ __forceinline__ bool op_attn(const Params& p, Smem& S, const int32_t* t) {
  Cons<ONE, TR> c(p, S, t);
  const bool ok = c.template attn<D>();
  c.save();
  return ok;
}

template <bool ONE, bool TR, int D>
__device__ __forceinline__ bool op_combine(const Params& p, Smem& S, const int32_t* t) {
  Cons<ONE, TR> c(p, S, t);
  const bool ok = c.template combine<D>();
  c.save();
  return ok;
}

// consumer main loop: take the next resolved task, run it, record its timeline.
// ONE: the batch has one token (one-token GEMV paths only; a separate kernel
// instance keeps each instance's union of inlined paths within registers).
// TR: the timeline is recorded (an instance of its own, so the timed
// instances carry no clock reads).
template <bool ONE, bool TR, bool F8>
__device__ __forceinline__ void consumer_loop(const Params& p, Smem& S) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t task_seq = 0;
  int n_rec = 0;
  while (true) {
    const uint32_t slot = task_seq % kTaskSlots;
    if (!wait_phase(p, &S.tfull[slot], (task_seq / kTaskSlots) & 1u)) {
      if (tid == 0) report(p, DEV_SMEM_TIMEOUT, -1, -1, -1, 0, 0);
      break;
    }
    const int32_t* t = S.task[slot];
    task_seq++;
    const int op = t[R_OP];
    if (op == OP_END) break;
    const unsigned long long t_start = TR ? gtime_ns() : 0ull;
    if (TR && tid == 0) {
      S.t_ready = t_start;
      S.t_mark[0] = S.t_mark[1] = S.t_mark[2] = S.t_mark[3] = t_start;
      S.t_swait = 0;
    }
    bool ok = false;
    switch (op) {
      case OP_P1:
      case OP_UP:
      case OP_DOWN:
      case OP_OUT:
      case OP_FINAL: {
        const int nt = t[R_NT];
        // one token: whole rows per warp, by the row's length; more tokens:
        // up to eight per pass
        if constexpr (ONE) {
          ok = op_row<true, TR, F8>(p, S, t);
        } else {
          ok = op_chunk<false, TR>(p, S, t);
        }
        (void)nt;
        break;
      }
      case OP_ROUTE: ok = op_route<ONE, TR>(p, S, t); break;
      case OP_ATTN: ok = (p.d == 128) ? op_attn<ONE, TR, 128>(p, S, t) : op_attn<ONE, TR, 64>(p, S, t); break;
      case OP_COMBINE: ok = (p.d == 128) ? op_combine<ONE, TR, 128>(p, S, t) : op_combine<ONE, TR, 64>(p, S, t); break;
      default: ok = false; break;
    }
    if (TR && tid == 0 && n_rec < p.trace_cap) {
      const unsigned long long t_end = gtime_ns();
      int32_t* rec = p.trace + ((size_t)blockIdx.x * p.trace_cap + n_rec) * kTraceWords;
      rec[0] = op;
      rec[1] = t[R_LAYER];
      rec[2] = op == OP_ATTN ? t[R_ITEM] : t[R_ROW0];
      rec[3] = (int32_t)(uint32_t)(t_start & 0xffffffffull);
      rec[4] = (int32_t)(uint32_t)(t_start >> 32);
      rec[5] = (int32_t)(S.t_ready - t_start);
      rec[6] = (int32_t)(t_end - t_start);
      rec[7] = blockIdx.x;
      for (int k = 0; k < 3; k++) rec[8 + k] = (int32_t)(S.t_mark[k] - t_start);
      rec[11] = t[R_KIND];
      rec[12] = t[R_NROWS];
      rec[13] = (int32_t)((uint32_t)t[R_PCOMMIT] - (uint32_t)t_start);
      rec[14] = t[R_PISSUE] ? (int32_t)((uint32_t)t[R_PISSUE] - (uint32_t)t_start) : 0;
      rec[15] = (int32_t)S.t_swait;
      n_rec++;
    }
    // the task's words are no longer needed: hand the slot back to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.tempty[slot]);
    if (!ok || S.abort_flag) {
      // a wait gave up (reported here as a time-out unless a report came first)
      if (tid == 0) report(p, DEV_SMEM_TIMEOUT, t[R_TASK], op, -1, 0, 0);
      break;
    }
  }
}

template <bool ONE, bool TR, bool F8 = false>
__global__ void __launch_bounds__(kThreads, 1) mk_step_kernel(const __grid_constant__ Params p) {
  static_assert(kThreads == 384 && kLaunchRegs == 168, "register split assumes 384 threads x 168");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + pad);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    for (int s = 0; s < kTaskSlots; s++) {
      mbar_init(&S.tfull[s], 1);
      mbar_init(&S.tempty[s], kConsumerWarps);
    }
    mbar_init(&S.cbar, kConsumerWarps);
    mbar_init(&S.route_bar, 1);
    for (int w = 0; w < kConsumerWarps; w++) {
      S.cstage[w] = S.cphase[w] = S.cchunk[w] = 0;
      S.seen_bar[w] = -1;
      S.seen_tgt[w] = 0;
    }
    S.abort_flag = 0;
    S.xq_layer = -1;
    mbar_fence_init();
  }
  __syncthreads();
  const int wid = threadIdx.x >> 5;
  if (wid >= kConsumerWarps) {
    // producer warpgroup: one warp streams, the other three only give their
    // registers back
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs) : "memory");
    if (wid == kConsumerWarps) {
      Prod<ONE, TR, F8> pr(p, S);
      pr.run();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs) : "memory");
    consumer_loop<ONE, TR, F8>(p, S);
  }
}

// the four kernel instances: (one token, several) x (timeline off, on)
// and, for one token with 8-bit experts, two more (timeline off, on), so that
// the BF16 instances carry none of the 8-bit paths
constexpr int kNumStepKernels = 6;
static const void* const kStepKernels[kNumStepKernels] = {
    (const void*)mk_step_kernel<false, false>, (const void*)mk_step_kernel<true, false>,
    (const void*)mk_step_kernel<false, true>, (const void*)mk_step_kernel<true, true>,
    (const void*)mk_step_kernel<true, false, true>, (const void*)mk_step_kernel<true, true, true>};

// registers per thread every kernel instance was built with (the split above
// needs kLaunchRegs); -1 if they differ or cannot be read
int step_kernel_regs() {
  int regs = -1;
  for (int i = 0; i < kNumStepKernels; i++) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, kStepKernels[i]) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
    if (i > 0 && a.numRegs != regs) return -1;
    regs = a.numRegs;
  }
  return regs;
}

size_t step_smem_bytes() { return kSmemBytes; }

// w_down of one layer, [E][H][I] -> [E][I/8][H][8]: block (e, 32 rows, 32
// groups) through shared memory, so both the reads (along a row) and the
// writes (along a group's rows) are 512-byte runs
__global__ void __launch_bounds__(256) relayout_down_kernel(const uint16_t* __restrict__ src,
                                                            uint16_t* __restrict__ dst, int E, int H, int I) {
  __shared__ uint4 tile[32][33];
  const int G = I / 8;
  const int gb = (G + 31) / 32, hb = (H + 31) / 32;
  const int e = blockIdx.x / (hb * gb), rem = blockIdx.x % (hb * gb);
  const int h0 = (rem / gb) * 32, g0 = (rem % gb) * 32;
  for (int k = threadIdx.x; k < 1024; k += 256) {
    const int r = k / 32, q = k % 32;
    if (h0 + r < H && g0 + q < G)
      tile[r][q] = *(const uint4*)(src + ((size_t)e * H + h0 + r) * I + (size_t)(g0 + q) * 8);
  }
  __syncthreads();
  for (int k = threadIdx.x; k < 1024; k += 256) {
    const int q = k / 32, r = k % 32;
    if (h0 + r < H && g0 + q < G)
      *(uint4*)(dst + (((size_t)e * G + g0 + q) * H + h0 + r) * 8) = tile[r][q];
  }
}

// the same blocking for 8-bit (E4M3) down projections: one thread per
// (expert, group, row) moves the row's 8 bytes of the group
__global__ void __launch_bounds__(256) relayout_down_e4m3_kernel(const uint8_t* __restrict__ src,
                                                                 uint8_t* __restrict__ dst, int E, int H, int I) {
  const size_t G = (size_t)I / 8, total = (size_t)E * G * H;
  for (size_t k = (size_t)blockIdx.x * 256 + threadIdx.x; k < total; k += (size_t)gridDim.x * 256) {
    const size_t h = k % H, g = (k / H) % G, e = k / ((size_t)H * G);
    *(uint2*)(dst + k * 8) = *(const uint2*)(src + (e * H + h) * I + g * 8);
  }
}

cudaError_t relayout_down_e4m3(const uint8_t* src, uint8_t* dst, int E, int H, int I) {
  if (I % 8 || (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 8)
    return cudaErrorInvalidValue;
  relayout_down_e4m3_kernel<<<1216, 256>>>(src, dst, E, H, I);
  return cudaGetLastError();
}

cudaError_t relayout_down(const uint16_t* src, uint16_t* dst, int E, int H, int I) {
  const int G = I / 8;
  const long long blocks = (long long)E * ((H + 31) / 32) * ((G + 31) / 32);
  if (blocks < 1 || blocks > 0x7fffffff) return cudaErrorInvalidValue;
  relayout_down_kernel<<<(unsigned)blocks, 256>>>(src, dst, E, H, I);
  return cudaGetLastError();
}

// the dynamic shared-memory limit is a per-device attribute of each kernel:
// set once on every device that launches the step
cudaError_t configure_step_kernels() {
  constexpr int kMaxDev = 64;
  static std::atomic<bool> configured[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev && configured[dev].load(std::memory_order_acquire)) return cudaSuccess;
  for (int i = 0; i < kNumStepKernels; i++) {
    e = cudaFuncSetAttribute(kStepKernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  if (dev >= 0 && dev < kMaxDev) configured[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

cudaError_t launch_step(const Params& p, int n_sm, cudaStream_t stream) {
  const cudaError_t ce = configure_step_kernels();
  if (ce != cudaSuccess) return ce;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_sm);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void* k = p.fp8 ? kStepKernels[4 + (p.trace != nullptr ? 1 : 0)]
                        : kStepKernels[(p.B == 1 ? 1 : 0) + (p.trace != nullptr ? 2 : 0)];
  void* args[1] = {(void*)&p};
  return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace mk
