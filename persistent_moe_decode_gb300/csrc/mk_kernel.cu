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
//  - §The task scheduler, dynamic part: ATTN / MOE claimers atomically take
//    the next item of a shared queue until it is exhausted;
//  - §Tasks: ATTN_DECODE over a partial KV slice, ATTN_COMBINE merging the
//    partial results.
//
// GB300 design (not the pages' H100 one):
//  - block = 8 consumer warps + 1 producer warp.  The producer resolves the
//    task list (descriptors, queue claims, page tables) and streams every
//    weight / KV byte HBM -> shared memory with 1-D bulk async copies into a
//    6-stage ring of 32 KB stages guarded by mbarriers.  The ring runs ahead
//    across task boundaries of different opcodes, so a task that waits for
//    its activations already has its weights in flight.
//  - narrow GEMV path (batch <= 8): a stage is up to 32 KB of whole
//    contiguous weight rows moved by ONE bulk copy (large copies are what
//    keep HBM busy); the warps split each row into segments, multiply on the
//    CUDA cores in fp32 against fp32 activations held in registers and reduce
//    with warp shuffles, then combine segments in a fixed order.
//  - wide GEMV path (batch 9..16): warp-level BF16 tensor-core MMA with the
//    weights as the 16-row operand and 16 tokens as the 16-wide operand, on
//    16-row stages padded for conflict-free fragment loads.
//  - attention: one queue item = one sequence, all KV heads, a range of
//    16-token pages (K and V of a page are each one contiguous copy).  QK^T
//    on the tensor cores with the fp32 query split into BF16 high + low
//    halves, online softmax in fp32, PV on the CUDA cores.  Separate combine
//    tasks merge the splits of one (sequence, KV head).
//  - the last router tile of a layer runs top-k and route setup (ticket
//    counter); the residual add + RMSNorm is one task per layer.
//  - every wait has a %globaltimer limit (the consumer warps' own barrier is
//    an mbarrier with a bounded wait, not bar.sync); on expiry the block
//    records the error, sets a global stop word that every other wait polls,
//    drains its own in-flight copies and returns.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mk_layout.h"
#include "mk_ptx.cuh"

namespace mk {

// ------------------------------------------------------------ shared memory
struct __align__(128) Smem {
  uint8_t stage[kStages][kStageBytes];
  float red[4096];                          // GEMV partials / attention merge
  float tile_out[64][kMaxBatch];            // reduced tile: [row][token]
  float pbuf[kConsumerWarps][16][8];        // attention probabilities of one page per warp
  float alpha[kConsumerWarps][8];           // attention rescale per head per warp
  float wstat[kConsumerWarps][8][2];        // attention (max, sum) per warp per head
  float nred[kConsumerWarps][kMaxBatch];    // norm reductions
  float rinv[kMaxBatch];
  int32_t sel[kMaxBatch][8];                // router top-k of the last tile
  int32_t task[kTaskSlots][kDescWords];     // resolved task ring
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[kTaskSlots];
  uint64_t tempty[kTaskSlots];
  uint64_t cbar;                            // bounded barrier of the 8 consumer warps
  uint32_t cstage[kConsumerWarps];          // per consumer warp: stages consumed
  uint32_t cphase[kConsumerWarps];          // per consumer warp: barrier phases passed
  unsigned long long t_ready;               // timeline: when the task's inputs were ready
  int32_t seen_bar[kConsumerWarps];         // per consumer warp: last counter waited on...
  int32_t seen_tgt[kConsumerWarps];         // ...and the target it reached (lower ones are free)
  unsigned long long t_mark[4];             // timeline: in-task phases (first stage, stages
                                            // done, reduce / merge done, epilogue done)
  volatile int32_t abort_flag;
  int32_t bcast;
};

// resolved task words (written by the producer into the task ring)
enum : int {
  R_OP = 0, R_LAYER, R_NST, R_K, R_NRG, R_VR0, R_VR1, R_W0, R_T0, R_W1, R_T1, R_SIG, R_INC,
  R_TILE, R_E, R_NTOK, R_OFF, R_TASK, R_B, R_G, R_TT0, R_TT1, R_POS, R_NSPLIT, R_ITEM, R_BASE,
  R_HEAD, R_J0, R_ROW0
};

// ---------------------------------------------------------------- errors
__device__ __forceinline__ bool stopped(const Params& p) {
  return *(volatile uint32_t*)&p.err[E_CODE] != 0;
}

__device__ void report(const Params& p, uint32_t code, int task, int op, int bar, uint32_t val,
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

// Bounded wait on a shared-memory mbarrier phase, called by a whole warp.  All
// lanes poll; lane 0 alone decides to give up (stop word or time limit) and the
// decision is broadcast, so the warp leaves together.  false = give up.
__device__ bool wait_phase(const Params& p, uint64_t* bar, uint32_t parity, int task, int op,
                           unsigned mult = 1) {
  bool done = mbar_try_wait(bar, parity);
  if (__all_sync(0xffffffffu, done)) return true;
  const unsigned long long t0 = gtime_ns();
  for (uint32_t it = 1;; ++it) {
    done = done || mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((it & 63u) == 0) {
      int give = 0;
      if ((threadIdx.x & 31) == 0) {
        if (stopped(p)) {
          give = 1;
        } else if (gtime_ns() - t0 > mult * p.timeout_ns) {
          report(p, DEV_SMEM_TIMEOUT, task, op, -1, 0, parity);
          give = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, give, 0)) return false;
    }
  }
}

// bounded spin on a global counter (Listing 2's wait, with a time limit)
__device__ bool spin_counter(const Params& p, int bar, uint32_t target, int task, int op) {
  const uint32_t* c = p.bars + bar;
  uint32_t v = ld_acquire_u32(c);
  if (v >= target) return true;
  const unsigned long long t0 = gtime_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(32);
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

__device__ __forceinline__ int rows_down(const Params& p) { return p.wide ? kRowsDownW : kRowsDownN; }
__device__ __forceinline__ int rows_lm(const Params& p) { return p.wide ? kRowsLMW : kRowsLMN; }

// split-KV stage geometry: pages of all KV heads per stage
__device__ __forceinline__ int attn_page_bytes(const Params& p) { return p.hkv * p.P * p.d * 2; }
__device__ __forceinline__ int attn_pps(const Params& p) {
  const int pb = attn_page_bytes(p);
  return pb >= kStageData / 2 ? 1 : (kStageData / 2) / pb;
}

// ===================================================================== producer
// One warp.  Resolves each descriptor (claiming queue items for the drain
// opcodes), publishes the resolved task in the task ring and streams the
// task's weight / KV stages into the stage ring.
struct Prod {
  const Params& p;
  Smem& S;
  int lane;
  uint32_t stage_seq = 0, task_seq = 0;
  bool ok = true;

  __device__ Prod(const Params& pp, Smem& ss) : p(pp), S(ss), lane(threadIdx.x & 31) {}

  // reserve the next task slot and write the resolved words (lane j writes word j)
  __device__ bool push(const int32_t (&w)[kDescWords], int task, int op) {
    const uint32_t slot = task_seq % kTaskSlots;
    if (!wait_phase(p, &S.tempty[slot], ((task_seq / kTaskSlots) & 1u) ^ 1u, task, op)) return false;
    int32_t mine = 0;
#pragma unroll
    for (int j = 0; j < kDescWords; j++)
      if (lane == j) mine = w[j];
    S.task[slot][lane] = mine;
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.tfull[slot]);
    task_seq++;
    return true;
  }

  __device__ bool acquire_stage(uint32_t& slot, int task, int op) {
    slot = stage_seq % kStages;
    return wait_phase(p, &S.empty[slot], ((stage_seq / kStages) & 1u) ^ 1u, task, op);
  }

  // narrow path: rows [row0, row0 + nrows) of a row-major [*, K] matrix, whole
  // rows, one bulk copy per stage
  __device__ bool stream_rows(const uint16_t* w, int row0, int nrows, int K, int task, int op) {
    const int rps = narrow_rows_per_stage(K);
    for (int done = 0; done < nrows; done += rps) {
      const int rows = min(rps, nrows - done);
      uint32_t slot;
      if (!acquire_stage(slot, task, op)) return false;
      if (lane == 0) {
        const uint32_t bytes = (uint32_t)(rows * K * 2);
        mbar_arrive_expect_tx(&S.full[slot], bytes);
        bulk_g2s(&S.stage[slot][0], w + (size_t)(row0 + done) * K, bytes, &S.full[slot]);
      }
      __syncwarp();
      stage_seq++;
    }
    return true;
  }

  __device__ static int nst_rows(int nrows, int K) {
    const int rps = narrow_rows_per_stage(K);
    return (nrows + rps - 1) / rps;
  }

  // wide path: rg0 rows [row0a, +vr0) of wa, rg1 rows [row0b, +vr1) of wb; columns
  // [col0, col0 + K) of rows `stride` elements apart; 16-row stages padded per row
  __device__ bool stream_padded(const uint16_t* wa, int row0a, int vr0, const uint16_t* wb,
                                int row0b, int vr1, int nrg, int stride, int col0, int K, int task,
                                int op) {
    const int nks = (K + kStageKcMax - 1) / kStageKcMax;
    const int kc = K / nks;
    const int pitch = kc * 2 + (((kc * 2) % 128) == 0 ? 64 : 0);
    for (int rg = 0; rg < nrg; rg++) {
      const uint16_t* w = rg ? wb : wa;
      const int row0 = rg ? row0b : row0a;
      const int vr = rg ? vr1 : vr0;
      for (int ks = 0; ks < nks; ks++) {
        uint32_t slot;
        if (!acquire_stage(slot, task, op)) return false;
        if (lane == 0) mbar_arrive_expect_tx(&S.full[slot], (uint32_t)(vr * kc * 2));
        __syncwarp();
        if (lane < vr) {
          const uint16_t* src = w + (size_t)(row0 + lane) * stride + col0 + ks * kc;
          bulk_g2s(&S.stage[slot][lane * pitch], src, (uint32_t)(kc * 2), &S.full[slot]);
        }
        stage_seq++;
      }
    }
    return true;
  }

  __device__ static int nst_padded(int nrg, int K) {
    return nrg * ((K + kStageKcMax - 1) / kStageKcMax);
  }

  // pages [pg0, pg0 + npages) of sequence b, all KV heads: K pages then V pages
  __device__ bool stream_attn(int layer, int b, int pg0, int npages, int task) {
    const int pb = attn_page_bytes(p);
    const int pps = attn_pps(p);
    const uint16_t* kp = p.k_pool[layer];
    const uint16_t* vp = p.v_pool[layer];
    const size_t page_elems = (size_t)p.hkv * p.P * p.d;
    for (int st = 0; st * pps < npages; st++) {
      const int n = min(pps, npages - st * pps);
      int pg = -1;
      if (lane < 2 * n) pg = p.page_tables[(size_t)b * p.max_pages + pg0 + st * pps + (lane % n)];
      const bool bad = (lane < 2 * n) && (pg < 0 || pg >= p.num_pages);
      if (__any_sync(0xffffffffu, bad)) {
        if (bad) report(p, DEV_BAD_PAGE, task, OP_ATTN, -1, (uint32_t)pg, (uint32_t)p.num_pages);
        return false;
      }
      uint32_t slot;
      if (!acquire_stage(slot, task, OP_ATTN)) return false;
      if (lane == 0) mbar_arrive_expect_tx(&S.full[slot], (uint32_t)(2 * n * pb));
      __syncwarp();
      if (lane < n) {
        bulk_g2s(&S.stage[slot][lane * pb], kp + (size_t)pg * page_elems, (uint32_t)pb, &S.full[slot]);
      } else if (lane < 2 * n) {
        bulk_g2s(&S.stage[slot][(pps + lane - n) * pb], vp + (size_t)pg * page_elems, (uint32_t)pb,
                 &S.full[slot]);
      }
      stage_seq++;
    }
    return true;
  }

  __device__ void run() {
    const int sm = blockIdx.x;
    const int t_begin = p.task_off[sm], t_end = p.task_off[sm + 1];
    const int H = p.H, d = p.d;
    const bool wide = p.wide != 0;
    for (int ti = t_begin; ti < t_end && ok; ti++) {
      const int32_t word = p.tasks[(size_t)ti * kDescWords + lane];
      const int op = __shfl_sync(0xffffffffu, word, F_OP);
      const int l = __shfl_sync(0xffffffffu, word, F_LAYER);
      const int tile = __shfl_sync(0xffffffffu, word, F_TILE);
      int32_t r[kDescWords];
#pragma unroll
      for (int j = 0; j < kDescWords; j++) r[j] = 0;
      r[R_OP] = op;
      r[R_LAYER] = l;
      r[R_TILE] = tile;
      r[R_TASK] = ti;
      r[R_W0] = __shfl_sync(0xffffffffu, word, F_W0);
      r[R_T0] = __shfl_sync(0xffffffffu, word, F_T0);
      r[R_W1] = __shfl_sync(0xffffffffu, word, F_W1);
      r[R_T1] = __shfl_sync(0xffffffffu, word, F_T1);
      r[R_SIG] = __shfl_sync(0xffffffffu, word, F_SIG);
      r[R_INC] = __shfl_sync(0xffffffffu, word, F_INC);
      const int pw = __shfl_sync(0xffffffffu, word, F_PW);
      const int pt = __shfl_sync(0xffffffffu, word, F_PT);

      if (op == OP_NORM || op == OP_COMBINE) {
        r[R_NST] = 0;
        r[R_NRG] = __shfl_sync(0xffffffffu, word, F_ARG);
        ok = push(r, ti, op);
      } else if (op == OP_QKV) {
        const int tph = d / 32;                  // tiles per head
        const int head = tile / tph, j0 = (tile % tph) * kRowsQKVHalf;
        const uint16_t* w = p.w_qkv[l];
        const int ra = head * d + j0, rb = head * d + d / 2 + j0;
        r[R_HEAD] = head;
        r[R_J0] = j0;
        r[R_K] = H;
        r[R_NRG] = 2;
        r[R_VR0] = r[R_VR1] = kRowsQKVHalf;
        if (!wide) {
          r[R_NST] = 2 * nst_rows(kRowsQKVHalf, H);
          ok = push(r, ti, op) && stream_rows(w, ra, kRowsQKVHalf, H, ti, op) &&
               stream_rows(w, rb, kRowsQKVHalf, H, ti, op);
        } else {
          r[R_NST] = nst_padded(2, H);
          ok = push(r, ti, op) && stream_padded(w, ra, 16, w, rb, 16, 2, H, 0, H, ti, op);
        }
      } else if (op == OP_ROUTER) {
        const int row0 = tile * kRowsRouter;
        const int vr = min(kRowsRouter, p.E - row0);
        r[R_K] = H;
        r[R_NRG] = 1;
        r[R_VR0] = vr;
        r[R_ROW0] = row0;
        if (!wide) {
          r[R_NST] = nst_rows(vr, H);
          ok = push(r, ti, op) && stream_rows(p.w_router[l], row0, vr, H, ti, op);
        } else {
          r[R_NST] = nst_padded(1, H);
          ok = push(r, ti, op) &&
               stream_padded(p.w_router[l], row0, vr, nullptr, 0, 0, 1, H, 0, H, ti, op);
        }
      } else if (op == OP_OPROJ) {
        const uint16_t* w = p.w_o[l];
        if (!wide) {
          const int row0 = tile * kRowsOProj, K = p.hq * d;
          r[R_ROW0] = row0;
          r[R_G] = 0;
          r[R_K] = K;
          r[R_NRG] = 1;
          r[R_VR0] = kRowsOProj;
          r[R_NST] = nst_rows(kRowsOProj, K);
          ok = push(r, ti, op) && stream_rows(w, row0, kRowsOProj, K, ti, op);
        } else {
          const int per = H / kRowsOProj;
          const int g = tile / per, row0 = (tile % per) * kRowsOProj;
          const int K = p.grp * d;
          r[R_ROW0] = row0;
          r[R_G] = g;
          r[R_K] = K;
          r[R_NRG] = 2;
          r[R_VR0] = r[R_VR1] = 16;
          r[R_NST] = nst_padded(2, K);
          ok = push(r, ti, op) &&
               stream_padded(w, row0, 16, w, row0 + 16, 16, 2, p.hq * d, g * K, K, ti, op);
        }
      } else if (op == OP_LMHEAD) {
        const int rl = rows_lm(p);
        const int row0 = tile * rl;
        const int nrows = min(rl, p.V - row0);
        r[R_ROW0] = row0;
        r[R_K] = H;
        if (!wide) {
          r[R_NRG] = 1;
          r[R_VR0] = nrows;
          r[R_NST] = nst_rows(nrows, H);
          ok = push(r, ti, op) && stream_rows(p.lm_head, row0, nrows, H, ti, op);
        } else {
          const int vr0 = min(16, nrows), vr1 = max(0, nrows - 16);
          r[R_NRG] = vr1 > 0 ? 2 : 1;
          r[R_VR0] = vr0;
          r[R_VR1] = vr1;
          r[R_NST] = nst_padded(r[R_NRG], H);
          ok = push(r, ti, op) && stream_padded(p.lm_head, row0, vr0, p.lm_head, row0 + 16, vr1,
                                                r[R_NRG], H, 0, H, ti, op);
        }
      } else if (op == OP_ATTN) {
        uint32_t* claim = p.bars + bar_index(p, l, p.bl.claim + Q_ATTN);
        const int pps = attn_pps(p);
        while (ok) {
          uint32_t item = 0;
          if (lane == 0) item = atomicAdd(claim, 1u);
          item = __shfl_sync(0xffffffffu, item, 0);
          if ((int)item >= p.n_attn_items) break;
          const int32_t iw = lane < 8 ? p.attn_items[(size_t)item * 8 + lane] : 0;
          const int b = __shfl_sync(0xffffffffu, iw, AI_B);
          const int t0 = __shfl_sync(0xffffffffu, iw, AI_T0);
          const int t1 = __shfl_sync(0xffffffffu, iw, AI_T1);
          r[R_B] = b;
          r[R_TT0] = t0;
          r[R_TT1] = t1;
          r[R_NSPLIT] = __shfl_sync(0xffffffffu, iw, AI_NSPLIT);
          r[R_BASE] = __shfl_sync(0xffffffffu, iw, AI_BASE);
          r[R_POS] = __shfl_sync(0xffffffffu, iw, AI_POS);
          r[R_ITEM] = (int)item;
          r[R_W0] = -1;                    // per-group waits happen inside the task
          r[R_SIG] = bar_index(p, l, p.bl.items + b);
          r[R_INC] = 1;
          const int pg0 = t0 / p.P, npages = (t1 + p.P - 1) / p.P - pg0;
          r[R_NST] = (npages + pps - 1) / pps;
          ok = push(r, ti, op) && stream_attn(l, b, pg0, npages, ti);
        }
      } else if (op == OP_MOE_UP || op == OP_MOE_DOWN) {
        // producer-side wait: the queue is written by the route setup of this layer
        bool ready = true;
        if (lane == 0) ready = spin_counter(p, pw, (uint32_t)pt, ti, op);
        ready = __shfl_sync(0xffffffffu, (int)ready, 0) != 0;
        if (!ready) { ok = false; break; }
        const bool up = op == OP_MOE_UP;
        const int n_items = __ldcg(&p.qmeta[l * 4 + (up ? 0 : 1)]);
        const int cap = up ? p.max_up : p.max_down;
        uint32_t* claim = p.bars + bar_index(p, l, p.bl.claim + (up ? Q_UP : Q_DOWN));
        while (ok) {
          uint32_t item = 0;
          if (lane == 0) item = atomicAdd(claim, 1u);
          item = __shfl_sync(0xffffffffu, item, 0);
          if ((int)item >= n_items) break;
          if (n_items > cap) {
            if (lane == 0) report(p, DEV_BAD_ITEM, ti, op, -1, (uint32_t)n_items, (uint32_t)cap);
            ok = false;
            break;
          }
          const int32_t qv = __ldcg(&(up ? p.upq : p.downq)[(size_t)l * cap + item]);
          const int e = qv >> 16, t = qv & 0xffff;
          const int cnt = __ldcg(&p.ecnt[l * p.E + e]);
          const int off = __ldcg(&p.eoff[l * (p.E + 1) + e]);
          r[R_E] = e;
          r[R_TILE] = t;
          r[R_NTOK] = cnt;
          r[R_OFF] = off;
          r[R_ITEM] = (int)item;
          if (up) {
            r[R_K] = H;
            r[R_NRG] = 2;
            r[R_VR0] = r[R_VR1] = kRowsUp;
            r[R_W0] = bar_index(p, l, p.bl.x);
            r[R_T0] = 1;
            r[R_SIG] = bar_index(p, l, p.bl.up + e);
            r[R_INC] = 1;
            const size_t eo = (size_t)e * p.I * H;
            const uint16_t* wg = p.w_gate[l] + eo;
            const uint16_t* wu = p.w_up[l] + eo;
            if (!wide) {
              r[R_NST] = 2 * nst_rows(kRowsUp, H);
              ok = push(r, ti, op) && stream_rows(wg, t * kRowsUp, kRowsUp, H, ti, op) &&
                   stream_rows(wu, t * kRowsUp, kRowsUp, H, ti, op);
            } else {
              r[R_NST] = nst_padded(2, H);
              ok = push(r, ti, op) &&
                   stream_padded(wg, t * kRowsUp, 16, wu, t * kRowsUp, 16, 2, H, 0, H, ti, op);
            }
          } else {
            const int rd = rows_down(p);
            r[R_K] = p.I;
            r[R_W0] = bar_index(p, l, p.bl.up + e);
            r[R_T0] = p.I / kRowsUp;
            r[R_SIG] = bar_index(p, l, p.bl.moe);
            r[R_INC] = cnt;
            r[R_ROW0] = t * rd;
            const uint16_t* w = p.w_down[l] + (size_t)e * H * p.I;
            if (!wide) {
              r[R_NRG] = 1;
              r[R_VR0] = rd;
              r[R_NST] = nst_rows(rd, p.I);
              ok = push(r, ti, op) && stream_rows(w, t * rd, rd, p.I, ti, op);
            } else {
              r[R_NRG] = 2;
              r[R_VR0] = r[R_VR1] = 16;
              r[R_NST] = nst_padded(2, p.I);
              ok = push(r, ti, op) &&
                   stream_padded(w, t * rd, 16, w, t * rd + 16, 16, 2, p.I, 0, p.I, ti, op);
            }
          }
        }
      } else {
        if (lane == 0) report(p, DEV_BAD_OP, ti, op, -1, 0, 0);
        ok = false;
      }
    }
    if (ok) {
      int32_t r[kDescWords];
#pragma unroll
      for (int j = 0; j < kDescWords; j++) r[j] = 0;
      r[R_OP] = OP_END;
      ok = push(r, -1, OP_END);
    }
    if (!ok) {
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
__device__ __forceinline__ void split_bf16(const float* v, uint32_t& hi, uint32_t& lo) {
  // v[0], v[1] -> packed high halves and packed remainders (x = hi + lo to ~2^-17)
  const uint16_t h0 = f2bf(v[0]), h1 = f2bf(v[1]);
  const uint16_t l0 = f2bf(v[0] - bf16f(h0)), l1 = f2bf(v[1] - bf16f(h1));
  hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
  lo = (uint32_t)l0 | ((uint32_t)l1 << 16);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  return (uint32_t)f2bf(a) | ((uint32_t)f2bf(b) << 16);
}

struct Cons {
  const Params& p;
  Smem& S;
  const int tid, warp, lane, gl, cq;   // gl = lane / 4 (MMA group), cq = lane % 4
  const int32_t* t;                 // resolved task words, in its shared-memory slot
  uint32_t stage_seq;               // stages this warp has consumed
  uint32_t cphase;                  // consumer-barrier phases this warp has passed

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
    const bool ok = wait_phase(p, &S.cbar, cphase & 1u, t[R_TASK], t[R_OP], 2);
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
    if (tid == 0) S.t_ready = gtime_ns();
    return ok;
  }

  // publish: every consumer's global stores are done; one thread releases the counter
  __device__ __forceinline__ bool signal(int bar, int inc) {
    if (!csync()) return false;
    if (bar >= 0 && tid == 0) {
      __threadfence();
      atomicAdd(p.bars + bar, (uint32_t)inc);
    }
    return true;
  }

  __device__ __forceinline__ bool stage_full(uint32_t& slot) {
    slot = stage_seq % kStages;
    if (!wait_phase(p, &S.full[slot], (stage_seq / kStages) & 1u, t[R_TASK], t[R_OP])) {
      S.abort_flag = 1;
      return false;
    }
    return true;
  }

  __device__ __forceinline__ void stage_release(uint32_t slot) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
    stage_seq++;
  }

  __device__ __forceinline__ int ntok() const {
    return (t[R_OP] == OP_MOE_UP || t[R_OP] == OP_MOE_DOWN) ? t[R_NTOK] : p.B;
  }

  // fp32 activation row (B operand) for token slot n of this task, or nullptr
  __device__ __forceinline__ const float* operand_row(int n) {
    const int op = t[R_OP], l = t[R_LAYER];
    const size_t Bm = (size_t)p.Bmax;
    switch (op) {
      case OP_QKV:
      case OP_ROUTER:
        return n < p.B ? p.x + ((size_t)l * Bm + n) * p.H : nullptr;
      case OP_LMHEAD:
        return n < p.B ? p.x + ((size_t)p.L * Bm + n) * p.H : nullptr;
      case OP_OPROJ:
        return n < p.B ? p.attn_out + ((size_t)l * Bm + n) * p.hq * p.d + (size_t)t[R_G] * p.grp * p.d
                       : nullptr;
      case OP_MOE_UP: {
        if (n >= t[R_NTOK]) return nullptr;
        const int entry = __ldcg(&p.elist[(size_t)l * Bm * p.topk + t[R_OFF] + n]);
        return p.x + ((size_t)l * Bm + entry / p.topk) * p.H;
      }
      case OP_MOE_DOWN:
        if (n >= t[R_NTOK]) return nullptr;
        return p.abuf + ((size_t)l * Bm * p.topk + t[R_OFF] + n) * p.I;
    }
    return nullptr;
  }

  // ------------------------------------------------------ narrow GEMV
  // y[row][n] = sum_k W[row][k] x[n][k] over whole rows streamed 32 KB per
  // stage.  The contraction is cut into 256-column segments; warp w serves
  // segment w % nsegp (+ nsegp, ...) of rows w / nsegp, + wps, ...; lane l
  // multiplies columns seg * 256 + 8 l .. + 8 against fp32 activations held
  // in registers.  RB rows x NB tokens run as independent FMA chains and are
  // reduced across the warp together (transposed butterfly: 9 shuffles for 8
  // sums).  Segments are summed in a fixed order at the end of the tile.
  template <int NB>
  __device__ __forceinline__ bool gemv_narrow() {
    constexpr int NSG = NB <= 4 ? 2 : 1;           // segments per warp held in registers
    constexpr int RB = 8 / NB;                     // rows per independent group (RB * NB = 8)
    if (!wait_counter(t[R_W0], t[R_T0])) return false;
    if (!wait_counter(t[R_W1], t[R_T1])) return false;
    const int K = t[R_K];
    const int nt = ntok();
    const int rps = narrow_rows_per_stage(K);
    const int ksg = K < 256 ? K : 256;
    const int nseg = K / ksg;
    const int nsegp = nseg < 8 ? nseg : 8;         // warps sharing one row's segments
    const int wps = 8 / nsegp;                     // warps per segment slot
    const bool active = warp < nsegp * wps;
    const int nsg = (nseg + nsegp - 1) / nsegp;    // segments per warp
    const bool lane_on = lane * 8 < ksg;
    float* part = S.red;                           // [tile_row][seg][token]
    const int seg0 = warp % nsegp;
    const int rwarp = warp / nsegp;

    float xr[NSG][NB][8];
    auto load_x = [&](int sg_first) {
#pragma unroll
      for (int q = 0; q < NSG; q++) {
        const int seg = seg0 + (sg_first + q) * nsegp;
#pragma unroll
        for (int b = 0; b < NB; b++) {
          const float* row = (active && seg < nseg && lane_on) ? operand_row(b) : nullptr;
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
          if (row) {
            a = __ldcg((const float4*)(row + seg * ksg + lane * 8));
            c = __ldcg((const float4*)(row + seg * ksg + lane * 8 + 4));
          }
          xr[q][b][0] = a.x; xr[q][b][1] = a.y; xr[q][b][2] = a.z; xr[q][b][3] = a.w;
          xr[q][b][4] = c.x; xr[q][b][5] = c.y; xr[q][b][6] = c.z; xr[q][b][7] = c.w;
        }
      }
    };
    const bool reload = nsg > NSG;                 // only NB = 8 with > 8 segments
    if (!reload) load_x(0);

    const int nblk = t[R_NRG];
    int tile_row0 = 0;
    for (int blk = 0; blk < nblk; blk++) {
      const int brows = blk ? t[R_VR1] : t[R_VR0];
      for (int done = 0; done < brows; done += rps) {
        const int rows = min(rps, brows - done);
        uint32_t slot;
        if (!stage_full(slot)) return false;
        if (tid == 0 && blk == 0 && done == 0) S.t_mark[0] = gtime_ns();
        const uint8_t* base = S.stage[slot];
        for (int sg0 = 0; sg0 < nsg; sg0 += NSG) {
          if (reload) load_x(sg0);
#pragma unroll
          for (int q = 0; q < NSG; q++) {
            const int seg = seg0 + (sg0 + q) * nsegp;
            if (active && seg < nseg) {
              for (int r0 = rwarp; r0 < rows; r0 += RB * wps) {
                // RB rows r0, r0 + wps, ... as independent chains
                float acc[RB][NB];
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
                    acc[rr][b] = a;
                  }
                }
                // transposed butterfly over the 8 sums v[i] = acc[i / NB][i % NB]
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; i++) v[i] = acc[i / NB][i % NB];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                  const bool up = lane & 16;
                  const float send = up ? v[i] : v[i + 4];
                  const float keep = up ? v[i + 4] : v[i];
                  v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
#pragma unroll
                for (int i = 0; i < 2; i++) {
                  const bool up = lane & 8;
                  const float send = up ? v[i] : v[i + 2];
                  const float keep = up ? v[i + 2] : v[i];
                  v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                {
                  const bool up = lane & 4;
                  const float send = up ? v[0] : v[1];
                  const float keep = up ? v[1] : v[0];
                  v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                }
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
                if ((lane & 3) == 0) {
                  const int i = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
                  const int rr = i / NB, b = i % NB;
                  const int r = r0 + rr * wps;
                  if (r < rows && b < nt)
                    part[((tile_row0 + done + r) * nseg + seg) * nt + b] = v[0];
                }
              }
            }
          }
        }
        stage_release(slot);
      }
      tile_row0 += brows;
    }
    if (tid == 0) S.t_mark[1] = gtime_ns();
    if (!csync()) return false;
    // fixed-order sum over the contraction segments, in the epilogue's item order
    const bool paired = t[R_OP] == OP_QKV || t[R_OP] == OP_MOE_UP;
    const int R = paired ? 16 : t[R_VR0] + (t[R_NRG] > 1 ? t[R_VR1] : 0);
    for (int i = tid; i < R * nt; i += 256) {
      const int n = i / R, row = i % R;
      float s0 = 0.f, s1 = 0.f;
      for (int sg = 0; sg < nseg; sg++) s0 += part[(row * nseg + sg) * nt + n];
      S.tile_out[row][n] = s0;
      if (paired) {
        for (int sg = 0; sg < nseg; sg++) s1 += part[((row + 16) * nseg + sg) * nt + n];
        S.tile_out[row + 16][n] = s1;
      }
    }
    if (tid == 0) S.t_mark[2] = gtime_ns();
    return true;
  }

  // -------------------------------------------------------- wide GEMV
  // Tensor-core MMA on padded 16-row stages of up to 1024 columns;
  // activations rounded to BF16.  Geometry is runtime, register slots are
  // compile-time (at most 2 column stages x 4 chunks per warp).
  __device__ __forceinline__ bool gemv_wide() {
    if (!wait_counter(t[R_W0], t[R_T0])) return false;
    if (!wait_counter(t[R_W1], t[R_T1])) return false;
    const int K = t[R_K];
    const int nks = (K + kStageKcMax - 1) / kStageKcMax;
    const int kc = K / nks;
    const int nch = kc / 32;
    const int cpw = (nch + 7) / 8;
    const int pitch = kc * 2 + (((kc * 2) % 128) == 0 ? 64 : 0);
    const int nt = ntok();
    const bool two = nt > 8;

    uint4 xr[8][2];
    {
      const float* r0 = operand_row(gl);
      const float* r1 = two ? operand_row(gl + 8) : nullptr;
#pragma unroll
      for (int ks = 0; ks < 2; ks++)
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const int ch = warp + 8 * j;
          const int k0 = ks * kc + ch * 32 + 8 * cq;
          const bool on = ks < nks && ch < nch;
#pragma unroll
          for (int hf = 0; hf < 2; hf++) {
            const float* rr = hf ? r1 : r0;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (on && rr) {
              const float4 a = __ldcg((const float4*)(rr + k0));
              const float4 c = __ldcg((const float4*)(rr + k0 + 4));
              v = make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(c.x, c.y),
                             pack_bf16(c.z, c.w));
            }
            xr[ks * 4 + j][hf] = v;
          }
        }
    }

    const int nrg = t[R_NRG];
    float* red = S.red;   // [rg][warp][lane][8]
#pragma unroll
    for (int rg = 0; rg < 2; rg++) {
      if (rg < nrg) {
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < 2; ks++) {
          if (ks < nks) {
            uint32_t slot;
            if (!stage_full(slot)) return false;
            const uint8_t* base = S.stage[slot];
#pragma unroll
            for (int j = 0; j < 4; j++) {
              const int ch = warp + 8 * j;
              if (j < cpw && ch < nch) {
                const uint8_t* a = base + gl * pitch + ch * 64 + cq * 16;
                const uint4 lo = lds128(a);
                const uint4 hi = lds128(a + 8 * pitch);
                const uint4 b0 = xr[ks * 4 + j][0];
                mma_bf16(acc[0], lo.x, hi.x, lo.y, hi.y, b0.x, b0.y);
                mma_bf16(acc[0], lo.z, hi.z, lo.w, hi.w, b0.z, b0.w);
                if (two) {
                  const uint4 b1 = xr[ks * 4 + j][1];
                  mma_bf16(acc[1], lo.x, hi.x, lo.y, hi.y, b1.x, b1.y);
                  mma_bf16(acc[1], lo.z, hi.z, lo.w, hi.w, b1.z, b1.w);
                }
              }
            }
            stage_release(slot);
          }
        }
        float4* dst = (float4*)&red[((rg * kConsumerWarps + warp) * 32 + lane) * 8];
        dst[0] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
        dst[1] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
      }
    }
    if (!csync()) return false;
    // fixed-order sum over the warps, in the epilogue's item order
    const bool paired = t[R_OP] == OP_QKV || t[R_OP] == OP_MOE_UP;
    const int R = paired ? 16 : t[R_VR0] + (nrg > 1 ? t[R_VR1] : 0);
    for (int i = tid; i < R * nt; i += 256) {
      const int n = i / R, row0 = i % R;
#pragma unroll
      for (int pr = 0; pr < 2; pr++) {
        if (pr == 1 && !paired) break;
        const int row = row0 + pr * 16;
        const int rg = row >> 4, r = row & 15;
        const int ln = (r & 7) * 4 + ((n & 7) >> 1);
        const int idx = (n >> 3) * 4 + (r >> 3) * 2 + (n & 1);
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; w++) s += red[((rg * kConsumerWarps + w) * 32 + ln) * 8 + idx];
        S.tile_out[row][n] = s;
      }
    }
    return true;
  }

  // ---------------------------------------------------------- epilogues
  __device__ __forceinline__ bool epi_qkv() {
    const int l = t[R_LAYER], head = t[R_HEAD], j0 = t[R_J0];
    const int d = p.d, hq = p.hq, hkv = p.hkv;
    const size_t Bm = (size_t)p.Bmax;
    const bool rot = head < hq + hkv;
    for (int i = tid; i < 16 * p.B; i += 256) {
      const int n = i / 16, r = i % 16;
      float x1 = S.tile_out[r][n], x2 = S.tile_out[16 + r][n];
      if (rot) {
        const float c = p.rope[((size_t)n * (d / 2) + j0 + r) * 2 + 0];
        const float s = p.rope[((size_t)n * (d / 2) + j0 + r) * 2 + 1];
        const float y1 = x1 * c - x2 * s, y2 = x2 * c + x1 * s;
        x1 = y1;
        x2 = y2;
      }
      if (head < hq) {
        float* q = p.q + ((size_t)l * Bm + n) * hq * d + (size_t)head * d;
        __stcg(q + j0 + r, x1);
        __stcg(q + j0 + d / 2 + r, x2);
      } else {
        const uint16_t b1 = f2bf(x1), b2 = f2bf(x2);
        const bool isk = head < hq + hkv;
        const int g = isk ? head - hq : head - hq - hkv;
        uint16_t* nb = (isk ? p.knew : p.vnew) + ((size_t)l * Bm + n) * hkv * d + (size_t)g * d;
        __stcg(nb + j0 + r, b1);
        __stcg(nb + j0 + d / 2 + r, b2);
        const int pos = p.pos[n];
        const int pg = p.page_tables[(size_t)n * p.max_pages + pos / p.P];
        uint16_t* pool = (isk ? p.k_pool : p.v_pool)[l] +
                         (((size_t)pg * hkv + g) * p.P + (pos % p.P)) * d;
        pool[j0 + r] = b1;
        pool[j0 + d / 2 + r] = b2;
      }
    }
    const int grp_of = head < hq ? head / p.grp : (head < hq + hkv ? head - hq : head - hq - hkv);
    return signal(bar_index(p, l, p.bl.qkv + grp_of), 1);
  }

  __device__ __forceinline__ bool route_setup(int l) {
    const int E = p.E, K = p.topk, B = p.B;
    const size_t Bm = (size_t)p.Bmax;
    // route-setup scratch lives in the reduction buffer, idle after the GEMV
    int32_t* ecount = (int32_t*)S.red;        // [256]
    int32_t* eoffs = ecount + 256;            // [257]
    int32_t* eact = eoffs + 257;              // [257]
    // top-k per token: one warp per token, value descending, index ascending on ties
    for (int n = warp; n < B; n += kConsumerWarps) {
      float v[8];
      const float* rl = p.rlog + ((size_t)l * Bm + n) * E;
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldcg(rl + e) : -INFINITY;
      }
      uint32_t taken = 0;
      float vals[8];
      int idxs[8];
#pragma unroll
      for (int j = 0; j < 8; j++) {
        vals[j] = 0.f;
        idxs[j] = 0;
        if (j < K) {
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
          vals[j] = bv;
          idxs[j] = bi;
        }
      }
      if (lane == 0) {
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < 8; j++)
          if (j < K) den += expf(vals[j] - vals[0]);
#pragma unroll
        for (int j = 0; j < 8; j++) {
          if (j < K) {
            p.ridx[((size_t)l * Bm + n) * K + j] = idxs[j];
            p.rw[((size_t)l * Bm + n) * K + j] = expf(vals[j] - vals[0]) / den;
            S.sel[n][j] = idxs[j];
          }
        }
      }
    }
    if (!csync()) return false;
    // per-expert counts (thread e), exclusive scans of counts and of active experts
    for (int e = tid; e < E; e += 256) {
      int c = 0;
      for (int n = 0; n < B; n++)
        for (int j = 0; j < K; j++) c += S.sel[n][j] == e;
      ecount[e] = c;
    }
    if (!csync()) return false;
    if (warp == 0) {
      // warp-wide exclusive scan over E <= 256 experts, 8 per lane
      int cnt[8], act[8], sc = 0, sa = 0;
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const int e = lane * 8 + i;
        cnt[i] = e < E ? ecount[e] : 0;
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
        if (e < E) { eoffs[e] = oc; eact[e] = oa; }
        oc += cnt[i];
        oa += act[i];
      }
      if (lane == 31) { eoffs[E] = ic; eact[E] = ia; }
    }
    if (!csync()) return false;
    const int nu = p.I / kRowsUp, nd = p.H / rows_down(p);
    for (int e = tid; e < E; e += 256) {
      const int c = ecount[e], off = eoffs[e];
      p.ecnt[l * E + e] = c;
      p.eoff[l * (E + 1) + e] = off;
      if (c > 0) {
        int i = 0;
        for (int n = 0; n < B; n++)
          for (int j = 0; j < K; j++)
            if (S.sel[n][j] == e) p.elist[(size_t)l * Bm * K + off + i++] = n * K + j;
        const int a = eact[e];
        for (int u = 0; u < nu; u++) p.upq[(size_t)l * p.max_up + a * nu + u] = (e << 16) | u;
        for (int r = 0; r < nd; r++) p.downq[(size_t)l * p.max_down + a * nd + r] = (e << 16) | r;
      }
    }
    if (tid == 0) {
      p.eoff[l * (E + 1) + E] = eoffs[E];
      p.qmeta[l * 4 + 0] = eact[E] * nu;
      p.qmeta[l * 4 + 1] = eact[E] * nd;
      p.qmeta[l * 4 + 2] = eact[E];
    }
    return signal(bar_index(p, l, p.bl.route), 1);
  }

  __device__ __forceinline__ bool epi_router() {
    const int l = t[R_LAYER], row0 = t[R_ROW0], vr = t[R_VR0];
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < vr * p.B; i += 256) {
      const int n = i / vr, r = i % vr;
      __stcg(p.rlog + ((size_t)l * Bm + n) * p.E + row0 + r, S.tile_out[r][n]);
    }
    if (!csync()) return false;
    if (tid == 0) {
      __threadfence();
      S.bcast = (int)atom_add_acq_rel(p.bars + bar_index(p, l, p.bl.tk_router), 1u);
    }
    if (!csync()) return false;
    const int ntiles = (p.E + kRowsRouter - 1) / kRowsRouter;
    if (S.bcast == ntiles - 1) {
      __threadfence();
      return route_setup(l);
    }
    return true;
  }

  __device__ __forceinline__ bool epi_oproj() {
    const int l = t[R_LAYER], g = t[R_G], row0 = t[R_ROW0];
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < kRowsOProj * p.B; i += 256) {
      const int n = i / kRowsOProj, r = i % kRowsOProj;
      __stcg(p.oproj + (((size_t)l * p.hkv + g) * Bm + n) * p.H + row0 + r, S.tile_out[r][n]);
    }
    return signal(t[R_SIG], t[R_INC]);
  }

  __device__ __forceinline__ bool epi_lmhead() {
    const int row0 = t[R_ROW0];
    const int rows = t[R_VR0] + (t[R_NRG] > 1 ? t[R_VR1] : 0);
    for (int i = tid; i < rows * p.B; i += 256) {
      const int n = i / rows, r = i % rows;
      p.logits[(size_t)n * p.V + row0 + r] = S.tile_out[r][n];
    }
    return csync();
  }

  __device__ __forceinline__ bool epi_up() {
    const int l = t[R_LAYER], u = t[R_TILE], nt = t[R_NTOK], off = t[R_OFF];
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < kRowsUp * nt; i += 256) {
      const int n = i / kRowsUp, r = i % kRowsUp;
      const float gt = S.tile_out[r][n], ut = S.tile_out[kRowsUp + r][n];
      const float a = gt / (1.f + expf(-gt)) * ut;
      __stcg(p.abuf + ((size_t)l * Bm * p.topk + off + n) * p.I + u * kRowsUp + r, a);
    }
    return signal(t[R_SIG], t[R_INC]);
  }

  __device__ __forceinline__ bool epi_down() {
    const int l = t[R_LAYER], nt = t[R_NTOK], off = t[R_OFF], row0 = t[R_ROW0];
    const int rd = rows_down(p);
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < rd * nt; i += 256) {
      const int n = i / rd, r = i % rd;
      const int entry = __ldcg(&p.elist[(size_t)l * Bm * p.topk + off + n]);
      const int b = entry / p.topk, j = entry % p.topk;
      const float w = __ldcg(&p.rw[((size_t)l * Bm + b) * p.topk + j]);
      __stcg(p.ybuf + (((size_t)l * Bm + b) * p.topk + j) * p.H + row0 + r, w * S.tile_out[r][n]);
    }
    return signal(t[R_SIG], t[R_INC]);
  }

  // ------------------------------------------------------------ RMSNorm
  // h_l = h_{l-1} + O-proj_{l-1} + sum_j y_{l-1}[j]  (the embedding row at l = 0);
  // x_l = h_l / sqrt(mean(h_l^2) + eps) * gain.  Each thread owns 4-column
  // groups and issues all of its loads before adding (fixed order).
  __device__ __forceinline__ bool norm() {
    if (!wait_counter(t[R_W0], t[R_T0])) return false;
    if (!wait_counter(t[R_W1], t[R_T1])) return false;
    const int l = t[R_LAYER], H = p.H, B = p.B, K = p.topk;
    const int nop = p.wide ? p.hkv : 1;
    const size_t Bm = (size_t)p.Bmax;
    const int H4 = H / 4;
    for (int n = 0; n < B; n++) {
      float ssl = 0.f;
      for (int i4 = tid; i4 < H4; i4 += 256) {
        float4 h;
        if (l == 0) {
          const uint2 e = *(const uint2*)(p.embed + (size_t)p.tokens[n] * H + i4 * 4);
          h = make_float4(bf16lo(e.x), bf16hi(e.x), bf16lo(e.y), bf16hi(e.y));
        } else {
          float4 src[1 + 8 + 8];
          src[0] = __ldcg((const float4*)(p.h + ((size_t)(l - 1) * Bm + n) * H) + i4);
#pragma unroll
          for (int g = 0; g < 8; g++)
            if (g < nop)
              src[1 + g] = __ldcg((const float4*)(p.oproj + (((size_t)(l - 1) * p.hkv + g) * Bm + n) * H) + i4);
#pragma unroll
          for (int j = 0; j < 8; j++)
            if (j < K)
              src[9 + j] = __ldcg((const float4*)(p.ybuf + (((size_t)(l - 1) * Bm + n) * K + j) * H) + i4);
          h = src[0];
#pragma unroll
          for (int g = 0; g < 8; g++)
            if (g < nop) { h.x += src[1 + g].x; h.y += src[1 + g].y; h.z += src[1 + g].z; h.w += src[1 + g].w; }
#pragma unroll
          for (int j = 0; j < 8; j++)
            if (j < K) { h.x += src[9 + j].x; h.y += src[9 + j].y; h.z += src[9 + j].z; h.w += src[9 + j].w; }
        }
        __stcg((float4*)(p.h + ((size_t)l * Bm + n) * H) + i4, h);
        ssl += h.x * h.x + h.y * h.y + h.z * h.z + h.w * h.w;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ssl += __shfl_xor_sync(0xffffffffu, ssl, o);
      if (lane == 0) S.nred[warp][n] = ssl;
    }
    if (!csync()) return false;
    if (tid < B) {
      float sum = 0.f;
      for (int w = 0; w < kConsumerWarps; w++) sum += S.nred[w][tid];
      S.rinv[tid] = 1.0f / sqrtf(sum / (float)H + p.rms_eps);
    }
    if (!csync()) return false;
    const uint16_t* gain = l < p.L ? p.attn_norm[l] : p.final_norm;
    for (int i4 = tid; i4 < H4; i4 += 256) {
      const uint2 gv = *(const uint2*)(gain + i4 * 4);
      const float g0 = bf16lo(gv.x), g1 = bf16hi(gv.x), g2 = bf16lo(gv.y), g3 = bf16hi(gv.y);
      for (int n = 0; n < B; n++) {
        const float4 h = __ldcg((const float4*)(p.h + ((size_t)l * Bm + n) * H) + i4);
        const float r = S.rinv[n];
        __stcg((float4*)(p.x + ((size_t)l * Bm + n) * H) + i4,
               make_float4(h.x * r * g0, h.y * r * g1, h.z * r * g2, h.w * r * g3));
      }
    }
    return signal(t[R_SIG], t[R_INC]);
  }

  // -------------------------------------------------------- attention
  // One split-KV item: sequence b, keys [tt0, tt1), every KV head.  Warp w
  // serves KV group g = w % hkv and every NWG-th page of the item.
  template <int D>
  __device__ __forceinline__ bool attn() {
    constexpr int DPL = D / 32;           // head dims per lane in PV
    const int hkv = p.hkv, grp = p.grp, P = p.P;
    const int NWG = kConsumerWarps / hkv;
    const int g = warp % hkv, jw = warp / hkv;
    const int l = t[R_LAYER], b = t[R_B];
    const int tt0 = t[R_TT0], tt1 = t[R_TT1], pos = t[R_POS];
    const size_t Bm = (size_t)p.Bmax;
    const int hb = P * D * 2;             // bytes of one head's 16-token page
    const int pb = hkv * hb;              // bytes of one page, all heads
    const int pps = attn_pps(p);
    // this step's QKV of every group must be done (q, and the new K/V)
    if (tid == 0) {
      for (int gg = 0; gg < hkv && !S.abort_flag; gg++)
        if (!spin_counter(p, bar_index(p, l, p.bl.qkv + gg), (uint32_t)((grp + 2) * (D / 32)),
                          t[R_TASK], OP_ATTN))
          S.abort_flag = 1;
    }
    if (!csync()) return false;
    if (tid == 0) S.t_ready = gtime_ns();

    // query fragments (B operand) split into BF16 high and low halves
    uint4 qh[D / 32], ql[D / 32];
    {
      const float* qrow = p.q + ((size_t)l * Bm + b) * p.hq * D + (size_t)(g * grp + gl) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ch++) {
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (gl < grp) {
          const float4 a = __ldcg((const float4*)(qrow + ch * 32 + 8 * cq));
          const float4 c = __ldcg((const float4*)(qrow + ch * 32 + 8 * cq + 4));
          v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
        }
        split_bf16(v + 0, qh[ch].x, ql[ch].x);
        split_bf16(v + 2, qh[ch].y, ql[ch].y);
        split_bf16(v + 4, qh[ch].z, ql[ch].z);
        split_bf16(v + 6, qh[ch].w, ql[ch].w);
      }
    }
    const uint16_t* kn = p.knew + ((size_t)l * Bm + b) * hkv * D + (size_t)g * D;
    const uint16_t* vn = p.vnew + ((size_t)l * Bm + b) * hkv * D + (size_t)g * D;

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[8][DPL];
#pragma unroll
    for (int h = 0; h < 8; h++)
#pragma unroll
      for (int j = 0; j < DPL; j++) o[h][j] = 0.f;

    const int pg0 = tt0 / P;
    const int npages = (tt1 + P - 1) / P - pg0;
    const int nst = t[R_NST];
    const float sc = p.attn_scale_log2;
    for (int st = 0; st < nst; st++) {
      uint32_t slot;
      if (!stage_full(slot)) return false;
      if (tid == 0 && st == 0) S.t_mark[0] = gtime_ns();
      for (int qi = 0; qi < pps; qi++) {
        const int page = st * pps + qi;
        if (page >= npages || page % NWG != jw) continue;
        uint8_t* kp = S.stage[slot] + qi * pb + g * hb;
        uint8_t* vp = S.stage[slot] + (pps + qi) * pb + g * hb;
        const int tk0 = (pg0 + page) * P;
        const bool has_new = pos >= tk0 && pos < tk0 + P;
        // the new token's K/V come from this step's QKV output, not the pool
        if (has_new) {
          const int row = pos - tk0;
          if (D == 128) {
            ((uint2*)(kp + row * D * 2))[lane] = __ldcg(((const uint2*)kn) + lane);
            ((uint2*)(vp + row * D * 2))[lane] = __ldcg(((const uint2*)vn) + lane);
          } else {
            ((uint32_t*)(kp + row * D * 2))[lane] = __ldcg(((const uint32_t*)kn) + lane);
            ((uint32_t*)(vp + row * D * 2))[lane] = __ldcg(((const uint32_t*)vn) + lane);
          }
          __syncwarp();
        }
        // scores: 16 tokens x 8 heads, q = high + low halves
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ch = 0; ch < D / 32; ch++) {
          const uint8_t* a = kp + gl * D * 2 + ch * 64 + cq * 16;
          const uint4 lo = lds128(a);
          const uint4 hi = lds128(a + 8 * D * 2);
          mma_bf16(s, lo.x, hi.x, lo.y, hi.y, qh[ch].x, qh[ch].y);
          mma_bf16(s, lo.z, hi.z, lo.w, hi.w, qh[ch].z, qh[ch].w);
          mma_bf16(s, lo.x, hi.x, lo.y, hi.y, ql[ch].x, ql[ch].y);
          mma_bf16(s, lo.z, hi.z, lo.w, hi.w, ql[ch].z, ql[ch].w);
        }
        const int lo_t = max(tt0 - tk0, 0), hi_t = min(tt1 - tk0, P);   // valid rows [lo_t, hi_t)
        const bool v0 = gl >= lo_t && gl < hi_t, v1 = gl + 8 >= lo_t && gl + 8 < hi_t;
        s[0] = v0 ? s[0] * sc : -INFINITY;
        s[1] = v0 ? s[1] * sc : -INFINITY;
        s[2] = v1 ? s[2] * sc : -INFINITY;
        s[3] = v1 ? s[3] * sc : -INFINITY;
        float pr[4];
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          float mx = fmaxf(s[hh], s[2 + hh]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m_run[hh], mx);
          const float al = (mn == -INFINITY) ? 1.f : exp2f(m_run[hh] - mn);
          pr[hh] = (mn == -INFINITY) ? 0.f : exp2f(s[hh] - mn);
          pr[2 + hh] = (mn == -INFINITY) ? 0.f : exp2f(s[2 + hh] - mn);
          float sm = pr[hh] + pr[2 + hh];
          sm += __shfl_xor_sync(0xffffffffu, sm, 4);
          sm += __shfl_xor_sync(0xffffffffu, sm, 8);
          sm += __shfl_xor_sync(0xffffffffu, sm, 16);
          l_run[hh] = l_run[hh] * al + sm;
          m_run[hh] = mn;
          if (gl == 0) S.alpha[warp][2 * cq + hh] = al;
        }
        S.pbuf[warp][gl][2 * cq] = pr[0];
        S.pbuf[warp][gl][2 * cq + 1] = pr[1];
        S.pbuf[warp][gl + 8][2 * cq] = pr[2];
        S.pbuf[warp][gl + 8][2 * cq + 1] = pr[3];
        __syncwarp();
        {
          const float4 a0 = *(const float4*)&S.alpha[warp][0];
          const float4 a1 = *(const float4*)&S.alpha[warp][4];
          const float al[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
          for (int h = 0; h < 8; h++)
#pragma unroll
            for (int j = 0; j < DPL; j++) o[h][j] *= al[h];
        }
#pragma unroll 2
        for (int tk = lo_t; tk < hi_t; tk++) {
          const float4 p0 = *(const float4*)&S.pbuf[warp][tk][0];
          const float4 p1 = *(const float4*)&S.pbuf[warp][tk][4];
          const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          float vv[DPL];
          if (DPL == 4) {
            const uint2 u = *(const uint2*)(vp + tk * D * 2 + lane * 8);
            vv[0] = bf16lo(u.x);
            vv[1] = bf16hi(u.x);
            vv[2 % DPL] = bf16lo(u.y);
            vv[3 % DPL] = bf16hi(u.y);
          } else {
            const uint32_t u = *(const uint32_t*)(vp + tk * D * 2 + lane * 4);
            vv[0] = bf16lo(u);
            vv[1 % DPL] = bf16hi(u);
          }
#pragma unroll
          for (int h = 0; h < 8; h++)
#pragma unroll
            for (int j = 0; j < DPL; j++) o[h][j] = fmaf(pv[h], vv[j], o[h][j]);
        }
        if (has_new) fence_proxy_async_smem();
        __syncwarp();
      }
      stage_release(slot);
    }

    if (tid == 0) S.t_mark[1] = gtime_ns();
    // merge the NWG warps of each KV group (fixed order), write the item's partials
    if (gl == 0) {
      S.wstat[warp][2 * cq][0] = m_run[0];
      S.wstat[warp][2 * cq][1] = l_run[0];
      S.wstat[warp][2 * cq + 1][0] = m_run[1];
      S.wstat[warp][2 * cq + 1][1] = l_run[1];
    }
    if (!csync()) return false;
    float myscale[8];
#pragma unroll
    for (int h = 0; h < 8; h++) {
      float mx = -INFINITY;
      for (int j = 0; j < NWG; j++) mx = fmaxf(mx, S.wstat[j * hkv + g][h][0]);
      const float mw = S.wstat[warp][h][0];
      myscale[h] = (mw == -INFINITY) ? 0.f : exp2f(mw - mx);
    }
    const int item = t[R_ITEM];
    float* red = S.red;   // [warp][8 heads][64 dims]
    constexpr int HALF = 64;
    constexpr int NPASS = D / HALF;
#pragma unroll
    for (int pass = 0; pass < NPASS; pass++) {
#pragma unroll
      for (int j = 0; j < DPL; j++) {
        const int dd = lane * DPL + j;
        if (dd >= pass * HALF && dd < (pass + 1) * HALF) {
#pragma unroll
          for (int h = 0; h < 8; h++) red[(warp * 8 + h) * 64 + (dd - pass * HALF)] = o[h][j] * myscale[h];
        }
      }
      if (!csync()) return false;
      for (int i = tid; i < hkv * grp * HALF; i += 256) {
        const int gg = i / (grp * HALF), h = (i / HALF) % grp, dl = i % HALF;
        float sum = 0.f;
        for (int j = 0; j < NWG; j++) sum += red[((j * hkv + gg) * 8 + h) * 64 + dl];
        const size_t it = ((size_t)item * hkv + gg) * grp + h;
        __stcg(p.attn_part + it * D + pass * HALF + dl, sum);
        if (pass == 0 && dl == 0) {
          float mx = -INFINITY;
          for (int j = 0; j < NWG; j++) mx = fmaxf(mx, S.wstat[j * hkv + gg][h][0]);
          float ls = 0.f;
          for (int j = 0; j < NWG; j++) {
            const float mw = S.wstat[j * hkv + gg][h][0];
            ls += (mw == -INFINITY) ? 0.f : S.wstat[j * hkv + gg][h][1] * exp2f(mw - mx);
          }
          __stcg(p.attn_ml + it * 2 + 0, mx);
          __stcg(p.attn_ml + it * 2 + 1, ls);
        }
      }
      if (!csync()) return false;
    }
    if (tid == 0) S.t_mark[2] = gtime_ns();
    return signal(t[R_SIG], t[R_INC]);
  }

  // ATTN_COMBINE of (sequence b, KV group g, heads [h0, h0 + hpt)): merge the
  // sequence's split-KV partials.  Warp w takes splits w, w + 8, ...; lane l
  // dims 4 l .. 4 l + 3; the warps' partial sums meet in shared memory and
  // are added in a fixed order.
  __device__ __forceinline__ bool combine() {
    const int l = t[R_LAYER], hkv = p.hkv, grp = p.grp, D = p.d;
    const int cpg = t[R_NRG];                  // combine tasks per (sequence, KV group)
    const int hp = grp / cpg;                  // heads per task
    const int b = t[R_TILE] / (hkv * cpg), g = (t[R_TILE] / cpg) % hkv, h0 = (t[R_TILE] % cpg) * hp;
    const int base = p.attn_meta[b * 2], nsplit = p.attn_meta[b * 2 + 1];
    if (!wait_counter(t[R_W0], nsplit)) return false;
    const size_t Bm = (size_t)p.Bmax;
    const bool lon = lane * 4 < D;
    // pass 1: per-head maximum
    float mx[8];
#pragma unroll
    for (int h = 0; h < 8; h++) mx[h] = -INFINITY;
    for (int s = warp; s < nsplit; s += kConsumerWarps) {
      const float* ml = p.attn_ml + ((size_t)(base + s) * hkv + g) * grp * 2;
#pragma unroll
      for (int h = 0; h < 8; h++)
        if (h < hp) mx[h] = fmaxf(mx[h], __ldcg(ml + (h0 + h) * 2));
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < 8; h++)
        if (h < hp) S.wstat[warp][h][0] = mx[h];
    }
    if (!csync()) return false;
#pragma unroll
    for (int h = 0; h < 8; h++) {
      if (h < hp) {
        float m = -INFINITY;
        for (int w = 0; w < kConsumerWarps; w++) m = fmaxf(m, S.wstat[w][h][0]);
        mx[h] = m;
      }
    }
    // pass 2: weighted sums of this warp's splits
    float num[8][4], den[8];
#pragma unroll
    for (int h = 0; h < 8; h++) {
      den[h] = 0.f;
      num[h][0] = num[h][1] = num[h][2] = num[h][3] = 0.f;
    }
#pragma unroll 2
    for (int s = warp; s < nsplit; s += kConsumerWarps) {
      const size_t it0 = ((size_t)(base + s) * hkv + g) * grp;
#pragma unroll
      for (int h = 0; h < 8; h++) {
        if (h < hp) {
          const float2 ml = __ldcg((const float2*)(p.attn_ml + (it0 + h0 + h) * 2));
          const float w = exp2f(ml.x - mx[h]);
          den[h] += w * ml.y;
          if (lon) {
            const float4 ov = __ldcg((const float4*)(p.attn_part + (it0 + h0 + h) * D + lane * 4));
            num[h][0] += w * ov.x;
            num[h][1] += w * ov.y;
            num[h][2] += w * ov.z;
            num[h][3] += w * ov.w;
          }
        }
      }
    }
    if (!csync()) return false;   // every warp has read the maxima
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < 8; h++)
        if (h < hp) S.wstat[warp][h][1] = den[h];
    }
    float* red = S.red;            // [warp][head][D] for up to 4 heads per pass
    for (int hb = 0; hb < hp; hb += 4) {
#pragma unroll
      for (int h = 0; h < 8; h++) {
        if (h >= hb && h < hb + 4 && h < hp && lon) {
          float* dst = red + ((size_t)(warp * 4 + (h - hb)) * D + lane * 4);
          dst[0] = num[h][0]; dst[1] = num[h][1]; dst[2] = num[h][2]; dst[3] = num[h][3];
        }
      }
      if (!csync()) return false;
      const int nh = min(4, hp - hb);
      for (int i = tid; i < nh * D; i += 256) {
        const int hh = i / D, dd = i % D;
        float sn = 0.f, sd = 0.f;
        for (int w = 0; w < kConsumerWarps; w++) {
          sn += red[(w * 4 + hh) * D + dd];
          sd += S.wstat[w][hb + hh][1];
        }
        __stcg(p.attn_out + ((size_t)l * Bm + b) * p.hq * D + (size_t)(g * grp + h0 + hb + hh) * D + dd,
               sn / sd);
      }
      if (!csync()) return false;
    }
    return signal(t[R_SIG], 1);
  }
};

// One out-of-line function per consumer path: each gets its own register
// allocation (the nine-warp block caps a thread at 168 registers, and the
// union of every path in one function would spill).  The per-warp pipeline
// counters travel through shared memory.
template <int NB>
__device__ __noinline__ bool op_gemv_narrow(const Params& p, Smem& S, const int32_t* t) {
  Cons c(p, S, t);
  const bool ok = c.gemv_narrow<NB>();
  c.save();
  return ok;
}

__device__ __noinline__ bool op_gemv_wide(const Params& p, Smem& S, const int32_t* t) {
  Cons c(p, S, t);
  const bool ok = c.gemv_wide();
  c.save();
  return ok;
}

__device__ __noinline__ bool op_epilogue(const Params& p, Smem& S, const int32_t* t) {
  Cons c(p, S, t);
  bool ok = false;
  switch (t[R_OP]) {
    case OP_QKV: ok = c.epi_qkv(); break;
    case OP_ROUTER: ok = c.epi_router(); break;
    case OP_OPROJ: ok = c.epi_oproj(); break;
    case OP_LMHEAD: ok = c.epi_lmhead(); break;
    case OP_MOE_UP: ok = c.epi_up(); break;
    case OP_MOE_DOWN: ok = c.epi_down(); break;
  }
  c.save();
  return ok;
}

template <int D>
__device__ __noinline__ bool op_attn(const Params& p, Smem& S, const int32_t* t) {
  Cons c(p, S, t);
  const bool ok = c.attn<D>();
  c.save();
  return ok;
}

__device__ __noinline__ bool op_norm(const Params& p, Smem& S, const int32_t* t) {
  Cons c(p, S, t);
  const bool ok = c.norm();
  c.save();
  return ok;
}

__device__ __noinline__ bool op_combine(const Params& p, Smem& S, const int32_t* t) {
  Cons c(p, S, t);
  const bool ok = c.combine();
  c.save();
  return ok;
}

__device__ __forceinline__ bool op_gemv(const Params& p, Smem& S, const int32_t* t) {
  if (p.wide) return op_gemv_wide(p, S, t);
  const int op = t[R_OP];
  const int nt = (op == OP_MOE_UP || op == OP_MOE_DOWN) ? t[R_NTOK] : p.B;
  bool ok;
  if (nt <= 1) ok = op_gemv_narrow<1>(p, S, t);
  else if (nt <= 2) ok = op_gemv_narrow<2>(p, S, t);
  else if (nt <= 4) ok = op_gemv_narrow<4>(p, S, t);
  else ok = op_gemv_narrow<8>(p, S, t);
  return ok && op_epilogue(p, S, t);
}

// consumer main loop: take the next resolved task, run it, record its timeline
__device__ __forceinline__ void consumer_loop(const Params& p, Smem& S) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t task_seq = 0;
  int n_rec = 0;
  while (true) {
    const uint32_t slot = task_seq % kTaskSlots;
    if (!wait_phase(p, &S.tfull[slot], (task_seq / kTaskSlots) & 1u, -1, -1)) break;
    const int32_t* t = S.task[slot];
    task_seq++;
    const int op = t[R_OP];
    if (op == OP_END) break;
    const unsigned long long t_start = gtime_ns();
    if (tid == 0) {
      S.t_ready = t_start;
      S.t_mark[0] = S.t_mark[1] = S.t_mark[2] = S.t_mark[3] = t_start;
    }
    bool ok = false;
    switch (op) {
      case OP_NORM: ok = op_norm(p, S, t); break;
      case OP_QKV:
      case OP_ROUTER:
      case OP_OPROJ:
      case OP_LMHEAD:
      case OP_MOE_UP:
      case OP_MOE_DOWN: ok = op_gemv(p, S, t); break;
      case OP_ATTN: ok = (p.d == 128) ? op_attn<128>(p, S, t) : op_attn<64>(p, S, t); break;
      case OP_COMBINE: ok = op_combine(p, S, t); break;
    }
    if (p.trace && tid == 0 && n_rec < p.trace_cap) {
      const unsigned long long t_end = gtime_ns();
      int32_t* rec = p.trace + ((size_t)blockIdx.x * p.trace_cap + n_rec) * 16;
      const bool item = op == OP_ATTN || op == OP_MOE_UP || op == OP_MOE_DOWN;
      rec[0] = op;
      rec[1] = t[R_LAYER];
      rec[2] = item ? t[R_ITEM] : t[R_TILE];
      rec[3] = (int32_t)(uint32_t)(t_start & 0xffffffffull);
      rec[4] = (int32_t)(uint32_t)(t_start >> 32);
      rec[5] = (int32_t)(S.t_ready - t_start);
      rec[6] = (int32_t)(t_end - t_start);
      rec[7] = blockIdx.x;
      for (int k = 0; k < 3; k++) rec[8 + k] = (int32_t)(S.t_mark[k] - t_start);
      n_rec++;
    }
    // the task's words are no longer needed: hand the slot back to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.tempty[slot]);
    if (!ok || S.abort_flag) break;
  }
}

__global__ void __launch_bounds__(kThreads, 1) mk_step_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
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
    for (int w = 0; w < kConsumerWarps; w++) S.cstage[w] = S.cphase[w] = 0;
    for (int w = 0; w < kConsumerWarps; w++) {
      S.seen_bar[w] = -1;
      S.seen_tgt[w] = 0;
    }
    S.abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if ((int)(threadIdx.x >> 5) == kConsumerWarps) {
    Prod pr(p, S);
    pr.run();
  } else {
    consumer_loop(p, S);
  }
}

size_t step_smem_bytes() { return sizeof(Smem); }

cudaError_t launch_step(const Params& p, int n_sm, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(mk_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(Smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_sm);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mk_step_kernel, p);
}

}  // namespace mk
