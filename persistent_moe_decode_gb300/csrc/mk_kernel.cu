// The persistent decode-step kernel for GB300 (sm_103a).
//
// "Inside the megakernel serving engine for North Mini Code":
//  - §What is a Megakernel / Fig 2: one thread block per SM stays resident for
//    the whole step and walks a host-built per-SM task list in global memory;
//  - §The threadblock shape / Listing 1: one fixed block shape for every
//    opcode, a warp that fetches descriptors ahead of the workers, worker
//    warps that never use __syncthreads (their own barrier excludes the
//    fetcher), weight tiles prefetched before the cross-SM wait on activations;
//  - §Barriers / Listing 2: counters in global memory, spun on with a
//    bounded wait, released after a fence, O(1) in fan-in and fan-out;
//  - §The task scheduler, dynamic part: ATTN / MOE claimers atomically take
//    the next item of a shared queue until it is exhausted.
//
// GB300 design (not the pages' H100 one):
//  - block = 8 consumer warps + 1 producer warp.  The producer resolves the
//    task list (descriptors, queue claims, page tables) and streams every
//    weight / KV byte HBM -> shared memory with 1-D bulk async copies into a
//    5-stage ring of 33 KB stages guarded by mbarriers.  Because each stage
//    holds up to 16 rows of any GEMV tile or 4 KV pages, the ring runs ahead
//    across task boundaries of different opcodes: a task waiting for its
//    activations already has its weights in flight.
//  - GEMV tiles use the warp-level BF16 tensor-core MMA with the weights as
//    the 16-row operand and up to 16 tokens as the 8/16-wide operand; the
//    eight warps split the contraction and reduce once per tile in shared
//    memory (fixed order: results are deterministic).
//  - split-KV attention: QK^T on the tensor cores (tokens x 8 query heads of
//    one GQA group), online softmax in fp32, PV on the CUDA cores; the last
//    split of a (sequence, KV head) merges all splits (ticket counter).
//  - the last router tile of a layer runs top-k and route setup (ticket
//    counter), the residual add + RMSNorm is one task per layer.
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
  float red[2][kConsumerWarps][32][8];      // per-tile cross-warp reduction / attention merge
  float tile_out[32][kMaxBatch];            // reduced tile: [row][token]
  float pbuf[kConsumerWarps][16][8];        // attention probabilities of one page per warp
  float alpha[kConsumerWarps][8];           // attention rescale per head per warp
  float wstat[kConsumerWarps][8][2];        // attention (max, sum) per warp per head
  float nred[kConsumerWarps][kMaxBatch];    // norm reductions
  float rinv[kMaxBatch];
  int32_t sel[kMaxBatch][8];                // router top-k of the last tile
  int32_t ecount[256];                      // route setup scratch
  int32_t eoffs[257];
  int32_t eact[257];
  int32_t task[kTaskSlots][kDescWords];     // resolved task ring
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[kTaskSlots];
  uint64_t tempty[kTaskSlots];
  uint64_t cbar;                            // bounded barrier of the 8 consumer warps
  volatile int32_t abort_flag;
  int32_t bcast;
};

// resolved task words (written by the producer into the task ring)
enum : int {
  R_OP = 0, R_LAYER, R_NST, R_K, R_NRG, R_VR0, R_VR1, R_W0, R_T0, R_W1, R_T1, R_SIG, R_INC,
  R_TILE, R_E, R_NTOK, R_OFF, R_TASK, R_B, R_G, R_TT0, R_TT1, R_POS, R_NSPLIT, R_ITEM, R_BASE,
  R_HEAD, R_J0
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

  // rg0 rows [row0a, +vr0) of wa, rg1 rows [row0b, +vr1) of wb; columns [col0, col0 + K)
  __device__ bool stream_gemv(const uint16_t* wa, int row0a, int vr0, const uint16_t* wb,
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

  // pages [pg0, pg0 + npages) of sequence b, KV head g: K pages then V pages per stage
  __device__ bool stream_attn(int layer, int b, int g, int pg0, int npages, int task) {
    const int pb = p.P * p.d * 2;
    const int pps = (kStageRows * kStageKcMax * 2) / (2 * pb);
    const uint16_t* kp = p.k_pool[layer];
    const uint16_t* vp = p.v_pool[layer];
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
        const uint16_t* src = kp + ((size_t)pg * p.hkv + g) * p.P * p.d;
        bulk_g2s(&S.stage[slot][lane * pb], src, (uint32_t)pb, &S.full[slot]);
      } else if (lane < 2 * n) {
        const uint16_t* src = vp + ((size_t)pg * p.hkv + g) * p.P * p.d;
        bulk_g2s(&S.stage[slot][pps * pb + (lane - n) * pb], src, (uint32_t)pb, &S.full[slot]);
      }
      stage_seq++;
    }
    return true;
  }

  __device__ static int nstages_gemv(int nrg, int K) {
    return nrg * ((K + kStageKcMax - 1) / kStageKcMax);
  }

  __device__ void run() {
    const int sm = blockIdx.x;
    const int t_begin = p.task_off[sm], t_end = p.task_off[sm + 1];
    const int L = p.L, H = p.H, d = p.d;
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

      if (op == OP_NORM) {
        r[R_NST] = 0;
        ok = push(r, ti, op);
      } else if (op == OP_QKV) {
        const int tph = d / 32;                  // tiles per head
        const int head = tile / tph, j0 = (tile % tph) * 16;
        r[R_HEAD] = head;
        r[R_J0] = j0;
        r[R_K] = H;
        r[R_NRG] = 2;
        r[R_VR0] = r[R_VR1] = 16;
        r[R_NST] = nstages_gemv(2, H);
        const uint16_t* w = p.w_qkv[l];
        ok = push(r, ti, op) &&
             stream_gemv(w, head * d + j0, 16, w, head * d + d / 2 + j0, 16, 2, H, 0, H, ti, op);
      } else if (op == OP_ROUTER) {
        const int row0 = tile * kRowsRouter;
        r[R_K] = H;
        r[R_NRG] = 1;
        r[R_VR0] = min(16, p.E - row0);
        r[R_NST] = nstages_gemv(1, H);
        ok = push(r, ti, op) &&
             stream_gemv(p.w_router[l], row0, r[R_VR0], nullptr, 0, 0, 1, H, 0, H, ti, op);
      } else if (op == OP_OPROJ) {
        const int per = H / kRowsOProj;
        const int g = tile / per, row0 = (tile % per) * kRowsOProj;
        const int K = p.grp * d;
        r[R_G] = g;
        r[R_K] = K;
        r[R_NRG] = 2;
        r[R_VR0] = r[R_VR1] = 16;
        r[R_NST] = nstages_gemv(2, K);
        const uint16_t* w = p.w_o[l];
        ok = push(r, ti, op) &&
             stream_gemv(w, row0, 16, w, row0 + 16, 16, 2, p.hq * d, g * K, K, ti, op);
      } else if (op == OP_LMHEAD) {
        const int row0 = tile * kRowsLM;
        const int vr0 = min(16, p.V - row0), vr1 = max(0, min(16, p.V - row0 - 16));
        r[R_K] = H;
        r[R_NRG] = vr1 > 0 ? 2 : 1;
        r[R_VR0] = vr0;
        r[R_VR1] = vr1;
        r[R_NST] = nstages_gemv(r[R_NRG], H);
        ok = push(r, ti, op) && stream_gemv(p.lm_head, row0, vr0, p.lm_head, row0 + 16, vr1,
                                            r[R_NRG], H, 0, H, ti, op);
      } else if (op == OP_ATTN) {
        uint32_t* claim = p.bars + bar_index(p, l, p.bl.claim + Q_ATTN);
        while (ok) {
          uint32_t item = 0;
          if (lane == 0) item = atomicAdd(claim, 1u);
          item = __shfl_sync(0xffffffffu, item, 0);
          if ((int)item >= p.n_attn_items) break;
          const int32_t iw = lane < 8 ? p.attn_items[(size_t)item * 8 + lane] : 0;
          const int b = __shfl_sync(0xffffffffu, iw, AI_B);
          const int g = __shfl_sync(0xffffffffu, iw, AI_G);
          const int t0 = __shfl_sync(0xffffffffu, iw, AI_T0);
          const int t1 = __shfl_sync(0xffffffffu, iw, AI_T1);
          r[R_B] = b;
          r[R_G] = g;
          r[R_TT0] = t0;
          r[R_TT1] = t1;
          r[R_NSPLIT] = __shfl_sync(0xffffffffu, iw, AI_NSPLIT);
          r[R_BASE] = __shfl_sync(0xffffffffu, iw, AI_BASE);
          r[R_POS] = __shfl_sync(0xffffffffu, iw, AI_POS);
          r[R_ITEM] = (int)item;
          r[R_W0] = bar_index(p, l, p.bl.qkv + g);
          r[R_T0] = (p.grp + 2) * (d / 32);
          r[R_SIG] = bar_index(p, l, p.bl.attn + g);
          r[R_INC] = 1;
          const int pg0 = t0 / p.P, npages = (t1 + p.P - 1) / p.P - pg0;
          const int pps = (kStageRows * kStageKcMax) / (2 * p.P * d);
          r[R_NST] = (npages + pps - 1) / pps;
          ok = push(r, ti, op) && stream_attn(l, b, g, pg0, npages, ti);
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
            r[R_VR0] = r[R_VR1] = 16;
            r[R_NST] = nstages_gemv(2, H);
            r[R_W0] = bar_index(p, l, p.bl.x);
            r[R_T0] = 1;
            r[R_SIG] = bar_index(p, l, p.bl.up + e);
            r[R_INC] = 1;
            const size_t eo = (size_t)e * p.I * H;
            ok = push(r, ti, op) && stream_gemv(p.w_gate[l] + eo, t * kRowsUp, 16, p.w_up[l] + eo,
                                                t * kRowsUp, 16, 2, H, 0, H, ti, op);
          } else {
            r[R_K] = p.I;
            r[R_NRG] = 2;
            r[R_VR0] = r[R_VR1] = 16;
            r[R_NST] = nstages_gemv(2, p.I);
            r[R_W0] = bar_index(p, l, p.bl.up + e);
            r[R_T0] = p.I / kRowsUp;
            r[R_SIG] = bar_index(p, l, p.bl.moe);
            r[R_INC] = cnt;
            const uint16_t* w = p.w_down[l] + (size_t)e * H * p.I;
            ok = push(r, ti, op) && stream_gemv(w, t * kRowsDown, 16, w, t * kRowsDown + 16, 16, 2,
                                                p.I, 0, p.I, ti, op);
          }
        }
      } else {
        if (lane == 0) report(p, DEV_BAD_OP, ti, op, -1, 0, 0);
        ok = false;
      }
    }
    (void)L;
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
      for (uint32_t s = first; s < n; s++) {
        const unsigned long long t0 = gtime_ns();
        while (!mbar_try_wait(&S.full[s % kStages], (s / kStages) & 1u)) {
          if (gtime_ns() - t0 > p.timeout_ns) break;
        }
      }
    }
  }
};

// ===================================================================== consumers
struct Cons {
  const Params& p;
  Smem& S;
  const int tid, warp, lane, gl, cq;   // gl = lane / 4 (MMA group), cq = lane % 4
  uint32_t stage_seq = 0;
  uint32_t cphase = 0;
  int32_t t[kDescWords];

  __device__ Cons(const Params& pp, Smem& ss)
      : p(pp), S(ss), tid(threadIdx.x), warp(threadIdx.x >> 5), lane(threadIdx.x & 31),
        gl((threadIdx.x & 31) >> 2), cq(threadIdx.x & 3) {}

  __device__ bool aborted() { return S.abort_flag != 0; }

  // Barrier of the 8 consumer warps (the producer never joins).  It is an
  // mbarrier with a bounded wait rather than bar.sync, so a warp that has
  // already left after an error cannot leave the others waiting forever.
  __device__ bool csync() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.cbar);
    const bool ok = wait_phase(p, &S.cbar, cphase & 1u, t[R_TASK], t[R_OP], 2);
    cphase++;
    if (!ok) S.abort_flag = 1;
    return ok && !aborted();
  }

  // cross-SM wait (thread 0 spins, the other consumers wait at the named barrier)
  __device__ bool wait_counter(int bar, int target) {
    if (bar < 0) return true;
    if (tid == 0) {
      if (!spin_counter(p, bar, (uint32_t)target, t[R_TASK], t[R_OP])) S.abort_flag = 1;
    }
    return csync();
  }

  // publish: every consumer's global stores are done; one thread releases the counter
  __device__ bool signal(int bar, int inc) {
    if (!csync()) return false;
    if (bar >= 0 && tid == 0) {
      __threadfence();
      atomicAdd(p.bars + bar, (uint32_t)inc);
    }
    return true;
  }

  __device__ bool stage_full(uint32_t& slot) {
    slot = stage_seq % kStages;
    if (!wait_phase(p, &S.full[slot], (stage_seq / kStages) & 1u, t[R_TASK], t[R_OP])) {
      S.abort_flag = 1;
      return false;
    }
    return true;
  }

  __device__ void stage_release(uint32_t slot) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
    stage_seq++;
  }

  // ------------------------------------------------------------------ GEMV
  // B-operand row (token) pointers for the two token halves this lane feeds.
  __device__ const uint16_t* operand_row(int n) {
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

  template <int K>
  __device__ bool gemv() {
    constexpr int NKS = (K + kStageKcMax - 1) / kStageKcMax;
    constexpr int KC = K / NKS;
    constexpr int NCH = KC / 32;             // 32-column chunks per stage row
    constexpr int CPW = (NCH + 7) / 8;       // chunks per warp per stage
    constexpr int PITCH = KC * 2 + (((KC * 2) % 128) == 0 ? 64 : 0);
    static_assert(KC % 32 == 0 && KC <= kStageKcMax, "unsupported contraction length");

    if (!wait_counter(t[R_W0], t[R_T0])) return false;
    if (!wait_counter(t[R_W1], t[R_T1])) return false;
    const int ntok = (t[R_OP] == OP_MOE_UP || t[R_OP] == OP_MOE_DOWN) ? t[R_NTOK] : p.B;
    const bool two = ntok > 8;

    // activation fragments for this warp's chunks, loaded once per tile
    uint4 xr[NKS * CPW][2];
    {
      const uint16_t* r0 = operand_row(gl);
      const uint16_t* r1 = two ? operand_row(gl + 8) : nullptr;
#pragma unroll
      for (int ks = 0; ks < NKS; ks++)
#pragma unroll
        for (int j = 0; j < CPW; j++) {
          const int ch = warp + 8 * j;
          const int k0 = ks * KC + ch * 32 + 8 * cq;
          uint4 z = make_uint4(0, 0, 0, 0);
          xr[ks * CPW + j][0] = (ch < NCH && r0) ? __ldcg((const uint4*)(r0 + k0)) : z;
          xr[ks * CPW + j][1] = (ch < NCH && r1) ? __ldcg((const uint4*)(r1 + k0)) : z;
        }
    }

    const int nrg = t[R_NRG];
#pragma unroll
    for (int rg = 0; rg < 2; rg++) {
      if (rg < nrg) {
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < NKS; ks++) {
          uint32_t slot;
          if (!stage_full(slot)) return false;
          const uint8_t* base = S.stage[slot];
#pragma unroll
          for (int j = 0; j < CPW; j++) {
            const int ch = warp + 8 * j;
            if (ch < NCH) {
              const uint8_t* a = base + gl * PITCH + ch * 64 + cq * 16;
              const uint4 lo = lds128(a);
              const uint4 hi = lds128(a + 8 * PITCH);
              const uint4 b0 = xr[ks * CPW + j][0];
              mma_bf16(acc[0], lo.x, hi.x, lo.y, hi.y, b0.x, b0.y);
              mma_bf16(acc[0], lo.z, hi.z, lo.w, hi.w, b0.z, b0.w);
              if (two) {
                const uint4 b1 = xr[ks * CPW + j][1];
                mma_bf16(acc[1], lo.x, hi.x, lo.y, hi.y, b1.x, b1.y);
                mma_bf16(acc[1], lo.z, hi.z, lo.w, hi.w, b1.z, b1.w);
              }
            }
          }
          stage_release(slot);
        }
        float4* dst = (float4*)&S.red[rg][warp][lane][0];
        dst[0] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
        dst[1] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
      }
    }
    if (!csync()) return false;
    // fixed-order reduction over the 8 warps: tile_out[rg * 16 + r][n]
    const int nout = nrg * 16 * ntok;
    for (int i = tid; i < nout; i += 256) {
      const int n = i % ntok, row = i / ntok;
      const int rg = row >> 4, r = row & 15;
      const int ln = (r & 7) * 4 + ((n & 7) >> 1);
      const int idx = (n >> 3) * 4 + (r >> 3) * 2 + (n & 1);
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; w++) s += S.red[rg][w][ln][idx];
      S.tile_out[row][n] = s;
    }
    if (!csync()) return false;
    return true;
  }

  __device__ bool run_gemv_k() {
    switch (t[R_K]) {
      case 128: return gemv<128>();
      case 256: return gemv<256>();
      case 512: return gemv<512>();
      case 768: return gemv<768>();
      case 1024: return gemv<1024>();
      case 2048: return gemv<2048>();
    }
    if (tid == 0) report(p, DEV_BAD_OP, t[R_TASK], t[R_OP], -1, (uint32_t)t[R_K], 0);
    S.abort_flag = 1;
    return false;
  }

  // ---------------------------------------------------------- epilogues
  __device__ bool epi_qkv() {
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
      const uint16_t b1 = f2bf(x1), b2 = f2bf(x2);
      if (head < hq) {
        uint16_t* q = p.q + ((size_t)l * Bm + n) * hq * d + (size_t)head * d;
        __stcg(q + j0 + r, b1);
        __stcg(q + j0 + d / 2 + r, b2);
      } else {
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

  __device__ bool route_setup(int l) {
    const int E = p.E, K = p.topk, B = p.B;
    const size_t Bm = (size_t)p.Bmax;
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
        vals[j] = bv;
        idxs[j] = bi;
      }
      if (lane == 0) {
        float den = 0.f;
        for (int j = 0; j < K; j++) den += expf(vals[j] - vals[0]);
        for (int j = 0; j < K; j++) {
          p.ridx[((size_t)l * Bm + n) * K + j] = idxs[j];
          p.rw[((size_t)l * Bm + n) * K + j] = expf(vals[j] - vals[0]) / den;
          S.sel[n][j] = idxs[j];
        }
      }
    }
    if (!csync()) return false;
    // per-expert counts (thread e), exclusive scans of counts and of active experts
    for (int e = tid; e < E; e += 256) {
      int c = 0;
      for (int n = 0; n < B; n++)
        for (int j = 0; j < K; j++) c += S.sel[n][j] == e;
      S.ecount[e] = c;
    }
    if (!csync()) return false;
    if (tid == 0) {
      int off = 0, act = 0;
      for (int e = 0; e < E; e++) {
        S.eoffs[e] = off;
        S.eact[e] = act;
        off += S.ecount[e];
        act += S.ecount[e] > 0;
      }
      S.eoffs[E] = off;
      S.eact[E] = act;
    }
    if (!csync()) return false;
    const int nu = p.I / kRowsUp, nd = p.H / kRowsDown;
    for (int e = tid; e < E; e += 256) {
      const int c = S.ecount[e], off = S.eoffs[e];
      p.ecnt[l * E + e] = c;
      p.eoff[l * (E + 1) + e] = off;
      if (c > 0) {
        int i = 0;
        for (int n = 0; n < B; n++)
          for (int j = 0; j < K; j++)
            if (S.sel[n][j] == e) p.elist[(size_t)l * Bm * K + off + i++] = n * K + j;
        const int a = S.eact[e];
        for (int u = 0; u < nu; u++) p.upq[(size_t)l * p.max_up + a * nu + u] = (e << 16) | u;
        for (int r = 0; r < nd; r++) p.downq[(size_t)l * p.max_down + a * nd + r] = (e << 16) | r;
      }
    }
    if (tid == 0) {
      p.eoff[l * (E + 1) + E] = S.eoffs[E];
      p.qmeta[l * 4 + 0] = S.eact[E] * nu;
      p.qmeta[l * 4 + 1] = S.eact[E] * nd;
      p.qmeta[l * 4 + 2] = S.eact[E];
    }
    return signal(bar_index(p, l, p.bl.route), 1);
  }

  __device__ bool epi_router() {
    const int l = t[R_LAYER], row0 = t[R_TILE] * kRowsRouter, vr = t[R_VR0];
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < 16 * p.B; i += 256) {
      const int n = i / 16, r = i % 16;
      if (r < vr) __stcg(p.rlog + ((size_t)l * Bm + n) * p.E + row0 + r, S.tile_out[r][n]);
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

  __device__ bool epi_oproj() {
    const int l = t[R_LAYER], g = t[R_G];
    const int row0 = (t[R_TILE] % (p.H / kRowsOProj)) * kRowsOProj;
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < 32 * p.B; i += 256) {
      const int n = i / 32, r = i % 32;
      __stcg(p.oproj + (((size_t)l * p.hkv + g) * Bm + n) * p.H + row0 + r, S.tile_out[r][n]);
    }
    return signal(t[R_SIG], t[R_INC]);
  }

  __device__ bool epi_lmhead() {
    const int row0 = t[R_TILE] * kRowsLM;
    const int rows = t[R_VR0] + (t[R_NRG] > 1 ? t[R_VR1] : 0);
    for (int i = tid; i < 32 * p.B; i += 256) {
      const int n = i / 32, r = i % 32;
      if (r < rows) p.logits[(size_t)n * p.V + row0 + r] = S.tile_out[r][n];
    }
    return csync();
  }

  __device__ bool epi_up() {
    const int l = t[R_LAYER], u = t[R_TILE], ntok = t[R_NTOK], off = t[R_OFF];
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < 16 * ntok; i += 256) {
      const int n = i / 16, r = i % 16;
      const float gt = S.tile_out[r][n], ut = S.tile_out[16 + r][n];
      const float a = gt / (1.f + expf(-gt)) * ut;
      __stcg(p.abuf + ((size_t)l * Bm * p.topk + off + n) * p.I + u * kRowsUp + r, f2bf(a));
    }
    return signal(t[R_SIG], t[R_INC]);
  }

  __device__ bool epi_down() {
    const int l = t[R_LAYER], tile = t[R_TILE], ntok = t[R_NTOK], off = t[R_OFF];
    const size_t Bm = (size_t)p.Bmax;
    for (int i = tid; i < 32 * ntok; i += 256) {
      const int n = i / 32, r = i % 32;
      const int entry = __ldcg(&p.elist[(size_t)l * Bm * p.topk + off + n]);
      const int b = entry / p.topk, j = entry % p.topk;
      const float w = __ldcg(&p.rw[((size_t)l * Bm + b) * p.topk + j]);
      __stcg(p.ybuf + (((size_t)l * Bm + b) * p.topk + j) * p.H + tile * kRowsDown + r,
             w * S.tile_out[r][n]);
    }
    return signal(t[R_SIG], t[R_INC]);
  }

  // ------------------------------------------------------------ RMSNorm
  // h_l = h_{l-1} + sum_g oproj_{l-1}[g] + sum_j y_{l-1}[j]  (embedding row at l = 0);
  // x_l = bf16(h_l / sqrt(mean(h_l^2) + eps) * gain)
  __device__ bool norm() {
    if (!wait_counter(t[R_W0], t[R_T0])) return false;
    if (!wait_counter(t[R_W1], t[R_T1])) return false;
    const int l = t[R_LAYER], H = p.H, B = p.B, K = p.topk;
    const size_t Bm = (size_t)p.Bmax;
    float ss[kMaxBatch];
#pragma unroll
    for (int n = 0; n < kMaxBatch; n++) ss[n] = 0.f;
    for (int i = tid; i < H; i += 256) {
#pragma unroll
      for (int n = 0; n < kMaxBatch; n++) {
        if (n < B) {
          float h;
          if (l == 0) {
            h = bf16f(p.embed[(size_t)p.tokens[n] * H + i]);
          } else {
            h = __ldcg(p.h + ((size_t)(l - 1) * Bm + n) * H + i);
            for (int g = 0; g < p.hkv; g++)
              h += __ldcg(p.oproj + (((size_t)(l - 1) * p.hkv + g) * Bm + n) * H + i);
            for (int j = 0; j < K; j++)
              h += __ldcg(p.ybuf + (((size_t)(l - 1) * Bm + n) * K + j) * H + i);
          }
          __stcg(p.h + ((size_t)l * Bm + n) * H + i, h);
          ss[n] += h * h;
        }
      }
    }
#pragma unroll
    for (int n = 0; n < kMaxBatch; n++) {
      float v = ss[n];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) S.nred[warp][n] = v;
    }
    if (!csync()) return false;
    if (tid < B) {
      float s = 0.f;
      for (int w = 0; w < kConsumerWarps; w++) s += S.nred[w][tid];
      S.rinv[tid] = 1.0f / sqrtf(s / (float)H + p.rms_eps);
    }
    if (!csync()) return false;
    const uint16_t* gain = l < p.L ? p.attn_norm[l] : p.final_norm;
    for (int i = tid; i < H; i += 256) {
      const float gi = bf16f(gain[i]);
      for (int n = 0; n < B; n++) {
        const float h = __ldcg(p.h + ((size_t)l * Bm + n) * H + i);
        __stcg(p.x + ((size_t)l * Bm + n) * H + i, f2bf(h * S.rinv[n] * gi));
      }
    }
    return signal(t[R_SIG], t[R_INC]);
  }

  // -------------------------------------------------------- attention
  template <int D>
  __device__ bool attn() {
    constexpr int DPL = D / 32;           // head dims per lane in PV
    constexpr int PB = 16 * D * 2;        // bytes of one 16-token page of one head
    constexpr int PPS = (kStageRows * kStageKcMax * 2) / (2 * PB);   // pages per stage
    constexpr int NWG = kConsumerWarps / PPS;                        // warp groups
    const int l = t[R_LAYER], b = t[R_B], g = t[R_G], grp = p.grp;
    const int tt0 = t[R_TT0], tt1 = t[R_TT1], pos = t[R_POS];
    const size_t Bm = (size_t)p.Bmax;
    if (!wait_counter(t[R_W0], t[R_T0])) return false;

    // query fragments (B operand): head gl of the group, dims ch*32 + 8*cq .. +8
    uint4 qf[D / 32];
    {
      const uint16_t* qrow = p.q + ((size_t)l * Bm + b) * p.hq * D + (size_t)(g * grp + gl) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ch++)
        qf[ch] = gl < grp ? __ldcg((const uint4*)(qrow + ch * 32 + 8 * cq)) : make_uint4(0, 0, 0, 0);
    }
    const uint16_t* kn = p.knew + ((size_t)l * Bm + b) * p.hkv * D + (size_t)g * D;
    const uint16_t* vn = p.vnew + ((size_t)l * Bm + b) * p.hkv * D + (size_t)g * D;

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[8][DPL];
#pragma unroll
    for (int h = 0; h < 8; h++)
#pragma unroll
      for (int j = 0; j < DPL; j++) o[h][j] = 0.f;

    const int pg0 = tt0 / 16;
    const int npages = (tt1 + 15) / 16 - pg0;
    const int nst = t[R_NST];
    const float sc = p.attn_scale_log2;
    for (int st = 0; st < nst; st++) {
      uint32_t slot;
      if (!stage_full(slot)) return false;
      const int pidx = warp - (st % NWG) * PPS;
      const int page = st * PPS + pidx;
      if (pidx >= 0 && pidx < PPS && page < npages) {
        uint8_t* kp = S.stage[slot] + pidx * PB;
        uint8_t* vp = S.stage[slot] + PPS * PB + pidx * PB;
        const int tk0 = (pg0 + page) * 16;
        // the new token's K/V come from this step's QKV output, not the pool
        if (pos >= tk0 && pos < tk0 + 16) {
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
        // scores: 16 tokens x 8 heads
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ch = 0; ch < D / 32; ch++) {
          const uint8_t* a = kp + gl * D * 2 + ch * 64 + cq * 16;
          const uint4 lo = lds128(a);
          const uint4 hi = lds128(a + 8 * D * 2);
          mma_bf16(s, lo.x, hi.x, lo.y, hi.y, qf[ch].x, qf[ch].y);
          mma_bf16(s, lo.z, hi.z, lo.w, hi.w, qf[ch].z, qf[ch].w);
        }
        const int lo_t = max(tt0 - tk0, 0), hi_t = min(tt1 - tk0, 16);   // valid rows [lo_t, hi_t)
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
        for (int tk = lo_t; tk < hi_t; tk++) {
          const float4 p0 = *(const float4*)&S.pbuf[warp][tk][0];
          const float4 p1 = *(const float4*)&S.pbuf[warp][tk][4];
          const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          float vv[DPL];
          if (DPL == 4) {
            const uint2 u = *(const uint2*)(vp + tk * D * 2 + lane * 8);
            vv[0] = bf16lo(u.x);
            vv[1] = bf16hi(u.x);
            vv[2] = bf16lo(u.y);
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
        if (pos >= tk0 && pos < tk0 + 16) fence_proxy_async_smem();
        __syncwarp();
      }
      stage_release(slot);
    }

    // merge the eight warps' partial softmax states (fixed order)
    if (gl == 0) {
      S.wstat[warp][2 * cq][0] = m_run[0];
      S.wstat[warp][2 * cq][1] = l_run[0];
      S.wstat[warp][2 * cq + 1][0] = m_run[1];
      S.wstat[warp][2 * cq + 1][1] = l_run[1];
    }
    if (!csync()) return false;
    float M[8], Ls[8], myscale[8];
#pragma unroll
    for (int h = 0; h < 8; h++) {
      float mx = -INFINITY;
      for (int w = 0; w < kConsumerWarps; w++) mx = fmaxf(mx, S.wstat[w][h][0]);
      float ls = 0.f;
      for (int w = 0; w < kConsumerWarps; w++) {
        const float mw = S.wstat[w][h][0];
        ls += (mw == -INFINITY) ? 0.f : S.wstat[w][h][1] * exp2f(mw - mx);
      }
      M[h] = mx;
      Ls[h] = ls;
      const float mw = S.wstat[warp][h][0];
      myscale[h] = (mw == -INFINITY) ? 0.f : exp2f(mw - mx);
    }
    const int item = t[R_ITEM], nsplit = t[R_NSPLIT];
    float* red = &S.red[0][0][0][0];   // [8 warps][8 heads][64 dims]
    constexpr int HALF = D < 64 ? D : 64;
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
      for (int i = tid; i < grp * HALF; i += 256) {
        const int h = i / HALF, dl = i % HALF, dd = pass * HALF + dl;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; w++) sum += red[(w * 8 + h) * 64 + dl];
        if (nsplit == 1) {
          __stcg(p.attn_out + ((size_t)l * Bm + b) * p.hq * D + (size_t)(g * grp + h) * D + dd,
                 f2bf(sum / Ls[h]));
        } else {
          __stcg(p.attn_part + ((size_t)item * grp + h) * D + dd, sum);
          if (dd == 0) {
            __stcg(p.attn_ml + ((size_t)item * grp + h) * 2 + 0, M[h]);
            __stcg(p.attn_ml + ((size_t)item * grp + h) * 2 + 1, Ls[h]);
          }
        }
      }
      if (!csync()) return false;
    }
    if (nsplit > 1) {
      // the last split of (sequence, KV head) to finish merges all of them
      if (tid == 0) {
        __threadfence();
        S.bcast = (int)atom_add_acq_rel(p.bars + bar_index(p, l, p.bl.tk_attn + b * p.hkv + g), 1u);
      }
      if (!csync()) return false;
      if (S.bcast != nsplit - 1) return true;
      __threadfence();
      const int base = t[R_BASE];
      for (int i = tid; i < grp * (D / 4); i += 256) {
        const int h = i / (D / 4), dq = (i % (D / 4)) * 4;
        float mx = -INFINITY;
        for (int sidx = 0; sidx < nsplit; sidx++)
          mx = fmaxf(mx, __ldcg(p.attn_ml + ((size_t)(base + sidx) * grp + h) * 2));
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        float den = 0.f;
        for (int sidx = 0; sidx < nsplit; sidx++) {
          const size_t it = (size_t)(base + sidx) * grp + h;
          const float w = exp2f(__ldcg(p.attn_ml + it * 2) - mx);
          den += w * __ldcg(p.attn_ml + it * 2 + 1);
          const float4 ov = __ldcg((const float4*)(p.attn_part + it * D + dq));
          num.x += w * ov.x;
          num.y += w * ov.y;
          num.z += w * ov.z;
          num.w += w * ov.w;
        }
        uint16_t* dst = p.attn_out + ((size_t)l * Bm + b) * p.hq * D + (size_t)(g * grp + h) * D + dq;
        const float inv = 1.f / den;
        __stcg(dst + 0, f2bf(num.x * inv));
        __stcg(dst + 1, f2bf(num.y * inv));
        __stcg(dst + 2, f2bf(num.z * inv));
        __stcg(dst + 3, f2bf(num.w * inv));
      }
    }
    return signal(t[R_SIG], t[R_INC]);
  }

  // ------------------------------------------------------------ main loop
  __device__ void run() {
    uint32_t task_seq = 0;
    while (true) {
      const uint32_t slot = task_seq % kTaskSlots;
      if (!wait_phase(p, &S.tfull[slot], (task_seq / kTaskSlots) & 1u, -1, -1)) break;
#pragma unroll
      for (int j = 0; j < kDescWords; j++) t[j] = S.task[slot][j];
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.tempty[slot]);
      task_seq++;
      const int op = t[R_OP];
      if (op == OP_END) break;
      bool ok = true;
      switch (op) {
        case OP_NORM: ok = norm(); break;
        case OP_QKV: ok = run_gemv_k() && epi_qkv(); break;
        case OP_ROUTER: ok = run_gemv_k() && epi_router(); break;
        case OP_OPROJ: ok = run_gemv_k() && epi_oproj(); break;
        case OP_LMHEAD: ok = run_gemv_k() && epi_lmhead(); break;
        case OP_MOE_UP: ok = run_gemv_k() && epi_up(); break;
        case OP_MOE_DOWN: ok = run_gemv_k() && epi_down(); break;
        case OP_ATTN: ok = (p.d == 128) ? attn<128>() : attn<64>(); break;
        default: ok = false;
      }
      if (!ok || aborted()) break;
    }
  }
};

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
    S.abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if ((int)(threadIdx.x >> 5) == kConsumerWarps) {
    Prod pr(p, S);
    pr.run();
  } else {
    Cons cs(p, S);
    cs.run();
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
