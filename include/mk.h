/*
 * mk.h — C ABI of the GB300 persistent MoE decode step.
 *
 * One decode step of a BF16 parallel-layer MoE transformer runs as ONE
 * persistent kernel: one thread block per SM stays resident for the whole
 * step and walks a host-built per-SM task list ("Inside the megakernel serving
 * engine for North Mini Code", §What is a Megakernel, Fig 2).  Dependencies
 * between tiles are global-memory counters that producers increment and
 * consumers spin on (§Barriers, Listing 2).  Work whose size depends on the
 * live sequence lengths or on the routing is cut at run time: the split-KV
 * items on the host; the routed experts' rows on the device once the routing
 * is known, into equal shares with one token and, with several tokens, into
 * fixed-size tiles that the expert-branch SMs claim from per-layer counters
 * (the pages' shared queues; §The task scheduler, the dynamic part).
 *
 * The host side mirrors the pages' decode service loop (§The serving engine
 * around the kernel: update_kv_page_tables, clear_scratch_and_barriers,
 * select_schedule(max_live_context), launch_megakernel):
 *   mk_create         validate the model, record the caller's weight and KV
 *                     pool pointers, allocate counters / scratch / queues;
 *   mk_schedule_step  snapshot one batch (tokens, page tables, lengths) into
 *                     the step's device state and pick the split-KV schedule;
 *   mk_decode_step    clear the counters and launch the persistent kernel;
 *   mk_step_status    read the device error word after the stream has synced.
 *
 * Conventions for every call:
 *   - Return 0 (MK_OK) or a negative MK_ERR_* code.  Nothing throws across
 *     the ABI; mk_strerror() names a code.
 *   - "device" pointers are CUDA global-memory addresses on the device that
 *     was current at mk_create; "host" pointers are ordinary host memory.
 *   - A handle is single-stream and not thread-safe: calls on one handle
 *     must not overlap.  Different handles are independent.
 *   - BF16 values are IEEE bfloat16 bit patterns; all layouts are row-major.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_ABI_VERSION 1

enum mk_status {
  MK_OK = 0,
  MK_ERR_BAD_CONFIG = -1,      /* unsupported or inconsistent model / config      */
  MK_ERR_OOM = -2,             /* device or pinned-host allocation failed         */
  MK_ERR_BAD_PAGE = -3,        /* a page index needed this step is out of range   */
  MK_ERR_BATCH_TOO_LARGE = -4, /* batch > config.max_batch or batch < 1           */
  MK_ERR_NOT_SCHEDULED = -5,   /* mk_decode_step without a preceding schedule     */
  MK_ERR_TIMEOUT = -6,         /* a device-side wait ran past config.timeout_ms   */
  MK_ERR_CUDA = -7,            /* a CUDA runtime call failed (no GPU, launch ...) */
  MK_ERR_BAD_ARG = -8,         /* NULL handle / pointer, bad length, bad token    */
  MK_ERR_DEVICE = -9           /* the kernel reported an inconsistent task/queue  */
};

/* Wave orders of the host scheduler when every SM runs every phase (§The
 * task scheduler, the static part: named waves per layer, one chosen order).
 * Each SM's list holds, per layer, one share of every wave:
 *   P1 (norm + router / QKV rows), ROUTE (top-k), ATTN (split-KV items),
 *   UP (expert gate/up rows), COMBINE (split merges), DOWN (expert down rows),
 *   OUT (O-proj rows). */
enum mk_wave_order {
  MK_WAVES_DEFAULT = 0,    /* P1, ROUTE, ATTN, UP, COMBINE, DOWN, OUT  */
  MK_WAVES_ATTN_FIRST = 1, /* P1, ROUTE, ATTN, COMBINE, UP, DOWN, OUT  */
  MK_WAVES_INTERLEAVED = 2 /* P1, ROUTE, UP, ATTN, DOWN, COMBINE, OUT  */
};

typedef struct {
  /* model (§Tasks: the decode graph; the parallel transformer layer) */
  int n_layers;       /* L                                                       */
  int hidden;         /* H; multiple of 32 and one of the supported K (below)    */
  int n_q_heads;      /* hq                                                      */
  int n_kv_heads;     /* hkv; hq % hkv == 0 and hq / hkv <= 8 (GQA group)        */
  int head_dim;       /* d: 64 or 128                                            */
  int n_experts;      /* E <= 256                                                */
  int top_k;          /* k <= 8                                                  */
  int moe_inter;      /* I (expert intermediate size)                            */
  int vocab;          /* V                                                       */
  int page_size;      /* KV page size in tokens: 16                              */
  double rope_theta;  /* RoPE base                                               */
  float rms_eps;      /* RMSNorm epsilon                                         */
  /* capacity */
  int max_batch;          /* 1..16 sequences per step                            */
  int max_pages_per_seq;  /* columns of the page table                           */
  int num_kv_pages;       /* pages in each layer's K (and V) pool                */
  int max_attn_items;     /* split-KV items per layer; 0 = 8192                  */
  /* schedule */
  int wave_order;         /* enum mk_wave_order                                  */
  int n_attn_claimers;    /* SMs that run the attention branch (split-KV items,
                             combines); the others run the routed experts
                             (routing, gate/up, down); every SM takes O-proj
                             rows.
                             0 = chosen per step from the KV bytes against the
                             experts' bytes; >= the SM count = every SM runs
                             every phase in wave_order                         */
  int n_moe_claimers;     /* with every SM running every phase: SMs that take
                             expert slices; 0 = all                             */
  int kv_split_tokens;    /* split-KV chunk (multiple of 64); 0 = per step       */
  int sm_cap;             /* use at most this many SMs; 0 = all                  */
  int timeout_ms;         /* device spin limit per wait; 0 = 2000                */
  int trace_records;      /* per-SM task timeline records kept; 0 = tracing off  */
  int moe_stage_depth;    /* batch 1: weight stages an expert-branch SM keeps in
                             flight (1..5); 0 = chosen per step: 3 when the
                             expert branch has more SMs than the attention
                             branch (its streams would otherwise take HBM
                             bandwidth from the attention branch, which is on
                             the critical path), else 5                      */
  int expert_format;      /* enum mk_expert_format: how w_gate / w_up / w_down
                             hold the routed experts' weights                 */
  int moe_claim_rows;     /* several tokens: > 0 (a multiple of 16) = the
                             expert-branch SMs claim tiles of this many rows
                             (gate/up pairs, or down rows) one at a time from
                             a per-layer counter, so an SM whose tiles cost
                             more takes fewer (the pages' shared work queue:
                             "Inside the megakernel serving engine for North
                             Mini Code", §The task scheduler); 0 = chosen per
                             step: 128-row tiles from 4 tokens up, static
                             shares below; -1 = each expert-branch SM takes an
                             equal share of the routed experts' rows.
                             Results are identical either way.              */
} mk_config;

/* Weight format of the routed experts (mk_config.expert_format).
 *   MK_EXPERTS_BF16     w_gate / w_up / w_down are BF16 (below).
 *   MK_EXPERTS_FP8_E4M3 they hold bytes in the OCP 8-bit floating point
 *                       E4M3 encoding (bias 7, no infinities), one fp32
 *                       scale per output row in s_gate / s_up / s_down:
 *                       weight = scale[row] * e4m3(byte).  Supported with
 *                       max_batch == 1, hidden 256, 512, 1024 or 2048 and
 *                       moe_inter a multiple of 16 (else
 *                       MK_ERR_BAD_CONFIG).  Halves the experts' bytes, the
 *                       largest share of a decode step (the pages name 8-bit
 *                       weights as the next step on Blackwell: "Inside the
 *                       megakernel serving engine for North Mini Code",
 *                       §Next steps). */
enum mk_expert_format { MK_EXPERTS_BF16 = 0, MK_EXPERTS_FP8_E4M3 = 1 };

/*
 * Weights and KV pools, all owned by the caller, all device pointers, all
 * BF16.  They must stay valid until mk_destroy.  Per-layer arrays are HOST
 * arrays of L device pointers (copied at mk_create).
 *   embed, lm_head   [V][H]            (untied)
 *   final_norm       [H]               RMSNorm gain before the LM head
 *   attn_norm[l]     [H]               the layer's RMSNorm gain
 *   w_qkv[l]         [(hq + 2 hkv) d][H]  rows: q heads, then k heads, then v heads
 *   w_o[l]           [H][hq d]
 *   w_router[l]      [E][H]
 *   w_gate[l], w_up[l]  [E][I][H]
 *   w_down[l]        [E][H][I]          (read once, at mk_create: see there)
 *   s_gate[l], s_up[l]  [E][I] fp32,  s_down[l]  [E][H] fp32: the per-row
 *                    scales of 8-bit experts (MK_EXPERTS_FP8_E4M3; the three
 *                    matrices above then hold E4M3 bytes in the same
 *                    layouts); NULL with BF16 experts
 *   k_pool[l], v_pool[l]  [num_kv_pages][hkv][page_size][d]  (written: the
 *                    step stores its new K/V, post-RoPE, at position seq_len)
 * Every pointer must be 16-byte aligned.
 */
typedef struct {
  const void* embed;
  const void* lm_head;
  const void* final_norm;
  const void* const* attn_norm;
  const void* const* w_qkv;
  const void* const* w_o;
  const void* const* w_router;
  const void* const* w_gate;
  const void* const* w_up;
  const void* const* w_down;
  void* const* k_pool;
  void* const* v_pool;
  const void* const* s_gate;
  const void* const* s_up;
  const void* const* s_down;
} mk_weights;

/* Device error word, read by mk_step_status. */
typedef struct {
  int code;        /* MK_OK, MK_ERR_TIMEOUT, MK_ERR_DEVICE                   */
  int sm;          /* block that reported it                                 */
  int task;        /* index in that block's task list (-1: not a list task)  */
  int op;          /* opcode being executed                                  */
  int barrier;     /* counter index waited on (-1: a shared-memory wait)     */
  unsigned value;  /* counter value seen at the give-up time                 */
  unsigned target; /* value that was waited for                              */
} mk_error;

typedef struct mk_handle mk_handle;

/* Create a decoder on the current CUDA device.
 * Validates cfg (MK_ERR_BAD_CONFIG), copies the per-layer pointer arrays,
 * allocates the library-owned device state (counters, activations scratch,
 * queues, task lists: MK_ERR_OOM on failure) and builds the per-layer waves.
 *
 * Weight snapshot: mk_create also copies every layer's w_down into a
 * library-owned device array in a blocked layout, [L][E][I / 8][H][8]
 * elements (each 8-column group of an expert's down projection contiguous;
 * BF16, or E4M3 bytes with 8-bit experts), and the decode step reads that
 * copy, not w_down.  It costs L * E * I * H * 2 bytes (BF16; half with 8-bit
 * experts) of device memory (19.3 GB for L = 48, E = 128, I = 768, H = 2048), counted
 * in mk_device_bytes, and is made with a device-wide synchronize before
 * mk_create returns.  Changes the caller makes to w_down after mk_create are
 * therefore NOT seen by later steps: destroy and re-create the handle to pick
 * them up.  Every other weight and both KV pools are read in place.
 * On success *out owns that state until mk_destroy. */
int mk_create(const mk_config* cfg, const mk_weights* w, mk_handle** out);

/* Snapshot one decode batch (the park/resume rule of the pages' decode
 * service: the kernel never sees a half-updated batch).  All arrays are HOST
 * arrays and may be reused by the caller as soon as the call returns.
 *   batch        1..max_batch
 *   seq_ids      [batch] caller's ids (recorded, not interpreted); may be NULL
 *   tokens       [batch] input token of each sequence, 0 <= t < V
 *   page_tables  [batch][max_pages_per_seq] physical page of each 16-token
 *                logical page; entries past the needed pages are ignored
 *   seq_lens     [batch] tokens already cached; the step writes the new K/V
 *                at position seq_lens[i], whose page must already be present
 * Uploads the step state on `stream` (a cudaStream_t; NULL = default) and
 * picks the split-KV chunk from the longest live context.  The caller
 * increments seq_lens itself afterwards.  Errors: MK_ERR_BATCH_TOO_LARGE,
 * MK_ERR_BAD_PAGE (an index >= num_kv_pages or < 0 among the pages the step
 * reads, or seq_lens[i] + 1 > max_pages_per_seq * page_size), MK_ERR_BAD_ARG. */
int mk_schedule_step(mk_handle* h, int batch, const int32_t* seq_ids, const int32_t* tokens,
                     const int32_t* page_tables, const int32_t* seq_lens, void* stream);

/* Run the scheduled step on `stream`: zero the counters and launch the
 * persistent kernel (cooperative launch, one block per SM).  Writes the
 * logits, fp32 [batch][V], to the DEVICE buffer `logits` and the new K/V into
 * the pools.  Asynchronous: errors found by the kernel surface through
 * mk_step_status once the stream has synchronised. */
int mk_decode_step(mk_handle* h, float* logits, void* stream);

/* After the stream of the last mk_decode_step has synchronised: copy the
 * device error word into *out (may be NULL) and return its code. */
int mk_step_status(mk_handle* h, mk_error* out);

/* Routing of the last completed step, for checking: HOST arrays
 * idx int32 [L][batch][top_k] (best first) and w fp32 [L][batch][top_k]
 * (renormalised weights); either may be NULL.  Synchronous. */
int mk_get_routing(mk_handle* h, int32_t* idx, float* w);

/* Intermediate activations of the last completed step, for checking.
 * which: MK_SCRATCH_* below; layer in [0, L] where the kind allows it
 * (X and H take L for the final norm).  Copies min(bytes, size) bytes to the
 * HOST buffer dst and returns the full size in *size_out (may be NULL). */
enum mk_scratch {
  MK_SCRATCH_H = 0,       /* fp32 [batch][H]  residual entering the layer         */
  MK_SCRATCH_X = 1,       /* fp32 [batch][H]  normalised layer input              */
  MK_SCRATCH_QKV = 2,     /* fp32 [batch][(hq + 2 hkv) d]  q, k, v before RoPE    */
  MK_SCRATCH_ATTN = 3,    /* fp32 [batch][hq*d]   attention output                */
  MK_SCRATCH_ROUTER = 4,  /* fp32 [batch][E]  router logits                       */
  MK_SCRATCH_OPROJ = 5,   /* fp32 [batch][H]  O-proj output                       */
  MK_SCRATCH_MOE = 6      /* fp32 [batch][H]  weighted sum of the routed experts  */
};
int mk_read_scratch(mk_handle* h, int which, int layer, void* dst, size_t bytes,
                    size_t* size_out);

/* Per-SM task lists of the schedule for `batch` (built on demand), for
 * checking the host scheduler without a GPU: descriptors int32 [n][32] in
 * SM-major order and offsets int32 [n_sm + 1].  With tasks == NULL only the
 * sizes are returned.  Host-only; needs no device. */
int mk_plan(const mk_config* cfg, int n_sm, int batch, int32_t* tasks, int32_t* offsets,
            int* n_tasks_out, int* n_barriers_out);

/* The whole host schedule of one step, as mk_schedule_step builds it for the
 * lengths seq_lens [batch] (HOST array): the attention-branch size, the
 * split-KV items and the per-SM task lists, for checking the scheduler and
 * its counter accounting without a GPU.  Host-only; needs no device.
 *   info      int32 [9]: n_tasks, n_items, attention SMs, then the SM counts
 *             the kernel takes as counter targets (COMBINE, UP, DOWN and
 *             router-row SMs), the split-KV chunk (tokens; 0 = balanced page
 *             runs), counter words; always written
 *   tasks     int32 [n_tasks][32] descriptors, SM-major; task_off [n_sm + 1]
 *   items     int32 [n_items][8] split-KV items (sequence, split index, split
 *             count, first key, end key, first item of the sequence, new
 *             token's position, 0); item_off [n_sm + 1] items of each SM
 *   meta      int32 [batch][2]: first item and split count of each sequence
 * Any of tasks .. meta may be NULL (call once with NULL to size them).
 * Errors: MK_ERR_BAD_ARG, MK_ERR_BATCH_TOO_LARGE, MK_ERR_BAD_CONFIG. */
int mk_plan_step(const mk_config* cfg, int n_sm, int batch, const int32_t* seq_lens, int32_t* info,
                 int32_t* tasks, int32_t* task_off, int32_t* items, int32_t* item_off, int32_t* meta);

/* Testing aid for the device timeout path: add `delta` to the wait target of
 * the norm task of `layer` in the cached schedules, so that its counter wait
 * can never complete and runs out after config.timeout_ms (the kernel then
 * stops every block and reports MK_ERR_TIMEOUT).  delta = 0 restores it. */
int mk_debug_bump_wait(mk_handle* h, int layer, int delta);

/* Task timeline of the last completed step (config.trace_records > 0):
 * HOST buffer of int32 [n_sm][trace_records][16] records
 *   {op, layer, tile or queue item, t_start_lo, t_start_hi, ready_ns, end_ns, sm,
 *    first_stage_ns, stages_done_ns, reduced_ns, kind, rows, handed_ns, issued_ns,
 *    stage_wait_ns}
 * where t_start is the %globaltimer value (ns) when the block took the task,
 * ready_ns the offset at which its inputs were ready, end_ns the offset at
 * which it signalled completion and the next three the offsets at which its
 * first stage arrived, its last stage was consumed and its partial sums were
 * reduced (equal to the start where a task has no such phase); kind and rows
 * describe the piece (a GEMV chunk kind and its row count); handed_ns and
 * issued_ns are the (usually negative) offsets at which the streaming warp
 * handed the piece over and issued its first copy (0: no copy), stage_wait_ns
 * the time the block waited for its stages; unused records have op = -1.  Copies min(bytes, size) bytes; *size_out (may be NULL) gets
 * the full size. */
int mk_read_trace(mk_handle* h, void* dst, size_t bytes, size_t* size_out);

/* Integer results of the last completed step, for exact checks; recorded
 * only when the handle keeps the task timeline (config.trace_records > 0),
 * else MK_ERR_BAD_CONFIG.  Copies min(bytes, size) bytes to the HOST buffer
 * dst; *size_out (may be NULL) gets the full size.
 *   MK_DEBUG_ROUTE_GROUPS  int32 [L][386]: block 0's grouping of each layer's
 *       routing: n_act; the routed experts ascending (128 slots); the first
 *       grouped slot of each (129 slots, the last = the entry count); the
 *       grouped entries b * top_k + j, tokens ascending within an expert
 *       (128 slots); unused slots -1
 *   MK_DEBUG_PAGE_GATHER   int32 [batch][max_pages_per_seq]: the physical
 *       page the attention streamed for each logical page in layer 0, -1 for
 *       pages past the sequence
 *   MK_DEBUG_NEW_SLOT      int32 [batch]: the cache slot page * page_size +
 *       row where layer 0 wrote each sequence's new K/V */
enum mk_debug { MK_DEBUG_ROUTE_GROUPS = 0, MK_DEBUG_PAGE_GATHER = 1, MK_DEBUG_NEW_SLOT = 2 };
int mk_read_debug(mk_handle* h, int which, void* dst, size_t bytes, size_t* size_out);

/* Words of the fixed device-resident counter block used by
 * mk_decode_step_static (256 KB per device). */
#define MK_STATIC_COUNTER_WORDS 65536

/* mk_decode_step for callers that may not allocate device memory while they
 * run a step: a real-time serving loop that must not take the allocator's
 * locks or meet an out-of-memory failure between steps, or a host runtime
 * that owns every device allocation itself and forbids its plug-ins to call
 * cudaMalloc.  The megakernel serving engine it follows has no such call.
 *
 * mk_decode_step keeps the step's counters, queue claim heads and error words
 * in device memory the handle allocated; this call keeps them instead in one
 * file-scope device array of MK_STATIC_COUNTER_WORDS 32-bit words that the
 * library holds on every device where it is loaded, until the process exits.
 * It calls no allocating routine: the schedule is the one mk_schedule_step
 * built, the words the step uses are cleared to zero on `stream` before the
 * kernel, and after it the error words are copied on `stream` into the
 * handle's own error block, so mk_step_status reports the step as usual.
 * The results are the same as those of mk_decode_step for the same batch.
 *
 * Limit: a handle needs 32 + n_layers * round_up(8 + max_batch, 32) words;
 * with max_batch <= 16 that is 32 words per layer, so up to 2,047 layers fit.
 * A larger need returns MK_ERR_BAD_CONFIG.  Other errors: MK_ERR_NOT_SCHEDULED, MK_ERR_BAD_ARG
 * (NULL logits, or the current device is not the handle's), MK_ERR_CUDA.
 *
 * Sharing: every handle on a device uses the same array, and it keeps what
 * the last call left in it.  Two calls whose kernels overlap on the GPU
 * (other streams, other handles, other threads) race on it and corrupt each
 * other's step: serialise them.  mk_decode_step does not touch the array.
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and sets the kernel's
 * shared-memory limit there; make that first call before any stream capture. */
int mk_decode_step_static(mk_handle* h, float* logits, void* stream);

/* ---------------------------------------------------------------------
 * Decode service ("Inside the megakernel serving engine for North Mini
 * Code", §The serving engine around the kernel: the host loop and its
 * park / resume rule).  A loop thread owns the handle and, per step:
 * retires the requests that have all their tokens and admits waiting ones
 * into the free slots (only between steps: the kernel never sees a batch
 * half updated), builds the page tables and lengths of the live slots,
 * schedules the step for the longest live context (mk_schedule_step),
 * launches it, picks every sequence's greedy token on the device (largest
 * logit, ties to the lowest index) and feeds it to the next step on the
 * device.  The host records the tokens from small asynchronous copies, a few
 * steps later.  The loop parks when it has run the steps asked for and
 * resumes on mk_service_run.  Requests finish after max_new_tokens tokens.
 *
 * While a service exists it is the only user of its handle: make no other
 * call on the handle (except mk_destroy after mk_service_destroy).  The
 * service functions are thread-safe.
 */
typedef struct mk_service mk_service;

/* Start the loop thread on the handle's device (must be current).  logits:
 * DEVICE fp32 [max_batch][V] the caller owns; each step writes its live
 * sequences' logits there, position i = the i-th live slot.  Errors:
 * MK_ERR_BAD_ARG, MK_ERR_OOM. */
int mk_service_create(mk_handle* h, float* logits, mk_service** out);

/* Queue a request: a sequence whose first cached_len tokens are already in
 * the KV pools, on the caller's physical pages pages[0 .. n_pages) (HOST
 * array, copied) in logical order, covering every position the request will
 * write (n_pages * page_size >= cached_len + max_new_tokens); first_token is
 * its next input token.  The pages stay the caller's; it may reuse them once
 * the request is done.  *id_out gets the request id.  Errors: MK_ERR_BAD_ARG,
 * MK_ERR_BAD_PAGE. */
int mk_service_submit(mk_service* s, const int32_t* pages, int n_pages, int cached_len, int32_t first_token,
                      int max_new_tokens, int64_t* id_out);

/* Ask the loop for n_steps more steps (resume it if parked); returns at once.
 * Returns the sticky error of an earlier step, if any. */
int mk_service_run(mk_service* s, int n_steps);

/* Block until the loop has run every step asked for and parked (the stream
 * synchronised, every token recorded); returns MK_OK or the first error (a
 * failed call or the device status of the last step). */
int mk_service_wait(mk_service* s);

/* The tokens request `id` has generated so far (HOST int32, up to cap), their
 * count and whether the request is done.  Call after mk_service_wait for a
 * complete record. */
int mk_service_result(mk_service* s, int64_t id, int32_t* tokens, int cap, int* n_out, int* done);

/* The last step's batch, position by position (HOST arrays of max_batch, any
 * may be NULL): request ids, cached lengths before the step, input tokens;
 * *batch gets its size.  Call after mk_service_wait. */
int mk_service_batch(mk_service* s, int64_t* ids, int32_t* seq_lens, int32_t* tokens, int* batch);

/* Stop the loop (after the step in flight) and free the service. */
void mk_service_destroy(mk_service* s);

/* Library-owned device bytes (counters, scratch, queues, task lists). */
size_t mk_device_bytes(const mk_handle* h);
/* SMs the persistent grid uses. */
int mk_num_sms(const mk_handle* h);
/* Bytes mk_schedule_step uploads for `batch` sequences (host -> device). */
size_t mk_step_upload_bytes(const mk_handle* h, int batch);

void mk_destroy(mk_handle* h);
const char* mk_strerror(int code);
int mk_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
