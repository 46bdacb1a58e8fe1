// Decode service: the host loop around the persistent step kernel.
//
// "Inside the megakernel serving engine for North Mini Code", §The serving
// engine around the kernel: a loop thread owns the GPU; between two steps it
// retires the finished sequences and admits waiting ones (the park/resume
// rule: the batch changes only at a step boundary, so the kernel never sees a
// half-updated batch), updates the page tables, selects the schedule for the
// longest live context (mk_schedule_step) and launches the step.  The greedy
// token of every sequence is chosen on the device ("llama.cpp on V100",
// §GPU argmax: no logits travel to the host) and fed to the next step on the
// device; the host only learns the tokens a few steps later, from a ring of
// small asynchronous copies, to record them.
//
// Requests finish by length (max_new_tokens): the synthetic models here have
// no end-of-sequence token.  A request's pages are the caller's: the service
// reads them and the caller may reuse them once the request is done.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <condition_variable>
#include <deque>
#include <map>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "../../include/mk.h"

namespace mk {
int32_t* handle_tokens(mk_handle* h);
const mk_config* handle_config(const mk_handle* h);
int handle_device(const mk_handle* h);
}  // namespace mk

namespace {

// greedy token of each row of logits [B][V]: the largest value, ties to the
// lowest index (NaNs never win); one block per row
__global__ void __launch_bounds__(1024) argmax_rows_kernel(const float* __restrict__ logits, int V,
                                                          int32_t* __restrict__ out) {
  const float* row = logits + (size_t)blockIdx.x * V;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    const float v = row[i];
    if (v > best || (v == best && i < bi)) {
      best = v;
      bi = i;
    }
  }
  __shared__ float sv[32];
  __shared__ int si[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) {
      best = ov;
      bi = oi;
    }
  }
  if (lane == 0) {
    sv[warp] = best;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = (int)(blockDim.x >> 5);
    best = lane < nw ? sv[lane] : -INFINITY;
    bi = lane < nw ? si[lane] : 0x7fffffff;
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > best || (ov == best && oi < bi)) {
        best = ov;
        bi = oi;
      }
    }
    if (lane == 0) out[blockIdx.x] = bi == 0x7fffffff ? 0 : bi;
  }
}

// the step's input tokens: position i continues position prev_pos[i] of the
// previous step (its greedy token), or (prev_pos[i] < 0) keeps the first
// token of a request that joins now (uploaded with the schedule)
__global__ void feed_tokens_kernel(const int32_t* __restrict__ prev, const int32_t* __restrict__ prev_pos,
                                   int B, int32_t* __restrict__ tokens) {
  const int i = threadIdx.x;
  if (i < B && prev_pos[i] >= 0) tokens[i] = prev[prev_pos[i]];
}

struct Request {
  std::vector<int32_t> pages;
  int cached_len = 0;
  int32_t first_token = 0;
  int max_new = 0;
  int issued = 0;                 // steps launched for it
  std::vector<int32_t> tokens;    // generated tokens recorded so far
  int slot = -1;
  bool retired = false;
};

constexpr int kRing = 4;

struct RingSlot {
  int32_t* host = nullptr;        // pinned [max_batch]: the step's greedy tokens
  int32_t* prev = nullptr;        // pinned [max_batch]: the step's prev_pos, uploaded
  cudaEvent_t ev = nullptr;       // after both copies of the step
  std::vector<int64_t> ids;       // request at each position
  bool used = false;
};

}  // namespace

struct mk_service {
  mk_handle* h = nullptr;
  float* logits = nullptr;
  cudaStream_t stream = nullptr;
  int dev = 0, slots = 0, V = 0, MP = 0, P = 16;
  std::mutex mu;
  std::condition_variable cv_work, cv_idle;
  std::thread loop;
  bool stop = false, busy = false;
  int queued = 0;                 // steps asked for and not yet run
  int error = MK_OK;              // sticky
  int64_t next_id = 1;
  std::deque<int64_t> pending;
  std::map<int64_t, Request> reqs;
  std::vector<int64_t> slot_req;  // [slots], -1 free
  std::vector<int> slot_pos;      // position of each slot in the last step, -1 none
  // device / pinned
  int32_t* d_next[2] = {nullptr, nullptr};
  int32_t* d_prev_pos = nullptr;
  int parity = 0;
  RingSlot ring[kRing];
  int ring_next = 0;
  // the last step's composition
  std::vector<int64_t> last_ids;
  std::vector<int32_t> last_lens, last_issued;
  long long steps_run = 0;
};

namespace {

// record the tokens of a finished ring slot (its copy has completed); lock held
void drain_slot(mk_service* s, RingSlot& r) {
  for (size_t i = 0; i < r.ids.size(); i++) {
    auto it = s->reqs.find(r.ids[i]);
    if (it != s->reqs.end()) it->second.tokens.push_back(r.host[i]);
  }
  r.ids.clear();
  r.used = false;
}

// one step; called by the loop thread with the lock held, returns with it held
int run_step(mk_service* s, std::unique_lock<std::mutex>& lk) {
  // retire the requests that have all their tokens, admit waiting ones
  for (int k = 0; k < s->slots; k++) {
    if (s->slot_req[k] < 0) continue;
    Request& r = s->reqs[s->slot_req[k]];
    if (r.issued >= r.max_new) {
      r.retired = true;
      r.slot = -1;
      s->slot_req[k] = -1;
    }
  }
  for (int k = 0; k < s->slots && !s->pending.empty(); k++) {
    if (s->slot_req[k] >= 0) continue;
    const int64_t id = s->pending.front();
    s->pending.pop_front();
    s->slot_req[k] = id;
    s->reqs[id].slot = k;
  }
  // the batch: live slots in slot order
  std::vector<int64_t> ids;
  std::vector<int32_t> tokens, lens, prev, pt, sid, issued;
  std::vector<int> new_pos(s->slots, -1);
  for (int k = 0; k < s->slots; k++) {
    if (s->slot_req[k] < 0) continue;
    const Request& r = s->reqs[s->slot_req[k]];
    const int pos = (int)ids.size();
    new_pos[k] = pos;
    ids.push_back(s->slot_req[k]);
    sid.push_back((int32_t)s->slot_req[k]);
    issued.push_back(r.issued);
    lens.push_back(r.cached_len + r.issued);
    // first step of a request: its first token; later: the previous greedy token
    tokens.push_back(r.issued == 0 ? r.first_token : 0);
    prev.push_back(r.issued == 0 ? -1 : s->slot_pos[k]);
    for (int i = 0; i < s->MP; i++) pt.push_back(i < (int)r.pages.size() ? r.pages[i] : -1);
  }
  const int B = (int)ids.size();
  if (B == 0) return MK_OK;
  lk.unlock();
  int rc = MK_OK;
  RingSlot& ring = s->ring[s->ring_next];
  if (ring.used && cudaEventSynchronize(ring.ev) != cudaSuccess) rc = MK_ERR_CUDA;
  if (!rc) rc = mk_schedule_step(s->h, B, sid.data(), tokens.data(), pt.data(), lens.data(), s->stream);
  if (!rc) {
    // the ring slot's pinned buffers are free: its previous step's event has completed
    memcpy(ring.prev, prev.data(), (size_t)B * 4);
    const int cur = s->parity ^ 1;
    if (cudaMemcpyAsync(s->d_prev_pos, ring.prev, (size_t)B * 4, cudaMemcpyHostToDevice, s->stream) !=
        cudaSuccess)
      rc = MK_ERR_CUDA;
    if (!rc) {
      feed_tokens_kernel<<<1, 32, 0, s->stream>>>(s->d_next[s->parity], s->d_prev_pos, B,
                                                   mk::handle_tokens(s->h));
      if (cudaGetLastError() != cudaSuccess) rc = MK_ERR_CUDA;
    }
    if (!rc) rc = mk_decode_step(s->h, s->logits, s->stream);
    if (!rc) {
      argmax_rows_kernel<<<B, 1024, 0, s->stream>>>(s->logits, s->V, s->d_next[cur]);
      if (cudaGetLastError() != cudaSuccess) rc = MK_ERR_CUDA;
    }
    if (!rc && (cudaMemcpyAsync(ring.host, s->d_next[cur], (size_t)B * 4, cudaMemcpyDeviceToHost, s->stream) !=
                    cudaSuccess ||
                cudaEventRecord(ring.ev, s->stream) != cudaSuccess))
      rc = MK_ERR_CUDA;
    s->parity = cur;
  }
  lk.lock();
  if (rc) return rc;
  if (ring.used) drain_slot(s, ring);
  ring.ids = ids;
  ring.used = true;
  s->ring_next = (s->ring_next + 1) % kRing;
  for (int i = 0; i < B; i++) s->reqs[ids[i]].issued++;
  s->slot_pos = new_pos;
  s->last_ids = ids;
  s->last_lens = lens;
  s->last_issued = issued;
  s->steps_run++;
  return MK_OK;
}

// park: wait for the stream, record every outstanding token, read the step
// status; lock held
int park(mk_service* s, std::unique_lock<std::mutex>& lk) {
  lk.unlock();
  int rc = cudaStreamSynchronize(s->stream) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
  if (!rc && s->steps_run > 0) rc = mk_step_status(s->h, nullptr);
  lk.lock();
  for (int k = 0; k < kRing; k++) {
    RingSlot& r = s->ring[(s->ring_next + k) % kRing];
    if (r.used) drain_slot(s, r);
  }
  return rc;
}

void loop_main(mk_service* s) {
  cudaSetDevice(s->dev);
  std::unique_lock<std::mutex> lk(s->mu);
  while (true) {
    s->cv_work.wait(lk, [&] { return s->stop || s->queued > 0; });
    if (s->stop) break;
    s->busy = true;
    int rc = MK_OK;
    while (s->queued > 0 && !s->stop && rc == MK_OK) {
      rc = run_step(s, lk);
      s->queued--;
    }
    const int prc = park(s, lk);
    if (rc == MK_OK) rc = prc;
    if (rc != MK_OK && s->error == MK_OK) s->error = rc;
    s->queued = 0;
    s->busy = false;
    s->cv_idle.notify_all();
  }
}

void free_service(mk_service* s) {
  if (s->stream) cudaStreamSynchronize(s->stream);
  for (auto& r : s->ring) {
    if (r.host) cudaFreeHost(r.host);
    if (r.prev) cudaFreeHost(r.prev);
    if (r.ev) cudaEventDestroy(r.ev);
  }
  cudaFree(s->d_next[0]);
  cudaFree(s->d_next[1]);
  cudaFree(s->d_prev_pos);
  if (s->stream) cudaStreamDestroy(s->stream);
  delete s;
}

}  // namespace

extern "C" {

int mk_service_create(mk_handle* h, float* logits, mk_service** out) {
  if (!h || !logits || !out) return MK_ERR_BAD_ARG;
  *out = nullptr;
  mk_service* s = new (std::nothrow) mk_service();
  if (!s) return MK_ERR_OOM;
  const mk_config* c = mk::handle_config(h);
  s->h = h;
  s->logits = logits;
  s->dev = mk::handle_device(h);
  s->slots = c->max_batch;
  s->V = c->vocab;
  s->MP = c->max_pages_per_seq;
  s->P = c->page_size;
  s->slot_req.assign(s->slots, -1);
  s->slot_pos.assign(s->slots, -1);
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != s->dev) {
    cudaGetLastError();
    delete s;
    return MK_ERR_BAD_ARG;
  }
  bool ok = cudaStreamCreateWithFlags(&s->stream, cudaStreamNonBlocking) == cudaSuccess &&
            cudaMalloc(&s->d_next[0], (size_t)s->slots * 4) == cudaSuccess &&
            cudaMalloc(&s->d_next[1], (size_t)s->slots * 4) == cudaSuccess &&
            cudaMalloc(&s->d_prev_pos, (size_t)s->slots * 4) == cudaSuccess;
  for (auto& r : s->ring)
    ok = ok && cudaMallocHost(&r.host, (size_t)s->slots * 4) == cudaSuccess &&
         cudaMallocHost(&r.prev, (size_t)s->slots * 4) == cudaSuccess &&
         cudaEventCreateWithFlags(&r.ev, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaMemset(s->d_next[0], 0, (size_t)s->slots * 4) == cudaSuccess &&
       cudaMemset(s->d_next[1], 0, (size_t)s->slots * 4) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    free_service(s);
    return MK_ERR_OOM;
  }
  try {
    s->loop = std::thread(loop_main, s);
  } catch (...) {
    free_service(s);
    return MK_ERR_OOM;
  }
  *out = s;
  return MK_OK;
}

int mk_service_submit(mk_service* s, const int32_t* pages, int n_pages, int cached_len, int32_t first_token,
                      int max_new_tokens, int64_t* id_out) {
  if (!s || !pages || n_pages < 1 || cached_len < 0 || max_new_tokens < 1) return MK_ERR_BAD_ARG;
  if (first_token < 0 || first_token >= s->V) return MK_ERR_BAD_ARG;
  // every position the request will write must have its page
  const long long need = ((long long)cached_len + max_new_tokens + s->P - 1) / s->P;
  if (n_pages > s->MP || need > n_pages) return MK_ERR_BAD_PAGE;
  const mk_config* c = mk::handle_config(s->h);
  for (int i = 0; i < n_pages; i++)
    if (pages[i] < 0 || pages[i] >= c->num_kv_pages) return MK_ERR_BAD_PAGE;
  std::lock_guard<std::mutex> g(s->mu);
  Request r;
  r.pages.assign(pages, pages + n_pages);
  r.cached_len = cached_len;
  r.first_token = first_token;
  r.max_new = max_new_tokens;
  const int64_t id = s->next_id++;
  if (id > 0x7fffffffll) return MK_ERR_BAD_ARG;
  s->reqs.emplace(id, std::move(r));
  s->pending.push_back(id);
  if (id_out) *id_out = id;
  return MK_OK;
}

int mk_service_run(mk_service* s, int n_steps) {
  if (!s || n_steps < 0) return MK_ERR_BAD_ARG;
  std::lock_guard<std::mutex> g(s->mu);
  if (s->error) return s->error;
  s->queued += n_steps;
  s->cv_work.notify_one();
  return MK_OK;
}

int mk_service_wait(mk_service* s) {
  if (!s) return MK_ERR_BAD_ARG;
  std::unique_lock<std::mutex> lk(s->mu);
  s->cv_idle.wait(lk, [&] { return s->queued == 0 && !s->busy; });
  return s->error;
}

int mk_service_result(mk_service* s, int64_t id, int32_t* tokens, int cap, int* n_out, int* done) {
  if (!s) return MK_ERR_BAD_ARG;
  std::lock_guard<std::mutex> g(s->mu);
  auto it = s->reqs.find(id);
  if (it == s->reqs.end()) return MK_ERR_BAD_ARG;
  const Request& r = it->second;
  const int n = (int)r.tokens.size();
  if (tokens && cap > 0) memcpy(tokens, r.tokens.data(), (size_t)std::min(n, cap) * 4);
  if (n_out) *n_out = n;
  if (done) *done = (r.retired || r.issued >= r.max_new) && n == r.max_new;
  return MK_OK;
}

int mk_service_batch(mk_service* s, int64_t* ids, int32_t* seq_lens, int32_t* tokens, int* batch) {
  if (!s || !batch) return MK_ERR_BAD_ARG;
  std::lock_guard<std::mutex> g(s->mu);
  const int B = (int)s->last_ids.size();
  *batch = B;
  for (int i = 0; i < B; i++) {
    if (ids) ids[i] = s->last_ids[i];
    if (seq_lens) seq_lens[i] = s->last_lens[i];
    if (tokens) {
      const Request& r = s->reqs[s->last_ids[i]];
      const int k = s->last_issued[i];
      // the step's input: the first token, or the token the step before produced
      tokens[i] = k == 0 ? r.first_token : (k - 1 < (int)r.tokens.size() ? r.tokens[k - 1] : -1);
    }
  }
  return MK_OK;
}

void mk_service_destroy(mk_service* s) {
  if (!s) return;
  {
    std::lock_guard<std::mutex> g(s->mu);
    s->stop = true;
    s->cv_work.notify_all();
  }
  if (s->loop.joinable()) s->loop.join();
  free_service(s);
}

}  // extern "C"
