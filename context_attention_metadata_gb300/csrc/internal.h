// Internal declarations shared by the translation units of libmarble (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/marble.h"

namespace marble {

// Per-block summary of the metadata tracks (MARBLE s03 "Block classification"): min and
// max of each track plus a 64-bit bitmap of the segment ids the block holds.
struct Summary {
  int slo, shi;    // sample id
  int nlo, nhi;    // noise id
  int glo, ghi;    // segment id over tokens with seg >= 0 (INT_MAX / -1 when none)
  int plo, phi;    // original position
  unsigned long long gbits;  // OR of 1 << (seg mod 64) over tokens with seg >= 0
  int flags;       // bit 0: some token has seg >= 0; bit 1: every token has seg >= 0
  int pad;
};

// chunk-layout search (plan.cu): the finest chunk count for nb blocks and P ranks, and the
// search over the pairs wf [Kf][Kf] between the finest chunks
int finest_chunks(int64_t nb, int P);
void chunk_layout_host(const std::vector<int64_t>& wf, int Kf, int P, int64_t tau, int* k,
                       std::vector<int>* rank, int64_t* cost, int64_t* step);

}  // namespace marble

struct marble_plan {
  int device = 0;
  int64_t n = 0, nb = 0;
  int P = 1, W = 0, order = 0, chunk_tokens = 0;
  int64_t range_cost = 0;                       // CHUNK_SEARCH: tau
  cudaStream_t build_stream = nullptr;          // the stream marble_plan ran on
  int64_t chunks_per_rank = 0, layout_cost = 0, layout_step_cost = 0;  // its result
  unsigned long long* shard_pairs = nullptr;    // [P*P] statistics: legal pairs per shard pair
  int32_t* kiv = nullptr;       // [2*n] new order: lo, hi of every key's visible query interval
  uint8_t* iv_block = nullptr;  // [nb] new order: 1 if every key of the block is exact
  int4* kiv_chunk = nullptr;    // [nb*4] per 32 keys: min lo, max lo, min hi, max hi
  int64_t bps = 0;           // blocks per shard
  int64_t nnz = 0, needed_total = 0;
  // device arrays (owned)
  marble::Summary* summ = nullptr;   // [nb], original block order
  int32_t* band = nullptr;           // [2*nb] candidate kv range per block (lo, hi incl.)
  int64_t* row_ptr = nullptr;        // [nb+1] tile map, original coordinates
  int32_t* col = nullptr;            // [nnz]
  uint8_t* tag = nullptr;            // [nnz]
  int32_t* block_perm = nullptr;     // [nb] new -> original
  int32_t* inv_block_perm = nullptr; // [nb] original -> new
  int32_t* perm = nullptr;           // [n] new token -> original token
  int32_t* tracks = nullptr;         // [4*n] sample, seg, noise, pos (new order)
  int64_t* step_ptr = nullptr;       // [nb*P+1]
  int32_t* step_col = nullptr;       // [nnz]
  uint8_t* step_tag = nullptr;       // [nnz]
  int64_t* colT_ptr = nullptr;       // [nb*P+1]
  int32_t* colT_row = nullptr;       // [nnz]
  uint8_t* colT_tag = nullptr;       // [nnz]
  int64_t* needed_ptr = nullptr;     // [P+1]
  int32_t* needed = nullptr;         // [needed_total]
  // work lists of the persistent kernels: for shard s and option k (k < P: kv shard k of
  // the forward / q shard k of the key-side backward; k == P: every shard), the blocks of
  // shard s with a non-empty list, longest list first
  int32_t* fwd_order = nullptr;      // [P*(P+1)*bps] over step_ptr (q blocks)
  int32_t* fwd_nwork = nullptr;      // [P*(P+1)]
  int32_t* bwd_order = nullptr;      // [P*(P+1)*bps] over colT_ptr (kv blocks)
  int32_t* bwd_nwork = nullptr;      // [P*(P+1)]
  std::vector<int32_t> h_fwd_nwork, h_bwd_nwork;
  // the fused forward: row lists in ring order (same CSR ranges as step_ptr over all kv
  // shards) and the work order of every block of the pack, longest row first
  int32_t* ring_col = nullptr;       // [nnz]
  uint8_t* ring_tag = nullptr;       // [nnz]
  int32_t* fwd_order_all = nullptr;  // [nb]
  int32_t* fwd_nwork_all = nullptr;  // [1]
  int32_t h_fwd_nwork_all = 0;
  // compact tile numbering of each step (the backward's dS tiles): step_off[nq*(P+1)+opt] is
  // the number of tiles of the q blocks before nq in its q shard, for option opt (kv shard opt,
  // or every kv shard when opt == P); colT_j[e] the index of column-list entry e's kv block in
  // its q block's list for that kv shard
  int32_t* step_off = nullptr;       // [nb*(P+1)]
  int64_t* step_tiles = nullptr;     // [P*(P+1)] tiles per (q shard, option)
  int64_t* step_max = nullptr;       // [P*(P+1)] longest q-block list per (q shard, option)
  int32_t* colT_j = nullptr;         // [nnz]
  std::vector<int64_t> h_step_tiles;
  std::vector<int64_t> h_step_max;        // [P*(P+1)] longest list of a q block in the step
  // backward scratch: bf16 dS^T tiles of two steps (allocated by the first backward call)
  mutable std::mutex scratch_mu;
  mutable void* ds_scratch = nullptr;
  mutable size_t ds_scratch_bytes = 0;
  // ticket counters of the persistent kernels: launch i uses pair (i mod kSchedSlots); the
  // last CTA of a launch puts its pair back to zero
  unsigned* sched = nullptr;         // [2*kSchedSlots]
  mutable std::atomic<unsigned> sched_next{0};
  unsigned* err = nullptr;           // device error word
  unsigned long long* counters = nullptr;  // [8] device scratch for statistics
  std::vector<int64_t> h_needed_ptr;      // host copy of needed_ptr
  std::vector<void*> owned;
  // the last use of the plan on each stream a call ran on (an event recorded after the
  // call's work): marble_plan_destroy frees the workspace in stream order after all of them
  mutable std::mutex use_mu;
  mutable std::vector<std::pair<cudaStream_t, cudaEvent_t>> uses;
};

namespace marble {

// An NVTX range named after the API call, open for the call's host-side duration, so that
// a profiler timeline shows which call queued which kernels (no cost without a profiler).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kSchedSlots = 256;

// a ticket-counter pair of `p` for one persistent-kernel launch
inline unsigned* sched_slot(const marble_plan_t* p) {
  const unsigned i = p->sched_next.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots;
  return p->sched + 2 * i;
}

// true for device or managed memory of the current context (api.cu)
bool is_device_ptr(const void* p);

// record that work using plan `p` has been queued on `s` (api.cu); every call that
// launches work on a plan's memory records it before returning
void plan_used(const marble_plan_t* p, cudaStream_t s);

// Small transfers between the device and pageable host memory (the planner's sizes and
// work counts, the error word, statistics) go through a pinned buffer of the calling thread
// (api.cu).  A copy to or from pageable memory is carried out by the copy engines on pages
// the driver has to resolve on the fly, and a training loop's large input and output copies
// then wait behind it; pinned memory needs no such step.  read_back queues a copy of every
// part into the buffer on `s`, synchronises `s` and copies the parts out; write_to_device
// copies `bytes` from `host` into the buffer, queues the copy to `dev` on `s` and
// synchronises `s`.  The buffer grows as needed and lives as long as the thread.
struct HostPart {
  void* host;
  const void* dev;
  size_t bytes;
};
cudaError_t read_back(cudaStream_t s, std::initializer_list<HostPart> parts);
cudaError_t write_to_device(cudaStream_t s, void* dev, const void* host, size_t bytes);

// dS^T scratch buffers of destroyed plans, kept per device for the next plans' backward calls
// (api.cu).  scratch_put hands over a buffer whose last use completes with `ready` (the cache
// owns the event); scratch_take returns a cached buffer of at least `bytes` bytes and at most
// twice that (the oldest such) after making `s` wait for its `ready`, or nullptr.  A buffer reused this way
// stays with the stream order of its previous owner, where a new pool allocation on another
// stream would make the pool map fresh memory while the old buffer's free is still queued.
void scratch_put(int device, void* ptr, size_t bytes, cudaEvent_t ready);
void* scratch_take(size_t bytes, cudaStream_t s, size_t* got);

// error reporting (api.cu)
void set_error(const std::string& msg);
marble_status_t fail(marble_status_t st, const std::string& msg);
marble_status_t cuda_fail(cudaError_t e, const char* what);
uint64_t wait_limit_ns();

// planner (plan.cu)
marble_status_t build_plan(const marble_plan_desc_t* d, cudaStream_t s, marble_plan_t* p);
marble_status_t plan_legal_pairs(const marble_plan_t* p, cudaStream_t s, int64_t* pairs,
                                 int64_t* n_full, int64_t* n_partial, int64_t* step_pairs);

// elementwise kernels (misc.cu)
cudaError_t launch_permute(const marble_plan_t* p, const void* src, void* dst, int64_t row_bytes,
                           int inverse, cudaStream_t s);
cudaError_t launch_permute_cast_bf16(const marble_plan_t* p, const float* src, void* dst,
                                     int64_t row_elems, int inverse, cudaStream_t s);
cudaError_t launch_cast_bf16(const float* src, void* dst, int64_t n, cudaStream_t s);
cudaError_t launch_finalize(const marble_plan_t* p, const float* o_acc, const float* m,
                            const float* l, int hq, int d, void* o, float* lse, cudaStream_t s);
cudaError_t launch_bwd_prep(const marble_plan_t* p, const void* o, const void* d_o, int hq, int d,
                            float* delta, cudaStream_t s);
cudaError_t launch_debug_wait(unsigned* err, uint64_t limit_ns, cudaStream_t s);

// attention (attn_fwd.cu, attn_bwd.cu): a list of ring steps launched back to back on `s`
marble_status_t run_attn_fwd(const marble_plan_t* p, const marble_qkv_t* qkv, int n_steps,
                             const int* q_shards, const int* kv_shards, const uint32_t* flags,
                             const marble_state_t* st, cudaStream_t s);
// the fused ring (attn_fwd.cu, attn_bwd.cu): every ring step of the pass in one forward
// launch, and one dK/dV launch per kv shard over its ring
marble_status_t run_attn_fwd_fused(const marble_plan_t* p, const marble_qkv_t* qkv,
                                   const marble_state_t* st, cudaStream_t s);
marble_status_t run_attn_bwd_fused(const marble_plan_t* p, const marble_qkv_t* qkv,
                                   const void* d_o, const float* lse, const float* delta,
                                   float* dq, float* dk, float* dv, cudaStream_t s);
marble_status_t run_attn_bwd(const marble_plan_t* p, const marble_qkv_t* qkv, const void* d_o,
                             const float* lse, const float* delta, int n_steps,
                             const int* q_shards, const int* kv_shards, float* dq, float* dk,
                             float* dv, cudaStream_t s);

// true the first time it is called for (key, current device); used for per-device set-up
bool once_per_device(int key);

// Device memory of plans, planner temporaries and the backward scratch comes from a
// library-owned memory pool per device, allocated and freed in stream order: no call
// synchronises the device (cudaFree does), and freed blocks stay in the pool for the next
// plan.
cudaError_t dev_alloc(void** p, size_t bytes, cudaStream_t s);
cudaError_t dev_free(void* p, cudaStream_t s);

// side stream idx of the current device (nullptr if it cannot be created or idx is at or
// above the cap of marble_set_side_streams), and an ordering edge from everything queued on
// `from` so far to everything queued on `to` afterwards
constexpr int kSideStreams = 4;
cudaStream_t side_stream(int idx = 0);
cudaError_t stream_fork(cudaStream_t from, cudaStream_t to);

// per-kernel timing (marble_timing_enable): kinds of kernels, and a span of launches of one
// kind on one stream, opened before the first launch and closed after the last
enum TimingKind { kTimeFwd = 0, kTimeDq = 1, kTimeDkdv = 2 };
bool timing_on();
int timing_begin(cudaStream_t s);  // -1 when timing is off
void timing_end(int span, cudaStream_t s, int kind, int launches);

}  // namespace marble
