// C ABI of libmarble: argument validation, plan lifetime, statistics and exports, and
// the launches of the planner, attention and helper kernels.  Declarations and the
// contract of every call are in include/marble.h.
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <map>
#include <set>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace marble {

static thread_local std::string g_last_error;
static uint64_t g_wait_limit_ns = 0;

void set_error(const std::string& msg) { g_last_error = msg; }

marble_status_t fail(marble_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

marble_status_t cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return MARBLE_ERR_CUDA;
}

uint64_t wait_limit_ns() {
  if (g_wait_limit_ns == 0) {
    const char* env = std::getenv("MARBLE_WAIT_LIMIT_MS");
    uint64_t ms = env ? std::strtoull(env, nullptr, 10) : 0;
    g_wait_limit_ns = ms ? ms * 1000000ull : 2000000000ull;
  }
  return g_wait_limit_ns;
}

bool once_per_device(int key) {
  static std::mutex mu;
  static std::set<std::pair<int, int>> seen;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  return seen.insert({key, dev}).second;
}

// the most side streams the step-list calls may use (marble_set_side_streams)
std::atomic<int> g_side_limit{kSideStreams};

static cudaMemPool_t mem_pool() {
  static std::mutex mu;
  static std::map<int, cudaMemPool_t> pools;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = pools.find(dev);
  if (it != pools.end()) return it->second;
  cudaMemPoolProps props;
  memset(&props, 0, sizeof(props));
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  cudaMemPool_t pool = nullptr;
  if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  uint64_t keep = UINT64_MAX;  // freed blocks stay in the pool
  cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
  pools[dev] = pool;
  return pool;
}

cudaError_t dev_alloc(void** p, size_t bytes, cudaStream_t s) {
  cudaMemPool_t pool = mem_pool();
  if (!pool) return cudaErrorMemoryAllocation;
  return cudaMallocFromPoolAsync(p, bytes, pool, s);
}

cudaError_t dev_free(void* p, cudaStream_t s) { return cudaFreeAsync(p, s); }

// Side streams, created once per device and index: work queued on one between a fork from
// `s` and the join back into `s` runs after everything queued on `s` before the fork, and
// everything queued on `s` after the join runs after it.

cudaStream_t side_stream(int idx) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, cudaStream_t> streams;
  if (idx < 0 || idx >= kSideStreams || idx >= g_side_limit.load()) return nullptr;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = streams.find({dev, idx});
  if (it != streams.end()) return it->second;
  cudaStream_t st = nullptr;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  streams[{dev, idx}] = st;
  return st;
}

namespace {
struct TimingSpan {
  cudaEvent_t a = nullptr, b = nullptr;
  int kind = 0, launches = 0;
};
std::mutex g_timing_mu;
bool g_timing = false;
std::vector<TimingSpan> g_spans;
}  // namespace

bool timing_on() {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  return g_timing;
}

int timing_begin(cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  if (!g_timing) return -1;
  TimingSpan t;
  if (cudaEventCreate(&t.a) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  cudaEventRecord(t.a, s);
  g_spans.push_back(t);
  return (int)g_spans.size() - 1;
}

void timing_end(int span, cudaStream_t s, int kind, int launches) {
  if (span < 0) return;
  std::lock_guard<std::mutex> lock(g_timing_mu);
  if (span >= (int)g_spans.size()) return;
  TimingSpan& t = g_spans[span];
  if (cudaEventCreate(&t.b) != cudaSuccess) {
    (void)cudaGetLastError();
    t.b = nullptr;
    return;
  }
  cudaEventRecord(t.b, s);
  t.kind = kind;
  t.launches = launches;
}

void plan_used(const marble_plan_t* p, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(p->use_mu);
  cudaEvent_t ev = nullptr;
  for (auto& u : p->uses)
    if (u.first == s) ev = u.second;
  if (!ev) {
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
      (void)cudaGetLastError();
      return;
    }
    p->uses.push_back({s, ev});
  }
  if (cudaEventRecord(ev, s) != cudaSuccess) (void)cudaGetLastError();
}

// the stream on which plans of the current device are freed (created once per device)
static cudaStream_t teardown_stream() {
  static std::mutex mu;
  static std::map<int, cudaStream_t> streams;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = streams.find(dev);
  if (it != streams.end()) return it->second;
  cudaStream_t st = nullptr;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  streams[dev] = st;
  return st;
}

// cached dS^T scratch buffers per device: at most kScratchKept; a buffer put beyond that
// goes back to the pool, in stream order after its last use
namespace {
constexpr size_t kScratchKept = 2;
struct CachedScratch {
  void* ptr;
  size_t bytes;
  cudaEvent_t ready;
};
std::mutex g_scratch_mu;
std::map<int, std::vector<CachedScratch>> g_scratch;
}  // namespace

void scratch_put(int device, void* ptr, size_t bytes, cudaEvent_t ready) {
  std::vector<CachedScratch> drop;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    auto& v = g_scratch[device];
    v.push_back({ptr, bytes, ready});
    while (v.size() > kScratchKept) {
      drop.push_back(v.front());
      v.erase(v.begin());
    }
  }
  for (auto& c : drop) {
    cudaStream_t fs = teardown_stream();
    if (fs && cudaStreamWaitEvent(fs, c.ready, 0) == cudaSuccess) dev_free(c.ptr, fs);
    cudaEventDestroy(c.ready);
  }
}

void* scratch_take(size_t bytes, cudaStream_t s, size_t* got) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  CachedScratch c{nullptr, 0, nullptr};
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    auto it = g_scratch.find(dev);
    if (it == g_scratch.end()) return nullptr;
    auto& v = it->second;
    // the oldest buffer that fits without holding more than twice the need
    for (size_t i = 0; i < v.size(); ++i) {
      if (v[i].bytes >= bytes && v[i].bytes / 2 <= bytes) {
        c = v[i];
        v.erase(v.begin() + (long)i);
        break;
      }
    }
  }
  if (!c.ptr) return nullptr;
  if (cudaStreamWaitEvent(s, c.ready, 0) != cudaSuccess) {
    // not usable on this stream: back to the pool after its last use
    (void)cudaGetLastError();
    cudaStream_t fs = teardown_stream();
    if (fs && cudaStreamWaitEvent(fs, c.ready, 0) == cudaSuccess) dev_free(c.ptr, fs);
    cudaEventDestroy(c.ready);
    return nullptr;
  }
  cudaEventDestroy(c.ready);  // released once the wait above has been satisfied
  *got = c.bytes;
  return c.ptr;
}

// the calling thread's pinned staging buffer, grown to at least `bytes`
static void* pinned_stage(size_t bytes, cudaError_t* err) {
  thread_local void* buf = nullptr;
  thread_local size_t cap = 0;
  if (bytes > cap) {
    size_t want = cap ? cap : 4096;
    while (want < bytes) want *= 2;
    void* q = nullptr;
    const cudaError_t e = cudaHostAlloc(&q, want, cudaHostAllocDefault);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    if (buf) cudaFreeHost(buf);
    buf = q;
    cap = want;
  }
  *err = cudaSuccess;
  return buf;
}

static size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

cudaError_t read_back(cudaStream_t s, std::initializer_list<HostPart> parts) {
  size_t total = 0;
  for (const HostPart& h : parts) total += round16(h.bytes);
  cudaError_t e = cudaSuccess;
  uint8_t* stage = static_cast<uint8_t*>(pinned_stage(total, &e));
  if (!stage) return e;
  size_t off = 0;
  for (const HostPart& h : parts) {
    if (h.bytes) {
      e = cudaMemcpyAsync(stage + off, h.dev, h.bytes, cudaMemcpyDeviceToHost, s);
      if (e != cudaSuccess) return e;
    }
    off += round16(h.bytes);
  }
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  off = 0;
  for (const HostPart& h : parts) {
    if (h.bytes) memcpy(h.host, stage + off, h.bytes);
    off += round16(h.bytes);
  }
  return cudaSuccess;
}

cudaError_t write_to_device(cudaStream_t s, void* dev, const void* host, size_t bytes) {
  if (!bytes) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  void* stage = pinned_stage(bytes, &e);
  if (!stage) return e;
  // every user of the buffer synchronises its stream before returning: no copy still reads it
  memcpy(stage, host, bytes);
  e = cudaMemcpyAsync(dev, stage, bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

cudaError_t stream_fork(cudaStream_t from, cudaStream_t to) {
  cudaEvent_t e;
  cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
  if (r != cudaSuccess) return r;
  r = cudaEventRecord(e, from);
  if (r == cudaSuccess) r = cudaStreamWaitEvent(to, e, 0);
  cudaEventDestroy(e);  // released once the recorded work completes
  return r;
}

// true for device or managed memory of the current context
bool is_device_ptr(const void* p) {
  if (!p) return false;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static marble_status_t check_tensor(const void* p, const char* name) {
  if (!p) return fail(MARBLE_ERR_INVALID_ARG, std::string(name) + " is null");
  if (!aligned16(p)) return fail(MARBLE_ERR_INVALID_ARG, std::string(name) + " is not 16-byte aligned");
  if (!is_device_ptr(p)) return fail(MARBLE_ERR_INVALID_ARG, std::string(name) + " is not device memory");
  return MARBLE_OK;
}

static marble_status_t check_qkv(const marble_plan_t* p, const marble_qkv_t* qkv) {
  if (!qkv) return fail(MARBLE_ERR_INVALID_ARG, "qkv is null");
  if (qkv->d != 64 && qkv->d != 128)
    return fail(MARBLE_ERR_INVALID_ARG, "head dim d must be 64 or 128");
  if (qkv->hq < 1 || qkv->hkv < 1 || qkv->hq % qkv->hkv)
    return fail(MARBLE_ERR_INVALID_ARG, "hq must be a positive multiple of hkv");
  if ((int64_t)p->bps * qkv->hq > INT_MAX)
    return fail(MARBLE_ERR_UNSUPPORTED, "too many (block, head) work units per shard");
  if (!(qkv->scale >= 0.f) || std::isinf(qkv->scale))
    return fail(MARBLE_ERR_INVALID_ARG, "scale must be finite and >= 0 (0 = 1/sqrt(d))");
  marble_status_t st;
  if ((st = check_tensor(qkv->q, "q")) != MARBLE_OK) return st;
  if ((st = check_tensor(qkv->k, "k")) != MARBLE_OK) return st;
  if ((st = check_tensor(qkv->v, "v")) != MARBLE_OK) return st;
  return MARBLE_OK;
}

static marble_status_t check_shards(const marble_plan_t* p, int q_shard, int kv_shard) {
  if (q_shard < 0 || q_shard >= p->P)
    return fail(MARBLE_ERR_INVALID_ARG, "q_shard out of range");
  if (kv_shard != MARBLE_KV_NEEDED && (kv_shard < 0 || kv_shard >= p->P))
    return fail(MARBLE_ERR_INVALID_ARG, "kv_shard out of range");
  return MARBLE_OK;
}

}  // namespace marble

using namespace marble;

#define MARBLE_API extern "C" __attribute__((visibility("default")))

MARBLE_API marble_status_t marble_plan(const marble_plan_desc_t* d, marble_stream_t stream,
                                       marble_plan_t** out) {
  NvtxRange nvtx_("marble_plan");
  if (!d || !out) return fail(MARBLE_ERR_INVALID_ARG, "desc and out must be non-null");
  *out = nullptr;
  if (d->n_tokens <= 0 || d->n_tokens % MARBLE_BLOCK || d->n_tokens >= (int64_t)INT_MAX)
    return fail(MARBLE_ERR_INVALID_ARG, "n_tokens must be a positive multiple of 128 below 2^31");
  if (d->window < 0) return fail(MARBLE_ERR_INVALID_ARG, "window must be >= 0");
  if (d->num_shards < 1 || d->num_shards > 256)
    return fail(MARBLE_ERR_INVALID_ARG, "num_shards must be in [1, 256]");
  const int64_t nb = d->n_tokens / MARBLE_BLOCK;
  if (nb % d->num_shards)
    return fail(MARBLE_ERR_INVALID_ARG, "number of 128-token blocks must be divisible by num_shards");
  if (d->order < MARBLE_ORDER_CONTIGUOUS || d->order > MARBLE_ORDER_CHUNK_SEARCH)
    return fail(MARBLE_ERR_INVALID_ARG, "unknown order");
  if (d->order == MARBLE_ORDER_CHUNK_SEARCH && d->range_cost < 0)
    return fail(MARBLE_ERR_INVALID_ARG, "range_cost must be >= 0");
  if (d->order == MARBLE_ORDER_PTRR_CHUNK) {
    if (d->chunk_tokens <= 0 || d->chunk_tokens % MARBLE_BLOCK || d->n_tokens % d->chunk_tokens ||
        (d->n_tokens / d->chunk_tokens) % d->num_shards)
      return fail(MARBLE_ERR_INVALID_ARG,
                  "chunk_tokens must be a multiple of 128 dividing n_tokens into a multiple of "
                  "num_shards chunks");
  }
  if (!is_device_ptr(d->sample_id) || !is_device_ptr(d->seg_id) || !is_device_ptr(d->noise_id))
    return fail(MARBLE_ERR_INVALID_ARG, "track arrays must be device memory");
  if (d->pos_id && !is_device_ptr(d->pos_id))
    return fail(MARBLE_ERR_INVALID_ARG, "pos_id must be device memory");
  marble_plan_t* p = new (std::nothrow) marble_plan_t();
  if (!p) return fail(MARBLE_ERR_OOM, "host allocation failed");
  cudaGetDevice(&p->device);
  p->n = d->n_tokens;
  p->nb = nb;
  p->P = d->num_shards;
  p->W = d->window;
  p->order = d->order;
  p->chunk_tokens = d->chunk_tokens;
  p->range_cost = d->order == MARBLE_ORDER_CHUNK_SEARCH ? d->range_cost : 0;
  p->bps = nb / d->num_shards;
  marble_status_t st = build_plan(d, (cudaStream_t)stream, p);
  plan_used(p, (cudaStream_t)stream);  // the planner's kernels, also on failure
  if (st != MARBLE_OK) {
    std::string msg = g_last_error;
    marble_plan_destroy(p);
    g_last_error = msg;
    return st;
  }
  *out = p;
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_plan_destroy(marble_plan_t* p) {
  NvtxRange nvtx_("marble_plan_destroy");
  if (!p) return MARBLE_OK;
  // Free in stream order, without synchronising anything: a library stream of the plan's
  // device waits for the last recorded use of the plan on every stream that used it, then
  // returns the workspace to the memory pool.  The host object goes at once.
  int prev = 0;
  cudaError_t err = cudaGetDevice(&prev);
  if (err == cudaSuccess && prev != p->device) err = cudaSetDevice(p->device);
  cudaStream_t fs = err == cudaSuccess ? teardown_stream() : nullptr;
  if (err == cudaSuccess && !fs) err = cudaErrorUnknown;
  {
    std::lock_guard<std::mutex> lock(p->use_mu);
    for (auto& u : p->uses) {
      if (err == cudaSuccess) err = cudaStreamWaitEvent(fs, u.second, 0);
      cudaEventDestroy(u.second);  // released once the recorded work completes
    }
    p->uses.clear();
  }
  if (err == cudaSuccess) {
    for (void* q : p->owned) {
      const cudaError_t e = dev_free(q, fs);
      if (err == cudaSuccess) err = e;
    }
    if (p->ds_scratch) {
      // the dS^T scratch goes to the cache for the next plan's backward, ready once the
      // teardown stream has passed the plan's last uses
      cudaEvent_t ready = nullptr;
      cudaError_t e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventRecord(ready, fs);
      if (e == cudaSuccess) {
        scratch_put(p->device, p->ds_scratch, p->ds_scratch_bytes, ready);
      } else {
        if (ready) cudaEventDestroy(ready);
        e = dev_free(p->ds_scratch, fs);
      }
      if (err == cudaSuccess) err = e;
    }
  }
  if (prev != p->device) cudaSetDevice(prev);
  delete p;
  if (err != cudaSuccess) return cuda_fail(err, "marble_plan_destroy: stream-ordered free");
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_chunk_layout_search(const int64_t* block_pairs, int64_t n_blocks,
                                                      int32_t num_shards, int64_t range_cost,
                                                      int32_t* chunk_rank, int64_t* out) {
  NvtxRange nvtx_("marble_chunk_layout_search");
  if (!block_pairs || !chunk_rank || !out)
    return fail(MARBLE_ERR_INVALID_ARG, "block_pairs, chunk_rank and out must be non-null");
  if (num_shards < 1 || num_shards > 256 || n_blocks < 1 || n_blocks % num_shards)
    return fail(MARBLE_ERR_INVALID_ARG, "n_blocks must be a positive multiple of num_shards <= 256");
  if (n_blocks > 65536) return fail(MARBLE_ERR_INVALID_ARG, "n_blocks must be <= 65536");
  if (range_cost < 0) return fail(MARBLE_ERR_INVALID_ARG, "range_cost must be >= 0");
  const int Kf = marble::finest_chunks(n_blocks, num_shards);
  const int64_t cs = n_blocks / Kf;
  std::vector<int64_t> wf((size_t)Kf * Kf, 0);
  for (int64_t a = 0; a < n_blocks; ++a)
    for (int64_t b = 0; b < n_blocks; ++b) {
      const int64_t v = block_pairs[a * n_blocks + b];
      if (v < 0) return fail(MARBLE_ERR_INVALID_ARG, "block_pairs must be >= 0");
      wf[(size_t)(a / cs) * Kf + b / cs] += v;
    }
  int k = 0;
  std::vector<int> rank;
  marble::chunk_layout_host(wf, Kf, num_shards, range_cost, &k, &rank, &out[1], &out[2]);
  out[0] = k;
  for (size_t u = 0; u < rank.size(); ++u) chunk_rank[u] = rank[u];
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_layout_vision_groups(const int32_t* sample, const int32_t* seg,
                                                       int64_t n, int32_t* perm) {
  NvtxRange nvtx_("marble_layout_vision_groups");
  if (!sample || !seg || !perm) return fail(MARBLE_ERR_INVALID_ARG, "arrays must be non-null");
  if (n < 0 || n >= (int64_t)INT_MAX) return fail(MARBLE_ERR_INVALID_ARG, "bad n");
  for (int64_t i = 0; i < n; ++i)
    if ((i > 0 && sample[i] < sample[i - 1]) || sample[i] < 0 || seg[i] < -1)
      return fail(MARBLE_ERR_INVALID_ARG,
                  "sample ids must be >= 0 and non-decreasing, seg ids >= -1");
  int64_t o = 0;
  std::map<int32_t, int> nruns;
  std::vector<std::pair<int64_t, int64_t>> runs, grouped;
  for (int64_t a = 0; a < n;) {
    int64_t b = a;
    while (b < n && sample[b] == sample[a]) ++b;  // the sample [a, b)
    runs.clear();
    nruns.clear();
    for (int64_t i = a; i < b;) {
      int64_t j = i + 1;
      while (j < b && seg[j] == seg[i]) ++j;
      runs.push_back({i, j});
      if (seg[i] >= 0) ++nruns[seg[i]];
      i = j;
    }
    grouped.clear();
    for (const auto& r : runs) {
      const int32_t g = seg[r.first];
      if (g >= 0 && nruns[g] > 1) {
        grouped.push_back(r);
      } else {
        for (int64_t t = r.first; t < r.second; ++t) perm[o++] = (int32_t)t;
      }
    }
    for (auto it = grouped.rbegin(); it != grouped.rend(); ++it)
      for (int64_t t = it->first; t < it->second; ++t) perm[o++] = (int32_t)t;
    a = b;
  }
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_plan_stats(const marble_plan_t* p, marble_stream_t stream,
                                             marble_plan_stats_t* out) {
  NvtxRange nvtx_("marble_plan_stats");
  if (!p || !out) return fail(MARBLE_ERR_INVALID_ARG, "plan and out must be non-null");
  cudaStream_t s = (cudaStream_t)stream;
  memset(out, 0, sizeof(*out));
  out->n_tokens = p->n;
  out->n_blocks = p->nb;
  out->num_shards = p->P;
  out->nnz = p->nnz;
  marble_status_t st = plan_legal_pairs(p, s, &out->legal_pairs, &out->n_full, &out->n_partial,
                                        &out->step_cost_pairs);
  plan_used(p, s);
  if (st != MARBLE_OK) return st;
  const int64_t np = p->nb * p->P + 1;
  std::vector<int64_t> ptr(np);
  std::vector<int64_t> nptr(p->P + 1);
  std::vector<int32_t> needed(p->needed_total);
  const cudaError_t e = read_back(s, {{ptr.data(), p->step_ptr, (size_t)np * 8},
                                      {nptr.data(), p->needed_ptr, (size_t)(p->P + 1) * 8},
                                      {needed.data(), p->needed, (size_t)p->needed_total * 4}});
  if (e != cudaSuccess) return cuda_fail(e, "marble_plan_stats copies");
  const int P = p->P;
  std::vector<int64_t> W((size_t)P * P, 0);
  for (int64_t nq = 0; nq < p->nb; ++nq)
    for (int j = 0; j < P; ++j)
      W[(nq / p->bps) * P + j] += ptr[nq * P + j + 1] - ptr[nq * P + j];
  int64_t mx = 0, sum = 0, sc = 0;
  for (int r = 0; r < P; ++r) {
    int64_t c = 0;
    for (int j = 0; j < P; ++j) c += W[r * P + j];
    mx = c > mx ? c : mx;
    sum += c;
  }
  for (int s2 = 0; s2 < P; ++s2) {
    int64_t best = 0;
    for (int r = 0; r < P; ++r) {
      const int64_t v = W[r * P + ((r - s2) % P + P) % P];
      best = v > best ? v : best;
    }
    sc += best;
  }
  out->shard_cost_max = mx;
  out->shard_cost_sum = sum;
  out->step_cost = sc;
  out->needed_total = p->needed_total;
  int64_t remote = 0;
  for (int r = 0; r < P; ++r)
    for (int64_t x = nptr[r]; x < nptr[r + 1]; ++x)
      remote += (needed[x] / p->bps) != r;
  out->needed_remote = remote;
  out->chunks_per_rank = p->chunks_per_rank;
  out->layout_cost = p->layout_cost;
  out->layout_step_cost = p->layout_step_cost;
  return MARBLE_OK;
}

static bool field_info(const marble_plan_t* p, int32_t field, const void** src, size_t* bytes) {
  const int64_t n = p->n, nb = p->nb, P = p->P;
  switch (field) {
    case MARBLE_FIELD_PERM: *src = p->perm; *bytes = n * 4; return true;
    case MARBLE_FIELD_BLOCK_PERM: *src = p->block_perm; *bytes = nb * 4; return true;
    case MARBLE_FIELD_TRACKS_PERM: *src = p->tracks; *bytes = 4 * n * 4; return true;
    case MARBLE_FIELD_TILE_ROWPTR: *src = p->row_ptr; *bytes = (nb + 1) * 8; return true;
    case MARBLE_FIELD_TILE_COL: *src = p->col; *bytes = p->nnz * 4; return true;
    case MARBLE_FIELD_TILE_TAG: *src = p->tag; *bytes = p->nnz; return true;
    case MARBLE_FIELD_STEP_PTR: *src = p->step_ptr; *bytes = (nb * P + 1) * 8; return true;
    case MARBLE_FIELD_STEP_COL: *src = p->step_col; *bytes = p->nnz * 4; return true;
    case MARBLE_FIELD_STEP_TAG: *src = p->step_tag; *bytes = p->nnz; return true;
    case MARBLE_FIELD_COLT_PTR: *src = p->colT_ptr; *bytes = (nb * P + 1) * 8; return true;
    case MARBLE_FIELD_COLT_ROW: *src = p->colT_row; *bytes = p->nnz * 4; return true;
    case MARBLE_FIELD_COLT_TAG: *src = p->colT_tag; *bytes = p->nnz; return true;
    case MARBLE_FIELD_NEEDED_PTR: *src = p->needed_ptr; *bytes = (P + 1) * 8; return true;
    case MARBLE_FIELD_NEEDED: *src = p->needed; *bytes = p->needed_total * 4; return true;
    case MARBLE_FIELD_KEY_INTERVALS: *src = p->kiv; *bytes = 2 * n * 4; return true;
    case MARBLE_FIELD_INTERVAL_BLOCKS: *src = p->iv_block; *bytes = nb; return true;
    default: return false;
  }
}

MARBLE_API marble_status_t marble_plan_field_bytes(const marble_plan_t* p, int32_t field,
                                                   size_t* bytes) {
  const void* src = nullptr;
  if (!p || !bytes) return fail(MARBLE_ERR_INVALID_ARG, "plan and bytes must be non-null");
  if (!field_info(p, field, &src, bytes)) return fail(MARBLE_ERR_INVALID_ARG, "unknown field");
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_plan_export(const marble_plan_t* p, int32_t field, void* dst,
                                              size_t bytes, marble_stream_t stream) {
  NvtxRange nvtx_("marble_plan_export");
  const void* src = nullptr;
  size_t want = 0;
  if (!p || (!dst && bytes)) return fail(MARBLE_ERR_INVALID_ARG, "plan and dst must be non-null");
  if (!field_info(p, field, &src, &want)) return fail(MARBLE_ERR_INVALID_ARG, "unknown field");
  if (bytes != want) return fail(MARBLE_ERR_INVALID_ARG, "bytes does not match the field size");
  if (!bytes) return MARBLE_OK;
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "marble_plan_export");
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_permute(const marble_plan_t* p, const void* src, void* dst,
                                          int64_t row_bytes, int32_t inverse,
                                          marble_stream_t stream) {
  NvtxRange nvtx_("marble_permute");
  if (!p) return fail(MARBLE_ERR_INVALID_ARG, "plan is null");
  if (row_bytes <= 0 || row_bytes % 4)
    return fail(MARBLE_ERR_INVALID_ARG, "row_bytes must be a positive multiple of 4");
  marble_status_t st;
  if ((st = check_tensor(src, "src")) != MARBLE_OK) return st;
  if ((st = check_tensor(dst, "dst")) != MARBLE_OK) return st;
  const char* a = static_cast<const char*>(src);
  const char* b = static_cast<const char*>(dst);
  const int64_t bytes = p->n * row_bytes;
  if (a < b + bytes && b < a + bytes) return fail(MARBLE_ERR_INVALID_ARG, "src and dst overlap");
  cudaError_t e = launch_permute(p, src, dst, row_bytes, inverse ? 1 : 0, (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "marble_permute launch");
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_permute_cast_bf16(const marble_plan_t* p, const float* src,
                                                    void* dst, int64_t row_elems,
                                                    int32_t inverse, marble_stream_t stream) {
  NvtxRange nvtx_("marble_permute_cast_bf16");
  if (!p) return fail(MARBLE_ERR_INVALID_ARG, "plan is null");
  if (row_elems <= 0 || row_elems % 4)
    return fail(MARBLE_ERR_INVALID_ARG, "row_elems must be a positive multiple of 4");
  marble_status_t st;
  if ((st = check_tensor(src, "src")) != MARBLE_OK) return st;
  if ((st = check_tensor(dst, "dst")) != MARBLE_OK) return st;
  const char* a = reinterpret_cast<const char*>(src);
  const char* b = static_cast<const char*>(dst);
  if (a < b + p->n * row_elems * 2 && b < a + p->n * row_elems * 4)
    return fail(MARBLE_ERR_INVALID_ARG, "src and dst overlap");
  cudaError_t e = launch_permute_cast_bf16(p, src, dst, row_elems, inverse ? 1 : 0,
                                           (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "marble_permute_cast_bf16 launch");
  return MARBLE_OK;
}

constexpr uint32_t kMergeBits = MARBLE_STEP_BF16_MERGE | MARBLE_STEP_FP32_MERGE;

// known bits only, and at most one merge variant
static bool step_flags_ok(uint32_t f) {
  return !(f & ~(MARBLE_STEP_FIRST | kMergeBits)) && (f & kMergeBits) != kMergeBits;
}

MARBLE_API marble_status_t marble_attn_step(const marble_plan_t* p, const marble_qkv_t* qkv,
                                            int32_t q_shard, int32_t kv_shard,
                                            const marble_state_t* state, uint32_t flags,
                                            marble_stream_t stream) {
  NvtxRange nvtx_("marble_attn_step");
  if (!p || !state) return fail(MARBLE_ERR_INVALID_ARG, "plan and state must be non-null");
  marble_status_t st;
  if ((st = check_qkv(p, qkv)) != MARBLE_OK) return st;
  if ((st = check_shards(p, q_shard, kv_shard)) != MARBLE_OK) return st;
  if ((st = check_tensor(state->o_acc, "state.o_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(state->m, "state.m")) != MARBLE_OK) return st;
  if ((st = check_tensor(state->l, "state.l")) != MARBLE_OK) return st;
  if (!step_flags_ok(flags)) return fail(MARBLE_ERR_INVALID_ARG, "unknown or conflicting flags");
  st = run_attn_fwd(p, qkv, 1, &q_shard, &kv_shard, &flags, state, (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  return st;
}

static marble_status_t check_step_list(const marble_plan_t* p, int32_t n_steps,
                                       const int32_t* q_shards, const int32_t* kv_shards) {
  if (n_steps < 0) return fail(MARBLE_ERR_INVALID_ARG, "n_steps must be >= 0");
  if (n_steps > 0 && (!q_shards || !kv_shards))
    return fail(MARBLE_ERR_INVALID_ARG, "step arrays must be non-null");
  for (int32_t i = 0; i < n_steps; ++i) {
    marble_status_t st = check_shards(p, q_shards[i], kv_shards[i]);
    if (st != MARBLE_OK) return st;
  }
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_attn_steps(const marble_plan_t* p, const marble_qkv_t* qkv,
                                             int32_t n_steps, const int32_t* q_shards,
                                             const int32_t* kv_shards, const uint32_t* flags,
                                             const marble_state_t* state,
                                             marble_stream_t stream) {
  NvtxRange nvtx_("marble_attn_steps");
  if (!p || !state) return fail(MARBLE_ERR_INVALID_ARG, "plan and state must be non-null");
  marble_status_t st;
  if ((st = check_qkv(p, qkv)) != MARBLE_OK) return st;
  if ((st = check_step_list(p, n_steps, q_shards, kv_shards)) != MARBLE_OK) return st;
  if (n_steps > 0 && !flags) return fail(MARBLE_ERR_INVALID_ARG, "flags must be non-null");
  for (int32_t i = 0; i < n_steps; ++i) {
    if (!step_flags_ok(flags[i]))
      return fail(MARBLE_ERR_INVALID_ARG, "unknown or conflicting flags");
    if ((flags[i] ^ flags[0]) & kMergeBits)
      return fail(MARBLE_ERR_INVALID_ARG, "the merge flags differ between steps");
  }
  if ((st = check_tensor(state->o_acc, "state.o_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(state->m, "state.m")) != MARBLE_OK) return st;
  if ((st = check_tensor(state->l, "state.l")) != MARBLE_OK) return st;
  if (n_steps == 0) return MARBLE_OK;
  st = run_attn_fwd(p, qkv, n_steps, q_shards, kv_shards, flags, state, (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  return st;
}

MARBLE_API marble_status_t marble_attn_bwd_steps(const marble_plan_t* p, const marble_qkv_t* qkv,
                                                 const void* d_o, const float* lse,
                                                 const float* delta, int32_t n_steps,
                                                 const int32_t* q_shards,
                                                 const int32_t* kv_shards, float* dq_acc,
                                                 float* dk_acc, float* dv_acc,
                                                 marble_stream_t stream) {
  NvtxRange nvtx_("marble_attn_bwd_steps");
  if (!p) return fail(MARBLE_ERR_INVALID_ARG, "plan is null");
  marble_status_t st;
  if ((st = check_qkv(p, qkv)) != MARBLE_OK) return st;
  if ((st = check_step_list(p, n_steps, q_shards, kv_shards)) != MARBLE_OK) return st;
  if ((st = check_tensor(d_o, "d_o")) != MARBLE_OK) return st;
  if ((st = check_tensor(lse, "lse")) != MARBLE_OK) return st;
  if ((st = check_tensor(delta, "delta")) != MARBLE_OK) return st;
  if ((st = check_tensor(dq_acc, "dq_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(dk_acc, "dk_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(dv_acc, "dv_acc")) != MARBLE_OK) return st;
  if (n_steps == 0) return MARBLE_OK;
  st = run_attn_bwd(p, qkv, d_o, lse, delta, n_steps, q_shards, kv_shards, dq_acc, dk_acc,
                    dv_acc, (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  return st;
}

MARBLE_API marble_status_t marble_attn_fwd_fused(const marble_plan_t* p, const marble_qkv_t* qkv,
                                                 const marble_state_t* state,
                                                 marble_stream_t stream) {
  NvtxRange nvtx_("marble_attn_fwd_fused");
  if (!p || !state) return fail(MARBLE_ERR_INVALID_ARG, "plan and state must be non-null");
  marble_status_t st;
  if ((st = check_qkv(p, qkv)) != MARBLE_OK) return st;
  if ((st = check_tensor(state->o_acc, "state.o_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(state->m, "state.m")) != MARBLE_OK) return st;
  if ((st = check_tensor(state->l, "state.l")) != MARBLE_OK) return st;
  st = run_attn_fwd_fused(p, qkv, state, (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  return st;
}

MARBLE_API marble_status_t marble_attn_bwd_fused(const marble_plan_t* p, const marble_qkv_t* qkv,
                                                 const void* d_o, const float* lse,
                                                 const float* delta, float* dq_acc,
                                                 float* dk_acc, float* dv_acc,
                                                 marble_stream_t stream) {
  NvtxRange nvtx_("marble_attn_bwd_fused");
  if (!p) return fail(MARBLE_ERR_INVALID_ARG, "plan is null");
  marble_status_t st;
  if ((st = check_qkv(p, qkv)) != MARBLE_OK) return st;
  if ((st = check_tensor(d_o, "d_o")) != MARBLE_OK) return st;
  if ((st = check_tensor(lse, "lse")) != MARBLE_OK) return st;
  if ((st = check_tensor(delta, "delta")) != MARBLE_OK) return st;
  if ((st = check_tensor(dq_acc, "dq_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(dk_acc, "dk_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(dv_acc, "dv_acc")) != MARBLE_OK) return st;
  st = run_attn_bwd_fused(p, qkv, d_o, lse, delta, dq_acc, dk_acc, dv_acc, (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  return st;
}

MARBLE_API marble_status_t marble_attn_finalize(const marble_plan_t* p,
                                                const marble_state_t* state, int32_t hq,
                                                int32_t d, void* o_bf16, float* lse,
                                                marble_stream_t stream) {
  NvtxRange nvtx_("marble_attn_finalize");
  if (!p || !state) return fail(MARBLE_ERR_INVALID_ARG, "plan and state must be non-null");
  if (d != 64 && d != 128) return fail(MARBLE_ERR_INVALID_ARG, "d must be 64 or 128");
  if (hq < 1) return fail(MARBLE_ERR_INVALID_ARG, "hq must be >= 1");
  marble_status_t st;
  if ((st = check_tensor(state->o_acc, "state.o_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(state->m, "state.m")) != MARBLE_OK) return st;
  if ((st = check_tensor(state->l, "state.l")) != MARBLE_OK) return st;
  if ((st = check_tensor(o_bf16, "o")) != MARBLE_OK) return st;
  if ((st = check_tensor(lse, "lse")) != MARBLE_OK) return st;
  cudaError_t e = launch_finalize(p, state->o_acc, state->m, state->l, hq, d, o_bf16, lse,
                                  (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "marble_attn_finalize launch");
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_attn_bwd_prep(const marble_plan_t* p, const void* o,
                                                const void* d_o, int32_t hq, int32_t d,
                                                float* delta, marble_stream_t stream) {
  NvtxRange nvtx_("marble_attn_bwd_prep");
  if (!p) return fail(MARBLE_ERR_INVALID_ARG, "plan is null");
  if (d != 64 && d != 128) return fail(MARBLE_ERR_INVALID_ARG, "d must be 64 or 128");
  if (hq < 1) return fail(MARBLE_ERR_INVALID_ARG, "hq must be >= 1");
  marble_status_t st;
  if ((st = check_tensor(o, "o")) != MARBLE_OK) return st;
  if ((st = check_tensor(d_o, "d_o")) != MARBLE_OK) return st;
  if ((st = check_tensor(delta, "delta")) != MARBLE_OK) return st;
  cudaError_t e = launch_bwd_prep(p, o, d_o, hq, d, delta, (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "marble_attn_bwd_prep launch");
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_attn_bwd(const marble_plan_t* p, const marble_qkv_t* qkv,
                                           const void* d_o, const float* lse,
                                           const float* delta, int32_t q_shard,
                                           int32_t kv_shard, float* dq_acc, float* dk_acc,
                                           float* dv_acc, uint32_t flags,
                                           marble_stream_t stream) {
  NvtxRange nvtx_("marble_attn_bwd");
  if (!p) return fail(MARBLE_ERR_INVALID_ARG, "plan is null");
  marble_status_t st;
  if ((st = check_qkv(p, qkv)) != MARBLE_OK) return st;
  if ((st = check_shards(p, q_shard, kv_shard)) != MARBLE_OK) return st;
  if ((st = check_tensor(d_o, "d_o")) != MARBLE_OK) return st;
  if ((st = check_tensor(lse, "lse")) != MARBLE_OK) return st;
  if ((st = check_tensor(delta, "delta")) != MARBLE_OK) return st;
  if ((st = check_tensor(dq_acc, "dq_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(dk_acc, "dk_acc")) != MARBLE_OK) return st;
  if ((st = check_tensor(dv_acc, "dv_acc")) != MARBLE_OK) return st;
  if (flags != 0) return fail(MARBLE_ERR_INVALID_ARG, "flags must be 0");
  st = run_attn_bwd(p, qkv, d_o, lse, delta, 1, &q_shard, &kv_shard, dq_acc, dk_acc, dv_acc,
                    (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  return st;
}

MARBLE_API marble_status_t marble_cast_bf16(const float* src, void* dst, int64_t n,
                                            marble_stream_t stream) {
  NvtxRange nvtx_("marble_cast_bf16");
  if (n < 0 || n % 4) return fail(MARBLE_ERR_INVALID_ARG, "n must be a non-negative multiple of 4");
  if (n == 0) return MARBLE_OK;
  marble_status_t st;
  if ((st = check_tensor(src, "src")) != MARBLE_OK) return st;
  if ((st = check_tensor(dst, "dst")) != MARBLE_OK) return st;
  cudaError_t e = launch_cast_bf16(src, dst, n, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "marble_cast_bf16 launch");
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_check(const marble_plan_t* p, marble_stream_t stream) {
  NvtxRange nvtx_("marble_check");
  if (!p) return fail(MARBLE_ERR_INVALID_ARG, "plan is null");
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "asynchronous CUDA error");
  unsigned h = 0;
  e = read_back((cudaStream_t)stream, {{&h, p->err, sizeof(unsigned)}});
  if (e != cudaSuccess) return cuda_fail(e, "reading the plan's error word");
  if (h) {
    e = cudaMemset(p->err, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the plan's error word");
    if (h & kErrTimeout)
      return fail(MARBLE_ERR_TIMEOUT, "a bounded in-kernel wait ran out (error word " +
                                          std::to_string(h) + ")");
    return fail(MARBLE_ERR_CUDA, "device error word " + std::to_string(h));
  }
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_set_side_streams(int32_t n) {
  if (n < 0 || n > kSideStreams) return fail(MARBLE_ERR_INVALID_ARG, "n must be in [0, 4]");
  g_side_limit.store(n);
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_release_memory(void) {
  NvtxRange nvtx_("marble_release_memory");
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "marble_release_memory");
  std::vector<CachedScratch> drop;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    auto it = g_scratch.find(dev);
    if (it != g_scratch.end()) drop.swap(it->second);
  }
  cudaStream_t fs = teardown_stream();
  if (!fs) return cuda_fail(cudaErrorUnknown, "marble_release_memory: teardown stream");
  for (auto& c : drop) {
    cudaError_t e = cudaStreamWaitEvent(fs, c.ready, 0);
    if (e == cudaSuccess) e = dev_free(c.ptr, fs);
    cudaEventDestroy(c.ready);
    if (err == cudaSuccess) err = e;
  }
  const cudaError_t e = cudaStreamSynchronize(fs);
  if (err == cudaSuccess) err = e;
  cudaMemPool_t pool = mem_pool();
  if (err == cudaSuccess && pool) err = cudaMemPoolTrimTo(pool, 0);
  if (err != cudaSuccess) return cuda_fail(err, "marble_release_memory");
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) return fail(MARBLE_ERR_INVALID_ARG, "limit must be > 0");
  g_wait_limit_ns = ns;
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_timing_enable(int on) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  g_timing = on != 0;
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_timing_read(double* out) {
  if (!out) return fail(MARBLE_ERR_INVALID_ARG, "out is null");
  std::lock_guard<std::mutex> lock(g_timing_mu);
  for (int i = 0; i < 6; ++i) out[i] = 0.0;
  cudaError_t err = cudaSuccess;
  for (TimingSpan& t : g_spans) {
    if (t.b) {
      float ms = 0.f;
      cudaError_t e = cudaEventSynchronize(t.b);
      if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.a, t.b);
      if (e == cudaSuccess && t.kind >= 0 && t.kind < 3) {
        out[2 * t.kind] += ms;
        out[2 * t.kind + 1] += t.launches;
      } else if (e != cudaSuccess) {
        err = e;
      }
      cudaEventDestroy(t.b);
    }
    if (t.a) cudaEventDestroy(t.a);
  }
  g_spans.clear();
  if (err != cudaSuccess) return cuda_fail(err, "marble_timing_read");
  return MARBLE_OK;
}

MARBLE_API marble_status_t marble_debug_wait_timeout(const marble_plan_t* p, uint64_t limit_ns,
                                                     marble_stream_t stream) {
  if (!p) return fail(MARBLE_ERR_INVALID_ARG, "plan is null");
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(MARBLE_ERR_INVALID_ARG, "limit_ns must be in (0, 10 s]");
  cudaError_t e = launch_debug_wait(p->err, limit_ns, (cudaStream_t)stream);
  plan_used(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "marble_debug_wait_timeout launch");
  return MARBLE_OK;
}

MARBLE_API const char* marble_last_error(void) { return g_last_error.c_str(); }

MARBLE_API const char* marble_version(void) { return "marble-gb300 0.1 (sm_103a)"; }
