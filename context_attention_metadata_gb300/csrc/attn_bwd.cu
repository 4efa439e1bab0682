// Backward ring step: fp32 dQ / dK / dV accumulation for the tiles between one q shard
// and one kv shard (or every needed kv block), against the FINAL LSE.
//
// MARBLE post, s03 "Exact ring attention accumulation": each step runs the attention
// backward against the final LSE, starting from an fp32 dQ accumulator carried across
// steps, while each kv shard's fp32 dK/dV accumulator travels with the shard; s03 closing
// rule: gradients summed across calls are summed in fp32.
//
// Per tile (S = Q K^T * scale, P = exp(S - LSE), dP = dO V^T, dS = P * (dP - delta)):
//   dV += P^T dO,  dK += scale * dS^T Q,  dQ += scale * dS K.
// Two kernels, so that every accumulator tile has one owner per launch and the kernels never
// add partial tiles of the same accumulator concurrently:
//   k_bwd_dkdv  KV-stationary units (kv block, kv head), looping over the q heads of the
//               group and the q blocks listed for the block: S^T = K Q^T and dP^T = V dO^T in
//               TMEM, P^T and dS^T (bf16) back into TMEM, dV += P^T dO and dK += dS^T Q with
//               dO and Q read MN-major; it also stores each bf16 dS^T tile to a scratch slot
//               numbered by the step's tile order.
//   k_bwd_dq    Q-stationary units (q block, q head): dQ += dS K, a GEMM over the unit's
//               dS^T tiles (read MN-major) and K tiles, after the step's dK/dV kernel.
// Both are persistent (one CTA per SM) and take their units from a ticket counter in the
// plan's order (longest list first), through a 4-entry queue in shared memory.  Warps of the
// dK/dV kernel (the dQ GEMM's are listed with it below):
//   warp 0      TMA producer: the unit's stationary tiles into one slot (refilled once the
//               unit's last score MMAs have read it), the streamed tiles through two stages
//   warp 1      TMEM allocation and MMA issue
//   warp 2      scheduler: ticket -> unit -> queue
//   warp 3      dS^T store: the staged dS^T boxes to the scratch, by TMA
//   warps 4..11 elementwise, four warps (one thread per TMEM lane) for each 64-column half
//               of a tile, with most of the block's registers (warpgroup 0 gives its share
//               up).  At a unit's end the same warps read the fp32 accumulators out of TMEM
//               (releasing them for the next unit, whose first MMAs are already under way),
//               stage them in a shared-memory slot the unit no longer needs and add them to
//               the global accumulators with TMA fp32 reduce-adds (no load).
// Masks only on partial tiles.
#include <math.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tma_host.h"

namespace marble {
namespace {

constexpr int kThreads = 384;  // producer, MMA, scheduler, dS store, 8 elementwise warps
constexpr int kWarpSched = 2;
constexpr int kWarpStore = 3;
// registers per thread: the launch gives every thread 168 (384 x 168 of the SM's 65,536);
// warpgroup 0 (producer, MMA, scheduler, store) hands 112 of each of its threads' to the two
// elementwise warpgroups: 128 x 56 + 256 x 224 = 384 x 168
constexpr int kRegsCtl = 56;
constexpr int kRegsElem = 224;
static_assert(128 * kRegsCtl + 256 * kRegsElem <= kThreads * 168, "register split");
constexpr int kQueue = 4;
constexpr int kDsBufs = 4;        // steps whose dS^T tiles the scratch holds at once (at most)
constexpr size_t kDsScratchCap = size_t(32) << 30;  // fewer buffers (down to 2) above this
constexpr int kDkdvStreams = 4;   // side streams of the dK/dV launches
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxShards = 256;   // the most virtual shards a plan has

struct BwdParams {
  CUtensorMap q_map, k_map, v_map, do_map;
  CUtensorMap dq_map, dk_map, dv_map;  // fp32 accumulators, box 32 x 128 x 1, 128-byte swizzle
  CUtensorMap ds_map;  // bf16 dS^T scratch tiles [slot][128 kv rows][128 q cols], box 64 x 128
  const int64_t* step_ptr;   // row lists (dQ kernel)
  const int32_t* step_col;
  const uint8_t* step_tag;
  const int64_t* colT_ptr;   // column lists (dK/dV kernel)
  const int32_t* colT_row;
  const uint8_t* colT_tag;
  const int64_t* needed_ptr;
  const int32_t* needed;
  const int32_t* order;      // work order of the launch (blocks of one shard, longest first)
  const int32_t* step_off;   // [nb][P+1] tiles of the q shard's earlier q blocks in a step
  const int32_t* colT_j;     // [nnz] index of a column-list entry in its q block's row list
  long long ds_slot0;        // first scratch slot of this step's dS^T tiles
  // fused ring (ring_len > 0, dK/dV kernel only): kv shard kv_shard over ring steps
  // [ring_s0, ring_s0 + ring_len), i.e. q shards (kv_shard + s) mod P, its dK/dV kept on chip
  // across them; the dS^T tile of q block nq lands at ds_base[nq / bps] + (its index in the
  // step's numbering) * hq + head
  int ring_s0, ring_len;
  // whole rows (whole != 0; 2: the dQ GEMM over every q block): the dK/dV kernel stores the
  // dS^T tile of row-list entry e (the plan's row lists, every kv shard) of a q block of shard
  // r at slot ds_base[r] + e * hq + head, and the dQ kernel runs one unit per (q block, q head)
  // over the block's whole row
  int whole;
  long long ds_base[kMaxShards];
  unsigned* sched;           // ticket counter pair of the launch
  const int32_t* tracks;     // [4][n] plan order
  const int32_t* kiv;        // [2][n] lo, hi of every key's visible-query interval
  const int32_t* qidx;       // [n] plan order -> index in the given token order (the plan's perm)
  const uint8_t* iv_block;   // [nb] 1: every key of the block has an exact interval
  const float* lse;          // [hq][n] natural log
  const float* delta;        // [hq][n]
  float* dq;
  float* dk;
  float* dv;
  unsigned* err;
  unsigned long long wait_ns;
  long long n;
  int P, bps, q_shard, kv_shard;
  int hq, hkv, group;
  int nwork;                 // units with a non-empty list
  int W;
  float scale, sl2;
};

// queue entry: head, block (plan order), list start and length; a dK/dV unit of the fused
// ring may have its list in two pieces of the column CSR: entries [0, La) at e0 + x, the
// rest at e1 + (x - La)
struct Queue {
  int head[kQueue];  // -1: no more work
  int blk[kQueue];
  int T[kQueue];
  int La[kQueue];
  long long e0[kQueue];
  long long e1[kQueue];
};

__device__ __forceinline__ int64_t list_entry(int64_t e0, int64_t e1, int La, int x) {
  return x < La ? e0 + x : e1 + (x - La);
}

// ticket -> unit of the dQ kernel: q head h (innermost), q block of the order
__device__ __forceinline__ void dq_unit(const BwdParams& p, unsigned t, int* h, int* blk,
                                        int64_t* e0, int* T) {
  int64_t nq, a, b;
  if (p.whole) {
    // over every q block of the pack (whole == 2) the q heads go outermost, so that the units
    // in flight read one head's K from L2; per q shard they go innermost
    if (p.whole == 2) {
      const unsigned nbk = (unsigned)(p.nwork / p.hq);
      *h = (int)(t / nbk);
      nq = p.order[t % nbk];
    } else {
      *h = (int)(t % (unsigned)p.hq);
      nq = (int64_t)p.q_shard * p.bps + p.order[t / (unsigned)p.hq];
    }
    *blk = (int)nq;
    *e0 = p.step_ptr[nq * p.P];
    *T = (int)(p.step_ptr[nq * p.P + p.P] - *e0);
    return;
  }
  *h = (int)(t % (unsigned)p.hq);
  nq = (int64_t)p.q_shard * p.bps + p.order[t / (unsigned)p.hq];
  if (p.kv_shard >= 0) {
    a = p.step_ptr[nq * p.P + p.kv_shard];
    b = p.step_ptr[nq * p.P + p.kv_shard + 1];
  } else {
    a = p.step_ptr[nq * p.P];
    b = p.step_ptr[nq * p.P + p.P];
  }
  *blk = (int)nq;
  *e0 = a;
  *T = (int)(b - a);
}

// ticket -> unit of the dK/dV kernel: kv head (innermost), kv block of the order (or of the
// needed list); T = number of listed q blocks (items = T x group).  In the fused ring the
// list runs over the q shards of the ring range, in ring order: one CSR range, or two when
// the range wraps past the last shard.
__device__ __forceinline__ void dkdv_unit(const BwdParams& p, unsigned t, int* kh, int* blk,
                                          int64_t* c0, int* T, int64_t* c1, int* La) {
  *kh = (int)(t % (unsigned)p.hkv);
  const unsigned i = t / (unsigned)p.hkv;
  int64_t nk;
  if (p.kv_shard >= 0)
    nk = (int64_t)p.kv_shard * p.bps + p.order[i];
  else
    nk = p.needed[p.needed_ptr[p.q_shard] + i];
  *blk = (int)nk;
  if (p.ring_len > 0) {
    const int a = (p.kv_shard + p.ring_s0) % p.P, b = a + p.ring_len;
    *c0 = p.colT_ptr[nk * p.P + a];
    if (b <= p.P) {
      *La = *T = (int)(p.colT_ptr[nk * p.P + b] - *c0);
      *c1 = 0;
    } else {
      *La = (int)(p.colT_ptr[nk * p.P + p.P] - *c0);
      *c1 = p.colT_ptr[nk * p.P];
      *T = *La + (int)(p.colT_ptr[nk * p.P + (b - p.P)] - *c1);
    }
    return;
  }
  *c0 = p.colT_ptr[nk * p.P + p.q_shard];
  *La = *T = (int)(p.colT_ptr[nk * p.P + p.q_shard + 1] - *c0);
  *c1 = 0;
}

// scheduler loop (one lane): post units until the tickets run out, then a terminator.  An
// entry is rewritten only once every role has released it.
template <bool kDQ>
__device__ void schedule(const BwdParams& p, Queue& queue, uint64_t* ufull, uint64_t* uempty,
                         const WaitCtx& w) {
  for (int uc = 0;; ++uc) {
    const int slot = uc % kQueue;
    if (uc >= kQueue && !mbar_wait(&uempty[slot], ((uc / kQueue) - 1) & 1, w)) return;
    int hd = -1, blk = 0, T = 0, La = 0;
    int64_t e0 = 0, e1 = 0;
    while (true) {  // units with an empty list (needed-block mode, part of a ring) are skipped
      const unsigned t = atomicAdd(p.sched, 1u);
      if (t >= (unsigned)p.nwork) {
        hd = -1;
        break;
      }
      if (kDQ) {
        dq_unit(p, t, &hd, &blk, &e0, &T);
        La = T;
      } else {
        dkdv_unit(p, t, &hd, &blk, &e0, &T, &e1, &La);
      }
      if (T > 0) break;
    }
    queue.head[slot] = hd;
    queue.blk[slot] = blk;
    queue.T[slot] = T;
    queue.La[slot] = La;
    queue.e0[slot] = e0;
    queue.e1[slot] = e1;
    mbar_arrive(&ufull[slot]);
    if (hd < 0) return;
  }
}

// the last CTA of a launch to finish puts the ticket counter pair back to zero
__device__ __forceinline__ void release_tickets(const BwdParams& p) {
  __threadfence();
  if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
    atomicExch(p.sched, 0u);
    atomicExch(p.sched + 1, 0u);
  }
}

// ======================================================================================
// dQ (Q-stationary GEMM over the dS^T tiles the dK/dV kernel wrote)
// ======================================================================================
// For a unit (q block, q head): dQ += dS K over the unit's tiles, A = dS read MN-major from
// the step's scratch tile [kv rows][q columns], B = K read MN-major; dq_acc += scale * dQ at
// the unit's end.  The dS^T tile and the K tile of each tile stream through three stages.
// The accumulator alternates between two TMEM buffers by unit, so that the epilogue warps
// read one out (and add it to dq_acc through staged boxes and TMA reduce-adds) while the
// tensor core accumulates the next unit in the other.
enum {
  G_FULL0, G_FULL1, G_FULL2, G_EMPTY0, G_EMPTY1, G_EMPTY2, G_OFULL0, G_OFULL1, G_OFREE0,
  G_OFREE1, G_STG, G_STGFREE, G_UFULL0, G_UEMPTY0 = G_UFULL0 + kQueue,
  G_DRAIN = G_UEMPTY0 + kQueue, G_NUM
};
constexpr int kGThreads = 224;  // producer, MMA, 4 epilogue warps, scheduler
constexpr int kGWarpSched = 6;

__host__ __device__ constexpr int dqg_arrivals(int b) {
  return (b == G_OFREE0 || b == G_OFREE1 || b == G_STG ||
          (b >= G_UEMPTY0 && b < G_UEMPTY0 + kQueue))
             ? 128
             : 1;
}

// shared memory of the dQ GEMM: three stages of (dS^T tile, two 16 KB boxes | K tile), then
// a staging area of two fp32 boxes
template <int D>
struct DqSmem {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kDs = 32768;
  static constexpr int kStage = kDs + kTile;
  static constexpr int kStg = 3 * kStage;
  static constexpr int kEnd = kStg + 32768;
  static constexpr size_t bytes() { return (size_t)kEnd + 1024; }
};
static_assert(DqSmem<128>::bytes() <= 232448 - 1024, "shared memory budget");

template <int D>
__global__ void __launch_bounds__(kGThreads, 1) k_bwd_dq(const __grid_constant__ BwdParams p) {
  using L = DqSmem<D>;
  constexpr int kTile = L::kTile;
  constexpr int kAtoms = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sStg = smem + L::kStg;
  __shared__ __align__(8) uint64_t bar[G_NUM];
  __shared__ Queue queue;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WaitCtx w{p.wait_ns, p.err, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int b = 0; b < G_NUM; ++b) mbar_init(&bar[b], dqg_arrivals(b));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tQ = tmem_base;  // dQ buffers at +0 and +128
  const int opt = p.kv_shard >= 0 ? p.kv_shard : p.P;  // the step's list option

  if (warp == kGWarpSched) {
    if (lane == 0) schedule<true>(p, queue, &bar[G_UFULL0], &bar[G_UEMPTY0], w);
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.ds_map);
      tma_prefetch_desc(&p.k_map);
    }
    int uc = 0, g = 0, fills[3] = {0, 0, 0};
    bool ok = true;
    while (ok) {
      const int slot = uc % kQueue;
      if (!wait_all(&bar[G_UFULL0 + slot], (uc / kQueue) & 1, w)) break;
      const int h = queue.head[slot];
      if (h < 0) break;
      const int64_t nq = queue.blk[slot];
      const int T = queue.T[slot];
      const int64_t e0 = queue.e0[slot];
      const int kvh = h / p.group;
      // the unit's first dS^T slot: by row-list entry (whole backward) or in the step's order
      const int64_t sl0 = p.whole ? p.ds_base[nq / p.bps] + e0 * p.hq + h
                                  : p.ds_slot0 + p.step_off[nq * (p.P + 1) + opt] * p.hq + h;
      for (int j = 0; j < T; ++j, ++g) {
        const int s = g % 3;
        if (g >= 3 && !wait_all(&bar[G_EMPTY0 + s], ((g / 3) - 1) & 1, w)) { ok = false; break; }
        if (lane == 0) {
          const int nk = p.step_col[e0 + j];
          const int64_t sl = sl0 + (int64_t)j * p.hq;
          uint8_t* st = smem + s * L::kStage;
          mbar_arrive_expect_tx(&bar[G_FULL0 + s], L::kDs + kTile);
          tma_load_3d(st, &p.ds_map, &bar[G_FULL0 + s], 0, (int)(sl * 128), 0);
          tma_load_3d(st + 16384, &p.ds_map, &bar[G_FULL0 + s], 64, (int)(sl * 128), 0);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_3d(st + L::kDs + a * 16384, &p.k_map, &bar[G_FULL0 + s], a * 64, nk * 128,
                        kvh);
        }
        ++fills[s];
      }
      ++uc;
    }
    if (lane == 0)
      for (int s = 0; s < 3; ++s)
        if (fills[s]) drain_wait(&bar[G_FULL0 + s], (fills[s] - 1) & 1, p.wait_ns, p.err);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kId = idesc_bf16(128, D, true, true);  // A and B both MN-major
      int uc = 0, g = 0;
      bool ok = true;
      while (ok) {
        const int slot = uc % kQueue;
        if (!mbar_wait(&bar[G_UFULL0 + slot], (uc / kQueue) & 1, w)) break;
        if (queue.head[slot] < 0) break;
        const int T = queue.T[slot];
        const uint32_t ob = (uint32_t)(uc & 1);
        for (int j = 0; j < T; ++j, ++g) {
          const int s = g % 3;
          if (!mbar_wait(&bar[G_FULL0 + s], (g / 3) & 1, w)) { ok = false; break; }
          // the unit's first MMA overwrites its buffer: the unit two back must be read out
          if (j == 0 && uc >= 2 && !mbar_wait(&bar[G_OFREE0 + ob], ((uc >> 1) - 1) & 1, w)) { ok = false; break; }
          tc_fence_after();
          const uint32_t aS = smem_u32(smem + s * L::kStage), aK = aS + L::kDs;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ss(tQ + ob * 128, sdesc_sw128(aS + k * 2048, 16384, 1024),
                   sdesc_sw128(aK + k * 2048, 16384, 1024), kId, (j > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bar[G_EMPTY0 + s]);
          if (j == T - 1) mma_commit(&bar[G_OFULL0 + ob]);
        }
        ++uc;
      }
      mma_commit(&bar[G_DRAIN]);
      drain_wait(&bar[G_DRAIN], 0, p.wait_ns, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    // one thread per row (warp w owns TMEM lane quarter w & 3)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    int uc = 0, k = 0;  // units, staging rounds
    bool ok = true;
    while (ok) {
      const int slot = uc % kQueue;
      if (!wait_all(&bar[G_UFULL0 + slot], (uc / kQueue) & 1, w)) break;
      const int h = queue.head[slot];
      if (h < 0) break;
      const int64_t nq = queue.blk[slot];
      const uint32_t ob = (uint32_t)(uc & 1);
      if (!wait_all(&bar[G_OFULL0 + ob], (uc >> 1) & 1, w)) break;
      tc_fence_after();
      // the unit's last MMA is done: the producer and the MMA thread are past its entry
      mbar_arrive(&bar[G_UEMPTY0 + slot]);
      // dq_acc += scale * dQ, 64 columns (two staged 128 x 32 boxes) per round
#pragma unroll 1
      for (int r = 0; r < D / 64; ++r, ++k) {
        uint32_t x[2][32];
        tmem_ld32(tQ + ob * 128 + lb + (2 * r) * 32, x[0]);
        tmem_ld32(tQ + ob * 128 + lb + (2 * r + 1) * 32, x[1]);
        tmem_ld_wait();
        if (r == D / 64 - 1) {
          tc_fence_before();
          mbar_arrive(&bar[G_OFREE0 + ob]);  // the buffer can take unit uc + 2
        }
        if (k > 0 && !wait_all(&bar[G_STGFREE], (k - 1) & 1, w)) { ok = false; break; }
        fence_proxy_async_smem();
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          float v[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) v[t] = p.scale * __uint_as_float(x[cb][t]);
          stage_row32(sStg + cb * 16384, row, v);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar[G_STG]);
        if (row == 0) {
          if (mbar_wait(&bar[G_STG], k & 1, w)) {
            for (int cb = 0; cb < 2; ++cb)
              tma_reduce_add_3d(&p.dq_map, sStg + cb * 16384, (2 * r + cb) * 32, (int)(nq * 128), h);
            bulk_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&bar[G_STGFREE]);
        }
      }
      ++uc;
    }
    if (row == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
  if (threadIdx.x == 0) release_tickets(p);
}

// ======================================================================================
// dK / dV (KV-stationary)
// ======================================================================================
// TMEM: two 128-column score regions R0, R1 and the accumulators dV [256, 384), dK [384, 512).
// Item g (counted over all units of the CTA) puts S^T(g) = K Q^T in R[g & 1] and
// dP^T(g) = V dO^T in R[(g + 1) & 1], full width (N = 128 q columns).  The elementwise warps
// load both into registers and say so (YFREE); the dP^T region is then free, and the MMA
// thread issues S^T(g + 1) into it while the warps compute.  Each half of the warps writes
// its bf16 P^T and dS^T into the 64 columns of S^T(g)'s region it has itself read (P^T of q
// columns [64 h, 64 h + 64) in columns [64 h, 64 h + 32), dS^T in [64 h + 32, 64 h + 64)),
// so no half waits for the other (PFULL); the MMA thread
// issues dV += P^T dO and dK += dS^T Q (A from TMEM, K = 128 q), then dP^T(g + 1) into the
// same region, which the tensor core writes only after the two accumulations have read it
// (tcgen05.mma instructions of one thread execute in issue order).  Per item: 32 MMA
// instructions, all N = 128.
// Each half stages its bf16 dS^T (128 kv rows x 64 q columns) in a shared box of its own, from
// which a lane of the store warp writes it to the step's scratch tile with a TMA store.
// The epilogue stages dV, then dK, in the Q/dO stage of the unit's last item (free once the
// unit's last MMAs are done; the epilogue hands it back to the producer) and adds them to
// dv_acc / dk_acc with TMA reduce-adds.
enum {
  K_KVFULL, K_KVEMPTY, K_QFULL0, K_QFULL1, K_QEMPTY0, K_QEMPTY1, K_SDP, K_YFREE, K_PFULL,
  K_ACCFULL, K_ACCFREE, K_STG0, K_STG1, K_STGR0, K_STGR1, K_TRK00, K_TRK01, K_TRK10, K_TRK11,
  K_DSSTG0, K_DSSTG1, K_DSFREE0, K_DSFREE1, K_UFULL0, K_UEMPTY0 = K_UFULL0 + kQueue,
  K_DRAIN = K_UEMPTY0 + kQueue, K_NUM
};

__host__ __device__ constexpr int dkdv_arrivals(int b) {
  return (b == K_ACCFREE || b == K_YFREE || b == K_PFULL ||
          (b >= K_UEMPTY0 && b < K_UEMPTY0 + kQueue))
             ? 256
             : ((b == K_STG0 || b == K_STG1 || b == K_DSSTG0 || b == K_DSSTG1 ||
                 (b >= K_TRK00 && b <= K_TRK11))
                    ? 128
                    : 1);
}

// The kernel's shared variables, kept at the end of the dynamic shared memory (the kernel
// has no static shared memory, so that the 1024-byte-aligned layout fits without slack).
struct DkdvShared {
  uint64_t bar[K_NUM];
  Queue queue;
  uint32_t tmem_base;
  int abort_flag;
  int epi_count;
  long long ds_mail[2];  // per half: scratch slot of the staged dS^T (-1: no more)
};

// shared memory of the dK/dV kernel: K, V, two Q/dO stages (6 tiles), one 16 KB dS^T box per
// half, per-half staging of LSE and delta, then the shared variables
template <int D>
struct DkdvSmem {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kDS = 6 * kTile;
  static constexpr int kStg = kDS + 2 * 16384;
  static constexpr int kVars = kStg + 2 * 2 * 128 * 4;
  static constexpr size_t bytes() { return (size_t)kVars + sizeof(DkdvShared); }
};
static_assert(DkdvSmem<128>::bytes() <= 232448, "shared memory budget");

template <int D>
__global__ void __launch_bounds__(kThreads, 1) k_bwd_dkdv(const __grid_constant__ BwdParams p) {
  using Lay = DkdvSmem<D>;
  constexpr int kTile = Lay::kTile;
  constexpr int kAtoms = D / 64;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The layout needs a 1024-byte-aligned base (TMA boxes and MMA operands with 128-byte
  // swizzle) and uses the dynamic shared memory to the last byte, with no room to realign:
  // a base that is not aligned is reported through the error word, before any barrier, TMEM
  // or TMA is touched.
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadPlanSize);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem;
  uint8_t* sV = smem + kTile;
  uint8_t* sQ0 = smem + 2 * kTile;  // stage s: Q at 2+2s, dO at 3+2s
  uint8_t* sDS = smem + Lay::kDS;   // half h's dS^T box at sDS + 16384 h
  // per half and buffer: lse2[64] | delta[64]
  float* stg = reinterpret_cast<float*>(smem + Lay::kStg);
  DkdvShared& sv = *reinterpret_cast<DkdvShared*>(smem + Lay::kVars);
  uint64_t* bar = sv.bar;
  Queue& queue = sv.queue;
  uint32_t& tmem_base = sv.tmem_base;
  int& abort_flag = sv.abort_flag;
  int& epi_count = sv.epi_count;
  long long* ds_mail = sv.ds_mail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long n = p.n;
  WaitCtx w{p.wait_ns, p.err, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    epi_count = 0;
    for (int b = 0; b < K_NUM; ++b) mbar_init(&bar[b], dkdv_arrivals(b));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // score regions R0, R1; item g: S^T in R[g & 1], dP^T in R[(g + 1) & 1]
  const uint32_t tR0 = tmem_base;
  const uint32_t tdV = tmem_base + 256;   // dV fp32 [256, 256+D)
  const uint32_t tdK = tmem_base + 384;   // dK fp32 [384, 384+D)

  if (warp < 4) {
  // warpgroup 0: scheduler, producer, MMA issuer, dS^T store, with few registers
  regs_shrink<kRegsCtl>();
  if (warp == kWarpSched) {
    if (lane == 0) schedule<false>(p, queue, &bar[K_UFULL0], &bar[K_UEMPTY0], w);
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.q_map);
      tma_prefetch_desc(&p.k_map);
      tma_prefetch_desc(&p.v_map);
      tma_prefetch_desc(&p.do_map);
    }
    int uc = 0, g = 0, kv_fills = 0, q_fills[2] = {0, 0};
    bool ok = true;
    while (ok) {
      const int slot = uc % kQueue;
      if (!wait_all(&bar[K_UFULL0 + slot], (uc / kQueue) & 1, w)) break;
      const int kh = queue.head[slot];
      if (kh < 0) break;
      const int64_t nk = queue.blk[slot];
      const int L = queue.T[slot], La = queue.La[slot];
      const int64_t c0 = queue.e0[slot], c1 = queue.e1[slot];
      const int items = L * p.group;
      // K and V of the unit once the previous unit's last S^T / dP^T have read the slot
      if (uc >= 1 && !wait_all(&bar[K_KVEMPTY], (uc - 1) & 1, w)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar[K_KVFULL], 2 * kTile);
        for (int a = 0; a < kAtoms; ++a) {
          tma_load_3d(sK + a * 16384, &p.k_map, &bar[K_KVFULL], a * 64, (int)(nk * 128), kh);
          tma_load_3d(sV + a * 16384, &p.v_map, &bar[K_KVFULL], a * 64, (int)(nk * 128), kh);
        }
      }
      ++kv_fills;
      for (int it = 0; it < items; ++it) {
        const int s = g & 1;
        if (g >= 2 && !wait_all(&bar[K_QEMPTY0 + s], ((g >> 1) - 1) & 1, w)) { ok = false; break; }
        const int h = kh * p.group + it / L;
        const int nqb = p.colT_row[list_entry(c0, c1, La, it % L)];
        if (lane == 0) {
          uint8_t* sQ = sQ0 + s * 2 * kTile;
          uint8_t* sDO = sQ + kTile;
          mbar_arrive_expect_tx(&bar[K_QFULL0 + s], 2 * kTile);
          for (int a = 0; a < kAtoms; ++a) {
            tma_load_3d(sQ + a * 16384, &p.q_map, &bar[K_QFULL0 + s], a * 64, nqb * 128, h);
            tma_load_3d(sDO + a * 16384, &p.do_map, &bar[K_QFULL0 + s], a * 64, nqb * 128, h);
          }
        }
        ++q_fills[s];
        ++g;
      }
      ++uc;
    }
    if (lane == 0) {
      if (kv_fills) drain_wait(&bar[K_KVFULL], (kv_fills - 1) & 1, p.wait_ns, p.err);
      for (int s = 0; s < 2; ++s)
        if (q_fills[s]) drain_wait(&bar[K_QFULL0 + s], (q_fills[s] - 1) & 1, p.wait_ns, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdAcc = idesc_bf16(128, D, false, true);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      // S^T(gg) = K Q^T into R[gg & 1]; dP^T(gg) = V dO^T into R[(gg + 1) & 1]
      auto issue_scores = [&](int gg, bool dp) {
        const uint32_t aQ = smem_u32(sQ0 + (gg & 1) * 2 * kTile) + (dp ? kTile : 0);
        const uint32_t aA = dp ? aV : aK;
        const uint32_t d = tR0 + (uint32_t)(((gg + (dp ? 1 : 0)) & 1) * 128);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(d, sdesc_sw128(aA + off, 16, 1024), sdesc_sw128(aQ + off, 16, 1024), kIdS, k > 0);
        }
      };
      // dV += P^T dO, dK += dS^T Q over the 128 q columns, 16 per MMA: the P^T of q columns
      // [16 kk, 16 kk + 16) sits in columns 64 (kk / 4) + 8 (kk % 4) of R[gg & 1], the dS^T 32
      // columns further
      auto issue_acc = [&](int gg, bool first) {
        const uint32_t aQ = smem_u32(sQ0 + (gg & 1) * 2 * kTile), aDO = aQ + kTile;
        const uint32_t r = tR0 + (uint32_t)((gg & 1) * 128);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tdV, r + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_sw128(aDO + kk * 2048, 16384, 1024),
                 kIdAcc, (first && kk == 0) ? 0u : 1u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tdK, r + (kk >> 2) * 64 + 32 + (kk & 3) * 8,
                 sdesc_sw128(aQ + kk * 2048, 16384, 1024), kIdAcc, (first && kk == 0) ? 0u : 1u);
      };
      int uc = 0, j = 0, g = 0, items = 0;
      bool ok = mbar_wait(&bar[K_UFULL0], 0, w) && queue.head[0] >= 0;
      if (ok) {
        items = queue.T[0] * p.group;
        ok = mbar_wait(&bar[K_KVFULL], 0, w) && mbar_wait(&bar[K_QFULL0], 0, w);
      }
      if (ok) {
        tc_fence_after();
        issue_scores(0, false);
        issue_scores(0, true);
        mma_commit(&bar[K_SDP]);
        if (items == 1) mma_commit(&bar[K_KVEMPTY]);  // the unit's last read of K and V
      }
      while (ok) {
        // the item after g: the next of this unit, or the first of the next unit
        bool nxt = true, newu = false;
        int itn = items;
        if (j + 1 == items) {
          const int slot = (uc + 1) % kQueue;
          if (!mbar_wait(&bar[K_UFULL0 + slot], ((uc + 1) / kQueue) & 1, w)) break;
          if (queue.head[slot] < 0) {
            nxt = false;
          } else {
            newu = true;
            itn = queue.T[slot] * p.group;
          }
        }
        // S^T(g + 1) into dP^T(g)'s region once every elementwise thread holds its scores;
        // at a unit's end it waits until item g's accumulations are issued (below), so that
        // the load of the next unit's K and V does not hold back the unit's last dV / dK
        auto next_scores = [&]() -> bool {
          if (!mbar_wait(&bar[K_YFREE], g & 1, w)) return false;
          if (newu && !mbar_wait(&bar[K_KVFULL], (uc + 1) & 1, w)) return false;
          if (!mbar_wait(&bar[K_QFULL0 + ((g + 1) & 1)], ((g + 1) >> 1) & 1, w)) return false;
          tc_fence_after();
          issue_scores(g + 1, false);
          return true;
        };
        if (nxt && !newu && !next_scores()) break;
        // dV / dK of item g once its P^T / dS^T are in TMEM; a unit's first accumulation
        // overwrites dV / dK, so the previous unit's must have been read out
        if (!mbar_wait(&bar[K_PFULL], g & 1, w)) break;
        if (j == 0 && uc >= 1 && !mbar_wait(&bar[K_ACCFREE], (uc - 1) & 1, w)) break;
        tc_fence_after();
        issue_acc(g, j == 0);
        // the unit's last Q/dO stage is handed back by the epilogue, which stages in it
        if (j == items - 1)
          mma_commit(&bar[K_ACCFULL]);
        else
          mma_commit(&bar[K_QEMPTY0 + (g & 1)]);
        if (!nxt) break;
        if (newu && !next_scores()) break;
        // dP^T(g + 1) into S^T(g)'s region, after the accumulations that read it
        issue_scores(g + 1, true);
        mma_commit(&bar[K_SDP]);
        if ((newu && itn == 1) || (!newu && j + 2 == items)) mma_commit(&bar[K_KVEMPTY]);
        ++g;
        if (newu) {
          ++uc;
          j = 0;
          items = itn;
        } else {
          ++j;
        }
      }
      mma_commit(&bar[K_DRAIN]);
      drain_wait(&bar[K_DRAIN], 0, p.wait_ns, p.err);
    }
    __syncwarp();
  } else if (warp == kWarpStore) {
    // ------------------------------------------------------------------ dS^T store
    // lane h writes half h's staged dS^T boxes to the scratch, one TMA store per item, and
    // hands the box back once the TMA has read it, so that no elementwise warp waits for it
    if (lane < 2) {
      const int half = lane;
      for (int g = 0;; ++g) {
        if (!mbar_wait(&bar[K_DSSTG0 + half], (uint32_t)(g & 1), w)) break;
        const long long slot_ds = ds_mail[half];
        if (slot_ds < 0) break;
        tma_store_3d(&p.ds_map, sDS + half * 16384, half * 64, (int)(slot_ds * 128), 0);
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(&bar[K_DSFREE0 + half]);
      }
      // the global writes of every store this lane issued have completed
      bulk_wait_all();
    }
    __syncwarp();
  }
  } else {
    // ------------------------------------------------------------------ elementwise
    // warpgroups 1 and 2, with the registers warpgroup 0 gave up; four warps per half:
    // `half` owns q columns [64 half, 64 half + 64), one kv row a thread
    regs_grow<kRegsElem>();
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int row = quarter * 32 + lane;  // kv row of the tile
    const int hr = row & 63;
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.sl2;
    int uc = 0, g = 0, rc = 0;  // rc: this half's epilogue rounds
    bool ok = true;
    while (ok) {
      const int slot = uc % kQueue;
      if (!wait_all(&bar[K_UFULL0 + slot], (uc / kQueue) & 1, w)) break;
      const int kh = queue.head[slot];
      if (kh < 0) {
        // no more work: each half posts the end of its dS^T stores once its last one is read
        if (row == 0) {
          if (g >= 1) mbar_wait(&bar[K_DSFREE0 + half], (uint32_t)((g - 1) & 1), w);
          ds_mail[half] = -1;
        }
        mbar_arrive(&bar[K_DSSTG0 + half]);
        break;
      }
      const int64_t nk = queue.blk[slot];
      const int L = queue.T[slot], La = queue.La[slot];
      const int64_t c0 = queue.e0[slot], c1 = queue.e1[slot];
      const int items = L * p.group;
      const int64_t tk = nk * 128 + row;
      const int sk = p.tracks[tk], gk = p.tracks[n + tk], zk = p.tracks[2 * n + tk],
                pk = p.tracks[3 * n + tk];
      // every key of the unit's block has an exact visible-query interval: partial tiles test
      // lo_k <= i_q < hi_k instead of the four-track predicate
      const bool ivt = p.iv_block[nk] != 0;
      const int klo = p.kiv[tk], khi = p.kiv[n + tk];
      for (int it = 0; it < items; ++it, ++g) {
        const int h = kh * p.group + it / L;
        const int64_t e = list_entry(c0, c1, La, it % L);
        const int64_t qrow = (int64_t)p.colT_row[e] * 128 + half * 64 + hr;
        const bool partial = p.colT_tag[e] == MARBLE_TILE_PARTIAL;
        // the tile's dS^T scratch slot (row 0 of the half), looked up now so that the loads
        // are done by the time the box is full: its row-list entry (whole rows), or the step's
        // tiles in row-list order; q heads innermost
        long long slot_ds = 0;
        if (row == 0) {
          const int64_t nq = p.colT_row[e];
          if (p.whole) {
            slot_ds = p.ds_base[nq / p.bps] +
                      (p.step_ptr[nq * p.P + nk / p.bps] + p.colT_j[e]) * p.hq + h;
          } else {
            const int opt = p.kv_shard >= 0 ? p.kv_shard : p.P;
            int64_t jj = p.colT_j[e];
            if (opt == p.P) jj += p.step_ptr[nq * p.P + nk / p.bps] - p.step_ptr[nq * p.P];
            const long long base = p.ring_len > 0 ? p.ds_base[nq / p.bps] : p.ds_slot0;
            slot_ds = base + ((int64_t)p.step_off[nq * (p.P + 1) + opt] + jj) * p.hq + h;
          }
        }
        // stage this half's per-query LSE (base 2) and delta (threads of rows [0, 64))
        const int b = g & 1;
        float* lse2s = stg + (half * 2 + b) * 128;
        float* dls = lse2s + 64;
        if ((row >> 6) == 0) {
          const float l2 = p.lse[(int64_t)h * n + qrow] * kLog2e;
          lse2s[hr] = (l2 == -INFINITY) ? INFINITY : l2;
          dls[hr] = p.delta[(int64_t)h * n + qrow];
        }
        mbar_arrive(&bar[K_TRK00 + half * 2 + b]);
        uint32_t lm[2] = {~0u, ~0u};
        if (partial && ivt) {
          // lo_k <= i_q < hi_k, i_q the query's index in the given token order.  The plan moves
          // whole 128-token blocks, so the half's 64 queries have the consecutive indices
          // i0, i0 + 1, ..., and the legal ones are the columns [lo_k - i0, hi_k - i0) cut to
          // [0, 64): one range of bits
          const int64_t i0 = (int64_t)p.qidx[(int64_t)p.colT_row[e] * 128] + half * 64;
          const int64_t a = min(max((int64_t)klo - i0, (int64_t)0), (int64_t)64);
          const int64_t c = min(max((int64_t)khi - i0, (int64_t)0), (int64_t)64);
          const uint64_t below_c = c >= 64 ? ~0ull : ((1ull << c) - 1ull);
          const uint64_t below_a = a >= 64 ? ~0ull : ((1ull << a) - 1ull);
          const uint64_t bits = a < c ? (below_c & ~below_a) : 0ull;
          lm[0] = (uint32_t)bits;
          lm[1] = (uint32_t)(bits >> 32);
        } else if (partial) {
          // the half's 64 queries' tracks, read straight from global memory (the same
          // addresses for every lane: broadcast loads), four queries per load
          const int32_t* qt = p.tracks + (int64_t)p.colT_row[e] * 128 + half * 64;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t bits = 0;
#pragma unroll
            for (int t2 = 0; t2 < 32; t2 += 4) {
              const int q = cc * 32 + t2;
              const int4 s4 = __ldg(reinterpret_cast<const int4*>(qt + q));
              const int4 g4 = __ldg(reinterpret_cast<const int4*>(qt + n + q));
              const int4 z4 = __ldg(reinterpret_cast<const int4*>(qt + 2 * n + q));
              const int4 p4 = __ldg(reinterpret_cast<const int4*>(qt + 3 * n + q));
              bits |= (mask_legal(s4.x, g4.x, z4.x, p4.x, sk, gk, zk, pk, p.W) ? 1u : 0u) << t2;
              bits |= (mask_legal(s4.y, g4.y, z4.y, p4.y, sk, gk, zk, pk, p.W) ? 1u : 0u) << (t2 + 1);
              bits |= (mask_legal(s4.z, g4.z, z4.z, p4.z, sk, gk, zk, pk, p.W) ? 1u : 0u) << (t2 + 2);
              bits |= (mask_legal(s4.w, g4.w, z4.w, p4.w, sk, gk, zk, pk, p.W) ? 1u : 0u) << (t2 + 3);
            }
            lm[cc] = bits;
          }
        }
        // a partial tile on which every row of this warp keeps all 64 of its columns needs no
        // mask
        const bool masked = partial && __any_sync(0xffffffffu, (lm[0] & lm[1]) != ~0u);
        if (!wait_all(&bar[K_TRK00 + half * 2 + b], (g >> 1) & 1, w)) { ok = false; break; }
        if (!wait_all(&bar[K_SDP], g & 1, w)) { ok = false; break; }
        // the scores of the unit's first item are issued: every role has read the queue entry
        if (it == 0) mbar_arrive(&bar[K_UEMPTY0 + slot]);
        tc_fence_after();
        const uint32_t rS = tR0 + (uint32_t)((g & 1) * 128);        // S^T(g), then P^T / dS^T
        const uint32_t rP = tR0 + (uint32_t)(((g + 1) & 1) * 128);  // dP^T(g)
        uint32_t vs[2][32], vp[2][32];
        tmem_ld32(rS + lb + half * 64, vs[0]);
        tmem_ld32(rS + lb + half * 64 + 32, vs[1]);
        tmem_ld32(rP + lb + half * 64, vp[0]);
        tmem_ld32(rP + lb + half * 64 + 32, vp[1]);
        tmem_ld_wait();
        // this thread holds its scores: once every thread has, dP^T(g)'s region may take
        // S^T(g + 1); the columns of S^T(g)'s region this half read take its P^T / dS^T
        tc_fence_before();
        mbar_arrive(&bar[K_YFREE]);
        // the half's dS^T box takes this item's tile once its previous store has read it (long
        // done, normally): each 32-column chunk goes to the box as soon as it is packed
        if (g >= 1 && !wait_all(&bar[K_DSFREE0 + half], (uint32_t)((g - 1) & 1), w)) { ok = false; break; }
        fence_proxy_async_smem();
        uint8_t* box_row = sDS + half * 16384 + row * 128;
        // P^T = exp2(s * scale * log2 e - lse2[q]), dS^T = P^T (dP^T - delta[q]); the per-query
        // LSE and delta are read four at a time.  Two copies of the loop, chosen per warp: with
        // the mask's select, and without it (full tiles, and partial ones whose rows in this
        // warp keep every column)
        auto elementwise = [&](auto with_mask) {
          constexpr bool kMasked = decltype(with_mask)::value;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t pk16[16], dk16[16];
#pragma unroll
            for (int t = 0; t < 32; t += 4) {
              const int q0 = cc * 32 + t;
              const float4 l4 = *reinterpret_cast<const float4*>(lse2s + q0);
              const float4 d4 = *reinterpret_cast<const float4*>(dls + q0);
              const float lq[4] = {l4.x, l4.y, l4.z, l4.w}, dq4[4] = {d4.x, d4.y, d4.z, d4.w};
              float pv[4], dv4[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float ex = fast_exp2(fmaf(__uint_as_float(vs[cc][t + u]), sl2, -lq[u]));
                pv[u] = (kMasked && !((lm[cc] >> (t + u)) & 1u)) ? 0.f : ex;
                dv4[u] = pv[u] * (__uint_as_float(vp[cc][t + u]) - dq4[u]);
              }
              pk16[t >> 1] = pack_bf16(pv[0], pv[1]);
              pk16[(t >> 1) + 1] = pack_bf16(pv[2], pv[3]);
              dk16[t >> 1] = pack_bf16(dv4[0], dv4[1]);
              dk16[(t >> 1) + 1] = pack_bf16(dv4[2], dv4[3]);
            }
            // q columns [32 cc, 32 cc + 32) of this half: 16-byte chunks 4 cc .. 4 cc + 3 of the
            // row, 128-byte swizzled as the TMA store reads them
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(box_row + (((4 * cc + c) ^ (row & 7)) << 4)) =
                  make_uint4(dk16[4 * c], dk16[4 * c + 1], dk16[4 * c + 2], dk16[4 * c + 3]);
            // q column pair c of this half -> P^T column 64 half + c, dS^T column 64 half + 32 + c
            tmem_st16(rS + lb + half * 64 + cc * 16, pk16);
            tmem_st16(rS + lb + half * 64 + 32 + cc * 16, dk16);
          }
        };
        if (masked)
          elementwise(std::true_type{});
        else
          elementwise(std::false_type{});
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[K_PFULL]);
        // ---- this half's bf16 dS^T (its 64 q columns, staged in its box above) to the tile's
        // scratch slot for the dQ GEMM
        if (row == 0) ds_mail[half] = slot_ds;
        fence_proxy_async_smem();
        mbar_arrive(&bar[K_DSSTG0 + half]);
      }
      if (!ok) break;
      // ---- the unit's dV and dK (dv_acc += dV, dk_acc += scale * dK): round 0 stages this
      // half's dV columns, round 1 its dK columns, as 128 x 32 fp32 boxes in the Q/dO stage of
      // the unit's last item, each added by a TMA reduce-add.  Every thread waits on each
      // unit's phase in order, so no wait runs two phases ahead.
      if (!wait_all(&bar[K_ACCFULL], uc & 1, w)) break;
      tc_fence_after();
      constexpr int kB = D / 64;  // boxes per half and round
      uint8_t* boxes = sQ0 + ((g - 1) & 1) * 2 * kTile + half * kB * 16384;
#pragma unroll 1
      for (int r = 0; r < 2; ++r, ++rc) {
        const uint32_t tacc = r == 0 ? tdV : tdK;
        const float sc = r == 0 ? 1.f : p.scale;
        uint32_t x[kB][32];
#pragma unroll
        for (int cb = 0; cb < kB; ++cb) tmem_ld32(tacc + lb + (half * kB + cb) * 32, x[cb]);
        tmem_ld_wait();
        if (r == 1) {
          tc_fence_before();
          mbar_arrive(&bar[K_ACCFREE]);  // the next unit's dV / dK MMAs may overwrite TMEM
        }
        // the boxes are free once this half's previous round has been read by its TMA
        if (rc > 0 && !wait_all(&bar[K_STGR0 + half], (rc - 1) & 1, w)) { ok = false; break; }
        fence_proxy_async_smem();
#pragma unroll
        for (int cb = 0; cb < kB; ++cb) {
          float v[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) v[t] = sc * __uint_as_float(x[cb][t]);
          stage_row32(boxes + cb * 16384, row, v);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar[K_STG0 + half]);
        if (row == 0) {
          if (mbar_wait(&bar[K_STG0 + half], rc & 1, w)) {
#pragma unroll
            for (int cb = 0; cb < kB; ++cb)
              tma_reduce_add_3d(r == 0 ? (const void*)&p.dv_map : (const void*)&p.dk_map,
                                boxes + cb * 16384, (half * kB + cb) * 32, (int)(nk * 128), kh);
            bulk_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&bar[K_STGR0 + half]);
          // the second half to finish hands the Q/dO stage back to the producer
          if (r == 1 && atomicAdd(&epi_count, 1) == 1) {
            epi_count = 0;
            mbar_arrive(&bar[K_QEMPTY0 + ((g - 1) & 1)]);
          }
        }
      }
      ++uc;
    }
    // the global writes of every TMA reduce this thread issued have completed
    if (row == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
  if (threadIdx.x == 0) release_tickets(p);
}

template <int D>
size_t dkdv_smem() {
  return DkdvSmem<D>::bytes();
}

// everything of a backward call but the step, its work list and the scratch: encoded once
template <int D>
marble_status_t prepare_bwd(const marble_plan_t* pl, const marble_qkv_t* qkv, const void* d_o,
                            const float* lse, const float* delta, float* dq, float* dk, float* dv,
                            BwdParams* out) {
  BwdParams& prm = *out;
  memset(&prm, 0, sizeof(prm));
  const int64_t n = pl->n;
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_rows_map(&prm.q_map, qkv->q, bf, 2, n, qkv->hq, D, 64, 128, sw) ||
      !make_rows_map(&prm.k_map, qkv->k, bf, 2, n, qkv->hkv, D, 64, 128, sw) ||
      !make_rows_map(&prm.v_map, qkv->v, bf, 2, n, qkv->hkv, D, 64, 128, sw) ||
      !make_rows_map(&prm.do_map, d_o, bf, 2, n, qkv->hq, D, 64, 128, sw) ||
      !make_rows_map(&prm.dq_map, dq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, n, qkv->hq, D, 32, 128,
                     sw) ||
      !make_rows_map(&prm.dk_map, dk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, n, qkv->hkv, D, 32, 128,
                     sw) ||
      !make_rows_map(&prm.dv_map, dv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, n, qkv->hkv, D, 32, 128,
                     sw))
    return fail(MARBLE_ERR_CUDA, "cuTensorMapEncodeTiled failed for Q/K/V/dO/accumulators");
  prm.step_ptr = pl->step_ptr;
  prm.step_col = pl->step_col;
  prm.step_tag = pl->step_tag;
  prm.colT_ptr = pl->colT_ptr;
  prm.colT_row = pl->colT_row;
  prm.colT_tag = pl->colT_tag;
  prm.needed_ptr = pl->needed_ptr;
  prm.needed = pl->needed;
  prm.tracks = pl->tracks;
  prm.kiv = pl->kiv;
  prm.qidx = pl->perm;
  prm.iv_block = pl->iv_block;
  prm.lse = lse;
  prm.delta = delta;
  prm.dq = dq;
  prm.dk = dk;
  prm.dv = dv;
  prm.err = pl->err;
  prm.wait_ns = wait_limit_ns();
  prm.n = n;
  prm.P = pl->P;
  prm.bps = (int)pl->bps;
  prm.hq = qkv->hq;
  prm.hkv = qkv->hkv;
  prm.group = qkv->hq / qkv->hkv;
  prm.W = pl->W;
  prm.scale = qkv->scale > 0.f ? qkv->scale : 1.0f / sqrtf((float)D);
  prm.sl2 = prm.scale * kLog2e;
  prm.step_off = pl->step_off;
  prm.colT_j = pl->colT_j;
  if (once_per_device(D == 128 ? 3 : 4)) {
    cudaError_t e = cudaFuncSetAttribute(k_bwd_dq<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)DqSmem<D>::bytes());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_bwd_dkdv<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)dkdv_smem<D>());
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd)");
  }
  {
    // the dK/dV kernel's warpgroups trade registers among themselves: the block must be
    // launched with at least the registers the two budgets add up to, or the growing
    // warpgroups would wait for registers that never come (checked on every call)
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, k_bwd_dkdv<D>);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(k_bwd_dkdv)");
    if ((long long)fa.numRegs * kThreads < 128LL * kRegsCtl + 256LL * kRegsElem)
      return fail(MARBLE_ERR_UNSUPPORTED, "dK/dV kernel built with " + std::to_string(fa.numRegs) +
                                              " registers per thread, fewer than its split needs");
  }
  return MARBLE_OK;
}

// The plan-owned scratch for bf16 dS^T tiles: at least `need` bytes, and its tensor map as
// [slots * 128 rows] x 128 columns with 64 x 128 boxes.
marble_status_t ds_scratch(const marble_plan_t* pl, size_t slots, cudaStream_t s, BwdParams* prm) {
  std::lock_guard<std::mutex> lock(pl->scratch_mu);
  const size_t need = slots * 32768;
  if (need > pl->ds_scratch_bytes) {
    // earlier calls joined their side streams back into their stream, and calls on one plan
    // are ordered: freeing in the order of `s` is safe
    if (pl->ds_scratch) {
      dev_free(pl->ds_scratch, s);
      pl->ds_scratch = nullptr;
      pl->ds_scratch_bytes = 0;
    }
    size_t got = need;
    void* q = scratch_take(need, s, &got);
    if (!q && dev_alloc(&q, need, s) != cudaSuccess) {
      (void)cudaGetLastError();
      return fail(MARBLE_ERR_OOM, "allocation of the backward dS scratch failed (" +
                                      std::to_string(need) + " bytes)");
    }
    pl->ds_scratch = q;
    pl->ds_scratch_bytes = got;
  }
  if (slots > 0 && !make_rows_map(&prm->ds_map, pl->ds_scratch, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                  2, (int64_t)slots * 128, 1, 128, 64, 128,
                                  CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(MARBLE_ERR_CUDA, "cuTensorMapEncodeTiled failed for the dS scratch");
  return MARBLE_OK;
}

int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

// dQ GEMM of step (q shard r, kv shard or every needed block), reading dS^T slots from slot0
template <int D>
void launch_dq(const marble_plan_t* pl, const BwdParams& prm, int r, int j, long long slot0,
               int hq, int sms, cudaStream_t s) {
  const int P = pl->P;
  BwdParams pq = prm;
  pq.q_shard = r;
  pq.kv_shard = j;
  pq.ds_slot0 = slot0;
  pq.ring_len = 0;
  const int64_t seg = (int64_t)r * (P + 1) + (j >= 0 ? j : P);
  pq.order = pl->fwd_order + seg * pl->bps;
  pq.nwork = pl->h_fwd_nwork[seg] * hq;
  if (pq.nwork > 0) {
    pq.sched = sched_slot(pl);
    const int span = timing_begin(s);
    k_bwd_dq<D><<<(unsigned)(pq.nwork < sms ? pq.nwork : sms), kGThreads, DqSmem<D>::bytes(), s>>>(pq);
    timing_end(span, s, kTimeDq, 1);
  }
}

// The cap on the dS^T scratch: kDsScratchCap, or less when MARBLE_DS_SCRATCH_CAP_MB says so
// (tests use it to reach the paths that larger packs take).
size_t scratch_cap() {
  size_t cap = kDsScratchCap;
  if (const char* env = std::getenv("MARBLE_DS_SCRATCH_CAP_MB")) {
    const unsigned long long mb = std::strtoull(env, nullptr, 10);
    if (mb > 0 && (mb << 20) < cap) cap = (size_t)(mb << 20);
  }
  return cap;
}

// the whole backward's dQ GEMM over whole rows: every (q block, q head) of the pack with tiles
// (q_shard < 0), or those of one q shard; at most `ctas` CTAs
template <int D>
void launch_dq_whole(const marble_plan_t* pl, const BwdParams& prm, int q_shard, int hq,
                     int ctas, cudaStream_t s) {
  BwdParams pq = prm;
  pq.whole = 1;
  pq.kv_shard = -1;
  pq.ring_len = 0;
  if (q_shard < 0) {
    pq.whole = 2;
    pq.q_shard = 0;
    pq.order = pl->fwd_order_all;
    pq.nwork = pl->h_fwd_nwork_all * hq;
  } else {
    const int64_t seg = (int64_t)q_shard * (pl->P + 1) + pl->P;
    pq.q_shard = q_shard;
    pq.order = pl->fwd_order + seg * pl->bps;
    pq.nwork = pl->h_fwd_nwork[seg] * hq;
  }
  if (pq.nwork > 0) {
    pq.sched = sched_slot(pl);
    const int span = timing_begin(s);
    k_bwd_dq<D><<<(unsigned)(pq.nwork < ctas ? pq.nwork : ctas), kGThreads, DqSmem<D>::bytes(), s>>>(pq);
    timing_end(span, s, kTimeDq, 1);
  }
}

// The whole backward keeps every tile's dS^T (nnz x hq slots of 32 KB) and runs the dQ GEMM
// once, after every dK/dV launch: dQ of a q block then accumulates its whole row in TMEM and
// is added to dq_acc once, instead of once per ring step.  It is taken when the scratch fits
// the cap.
size_t whole_slots(const marble_plan_t* pl, int hq) {
  const size_t slots = (size_t)pl->nnz * (size_t)hq;
  return slots * 32768 <= scratch_cap() ? slots : 0;
}

// Whole-row dQ for a full ring list: the dK/dV launch of every step (kv shard j on side
// stream j mod kDkdvStreams, so that the launches adding into one kv shard's dK/dV rows stay in
// order) and dQ GEMMs over whole rows (stream s, after the side streams' launches so far).  The
// dS^T tiles of q shard r sit at ds_base[r] + e * hq + head (e the row-list entry):
//   nbuf >= P  every q shard has its own place in one array (ds_base = 0), and one dQ GEMM
//              over every q block follows all dK/dV launches;
//   otherwise  the list holds each q shard's steps in one run, the k-th q shard of the list
//              takes buffer k mod nbuf of buf_slots slots, its dQ GEMM follows its last step
//              (overlapping the dK/dV launches of the steps after it), and its first dK/dV
//              launch waits until the dQ GEMM of the q shard nbuf runs earlier has read that
//              buffer.
template <int D>
marble_status_t launch_whole(const marble_plan_t* pl, const marble_qkv_t* qkv, BwdParams prm,
                             int n_steps, const int* q_shards, const int* kv_shards, int nbuf,
                             int64_t buf_slots, cudaStream_t s) {
  const int smem_k = (int)dkdv_smem<D>();
  const int sms = sm_count();
  const int P = pl->P;
  const int64_t hq = qkv->hq;
  const bool all = nbuf >= P;
  marble_status_t rc = ds_scratch(pl, all ? whole_slots(pl, (int)hq) : (size_t)(nbuf * buf_slots),
                                  s, &prm);
  if (rc != MARBLE_OK) return rc;
  prm.whole = 1;
  prm.ds_slot0 = 0;
  // first row-list entry of every q shard
  std::vector<int64_t> first(P + 1, 0);
  for (int r = 0; r < P; ++r) first[r + 1] = first[r] + pl->h_step_tiles[(size_t)r * (P + 1) + P];
  cudaStream_t sk[kDkdvStreams];
  int nsk = 0;
  for (int k = 0; k < kDkdvStreams; ++k) {
    cudaStream_t x = side_stream(k);
    if (!x) break;
    cudaError_t e = stream_fork(s, x);
    if (e != cudaSuccess) return cuda_fail(e, "fork of the backward streams");
    sk[nsk++] = x;
  }
  if (nsk == 0) sk[nsk++] = s;
  const bool overlap = sk[0] != s;
  // with side streams, a dK/dV launch takes at most half the SMs: launches of different kv
  // shards then share the GPU instead of one waiting for the other's tail
  const int cap = overlap ? (sms + 1) / 2 : sms;
  std::vector<int> issued(P, 0);
  std::vector<cudaEvent_t> ev_buf(all ? 0 : nbuf, nullptr);
  int shards_begun = 0;
  cudaError_t err = cudaSuccess;
  for (int i = 0; i < n_steps && err == cudaSuccess; ++i) {
    const int r = q_shards[i];
    if (issued[r] == 0 && !all) {
      // the q shard's buffer: free once the dQ GEMM that last read it is done
      const int k = shards_begun % nbuf;
      prm.ds_base[r] = (long long)k * buf_slots - first[r] * hq;
      if (ev_buf[k] && overlap)
        for (int x = 0; x < nsk && err == cudaSuccess; ++x)
          err = cudaStreamWaitEvent(sk[x], ev_buf[k], 0);
      ++shards_begun;
    }
    BwdParams pk = prm;
    pk.q_shard = r;
    pk.kv_shard = kv_shards[i];
    const int64_t seg = (int64_t)pk.kv_shard * (P + 1) + r;
    pk.order = pl->bwd_order + seg * pl->bps;
    pk.nwork = pl->h_bwd_nwork[seg] * qkv->hkv;
    if (pk.nwork > 0 && err == cudaSuccess) {
      const cudaStream_t sks = sk[pk.kv_shard % nsk];
      pk.sched = sched_slot(pl);
      const int span = timing_begin(sks);
      k_bwd_dkdv<D><<<(unsigned)(pk.nwork < cap ? pk.nwork : cap), kThreads, smem_k, sks>>>(pk);
      timing_end(span, sks, kTimeDkdv, 1);
    }
    if (++issued[r] == P && !all && err == cudaSuccess) {
      for (int k = 0; k < nsk && err == cudaSuccess; ++k)
        if (sk[k] != s) err = stream_fork(sk[k], s);
      // held to half the SMs while dK/dV launches follow (enough for the memory bandwidth it
      // is bound by); the last one has the GPU to itself
      const int ctas = (overlap && i + 1 < n_steps) ? std::max(1, sms / 2) : sms;
      if (err == cudaSuccess) launch_dq_whole<D>(pl, prm, r, (int)hq, ctas, s);
      if (err == cudaSuccess) {
        const int k = (shards_begun - 1) % nbuf;
        if (ev_buf[k]) cudaEventDestroy(ev_buf[k]);
        ev_buf[k] = nullptr;
        err = cudaEventCreateWithFlags(&ev_buf[k], cudaEventDisableTiming);
        if (err == cudaSuccess) err = cudaEventRecord(ev_buf[k], s);
      }
    }
  }
  for (int k = 0; k < nsk && err == cudaSuccess; ++k)
    if (sk[k] != s) err = stream_fork(sk[k], s);
  for (cudaEvent_t ev : ev_buf)
    if (ev) cudaEventDestroy(ev);
  if (err != cudaSuccess) return cuda_fail(err, "ordering of the backward streams");
  // every tile of the pack at once: one dQ GEMM over every q block's whole row at the end
  // (one launch balances the rows of all q shards; q shard by q shard in the gaps between
  // dK/dV launches measured slower)
  if (all) launch_dq_whole<D>(pl, prm, -1, (int)hq, sms, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch of the backward kernels");
  return MARBLE_OK;
}

// How a full ring list can run with whole-row dQ (launch_whole): 0 if it cannot; else the
// number of q-shard buffers (P: the whole pack at once) and, below P, each buffer's slots.
// Below P the list must hold each q shard's steps in one run.  A dQ GEMM unit is a q block's
// whole row: when the longest row is more than half a CTA's share of its launch, that one
// unit would set the launch's length, and the per-step GEMMs (rows cut at kv shards) are
// taken instead.
// no q block's whole row longer than half a CTA's share of `tiles` rows' worth of units
// (MARBLE_WHOLE_ROWS=always skips the test; tests use it to reach these paths on small packs)
bool rows_balance(int64_t longest, int64_t tiles, int hq) {
  const char* env = std::getenv("MARBLE_WHOLE_ROWS");
  if (env && std::strcmp(env, "always") == 0) return true;
  return 2 * longest * sm_count() <= tiles * (int64_t)hq;
}

// every tile of the pack at once, with one dQ GEMM over all q blocks
bool whole_all(const marble_plan_t* pl, int hq) {
  if (whole_slots(pl, hq) == 0) return false;
  int64_t longest = 0;
  for (int r = 0; r < pl->P; ++r)
    longest = std::max(longest, pl->h_step_max[(size_t)r * (pl->P + 1) + pl->P]);
  return rows_balance(longest, pl->nnz, hq);
}

int whole_plan(const marble_plan_t* pl, int hq, int n_steps, const int* q_shards,
               const int* kv_shards, int64_t* buf_slots) {
  const int P = pl->P;
  if (n_steps != P * P) return 0;
  std::vector<uint8_t> seen((size_t)P * P, 0), begun(P, 0);
  bool runs = true;
  for (int i = 0; i < n_steps; ++i) {
    const int r = q_shards[i], j = kv_shards[i];
    if (j < 0 || seen[(size_t)r * P + j]) return 0;
    seen[(size_t)r * P + j] = 1;
    if (i % P == 0) {
      if (begun[r]) runs = false;
      begun[r] = 1;
    } else if (r != q_shards[i - 1]) {
      runs = false;
    }
  }
  if (whole_all(pl, hq)) return P;
  if (!runs) return 0;
  int64_t mx = 0;
  for (int r = 0; r < P; ++r) {
    const int64_t tiles = pl->h_step_tiles[(size_t)r * (P + 1) + P];
    if (!rows_balance(pl->h_step_max[(size_t)r * (P + 1) + P], tiles, hq)) return 0;
    mx = std::max(mx, tiles);
  }
  *buf_slots = mx * hq;
  const int64_t nbuf = (int64_t)(scratch_cap() / ((size_t)std::max<int64_t>(*buf_slots, 1) * 32768));
  return nbuf >= 2 ? (int)std::min<int64_t>(nbuf, P - 1) : 0;
}

template <int D>
marble_status_t launch_steps(const marble_plan_t* pl, const marble_qkv_t* qkv, const void* d_o,
                             const float* lse, const float* delta, int n_steps,
                             const int* q_shards, const int* kv_shards, float* dq, float* dk,
                             float* dv, cudaStream_t s) {
  BwdParams prm;
  marble_status_t rc = prepare_bwd<D>(pl, qkv, d_o, lse, delta, dq, dk, dv, &prm);
  if (rc != MARBLE_OK) return rc;
  const int smem_k = (int)dkdv_smem<D>();
  const int sms = sm_count();
  const int P = pl->P;
  // a list that holds every (q shard, kv shard) step of the ring exactly once runs with
  // whole-row dQ GEMMs when its scratch allows (launch_whole)
  {
    int64_t buf_slots = 0;
    const int nbuf = whole_plan(pl, qkv->hq, n_steps, q_shards, kv_shards, &buf_slots);
    if (nbuf > 0)
      return launch_whole<D>(pl, qkv, prm, n_steps, q_shards, kv_shards, nbuf, buf_slots, s);
  }
  // scratch for the bf16 dS^T tiles of kDsBufs steps: the dQ GEMM of step i reads buffer
  // i mod kDsBufs while the dK/dV kernels of the next steps write the others
  int64_t max_tiles = 0;  // the largest step of this call
  for (int i = 0; i < n_steps; ++i) {
    const int64_t t =
        pl->h_step_tiles[(size_t)q_shards[i] * (P + 1) + (kv_shards[i] >= 0 ? kv_shards[i] : P)];
    max_tiles = t > max_tiles ? t : max_tiles;
  }
  const int64_t buf_slots = max_tiles * qkv->hq;
  const int nbuf = (int)std::max<int64_t>(
      2, std::min<int64_t>(kDsBufs, (int64_t)(scratch_cap() / ((size_t)std::max<int64_t>(
                                                                 buf_slots, 1) * 32768))));
  rc = ds_scratch(pl, (size_t)(nbuf * buf_slots), s, &prm);
  if (rc != MARBLE_OK) return rc;
  // Step i: the dK/dV kernel (a side stream) writes the step's dS^T tiles into buffer
  // i mod nbuf of the scratch, then the dQ GEMM (stream s) reads them; dK/dV of step
  // i + nbuf waits until the dQ GEMM of step i has finished with that buffer.  dK/dV of kv
  // shard j runs on side stream j mod kDkdvStreams, so that the launches of one kv shard
  // (which add into the same dK/dV rows) stay in order while consecutive steps (different kv
  // shards) overlap one another and the dQ GEMMs.  With every needed block at once, all
  // dK/dV launches share one side stream.
  const bool needed_mode = n_steps > 0 && kv_shards[0] < 0;
  cudaStream_t sk[kDkdvStreams];
  int nsk = 0;
  for (int k = 0; k < (needed_mode ? 1 : kDkdvStreams); ++k) {
    cudaStream_t x = side_stream(k);
    if (!x) break;
    cudaError_t e = stream_fork(s, x);
    if (e != cudaSuccess) return cuda_fail(e, "fork of the backward streams");
    sk[nsk++] = x;
  }
  if (nsk == 0) sk[nsk++] = s;
  const cudaStream_t s2 = sk[0];
  std::vector<cudaEvent_t> ev_k(n_steps, nullptr), ev_q(n_steps, nullptr);
  auto make_event = [](cudaEvent_t* ev) {
    return cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  };
  cudaError_t err = cudaSuccess;
  for (int i = 0; i < n_steps && err == cudaSuccess; ++i) {
    prm.q_shard = q_shards[i];
    prm.kv_shard = kv_shards[i];
    prm.ds_slot0 = (long long)(i % nbuf) * buf_slots;
    // dK/dV: the kv blocks of the kv shard listed for the q shard (longest list first), or
    // the q shard's needed kv blocks
    {
      BwdParams pk = prm;
      if (pk.kv_shard >= 0) {
        const int64_t seg = (int64_t)pk.kv_shard * (P + 1) + pk.q_shard;
        pk.order = pl->bwd_order + seg * pl->bps;
        pk.nwork = pl->h_bwd_nwork[seg] * qkv->hkv;
      } else {
        pk.order = nullptr;
        pk.nwork = (int)(pl->h_needed_ptr[pk.q_shard + 1] - pl->h_needed_ptr[pk.q_shard]) *
                   qkv->hkv;
      }
      const cudaStream_t sks = sk[pk.kv_shard >= 0 ? pk.kv_shard % nsk : 0];
      if (sks != s && i >= nbuf) err = cudaStreamWaitEvent(sks, ev_q[i - nbuf], 0);
      if (pk.nwork > 0 && err == cudaSuccess) {
        pk.sched = sched_slot(pl);
        const int span = timing_begin(sks);
        // with several side streams, at most half the SMs (as in launch_whole)
        const int cap = (sks != s && nsk > 1) ? (sms + 1) / 2 : sms;
        k_bwd_dkdv<D><<<(unsigned)(pk.nwork < cap ? pk.nwork : cap), kThreads, smem_k, sks>>>(pk);
        timing_end(span, sks, kTimeDkdv, 1);
      }
      if (sks != s && err == cudaSuccess) {
        err = make_event(&ev_k[i]);
        if (err == cudaSuccess) err = cudaEventRecord(ev_k[i], sks);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(s, ev_k[i], 0);
      }
    }
    // dQ GEMM: the q blocks of the q shard with tiles in this step, longest list first
    if (err == cudaSuccess) {
      launch_dq<D>(pl, prm, prm.q_shard, prm.kv_shard, prm.ds_slot0, qkv->hq, sms, s);
      if (s2 != s) {
        err = make_event(&ev_q[i]);
        if (err == cudaSuccess) err = cudaEventRecord(ev_q[i], s);
      }
    }
  }
  for (int k = 0; k < nsk && err == cudaSuccess; ++k)
    if (sk[k] != s) err = stream_fork(sk[k], s);
  for (cudaEvent_t ev : ev_k)
    if (ev) cudaEventDestroy(ev);
  for (cudaEvent_t ev : ev_q)
    if (ev) cudaEventDestroy(ev);
  if (err != cudaSuccess) return cuda_fail(err, "ordering of the backward streams");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch of the backward kernels");
  return MARBLE_OK;
}

// The fused ring: for every kv shard j, one dK/dV launch over the ring steps of a range
// (q shards j, j + 1, ... in ring order; the whole ring unless its dS^T tiles exceed the
// scratch cap), keeping the kv blocks' dK/dV in TMEM across all of them and adding them to
// dk_acc / dv_acc once per range; then the range's dQ GEMMs, one per step (q shard, j), on
// the caller's stream.  Ranges of one kv shard run in order on one side stream.
template <int D>
marble_status_t launch_fused(const marble_plan_t* pl, const marble_qkv_t* qkv, const void* d_o,
                             const float* lse, const float* delta, float* dq, float* dk,
                             float* dv, cudaStream_t s) {
  BwdParams prm;
  marble_status_t rc = prepare_bwd<D>(pl, qkv, d_o, lse, delta, dq, dk, dv, &prm);
  if (rc != MARBLE_OK) return rc;
  const int smem_k = (int)dkdv_smem<D>();
  const int sms = sm_count();
  const int P = pl->P;
  const int64_t hq = qkv->hq;
  if (whole_all(pl, (int)hq)) {
    // the whole backward: one dK/dV launch per kv shard over its whole ring, storing every
    // dS^T tile by its row-list entry, then one dQ GEMM over every q block
    rc = ds_scratch(pl, whole_slots(pl, (int)hq), s, &prm);
    if (rc != MARBLE_OK) return rc;
    prm.whole = 1;
    cudaStream_t sk[kDkdvStreams];
    int nsk = 0;
    for (int k = 0; k < kDkdvStreams; ++k) {
      cudaStream_t x = side_stream(k);
      if (!x) break;
      cudaError_t e = stream_fork(s, x);
      if (e != cudaSuccess) return cuda_fail(e, "fork of the backward streams");
      sk[nsk++] = x;
    }
    if (nsk == 0) sk[nsk++] = s;
    for (int j = 0; j < P; ++j) {
      BwdParams pk = prm;
      pk.kv_shard = j;
      pk.q_shard = 0;
      pk.ring_s0 = 0;
      pk.ring_len = P;
      const int64_t seg = (int64_t)j * (P + 1) + P;
      pk.order = pl->bwd_order + seg * pl->bps;
      pk.nwork = pl->h_bwd_nwork[seg] * qkv->hkv;
      if (pk.nwork > 0) {
        const cudaStream_t sks = sk[j % nsk];
        pk.sched = sched_slot(pl);
        const int span = timing_begin(sks);
        // with several side streams, at most half the SMs (as in launch_whole; measured a
        // little faster here, slower in the ranges below, whose dQ GEMMs interleave)
        const int cap = nsk > 1 ? (sms + 1) / 2 : sms;
        k_bwd_dkdv<D><<<(unsigned)(pk.nwork < cap ? pk.nwork : cap), kThreads, smem_k, sks>>>(pk);
        timing_end(span, sks, kTimeDkdv, 1);
      }
    }
    cudaError_t err = cudaSuccess;
    for (int k = 0; k < nsk && err == cudaSuccess; ++k)
      if (sk[k] != s) err = stream_fork(sk[k], s);
    if (err != cudaSuccess) return cuda_fail(err, "ordering of the fused backward streams");
    launch_dq_whole<D>(pl, prm, -1, (int)hq, sms, s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch of the fused backward kernels");
    return MARBLE_OK;
  }
  // ranges of ring steps: consecutive q shards of one kv shard whose dS^T tiles fit in half
  // the scratch cap (two ranges in flight); MARBLE_DS_SCRATCH_CAP_MB lowers the cap (tests)
  struct Range { int j, s0, len; int64_t tiles; };
  std::vector<Range> ranges;
  const size_t cap = scratch_cap();
  const int64_t cap_slots = (int64_t)(cap / 2 / 32768);
  int64_t buf_slots = 0;
  for (int j = 0; j < P; ++j) {
    int s0 = 0;
    int64_t acc = 0;
    for (int st = 0; st < P; ++st) {
      const int r = (j + st) % P;
      const int64_t t = pl->h_step_tiles[(size_t)r * (P + 1) + j];
      if (st > s0 && (acc + t) * hq > cap_slots) {
        ranges.push_back({j, s0, st - s0, acc});
        buf_slots = std::max(buf_slots, acc * hq);
        s0 = st;
        acc = 0;
      }
      acc += t;
    }
    ranges.push_back({j, s0, P - s0, acc});
    buf_slots = std::max(buf_slots, acc * hq);
  }
  const int nbuf = 2;
  rc = ds_scratch(pl, (size_t)(nbuf * buf_slots), s, &prm);
  if (rc != MARBLE_OK) return rc;
  cudaStream_t sk[kDkdvStreams];
  int nsk = 0;
  for (int k = 0; k < kDkdvStreams; ++k) {
    cudaStream_t x = side_stream(k);
    if (!x) break;
    cudaError_t e = stream_fork(s, x);
    if (e != cudaSuccess) return cuda_fail(e, "fork of the backward streams");
    sk[nsk++] = x;
  }
  if (nsk == 0) sk[nsk++] = s;
  const int nr = (int)ranges.size();
  std::vector<cudaEvent_t> ev_q(nr, nullptr);
  cudaError_t err = cudaSuccess;
  for (int i = 0; i < nr && err == cudaSuccess; ++i) {
    const Range& g = ranges[i];
    BwdParams pk = prm;
    pk.kv_shard = g.j;
    pk.q_shard = 0;
    pk.ring_s0 = g.s0;
    pk.ring_len = g.len;
    long long base = (long long)(i % nbuf) * buf_slots;
    for (int st = g.s0; st < g.s0 + g.len; ++st) {
      const int r = (g.j + st) % P;
      pk.ds_base[r] = base;
      base += (long long)pl->h_step_tiles[(size_t)r * (P + 1) + g.j] * hq;
    }
    // every kv block of shard j with a tile anywhere in its column (blocks without one in this
    // range are skipped by the scheduler)
    const int64_t seg = (int64_t)g.j * (P + 1) + P;
    pk.order = pl->bwd_order + seg * pl->bps;
    pk.nwork = pl->h_bwd_nwork[seg] * qkv->hkv;
    const cudaStream_t sks = sk[g.j % nsk];
    if (sks != s && i >= nbuf) err = cudaStreamWaitEvent(sks, ev_q[i - nbuf], 0);
    if (pk.nwork > 0 && err == cudaSuccess) {
      pk.sched = sched_slot(pl);
      const int span = timing_begin(sks);
      k_bwd_dkdv<D><<<(unsigned)(pk.nwork < sms ? pk.nwork : sms), kThreads, smem_k, sks>>>(pk);
      timing_end(span, sks, kTimeDkdv, 1);
    }
    if (sks != s && err == cudaSuccess) err = stream_fork(sks, s);
    for (int st = g.s0; st < g.s0 + g.len && err == cudaSuccess; ++st) {
      const int r = (g.j + st) % P;
      launch_dq<D>(pl, prm, r, g.j, pk.ds_base[r], (int)hq, sms, s);
    }
    if (err == cudaSuccess && sks != s) {
      err = cudaEventCreateWithFlags(&ev_q[i], cudaEventDisableTiming);
      if (err == cudaSuccess) err = cudaEventRecord(ev_q[i], s);
    }
  }
  for (int k = 0; k < nsk && err == cudaSuccess; ++k)
    if (sk[k] != s) err = stream_fork(sk[k], s);
  for (cudaEvent_t ev : ev_q)
    if (ev) cudaEventDestroy(ev);
  if (err != cudaSuccess) return cuda_fail(err, "ordering of the fused backward streams");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch of the fused backward kernels");
  return MARBLE_OK;
}

}  // namespace

marble_status_t run_attn_bwd_fused(const marble_plan_t* p, const marble_qkv_t* qkv,
                                   const void* d_o, const float* lse, const float* delta,
                                   float* dq, float* dk, float* dv, cudaStream_t s) {
  if (p->P > kMaxShards) return fail(MARBLE_ERR_UNSUPPORTED, "more than 256 shards");
  if (qkv->d == 128) return launch_fused<128>(p, qkv, d_o, lse, delta, dq, dk, dv, s);
  if (qkv->d == 64) return launch_fused<64>(p, qkv, d_o, lse, delta, dq, dk, dv, s);
  return fail(MARBLE_ERR_UNSUPPORTED, "head dim must be 64 or 128");
}

marble_status_t run_attn_bwd(const marble_plan_t* p, const marble_qkv_t* qkv, const void* d_o,
                             const float* lse, const float* delta, int n_steps,
                             const int* q_shards, const int* kv_shards, float* dq, float* dk,
                             float* dv, cudaStream_t s) {
  if (qkv->d == 128)
    return launch_steps<128>(p, qkv, d_o, lse, delta, n_steps, q_shards, kv_shards, dq, dk, dv, s);
  if (qkv->d == 64)
    return launch_steps<64>(p, qkv, d_o, lse, delta, n_steps, q_shards, kv_shards, dq, dk, dv, s);
  return fail(MARBLE_ERR_UNSUPPORTED, "head dim must be 64 or 128");
}

}  // namespace marble
