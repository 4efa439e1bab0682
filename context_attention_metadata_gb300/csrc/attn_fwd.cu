// Forward ring step: update the fp32 online-softmax state (O_acc, m, l) of one q shard
// against the tiles the plan lists for one kv shard (or for all needed kv blocks).
//
// MARBLE post, s03 "Exact ring attention accumulation": each ring step is the usual
// FlashAttention loop over a different set of key/value blocks; the fp32 accumulator, m
// and l stay in HBM between calls and are resumed on every call but the first; only
// the last call normalises.  RingAttention tutorial, "The Online Softmax Formulation":
// the recurrence m_new = max(m, rowmax S), rescale by exp(m - m_new), add exp(S - m_new).
//
// Kernel structure (sm_103a): one persistent CTA per SM takes work units (q block, q head)
// from a shared ticket counter, in the plan's order for the step (longest tile list first),
// and runs them through a pipeline of warp roles that meet at mbarriers:
//   warp 14     scheduler: draws a ticket, turns it into a unit and its tile-list range and
//               posts it in a 4-entry queue in shared memory; every other role reads the
//               queue in order, and the epilogue frees an entry once all roles are past it.
//   warp 0      TMA producer: Q of each unit into one of two slots, K_j and V_j through
//               two-slot rings.
//   warp 1      allocates all 512 TMEM columns: S double buffer [0,128) and [128,256),
//               O double buffer [256,384) and [384,512) (units alternate); lane 0 issues
//               tcgen05.mma -- S = Q K^T up to two tiles ahead of the softmax, O += P V with P
//               as bf16 in TMEM over its S buffer and V read MN-major -- polling its inputs
//               and issuing whichever of the next PV and the next S is ready.
//   warps 2..9  softmax: two warps per TMEM lane quarter, each owning 64 of a row's 128
//               columns; the row max is exchanged through shared memory.  Row max, exp2,
//               row sum, bf16 P back into TMEM, lazy O rescale; at a unit's end they hand
//               the row's (m, l) to the epilogue and go on with the next unit at once.  On
//               partial tiles they stage the keys' tracks and evaluate the mask once per
//               pair; full tiles skip it; empty tiles are never listed, so never loaded.
//   warps 10..13 epilogue, one thread per row: merge the unit's (O, m, l) into the stored
//               state through a staged TMA store / reduce-add, while the softmax warps and
//               the tensor core work on the next unit in the other O buffer.
// Scores are kept in base-2 units (s * scale * log2 e); the stored m is in the same units
// and always an integer, so that every rescale (lazy, when the max grows past 2^8, within
// a call; and the merge with the stored state) multiplies by an exact power of two.
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tma_host.h"

namespace marble {
namespace {

constexpr int kThreads = 480;              // 15 warps, roles above
constexpr int kSoftmax = 256;              // softmax threads (warps 2..9)
constexpr int kEpi = 128;                  // epilogue threads (warps 10..13)
constexpr int kWarpEpi0 = 10;
constexpr int kWarpSched = 14;
constexpr float kRescaleThreshold = 8.0f;  // base-2 units: rescale O when max grows > 2^8
constexpr int kQueue = 4;                  // work-queue entries

enum {
  B_QFULL0, B_QFULL1, B_QEMPTY0, B_QEMPTY1,  // Q slots (unit & 1): fill / last S of the unit
  B_KFULL0, B_KFULL1, B_KEMPTY0, B_KEMPTY1,  // K ring (slot = tile & 1): fill / S done
  B_VFULL0, B_VFULL1, B_VEMPTY0, B_VEMPTY1,  // V ring: fill / PV done
  B_SFULL0, B_SFULL1,                // S buffer (tile & 1) computed
  B_PFULL0, B_PFULL1,                // P written over S buffer (256 softmax arrivals)
  B_PVDONE,                          // one phase per tile: its PV has completed
  B_OFULL0, B_OFULL1,                // O buffer (unit & 1): the unit's last PV completed
  B_OFREE0, B_OFREE1,                // O buffer read out by the epilogue (128 arrivals)
  B_MX0, B_MX1,                      // per-row max exchanged between the two halves
  B_TRK0, B_TRK1,                    // key tracks of a partial tile staged
  B_EPIRDY0, B_EPIRDY1,              // (m, l) of the unit handed over (256 arrivals)
  B_HFREE0, B_HFREE1,                // hand-over slot read by the epilogue (128 arrivals)
  B_EVOTE,                           // per unit: epilogue's merge-mode vote (128 arrivals)
  B_STG,                             // per staging round: rows written (128 arrivals)
  B_STGFREE,                         // per staging round: the TMA has read the staging box
  B_UFULL0,                          // queue entry posted (kQueue barriers)
  B_UEMPTY0 = B_UFULL0 + kQueue,     // queue entry released (kQueue barriers)
  B_DRAIN = B_UEMPTY0 + kQueue,
  B_NUM
};

__host__ __device__ constexpr int arrivals(int b) {
  return (b == B_PFULL0 || b == B_PFULL1 || b == B_MX0 || b == B_MX1 || b == B_TRK0 ||
          b == B_TRK1 || b == B_EPIRDY0 || b == B_EPIRDY1)
             ? kSoftmax
             : ((b == B_OFREE0 || b == B_OFREE1 || b == B_HFREE0 || b == B_HFREE1 ||
                 b == B_EVOTE || b == B_STG)
                    ? kEpi
                    : 1);
}

struct FwdParams {
  CUtensorMap q_map, k_map, v_map;
  CUtensorMap o_map;  // fp32 O_acc, box 32 x 128 x 1, 128-byte swizzle
  const int64_t* step_ptr;
  const int32_t* step_col;
  const uint8_t* step_tag;
  const int32_t* tracks;  // [4][n] sample, seg, noise, pos in plan order
  const int32_t* order;   // work order of this step: q blocks of the shard, longest first
  unsigned* sched;        // ticket counter pair of this launch
  float* o_acc;
  float* m;
  float* l;
  unsigned* err;
  unsigned long long wait_ns;
  long long n;
  int P, bps, q_shard, kv_shard;
  int hq, group;
  int units;  // bps * hq
  int nwork;  // units with at least one tile: nonempty blocks of the order x hq
  int W;
  int first;
  int lse_merge;   // 0 carried state; 1 merge of bf16 partials (standard ring); 2 of fp32 ones
  const int32_t* kiv;       // [2][n] lo, hi of every key's visible-query interval
  const int4* kiv_chunk;    // [nb*4] per 32 keys: min lo, max lo, min hi, max hi
  const int32_t* qidx;      // [n] plan order -> index in the given token order (the plan's perm)
  const uint8_t* iv_block;  // [nb] 1: every key of the block has an exact interval
  float scale_log2;
};

// list range of work unit u = h * bps + i (q block i of the shard, q head h)
__device__ __forceinline__ int unit_tiles(const FwdParams& p, int u, int64_t* e0) {
  const int i = u % p.bps;
  const int64_t nq = (int64_t)p.q_shard * p.bps + i;
  int64_t a, b;
  if (p.kv_shard >= 0) {
    a = p.step_ptr[nq * p.P + p.kv_shard];
    b = p.step_ptr[nq * p.P + p.kv_shard + 1];
  } else {
    a = p.step_ptr[nq * p.P];
    b = p.step_ptr[nq * p.P + p.P];
  }
  *e0 = a;
  return (int)(b - a);
}

// the work queue in shared memory: entry uc of this CTA sits in slot uc % kQueue
struct Queue {
  int unit[kQueue];  // -1: no more work
  int T[kQueue];
  long long e0[kQueue];
};

// two-slot rings indexed by the tile counter g: slot g & 1, phase parity (g >> 1) & 1
__device__ __forceinline__ uint32_t ring_slot(int g) { return (uint32_t)(g & 1); }
__device__ __forceinline__ uint32_t ring_parity(int g) { return (uint32_t)((g >> 1) & 1); }

// shared memory: Q (2) | K ring (2) | V ring (2) | staging (one 128 x 32 fp32 box) | key
// tracks [2][4][128] int32 | row-max exchange [2][2][128] f32 | hand-over m [2][128] and
// l [2][2][128] f32
template <int D>
struct Smem {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = 2 * kTile;
  static constexpr int kV = 4 * kTile;
  static constexpr int kStg = 6 * kTile;
  static constexpr int kTrk = kStg + 16384;
  static constexpr int kMx = kTrk + 2 * 512 * 4;
  static constexpr int kHm = kMx + 2 * 2 * 128 * 4;
  static constexpr int kHl = kHm + 2 * 128 * 4;
  static constexpr int kEnd = kHl + 2 * 2 * 128 * 4;
  static constexpr size_t bytes() { return (size_t)kEnd + 1024; }  // + alignment slack
};
static_assert(Smem<128>::bytes() <= 232448, "shared memory budget");

template <int D>
__global__ void __launch_bounds__(kThreads, 1) k_attn_fwd(const __grid_constant__ FwdParams p) {
  using L = Smem<D>;
  constexpr int kTile = L::kTile;
  constexpr int kAtoms = D / 64;  // 128-byte swizzle atoms along d
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem + L::kQ;  // slot b at sQ + b * kTile
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  uint8_t* sStg = smem + L::kStg;
  int32_t* ktr = reinterpret_cast<int32_t*>(smem + L::kTrk);
  float* mxs = reinterpret_cast<float*>(smem + L::kMx);
  float* hm = reinterpret_cast<float*>(smem + L::kHm);
  float* hl = reinterpret_cast<float*>(smem + L::kHl);
  __shared__ __align__(8) uint64_t bar[B_NUM];
  __shared__ Queue queue;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int epi_mode[2];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long n = p.n;
  WaitCtx w{p.wait_ns, p.err, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    epi_mode[0] = epi_mode[1] = 0;
    for (int b = 0; b < B_NUM; ++b) mbar_init(&bar[b], arrivals(b));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = tmem_base;        // S buffers at +0 and +128
  const uint32_t tO = tmem_base + 256;  // O buffers at +0 and +128

  if (warp == kWarpSched) {
    // ------------------------------------------------------------------ scheduler
    if (lane == 0) {
      for (int uc = 0;; ++uc) {
        const int slot = uc % kQueue;
        if (uc >= kQueue && !mbar_wait(&bar[B_UEMPTY0 + slot], ((uc / kQueue) - 1) & 1, w)) break;
        int unit = -1, T = 0;
        int64_t e0 = 0;
        // longest lists first, the q heads of a block one after the other
        const unsigned t = atomicAdd(p.sched, 1u);
        if (t < (unsigned)p.nwork) {
          unit = (int)(t % (unsigned)p.hq) * p.bps + p.order[t / (unsigned)p.hq];
          T = unit_tiles(p, unit, &e0);
        }
        queue.unit[slot] = unit;
        queue.T[slot] = T;
        queue.e0[slot] = e0;
        mbar_arrive(&bar[B_UFULL0 + slot]);
        if (unit < 0) break;
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.q_map);
      tma_prefetch_desc(&p.k_map);
      tma_prefetch_desc(&p.v_map);
      tma_prefetch_desc(&p.o_map);
    }
    int uc = 0, g = 0;          // units reached, tiles reached
    int q_fills = 0, k_fills = 0, v_fills = 0;  // copies issued (fill t of K/V is tile t)
    bool ok = true;
    while (ok) {
      const int slot = uc % kQueue;
      if (!wait_all(&bar[B_UFULL0 + slot], (uc / kQueue) & 1, w)) break;
      const int unit = queue.unit[slot];
      if (unit < 0) break;
      const int T = queue.T[slot];
      const int64_t e0 = queue.e0[slot];
      const int h = unit / p.bps;
      const int kvh = h / p.group;
      const int64_t nq = (int64_t)p.q_shard * p.bps + unit % p.bps;
      // Q of the unit once the unit two back has finished reading the slot
      const int qb = uc & 1;
      if (uc >= 2 && !wait_all(&bar[B_QEMPTY0 + qb], ((uc >> 1) - 1) & 1, w)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar[B_QFULL0 + qb], kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(sQ + qb * kTile + a * 16384, &p.q_map, &bar[B_QFULL0 + qb], a * 64,
                      (int)(nq * 128), h);
      }
      ++q_fills;
      for (int j = 0; j < T; ++j, ++g) {
        const int nk = p.step_col[e0 + j];
        const uint32_t s = ring_slot(g);
        if (g >= 2 && !wait_all(&bar[B_KEMPTY0 + s], ring_parity(g - 2), w)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar[B_KFULL0 + s], kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_3d(sK + s * kTile + a * 16384, &p.k_map, &bar[B_KFULL0 + s], a * 64,
                        nk * 128, kvh);
        }
        ++k_fills;
        if (g >= 2 && !wait_all(&bar[B_VEMPTY0 + s], ring_parity(g - 2), w)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar[B_VFULL0 + s], kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_3d(sV + s * kTile + a * 16384, &p.v_map, &bar[B_VFULL0 + s], a * 64,
                        nk * 128, kvh);
        }
        ++v_fills;
      }
      ++uc;
    }
    // never leave the CTA with a copy still landing in its shared memory: the fills of a
    // slot complete in order, so waiting for the latest fill of each slot suffices (Q fill
    // f went to slot f & 1, K and V fill t to ring slot t & 1)
    if (lane == 0) {
      for (int f = q_fills - 1; f >= 0 && f >= q_fills - 2; --f)
        drain_wait(&bar[B_QFULL0 + (f & 1)], (f >> 1) & 1, p.wait_ns, p.err);
      for (int t = k_fills - 1; t >= 0 && t >= k_fills - 2; --t)
        drain_wait(&bar[B_KFULL0 + ring_slot(t)], ring_parity(t), p.wait_ns, p.err);
      for (int t = v_fills - 1; t >= 0 && t >= v_fills - 2; --t)
        drain_wait(&bar[B_VFULL0 + ring_slot(t)], ring_parity(t), p.wait_ns, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);
      const uint32_t aQ0 = smem_u32(sQ), aK0 = smem_u32(sK), aV0 = smem_u32(sV);
      // Event loop over two cursors into the work queue: issue whichever of the next PV
      // (priority: it feeds the softmax and the epilogue) and the next S (at most two tiles
      // ahead of the next PV) has its inputs ready, polling with non-blocking tests.
      struct Cur {
        int uc, j, g, T, state;  // state: 0 waiting for queue entry uc, 1 in a unit, 2 done
      };
      Cur cs{0, 0, 0, 0, 0}, cp{0, 0, 0, 0, 0};
      auto fetch = [&](Cur& c) {
        if (c.state != 0) return;
        const int slot = c.uc % kQueue;
        if (!mbar_test(&bar[B_UFULL0 + slot], (c.uc / kQueue) & 1)) return;
        c.state = queue.unit[slot] < 0 ? 2 : 1;
        c.T = queue.T[slot];
        c.j = 0;
      };
      auto advance = [](Cur& c) {
        ++c.g;
        if (++c.j == c.T) {
          ++c.uc;
          c.state = 0;
        }
      };
      uint64_t t_idle = 0;
      uint32_t idle = 0;
      while (cs.state != 2 || cp.state != 2) {
        fetch(cs);
        fetch(cp);
        bool progressed = false;
        if (cp.state == 1) {
          const int g = cp.g;
          const uint32_t b = (uint32_t)(g & 1), s = ring_slot(g), ob = (uint32_t)(cp.uc & 1);
          // the first PV of a unit overwrites its O buffer: the unit two back must be read out
          const bool ready =
              mbar_test(&bar[B_PFULL0 + b], (g >> 1) & 1) &&
              mbar_test(&bar[B_VFULL0 + s], ring_parity(g)) &&
              (cp.j != 0 || cp.uc < 2 || mbar_test(&bar[B_OFREE0 + ob], ((cp.uc >> 1) - 1) & 1));
          if (ready) {
            tc_fence_after();
            const uint32_t aV = aV0 + s * kTile;
            // P of half h sits in columns [64 h, 64 h + 32) of the S buffer
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ts(tO + ob * 128, tS + b * 128 + (k >> 2) * 64 + (k & 3) * 8,
                     sdesc_sw128(aV + k * 2048, 16384, 1024), kIdO, (cp.j > 0 || k > 0) ? 1u : 0u);
            mma_commit(&bar[B_PVDONE]);
            mma_commit(&bar[B_VEMPTY0 + s]);
            if (cp.j == cp.T - 1) mma_commit(&bar[B_OFULL0 + ob]);
            advance(cp);
            progressed = true;
          }
        }
        if (cs.state == 1 && cs.g < cp.g + 2) {
          const int g = cs.g;
          const uint32_t b = (uint32_t)(g & 1), s = ring_slot(g), qb = (uint32_t)(cs.uc & 1);
          // S(g) overwrites the P of tile g - 2, which PV(g - 2) reads: the PV is issued already
          // (S runs at most two tiles ahead of the next PV), and tcgen05.mma instructions of one
          // thread execute in issue order, so no wait for its completion is needed
          const bool ready = (cs.j != 0 || mbar_test(&bar[B_QFULL0 + qb], (cs.uc >> 1) & 1)) &&
                             mbar_test(&bar[B_KFULL0 + s], ring_parity(g));
          if (ready) {
            tc_fence_after();
            const uint32_t aQ = aQ0 + qb * kTile, aK = aK0 + s * kTile;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
              mma_ss(tS + b * 128, sdesc_sw128(aQ + off, 16, 1024),
                     sdesc_sw128(aK + off, 16, 1024), kIdS, k > 0);
            }
            mma_commit(&bar[B_SFULL0 + b]);
            mma_commit(&bar[B_KEMPTY0 + s]);
            if (cs.j == cs.T - 1) mma_commit(&bar[B_QEMPTY0 + qb]);  // the unit's last read of Q
            advance(cs);
            progressed = true;
          }
        }
        if (progressed) {
          idle = 0;
        } else {
          // the clock is read only while idle, so that it never delays an issue
          __nanosleep(32);
          if ((++idle & 63) == 0) {
            if (*w.abort) break;
            const uint64_t now = globaltimer_ns();
            if (idle == 64) {
              t_idle = now;
            } else if (now - t_idle > p.wait_ns) {
              atomicOr(p.err, kErrTimeout);
              *w.abort = 1;
              break;
            }
          }
        }
      }
      // every MMA issued by this thread has completed before TMEM is released
      mma_commit(&bar[B_DRAIN]);
      drain_wait(&bar[B_DRAIN], 0, p.wait_ns, p.err);
    }
    __syncwarp();
  }
  else if (warp < kWarpEpi0) {
    // ------------------------------------------------------------------ softmax warps
    // two warps per TMEM lane quarter: `half` owns S columns [64 half, 64 half + 64) and O
    // columns [D/2 half, D/2 half + D/2) of its row
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    int uc = 0, g = 0, n_partial = 0;
    bool ok = true;
    while (ok) {
      const int slot = uc % kQueue;
      if (!wait_all(&bar[B_UFULL0 + slot], (uc / kQueue) & 1, w)) break;
      const int unit = queue.unit[slot];
      if (unit < 0) break;
      const int T = queue.T[slot];
      const int64_t e0 = queue.e0[slot];
      const int64_t tq = ((int64_t)p.q_shard * p.bps + unit % p.bps) * 128 + row;
      const int sq = p.tracks[tq], gq = p.tracks[n + tq], zq = p.tracks[2 * n + tq],
                pq = p.tracks[3 * n + tq];
      const int iq = p.qidx[tq];  // the interval test's coordinate: the query's index
      const uint32_t ob = tO + (uint32_t)(uc & 1) * 128;
      float m_run = -INFINITY, l_h = 0.f;
      for (int j = 0; j < T; ++j, ++g) {
        const uint32_t b = (uint32_t)(g & 1);
        const bool partial = p.step_tag[e0 + j] == MARBLE_TILE_PARTIAL;
        uint32_t lm[2] = {~0u, ~0u};  // legal-key bits of this row in this half's 64 columns
        const int64_t kb = partial ? p.step_col[e0 + j] : 0;
        // every key of the block has an exact visible-query interval: the test is
        // lo_k <= i_q < hi_k (i_q the query's index in the given token order), with the half's
        // 64 (lo, hi) pairs read straight from global memory (the same addresses for every
        // lane: broadcast loads)
        const bool ivt = partial && p.iv_block[kb] != 0;
        if (ivt) {
          // per 32-key chunk, its keys' (min lo, max lo, min hi, max hi) first: a row inside
          // every interval takes all 32 keys and a row outside all of them none; the keys are
          // tested one by one only when some row of the warp is neither
          const int32_t* klo = p.kiv + kb * 128 + half * 64;
          const int32_t* khi = klo + n;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int4 cs = __ldg(p.kiv_chunk + kb * 4 + half * 2 + cc);
            const bool all = iq >= cs.y && iq < cs.z;
            const bool none = iq < cs.x || iq >= cs.w;
            uint32_t bits = all ? ~0u : 0u;
            if (__any_sync(0xffffffffu, !(all || none))) {
              bits = 0;
#pragma unroll
              for (int t2 = 0; t2 < 32; t2 += 4) {
                const int4 l4 = __ldg(reinterpret_cast<const int4*>(klo + cc * 32 + t2));
                const int4 h4 = __ldg(reinterpret_cast<const int4*>(khi + cc * 32 + t2));
                bits |= ((iq >= l4.x) & (iq < h4.x) ? 1u : 0u) << t2;
                bits |= ((iq >= l4.y) & (iq < h4.y) ? 1u : 0u) << (t2 + 1);
                bits |= ((iq >= l4.z) & (iq < h4.z) ? 1u : 0u) << (t2 + 2);
                bits |= ((iq >= l4.w) & (iq < h4.w) ? 1u : 0u) << (t2 + 3);
              }
            }
            lm[cc] = bits;
          }
        } else if (partial) {
          // stage the 128 keys' tracks in one of two buffers (the two halves load two tracks
          // each); every softmax thread arrives before any reads, so a buffer is rewritten
          // only after every thread left its previous use
          const int bb = n_partial & 1;
          const uint32_t par = (n_partial >> 1) & 1;
          ++n_partial;
          int32_t* kt = ktr + bb * 512;
          const int64_t t = kb * 128 + row;
          if (half == 0) {
            kt[row] = p.tracks[t];
            kt[128 + row] = p.tracks[n + t];
          } else {
            kt[256 + row] = p.tracks[2 * n + t];
            kt[384 + row] = p.tracks[3 * n + t];
          }
          mbar_arrive(&bar[B_TRK0 + bb]);
          if (!wait_all(&bar[B_TRK0 + bb], par, w)) { ok = false; break; }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int kc0 = (2 * half + cc) * 32;
            uint32_t bits = 0;
#pragma unroll
            for (int t2 = 0; t2 < 32; ++t2) {
              const int kc = kc0 + t2;
              bits |= (mask_legal(sq, gq, zq, pq, kt[kc], kt[128 + kc], kt[256 + kc],
                                  kt[384 + kc], p.W) ? 1u : 0u) << t2;
            }
            lm[cc] = bits;
          }
        }
        // a partial tile on which every row of this warp keeps all 64 of its keys takes the
        // full-tile path below
        const bool masked = partial && __any_sync(0xffffffffu, (lm[0] & lm[1]) != ~0u);
        if (!wait_all(&bar[B_SFULL0 + b], (g >> 1) & 1, w)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sb = tS + b * 128;
        uint32_t v[2][32];
        tmem_ld32(sb + lb + (2 * half) * 32, v[0]);
        tmem_ld32(sb + lb + (2 * half + 1) * 32, v[1]);
        tmem_ld_wait();
        // this half's row maximum of the scaled, masked scores; where a key is masked the
        // scaled scores (-inf where masked) replace v, otherwise v keeps the raw scores
        // (scaling by a positive constant commutes with the maximum, and P takes one FMA below)
        float mx = -INFINITY;
        if (masked) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              const float s = ((lm[cc] >> t) & 1u) ? __uint_as_float(v[cc][t]) * sl2 : -INFINITY;
              v[cc][t] = __float_as_uint(s);
              mx = fmaxf(mx, s);
            }
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int t = 0; t < 32; ++t) mx = fmaxf(mx, __uint_as_float(v[cc][t]));
          mx *= sl2;
        }
        float* mxb = mxs + b * 256;
        mxb[half * 128 + row] = mx;
        mbar_arrive(&bar[B_MX0 + b]);
        if (!wait_all(&bar[B_MX0 + b], (g >> 1) & 1, w)) { ok = false; break; }
        mx = fmaxf(mx, mxb[(1 - half) * 128 + row]);
        // the running max is kept integral (base 2): every rescale factor below is then an
        // exact power of two, and bf16 rounding of P does not depend on which keys a step
        // happened to see first
        const float m_new = ceilf(mx);
        const bool grow = m_new > m_run + kRescaleThreshold;
        const bool need = grow && (m_run != -INFINITY);  // earlier tiles of this unit to rescale
        const float alpha = need ? ldexpf(1.f, (int)(m_run - m_new)) : 1.f;
        if (grow) {
          l_h *= alpha;
          m_run = m_new;
        }
        // tcgen05.ld/st are warp-collective: the whole warp rescales when any of its rows
        // must (alpha = 1 on the others).  A row that needs it has a finite max from an
        // earlier tile of this unit, so PV(g-1) is the accumulation to wait for.
        if (__any_sync(0xffffffffu, need)) {
          if (!wait_all(&bar[B_PVDONE], (g - 1) & 1, w)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < D / 64; ++cc) {
            const uint32_t col = half * (D / 2) + cc * 32;
            uint32_t x[32];
            tmem_ld32(ob + lb + col, x);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < 32; ++t) x[t] = __float_as_uint(__uint_as_float(x[t]) * alpha);
            tmem_st32(ob + lb + col, x);
          }
        }
        // P = exp2(s - m_run) as bf16, packed into columns [64 half, 64 half + 32) of the S
        // buffer: inside the fp32 columns this warp has just read
        const float base = (m_run == -INFINITY) ? 0.f : m_run;
        // v holds scaled scores where keys were masked, raw ones otherwise
        const float vs = masked ? 1.f : sl2;
        float rs = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            const float p0 = fast_exp2(fmaf(__uint_as_float(v[cc][t]), vs, -base));
            const float p1 = fast_exp2(fmaf(__uint_as_float(v[cc][t + 1]), vs, -base));
            rs += p0 + p1;
            pk[t >> 1] = pack_bf16(p0, p1);
          }
          tmem_st16(sb + lb + half * 64 + cc * 16, pk);
        }
        tmem_st_wait();
        l_h += rs;
        tc_fence_before();
        mbar_arrive(&bar[B_PFULL0 + b]);
      }
      if (!ok) break;
      // hand the unit's (m, l) to the epilogue once it has read the slot's previous use
      const int ub = uc & 1;
      if (uc >= 2 && !wait_all(&bar[B_HFREE0 + ub], ((uc >> 1) - 1) & 1, w)) break;
      if (half == 0) hm[ub * 128 + row] = m_run;
      hl[(ub * 2 + half) * 128 + row] = l_h;
      mbar_arrive(&bar[B_EPIRDY0 + ub]);
      ++uc;
    }
  }
  else {
    // ------------------------------------------------------------------ epilogue warps
    // one thread per row (warp w owns TMEM lane quarter w & 3)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    if (p.first) {
      // rows of units without a tile in this step start from (O = 0, m = -inf, l = 0)
      for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        int64_t e0;
        if (unit_tiles(p, u, &e0) != 0) continue;
        const int h = u / p.bps;
        const int64_t tq = ((int64_t)p.q_shard * p.bps + u % p.bps) * 128 + row;
        p.m[(int64_t)h * n + tq] = -INFINITY;
        p.l[(int64_t)h * n + tq] = 0.f;
        float4* o = reinterpret_cast<float4*>(p.o_acc + (tq * p.hq + h) * D);
#pragma unroll 8
        for (int t = 0; t < D / 4; ++t) o[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    // Merge each unit's (O, m, l) into the stored state through one staged fp32 box of 32
    // columns at a time:
    //   FIRST         the tile is stored (TMA store);
    //   otherwise     the stored max is kept unless some row's max grew past it by more
    //                 than the lazy threshold, so the update is a pure addition of
    //                 O_call * 2^(m_call - m_stored): a TMA fp32 reduce-add, no load;
    //   some row grew exact merge with the stored tile (loaded by the row threads), then a
    //                 TMA store.
    //   LSE merge     the call's output is normalised into a partial, merged with the
    //                 stored (normalised) output by log-sum-exp weights and stored; m then
    //                 holds the running base-2 LSE and l is 1 (0 for a row that has seen no
    //                 legal key), which the finalize reads unchanged.  Partial and merged
    //                 output are rounded to bf16 (the standard ring merge, kept for
    //                 comparison) or kept in fp32 (merging fp32 partials: exact to fp32).
    int uc = 0, k = 0;  // units merged, staging rounds
    bool ok = true;
    while (ok) {
      const int slot = uc % kQueue;
      if (!wait_all(&bar[B_UFULL0 + slot], (uc / kQueue) & 1, w)) break;
      const int unit = queue.unit[slot];
      if (unit < 0) break;
      const int h = unit / p.bps;
      const int64_t q0 = ((int64_t)p.q_shard * p.bps + unit % p.bps) * 128;
      const int64_t tq = q0 + row;
      const int64_t gi = (int64_t)h * n + tq;
      float m_old = -INFINITY, l_old = 0.f;
      if (!p.first) {
        m_old = p.m[gi];
        l_old = p.l[gi];
      }
      const int ub = uc & 1;
      if (!wait_all(&bar[B_EPIRDY0 + ub], (uc >> 1) & 1, w)) break;
      const float m_run = hm[ub * 128 + row];
      const float l_run = hl[ub * 256 + row] + hl[ub * 256 + 128 + row];
      mbar_arrive(&bar[B_HFREE0 + ub]);
      // the merge mode is one per unit: the four warps vote
      const bool grows = !p.first && m_old != -INFINITY && m_run > m_old + kRescaleThreshold;
      if (__any_sync(0xffffffffu, grows) && lane == 0) atomicOr(&epi_mode[uc & 1], 1);
      mbar_arrive(&bar[B_EVOTE]);
      if (!wait_all(&bar[B_EVOTE], uc & 1, w)) break;
      const int mode = p.lse_merge ? 3 : p.first ? 0 : (epi_mode[uc & 1] ? 2 : 1);
      // every epilogue thread has read the other flag (before this vote), and none can vote
      // on the next unit before row 0 has passed its first staging round of this one
      if (row == 0) epi_mode[(uc + 1) & 1] = 0;
      if (!wait_all(&bar[B_OFULL0 + ub], (uc >> 1) & 1, w)) break;
      tc_fence_after();
      // every role is past queue entry uc: the producer and the S cursor before the last S,
      // the PV cursor before the last PV, the softmax before the hand-over, and this group
      // before the vote
      if (row == 0) mbar_arrive(&bar[B_UEMPTY0 + slot]);
      float a_new = 1.f, a_old = 0.f, m_out = m_run, l_out = l_run;
      if (mode == 1) {
        m_out = (m_old == -INFINITY) ? m_run : m_old;
        a_new = (m_run == -INFINITY) ? 0.f : ldexpf(1.f, (int)fmaxf(m_run - m_out, -1000.f));
        l_out = l_old + l_run * a_new;
      } else if (mode == 2) {
        m_out = fmaxf(m_old, m_run);  // both integral: the factors are exact powers of two
        a_old = (m_old == -INFINITY) ? 0.f : ldexpf(1.f, (int)fmaxf(m_old - m_out, -1000.f));
        a_new = (m_run == -INFINITY) ? 0.f : ldexpf(1.f, (int)fmaxf(m_run - m_out, -1000.f));
        l_out = l_old * a_old + l_run * a_new;
      } else if (mode == 3) {
        // log-sum-exp merge in base 2: b = the call's LSE, m_old = the stored one
        const float b = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
        const float hi = fmaxf(m_old, b), lo = fminf(m_old, b);
        m_out = lo == -INFINITY ? hi : hi + log1pf(exp2f(lo - hi)) * 1.4426950408889634f;
        a_old = m_old == -INFINITY ? 0.f : exp2f(m_old - m_out);
        a_new = b == -INFINITY ? 0.f : exp2f(b - m_out);  // weight of the normalised partial
        l_out = m_out == -INFINITY ? 0.f : 1.f;
      }
      p.m[gi] = m_out;
      p.l[gi] = l_out;
      const uint32_t ob = tO + (uint32_t)ub * 128;
      const float4* src = reinterpret_cast<const float4*>(p.o_acc + (tq * p.hq + h) * D);
#pragma unroll 1
      for (int r = 0; r < D / 32; ++r, ++k) {
        if (k > 0 && !wait_all(&bar[B_STGFREE], (k - 1) & 1, w)) { ok = false; break; }
        uint32_t x[32];
        tmem_ld32(ob + lb + r * 32, x);
        tmem_ld_wait();
        if (r == D / 32 - 1) {
          // the O buffer can take unit uc + 2
          tc_fence_before();
          mbar_arrive(&bar[B_OFREE0 + ub]);
        }
        float vals[32];
        if (mode == 3) {
          // rnd(O_old * a_old + rnd(O_call / l_call) * a_new), rnd = bf16 rounding or none
          const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
          const bool rb = p.lse_merge == 1;
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const float o = __uint_as_float(x[t]) * inv_l;
            vals[t] = (rb ? bf16_round(o) : o) * a_new;
          }
          if (!p.first) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 o = src[r * 8 + t];
              vals[4 * t] = fmaf(o.x, a_old, vals[4 * t]);
              vals[4 * t + 1] = fmaf(o.y, a_old, vals[4 * t + 1]);
              vals[4 * t + 2] = fmaf(o.z, a_old, vals[4 * t + 2]);
              vals[4 * t + 3] = fmaf(o.w, a_old, vals[4 * t + 3]);
            }
          }
          if (rb) {
#pragma unroll
            for (int t = 0; t < 32; ++t) vals[t] = bf16_round(vals[t]);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) vals[t] = __uint_as_float(x[t]) * a_new;
        }
        if (mode == 2) {
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float4 o = src[r * 8 + t];
            vals[4 * t] += o.x * a_old;
            vals[4 * t + 1] += o.y * a_old;
            vals[4 * t + 2] += o.z * a_old;
            vals[4 * t + 3] += o.w * a_old;
          }
        }
        stage_row32(sStg, row, vals);
        fence_proxy_async_smem();
        mbar_arrive(&bar[B_STG]);
        if (row == 0) {
          if (mbar_wait(&bar[B_STG], k & 1, w)) {
            if (mode == 1)
              tma_reduce_add_3d(&p.o_map, sStg, r * 32, (int)q0, h);
            else
              tma_store_3d(&p.o_map, sStg, r * 32, (int)q0, h);
            bulk_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&bar[B_STGFREE]);
        }
      }
      ++uc;
    }
    // the global writes of every TMA store / reduce this thread issued have completed
    if (row == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
  if (threadIdx.x == 0) {
    // every CTA of the launch has drawn its last ticket once it gets here: the last one to
    // arrive puts the counter pair back to zero for a later launch
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
  }
}

// everything but the shard pair, the FIRST flag and the work list: encoded once per call
template <int D>
marble_status_t prepare(const marble_plan_t* pl, const marble_qkv_t* qkv,
                        const marble_state_t* st, FwdParams* prm) {
  memset(prm, 0, sizeof(*prm));
  const int64_t n = pl->n;
  if (!make_rows_map(&prm->q_map, qkv->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, n, qkv->hq, D, 64,
                     128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_rows_map(&prm->k_map, qkv->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, n, qkv->hkv, D, 64,
                     128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_rows_map(&prm->v_map, qkv->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, n, qkv->hkv, D, 64,
                     128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_rows_map(&prm->o_map, st->o_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, n, qkv->hq, D, 32,
                     128, CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(MARBLE_ERR_CUDA, "cuTensorMapEncodeTiled failed for Q/K/V/O_acc");
  prm->step_ptr = pl->step_ptr;
  prm->step_col = pl->step_col;
  prm->step_tag = pl->step_tag;
  prm->tracks = pl->tracks;
  prm->kiv = pl->kiv;
  prm->kiv_chunk = pl->kiv_chunk;
  prm->qidx = pl->perm;
  prm->iv_block = pl->iv_block;
  prm->o_acc = st->o_acc;
  prm->m = st->m;
  prm->l = st->l;
  prm->err = pl->err;
  prm->wait_ns = wait_limit_ns();
  prm->n = n;
  prm->P = pl->P;
  prm->bps = (int)pl->bps;
  prm->hq = qkv->hq;
  prm->group = qkv->hq / qkv->hkv;
  prm->units = (int)(pl->bps * qkv->hq);
  prm->W = pl->W;
  const float scale = qkv->scale > 0.f ? qkv->scale : 1.0f / sqrtf((float)D);
  prm->scale_log2 = scale * 1.4426950408889634f;
  if (once_per_device(D == 128 ? 1 : 2)) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_fwd<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Smem<D>::bytes());
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(k_attn_fwd)");
  }
  return MARBLE_OK;
}

template <int D>
marble_status_t launch_steps(const marble_plan_t* pl, const marble_qkv_t* qkv, int n_steps,
                             const int* q_shards, const int* kv_shards, const uint32_t* flags,
                             const marble_state_t* st, cudaStream_t s) {
  FwdParams base;
  marble_status_t rc = prepare<D>(pl, qkv, st, &base);
  if (rc != MARBLE_OK) return rc;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Steps of different q shards touch disjoint rows of the state: q shard r runs on stream
  // r mod ns (the caller's stream and up to three side streams), so that the tails of
  // launches of different shards overlap.  Steps of one q shard stay in order on one stream.
  constexpr int kFwdSide = 3;
  cudaStream_t st_of[1 + kFwdSide] = {s};
  int ns = 1;
  if (n_steps > 1)
    for (int k = 0; k < kFwdSide; ++k) {
      cudaStream_t x = side_stream(k);
      if (!x) break;
      cudaError_t e = stream_fork(s, x);
      if (e != cudaSuccess) return cuda_fail(e, "fork of the forward streams");
      st_of[ns++] = x;
    }
  int span[1 + kFwdSide], launches[1 + kFwdSide] = {0};
  for (int k = 0; k < ns; ++k) span[k] = timing_begin(st_of[k]);
  for (int i = 0; i < n_steps; ++i) {
    FwdParams prm = base;
    prm.q_shard = q_shards[i];
    prm.kv_shard = kv_shards[i];
    prm.first = (flags[i] & MARBLE_STEP_FIRST) ? 1 : 0;
    prm.lse_merge = (flags[i] & MARBLE_STEP_BF16_MERGE) ? 1 : (flags[i] & MARBLE_STEP_FP32_MERGE) ? 2 : 0;
    const int64_t seg = (int64_t)prm.q_shard * (pl->P + 1) + (prm.kv_shard >= 0 ? prm.kv_shard : pl->P);
    prm.order = pl->fwd_order + seg * pl->bps;
    prm.nwork = pl->h_fwd_nwork[seg] * qkv->hq;
    if (prm.nwork == 0 && !prm.first) continue;  // nothing to add to the state
    prm.sched = sched_slot(pl);
    // persistent: one CTA per SM (each takes all 512 TMEM columns); the FIRST call also
    // initialises the units without tiles, spread over the whole grid
    const int want = prm.first ? base.units : prm.nwork;
    // with side streams, a launch takes at most half the SMs: launches of different q shards
    // then share the GPU instead of one waiting for the other's tail
    const int cap = ns > 1 ? (sms + 1) / 2 : sms;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    const int k = prm.q_shard % ns;
    k_attn_fwd<D><<<grid, kThreads, Smem<D>::bytes(), st_of[k]>>>(prm);
    ++launches[k];
  }
  for (int k = 0; k < ns; ++k) timing_end(span[k], st_of[k], kTimeFwd, launches[k]);
  for (int k = 1; k < ns; ++k) {
    cudaError_t e = stream_fork(st_of[k], s);
    if (e != cudaSuccess) return cuda_fail(e, "join of the forward streams");
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch k_attn_fwd");
  return MARBLE_OK;
}

// The fused forward: one launch over every (q block, q head) of every shard, each row
// walking its tiles in ring order (kv shard (r - s) mod P at step s, the plan's ring-ordered
// copy of its lists) with the fp32 state held on chip from the first step to the last; the
// state is written once, as the FIRST step of the per-step path writes it.
template <int D>
marble_status_t launch_fused(const marble_plan_t* pl, const marble_qkv_t* qkv,
                             const marble_state_t* st, cudaStream_t s) {
  FwdParams prm;
  marble_status_t rc = prepare<D>(pl, qkv, st, &prm);
  if (rc != MARBLE_OK) return rc;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // every block of the pack as one shard of nb blocks, whole rows, ring-ordered lists
  prm.bps = (int)pl->nb;
  prm.q_shard = 0;
  prm.kv_shard = -1;
  prm.first = 1;
  prm.lse_merge = 0;
  prm.step_col = pl->ring_col;
  prm.step_tag = pl->ring_tag;
  prm.order = pl->fwd_order_all;
  prm.units = (int)(pl->nb * qkv->hq);
  prm.nwork = pl->h_fwd_nwork_all * qkv->hq;
  prm.sched = sched_slot(pl);
  const unsigned grid = (unsigned)(prm.units < sms ? prm.units : sms);
  const int span = timing_begin(s);
  k_attn_fwd<D><<<grid, kThreads, Smem<D>::bytes(), s>>>(prm);
  timing_end(span, s, kTimeFwd, 1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch k_attn_fwd (fused)");
  return MARBLE_OK;
}

}  // namespace

marble_status_t run_attn_fwd_fused(const marble_plan_t* p, const marble_qkv_t* qkv,
                                   const marble_state_t* st, cudaStream_t s) {
  if ((int64_t)p->nb * qkv->hq > INT_MAX)
    return fail(MARBLE_ERR_UNSUPPORTED, "too many (block, head) work units");
  if (qkv->d == 128) return launch_fused<128>(p, qkv, st, s);
  if (qkv->d == 64) return launch_fused<64>(p, qkv, st, s);
  return fail(MARBLE_ERR_UNSUPPORTED, "head dim must be 64 or 128");
}

marble_status_t run_attn_fwd(const marble_plan_t* p, const marble_qkv_t* qkv, int n_steps,
                             const int* q_shards, const int* kv_shards, const uint32_t* flags,
                             const marble_state_t* st, cudaStream_t s) {
  if (qkv->d == 128) return launch_steps<128>(p, qkv, n_steps, q_shards, kv_shards, flags, st, s);
  if (qkv->d == 64) return launch_steps<64>(p, qkv, n_steps, q_shards, kv_shards, flags, st, s);
  return fail(MARBLE_ERR_UNSUPPORTED, "head dim must be 64 or 128");
}

}  // namespace marble
