// Forward ring step: update the fp32 online-softmax state (O_acc, m, l) of one q shard
// against the tiles the plan lists for one kv shard (or for all needed kv blocks).
//
// MARBLE post, s03 "Exact ring attention accumulation": each ring step is the usual
// FlashAttention loop over a different set of key/value blocks; the fp32 accumulator, m
// and l stay in HBM between calls and are resumed on every call but the first; only
// the last call normalises.  RingAttention tutorial, "The Online Softmax Formulation":
// the recurrence m_new = max(m, rowmax S), rescale by exp(m - m_new), add exp(S - m_new).
//
// Kernel structure (sm_103a): one CTA per (q block, q head) work unit, two CTAs per SM.
//   warp 0      TMA producer: Q tile once, then K_j and V_j of every listed tile (single
//               slot each; K_j+1 streams in while tile j's softmax and PV run).
//   warp 1      allocates 256 TMEM columns; lane 0 issues tcgen05.mma:
//                 S = Q K_j^T  (SS, 128x128, fp32 in TMEM columns [0,128))
//                 O += P_j V_j (TS: P as bf16 in TMEM columns [0,64) over S; V MN-major)
//   warps 2..5  one thread per query row (TMEM lane): row max, exp2, row sum, bf16 P
//               back into TMEM, lazy O rescale, and the final merge with the stored state;
//               on partial tiles they first stage the keys' metadata tracks in shared
//               memory and evaluate the mask once per pair into a 128-bit row mask.
// Full tiles skip the mask; partial tiles evaluate the packed-mask predicate per pair;
// empty tiles are never listed, so never loaded.  Scores are kept in base-2 units
// (s * scale * log2 e); the stored m is in the same units and always an integer, so that
// every rescale (lazy, by at least 2^8, within a call; and the merge with the stored
// state) multiplies by an exact power of two.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tma_host.h"

namespace marble {
namespace {

constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kPrefetchTiles = 64;  // L2 prefetch depth per unit  // base-2 units: rescale O when max grows > 2^8

enum {
  B_QFULL, B_KFULL, B_VFULL, B_KEMPTY, B_VEMPTY, B_SFULL, B_PFULL, B_OFULL, B_DRAIN,
  B_TRK0, B_TRK1, B_EPI0, B_EPI1, B_NUM
};

struct FwdParams {
  CUtensorMap q_map, k_map, v_map;
  CUtensorMap o_map;  // fp32 O_acc, box 32 x 128 x 1, 128-byte swizzle
  const int64_t* step_ptr;
  const int32_t* step_col;
  const uint8_t* step_tag;
  const int32_t* tracks;  // [4][n] sample, seg, noise, pos in plan order
  float* o_acc;
  float* m;
  float* l;
  unsigned* err;
  unsigned long long wait_ns;
  long long n;
  int P, bps, q_shard, kv_shard;
  int hq, group;
  int W;
  int first;
  float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2) k_attn_fwd(const __grid_constant__ FwdParams p) {
  constexpr int kTile = 128 * D * 2;  // bytes of one bf16 128 x D tile
  constexpr int kAtoms = D / 64;      // 128-byte swizzle atoms along d
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kTile;
  uint8_t* sV = smem + 2 * kTile;
  int32_t* ktr = reinterpret_cast<int32_t*>(smem + 3 * kTile);  // [2][4][128]
  __shared__ __align__(8) uint64_t bar[B_NUM];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int epi_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x / p.bps, i = blockIdx.x % p.bps;
  const long long n = p.n;
  const int64_t nq = (int64_t)p.q_shard * p.bps + i;
  int64_t e0, e1;
  if (p.kv_shard >= 0) {
    e0 = p.step_ptr[nq * p.P + p.kv_shard];
    e1 = p.step_ptr[nq * p.P + p.kv_shard + 1];
  } else {
    e0 = p.step_ptr[nq * p.P];
    e1 = p.step_ptr[nq * p.P + p.P];
  }
  const int T = (int)(e1 - e0);

  if (T == 0) {
    if (!p.first) return;
    // rows with no tile on their first step start from (O = 0, m = -inf, l = 0)
    for (int r = threadIdx.x; r < 128; r += kThreads) {
      p.m[(int64_t)h * n + nq * 128 + r] = -INFINITY;
      p.l[(int64_t)h * n + nq * 128 + r] = 0.f;
    }
    for (int idx = threadIdx.x; idx < 128 * (D / 4); idx += kThreads) {
      const int r = idx / (D / 4), c = idx % (D / 4);
      float4* o = reinterpret_cast<float4*>(p.o_acc + ((nq * 128 + r) * p.hq + h) * D) + c;
      *o = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }

  WaitCtx w{p.wait_ns, p.err, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar[B_QFULL], 1);
    mbar_init(&bar[B_KFULL], 1);
    mbar_init(&bar[B_VFULL], 1);
    mbar_init(&bar[B_KEMPTY], 1);
    mbar_init(&bar[B_VEMPTY], 1);
    mbar_init(&bar[B_SFULL], 1);
    mbar_init(&bar[B_PFULL], 128);
    mbar_init(&bar[B_OFULL], 1);
    mbar_init(&bar[B_DRAIN], 1);
    mbar_init(&bar[B_TRK0], 128);
    mbar_init(&bar[B_TRK1], 128);
    mbar_init(&bar[B_EPI0], 128);
    mbar_init(&bar[B_EPI1], 128);
    epi_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = tmem_base;        // S (fp32, 128 cols); P (bf16) in cols [0, 64)
  const uint32_t tO = tmem_base + 128;  // O (fp32, D cols)
  const int kvh = h / p.group;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.q_map);
      tma_prefetch_desc(&p.k_map);
      tma_prefetch_desc(&p.v_map);
      mbar_arrive_expect_tx(&bar[B_QFULL], kTile);
      for (int a = 0; a < kAtoms; ++a)
        tma_load_3d(sQ + a * 16384, &p.q_map, &bar[B_QFULL], a * 64, (int)(nq * 128), h);
    }
    // pull the unit's K/V tiles toward L2 ahead of their loads (single smem slots)
    for (int j = lane; j < T && j < kPrefetchTiles; j += 32) {
      const int nk = p.step_col[e0 + j];
      for (int a = 0; a < kAtoms; ++a) {
        tma_prefetch_l2_3d(&p.k_map, a * 64, nk * 128, kvh);
        tma_prefetch_l2_3d(&p.v_map, a * 64, nk * 128, kvh);
      }
    }
    int kfill = 0, vfill = 0;
    for (int j = 0; j < T; ++j) {
      const int nk = p.step_col[e0 + j];
      if (j > 0 && !warp_wait(&bar[B_KEMPTY], (j - 1) & 1, w)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar[B_KFULL], kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(sK + a * 16384, &p.k_map, &bar[B_KFULL], a * 64, nk * 128, kvh);
      }
      ++kfill;
      if (j > 0 && !warp_wait(&bar[B_VEMPTY], (j - 1) & 1, w)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar[B_VFULL], kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(sV + a * 16384, &p.v_map, &bar[B_VFULL], a * 64, nk * 128, kvh);
      }
      ++vfill;
    }
    // never leave the CTA with a copy still landing in its shared memory
    if (lane == 0) {
      drain_wait(&bar[B_QFULL], 0, p.wait_ns, p.err);
      if (kfill) drain_wait(&bar[B_KFULL], (kfill - 1) & 1, p.wait_ns, p.err);
      if (vfill) drain_wait(&bar[B_VFULL], (vfill - 1) & 1, p.wait_ns, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
      bool ok = mbar_wait(&bar[B_QFULL], 0, w);
      for (int j = 0; ok && j < T; ++j) {
        if (!mbar_wait(&bar[B_KFULL], j & 1, w)) break;
        // S/P columns are free once the previous PV has consumed P
        if (j > 0 && !mbar_wait(&bar[B_OFULL], (j - 1) & 1, w)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(tS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024), kIdS,
                 k > 0);
        }
        mma_commit(&bar[B_SFULL]);
        mma_commit(&bar[B_KEMPTY]);
        if (!mbar_wait(&bar[B_PFULL], j & 1, w)) break;
        if (!mbar_wait(&bar[B_VFULL], j & 1, w)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tO, tS + k * 8, sdesc_sw128(aV + k * 2048, 16384, 1024), kIdO,
                 (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(&bar[B_OFULL]);
        mma_commit(&bar[B_VEMPTY]);
      }
      // every MMA issued by this thread has completed before TMEM is released
      mma_commit(&bar[B_DRAIN]);
      drain_wait(&bar[B_DRAIN], 0, p.wait_ns, p.err);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax warps
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    const int64_t tq = nq * 128 + row;
    const int sq = p.tracks[tq], gq = p.tracks[n + tq], zq = p.tracks[2 * n + tq],
              pq = p.tracks[3 * n + tq];
    const float sl2 = p.scale_log2;
    const int W = p.W;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int n_partial = 0;
    for (int j = 0; j < T; ++j) {
      const bool partial = p.step_tag[e0 + j] == MARBLE_TILE_PARTIAL;
      uint32_t lm[4] = {~0u, ~0u, ~0u, ~0u};  // legal-key bits of this row in tile j
      if (partial) {
        // stage the 128 keys' tracks in one of two buffers; all 128 rows arrive before
        // any reads, so a buffer is rewritten only after every row left its last use
        const int b = n_partial & 1;
        const uint32_t par = (n_partial >> 1) & 1;
        ++n_partial;
        int32_t* kt = ktr + b * 512;
        const int64_t t = (int64_t)p.step_col[e0 + j] * 128 + row;
        kt[row] = p.tracks[t];
        kt[128 + row] = p.tracks[n + t];
        kt[256 + row] = p.tracks[2 * n + t];
        kt[384 + row] = p.tracks[3 * n + t];
        mbar_arrive(&bar[B_TRK0 + b]);
        if (!wait_all(&bar[B_TRK0 + b], par, w)) { ok = false; break; }
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t bits = 0;
#pragma unroll
          for (int t2 = 0; t2 < 32; ++t2) {
            const int kc = c * 32 + t2;
            const int dp = pq - kt[384 + kc];
            const bool legal = ((dp >= 0 && dp < W) || (gq >= 0 && gq == kt[128 + kc])) &&
                               (kt[256 + kc] < 0 || kt[256 + kc] == zq) && (kt[kc] == sq);
            bits |= (legal ? 1u : 0u) << t2;
          }
          lm[c] = bits;
        }
      }
      if (!wait_all(&bar[B_SFULL], j & 1, w)) { ok = false; break; }
      tc_fence_after();
      // pass 1: row maximum of the scaled, masked scores
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + lb + c * 32, v);
        tmem_ld_wait();
        if (partial) {
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const float s = ((lm[c] >> t) & 1u) ? __uint_as_float(v[t]) * sl2 : -INFINITY;
            mx = fmaxf(mx, s);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) mx = fmaxf(mx, __uint_as_float(v[t]) * sl2);
        }
      }
      // the running max is kept integral (base 2): every rescale factor below is then an
      // exact power of two, and bf16 rounding of P does not depend on which keys a step
      // happened to see first
      const float m_new = ceilf(mx);
      const bool grow = m_new > m_run + kRescaleThreshold;
      const bool need = grow && (m_run != -INFINITY);  // earlier tiles of this call to rescale
      const float alpha = need ? ldexpf(1.f, (int)(m_run - m_new)) : 1.f;
      if (grow) {
        l_run *= alpha;
        m_run = m_new;
      }
      // tcgen05.ld/st are warp-collective: the whole warp rescales when any of its rows
      // must (alpha = 1 on the others).  A row that needs it has a finite max from an
      // earlier tile, so j >= 1 and PV_{j-1} is the accumulation to wait for.
      if (__any_sync(0xffffffffu, need)) {
        if (!wait_all(&bar[B_OFULL], (j - 1) & 1, w)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tO + lb + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * alpha);
          tmem_st32(tO + lb + c * 32, v);
        }
      }
      // pass 2: P = exp2(s - m_run) as bf16 into TMEM over the consumed S columns
      const float base = (m_run == -INFINITY) ? 0.f : m_run;
      float rs = 0.f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + lb + c * 32, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          float s0 = __uint_as_float(v[t]) * sl2, s1 = __uint_as_float(v[t + 1]) * sl2;
          if (!((lm[c] >> t) & 1u)) s0 = -INFINITY;
          if (!((lm[c] >> (t + 1)) & 1u)) s1 = -INFINITY;
          const float p0 = fast_exp2(s0 - base), p1 = fast_exp2(s1 - base);
          rs += p0 + p1;
          pk[t >> 1] = pack_bf16(p0, p1);
        }
        tmem_st16(tS + lb + c * 16, pk);
      }
      tmem_st_wait();
      l_run += rs;
      tc_fence_before();
      mbar_arrive(&bar[B_PFULL]);
    }
    // epilogue: merge this call's (O, m, l) into the stored state through a staged tile.
    //   FIRST             the tile is stored (TMA store);
    //   otherwise         the stored max is kept unless some row's max grew past it by more
    //                     than the lazy threshold, so the update is a pure addition of
    //                     O_call * 2^(m_call - m_stored): a TMA fp32 reduce-add, no load;
    //   some row grew     exact merge with the stored tile (loaded by the row threads),
    //                     then a TMA store.
    // Q and K slots (all MMAs are done) hold the staging tile: D/32 boxes of 128 x 32 fp32.
    ok = __all_sync(0xffffffffu, ok);
    if (ok && !wait_all(&bar[B_OFULL], (T - 1) & 1, w)) ok = false;
    tc_fence_after();
    const int64_t gi = (int64_t)h * n + tq;
    float m_old = -INFINITY, l_old = 0.f;
    if (!p.first) {
      m_old = p.m[gi];
      l_old = p.l[gi];
    }
    const bool grows = !p.first && m_old != -INFINITY && m_run > m_old + kRescaleThreshold;
    if (__any_sync(0xffffffffu, grows) && lane == 0) atomicOr(&epi_flag, 1);
    mbar_arrive(&bar[B_EPI0]);
    if (ok && !wait_all(&bar[B_EPI0], 0, w)) ok = false;
    const int mode = p.first ? 0 : (epi_flag ? 2 : 1);
    uint8_t* stg = smem;
    if (ok) {
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
      }
      const float* orow = p.o_acc + (tq * p.hq + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t x[32];
        tmem_ld32(tO + lb + c * 32, x);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] = __uint_as_float(x[t]) * a_new;
        if (mode == 2) {
          const float4* src = reinterpret_cast<const float4*>(orow + c * 32);
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float4 o = src[t];
            v[4 * t] += o.x * a_old;
            v[4 * t + 1] += o.y * a_old;
            v[4 * t + 2] += o.z * a_old;
            v[4 * t + 3] += o.w * a_old;
          }
        }
        stage_row32(stg + c * 16384, row, v);
      }
      fence_proxy_async_smem();
      p.m[gi] = m_out;
      p.l[gi] = l_out;
    }
    mbar_arrive(&bar[B_EPI1]);
    if (row == 0 && ok && mbar_wait(&bar[B_EPI1], 0, w)) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        if (mode == 1)
          tma_reduce_add_3d(&p.o_map, stg + c * 16384, c * 32, (int)(nq * 128), h);
        else
          tma_store_3d(&p.o_map, stg + c * 16384, c * 32, (int)(nq * 128), h);
      }
      bulk_commit();
      bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
}

template <int D>
size_t fwd_smem() {
  // at least ~100 KB so that exactly two CTAs share an SM (two 256-column TMEM halves)
  size_t smem = 3 * (128 * D * 2) + 4096 + 1024;
  return smem < 100 * 1024 ? 100 * 1024 : smem;
}

// everything but the shard pair and the FIRST flag: encoded once per call
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
  prm->W = pl->W;
  const float scale = qkv->scale > 0.f ? qkv->scale : 1.0f / sqrtf((float)D);
  prm->scale_log2 = scale * 1.4426950408889634f;
  if (once_per_device(D == 128 ? 1 : 2)) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_fwd<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)fwd_smem<D>());
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
  const unsigned grid = (unsigned)(pl->bps * qkv->hq);
  for (int i = 0; i < n_steps; ++i) {
    FwdParams prm = base;
    prm.q_shard = q_shards[i];
    prm.kv_shard = kv_shards[i];
    prm.first = (flags[i] & MARBLE_STEP_FIRST) ? 1 : 0;
    k_attn_fwd<D><<<grid, kThreads, fwd_smem<D>(), s>>>(prm);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch k_attn_fwd");
  return MARBLE_OK;
}

}  // namespace

marble_status_t run_attn_fwd(const marble_plan_t* p, const marble_qkv_t* qkv, int n_steps,
                             const int* q_shards, const int* kv_shards, const uint32_t* flags,
                             const marble_state_t* st, cudaStream_t s) {
  if (qkv->d == 128) return launch_steps<128>(p, qkv, n_steps, q_shards, kv_shards, flags, st, s);
  if (qkv->d == 64) return launch_steps<64>(p, qkv, n_steps, q_shards, kv_shards, flags, st, s);
  return fail(MARBLE_ERR_UNSUPPORTED, "head dim must be 64 or 128");
}

}  // namespace marble
