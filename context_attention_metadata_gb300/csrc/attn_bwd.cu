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
// Two kernels, so that every accumulator has exactly one owner per launch and no atomics
// are needed (a fused kernel would scatter one fp32 dQ tile per (q, kv) tile):
//   k_bwd_dq    Q-stationary, one CTA per (q block, q head): S and dP in TMEM, dS (bf16)
//               back into TMEM over S, dQ += dS K with K read MN-major from the K tile
//               already staged for S; at the end dq_acc += scale * dQ by a TMA reduce-add.
//   k_bwd_dkdv  KV-stationary, one CTA per (kv block, kv head), looping over the q heads of
//               its group and the q blocks listed for it: S^T = K Q^T and dP^T = V dO^T in
//               TMEM, P^T and dS^T (bf16) back into TMEM, dV += P^T dO and dK += dS^T Q with
//               dO and Q read MN-major; at the end dv_acc += dV, dk_acc += scale * dK by TMA
//               reduce-adds.
// Both: warp 0 TMA producer (two stages), warp 1 TMEM allocation + MMA issue, warps 2..9
// elementwise, four warps (one thread per TMEM lane) for each 64-column half of a tile; the
// halves run as two chains offset in time so that the tensor core works on one half while
// the other half's elementwise stage runs.  Masks only on partial tiles.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tma_host.h"

namespace marble {
namespace {

constexpr int kThreads = 320;  // producer, MMA, 8 elementwise warps (2 per lane quarter)
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPrefetchTiles = 64;  // L2 prefetch depth per unit

struct BwdParams {
  CUtensorMap q_map, k_map, v_map, do_map;
  CUtensorMap dq_map, dk_map, dv_map;  // fp32 accumulators, box 32 x 128 x 1, 128-byte swizzle
  const int64_t* step_ptr;   // row lists (dQ kernel)
  const int32_t* step_col;
  const uint8_t* step_tag;
  const int64_t* colT_ptr;   // column lists (dK/dV kernel)
  const int32_t* colT_row;
  const uint8_t* colT_tag;
  const int64_t* needed_ptr;
  const int32_t* needed;
  const int32_t* tracks;     // [4][n] plan order
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
  int W;
  float scale, sl2;
};

// ======================================================================================
// dQ (Q-stationary)
// ======================================================================================
// The tile's 128 kv columns are worked as two halves (h = 0, 1) that run as two chains
// offset in time: while the elementwise warps of one half compute dS, the tensor core runs
// the other half's MMAs.  Per tile j and half h:
//   S_h = Q K_h^T and dP_h = dO V_h^T (N = 64)  ->  elementwise: dS_h (bf16) over S_h
//   ->  dQ += dS_h K_h (K = 64).
// S alternates between two TMEM buffers by tile, so S_h(j+1) never overwrites the dS_h(j)
// that dQ_h(j) reads; dP has one buffer, rewritten once the elementwise has loaded it.
enum { Q_QFULL, Q_KVFULL0, Q_KVFULL1, Q_KVEMPTY0, Q_KVEMPTY1, Q_SFULL0, Q_SFULL1, Q_PFULL0,
       Q_PFULL1, Q_DQDONE0, Q_DQDONE1, Q_DRAIN, Q_TRK00, Q_TRK01, Q_TRK10, Q_TRK11, Q_EPI,
       Q_NUM };

template <int D>
__global__ void __launch_bounds__(kThreads, 1) k_bwd_dq(const __grid_constant__ BwdParams p) {
  constexpr int kTile = 128 * D * 2;
  constexpr int kAtoms = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + kTile;
  uint8_t* sK0 = smem + 2 * kTile;  // stage s: K at 2+2s, V at 3+2s
  int32_t* ktr = reinterpret_cast<int32_t*>(smem + 6 * kTile);  // [half][buffer][4][64]
  __shared__ __align__(8) uint64_t bar[Q_NUM];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

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
  if (T == 0) return;

  WaitCtx w{p.wait_ns, p.err, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int b = 0; b < Q_NUM; ++b) {
      const int cnt = (b == Q_EPI) ? 256
                      : (b == Q_PFULL0 || b == Q_PFULL1 || b == Q_TRK00 || b == Q_TRK01 ||
                         b == Q_TRK10 || b == Q_TRK11)
                          ? 128
                          : 1;
      mbar_init(&bar[b], cnt);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // S buffers fp32 at [0,128) (even tiles) and [384,512) (odd tiles); dS_h bf16 is packed into
  // columns [64h, 64h + 32) of its S buffer, inside the fp32 columns half h has read.
  // dP fp32 [128,256); dQ fp32 [256, 256+D).
  const uint32_t tS0 = tmem_base, tS1 = tmem_base + 384;
  const uint32_t tP = tmem_base + 128;
  const uint32_t tQ = tmem_base + 256;
  const int kvh = h / p.group;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.q_map);
      tma_prefetch_desc(&p.k_map);
      tma_prefetch_desc(&p.v_map);
      tma_prefetch_desc(&p.do_map);
      mbar_arrive_expect_tx(&bar[Q_QFULL], 2 * kTile);
      for (int a = 0; a < kAtoms; ++a) {
        tma_load_3d(sQ + a * 16384, &p.q_map, &bar[Q_QFULL], a * 64, (int)(nq * 128), h);
        tma_load_3d(sDO + a * 16384, &p.do_map, &bar[Q_QFULL], a * 64, (int)(nq * 128), h);
      }
    }
    int fills[2] = {0, 0};
    for (int j = 0; j < T; ++j) {
      const int s = j & 1;
      if (j >= 2 && !warp_wait(&bar[Q_KVEMPTY0 + s], ((j >> 1) - 1) & 1, w)) break;
      const int nk = p.step_col[e0 + j];
      if (lane == 0) {
        uint8_t* sK = sK0 + s * 2 * kTile;
        uint8_t* sV = sK + kTile;
        mbar_arrive_expect_tx(&bar[Q_KVFULL0 + s], 2 * kTile);
        for (int a = 0; a < kAtoms; ++a) {
          tma_load_3d(sK + a * 16384, &p.k_map, &bar[Q_KVFULL0 + s], a * 64, nk * 128, kvh);
          tma_load_3d(sV + a * 16384, &p.v_map, &bar[Q_KVFULL0 + s], a * 64, nk * 128, kvh);
        }
      }
      ++fills[s];
      if (j == 1) {
        // pull the later K/V tiles toward L2 once the first two loads are queued
        for (int jj = 2 + lane; jj < T && jj < kPrefetchTiles; jj += 32) {
          const int nkk = p.step_col[e0 + jj];
          for (int a = 0; a < kAtoms; ++a) {
            tma_prefetch_l2_3d(&p.k_map, a * 64, nkk * 128, kvh);
            tma_prefetch_l2_3d(&p.v_map, a * 64, nkk * 128, kvh);
          }
        }
      }
    }
    if (lane == 0) {
      drain_wait(&bar[Q_QFULL], 0, p.wait_ns, p.err);
      for (int s = 0; s < 2; ++s)
        if (fills[s]) drain_wait(&bar[Q_KVFULL0 + s], (fills[s] - 1) & 1, p.wait_ns, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 64, false, false);
      constexpr uint32_t kIdQ = idesc_bf16(128, D, false, true);
      const uint32_t aQ = smem_u32(sQ), aDO = smem_u32(sDO);
      // S_hh(jj) and dP_hh(jj): kv rows [64 hh, 64 hh + 64) of stage jj & 1
      auto issue_s = [&](int jj, int hh) {
        const uint32_t aK = smem_u32(sK0 + (jj & 1) * 2 * kTile) + hh * 8192, aV = aK + kTile;
        const uint32_t ts = ((jj & 1) ? tS1 : tS0) + hh * 64;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(ts, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024), kIdS,
                 k > 0);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(tP + hh * 64, sdesc_sw128(aDO + off, 16, 1024), sdesc_sw128(aV + off, 16, 1024),
                 kIdS, k > 0);
        }
        mma_commit(&bar[Q_SFULL0 + hh]);
      };
      bool ok = mbar_wait(&bar[Q_QFULL], 0, w) && mbar_wait(&bar[Q_KVFULL0], 0, w);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(0, 1);
      }
      for (int j = 0; ok && j < T; ++j) {
        const int s = j & 1;
        const bool nxt = j + 1 < T;
        if (nxt && !mbar_wait(&bar[Q_KVFULL0 + ((j + 1) & 1)], ((j + 1) >> 1) & 1, w)) break;
        for (int hh = 0; hh < 2; ++hh) {
          if (!mbar_wait(&bar[Q_PFULL0 + hh], j & 1, w)) { ok = false; break; }
          // S_hh(j+1) goes to the buffer dQ_hh(j-1) read: wait for it before dQ_hh(j) is
          // issued, so that the wait is on the phase just before the one in flight
          if (nxt && j >= 1 && !mbar_wait(&bar[Q_DQDONE0 + hh], (j - 1) & 1, w)) { ok = false; break; }
          tc_fence_after();
          const uint32_t aK = smem_u32(sK0 + s * 2 * kTile);
          const uint32_t ts = (s ? tS1 : tS0) + hh * 64;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tQ, ts + kk * 8, sdesc_sw128(aK + (4 * hh + kk) * 2048, 16384, 1024), kIdQ,
                   (j > 0 || hh > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar[Q_DQDONE0 + hh]);
          if (hh == 1) mma_commit(&bar[Q_KVEMPTY0 + s]);
          if (nxt) issue_s(j + 1, hh);
        }
      }
      mma_commit(&bar[Q_DRAIN]);
      drain_wait(&bar[Q_DRAIN], 0, p.wait_ns, p.err);
    }
    __syncwarp();
  } else {
    // four warps per half: `half` owns kv columns [64 half, 64 half + 64), one row a thread
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const int hr = row & 63;  // this thread's share of the half's key tracks
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    const int64_t tq = nq * 128 + row;
    const int sq = p.tracks[tq], gq = p.tracks[n + tq], zq = p.tracks[2 * n + tq],
              pq = p.tracks[3 * n + tq];
    float lse2 = p.lse[(int64_t)h * n + tq] * kLog2e;
    if (lse2 == -INFINITY) lse2 = INFINITY;  // a row with no legal key: every P is 0
    const float dlt = p.delta[(int64_t)h * n + tq];
    const float sl2 = p.sl2;
    bool ok = true;
    int n_partial = 0;
    for (int j = 0; j < T; ++j) {
      const bool partial = p.step_tag[e0 + j] == MARBLE_TILE_PARTIAL;
      uint32_t lm[2] = {~0u, ~0u};  // legal-key bits of this row in this half's 64 columns
      if (partial) {
        // the half's 64 keys' tracks, two per thread, in one of two buffers
        const int b = n_partial & 1;
        const uint32_t par = (n_partial >> 1) & 1;
        ++n_partial;
        int32_t* kt = ktr + (half * 2 + b) * 256;
        const int64_t t = (int64_t)p.step_col[e0 + j] * 128 + half * 64 + hr;
        const int tr0 = (row >> 6) * 2;  // tracks tr0, tr0 + 1
        kt[tr0 * 64 + hr] = p.tracks[tr0 * n + t];
        kt[(tr0 + 1) * 64 + hr] = p.tracks[(tr0 + 1) * n + t];
        mbar_arrive(&bar[Q_TRK00 + half * 2 + b]);
        if (!wait_all(&bar[Q_TRK00 + half * 2 + b], par, w)) { ok = false; break; }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t bits = 0;
#pragma unroll
          for (int t2 = 0; t2 < 32; ++t2) {
            const int kc = cc * 32 + t2;
            bits |= (mask_legal(sq, gq, zq, pq, kt[kc], kt[64 + kc], kt[128 + kc], kt[192 + kc],
                                p.W) ? 1u : 0u) << t2;
          }
          lm[cc] = bits;
        }
      }
      if (!wait_all(&bar[Q_SFULL0 + half], j & 1, w)) { ok = false; break; }
      tc_fence_after();
      const uint32_t ts = ((j & 1) ? tS1 : tS0) + half * 64;
      uint32_t vs[2][32], vp[2][32];
      tmem_ld32(ts + lb, vs[0]);
      tmem_ld32(ts + lb + 32, vs[1]);
      tmem_ld32(tP + lb + half * 64, vp[0]);
      tmem_ld32(tP + lb + half * 64 + 32, vp[1]);
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          const bool l0 = (lm[cc] >> t) & 1u, l1 = (lm[cc] >> (t + 1)) & 1u;
          const float p0 = l0 ? fast_exp2(__uint_as_float(vs[cc][t]) * sl2 - lse2) : 0.f;
          const float p1 = l1 ? fast_exp2(__uint_as_float(vs[cc][t + 1]) * sl2 - lse2) : 0.f;
          const float d0 = p0 * (__uint_as_float(vp[cc][t]) - dlt);
          const float d1 = p1 * (__uint_as_float(vp[cc][t + 1]) - dlt);
          pk[t >> 1] = pack_bf16(d0, d1);
        }
        tmem_st16(ts + lb + cc * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[Q_PFULL0 + half]);
    }
    // epilogue: dq_acc += scale * dQ as a TMA fp32 reduce-add of a tile staged in the Q/dO
    // slots (all MMAs are done), D/32 boxes of 128 x 32 fp32: no load of dq_acc.  The MMA
    // thread's final commit has one phase, so it is safe to wait on from either half (a
    // per-tile barrier could be two phases behind while the other half is still working).
    ok = __all_sync(0xffffffffu, ok);
    if (ok && !wait_all(&bar[Q_DRAIN], 0, w)) ok = false;
    tc_fence_after();
    uint8_t* stg = smem;
    if (ok) {
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        uint32_t x[32];
        tmem_ld32(tQ + lb + c * 32, x);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] = p.scale * __uint_as_float(x[t]);
        stage_row32(stg + c * 16384, row, v);
      }
      fence_proxy_async_smem();
    }
    mbar_arrive(&bar[Q_EPI]);
    if (row == 0 && half == 0 && ok && mbar_wait(&bar[Q_EPI], 0, w)) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c)
        tma_reduce_add_3d(&p.dq_map, stg + c * 16384, c * 32, (int)(nq * 128), h);
      bulk_commit();
      bulk_wait_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ======================================================================================
// dK / dV (KV-stationary)
// ======================================================================================
// As in the dQ kernel, the item's 128 q columns are worked as two halves that run as two
// chains offset in time.  Per item j and half h:
//   S^T_h = K Q_h^T and dP^T_h = V dO_h^T (N = 64)  ->  elementwise: P^T_h and dS^T_h (bf16)
//   over them  ->  dV += P^T_h dO_h and dK += dS^T_h Q_h (K = 64).
// With dV and dK resident, TMEM holds one S^T / dP^T buffer: S^T_h(j+1) is issued once the
// MMAs of half h of item j have completed, while the other half's elementwise runs.
enum { K_KVFULL, K_QFULL0, K_QFULL1, K_QEMPTY0, K_QEMPTY1, K_SFULL0, K_SFULL1, K_PFULL0,
       K_PFULL1, K_CONS0, K_CONS1, K_DRAIN, K_TRK00, K_TRK01, K_TRK10, K_TRK11, K_EPI, K_NUM };

template <int D>
__global__ void __launch_bounds__(kThreads, 1) k_bwd_dkdv(const __grid_constant__ BwdParams p) {
  constexpr int kTile = 128 * D * 2;
  constexpr int kAtoms = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sK = smem;
  uint8_t* sV = smem + kTile;
  uint8_t* sQ0 = smem + 2 * kTile;  // stage s: Q at 2+2s, dO at 3+2s
  // per half and buffer: lse2[64] | delta[64] | tracks [4][64]
  float* stg = reinterpret_cast<float*>(smem + 6 * kTile);
  __shared__ __align__(8) uint64_t bar[K_NUM];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long n = p.n;
  int64_t nk;
  int kh;
  if (p.kv_shard >= 0) {
    kh = blockIdx.x / p.bps;
    nk = (int64_t)p.kv_shard * p.bps + blockIdx.x % p.bps;
  } else {
    const int64_t cnt = p.needed_ptr[p.q_shard + 1] - p.needed_ptr[p.q_shard];
    kh = (int)(blockIdx.x / cnt);
    nk = p.needed[p.needed_ptr[p.q_shard] + blockIdx.x % cnt];
  }
  const int64_t c0 = p.colT_ptr[nk * p.P + p.q_shard];
  const int L = (int)(p.colT_ptr[nk * p.P + p.q_shard + 1] - c0);
  const int T = L * p.group;  // items: (q head of the group, listed q block)
  if (T == 0) return;

  WaitCtx w{p.wait_ns, p.err, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int b = 0; b < K_NUM; ++b) {
      const int cnt = (b == K_EPI) ? 256
                      : (b == K_PFULL0 || b == K_PFULL1 || b == K_TRK00 || b == K_TRK01 ||
                         b == K_TRK10 || b == K_TRK11)
                          ? 128
                          : 1;
      mbar_init(&bar[b], cnt);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // S^T fp32 [0,128) and dP^T fp32 [128,256), half h in columns [64h, 64h + 64) of each;
  // P^T_h / dS^T_h bf16 packed into columns [64h, 64h + 32) of the same region
  const uint32_t tS = tmem_base;
  const uint32_t tP = tmem_base + 128;
  const uint32_t tdV = tmem_base + 256;   // dV fp32 [256, 256+D)
  const uint32_t tdK = tmem_base + 384;   // dK fp32 [384, 384+D)

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.q_map);
      tma_prefetch_desc(&p.k_map);
      tma_prefetch_desc(&p.v_map);
      tma_prefetch_desc(&p.do_map);
      mbar_arrive_expect_tx(&bar[K_KVFULL], 2 * kTile);
      for (int a = 0; a < kAtoms; ++a) {
        tma_load_3d(sK + a * 16384, &p.k_map, &bar[K_KVFULL], a * 64, (int)(nk * 128), kh);
        tma_load_3d(sV + a * 16384, &p.v_map, &bar[K_KVFULL], a * 64, (int)(nk * 128), kh);
      }
    }
    int fills[2] = {0, 0};
    for (int it = 0; it < T; ++it) {
      const int s = it & 1;
      if (it >= 2 && !warp_wait(&bar[K_QEMPTY0 + s], ((it >> 1) - 1) & 1, w)) break;
      const int h = kh * p.group + it / L;
      const int nqb = p.colT_row[c0 + it % L];
      if (lane == 0) {
        uint8_t* sQ = sQ0 + s * 2 * kTile;
        uint8_t* sDO = sQ + kTile;
        mbar_arrive_expect_tx(&bar[K_QFULL0 + s], 2 * kTile);
        for (int a = 0; a < kAtoms; ++a) {
          tma_load_3d(sQ + a * 16384, &p.q_map, &bar[K_QFULL0 + s], a * 64, nqb * 128, h);
          tma_load_3d(sDO + a * 16384, &p.do_map, &bar[K_QFULL0 + s], a * 64, nqb * 128, h);
        }
      }
      ++fills[s];
      if (it == 1) {
        // pull the later items' Q/dO tiles toward L2 once the first two loads are queued
        for (int i2 = 2 + lane; i2 < T && i2 < kPrefetchTiles; i2 += 32) {
          const int h2 = kh * p.group + i2 / L;
          const int nq2 = p.colT_row[c0 + i2 % L];
          for (int a = 0; a < kAtoms; ++a) {
            tma_prefetch_l2_3d(&p.q_map, a * 64, nq2 * 128, h2);
            tma_prefetch_l2_3d(&p.do_map, a * 64, nq2 * 128, h2);
          }
        }
      }
    }
    if (lane == 0) {
      drain_wait(&bar[K_KVFULL], 0, p.wait_ns, p.err);
      for (int s = 0; s < 2; ++s)
        if (fills[s]) drain_wait(&bar[K_QFULL0 + s], (fills[s] - 1) & 1, p.wait_ns, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 64, false, false);
      constexpr uint32_t kIdAcc = idesc_bf16(128, D, false, true);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      // S^T_hh(it) and dP^T_hh(it): q rows [64 hh, 64 hh + 64) of stage it & 1
      auto issue_s = [&](int it, int hh) {
        const uint32_t aQ = smem_u32(sQ0 + (it & 1) * 2 * kTile) + hh * 8192, aDO = aQ + kTile;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(tS + hh * 64, sdesc_sw128(aK + off, 16, 1024), sdesc_sw128(aQ + off, 16, 1024),
                 kIdS, k > 0);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(tP + hh * 64, sdesc_sw128(aV + off, 16, 1024), sdesc_sw128(aDO + off, 16, 1024),
                 kIdS, k > 0);
        }
        mma_commit(&bar[K_SFULL0 + hh]);
      };
      bool ok = mbar_wait(&bar[K_KVFULL], 0, w) && mbar_wait(&bar[K_QFULL0], 0, w);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(0, 1);
      }
      for (int it = 0; ok && it < T; ++it) {
        const int s = it & 1;
        const bool nxt = it + 1 < T;
        if (nxt && !mbar_wait(&bar[K_QFULL0 + ((it + 1) & 1)], ((it + 1) >> 1) & 1, w)) break;
        const uint32_t aQ = smem_u32(sQ0 + s * 2 * kTile), aDO = aQ + kTile;
        for (int hh = 0; hh < 2; ++hh) {
          if (!mbar_wait(&bar[K_PFULL0 + hh], it & 1, w)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tdV, tS + hh * 64 + kk * 8,
                   sdesc_sw128(aDO + (4 * hh + kk) * 2048, 16384, 1024), kIdAcc,
                   (it > 0 || hh > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tdK, tP + hh * 64 + kk * 8,
                   sdesc_sw128(aQ + (4 * hh + kk) * 2048, 16384, 1024), kIdAcc,
                   (it > 0 || hh > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar[K_CONS0 + hh]);
          if (hh == 1) mma_commit(&bar[K_QEMPTY0 + s]);
          if (nxt) {
            // half hh of the S^T / dP^T buffer is free once these MMAs have read P^T / dS^T
            if (!mbar_wait(&bar[K_CONS0 + hh], it & 1, w)) { ok = false; break; }
            tc_fence_after();
            issue_s(it + 1, hh);
          }
        }
      }
      mma_commit(&bar[K_DRAIN]);
      drain_wait(&bar[K_DRAIN], 0, p.wait_ns, p.err);
    }
    __syncwarp();
  } else {
    // four warps per half: `half` owns q columns [64 half, 64 half + 64), one kv row a thread
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;  // kv row of the tile
    const int hr = row & 63;
    const uint32_t lb = (uint32_t)(quarter * 32) << 16;
    const int64_t tk = nk * 128 + row;
    const int sk = p.tracks[tk], gk = p.tracks[n + tk], zk = p.tracks[2 * n + tk],
              pk = p.tracks[3 * n + tk];
    const float sl2 = p.sl2;
    bool ok = true;
    for (int it = 0; it < T; ++it) {
      const int h = kh * p.group + it / L;
      const int64_t e = c0 + it % L;
      const int64_t qrow = (int64_t)p.colT_row[e] * 128 + half * 64 + hr;
      const bool partial = p.colT_tag[e] == MARBLE_TILE_PARTIAL;
      // stage this half's per-query LSE (base 2), delta and, on partial tiles, tracks: the
      // first 64 threads of the half the two floats, the other 64 the four tracks
      const int b = it & 1;
      float* lse2s = stg + (half * 2 + b) * 384;
      float* dls = lse2s + 64;
      int32_t* qt = reinterpret_cast<int32_t*>(lse2s + 128);
      if ((row >> 6) == 0) {
        const float l2 = p.lse[(int64_t)h * n + qrow] * kLog2e;
        lse2s[hr] = (l2 == -INFINITY) ? INFINITY : l2;
        dls[hr] = p.delta[(int64_t)h * n + qrow];
      } else if (partial) {
        qt[hr] = p.tracks[qrow];
        qt[64 + hr] = p.tracks[n + qrow];
        qt[128 + hr] = p.tracks[2 * n + qrow];
        qt[192 + hr] = p.tracks[3 * n + qrow];
      }
      mbar_arrive(&bar[K_TRK00 + half * 2 + b]);
      if (!wait_all(&bar[K_TRK00 + half * 2 + b], (it >> 1) & 1, w)) { ok = false; break; }
      uint32_t lm[2] = {~0u, ~0u};
      if (partial) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t bits = 0;
#pragma unroll
          for (int t2 = 0; t2 < 32; ++t2) {
            const int q = cc * 32 + t2;
            bits |= (mask_legal(qt[q], qt[64 + q], qt[128 + q], qt[192 + q], sk, gk, zk, pk,
                                p.W) ? 1u : 0u) << t2;
          }
          lm[cc] = bits;
        }
      }
      if (!wait_all(&bar[K_SFULL0 + half], it & 1, w)) { ok = false; break; }
      tc_fence_after();
      uint32_t vs[2][32], vp[2][32];
      tmem_ld32(tS + lb + half * 64, vs[0]);
      tmem_ld32(tS + lb + half * 64 + 32, vs[1]);
      tmem_ld32(tP + lb + half * 64, vp[0]);
      tmem_ld32(tP + lb + half * 64 + 32, vp[1]);
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t pk16[16], dk16[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          const int q0 = cc * 32 + t;
          const bool l0 = (lm[cc] >> t) & 1u, l1 = (lm[cc] >> (t + 1)) & 1u;
          const float p0 = l0 ? fast_exp2(__uint_as_float(vs[cc][t]) * sl2 - lse2s[q0]) : 0.f;
          const float p1 =
              l1 ? fast_exp2(__uint_as_float(vs[cc][t + 1]) * sl2 - lse2s[q0 + 1]) : 0.f;
          const float d0 = p0 * (__uint_as_float(vp[cc][t]) - dls[q0]);
          const float d1 = p1 * (__uint_as_float(vp[cc][t + 1]) - dls[q0 + 1]);
          pk16[t >> 1] = pack_bf16(p0, p1);
          dk16[t >> 1] = pack_bf16(d0, d1);
        }
        tmem_st16(tS + lb + half * 64 + cc * 16, pk16);
        tmem_st16(tP + lb + half * 64 + cc * 16, dk16);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[K_PFULL0 + half]);
    }
    // epilogue: dv_acc += dV and dk_acc += scale * dK as TMA fp32 reduce-adds of tiles staged
    // in the K/V and first Q/dO slots (all MMAs are done): no load of the accumulators.  The
    // MMA thread's final commit has one phase, so it is safe to wait on from either half.
    ok = __all_sync(0xffffffffu, ok);
    if (ok && !wait_all(&bar[K_DRAIN], 0, w)) ok = false;
    tc_fence_after();
    uint8_t* stv = smem;
    uint8_t* stk = smem + (D / 32) * 16384;
    if (ok) {
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        uint32_t xv[32], xk[32];
        tmem_ld32(tdV + lb + c * 32, xv);
        tmem_ld32(tdK + lb + c * 32, xk);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] = __uint_as_float(xv[t]);
        stage_row32(stv + c * 16384, row, v);
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] = p.scale * __uint_as_float(xk[t]);
        stage_row32(stk + c * 16384, row, v);
      }
      fence_proxy_async_smem();
    }
    mbar_arrive(&bar[K_EPI]);
    if (row == 0 && half == 0 && ok && mbar_wait(&bar[K_EPI], 0, w)) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        tma_reduce_add_3d(&p.dv_map, stv + c * 16384, c * 32, (int)(nk * 128), kh);
        tma_reduce_add_3d(&p.dk_map, stk + c * 16384, c * 32, (int)(nk * 128), kh);
      }
      bulk_commit();
      bulk_wait_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int D>
size_t bwd_smem() {
  // one CTA per SM: each CTA owns all 512 TMEM columns
  size_t smem = 6 * (128 * D * 2) + 2 * 2 * 384 * 4 + 1024;
  return smem < 120 * 1024 ? 120 * 1024 : smem;
}

template <int D>
marble_status_t launch_steps(const marble_plan_t* pl, const marble_qkv_t* qkv, const void* d_o,
                             const float* lse, const float* delta, int n_steps,
                             const int* q_shards, const int* kv_shards, float* dq, float* dk,
                             float* dv, cudaStream_t s) {
  BwdParams prm;
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
  const size_t smem = bwd_smem<D>();
  if (once_per_device(D == 128 ? 3 : 4)) {
    cudaError_t e = cudaFuncSetAttribute(k_bwd_dq<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_bwd_dkdv<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd)");
  }
  for (int i = 0; i < n_steps; ++i) {
    prm.q_shard = q_shards[i];
    prm.kv_shard = kv_shards[i];
    k_bwd_dq<D><<<(unsigned)(pl->bps * qkv->hq), kThreads, smem, s>>>(prm);
    int64_t units;
    if (prm.kv_shard >= 0)
      units = pl->bps * qkv->hkv;
    else
      units = (pl->h_needed_ptr[prm.q_shard + 1] - pl->h_needed_ptr[prm.q_shard]) * qkv->hkv;
    if (units > 0) k_bwd_dkdv<D><<<(unsigned)units, kThreads, smem, s>>>(prm);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch of the backward kernels");
  return MARBLE_OK;
}

}  // namespace

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
