// Mask-metadata -> tile map planner, token order and per-step tile lists, all on device.
//
// MARBLE post, s03 "Block classification": per 128-token block, cheap summaries (min/max
// of every track and a small segment bitmap) let one test per block pair decide whether
// the pair is full (provably all legal), empty (provably none legal) or partial.  s03
// "PTRR": sort query blocks by cost, deal them to ranks in rounds of R with every other
// round reversed, keep each rank's blocks in sequence order.  s03 "Chunked ring
// attention": PTRR's rule over contiguous chunks.  s04 "Sparse all-to-all": the key/value
// blocks each rank's queries need.  s04 "Layout transforms": tokens are permuted once and
// carry their metadata and original position.
//
// The candidate band: sample ids are non-decreasing along the pack, so every block
// outside [first block whose max sample >= this block's min sample, last block whose min
// sample <= this block's max sample] has a disjoint sample range and is empty by the
// sample test; classification only visits the band.
#include <algorithm>
#include <climits>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace marble {
namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ------------------------------------------------------------------------------------
// a1 + a2: validation and block summaries (one warp per block, 4 tokens per lane)
// ------------------------------------------------------------------------------------
__global__ void k_summaries(const int32_t* __restrict__ sample, const int32_t* __restrict__ seg,
                            const int32_t* __restrict__ noise, const int32_t* __restrict__ pos,
                            int64_t nb, Summary* __restrict__ out, unsigned* err) {
  const int lane = threadIdx.x & 31;
  const int64_t b = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (b >= nb) return;
  const int64_t t0 = b * kBlock + lane * 4;
  int slo = INT_MAX, shi = INT_MIN, nlo = INT_MAX, nhi = INT_MIN, glo = INT_MAX, ghi = -1;
  int plo = INT_MAX, phi = INT_MIN;  // positions: the index unless a position track is given
  unsigned blo = 0, bhi = 0;
  bool any_seg = false, all_seg = true, bad = false;
  int prev = t0 > 0 ? sample[t0 - 1] : INT_MIN;
  for (int i = 0; i < 4; ++i) {
    const int s = sample[t0 + i], g = seg[t0 + i], z = noise[t0 + i];
    const int ps = pos ? pos[t0 + i] : (int)(t0 + i);
    bad |= (s < 0) | (g < -1) | (z < -1) | (s < prev) | (ps < 0);
    plo = min(plo, ps);
    phi = max(phi, ps);
    prev = s;
    slo = min(slo, s); shi = max(shi, s);
    nlo = min(nlo, z); nhi = max(nhi, z);
    if (g >= 0) {
      any_seg = true;
      glo = min(glo, g); ghi = max(ghi, g);
      const int bit = g & 63;
      if (bit < 32) blo |= 1u << bit; else bhi |= 1u << (bit - 32);
    } else {
      all_seg = false;
    }
  }
  const unsigned full = 0xffffffffu;
  slo = __reduce_min_sync(full, slo); shi = __reduce_max_sync(full, shi);
  nlo = __reduce_min_sync(full, nlo); nhi = __reduce_max_sync(full, nhi);
  glo = __reduce_min_sync(full, glo); ghi = __reduce_max_sync(full, ghi);
  plo = __reduce_min_sync(full, plo); phi = __reduce_max_sync(full, phi);
  blo = __reduce_or_sync(full, blo); bhi = __reduce_or_sync(full, bhi);
  const bool has = __any_sync(full, any_seg);
  const bool all = __all_sync(full, all_seg);
  if (__any_sync(full, bad) && lane == 0) atomicOr(err, kErrBadTracks);
  if (lane == 0) {
    Summary r;
    r.slo = slo; r.shi = shi; r.nlo = nlo; r.nhi = nhi; r.glo = glo; r.ghi = ghi;
    r.plo = plo; r.phi = phi;
    r.gbits = ((unsigned long long)bhi << 32) | blo;
    r.flags = (has ? 1 : 0) | (all ? 2 : 0);
    r.pad = 0;
    out[b] = r;
  }
}

// candidate band [lo, hi] of every block by binary search over the non-decreasing
// per-block sample bounds
__global__ void k_band(const Summary* __restrict__ s, int64_t nb, int32_t* __restrict__ band) {
  const int64_t a = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (a >= nb) return;
  const int slo = s[a].slo, shi = s[a].shi;
  int64_t lo = 0, hi = a;  // first b with s[b].shi >= slo (b <= a holds)
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (s[mid].shi >= slo) hi = mid; else lo = mid + 1;
  }
  band[2 * a] = (int32_t)lo;
  lo = a; hi = nb;  // first b with s[b].slo > shi
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (s[mid].slo > shi) hi = mid; else lo = mid + 1;
  }
  band[2 * a + 1] = (int32_t)(lo - 1);
}

// a3: the summary rule (full = 1, partial = 2, empty = 0) for q block A, k block B
__device__ __forceinline__ int classify(const Summary& A, const Summary& B, int W) {
  const bool samp_all = A.slo == A.shi && A.shi == B.slo && B.slo == B.shi;
  const bool samp_none = A.shi < B.slo || B.shi < A.slo;
  const bool caus_all = (A.plo - B.phi >= 0) && (A.phi - B.plo < W);
  const bool caus_none = (A.phi - B.plo < 0) || (A.plo - B.phi >= W);
  const bool hasA = A.flags & 1, hasB = B.flags & 1;
  const bool allA = A.flags & 2, allB = B.flags & 2;
  const bool span_all = allA && allB && A.glo == A.ghi && A.ghi == B.glo && B.glo == B.ghi;
  const bool span_none =
      !hasA || !hasB || (A.gbits & B.gbits) == 0ull || A.ghi < B.glo || B.ghi < A.glo;
  const bool noise_all =
      B.nhi < 0 || (A.nlo == A.nhi && A.nhi == B.nlo && B.nlo == B.nhi && B.nhi >= 0);
  const bool noise_none = B.nlo >= 0 && (A.nhi < B.nlo || B.nhi < A.nlo);
  if (samp_none || noise_none || (caus_none && span_none)) return 0;
  if (samp_all && noise_all && (caus_all || span_all)) return MARBLE_TILE_FULL;
  return MARBLE_TILE_PARTIAL;
}

// one warp per q block: count non-empty tiles of the row
__global__ void k_tiles_count(const Summary* __restrict__ s, const int32_t* __restrict__ band,
                              int64_t nb, int W, int32_t* __restrict__ cnt) {
  const int lane = threadIdx.x & 31;
  const int64_t a = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (a >= nb) return;
  const Summary A = s[a];
  const int lo = band[2 * a], hi = band[2 * a + 1];
  int c = 0;
  for (int b0 = lo; b0 <= hi; b0 += 32) {
    const int b = b0 + lane;
    const int t = b <= hi ? classify(A, s[b], W) : 0;
    c += __popc(__ballot_sync(0xffffffffu, t != 0));
  }
  if (lane == 0) cnt[a] = c;
}

// one warp per q block: write the row's tiles in ascending kv block order
__global__ void k_tiles_write(const Summary* __restrict__ s, const int32_t* __restrict__ band,
                              const int64_t* __restrict__ row_ptr, int64_t nb, int W,
                              int32_t* __restrict__ col, uint8_t* __restrict__ tag) {
  const int lane = threadIdx.x & 31;
  const int64_t a = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (a >= nb) return;
  const Summary A = s[a];
  const int lo = band[2 * a], hi = band[2 * a + 1];
  int64_t out = row_ptr[a];
  for (int b0 = lo; b0 <= hi; b0 += 32) {
    const int b = b0 + lane;
    const int t = b <= hi ? classify(A, s[b], W) : 0;
    const unsigned m = __ballot_sync(0xffffffffu, t != 0);
    if (t) {
      const int64_t o = out + __popc(m & lanemask_lt());
      col[o] = b;
      tag[o] = (uint8_t)t;
    }
    out += __popc(m);
  }
}

// exclusive scan of n counters into out[0..n] (out[n] = total); one CTA, each thread owns
// a contiguous chunk
template <typename T>
__global__ void k_scan(const T* __restrict__ in, int64_t n, int64_t* __restrict__ out) {
  __shared__ int64_t ws[32];
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, wid = tid >> 5;
  const int64_t per = (n + nt - 1) / nt;
  const int64_t a = min(n, (int64_t)tid * per), b = min(n, a + per);
  int64_t sum = 0;
  for (int64_t i = a; i < b; ++i) sum += (int64_t)in[i];
  int64_t x = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int64_t y = lane < (nt >> 5) ? ws[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    ws[lane] = y;
  }
  __syncthreads();
  int64_t run = (wid ? ws[wid - 1] : 0) + x - sum;
  for (int64_t i = a; i < b; ++i) {
    out[i] = run;
    run += (int64_t)in[i];
  }
  if (tid == nt - 1) out[n] = run;
}

// ------------------------------------------------------------------------------------
// a4: order
// ------------------------------------------------------------------------------------
__global__ void k_unit_cost(const int32_t* __restrict__ cnt, int ub, int64_t units,
                            int32_t* __restrict__ ucost) {
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  int c = 0;
  for (int i = 0; i < ub; ++i) c += cnt[u * ub + i];
  ucost[u] = c;
}

// PTRR rank of every unit: its position in the (cost desc, index asc) order decides the
// round t and slot i; even rounds deal slots to ranks 0..P-1, odd rounds to P-1..0.
__global__ void k_ptrr_rank(const int32_t* __restrict__ ucost, int64_t U, int P,
                            int32_t* __restrict__ rank_of) {
  __shared__ int32_t tile[1024];
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int cu = u < U ? ucost[u] : 0;
  int64_t pos = 0;
  for (int64_t v0 = 0; v0 < U; v0 += 1024) {
    __syncthreads();
    for (int i = threadIdx.x; i < 1024; i += blockDim.x)
      tile[i] = (v0 + i < U) ? ucost[v0 + i] : INT_MIN;
    __syncthreads();
    const int lim = (int)min((int64_t)1024, U - v0);
    for (int i = 0; i < lim; ++i) {
      const int cv = tile[i];
      pos += (cv > cu) || (cv == cu && v0 + i < u);
    }
  }
  if (u < U) {
    const int64_t t = pos / P, i = pos % P;
    rank_of[u] = (int32_t)((t & 1) ? (P - 1 - i) : i);
  }
}

// slot of every unit inside its rank: ascending unit index
__global__ void k_ptrr_place(const int32_t* __restrict__ rank_of, int64_t U, int P,
                             int32_t* __restrict__ unit_new) {
  __shared__ int32_t tile[1024];
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int ru = u < U ? rank_of[u] : -1;
  int64_t idx = 0;
  const int64_t last = min(U, ((int64_t)blockIdx.x + 1) * blockDim.x);
  for (int64_t v0 = 0; v0 < last; v0 += 1024) {
    __syncthreads();
    for (int i = threadIdx.x; i < 1024; i += blockDim.x)
      tile[i] = (v0 + i < U) ? rank_of[v0 + i] : -2;
    __syncthreads();
    const int lim = (int)min((int64_t)1024, U - v0);
    for (int i = 0; i < lim; ++i) idx += (v0 + i < u) && (tile[i] == ru);
  }
  if (u < U) unit_new[u] = (int32_t)((int64_t)ru * (U / P) + idx);
}

__global__ void k_block_perm(const int32_t* __restrict__ unit_new, int ub, int64_t nb,
                             int32_t* __restrict__ block_perm, int32_t* __restrict__ inv) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nb) return;
  const int64_t nbk = unit_new ? (int64_t)unit_new[b / ub] * ub + (b % ub) : b;
  block_perm[nbk] = (int32_t)b;
  inv[b] = (int32_t)nbk;
}

__global__ void k_perm_tracks(const int32_t* __restrict__ block_perm,
                              const int32_t* __restrict__ sample, const int32_t* __restrict__ seg,
                              const int32_t* __restrict__ noise, const int32_t* __restrict__ pos,
                              int64_t n,
                              int32_t* __restrict__ perm, int32_t* __restrict__ tracks) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n) return;
  const int64_t o = (int64_t)block_perm[t >> 7] * kBlock + (t & (kBlock - 1));
  perm[t] = (int32_t)o;
  tracks[t] = sample[o];
  tracks[n + t] = seg[o];
  tracks[2 * n + t] = noise[o];
  tracks[3 * n + t] = pos ? pos[o] : (int32_t)o;
}

// ------------------------------------------------------------------------------------
// key intervals: per key, the interval [lo, hi) of query indices that see it, and whether
// every query inside sees it (the fast mask test of partial tiles)
// ------------------------------------------------------------------------------------
// first / last index and size of every segment id and noise id below n
__global__ void k_iv_tables(const int32_t* __restrict__ seg, const int32_t* __restrict__ noise,
                            int64_t n, int32_t* __restrict__ gfirst, int32_t* __restrict__ glast,
                            int32_t* __restrict__ gcount, int32_t* __restrict__ zfirst,
                            int32_t* __restrict__ zlast, int32_t* __restrict__ zcount) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int g = seg[i], z = noise[i];
  if (g >= 0 && g < n) {
    atomicMin(&gfirst[g], (int)i);
    atomicMax(&glast[g], (int)i);
    atomicAdd(&gcount[g], 1);
  }
  if (z >= 0 && z < n) {
    atomicMin(&zfirst[z], (int)i);
    atomicMax(&zlast[z], (int)i);
    atomicAdd(&zcount[z], 1);
  }
}

// Per key k of sample run [a, b): the causal queries form [k, min(k + W, b)); a key of a
// span or group is also seen by the whole segment, and a noise key only by its noise span.
// With the segment and the noise span each one run inside the sample, the visible set is
// (causal u segment) n noise span, an interval; otherwise the key is not exact.  iv_orig
// (per original block, preset to 1) is cleared by any key that is not exact.
__global__ void k_iv_keys(const int32_t* __restrict__ sample, const int32_t* __restrict__ seg,
                          const int32_t* __restrict__ noise, int64_t n, int W,
                          const int32_t* __restrict__ gfirst, const int32_t* __restrict__ glast,
                          const int32_t* __restrict__ gcount, const int32_t* __restrict__ zfirst,
                          const int32_t* __restrict__ zlast, const int32_t* __restrict__ zcount,
                          int32_t* __restrict__ lo_out, int32_t* __restrict__ hi_out,
                          uint8_t* __restrict__ iv_orig) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  const int s = sample[k];
  int64_t a = 0, b = k;  // a = first index of the sample (sample ids are non-decreasing)
  while (a < b) {
    const int64_t m = (a + b) >> 1;
    if (sample[m] < s) a = m + 1; else b = m;
  }
  int64_t lo2 = k + 1, b2 = n;  // b2 = one past the last index of the sample
  while (lo2 < b2) {
    const int64_t m = (lo2 + b2) >> 1;
    if (sample[m] <= s) lo2 = m + 1; else b2 = m;
  }
  b = b2;
  int64_t lo = k, hi = min(b, k + (int64_t)W);  // causal part, empty when W == 0
  bool ex = true;
  const int g = seg[k], z = noise[k];
  if (g >= 0) {
    if (g < n && gcount[g] == glast[g] - gfirst[g] + 1 && gfirst[g] >= a && glast[g] < b) {
      lo = hi > lo ? min(lo, (int64_t)gfirst[g]) : (int64_t)gfirst[g];
      hi = max(hi, (int64_t)glast[g] + 1);
    } else {
      ex = false;
    }
  }
  if (z >= 0) {
    if (z < n && zcount[z] == zlast[z] - zfirst[z] + 1 && zfirst[z] >= a && zlast[z] < b) {
      lo = max(lo, (int64_t)zfirst[z]);
      hi = min(hi, (int64_t)zlast[z] + 1);
    } else {
      ex = false;
    }
  }
  if (hi <= lo) lo = hi = 0;  // seen by no query
  lo_out[k] = (int32_t)lo;
  hi_out[k] = (int32_t)hi;
  if (!ex) iv_orig[k >> 7] = 0;
}

// Key intervals of a pack given with a position track (a permuted pack, MARBLE s04 "Layout
// transforms"), on globally causal layers.  Key k is seen causally by the queries of its
// sample at a position >= pos[k]; the layout transform is what makes the visible queries
// one range of indices.  Here every key gets a hull [lo, hi) that provably holds all of its
// visible queries, and a warp then checks the predicate on every query of the hull: the key
// is exact when all of them see it.
//   causal hull  the smallest and largest index among the sample's tokens at a position
//                >= pos[k], from suffix minima / maxima over positions (this needs positions
//                that are a permutation of [0, n) with each sample holding one range of
//                them: checked, and otherwise no key is exact);
//   segment      every token of k's segment id lies in [gfirst, glast], cut to the sample;
//   noise        a noise key is seen only inside [zfirst, zlast].
// inv[position] = index.
__global__ void k_pos_inv(const int32_t* __restrict__ pos, int64_t n, int32_t* __restrict__ inv,
                          unsigned* __restrict__ bad) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int p = pos[i];
  if (p < 0 || p >= n || atomicCAS(&inv[p], -1, (int)i) != -1) atomicOr(bad, 1u);
}

__device__ __forceinline__ void sample_run(const int32_t* __restrict__ sample, int64_t n,
                                           int64_t k, int64_t* a_out, int64_t* b_out) {
  const int s = sample[k];
  int64_t a = 0, b = k;
  while (a < b) {
    const int64_t m = (a + b) >> 1;
    if (sample[m] < s) a = m + 1; else b = m;
  }
  int64_t lo2 = k + 1, b2 = n;
  while (lo2 < b2) {
    const int64_t m = (lo2 + b2) >> 1;
    if (sample[m] <= s) lo2 = m + 1; else b2 = m;
  }
  *a_out = a;
  *b_out = b2;
}

// per sample run [a, b) of indices: min and max position, kept at the run's first index
__global__ void k_pos_runs(const int32_t* __restrict__ sample, const int32_t* __restrict__ pos,
                           int64_t n, int32_t* __restrict__ rmin, int32_t* __restrict__ rmax) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  int64_t a, b;
  sample_run(sample, n, k, &a, &b);
  atomicMin(&rmin[a], pos[k]);
  atomicMax(&rmax[a], pos[k]);
}

// the sample id of every position, and a flag if some sample's positions are not one range
__global__ void k_pos_check(const int32_t* __restrict__ sample, const int32_t* __restrict__ pos,
                            int64_t n, const int32_t* __restrict__ rmin,
                            const int32_t* __restrict__ rmax, int32_t* __restrict__ psample,
                            unsigned* __restrict__ bad) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  int64_t a, b;
  sample_run(sample, n, k, &a, &b);
  if (k == a && (int64_t)rmax[a] - rmin[a] + 1 != b - a) atomicOr(bad, 1u);
  const int p = pos[k];
  if (p >= 0 && p < n) psample[p] = sample[k];  // out-of-range positions were flagged
}

// Suffix minimum and maximum of inv[] over positions >= p within the sample of position p,
// by one CTA walking the positions downward in chunks of 1024 (a segmented scan; a segment
// is a sample's range of positions).
__global__ void __launch_bounds__(1024) k_pos_suffix(const int32_t* __restrict__ inv,
                                                     const int32_t* __restrict__ psample,
                                                     int64_t n, int32_t* __restrict__ smin,
                                                     int32_t* __restrict__ smax) {
  __shared__ int vmin[1024], vmax[1024], head[1024];
  __shared__ int cmin_c, cmax_c, cs_c;
  const int t = threadIdx.x;
  if (t == 0) {
    cmin_c = INT_MAX;
    cmax_c = INT_MIN;
    cs_c = INT_MIN;  // sample of the lowest position of the previous (higher) chunk
  }
  __syncthreads();
  for (int64_t top = n; top > 0; top -= 1024) {
    // element t of the chunk is position top - 1 - t (walking down)
    const int64_t p = top - 1 - t;
    const bool ok = p >= 0;
    const int sp = ok ? psample[p] : INT_MIN;
    int mn = ok ? inv[p] : INT_MAX, mx = ok ? inv[p] : INT_MIN;
    // a segment starts at element t if position p + 1 belongs to another sample; element 0
    // continues the previous chunk's segment when the sample matches
    int hd;
    if (t == 0) {
      hd = sp != cs_c;
      if (!hd) {
        mn = min(mn, cmin_c);
        mx = max(mx, cmax_c);
      }
    } else {
      hd = ok && psample[p + 1] != sp;
    }
    vmin[t] = mn;
    vmax[t] = mx;
    head[t] = hd;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      int a = vmin[t], b = vmax[t], h = head[t];
      if (t >= off && !h) {
        a = min(a, vmin[t - off]);
        b = max(b, vmax[t - off]);
        h = head[t - off];
      }
      __syncthreads();
      vmin[t] = a;
      vmax[t] = b;
      head[t] = h;
      __syncthreads();
    }
    if (ok) {
      smin[p] = vmin[t];
      smax[p] = vmax[t];
    }
    __syncthreads();
    if (t == 1023 || p == 0) {
      cmin_c = vmin[t];
      cmax_c = vmax[t];
      cs_c = sp;
    }
    __syncthreads();
  }
}

// the hull of every key (see above); with invalid positions every key is marked inexact
__global__ void k_iv_hull_pos(const int32_t* __restrict__ sample, const int32_t* __restrict__ seg,
                              const int32_t* __restrict__ noise, const int32_t* __restrict__ pos,
                              int64_t n, const int32_t* __restrict__ gfirst,
                              const int32_t* __restrict__ glast, const int32_t* __restrict__ zfirst,
                              const int32_t* __restrict__ zlast, const int32_t* __restrict__ smin,
                              const int32_t* __restrict__ smax, const unsigned* __restrict__ bad,
                              int32_t* __restrict__ lo_out, int32_t* __restrict__ hi_out,
                              uint8_t* __restrict__ iv_orig) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  if (*bad) {
    lo_out[k] = hi_out[k] = 0;
    iv_orig[k >> 7] = 0;
    return;
  }
  int64_t a, b;
  sample_run(sample, n, k, &a, &b);
  const int p = pos[k];
  int64_t lo = smin[p], hi = (int64_t)smax[p] + 1;  // holds k itself
  const int g = seg[k], z = noise[k];
  if (g >= 0) {
    if (g < n) {
      lo = min(lo, max(a, (int64_t)gfirst[g]));
      hi = max(hi, min(b, (int64_t)glast[g] + 1));
    } else {
      lo = a;  // no table for this id: the whole sample
      hi = b;
    }
  }
  if (z >= 0 && z < n) {
    lo = max(lo, (int64_t)zfirst[z]);
    hi = min(hi, (int64_t)zlast[z] + 1);
  }
  if (hi <= lo) lo = hi = 0;
  lo_out[k] = (int32_t)lo;
  hi_out[k] = (int32_t)hi;
}

// one warp per key: clears the key's block flag unless every query of its hull sees it
__global__ void k_iv_verify(const int32_t* __restrict__ sample, const int32_t* __restrict__ seg,
                            const int32_t* __restrict__ noise, const int32_t* __restrict__ pos,
                            int64_t n, const int32_t* __restrict__ lo_in,
                            const int32_t* __restrict__ hi_in, uint8_t* __restrict__ iv_orig) {
  const int lane = threadIdx.x & 31;
  const int64_t k = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (k >= n) return;
  const int64_t lo = lo_in[k], hi = hi_in[k];
  if (hi <= lo || !iv_orig[k >> 7]) return;  // nothing to check, or the block is off already
  const int sk = sample[k], gk = seg[k], zk = noise[k], pk = pos[k];
  for (int64_t q0 = lo; q0 < hi; q0 += 32) {
    const int64_t q = q0 + lane;
    bool ok = true;
    if (q < hi)
      ok = mask_legal(sample[q], seg[q], noise[q], pos[q], sk, gk, zk, pk, MARBLE_WINDOW_INF);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) iv_orig[k >> 7] = 0;
      return;
    }
  }
}

// intervals and block flags into the new order
__global__ void k_perm_iv(const int32_t* __restrict__ perm, const int32_t* __restrict__ block_perm,
                          const int32_t* __restrict__ lo, const int32_t* __restrict__ hi,
                          const uint8_t* __restrict__ iv_orig, int64_t n,
                          int32_t* __restrict__ kiv, uint8_t* __restrict__ iv_block) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n) return;
  const int64_t o = perm[t];
  kiv[t] = lo[o];
  kiv[n + t] = hi[o];
  if ((t & (kBlock - 1)) == 0) iv_block[t >> 7] = iv_orig[block_perm[t >> 7]];
}

// per 32-key chunk of the new order: (min lo, max lo, min hi, max hi) of its keys' intervals,
// one warp per chunk.  A query index i with max lo <= i < min hi lies in every key's interval
// of the chunk; one with i < min lo or i >= max hi in none.
__global__ void k_iv_chunks(const int32_t* __restrict__ kiv, int64_t n, int4* __restrict__ out) {
  const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (c * 32 >= n) return;
  const int64_t t = c * 32 + lane;
  const int lo = kiv[t], hi = kiv[n + t];
  int4 r;
  r.x = __reduce_min_sync(0xffffffffu, lo);
  r.y = __reduce_max_sync(0xffffffffu, lo);
  r.z = __reduce_min_sync(0xffffffffu, hi);
  r.w = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) out[c] = r;
}

// ------------------------------------------------------------------------------------
// a5: per-step lists
// ------------------------------------------------------------------------------------
// rows: new q block nq (forward / dQ lists keyed (nq, kv shard j))
__global__ void k_step_count(const int64_t* __restrict__ row_ptr, const int32_t* __restrict__ col,
                             const int32_t* __restrict__ block_perm,
                             const int32_t* __restrict__ inv, int64_t nb, int P, int64_t bps,
                             int32_t* __restrict__ cnt) {
  const int lane = threadIdx.x & 31;
  const int64_t nq = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (nq >= nb) return;
  const int64_t qb = block_perm[nq];
  const int64_t a = row_ptr[qb], e = row_ptr[qb + 1];
  for (int64_t i0 = a; i0 < e; i0 += 32) {
    const int64_t i = i0 + lane;
    const bool ok = i < e;
    const unsigned act = __ballot_sync(0xffffffffu, ok);
    if (ok) {
      const int j = (int)(inv[col[i]] / bps);
      const unsigned peers = __match_any_sync(act, j);
      if ((peers & lanemask_lt()) == 0) atomicAdd(&cnt[nq * P + j], __popc(peers));
    }
  }
}

__global__ void k_step_write(const int64_t* __restrict__ row_ptr, const int32_t* __restrict__ col,
                             const uint8_t* __restrict__ tag,
                             const int32_t* __restrict__ block_perm,
                             const int32_t* __restrict__ inv, int64_t nb, int P, int64_t bps,
                             const int64_t* __restrict__ step_ptr, int32_t* __restrict__ out_col,
                             uint8_t* __restrict__ out_tag) {
  extern __shared__ int64_t offs_all[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int64_t* offs = offs_all + (int64_t)w * P;
  const int64_t nq = (int64_t)blockIdx.x * kWarpsPerCta + w;
  if (nq >= nb) return;
  for (int j = lane; j < P; j += 32) offs[j] = step_ptr[nq * P + j];
  __syncwarp();
  const int64_t qb = block_perm[nq];
  const int64_t a = row_ptr[qb], e = row_ptr[qb + 1];
  for (int64_t i0 = a; i0 < e; i0 += 32) {
    const int64_t i = i0 + lane;
    const bool ok = i < e;
    const unsigned act = __ballot_sync(0xffffffffu, ok);
    int j = 0;
    unsigned peers = 0;
    int64_t o = 0;
    if (ok) {
      const int nk = inv[col[i]];
      j = (int)(nk / bps);
      peers = __match_any_sync(act, j);
      o = offs[j] + __popc(peers & lanemask_lt());
      out_col[o] = nk;
      out_tag[o] = tag[i];
    }
    __syncwarp();
    if (ok && (peers & lanemask_lt()) == 0) offs[j] += __popc(peers);
    __syncwarp();
  }
}

// The row lists in ring order, for the fused forward: q block nq of shard r visits kv shard
// (r - s) mod P at step s (MARBLE s03 ring pairing), so its entries are copied segment by
// segment, kv shard r first, then r - 1, ..., wrapping round to r + 1.  Same CSR ranges as
// step_ptr[nq * P] .. step_ptr[nq * P + P]; one warp per q block.
__global__ void k_ring_write(const int64_t* __restrict__ step_ptr,
                             const int32_t* __restrict__ step_col,
                             const uint8_t* __restrict__ step_tag, int64_t nb, int P, int64_t bps,
                             int32_t* __restrict__ ring_col, uint8_t* __restrict__ ring_tag) {
  const int lane = threadIdx.x & 31;
  const int64_t nq = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (nq >= nb) return;
  const int r = (int)(nq / bps);
  int64_t o = step_ptr[nq * P];
  for (int st = 0; st < P; ++st) {
    const int j = (r - st + P) % P;
    const int64_t a = step_ptr[nq * P + j], e = step_ptr[nq * P + j + 1];
    for (int64_t i = a + lane; i < e; i += 32) {
      ring_col[o + (i - a)] = step_col[i];
      ring_tag[o + (i - a)] = step_tag[i];
    }
    o += e - a;
  }
}

// columns: original kv block B (dK/dV lists keyed (nk, q shard r)), visiting the band of
// q blocks in ascending original order and classifying (A, B) directly
template <bool kWrite>
__global__ void k_colT(const Summary* __restrict__ s, const int32_t* __restrict__ band,
                       const int32_t* __restrict__ inv, int64_t nb, int W, int P, int64_t bps,
                       int32_t* __restrict__ cnt, const int64_t* __restrict__ colT_ptr,
                       int32_t* __restrict__ out_row, uint8_t* __restrict__ out_tag) {
  extern __shared__ int64_t offs_all[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t b = (int64_t)blockIdx.x * kWarpsPerCta + w;
  if (b >= nb) return;
  const int64_t nk = inv[b];
  int64_t* offs = offs_all + (int64_t)w * P;
  if (kWrite) {
    for (int r = lane; r < P; r += 32) offs[r] = colT_ptr[nk * P + r];
    __syncwarp();
  }
  const Summary B = s[b];
  const int lo = band[2 * b], hi = band[2 * b + 1];  // the band is symmetric
  for (int a0 = lo; a0 <= hi; a0 += 32) {
    const int a = a0 + lane;
    const int t = a <= hi ? classify(s[a], B, W) : 0;
    const unsigned act = __ballot_sync(0xffffffffu, t != 0);
    int r = 0;
    unsigned peers = 0;
    if (t) {
      const int nq = inv[a];
      r = (int)(nq / bps);
      peers = __match_any_sync(act, r);
      if (kWrite) {
        const int64_t o = offs[r] + __popc(peers & lanemask_lt());
        out_row[o] = nq;
        out_tag[o] = (uint8_t)t;
      } else if ((peers & lanemask_lt()) == 0) {
        atomicAdd(&cnt[nk * P + r], __popc(peers));
      }
    }
    if (kWrite) {
      __syncwarp();
      if (t && (peers & lanemask_lt()) == 0) offs[r] += __popc(peers);
      __syncwarp();
    }
  }
}

// Positions of the column-list entries in the row lists: for the entry of (kv block nk, q
// shard r) that lists q block nq, the index of nk within nq's list for kv shard nk / bps.  Both
// lists are sorted by original block index, so a binary search on it finds the entry.
__global__ void k_colT_pos(const int64_t* __restrict__ colT_ptr, const int32_t* __restrict__ colT_row,
                           const int64_t* __restrict__ step_ptr, const int32_t* __restrict__ step_col,
                           const int32_t* __restrict__ block_perm, int64_t nb, int P, int64_t bps,
                           int32_t* __restrict__ colT_j) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);  // nk * P + r
  if (row >= nb * P) return;
  const int64_t nk = row / P;
  const int s = (int)(nk / bps);
  const int32_t key = block_perm[nk];
  for (int64_t e = colT_ptr[row] + lane; e < colT_ptr[row + 1]; e += 32) {
    const int64_t nq = colT_row[e];
    const int64_t base = step_ptr[nq * P + s];
    int64_t lo = base, hi = step_ptr[nq * P + s + 1] - 1;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (block_perm[step_col[mid]] < key)
        lo = mid + 1;
      else
        hi = mid;
    }
    colT_j[e] = (int32_t)(lo - base);
  }
}

// Compact numbering of one step's tiles (one CTA per (q shard r, option opt); option opt < P
// is kv shard opt, option P every kv shard): step_off[nq * (P+1) + opt] = number of tiles of
// the q blocks of shard r before nq; step_tiles[r * (P+1) + opt] = the step's total.
__global__ void __launch_bounds__(1024) k_step_off(const int64_t* __restrict__ step_ptr, int P,
                                                   int64_t bps, int32_t* __restrict__ step_off,
                                                   int64_t* __restrict__ step_tiles,
                                                   int64_t* __restrict__ step_max) {
  __shared__ int64_t sc[1024];
  __shared__ int64_t carry;
  __shared__ unsigned long long longest;
  const int seg = blockIdx.x;
  const int r = seg / (P + 1), opt = seg % (P + 1);
  const int c_lo = opt < P ? opt : 0, c_hi = opt < P ? opt + 1 : P;
  const int t = threadIdx.x;
  if (t == 0) {
    carry = 0;
    longest = 0;
  }
  __syncthreads();
  for (int64_t i0 = 0; i0 < bps; i0 += 1024) {
    const int64_t i = i0 + t;
    int64_t len = 0;
    if (i < bps) {
      const int64_t nq = (int64_t)r * bps + i;
      len = step_ptr[nq * P + c_hi] - step_ptr[nq * P + c_lo];
      atomicMax(&longest, (unsigned long long)len);
    }
    sc[t] = len;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const int64_t v = t >= off ? sc[t - off] : 0;
      __syncthreads();
      sc[t] += v;
      __syncthreads();
    }
    if (i < bps) step_off[((int64_t)r * bps + i) * (P + 1) + opt] = (int32_t)(carry + sc[t] - len);
    __syncthreads();
    if (t == 1023) carry += sc[1023];
    __syncthreads();
  }
  if (t == 0) {
    step_tiles[seg] = carry;
    step_max[seg] = (int64_t)longest;
  }
}

// needed kv blocks of q shard r = kv blocks with a non-empty (kv block, r) list
template <bool kWrite>
__global__ void k_needed(const int64_t* __restrict__ colT_ptr, int64_t nb, int P,
                         int32_t* __restrict__ count, const int64_t* __restrict__ needed_ptr,
                         int32_t* __restrict__ needed) {
  __shared__ int ws[32];
  __shared__ int64_t carry;
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) carry = kWrite ? needed_ptr[r] : 0;
  __syncthreads();
  for (int64_t k0 = 0; k0 < nb; k0 += blockDim.x) {
    const int64_t k = k0 + tid;
    const int f = (k < nb) && (colT_ptr[k * P + r + 1] > colT_ptr[k * P + r]);
    const unsigned m = __ballot_sync(0xffffffffu, f);
    if (lane == 0) ws[wid] = __popc(m);
    __syncthreads();
    int before = 0, total = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
      if (i < wid) before += ws[i];
      total += ws[i];
    }
    if (kWrite && f) needed[carry + before + __popc(m & lanemask_lt())] = (int32_t)k;
    __syncthreads();
    if (tid == 0) carry += total;
    __syncthreads();
  }
  if (!kWrite && tid == 0) count[r] = (int32_t)carry;
}

// ------------------------------------------------------------------------------------
// statistics: legal pairs (full tiles 128*128, partial tiles evaluated pair by pair)
// ------------------------------------------------------------------------------------
__global__ void k_legal_pairs(const int64_t* __restrict__ row_ptr, const int32_t* __restrict__ col,
                              const uint8_t* __restrict__ tag, const int32_t* __restrict__ inv,
                              const int32_t* __restrict__ tracks, int64_t n, int64_t nb, int W,
                              int64_t bps, int P, unsigned long long* __restrict__ acc,
                              unsigned long long* __restrict__ shard_pairs) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
  const int32_t* smp = tracks;
  const int32_t* sg = tracks + n;
  const int32_t* nz = tracks + 2 * n;
  const int32_t* ps = tracks + 3 * n;
  unsigned long long legal = 0, nfull = 0, npart = 0;
  for (int64_t qb = warp0; qb < nb; qb += nwarps) {
    const int64_t qn = (int64_t)inv[qb] * kBlock;
    for (int64_t e = row_ptr[qb]; e < row_ptr[qb + 1]; ++e) {
      // W[q shard, kv shard] in legal pairs
      unsigned long long* wsh = shard_pairs + (inv[qb] / bps) * P + inv[col[e]] / bps;
      if (tag[e] == MARBLE_TILE_FULL) {
        if (lane == 0) {
          legal += kBlock * kBlock;
          ++nfull;
          atomicAdd(wsh, (unsigned long long)(kBlock * kBlock));
        }
        continue;
      }
      if (lane == 0) ++npart;
      const int64_t kn = (int64_t)inv[col[e]] * kBlock;
      unsigned long long tile = 0;
      for (int qi = lane; qi < kBlock; qi += 32) {
        const int64_t q = qn + qi;
        const int sq = smp[q], gq = sg[q], zq = nz[q], pq = ps[q];
        int c = 0;
        for (int ki = 0; ki < kBlock; ++ki) {
          const int64_t k = kn + ki;
          const int dp = pq - ps[k];
          const bool causal = dp >= 0 && dp < W;
          const bool span = gq >= 0 && sg[k] == gq;
          const bool keep = nz[k] < 0 || nz[k] == zq;
          c += (causal || span) && keep && smp[k] == sq;
        }
        legal += c;
        tile += c;
      }
      for (int o = 16; o; o >>= 1) tile += __shfl_xor_sync(0xffffffffu, tile, o);
      if (lane == 0 && tile) atomicAdd(wsh, tile);
    }
  }
  for (int o = 16; o; o >>= 1) {
    legal += __shfl_xor_sync(0xffffffffu, legal, o);
  }
  if (lane == 0) {
    atomicAdd(&acc[0], legal);
    atomicAdd(&acc[1], nfull);
    atomicAdd(&acc[2], npart);
  }
}

// chunk-layout search input: legal pairs between every pair of chunks of cs blocks (original
// order), full tiles 128 * 128, partial tiles counted pair by pair; one warp per q block
__global__ void k_chunk_pairs(const int64_t* __restrict__ row_ptr, const int32_t* __restrict__ col,
                              const uint8_t* __restrict__ tag, const int32_t* __restrict__ sample,
                              const int32_t* __restrict__ seg, const int32_t* __restrict__ noise,
                              const int32_t* __restrict__ pos, int64_t nb, int W, int cs, int K,
                              unsigned long long* __restrict__ wc) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
  for (int64_t qb = warp0; qb < nb; qb += nwarps) {
    for (int64_t e = row_ptr[qb]; e < row_ptr[qb + 1]; ++e) {
      const int64_t kb = col[e];
      unsigned long long c = 0;
      if (tag[e] == MARBLE_TILE_FULL) {
        c = lane == 0 ? (unsigned long long)(kBlock * kBlock) : 0ull;
      } else {
        for (int qi = lane; qi < kBlock; qi += 32) {
          const int64_t q = qb * kBlock + qi;
          const int sq = sample[q], gq = seg[q], zq = noise[q], pq = pos ? pos[q] : (int)q;
          for (int ki = 0; ki < kBlock; ++ki) {
            const int64_t k = kb * kBlock + ki;
            c += mask_legal(sq, gq, zq, pq, sample[k], seg[k], noise[k], pos ? pos[k] : (int)k, W);
          }
        }
      }
      for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (lane == 0 && c) atomicAdd(&wc[(qb / cs) * K + kb / cs], c);
    }
  }
}

inline unsigned grid_for(int64_t items, int per_cta) {
  return (unsigned)((items + per_cta - 1) / per_cta);
}

}  // namespace

// ------------------------------------------------------------------------------------
// host driver
// ------------------------------------------------------------------------------------
#define MARBLE_CK(call)                                   \
  do {                                                    \
    cudaError_t e_ = (call);                              \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);   \
  } while (0)

template <typename T>
static marble_status_t dalloc(marble_plan_t* p, T** ptr, size_t count) {
  void* q = nullptr;
  const size_t bytes = count * sizeof(T) > 0 ? count * sizeof(T) : 16;
  cudaError_t e = dev_alloc(&q, bytes, p->build_stream);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(MARBLE_ERR_OOM, "allocation of plan workspace failed (" +
                                    std::to_string(bytes) + " bytes)");
  }
  p->owned.push_back(q);
  *ptr = static_cast<T*>(q);
  return MARBLE_OK;
}

// Work order of the persistent attention kernels (one CTA of 1024 threads per segment):
// segment (s, k) lists the blocks i of shard s whose list for option k is non-empty --
// option k < P counts the entries of column k of row s*bps+i of `ptr`, option P the whole
// row -- sorted by that count, longest first (counts above 1023 share a bucket).  Equal
// counts come out in no fixed order: each unit's result does not depend on where or when
// it runs.
__device__ void work_order_segment(const int64_t* __restrict__ ptr, int P, int64_t bps, int s,
                                   int c_lo, int c_hi, int32_t* __restrict__ out,
                                   int32_t* __restrict__ nwork_out);

__global__ void __launch_bounds__(1024) k_work_order(const int64_t* __restrict__ ptr, int P,
                                                     int64_t bps, int32_t* __restrict__ order,
                                                     int32_t* __restrict__ nwork) {
  const int seg = blockIdx.x;
  const int s = seg / (P + 1), k = seg % (P + 1);
  const int c_lo = k < P ? k : 0, c_hi = k < P ? k + 1 : P;
  work_order_segment(ptr, P, bps, s, c_lo, c_hi, order + (int64_t)seg * bps, nwork + seg);
}

// the same order over every block of the pack, by the length of its whole row (every kv
// shard): the work order of the fused forward (one CTA)
__global__ void __launch_bounds__(1024) k_work_order_all(const int64_t* __restrict__ ptr, int P,
                                                         int64_t nb, int32_t* __restrict__ order,
                                                         int32_t* __restrict__ nwork) {
  work_order_segment(ptr, P, nb, 0, 0, P, order, nwork);
}

__device__ void work_order_segment(const int64_t* __restrict__ ptr, int P, int64_t bps, int s,
                                   int c_lo, int c_hi, int32_t* __restrict__ out,
                                   int32_t* __restrict__ nwork_out) {
  __shared__ int hist[1024];
  __shared__ int scan[1024];
  hist[threadIdx.x] = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < bps; i += blockDim.x) {
    const int64_t r = (int64_t)s * bps + i;
    const int64_t c = ptr[r * P + c_hi] - ptr[r * P + c_lo];
    if (c > 0) atomicAdd(&hist[c < 1023 ? c : 1023], 1);
  }
  __syncthreads();
  // inclusive scan of the histogram read from the top bucket down (Hillis-Steele)
  const int t = threadIdx.x;
  scan[t] = hist[1023 - t];
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int v = t >= off ? scan[t - off] : 0;
    __syncthreads();
    scan[t] += v;
    __syncthreads();
  }
  // first output position of bucket b = entries in buckets above b
  const int b = 1023 - t;
  const int start = scan[t] - hist[b];
  __syncthreads();
  hist[b] = start;  // reused as the bucket cursors
  if (t == 1023) *nwork_out = scan[1023];
  __syncthreads();
  for (int64_t i = threadIdx.x; i < bps; i += blockDim.x) {
    const int64_t r = (int64_t)s * bps + i;
    const int64_t c = ptr[r * P + c_hi] - ptr[r * P + c_lo];
    if (c > 0) out[atomicAdd(&hist[c < 1023 ? c : 1023], 1)] = (int32_t)i;
  }
}

// ------------------------------------------------------------------------------------
// chunk-layout search (host): see MARBLE_ORDER_CHUNK_SEARCH in marble.h
// ------------------------------------------------------------------------------------
constexpr int kMaxChunks = 1024;
constexpr int kMaxSwapPasses = 64;

// sum over steps s of max over ranks r of W[r, (r - s) mod P]
static int64_t layout_step_cost(const std::vector<int64_t>& Wr, int P) {
  int64_t c = 0;
  for (int s = 0; s < P; ++s) {
    int64_t m = Wr[(size_t)(P - s) % P];  // r = 0
    for (int r = 1; r < P; ++r) m = std::max(m, Wr[(size_t)r * P + (r - s + P) % P]);
    c += m;
  }
  return c;
}

// PTRR's dealing over K units: (cost desc, index asc) order, round t of P units to ranks
// 0..P-1 (t even) or P-1..0 (t odd)
static void ptrr_deal(const std::vector<int64_t>& cost, int P, std::vector<int>& rank) {
  const int K = (int)cost.size();
  std::vector<int> order(K);
  for (int u = 0; u < K; ++u) order[u] = u;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  rank.assign(K, 0);
  for (int i = 0; i < K; ++i) {
    const int t = i / P, slot = i % P;
    rank[order[i]] = (t & 1) ? P - 1 - slot : slot;
  }
}

struct LayoutChoice {
  int k = 0;
  std::vector<int> rank;  // rank of every chunk
  int64_t C = 0, step = 0;
};

// search over one chunk count: K = k * P chunks, Wc [K][K] legal pairs between chunks
static void search_chunks(const std::vector<int64_t>& Wc, int K, int P, std::vector<int>& rank,
                          int64_t* step) {
  std::vector<int64_t> Wr((size_t)P * P);
  auto rank_work = [&](const std::vector<int>& rk) {
    std::fill(Wr.begin(), Wr.end(), 0);
    for (int a = 0; a < K; ++a)
      for (int b = 0; b < K; ++b) Wr[(size_t)rk[a] * P + rk[b]] += Wc[(size_t)a * K + b];
    return layout_step_cost(Wr, P);
  };
  std::vector<int64_t> work(K, 0), zero(K, 0);
  for (int a = 0; a < K; ++a)
    for (int b = 0; b < K; ++b) work[a] += Wc[(size_t)a * K + b];
  std::vector<int> ra, rb;
  ptrr_deal(work, P, ra);
  ptrr_deal(zero, P, rb);
  const int64_t ca = rank_work(ra), cb = rank_work(rb);
  rank = ca <= cb ? ra : rb;
  int64_t cur = rank_work(rank);  // leaves Wr for the chosen start
  // per chunk: its work towards / from every rank
  std::vector<int64_t> srow((size_t)K * P, 0), scol((size_t)K * P, 0);
  for (int a = 0; a < K; ++a)
    for (int b = 0; b < K; ++b) {
      srow[(size_t)a * P + rank[b]] += Wc[(size_t)a * K + b];
      scol[(size_t)b * P + rank[a]] += Wc[(size_t)a * K + b];
    }
  std::vector<int64_t> W2((size_t)P * P);
  for (int pass = 0; pass < kMaxSwapPasses; ++pass) {
    bool swapped = false;
    for (int a = 0; a < K; ++a)
      for (int b = a + 1; b < K; ++b) {
        const int x = rank[a], y = rank[b];
        if (x == y) continue;
        // chunk a moves from rank x to y, chunk b from y to x
        const int64_t waa = Wc[(size_t)a * K + a], wbb = Wc[(size_t)b * K + b];
        const int64_t wab = Wc[(size_t)a * K + b], wba = Wc[(size_t)b * K + a];
        W2 = Wr;
        for (int j = 0; j < P; ++j) {
          // a's and b's work towards the other chunks of rank j
          const int64_t ta = srow[(size_t)a * P + j] - (j == x ? waa : 0) - (j == y ? wab : 0);
          const int64_t tb = srow[(size_t)b * P + j] - (j == x ? wba : 0) - (j == y ? wbb : 0);
          W2[(size_t)x * P + j] += tb - ta;
          W2[(size_t)y * P + j] += ta - tb;
          // the other chunks of rank j towards a and b
          const int64_t ua = scol[(size_t)a * P + j] - (j == x ? waa : 0) - (j == y ? wba : 0);
          const int64_t ub = scol[(size_t)b * P + j] - (j == x ? wab : 0) - (j == y ? wbb : 0);
          W2[(size_t)j * P + x] += ub - ua;
          W2[(size_t)j * P + y] += ua - ub;
        }
        W2[(size_t)x * P + x] += wbb - waa;
        W2[(size_t)y * P + y] += waa - wbb;
        W2[(size_t)x * P + y] += wba - wab;
        W2[(size_t)y * P + x] += wab - wba;
        const int64_t c = layout_step_cost(W2, P);
        if (c >= cur) continue;
        cur = c;
        swapped = true;
        Wr = W2;
        for (int z = 0; z < K; ++z) {
          const int64_t dz = Wc[(size_t)z * K + b] - Wc[(size_t)z * K + a];
          srow[(size_t)z * P + x] += dz;
          srow[(size_t)z * P + y] -= dz;
          const int64_t ez = Wc[(size_t)b * K + z] - Wc[(size_t)a * K + z];
          scol[(size_t)z * P + x] += ez;
          scol[(size_t)z * P + y] -= ez;
        }
        rank[a] = y;
        rank[b] = x;
      }
    if (!swapped) break;
  }
  *step = cur;
}

// the layout with the lowest C over 1, 2, 4, ..., 64 chunks per rank; Wf [Kf][Kf] holds
// the pairs between the finest chunks (Kf = kf * P, kf the largest candidate)
static LayoutChoice choose_layout(const std::vector<int64_t>& Wf, int Kf, int P, int64_t tau) {
  LayoutChoice best;
  const int kf = Kf / P;
  for (int k = 1; k <= kf; k *= 2) {
    const int K = k * P, f = kf / k;
    std::vector<int64_t> Wc((size_t)K * K, 0);
    for (int a = 0; a < Kf; ++a)
      for (int b = 0; b < Kf; ++b) Wc[(size_t)(a / f) * K + b / f] += Wf[(size_t)a * Kf + b];
    std::vector<int> rank;
    int64_t step = 0;
    search_chunks(Wc, K, P, rank, &step);
    const int64_t C = step + tau * P * k;
    if (best.k == 0 || C < best.C) {
      best.k = k;
      best.rank = rank;
      best.C = C;
      best.step = step;
    }
  }
  return best;
}

// the finest chunk count the search tries: k * P chunks with k = 1, 2, 4, ..., 64 dividing
// the blocks evenly, at most kMaxChunks in all
int finest_chunks(int64_t nb, int P) {
  int kf = 1;
  while (kf * 2 <= 64 && (int64_t)kf * 2 * P <= kMaxChunks && nb % ((int64_t)kf * 2 * P) == 0)
    kf *= 2;
  return kf * P;
}

void chunk_layout_host(const std::vector<int64_t>& wf, int Kf, int P, int64_t tau, int* k,
                       std::vector<int>* rank, int64_t* cost, int64_t* step) {
  const LayoutChoice L = choose_layout(wf, Kf, P, tau);
  *k = L.k;
  *rank = L.rank;
  *cost = L.C;
  *step = L.step;
}

#define MARBLE_TRY(x)                     \
  do {                                    \
    marble_status_t st_ = (x);            \
    if (st_ != MARBLE_OK) return st_;     \
  } while (0)

marble_status_t build_plan(const marble_plan_desc_t* d, cudaStream_t s, marble_plan_t* p) {
  p->build_stream = s;
  const int64_t n = p->n, nb = p->nb;
  const int P = p->P, W = p->W;
  const int64_t bps = p->bps;
  const int threads = 256;
  const int warp_ctas = (int)grid_for(nb, kWarpsPerCta);

  MARBLE_TRY(dalloc(p, &p->err, 4));
  MARBLE_TRY(dalloc(p, &p->counters, 8));
  MARBLE_TRY(dalloc(p, &p->shard_pairs, (size_t)P * P));
  MARBLE_TRY(dalloc(p, &p->summ, nb));
  MARBLE_TRY(dalloc(p, &p->band, 2 * nb));
  MARBLE_TRY(dalloc(p, &p->row_ptr, nb + 1));
  MARBLE_TRY(dalloc(p, &p->block_perm, nb));
  MARBLE_TRY(dalloc(p, &p->inv_block_perm, nb));
  MARBLE_TRY(dalloc(p, &p->perm, n));
  MARBLE_TRY(dalloc(p, &p->tracks, 4 * n));
  MARBLE_TRY(dalloc(p, &p->step_ptr, nb * P + 1));
  MARBLE_TRY(dalloc(p, &p->colT_ptr, nb * P + 1));
  MARBLE_TRY(dalloc(p, &p->needed_ptr, P + 1));
  MARBLE_TRY(dalloc(p, &p->fwd_order, (size_t)P * (P + 1) * bps));
  MARBLE_TRY(dalloc(p, &p->fwd_nwork, (size_t)P * (P + 1)));
  MARBLE_TRY(dalloc(p, &p->bwd_order, (size_t)P * (P + 1) * bps));
  MARBLE_TRY(dalloc(p, &p->bwd_nwork, (size_t)P * (P + 1)));
  MARBLE_TRY(dalloc(p, &p->sched, 2 * kSchedSlots));
  MARBLE_TRY(dalloc(p, &p->step_off, (size_t)nb * (P + 1)));
  MARBLE_TRY(dalloc(p, &p->step_tiles, (size_t)P * (P + 1)));
  MARBLE_TRY(dalloc(p, &p->step_max, (size_t)P * (P + 1)));
  // scratch: counters of the two-pass compactions and the order builder
  int32_t *cnt = nullptr, *cnt2 = nullptr, *cntT = nullptr, *ucost = nullptr,
          *rank_of = nullptr, *unit_new = nullptr, *ncount = nullptr;
  std::vector<void*> scratch;
  auto salloc = [&](int32_t** ptr, size_t count) -> marble_status_t {
    void* q = nullptr;
    cudaError_t e = dev_alloc(&q, (count ? count : 1) * sizeof(int32_t), s);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return fail(MARBLE_ERR_OOM, "allocation of planner scratch failed");
    }
    scratch.push_back(q);
    *ptr = static_cast<int32_t*>(q);
    return MARBLE_OK;
  };
  struct Freer {
    std::vector<void*>* v;
    cudaStream_t s;
    ~Freer() {
      for (void* q : *v) dev_free(q, s);  // in stream order, after the kernels that use it
    }
  } freer{&scratch, s};
  const int ub = (p->order == MARBLE_ORDER_PTRR_CHUNK) ? p->chunk_tokens / kBlock : 1;
  const int64_t units = nb / ub;
  MARBLE_TRY(salloc(&cnt, nb));
  MARBLE_TRY(salloc(&cnt2, nb * P));
  MARBLE_TRY(salloc(&cntT, nb * P));
  MARBLE_TRY(salloc(&ucost, units));
  MARBLE_TRY(salloc(&rank_of, units));
  MARBLE_TRY(salloc(&unit_new, nb));  // the searched chunk layout has at most nb units
  MARBLE_TRY(salloc(&ncount, P));

  MARBLE_CK(cudaMemsetAsync(p->err, 0, 4 * sizeof(unsigned), s));
  MARBLE_CK(cudaMemsetAsync(p->counters, 0, 8 * sizeof(unsigned long long), s));
  MARBLE_CK(cudaMemsetAsync(p->sched, 0, 2 * kSchedSlots * sizeof(unsigned), s));
  MARBLE_CK(cudaMemsetAsync(cnt2, 0, nb * P * sizeof(int32_t), s));
  MARBLE_CK(cudaMemsetAsync(cntT, 0, nb * P * sizeof(int32_t), s));

  // a1 + a2
  k_summaries<<<warp_ctas, 32 * kWarpsPerCta, 0, s>>>(d->sample_id, d->seg_id, d->noise_id,
                                                      d->pos_id, nb, p->summ, p->err);
  MARBLE_CK(cudaGetLastError());
  unsigned herr = 0;
  MARBLE_CK(read_back(s, {{&herr, p->err, sizeof(unsigned)}}));
  if (herr & kErrBadTracks)
    return fail(MARBLE_ERR_INVALID_ARG,
                "metadata check failed: sample ids must be >= 0 and non-decreasing, seg and "
                "noise ids >= -1, positions >= 0");

  // a3
  k_band<<<grid_for(nb, threads), threads, 0, s>>>(p->summ, nb, p->band);
  k_tiles_count<<<warp_ctas, 32 * kWarpsPerCta, 0, s>>>(p->summ, p->band, nb, W, cnt);
  k_scan<int32_t><<<1, 1024, 0, s>>>(cnt, nb, p->row_ptr);
  MARBLE_CK(cudaGetLastError());
  int64_t nnz = 0;
  MARBLE_CK(read_back(s, {{&nnz, p->row_ptr + nb, sizeof(int64_t)}}));
  p->nnz = nnz;
  MARBLE_TRY(dalloc(p, &p->col, nnz));
  MARBLE_TRY(dalloc(p, &p->tag, nnz));
  MARBLE_TRY(dalloc(p, &p->step_col, nnz));
  MARBLE_TRY(dalloc(p, &p->step_tag, nnz));
  MARBLE_TRY(dalloc(p, &p->colT_row, nnz));
  MARBLE_TRY(dalloc(p, &p->colT_tag, nnz));
  MARBLE_TRY(dalloc(p, &p->colT_j, nnz));
  k_tiles_write<<<warp_ctas, 32 * kWarpsPerCta, 0, s>>>(p->summ, p->band, p->row_ptr, nb, W,
                                                        p->col, p->tag);
  MARBLE_CK(cudaGetLastError());

  // a4
  if (p->order == MARBLE_ORDER_CONTIGUOUS) {
    k_block_perm<<<grid_for(nb, threads), threads, 0, s>>>(nullptr, 1, nb, p->block_perm,
                                                            p->inv_block_perm);
  } else if (p->order == MARBLE_ORDER_CHUNK_SEARCH) {
    // legal pairs between the finest chunks (the most chunks per rank the search tries),
    // then the search on the host
    const int Kf = finest_chunks(nb, P);
    const int cs = (int)(nb / Kf);
    void* wq = nullptr;
    cudaError_t e = dev_alloc(&wq, (size_t)Kf * Kf * sizeof(unsigned long long), s);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return fail(MARBLE_ERR_OOM, "allocation of the chunk-pair matrix failed");
    }
    scratch.push_back(wq);
    auto* wc = static_cast<unsigned long long*>(wq);
    MARBLE_CK(cudaMemsetAsync(wc, 0, (size_t)Kf * Kf * sizeof(unsigned long long), s));
    k_chunk_pairs<<<warp_ctas, 32 * kWarpsPerCta, 0, s>>>(p->row_ptr, p->col, p->tag, d->sample_id,
                                                          d->seg_id, d->noise_id, d->pos_id, nb, W,
                                                          cs, Kf, wc);
    MARBLE_CK(cudaGetLastError());
    std::vector<int64_t> wf((size_t)Kf * Kf);
    MARBLE_CK(read_back(s, {{wf.data(), wc, wf.size() * sizeof(int64_t)}}));
    const LayoutChoice L = choose_layout(wf, Kf, P, p->range_cost);
    const int K = L.k * P;
    std::vector<int32_t> un(K), seen(P, 0);
    for (int u = 0; u < K; ++u) un[u] = L.rank[u] * L.k + seen[L.rank[u]]++;
    MARBLE_CK(write_to_device(s, unit_new, un.data(), K * sizeof(int32_t)));
    k_block_perm<<<grid_for(nb, threads), threads, 0, s>>>(unit_new, (int)(nb / K), nb,
                                                            p->block_perm, p->inv_block_perm);
    p->chunks_per_rank = L.k;
    p->layout_cost = L.C;
    p->layout_step_cost = L.step;
  } else {
    k_unit_cost<<<grid_for(units, threads), threads, 0, s>>>(cnt, ub, units, ucost);
    k_ptrr_rank<<<grid_for(units, threads), threads, 0, s>>>(ucost, units, P, rank_of);
    k_ptrr_place<<<grid_for(units, threads), threads, 0, s>>>(rank_of, units, P, unit_new);
    k_block_perm<<<grid_for(nb, threads), threads, 0, s>>>(unit_new, ub, nb, p->block_perm,
                                                            p->inv_block_perm);
  }
  k_perm_tracks<<<grid_for(n, threads), threads, 0, s>>>(p->block_perm, d->sample_id, d->seg_id,
                                                          d->noise_id, d->pos_id, n, p->perm,
                                                          p->tracks);
  MARBLE_CK(cudaGetLastError());

  // key intervals (all blocks flagged 0 when switched off: partial tiles then always
  // evaluate the four-track predicate)
  MARBLE_TRY(dalloc(p, &p->kiv, 2 * n));
  MARBLE_TRY(dalloc(p, &p->iv_block, nb));
  MARBLE_TRY(dalloc(p, &p->kiv_chunk, nb * 4));
  MARBLE_CK(cudaMemsetAsync(p->kiv_chunk, 0, nb * 4 * sizeof(int4), s));
  MARBLE_CK(cudaMemsetAsync(p->kiv, 0, 2 * n * sizeof(int32_t), s));
  MARBLE_CK(cudaMemsetAsync(p->iv_block, 0, nb, s));
  // With a position track the causal part of an interval comes from the positions, on
  // globally causal layers (with a window the causal queries need not form one range)
  const bool use_pos = d->pos_id != nullptr;
  if (!d->no_key_intervals && (!use_pos || W == MARBLE_WINDOW_INF)) {
    int32_t *tab = nullptr, *klo = nullptr;
    MARBLE_TRY(salloc(&tab, 6 * n));
    MARBLE_TRY(salloc(&klo, 2 * n + (nb + 3) / 4));

    int32_t *gfirst = tab, *glast = tab + n, *gcount = tab + 2 * n, *zfirst = tab + 3 * n,
            *zlast = tab + 4 * n, *zcount = tab + 5 * n;
    uint8_t* iv_orig = reinterpret_cast<uint8_t*>(klo + 2 * n);
    MARBLE_CK(cudaMemsetAsync(gfirst, 0x7f, n * sizeof(int32_t), s));
    MARBLE_CK(cudaMemsetAsync(glast, 0xff, n * sizeof(int32_t), s));
    MARBLE_CK(cudaMemsetAsync(gcount, 0, n * sizeof(int32_t), s));
    MARBLE_CK(cudaMemsetAsync(zfirst, 0x7f, n * sizeof(int32_t), s));
    MARBLE_CK(cudaMemsetAsync(zlast, 0xff, n * sizeof(int32_t), s));
    MARBLE_CK(cudaMemsetAsync(zcount, 0, n * sizeof(int32_t), s));
    MARBLE_CK(cudaMemsetAsync(iv_orig, 1, nb, s));
    k_iv_tables<<<grid_for(n, threads), threads, 0, s>>>(d->seg_id, d->noise_id, n, gfirst, glast,
                                                        gcount, zfirst, zlast, zcount);
    if (!use_pos) {
      k_iv_keys<<<grid_for(n, threads), threads, 0, s>>>(d->sample_id, d->seg_id, d->noise_id, n,
                                                        W, gfirst, glast, gcount, zfirst, zlast,
                                                        zcount, klo, klo + n, iv_orig);
    } else {
      int32_t *inv = nullptr, *rmin = nullptr, *rmax = nullptr, *psample = nullptr,
              *smin = nullptr, *smax = nullptr, *badw = nullptr;
      MARBLE_TRY(salloc(&inv, n));
      MARBLE_TRY(salloc(&rmin, n));
      MARBLE_TRY(salloc(&rmax, n));
      MARBLE_TRY(salloc(&psample, n));
      MARBLE_TRY(salloc(&smin, n));
      MARBLE_TRY(salloc(&smax, n));
      MARBLE_TRY(salloc(&badw, 1));
      unsigned* bad = reinterpret_cast<unsigned*>(badw);
      MARBLE_CK(cudaMemsetAsync(inv, 0xff, n * sizeof(int32_t), s));
      MARBLE_CK(cudaMemsetAsync(rmin, 0x7f, n * sizeof(int32_t), s));
      MARBLE_CK(cudaMemsetAsync(rmax, 0x80, n * sizeof(int32_t), s));
      MARBLE_CK(cudaMemsetAsync(bad, 0, sizeof(unsigned), s));
      k_pos_inv<<<grid_for(n, threads), threads, 0, s>>>(d->pos_id, n, inv, bad);
      k_pos_runs<<<grid_for(n, threads), threads, 0, s>>>(d->sample_id, d->pos_id, n, rmin, rmax);
      k_pos_check<<<grid_for(n, threads), threads, 0, s>>>(d->sample_id, d->pos_id, n, rmin, rmax,
                                                          psample, bad);
      k_pos_suffix<<<1, 1024, 0, s>>>(inv, psample, n, smin, smax);
      k_iv_hull_pos<<<grid_for(n, threads), threads, 0, s>>>(
          d->sample_id, d->seg_id, d->noise_id, d->pos_id, n, gfirst, glast, zfirst, zlast, smin,
          smax, bad, klo, klo + n, iv_orig);
      k_iv_verify<<<grid_for(n, kWarpsPerCta), 32 * kWarpsPerCta, 0, s>>>(
          d->sample_id, d->seg_id, d->noise_id, d->pos_id, n, klo, klo + n, iv_orig);
    }
    k_perm_iv<<<grid_for(n, threads), threads, 0, s>>>(p->perm, p->block_perm, klo, klo + n,
                                                      iv_orig, n, p->kiv, p->iv_block);
    k_iv_chunks<<<grid_for(n, threads), threads, 0, s>>>(p->kiv, n, p->kiv_chunk);
    MARBLE_CK(cudaGetLastError());
  }

  // a5: forward lists
  const size_t offs_smem = (size_t)kWarpsPerCta * P * sizeof(int64_t);
  k_step_count<<<warp_ctas, 32 * kWarpsPerCta, 0, s>>>(p->row_ptr, p->col, p->block_perm,
                                                       p->inv_block_perm, nb, P, bps, cnt2);
  k_scan<int32_t><<<1, 1024, 0, s>>>(cnt2, nb * P, p->step_ptr);
  k_step_write<<<warp_ctas, 32 * kWarpsPerCta, offs_smem, s>>>(
      p->row_ptr, p->col, p->tag, p->block_perm, p->inv_block_perm, nb, P, bps, p->step_ptr,
      p->step_col, p->step_tag);
  MARBLE_CK(cudaGetLastError());
  // column lists
  k_colT<false><<<warp_ctas, 32 * kWarpsPerCta, offs_smem, s>>>(
      p->summ, p->band, p->inv_block_perm, nb, W, P, bps, cntT, nullptr, nullptr, nullptr);
  k_scan<int32_t><<<1, 1024, 0, s>>>(cntT, nb * P, p->colT_ptr);
  k_colT<true><<<warp_ctas, 32 * kWarpsPerCta, offs_smem, s>>>(
      p->summ, p->band, p->inv_block_perm, nb, W, P, bps, nullptr, p->colT_ptr, p->colT_row,
      p->colT_tag);
  MARBLE_CK(cudaGetLastError());
  // needed index
  k_needed<false><<<P, 1024, 0, s>>>(p->colT_ptr, nb, P, ncount, nullptr, nullptr);
  k_scan<int32_t><<<1, 1024, 0, s>>>(ncount, P, p->needed_ptr);
  MARBLE_CK(cudaGetLastError());
  p->h_needed_ptr.resize(P + 1);
  MARBLE_CK(read_back(s, {{p->h_needed_ptr.data(), p->needed_ptr, (P + 1) * sizeof(int64_t)}}));
  const int64_t ntot = p->h_needed_ptr[P];
  p->needed_total = ntot;
  MARBLE_TRY(dalloc(p, &p->needed, ntot));
  k_needed<true><<<P, 1024, 0, s>>>(p->colT_ptr, nb, P, nullptr, p->needed_ptr, p->needed);
  MARBLE_CK(cudaGetLastError());
  // positions of the column-list entries in the row lists, and each step's tile numbering
  k_colT_pos<<<(unsigned)grid_for(nb * P, kWarpsPerCta), 32 * kWarpsPerCta, 0, s>>>(
      p->colT_ptr, p->colT_row, p->step_ptr, p->step_col, p->block_perm, nb, P, bps, p->colT_j);
  k_step_off<<<P * (P + 1), 1024, 0, s>>>(p->step_ptr, P, bps, p->step_off, p->step_tiles,
                                          p->step_max);
  MARBLE_CK(cudaGetLastError());
  // work order of the persistent kernels
  k_work_order<<<P * (P + 1), 1024, 0, s>>>(p->step_ptr, P, bps, p->fwd_order, p->fwd_nwork);
  k_work_order<<<P * (P + 1), 1024, 0, s>>>(p->colT_ptr, P, bps, p->bwd_order, p->bwd_nwork);
  MARBLE_CK(cudaGetLastError());
  // the fused forward: row lists in ring order and the order of all blocks
  MARBLE_TRY(dalloc(p, &p->ring_col, nnz));
  MARBLE_TRY(dalloc(p, &p->ring_tag, nnz));
  MARBLE_TRY(dalloc(p, &p->fwd_order_all, nb));
  MARBLE_TRY(dalloc(p, &p->fwd_nwork_all, 1));
  k_ring_write<<<warp_ctas, 32 * kWarpsPerCta, 0, s>>>(p->step_ptr, p->step_col, p->step_tag, nb,
                                                       P, bps, p->ring_col, p->ring_tag);
  k_work_order_all<<<1, 1024, 0, s>>>(p->step_ptr, P, nb, p->fwd_order_all, p->fwd_nwork_all);
  MARBLE_CK(cudaGetLastError());
  p->h_fwd_nwork.resize((size_t)P * (P + 1));
  p->h_bwd_nwork.resize((size_t)P * (P + 1));
  p->h_step_tiles.resize((size_t)P * (P + 1));
  p->h_step_max.resize((size_t)P * (P + 1));
  const size_t pp = (size_t)P * (P + 1);
  MARBLE_CK(read_back(s, {{&p->h_fwd_nwork_all, p->fwd_nwork_all, sizeof(int32_t)},
                          {p->h_fwd_nwork.data(), p->fwd_nwork, pp * sizeof(int32_t)},
                          {p->h_bwd_nwork.data(), p->bwd_nwork, pp * sizeof(int32_t)},
                          {p->h_step_tiles.data(), p->step_tiles, pp * sizeof(int64_t)},
                          {p->h_step_max.data(), p->step_max, pp * sizeof(int64_t)}}));
  return MARBLE_OK;
}

marble_status_t plan_legal_pairs(const marble_plan_t* p, cudaStream_t s, int64_t* pairs,
                                 int64_t* n_full, int64_t* n_partial, int64_t* step_pairs) {
  MARBLE_CK(cudaMemsetAsync(p->counters, 0, 3 * sizeof(unsigned long long), s));
  MARBLE_CK(cudaMemsetAsync(p->shard_pairs, 0, (size_t)p->P * p->P * sizeof(unsigned long long), s));
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const unsigned ctas = (unsigned)std::min<int64_t>(grid_for(p->nb, kWarpsPerCta), 8 * sms);
  k_legal_pairs<<<ctas, 32 * kWarpsPerCta, 0, s>>>(p->row_ptr, p->col, p->tag,
                                                   p->inv_block_perm, p->tracks, p->n, p->nb,
                                                   p->W, p->bps, p->P, p->counters,
                                                   p->shard_pairs);
  MARBLE_CK(cudaGetLastError());
  unsigned long long h[3] = {0, 0, 0};
  std::vector<int64_t> w((size_t)p->P * p->P);
  MARBLE_CK(read_back(s, {{h, p->counters, sizeof(h)},
                          {w.data(), p->shard_pairs, w.size() * sizeof(int64_t)}}));
  *step_pairs = layout_step_cost(w, p->P);
  *pairs = (int64_t)h[0];
  *n_full = (int64_t)h[1];
  *n_partial = (int64_t)h[2];
  return MARBLE_OK;
}

}  // namespace marble

// ======================================================================================
// Tile map into caller buffers, without allocating
// ======================================================================================
// Some callers cannot call cudaMalloc: a planner that runs for every packed batch on a
// data-loader stream while the previous training step is still running must not pay the
// device-wide synchronisation cudaMalloc may imply, and a process whose device memory is
// owned by another allocator (a framework's caching allocator that has reserved the pool,
// or a fixed per-process budget) cannot obtain memory outside it.  For them,
// marble_tile_map_static builds the global tile map with the same kernels as marble_plan,
// keeping its intermediate scratch (per-block summaries, candidate bands, per-row counts
// and a validation word) in the file-scope array below instead of allocated memory.  The
// array is part of the module image: every GPU that loads the library holds it until the
// process exits.
namespace marble {
namespace {

constexpr int64_t kStaticMaxBlocks = MARBLE_TILE_MAP_STATIC_MAX_TOKENS / kBlock;
constexpr size_t kStaticSummaryBytes = kStaticMaxBlocks * sizeof(Summary);
constexpr size_t kStaticBandBytes = kStaticMaxBlocks * 2 * sizeof(int32_t);
constexpr size_t kStaticCountBytes = kStaticMaxBlocks * sizeof(int32_t);
constexpr size_t kStaticScratchBytes =
    kStaticSummaryBytes + kStaticBandBytes + kStaticCountBytes + 256;

// In host code this name is only a host-side stand-in for the device array: its address
// must be obtained with cudaGetSymbolAddress on each device (see static_scratch()).
static __device__ __align__(256) unsigned char g_tile_map_scratch[kStaticScratchBytes];

// writes the tiles of each row whose CSR index is below `capacity`
__global__ void k_tiles_write_capped(const Summary* __restrict__ s,
                                     const int32_t* __restrict__ band,
                                     const int64_t* __restrict__ row_ptr, int64_t nb, int W,
                                     int64_t capacity, int32_t* __restrict__ col,
                                     uint8_t* __restrict__ tag) {
  const int lane = threadIdx.x & 31;
  const int64_t a = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (a >= nb) return;
  const Summary A = s[a];
  const int lo = band[2 * a], hi = band[2 * a + 1];
  int64_t out = row_ptr[a];
  for (int b0 = lo; b0 <= hi; b0 += 32) {
    const int b = b0 + lane;
    const int t = b <= hi ? classify(A, s[b], W) : 0;
    const unsigned m = __ballot_sync(0xffffffffu, t != 0);
    if (t) {
      const int64_t o = out + __popc(m & lanemask_lt());
      if (o < capacity) {
        col[o] = b;
        tag[o] = (uint8_t)t;
      }
    }
    out += __popc(m);
  }
}

// metadata that failed validation is reported in the output itself: row_ptr[0] = -1
__global__ void k_flag_invalid(const unsigned* __restrict__ err, int64_t* __restrict__ row_ptr) {
  if (threadIdx.x == 0 && (*err & kErrBadTracks)) row_ptr[0] = -1;
}

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};

// Device address of the scratch array on the current device, looked up once per device.
// The address belongs to the device's primary context: after cudaDeviceReset the module
// is loaded anew and the cached address no longer applies (documented in marble.h).
marble_status_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(MARBLE_ERR_UNSUPPORTED, "device ordinal >= 64");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_tile_map_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(tile-map scratch)");
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return MARBLE_OK;
}

}  // namespace
}  // namespace marble

extern "C" __attribute__((visibility("default"))) marble_status_t marble_tile_map_static(
    int64_t n_tokens, const int32_t* sample_id, const int32_t* seg_id, const int32_t* noise_id,
    int32_t window, int64_t* row_ptr, int32_t* col, uint8_t* tag, int64_t capacity,
    marble_stream_t stream) {
  using namespace marble;
  NvtxRange nvtx_("marble_tile_map_static");
  if (n_tokens <= 0 || n_tokens % kBlock)
    return fail(MARBLE_ERR_INVALID_ARG, "n_tokens must be a positive multiple of 128");
  if (n_tokens > MARBLE_TILE_MAP_STATIC_MAX_TOKENS)
    return fail(MARBLE_ERR_INVALID_ARG,
                "n_tokens exceeds MARBLE_TILE_MAP_STATIC_MAX_TOKENS (" +
                    std::to_string((long long)MARBLE_TILE_MAP_STATIC_MAX_TOKENS) +
                    "), the size of the static scratch; use marble_plan instead");
  if (window < 0) return fail(MARBLE_ERR_INVALID_ARG, "window must be >= 0");
  if (capacity < 0) return fail(MARBLE_ERR_INVALID_ARG, "capacity must be >= 0");
  if (!sample_id || !seg_id || !noise_id || !row_ptr || (capacity > 0 && (!col || !tag)))
    return fail(MARBLE_ERR_INVALID_ARG, "null pointer");
  // every pointer goes straight to a kernel: host or foreign memory is refused here
  if (!is_device_ptr(sample_id) || !is_device_ptr(seg_id) || !is_device_ptr(noise_id) ||
      !is_device_ptr(row_ptr) || (capacity > 0 && (!is_device_ptr(col) || !is_device_ptr(tag))))
    return fail(MARBLE_ERR_INVALID_ARG,
                "sample_id, seg_id, noise_id, row_ptr, col and tag must be device memory");
  void* base = nullptr;
  marble_status_t st = static_scratch(&base);
  if (st != MARBLE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t nb = n_tokens / kBlock;
  unsigned char* scratch = static_cast<unsigned char*>(base);
  Summary* summ = reinterpret_cast<Summary*>(scratch);
  int32_t* band = reinterpret_cast<int32_t*>(scratch + kStaticSummaryBytes);
  int32_t* cnt = reinterpret_cast<int32_t*>(scratch + kStaticSummaryBytes + kStaticBandBytes);
  unsigned* err = reinterpret_cast<unsigned*>(scratch + kStaticSummaryBytes + kStaticBandBytes +
                                              kStaticCountBytes);
  const int warp_ctas = (int)grid_for(nb, kWarpsPerCta);
  // the validation word accumulates with atomicOr: it must start at zero on every call
  MARBLE_CK(cudaMemsetAsync(err, 0, sizeof(unsigned), s));
  k_summaries<<<warp_ctas, 32 * kWarpsPerCta, 0, s>>>(sample_id, seg_id, noise_id, nullptr, nb,
                                                      summ, err);
  k_band<<<grid_for(nb, 256), 256, 0, s>>>(summ, nb, band);
  k_tiles_count<<<warp_ctas, 32 * kWarpsPerCta, 0, s>>>(summ, band, nb, window, cnt);
  k_scan<int32_t><<<1, 1024, 0, s>>>(cnt, nb, row_ptr);
  k_tiles_write_capped<<<warp_ctas, 32 * kWarpsPerCta, 0, s>>>(summ, band, row_ptr, nb, window,
                                                               capacity, col, tag);
  k_flag_invalid<<<1, 32, 0, s>>>(err, row_ptr);
  MARBLE_CK(cudaGetLastError());
  return MARBLE_OK;
}
