// HBM-bound helpers: token permutation (MARBLE s04 "Layout transforms"), the final
// normalisation (MARBLE s03: only the last call normalises, writes the LSE and casts to
// bf16), the backward preprocessing delta = rowsum(dO * O), an fp32 -> bf16 cast and the
// bounded-wait self test.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace marble {
namespace {

// dst row i <- src row perm[i]  (inverse: dst row perm[i] <- src row i), rows of `chunks`
// 16-byte chunks.  A block moves kRows rows at a time, so that each thread has kRows loads in
// flight before its first store.  CAST: a source chunk is 4 fp32, written as 4 bf16 (round
// to nearest even) into rows of `chunks` 8-byte chunks.
constexpr int kRows = 4;

template <bool CAST>
__global__ void k_permute_rows(const int32_t* __restrict__ perm, const uint4* __restrict__ src,
                               void* __restrict__ dst, int64_t n, int chunks, int inverse) {
  for (int64_t r0 = (int64_t)blockIdx.x * kRows; r0 < n; r0 += (int64_t)gridDim.x * kRows) {
    int64_t from[kRows], to[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const int64_t r = r0 + j < n ? r0 + j : r0;
      const int64_t o = perm[r];
      from[j] = inverse ? r : o;
      to[j] = inverse ? o : r;
    }
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      uint4 v[kRows];
#pragma unroll
      for (int j = 0; j < kRows; ++j)
        if (r0 + j < n) v[j] = src[from[j] * chunks + c];
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        if (r0 + j >= n) continue;
        if constexpr (CAST) {
          const float4 f = *reinterpret_cast<const float4*>(&v[j]);
          static_cast<uint2*>(dst)[to[j] * chunks + c] =
              make_uint2(pack_bf16(f.x, f.y), pack_bf16(f.z, f.w));
        } else {
          static_cast<uint4*>(dst)[to[j] * chunks + c] = v[j];
        }
      }
    }
  }
}

__global__ void k_permute4(const int32_t* __restrict__ perm, const uint32_t* __restrict__ src,
                           uint32_t* __restrict__ dst, int64_t n, int64_t words, int inverse) {
  const int64_t total = n * words;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = x / words, c = x % words;
    const int64_t o = perm[r];
    if (inverse)
      dst[o * words + c] = src[r * words + c];
    else
      dst[r * words + c] = src[o * words + c];
  }
}

__global__ void k_cast_bf16(const float4* __restrict__ src, uint2* __restrict__ dst, int64_t n4) {
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n4;
       x += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = src[x];
    dst[x] = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
  }
}

// One group of D/8 threads per (token, head) row: 8 elements per thread.
template <int D>
__global__ void k_finalize(const float* __restrict__ o_acc, const float* __restrict__ m,
                           const float* __restrict__ l, int64_t n, int hq,
                           __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  constexpr int kTpr = D / 8;
  const int64_t rows = n * hq;
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = x / kTpr;
  const int part = (int)(x % kTpr);
  if (row >= rows) return;
  const int64_t t = row / hq;
  const int h = (int)(row % hq);
  const float lv = l[(int64_t)h * n + t];
  const float inv = lv > 0.f ? 1.f / lv : 0.f;
  const float4* src = reinterpret_cast<const float4*>(o_acc + row * D + part * 8);
  const float4 a = src[0], b = src[1];
  uint4 out;
  out.x = pack_bf16(a.x * inv, a.y * inv);
  out.y = pack_bf16(a.z * inv, a.w * inv);
  out.z = pack_bf16(b.x * inv, b.y * inv);
  out.w = pack_bf16(b.z * inv, b.w * inv);
  *reinterpret_cast<uint4*>(o + row * D + part * 8) = out;
  if (part == 0) {
    // natural-log LSE from base-2 state: (m + log2 l) * ln 2
    lse[(int64_t)h * n + t] =
        lv > 0.f ? (m[(int64_t)h * n + t] + log2f(lv)) * 0.69314718055994531f : -INFINITY;
  }
}

template <int D>
__global__ void k_bwd_prep(const __nv_bfloat16* __restrict__ o,
                           const __nv_bfloat16* __restrict__ d_o, int64_t n, int hq,
                           float* __restrict__ delta) {
  constexpr int kTpr = D / 8;
  const int64_t rows = n * hq;
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = x / kTpr;
  const int part = (int)(x % kTpr);
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + part * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(d_o + row * D + part * 8);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 fa = __bfloat1622float2(pa[k]), fb = __bfloat1622float2(pb[k]);
      acc += fa.x * fb.x + fa.y * fb.y;
    }
  }
  // reduce over the kTpr threads of the row (kTpr divides 32, rows aligned to groups)
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) {
    const int64_t t = row / hq;
    const int h = (int)(row % hq);
    delta[(int64_t)h * n + t] = acc;
  }
}

__global__ void k_debug_wait(unsigned* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtx w{limit_ns, err, &abort_flag};
    (void)mbar_wait(&bar, 0, w);  // nothing ever arrives: runs out after limit_ns
  }
  __syncthreads();
}

// grid for grid-stride kernels (capped)
unsigned grid_of(int64_t items, int threads) {
  int64_t g = (items + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > 1048576) g = 1048576;
  return (unsigned)g;
}

// grid covering every item once (one thread per item)
unsigned grid_exact(int64_t items, int threads) {
  int64_t g = (items + threads - 1) / threads;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

// threads per block of k_permute_rows: one 16-byte chunk each, up to 256
static int row_threads(int64_t chunks) {
  return chunks >= 256 ? 256 : (int)((chunks + 31) / 32 * 32);
}

cudaError_t launch_permute(const marble_plan_t* p, const void* src, void* dst, int64_t row_bytes,
                           int inverse, cudaStream_t s) {
  if (row_bytes % 16 == 0) {
    const int64_t chunks = row_bytes / 16;
    k_permute_rows<false><<<grid_of(p->n, kRows), row_threads(chunks), 0, s>>>(
        p->perm, static_cast<const uint4*>(src), dst, p->n, (int)chunks, inverse);
  } else {
    const int64_t words = row_bytes / 4;
    k_permute4<<<grid_of(p->n * words, 256), 256, 0, s>>>(
        p->perm, static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), p->n, words,
        inverse);
  }
  return cudaGetLastError();
}

cudaError_t launch_permute_cast_bf16(const marble_plan_t* p, const float* src, void* dst,
                                     int64_t row_elems, int inverse, cudaStream_t s) {
  const int64_t chunks = row_elems / 4;
  k_permute_rows<true><<<grid_of(p->n, kRows), row_threads(chunks), 0, s>>>(
      p->perm, reinterpret_cast<const uint4*>(src), dst, p->n, (int)chunks, inverse);
  return cudaGetLastError();
}

cudaError_t launch_cast_bf16(const float* src, void* dst, int64_t n, cudaStream_t s) {
  const int64_t n4 = n / 4;
  k_cast_bf16<<<grid_of(n4, 256), 256, 0, s>>>(reinterpret_cast<const float4*>(src),
                                               static_cast<uint2*>(dst), n4);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const marble_plan_t* p, const float* o_acc, const float* m,
                            const float* l, int hq, int d, void* o, float* lse, cudaStream_t s) {
  const int64_t threads = p->n * hq * (d / 8);
  if (d == 128)
    k_finalize<128><<<grid_exact(threads, 256), 256, 0, s>>>(
        o_acc, m, l, p->n, hq, static_cast<__nv_bfloat16*>(o), lse);
  else
    k_finalize<64><<<grid_exact(threads, 256), 256, 0, s>>>(
        o_acc, m, l, p->n, hq, static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const marble_plan_t* p, const void* o, const void* d_o, int hq, int d,
                            float* delta, cudaStream_t s) {
  const int64_t threads = p->n * hq * (d / 8);
  if (d == 128)
    k_bwd_prep<128><<<grid_exact(threads, 256), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), p->n, hq,
        delta);
  else
    k_bwd_prep<64><<<grid_exact(threads, 256), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), p->n, hq,
        delta);
  return cudaGetLastError();
}

cudaError_t launch_debug_wait(unsigned* err, uint64_t limit_ns, cudaStream_t s) {
  k_debug_wait<<<1, 32, 0, s>>>(err, (unsigned long long)limit_ns);
  return cudaGetLastError();
}

}  // namespace marble
