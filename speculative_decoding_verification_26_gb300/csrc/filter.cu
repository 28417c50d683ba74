// filter.cu -- top-k / top-p filtering of logit rows before verification.
//
// The tutorial page "5.1 投机解码核心原理", section 2.1: p and q are the
// distributions actually sampled from, with temperature, top-k and top-p
// already applied when they are used.  Per row, by value (ties stay
// together):
//   top-k (1 <= k < V): keep x >= the k-th largest logit;
//   top-p (0 < top_p < 1), on the distribution left by top-k at the row's
//   temperature: keep x >= t*, the largest value whose upper mass
//   {x >= t*} reaches top_p;
//   a removed logit becomes -inf, in place.
//
// One CTA per row (grid-stride over rows).  Logits map to order-preserving
// integer keys (-0 folded into +0, so equal values have equal keys); each
// threshold is found by a most-significant-digit-first radix descent over the
// keys, 8 bits a level (2 levels for bf16, 4 for fp32), one histogram pass
// over the row per level.  top-k counts keys; top-p sums the tokens' weights
// 2^{(x - m) c} as 64-bit fixed-point integers (2^(61 - ceil(log2 V)) per unit
// of the row maximum's weight), so every sum is exact in its own arithmetic
// and the result does not depend on the order of the atomics.  Logits near the
// row max share their leading key bits, so a histogram keeps one copy of each
// bucket per lane (64 KB of dynamic shared memory), summed per bucket after
// the pass: the atomics of a warp never meet on one address.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace sv {
namespace {

constexpr int kFiltThreads = 512;

template <int DT>
struct Keys;
template <>
struct Keys<SPEC_BF16> {
  static constexpr int kLevels = 2;
  __device__ __forceinline__ static uint32_t raw(const unsigned char* row, int v) {
    return reinterpret_cast<const uint16_t*>(row)[v];
  }
  __device__ __forceinline__ static float value(uint32_t h) { return __uint_as_float(h << 16); }
  __device__ __forceinline__ static uint32_t key(uint32_t h) {
    if (h == 0x8000u) h = 0u;                              // -0 -> +0
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
  }
  __device__ __forceinline__ static void kill(unsigned char* row, int v) {
    reinterpret_cast<uint16_t*>(row)[v] = 0xFF80u;         // -inf
  }
};
template <>
struct Keys<SPEC_F32> {
  static constexpr int kLevels = 4;
  __device__ __forceinline__ static uint32_t raw(const unsigned char* row, int v) {
    return reinterpret_cast<const uint32_t*>(row)[v];
  }
  __device__ __forceinline__ static float value(uint32_t u) { return __uint_as_float(u); }
  __device__ __forceinline__ static uint32_t key(uint32_t u) {
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  __device__ __forceinline__ static void kill(unsigned char* row, int v) {
    reinterpret_cast<uint32_t*>(row)[v] = 0xFF800000u;
  }
};

// Bucket d's total from its 32 lane copies (threads 0..255, one bucket each;
// integer sums, so the order does not matter).
__device__ __forceinline__ void bucket_totals(const unsigned long long* h, unsigned long long* b, int tid) {
  if (tid < 256) {
    unsigned long long t = 0ull;
#pragma unroll 8
    for (int l = 0; l < 32; ++l) t += h[tid * 32 + ((l + tid) & 31)];   // staggered: no bank conflicts
    b[tid] = t;
  }
}

template <int DT>
__global__ void __launch_bounds__(kFiltThreads, 2) filter_kernel(const __grid_constant__ FiltParams P) {
  using K = Keys<DT>;
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  constexpr int kKeyBits = 8 * ES;
  extern __shared__ unsigned long long s_h[];            // [256 buckets][32 lanes]
  __shared__ unsigned long long s_b[256];                  // bucket totals
  __shared__ float s_max[kFiltThreads / 32];
  __shared__ int s_bad[kFiltThreads / 32];
  __shared__ uint32_t s_prefix;
  __shared__ unsigned long long s_above, s_total;
  const int V = P.V, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int r = blockIdx.x; r < P.n; r += gridDim.x) {
    unsigned char* row = P.logits + (size_t)r * V * ES;
    const int k = P.top_k ? P.top_k[r] : 0;
    const float tp = P.top_p ? P.top_p[r] : 1.f;
    const float T = P.temperature ? P.temperature[r] : 1.f;
    const bool use_k = k >= 1 && k < V, use_p = tp > 0.f && tp < 1.f;
    if (!use_k && !use_p) {
      if (tid == 0 && P.status) P.status[r] = 0;
      continue;
    }
    if (use_p && !temperature_ok(T)) {
      if (tid == 0 && P.status) P.status[r] = SPEC_ST_BAD_TEMPERATURE;
      continue;
    }
    // pass 0: a NaN or +inf logit, and the row max
    float m = -INFINITY;
    int bad = 0;
    for (int v = tid; v < V; v += kFiltThreads) {
      const float x = K::value(K::raw(row, v));
      bad |= (x != x) || x == INFINITY;
      m = fmaxf(m, x);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      bad |= __shfl_xor_sync(0xffffffffu, bad, off);
    }
    if (lane == 0) { s_max[warp] = m; s_bad[warp] = bad; }
    __syncthreads();
    m = s_max[0];
    bad = s_bad[0];
    for (int w = 1; w < kFiltThreads / 32; ++w) { m = fmaxf(m, s_max[w]); bad |= s_bad[w]; }
    __syncthreads();
    if (bad || m == -INFINITY) {
      if (tid == 0 && P.status) P.status[r] = SPEC_ST_NONFINITE;
      continue;
    }

    // top-k: the key of the k-th largest logit (radix descent on counts)
    uint32_t thr = 0u;                                    // keep keys >= thr
    if (use_k) {
      uint32_t prefix = 0u;
      unsigned long long above = 0ull;                    // keys above the prefix's range
      for (int L = 0; L < K::kLevels; ++L) {
        const int sh = kKeyBits - 8 * (L + 1);
        for (int i = tid; i < 256 * 32; i += kFiltThreads) s_h[i] = 0ull;
        __syncthreads();
        for (int v = tid; v < V; v += kFiltThreads) {
          const uint32_t key = K::key(K::raw(row, v));
          if (L == 0 || (key >> (sh + 8)) == (prefix >> (sh + 8)))
            atomicAdd(&s_h[((key >> sh) & 255u) * 32 + lane], 1ull);
        }
        __syncthreads();
        bucket_totals(s_h, s_b, tid);
        __syncthreads();
        if (tid == 0) {
          unsigned long long cum = above;
          int d = 255;
          for (; d > 0; --d) {
            if (cum + s_b[d] >= (unsigned long long)k) break;
            cum += s_b[d];
          }
          s_prefix = prefix | ((uint32_t)d << sh);
          s_above = cum;
        }
        __syncthreads();
        prefix = s_prefix;
        above = s_above;
        __syncthreads();
      }
      thr = prefix;
    }

    // top-p: the key of t* (radix descent on fixed-point masses)
    if (use_p) {
      const float c = scale_of(T);
      const float c_lo = (float)(1.4426950408889634 / (double)T - (double)c);
      const float ks = scale_k(c, c_lo);
      const float nr = -ref_of(m, c);
      int lg = 0;
      while ((1 << lg) < V) ++lg;
      const float unit = __int_as_float((127 + 61 - lg) << 23);   // 2^(61 - ceil(log2 V))
      auto weight = [&](float x) -> unsigned long long {
        const float w = ex2(stretch(fmaf(x, c, nr), ks));
        return __float2ull_rz(w * unit);
      };
      // total mass of the tokens top-k keeps
      if (tid == 0) s_total = 0ull;
      __syncthreads();
      unsigned long long part = 0ull;
      for (int v = tid; v < V; v += kFiltThreads) {
        const uint32_t h = K::raw(row, v);
        if (K::key(h) >= thr) part += weight(K::value(h));
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      if (lane == 0) atomicAdd(&s_total, part);
      __syncthreads();
      const double need = (double)tp * (double)s_total;   // upper mass to reach
      uint32_t prefix = 0u;
      unsigned long long above = 0ull;
      for (int L = 0; L < K::kLevels; ++L) {
        const int sh = kKeyBits - 8 * (L + 1);
        for (int i = tid; i < 256 * 32; i += kFiltThreads) s_h[i] = 0ull;
        __syncthreads();
        for (int v = tid; v < V; v += kFiltThreads) {
          const uint32_t h = K::raw(row, v);
          const uint32_t key = K::key(h);
          if (key >= thr && (L == 0 || (key >> (sh + 8)) == (prefix >> (sh + 8))))
            atomicAdd(&s_h[((key >> sh) & 255u) * 32 + lane], weight(K::value(h)));
        }
        __syncthreads();
        bucket_totals(s_h, s_b, tid);
        __syncthreads();
        if (tid == 0) {
          unsigned long long cum = above;
          int d = 255;
          for (; d > 0; --d) {
            if ((double)(cum + s_b[d]) >= need) break;
            cum += s_b[d];
          }
          s_prefix = prefix | ((uint32_t)d << sh);
          s_above = cum;
        }
        __syncthreads();
        prefix = s_prefix;
        above = s_above;
        __syncthreads();
      }
      if (prefix > thr) thr = prefix;
    }

    // the removed logits become -inf
    for (int v = tid; v < V; v += kFiltThreads)
      if (K::key(K::raw(row, v)) < thr) K::kill(row, v);
    if (tid == 0 && P.status) P.status[r] = 0;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_filter(const FiltParams& P, int grid, cudaStream_t s) {
  constexpr int kSmem = 256 * 32 * (int)sizeof(unsigned long long);   // per-lane bucket copies
  cudaError_t e;
  if (P.dtype == SPEC_BF16) {
    e = cudaFuncSetAttribute(filter_kernel<SPEC_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess) filter_kernel<SPEC_BF16><<<grid, kFiltThreads, kSmem, s>>>(P);
  } else {
    e = cudaFuncSetAttribute(filter_kernel<SPEC_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess) filter_kernel<SPEC_F32><<<grid, kFiltThreads, kSmem, s>>>(P);
  }
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace sv
