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
// One CTA per row (grid-stride over rows, two CTAs per SM, so the rows in
// flight fit in L2 and the passes after the first mostly hit it).  Logits map
// to order-preserving integer keys (-0 folded into +0, so equal values have
// equal keys); each threshold is found by a most-significant-digit-first radix
// descent over the keys, 8 bits a level (2 levels for bf16, 4 for fp32).
// top-k counts keys; top-p sums the tokens' weights 2^{(x - m) c} as 64-bit
// fixed-point integers (2^(61 - ceil(log2 V)) per unit of the row maximum's
// weight), so every histogram sum is exact in its own arithmetic and the
// result does not depend on the order of the atomics.  Logits near the row max share their
// leading key bits, so a histogram keeps one copy of each bucket per lane,
// summed per bucket after the pass: the atomics of a warp never meet on one
// address; a thread also merges runs of its own elements that fall in one
// bucket before adding a mass (integer sums: still exact).
//
// Passes over the row (16-byte loads, four in flight per thread; bf16 pairs
// are compared and maxed as packed bf16x2, so a pass costs a few instructions
// per element):
//   A: the row max and the non-finite check;
//   S + C (top-k, k <= 512): over a quarter of the row, the k-th largest of the
//      512 threads' own maxima is a lower bound of the k-th largest logit (k
//      threads each hold an element that large), so pass A also copies the
//      logits at or above it -- a few times k of them -- to shared memory, and
//      every level, top-k's and top-p's, runs on that list.  For larger k, or
//      when the list would pass kCap, the first top-k level counts the whole
//      row, and its keys at or above the chosen bucket are copied instead when
//      they fit;
//   S + C (top-p alone): the sample's max m_s is a provisional reference, so
//      pass A also sums the whole row's mass on it in registers (each 16-byte
//      vector's weights by a fixed tree, then a compensated fp32 sum per
//      thread, reduced in fp64 in a fixed order: ~2e-7 relative,
//      deterministic), rescaled to the row max by 2^{(R(m_s) - R(m))(1 + k)},
//      and copies the logits above the 256th largest sampled thread maximum;
//      when those carry at least top_p of the total in exact fixed point (on
//      the row max), t* is among them and the levels run on the list.  A
//      weight that overflows on m_s voids the list (the exact path runs);
//      with no finite m_s, pass A takes the max alone and a pass C does the
//      rest on the row max;
//   else one pass per remaining level (a packed range test first, the exact
//      key test on the few elements inside);
//   K: the removed logits become -inf: on a list, -inf stores over the whole
//      row (no read) and the list's kept logits put back at their indices;
//      else a 16-byte store where any element changed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace sv {
namespace {

constexpr int kFiltThreads = 512;
constexpr int kUnroll = 4;                                 // 16-byte loads in flight per thread
constexpr int kCap = 4096;                                 // candidate list (index << 32 | raw)
constexpr int kRankP = 384;                                // top-p alone: the list's bound, a thread-max rank
constexpr int kRankPS = 256;                               // the same over a quarter-row sample
constexpr int kHistWords = 256 * 32;                       // [bucket][lane] copies
constexpr int kFiltSmem = kHistWords * 8 + kCap * 8;       // 96 KB dynamic

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
  __nv_bfloat162 v;
  memcpy(&v, &w, 4);
  return v;
}
__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) {
  uint32_t w;
  memcpy(&w, &v, 4);
  return w;
}

template <int DT>
struct Keys;
template <>
struct Keys<SPEC_BF16> {
  static constexpr int kLevels = 2, kES = 2;
  static constexpr uint32_t kNegInf = 0xFF80u, kKeyNegInf = 0x007Fu, kKeyPosInf = 0xFF80u;
  __device__ __forceinline__ static uint32_t raw(const unsigned char* row, int v) {
    return reinterpret_cast<const uint16_t*>(row)[v];
  }
  __device__ __forceinline__ static float value(uint32_t h) { return __uint_as_float(h << 16); }
  __device__ __forceinline__ static uint32_t key(uint32_t h) {
    if (h == 0x8000u) h = 0u;                              // -0 -> +0
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
  }
  __device__ __forceinline__ static uint32_t unkey(uint32_t k) { return k >= 0x8000u ? k ^ 0x8000u : (~k & 0xFFFFu); }
  __device__ __forceinline__ static void kill(unsigned char* row, int v) {
    reinterpret_cast<uint16_t*>(row)[v] = (uint16_t)kNegInf;
  }
};
template <>
struct Keys<SPEC_F32> {
  static constexpr int kLevels = 4, kES = 4;
  static constexpr uint32_t kNegInf = 0xFF800000u, kKeyNegInf = 0x007FFFFFu, kKeyPosInf = 0xFF800000u;
  __device__ __forceinline__ static uint32_t raw(const unsigned char* row, int v) {
    return reinterpret_cast<const uint32_t*>(row)[v];
  }
  __device__ __forceinline__ static float value(uint32_t u) { return __uint_as_float(u); }
  __device__ __forceinline__ static uint32_t key(uint32_t u) {
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  __device__ __forceinline__ static uint32_t unkey(uint32_t k) { return k >= 0x80000000u ? k ^ 0x80000000u : ~k; }
  __device__ __forceinline__ static void kill(unsigned char* row, int v) {
    reinterpret_cast<uint32_t*>(row)[v] = kNegInf;
  }
};

// The value a key stands for, as a float: for a key k of a finite or infinite
// logit, x >= value_of(k) holds exactly when key(x) >= k, and x < value_of(k)
// exactly when key(x) < k, for every non-NaN x (keys of NaN patterns map to
// -inf below the keys of -inf and to +inf above those of +inf).
template <int DT>
__device__ __forceinline__ float value_of(uint32_t k) {
  using K = Keys<DT>;
  if (k <= K::kKeyNegInf) return -INFINITY;
  if (k >= K::kKeyPosInf) return INFINITY;
  return K::value(K::unkey(k));
}

// Split of a row into a scalar head up to the first 16-byte boundary, a body
// of 16-byte vectors and a scalar tail.
template <int DT>
struct Span {
  int head, nvec, tail0;
  __device__ __forceinline__ Span(const unsigned char* row, int V) {
    constexpr int ES = Keys<DT>::kES, PER = 16 / ES;
    const int mis = (int)(reinterpret_cast<uintptr_t>(row) & 15u);
    head = mis ? (16 - mis) / ES : 0;
    if (head > V) head = V;
    nvec = (V - head) / PER;
    tail0 = head + nvec * PER;
  }
};

// fe(raw, v) for each element v of the head and tail, fw(word, v) for each
// 32-bit word of the body (one fp32 element, or two bf16 elements, element v
// in the low half and v + 1 in the high half), in no particular order.
template <int DT, class FE, class FW>
__device__ __forceinline__ void each_word_at(const unsigned char* row, int V, FE&& fe, FW&& fw) {
  using K = Keys<DT>;
  constexpr int PER = 16 / K::kES, WS = PER / 4;         // elements per vector / per word
  const Span<DT> sp(row, V);
  const int tid = threadIdx.x;
  if (tid < sp.head) fe(K::raw(row, tid), tid);
  const uint4* body = reinterpret_cast<const uint4*>(row + (size_t)sp.head * K::kES);
  auto vec = [&](const uint4& w, int i) {
    const int v = sp.head + i * PER;
    fw(w.x, v); fw(w.y, v + WS); fw(w.z, v + 2 * WS); fw(w.w, v + 3 * WS);
  };
  int i = tid;
  for (; i + (kUnroll - 1) * kFiltThreads < sp.nvec; i += kUnroll * kFiltThreads) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) w[u] = body[i + u * kFiltThreads];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) vec(w[u], i + u * kFiltThreads);
  }
  for (; i < sp.nvec; i += kFiltThreads) vec(body[i], i);
  for (int v = sp.tail0 + tid; v < V; v += kFiltThreads) fe(K::raw(row, v), v);
}

// fe(raw, v) for each element v of the head and tail, fv(vector, v) for each
// 16-byte vector of the body (its first element is v), in no particular order.
template <int DT, class FE, class FV>
__device__ __forceinline__ void each_vec_at(const unsigned char* row, int V, FE&& fe, FV&& fv) {
  using K = Keys<DT>;
  constexpr int PER = 16 / K::kES;
  const Span<DT> sp(row, V);
  const int tid = threadIdx.x;
  if (tid < sp.head) fe(K::raw(row, tid), tid);
  const uint4* body = reinterpret_cast<const uint4*>(row + (size_t)sp.head * K::kES);
  int i = tid;
  for (; i + (kUnroll - 1) * kFiltThreads < sp.nvec; i += kUnroll * kFiltThreads) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) w[u] = body[i + u * kFiltThreads];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) fv(w[u], sp.head + (i + u * kFiltThreads) * PER);
  }
  for (; i < sp.nvec; i += kFiltThreads) fv(body[i], sp.head + i * PER);
  for (int v = sp.tail0 + tid; v < V; v += kFiltThreads) fe(K::raw(row, v), v);
}

// The same without the element indices.
template <int DT, class FE, class FW>
__device__ __forceinline__ void each_word(const unsigned char* row, int V, FE&& fe, FW&& fw) {
  each_word_at<DT>(row, V, [&](uint32_t h, int) { fe(h); }, [&](uint32_t w, int) { fw(w); });
}

// f(raw) for every element of the row, in no particular order.
template <int DT, class F>
__device__ __forceinline__ void each_raw(const unsigned char* row, int V, F&& f) {
  if constexpr (DT == SPEC_BF16) {
    each_word<DT>(row, V, f, [&](uint32_t w) { f(w & 0xFFFFu); f(w >> 16); });
  } else {
    each_word<DT>(row, V, f, f);
  }
}

// f(raw, v) for every element v of the row, in no particular order.
template <int DT, class F>
__device__ __forceinline__ void each_raw_at(const unsigned char* row, int V, F&& f) {
  if constexpr (DT == SPEC_BF16) {
    each_word_at<DT>(row, V, f, [&](uint32_t w, int v) { f(w & 0xFFFFu, v); f(w >> 16, v + 1); });
  } else {
    each_word_at<DT>(row, V, f, f);
  }
}

// f(raw, v) for every element x with lo <= x <= hi (and perhaps a few more: a
// packed range test on bf16 pairs, which f must follow with its exact test).
template <int DT, class F>
__device__ __forceinline__ void each_in_range_at(const unsigned char* row, int V, float lo, float hi, F&& f) {
  using K = Keys<DT>;
  auto fe = [&](uint32_t h, int v) {
    const float x = K::value(h);
    if (x >= lo && x <= hi) f(h, v);
  };
  if constexpr (DT == SPEC_BF16) {
    const __nv_bfloat162 lo2 = __float2bfloat162_rn(lo), hi2 = __float2bfloat162_rn(hi);
    each_word_at<DT>(row, V, fe, [&](uint32_t w, int v) {
      const uint32_t in = __hge2_mask(as_bf2(w), lo2) & __hle2_mask(as_bf2(w), hi2);
      if (in) {
        if (in & 0xFFFFu) f(w & 0xFFFFu, v);
        if (in >> 16) f(w >> 16, v + 1);
      }
    });
  } else {
    each_word_at<DT>(row, V, fe, fe);
  }
}

template <int DT, class F>
__device__ __forceinline__ void each_in_range(const unsigned char* row, int V, float lo, float hi, F&& f) {
  each_in_range_at<DT>(row, V, lo, hi, [&](uint32_t h, int) { f(h); });
}

// Every logit of the row becomes -inf (stores only: the row is not read).
template <int DT>
__device__ __forceinline__ void fill_neg_inf(unsigned char* row, int V) {
  using K = Keys<DT>;
  const Span<DT> sp(row, V);
  const int tid = threadIdx.x;
  if (tid < sp.head) K::kill(row, tid);
  constexpr uint32_t w = DT == SPEC_BF16 ? K::kNegInf * 0x00010001u : K::kNegInf;
  uint4* body = reinterpret_cast<uint4*>(row + (size_t)sp.head * K::kES);
  for (int i = tid; i < sp.nvec; i += kFiltThreads) body[i] = make_uint4(w, w, w, w);
  for (int v = sp.tail0 + tid; v < V; v += kFiltThreads) K::kill(row, v);
}

// Every logit below t becomes -inf.
template <int DT>
__device__ __forceinline__ void kill_below(unsigned char* row, int V, float t) {
  using K = Keys<DT>;
  const Span<DT> sp(row, V);
  const int tid = threadIdx.x;
  if (tid < sp.head && K::value(K::raw(row, tid)) < t) K::kill(row, tid);
  uint4* body = reinterpret_cast<uint4*>(row + (size_t)sp.head * K::kES);
  const __nv_bfloat162 t2 = __float2bfloat162_rn(t);
  auto word = [&](uint32_t w) -> uint32_t {
    if constexpr (DT == SPEC_BF16) {
      const uint32_t lt = __hlt2_mask(as_bf2(w), t2);
      return (w & ~lt) | (K::kNegInf * 0x00010001u & lt);
    } else {
      return __uint_as_float(w) < t ? K::kNegInf : w;
    }
  };
  auto fix = [&](uint4& w) -> bool {
    const uint4 o = w;
    w.x = word(w.x); w.y = word(w.y); w.z = word(w.z); w.w = word(w.w);
    return ((o.x ^ w.x) | (o.y ^ w.y) | (o.z ^ w.z) | (o.w ^ w.w)) != 0u;
  };
  int i = tid;
  for (; i + (kUnroll - 1) * kFiltThreads < sp.nvec; i += kUnroll * kFiltThreads) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) w[u] = body[i + u * kFiltThreads];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (fix(w[u])) body[i + u * kFiltThreads] = w[u];
  }
  for (; i < sp.nvec; i += kFiltThreads) {
    uint4 w = body[i];
    if (fix(w)) body[i] = w;
  }
  for (int v = sp.tail0 + tid; v < V; v += kFiltThreads)
    if (K::value(K::raw(row, v)) < t) K::kill(row, v);
}

// Bucket d's total from its 32 lane copies (threads 0..255, one bucket each;
// integer sums, so the order does not matter).
template <class T>
__device__ __forceinline__ void bucket_totals(const T* h, unsigned long long* b, int tid) {
  if (tid < 256) {
    unsigned long long t = 0ull;
#pragma unroll 8
    for (int l = 0; l < 32; ++l) t += h[tid * 32 + ((l + tid) & 31)];   // staggered: no bank conflicts
    b[tid] = t;
  }
}

// One level of the descent, by warp 0: scanning buckets from 255 down with
// cum starting at `above`, the first bucket d where cum + b[d] reaches need
// (bucket 0 if none before it), with cum = the measure above d.  Lane l takes
// buckets 255-8l .. 248-8l; the crossing lane is found by a scan and a ballot
// (the test is monotone in d), then walks its own eight buckets.
__device__ __forceinline__ void descend(const unsigned long long* b, unsigned long long above, double need,
                                        int lane, int* s_d, unsigned long long* s_cum,
                                        unsigned long long* s_in) {
  unsigned long long sum = 0ull;
#pragma unroll
  for (int j = 0; j < 8; ++j) sum += b[255 - 8 * lane - j];
  unsigned long long incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  const unsigned mask = __ballot_sync(0xffffffffu, (double)(above + incl) >= need);
  const int src = mask ? __ffs(mask) - 1 : 31;
  if (lane == src) {
    unsigned long long cum = above + (incl - sum);
    int d = 0;
    unsigned long long in = 0ull;
    for (int j = 0; j < 8; ++j) {
      d = 255 - 8 * lane - j;
      in = b[d];
      if (d == 0 || (double)(cum + in) >= need) break;
      cum += in;
    }
    *s_d = d;
    *s_cum = cum;
    *s_in = in;
  }
}

__device__ __forceinline__ unsigned long long warp_sum(unsigned long long x) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

template <int DT>
__global__ void __launch_bounds__(kFiltThreads, 2) filter_kernel(const __grid_constant__ FiltParams P) {
  using K = Keys<DT>;
  constexpr int kKeyBits = 8 * K::kES;
  extern __shared__ __align__(16) unsigned long long s_h[];   // [256 buckets][32 lanes], then the list
  uint32_t* const s_cnt = reinterpret_cast<uint32_t*>(s_h);
  unsigned long long* const s_cand = s_h + kHistWords;       // (element index << 32) | raw
  __shared__ unsigned long long s_b[256];                      // bucket totals
  __shared__ __align__(16) float s_tmax[kFiltThreads];         // each thread's own max
  __shared__ float s_max[kFiltThreads / 32];
  __shared__ double s_dsum[kFiltThreads / 32];                 // warp parts of the row's total
  __shared__ int s_d, s_n;
  __shared__ unsigned long long s_cum, s_in, s_sum;
  const int V = P.V, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  auto zero_hist = [&](int words64) {
    uint4* z = reinterpret_cast<uint4*>(s_h);
    for (int i = tid; i < words64 / 2; i += kFiltThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
  };
  auto block_max = [&](float v) -> float {   // every thread gets the CTA's max of v
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if (lane == 0) s_max[warp] = v;
    __syncthreads();
    float r = s_max[0];
    for (int w = 1; w < kFiltThreads / 32; ++w) r = fmaxf(r, s_max[w]);
    __syncthreads();
    return r;
  };

  auto rank_bound = [&](float mt, int rank) -> float {   // the rank-th largest thread max (rank <= threads)
    s_tmax[tid] = mt;
    __syncthreads();
    int c = 0;
    const float4* t4 = reinterpret_cast<const float4*>(s_tmax);
#pragma unroll 4
    for (int j = 0; j < kFiltThreads / 4; ++j) {
      const float4 q = t4[j];
      c += (q.x >= mt) + (q.y >= mt) + (q.z >= mt) + (q.w >= mt);
    }
    return block_max(c >= rank ? mt : -INFINITY);
  };
  auto block_sum = [&](unsigned long long v) -> unsigned long long {   // s_sum must be zero before
    v = warp_sum(v);
    if (lane == 0 && v) atomicAdd(&s_sum, v);
    __syncthreads();
    const unsigned long long t = s_sum;
    __syncthreads();
    return t;
  };

  auto block_dsum = [&](double v) -> double {   // fixed-order fp64 sum over the CTA
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) s_dsum[warp] = v;
    __syncthreads();
    double t = 0.0;
    for (int w = 0; w < kFiltThreads / 32; ++w) t += s_dsum[w];
    __syncthreads();
    return t;
  };

  for (int r = blockIdx.x; r < P.n; r += gridDim.x) {
    unsigned char* row = P.logits + (size_t)r * V * K::kES;
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

    // pass A: the row max and a NaN or +inf logit; with a large k, also top-k's
    // first level (counts of the keys' top byte)
    constexpr int sh0 = kKeyBits - 8;
    const bool by_sample = use_k && k <= kFiltThreads;
    const bool hist_in_a = use_k && !by_sample;
    const bool p_alone = use_p && !use_k;
    // top-p's scale: log2(e)/T as c + c_lo, applied as a stretch by ks
    float c = 0.f, ks = 0.f, unit = 0.f;
    if (use_p) {
      c = scale_of(T);
      const float c_lo = (float)(1.4426950408889634 / (double)T - (double)c);
      ks = scale_k(c, c_lo);
      int lg = 0;
      while ((1 << lg) < V) ++lg;
      unit = __int_as_float((127 + 61 - lg) << 23);        // 2^(61 - ceil(log2 V))
    }
    // pass S: each thread's max over a quarter of the row (every fourth block
    // of kFiltThreads vectors).  Any subset's k-th largest thread max bounds
    // the row's k-th largest logit from below; the CTA's max of it is a
    // provisional reference for top-p's weights.
    float ms = -INFINITY;
    if (by_sample || p_alone) {
      const Span<DT> sp(row, V);
      const uint4* body = reinterpret_cast<const uint4*>(row + (size_t)sp.head * K::kES);
#pragma unroll 4
      for (int i = tid; i < sp.nvec; i += 4 * kFiltThreads) {
        const uint4 w = body[i];
        if constexpr (DT == SPEC_BF16) {
          __nv_bfloat162 a = __hmax2(__hmax2(as_bf2(w.x), as_bf2(w.y)), __hmax2(as_bf2(w.z), as_bf2(w.w)));
          const uint32_t b = bf2_bits(a);
          ms = fmaxf(ms, fmaxf(K::value(b & 0xFFFFu), K::value(b >> 16)));
        } else {
          ms = fmaxf(ms, fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                               fmaxf(__uint_as_float(w.z), __uint_as_float(w.w))));
        }
      }
    }
    const float m_s = p_alone ? block_max(ms) : -INFINITY;
    const bool fused_p = p_alone && m_s > -INFINITY && m_s < INFINITY;
    auto put = [&](uint32_t h, int v) {   // onto the list
      const int slot = atomicAdd(&s_n, 1);
      if (slot < kCap) s_cand[slot] = ((unsigned long long)v << 32) | h;
    };
    float mt = -INFINITY;                                      // this thread's max
    int bad = 0;
    double tot_s = 0.0;                                        // top-p alone: the mass on m_s
    if (hist_in_a) {
      zero_hist(kHistWords / 2);
      __syncthreads();
      each_raw<DT>(row, V, [&](uint32_t h) {
        const float x = K::value(h);
        bad |= (x != x) || x == INFINITY;
        mt = fmaxf(mt, x);
        atomicAdd(&s_cnt[((K::key(h) >> sh0) & 255u) * 32 + lane], 1u);
      });
    } else if (by_sample) {
      // pass A with C: the max, the non-finite check, and every logit >= the
      // k-th largest sampled thread max to the list
      const float lb = rank_bound(ms, k);
      if (tid == 0) s_n = 0;
      __syncthreads();
      if constexpr (DT == SPEC_BF16) {
        __nv_bfloat162 mx = as_bf2(K::kNegInf * 0x00010001u);
        const __nv_bfloat162 lb2 = __float2bfloat162_rn(lb);
        each_word_at<DT>(
            row, V,
            [&](uint32_t h, int v) {
              mx = __hmax2_nan(mx, as_bf2(h * 0x00010001u));
              if (K::value(h) >= lb) put(h, v);
            },
            [&](uint32_t w, int v) {
              mx = __hmax2_nan(mx, as_bf2(w));
              const uint32_t in = __hge2_mask(as_bf2(w), lb2);
              if (in) {
                if (in & 0xFFFFu) put(w & 0xFFFFu, v);
                if (in >> 16) put(w >> 16, v + 1);
              }
            });
        const uint32_t b = bf2_bits(mx);
        const float lo = K::value(b & 0xFFFFu), hi = K::value(b >> 16);
        bad = (lo != lo) || (hi != hi) || lo == INFINITY || hi == INFINITY;
        mt = fmaxf(lo, hi);
      } else {
        each_raw_at<DT>(row, V, [&](uint32_t h, int v) {
          const float x = K::value(h);
          bad |= (x != x) || x == INFINITY;
          mt = fmaxf(mt, x);
          if (x >= lb) put(h, v);
        });
      }
    } else if (fused_p) {
      // pass A with C for top-p alone: the max, the non-finite check, the row's
      // mass on the reference m_s (a compensated fp32 sum per thread; rescaled
      // to the row max below) and the logits above a sampled thread-max rank
      const float lb = rank_bound(ms, kRankPS);
      const float nrs = -ref_of(m_s, c);
      if (tid == 0) s_n = 0;
      __syncthreads();
      // a vector's weights are summed by a fixed tree, and only that sum
      // enters the compensated sum: a short serial chain per 16 bytes
      float sf = 0.f, cf = 0.f;
      auto kahan = [&](float y) {
        y -= cf;
        const float t = sf + y;
        cf = (t - sf) - y;
        sf = t;
      };
      auto wt = [&](float x) { return ex2(stretch(fmaf(x, c, nrs), ks)); };
      auto one = [&](uint32_t h, int v) {   // a head or tail element
        const float x = K::value(h);
        kahan(wt(x));
        if (x >= lb) put(h, v);
      };
      if constexpr (DT == SPEC_BF16) {
        __nv_bfloat162 mx = as_bf2(K::kNegInf * 0x00010001u);
        const __nv_bfloat162 lb2 = __float2bfloat162_rn(lb);
        each_vec_at<DT>(
            row, V,
            [&](uint32_t h, int v) {
              mx = __hmax2_nan(mx, as_bf2(h * 0x00010001u));
              one(h, v);
            },
            [&](const uint4& q, int v) {
              const uint32_t w[4] = {q.x, q.y, q.z, q.w};
              float e[8];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                mx = __hmax2_nan(mx, as_bf2(w[j]));
                e[2 * j] = wt(K::value(w[j] & 0xFFFFu));
                e[2 * j + 1] = wt(K::value(w[j] >> 16));
              }
              kahan(((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7])));
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t in = __hge2_mask(as_bf2(w[j]), lb2);
                if (in) {
                  if (in & 0xFFFFu) put(w[j] & 0xFFFFu, v + 2 * j);
                  if (in >> 16) put(w[j] >> 16, v + 2 * j + 1);
                }
              }
            });
        const uint32_t b = bf2_bits(mx);
        const float lo = K::value(b & 0xFFFFu), hi = K::value(b >> 16);
        bad = (lo != lo) || (hi != hi) || lo == INFINITY || hi == INFINITY;
        mt = fmaxf(lo, hi);
      } else {
        auto chk = [&](float x) {
          bad |= (x != x) || x == INFINITY;
          mt = fmaxf(mt, x);
        };
        each_vec_at<DT>(
            row, V,
            [&](uint32_t h, int v) {
              chk(K::value(h));
              one(h, v);
            },
            [&](const uint4& q, int v) {
              const float x[4] = {__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z),
                                  __uint_as_float(q.w)};
#pragma unroll
              for (int j = 0; j < 4; ++j) chk(x[j]);
              kahan((wt(x[0]) + wt(x[1])) + (wt(x[2]) + wt(x[3])));
              const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (x[j] >= lb) put(u[j], v + j);
            });
      }
      tot_s = block_dsum((double)sf - (double)cf);
    } else if constexpr (DT == SPEC_BF16) {
      __nv_bfloat162 mx = as_bf2(K::kNegInf * 0x00010001u);
      each_word<DT>(row, V, [&](uint32_t h) { mx = __hmax2_nan(mx, as_bf2(h * 0x00010001u)); },
                    [&](uint32_t w) { mx = __hmax2_nan(mx, as_bf2(w)); });
      const uint32_t b = bf2_bits(mx);
      const float lo = K::value(b & 0xFFFFu), hi = K::value(b >> 16);
      bad = (lo != lo) || (hi != hi) || lo == INFINITY || hi == INFINITY;
      mt = fmaxf(lo, hi);
    } else {
      each_raw<DT>(row, V, [&](uint32_t h) {
        const float x = K::value(h);
        bad |= (x != x) || x == INFINITY;
        mt = fmaxf(mt, x);
      });
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0 && P.status) P.status[r] = SPEC_ST_NONFINITE;
      continue;
    }
    const float m = block_max(mt);
    if (m == -INFINITY) {
      if (tid == 0 && P.status) P.status[r] = SPEC_ST_NONFINITE;
      continue;
    }

    // the keys later levels look at: the whole row, or the list C collects
    bool on_list = false;
    int n_list = 0;
    auto each_key = [&](auto&& f) {
      if (on_list) {
        for (int i = tid; i < n_list; i += kFiltThreads) f((uint32_t)s_cand[i]);
      } else {
        each_raw<DT>(row, V, f);
      }
    };
    auto collect = [&](float lo) {   // pass C: every logit >= lo, to the list (any order)
      if (tid == 0) s_n = 0;
      __syncthreads();
      each_in_range_at<DT>(row, V, lo, INFINITY, [&](uint32_t h, int v) {
        if (K::value(h) >= lo) {
          const int slot = atomicAdd(&s_n, 1);
          if (slot < kCap) s_cand[slot] = ((unsigned long long)v << 32) | h;
        }
      });
      __syncthreads();
      if (s_n <= kCap) {
        on_list = true;
        n_list = s_n;
      }
      __syncthreads();
    };

    // top-k: the key of the k-th largest logit (radix descent on counts)
    uint32_t thr = 0u;                                         // keep keys >= thr
    if (use_k) {
      uint32_t prefix = 0u;
      unsigned long long above = 0ull;
      int L = 0;
      auto count_level = [&](int lv) {   // histogram of level lv among the prefix's keys, then descend
        const int sh = kKeyBits - 8 * (lv + 1);
        zero_hist(kHistWords / 2);
        __syncthreads();
        each_key([&](uint32_t h) {
          const uint32_t key = K::key(h);
          if (lv == 0 || (key >> (sh + 8)) == (prefix >> (sh + 8)))
            atomicAdd(&s_cnt[((key >> sh) & 255u) * 32 + lane], 1u);
        });
        __syncthreads();
      };
      auto pick = [&](int lv) {
        bucket_totals(s_cnt, s_b, tid);
        __syncthreads();
        if (warp == 0) descend(s_b, above, (double)k, lane, &s_d, &s_cum, &s_in);
        __syncthreads();
        prefix |= (uint32_t)s_d << (kKeyBits - 8 * (lv + 1));
        above = s_cum;
      };
      if (by_sample && s_n <= kCap) {   // the list pass A filled
        on_list = true;
        n_list = s_n;
      }
      if (!on_list) {
        if (!hist_in_a) count_level(0);
        pick(0);
        L = 1;
        if (above + s_in <= (unsigned long long)kCap) collect(value_of<DT>(prefix));
      }
      for (; L < K::kLevels; ++L) {
        count_level(L);
        pick(L);
      }
      thr = prefix;
    }

    // top-p: the key of t* (radix descent on fixed-point masses)
    if (use_p) {
      const float nr = -ref_of(m, c);
      auto weight = [&](float x) -> unsigned long long {
        const float w = ex2(stretch(fmaf(x, c, nr), ks));
        return __float2ull_rz(w * unit);
      };
      double need = -1.0;                                      // known before the levels when >= 0
      if (!use_k) {
        double tot;                                            // the row's mass on the row max
        if (fused_p) {   // pass A summed it on m_s: 2^{(R(m_s) - R(m))(1 + ks)} rescales it
          tot = tot_s * exp2(((double)ref_of(m_s, c) - (double)ref_of(m, c)) * (1.0 + (double)ks));
        } else {
          // pass C: the row's total mass, and the logits at or above a bound
          const float lb = rank_bound(mt, kRankP);
          if (tid == 0) s_n = 0;
          __syncthreads();
          float sf = 0.f, cf = 0.f;                            // compensated (Kahan) fp32 sum
          each_raw_at<DT>(row, V, [&](uint32_t h, int v) {
            const float x = K::value(h);
            const float y = ex2(stretch(fmaf(x, c, nr), ks)) - cf;
            const float t = sf + y;
            cf = (t - sf) - y;
            sf = t;
            if (x >= lb) put(h, v);
          });
          tot = block_dsum((double)sf - (double)cf);         // fixed-order fp64 reduction
        }
        const double want = (double)tp * tot * (double)unit;
        if (s_n <= kCap) {   // the list's own mass: t* is on it when that reaches the target
          if (tid == 0) s_sum = 0ull;
          __syncthreads();
          const int nl = s_n;
          unsigned long long lm = 0ull;
          for (int i = tid; i < nl; i += kFiltThreads) lm += weight(K::value((uint32_t)s_cand[i]));
          if ((double)block_sum(lm) >= want) {
            on_list = true;
            n_list = nl;
            need = want;
          }
        }
      }
      uint32_t prefix = 0u;
      unsigned long long above = 0ull;
      for (int L = 0; L < K::kLevels; ++L) {
        const int sh = kKeyBits - 8 * (L + 1);
        zero_hist(kHistWords);
        __syncthreads();
        uint32_t cb = 0xFFFFFFFFu;                             // this thread's pending bucket and mass:
        unsigned long long ca = 0ull;                          // neighbours often share a bucket
        auto add = [&](uint32_t h) {
          const uint32_t key = K::key(h);
          if (key >= thr && (L == 0 || (key >> (sh + 8)) == (prefix >> (sh + 8)))) {
            const unsigned long long w = weight(K::value(h));
            const uint32_t bk = (key >> sh) & 255u;
            if (bk != cb) { if (ca) atomicAdd(&s_h[cb * 32 + lane], ca); cb = bk; ca = w; } else ca += w;
          }
        };
        if (L == 0 || on_list) {
          each_key(add);
        } else {   // the prefix's key range, by a packed value test first
          const uint32_t lo_key = (prefix >> (sh + 8)) << (sh + 8);
          const uint32_t hi_key = lo_key | ((2u << (sh + 7)) - 1u);
          each_in_range<DT>(row, V, value_of<DT>(lo_key > thr ? lo_key : thr), value_of<DT>(hi_key), add);
        }
        if (ca) atomicAdd(&s_h[cb * 32 + lane], ca);
        __syncthreads();
        bucket_totals(s_h, s_b, tid);
        __syncthreads();
        if (warp == 0) {
          if (L == 0 && need < 0.0) {   // the total mass of what top-k keeps, and the upper mass to reach
            unsigned long long t = 0ull;
#pragma unroll
            for (int j = 0; j < 8; ++j) t += s_b[lane * 8 + j];
            need = (double)tp * (double)warp_sum(t);
          }
          descend(s_b, above, need, lane, &s_d, &s_cum, &s_in);
        }
        __syncthreads();
        prefix |= (uint32_t)s_d << sh;
        above = s_cum;
      }
      if (prefix > thr) thr = prefix;
    }

    // pass K: the removed logits become -inf.  On the list every kept logit is
    // known with its index: fill the row, then put those back (no row read).
    if (on_list) {
      fill_neg_inf<DT>(row, V);
      __syncthreads();
      for (int i = tid; i < n_list; i += kFiltThreads) {
        const unsigned long long e = s_cand[i];
        const uint32_t h = (uint32_t)e;
        if (K::key(h) >= thr) {
          const int v = (int)(e >> 32);
          if constexpr (DT == SPEC_BF16) reinterpret_cast<uint16_t*>(row)[v] = (uint16_t)h;
          else reinterpret_cast<uint32_t*>(row)[v] = h;
        }
      }
    } else if (thr > 0u) {
      kill_below<DT>(row, V, value_of<DT>(thr));
    }
    if (tid == 0 && P.status) P.status[r] = 0;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_filter(const FiltParams& P, int grid, cudaStream_t s) {
  cudaError_t e;
  if (P.dtype == SPEC_BF16) {
    e = cudaFuncSetAttribute(filter_kernel<SPEC_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFiltSmem);
    if (e == cudaSuccess) filter_kernel<SPEC_BF16><<<grid, kFiltThreads, kFiltSmem, s>>>(P);
  } else {
    e = cudaFuncSetAttribute(filter_kernel<SPEC_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFiltSmem);
    if (e == cudaSuccess) filter_kernel<SPEC_F32><<<grid, kFiltThreads, kFiltSmem, s>>>(P);
  }
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace sv
