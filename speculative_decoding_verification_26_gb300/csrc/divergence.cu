// divergence.cu -- per-position divergence statistics of a draft chain.
//
// For each request b and position i < gamma_b, with p = softmax(target row
// i / T_b) and q = softmax(draft row i / T_b), five statistics in bits:
//   A   = sum_v min(p(v), q(v))  (= 1 - TV(p, q), the position's expected
//         acceptance: tutorial page "5.1 投机解码核心原理", section 4.3);
//   L1  = sum_v |p(v) - q(v)|    (the L1 / TV distance of the DLite page's
//         distillation loss, an input of the DDTE page's selector);
//   KL(p||q) = sum p log2(p/q), KL(q||p) (forward KL of the DLite page, the
//         DDTE page's "bidirectional KL"), and H(p) = -sum p log2 p (the
//         target entropy of the DDTE page's selector inputs).
//
// divergence_kernel is persistent, one CTA per SM, looping over the (request,
// position) pairs.  A pair is read twice: pass 1 keeps an online max and sum
// of both rows per thread (the exponent of the verify kernel: fl(x c - R(m))
// stretched by the scale's remainder, see ref_of), reduced over the CTA; pass 2
// re-reads the pair (from L2: at most one pair per SM is in flight, ~92 MB
// for 152 SMs at V = 151 936 bf16) and sums the per-token terms with the final
// row sums known.  Every term of pass 2 is non-negative or a difference of
// two small logarithms, so no sum cancels between large partials: A, L1 and
// H near 0 or 1 keep their relative precision.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace sv {
namespace {

constexpr int kDivThreads = 512;
constexpr int kDivWarps = kDivThreads / 32;
constexpr int kLoadsAhead = 4;      // 16-byte vectors per row a thread has in flight

struct Acc {
  float m, s;       // running max and sum of 2^a (relative to R(m))
};

__device__ __forceinline__ void acc_reset(Acc& a) { a.m = -INFINITY; a.s = 0.f; }

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Add logits x[0..n) to a running (m, s) with the shared exponent rule.
template <int N>
__device__ __forceinline__ void acc_add(Acc& a, const float (&x)[N], float c, float ks) {
  float vm = -INFINITY;
#pragma unroll
  for (int k = 0; k < N; ++k) vm = fmaxf(vm, x[k]);
  if (vm > a.m) {
    if (a.m != -INFINITY) a.s *= ex2(stretch(__fsub_rn(ref_of(a.m, c), ref_of(vm, c)), ks));
    a.m = vm;
  }
  if (a.m == -INFINITY) return;
  const float nr = -ref_of(a.m, c);
  if constexpr (N % 2 == 0) {   // packed fp32 pairs: the same roundings per lane
    const float2 C2 = f2(c, c), K2 = f2(ks, ks), NR2 = f2(nr, nr);
    float2 t2 = f2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < N; k += 2) {
      float2 e = __ffma2_rn(f2(x[k], x[k + 1]), C2, NR2);
      e = __ffma2_rn(e, K2, e);                           // stretch
      t2 = __fadd2_rn(t2, f2(ex2(e.x), ex2(e.y)));
    }
    a.s += t2.x + t2.y;
  } else {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < N; ++k) t += ex2(stretch(fmaf(x[k], c, nr), ks));
    a.s += t;
  }
}

// Merge two partials (the online-softmax rule).
__device__ __forceinline__ Acc acc_merge(Acc a, Acc b, float c, float ks) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return a;
  Acc o;
  o.m = m;
  o.s = 0.f;
  if (a.s != 0.f) o.s += a.s * ex2(stretch(__fsub_rn(ref_of(a.m, c), ref_of(m, c)), ks));
  if (b.s != 0.f) o.s += b.s * ex2(stretch(__fsub_rn(ref_of(b.m, c), ref_of(m, c)), ks));
  return o;
}

// The five sums of pass 2 (per thread, then over the CTA).
struct Sums {
  float A, L1, kpq, kqp, H;
};

template <int DT>
struct Row;
template <>
struct Row<SPEC_BF16> {
  static constexpr int N = 8;   // logits per 16-byte vector
  __device__ __forceinline__ static void unpack(uint4 w, float (&x)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) { x[2 * k] = bf16_lo(u[k]); x[2 * k + 1] = bf16_hi(u[k]); }
  }
};
template <>
struct Row<SPEC_F32> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(uint4 w, float (&x)[4]) {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
};

// Tokens of one thread per step: vectors when every row is 16-byte aligned,
// else single logits (coalesced scalar loads).
template <int DT, class F>
__device__ __forceinline__ void for_pair(const unsigned char* trow, const unsigned char* drow, int V, bool vec, F&& f) {
  constexpr int N = Row<DT>::N;
  if (vec) {
    // kLoadsAhead vectors of each row are loaded before any is used (enough
    // bytes in flight per SM for HBM); the thread still visits its vectors
    // v, v + kDivThreads, ... in order
    constexpr int U = kLoadsAhead;
    const uint4* tv = reinterpret_cast<const uint4*>(trow);
    const uint4* dv = reinterpret_cast<const uint4*>(drow);
    const int nv = V / N;
    for (int v0 = threadIdx.x; v0 < nv; v0 += kDivThreads * U) {
      uint4 wt[U], wd[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * kDivThreads;
        if (v < nv) {
          wt[u] = __ldg(tv + v);
          wd[u] = __ldg(dv + v);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (v0 + u * kDivThreads < nv) {
          float xt[N], xd[N];
          Row<DT>::unpack(wt[u], xt);
          Row<DT>::unpack(wd[u], xd);
          f(xt, xd);
        }
      }
    }
  } else {
    for (int e = threadIdx.x; e < V; e += kDivThreads) {
      float xt[1] = {load_logit(trow, DT, e)}, xd[1] = {load_logit(drow, DT, e)};
      f(xt, xd);
    }
  }
}

__device__ __forceinline__ bool bad_logit(float x) { return x != x || x == INFINITY; }

template <int DT>
__global__ void __launch_bounds__(kDivThreads, 1) divergence_kernel(const __grid_constant__ DivParams P) {
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  __shared__ Acc s_p[kDivWarps], s_q[kDivWarps];
  __shared__ Sums s_sum[kDivWarps];
  __shared__ int s_bad[kDivWarps];  // per warp: a NaN or +inf logit in the pair
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = P.G, V = P.V;
  const int npairs = P.B * G;
  for (int pair = blockIdx.x; pair < npairs; pair += gridDim.x) {
    const int b = pair / G, i = pair % G;
    float* out = P.stats + (size_t)pair * 5;
    const int gam = P.gamma ? P.gamma[b] : G;
    const float T = P.temperature[b];
    int st = 0;
    if (gam < 0 || gam > G) st |= SPEC_ST_BAD_GAMMA;
    if (!temperature_ok(T)) st |= SPEC_ST_BAD_TEMPERATURE;
    if (st != 0 || i >= gam) {
      if (threadIdx.x < 5) out[threadIdx.x] = __int_as_float(0x7fc00000);
      if (threadIdx.x == 0 && st != 0 && i == 0 && P.status) atomicOr(P.status + b, st);
      continue;
    }
    const float c = scale_of(T);
    const float c_lo = (float)(1.4426950408889634 / (double)T - (double)c);
    const float ks = scale_k(c, c_lo);
    const unsigned char* trow = P.target + (size_t)((long long)b * (G + 1) + i) * V * ES;
    const unsigned char* drow = P.draft + (size_t)((long long)b * G + i) * V * ES;
    const bool vec = P.aligned;

    // pass 1: the max and sum of each row
    Acc ap, aq;
    acc_reset(ap);
    acc_reset(aq);
    bool bad = false;
    for_pair<DT>(trow, drow, V, vec, [&](auto& xt, auto& xd) {
      constexpr int n = sizeof(xt) / sizeof(float);
#pragma unroll
      for (int k = 0; k < n; ++k) bad |= bad_logit(xt[k]) || bad_logit(xd[k]);
      acc_add(ap, xt, c, ks);
      acc_add(aq, xd, c, ks);
    });
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      Acc o;
      o.m = __shfl_xor_sync(0xffffffffu, ap.m, off); o.s = __shfl_xor_sync(0xffffffffu, ap.s, off);
      ap = acc_merge(ap, o, c, ks);
      o.m = __shfl_xor_sync(0xffffffffu, aq.m, off); o.s = __shfl_xor_sync(0xffffffffu, aq.s, off);
      aq = acc_merge(aq, o, c, ks);
    }
    const bool wbad = __any_sync(0xffffffffu, bad);
    if (lane == 0) { s_p[warp] = ap; s_q[warp] = aq; s_bad[warp] = wbad; }
    __syncthreads();
    Acc fp = s_p[0], fq = s_q[0];
    int any_bad = s_bad[0];
    for (int w = 1; w < kDivWarps; ++w) {     // fixed order: every thread gets the same bits
      fp = acc_merge(fp, s_p[w], c, ks);
      fq = acc_merge(fq, s_q[w], c, ks);
      any_bad |= s_bad[w];
    }
    const bool row_bad = any_bad != 0 || fp.m == -INFINITY || fq.m == -INFINITY;
    if (row_bad) {
      if (threadIdx.x < 5) out[threadIdx.x] = __int_as_float(0x7fc00000);
      if (threadIdx.x == 0 && P.status) atomicOr(P.status + b, SPEC_ST_NONFINITE);
      __syncthreads();      // the shared partials are rewritten by the next pair
      continue;
    }

    // pass 2: the per-token terms with the final sums
    const float rp = 1.f / fp.s, rq = 1.f / fq.s;
    const float lsp = log2f(fp.s), lsq = log2f(fq.s);
    const float nrp = -ref_of(fp.m, c), nrq = -ref_of(fq.m, c);
    Sums sm{0.f, 0.f, 0.f, 0.f, 0.f};
    const float2 C2 = f2(c, c), K2 = f2(ks, ks), NRP2 = f2(nrp, nrp), NRQ2 = f2(nrq, nrq);
    const float2 RP2 = f2(rp, rp), RQ2 = f2(rq, rq), NLSP2 = f2(-lsp, -lsp), NLSQ2 = f2(-lsq, -lsq);
    const float2 M1 = f2(-1.f, -1.f);
    for_pair<DT>(trow, drow, V, vec, [&](auto& xt, auto& xd) {
      constexpr int n = sizeof(xt) / sizeof(float);
      Sums v{0.f, 0.f, 0.f, 0.f, 0.f};        // the vector's terms first, then the thread's sums
      if constexpr (n % 2 == 0) {
        // token pairs in packed fp32 (each lane rounds as the scalar form);
        // the KL and entropy terms stay per token, guarded for p or q = 0
        float2 vA = f2(0.f, 0.f), vL1 = f2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < n; k += 2) {
          float2 a1 = __ffma2_rn(f2(xt[k], xt[k + 1]), C2, NRP2);
          a1 = __ffma2_rn(a1, K2, a1);
          float2 a2 = __ffma2_rn(f2(xd[k], xd[k + 1]), C2, NRQ2);
          a2 = __ffma2_rn(a2, K2, a2);
          const float2 p = __fmul2_rn(f2(ex2(a1.x), ex2(a1.y)), RP2);
          const float2 q = __fmul2_rn(f2(ex2(a2.x), ex2(a2.y)), RQ2);
          const float2 lp = __fadd2_rn(a1, NLSP2), lq = __fadd2_rn(a2, NLSQ2);   // log2 p, log2 q
          const float2 d = __ffma2_rn(lq, M1, lp);          // log2 p - log2 q
          const float2 pq = __ffma2_rn(q, M1, p);           // p - q
          vA = __fadd2_rn(vA, f2(fminf(p.x, q.x), fminf(p.y, q.y)));
          vL1 = __fadd2_rn(vL1, f2(fabsf(pq.x), fabsf(pq.y)));
          if (p.x > 0.f) { v.kpq = fmaf(p.x, d.x, v.kpq); v.H = fmaf(-p.x, lp.x, v.H); }
          if (q.x > 0.f) v.kqp = fmaf(-q.x, d.x, v.kqp);
          if (p.y > 0.f) { v.kpq = fmaf(p.y, d.y, v.kpq); v.H = fmaf(-p.y, lp.y, v.H); }
          if (q.y > 0.f) v.kqp = fmaf(-q.y, d.y, v.kqp);
        }
        v.A = vA.x + vA.y;
        v.L1 = vL1.x + vL1.y;
      } else {
#pragma unroll
        for (int k = 0; k < n; ++k) {
          const float a1 = stretch(fmaf(xt[k], c, nrp), ks), a2 = stretch(fmaf(xd[k], c, nrq), ks);
          const float p = ex2(a1) * rp, q = ex2(a2) * rq;
          const float lp = a1 - lsp, lq = a2 - lsq;   // log2 p, log2 q
          v.A += fminf(p, q);
          v.L1 += fabsf(p - q);
          if (p > 0.f) { v.kpq += p * (lp - lq); v.H -= p * lp; }
          if (q > 0.f) v.kqp += q * (lq - lp);
        }
      }
      sm.A += v.A; sm.L1 += v.L1; sm.kpq += v.kpq; sm.kqp += v.kqp; sm.H += v.H;
    });
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      sm.A += __shfl_xor_sync(0xffffffffu, sm.A, off);
      sm.L1 += __shfl_xor_sync(0xffffffffu, sm.L1, off);
      sm.kpq += __shfl_xor_sync(0xffffffffu, sm.kpq, off);
      sm.kqp += __shfl_xor_sync(0xffffffffu, sm.kqp, off);
      sm.H += __shfl_xor_sync(0xffffffffu, sm.H, off);
    }
    if (lane == 0) s_sum[warp] = sm;
    __syncthreads();
    if (threadIdx.x == 0) {
      Sums t = s_sum[0];
      for (int w = 1; w < kDivWarps; ++w) {
        t.A += s_sum[w].A; t.L1 += s_sum[w].L1; t.kpq += s_sum[w].kpq; t.kqp += s_sum[w].kqp; t.H += s_sum[w].H;
      }
      out[0] = t.A; out[1] = t.L1; out[2] = t.kpq; out[3] = t.kqp; out[4] = t.H;
    }
    __syncthreads();        // the shared partials are rewritten by the next pair
  }
}

}  // namespace

cudaError_t launch_divergence(const DivParams& P, int grid, cudaStream_t s) {
  if (P.dtype == SPEC_BF16) divergence_kernel<SPEC_BF16><<<grid, kDivThreads, 0, s>>>(P);
  else divergence_kernel<SPEC_F32><<<grid, kDivThreads, 0, s>>>(P);
  return cudaGetLastError();
}

}  // namespace sv
