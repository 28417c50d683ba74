// gamma.cu -- the SpecKV gamma selector on the draft signals.
//
// The SpecKV page ("接受率预测与 gamma 选择", acceptance prediction and gamma
// selection): with the context x = [mean H, mean c, max H, min c, comp] of a
// request, a regressor f(x, gamma) predicts the acceptance rate; the expected
// tokens of a step are f(x, gamma) gamma + 1 and the policy takes
// gamma* = argmax over gamma in {2, 4, 6, 8}; f is an MLP with 16 hidden
// units.  Here its inputs are [x, gamma], standardised as (z - mu) / sd, with
// one ReLU hidden layer and an identity output; ties go to the smaller gamma.
// One thread per request; the 141 model values are staged in shared memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace sv {
namespace {

constexpr int kGselThreads = 256;

__global__ void __launch_bounds__(kGselThreads) gamma_select_kernel(const float* __restrict__ signals,
                                                                    const float* __restrict__ comp,
                                                                    const float* __restrict__ model, int B,
                                                                    int32_t* __restrict__ gamma_star,
                                                                    float* __restrict__ expected) {
  __shared__ float m[kGammaModelFloats];
  for (int k = threadIdx.x; k < kGammaModelFloats; k += blockDim.x) m[k] = model[k];
  __syncthreads();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const float* mu = m;
  const float* sd = m + 6;
  const float* W1 = m + 12;
  const float* b1 = m + 108;
  const float* w2 = m + 124;
  const float b2 = m[140];
  const float4 s = reinterpret_cast<const float4*>(signals)[b];   // mean H, max H, mean c, min c
  const float x[5] = {s.x, s.z, s.y, s.w, comp ? comp[b] : 0.f};  // [mean H, mean c, max H, min c, comp]
  bool finite = true;
#pragma unroll
  for (int k = 0; k < 5; ++k) finite &= isfinite(x[k]);
  float z[6];
#pragma unroll
  for (int k = 0; k < 5; ++k) z[k] = (x[k] - mu[k]) / sd[k];
  int best = -1;
  float bestE = -INFINITY;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int g = 2 + 2 * j;
    z[5] = ((float)g - mu[5]) / sd[5];
    float f = b2;
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      float a = b1[h];
#pragma unroll
      for (int k = 0; k < 6; ++k) a = fmaf(W1[h * 6 + k], z[k], a);
      f = fmaf(w2[h], fmaxf(a, 0.f), f);
    }
    const float E = finite ? fmaf(f, (float)g, 1.f) : __int_as_float(0x7fc00000);
    if (finite && E > bestE) {
      bestE = E;
      best = g;
    }
    if (expected) expected[(size_t)b * 4 + j] = E;
  }
  gamma_star[b] = finite ? best : -1;
}

}  // namespace

cudaError_t launch_gamma_select(const float* signals, const float* comp, const float* model, int B,
                                int32_t* gamma_star, float* expected, cudaStream_t s) {
  const int grid = (B + kGselThreads - 1) / kGselThreads;
  gamma_select_kernel<<<grid, kGselThreads, 0, s>>>(signals, comp, model, B, gamma_star, expected);
  return cudaGetLastError();
}

}  // namespace sv
