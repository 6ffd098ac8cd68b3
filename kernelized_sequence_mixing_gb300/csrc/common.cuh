// Device helpers shared by the library's kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace linattn {

// phi(x) = elu(x) + 1 with alpha = 1: x + 1 for x > 0, exp(x) otherwise
// ("Linear Attention Mechanisms" (dileepadev.github.io), "Choosing the
// Feature Map", ELU-based features).  exp(x) is taken directly rather than as
// (exp(x) - 1) + 1, so phi stays positive and exact at 0.
__device__ __forceinline__ float phi_f32(float x) {
  return x > 0.f ? x + 1.f : expf(x);
}

// The feature map a kernel applies to its q, k inputs: phi, or the identity
// when the inputs already are features.
template <bool IDENT>
__device__ __forceinline__ float feat_f32(float x) {
  if constexpr (IDENT) return x;
  else return phi_f32(x);
}

template <typename T> struct io;
template <> struct io<float> {
  static __device__ __forceinline__ float load(const float *p) { return *p; }
  static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
};
template <> struct io<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
  }
};

// gamma^k for k = 0..n, built in fp64 by repeated multiplication and rounded
// once to fp32 (gamma^0 = 1 also for gamma = 0).  One thread writes it.
__device__ __forceinline__ void build_pow_table(float *G, int n, float gamma) {
  double g = 1.0;
  for (int k = 0; k <= n; ++k) {
    G[k] = (float)g;
    g *= (double)gamma;
  }
}

}  // namespace linattn
