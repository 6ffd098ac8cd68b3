// One recurrent decode step, in place on the fp32 state.
//
// "Linear Attention Mechanisms" (dileepadev.github.io), "Recurrent
// Reformulation": S <- gamma S + phi(k) v^T, z <- gamma z + phi(k), then
// o = phi(q)^T S / (phi(q) . z + eps) with the updated state.  The gated form
// of "Gating and Selective State Updates" scales row d of S and entry d of z
// by a[d] instead of one gamma per head (a gate per key feature).  Per token this
// reads and rewrites the whole D x Dv state, so the step is bound by HBM
// bandwidth: the kernel streams each state once with 16-byte accesses, keeps
// every load of a thread in flight at once, and fuses the read-out into the
// update so the state is touched exactly once.
//
// One CTA per (batch, head).  Lane l of every warp owns Dv/32 consecutive
// columns; warp w owns rows d = w*D/8 .. (w+1)*D/8 - 1.  The read-out is a
// column sum over d: per-warp partial sums meet in shared memory.
#include "common.cuh"
#include "kernels.h"

namespace linattn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int N>
struct vec;
template <>
struct vec<4> {
  using type = float4;
};
template <>
struct vec<2> {
  using type = float2;
};

__device__ __forceinline__ void to_arr(const float4 &x, float *a) {
  a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
}
__device__ __forceinline__ void to_arr(const float2 &x, float *a) {
  a[0] = x.x; a[1] = x.y;
}
__device__ __forceinline__ float4 from_arr4(const float *a) {
  return make_float4(a[0], a[1], a[2], a[3]);
}
__device__ __forceinline__ float2 from_arr2(const float *a) {
  return make_float2(a[0], a[1]);
}

// MODE: kPlain (no decay), kGamma (one gamma per head), kGate (a[d] per key
// feature, a: [B*H][D] fp32).
enum { kPlain = 0, kGamma = 1, kGate = 2 };

template <int D, int DV, int MODE, typename T>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const T *__restrict__ q, const T *__restrict__ k,
                  const T *__restrict__ v, const float *__restrict__ a,
                  float *__restrict__ S, float *__restrict__ z, T *__restrict__ o,
                  int H, float eps, const __grid_constant__ Gammas gam) {
  constexpr int EPL = DV / 32;         // columns per lane
  constexpr int RPW = D / kWarps;      // rows per warp
  using V = typename vec<EPL>::type;
  __shared__ float fq[D], fk[D], vv[DV], ga[D];
  __shared__ float part[kWarps][DV];
  __shared__ float qz_part[kWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = blockIdx.x;
  const float g = MODE == kGamma ? gam.g[u % H] : 1.f;
  float *Su = S + u * (int64_t)D * DV;
  const int e0 = lane * EPL;
  const int d0 = warp * RPW;

  // Issue every state load of this thread before anything else.
  float s[RPW][EPL];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const V x = __ldcs(reinterpret_cast<const V *>(Su + (int64_t)(d0 + r) * DV + e0));
    to_arr(x, s[r]);
  }
  for (int i = tid; i < D; i += kThreads) {
    fq[i] = phi_f32(io<T>::load(q + u * D + i));
    fk[i] = phi_f32(io<T>::load(k + u * D + i));
    if (MODE == kGate) ga[i] = a[u * D + i];
  }
  for (int i = tid; i < DV; i += kThreads) vv[i] = io<T>::load(v + u * DV + i);
  __syncthreads();
  // z update and the phi(q).z partial sums (threads 0..D-1)
  float qz = 0.f;
  if (tid < D) {
    const float gz = MODE == kGate ? ga[tid] : g;
    const float zn = MODE != kPlain ? fmaf(gz, z[u * D + tid], fk[tid]) : z[u * D + tid] + fk[tid];
    z[u * D + tid] = zn;
    qz = fq[tid] * zn;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) qz += __shfl_xor_sync(0xffffffffu, qz, off);
  if (lane == 0) qz_part[warp] = qz;

  float ve[EPL], acc[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    ve[j] = vv[e0 + j];
    acc[j] = 0.f;
  }
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const float kd = fk[d0 + r], qd = fq[d0 + r];
    const float gr = MODE == kGate ? ga[d0 + r] : g;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const float sn = MODE != kPlain ? fmaf(gr, s[r][j], kd * ve[j]) : fmaf(kd, ve[j], s[r][j]);
      s[r][j] = sn;
      acc[j] = fmaf(qd, sn, acc[j]);
    }
    V out;
    if constexpr (EPL == 4) out = from_arr4(s[r]); else out = from_arr2(s[r]);
    __stcs(reinterpret_cast<V *>(Su + (int64_t)(d0 + r) * DV + e0), out);
  }
#pragma unroll
  for (int j = 0; j < EPL; ++j) part[warp][e0 + j] = acc[j];
  __syncthreads();
  float den = eps;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) den += qz_part[w];
  for (int e = tid; e < DV; e += kThreads) {
    float num = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) num += part[w][e];
    io<T>::store(o + u * DV + e, num / den);
  }
}

template <int D, int DV, int MODE, typename T>
cudaError_t dec_typed(const void *q, const void *k, const void *v, const float *a,
                      float *S, float *z, void *o, int BH, int H, float eps,
                      const Gammas &g, cudaStream_t s) {
  decode_kernel<D, DV, MODE, T><<<(unsigned)BH, kThreads, 0, s>>>(
      static_cast<const T *>(q), static_cast<const T *>(k),
      static_cast<const T *>(v), a, S, z, static_cast<T *>(o), H, eps, g);
  return cudaGetLastError();
}

template <int D, int DV, typename T>
cudaError_t dec_mode(const void *q, const void *k, const void *v, const float *a,
                     float *S, float *z, void *o, int BH, int H, int mode, float eps,
                     const Gammas &g, cudaStream_t s) {
  if (mode == kGate) return dec_typed<D, DV, kGate, T>(q, k, v, a, S, z, o, BH, H, eps, g, s);
  if (mode == kGamma) return dec_typed<D, DV, kGamma, T>(q, k, v, a, S, z, o, BH, H, eps, g, s);
  return dec_typed<D, DV, kPlain, T>(q, k, v, a, S, z, o, BH, H, eps, g, s);
}

template <typename T>
cudaError_t dec_shape(const void *q, const void *k, const void *v, const float *a,
                      float *S, float *z, void *o, int BH, int H, int D, int Dv,
                      int mode, float eps, const Gammas &g, cudaStream_t s) {
  if (D == 64 && Dv == 64) return dec_mode<64, 64, T>(q, k, v, a, S, z, o, BH, H, mode, eps, g, s);
  if (D == 64 && Dv == 128) return dec_mode<64, 128, T>(q, k, v, a, S, z, o, BH, H, mode, eps, g, s);
  if (D == 128 && Dv == 64) return dec_mode<128, 64, T>(q, k, v, a, S, z, o, BH, H, mode, eps, g, s);
  if (D == 128 && Dv == 128) return dec_mode<128, 128, T>(q, k, v, a, S, z, o, BH, H, mode, eps, g, s);
  return cudaErrorNotSupported;
}

cudaError_t dec_dispatch(const void *q, const void *k, const void *v, const float *a,
                         float *S, float *z, void *o, int B, int H, int D, int Dv, int mode,
                         const Gammas &g, float eps, Dtype dt, cudaStream_t s) {
  const int BH = B * H;
  return dt == kF32
             ? dec_shape<float>(q, k, v, a, S, z, o, BH, H, D, Dv, mode, eps, g, s)
             : dec_shape<__nv_bfloat16>(q, k, v, a, S, z, o, BH, H, D, Dv, mode, eps, g, s);
}

}  // namespace

cudaError_t launch_decode_step(const void *q, const void *k, const void *v,
                               float *S, float *z, void *o, int B, int H,
                               int D, int Dv, bool decay, const Gammas &g,
                               float eps, Dtype dt, cudaStream_t s) {
  return dec_dispatch(q, k, v, nullptr, S, z, o, B, H, D, Dv, decay ? kGamma : kPlain, g, eps,
                      dt, s);
}

cudaError_t launch_decode_gated(const void *q, const void *k, const void *v, const float *a,
                                float *S, float *z, void *o, int B, int H, int D, int Dv,
                                float eps, Dtype dt, cudaStream_t s) {
  Gammas none;
  for (int h = 0; h < kMaxHeads; ++h) none.g[h] = 1.f;
  return dec_dispatch(q, k, v, a, S, z, o, B, H, D, Dv, kGate, none, eps, dt, s);
}

}  // namespace linattn
