// Causal linear attention on CUDA cores (fp32 FFMA), chunked.
//
// The causal recurrence of "Linear Attention Mechanisms" (dileepadev.github.io),
// "Recurrent Reformulation", with the fixed decay of "Gating and Selective
// State Updates", evaluated a chunk of kC tokens at a time.  Within a chunk
// starting at c0, for local rows t and columns s (s <= t):
//   A_ts  = gamma^(t-s) phi(q_t).phi(k_s)
//   o_t   = (sum_s A_ts v_s + gamma^(t+1) phi(q_t)^T S_prev)
//           / (sum_s A_ts + gamma^(t+1) phi(q_t).z_prev + eps)
//   S_new = gamma^n S_prev + sum_s gamma^(n-1-s) phi(k_s) v_s^T  (n = rows)
//   z_new = gamma^n z_prev + sum_s gamma^(n-1-s) phi(k_s)
// which is the token-by-token recurrence regrouped: no term is dropped or
// approximated, only the summation order differs.
//
// All arithmetic is fp32.  This is the path for fp32 inputs (whose tolerance
// the bf16 tensor-core operands cannot meet) and the general fallback for
// shapes outside the tensor-core kernel's envelope.  One CTA owns one
// (batch, head) and a 32-column slice of Dv; the state slice S[:, slice] and
// z live in shared memory for the whole sequence.
#include "common.cuh"
#include "kernels.h"

namespace linattn {
namespace {

constexpr int kC = 64;  // tokens per chunk
constexpr int kThreads = 256;
constexpr int kLd = kC + 4;  // row stride of the transposed phi tiles
constexpr int kDvs = 32;     // Dv columns per CTA

template <int D>
struct SimtLayout {
  static constexpr int fqT = D * kLd;
  static constexpr int fkT = D * kLd;
  static constexpr int A = kC * (kC + 1);
  static constexpr int vs = kC * kDvs;
  static constexpr int S = D * kDvs;
  static constexpr int z = D;
  static constexpr int G = kC + 4;
  static constexpr int den = kC;
  static constexpr int total = fqT + fkT + A + vs + S + z + G + den;
  static constexpr size_t bytes = sizeof(float) * total;
};

template <int D, int DV, bool DECAY, bool IDENT, typename T>
__global__ void __launch_bounds__(kThreads)
    causal_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                       const T *__restrict__ v, T *__restrict__ o, int H,
                       int N, float eps, const __grid_constant__ Gammas gam) {
  extern __shared__ float4 smem4[];
  using L = SimtLayout<D>;
  float *fqT = reinterpret_cast<float *>(smem4);  // [D][kLd]  phi(q)^T
  float *fkT = fqT + L::fqT;                      // [D][kLd]  phi(k)^T
  float *As = fkT + L::fkT;                       // [kC][kC+1]
  float *vs = As + L::A;                          // [kC][kDvs]
  float *Ss = vs + L::vs;                         // [D][kDvs] state slice
  float *zs = Ss + L::S;                          // [D]
  float *G = zs + L::z;                           // gamma^k, k = 0..kC
  float *den = G + L::G;                          // [kC]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t bh = blockIdx.x;
  const int h = (int)(bh % H);
  const int e0 = blockIdx.y * kDvs;
  const T *qh = q + bh * (int64_t)N * D;
  const T *kh = k + bh * (int64_t)N * D;
  const T *vh = v + bh * (int64_t)N * DV;
  T *oh = o + bh * (int64_t)N * DV;

  for (int i = tid; i < D * kDvs; i += kThreads) Ss[i] = 0.f;
  for (int i = tid; i < D; i += kThreads) zs[i] = 0.f;
  if (tid == 0) {
    if (DECAY)
      build_pow_table(G, kC, gam.g[h]);
    else
      for (int i = 0; i <= kC; ++i) G[i] = 1.f;
  }
  __syncthreads();

  const int ty = tid >> 4, tx = tid & 15;  // 16 x 16 grid over the A tile
  for (int c0 = 0; c0 < N; c0 += kC) {
    const int nv = min(kC, N - c0);
    // 1. phi(q), phi(k) transposed into shared memory; v slice.  Rows past
    //    the end of the sequence are zero.  Every load of the chunk is issued
    //    before any is used, so the chunk pays one memory latency, not one
    //    per loop step.
    {
      constexpr int kQK = kC * D / kThreads, kV = kC * kDvs / kThreads;
      float xq[kQK], xk[kQK], xv[kV];
#pragma unroll
      for (int it = 0; it < kQK; ++it) {
        const int i = tid + it * kThreads, t = i / D, d = i % D;
        xq[it] = t < nv ? io<T>::load(qh + (int64_t)(c0 + t) * D + d) : 0.f;
        xk[it] = t < nv ? io<T>::load(kh + (int64_t)(c0 + t) * D + d) : 0.f;
      }
#pragma unroll
      for (int it = 0; it < kV; ++it) {
        const int i = tid + it * kThreads, t = i / kDvs, e = i % kDvs;
        xv[it] = t < nv ? io<T>::load(vh + (int64_t)(c0 + t) * DV + e0 + e) : 0.f;
      }
#pragma unroll
      for (int it = 0; it < kQK; ++it) {
        const int i = tid + it * kThreads, t = i / D, d = i % D;
        fqT[d * kLd + t] = t < nv ? feat_f32<IDENT>(xq[it]) : 0.f;
        fkT[d * kLd + t] = t < nv ? feat_f32<IDENT>(xk[it]) : 0.f;
      }
#pragma unroll
      for (int it = 0; it < kV; ++it) vs[tid + it * kThreads] = xv[it];
    }
    __syncthreads();

    // 2. A tile (masked, decayed) and the denominators.
    {
      float acc[4][4] = {};
#pragma unroll 4
      for (int d = 0; d < D; ++d) {
        const float4 a = *reinterpret_cast<const float4 *>(fqT + d * kLd + ty * 4);
        const float4 b = *reinterpret_cast<const float4 *>(fkT + d * kLd + tx * 4);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      float rs[4], qz[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = ty * 4 + i;
        rs[i] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int s = tx * 4 + j;
          float a = 0.f;
          if (s <= t) a = DECAY ? acc[i][j] * G[t - s] : acc[i][j];
          As[t * (kC + 1) + s] = a;
          rs[i] += a;
        }
        float p = 0.f;  // phi(q_t) . z_prev, split over the 16 tx lanes
        for (int d = tx; d < D; d += 16) p = fmaf(fqT[d * kLd + t], zs[d], p);
        qz[i] = p;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {
          rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], off);
          qz[i] += __shfl_xor_sync(0xffffffffu, qz[i], off);
        }
      }
      if (tx == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = ty * 4 + i;
          den[t] = rs[i] + G[t + 1] * qz[i] + eps;
        }
      }
    }
    __syncthreads();

    // 3. o_t = (A_t. V + gamma^(t+1) phi(q_t)^T S_prev) / den_t.
    //    Warp w owns rows 8w..8w+7, lane owns column e0 + lane.
    {
      constexpr int R = kC / 8;
      const int t0 = warp * R;
      float num[R], inter[R];
#pragma unroll
      for (int r = 0; r < R; ++r) num[r] = inter[r] = 0.f;
      for (int s = 0; s < kC; ++s) {
        const float vv = vs[s * kDvs + lane];
#pragma unroll
        for (int r = 0; r < R; ++r) num[r] = fmaf(As[(t0 + r) * (kC + 1) + s], vv, num[r]);
      }
#pragma unroll 4
      for (int d = 0; d < D; ++d) {
        const float sv = Ss[d * kDvs + lane];
        const float4 f0 = *reinterpret_cast<const float4 *>(fqT + d * kLd + t0);
        const float4 f1 = *reinterpret_cast<const float4 *>(fqT + d * kLd + t0 + 4);
        const float fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
        for (int r = 0; r < R; ++r) inter[r] = fmaf(fv[r], sv, inter[r]);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int t = t0 + r;
        if (t < nv)
          io<T>::store(oh + (int64_t)(c0 + t) * DV + e0 + lane,
                       (num[r] + G[t + 1] * inter[r]) / den[t]);
      }
    }
    __syncthreads();

    // 4. State carry: S = gamma^n S + sum_s gamma^(n-1-s) phi(k_s) v_s^T and
    //    z likewise.  Warp w owns rows d = w, w+8, ...
    {
      const float gn = G[nv];
      for (int d = warp; d < D; d += 8) {
        float acc = 0.f, zp = 0.f;
        for (int s = 0; s < nv; ++s) {
          const float f = DECAY ? fkT[d * kLd + s] * G[nv - 1 - s] : fkT[d * kLd + s];
          acc = fmaf(f, vs[s * kDvs + lane], acc);
        }
        for (int s = lane; s < nv; s += 32)
          zp += DECAY ? fkT[d * kLd + s] * G[nv - 1 - s] : fkT[d * kLd + s];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) zp += __shfl_xor_sync(0xffffffffu, zp, off);
        Ss[d * kDvs + lane] = fmaf(gn, Ss[d * kDvs + lane], acc);
        if (lane == 0) zs[d] = fmaf(gn, zs[d], zp);
      }
    }
    __syncthreads();
  }
}

template <int D, int DV, bool DECAY, bool IDENT, typename T>
cudaError_t launch_typed(const Problem &p, const Gammas &g, cudaStream_t s) {
  auto kern = causal_simt_kernel<D, DV, DECAY, IDENT, T>;
  const size_t smem = SimtLayout<D>::bytes;
  cudaError_t err = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)(p.B * p.H), DV / kDvs);
  kern<<<grid, kThreads, smem, s>>>(
      static_cast<const T *>(p.q), static_cast<const T *>(p.k),
      static_cast<const T *>(p.v), static_cast<T *>(p.o), p.H, p.N, p.eps, g);
  return cudaGetLastError();
}

template <int D, int DV, typename T>
cudaError_t launch_decay(const Problem &p, const Gammas &g, cudaStream_t s) {
  if (p.ident)
    return p.decay ? launch_typed<D, DV, true, true, T>(p, g, s)
                   : launch_typed<D, DV, false, true, T>(p, g, s);
  return p.decay ? launch_typed<D, DV, true, false, T>(p, g, s)
                 : launch_typed<D, DV, false, false, T>(p, g, s);
}

template <typename T>
cudaError_t launch_shape(const Problem &p, const Gammas &g, cudaStream_t s) {
  if (p.D == 64 && p.Dv == 64) return launch_decay<64, 64, T>(p, g, s);
  if (p.D == 64 && p.Dv == 128) return launch_decay<64, 128, T>(p, g, s);
  if (p.D == 128 && p.Dv == 64) return launch_decay<128, 64, T>(p, g, s);
  if (p.D == 128 && p.Dv == 128) return launch_decay<128, 128, T>(p, g, s);
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_causal_simt(const Problem &p, const Gammas &g,
                               cudaStream_t s) {
  return p.dtype == kF32 ? launch_shape<float>(p, g, s)
                         : launch_shape<__nv_bfloat16>(p, g, s);
}

}  // namespace linattn
