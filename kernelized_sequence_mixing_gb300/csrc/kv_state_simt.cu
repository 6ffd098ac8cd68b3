// Key/value state reduction and the non-causal read-out on CUDA cores.
//
//   S = sum_j w_j phi(k_j) v_j^T,  z = sum_j w_j phi(k_j)
// with w_j = 1 for the non-causal form ("Linear Attention Mechanisms"
// (dileepadev.github.io), "The Kernel Trick for Attention": S and z are
// computed once over every key) and w_j = gamma^(N-1-j) for the state a
// causal pass leaves behind (the prefill of the decode loop; decay as in
// "Gating and Selective State Updates").  The sequence is split into
// segments reduced in parallel; partial states are summed in a fixed order
// so repeated runs give identical bits.
//
//   o_i = phi(q_i)^T S / (phi(q_i) . z + eps)
// is the non-causal read-out, the same S and z for every query.
#include "common.cuh"
#include "kernels.h"

namespace linattn {
namespace {

constexpr int kThreads = 256;
constexpr int kTok = 32;            // tokens staged per tile
constexpr int kSplitTokens = 4096;  // tokens per split of the reduction

// The y extent of a grid is at most 65535; larger counts are strided.
inline int grid_y(int64_t n) { return (int)(n < 1 ? 1 : (n > 65535 ? 65535 : n)); }

// grid (BH, min(nsplit, 65535)); S_out/z_out indexed by (split * BH + bh).
template <int D, int DV, bool DECAY, bool IDENT, typename T>
__global__ void __launch_bounds__(kThreads)
    kv_partial_kernel(const T *__restrict__ k, const T *__restrict__ v,
                      float *__restrict__ S_out, float *__restrict__ z_out,
                      int H, int N, int split_len, int nsplit,
                      const __grid_constant__ Gammas gam) {
  constexpr int RD = D / 16, RE = DV / 16;
  __shared__ __align__(16) float fk[kTok][D];
  __shared__ __align__(16) float vs[kTok][DV];
  __shared__ float wt[kTok];

  const int tid = threadIdx.x;
  const int td = tid >> 4, te = tid & 15;
  const int64_t bh = blockIdx.x;
  const int64_t BH = gridDim.x;
  const int h = (int)(bh % H);
  const T *kh = k + bh * (int64_t)N * D;
  const T *vh = v + bh * (int64_t)N * DV;
  const double gamma = DECAY ? (double)gam.g[h] : 1.0;
  // splits beyond the grid's y extent (at most 65535) are taken in strides
  for (int sp = blockIdx.y; sp < nsplit; sp += gridDim.y) {
    const int64_t j0 = (int64_t)sp * split_len;
    const int j1 = (int)min((int64_t)N, j0 + split_len);

    float acc[RD][RE] = {};
    float zacc[RD] = {};
    for (int t0 = (int)j0; t0 < j1; t0 += kTok) {
      const int nv = min(kTok, j1 - t0);
      if (DECAY && tid < kTok) {
        // gamma^(N-1-j), in fp64 then rounded once
        wt[tid] = tid < nv ? (float)pow(gamma, (double)(N - 1 - (t0 + tid))) : 0.f;
      }
      if (DECAY) __syncthreads();
      for (int i = tid; i < kTok * D; i += kThreads) {
        const int t = i / D, d = i % D;
        float x = 0.f;
        if (t < nv) {
          x = feat_f32<IDENT>(io<T>::load(kh + (int64_t)(t0 + t) * D + d));
          if (DECAY) x *= wt[t];
        }
        fk[t][d] = x;
      }
      for (int i = tid; i < kTok * DV; i += kThreads) {
        const int t = i / DV, e = i % DV;
        vs[t][e] = t < nv ? io<T>::load(vh + (int64_t)(t0 + t) * DV + e) : 0.f;
      }
      __syncthreads();
      for (int s = 0; s < nv; ++s) {
        float a[RD], b[RE];
#pragma unroll
        for (int i = 0; i < RD; ++i) a[i] = fk[s][td * RD + i];
#pragma unroll
        for (int j = 0; j < RE; ++j) b[j] = vs[s][te * RE + j];
#pragma unroll
        for (int i = 0; i < RD; ++i) {
#pragma unroll
          for (int j = 0; j < RE; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          zacc[i] += a[i];
        }
      }
      __syncthreads();
    }
    const int64_t u = (int64_t)sp * BH + bh;
    float *So = S_out + u * (int64_t)D * DV;
#pragma unroll
    for (int i = 0; i < RD; ++i)
#pragma unroll
      for (int j = 0; j < RE; ++j) So[(td * RD + i) * DV + te * RE + j] = acc[i][j];
    if (te == 0) {
#pragma unroll
      for (int i = 0; i < RD; ++i) z_out[u * D + td * RD + i] = zacc[i];
    }
  }
}

// out[i] = sum over splits of part[sp][i], in split order.
__global__ void __launch_bounds__(kThreads)
    kv_reduce_kernel(const float *__restrict__ part, float *__restrict__ out,
                     int64_t n, int nsplit) {
  const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (i >= n) return;
  float s = 0.f;
  for (int sp = 0; sp < nsplit; ++sp) s += part[(int64_t)sp * n + i];
  out[i] = s;
}

// grid (BH, min(ceil(N / kRowsPerCta), 65535)).
constexpr int kRowTile = 64;
constexpr int kRowsPerCta = 256;

template <int D, int DV, bool IDENT, typename T>
__global__ void __launch_bounds__(kThreads)
    nc_apply_kernel(const T *__restrict__ q, const float *__restrict__ S,
                    const float *__restrict__ z, T *__restrict__ o, int N,
                    float eps) {
  constexpr int RT = kRowTile / 16, RE = DV / 16;
  extern __shared__ float4 smem4[];
  float *Ss = reinterpret_cast<float *>(smem4);  // [D][DV]
  float *zs = Ss + D * DV;                       // [D]
  float *fq = zs + D;                            // [kRowTile][D + 1]

  const int tid = threadIdx.x, tt = tid >> 4, te = tid & 15;
  const int64_t bh = blockIdx.x;
  const T *qh = q + bh * (int64_t)N * D;
  T *oh = o + bh * (int64_t)N * DV;
  for (int i = tid; i < D * DV; i += kThreads) Ss[i] = S[bh * D * DV + i];
  for (int i = tid; i < D; i += kThreads) zs[i] = z[bh * D + i];

  // row blocks beyond the grid's y extent (at most 65535) are taken in strides
  const int nblk = (N + kRowsPerCta - 1) / kRowsPerCta;
  for (int blk = blockIdx.y; blk < nblk; blk += gridDim.y) {
    const int r_begin = blk * kRowsPerCta;
    const int r_end = min(N, r_begin + kRowsPerCta);
    for (int r0 = r_begin; r0 < r_end; r0 += kRowTile) {
      const int nv = min(kRowTile, r_end - r0);
      __syncthreads();
      for (int i = tid; i < kRowTile * D; i += kThreads) {
        const int t = i / D, d = i % D;
        fq[t * (D + 1) + d] = t < nv ? feat_f32<IDENT>(io<T>::load(qh + (int64_t)(r0 + t) * D + d)) : 0.f;
      }
      __syncthreads();
      float acc[RT][RE] = {};
      float dn[RT] = {};
      for (int d = 0; d < D; ++d) {
        float b[RE];
#pragma unroll
        for (int j = 0; j < RE; ++j) b[j] = Ss[d * DV + te * RE + j];
        const float zd = zs[d];
#pragma unroll
        for (int i = 0; i < RT; ++i) {
          const float a = fq[(tt * RT + i) * (D + 1) + d];
          dn[i] = fmaf(a, zd, dn[i]);
#pragma unroll
          for (int j = 0; j < RE; ++j) acc[i][j] = fmaf(a, b[j], acc[i][j]);
        }
      }
#pragma unroll
      for (int i = 0; i < RT; ++i) {
        const int t = tt * RT + i;
        if (t < nv) {
          const float dd = dn[i] + eps;
#pragma unroll
          for (int j = 0; j < RE; ++j)
            io<T>::store(oh + (int64_t)(r0 + t) * DV + te * RE + j, acc[i][j] / dd);
        }
      }
    }
  }
}

template <int D, int DV, bool DECAY, bool IDENT, typename T>
cudaError_t kv_typed(const void *k, const void *v, float *S, float *z,
                     float *part, int BH, int H, int N, const Gammas &g,
                     cudaStream_t s) {
  const int nsplit = kv_state_num_splits(BH, N);
  const int64_t nS = (int64_t)BH * D * DV, nz = (int64_t)BH * D;
  float *So = nsplit == 1 ? S : part;
  float *zo = nsplit == 1 ? z : part + (int64_t)nsplit * nS;
  dim3 grid((unsigned)BH, (unsigned)grid_y(nsplit));
  kv_partial_kernel<D, DV, DECAY, IDENT, T><<<grid, kThreads, 0, s>>>(
      static_cast<const T *>(k), static_cast<const T *>(v), So, zo, H, N,
      kSplitTokens, nsplit, g);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || nsplit == 1) return err;
  kv_reduce_kernel<<<(unsigned)((nS + kThreads - 1) / kThreads), kThreads, 0, s>>>(
      part, S, nS, nsplit);
  kv_reduce_kernel<<<(unsigned)((nz + kThreads - 1) / kThreads), kThreads, 0, s>>>(
      part + (int64_t)nsplit * nS, z, nz, nsplit);
  return cudaGetLastError();
}

template <int D, int DV, typename T>
cudaError_t kv_decay(const void *k, const void *v, float *S, float *z,
                     float *part, int BH, int H, int N, bool decay, bool ident,
                     const Gammas &g, cudaStream_t s) {
  if (ident)
    return decay ? kv_typed<D, DV, true, true, T>(k, v, S, z, part, BH, H, N, g, s)
                 : kv_typed<D, DV, false, true, T>(k, v, S, z, part, BH, H, N, g, s);
  return decay ? kv_typed<D, DV, true, false, T>(k, v, S, z, part, BH, H, N, g, s)
               : kv_typed<D, DV, false, false, T>(k, v, S, z, part, BH, H, N, g, s);
}

template <typename T>
cudaError_t kv_shape(const void *k, const void *v, float *S, float *z,
                     float *part, int BH, int H, int N, int D, int Dv,
                     bool decay, bool ident, const Gammas &g, cudaStream_t s) {
  if (D == 64 && Dv == 64) return kv_decay<64, 64, T>(k, v, S, z, part, BH, H, N, decay, ident, g, s);
  if (D == 64 && Dv == 128) return kv_decay<64, 128, T>(k, v, S, z, part, BH, H, N, decay, ident, g, s);
  if (D == 128 && Dv == 64) return kv_decay<128, 64, T>(k, v, S, z, part, BH, H, N, decay, ident, g, s);
  if (D == 128 && Dv == 128) return kv_decay<128, 128, T>(k, v, S, z, part, BH, H, N, decay, ident, g, s);
  return cudaErrorNotSupported;
}

template <int D, int DV, bool IDENT, typename T>
cudaError_t apply_typed(const void *q, const float *S, const float *z, void *o,
                        int BH, int N, float eps, cudaStream_t s) {
  auto kern = nc_apply_kernel<D, DV, IDENT, T>;
  const size_t smem = sizeof(float) * ((size_t)D * DV + D + kRowTile * (D + 1));
  cudaError_t err = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)BH, (unsigned)grid_y((N + kRowsPerCta - 1) / kRowsPerCta));
  kern<<<grid, kThreads, smem, s>>>(static_cast<const T *>(q), S, z,
                                    static_cast<T *>(o), N, eps);
  return cudaGetLastError();
}

template <bool IDENT, typename T>
cudaError_t apply_shape(const void *q, const float *S, const float *z, void *o,
                        int BH, int N, int D, int Dv, float eps,
                        cudaStream_t s) {
  if (D == 64 && Dv == 64) return apply_typed<64, 64, IDENT, T>(q, S, z, o, BH, N, eps, s);
  if (D == 64 && Dv == 128) return apply_typed<64, 128, IDENT, T>(q, S, z, o, BH, N, eps, s);
  if (D == 128 && Dv == 64) return apply_typed<128, 64, IDENT, T>(q, S, z, o, BH, N, eps, s);
  if (D == 128 && Dv == 128) return apply_typed<128, 128, IDENT, T>(q, S, z, o, BH, N, eps, s);
  return cudaErrorNotSupported;
}

template <int D, int DV, bool DECAY, typename T>
cudaError_t kv_typed_n(const void *k, const void *v, float *S, float *z, float *part,
                       int BH, int H, int N, int nsplit, int split_len, const Gammas &g,
                       cudaStream_t s) {
  const int64_t nS = (int64_t)BH * D * DV, nz = (int64_t)BH * D;
  float *So = nsplit == 1 ? S : part;
  float *zo = nsplit == 1 ? z : part + (int64_t)nsplit * nS;
  dim3 grid((unsigned)BH, (unsigned)grid_y(nsplit));
  kv_partial_kernel<D, DV, DECAY, false, T><<<grid, kThreads, 0, s>>>(
      static_cast<const T *>(k), static_cast<const T *>(v), So, zo, H, N, split_len, nsplit, g);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || nsplit == 1) return err;
  kv_reduce_kernel<<<(unsigned)((nS + kThreads - 1) / kThreads), kThreads, 0, s>>>(
      part, S, nS, nsplit);
  kv_reduce_kernel<<<(unsigned)((nz + kThreads - 1) / kThreads), kThreads, 0, s>>>(
      part + (int64_t)nsplit * nS, z, nz, nsplit);
  return cudaGetLastError();
}

template <typename T>
cudaError_t kv_shape_n(const void *k, const void *v, float *S, float *z, float *part,
                       int BH, int H, int N, int D, int Dv, int nsplit, int split_len,
                       const Gammas &g, cudaStream_t s) {
  if (D == 64 && Dv == 64) return kv_typed_n<64, 64, false, T>(k, v, S, z, part, BH, H, N, nsplit, split_len, g, s);
  if (D == 64 && Dv == 128) return kv_typed_n<64, 128, false, T>(k, v, S, z, part, BH, H, N, nsplit, split_len, g, s);
  if (D == 128 && Dv == 64) return kv_typed_n<128, 64, false, T>(k, v, S, z, part, BH, H, N, nsplit, split_len, g, s);
  if (D == 128 && Dv == 128) return kv_typed_n<128, 128, false, T>(k, v, S, z, part, BH, H, N, nsplit, split_len, g, s);
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_kv_state_splits(const void *k, const void *v, float *S, float *z,
                                   float *partials, int B, int H, int N, int D, int Dv,
                                   int nsplit, const Gammas &g, Dtype dt, cudaStream_t s) {
  const int BH = B * H;
  if (nsplit < 1) return cudaErrorInvalidValue;
  const int split_len = N > 0 ? (N + nsplit - 1) / nsplit : 1;
  return dt == kF32
             ? kv_shape_n<float>(k, v, S, z, partials, BH, H, N, D, Dv, nsplit, split_len, g, s)
             : kv_shape_n<__nv_bfloat16>(k, v, S, z, partials, BH, H, N, D, Dv, nsplit, split_len, g, s);
}

int kv_state_num_splits(int BH, int N) {
  (void)BH;
  return N <= kSplitTokens ? 1 : (N + kSplitTokens - 1) / kSplitTokens;
}

size_t kv_state_workspace_bytes(int BH, int N, int D, int Dv) {
  const int nsplit = kv_state_num_splits(BH, N);
  return nsplit == 1 ? 0
                     : sizeof(float) * (size_t)nsplit * BH * ((size_t)D * Dv + D);
}

cudaError_t launch_kv_state(const void *k, const void *v, float *S, float *z,
                            float *partials, int B, int H, int N, int D,
                            int Dv, bool decay, const Gammas &g, Dtype dt,
                            cudaStream_t s, bool ident) {
  const int BH = B * H;
  return dt == kF32
             ? kv_shape<float>(k, v, S, z, partials, BH, H, N, D, Dv, decay, ident, g, s)
             : kv_shape<__nv_bfloat16>(k, v, S, z, partials, BH, H, N, D, Dv, decay, ident, g, s);
}

cudaError_t launch_noncausal_apply(const void *q, const float *S,
                                   const float *z, void *o, int BH, int N,
                                   int D, int Dv, float eps, Dtype dt,
                                   cudaStream_t s, bool ident) {
  if (ident)
    return dt == kF32 ? apply_shape<true, float>(q, S, z, o, BH, N, D, Dv, eps, s)
                      : apply_shape<true, __nv_bfloat16>(q, S, z, o, BH, N, D, Dv, eps, s);
  return dt == kF32
             ? apply_shape<false, float>(q, S, z, o, BH, N, D, Dv, eps, s)
             : apply_shape<false, __nv_bfloat16>(q, S, z, o, BH, N, D, Dv, eps, s);
}

}  // namespace linattn
