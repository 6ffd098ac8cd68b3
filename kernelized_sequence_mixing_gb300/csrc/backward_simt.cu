// Backward pass of causal linear attention (with the per-head decay), fp32 on
// CUDA cores.
//
// The forward is the causal form of "Linear Attention Mechanisms"
// (dileepadev.github.io), "Recurrent Reformulation", with the decay of
// "Gating and Selective State Updates": with w_ij = gamma^(i-j) phi(q_i).phi(k_j)
// (j <= i), n_i = sum_j w_ij v_j, d_i = sum_j w_ij + eps, o_i = n_i / d_i.  For
// an upstream gradient g_i, with gt_i = g_i / d_i and c_i = gt_i . o_i, the
// chain rule through the quotient gives dL/dw_ij = gt_i . v_j - c_i, and
//   dphi(q)_i = sum_(j<=i) gamma^(i-j) (gt_i . v_j - c_i) phi(k_j)
//   dv_j      = sum_(i>=j) gamma^(i-j) (phi(k_j) . phi(q_i)) gt_i
//   dphi(k)_j = sum_(i>=j) gamma^(i-j) (v_j . gt_i - c_i) phi(q_i)
// then dq = dphi(q) * phi'(q), dk likewise (phi'(x) = 1 for x > 0, exp(x)
// otherwise, i.e. min(phi(x), 1)).
//
// Every one of these, and the forward's n and d, is an instance of one
// unnormalised decayed causal product
//   y_t = sum_(s<=t) gamma^(t-s) (a_t . b_s) c_s      (or s >= t, reversed)
// over per-token vectors a, b (length DA) and c (length DC):
//   n, d - eps : a = phi(q),    b = phi(k),     c = [v | 1]
//   dphi(q)    : a = [gt | c],  b = [v | -1],   c = phi(k)
//   dv         : a = phi(k),    b = phi(q),     c = gt        (reversed)
//   dphi(k)    : a = [v | -1],  b = [gt | c],   c = phi(q)    (reversed)
// (the augmented vectors are padded with zeros to a multiple of 4).  The
// product runs chunked, like the forward: per chunk of 64 tokens the masked,
// decayed A = a b^T, y = A c + gamma^(...) a^T H, and the carried state
// H = sum gamma^(...) b c^T updated; one CTA per (batch, head) and 32-column
// slice of c, the chunks in sequence.  Small elementwise kernels build the
// operands and finish the gradients.  All arithmetic is fp32; the operands
// live in an fp32 workspace.
#include "common.cuh"
#include "kernels.h"

namespace linattn {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr int kLd = kC + 4;
constexpr int kCs = 32;  // columns of c per CTA

template <int DA>
struct ProdLayout {
  static constexpr int aT = DA * kLd, bT = DA * kLd, A = kC * (kC + 1), cs = kC * kCs,
                       H = DA * kCs, G = kC + 4;
  static constexpr size_t bytes = sizeof(float) * (aT + bT + A + cs + H + G);
};

// grid: x = (batch, head), y = ceil(DC / 32).  a, b: [BH][N][DA]; c, y:
// [BH][N][DC], fp32.
template <int DA, int DC, bool REV>
__global__ void __launch_bounds__(kThreads)
    causal_product_kernel(const float *__restrict__ a, const float *__restrict__ b,
                          const float *__restrict__ c, float *__restrict__ y, int H, int N,
                          const __grid_constant__ Gammas gam) {
  extern __shared__ float4 smem4[];
  using L = ProdLayout<DA>;
  float *aT = reinterpret_cast<float *>(smem4);  // [DA][kLd]
  float *bT = aT + L::aT;                        // [DA][kLd]
  float *As = bT + L::bT;                        // [kC][kC+1]
  float *cs = As + L::A;                         // [kC][kCs]
  float *Hs = cs + L::cs;                        // [DA][kCs]
  float *G = Hs + L::H;                          // gamma^k, k = 0..kC

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t bh = blockIdx.x;
  const int e0 = blockIdx.y * kCs;
  const int ncol = min(kCs, DC - e0);
  const float *ah = a + bh * N * DA;
  const float *bh_ = b + bh * N * DA;
  const float *ch = c + bh * N * DC;
  float *yh = y + bh * N * DC;

  for (int i = tid; i < DA * kCs; i += kThreads) Hs[i] = 0.f;
  if (tid == 0) build_pow_table(G, kC, gam.g[bh % H]);
  __syncthreads();

  const int ty = tid >> 4, tx = tid & 15;
  const int nch = (N + kC - 1) / kC;
  for (int ci = 0; ci < nch; ++ci) {
    const int cidx = REV ? nch - 1 - ci : ci;
    const int c0 = cidx * kC, nv = min(kC, N - c0);
    for (int i = tid; i < kC * DA; i += kThreads) {
      const int t = i / DA, d = i % DA;
      float xa = 0.f, xb = 0.f;
      if (t < nv) {
        xa = ah[(int64_t)(c0 + t) * DA + d];
        xb = bh_[(int64_t)(c0 + t) * DA + d];
      }
      aT[d * kLd + t] = xa;
      bT[d * kLd + t] = xb;
    }
    for (int i = tid; i < kC * kCs; i += kThreads) {
      const int t = i / kCs, e = i % kCs;
      cs[i] = (t < nv && e < ncol) ? ch[(int64_t)(c0 + t) * DC + e0 + e] : 0.f;
    }
    __syncthreads();
    // A_ts = gamma^|t-s| a_t . b_s on s <= t (forward) or s >= t (reversed)
    {
      float acc[4][4] = {};
#pragma unroll 4
      for (int d = 0; d < DA; ++d) {
        const float4 x = *reinterpret_cast<const float4 *>(aT + d * kLd + ty * 4);
        const float4 w = *reinterpret_cast<const float4 *>(bT + d * kLd + tx * 4);
        const float xv[4] = {x.x, x.y, x.z, x.w};
        const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = ty * 4 + i, s = tx * 4 + j;
          const bool in = REV ? s >= t : s <= t;
          As[t * (kC + 1) + s] = in ? acc[i][j] * G[REV ? s - t : t - s] : 0.f;
        }
    }
    __syncthreads();
    // y_t = A_t. c + gamma^k a_t^T H, k = t + 1 (forward) or nv - t (reversed);
    // warp w owns rows 8w..8w+7, lane owns column e0 + lane
    {
      constexpr int R = kC / 8;
      const int t0 = warp * R;
      float num[R], inter[R];
#pragma unroll
      for (int r = 0; r < R; ++r) num[r] = inter[r] = 0.f;
      for (int s = 0; s < kC; ++s) {
        const float cv = cs[s * kCs + lane];
#pragma unroll
        for (int r = 0; r < R; ++r) num[r] = fmaf(As[(t0 + r) * (kC + 1) + s], cv, num[r]);
      }
#pragma unroll 4
      for (int d = 0; d < DA; ++d) {
        const float hv = Hs[d * kCs + lane];
        const float4 f0 = *reinterpret_cast<const float4 *>(aT + d * kLd + t0);
        const float4 f1 = *reinterpret_cast<const float4 *>(aT + d * kLd + t0 + 4);
        const float fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
        for (int r = 0; r < R; ++r) inter[r] = fmaf(fv[r], hv, inter[r]);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int t = t0 + r;
        if (t < nv && lane < ncol)
          yh[(int64_t)(c0 + t) * DC + e0 + lane] = fmaf(G[REV ? nv - t : t + 1], inter[r], num[r]);
      }
    }
    __syncthreads();
    // H = gamma^nv H + sum_s gamma^k b_s c_s^T, k = nv - 1 - s (forward) or s
    // (reversed: H relative to the chunk's first token)
    {
      const float gn = G[nv];
      for (int d = warp; d < DA; d += 8) {
        float acc = 0.f;
        for (int s = 0; s < nv; ++s)
          acc = fmaf(bT[d * kLd + s] * G[REV ? s : nv - 1 - s], cs[s * kCs + lane], acc);
        Hs[d * kCs + lane] = fmaf(gn, Hs[d * kCs + lane], acc);
      }
    }
    __syncthreads();
  }
}

template <int DA, int DC, bool REV>
cudaError_t product_launch(const float *a, const float *b, const float *c, float *y, int BH,
                           int H, int N, const Gammas &g, cudaStream_t s) {
  auto kern = causal_product_kernel<DA, DC, REV>;
  const size_t smem = ProdLayout<DA>::bytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3((unsigned)BH, (DC + kCs - 1) / kCs), kThreads, smem, s>>>(a, b, c, y, H, N, g);
  return cudaGetLastError();
}

// Operands: fq = phi(q), fk = phi(k) [.][D]; vp = [v | 1 | 0 0 0],
// vm = [v | -1 | 0 0 0] [.][Dv + 4]; one thread per (row, column).
template <typename T>
__global__ void bwd_prep_kernel(const T *__restrict__ q, const T *__restrict__ k,
                                const T *__restrict__ v, float *__restrict__ fq,
                                float *__restrict__ fk, float *__restrict__ vp,
                                float *__restrict__ vm, int64_t rows, int D, int Dv) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int W = D + Dv + 4;
  if (i >= rows * W) return;
  const int64_t r = i / W;
  const int col = static_cast<int>(i % W);
  if (col < D) {
    fq[r * D + col] = phi_f32(io<T>::load(q + r * D + col));
    fk[r * D + col] = phi_f32(io<T>::load(k + r * D + col));
  } else {
    const int e = col - D;
    const float x = e < Dv ? io<T>::load(v + r * Dv + e) : (e == Dv ? 1.f : 0.f);
    vp[r * (Dv + 4) + e] = x;
    vm[r * (Dv + 4) + e] = e == Dv ? -1.f : x;
  }
}

// From nd = [n | d - eps]: o = n / d, gt = g / d, c = gt . o; writes
// gc = [gt | c | 0 0 0] and gt.  One warp per row.
template <typename T>
__global__ void bwd_mid_kernel(const float *__restrict__ nd, const T *__restrict__ g,
                               float *__restrict__ gc, float *__restrict__ gt, int64_t rows,
                               int Dv, float eps) {
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const float *ndr = nd + r * (Dv + 4);
  const float den = ndr[Dv] + eps;
  float cp = 0.f;
  for (int e = lane; e < Dv; e += 32) {
    const float o = ndr[e] / den;
    const float gv = io<T>::load(g + r * Dv + e) / den;
    gc[r * (Dv + 4) + e] = gv;
    gt[r * Dv + e] = gv;
    cp = fmaf(gv, o, cp);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) cp += __shfl_xor_sync(0xffffffffu, cp, off);
  if (lane < 4) gc[r * (Dv + 4) + Dv + lane] = lane == 0 ? cp : 0.f;
}

// dq = dphi(q) min(phi(q), 1), dk likewise, dv as it is; cast to T.
template <typename T>
__global__ void bwd_final_kernel(const float *__restrict__ dfq, const float *__restrict__ dfk,
                                 const float *__restrict__ dvf, const float *__restrict__ fq,
                                 const float *__restrict__ fk, T *__restrict__ dq,
                                 T *__restrict__ dk, T *__restrict__ dv, int64_t rows, int D,
                                 int Dv) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int W = 2 * D + Dv;
  if (i >= rows * W) return;
  const int64_t r = i / W;
  const int col = static_cast<int>(i % W);
  if (col < D) {
    io<T>::store(dq + r * D + col, dfq[r * D + col] * fminf(fq[r * D + col], 1.f));
  } else if (col < 2 * D) {
    const int d = col - D;
    io<T>::store(dk + r * D + d, dfk[r * D + d] * fminf(fk[r * D + d], 1.f));
  } else {
    const int e = col - 2 * D;
    io<T>::store(dv + r * Dv + e, dvf[r * Dv + e]);
  }
}

template <int D, int DV, typename T>
cudaError_t backward_typed(const Problem &p, const void *dO, void *dq, void *dk, void *dv,
                           const Gammas &g, float *ws, cudaStream_t s) {
  constexpr int DV4 = DV + 4;
  const int BH = p.B * p.H;
  const int64_t rows = static_cast<int64_t>(BH) * p.N;
  float *fq = ws, *fk = fq + rows * D, *vp = fk + rows * D, *vm = vp + rows * DV4,
        *nd = vm + rows * DV4, *gc = nd + rows * DV4, *gt = gc + rows * DV4,
        *dfq = gt + rows * DV, *dfk = dfq + rows * D, *dvf = dfk + rows * D;
  cudaError_t e;
  {
    const int64_t n = rows * (D + DV + 4);
    bwd_prep_kernel<T><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
        static_cast<const T *>(p.q), static_cast<const T *>(p.k), static_cast<const T *>(p.v), fq,
        fk, vp, vm, rows, D, DV);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = product_launch<D, DV4, false>(fq, fk, vp, nd, BH, p.H, p.N, g, s)) != cudaSuccess) return e;
  bwd_mid_kernel<T><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, s>>>(
      nd, static_cast<const T *>(dO), gc, gt, rows, DV, p.eps);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = product_launch<DV4, D, false>(gc, vm, fk, dfq, BH, p.H, p.N, g, s)) != cudaSuccess) return e;
  if ((e = product_launch<D, DV, true>(fk, fq, gt, dvf, BH, p.H, p.N, g, s)) != cudaSuccess) return e;
  if ((e = product_launch<DV4, D, true>(vm, gc, fq, dfk, BH, p.H, p.N, g, s)) != cudaSuccess) return e;
  {
    const int64_t n = rows * (2 * D + DV);
    bwd_final_kernel<T><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
        dfq, dfk, dvf, fq, fk, static_cast<T *>(dq), static_cast<T *>(dk), static_cast<T *>(dv),
        rows, D, DV);
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t backward_shape(const Problem &p, const void *dO, void *dq, void *dk, void *dv,
                           const Gammas &g, float *ws, cudaStream_t s) {
  if (p.D == 64 && p.Dv == 64) return backward_typed<64, 64, T>(p, dO, dq, dk, dv, g, ws, s);
  if (p.D == 64 && p.Dv == 128) return backward_typed<64, 128, T>(p, dO, dq, dk, dv, g, ws, s);
  if (p.D == 128 && p.Dv == 64) return backward_typed<128, 64, T>(p, dO, dq, dk, dv, g, ws, s);
  if (p.D == 128 && p.Dv == 128) return backward_typed<128, 128, T>(p, dO, dq, dk, dv, g, ws, s);
  return cudaErrorNotSupported;
}

}  // namespace

size_t backward_workspace_bytes(int BH, int N, int D, int Dv) {
  const size_t rows = static_cast<size_t>(BH) * N;
  return sizeof(float) * rows * (4 * static_cast<size_t>(D) + 4 * (Dv + 4) + 2 * Dv);
}

cudaError_t launch_backward(const Problem &p, const void *dO, void *dq, void *dk, void *dv,
                            const Gammas &g, void *ws, cudaStream_t s) {
  float *w = static_cast<float *>(ws);
  return p.dtype == kF32 ? backward_shape<float>(p, dO, dq, dk, dv, g, w, s)
                         : backward_shape<__nv_bfloat16>(p, dO, dq, dk, dv, g, w, s);
}

}  // namespace linattn
