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
constexpr int kLdA = kC + 4;  // row stride of the transposed A tile
constexpr int kCs = 32;       // columns of c per CTA

template <int DA>
struct ProdLayout {
  static constexpr int aT = DA * kC, bT = DA * kC, A = kC * kLdA, cs = kC * kCs, H = DA * kCs,
                       G = kC + 4;
  static constexpr size_t bytes = sizeof(float) * (aT + bT + A + cs + H + G);
};

struct ProdArgs {
  const float *a, *b, *c;
  float *y;
  float *rec;  // per-part states [B*H][P][DA][DC] (P > 1)
};

enum { kPassOut = 0, kPassState = 1 };

__host__ __device__ inline int part_chunk(int p, int P, int nch) {
  return static_cast<int>((static_cast<long long>(p) * nch) / P);
}

// One CTA of the product over a (batch, head) and 32-column slice of c:
// a, b [BH][N][DA]; c, y [BH][N][DC], fp32.  Per 64-token chunk:
//   load   item (t = i mod 64, column quad i / 64): 16-byte loads of a row's
//          quad, stored transposed ([column][token]) by consecutive lanes at
//          consecutive tokens;
//   A      16 x 16 threads, 4 x 4 register tiles of a b^T, masked and decayed,
//          stored transposed ([s][t]);
//   y      4 tokens x 2 columns per thread: y = A c + gamma^k a^T H;
//   H      4 rows x 4 columns per item: H = gamma^nv H + sum_s gamma^k b_s c_s^T.
// Sequence parts: part `part` of P covers whole chunks [cb, ce).  The output
// pass starts from the state the scan left for it (forward: the state after
// part - 1; reversed: the state before part + 1) and the state pass only
// carries H from zero over its part and stores it.
template <int DA, int DC, bool REV, int PASS>
__device__ __forceinline__ void product_body(const ProdArgs &pa, int64_t bh, int part, int P,
                                             int slice, int H, int N, const Gammas &gam,
                                             float *smem) {
  using L = ProdLayout<DA>;
  float *aT = smem;          // [DA][kC]
  float *bT = aT + L::aT;    // [DA][kC]
  float *AT = bT + L::bT;    // [kC][kLdA]
  float *cs = AT + L::A;     // [kC][kCs]
  float *Hs = cs + L::cs;    // [DA][kCs]
  float *G = Hs + L::H;      // gamma^k, k = 0..kC
  constexpr int DQ = DA / 4;

  const int tid = threadIdx.x;
  const int e0 = slice * kCs;
  const int ncol = min(kCs, DC - e0);
  const float *ah = pa.a + bh * N * DA;
  const float *bhp = pa.b + bh * N * DA;
  const float *ch = pa.c + bh * N * DC;
  float *yh = pa.y + bh * N * DC;

  const size_t rstride = static_cast<size_t>(DA) * DC;
  const int pin = REV ? part + 1 : part - 1;  // the part whose scanned state starts this one
  if (PASS == kPassOut && pin >= 0 && pin < P) {
    const float *r = pa.rec + (static_cast<size_t>(bh) * P + pin) * rstride;
    for (int i = tid; i < DA * kCs; i += kThreads) {
      const int d = i / kCs, e = i % kCs;
      Hs[i] = e < ncol ? r[d * DC + e0 + e] : 0.f;
    }
  } else {
    for (int i = tid; i < DA * kCs; i += kThreads) Hs[i] = 0.f;
  }
  if (tid == 0) build_pow_table(G, kC, gam.g[bh % H]);
  __syncthreads();

  const int nch_all = (N + kC - 1) / kC;
  const int cb = part_chunk(part, P, nch_all), ce = part_chunk(part + 1, P, nch_all);
  for (int ci = 0; ci < ce - cb; ++ci) {
    const int cidx = REV ? ce - 1 - ci : cb + ci;
    const int c0 = cidx * kC, nv = min(kC, N - c0);
    for (int i = tid; i < kC * DQ; i += kThreads) {
      const int t = i & (kC - 1), q4 = i >> 6;
      float4 xa = make_float4(0.f, 0.f, 0.f, 0.f), xb = xa;
      if (t < nv) {
        if (PASS == kPassOut)
          xa = *reinterpret_cast<const float4 *>(ah + (int64_t)(c0 + t) * DA + 4 * q4);
        xb = *reinterpret_cast<const float4 *>(bhp + (int64_t)(c0 + t) * DA + 4 * q4);
      }
      if (PASS == kPassOut) {
        aT[(4 * q4 + 0) * kC + t] = xa.x;
        aT[(4 * q4 + 1) * kC + t] = xa.y;
        aT[(4 * q4 + 2) * kC + t] = xa.z;
        aT[(4 * q4 + 3) * kC + t] = xa.w;
      }
      bT[(4 * q4 + 0) * kC + t] = xb.x;
      bT[(4 * q4 + 1) * kC + t] = xb.y;
      bT[(4 * q4 + 2) * kC + t] = xb.z;
      bT[(4 * q4 + 3) * kC + t] = xb.w;
    }
    for (int i = tid; i < kC * (kCs / 4); i += kThreads) {
      const int t = i >> 3, q4 = i & 7;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < nv && 4 * q4 < ncol) {
        const float *src = ch + (int64_t)(c0 + t) * DC + e0 + 4 * q4;
        if (DC % 4 == 0) {
          x = *reinterpret_cast<const float4 *>(src);
        } else {
          x.x = src[0];
          if (4 * q4 + 1 < ncol) x.y = src[1];
          if (4 * q4 + 2 < ncol) x.z = src[2];
          if (4 * q4 + 3 < ncol) x.w = src[3];
        }
      }
      *reinterpret_cast<float4 *>(cs + t * kCs + 4 * q4) = x;
    }
    __syncthreads();
    // A_ts = gamma^|t-s| a_t . b_s on s <= t (forward) or s >= t (reversed)
    if (PASS == kPassOut) {
      const int ty = tid >> 4, tx = tid & 15;
      float acc[4][4] = {};
      if (REV ? tx >= ty : tx <= ty) {
#pragma unroll 4
        for (int d = 0; d < DA; ++d) {
          const float4 x = *reinterpret_cast<const float4 *>(aT + d * kC + 4 * ty);
          const float4 w = *reinterpret_cast<const float4 *>(bT + d * kC + 4 * tx);
          const float xv[4] = {x.x, x.y, x.z, x.w};
          const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float col[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = 4 * ty + i, sidx = 4 * tx + j;
          const bool in = REV ? sidx >= t : sidx <= t;
          col[i] = in ? acc[i][j] * G[REV ? sidx - t : t - sidx] : 0.f;
        }
        *reinterpret_cast<float4 *>(AT + (4 * tx + j) * kLdA + 4 * ty) =
            make_float4(col[0], col[1], col[2], col[3]);
      }
    }
    if (PASS == kPassOut) __syncthreads();
    // y_t = A_t. c + gamma^k a_t^T H, k = t + 1 (forward) or nv - t (reversed)
    if (PASS == kPassOut) {
      const int ep = tid & 15, tg = tid >> 4;
      float acc[4][2] = {};
      const int s0 = REV ? 4 * tg : 0, s1 = REV ? kC : 4 * tg + 4;
      for (int sidx = s0; sidx < s1; ++sidx) {
        const float4 w = *reinterpret_cast<const float4 *>(AT + sidx * kLdA + 4 * tg);
        const float2 x = *reinterpret_cast<const float2 *>(cs + sidx * kCs + 2 * ep);
        const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i][0] = fmaf(wv[i], x.x, acc[i][0]);
          acc[i][1] = fmaf(wv[i], x.y, acc[i][1]);
        }
      }
      float inter[4][2] = {};
#pragma unroll 4
      for (int d = 0; d < DA; ++d) {
        const float4 f = *reinterpret_cast<const float4 *>(aT + d * kC + 4 * tg);
        const float2 hv = *reinterpret_cast<const float2 *>(Hs + d * kCs + 2 * ep);
        const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          inter[i][0] = fmaf(fv[i], hv.x, inter[i][0]);
          inter[i][1] = fmaf(fv[i], hv.y, inter[i][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 4 * tg + i;
        if (t >= nv) continue;
        const float gk = G[REV ? nv - t : t + 1];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
          if (2 * ep + jj < ncol)
            yh[(int64_t)(c0 + t) * DC + e0 + 2 * ep + jj] = fmaf(gk, inter[i][jj], acc[i][jj]);
      }
    }
    if (PASS == kPassOut) __syncthreads();
    // H = gamma^nv H + sum_s w_s b_s c_s^T, w_s = gamma^(nv-1-s) (forward) or
    // gamma^s (reversed: H relative to the chunk's first token)
    {
      const float gn = G[nv];
      for (int it = tid; it < DQ * (kCs / 4); it += kThreads) {
        const int dq = it >> 3, eq = it & 7;
        float acc[4][4] = {};
        for (int sidx = 0; sidx < kC; sidx += 4) {
          float4 kb[4], vv[4];
#pragma unroll
          for (int r = 0; r < 4; ++r)
            kb[r] = *reinterpret_cast<const float4 *>(bT + (4 * dq + r) * kC + sidx);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            vv[j] = *reinterpret_cast<const float4 *>(cs + (sidx + j) * kCs + 4 * eq);
          float wgt[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int sj = sidx + j;
            wgt[j] = sj < nv ? G[REV ? sj : nv - 1 - sj] : 0.f;
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float kr[4] = {kb[r].x * wgt[0], kb[r].y * wgt[1], kb[r].z * wgt[2],
                                 kb[r].w * wgt[3]};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              acc[r][0] = fmaf(kr[j], vv[j].x, acc[r][0]);
              acc[r][1] = fmaf(kr[j], vv[j].y, acc[r][1]);
              acc[r][2] = fmaf(kr[j], vv[j].z, acc[r][2]);
              acc[r][3] = fmaf(kr[j], vv[j].w, acc[r][3]);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float4 *hp = reinterpret_cast<float4 *>(Hs + (4 * dq + r) * kCs + 4 * eq);
          float4 h = *hp;
          h.x = fmaf(gn, h.x, acc[r][0]);
          h.y = fmaf(gn, h.y, acc[r][1]);
          h.z = fmaf(gn, h.z, acc[r][2]);
          h.w = fmaf(gn, h.w, acc[r][3]);
          *hp = h;
        }
      }
    }
    __syncthreads();
  }
  if (PASS == kPassState) {
    float *r = pa.rec + (static_cast<size_t>(bh) * P + part) * rstride;
    for (int i = tid; i < DA * kCs; i += kThreads) {
      const int d = i / kCs, e = i % kCs;
      if (e < ncol) r[d * DC + e0 + e] = Hs[i];
    }
  }
}

// The scan over parts of one product, in place over the records of one
// (batch, head): forward, record p (the state of part p from zero, relative
// to its last token) becomes the state after parts 0..p, S(p) =
// gamma^len(p) S(p-1) + rec(p), for p < P - 1; reversed, record p (relative
// to its first token) becomes the state of parts p..P-1, for p > 0.
constexpr int kMaxParts = 64;

// gamma^len(p) for every part, once per CTA (one fp64 power per part, from
// threads 0..P-1).
__device__ __forceinline__ void part_weights(float *w, int P, int N, float gamma) {
  const int nch_all = (N + kC - 1) / kC;
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int t0 = part_chunk(p, P, nch_all) * kC;
    const int t1 = min(N, part_chunk(p + 1, P, nch_all) * kC);
    w[p] = static_cast<float>(pow(static_cast<double>(gamma), static_cast<double>(t1 - t0)));
  }
  __syncthreads();
}

template <int DA, int DC, bool REV>
__device__ __forceinline__ void scan_body(float *rec, int64_t bh, int P, const float *w) {
  const int i = blockIdx.y * blockDim.x + threadIdx.x;
  if (i >= DA * DC) return;
  const size_t rstride = static_cast<size_t>(DA) * DC;
  float *r = rec + static_cast<size_t>(bh) * P * rstride + i;
  float carry = 0.f;
  for (int j = 0; j < P - 1; ++j) {
    const int p = REV ? P - 1 - j : j;
    carry = fmaf(w[p], carry, r[p * rstride]);
    r[p * rstride] = carry;
  }
}

// grid x = (batch, head) * parts of this pass + part: the output pass has P
// parts; the state pass P - 1 (every part but the last one in scan order).
__device__ __forceinline__ void pass_part(int PASS_, bool rev, int P, int64_t *bh, int *part) {
  const int pg = PASS_ == kPassOut ? P : P - 1;
  *bh = blockIdx.x / pg;
  *part = blockIdx.x % pg + (PASS_ == kPassState && rev ? 1 : 0);
}

// One product: grid y = ceil(DC / 32) column slices.
template <int DA, int DC, bool REV, int PASS>
__global__ void __launch_bounds__(kThreads, 2)
    causal_product_kernel(ProdArgs pa, int P, int H, int N, const __grid_constant__ Gammas gam) {
  extern __shared__ float4 smem4[];
  int64_t bh;
  int part;
  pass_part(PASS, REV, P, &bh, &part);
  product_body<DA, DC, REV, PASS>(pa, bh, part, P, blockIdx.y, H, N, gam,
                                  reinterpret_cast<float *>(smem4));
}

// The three gradient products in one launch (grid z = 0, 1, 2):
//   dphi(q) <DV4, D, forward>, dv <D, DV, reversed>, dphi(k) <DV4, D, reversed>.
template <int D, int DV, int PASS>
__global__ void __launch_bounds__(kThreads, 2)
    gradient_products_kernel(ProdArgs p0, ProdArgs p1, ProdArgs p2, int P, int H, int N,
                             const __grid_constant__ Gammas gam) {
  extern __shared__ float4 smem4[];
  float *sm = reinterpret_cast<float *>(smem4);
  constexpr int DV4 = DV + 4;
  int64_t bh;
  int part;
  if (blockIdx.z == 0) {
    pass_part(PASS, false, P, &bh, &part);
    if (blockIdx.y < (D + kCs - 1) / kCs)
      product_body<DV4, D, false, PASS>(p0, bh, part, P, blockIdx.y, H, N, gam, sm);
  } else if (blockIdx.z == 1) {
    pass_part(PASS, true, P, &bh, &part);
    if (blockIdx.y < (DV + kCs - 1) / kCs)
      product_body<D, DV, true, PASS>(p1, bh, part, P, blockIdx.y, H, N, gam, sm);
  } else {
    pass_part(PASS, true, P, &bh, &part);
    if (blockIdx.y < (D + kCs - 1) / kCs)
      product_body<DV4, D, true, PASS>(p2, bh, part, P, blockIdx.y, H, N, gam, sm);
  }
}

// Scans: grid x = (batch, head), y = blocks of 256 state entries.
template <int DA, int DC, bool REV>
__global__ void __launch_bounds__(256)
    product_scan_kernel(float *rec, int P, int H, int N, const __grid_constant__ Gammas gam) {
  __shared__ float w[kMaxParts];
  part_weights(w, P, N, gam.g[blockIdx.x % H]);
  scan_body<DA, DC, REV>(rec, blockIdx.x, P, w);
}
template <int D, int DV>
__global__ void __launch_bounds__(256)
    gradient_scan_kernel(float *r0, float *r1, float *r2, int P, int H, int N,
                         const __grid_constant__ Gammas gam) {
  constexpr int DV4 = DV + 4;
  __shared__ float w[kMaxParts];
  part_weights(w, P, N, gam.g[blockIdx.x % H]);
  if (blockIdx.z == 0) scan_body<DV4, D, false>(r0, blockIdx.x, P, w);
  else if (blockIdx.z == 1) scan_body<D, DV, true>(r1, blockIdx.x, P, w);
  else scan_body<DV4, D, true>(r2, blockIdx.x, P, w);
}

int num_sms_bwd() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// Parts per (batch, head): the count minimising a wave model of the output
// pass plus the state pass (measured at about 0.3 of it), with
// waves(n) = ceil(ctas_per_part * n / (2 CTAs per SM x SMs)), plus a fixed
// cost per part (its records, its start-up) of 0.01 of a full-sequence pass;
// at most one part per 2 chunks and kMaxParts.
int product_parts(long long ctas_per_part, int N) {
  const long long nch = (N + kC - 1) / kC;
  const long long slots = 2LL * num_sms_bwd();
  auto waves = [&](long long n) { return (ctas_per_part * n + slots - 1) / slots; };
  const long long pmax = nch / 2 < kMaxParts ? nch / 2 : kMaxParts;
  long long best = 1;
  double best_t = static_cast<double>(waves(1));
  for (long long P = 2; P <= pmax; ++P) {
    const double t =
        (static_cast<double>(waves(P)) + 0.3 * static_cast<double>(waves(P - 1))) / P + 0.01 * P;
    if (t < best_t * 0.97) {
      best_t = t;
      best = P;
    }
  }
  return static_cast<int>(best);
}

template <int DA, int DC, bool REV>
cudaError_t product_launch(const float *a, const float *b, const float *c, float *y, float *rec,
                           int P, int BH, int H, int N, const Gammas &g, cudaStream_t s) {
  const size_t smem = ProdLayout<DA>::bytes;
  const unsigned ny = (DC + kCs - 1) / kCs;
  const ProdArgs pa{a, b, c, y, rec};
  cudaError_t e;
  if (P > 1) {
    auto ks = causal_product_kernel<DA, DC, REV, kPassState>;
    if ((e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return e;
    ks<<<dim3((unsigned)(BH * (P - 1)), ny), kThreads, smem, s>>>(pa, P, H, N, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    product_scan_kernel<DA, DC, REV><<<dim3((unsigned)BH, (DA * DC + 255) / 256), 256, 0, s>>>(
        rec, P, H, N, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  auto ko = causal_product_kernel<DA, DC, REV, kPassOut>;
  if ((e = cudaFuncSetAttribute(ko, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return e;
  ko<<<dim3((unsigned)(BH * P), ny), kThreads, smem, s>>>(pa, P, H, N, g);
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

// Parts of the forward-recompute product and of the gradient products, and
// the floats of their per-part records.
struct BwdPlan {
  int P_nd, P_g;
  size_t rec_nd, rec_g0, rec_g1, rec_g2;
};

BwdPlan bwd_plan(int BH, int N, int D, int Dv) {
  BwdPlan pl;
  const int Dv4 = Dv + 4;
  const int ny = ((D > Dv ? D : Dv) + kCs - 1) / kCs;
  pl.P_nd = product_parts(static_cast<long long>(BH) * ((Dv4 + kCs - 1) / kCs), N);
  pl.P_g = product_parts(static_cast<long long>(BH) * ny * 3, N);
  const size_t bn = static_cast<size_t>(BH) * pl.P_nd, bg = static_cast<size_t>(BH) * pl.P_g;
  pl.rec_nd = pl.P_nd > 1 ? bn * D * Dv4 : 0;
  pl.rec_g0 = pl.P_g > 1 ? bg * Dv4 * D : 0;
  pl.rec_g1 = pl.P_g > 1 ? bg * D * Dv : 0;
  pl.rec_g2 = pl.rec_g0;
  return pl;
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
  const BwdPlan pl = bwd_plan(BH, p.N, D, DV);
  float *rec_nd = dvf + rows * DV, *rec_g0 = rec_nd + pl.rec_nd, *rec_g1 = rec_g0 + pl.rec_g0,
        *rec_g2 = rec_g1 + pl.rec_g1;
  cudaError_t e;
  {
    const int64_t n = rows * (D + DV + 4);
    bwd_prep_kernel<T><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
        static_cast<const T *>(p.q), static_cast<const T *>(p.k), static_cast<const T *>(p.v), fq,
        fk, vp, vm, rows, D, DV);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = product_launch<D, DV4, false>(fq, fk, vp, nd, rec_nd, pl.P_nd, BH, p.H, p.N, g, s)) !=
      cudaSuccess)
    return e;
  bwd_mid_kernel<T><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, s>>>(
      nd, static_cast<const T *>(dO), gc, gt, rows, DV, p.eps);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    // dphi(q), dv and dphi(k) are independent: one launch per pass, grid z
    // selects the product
    const size_t smem = ProdLayout<(DV4 > D ? DV4 : D)>::bytes;
    const unsigned ny = ((D > DV ? D : DV) + kCs - 1) / kCs;
    const ProdArgs a0{gc, vm, fk, dfq, rec_g0}, a1{fk, fq, gt, dvf, rec_g1},
        a2{vm, gc, fq, dfk, rec_g2};
    const int P = pl.P_g;
    if (P > 1) {
      auto ks = gradient_products_kernel<D, DV, kPassState>;
      if ((e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
          cudaSuccess)
        return e;
      ks<<<dim3((unsigned)(BH * (P - 1)), ny, 3), kThreads, smem, s>>>(a0, a1, a2, P, p.H, p.N, g);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      constexpr int kMaxEntries = (DV4 * D > D * DV ? DV4 * D : D * DV);
      gradient_scan_kernel<D, DV><<<dim3((unsigned)BH, (kMaxEntries + 255) / 256, 3), 256, 0, s>>>(
          rec_g0, rec_g1, rec_g2, P, p.H, p.N, g);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    auto ko = gradient_products_kernel<D, DV, kPassOut>;
    if ((e = cudaFuncSetAttribute(ko, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    ko<<<dim3((unsigned)(BH * P), ny, 3), kThreads, smem, s>>>(a0, a1, a2, P, p.H, p.N, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
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
  const BwdPlan pl = bwd_plan(BH, N, D, Dv);
  return sizeof(float) * (rows * (4 * static_cast<size_t>(D) + 4 * (Dv + 4) + 2 * Dv) +
                          pl.rec_nd + pl.rec_g0 + pl.rec_g1 + pl.rec_g2);
}

int backward_launches(int BH, int N, int D, int Dv) {
  const BwdPlan pl = bwd_plan(BH, N, D, Dv);
  return 3 + (pl.P_nd > 1 ? 3 : 1) + (pl.P_g > 1 ? 3 : 1);
}

cudaError_t launch_backward(const Problem &p, const void *dO, void *dq, void *dk, void *dv,
                            const Gammas &g, void *ws, cudaStream_t s) {
  float *w = static_cast<float *>(ws);
  return p.dtype == kF32 ? backward_shape<float>(p, dO, dq, dk, dv, g, w, s)
                         : backward_shape<__nv_bfloat16>(p, dO, dq, dk, dv, g, w, s);
}

}  // namespace linattn
