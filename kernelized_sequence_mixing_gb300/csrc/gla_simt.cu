// Gated causal linear attention on CUDA cores (fp32), chunked and split into
// sequence parts.
//
// "Linear Attention Mechanisms" (dileepadev.github.io), "Gating and Selective
// State Updates", gated linear attention: S_t = G_t (.) S_(t-1) + phi(k_t) v_t^T
// with a data-dependent gate G_t in [0, 1]^(D x Dv).  The gate is one value per
// key feature and step, G_t = a_t 1^T (row d of the state is scaled by
// a_t[d]); the normaliser is gated the same way, z_t = a_t (.) z_(t-1) +
// phi(k_t), and o_t = phi(q_t)^T S_t / (phi(q_t) . z_t + eps).
//
// Chunk form.  Within a chunk with local index t and per-feature prefix
// products c_t = a_0 (.) ... (.) a_t, the recurrence unrolls to
//   S_t = diag(c_t) S_in + sum_(s<=t) diag(c_t / c_s) phi(k_s) v_s^T.
// With qc_t = c_t (.) phi(q_t) and kc_s = phi(k_s) / c_s:
//   o_t   = (sum_(s<=t) (qc_t . kc_s) v_s + qc_t^T S_in)
//           / (sum_(s<=t) qc_t . kc_s + qc_t . z_in + eps)
//   S_out = diag(c_last) (S_in + sum_s kc_s v_s^T), z likewise.
// Dividing by c_s is safe while every feature keeps c_last >= 2^-100 over the
// chunk: then kc_s <= 2^100 phi(k_s) and every product stays inside fp32
// range.  A chunk that forgets harder than that in some feature runs the
// token recurrence itself instead, which is exact for every gate in [0, 1],
// 0 included.
//
// Sequence parts.  The tokens of one (batch, head) split into P parts of whole
// chunks.  The state pass gives every part but the last its own end state
// from zero, A_p = sum_(s in p) diag(prod_(u>s in p) a_u) phi(k_s) v_s^T (the
// suffix products are at most 1, so no threshold is needed), and its gate
// product g_p.  A scan turns the records into the state after each part,
// S_after(p) = diag(g_p) S_after(p-1) + A_p, and the output pass runs each
// part from the state after the previous one.  One CTA owns one (batch, head,
// part) and a 32-column slice of Dv.
#include "common.cuh"
#include "kernels.h"

namespace linattn {
namespace {

constexpr int kC = 64;        // tokens per chunk
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kLd = kC + 4;   // row stride of the transposed tiles
constexpr int kDvs = 32;      // Dv columns per CTA
constexpr float kMinProd = 0x1p-100f;

template <int D>
struct GlaLayout {
  static constexpr int tile = D * kLd;
  static constexpr int total = 3 * tile + kC * kDvs + D * kDvs + 3 * D + kC +
                               2 * kWarps * kDvs + 2 * kWarps;
  static constexpr size_t bytes = sizeof(float) * total;
};
// the masked A tile reuses the gate tile once the prefix products are taken
static_assert(kC * (kC + 1) <= 64 * kLd, "A tile must fit in the gate tile");

enum { kPassState = 0, kPassOut = 1 };

__host__ __device__ inline int part_chunk(int p, int P, int nch) {
  return static_cast<int>((static_cast<long long>(p) * nch) / P);
}

template <int D, int DV>
__host__ __device__ constexpr size_t record_floats() {
  return static_cast<size_t>(D) * DV + 2 * D;  // A_p | z part | g_p
}

// Row d of the state slice: S = c (S + sum_s kc_s v_s) when `fold`, else
// S = c S + sum_s kc_s v_s; z likewise.  Warp w owns rows d = w, w + 8, ...
template <int D>
__device__ __forceinline__ void state_update(float *Ss, float *zs, const float *fkT,
                                             const float *vs, const float *cl, int nv,
                                             bool fold, int warp, int lane) {
  for (int d = warp; d < D; d += kWarps) {
    float acc = 0.f, zp = 0.f;
    for (int s = 0; s < nv; ++s) acc = fmaf(fkT[d * kLd + s], vs[s * kDvs + lane], acc);
    for (int s = lane; s < nv; s += 32) zp += fkT[d * kLd + s];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zp += __shfl_xor_sync(0xffffffffu, zp, off);
    const float c = cl[d];
    if (fold) {
      Ss[d * kDvs + lane] = c * (Ss[d * kDvs + lane] + acc);
      if (lane == 0) zs[d] = c * (zs[d] + zp);
    } else {
      Ss[d * kDvs + lane] = fmaf(c, Ss[d * kDvs + lane], acc);
      if (lane == 0) zs[d] = fmaf(c, zs[d], zp);
    }
  }
}

// grid: x = (batch, head) * Pg + part, y = Dv / 32; Pg = P - 1 for the state
// pass (the last part needs no record), P for the output pass.
template <int D, int DV, int PASS, typename T>
__global__ void __launch_bounds__(kThreads)
    gla_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                    const T *__restrict__ v, const float *__restrict__ a,
                    T *__restrict__ o, float *__restrict__ rec,
                    float *__restrict__ S_out, float *__restrict__ z_out, int N,
                    int P, int Pg, float eps) {
  extern __shared__ float4 smem4[];
  using L = GlaLayout<D>;
  float *fqT = reinterpret_cast<float *>(smem4);  // [D][kLd] phi(q)^T, then qc^T
  float *fkT = fqT + L::tile;                     // [D][kLd] phi(k)^T, then kc^T
  float *aT = fkT + L::tile;                      // [D][kLd] gates^T
  float *As = aT;                                 // [kC][kC+1] masked A tile
  float *vs = aT + L::tile;                       // [kC][kDvs]
  float *Ss = vs + kC * kDvs;                     // [D][kDvs] state slice
  float *zs = Ss + D * kDvs;                      // [D]
  float *cl = zs + D;                             // [D] c_last of the chunk
  float *gp = cl + D;                             // [D] gate product of the part
  float *den = gp + D;                            // [kC]
  float *red = den + kC;                          // [2][kWarps][kDvs]
  float *redz = red + 2 * kWarps * kDvs;          // [2][kWarps]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = blockIdx.x / Pg, part = blockIdx.x % Pg;
  const int e0 = blockIdx.y * kDvs;
  const int nch = (N + kC - 1) / kC;
  const int cb = part_chunk(part, P, nch), ce = part_chunk(part + 1, P, nch);
  constexpr size_t R = record_floats<D, DV>();
  const int64_t qk0 = static_cast<int64_t>(bh) * N * D;
  const int64_t v0 = static_cast<int64_t>(bh) * N * DV;

  if (PASS == kPassOut && part > 0) {
    const float *r = rec + (static_cast<size_t>(bh) * (P - 1) + part - 1) * R;
    for (int i = tid; i < D * kDvs; i += kThreads)
      Ss[i] = r[(i / kDvs) * DV + e0 + i % kDvs];
    for (int i = tid; i < D; i += kThreads) zs[i] = r[D * DV + i];
  } else {
    for (int i = tid; i < D * kDvs; i += kThreads) Ss[i] = 0.f;
    for (int i = tid; i < D; i += kThreads) zs[i] = 0.f;
  }
  for (int i = tid; i < D; i += kThreads) gp[i] = 1.f;
  __syncthreads();

  const int ty = tid >> 4, tx = tid & 15;  // 16 x 16 grid over the A tile
  for (int c = cb; c < ce; ++c) {
    const int c0 = c * kC, nv = min(kC, N - c0);
    // 1. phi(q), phi(k) and the gates, transposed; the v slice.  Rows past the
    //    end of the sequence: zero features, gate 1.
    for (int i = tid; i < kC * D; i += kThreads) {
      const int t = i / D, d = i % D;
      float xq = 0.f, xk = 0.f, xa = 1.f;
      if (t < nv) {
        const int64_t off = qk0 + static_cast<int64_t>(c0 + t) * D + d;
        if (PASS == kPassOut) xq = phi_f32(io<T>::load(q + off));
        xk = phi_f32(io<T>::load(k + off));
        xa = a[off];
      }
      if (PASS == kPassOut) fqT[d * kLd + t] = xq;
      fkT[d * kLd + t] = xk;
      aT[d * kLd + t] = xa;
    }
    for (int i = tid; i < kC * kDvs; i += kThreads) {
      const int t = i / kDvs, e = i % kDvs;
      vs[i] = t < nv ? io<T>::load(v + v0 + static_cast<int64_t>(c0 + t) * DV + e0 + e) : 0.f;
    }
    __syncthreads();

    if (PASS == kPassState) {
      // suffix products: kc_s = phi(k_s) prod_(u>s) a_u, c_last = prod a
      if (tid < D) {
        float suf = 1.f;
        for (int t = kC - 1; t >= 0; --t) {
          fkT[tid * kLd + t] *= suf;
          suf *= aT[tid * kLd + t];
        }
        cl[tid] = suf;
        gp[tid] *= suf;
      }
      __syncthreads();
      state_update<D>(Ss, zs, fkT, vs, cl, nv, false, warp, lane);
      __syncthreads();
      continue;
    }

    bool hard = false;  // some feature forgets below 2^-100 within the chunk
    if (tid < D) {
      float cp = 1.f;
      for (int t = 0; t < nv; ++t) cp *= aT[tid * kLd + t];
      hard = !(cp >= kMinProd);
    }
    if (!__syncthreads_or(hard)) {
      // 2. prefix products: qc_t = c_t phi(q_t), kc_s = phi(k_s) / c_s
      if (tid < D) {
        float cp = 1.f;
        for (int t = 0; t < kC; ++t) {
          cp *= aT[tid * kLd + t];
          fqT[tid * kLd + t] *= cp;
          fkT[tid * kLd + t] /= cp;
        }
        cl[tid] = cp;
      }
      __syncthreads();
      // 3. masked A tile and the denominators
      {
        float acc[4][4] = {};
#pragma unroll 4
        for (int d = 0; d < D; ++d) {
          const float4 x = *reinterpret_cast<const float4 *>(fqT + d * kLd + ty * 4);
          const float4 y = *reinterpret_cast<const float4 *>(fkT + d * kLd + tx * 4);
          const float xv[4] = {x.x, x.y, x.z, x.w};
          const float yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], yv[j], acc[i][j]);
        }
        float rs[4], qz[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = ty * 4 + i;
          rs[i] = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int s = tx * 4 + j;
            const float x = s <= t ? acc[i][j] : 0.f;
            As[t * (kC + 1) + s] = x;
            rs[i] += x;
          }
          float p = 0.f;  // qc_t . z_in, split over the 16 tx lanes
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
          for (int i = 0; i < 4; ++i) den[ty * 4 + i] = rs[i] + qz[i] + eps;
        }
      }
      __syncthreads();
      // 4. o_t = (A_t. V + qc_t^T S_in) / den_t; warp w owns rows 8w..8w+7
      {
        constexpr int Rw = kC / kWarps;
        const int t0 = warp * Rw;
        float num[Rw];
#pragma unroll
        for (int r = 0; r < Rw; ++r) num[r] = 0.f;
        for (int s = 0; s < kC; ++s) {
          const float vv = vs[s * kDvs + lane];
#pragma unroll
          for (int r = 0; r < Rw; ++r) num[r] = fmaf(As[(t0 + r) * (kC + 1) + s], vv, num[r]);
        }
#pragma unroll 4
        for (int d = 0; d < D; ++d) {
          const float sv = Ss[d * kDvs + lane];
          const float4 f0 = *reinterpret_cast<const float4 *>(fqT + d * kLd + t0);
          const float4 f1 = *reinterpret_cast<const float4 *>(fqT + d * kLd + t0 + 4);
          const float fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
          for (int r = 0; r < Rw; ++r) num[r] = fmaf(fv[r], sv, num[r]);
        }
#pragma unroll
        for (int r = 0; r < Rw; ++r) {
          const int t = t0 + r;
          if (t < nv)
            io<T>::store(o + v0 + static_cast<int64_t>(c0 + t) * DV + e0 + lane, num[r] / den[t]);
        }
      }
      __syncthreads();
      // 5. S = diag(c_last) (S + sum_s kc_s v_s^T), z likewise
      state_update<D>(Ss, zs, fkT, vs, cl, nv, true, warp, lane);
      __syncthreads();
    } else {
      // The token recurrence: thread (warp w, lane e) owns S[d][e] for
      // d = w, w + 8, ...; lane 0 also owns z[d].  Partial read-outs meet in a
      // double-buffered reduction, so one barrier per token suffices.
      for (int t = 0; t < nv; ++t) {
        const float ve = vs[t * kDvs + lane];
        float num = 0.f, qz = 0.f;
        for (int d = warp; d < D; d += kWarps) {
          const float al = aT[d * kLd + t], fk = fkT[d * kLd + t], fq = fqT[d * kLd + t];
          const float sn = fmaf(al, Ss[d * kDvs + lane], fk * ve);
          Ss[d * kDvs + lane] = sn;
          num = fmaf(fq, sn, num);
          if (lane == 0) {
            const float zn = fmaf(al, zs[d], fk);
            zs[d] = zn;
            qz = fmaf(fq, zn, qz);
          }
        }
        float *rb = red + (t & 1) * kWarps * kDvs;
        float *rz = redz + (t & 1) * kWarps;
        rb[warp * kDvs + lane] = num;
        if (lane == 0) rz[warp] = qz;
        __syncthreads();
        if (warp == 0) {
          float n = 0.f, dz = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            n += rb[w * kDvs + lane];
            dz += rz[w];
          }
          io<T>::store(o + v0 + static_cast<int64_t>(c0 + t) * DV + e0 + lane, n / (dz + eps));
        }
      }
      __syncthreads();
    }
  }

  if (PASS == kPassState) {
    float *r = rec + (static_cast<size_t>(bh) * (P - 1) + part) * R;
    for (int i = tid; i < D * kDvs; i += kThreads) r[(i / kDvs) * DV + e0 + i % kDvs] = Ss[i];
    if (blockIdx.y == 0)
      for (int i = tid; i < D; i += kThreads) {
        r[D * DV + i] = zs[i];
        r[D * DV + D + i] = gp[i];
      }
  } else if (S_out && part == P - 1) {
    float *Sb = S_out + static_cast<size_t>(bh) * D * DV;
    for (int i = tid; i < D * kDvs; i += kThreads) Sb[(i / kDvs) * DV + e0 + i % kDvs] = Ss[i];
    if (blockIdx.y == 0)
      for (int i = tid; i < D; i += kThreads) z_out[static_cast<size_t>(bh) * D + i] = zs[i];
  }
}

// In place over the records of one (batch, head): record p becomes the state
// after part p, S_after(p) = g_p (.) S_after(p-1) + A_p (rows scaled by g_p).
// grid: x = (batch, head), y = blocks over the D*Dv + D state entries.
template <int D, int DV>
__global__ void __launch_bounds__(256) gla_scan_kernel(float *__restrict__ rec, int P) {
  constexpr size_t R = record_floats<D, DV>();
  const int i = blockIdx.y * blockDim.x + threadIdx.x;
  if (i >= D * DV + D) return;
  const int d = i < D * DV ? i / DV : i - D * DV;
  float *r = rec + static_cast<size_t>(blockIdx.x) * (P - 1) * R;
  float carry = 0.f;
  for (int p = 0; p < P - 1; ++p) {
    float *rp = r + p * R;
    carry = fmaf(rp[D * DV + D + d], carry, rp[i]);
    rp[i] = carry;
  }
}

int num_sms_gla() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

template <int D, int DV, typename T>
cudaError_t gla_typed(const Problem &p, const float *a, float *ws, int P, float *S_out,
                      float *z_out, cudaStream_t s) {
  const int BH = p.B * p.H;
  const size_t smem = GlaLayout<D>::bytes;
  auto kst = gla_simt_kernel<D, DV, kPassState, T>;
  auto kout = gla_simt_kernel<D, DV, kPassOut, T>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kst, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(kout, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return e;
  const T *q = static_cast<const T *>(p.q), *k = static_cast<const T *>(p.k),
          *v = static_cast<const T *>(p.v);
  T *o = static_cast<T *>(p.o);
  if (P > 1) {
    kst<<<dim3((unsigned)(BH * (P - 1)), DV / kDvs), kThreads, smem, s>>>(
        q, k, v, a, o, ws, nullptr, nullptr, p.N, P, P - 1, p.eps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    gla_scan_kernel<D, DV><<<dim3((unsigned)BH, (D * DV + D + 255) / 256), 256, 0, s>>>(ws, P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  kout<<<dim3((unsigned)(BH * P), DV / kDvs), kThreads, smem, s>>>(
      q, k, v, a, o, ws, S_out, z_out, p.N, P, P, p.eps);
  return cudaGetLastError();
}

template <typename T>
cudaError_t gla_shape(const Problem &p, const float *a, float *ws, int P, float *S_out,
                      float *z_out, cudaStream_t s) {
  if (p.D == 64 && p.Dv == 64) return gla_typed<64, 64, T>(p, a, ws, P, S_out, z_out, s);
  if (p.D == 64 && p.Dv == 128) return gla_typed<64, 128, T>(p, a, ws, P, S_out, z_out, s);
  if (p.D == 128 && p.Dv == 64) return gla_typed<128, 64, T>(p, a, ws, P, S_out, z_out, s);
  if (p.D == 128 && p.Dv == 128) return gla_typed<128, 128, T>(p, a, ws, P, S_out, z_out, s);
  return cudaErrorNotSupported;
}

}  // namespace

int gla_parts(int BH, int N, int Dv) {
  if (BH <= 0 || N <= 0) return 1;
  const long long nch = (N + kC - 1) / kC;
  const long long ctas = static_cast<long long>(BH) * (Dv / kDvs);
  long long P = (2LL * num_sms_gla() + ctas - 1) / ctas;
  if (P > nch) P = nch;
  if (P < 1) P = 1;
  return static_cast<int>(P);
}

size_t gla_workspace_bytes(int BH, int P, int D, int Dv) {
  if (P <= 1) return 0;
  return sizeof(float) * static_cast<size_t>(BH) * (P - 1) *
         (static_cast<size_t>(D) * Dv + 2 * static_cast<size_t>(D));
}

cudaError_t launch_gla_simt(const Problem &p, const float *a, void *ws, int P, float *S_out,
                            float *z_out, cudaStream_t s) {
  if (P < 1 || (P > 1 && !ws)) return cudaErrorInvalidValue;
  float *w = static_cast<float *>(ws);
  return p.dtype == kF32 ? gla_shape<float>(p, a, w, P, S_out, z_out, s)
                         : gla_shape<__nv_bfloat16>(p, a, w, P, S_out, z_out, s);
}

}  // namespace linattn
