// Gated causal linear attention on CUDA cores (fp32), chunked and split into
// sequence parts.
//
// "Linear Attention Mechanisms" (dileepadev.github.io), "Gating and Selective
// State Updates", gated linear attention: S_t = G_t (.) S_(t-1) + phi(k_t) v_t^T,
// where G_t has the state's D x Dv shape, entries in [0, 1], and is computed
// from step t's input.  Here the gate is one value per key feature and step,
// G_t = a_t 1^T (row d of the state is scaled by a_t[d]); the normaliser is
// gated the same way, z_t = a_t (.) z_(t-1) + phi(k_t), and
// o_t = phi(q_t)^T S_t / (phi(q_t) . z_t + eps).
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
// part from the state after the previous one.
//
// One CTA (8 warps) owns one (batch, head, part) and a 32-column slice of Dv;
// about 109 KB of shared memory at D = 128, so two CTAs share an SM and one
// loads while the other computes.  Per chunk:
//   load   lane l of warp w holds tokens l and 32 + l of feature groups
//          {w, w + 8} (8 features each): 16-byte loads, the prefix (or
//          suffix) products of the gates by warp shuffles, the scaled
//          features stored transposed ([feature][token]) without bank
//          conflicts;
//   A      16 x 16 threads, 4 x 4 register tiles of qc kc^T, masked, stored
//          transposed ([s][t]);
//   output 4 tokens x 2 columns per thread (two shared loads per 8 FMAs);
//   state  4 feature rows x 4 columns per thread (two 16-byte shared loads
//          per 16 FMAs).
#include "common.cuh"
#include "kernels.h"

namespace linattn {
namespace {

constexpr int kC = 64;        // tokens per chunk
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kLdA = kC + 4;  // row stride of the transposed A tile
constexpr int kDvs = 32;      // Dv columns per CTA
constexpr float kMinProd = 0x1p-100f;

template <int D>
struct GlaLayout {
  static constexpr int tile = D * kC;  // [D][kC] transposed features
  static constexpr int total = 2 * tile + kC * kLdA + kC * kDvs + D * kDvs + 3 * D + kC +
                               2 * kWarps * kDvs + 2 * kWarps;
  static constexpr size_t bytes = sizeof(float) * total;
};

enum { kPassState = 0, kPassOut = 1 };

__host__ __device__ inline int part_chunk(int p, int P, int nch) {
  return static_cast<int>((static_cast<long long>(p) * nch) / P);
}

template <int D, int DV>
__host__ __device__ constexpr size_t record_floats() {
  return static_cast<size_t>(D) * DV + 2 * D;  // A_p | z part | g_p
}

// 8 consecutive values widened to fp32 (16-byte aligned source).
__device__ __forceinline__ void load8(const float *p, float *x) {
  const float4 a = *reinterpret_cast<const float4 *>(p);
  const float4 b = *reinterpret_cast<const float4 *>(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float *x) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void store2(float *p, float a, float b) {
  *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}
__device__ __forceinline__ void store2(__nv_bfloat16 *p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}

// Inclusive products along the warp: lane l gets x_0 * ... * x_l.
__device__ __forceinline__ float scan_prod(float x, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x *= y;
  }
  return x;
}
// Inclusive suffix products: lane l gets x_l * ... * x_31.
__device__ __forceinline__ float scan_prod_rev(float x, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_down_sync(0xffffffffu, x, off);
    if (lane + off < 32) x *= y;
  }
  return x;
}

// One (batch, head, part) and 32-column slice of Dv: vb = (batch, head) * Pg
// + part, the slice blockIdx.y; Pg = P - 1 for the state pass (the last part
// needs no record), P for the output pass.
template <int D, int DV, int PASS, typename T>
__device__ __forceinline__ void gla_simt_block(const T *__restrict__ q, const T *__restrict__ k,
                                               const T *__restrict__ v, const float *__restrict__ a,
                                               T *__restrict__ o, float *__restrict__ rec,
                                               float *__restrict__ S_out, float *__restrict__ z_out,
                                               int N, int P, int Pg, float eps, int vb) {
  constexpr int NG = D / 64;  // feature groups of 8 per warp
  constexpr int RD = D / 32;  // state rows per thread
  extern __shared__ float4 smem4[];
  using L = GlaLayout<D>;
  float *fq = reinterpret_cast<float *>(smem4);  // [D][kC] qc (or phi(q))
  float *fk = fq + L::tile;                      // [D][kC] kc (or phi(k))
  float *AT = fk + L::tile;                      // [kC][kLdA] masked A, transposed
  float *vs = AT + kC * kLdA;                    // [kC][kDvs]
  float *Ss = vs + kC * kDvs;                    // [D][kDvs] state slice
  float *zs = Ss + D * kDvs;                     // [D]
  float *cl = zs + D;                            // [D] c_last of the chunk
  float *gp = cl + D;                            // [D] gate product of the part
  float *den = gp + D;                           // [kC]
  float *red = den + kC;                         // [2][kWarps][kDvs]
  float *redz = red + 2 * kWarps * kDvs;         // [2][kWarps]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = vb / Pg, part = vb % Pg;
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

  for (int c = cb; c < ce; ++c) {
    const int c0 = c * kC, nv = min(kC, N - c0);
    // ---- load: tokens t = lane + 32 h, features 8 g .. 8 g + 7 for the
    // groups g = w + 8 gi.  phi(q), phi(k) go to shared memory as they are
    // (transposed; rows past the end are 0), the gates stay in registers.
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = lane + 32 * h, g = warp + kWarps * gi;
        float xk[8], xq[8];
        if (t < nv) {
          const int64_t off = qk0 + static_cast<int64_t>(c0 + t) * D + 8 * g;
          load8(k + off, xk);
          if (PASS == kPassOut) load8(q + off, xq);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            xk[j] = phi_f32(xk[j]);
            if (PASS == kPassOut) xq[j] = phi_f32(xq[j]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) xk[j] = xq[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          fk[(8 * g + j) * kC + t] = xk[j];
          if (PASS == kPassOut) fq[(8 * g + j) * kC + t] = xq[j];
        }
      }
    float xa[NG][2][8];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = lane + 32 * h, g = warp + kWarps * gi;
        if (t < nv) {
          load8(a + qk0 + static_cast<int64_t>(c0 + t) * D + 8 * g, xa[gi][h]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) xa[gi][h][j] = 1.f;
        }
      }
    {
      const int row = tid >> 2, col = 8 * (tid & 3);
      float xv[8];
      if (row < nv) {
        load8(v + v0 + static_cast<int64_t>(c0 + row) * DV + e0 + col, xv);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) xv[j] = 0.f;
      }
      *reinterpret_cast<float4 *>(vs + row * kDvs + col) = make_float4(xv[0], xv[1], xv[2], xv[3]);
      *reinterpret_cast<float4 *>(vs + row * kDvs + col + 4) = make_float4(xv[4], xv[5], xv[6], xv[7]);
    }

    if (PASS == kPassState) {
      // exclusive suffix products: kc_s = phi(k_s) prod_(u>s) a_u (each
      // thread rescales the entries it stored itself)
#pragma unroll
      for (int gi = 0; gi < NG; ++gi)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float s1 = scan_prod_rev(xa[gi][1][j], lane);
          const float p1 = __shfl_sync(0xffffffffu, s1, 0);
          const float s0 = scan_prod_rev(xa[gi][0][j], lane) * p1;
          float e1 = __shfl_down_sync(0xffffffffu, s1, 1);
          float e0x = __shfl_down_sync(0xffffffffu, s0, 1);
          if (lane == 31) {
            e1 = 1.f;
            e0x = p1;
          }
          const int d = 8 * (warp + kWarps * gi) + j;
          fk[d * kC + lane] *= e0x;
          fk[d * kC + 32 + lane] *= e1;
          if (lane == 0) {
            cl[d] = s0;
            gp[d] *= s0;
          }
        }
      __syncthreads();
    } else {
      // inclusive prefix products c_t; a chunk is hard if some feature's
      // product over the chunk falls below 2^-100 (or is NaN)
      bool hard = false;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float c0v = scan_prod(xa[gi][0][j], lane);
          const float c1v = scan_prod(xa[gi][1][j], lane) * __shfl_sync(0xffffffffu, c0v, 31);
          const float tot = __shfl_sync(0xffffffffu, c1v, 31);
          hard |= !(tot >= kMinProd);
          xa[gi][0][j] = c0v;
          xa[gi][1][j] = c1v;
        }
      if (!__syncthreads_or(hard)) {
        // qc = c_t phi(q_t), kc = phi(k_t) / c_t on the thread's own entries
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int d = 8 * (warp + kWarps * gi) + j;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              fq[d * kC + 32 * h + lane] *= xa[gi][h][j];
              fk[d * kC + 32 * h + lane] /= xa[gi][h][j];
            }
            if (lane == 31) cl[d] = xa[gi][1][j];
          }
        __syncthreads();
        // ---- A = qc kc^T masked (s <= t), stored as AT[s][t]; denominators
        {
          const int ty = tid >> 4, tx = tid & 15;
          float acc[4][4] = {};
          if (tx <= ty) {
#pragma unroll 4
            for (int d = 0; d < D; ++d) {
              const float4 x = *reinterpret_cast<const float4 *>(fq + d * kC + 4 * ty);
              const float4 y = *reinterpret_cast<const float4 *>(fk + d * kC + 4 * tx);
              const float xv[4] = {x.x, x.y, x.z, x.w};
              const float yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
              for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], yv[j], acc[i][j]);
            }
          }
          float rs[4], qz[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int t = 4 * ty + i;
            rs[i] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (4 * tx + j > t) acc[i][j] = 0.f;
              rs[i] += acc[i][j];
            }
            float p = 0.f;  // qc_t . z_in, split over the 16 tx lanes
            for (int d = tx; d < D; d += 16) p = fmaf(fq[d * kC + t], zs[d], p);
            qz[i] = p;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float4 *>(AT + (4 * tx + j) * kLdA + 4 * ty) =
                make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
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
            for (int i = 0; i < 4; ++i) den[4 * ty + i] = rs[i] + qz[i] + eps;
          }
        }
        __syncthreads();
        // ---- o_t = (A_t. V + qc_t^T S_in) / den_t: 4 tokens x 2 columns
        {
          const int ep = tid & 15, tg = tid >> 4;
          float num[4][2] = {};
          const int smax = 4 * tg + 4;
          for (int s = 0; s < smax; ++s) {
            const float4 w = *reinterpret_cast<const float4 *>(AT + s * kLdA + 4 * tg);
            const float2 x = *reinterpret_cast<const float2 *>(vs + s * kDvs + 2 * ep);
            const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              num[i][0] = fmaf(wv[i], x.x, num[i][0]);
              num[i][1] = fmaf(wv[i], x.y, num[i][1]);
            }
          }
#pragma unroll 4
          for (int d = 0; d < D; ++d) {
            const float4 f = *reinterpret_cast<const float4 *>(fq + d * kC + 4 * tg);
            const float2 sv = *reinterpret_cast<const float2 *>(Ss + d * kDvs + 2 * ep);
            const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              num[i][0] = fmaf(fv[i], sv.x, num[i][0]);
              num[i][1] = fmaf(fv[i], sv.y, num[i][1]);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int t = 4 * tg + i;
            if (t < nv) {
              const float dn = den[t];
              store2(o + v0 + static_cast<int64_t>(c0 + t) * DV + e0 + 2 * ep, num[i][0] / dn,
                     num[i][1] / dn);
            }
          }
        }
        __syncthreads();
      } else {
        // ---- the token recurrence on raw features: thread (warp w, lane e)
        // owns S[d][e] for d = w, w + 8, ...; lane 0 also owns z[d].  Partial
        // read-outs meet in a double-buffered reduction (one barrier a token).
        // The raw features are already in shared memory (the barrier above).
        const float *ac = a + qk0 + static_cast<int64_t>(c0) * D;
        for (int t = 0; t < nv; ++t) {
          const float ve = vs[t * kDvs + lane];
          float num = 0.f, qzp = 0.f;
          for (int d = warp; d < D; d += kWarps) {
            const float al = ac[t * D + d], fkv = fk[d * kC + t], fqv = fq[d * kC + t];
            const float sn = fmaf(al, Ss[d * kDvs + lane], fkv * ve);
            Ss[d * kDvs + lane] = sn;
            num = fmaf(fqv, sn, num);
            if (lane == 0) {
              const float zn = fmaf(al, zs[d], fkv);
              zs[d] = zn;
              qzp = fmaf(fqv, zn, qzp);
            }
          }
          float *rb = red + (t & 1) * kWarps * kDvs;
          float *rz = redz + (t & 1) * kWarps;
          rb[warp * kDvs + lane] = num;
          if (lane == 0) rz[warp] = qzp;
          __syncthreads();
          if (warp == 0) {
            float n = 0.f, dz = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
              n += rb[w * kDvs + lane];
              dz += rz[w];
            }
            const float ov = n / (dz + eps);
            o[v0 + static_cast<int64_t>(c0 + t) * DV + e0 + lane] =
                static_cast<T>(ov);
          }
        }
        __syncthreads();
        continue;
      }
    }
    // ---- state: S = c_last (S + sum kc v) (output pass) or c_last S +
    // sum kc v (state pass); z likewise.  4 (D = 128) or 2 feature rows x 4
    // columns per thread.
    {
      const int eq = tid & 7, dq = tid >> 3;
      float acc[RD][4] = {}, zp[RD] = {};
#pragma unroll 2
      for (int s = 0; s < kC; s += 4) {
        float4 kv[RD], vv[4];
#pragma unroll
        for (int r = 0; r < RD; ++r)
          kv[r] = *reinterpret_cast<const float4 *>(fk + (RD * dq + r) * kC + s);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          vv[j] = *reinterpret_cast<const float4 *>(vs + (s + j) * kDvs + 4 * eq);
#pragma unroll
        for (int r = 0; r < RD; ++r) {
          const float kr[4] = {kv[r].x, kv[r].y, kv[r].z, kv[r].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[r][0] = fmaf(kr[j], vv[j].x, acc[r][0]);
            acc[r][1] = fmaf(kr[j], vv[j].y, acc[r][1]);
            acc[r][2] = fmaf(kr[j], vv[j].z, acc[r][2]);
            acc[r][3] = fmaf(kr[j], vv[j].w, acc[r][3]);
            zp[r] += kr[j];
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RD; ++r) {
        const int d = RD * dq + r;
        const float cv = cl[d];
        float4 *sp = reinterpret_cast<float4 *>(Ss + d * kDvs + 4 * eq);
        float4 sv = *sp;
        if (PASS == kPassOut) {
          sv.x = cv * (sv.x + acc[r][0]);
          sv.y = cv * (sv.y + acc[r][1]);
          sv.z = cv * (sv.z + acc[r][2]);
          sv.w = cv * (sv.w + acc[r][3]);
          if (eq == 0) zs[d] = cv * (zs[d] + zp[r]);
        } else {
          sv.x = fmaf(cv, sv.x, acc[r][0]);
          sv.y = fmaf(cv, sv.y, acc[r][1]);
          sv.z = fmaf(cv, sv.z, acc[r][2]);
          sv.w = fmaf(cv, sv.w, acc[r][3]);
          if (eq == 0) zs[d] = fmaf(cv, zs[d], zp[r]);
        }
        *sp = sv;
      }
    }
    __syncthreads();
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

// grid: x strides over the nvb = (batch, head) * Pg blocks of
// gla_simt_block, y = Dv / 32.  Behind the tensor-core form (only_if set)
// the grid is one wave, so that it costs one wave of early exits when that
// form covered every chunk.
template <int D, int DV, int PASS, typename T>
__global__ void __launch_bounds__(kThreads, 2)
    gla_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                    const T *__restrict__ v, const float *__restrict__ a,
                    T *__restrict__ o, float *__restrict__ rec,
                    float *__restrict__ S_out, float *__restrict__ z_out, int N,
                    int P, int Pg, float eps, int nvb, const int *__restrict__ only_if) {
  if (only_if && *only_if == 0) return;  // uniform: the tensor-core form ran
  for (int vb = blockIdx.x; vb < nvb; vb += gridDim.x) {
    gla_simt_block<D, DV, PASS, T>(q, k, v, a, o, rec, S_out, z_out, N, P, Pg, eps, vb);
    __syncthreads();  // shared memory is reused by the next block
  }
}

// In place over the records of one (batch, head): record p becomes the state
// after part p, S_after(p) = g_p (.) S_after(p-1) + A_p (rows scaled by g_p).
// grid: x strides over the BH (batch, head) pairs, y = blocks over the
// D*Dv + D state entries.
template <int D, int DV>
__global__ void __launch_bounds__(256) gla_scan_kernel(float *__restrict__ rec, int P, int BH,
                                                      const int *__restrict__ only_if) {
  if (only_if && *only_if == 0) return;
  constexpr size_t R = record_floats<D, DV>();
  const int i = blockIdx.y * blockDim.x + threadIdx.x;
  if (i >= D * DV + D) return;
  const int d = i < D * DV ? i / DV : i - D * DV;
  for (int bh = blockIdx.x; bh < BH; bh += gridDim.x) {
    float *r = rec + static_cast<size_t>(bh) * (P - 1) * R;
    float carry = 0.f;
    for (int p = 0; p < P - 1; ++p) {
      float *rp = r + p * R;
      carry = fmaf(rp[D * DV + D + d], carry, rp[i]);
      rp[i] = carry;
    }
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
                      float *z_out, const int *only_if, cudaStream_t s) {
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
  // behind the tensor-core form: grids of one wave (two CTAs per SM of the
  // passes, eight of the scan), strided over the blocks
  const long long sms = num_sms_gla();
  auto cap = [&](long long nblocks, long long per_wave) {
    return static_cast<unsigned>(only_if && nblocks > per_wave ? per_wave : nblocks);
  };
  const int ys = DV / kDvs, yscan = (D * DV + D + 255) / 256;
  const long long pass_wave = (2 * sms + ys - 1) / ys, scan_wave = (8 * sms + yscan - 1) / yscan;
  if (P > 1) {
    const int nvb = BH * (P - 1);
    kst<<<dim3(cap(nvb, pass_wave), ys), kThreads, smem, s>>>(q, k, v, a, o, ws, nullptr, nullptr, p.N,
                                                              P, P - 1, p.eps, nvb, only_if);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    gla_scan_kernel<D, DV><<<dim3(cap(BH, scan_wave), yscan), 256, 0, s>>>(ws, P, BH, only_if);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int nvb = BH * P;
  kout<<<dim3(cap(nvb, pass_wave), ys), kThreads, smem, s>>>(q, k, v, a, o, ws, S_out, z_out, p.N, P, P,
                                                             p.eps, nvb, only_if);
  return cudaGetLastError();
}

template <typename T>
cudaError_t gla_shape(const Problem &p, const float *a, float *ws, int P, float *S_out,
                      float *z_out, const int *only_if, cudaStream_t s) {
  if (p.D == 64 && p.Dv == 64) return gla_typed<64, 64, T>(p, a, ws, P, S_out, z_out, only_if, s);
  if (p.D == 64 && p.Dv == 128) return gla_typed<64, 128, T>(p, a, ws, P, S_out, z_out, only_if, s);
  if (p.D == 128 && p.Dv == 64) return gla_typed<128, 64, T>(p, a, ws, P, S_out, z_out, only_if, s);
  if (p.D == 128 && p.Dv == 128) return gla_typed<128, 128, T>(p, a, ws, P, S_out, z_out, only_if, s);
  return cudaErrorNotSupported;
}

// phi for operands rounded to bf16 next: __expf's error (a few fp32 ulp at
// the inputs' scale) is far below bf16's 2^-8 spacing, and it avoids the
// accurate expf's range reduction (branches and FMAs that held this
// HBM-bound kernel to about 0.8 of its bandwidth)
__device__ __forceinline__ float phi_bf16_operand(float x) { return x > 0.f ? x + 1.f : __expf(x); }

// barrier 1 or 2 (the block's first or second 64-thread half), with
// immediate ids so that only those barriers are reserved
__device__ __forceinline__ void half_sync(int half) {
  if (half == 0)
    asm volatile("bar.sync 1, 64;" ::: "memory");
  else
    asm volatile("bar.sync 2, 64;" ::: "memory");
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// The operands of the gated tensor-core form (D = 128): per 128-token chunk
// and feature d, with the suffix products r_t = a_(t+1) ... a_(last token of
// the chunk),
//   qh_t = phi(q_t) / r_t,   kh_t = phi(k_t) r_t   (bf16),
// and the chunk's gate product a_(first) ... a_(last) (fp32), so that within
// a chunk qh_t . kh_s = sum_d phi(q_t)[d] phi(k_s)[d] prod_(u=s+1..t) a_u[d]
// for s <= t, and the state carried from the previous chunk enters token t
// as qh_t . (gate product) S.  A chunk whose gate product falls below 2^-93
// in some feature (r_t could leave the bf16 range) sets *hard.
// With P > 1 parts per (batch, head) (the part split of the 128-token
// kernel), the block that finishes the last chunk of a part also writes that
// part's gate tables: per chunk c of part q, gsuf[c] = the product of gp over
// the chunks after c in q, and gpart[q] = the product of gp over q.  Each
// block publishes its gp behind a fence and counts itself in done[bh * P + q]
// (zero at launch); the block whose count completes the part reads the
// others' gp from L2.  Nothing waits.
// grid: ceil(B*H*chunks / 2) blocks of 128 threads, two chunks per block
// (64 threads each, synchronised by their own named barrier); thread j of a
// chunk owns features 2j, 2j + 1 and walks the chunk's tokens from the last,
// loading kT tokens before it computes and stores the first of them, so that
// each warp keeps kT rows of reads in flight (eight gave 0.89 of the copy
// bandwidth; wider accesses per thread with fewer warps were slower, and
// blocks of one chunk 3% slower than of two).
__global__ void __launch_bounds__(128)
    gla_tc_prep_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                       const float *__restrict__ a, __nv_bfloat16 *__restrict__ qh,
                       __nv_bfloat16 *__restrict__ kh, float *__restrict__ gp,
                       float *__restrict__ gsuf, float *__restrict__ gpart,
                       unsigned *__restrict__ done, int *__restrict__ hard, int N, int P,
                       long long items) {
  constexpr int kD128 = 128, kC128 = 128, kT = 8;
  const int half = threadIdx.x >> 6;  // chunk of the block, and its barrier
  const long long item = static_cast<long long>(blockIdx.x) * 2 + half;
  if (item >= items) return;  // the second chunk of the last block: whole half
  const int j = threadIdx.x & 63;
  const int nch = (N + kC128 - 1) / kC128;
  const int64_t bh = item / nch;
  const int c = static_cast<int>(item % nch);
  const int c0 = c * kC128, nv = min(kC128, N - c0);
  const int64_t base = (bh * N + c0) * kD128 + 2 * j;
  float r0 = 1.f, r1 = 1.f;
  for (int t0 = nv - 1; t0 >= 0; t0 -= kT) {
    uint32_t wq[kT], wk[kT];
    float2 ga[kT];
#pragma unroll
    for (int u = 0; u < kT; ++u) {
      if (t0 - u < 0) break;
      const int64_t off = base + static_cast<int64_t>(t0 - u) * kD128;
      wq[u] = __ldcs(reinterpret_cast<const unsigned int *>(q + off));
      wk[u] = __ldcs(reinterpret_cast<const unsigned int *>(k + off));
      ga[u] = __ldcs(reinterpret_cast<const float2 *>(a + off));
    }
#pragma unroll
    for (int u = 0; u < kT; ++u) {
      if (t0 - u < 0) break;
      const int64_t off = base + static_cast<int64_t>(t0 - u) * kD128;
      const float q0 = __uint_as_float(wq[u] << 16), q1 = __uint_as_float(wq[u] & 0xffff0000u);
      const float k0 = __uint_as_float(wk[u] << 16), k1 = __uint_as_float(wk[u] & 0xffff0000u);
      // r stays within [2^-93, 1] on every chunk not flagged hard, where the
      // fast divide is within 2 ulp of fp32 before the bf16 rounding
      __stcs(reinterpret_cast<unsigned int *>(qh + off),
             bf16x2_bits(__fdividef(phi_bf16_operand(q0), r0), __fdividef(phi_bf16_operand(q1), r1)));
      __stcs(reinterpret_cast<unsigned int *>(kh + off),
             bf16x2_bits(phi_bf16_operand(k0) * r0, phi_bf16_operand(k1) * r1));
      r0 *= ga[u].x;
      r1 *= ga[u].y;
    }
  }
  *reinterpret_cast<float2 *>(gp + (bh * nch + c) * kD128 + 2 * j) = make_float2(r0, r1);
  if (!(r0 >= 0x1p-93f) || !(r1 >= 0x1p-93f)) *hard = 1;
  if (P <= 1) return;
  // the part of chunk c: the first nch % P parts have one chunk more
  const int base_n = nch / P, rem = nch % P;
  const int part = c < rem * (base_n + 1) ? c / (base_n + 1) : rem + (c - rem * (base_n + 1)) / base_n;
  const int cb = chunk_part_begin(part, P, nch), ce = chunk_part_begin(part + 1, P, nch);
  __shared__ unsigned last[2];
  __threadfence();
  half_sync(half);
  if (j == 0) last[half] = atomicAdd(done + bh * P + part, 1u) == static_cast<unsigned>(ce - cb - 1);
  half_sync(half);
  if (!last[half]) return;
  __threadfence();
  float s0 = 1.f, s1 = 1.f;
  for (int c1 = ce - 1; c1 >= cb; c1 -= kT) {
    float2 g[kT];
#pragma unroll
    for (int u = 0; u < kT; ++u)
      if (c1 - u >= cb) g[u] = __ldcg(reinterpret_cast<const float2 *>(gp + (bh * nch + c1 - u) * kD128 + 2 * j));
#pragma unroll
    for (int u = 0; u < kT; ++u)
      if (c1 - u >= cb) {
        *reinterpret_cast<float2 *>(gsuf + (bh * nch + c1 - u) * kD128 + 2 * j) = make_float2(s0, s1);
        s0 *= g[u].x;
        s1 *= g[u].y;
      }
  }
  *reinterpret_cast<float2 *>(gpart + (bh * P + part) * kD128 + 2 * j) = make_float2(s0, s1);
}

}  // namespace

// Parts per (batch, head): the count that minimises the estimated time, in
// units of one part's output pass over the whole sequence, of
//   waves(P) / P  (output pass)  +  0.25 waves(P - 1) / P  (state pass),
// with waves(n) = ceil(B*H*(Dv/32)*n / (2 CTAs per SM x SMs)), at most one
// part per 64-token chunk.
int gla_parts(int BH, int N, int Dv) {
  if (BH <= 0 || N <= 0) return 1;
  const long long nch = (N + kC - 1) / kC;
  const long long ctas = static_cast<long long>(BH) * (Dv / kDvs);
  const long long slots = 2LL * num_sms_gla();
  auto waves = [&](long long n) { return (ctas * n + slots - 1) / slots; };
  const long long pmax = nch < 64 ? nch : 64;
  long long best = 1;
  double best_t = static_cast<double>(waves(1));
  for (long long P = 2; P <= pmax; ++P) {
    const double t = (static_cast<double>(waves(P)) + 0.25 * static_cast<double>(waves(P - 1))) / P;
    if (t < best_t * 0.98) {
      best_t = t;
      best = P;
    }
  }
  return static_cast<int>(best);
}

size_t gla_workspace_bytes(int BH, int P, int D, int Dv) {
  if (P <= 1) return 0;
  return sizeof(float) * static_cast<size_t>(BH) * (P - 1) *
         (static_cast<size_t>(D) * Dv + 2 * static_cast<size_t>(D));
}

cudaError_t launch_gla_simt(const Problem &p, const float *a, void *ws, int P, float *S_out,
                            float *z_out, cudaStream_t s, const int *only_if) {
  if (P < 1 || (P > 1 && !ws)) return cudaErrorInvalidValue;
  float *w = static_cast<float *>(ws);
  return p.dtype == kF32 ? gla_shape<float>(p, a, w, P, S_out, z_out, only_if, s)
                         : gla_shape<__nv_bfloat16>(p, a, w, P, S_out, z_out, only_if, s);
}

bool gla_tc_supported(const Problem &p) {
  return p.dtype == kBF16 && p.D == 128 && p.Dv == 128 && p.N > 0 &&
         static_cast<long long>(p.B) * p.H >= 8;
}

// the hard flag and the per-(batch, head, part) chunk counts of the prep kernel
static size_t gla_tc_header_bytes(int BH, int P) {
  return (sizeof(int) + sizeof(unsigned) * static_cast<size_t>(BH) * P + 255) & ~static_cast<size_t>(255);
}

size_t gla_tc_workspace_bytes(int BH, int N) {
  const size_t rows = static_cast<size_t>(BH) * N;
  const size_t nch = (static_cast<size_t>(N) + 127) / 128;
  const int P = chunk128_parts(BH, N);
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  // [hard flag, per-part chunk counts][qh][kh][gp][gsuf][gpart][chunk kernel]
  return gla_tc_header_bytes(BH, P) + 2 * up(rows * 128 * 2) + 2 * up(static_cast<size_t>(BH) * nch * 128 * 4) +
         up(static_cast<size_t>(BH) * P * 128 * 4) + up(chunk128_workspace_bytes(BH, P));
}

cudaError_t launch_gla_tc(const Problem &p, const float *a, void *ws, cudaStream_t s,
                          const int **hard_out, float *S_out, float *z_out) {
  if (!gla_tc_supported(p)) return cudaErrorNotSupported;
  const int BH = p.B * p.H;
  const size_t rows = static_cast<size_t>(BH) * p.N;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  uint8_t *w = static_cast<uint8_t *>(ws);
  const int P = chunk128_parts(BH, p.N);
  const size_t hdr = gla_tc_header_bytes(BH, P);
  int *hard = reinterpret_cast<int *>(w);
  unsigned *done = reinterpret_cast<unsigned *>(w + sizeof(int));
  __nv_bfloat16 *qh = reinterpret_cast<__nv_bfloat16 *>(w + hdr);
  __nv_bfloat16 *kh = reinterpret_cast<__nv_bfloat16 *>(w + hdr + up(rows * 128 * 2));
  const int nch = (p.N + 127) / 128;
  const size_t ntab = up(static_cast<size_t>(BH) * nch * 128 * 4);
  float *gp = reinterpret_cast<float *>(w + hdr + 2 * up(rows * 128 * 2));
  float *gsuf = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(gp) + ntab);
  float *gpart = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(gsuf) + ntab);
  void *cws = reinterpret_cast<uint8_t *>(gpart) + up(static_cast<size_t>(BH) * P * 128 * 4);
  cudaError_t e = cudaMemsetAsync(w, 0, sizeof(int) + sizeof(unsigned) * static_cast<size_t>(BH) * P, s);
  if (e != cudaSuccess) return e;
  // two (batch, head, chunk) items per block; the gate tables come from the
  // item that completes each part
  const long long items = static_cast<long long>(BH) * nch;
  gla_tc_prep_kernel<<<(unsigned)((items + 1) / 2), 128, 0, s>>>(
      static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k), a, qh, kh,
      gp, gsuf, gpart, done, hard, p.N, P, items);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  Problem pf = p;
  pf.q = qh;
  pf.k = kh;
  pf.ident = true;
  *hard_out = hard;
  return launch_gated_chunk128(pf, gp, gsuf, gpart, hard, cws, P, s, S_out, z_out);
}

}  // namespace linattn
