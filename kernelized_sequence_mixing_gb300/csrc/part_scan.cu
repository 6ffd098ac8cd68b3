// Scan over the per-part contributions of the sequence-parallel tensor-core
// kernels (CUDA cores, fp32).
//
// Each (batch, head) is cut into P parts of whole 64-token chunks; the state
// pass leaves A_p = sum_(s in part p) gamma^(e_p - s) phi(k_s) [v_s | 1]^T
// (e_p = the part's last token).  The recurrence of "Linear Attention
// Mechanisms" (dileepadev.github.io), "Recurrent Reformulation", with the
// per-head decay of its "Gating and Selective State Updates", carries over
// whole parts as S_after(p) = gamma^len_p S_after(p-1) + A_p.  One thread per
// element of a (batch, head) record walks the parts in order.
#include "kernels.h"

namespace linattn {
namespace {

// One thread per 4 consecutive elements (records are multiples of 4 floats
// long); the records of up to 8 parts are loaded before they are combined.
__global__ void part_scan_kernel(float *rec, int BH, int H, int P, int N, int D, int Dv,
                                 const __grid_constant__ Gammas lg, int mode, float *S_out,
                                 float *z_out) {
  const long long rec4 = (static_cast<long long>(D) * Dv + D) / 4;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(BH) * rec4) return;
  const int bh = static_cast<int>(idx / rec4);
  const long long e4 = idx % rec4;
  const float l = lg.g[bh % H];
  const int nch = (N + 63) / 64, pbase = nch / P, prem = nch % P;
  float4 *r = reinterpret_cast<float4 *>(rec) + static_cast<size_t>(bh) * P * rec4 + e4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  // parts whose record is read: all but the last when computing start states
  const int nread = mode == kScanStarts ? P - 1 : P;
  for (int p0 = 0; p0 < P; p0 += 8) {
    float4 a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      a[j] = p0 + j < nread ? __ldcg(r + static_cast<size_t>(p0 + j) * rec4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int p = p0 + j;
      if (p >= P) break;
      if (mode == kScanSum) {
        acc.x += a[j].x;
        acc.y += a[j].y;
        acc.z += a[j].z;
        acc.w += a[j].w;
        continue;
      }
      // in place: slot p <- the state before part p
      if (mode == kScanStarts) __stcg(r + static_cast<size_t>(p) * rec4, acc);
      const int cb = p * pbase + min(p, prem), n = pbase + (p < prem ? 1 : 0);
      const int len = min(N, (cb + n) * 64) - cb * 64;
      const float g = exp2f(static_cast<float>(len) * l);
      acc.x = fmaf(g, acc.x, a[j].x);
      acc.y = fmaf(g, acc.y, a[j].y);
      acc.z = fmaf(g, acc.z, a[j].z);
      acc.w = fmaf(g, acc.w, a[j].w);
    }
  }
  if (mode == kScanSum) {
    r[0] = acc;
  } else if (mode == kScanFinal) {
    const float v[4] = {acc.x, acc.y, acc.z, acc.w};
    const long long nS = static_cast<long long>(D) * Dv;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const long long e = 4 * e4 + c;
      if (e < nS)
        S_out[static_cast<size_t>(bh) * nS + e] = v[c];
      else
        z_out[static_cast<size_t>(bh) * D + (e - nS)] = v[c];
    }
  }
}

}  // namespace

cudaError_t launch_part_scan(float *rec, int BH, int H, int P, int N, int D, int Dv,
                             const Gammas &lg, int mode, float *S_out, float *z_out,
                             cudaStream_t s) {
  const long long total = static_cast<long long>(BH) * ((static_cast<long long>(D) * Dv + D) / 4);
  if (total <= 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (blocks >= (1LL << 31)) return cudaErrorNotSupported;
  part_scan_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(rec, BH, H, P, N, D, Dv, lg, mode,
                                                                      S_out, z_out);
  return cudaGetLastError();
}

}  // namespace linattn
