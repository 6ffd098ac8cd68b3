// Backward of the causal (decayed) form on tcgen05 tensor cores, bf16, for
// Dv = 64.
//
// Method: the chain rule through o_i = n_i / d_i of "Linear Attention
// Mechanisms" (dileepadev.github.io), "Recurrent Reformulation" (the causal
// form trained in its parallel view), with the per-head decay of "Gating and
// Selective State Updates".  With w_ij = gamma^(i-j) phi(q_i).phi(k_j) for
// j <= i, gt_i = dL/do_i / d_i and c_i = gt_i . o_i, dL/dw_ij = gt_i . v_j - c_i
// and
//   dphi(q)_i = sum_(j <= i) gamma^(i-j) (gt_i . v_j - c_i) phi(k)_j
//   dphi(k)_j = sum_(i >= j) gamma^(i-j) (v_j . gt_i - c_i) phi(q)_i
//   dv_j      = sum_(i >= j) gamma^(i-j) (phi(k)_j . phi(q)_i) gt_i
// Each is a decayed causal product y_t = sum_s gamma^|t-s| (a_t . b_s) c_s,
// the form the chunked forward kernel computes without its division:
//   n, d  a = phi(q), b = phi(k), c = [v | 1]          forward (the forward)
//   dq    a = [gt | c], b = [v | -1], c = phi(k)       forward
//   dk    a = [v | -1], b = [gt | c], c = phi(q)       reversed
//   dv    a = phi(k), b = phi(q), c = gt               reversed (phi applied by the
//                                                      product itself, on raw
//                                                      reversed q and k)
// The scalar c_i rides in one more column of the augmented operands (width
// Dv + 1, padded with zeros to 128), so dL/dw_ij is the plain dot product
// of two rows and no separate scan of the decayed sums is needed.  A
// reversed product (s >= t) is the forward product over token-reversed
// operands; the prep kernel writes those operands in reversed order, and the
// product's epilogue writes its rows back in token order, multiplied by
// phi'(x) = 1 (x > 0), e^x (x <= 0) for dq and dk.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace linattn {
namespace {

using tc::pack_bf16x2;

constexpr int kDv = 64;   // value width of this path
constexpr int kAug = 128; // width of the augmented operands [gt | c | 0], [v | -1 | 0]

__device__ __forceinline__ float phi_f(float x) { return x > 0.f ? x + 1.f : __expf(x); }

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// One warp per row (token t of unit u): from the forward's undivided n and
// d - eps, o = n / d, gt = dL/do / d and c = gt . o, then the operands of the
// three gradient products, forward (row t) or token-reversed (row N - 1 - t
// of the same unit).  Lane l holds columns 2l, 2l + 1 of the Dv-wide rows.
// The dv product takes raw reversed q and k and maps them itself, so that
// phi and the decay scale round once, as in the forward.
template <int D>
__global__ void __launch_bounds__(256) bwd_tc_prep_kernel(
    const float *__restrict__ n, const float *__restrict__ den, const __nv_bfloat16 *__restrict__ dO,
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *__restrict__ A1, __nv_bfloat16 *__restrict__ B1,
    __nv_bfloat16 *__restrict__ C1, __nv_bfloat16 *__restrict__ A1r, __nv_bfloat16 *__restrict__ B1r,
    __nv_bfloat16 *__restrict__ Q2r, __nv_bfloat16 *__restrict__ G3r, __nv_bfloat16 *__restrict__ Kr,
    __nv_bfloat16 *__restrict__ Qr, int N, long long rows, float eps) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const long long u = row / N, t = row % N;
  const long long rrow = u * N + (N - 1 - t);
  const int e = 2 * lane;
  const float d = __ldg(den + row) + eps;
  const float2 n2 = __ldg(reinterpret_cast<const float2 *>(n + row * kDv + e));
  const uint32_t dow = __ldg(reinterpret_cast<const uint32_t *>(dO + row * kDv + e));
  const uint32_t vw = __ldg(reinterpret_cast<const uint32_t *>(v + row * kDv + e));
  const float2 do2 = bf16x2_to_f2(dow);
  const float inv = 1.f / d;
  const float g0 = do2.x * inv, g1 = do2.y * inv;
  float c = g0 * (n2.x * inv) + g1 * (n2.y * inv);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
  const uint32_t gb = pack_bf16x2(g0, g1);
  // [gt | c | 0] and [v | -1 | 0]: columns 2l, 2l + 1, then 64 + 2l, 65 + 2l
  const uint32_t ahi = lane == 0 ? pack_bf16x2(c, 0.f) : 0u;
  const uint32_t bhi = lane == 0 ? pack_bf16x2(-1.f, 0.f) : 0u;
  uint32_t *a1 = reinterpret_cast<uint32_t *>(A1 + row * kAug), *a1r = reinterpret_cast<uint32_t *>(A1r + rrow * kAug);
  uint32_t *b1 = reinterpret_cast<uint32_t *>(B1 + row * kAug), *b1r = reinterpret_cast<uint32_t *>(B1r + rrow * kAug);
  a1[lane] = gb;
  a1[32 + lane] = ahi;
  a1r[lane] = gb;
  a1r[32 + lane] = ahi;
  b1[lane] = vw;
  b1[32 + lane] = bhi;
  b1r[lane] = vw;
  b1r[32 + lane] = bhi;
  reinterpret_cast<uint32_t *>(G3r + rrow * kDv)[lane] = gb;
  // phi(k) (forward), phi(q) (reversed), raw k and q (reversed), D wide
#pragma unroll
  for (int j = 0; j < D / 64; ++j) {
    const long long c0 = 64 * j + e;
    const uint32_t kw = __ldg(reinterpret_cast<const uint32_t *>(k + row * D + c0));
    const uint32_t qw = __ldg(reinterpret_cast<const uint32_t *>(q + row * D + c0));
    const float2 k2 = bf16x2_to_f2(kw), q2 = bf16x2_to_f2(qw);
    *reinterpret_cast<uint32_t *>(C1 + row * D + c0) = pack_bf16x2(phi_f(k2.x), phi_f(k2.y));
    *reinterpret_cast<uint32_t *>(Q2r + rrow * D + c0) = pack_bf16x2(phi_f(q2.x), phi_f(q2.y));
    *reinterpret_cast<uint32_t *>(Kr + rrow * D + c0) = kw;
    *reinterpret_cast<uint32_t *>(Qr + rrow * D + c0) = qw;
  }
}

struct TcLayout {
  size_t n, den, A1, B1, A1r, B1r, C1, Q2r, G3r, Kr, Qr, chunk, total;
};

TcLayout tc_layout(int BH, int N, int D) {
  const size_t rows = static_cast<size_t>(BH) * N;
  const int P = chunk_parts(BH, N);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return o;
  };
  TcLayout L;
  L.n = take(rows * kDv * 4);
  L.den = take(rows * 4);
  L.A1 = take(rows * kAug * 2);
  L.B1 = take(rows * kAug * 2);
  L.A1r = take(rows * kAug * 2);
  L.B1r = take(rows * kAug * 2);
  L.C1 = take(rows * D * 2);
  L.Q2r = take(rows * D * 2);
  L.G3r = take(rows * kDv * 2);
  L.Kr = take(rows * D * 2);
  L.Qr = take(rows * D * 2);
  // the chunk kernel's flags and records, shared by the four products (they
  // run one after another on the stream); sized for the widest of them
  L.chunk = take(chunk_causal_workspace_bytes(BH, P, kAug, 128));
  L.total = off;
  return L;
}

}  // namespace

bool backward_tc_supported(const Problem &p, const Gammas &g) {
  if (p.dtype != kBF16 || p.Dv != kDv || (p.D != 64 && p.D != 128) || p.N <= 0 || p.ident) return false;
  // the four products run on the 64-token chunk kernel: its decay envelope
  Problem fwd = p;
  return chunk_tc_supported(fwd, g);
}

size_t backward_tc_workspace_bytes(int BH, int N, int D) { return tc_layout(BH, N, D).total; }

int backward_tc_launches() { return 5; }  // four chunk-kernel products and the prep kernel

cudaError_t launch_backward_tc(const Problem &p, const void *dO, void *dq, void *dk, void *dv,
                               const Gammas &g, void *ws, cudaStream_t s) {
  if (!backward_tc_supported(p, g) || !ws) return cudaErrorNotSupported;
  const int BH = p.B * p.H, N = p.N, D = p.D;
  const long long rows = static_cast<long long>(BH) * N;
  const TcLayout L = tc_layout(BH, N, D);
  uint8_t *w = static_cast<uint8_t *>(ws);
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16 *>(w + off); };
  float *n = reinterpret_cast<float *>(w + L.n), *den = reinterpret_cast<float *>(w + L.den);
  void *cws = w + L.chunk;
  const int P = chunk_parts(BH, N);
  // n, d - eps: the forward product without its division
  ChunkEpilogue ep0{n, den, nullptr, nullptr, 0};
  Problem p0 = p;
  p0.o = nullptr;
  cudaError_t e = launch_causal_chunk_epilogue(p0, g, cws, P, s, ep0);
  if (e != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  auto prep = D == 64 ? bwd_tc_prep_kernel<64> : bwd_tc_prep_kernel<128>;
  prep<<<blocks, 256, 0, s>>>(n, den, static_cast<const __nv_bfloat16 *>(dO),
                              static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k),
                              static_cast<const __nv_bfloat16 *>(p.v), bf(L.A1), bf(L.B1), bf(L.C1), bf(L.A1r),
                              bf(L.B1r), bf(L.Q2r), bf(L.G3r), bf(L.Kr), bf(L.Qr), N, rows, p.eps);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the three gradient products: dq and dk on operands already mapped
  // (identity feature map), dv on raw q and k (phi = elu + 1 in the kernel)
  auto product = [&](const void *a, const void *b, const void *c, int Da, int Dc, void *out,
                     const void *x, int rev, bool ident = true) {
    Problem pp{a, b, c, nullptr, p.B, p.H, N, Da, Dc, p.decay, 0.f, kBF16};
    pp.ident = ident;
    ChunkEpilogue ep{nullptr, nullptr, static_cast<__nv_bfloat16 *>(out),
                     static_cast<const __nv_bfloat16 *>(x), rev};
    return launch_causal_chunk_epilogue(pp, g, cws, P, s, ep);
  };
  if ((e = product(bf(L.A1), bf(L.B1), bf(L.C1), kAug, D, dq, p.q, 0)) != cudaSuccess) return e;
  if ((e = product(bf(L.B1r), bf(L.A1r), bf(L.Q2r), kAug, D, dk, p.k, 1)) != cudaSuccess) return e;
  return product(bf(L.Kr), bf(L.Qr), bf(L.G3r), D, kDv, dv, nullptr, 1, false);
}

}  // namespace linattn
