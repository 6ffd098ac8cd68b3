// Sequence-parallel linear attention on tcgen05 tensor cores (sm_103a).
//
// Method: the recurrence of "Linear Attention Mechanisms" (dileepadev.github.io),
// "Recurrent Reformulation", S_i = gamma S_(i-1) + phi(k_i) v_i^T,
// z_i = gamma z_(i-1) + phi(k_i), o_i = phi(q_i)^T S_i / (phi(q_i) . z_i + eps),
// with the fixed per-head decay gamma of its "Gating and Selective State
// Updates" (RetNet) on both S and z, and phi = elu + 1.  The non-causal form
// ("The Kernel Trick for Attention") is the same read-out with the sums taken
// once over all tokens and gamma = 1.
//
// Work split.  The tokens of each (batch, head) are cut into P parts of whole
// 64-token chunks so that B*H*P CTAs keep every SM busy even when B*H is
// small; one CTA owns one part with the full D x Dv state.
//
//   phase A  the part's own contribution to the state, summed in tensor
//            memory (M = D, N = Dv + 16, K = tokens; the operand phi(k) times
//            its decay factor is split into two bf16 numbers, so the sum
//            carries about 16 significant bits),
//              A_p = sum_(s in part) gamma^(e_p - s) phi(k_s) [v_s | 1]^T,
//            e_p = the part's last token.
//   causal mode (one kernel): the CTA of part p > 0 runs phase A over part
//            p - 1, publishes A_(p-1) for the later parts, reads A_j, j < p - 1
//            (published by the CTA of part j + 1; a flag per record), and
//            starts from the state before its part,
//              S0 = sum_(j < p) gamma^(c0 - E_j) A_j   (E_j = end of part j);
//            parts are handed out in part-major order by an atomic ticket, so
//            the CTAs it waits for have already started and every wait ends.
//            Part 0 starts from zero.  Then phase C runs the part's chunks.
//            For a chunk at c0 inside a decay window ending at E (windows of
//            W tokens from the part's start, W chosen so gamma^W stays far
//            above the bf16 range limit):
//              qh_t = gamma^(c0+t-E) phi(q_t),  kh_s = gamma^(E-c0-s) phi(k_s)
//              A'   = qh kh^T                 (= gamma^(t-s) phi(q_t).phi(k_s))
//              P    = A' masked to s <= t
//              O    = qh [T | z] + P [V | 1]  (numerators and the normaliser)
//              T   += kh^T [V | 1]
//            where T (fp32, tensor memory) is the state scaled to the window
//            end: T = sum_(s < c0) gamma^(E - s) phi(k_s) [v_s | 1].  Scaling
//            q and k to the same reference point makes O exact without
//            rescaling T per chunk; T is multiplied by gamma^W once per
//            window.  o_t = O[t, :Dv] / (O[t, Dv] + eps).
//   state mode: phase A only, A_p stored for a scan over the parts
//            (part_scan.cu): the final state of a prefill.  (The bf16
//            non-causal form has its own streaming passes, noncausal_tc.cu.)
//
// Every term of the token-by-token recurrence appears once; the regrouping
// changes only the order of summation and the rounding of the MMA operands
// to bf16.
//
// Warp roles (18 warps):
//   0-3   P: A' -> masked bf16 P in shared memory
//   4-7   state: the chain, T from the previous part's state, bf16 copy of
//         [T | z] for the MMA, window rescaling, the part's sum in state mode
//         (thread = row d of T)
//   8-11  output: O -> o rows (divide by the normaliser)
//   12-15 feature map: phi and the decay scale in place on the q, k tiles
//         (in phase A, warps 0-15 share this work)
//   16    TMA producer (q, k, v tiles into a ring of stages)
//   17    TMEM owner and MMA issuer
// Every wait is bounded; a CTA that gives up counts the failure in device
// memory, drains its in-flight copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace linattn {
namespace {

using namespace tc;

constexpr int kC = 64;          // tokens per chunk
constexpr int kThreads = 576;   // 18 warps
constexpr int kSmemMax = 227 * 1024;
constexpr int kBox = 8192;      // one TMA box: 64 rows x 128 bytes (64 bf16)
constexpr float kGammaMin = 0.35f;
constexpr float kLog2Floor = -93.0139f;  // log2(1e-28): smallest factor in a window

constexpr int kWarpS = 4;
constexpr int kWarpO = 8;
constexpr int kWarpPhi = 12;
constexpr int kWarpTma = 16;
constexpr int kWarpMma = 17;

enum Mode : int { kCausal = 0, kState = 1 };
constexpr int kMaxStages = 8;

template <int D, int DV, int MODE>
struct Lay {
  static constexpr bool STATE = MODE == kState;
  static constexpr int KB = D / 64, VB = DV / 64;
  static constexpr int NA = DV + 16;  // columns of [V | 1], [T | z] and O
  // Stage layout by mode:
  //   causal: q boxes | k boxes (and a zero box when D = 64) | v boxes | ones box
  //   state:  k boxes | low bf16 parts of kh | v boxes | ones box (Dv = 128)
  //   apply:  q boxes
  // In state mode the zero box (D = 64) and the ones box (Dv = 64) are one
  // shared copy after the stages, reached through per-stage descriptor
  // offsets, so that more stages fit.  The causal mode's first phase keeps
  // the low parts in the (then unused) q boxes.
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = STATE ? 0 : KB * kBox;
  static constexpr int kOffKlo = STATE ? KB * kBox : kOffQ;
  static constexpr int kOffV = STATE ? 2 * KB * kBox : kOffK + 2 * kBox;
  static constexpr bool kOnesInStage = !(STATE && DV == 64);
  static constexpr int kOffOnes = kOffV + VB * kBox;  // in-stage ones box
  static constexpr int kStageBytes =
      STATE ? kOffOnes + (kOnesInStage ? kBox : 0) : kOffOnes + kBox;
  static constexpr int kSharedBytes = STATE ? ((D == 64 ? kBox : 0) + (DV == 64 ? kBox : 0)) : 0;
  static constexpr int kPBytes = MODE == kCausal ? kC * 128 : 0;
  static constexpr int kSopAtom = D * 64;  // 32 columns of [T | z], 64-byte swizzle
  static constexpr int kSopBytes = STATE ? 0 : (DV / 32 + 1) * kSopAtom;
  static constexpr int kNumBars = 3 * kMaxStages + 12;
  static constexpr int kFixed =
      kSharedBytes + kPBytes + kSopBytes + kNumBars * 8 + 64 + 1024;
  static constexpr int kFit = (kSmemMax - kFixed) / kStageBytes;
  static constexpr int kStages = kFit > kMaxStages ? kMaxStages : kFit;
  static constexpr int kOffShared = kStages * kStageBytes;   // state: zero box, then ones box
  static constexpr int kOffZero = kOffShared;
  static constexpr int kOffSharedOnes = kOffShared + (D == 64 ? kBox : 0);
  static constexpr int kOffP = kOffShared + kSharedBytes;
  static constexpr int kOffSop = kOffP + kPBytes;
  static constexpr int kOffBar = kOffSop + kSopBytes;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 32;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  // tensor memory columns (fp32): A' (M = 64), T (M = 128), O double buffer
  // (M = 64); state mode uses only T, and allocates no more
  // than it uses (two apply CTAs can then share an SM)
  static constexpr uint32_t kColA = 0, kColT = STATE ? 0 : 64, kColO = 64 + NA;
  static constexpr uint32_t kTmemUsed = STATE ? NA : kColO + 2 * NA;
  static constexpr uint32_t kTmemCols = kTmemUsed <= 128 ? 128 : (kTmemUsed <= 256 ? 256 : 512);
  static_assert(kTmemUsed <= 512, "tensor memory");
  static_assert(kStages >= 3, "stages");
  static_assert(kAlloc <= kSmemMax, "shared memory");
  static_assert(kStageBytes % 1024 == 0 && kOffP % 1024 == 0 && kOffSop % 1024 == 0, "align");
};

struct ChunkParams {
  CUtensorMap tmQ, tmK, tmV;
  __nv_bfloat16 *o;
  // per-part records [B*H][rec_parts][D*Dv + D]: state mode writes A_p (S
  // rows, then z); causal mode A_(p-1) column-group-major (float4 of
  // columns 4g..4g+3 of row d at g * D + d, then z)
  float *rec;
  int *ws_flag;    // causal, P > 1: [B*H][P], 1 once A_p is published
  int *ws_ticket;  // causal, P > 1: part-major work counter
  unsigned int *timeouts;
  int BH, H, N, P, rec_parts;
  float eps;
  Gammas lg;  // log2(gamma) per head
  // causal-mode epilogue in place of o = O[:, :Dv] / (O[:, Dv] + eps):
  //   raw:  out_raw [B*H][N][Dv] fp32 = O[t, :Dv] and den_raw [B*H][N] fp32 =
  //         O[t, Dv] (the undivided numerators and normalisers);
  //   grad: grad_out [B*H][N][Dv] bf16 = O[t, :Dv] times phi'(x) elementwise,
  //         x = grad_in (bf16 [B*H][N][Dv]) at the same row, or 1 when
  //         grad_in is null; rev: row N - 1 - t of grad_out and grad_in
  //         (the output of a product over token-reversed operands, stored in
  //         token order).  phi'(x) = 1 for x > 0, e^x otherwise.
  float *out_raw, *den_raw;
  __nv_bfloat16 *grad_out;
  const __nv_bfloat16 *grad_in;
  int rev;
  // causal mode: parts skewed toward the front (the plain forward; the
  // backward's products run equal parts, which measured faster there)
  int skew;
};

// One output half-row (64 columns, starting at column c0) of the causal
// mode's epilogue: o = x / (den + eps) in bf16, or one of the raw and
// gradient forms (ChunkParams).
__device__ __forceinline__ void emit_half(const ChunkParams &p, size_t row, size_t grow, int DV, int c0,
                                          const float *x, float den, float inv) {
  if (p.out_raw) {
    float4 *dst = reinterpret_cast<float4 *>(p.out_raw + row * DV + c0);
#pragma unroll
    for (int q = 0; q < 16; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    if (c0 == 0) p.den_raw[row] = den;
  } else if (p.grad_out) {
    uint4 *dst = reinterpret_cast<uint4 *>(p.grad_out + grow * DV + c0);
    const uint4 *src = p.grad_in ? reinterpret_cast<const uint4 *>(p.grad_in + grow * DV + c0) : nullptr;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float m[8];
      if (src) {
        const uint4 w = __ldg(src + q);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = __uint_as_float(wv[e] << 16), b = __uint_as_float(wv[e] & 0xffff0000u);
          m[2 * e] = a > 0.f ? 1.f : __expf(a);
          m[2 * e + 1] = b > 0.f ? 1.f : __expf(b);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) m[e] = 1.f;
      }
      dst[q] = make_uint4(pack_bf16x2(x[8 * q] * m[0], x[8 * q + 1] * m[1]),
                          pack_bf16x2(x[8 * q + 2] * m[2], x[8 * q + 3] * m[3]),
                          pack_bf16x2(x[8 * q + 4] * m[4], x[8 * q + 5] * m[5]),
                          pack_bf16x2(x[8 * q + 6] * m[6], x[8 * q + 7] * m[7]));
    }
  } else {
    uint4 *dst = reinterpret_cast<uint4 *>(p.o + row * DV + c0);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      dst[q] = make_uint4(pack_bf16x2(x[8 * q + 0] * inv, x[8 * q + 1] * inv),
                          pack_bf16x2(x[8 * q + 2] * inv, x[8 * q + 3] * inv),
                          pack_bf16x2(x[8 * q + 4] * inv, x[8 * q + 5] * inv),
                          pack_bf16x2(x[8 * q + 6] * inv, x[8 * q + 7] * inv));
  }
}

// phi and the row scales in place on NB boxes of 64 rows x 128 bytes.  Thread
// tp (0..127) handles the 16-byte chunks tp + 128 m of every box, which lie in
// rows (tp / 8) + 16 m, m = 0..3.
template <int NB, bool IDENT>
__device__ __forceinline__ void map_boxes(uint8_t *box0, const uint32_t sc[4], int tp) {
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    uint4 x[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) x[m] = reinterpret_cast<const uint4 *>(box0 + b * kBox)[tp + 128 * m];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      x[m].x = feat_scale_bf16x2<IDENT>(x[m].x, sc[m]);
      x[m].y = feat_scale_bf16x2<IDENT>(x[m].y, sc[m]);
      x[m].z = feat_scale_bf16x2<IDENT>(x[m].z, sc[m]);
      x[m].w = feat_scale_bf16x2<IDENT>(x[m].w, sc[m]);
      reinterpret_cast<uint4 *>(box0 + b * kBox)[tp + 128 * m] = x[m];
    }
  }
}

// The same in fp32, leaving each value as the sum of two bf16 numbers: the
// rounded value in place and the rounding error in the matching position of
// lo0, so that an MMA pair over both carries about 16 significant bits.  Here
// 512 threads share the boxes: thread tp handles chunk tp of every box, all
// in row tp / 8, with the row scale sc.
template <int NB, bool IDENT>
__device__ __forceinline__ void map_boxes_split(uint8_t *box0, uint8_t *lo0, float sc, int tp) {
  uint4 x[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) x[b] = reinterpret_cast<const uint4 *>(box0 + b * kBox)[tp];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    {
      uint32_t w[4] = {x[b].x, x[b].y, x[b].z, x[b].w}, hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float a = __uint_as_float(h ? (w[k] & 0xffff0000u) : (w[k] << 16));
          v[h] = (IDENT ? a : __expf(fminf(a, 0.f)) + fmaxf(a, 0.f)) * sc;
        }
        hi[k] = pack_bf16x2(v[0], v[1]);
        const float h0 = __uint_as_float(hi[k] << 16), h1 = __uint_as_float(hi[k] & 0xffff0000u);
        lo[k] = pack_bf16x2(v[0] - h0, v[1] - h1);
      }
      reinterpret_cast<uint4 *>(box0 + b * kBox)[tp] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      reinterpret_cast<uint4 *>(lo0 + b * kBox)[tp] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
}

template <int D, int DV, int MODE, bool DECAY, bool IDENT>
__global__ void __launch_bounds__(kThreads, 1) chunk_tc_kernel(const __grid_constant__ ChunkParams p) {
  using L = Lay<D, DV, MODE>;
  constexpr int S = L::kStages;
  constexpr int NA = L::NA;
  constexpr bool kPhaseC = MODE == kCausal;
  constexpr size_t kRec = static_cast<size_t>(D) * DV + D;
  // identity features without decay: the feature map would multiply by one
  // (rows past the sequence end are already zero from the copy's bounds), so
  // the map warps only pass each stage on
  constexpr bool kMapNeeded = !(IDENT && !DECAY);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
  uint64_t *full = bars, *mapped = bars + kMaxStages, *empty = bars + 2 * kMaxStages;
  uint64_t *A_full = bars + 3 * kMaxStages, *A_free = A_full + 1, *P_full = A_full + 2;
  uint64_t *T_ready = A_full + 3, *T_free = A_full + 4, *S_full = A_full + 5, *S_free = A_full + 6;
  uint64_t *O_full = A_full + 7, *O_free = A_full + 9, *drain = A_full + 11;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffMisc + 4);
  int *item = reinterpret_cast<int *>(sm + L::kOffMisc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.BH, N = p.N, P = p.P;

  // ---- set-up: work item, constant operand blocks, barriers, TMEM ----
  const int prun = static_cast<int>(gridDim.x) / BH;  // parts run per (batch, head)
  if (tid == 0) {
    int t = static_cast<int>(blockIdx.x);
    if (MODE == kCausal && P > 1) t = atomicAdd(p.ws_ticket, 1);
    item[0] = t / BH;  // part (part-major order)
    item[1] = t % BH;  // batch * head
  }
  {
    // ones boxes (column 0 = 1 in each of the 64 rows), zero boxes (the
    // second 64-row atom of kh^T when D = 64), P and [T | z] buffers: zero
    constexpr int kBoxU4 = kBox / 16;
    for (int i = tid; i < S * kBoxU4; i += kThreads) {
      const int st = i / kBoxU4, j = i % kBoxU4;
      uint8_t *stg = sm + st * L::kStageBytes;
      if (L::kOnesInStage) reinterpret_cast<uint4 *>(stg + L::kOffOnes)[j] = make_uint4(0, 0, 0, 0);
      if (D == 64 && MODE == kCausal) reinterpret_cast<uint4 *>(stg + L::kOffK + kBox)[j] = make_uint4(0, 0, 0, 0);
    }
    uint4 *z4 = reinterpret_cast<uint4 *>(sm + L::kOffShared);
    for (int i = tid; i < (L::kSharedBytes + L::kPBytes + L::kSopBytes) / 16; i += kThreads)
      z4[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (L::kOnesInStage && tid < S * kC) {
    const int st = tid / kC, r = tid % kC;
    *reinterpret_cast<__nv_bfloat16 *>(sm + st * L::kStageBytes + L::kOffOnes + sw128_off(r, 0)) =
        __float2bfloat16_rn(1.f);
  }
  if (MODE == kState && DV == 64 && tid < kC)
    *reinterpret_cast<__nv_bfloat16 *>(sm + L::kOffSharedOnes + sw128_off(tid, 0)) =
        __float2bfloat16_rn(1.f);
  if (tid == 32 * kWarpTma) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&mapped[i], 16);
      mbar_init(&empty[i], 1);
    }
    mbar_init(A_full, 1);
    mbar_init(A_free, 4);
    mbar_init(P_full, 4);
    mbar_init(T_ready, 1);
    mbar_init(T_free, 4);
    mbar_init(S_full, 4);
    mbar_init(S_free, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&O_full[b], 1);
      mbar_init(&O_free[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, L::kTmemCols);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int part = item[0], bh = item[1];

  // the part: chunks [cb, cb + nch) of this (batch, head).  Phase A runs
  // over chunks [cbA, cbA + nA): the part itself in state mode, the previous
  // part in causal mode.
  const int nch_all = (N + kC - 1) / kC;
  const int pbase = nch_all / P, prem = nch_all % P;
  // Skewed parts (p.skew, causal mode, parts of 8 chunks or more): boundary
  // q moves q (P - q) / 2 chunks toward the end, so that earlier parts take
  // more chunks (a later part starts phase C later: its look-back waits for
  // more records, and part 0 has no phase A); for P = 4, 64 chunks split 17,
  // 17, 15, 15, about 3% faster than equal parts.  Every part keeps
  // pbase - (P - 1) / 2 >= 1 chunks: the host sets p.skew only then.
  const bool skew = MODE == kCausal && p.skew && pbase >= 8;
  auto part_begin = [&](int q) { return q * pbase + min(q, prem) + (skew ? q * (P - q) / 2 : 0); };
  const int cb = part_begin(part);
  const int nch = part_begin(part + 1) - cb;
  const int len = min(N, (cb + nch) * kC) - cb * kC;
  const bool hasA = MODE == kState || (MODE == kCausal && part > 0);
  const int cbA = MODE == kCausal && part > 0 ? part_begin(part - 1) : cb;
  const int nA = !hasA ? 0 : (MODE == kCausal ? cb - cbA : nch);
  (void)prun;
  const float lg = DECAY ? p.lg.g[bh % p.H] : 0.f;
  int WC = 64;  // chunks per decay window
  if (DECAY && lg < 0.f) {
    const float c = kLog2Floor / lg / 64.f;
    WC = c < 1.f ? 1 : (c > 64.f ? 64 : static_cast<int>(c));
  }
  const int W = kC * WC;

  // phase A feature map, kh_s = gamma^(e_p - s) phi(k_s).  State mode: warps
  // 0-15, thread tp maps row tp / 8 of every k box in fp32, split into bf16
  // high and low parts (low parts to the boxes at kOffKlo).  Causal mode: the
  // four feature-map warps, bf16 (tp = 0..127, rows tp / 8 + 16 m).
  auto phase_a_map = [&](int tp) {
    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nA; ++i) {
      if (!warp_wait(&full[s], ph, abort_flag, p.timeouts)) break;
      const int nv = min(kC, N - (cbA + i) * kC);
      uint8_t *st = sm + s * L::kStageBytes;
      const int e0 = kC * nA - 1 - kC * i;
      if (MODE == kState) {
        const int row = tp >> 3;
        float f = DECAY ? exp2f(static_cast<float>(e0 - row) * lg) : 1.f;
        if (row >= nv) f = 0.f;
        map_boxes_split<L::KB, IDENT>(st + L::kOffK, st + L::kOffKlo, f, tp);
      } else {
        uint32_t sc[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int t = (tp >> 3) + 16 * m;
          float f = DECAY ? exp2f(static_cast<float>(e0 - t) * lg) : 1.f;
          if (t >= nv) f = 0.f;
          sc[m] = pack_bf16x2(f, f);
        }
        if (kMapNeeded) map_boxes<L::KB, IDENT>(st + L::kOffK, sc, tp);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(&mapped[s], MODE == kState ? 1 : 4);
      if (++s == S) {
        s = 0;
        ph ^= 1;
      }
    }
  };

  // Causal mode, before phase C, by the state and output warps (w8 = 0..7:
  // rows 32 (w8 % 4) + lane, columns [Dv/2 (w8 / 4), + Dv/2); w8 >= 4 also
  // z).  The state before the part is S0 = sum_(j < part) gamma^(c0 - E_j)
  // A_j (c0 = the part's first token, E_j = the end of part j, A_j = part
  // j's own sum scaled to E_j).  This CTA's phase A summed A_(part-1) in
  // tensor memory; it is published for the later parts that need it
  // (column-group-major records: float4 of columns 4g..4g+3 of row d at
  // g * D + d, then z; a flag per record, release/acquire at GPU scope).
  // A_j for j < part - 1 was published by the CTA of part j + 1; parts are
  // started in part-major order by an atomic ticket, so every wait ends.
  // T = gamma^W S0 goes to tensor memory and, in bf16, to [T | z].
  auto look_back = [&](int w8, int c) {
    const int qd = w8 & 3, hf = w8 >> 2;
    const int d = 32 * qd + lane;
    const bool act = d < D, zcol = hf == 1;
    const uint32_t tT = tmem_addr(tmem, 32 * qd, L::kColT);
    uint8_t *sop = sm + L::kOffSop;
    constexpr int NG = DV / 64;  // 32-column groups per thread
    const int g0 = hf * NG;
    if (hasA) {
      warp_wait(T_ready, 0, abort_flag, p.timeouts);
      tc_fence_after();
      if (part < P - 1) {  // A_(part-1) is read by the parts after this one
        float *rec = p.rec + (static_cast<size_t>(bh) * P + part - 1) * kRec;
#pragma unroll 1
        for (int g = g0; g < g0 + NG; ++g) {
          float x[32];
          tmem_ld32(tT + 32 * g, x);
          tmem_wait_ld();
          if (act)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg(reinterpret_cast<float4 *>(rec) + (8 * g + q) * D + d,
                     make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
        }
        if (zcol) {
          const float zd = tmem_ld1(tT + DV);
          tmem_wait_ld();
          if (act) __stcg(rec + D * DV + d, zd);
        }
        __threadfence();
      }
    }
    named_sync(1, 256);
    if (hasA && part < P - 1 && c == 0) st_release_gpu(p.ws_flag + bh * P + part - 1, 1);
    if (part >= 2) {
      if (c == 0) {
        const long long t0 = clock64();
        for (int j = 0; j < part - 1 && !*abort_flag; ++j) {
          const int *f = p.ws_flag + bh * P + j;
          while (ld_acquire_gpu(f) == 0) {
            if (*abort_flag) break;
            if (clock64() - t0 > kWaitCycles) {
              *abort_flag = 1;
              atomicAdd(p.timeouts, 1u);
              break;
            }
            __nanosleep(32);
          }
        }
      }
      named_sync(1, 256);
    }
    const float gW = DECAY ? exp2f(static_cast<float>(W) * lg) : 1.f;
#pragma unroll 1
    for (int g = g0; g < g0 + NG; ++g) {
      float acc[32];
      if (hasA) {
        tmem_ld32(tT + 32 * g, acc);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = 0.f;
      }
      for (int j = 0; j < part - 1; ++j) {
        const float wj = DECAY ? exp2f(static_cast<float>((cb - part_begin(j + 1)) * kC) * lg) : 1.f;
        const float *rec = p.rec + (static_cast<size_t>(bh) * P + j) * kRec;
        float4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          v[q] = act ? __ldcg(reinterpret_cast<const float4 *>(rec) + (8 * g + q) * D + d)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          acc[4 * q] = fmaf(wj, v[q].x, acc[4 * q]);
          acc[4 * q + 1] = fmaf(wj, v[q].y, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(wj, v[q].z, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(wj, v[q].w, acc[4 * q + 3]);
        }
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[e] *= gW;
      tmem_st32(tT + 32 * g, acc);
      if (act) put_sop32(sop, L::kSopAtom, g, d, acc);
    }
    if (zcol) {
      float zz[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) zz[e] = 0.f;
      if (hasA) {
        zz[0] = tmem_ld1(tT + DV);
        tmem_wait_ld();
      }
      for (int j = 0; j < part - 1; ++j) {
        const float wj = DECAY ? exp2f(static_cast<float>((cb - part_begin(j + 1)) * kC) * lg) : 1.f;
        const float *rec = p.rec + (static_cast<size_t>(bh) * P + j) * kRec;
        if (act) zz[0] = fmaf(wj, __ldcg(rec + D * DV + d), zz[0]);
      }
      zz[0] *= gW;
      tmem_st16(tT + DV, zz);
      if (act) put_sop16(sop, L::kSopAtom, DV / 32, d, zz);
    }
    tmem_wait_st();
    tc_fence_before();
    fence_async_smem();
    named_sync(1, 256);
  };

  if (warp == kWarpTma) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmK);
      prefetch_tmap(&p.tmV);
      if (kPhaseC) prefetch_tmap(&p.tmQ);
    }
    const int nC = kPhaseC ? nch : 0;
    int s = 0, issued = 0;
    uint32_t ph = 0;
    for (int it = 0; it < nA + nC; ++it) {
      if (!warp_wait(&empty[s], ph ^ 1, abort_flag, p.timeouts)) break;
      if (lane == 0) {
        const bool phaseA = it < nA;
        const int row = (phaseA ? cbA + it : cb + it - nA) * kC;
        const bool wq = !phaseA, wkv = true;
        uint8_t *st = sm + s * L::kStageBytes;
        mbar_arrive_expect_tx(&full[s], (wq ? L::KB * kBox : 0) + (wkv ? (L::KB + L::VB) * kBox : 0));
        if (wq)
#pragma unroll
          for (int kb = 0; kb < L::KB; ++kb)
            tma_load_3d(st + L::kOffQ + kb * kBox, &p.tmQ, kb * 64, row, bh, &full[s]);
        if (wkv) {
#pragma unroll
          for (int kb = 0; kb < L::KB; ++kb)
            tma_load_3d(st + L::kOffK + kb * kBox, &p.tmK, kb * 64, row, bh, &full[s]);
#pragma unroll
          for (int vb = 0; vb < L::VB; ++vb)
            tma_load_3d(st + L::kOffV + vb * kBox, &p.tmV, vb * 64, row, bh, &full[s]);
        }
      }
      __syncwarp();
      issued = it + 1;
      if (++s == S) {
        s = 0;
        ph ^= 1;
      }
    }
    if (*abort_flag && lane == 0) {  // let every issued copy land before the CTA exits
      for (int c = issued > S ? issued - S : 0; c < issued; ++c)
        mbar_wait_drain(&full[c % S], (c / S) & 1);
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer: lane 0 alone ----------------
    // One thread waits and issues: a warp-wide loop paid a vote and a
    // reconvergence around every wait and every issue, which kept the tensor
    // pipe idle most of each chunk (its own MMAs need about 850 cycles of a
    // chunk's 2700 at D = Dv = 64).
    if (lane == 0) {
      constexpr uint32_t ID_A = idesc_bf16(64, 64, false, false);
      constexpr uint32_t ID_DS = idesc_bf16(128, NA, true, true);
      constexpr uint32_t ID_O = idesc_bf16(64, NA, false, true);
      constexpr uint64_t kStageU = L::kStageBytes >> 4;
      const uint32_t base = smem_u32(sm);
      // q, k: K-major (K = d); kh^T: MN-major (M = d, K = tokens); [V | 1]:
      // MN-major (N = value column, K = tokens); P: K-major; [T | z]: MN-major
      // (N = value column, K = d).  Variants differ in the start address only.
      const uint64_t dq0 = smem_desc(base + L::kOffQ, 16, 1024, kSw128);
      const uint64_t dk0 = smem_desc(base + L::kOffK, 16, 1024, kSw128);
      // kh^T (its low parts) and [V | 1]: the second atom (zero box, ones box)
      // is in the stage at the next box, except where it is a shared copy
      const uint64_t dkt0 = smem_desc(base + L::kOffK, kBox, 1024, kSw128);
      const uint64_t dktlo0 = smem_desc(base + L::kOffKlo, (MODE == kCausal && D == 64) ? 2 * kBox : kBox, 1024, kSw128);
      const uint64_t dv0 = smem_desc(base + L::kOffV, kBox, 1024, kSw128);
      // state mode, per stage: start address field as usual, LBO to the shared box
      auto desc_state = [&](int st, int off, bool shared, int shared_off) {
        const uint32_t a = base + st * L::kStageBytes + off;
        return smem_desc(a, shared ? base + shared_off - a : kBox, 1024, kSw128);
      };
      const uint64_t dp0 = smem_desc(base + L::kOffP, 16, 1024, kSw128);
      const uint64_t dsop0 = smem_desc(base + L::kOffSop, L::kSopAtom, 512, kSw64);
      const uint32_t tA = tmem + L::kColA, tT = tmem + L::kColT;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      // phase A: T = kh^T [V | 1] over the part
      for (int i = 0; i < nA; ++i) {
        if (!mbar_wait(&mapped[s], ph, abort_flag, p.timeouts)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>(s) * kStageU;
        if (MODE == kState) {
          const uint64_t dk = desc_state(s, L::kOffK, D == 64, L::kOffZero);
          const uint64_t dl = desc_state(s, L::kOffKlo, D == 64, L::kOffZero);
          const uint64_t dv = desc_state(s, L::kOffV, DV == 64, L::kOffSharedOnes);
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk) {
            mma_bf16(tT, dk + kk * 128, dv + kk * 128, ID_DS, (i > 0 || kk > 0) ? 1u : 0u);
            mma_bf16(tT, dl + kk * 128, dv + kk * 128, ID_DS, 1u);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk)
            mma_bf16(tT, dkt0 + so + kk * 128, dv0 + so + kk * 128, ID_DS, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
      if (ok && hasA) {
        mma_commit(T_ready);
      }
      // phase C.  Iteration i issues chunk i+1's A' first, then chunk i's
      // [dS | dz], inter- and intra-chunk MMAs, so the P warps turn A'_(i+1)
      // into P while the tensor pipe works on chunk i: every wait below has
      // about a chunk of queued work in front of it.  (A' has one buffer: the
      // P warps have read A'_i long before A'_(i+1) is issued.)
      auto issue_a = [&](int j, int st) -> bool {  // A'_j = qh kh^T (M 64 t, N 64 s, K = D)
        if (!mbar_wait(A_free, (j & 1) ^ 1, abort_flag, p.timeouts)) return false;
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>(st) * kStageU;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = so + (kk >> 2) * (kBox >> 4) + (kk & 3) * 2;
          mma_bf16(tA, dq0 + off, dk0 + off, ID_A, kk > 0 ? 1u : 0u);
        }
        mma_commit(A_full);
        return true;
      };
      if (ok && kPhaseC && nch > 0 && MODE == kCausal) {
        if (!mbar_wait(&mapped[s], ph, abort_flag, p.timeouts) || !issue_a(0, s)) ok = false;
      }
      for (int i = 0; ok && kPhaseC && i < nch; ++i) {
        const int b = i & 1;
        const uint32_t u = static_cast<uint32_t>(i >> 1);
        const uint64_t so = static_cast<uint64_t>(s) * kStageU;
        int s1 = s + 1;
        uint32_t ph1 = ph;
        if (s1 == S) {
          s1 = 0;
          ph1 ^= 1;
        }
        if (MODE == kCausal) {
          if (i + 1 < nch) {
            if (!mbar_wait(&mapped[s1], ph1, abort_flag, p.timeouts)) break;
            if (!issue_a(i + 1, s1)) break;
            // T += kh^T [V | 1]: not needed after the last chunk
            if (!mbar_wait(T_free, i & 1, abort_flag, p.timeouts)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kC / 16; ++kk)
              mma_bf16(tT, dkt0 + so + kk * 128, dv0 + so + kk * 128, ID_DS, 1u);
            mma_commit(T_ready);
          }
        }
        // O = qh [T | z]  (M 64, N Dv + 16, K = D)
        if (!mbar_wait(&O_free[b], (u & 1) ^ 1, abort_flag, p.timeouts)) break;
        if (!mbar_wait(S_full, static_cast<uint32_t>(i & 1), abort_flag, p.timeouts)) break;
        tc_fence_after();
        const uint32_t tO = tmem + L::kColO + b * NA;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16(tO, dq0 + so + (kk >> 2) * (kBox >> 4) + (kk & 3) * 2, dsop0 + kk * 64, ID_O,
                   kk > 0 ? 1u : 0u);
        if (MODE == kCausal) mma_commit(S_free);
        if (MODE == kCausal) {
          // O += P [V | 1]  (M 64, N Dv + 16, K 64 tokens)
          if (!mbar_wait(P_full, i & 1, abort_flag, p.timeouts)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk) mma_bf16(tO, dp0 + kk * 2, dv0 + so + kk * 128, ID_O, 1u);
        }
        mma_commit(&O_full[b]);
        mma_commit(&empty[s]);
        s = s1;
        ph = ph1;
      }
      // every MMA issued has completed before TMEM is released
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= kWarpPhi) {
    // ---------------- feature map and decay scales, in place ----------------
    // phase A (warps 0-15, see below) comes first; this loop is phase C
    const int tp = tid - kWarpPhi * 32;
    const int r0 = tp >> 3;
    if (hasA) phase_a_map(MODE == kState ? tid : tp);
    int s = nA % S;
    uint32_t ph = static_cast<uint32_t>((nA / S) & 1);
    for (int i = 0; kPhaseC && i < nch; ++i) {
      if (!warp_wait(&full[s], ph, abort_flag, p.timeouts)) break;
      const int nv = min(kC, N - (cb + i) * kC);
      uint8_t *st = sm + s * L::kStageBytes;
      {
        // kh_s = gamma^(E - s) phi(k_s); rows past the sequence end are zero
        const int e0 = W - 1 - kC * (i % WC);
        uint32_t sc[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int t = r0 + 16 * m;
          float f = DECAY ? exp2f(static_cast<float>(e0 - t) * lg) : 1.f;
          if (t >= nv) f = 0.f;
          sc[m] = pack_bf16x2(f, f);
        }
        if (kMapNeeded) map_boxes<L::KB, IDENT>(st + L::kOffK, sc, tp);
      }
      {
        // qh_t = gamma^(t - E) phi(q_t)
        const int e0 = kC * (i % WC) - (W - 1);
        uint32_t sc[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float f = DECAY ? exp2f(static_cast<float>(e0 + r0 + 16 * m) * lg) : 1.f;
          sc[m] = pack_bf16x2(f, f);
        }
        if (kMapNeeded) map_boxes<L::KB, IDENT>(st + L::kOffQ, sc, tp);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(&mapped[s], 4);
      if (++s == S) {
        s = 0;
        ph ^= 1;
      }
    }
  } else if (warp >= kWarpO) {
    // ---------------- output rows ----------------
    if (MODE == kState) phase_a_map(tid);
    const int w = warp - kWarpO;  // TMEM lane quadrant
    if (MODE == kCausal) look_back(4 + w, 128 + tid - kWarpO * 32);
    const int t = 16 * w + lane;  // M = 64 layout: rows 16w..16w+15 in lanes 0..15
    for (int i = 0; kPhaseC && i < nch; ++i) {
      const int b = i & 1;
      const uint32_t u = static_cast<uint32_t>(i >> 1);
      if (!warp_wait(&O_full[b], u & 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      const uint32_t tO = tmem_addr(tmem, 32 * w, L::kColO + b * NA);
      const int nv = min(kC, N - (cb + i) * kC);
      const bool row_ok = lane < 16 && t < nv;
      // this thread's row of the output (and its place in token order for a
      // product over token-reversed operands)
      const int tok = (cb + i) * kC + t;
      const size_t row = static_cast<size_t>(bh) * N + tok;
      const size_t grow = static_cast<size_t>(bh) * N + (p.rev ? N - 1 - tok : tok);
      float x[64], dz[16];
      tmem_ld16(tO + DV, dz);
      tmem_ld32(tO, x);
      tmem_ld32(tO + 32, x + 32);
      tmem_wait_ld();
      const float inv = 1.f / (dz[0] + p.eps);
      if (DV == 64) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&O_free[b]);
      }
      if (row_ok) emit_half(p, row, grow, DV, 0, x, dz[0], inv);
      if (DV == 128) {
        tmem_ld32(tO + 64, x);
        tmem_ld32(tO + 96, x + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&O_free[b]);
        if (row_ok) emit_half(p, row, grow, DV, 64, x, dz[0], inv);
      }
    }
  } else if (warp >= kWarpS) {
    // ---------------- state: thread d owns row d of T ----------------
    const int w = warp - kWarpS;
    const int d = 32 * w + lane;
    const bool act = d < D;
    const uint32_t tT = tmem_addr(tmem, 32 * w, L::kColT);
    uint8_t *sop = sm + L::kOffSop;
    constexpr int kAtom = L::kSopAtom;
    if (MODE == kState) phase_a_map(tid);
    if (MODE == kState) {
      // A_p = gamma^(e_p - E) T: T is scaled to the chunk-aligned end E of
      // the part; e_p = its last token (they differ only for a ragged end)
      const float corr = DECAY ? exp2f(-static_cast<float>(kC * nch - len) * lg) : 1.f;
      warp_wait(T_ready, 0, abort_flag, p.timeouts);
      tc_fence_after();
      float *aS = p.rec + (static_cast<size_t>(bh) * p.rec_parts + part) * kRec;
#pragma unroll 1
      for (int cc = 0; cc < DV / 32; cc += 2) {
        float x0[32], x1[32];
        tmem_ld32(tT + 32 * cc, x0);
        tmem_ld32(tT + 32 * cc + 32, x1);
        tmem_wait_ld();
        if (act) {
          float4 *dst = reinterpret_cast<float4 *>(aS + d * DV + 32 * cc);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            dst[q] = make_float4(corr * x0[4 * q], corr * x0[4 * q + 1], corr * x0[4 * q + 2], corr * x0[4 * q + 3]);
            dst[8 + q] = make_float4(corr * x1[4 * q], corr * x1[4 * q + 1], corr * x1[4 * q + 2], corr * x1[4 * q + 3]);
          }
        }
      }
      float tz[16];
      tmem_ld16(tT + DV, tz);
      tmem_wait_ld();
      if (act) aS[D * DV + d] = corr * tz[0];
    } else {
      look_back(w, tid - kWarpS * 32);
      const float gW = DECAY ? exp2f(static_cast<float>(W) * lg) : 1.f;
      if (kPhaseC) {
        if (lane == 0) {  // both warp groups are done (look_back ends with a barrier)
          mbar_arrive(T_free);
          mbar_arrive(S_full);
        }
        // per chunk: after T += kh^T [V | 1] of chunk i-1, publish bf16 [T | z]
        // for chunk i (rescaled when chunk i opens a new decay window)
        for (int i = 1; i < nch; ++i) {
          if (!warp_wait(T_ready, static_cast<uint32_t>((i - 1 + (hasA ? 1 : 0)) & 1), abort_flag,
                         p.timeouts))
            break;
          tc_fence_after();
          const bool rebase = DECAY && (i % WC == 0);
          if (!warp_wait(S_free, static_cast<uint32_t>((i - 1) & 1), abort_flag, p.timeouts)) break;
          // two 32-column tiles at a time, or one where the decay rescale is
          // compiled in (two spilled there)
          constexpr int kTiles = DECAY ? 1 : 2;
#pragma unroll 1
          for (int cc = 0; cc < DV / 32; cc += kTiles) {
            float x[kTiles][32];
#pragma unroll
            for (int u = 0; u < kTiles; ++u) tmem_ld32(tT + 32 * (cc + u), x[u]);
            tmem_wait_ld();
            if (rebase) {
#pragma unroll
              for (int u = 0; u < kTiles; ++u) {
#pragma unroll
                for (int e = 0; e < 32; ++e) x[u][e] *= gW;
                tmem_st32(tT + 32 * (cc + u), x[u]);
              }
            }
            if (act)
#pragma unroll
              for (int u = 0; u < kTiles; ++u) put_sop32(sop, kAtom, cc + u, d, x[u]);
          }
          {
            float x0[16];
            tmem_ld16(tT + DV, x0);
            tmem_wait_ld();
            if (rebase) {
#pragma unroll
              for (int e = 0; e < 16; ++e) x0[e] *= gW;
              tmem_st16(tT + DV, x0);
            }
            if (act) put_sop16(sop, kAtom, DV / 32, d, x0);
          }
          if (rebase) tmem_wait_st();
          tc_fence_before();
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(T_free);
            mbar_arrive(S_full);
          }
        }
      }
    }
  } else {
    // ---------------- P = A' masked to s <= t, bf16, 128-byte swizzled ----------------
    if (MODE == kState) phase_a_map(tid);
    const int w = warp;  // TMEM lane quadrant
    const int t = 16 * w + lane;
    for (int i = 0; MODE == kCausal && i < nch; ++i) {
      if (!warp_wait(A_full, i & 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      float a[64];
      tmem_ld32(tmem_addr(tmem, 32 * w, L::kColA), a);
      if (w >= 2) tmem_ld32(tmem_addr(tmem, 32 * w, L::kColA + 32), a + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(A_free);
      // P of the previous chunk has been consumed by its MMA
      if (i > 0 && !warp_wait(&O_full[(i - 1) & 1], static_cast<uint32_t>(((i - 1) >> 1) & 1),
                              abort_flag, p.timeouts))
        break;
      if (lane < 16) {
        uint8_t *prow = sm + L::kOffP;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (8 * j <= t) {  // chunks wholly above the diagonal stay zero
            uint32_t wv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int s0 = 8 * j + 2 * q;
              wv[q] = pack_bf16x2(s0 <= t ? a[s0] : 0.f, s0 + 1 <= t ? a[s0 + 1] : 0.f);
            }
            *reinterpret_cast<uint4 *>(prow + sw128_off(t, 16 * j)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(P_full);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, L::kTmemCols);
}

template <int D, int DV, int MODE, bool DECAY, bool IDENT>
cudaError_t launch_typed(const ChunkParams &prm, int grid, cudaStream_t s) {
  auto kern = chunk_tc_kernel<D, DV, MODE, DECAY, IDENT>;
  const int smem = Lay<D, DV, MODE>::kAlloc;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  kern<<<grid, kThreads, smem, s>>>(prm);
  return cudaGetLastError();
}

template <int MODE, bool DECAY, bool IDENT>
cudaError_t launch_dims(const ChunkParams &prm, int D, int DV, int grid, cudaStream_t s) {
  if (D == 64)
    return DV == 64 ? launch_typed<64, 64, MODE, DECAY, IDENT>(prm, grid, s)
                    : launch_typed<64, 128, MODE, DECAY, IDENT>(prm, grid, s);
  return DV == 64 ? launch_typed<128, 64, MODE, DECAY, IDENT>(prm, grid, s)
                  : launch_typed<128, 128, MODE, DECAY, IDENT>(prm, grid, s);
}

template <int MODE>
cudaError_t launch_mode(const ChunkParams &prm, bool decay, bool ident, int D, int DV, int grid,
                        cudaStream_t s) {
  if (ident)
    return decay ? launch_dims<MODE, true, true>(prm, D, DV, grid, s)
                 : launch_dims<MODE, false, true>(prm, D, DV, grid, s);
  return decay ? launch_dims<MODE, true, false>(prm, D, DV, grid, s)
               : launch_dims<MODE, false, false>(prm, D, DV, grid, s);
}

int num_sms() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!n[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    n[dev] = v;
  }
  return n[dev];
}

bool dims_ok(int D, int Dv) { return (D == 64 || D == 128) && (Dv == 64 || Dv == 128); }

bool setup_params(ChunkParams *prm, const void *q, const void *k, const void *v, int BH, int N,
                  int D, int Dv, int H, const Gammas &g, bool decay) {
  if (q && !make_tmap_3d_bf16(&prm->tmQ, q, D, N, BH, 64, kC, 128)) return false;
  if (!make_tmap_3d_bf16(&prm->tmK, k, D, N, BH, 64, kC, 128)) return false;
  if (!make_tmap_3d_bf16(&prm->tmV, v, Dv, N, BH, 64, kC, 128)) return false;
  if (!q) prm->tmQ = prm->tmK;
  prm->timeouts = wait_timeout_counter();
  if (!prm->timeouts) return false;
  prm->BH = BH;
  prm->H = H;
  prm->N = N;
  prm->lg = log2_gammas(g, H, decay);
  return true;
}

}  // namespace

Gammas log2_gammas(const Gammas &g, int H, bool decay) {
  Gammas lg;
  for (int h = 0; h < kMaxHeads; ++h)
    lg.g[h] = (decay && h < H) ? static_cast<float>(log2(static_cast<double>(g.g[h]))) : 0.f;
  return lg;
}

int chunk_parts(int BH, int N) {
  // A CTA's time is about its phase A (0.3 of its phase C per chunk) plus the
  // chain links before it plus its phase C, and a second wave of CTAs
  // repeats the whole critical path.  So: at most one wave, and no more
  // parts than minimise phase C + chain, P ~ sqrt(nch * 3 / 7) with a chain
  // link worth about 3 chunks of phase C.
  const int nch = (N + kC - 1) / kC;
  if (BH <= 0 || nch <= 0) return 1;
  int P = num_sms() / BH;
  const int pmax = static_cast<int>(sqrt(0.43 * nch));
  if (P > pmax) P = pmax;
  if (P > nch) P = nch;
  return P < 1 ? 1 : P;
}

namespace {
// CTAs of the state-mode kernel that run at once on one SM: its occupancy
// by shared memory and registers, capped by its tensor-memory columns (an
// allocation that does not fit waits for another CTA to free its columns).
template <int D, int DV>
int state_ctas_per_sm() {
  using L = Lay<D, DV, kState>;
  auto kern = chunk_tc_kernel<D, DV, kState, false, false>;
  int occ = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, L::kAlloc) != cudaSuccess)
    occ = 1;
  const int tmem_cap = static_cast<int>(512 / L::kTmemCols);
  occ = occ < tmem_cap ? occ : tmem_cap;
  return occ < 1 ? 1 : occ;
}
}  // namespace

int chunk_state_parts(int BH, int N, int D, int Dv) {
  // state and apply passes: parts are independent (no chain), each CTA's
  // time is proportional to its part's length, and whole waves of CTAs run
  // at once; so P minimises waves(P) / P, waves(P) = ceil(B*H*P / slots),
  // plus a small cost per part (its record and its share of the scan)
  const int nch = (N + kC - 1) / kC;
  if (BH <= 0 || nch <= 0) return 1;
  int per_sm = 1;
  if (D == 64 && Dv == 64) per_sm = state_ctas_per_sm<64, 64>();
  else if (D == 64) per_sm = state_ctas_per_sm<64, 128>();
  else if (Dv == 64) per_sm = state_ctas_per_sm<128, 64>();
  else per_sm = state_ctas_per_sm<128, 128>();
  const long long slots = static_cast<long long>(num_sms()) * per_sm;
  const int pmax = nch < 64 ? nch : 64;
  int best = 1;
  double best_t = 1e30;
  for (int P = 1; P <= pmax; ++P) {
    const long long waves = (static_cast<long long>(BH) * P + slots - 1) / slots;
    const double t = static_cast<double>(waves) / P + 0.002 * P;
    if (t < best_t - 1e-9) {
      best_t = t;
      best = P;
    }
  }
  return best;
}

size_t chunk_workspace_bytes(int BH, int P, int D, int Dv) {
  return sizeof(float) * static_cast<size_t>(BH) * P * (static_cast<size_t>(D) * Dv + D);
}

namespace {
size_t causal_flag_bytes(int BH, int P) {
  const size_t flags = (static_cast<size_t>(BH) * P + 1) * sizeof(int);
  return (flags + 255) & ~static_cast<size_t>(255);
}
}  // namespace

size_t chunk_causal_workspace_bytes(int BH, int P, int D, int Dv) {
  return P <= 1 ? 0 : causal_flag_bytes(BH, P) + chunk_workspace_bytes(BH, P, D, Dv);
}

bool chunk_tc_supported(const Problem &p, const Gammas &g) {
  if (p.dtype != kBF16 || !dims_ok(p.D, p.Dv) || p.N <= 0) return false;
  const long long rows = static_cast<long long>(p.B) * p.H;
  if (rows <= 0 || rows * chunk_parts(static_cast<int>(rows), p.N) >= (1LL << 31)) return false;
  if (p.decay)
    for (int h = 0; h < p.H; ++h)
      if (!(g.g[h] >= kGammaMin)) return false;
  return true;
}

cudaError_t launch_causal_chunk(const Problem &p, const Gammas &g, void *ws, int P, cudaStream_t s) {
  if (!chunk_tc_supported(p, g)) return cudaErrorNotSupported;
  const int BH = p.B * p.H;
  ChunkParams prm = {};
  if (!setup_params(&prm, p.q, p.k, p.v, BH, p.N, p.D, p.Dv, p.H, g, p.decay))
    return cudaErrorNotSupported;
  prm.o = static_cast<__nv_bfloat16 *>(p.o);
  prm.P = P;
  prm.rec_parts = P;
  prm.eps = p.eps;
  // skewed parts only while the last part keeps a chunk: the skew moves its
  // start (P - 1) / 2 chunks later (true of every part count chunk_parts
  // gives; a caller's larger P falls back to equal parts)
  const int nch_all = (p.N + kC - 1) / kC;
  prm.skew = P >= 1 && nch_all / P - (P - 1) / 2 >= 1;
  if (P > 1) {
    if (!ws) return cudaErrorInvalidValue;
    // flags and ticket start at zero; the records need no initialisation
    const size_t fb = causal_flag_bytes(BH, P);
    prm.ws_flag = static_cast<int *>(ws);
    prm.ws_ticket = prm.ws_flag + static_cast<size_t>(BH) * P;
    prm.rec = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + fb);
    cudaError_t e = cudaMemsetAsync(ws, 0, (static_cast<size_t>(BH) * P + 1) * sizeof(int), s);
    if (e != cudaSuccess) return e;
  }
  return launch_mode<kCausal>(prm, p.decay, p.ident, p.D, p.Dv, BH * P, s);
}

cudaError_t launch_causal_chunk_epilogue(const Problem &p, const Gammas &g, void *ws, int P,
                                         cudaStream_t s, const ChunkEpilogue &ep) {
  if (!chunk_tc_supported(p, g) || !(ep.out_raw ? ep.den_raw != nullptr : ep.grad_out != nullptr))
    return cudaErrorNotSupported;
  const int BH = p.B * p.H;
  ChunkParams prm = {};
  if (!setup_params(&prm, p.q, p.k, p.v, BH, p.N, p.D, p.Dv, p.H, g, p.decay))
    return cudaErrorNotSupported;
  prm.out_raw = ep.out_raw;
  prm.den_raw = ep.den_raw;
  prm.grad_out = ep.out_raw ? nullptr : ep.grad_out;
  prm.grad_in = ep.grad_in;
  prm.rev = ep.rev;
  prm.P = P;
  prm.rec_parts = P;
  prm.eps = p.eps;
  if (P > 1) {
    if (!ws) return cudaErrorInvalidValue;
    const size_t fb = causal_flag_bytes(BH, P);
    prm.ws_flag = static_cast<int *>(ws);
    prm.ws_ticket = prm.ws_flag + static_cast<size_t>(BH) * P;
    prm.rec = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + fb);
    cudaError_t e = cudaMemsetAsync(ws, 0, (static_cast<size_t>(BH) * P + 1) * sizeof(int), s);
    if (e != cudaSuccess) return e;
  }
  return launch_mode<kCausal>(prm, p.decay, p.ident, p.D, p.Dv, BH * P, s);
}

cudaError_t launch_prefill_chunk(const void *k, const void *v, float *S, float *z, int B, int H,
                                 int N, int D, int Dv, bool decay, const Gammas &g, void *ws,
                                 int P, cudaStream_t s) {
  const Problem pr{nullptr, k, v, nullptr, B, H, N, D, Dv, decay, 0.f, kBF16};
  if (!chunk_tc_supported(pr, g) || !ws) return cudaErrorNotSupported;
  const int BH = B * H;
  ChunkParams prm = {};
  if (!setup_params(&prm, nullptr, k, v, BH, N, D, Dv, H, g, decay)) return cudaErrorNotSupported;
  prm.P = P;
  prm.rec_parts = P;
  prm.rec = static_cast<float *>(ws);
  cudaError_t e = launch_mode<kState>(prm, decay, false, D, Dv, BH * P, s);
  if (e != cudaSuccess) return e;
  return launch_part_scan(prm.rec, BH, H, P, N, D, Dv, prm.lg, kScanFinal, S, z, s);
}

}  // namespace linattn
