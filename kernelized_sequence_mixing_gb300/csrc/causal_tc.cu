// Causal linear attention on tcgen05 tensor cores (sm_103a).
//
// Method: the causal recurrence of "Linear Attention Mechanisms"
// (dileepadev.github.io), "Recurrent Reformulation", with the fixed decay
// gamma of its "Gating and Selective State Updates" (RetNet) on both S and z,
// evaluated chunkwise.  For a chunk of kC = 64 tokens starting at c0 (local
// indices t, s) and the state (S, z) left by the tokens before it:
//
//   qh_t = gamma^t phi(q_t),  kh_s = gamma^-s phi(k_s)        (bf16 operands)
//   A'   = qh kh^T            -> A'_ts = gamma^(t-s) phi(q_t).phi(k_s)
//   P    = A' masked to s <= t (bf16)
//   [num | den]_intra  = P  [V | 1]
//   [num | den]_inter  = qh [S | z]                       (S, z as bf16)
//   o_t  = (num_intra + gamma num_inter) / (den_intra + gamma den_inter + eps)
//   [dS | dz] = kh^T [V | 1]
//   S <- gamma^64 S + gamma^63 dS,   z <- gamma^64 z + gamma^63 dz  (fp32)
//
// Every term of the token-by-token recurrence appears exactly once; the
// regrouping changes only the order of summation and the rounding of the
// matrix-multiply operands to bf16.  Folding gamma^t and gamma^-s into the
// operands keeps both factors within bf16 range for gamma >= kGammaMin; the
// launcher sends smaller decays to the CUDA-core kernel.
//
// Work split: one CTA per (batch*head, 32-column slice of Dv), so the D x 32
// state slice and its normaliser column live on one SM for the whole
// sequence.  Warp roles (14 warps):
//   0-3   state and P: build P from A' (TMEM -> bf16 smem), then carry the
//         fp32 state in registers (thread = row d) and publish its bf16 copy
//   4-7   output: combine intra/inter accumulators, divide, store bf16 rows
//   8-11  feature map: phi and the decay scales, in place on the TMA tiles
//   12    TMA producer (q, k tiles and the v slice, 4-stage ring)
//   13    TMEM owner and single-thread MMA issuer
// Every wait is bounded; a CTA that gives up counts the failure in device
// memory, drains its in-flight copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace linattn {
namespace {

using namespace tc;

constexpr int kC = 64;       // tokens per chunk
constexpr int kDvs = 32;     // value columns per CTA
constexpr int kNaug = 48;    // kDvs + normaliser column, padded to a multiple of 16
constexpr int kStages = 4;   // TMA ring depth
constexpr int kThreads = 448;
constexpr float kGammaMin = 0.35f;

constexpr int kWarpEpY = 4;
constexpr int kWarpPhi = 8;
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;

// tensor-memory columns (fp32 accumulators)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0;        // 2 x 64   (M = 64 rows: 16 lanes per quadrant)
constexpr uint32_t kColDS = 128;     // 2 x 64   (48 used; M = 128 rows d)
constexpr uint32_t kColInter = 256;  // 2 x 64   (48 used)
constexpr uint32_t kColIntra = 384;  // 2 x 64   (48 used)

template <int D>
struct Layout {
  static constexpr int KB = D / 64;              // 128-byte column blocks of a q/k row
  static constexpr int kBlk = kC * 128;          // one [64 rows][128 B] block
  static constexpr int kQBytes = KB * kBlk;
  static constexpr int kKBytes = 2 * kBlk;       // second block is zero when D = 64
  static constexpr int kVBytes = kC * 64;        // [64 rows][32 bf16], 64-byte swizzle
  static constexpr int kStageBytes = kQBytes + kKBytes + kVBytes;
  static constexpr int kOffOnes = kStages * kStageBytes;  // [64][32] with column 0 = 1
  static constexpr int kOffP = kOffOnes + kVBytes;        // 2 x [64 t][64 s]
  static constexpr int kSBlk = kNaug * 128;               // [48 e][64 d] block
  static constexpr int kSBytes = KB * kSBlk;
  static constexpr int kOffS = kOffP + 2 * kBlk;          // 2 x S buffers
  static constexpr int kOffTab = kOffS + 2 * kSBytes;     // gamma^t, gamma^-s (fp32)
  static constexpr int kNumBars = 3 * kStages + 21;
  static constexpr int kOffBar = kOffTab + 2 * kC * 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kStageBytes % 1024 == 0 && kOffP % 1024 == 0 && kOffS % 1024 == 0, "align");
};

struct TcParams {
  CUtensorMap tmQ, tmK, tmV;
  __nv_bfloat16 *o;
  unsigned int *timeouts;
  int H, N, Dv;
  float eps;
  Gammas gam;
};

// phi(x) = elu(x) + 1 on a pair of bf16 values, times a per-row scale:
// exp(min(x, 0)) + max(x, 0), with exp(y) = 2^(y log2 e) on the packed bf16
// exp2 unit.  log2 e is split into a bf16 head and tail so that the argument
// carries one rounding only.
__device__ __forceinline__ uint32_t phi_scale_bf16x2(uint32_t w, uint32_t scale2) {
  const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&w);
  const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
  const __nv_bfloat162 l2e_hi = __float2bfloat162_rn(1.4453125f);
  const __nv_bfloat162 l2e_lo = __float2bfloat162_rn(1.4426950408889634f - 1.4453125f);
  const __nv_bfloat162 m = __hmin2(x, zero);
  const __nv_bfloat162 a = __hfma2(m, l2e_hi, __hmul2(m, l2e_lo));
  uint32_t au = *reinterpret_cast<const uint32_t *>(&a), eu;
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(eu) : "r"(au));
  const __nv_bfloat162 e = *reinterpret_cast<const __nv_bfloat162 *>(&eu);
  __nv_bfloat162 r = __hadd2(e, __hmax2(x, zero));
  r = __hmul2(r, *reinterpret_cast<const __nv_bfloat162 *>(&scale2));
  return *reinterpret_cast<const uint32_t *>(&r);
}

// In place on a TMA-loaded [64 rows][D] tile (KB blocks of 128-byte swizzled
// rows): phi, then row r scaled by tab[r]; rows >= nv zeroed when `mask_tail`.
template <int D, bool DECAY>
__device__ __forceinline__ void phi_tile(uint8_t *tile, const float *tab, int nv,
                                         bool mask_tail, int tp) {
  constexpr int kChunks = (D / 64) * 512;  // 16-byte chunks
#pragma unroll 4
  for (int j = tp; j < kChunks; j += 128) {
    const int row = (j >> 3) & 63;
    float sc = DECAY ? tab[row] : 1.f;
    if (mask_tail && row >= nv) sc = 0.f;
    const uint32_t s2 = pack_bf16x2(sc, sc);
    uint4 *ptr = reinterpret_cast<uint4 *>(tile) + j;
    uint4 x = *ptr;
    x.x = phi_scale_bf16x2(x.x, s2);
    x.y = phi_scale_bf16x2(x.y, s2);
    x.z = phi_scale_bf16x2(x.z, s2);
    x.w = phi_scale_bf16x2(x.w, s2);
    *ptr = x;
  }
}

template <int D, bool DECAY>
__global__ void __launch_bounds__(kThreads, 1) causal_tc_kernel(const __grid_constant__ TcParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
  uint64_t *full_raw = bars, *full_phi = bars + kStages, *empty = bars + 2 * kStages;
  uint64_t *A_full = bars + 3 * kStages, *A_empty = A_full + 2;
  uint64_t *P_full = A_full + 4, *P_empty = A_full + 6;
  uint64_t *dS_full = A_full + 8, *dS_empty = A_full + 10;
  uint64_t *S_full = A_full + 12, *S_empty = A_full + 14;
  uint64_t *O_full = A_full + 16, *O_empty = A_full + 18;
  uint64_t *drain = A_full + 20;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffMisc + 4);
  float *gq = reinterpret_cast<float *>(sm + L::kOffTab);
  float *gk = gq + kC;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = blockIdx.x * kDvs;
  const int bh = blockIdx.y;
  const int N = p.N;
  const int nchunks = (N + kC - 1) / kC;
  const float gamma = DECAY ? p.gam.g[bh % p.H] : 1.f;

  // ---- set-up: constant operand blocks, decay tables, barriers, TMEM ----
  {
    uint4 *z4 = reinterpret_cast<uint4 *>(sm + L::kOffOnes);
    const int n4 = (L::kOffTab - L::kOffOnes) / 16;  // ones block, P and S buffers
    for (int i = tid; i < n4; i += kThreads) z4[i] = make_uint4(0, 0, 0, 0);
    if (D == 64) {
      for (int s = 0; s < kStages; ++s) {
        uint4 *kz = reinterpret_cast<uint4 *>(sm + s * L::kStageBytes + L::kQBytes + L::kBlk);
        for (int i = tid; i < L::kBlk / 16; i += kThreads) kz[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  __syncthreads();
  if (tid < kC) {  // ones column of the value operand: row tid, column 0
    *reinterpret_cast<__nv_bfloat16 *>(sm + L::kOffOnes + tid * 64 + ((((tid >> 1) & 3)) << 4)) =
        __float2bfloat16_rn(1.f);
  }
  if (tid == 32) {
    double g = 1.0;
    for (int t = 0; t < kC; ++t) {
      gq[t] = static_cast<float>(g);
      gk[t] = static_cast<float>(1.0 / g);
      g *= static_cast<double>(gamma);
    }
  }
  if (tid == 64) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_raw[s], 1);
      mbar_init(&full_phi[s], 4);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&A_full[b], 1);
      mbar_init(&A_empty[b], 4);
      mbar_init(&P_full[b], 4);
      mbar_init(&P_empty[b], 1);
      mbar_init(&dS_full[b], 1);
      mbar_init(&dS_empty[b], 4);
      mbar_init(&S_full[b], 4);
      mbar_init(&S_empty[b], 1);
      mbar_init(&O_full[b], 1);
      mbar_init(&O_empty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, kTmemCols);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmQ);
      prefetch_tmap(&p.tmK);
      prefetch_tmap(&p.tmV);
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        if (!mbar_wait(&empty[s], ((c / kStages) & 1) ^ 1, abort_flag, p.timeouts)) break;
        uint8_t *st = sm + s * L::kStageBytes;
        mbar_arrive_expect_tx(&full_raw[s], 2 * L::kQBytes + L::kVBytes);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
          tma_load_3d(st + kb * L::kBlk, &p.tmQ, kb * 64, c * kC, bh, &full_raw[s]);
          tma_load_3d(st + L::kQBytes + kb * L::kBlk, &p.tmK, kb * 64, c * kC, bh, &full_raw[s]);
        }
        tma_load_3d(st + L::kQBytes + L::kKBytes, &p.tmV, e0, c * kC, bh, &full_raw[s]);
        issued = c + 1;
      }
      if (*abort_flag) {  // let every issued copy land before the CTA exits
        for (int c = issued > kStages ? issued - kStages : 0; c < issued; ++c)
          mbar_wait_drain(&full_raw[c % kStages], (c / kStages) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t ID_A = idesc_bf16(64, 64, false, false);
      constexpr uint32_t ID_DS = idesc_bf16(128, kNaug, true, true);
      constexpr uint32_t ID_INTER = idesc_bf16(64, kNaug, false, false);
      constexpr uint32_t ID_INTRA = idesc_bf16(64, kNaug, false, true);
      const uint32_t base = smem_u32(sm);
      const uint32_t ones = base + L::kOffOnes;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages, b = c & 1;
        const uint32_t ub = static_cast<uint32_t>(c >> 1);
        if (!mbar_wait(&full_phi[s], (c / kStages) & 1, abort_flag, p.timeouts)) break;
        tc_fence_after();
        const uint32_t q0 = base + s * L::kStageBytes;
        const uint32_t k0 = q0 + L::kQBytes;
        const uint32_t v0 = k0 + L::kKBytes;
        // A' = qh kh^T  (M 64 tokens, N 64 tokens, K = D)
        if (!mbar_wait(&A_empty[b], (ub & 1) ^ 1, abort_flag, p.timeouts)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kBlk + (kk & 3) * 32;
          mma_bf16(tmem + kColA + 64 * b, smem_desc(q0 + off, 16, 1024, kSw128),
                   smem_desc(k0 + off, 16, 1024, kSw128), ID_A, kk > 0);
        }
        mma_commit(&A_full[b]);
        // [dS | dz] = kh^T [V | 1]  (M 128 = d, N 48, K 64 tokens)
        if (!mbar_wait(&dS_empty[b], (ub & 1) ^ 1, abort_flag, p.timeouts)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          mma_bf16(tmem + kColDS + 64 * b, smem_desc(k0 + kk * 2048, L::kBlk, 1024, kSw128),
                   smem_desc(v0 + kk * 1024, ones - v0, 512, kSw64), ID_DS, kk > 0);
        }
        mma_commit(&dS_full[b]);
        // inter = qh [S | z] with the state before this chunk
        if (!mbar_wait(&O_empty[b], (ub & 1) ^ 1, abort_flag, p.timeouts)) break;
        tc_fence_after();
        if (c > 0) {
          const int sb = (c - 1) & 1;
          if (!mbar_wait(&S_full[sb], ((c - 1) >> 1) & 1, abort_flag, p.timeouts)) break;
          tc_fence_after();
          const uint32_t s0 = base + L::kOffS + sb * L::kSBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            mma_bf16(tmem + kColInter + 64 * b,
                     smem_desc(q0 + (kk >> 2) * L::kBlk + (kk & 3) * 32, 16, 1024, kSw128),
                     smem_desc(s0 + (kk >> 2) * L::kSBlk + (kk & 3) * 32, 16, 1024, kSw128),
                     ID_INTER, kk > 0);
          }
          mma_commit(&S_empty[sb]);
        }
        // intra = P [V | 1]
        if (!mbar_wait(&P_full[b], ub & 1, abort_flag, p.timeouts)) break;
        tc_fence_after();
        const uint32_t p0 = base + L::kOffP + b * L::kBlk;
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          mma_bf16(tmem + kColIntra + 64 * b, smem_desc(p0 + kk * 32, 16, 1024, kSw128),
                   smem_desc(v0 + kk * 1024, ones - v0, 512, kSw64), ID_INTRA, kk > 0);
        }
        mma_commit(&P_empty[b]);
        mma_commit(&O_full[b]);
        mma_commit(&empty[s]);
      }
      // every MMA issued has completed before TMEM is released
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= kWarpPhi) {
    // ---------------- feature map ----------------
    const int tp = tid - kWarpPhi * 32;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kStages;
      if (!mbar_wait(&full_raw[s], (c / kStages) & 1, abort_flag, p.timeouts)) break;
      const int nv = min(kC, N - c * kC);
      uint8_t *st = sm + s * L::kStageBytes;
      phi_tile<D, DECAY>(st, gq, nv, false, tp);
      phi_tile<D, DECAY>(st + L::kQBytes, gk, nv, true, tp);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_phi[s]);
    }
  } else if (warp >= kWarpEpY) {
    // ---------------- output rows ----------------
    const int w = warp - kWarpEpY;  // TMEM lane quadrant
    const int t = 16 * w + lane;    // M = 64 layout: rows 16w..16w+15 in lanes 0..15
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      const uint32_t ub = static_cast<uint32_t>(c >> 1);
      if (!mbar_wait(&O_full[b], ub & 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      float in[32], it[32];
      tmem_ld32(tmem_addr(tmem, 32 * w, kColIntra + 64 * b), in);
      const float din = tmem_ld1(tmem_addr(tmem, 32 * w, kColIntra + 64 * b + 32));
      float dit = 0.f;
      if (c > 0) {
        tmem_ld32(tmem_addr(tmem, 32 * w, kColInter + 64 * b), it);
        dit = tmem_ld1(tmem_addr(tmem, 32 * w, kColInter + 64 * b + 32));
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) it[e] = 0.f;
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&O_empty[b]);
      const int nv = min(kC, N - c * kC);
      if (lane < 16 && t < nv) {
        const float inv = 1.f / (din + gamma * dit + p.eps);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2((in[2 * i] + gamma * it[2 * i]) * inv,
                              (in[2 * i + 1] + gamma * it[2 * i + 1]) * inv);
        uint4 *dst = reinterpret_cast<uint4 *>(
            p.o + (static_cast<size_t>(bh) * N + c * kC + t) * p.Dv + e0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  } else {
    // ---------------- P construction and state carry ----------------
    const int w = warp;  // TMEM lane quadrant
    const int t = 16 * w + lane;
    const int d = 32 * w + lane;
    float S[32], z = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) S[e] = 0.f;
    double gC = 1.0, gC1 = 1.0;
    for (int i = 0; i < kC; ++i) {
      gC1 = gC;
      gC *= static_cast<double>(gamma);
    }
    const float g64 = static_cast<float>(gC), g63 = static_cast<float>(gC1);
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      const uint32_t ub = static_cast<uint32_t>(c >> 1);
      // P = A' masked to s <= t, as bf16 in the 128-byte swizzled K-major tile
      if (!mbar_wait(&A_full[b], ub & 1, abort_flag, p.timeouts)) break;
      if (!mbar_wait(&P_empty[b], (ub & 1) ^ 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      float a[64];
      tmem_ld32(tmem_addr(tmem, 32 * w, kColA + 64 * b), a);
      if (w >= 2) tmem_ld32(tmem_addr(tmem, 32 * w, kColA + 64 * b + 32), a + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&A_empty[b]);
      if (lane < 16) {
        uint8_t *prow = sm + L::kOffP + b * L::kBlk;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (8 * j <= t) {  // chunks wholly above the diagonal stay zero
            uint32_t wv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int s0 = 8 * j + 2 * q;
              wv[q] = pack_bf16x2(s0 <= t ? a[s0] : 0.f, s0 + 1 <= t ? a[s0 + 1] : 0.f);
            }
            *reinterpret_cast<uint4 *>(prow + sw128_off(t, 16 * j)) =
                make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&P_full[b]);

      // state carry: thread d owns row d of the fp32 state slice
      if (!mbar_wait(&dS_full[b], ub & 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      float ds[32];
      tmem_ld32(tmem_addr(tmem, 32 * w, kColDS + 64 * b), ds);
      const float dz = tmem_ld1(tmem_addr(tmem, 32 * w, kColDS + 64 * b + 32));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dS_empty[b]);
      if (d < D) {
#pragma unroll
        for (int e = 0; e < 32; ++e) S[e] = DECAY ? fmaf(g64, S[e], g63 * ds[e]) : S[e] + ds[e];
        z = DECAY ? fmaf(g64, z, g63 * dz) : z + dz;
      }
      if (!mbar_wait(&S_empty[c & 1], ((c >> 1) & 1) ^ 1, abort_flag, p.timeouts)) break;
      if (d < D) {
        uint8_t *sb = sm + L::kOffS + (c & 1) * L::kSBytes + (d >> 6) * L::kSBlk;
        const int byte = (d & 63) * 2;
#pragma unroll
        for (int e = 0; e < 32; ++e)
          *reinterpret_cast<__nv_bfloat16 *>(sb + sw128_off(e, byte)) = __float2bfloat16_rn(S[e]);
        *reinterpret_cast<__nv_bfloat16 *>(sb + sw128_off(32, byte)) = __float2bfloat16_rn(z);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S_full[c & 1]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

template <int D, bool DECAY>
cudaError_t launch_typed(const TcParams &prm, int slices, int BH, cudaStream_t s) {
  auto kern = causal_tc_kernel<D, DECAY>;
  const int smem = Layout<D>::kAlloc;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  dim3 grid(static_cast<unsigned>(slices), static_cast<unsigned>(BH));
  kern<<<grid, kThreads, smem, s>>>(prm);
  return cudaGetLastError();
}

}  // namespace

bool causal_tc_supported(const Problem &p, const Gammas &g) {
  if (p.dtype != kBF16) return false;
  if ((p.D != 64 && p.D != 128) || (p.Dv != 64 && p.Dv != 128)) return false;
  const long long BH = static_cast<long long>(p.B) * p.H;
  if (BH > 65535 || p.N <= 0) return false;
  if (p.decay)
    for (int h = 0; h < p.H; ++h)
      if (!(g.g[h] >= kGammaMin)) return false;
  return true;
}

cudaError_t launch_causal_tc(const Problem &p, const Gammas &g, cudaStream_t s) {
  if (!causal_tc_supported(p, g)) return cudaErrorNotSupported;
  const int BH = p.B * p.H;
  TcParams prm;
  if (!make_tmap_3d_bf16(&prm.tmQ, p.q, p.D, p.N, BH, 64, kC, 128) ||
      !make_tmap_3d_bf16(&prm.tmK, p.k, p.D, p.N, BH, 64, kC, 128) ||
      !make_tmap_3d_bf16(&prm.tmV, p.v, p.Dv, p.N, BH, kDvs, kC, 64))
    return cudaErrorNotSupported;
  prm.o = static_cast<__nv_bfloat16 *>(p.o);
  prm.timeouts = wait_timeout_counter();
  if (!prm.timeouts) return cudaErrorUnknown;
  prm.H = p.H;
  prm.N = p.N;
  prm.Dv = p.Dv;
  prm.eps = p.eps;
  prm.gam = g;
  const int slices = p.Dv / kDvs;
  if (p.D == 64)
    return p.decay ? launch_typed<64, true>(prm, slices, BH, s)
                   : launch_typed<64, false>(prm, slices, BH, s);
  return p.decay ? launch_typed<128, true>(prm, slices, BH, s)
                 : launch_typed<128, false>(prm, slices, BH, s);
}

}  // namespace linattn
