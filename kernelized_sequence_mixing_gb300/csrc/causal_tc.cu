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
// sequence.  The Dv/32 CTAs of one (batch, head) form a thread-block cluster
// and share the feature-map work: CTA r loads only rows
// [r*64/NS, (r+1)*64/NS) of each q and k chunk (plus its own v slice) into a
// small private ring, maps them, and pushes the mapped rows into every peer's
// operand stage with one bulk DSMEM copy per peer, so each q/k element is read
// from L2 and mapped once per cluster.  The operand stage interleaves the
// 128-byte blocks of q and k per 8-row group, which makes a CTA's rows one
// contiguous region.  A stage is refilled only when every CTA of the cluster
// has released it (multicast MMA commits); the private ring decouples the
// HBM latency from that release.  Warp roles (18 warps):
//   0-3   P: build P from A' (TMEM -> bf16 smem, masked)
//   4-7   state: carry the fp32 state slice in registers (thread = row d)
//         and publish its bf16 copy for the next chunk's inter-chunk MMA
//   8-11  output: combine intra/inter accumulators, divide, store bf16 rows
//   12-15 feature map: phi and the decay scales on this CTA's rows, copy of
//         the v slice, push to the peers
//   16    TMA producer of this CTA's q, k rows (private ring)
//   17    TMEM owner and MMA issuer
//   18    TMA producer of the v slice (its own ring)
// The single-issuer roles (16-18) run their loops warp-wide, waits included,
// and let lane 0 issue each copy, MMA or commit, so their warps never diverge
// for longer than one issue block.
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
constexpr int kVSlots = 4;   // v-slice ring depth
constexpr int kThreads = 608;
constexpr float kGammaMin = 0.35f;
constexpr int kSmemMax = 227 * 1024;

constexpr int kWarpS = 4;
constexpr int kWarpO = 8;
constexpr int kWarpPhi = 12;
constexpr int kWarpTma = 16;   // own q/k rows
constexpr int kWarpMma = 17;
constexpr int kWarpTmaV = 18;  // v slices

// tensor-memory columns (fp32 accumulators)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0;        // 2 x 64   (M = 64 rows: 16 lanes per quadrant)
constexpr uint32_t kColDS = 128;     // 2 x 64   (48 used; M = 128 rows d)
constexpr uint32_t kColInter = 256;  // 2 x 64   (48 used)
constexpr uint32_t kColIntra = 384;  // 2 x 64   (48 used)

template <int D, int NS>
struct Layout {
  static constexpr int KB = D / 64;              // 128-byte column blocks of a q/k row
  static constexpr int R = kC / NS;              // q/k rows loaded and mapped per CTA
  // q/k operand stage: for each 8-row group g, NB consecutive 1 KB blocks
  // [q block 0..KB-1 | k block 0..KB-1 | zero block when D = 64]
  static constexpr int NB = D == 128 ? 4 : 3;
  static constexpr int kGroup = NB * 1024;       // stride of 8-row groups (SBO)
  static constexpr int kStageBytes = 8 * kGroup;
  static constexpr int kOwnOff = (R / 8) * kGroup;   // offset of rank r's rows: r * kOwnOff
  static constexpr int kOwnBytes = (R / 8) * kGroup; // pushed to each peer
  static constexpr int kPeerBytes = (NS - 1) * kOwnBytes;
  static constexpr int kVBytes = kC * 64;        // v slice [64 rows][32 bf16], 64-byte swizzle
  // private ring slot: own q rows, own k rows (KB blocks of [R][128 B])
  static constexpr int kRawQK = KB * R * 128;
  static constexpr int kRawBytes = 2 * kRawQK;
  static constexpr int kSBlk = D * 64;                    // [D rows d][32 e], 64-byte swizzle
  static constexpr int kSBytes = 2 * kSBlk;               // S block + normaliser block
  static constexpr int kFixed = kVSlots * kVBytes + kVBytes + 2 * kC * 128 + 2 * kSBytes +
                                2 * kC * 4 + 64 * 8 + 16 + 1024;
  // q/k stages: 4 if two or more private slots still fit, else 3
  static constexpr int kStages =
      (kSmemMax - kFixed - 4 * kStageBytes) / kRawBytes >= 2 ? 4 : 3;
  static constexpr int kRawFit = (kSmemMax - kFixed - kStages * kStageBytes) / kRawBytes;
  static constexpr int kRaw = kRawFit >= 4 ? 4 : kRawFit;
  static constexpr int kOffV = kStages * kStageBytes;
  static constexpr int kOffRaw = kOffV + kVSlots * kVBytes;
  static constexpr int kOffOnes = kOffRaw + kRaw * kRawBytes;  // [64][32] with column 0 = 1
  static constexpr int kOffP = kOffOnes + kVBytes;             // 2 x [64 t][64 s]
  static constexpr int kOffS = kOffP + 2 * kC * 128;           // 2 x S buffers
  static constexpr int kOffTab = kOffS + 2 * kSBytes;          // gamma^t, gamma^-s (fp32)
  static constexpr int kOffBar = kOffTab + 2 * kC * 4;
  static constexpr int kNumBars = 7 * 4 + 21;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kRaw >= 2, "shared memory");
  static_assert(kAlloc <= kSmemMax, "shared memory");
  static_assert(kStageBytes % 1024 == 0 && kRawBytes % 1024 == 0 && kOffRaw % 1024 == 0 &&
                    kOffP % 1024 == 0 && kOffS % 1024 == 0 && kOffOnes % 1024 == 0,
                "align");
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

// Maps this CTA's rows of one chunk from the private ring slot into the
// q/k operand stage: phi, the row scale (gamma^t for q, gamma^-s for k; k rows
// at or past nv are zeroed), then placed in the interleaved group layout.  The
// 128-byte swizzle pattern depends on row % 8 only, and the own rows start on
// an 8-row boundary, so 16-byte chunks move without re-swizzling.
template <int D, int NS, bool DECAY>
__device__ __forceinline__ void map_rows(const uint8_t *raw, uint8_t *stage, int row0,
                                         const float *gq, const float *gk, int nv, int tp) {
  using L = Layout<D, NS>;
  constexpr int kPerBlk = L::R * 8;              // 16-byte chunks of our rows in one block
  constexpr int kQK = 2 * L::KB * kPerBlk;       // q and k chunks
  constexpr int kIter = (kQK + 127) / 128;
  uint4 x[kIter];
  uint32_t s2[kIter];
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int j = tp + 128 * i;
    if (j < kQK) {
      x[i] = reinterpret_cast<const uint4 *>(raw)[j];
      const bool is_k = j >= L::KB * kPerBlk;
      const int row = row0 + ((j % kPerBlk) >> 3);
      float sc = DECAY ? (is_k ? gk[row] : gq[row]) : 1.f;
      if (is_k && row >= nv) sc = 0.f;
      s2[i] = pack_bf16x2(sc, sc);
    }
  }
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int j = tp + 128 * i;
    if (j < kQK) {
      x[i].x = phi_scale_bf16x2(x[i].x, s2[i]);
      x[i].y = phi_scale_bf16x2(x[i].y, s2[i]);
      x[i].z = phi_scale_bf16x2(x[i].z, s2[i]);
      x[i].w = phi_scale_bf16x2(x[i].w, s2[i]);
      // raw chunk j: block bb (q blocks then k blocks), own row rr, chunk cc
      const int bb = j / kPerBlk, jj = j % kPerBlk;
      const int row = row0 + (jj >> 3), cc = jj & 7;
      uint8_t *dst = stage + (row >> 3) * L::kGroup + bb * 1024 + (row & 7) * 128 + cc * 16;
      *reinterpret_cast<uint4 *>(dst) = x[i];
    }
  }
}

template <int D, int NS, bool DECAY>
__global__ void __launch_bounds__(kThreads, 1) causal_tc_kernel(const __grid_constant__ TcParams p) {
  using L = Layout<D, NS>;
  constexpr int RAW = L::kRaw;
  constexpr int QKS = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
  uint64_t *raw_full = bars, *raw_empty = bars + 4;
  uint64_t *v_full = bars + 8, *v_empty = bars + 12;
  uint64_t *qk_full = bars + 16, *qk_empty = bars + 20;
  uint64_t *mapped = bars + 24;  // the four feature-map warps finished a stage
  uint64_t *A_full = bars + 28, *A_empty = A_full + 2;
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
  const uint32_t rank = cluster_ctarank();
  const int row0 = static_cast<int>(rank) * L::R;  // this CTA's q/k rows in a chunk
  const int N = p.N;
  const int nchunks = (N + kC - 1) / kC;
  const float gamma = DECAY ? p.gam.g[bh % p.H] : 1.f;

  // ---- set-up: constant operand blocks, decay tables, barriers, TMEM ----
  {
    uint4 *z4 = reinterpret_cast<uint4 *>(sm + L::kOffOnes);
    const int n4 = (L::kOffTab - L::kOffOnes) / 16;  // ones block, P and S buffers
    for (int i = tid; i < n4; i += kThreads) z4[i] = make_uint4(0, 0, 0, 0);
    if (D == 64) {  // zero block of every group (rows d >= 64 of the k^T operand)
      for (int i = tid; i < QKS * 8 * 64; i += kThreads) {
        const int st = i / 512, g = (i / 64) % 8, c16 = i % 64;
        reinterpret_cast<uint4 *>(sm + st * L::kStageBytes + g * L::kGroup + 2 * 1024)[c16] =
            make_uint4(0, 0, 0, 0);
      }
    }
  }
  __syncthreads();
  if (tid < kC) {  // ones column of the value operand: row tid, column 0
    *reinterpret_cast<__nv_bfloat16 *>(sm + L::kOffOnes + sw64_off(tid, 0)) =
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
    for (int r = 0; r < 4; ++r) {
      mbar_init(&raw_full[r], 1);
      mbar_init(&raw_empty[r], 1);
      mbar_init(&v_full[r], 1);
      mbar_init(&v_empty[r], 1);
      mbar_init(&qk_full[r], 1);
      mbar_init(&qk_empty[r], NS);
      mbar_init(&mapped[r], 4);
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
  cluster_sync();  // peers' barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ---------------- TMA producer: own q/k rows ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmQ);
      prefetch_tmap(&p.tmK);
    }
    int issued = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int r = c % RAW;
      if (!warp_wait(&raw_empty[r], ((c / RAW) & 1) ^ 1, abort_flag, p.timeouts)) break;
      if (lane == 0) {
        uint8_t *slot = sm + L::kOffRaw + r * L::kRawBytes;
        mbar_arrive_expect_tx(&raw_full[r], L::kRawBytes);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb) {
          tma_load_3d(slot + kb * L::R * 128, &p.tmQ, kb * 64, c * kC + row0, bh, &raw_full[r]);
          tma_load_3d(slot + L::kRawQK + kb * L::R * 128, &p.tmK, kb * 64, c * kC + row0, bh,
                      &raw_full[r]);
        }
      }
      __syncwarp();
      issued = c + 1;
    }
    if (*abort_flag && lane == 0) {  // let every issued copy land before the CTA exits
      for (int c = issued > RAW ? issued - RAW : 0; c < issued; ++c)
        mbar_wait_drain(&raw_full[c % RAW], (c / RAW) & 1);
    }
  } else if (warp == kWarpTmaV) {
    // ---------------- TMA producer: v slice ----------------
    if (lane == 0) prefetch_tmap(&p.tmV);
    int issued = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int r = c % kVSlots;
      if (!warp_wait(&v_empty[r], ((c / kVSlots) & 1) ^ 1, abort_flag, p.timeouts)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&v_full[r], L::kVBytes);
        tma_load_3d(sm + L::kOffV + r * L::kVBytes, &p.tmV, e0, c * kC, bh, &v_full[r]);
      }
      __syncwarp();
      issued = c + 1;
    }
    if (*abort_flag && lane == 0) {
      for (int c = issued > kVSlots ? issued - kVSlots : 0; c < issued; ++c)
        mbar_wait_drain(&v_full[c % kVSlots], (c / kVSlots) & 1);
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer (warp-wide loop, lane 0 issues) ----------------
    {
      const bool leader = lane == 0;
      constexpr uint32_t ID_A = idesc_bf16(64, 64, false, false);
      constexpr uint32_t ID_DS = idesc_bf16(128, kNaug, true, true);
      constexpr uint32_t ID_O = idesc_bf16(64, kNaug, false, true);
      constexpr uint16_t kAll = static_cast<uint16_t>((1u << NS) - 1);
      // Every descriptor is built once; per-stage, per-buffer and per-k-step
      // variants differ only in the start-address field (bits 0-13, in
      // 16-byte units), so they are formed by adding constants.  All shared
      // addresses are below 256 KB, so the additions never carry out of it.
      const uint32_t base = smem_u32(sm);
      const uint32_t ones = base + L::kOffOnes;
      constexpr uint64_t kStageU = L::kStageBytes >> 4;
      constexpr uint64_t kVU = L::kVBytes >> 4;
      const uint64_t dq0 = smem_desc(base, 16, L::kGroup, kSw128);                  // q, K-major
      const uint64_t dk0 = smem_desc(base + L::KB * 1024, 16, L::kGroup, kSw128);  // k, K-major
      const uint64_t dkt0 = smem_desc(base + L::KB * 1024, 1024, L::kGroup, kSw128);  // k^T, MN
      const uint64_t dv0 = smem_desc(base + L::kOffV, ones - (base + L::kOffV), 512, kSw64);
      const uint64_t dp0 = smem_desc(base + L::kOffP, 16, 1024, kSw128);
      const uint64_t ds0 = smem_desc(base + L::kOffS, L::kSBlk, 512, kSw64);
      auto stage_add = [](uint64_t d, int s) { return d + static_cast<uint64_t>(s) * kStageU; };
      // v slot r: start + r*kV; its LBO (distance to the ones block) shrinks alike
      auto v_desc = [&](int r) {
        const uint64_t o = static_cast<uint64_t>(r) * kVU;
        return dv0 + o - (o << 16);
      };
      // Chunk c+1's A' and [dS | dz] depend only on its own tiles, so they are
      // issued before chunk c's intra-chunk MMA waits for P: the tensor pipe
      // keeps working while the P warps turn A'_c into P_c.
      auto issue_independent = [&](int c) -> bool {
        const int s = c % QKS, b = c & 1, vr = c % kVSlots;
        const uint32_t ub = static_cast<uint32_t>(c >> 1);
        if (!warp_wait(&qk_full[s], (c / QKS) & 1, abort_flag, p.timeouts)) return false;
        const uint64_t dq = stage_add(dq0, s), dk = stage_add(dk0, s), dkt = stage_add(dkt0, s);
        if (!warp_wait(&A_empty[b], (ub & 1) ^ 1, abort_flag, p.timeouts)) return false;
        tc_fence_after();
        // A' = qh kh^T  (M 64 tokens, N 64 tokens, K = D)
        const uint32_t ta = tmem + kColA + 64 * b;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = (kk >> 2) * 64 + (kk & 3) * 2;
            mma_bf16(ta, dq + off, dk + off, ID_A, kk > 0);
          }
          mma_commit(&A_full[b]);
        }
        __syncwarp();
        // [dS | dz] = kh^T [V | 1]  (M 128 = d: k blocks 1 KB apart, N 48, K 64 tokens)
        if (!warp_wait(&v_full[vr], (c / kVSlots) & 1, abort_flag, p.timeouts)) return false;
        if (!warp_wait(&dS_empty[b], (ub & 1) ^ 1, abort_flag, p.timeouts)) return false;
        tc_fence_after();
        const uint64_t dv = v_desc(vr);
        const uint32_t tds = tmem + kColDS + 64 * b;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk)
            mma_bf16(tds, dkt + kk * (2 * L::kGroup >> 4), dv + kk * 64, ID_DS, kk > 0);
          mma_commit(&dS_full[b]);
        }
        __syncwarp();
        return true;
      };
      bool ok = nchunks > 0 ? issue_independent(0) : true;
      for (int c = 0; ok && c < nchunks; ++c) {
        const int s = c % QKS, b = c & 1, vr = c % kVSlots;
        const uint32_t ub = static_cast<uint32_t>(c >> 1);
        if (c + 1 < nchunks && !issue_independent(c + 1)) break;
        // inter = qh [S | z] with the state before this chunk
        if (!warp_wait(&O_empty[b], (ub & 1) ^ 1, abort_flag, p.timeouts)) break;
        if (c > 0) {
          const int sb = (c - 1) & 1;
          if (!warp_wait(&S_full[sb], ((c - 1) >> 1) & 1, abort_flag, p.timeouts)) break;
          tc_fence_after();
          const uint64_t dq = stage_add(dq0, s);
          const uint64_t dS = ds0 + static_cast<uint64_t>(sb) * (L::kSBytes >> 4);
          const uint32_t ti = tmem + kColInter + 64 * b;
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_bf16(ti, dq + (kk >> 2) * 64 + (kk & 3) * 2, dS + kk * 64, ID_O, kk > 0);
            mma_commit(&S_empty[sb]);
          }
          __syncwarp();
        }
        // the q/k stage has served A', [dS | dz] and inter: free it for every
        // CTA of the cluster without waiting for P
        if (leader) mma_commit_multicast(&qk_empty[s], kAll);
        __syncwarp();
        // intra = P [V | 1]
        if (!warp_wait(&P_full[b], ub & 1, abort_flag, p.timeouts)) break;
        tc_fence_after();
        const uint64_t dP = dp0 + static_cast<uint64_t>(b) * ((kC * 128) >> 4);
        const uint64_t dv = v_desc(vr);
        const uint32_t tn = tmem + kColIntra + 64 * b;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk) mma_bf16(tn, dP + kk * 2, dv + kk * 64, ID_O, kk > 0);
          mma_commit(&P_empty[b]);
          mma_commit(&O_full[b]);
          mma_commit(&v_empty[vr]);
        }
        __syncwarp();
      }
      // every MMA issued has completed before TMEM is released
      if (leader) {
        mma_commit(drain);
        mbar_wait_drain(drain, 0);
      }
      __syncwarp();
    }
  } else if (warp >= kWarpPhi) {
    // ---------------- feature map on own rows, pushed to the peers ----------------
    const int tp = tid - kWarpPhi * 32;
    const uint32_t base = smem_u32(sm);
    for (int c = 0; c < nchunks; ++c) {
      const int r = c % RAW, s = c % QKS;
      if (!warp_wait(&raw_full[r], (c / RAW) & 1, abort_flag, p.timeouts)) break;
      // every CTA of the cluster has finished with this stage
      if (!warp_wait(&qk_empty[s], ((c / QKS) & 1) ^ 1, abort_flag, p.timeouts)) break;
      const int nv = min(kC, N - c * kC);
      map_rows<D, NS, DECAY>(sm + L::kOffRaw + r * L::kRawBytes, sm + s * L::kStageBytes, row0,
                             gq, gk, nv, tp);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&mapped[s]);
      if (warp == kWarpPhi) {
        // one warp waits for the other three, then lane 0 pushes
        if (!warp_wait(&mapped[s], (c / QKS) & 1, abort_flag, p.timeouts)) break;
      }
      if (tp == 0) {
        mbar_arrive(&raw_empty[r]);
        const uint32_t own = base + s * L::kStageBytes + rank * L::kOwnOff;
#pragma unroll 1
        for (int j = 1; j < NS; ++j) {
          const uint32_t peer = (rank + j) % NS;
          bulk_copy_to_peer(map_to_cta(own, peer), own, L::kOwnBytes,
                            map_to_cta(smem_u32(&qk_full[s]), peer));
        }
        bulk_commit_group();
        mbar_arrive_expect_tx(&qk_full[s], L::kPeerBytes);
      }
    }
    if (tp == 0) bulk_wait_read_all();
  } else if (warp >= kWarpO) {
    // ---------------- output rows ----------------
    const int w = warp - kWarpO;  // TMEM lane quadrant
    const int t = 16 * w + lane;  // M = 64 layout: rows 16w..16w+15 in lanes 0..15
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      const uint32_t ub = static_cast<uint32_t>(c >> 1);
      if (!warp_wait(&O_full[b], ub & 1, abort_flag, p.timeouts)) break;
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
  } else if (warp >= kWarpS) {
    // ---------------- state carry: thread d owns row d of the fp32 state ----------------
    const int w = warp - kWarpS;
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
      if (!warp_wait(&dS_full[b], ub & 1, abort_flag, p.timeouts)) break;
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
      if (!warp_wait(&S_empty[c & 1], ((c >> 1) & 1) ^ 1, abort_flag, p.timeouts)) break;
      if (d < D) {
        // row d of [S | z] in the MN-major (64-byte swizzled) operand layout
        uint8_t *sb = sm + L::kOffS + (c & 1) * L::kSBytes;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4 *>(sb + sw64_off(d, 16 * q)) =
              make_uint4(pack_bf16x2(S[8 * q + 0], S[8 * q + 1]),
                         pack_bf16x2(S[8 * q + 2], S[8 * q + 3]),
                         pack_bf16x2(S[8 * q + 4], S[8 * q + 5]),
                         pack_bf16x2(S[8 * q + 6], S[8 * q + 7]));
        *reinterpret_cast<__nv_bfloat16 *>(sb + L::kSBlk + sw64_off(d, 0)) =
            __float2bfloat16_rn(z);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S_full[c & 1]);
    }
  } else {
    // ---------------- P = A' masked to s <= t, bf16, 128-byte swizzled ----------------
    const int w = warp;  // TMEM lane quadrant
    const int t = 16 * w + lane;
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      const uint32_t ub = static_cast<uint32_t>(c >> 1);
      if (!warp_wait(&A_full[b], ub & 1, abort_flag, p.timeouts)) break;
      if (!warp_wait(&P_empty[b], (ub & 1) ^ 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      float a[64];
      tmem_ld32(tmem_addr(tmem, 32 * w, kColA + 64 * b), a);
      if (w >= 2) tmem_ld32(tmem_addr(tmem, 32 * w, kColA + 64 * b + 32), a + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&A_empty[b]);
      if (lane < 16) {
        uint8_t *prow = sm + L::kOffP + b * (kC * 128);
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
    }
  }

  // no CTA leaves while a peer may still write into it or signal its barriers
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

template <int D, int NS, bool DECAY>
cudaError_t launch_typed(const TcParams &prm, int BH, cudaStream_t s) {
  auto kern = causal_tc_kernel<D, NS, DECAY>;
  const int smem = Layout<D, NS>::kAlloc;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(NS, static_cast<unsigned>(BH));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int D, int NS>
cudaError_t launch_decay(const TcParams &prm, bool decay, int BH, cudaStream_t s) {
  return decay ? launch_typed<D, NS, true>(prm, BH, s) : launch_typed<D, NS, false>(prm, BH, s);
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
  const int NS = p.Dv / kDvs;  // CTAs per (batch, head): one cluster
  const int R = kC / NS;       // q/k rows each CTA loads
  TcParams prm;
  if (!make_tmap_3d_bf16(&prm.tmQ, p.q, p.D, p.N, BH, 64, R, 128) ||
      !make_tmap_3d_bf16(&prm.tmK, p.k, p.D, p.N, BH, 64, R, 128) ||
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
  if (p.D == 64)
    return NS == 2 ? launch_decay<64, 2>(prm, p.decay, BH, s) : launch_decay<64, 4>(prm, p.decay, BH, s);
  return NS == 2 ? launch_decay<128, 2>(prm, p.decay, BH, s) : launch_decay<128, 4>(prm, p.decay, BH, s);
}

}  // namespace linattn
