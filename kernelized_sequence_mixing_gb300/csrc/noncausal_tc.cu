// Non-causal linear attention on tcgen05 tensor cores (sm_103a), bf16: the
// two streaming passes of "Linear Attention Mechanisms" (dileepadev.github.io),
// "The Kernel Trick for Attention": S = sum_j phi(k_j) v_j^T and
// z = sum_j phi(k_j) once per (batch, head), then
// o_i = phi(q_i)^T S / (phi(q_i) . z + eps) for every query (eps as in the
// NumPy listing of "Linear Attention Mechanisms" (sadullah.online)).
//
// Both passes are persistent: a grid of CTAs (one or two per SM) walks work
// items (batch-head, part), a part being a run of whole 128-token tiles, in
// round-robin order.  Each CTA streams its tiles through a ring of TMA
// stages; four warps apply the feature map in place; one thread issues the
// MMAs; fp32 accumulators live in tensor memory, two of them, so that one is
// drained while the other fills.
//
//   reduce:  per item, [S_p | z_p] = phi(K_p)^T [V_p | 1]  (M = D, padded to
//            128 rows with a zero block when D = 64; N = Dv + 16; K = tokens),
//            written as the part's record; a scan over the parts sums them.
//   apply:   per tile, [num | den] = phi(Q) [S | z]  (M = 128 tokens,
//            N = Dv + 16, K = D) and o = num / (den + eps).
//
// Operands are single bf16 values with fp32 accumulation: the output is
// bf16, so the split operands of the prefill's reduction (which keeps 1e-4 of
// fp64 for the decode state) are not needed here.
//
// Warp roles (10 warps): 0 TMA producer; 1 tensor-memory owner and MMA
// issuer; 2-5 feature map; 6-9 reduce: record writers (thread = row d of the
// state), apply: [S | z] operand writers and output rows (thread = token row).
// Every wait is bounded; a CTA that gives up counts the failure in device
// memory, drains its in-flight copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace linattn {
namespace {

using namespace tc;

constexpr int kT = 128;              // tokens per tile
constexpr int kBox = 128 * 128;      // one TMA box: 128 rows x 64 bf16, 128-byte swizzle
constexpr int kThreadsNc = 320;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpMap = 2, kWarpOut = 6;
constexpr int kMaxStages = 8;
constexpr int kSmemTwoPerSm = 113 * 1024;  // per CTA when two share an SM
constexpr int kSmemMax = 227 * 1024;

enum NcPass : int { kReduce = 0, kApply = 1 };

// Shared-memory plan of a pass.  Reduce stage: k boxes | v boxes (| ones box
// when Dv = 128); after the stages, a zero box (D = 64: the second 64-row
// block of the M = 128 operand kh^T) and, for Dv = 64, one ones box that
// every stage's [V | 1] reaches through its own descriptor stride.  Apply
// stage: q boxes; after the stages, [S | z] in 32-column atoms of D rows x
// 64 bytes (64-byte swizzle).
template <int D, int DV, int PASS>
struct NcLay {
  static constexpr int KB = D / 64, VB = DV / 64;
  static constexpr int NA = DV + 16;  // columns of [V | 1], [S | z], the accumulators
  static constexpr bool kOnesInStage = PASS == kReduce && DV == 128;
  static constexpr int kStageBytes = PASS == kReduce ? (KB + VB + (kOnesInStage ? 1 : 0)) * kBox : KB * kBox;
  static constexpr int kSopAtom = D * 64;
  static constexpr int kSharedBytes =
      PASS == kReduce ? ((D == 64 ? kBox : 0) + (kOnesInStage ? 0 : kBox)) : (DV / 32 + 1) * kSopAtom;
  static constexpr int kNumBars = 3 * kMaxStages + 8;
  static constexpr int kFixed = kSharedBytes + kNumBars * 8 + 32 + 1024;
  // two CTAs per SM when at least three stages fit in half the shared memory
  static constexpr int kFitHalf = (kSmemTwoPerSm - kFixed) / kStageBytes;
  static constexpr bool kTwoPerSm = kFitHalf >= 3 && 2 * NA <= 128 + 128;  // tensor memory: 256 each
  static constexpr int kFit = kTwoPerSm ? kFitHalf : (kSmemMax - kFixed) / kStageBytes;
  static constexpr int kStages = kFit > kMaxStages ? kMaxStages : kFit;
  static constexpr int kOffShared = kStages * kStageBytes;
  static constexpr int kOffZero = kOffShared;                                    // reduce, D = 64
  static constexpr int kOffOnes = kOffShared + (D == 64 ? kBox : 0);             // reduce, Dv = 64
  static constexpr int kOffSop = kOffShared;                                     // apply
  static constexpr int kOffBar = kOffShared + kSharedBytes;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kAlloc = kOffMisc + 32 + 1024;  // slack for the 1024-byte alignment
  static constexpr uint32_t kTmemCols = 2 * NA <= 256 ? 256 : 512;
  static_assert(kStages >= 2, "stages");
  static_assert(kAlloc <= kSmemMax, "shared memory");
  static_assert(kStageBytes % 1024 == 0 && kOffShared % 1024 == 0, "alignment");
};

struct NcParams {
  CUtensorMap tmA, tmB;  // reduce: k, v; apply: q (tmB unused)
  float *rec;            // [BH][rec_parts][D*Dv + D]; apply reads slot 0 (the sum over parts)
  __nv_bfloat16 *o;      // apply: [BH][N][Dv]
  unsigned int *timeouts;
  int BH, N, P, tpp;     // parts of this pass; tpp: tiles per part (the last may have fewer)
  int rec_parts;         // records per (batch, head)
  int o_v8;              // o is 32-byte aligned
  float eps;
};

// phi (or the identity) times a row factor in place on row r of a box:
// 8 chunks of 16 bytes, 128-byte swizzle.
template <bool IDENT>
__device__ __forceinline__ void map_box_row(uint8_t *box, int r, uint32_t sc) {
  uint4 x[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) x[c] = *reinterpret_cast<const uint4 *>(box + sw128_off(r, 16 * c));
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    x[c].x = feat_scale_bf16x2<IDENT>(x[c].x, sc);
    x[c].y = feat_scale_bf16x2<IDENT>(x[c].y, sc);
    x[c].z = feat_scale_bf16x2<IDENT>(x[c].z, sc);
    x[c].w = feat_scale_bf16x2<IDENT>(x[c].w, sc);
    *reinterpret_cast<uint4 *>(box + sw128_off(r, 16 * c)) = x[c];
  }
}

template <int D, int DV, int PASS, bool IDENT>
__global__ void __launch_bounds__(kThreadsNc) noncausal_tc_kernel(const __grid_constant__ NcParams p) {
  using L = NcLay<D, DV, PASS>;
  constexpr int S = L::kStages, NA = L::NA;
  constexpr size_t kRec = static_cast<size_t>(D) * DV + D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
  uint64_t *full = bars, *mapped = bars + kMaxStages, *empty = bars + 2 * kMaxStages;
  uint64_t *acc_full = bars + 3 * kMaxStages;  // [2] accumulator complete
  uint64_t *acc_free = acc_full + 2;           // [2] accumulator read
  uint64_t *sop_ready = acc_full + 4;          // apply: [S | z] written
  uint64_t *item_done = acc_full + 5;          // apply: every MMA of the item done
  uint64_t *drain = acc_full + 6;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N, P = p.P, tpp = p.tpp;
  const int ntile = (N + kT - 1) / kT;
  const int nitems = p.BH * P;

  // ---- set-up: constant operand blocks, barriers, tensor memory ----
  if (PASS == kReduce) {
    // zero box (D = 64) and ones boxes (column 0 = 1 in every row)
    for (int i = tid; i < L::kSharedBytes / 16; i += kThreadsNc)
      reinterpret_cast<uint4 *>(sm + L::kOffShared)[i] = make_uint4(0, 0, 0, 0);
    if (L::kOnesInStage)
      for (int i = tid; i < S * (kBox / 16); i += kThreadsNc)
        reinterpret_cast<uint4 *>(sm + (i / (kBox / 16)) * L::kStageBytes + (L::KB + L::VB) * kBox)
            [i % (kBox / 16)] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (tid < kT) {
      const __nv_bfloat16 one = __float2bfloat16_rn(1.f);
      if (L::kOnesInStage) {
        for (int st = 0; st < S; ++st)
          *reinterpret_cast<__nv_bfloat16 *>(sm + st * L::kStageBytes + (L::KB + L::VB) * kBox +
                                             sw128_off(tid, 0)) = one;
      } else {
        *reinterpret_cast<__nv_bfloat16 *>(sm + L::kOffOnes + sw128_off(tid, 0)) = one;
      }
    }
  }
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&mapped[i], 4);
      mbar_init(&empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_free[b], 4);
    }
    mbar_init(sop_ready, 4);
    mbar_init(item_done, 1);
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

  // the tiles [t0, t1) of item `it` (part of its batch-head)
  auto item_tiles = [&](int it, int *bh, int *part, int *t0, int *t1) {
    *bh = it / P;
    *part = it % P;
    *t0 = *part * tpp;
    *t1 = min(ntile, *t0 + tpp);
  };

  if (warp == kWarpTma) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmA);
      if (PASS == kReduce) prefetch_tmap(&p.tmB);
      int c = 0, issued = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < nitems; it += gridDim.x) {
        int bh, part, t0, t1;
        item_tiles(it, &bh, &part, &t0, &t1);
        for (int t = t0; t < t1; ++t, ++c) {
          const int s = c % S;
          if (!mbar_wait(&empty[s], ((c / S) & 1) ^ 1, abort_flag, p.timeouts)) {
            ok = false;
            break;
          }
          uint8_t *st = sm + s * L::kStageBytes;
          mbar_arrive_expect_tx(&full[s], (PASS == kReduce ? L::KB + L::VB : L::KB) * kBox);
#pragma unroll
          for (int b = 0; b < L::KB; ++b) tma_load_3d(st + b * kBox, &p.tmA, 64 * b, t * kT, bh, &full[s]);
          if (PASS == kReduce)
#pragma unroll
            for (int b = 0; b < L::VB; ++b)
              tma_load_3d(st + (L::KB + b) * kBox, &p.tmB, 64 * b, t * kT, bh, &full[s]);
          issued = c + 1;
        }
      }
      if (*abort_flag)  // let every issued copy land before the CTA exits
        for (int q = issued > S ? issued - S : 0; q < issued; ++q) mbar_wait_drain(&full[q % S], (q / S) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer ----------------
    const bool leader = lane == 0;
    const uint32_t base = smem_u32(sm);
    int c = 0, j = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < nitems; it += gridDim.x, ++j) {
      int bh, part, t0, t1;
      item_tiles(it, &bh, &part, &t0, &t1);
      if (PASS == kReduce) {
        // [S_p | z_p] += kh^T [V | 1] into accumulator j % 2 (M 128 d, N Dv + 16, K 128 tokens)
        constexpr uint32_t ID = idesc_bf16(128, NA, true, true);
        const int b = j & 1;
        if (!warp_wait(&acc_free[b], ((j >> 1) & 1) ^ 1, abort_flag, p.timeouts)) break;
        tc_fence_after();
        for (int t = t0; t < t1; ++t, ++c) {
          const int s = c % S;
          if (!warp_wait(&mapped[s], (c / S) & 1, abort_flag, p.timeouts)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            const uint32_t ks = base + s * L::kStageBytes, vs = ks + L::KB * kBox;
            // kh^T: M = d in 64-row blocks (the second one is the zero box when
            // D = 64); [V | 1]: N in 64-column blocks, the last one the ones box
            const uint64_t da = smem_desc(ks, D == 128 ? kBox : base + L::kOffZero - ks, 1024, kSw128);
            const uint64_t db = smem_desc(vs, L::kOnesInStage ? kBox : base + L::kOffOnes - vs, 1024, kSw128);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_bf16(tmem + b * NA, da + kk * 128, db + kk * 128, ID, (t > t0 || kk > 0) ? 1u : 0u);
            mma_commit(&empty[s]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (leader) mma_commit(&acc_full[b]);
        __syncwarp();
      } else {
        // [num | den] = qh [S | z]  (M 128 tokens, N Dv + 16, K = D), per tile
        constexpr uint32_t ID = idesc_bf16(128, NA, false, true);
        const uint64_t dsop = smem_desc(base + L::kOffSop, L::kSopAtom, 512, kSw64);
        if (!warp_wait(sop_ready, j & 1, abort_flag, p.timeouts)) break;
        for (int t = t0; t < t1; ++t, ++c) {
          const int s = c % S, b = c & 1;
          if (!warp_wait(&mapped[s], (c / S) & 1, abort_flag, p.timeouts) ||
              !warp_wait(&acc_free[b], ((c >> 1) & 1) ^ 1, abort_flag, p.timeouts)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            const uint64_t dq = smem_desc(base + s * L::kStageBytes, 16, 1024, kSw128);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_bf16(tmem + b * NA, dq + (kk >> 2) * (kBox >> 4) + (kk & 3) * 2, dsop + kk * 64, ID,
                       kk > 0 ? 1u : 0u);
            mma_commit(&empty[s]);
            mma_commit(&acc_full[b]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (leader) mma_commit(item_done);  // [S | z] may be replaced
        __syncwarp();
      }
    }
    // every MMA issued has completed before tensor memory is released
    if (leader) {
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp < kWarpOut) {
    // ---------------- feature map, thread = token row ----------------
    const int r = 32 * (warp - kWarpMap) + lane;
    int c = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < nitems; it += gridDim.x) {
      int bh, part, t0, t1;
      item_tiles(it, &bh, &part, &t0, &t1);
      for (int t = t0; t < t1; ++t, ++c) {
        const int s = c % S;
        if (!warp_wait(&full[s], (c / S) & 1, abort_flag, p.timeouts)) {
          ok = false;
          break;
        }
        // reduce: rows past the sequence end are zero (the copy filled them
        // with zeros, and phi(0) = 1); apply: those rows are not stored
        const uint32_t sc = PASS == kReduce && t * kT + r >= N ? 0u : pack_bf16x2(1.f, 1.f);
        uint8_t *st = sm + s * L::kStageBytes;
#pragma unroll
        for (int b = 0; b < L::KB; ++b) map_box_row<IDENT>(st + b * kBox, r, sc);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&mapped[s]);
      }
    }
  } else {
    const int w = warp & 3;        // tensor-memory lane quadrant
    const int row = 32 * w + lane; // reduce: row d of the state; apply: token row
    if (PASS == kReduce) {
      // ---------------- part records ----------------
      int j = 0;
      for (int it = blockIdx.x; it < nitems; it += gridDim.x, ++j) {
        int bh, part, t0, t1;
        item_tiles(it, &bh, &part, &t0, &t1);
        const int b = j & 1;
        if (!warp_wait(&acc_full[b], (j >> 1) & 1, abort_flag, p.timeouts)) break;
        tc_fence_after();
        const uint32_t ta = tmem_addr(tmem, 32 * w, b * NA);
        float *rec = p.rec + (static_cast<size_t>(bh) * P + part) * kRec;
#pragma unroll 1
        for (int cc = 0; cc < DV / 32; ++cc) {
          float x[32];
          tmem_ld32(ta + 32 * cc, x);
          tmem_wait_ld();
          if (row < D) {
            float4 *dst = reinterpret_cast<float4 *>(rec + static_cast<size_t>(row) * DV + 32 * cc);
#pragma unroll
            for (int q = 0; q < 8; ++q) __stcg(dst + q, make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
          }
        }
        const float zd = tmem_ld1(ta + DV);
        tmem_wait_ld();
        if (row < D) __stcg(rec + static_cast<size_t>(D) * DV + row, zd);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&acc_free[b]);
      }
    } else {
      // ---------------- [S | z] operand, then output rows ----------------
      uint8_t *sop = sm + L::kOffSop;
      int c = 0, j = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < nitems; it += gridDim.x, ++j) {
        int bh, part, t0, t1;
        item_tiles(it, &bh, &part, &t0, &t1);
        // the previous item's MMAs have read the old [S | z]
        if (j > 0 && !warp_wait(item_done, (j - 1) & 1, abort_flag, p.timeouts)) break;
        if (row < D) {
          const float *src = p.rec + static_cast<size_t>(bh) * p.rec_parts * kRec + static_cast<size_t>(row) * DV;
#pragma unroll 1
          for (int cc = 0; cc < DV / 32; ++cc) {
            float x[32];
            const float4 *s4 = reinterpret_cast<const float4 *>(src + 32 * cc);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 v4 = __ldcg(s4 + q);
              x[4 * q] = v4.x;
              x[4 * q + 1] = v4.y;
              x[4 * q + 2] = v4.z;
              x[4 * q + 3] = v4.w;
            }
            put_sop32(sop, L::kSopAtom, cc, row, x);
          }
          float zz[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) zz[e] = 0.f;
          zz[0] = __ldcg(p.rec + static_cast<size_t>(bh) * p.rec_parts * kRec + static_cast<size_t>(D) * DV + row);
          put_sop16(sop, L::kSopAtom, DV / 32, row, zz);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sop_ready);
        for (int t = t0; t < t1; ++t, ++c) {
          const int b = c & 1;
          if (!warp_wait(&acc_full[b], (c >> 1) & 1, abort_flag, p.timeouts)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ta = tmem_addr(tmem, 32 * w, b * NA);
          const int tok = t * kT + row;
          uint8_t *orow = reinterpret_cast<uint8_t *>(p.o + (static_cast<size_t>(bh) * N + tok) * DV);
          const float den = tmem_ld1(ta + DV);
          float x[DV / 2];
          uint32_t pk[DV / 4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // two halves of the row: Dv / 2 columns each
            if (DV == 64) {
              tmem_ld32(ta + 32 * h, x);
            } else {
              tmem_ld32(ta + 64 * h, x);
              tmem_ld32(ta + 64 * h + 32, x + 32);
            }
            tmem_wait_ld();
            if (h == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_relaxed(&acc_free[b]);
            }
            const float inv = 1.f / (den + p.eps);
#pragma unroll
            for (int e = 0; e < DV / 4; ++e) pk[e] = pack_bf16x2(x[2 * e] * inv, x[2 * e + 1] * inv);
            if (tok < N) {
              uint8_t *dst = orow + h * DV;  // DV / 2 bf16 = DV bytes
              if (p.o_v8) {
#pragma unroll
                for (int q = 0; q < DV / 32; ++q) st_global_v8(dst + 32 * q, pk + 8 * q);
              } else {
#pragma unroll
                for (int q = 0; q < DV / 16; ++q)
                  *reinterpret_cast<uint4 *>(dst + 16 * q) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
              }
            }
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, L::kTmemCols);
}

// Dynamic shared memory of a pass, and the whole of the SM's unified memory
// as shared memory (left to itself, the driver may size the carveout for
// one CTA and so keep the second CTA of a pass that plans two per SM off
// the SM).
template <typename K>
cudaError_t nc_set_attributes(K kern, int smem) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                              static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

template <int D, int DV, int PASS, bool IDENT>
int nc_grid() {
  // CTAs that run at once on the device: one or two per SM by the plan (the
  // shared-memory plan, at most 256 tensor-memory columns and 320 threads of
  // at most 102 registers each let two share an SM).  The passes have no
  // waits between CTAs, so a grid larger than what fits only runs longer.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  return sms * (NcLay<D, DV, PASS>::kTwoPerSm ? 2 : 1);
}

// Parts per (batch, head) for `slots` resident CTAs: the number of whole
// waves of equal items times the tiles of an item, plus a cost per part in
// tiles (the reduce pass: a record to write and scan; the apply pass: at
// each new item the pipeline drains while [S | z] is replaced).
int nc_parts(int BH, int ntile, int slots, double per_part) {
  int best = 1;
  double best_t = 1e300;
  const int pmax = ntile < 64 ? ntile : 64;
  for (int P = 1; P <= pmax; ++P) {
    const int tpp = (ntile + P - 1) / P;
    const int pe = (ntile + tpp - 1) / tpp;  // parts with at least one tile
    const long long items = static_cast<long long>(BH) * pe;
    const long long waves = (items + slots - 1) / slots;
    const double t = static_cast<double>(waves) * tpp + per_part * pe;
    if (t < best_t - 1e-9) {
      best_t = t;
      best = pe;
    }
  }
  return best;
}

template <int D, int DV, int PASS, bool IDENT>
cudaError_t nc_launch(const NcParams &prm, int grid, cudaStream_t s) {
  auto kern = noncausal_tc_kernel<D, DV, PASS, IDENT>;
  const int smem = NcLay<D, DV, PASS>::kAlloc;
  cudaError_t e = nc_set_attributes(kern, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreadsNc, smem, s>>>(prm);
  return cudaGetLastError();
}

struct NcPlan {
  int Pr, Pa, gr, ga;
};

template <int D, int DV, bool IDENT>
NcPlan nc_plan(int BH, int N) {
  const int ntile = (N + kT - 1) / kT;
  NcPlan pl;
  pl.gr = nc_grid<D, DV, kReduce, IDENT>();
  pl.ga = nc_grid<D, DV, kApply, IDENT>();
  pl.Pr = nc_parts(BH, ntile, pl.gr, 0.5);
  pl.Pa = nc_parts(BH, ntile, pl.ga, 3.0);
  const long long ir = static_cast<long long>(BH) * pl.Pr, ia = static_cast<long long>(BH) * pl.Pa;
  if (ir < pl.gr) pl.gr = static_cast<int>(ir);
  if (ia < pl.ga) pl.ga = static_cast<int>(ia);
  return pl;
}

template <bool IDENT>
NcPlan nc_plan_dims(int BH, int N, int D, int Dv) {
  if (D == 64) return Dv == 64 ? nc_plan<64, 64, IDENT>(BH, N) : nc_plan<64, 128, IDENT>(BH, N);
  return Dv == 64 ? nc_plan<128, 64, IDENT>(BH, N) : nc_plan<128, 128, IDENT>(BH, N);
}

template <int D, int DV, bool IDENT>
cudaError_t nc_run(const Problem &p, float *rec, const NcPlan &pl, cudaStream_t s) {
  const int BH = p.B * p.H, ntile = (p.N + kT - 1) / kT;
  NcParams prm = {};
  if (!make_tmap_3d_bf16(&prm.tmA, p.k, D, p.N, BH, 64, kT, 128) ||
      !make_tmap_3d_bf16(&prm.tmB, p.v, DV, p.N, BH, 64, kT, 128))
    return cudaErrorNotSupported;
  prm.timeouts = wait_timeout_counter();
  if (!prm.timeouts) return cudaErrorNotSupported;
  prm.rec = rec;
  prm.rec_parts = pl.Pr;
  prm.BH = BH;
  prm.N = p.N;
  prm.eps = p.eps;
  prm.P = pl.Pr;
  prm.tpp = (ntile + pl.Pr - 1) / pl.Pr;
  cudaError_t e = nc_launch<D, DV, kReduce, IDENT>(prm, pl.gr, s);
  if (e != cudaSuccess) return e;
  Gammas ones;
  for (int h = 0; h < kMaxHeads; ++h) ones.g[h] = 0.f;  // log2(1): no decay
  e = launch_part_scan(rec, BH, p.H, pl.Pr, p.N, D, DV, ones, kScanSum, nullptr, nullptr, s);
  if (e != cudaSuccess) return e;
  if (!make_tmap_3d_bf16(&prm.tmA, p.q, D, p.N, BH, 64, kT, 128)) return cudaErrorNotSupported;
  prm.o = static_cast<__nv_bfloat16 *>(p.o);
  prm.o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
  // the apply pass reads the sum from slot 0 of each (batch, head)
  prm.P = pl.Pa;
  prm.tpp = (ntile + pl.Pa - 1) / pl.Pa;
  return nc_launch<D, DV, kApply, IDENT>(prm, pl.ga, s);
}

template <bool IDENT>
cudaError_t nc_run_dims(const Problem &p, float *rec, const NcPlan &pl, cudaStream_t s) {
  if (p.D == 64)
    return p.Dv == 64 ? nc_run<64, 64, IDENT>(p, rec, pl, s) : nc_run<64, 128, IDENT>(p, rec, pl, s);
  return p.Dv == 64 ? nc_run<128, 64, IDENT>(p, rec, pl, s) : nc_run<128, 128, IDENT>(p, rec, pl, s);
}

}  // namespace

bool noncausal_tc_supported(const Problem &p) {
  return p.dtype == kBF16 && !p.decay && (p.D == 64 || p.D == 128) && (p.Dv == 64 || p.Dv == 128) &&
         p.N > 0 && static_cast<long long>(p.B) * p.H > 0;
}

size_t noncausal_tc_workspace_bytes(const Problem &p) {
  const int BH = p.B * p.H;
  const NcPlan pl = p.ident ? nc_plan_dims<true>(BH, p.N, p.D, p.Dv) : nc_plan_dims<false>(BH, p.N, p.D, p.Dv);
  return sizeof(float) * static_cast<size_t>(BH) * pl.Pr * (static_cast<size_t>(p.D) * p.Dv + p.D);
}

cudaError_t launch_noncausal_tc(const Problem &p, void *ws, cudaStream_t s) {
  if (!noncausal_tc_supported(p) || !ws) return cudaErrorNotSupported;
  const int BH = p.B * p.H;
  const NcPlan pl = p.ident ? nc_plan_dims<true>(BH, p.N, p.D, p.Dv) : nc_plan_dims<false>(BH, p.N, p.D, p.Dv);
  float *rec = static_cast<float *>(ws);
  return p.ident ? nc_run_dims<true>(p, rec, pl, s) : nc_run_dims<false>(p, rec, pl, s);
}

}  // namespace linattn
