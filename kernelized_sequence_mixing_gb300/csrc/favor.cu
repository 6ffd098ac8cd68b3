// Performer random-feature map:  phi(x) = r^(-1/2) exp(W x - |x|^2 / 2).
//
// "Linear Attention Mechanisms" (dileepadev.github.io), "Choosing the Feature
// Map": random features exp(w_j . x) over r directions w_j (Performer) and
// their positive, orthogonal variant (FAVOR+).  The -|x|^2/2 term is what
// makes the expectation the passage states, E[phi(q) . phi(k)] = exp(q . k),
// hold for w ~ N(0, I); the directions W [r][D] are the caller's (drawn once,
// iid or block-orthogonal).  The map runs once over the rows of q and once
// over the rows of k.
//
// bf16: a tcgen05 GEMM  U = X W^T  (128 rows of X per tile, all r columns,
// K = D) with the exponential fused into the epilogue, so X is read and phi
// written exactly once.  Persistent CTAs; warp 4 streams 128-row tiles of X
// by TMA into a 3-stage ring (W is loaded once per CTA), warp 5 issues the
// MMAs into one of two TMEM accumulators, warps 0-3 take |x|^2 of their row
// from the staged tile and turn their row of U into phi:
//   phi = exp2(u log2(e) - |x|^2 log2(e) / 2 - log2(r) / 2), rounded to bf16,
// staged per warp in 32 x 32 boxes and written by TMA tile stores.
// fp32: the same map on CUDA cores in fp32 (the tensor cores' tf32 operands
// would cost the exponent ~1e-3 of relative accuracy).
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace linattn {
namespace {
using namespace tc;

constexpr int kRows = 128;    // rows of X per tile
constexpr int kStages = 3;    // X ring
constexpr int kThreads = 192; // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr int kWarpTma = 4, kWarpMma = 5;
constexpr float kLog2e = 1.4426950408889634f;

// barriers
enum { kWFull = 0, kXFull = 1, kXEmpty = kXFull + kStages, kAccFull = kXEmpty + kStages,
       kAccEmpty = kAccFull + 2, kDrain = kAccEmpty + 2, kNumBars = kDrain + 1 };

template <int D, int R>
struct FavorLayout {
  static constexpr int kXBox = kRows * 128;        // 64 bf16 columns x 128 rows, SW128
  static constexpr int kXStage = (D / 64) * kXBox;
  static constexpr int kWBox = R * 128;            // 64 columns x R rows
  static constexpr int kW = (D / 64) * kWBox;
  static constexpr int kStgBox = 32 * 64;          // 32 rows x 32 bf16, SW64
  static constexpr int kStgWarp = (R / 32) * kStgBox;
  static constexpr int kOffW = 0;
  static constexpr int kOffX = kOffW + kW;
  static constexpr int kOffStg = kOffX + kStages * kXStage;  // phi staging, per warp
  static constexpr int kOffBar = kOffStg + 4 * kStgWarp;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static constexpr int kTmemCols = 2 * R;              // two accumulators
};

struct FavorParams {
  CUtensorMap tmX[2];  // rows of q, rows of k: [rows][D] bf16
  CUtensorMap tmW;     // [R][D] bf16
  CUtensorMap tmO[2];  // phi of q, of k: [rows][R] bf16, 32 x 32 boxes, SW64
  unsigned int *timeouts;
  long long rows;  // rows of each input
  int tiles1;      // tiles per input
  int nin;         // inputs: 2 (q and k) or 1 (q)
  float cst;       // -log2(r) / 2
};

template <int D, int R>
__global__ void __launch_bounds__(kThreads, 1) favor_tc_kernel(const __grid_constant__ FavorParams p) {
  using L = FavorLayout<D, R>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = p.nin * p.tiles1;
  const int my = static_cast<int>(blockIdx.x) < ntiles
                     ? (ntiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                     : 0;

  if (tid == 0) {
    mbar_init(&bar[kWFull], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar[kXFull + s], 1);
      mbar_init(&bar[kXEmpty + s], 1 + 4);  // the MMAs' commit + the 4 epilogue warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar[kAccFull + b], 1);
      mbar_init(&bar[kAccEmpty + b], 4);
    }
    mbar_init(&bar[kDrain], 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, L::kTmemCols);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto tile_of = [&](int j, int *which, long long *row0) {
    const int t = static_cast<int>(blockIdx.x) + j * static_cast<int>(gridDim.x);
    *which = t >= p.tiles1 ? 1 : 0;
    *row0 = static_cast<long long>(t - *which * p.tiles1) * kRows;
  };

  if (warp == kWarpTma) {
    // ---------------- TMA producer (lane 0) ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tmW);
      prefetch_tmap(&p.tmX[0]);
      prefetch_tmap(&p.tmX[1]);
      mbar_arrive_expect_tx(&bar[kWFull], L::kW);
#pragma unroll
      for (int b = 0; b < D / 64; ++b)
        tma_load_3d(sm + L::kOffW + b * L::kWBox, &p.tmW, 64 * b, 0, 0, &bar[kWFull]);
      int issued = 0;
      for (int j = 0; j < my; ++j) {
        const int s = j % kStages;
        const uint32_t ph = static_cast<uint32_t>((j / kStages) & 1);
        if (!mbar_wait(&bar[kXEmpty + s], ph ^ 1, abort_flag, p.timeouts)) break;
        int which;
        long long row0;
        tile_of(j, &which, &row0);
        mbar_arrive_expect_tx(&bar[kXFull + s], L::kXStage);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(sm + L::kOffX + s * L::kXStage + b * L::kXBox, &p.tmX[which], 64 * b,
                      static_cast<int>(row0), 0, &bar[kXFull + s]);
        issued = j + 1;
      }
      if (*abort_flag) {  // let every issued copy land before the CTA exits
        mbar_wait_drain(&bar[kWFull], 0);
        for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
          mbar_wait_drain(&bar[kXFull + j % kStages], (j / kStages) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer (warp-wide loop, lane 0 issues) ----------------
    const bool leader = lane == 0;
    constexpr uint32_t ID = idesc_bf16(kRows, R, false, false);
    const uint32_t base = smem_u32(sm);
    bool ok = warp_wait(&bar[kWFull], 0, abort_flag, p.timeouts);
    for (int j = 0; ok && j < my; ++j) {
      const int s = j % kStages, b = j & 1;
      if (!warp_wait(&bar[kXFull + s], (j / kStages) & 1, abort_flag, p.timeouts)) break;
      if (!warp_wait(&bar[kAccEmpty + b], ((j >> 1) & 1) ^ 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      if (leader) {
        const uint64_t da = smem_desc(base + L::kOffX + s * L::kXStage, 16, 1024, kSw128);
        const uint64_t db = smem_desc(base + L::kOffW, 16, 1024, kSw128);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16(tmem + b * R, da + (kk >> 2) * (L::kXBox >> 4) + (kk & 3) * 2,
                   db + (kk >> 2) * (L::kWBox >> 4) + (kk & 3) * 2, ID, kk > 0 ? 1u : 0u);
        mma_commit(&bar[kAccFull + b]);
        mma_commit(&bar[kXEmpty + s]);
      }
      __syncwarp();
    }
    // every MMA issued has completed before TMEM is released
    if (leader) {
      mma_commit(&bar[kDrain]);
      mbar_wait_drain(&bar[kDrain], 0);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: warp w owns rows 32 w .. 32 w + 31 ----------------
    // phi goes out through the warp's staging boxes (one per 32 columns) by
    // TMA tile stores; rows past the end are clipped by the store itself
    const int r = 32 * warp + lane;
    uint8_t *stg = sm + L::kOffStg + warp * L::kStgWarp;
    for (int j = 0; j < my; ++j) {
      const int s = j % kStages, b = j & 1;
      int which;
      long long row0;
      tile_of(j, &which, &row0);
      if (!warp_wait(&bar[kXFull + s], (j / kStages) & 1, abort_flag, p.timeouts)) break;
      // |x|^2 of the row from the staged tile (bf16 values, fp32 sums)
      float sq = 0.f;
      const uint8_t *xs = sm + L::kOffX + s * L::kXStage;
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 u = *reinterpret_cast<const uint4 *>(xs + bx * L::kXBox + sw128_off(r, 16 * c));
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(w4[i] << 16), hi = __uint_as_float(w4[i] & 0xffff0000u);
            sq = fmaf(lo, lo, sq);
            sq = fmaf(hi, hi, sq);
          }
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kXEmpty + s]);
      if (!warp_wait(&bar[kAccFull + b], (j >> 1) & 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      const float cst = fmaf(-0.5f * kLog2e, sq, p.cst);
      if (lane == 0) bulk_wait_group_read0();  // the previous tile's stores have read stg
      __syncwarp();
#pragma unroll
      for (int cc = 0; cc < R / 32; ++cc) {
        float x[32];
        tmem_ld32(tmem_addr(tmem, 32 * warp, b * R + 32 * cc), x);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(exp2f(fmaf(x[2 * i], kLog2e, cst)),
                              exp2f(fmaf(x[2 * i + 1], kLog2e, cst)));
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4 *>(stg + cc * L::kStgBox + sw64_off(lane, 16 * i)) =
              make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar[kAccEmpty + b]);
        if (row0 + 32 * warp < p.rows) {  // a box past the last row is not stored
#pragma unroll
          for (int cc = 0; cc < R / 32; ++cc)
            tma_store_3d(&p.tmO[which], stg + cc * L::kStgBox, 32 * cc,
                         static_cast<int>(row0) + 32 * warp, 0);
        }
        bulk_commit_group();
      }
    }
    if (lane == 0) bulk_wait_group0();  // every store complete before the CTA exits
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, L::kTmemCols);
}

// fp32 (or any dtype) on CUDA cores: 32 rows per CTA, 256 threads, each a
// 4-row x 4-column block of U = X W^T, W held transposed in shared memory.
constexpr int kSimtRows = 32;

template <int D, int R, typename T>
__global__ void __launch_bounds__(256) favor_simt_kernel(const T *__restrict__ x,
                                                         const T *__restrict__ W,
                                                         T *__restrict__ out, long long rows,
                                                         float cst) {
  extern __shared__ float4 smem4[];
  float *WT = reinterpret_cast<float *>(smem4);  // [D][R]
  float *xs = WT + D * R;                         // [D][kSimtRows + 4] transposed rows
  float *hs = xs + D * (kSimtRows + 4);           // [kSimtRows] -|x|^2 log2(e) / 2
  constexpr int kLdx = kSimtRows + 4;
  const int tid = threadIdx.x;
  const long long r0 = static_cast<long long>(blockIdx.x) * kSimtRows;
  for (int i = tid; i < D * R; i += 256) {
    const int j = i / D, d = i % D;
    WT[d * R + j] = io<T>::load(W + i);
  }
  for (int i = tid; i < kSimtRows * D; i += 256) {
    const int rr = i / D, d = i % D;
    xs[d * kLdx + rr] = r0 + rr < rows ? io<T>::load(x + (r0 + rr) * D + d) : 0.f;
  }
  __syncthreads();
  if (tid < kSimtRows) {
    float sq = 0.f;
    for (int d = 0; d < D; ++d) sq = fmaf(xs[d * kLdx + tid], xs[d * kLdx + tid], sq);
    hs[tid] = -0.5f * kLog2e * sq;
  }
  __syncthreads();
  // thread: rows 4 (tid / (R / 4)) .., columns 4 (tid % (R / 4)) ..
  constexpr int CQ = R / 4;  // column quads
  for (int blk = tid; blk < (kSimtRows / 4) * CQ; blk += 256) {
    const int rq = blk / CQ, cq = blk % CQ;
    float acc[4][4] = {};
    for (int d = 0; d < D; ++d) {
      const float4 xv = *reinterpret_cast<const float4 *>(xs + d * kLdx + 4 * rq);
      const float4 wv = *reinterpret_cast<const float4 *>(WT + d * R + 4 * cq);
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
      const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = fmaf(xa[i], wa[c], acc[i][c]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const long long row = r0 + 4 * rq + i;
      if (row >= rows) continue;
      const float h = hs[4 * rq + i] + cst;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        io<T>::store(out + row * R + 4 * cq + c, exp2f(fmaf(acc[i][c], kLog2e, h)));
    }
  }
}

int num_sms_favor() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

template <int D, int R>
cudaError_t favor_tc_launch(const void *q, const void *k, const void *W, void *fq, void *fk,
                            long long rows, cudaStream_t s) {
  using L = FavorLayout<D, R>;
  FavorParams prm;
  prm.nin = k ? 2 : 1;
  if (!make_tmap_3d_bf16(&prm.tmX[0], q, D, rows, 1, 64, kRows, 128) ||
      !make_tmap_3d_bf16(&prm.tmX[1], k ? k : q, D, rows, 1, 64, kRows, 128) ||
      !make_tmap_3d_bf16(&prm.tmW, W, D, R, 1, 64, R, 128) ||
      !make_tmap_3d_bf16(&prm.tmO[0], fq, R, rows, 1, 32, 32, 64) ||
      !make_tmap_3d_bf16(&prm.tmO[1], k ? fk : fq, R, rows, 1, 32, 32, 64))
    return cudaErrorInvalidValue;
  prm.timeouts = wait_timeout_counter();
  if (!prm.timeouts) return cudaErrorInvalidValue;
  prm.rows = rows;
  prm.tiles1 = static_cast<int>((rows + kRows - 1) / kRows);
  prm.cst = -0.5f * log2f(static_cast<float>(R));
  auto kern = favor_tc_kernel<D, R>;
  // at least 120 KB of shared memory, so one CTA holds an SM and its tensor
  // memory (up to 256 columns) never waits for another CTA's
  const int smem = L::kBytes > 120 * 1024 ? L::kBytes : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long ntiles = static_cast<long long>(prm.nin) * prm.tiles1;
  const int grid = static_cast<int>(ntiles < num_sms_favor() ? ntiles : num_sms_favor());
  kern<<<grid, kThreads, smem, s>>>(prm);
  return cudaGetLastError();
}

template <int D, int R, typename T>
cudaError_t favor_simt_launch(const void *q, const void *k, const void *W, void *fq, void *fk,
                              long long rows, cudaStream_t s) {
  auto kern = favor_simt_kernel<D, R, T>;
  const size_t smem = sizeof(float) * (static_cast<size_t>(D) * R + D * (kSimtRows + 4) + kSimtRows);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float cst = -0.5f * log2f(static_cast<float>(R));
  const unsigned grid = static_cast<unsigned>((rows + kSimtRows - 1) / kSimtRows);
  const T *Wt = static_cast<const T *>(W);
  kern<<<grid, 256, smem, s>>>(static_cast<const T *>(q), Wt, static_cast<T *>(fq), rows, cst);
  if ((e = cudaGetLastError()) != cudaSuccess || !k) return e;
  kern<<<grid, 256, smem, s>>>(static_cast<const T *>(k), Wt, static_cast<T *>(fk), rows, cst);
  return cudaGetLastError();
}

template <int D, int R>
cudaError_t favor_dispatch(const void *q, const void *k, const void *W, void *fq, void *fk,
                           long long rows, Dtype dt, cudaStream_t s) {
  if (dt == kBF16) return favor_tc_launch<D, R>(q, k, W, fq, fk, rows, s);
  return favor_simt_launch<D, R, float>(q, k, W, fq, fk, rows, s);
}

}  // namespace

cudaError_t launch_favor_features(const void *q, const void *k, const void *W, void *fq,
                                  void *fk, long long rows, int D, int R, Dtype dt,
                                  cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (D == 64 && R == 64) return favor_dispatch<64, 64>(q, k, W, fq, fk, rows, dt, s);
  if (D == 64 && R == 128) return favor_dispatch<64, 128>(q, k, W, fq, fk, rows, dt, s);
  if (D == 128 && R == 64) return favor_dispatch<128, 64>(q, k, W, fq, fk, rows, dt, s);
  if (D == 128 && R == 128) return favor_dispatch<128, 128>(q, k, W, fq, fk, rows, dt, s);
  return cudaErrorNotSupported;
}

}  // namespace linattn
