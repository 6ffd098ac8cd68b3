// sm_103a primitives for the tensor-core kernels: mbarriers with bounded
// waits, TMA tile loads, tcgen05 (UMMA) descriptors, MMA issue, commit and
// tensor-memory loads.  Written directly as inline PTX.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace linattn {
namespace tc {

// A wait gives up after this many SM clock cycles (about one second at the
// GB300's clocks); legitimate waits last microseconds.
constexpr long long kWaitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// Arrive without ordering this thread's earlier memory operations: for
// hand-offs whose consumer only reuses tensor memory (tcgen05.wait::ld and
// tcgen05.fence::before_thread_sync already order those reads), so the arrive
// does not wait for outstanding global stores.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t *bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// `count` arrivals at once
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// `limit` cycles, or as soon as another thread of the CTA has given up
// (*abort), counting its own failure in *timeouts (device memory); returns
// false in both cases.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity,
                                                volatile int *abort, unsigned int *timeouts,
                                                long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      atomicAdd(timeouts, 1u);
      return false;
    }
  }
}
// The kernels' waits: the limit is kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          volatile int *abort,
                                          unsigned int *timeouts) {
  return mbar_wait_limit(bar, parity, abort, timeouts, kWaitCycles);
}
// mbar_wait executed by a whole warp, agreeing on the outcome: if any lane
// gave up, every lane returns false, so the warp leaves its loop together.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          unsigned int *timeouts) {
  const bool ok = mbar_wait(bar, parity, abort, timeouts);
  return __all_sync(0xffffffffu, ok);
}
// Bounded wait used only while shutting down after an abort: waits for work
// already in flight (copies, MMAs) so that no engine still writes into shared
// or tensor memory when the CTA exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
}

// ---- TMA --------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int x,
                                            int y, int z, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// TMA tile store from shared memory (bulk-group completion), and the
// bulk-group bookkeeping of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *smem_src, int x,
                                             int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(smem_u32(smem_src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until the thread's committed bulk stores have read their shared memory
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// wait until the thread's committed bulk stores are complete
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// One 32-byte store of eight 32-bit words to global memory (the address must
// be 32-byte aligned): a whole sector per instruction and thread.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
// Prefetch a tile into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- named barriers -----------------------------------------------------------
// Named barrier among `count` threads (multiple of 32).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- fences -----------------------------------------------------------------
// generic-proxy shared-memory writes -> visible to the async proxy (MMA, TMA)
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- UMMA descriptors -------------------------------------------------------
enum Swizzle : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };

// Shared-memory matrix descriptor: start address, leading/stride byte
// offsets (in bytes, multiples of 16), descriptor version 1, swizzle mode.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              Swizzle sw) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(sw) << 61;
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulator.
// a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// ---- tensor memory ----------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit values: thread i of the warp receives lane
// (base lane + i), columns col..col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// one column
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
  return __uint_as_float(r);
}

// 32 lanes x 16 columns
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Stores: thread i of the warp writes lane (base lane + i).  The values are
// in tensor memory once tcgen05.wait::st has returned.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, int lane, int col) {
  return base + (static_cast<uint32_t>(lane) << 16) + static_cast<uint32_t>(col);
}

// ---- flags in global memory shared between CTAs ------------------------------
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---- packed bf16 helpers ------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

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

// phi (IDENT = false) or the identity (inputs already features), times the
// per-row scale, on a pair of bf16 values.
template <bool IDENT>
__device__ __forceinline__ uint32_t feat_scale_bf16x2(uint32_t w, uint32_t scale2) {
  if constexpr (IDENT) {
    const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&w),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&scale2));
    return *reinterpret_cast<const uint32_t *>(&r);
  } else {
    return phi_scale_bf16x2(w, scale2);
  }
}

// ---- swizzled shared-memory addressing ---------------------------------------
// Byte offset of (row, byte-in-row) in a tile of 128-byte rows with the
// 128-byte swizzle (16-byte chunk index XOR row % 8); tile 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128_off(int row, int byte) {
  return static_cast<uint32_t>(row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15)));
}
// The same for 64-byte rows with the 64-byte swizzle (chunk XOR (row/2) % 4);
// tile 512-byte aligned.
__device__ __forceinline__ uint32_t sw64_off(int row, int byte) {
  return static_cast<uint32_t>(row * 64 +
                               ((((byte >> 4) ^ ((row >> 1) & 3)) << 4) | (byte & 15)));
}

// Row d of [T | z] (fp32 values of 32 consecutive columns starting at column
// 32 * atom) into the MN-major, 64-byte-swizzled bf16 operand.
__device__ __forceinline__ void put_sop32(uint8_t *sop, int atom_bytes, int atom, int d,
                                          const float *x) {
  uint8_t *a = sop + atom * atom_bytes;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4 *>(a + sw64_off(d, 16 * q)) =
        make_uint4(pack_bf16x2(x[8 * q + 0], x[8 * q + 1]), pack_bf16x2(x[8 * q + 2], x[8 * q + 3]),
                   pack_bf16x2(x[8 * q + 4], x[8 * q + 5]), pack_bf16x2(x[8 * q + 6], x[8 * q + 7]));
}
__device__ __forceinline__ void put_sop16(uint8_t *sop, int atom_bytes, int atom, int d,
                                          const float *x) {
  uint8_t *a = sop + atom * atom_bytes;
#pragma unroll
  for (int q = 0; q < 2; ++q)
    *reinterpret_cast<uint4 *>(a + sw64_off(d, 16 * q)) =
        make_uint4(pack_bf16x2(x[8 * q + 0], x[8 * q + 1]), pack_bf16x2(x[8 * q + 2], x[8 * q + 3]),
                   pack_bf16x2(x[8 * q + 4], x[8 * q + 5]), pack_bf16x2(x[8 * q + 6], x[8 * q + 7]));
}

// D[tmem] (+)= A[tmem] * B[smem]^T: row m of A in tensor-memory lane m, its
// K values as bf16 pairs, 16 K values in 8 consecutive 32-bit columns.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

}  // namespace tc

// Host: encode a rank-3 bf16 tensor map over a dense [z][y][x] array
// (x innermost), box (box_x, box_y, 1), swizzle of 32, 64 or 128 bytes (0:
// none), zero fill out of bounds.  Returns false for another swizzle value
// or if the driver rejects the map.
bool make_tmap_3d_bf16(CUtensorMap *map, const void *base, uint64_t dim_x, uint64_t dim_y,
                       uint64_t dim_z, uint32_t box_x, uint32_t box_y, int swizzle_bytes);

// Host: device address of the wait-timeout counter on the current device
// (nullptr if it cannot be obtained).
unsigned int *wait_timeout_counter();

// Host: run the kernels' bounded mbarrier wait, with a limit of `cycles`,
// on a barrier nothing arrives on (one CTA of one warp); *gave_up (host)
// becomes 1 when the wait gave up and counted itself in the timeout counter.
// Synchronises the device.
cudaError_t wait_selftest(long long cycles, int *gave_up);

}  // namespace linattn
