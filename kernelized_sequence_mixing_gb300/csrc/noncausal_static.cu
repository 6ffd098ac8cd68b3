// Non-causal forward that allocates nothing: its scratch (the per-head S, z
// and the split partial sums) lives in a fixed array inside the library.
//
// Why: the regular non-causal forward takes a stream-ordered workspace with
// cudaMallocAsync.  Some callers cannot let a library allocate device memory:
// applications that reserve all of HBM up front in their own memory manager
// and forbid allocations by third-party code, and latency-critical loops
// (e.g. serving) where an allocation may stall on, or fail with, a full or
// fragmented memory pool.  This entry point uses memory that exists as soon
// as the library is loaded on a device.
#include <math.h>
#include <mutex>
#include <stdint.h>

#include "../../include/linattn.h"
#include "kernels.h"

using namespace linattn;

namespace {

// 32 MiB of scratch on every GPU that loads the library, kept until the
// process exits.
constexpr size_t kScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_nc_scratch[kScratchBytes];

// Device address of the scratch array on the current device.  The host-side
// name g_nc_scratch is only a stand-in, so the address is queried once per
// device (with that device current) and cached.
float *scratch_on_current_device() {
  constexpr int kMaxDev = 64;
  static void *addr[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_nc_scratch) != cudaSuccess || !p) return nullptr;
    addr[dev] = p;
  }
  return static_cast<float *>(addr[dev]);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" {

size_t la_forward_noncausal_static_limit(void) { return kScratchBytes; }

la_status_t la_forward_noncausal_static(const void *q, const void *k, const void *v, void *o,
                                        int B, int H, int N, int D, int Dv, float eps,
                                        la_dtype_t dtype, void *stream) {
  // argument checks first: a rejected call touches no device
  if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || N < 0 || D <= 0 || Dv <= 0) return LA_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || (Dv != 64 && Dv != 128)) return LA_ERR_UNSUPPORTED;
  if (H > kMaxHeads) return LA_ERR_UNSUPPORTED;
  if ((int64_t)B * H * (int64_t)(N > 0 ? N : 1) >= ((int64_t)1 << 31)) return LA_ERR_UNSUPPORTED;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)B * H * N;
  if (rows == 0) return LA_OK;
  if (!q || !k || !v || !o) return LA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return LA_ERR_INVALID_ARG;
  const size_t es = dtype == LA_F32 ? 4 : 2;
  const size_t nqk = (size_t)rows * D * es, nv = (size_t)rows * Dv * es;
  if (overlaps(o, nv, q, nqk) || overlaps(o, nv, k, nqk) || overlaps(o, nv, v, nv))
    return LA_ERR_INVALID_ARG;
  // scratch plan: S, z for every head, plus nsplit partial copies when the
  // sequence is reduced in parallel pieces; use as many splits as fit
  const int BH = B * H;
  const size_t per_state = sizeof(float) * (size_t)BH * ((size_t)D * Dv + D);
  if (per_state > kScratchBytes) return LA_ERR_UNSUPPORTED;
  int nsplit = kv_state_num_splits(BH, N);
  while (nsplit > 1 && per_state * (1 + (size_t)nsplit) > kScratchBytes) --nsplit;

  float *scratch = scratch_on_current_device();  // first call on a device: one query
  if (!scratch) return LA_ERR_CUDA;
  float *S = scratch;
  float *z = S + (size_t)BH * D * Dv;
  float *part = nsplit > 1 ? z + (size_t)BH * D : nullptr;
  Gammas g;
  for (int h = 0; h < kMaxHeads; ++h) g.g[h] = 1.f;
  const Dtype dt = dtype == LA_F32 ? kF32 : kBF16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // every scratch word read below is written earlier on the same stream in
  // this call, so nothing has to be cleared between calls
  cudaError_t e = launch_kv_state_splits(k, v, S, z, part, B, H, N, D, Dv, nsplit, g, dt, s);
  if (e == cudaSuccess) e = launch_noncausal_apply(q, S, z, o, BH, N, D, Dv, eps, dt, s);
  if (e == cudaErrorNotSupported) return LA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // extern "C"
