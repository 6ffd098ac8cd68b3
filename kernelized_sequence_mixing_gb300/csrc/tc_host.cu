// Host-side support for the tensor-core kernels: TMA tensor-map encoding and
// the device counter of abandoned (timed-out) waits.
#include <cudaTypedefs.h>
#include <mutex>

#include "tc_common.cuh"

namespace linattn {

// Counts waits that gave up in any tensor-core kernel on this device.
__device__ unsigned int g_wait_timeouts = 0;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

bool make_tmap_3d_bf16(CUtensorMap *map, const void *base, uint64_t dim_x, uint64_t dim_y,
                       uint64_t dim_z, uint32_t box_x, uint32_t box_y, int swizzle_bytes) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {dim_x, dim_y, dim_z};
  const cuuint64_t strides[2] = {dim_x * 2, dim_x * dim_y * 2};  // bytes, dims 1..2
  const cuuint32_t box[3] = {box_x, box_y, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMapSwizzle sw;
  switch (swizzle_bytes) {
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; break;
    case 0: sw = CU_TENSOR_MAP_SWIZZLE_NONE; break;
    default: return false;
  }
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

unsigned int *wait_timeout_counter() {
  constexpr int kMaxDev = 64;
  static unsigned int *addr[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wait_timeouts) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned int *>(p);
  }
  return addr[dev];
}

namespace {

// One thread waits, with the kernels' own bounded wait, for phase 0 of an
// mbarrier that nothing arrives on; it gives up after `cycles`, counts
// itself once in the timeout counter and reports.
__global__ void wait_selftest_kernel(long long cycles, int *result, unsigned int *timeouts) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  abort_flag = 0;
  tc::mbar_init_fence();
  const bool ok = tc::mbar_wait_limit(&bar, 0, &abort_flag, timeouts, cycles);
  *result = ok ? 0 : 1;
}

}  // namespace

cudaError_t wait_selftest(long long cycles, int *gave_up) {
  unsigned int *ctr = wait_timeout_counter();
  if (!ctr) return cudaErrorInvalidValue;
  int *d = nullptr;
  cudaError_t e = cudaMalloc(&d, sizeof(int));
  if (e != cudaSuccess) return e;
  wait_selftest_kernel<<<1, 32>>>(cycles, d, ctr);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  int h = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&h, d, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e == cudaSuccess) *gave_up = h;
  return e;
}

}  // namespace linattn
