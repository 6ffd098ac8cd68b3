// C ABI of the library: argument validation, workspace and dispatch.
//
// Every check runs before the first CUDA call, so a rejected call has no side
// effect on the device or the stream.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/linattn.h"
#include "kernels.h"
#include "tc_common.cuh"

using namespace linattn;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

size_t elem_size(la_dtype_t dt) { return dt == LA_F32 ? 4 : 2; }

bool supported_dim(int d) { return d == 64 || d == 128; }

// Common size/type checks.  Returns LA_OK or the first failure.
la_status_t check_sizes(int B, int H, int N, int D, int Dv, la_dtype_t dt) {
  if (dt != LA_F32 && dt != LA_BF16) return LA_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || N < 0 || D <= 0 || Dv <= 0) return LA_ERR_INVALID_ARG;
  if (!supported_dim(D) || !supported_dim(Dv)) return LA_ERR_UNSUPPORTED;
  if (H > kMaxHeads) return LA_ERR_UNSUPPORTED;
  if ((int64_t)B * H * (int64_t)(N > 0 ? N : 1) >= ((int64_t)1 << 31))
    return LA_ERR_UNSUPPORTED;
  return LA_OK;
}

// gamma: NULL (all 1) or H values in [0, 1].  Fills g and reports whether any
// value differs from 1.
la_status_t load_gammas(const float *gamma, int H, Gammas *g, bool *decay) {
  *decay = false;
  for (int h = 0; h < kMaxHeads; ++h) g->g[h] = 1.f;
  if (!gamma) return LA_OK;
  for (int h = 0; h < H; ++h) {
    const float x = gamma[h];
    if (!(x >= 0.f && x <= 1.f)) return LA_ERR_INVALID_ARG;  // also NaN
    g->g[h] = x;
    if (x != 1.f) *decay = true;
  }
  return LA_OK;
}

la_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return LA_OK;
  if (e == cudaErrorNotSupported) return LA_ERR_UNSUPPORTED;
  return LA_ERR_CUDA;
}

la_status_t run_forward(const Problem &p, const Gammas &g, int causal, cudaStream_t s);
la_status_t run_forward_host(const void *q, const void *k, const void *v, void *o, int B, int H,
                             int N, int D, int Dv, int causal, const Gammas &g, float eps, Dtype dt,
                             cudaStream_t s);

}  // namespace

extern "C" {

int la_causal_kernel(int B, int H, int N, int D, int Dv, const float *gamma,
                     la_dtype_t dtype) {
  la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return -static_cast<int>(st);
  Gammas g;
  bool decay = false;
  if ((st = load_gammas(gamma, H, &g, &decay)) != LA_OK) return -static_cast<int>(st);
  Problem p{nullptr, nullptr, nullptr, nullptr, B, H, N, D, Dv, decay, 0.f,
            dtype == LA_F32 ? kF32 : kBF16};
  if (chunk128_supported(p, g)) return 2;
  return chunk_tc_supported(p, g) ? 1 : 0;
}

int la_device_wait_timeouts(int reset) {
  unsigned int *ctr = wait_timeout_counter();
  if (!ctr) return -1;
  unsigned int v = 0;
  if (cudaMemcpy(&v, ctr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  if (reset) {
    const unsigned int zero = 0;
    if (cudaMemcpy(ctr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return -1;
  }
  return static_cast<int>(v);
}

const char *la_status_string(la_status_t s) {
  switch (s) {
    case LA_OK: return "ok";
    case LA_ERR_INVALID_ARG: return "invalid argument";
    case LA_ERR_UNSUPPORTED: return "unsupported shape or size";
    case LA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

la_status_t la_forward(const void *q, const void *k, const void *v, void *o,
                       int B, int H, int N, int D, int Dv, int causal,
                       const float *gamma, float eps, la_dtype_t dtype,
                       void *stream) {
  la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return st;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  Gammas g;
  bool decay = false;
  if ((st = load_gammas(gamma, H, &g, &decay)) != LA_OK) return st;
  if (!causal && decay) return LA_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)B * H * N;
  if (rows == 0) return LA_OK;
  if (!q || !k || !v || !o) return LA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return LA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t nqk = (size_t)rows * D * es, nv = (size_t)rows * Dv * es;
  if (overlaps(o, nv, q, nqk) || overlaps(o, nv, k, nqk) || overlaps(o, nv, v, nv))
    return LA_ERR_INVALID_ARG;

  Problem p{q, k, v, o, B, H, N, D, Dv, decay, eps,
            dtype == LA_F32 ? kF32 : kBF16};
  return run_forward(p, g, causal, static_cast<cudaStream_t>(stream));
}

la_status_t la_forward_host(const void *q, const void *k, const void *v, void *o,
                            int B, int H, int N, int D, int Dv, int causal,
                            const float *gamma, float eps, la_dtype_t dtype,
                            void *stream) {
  la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return st;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  Gammas g;
  bool decay = false;
  if ((st = load_gammas(gamma, H, &g, &decay)) != LA_OK) return st;
  if (!causal && decay) return LA_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)B * H * N;
  if (rows == 0) return LA_OK;
  if (!q || !k || !v || !o) return LA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t nqk = (size_t)rows * D * es, nv = (size_t)rows * Dv * es;
  if (overlaps(o, nv, q, nqk) || overlaps(o, nv, k, nqk) || overlaps(o, nv, v, nv))
    return LA_ERR_INVALID_ARG;
  return run_forward_host(q, k, v, o, B, H, N, D, Dv, causal, g, eps, dtype == LA_F32 ? kF32 : kBF16,
                          static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// The forward pass of a validated problem: picks the kernel, takes and
// returns the stream-ordered workspace.  p.ident: q, k already are features.
la_status_t run_forward(const Problem &p, const Gammas &g, int causal, cudaStream_t s) {
  const int BH = p.B * p.H;
  const int N = p.N, D = p.D, Dv = p.Dv;
  const void *k = p.k, *v = p.v, *q = p.q;
  void *o = p.o;
  const float eps = p.eps;
  const int B = p.B, H = p.H;
  if (causal) {
    if (chunk128_supported(p, g)) {
      // 128-token chunks (D = Dv = 128); parts as below
      const int P = chunk128_parts(BH, N);
      const size_t wsb = chunk128_workspace_bytes(BH, P);
      void *ws = nullptr;
      if (wsb && cudaMallocAsync(&ws, wsb, s) != cudaSuccess) return LA_ERR_CUDA;
      cudaError_t e = launch_causal_chunk128(p, g, ws, P, s);
      cudaError_t ef = ws ? cudaFreeAsync(ws, s) : cudaSuccess;
      if (e != cudaSuccess) return from_cuda(e);
      return from_cuda(ef);
    }
    if (chunk_tc_supported(p, g)) {
      // parts of the sequence run on separate SMs; the workspace carries the
      // state from one part to the next
      const int P = chunk_parts(BH, N);
      const size_t wsb = chunk_causal_workspace_bytes(BH, P, D, Dv);
      void *ws = nullptr;
      if (wsb && cudaMallocAsync(&ws, wsb, s) != cudaSuccess) return LA_ERR_CUDA;
      cudaError_t e = launch_causal_chunk(p, g, ws, P, s);
      cudaError_t ef = ws ? cudaFreeAsync(ws, s) : cudaSuccess;
      if (e != cudaSuccess) return from_cuda(e);
      return from_cuda(ef);
    }
    return from_cuda(launch_causal_simt(p, g, s));
  }
  // Non-causal: reduce S, z per (b, h) into a stream-ordered workspace, then
  // apply them to every query (bf16: persistent tensor-core passes).
  if (noncausal_tc_supported(p)) {
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, noncausal_tc_workspace_bytes(p), s) != cudaSuccess) return LA_ERR_CUDA;
    cudaError_t e = launch_noncausal_tc(p, ws, s);
    cudaError_t ef = cudaFreeAsync(ws, s);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(ef);
  }
  const size_t state_bytes = sizeof(float) * (size_t)BH * ((size_t)D * Dv + D);
  const size_t part_bytes = kv_state_workspace_bytes(BH, N, D, Dv);
  void *ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, state_bytes + part_bytes, s);
  if (e != cudaSuccess) return LA_ERR_CUDA;
  float *S = static_cast<float *>(ws);
  float *z = S + (size_t)BH * D * Dv;
  float *part = part_bytes ? z + (size_t)BH * D : nullptr;
  e = launch_kv_state(k, v, S, z, part, B, H, N, D, Dv, false, g, p.dtype, s, p.ident);
  if (e == cudaSuccess)
    e = launch_noncausal_apply(q, S, z, o, BH, N, D, Dv, eps, p.dtype, s, p.ident);
  cudaError_t ef = cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(ef);
}

// Copy streams of the current device for la_forward_host, created once and
// kept until the process exits.
bool copy_streams(cudaStream_t *up, cudaStream_t *down) {
  constexpr int kMaxDev = 64;
  static cudaStream_t ups[kMaxDev] = {}, downs[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!ups[dev]) {
    cudaStream_t a = nullptr, b = nullptr;
    if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess) {
      cudaStreamDestroy(a);
      return false;
    }
    ups[dev] = a;
    downs[dev] = b;
  }
  *up = ups[dev];
  *down = downs[dev];
  return true;
}

// The device-memory pool of la_forward_host's buffers on the current
// device: created once, it keeps released memory for the next call (a
// release threshold of "never"), so that a call does not map its buffers
// anew each time.
cudaMemPool_t host_path_pool() {
  constexpr int kMaxDev = 64;
  static cudaMemPool_t pools[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t keep = UINT64_MAX;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return nullptr;
    }
    pools[dev] = pool;
  }
  return pools[dev];
}

// Host buffers in, host buffer out, in groups of heads: group g's inputs go
// up on one copy stream, its forward runs on `s` once they have landed, its
// output comes down on a second copy stream once the forward is done, so
// that the uploads, the kernels and the downloads of different groups
// overlap.  A group is a run of heads of one batch entry (so each keeps its
// decays); device buffers for the whole problem are stream-ordered
// allocations on `s` from the library's pool, released on `s` after the
// last download.
la_status_t run_forward_host(const void *q, const void *k, const void *v, void *o, int B, int H,
                             int N, int D, int Dv, int causal, const Gammas &g, float eps, Dtype dt,
                             cudaStream_t s) {
  cudaStream_t up = nullptr, down = nullptr;
  if (!copy_streams(&up, &down)) return LA_ERR_CUDA;
  cudaMemPool_t pool = host_path_pool();
  if (!pool) return LA_ERR_CUDA;
  const size_t es = dt == kF32 ? 4 : 2;
  const size_t head_qk = (size_t)N * D * es, head_v = (size_t)N * Dv * es;
  const size_t nqk = (size_t)B * H * head_qk, nvv = (size_t)B * H * head_v;
  // about eight groups: enough to overlap, few enough that each forward
  // still spreads over the SMs
  const int groups_target = 8;
  int hs = (B * H + groups_target - 1) / groups_target;
  if (hs > H) hs = H;
  if (hs < 1) hs = 1;
  const int gpb = (H + hs - 1) / hs;  // groups per batch entry
  const int G = B * gpb;
  uint8_t *dbuf = nullptr;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void **>(&dbuf), 2 * nqk + 2 * nvv, pool, s) != cudaSuccess)
    return LA_ERR_CUDA;
  uint8_t *dq = dbuf, *dk = dq + nqk, *dv = dk + nqk, *dout = dv + nvv;
  std::vector<cudaEvent_t> ev(2 * G + 2, nullptr);
  la_status_t st = LA_OK;
  for (auto &e : ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) st = LA_ERR_CUDA;
  cudaEvent_t ev_alloc = ev[2 * G], ev_done = ev[2 * G + 1];
  auto ok = [&](cudaError_t e) {
    if (e != cudaSuccess && st == LA_OK) st = LA_ERR_CUDA;
    return st == LA_OK;
  };
  if (st == LA_OK && ok(cudaEventRecord(ev_alloc, s)) && ok(cudaStreamWaitEvent(up, ev_alloc, 0)) &&
      ok(cudaStreamWaitEvent(down, ev_alloc, 0))) {
    auto range = [&](int gi, int *b, int *h0, int *nh) {
      *b = gi / gpb;
      *h0 = (gi % gpb) * hs;
      *nh = H - *h0 < hs ? H - *h0 : hs;
    };
    // uploads, in group order
    for (int gi = 0; gi < G && st == LA_OK; ++gi) {
      int b, h0, nh;
      range(gi, &b, &h0, &nh);
      const size_t u0 = (size_t)b * H + h0;
      ok(cudaMemcpyAsync(dq + u0 * head_qk, static_cast<const uint8_t *>(q) + u0 * head_qk, nh * head_qk,
                         cudaMemcpyHostToDevice, up));
      ok(cudaMemcpyAsync(dk + u0 * head_qk, static_cast<const uint8_t *>(k) + u0 * head_qk, nh * head_qk,
                         cudaMemcpyHostToDevice, up));
      ok(cudaMemcpyAsync(dv + u0 * head_v, static_cast<const uint8_t *>(v) + u0 * head_v, nh * head_v,
                         cudaMemcpyHostToDevice, up));
      ok(cudaEventRecord(ev[gi], up));
    }
    // each group's forward once its inputs are on the device, then its download
    for (int gi = 0; gi < G && st == LA_OK; ++gi) {
      int b, h0, nh;
      range(gi, &b, &h0, &nh);
      const size_t u0 = (size_t)b * H + h0;
      if (!ok(cudaStreamWaitEvent(s, ev[gi], 0))) break;
      Gammas gg;
      for (int h = 0; h < kMaxHeads; ++h) gg.g[h] = h < nh ? g.g[h0 + h] : 1.f;
      bool gdecay = false;
      for (int h = 0; h < nh; ++h) gdecay = gdecay || gg.g[h] != 1.f;
      Problem pg{dq + u0 * head_qk, dk + u0 * head_qk, dv + u0 * head_v, dout + u0 * head_v, 1, nh, N,
                 D, Dv, gdecay, eps, dt};
      const la_status_t fs = run_forward(pg, gg, causal, s);
      if (fs != LA_OK) {
        st = fs;
        break;
      }
      if (!ok(cudaEventRecord(ev[G + gi], s)) || !ok(cudaStreamWaitEvent(down, ev[G + gi], 0))) break;
      ok(cudaMemcpyAsync(static_cast<uint8_t *>(o) + u0 * head_v, dout + u0 * head_v, nh * head_v,
                         cudaMemcpyDeviceToHost, down));
    }
  }
  // the caller's stream waits for every download before the buffers are
  // released (and before its own later work)
  if (ev_done && cudaEventRecord(ev_done, down) == cudaSuccess) cudaStreamWaitEvent(s, ev_done, 0);
  if (cudaFreeAsync(dbuf, s) != cudaSuccess && st == LA_OK) st = LA_ERR_CUDA;
  for (auto &e : ev)
    if (e) cudaEventDestroy(e);  // released once the work they mark is done
  return st;
}

}  // namespace

extern "C" {

la_status_t la_prefill_state(const void *k, const void *v, float *S, float *z,
                             int B, int H, int N, int D, int Dv,
                             const float *gamma, la_dtype_t dtype,
                             void *stream) {
  la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return st;
  Gammas g;
  bool decay = false;
  if ((st = load_gammas(gamma, H, &g, &decay)) != LA_OK) return st;
  const int BH = B * H;
  if (BH == 0) return LA_OK;
  if (!S || !z || !aligned16(S) || !aligned16(z)) return LA_ERR_INVALID_ARG;
  const size_t nS = sizeof(float) * (size_t)BH * D * Dv, nz = sizeof(float) * (size_t)BH * D;
  if (overlaps(S, nS, z, nz)) return LA_ERR_INVALID_ARG;
  if (N > 0) {
    if (!k || !v || !aligned16(k) || !aligned16(v)) return LA_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    const size_t nk = (size_t)BH * N * D * es, nv = (size_t)BH * N * Dv * es;
    if (overlaps(S, nS, k, nk) || overlaps(S, nS, v, nv) ||
        overlaps(z, nz, k, nk) || overlaps(z, nz, v, nv))
      return LA_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Problem pr{nullptr, k, v, nullptr, B, H, N, D, Dv, decay, 0.f,
                   dtype == LA_F32 ? kF32 : kBF16};
  if (N > 0 && chunk_tc_supported(pr, g)) {
    // tensor cores: per-part sums, then a scan over the parts
    const int P = chunk_state_parts(BH, N, D, Dv);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, chunk_workspace_bytes(BH, P, D, Dv), s) != cudaSuccess)
      return LA_ERR_CUDA;
    cudaError_t e = launch_prefill_chunk(k, v, S, z, B, H, N, D, Dv, decay, g, ws, P, s);
    cudaError_t ef = cudaFreeAsync(ws, s);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(ef);
  }
  const size_t part_bytes = kv_state_workspace_bytes(BH, N, D, Dv);
  void *ws = nullptr;
  if (part_bytes) {
    if (cudaMallocAsync(&ws, part_bytes, s) != cudaSuccess) return LA_ERR_CUDA;
  }
  cudaError_t e = launch_kv_state(k, v, S, z, static_cast<float *>(ws), B, H,
                                  N, D, Dv, decay, g,
                                  dtype == LA_F32 ? kF32 : kBF16, s);
  cudaError_t ef = ws ? cudaFreeAsync(ws, s) : cudaSuccess;
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(ef);
}

la_status_t la_forward_state(const void *q, const void *k, const void *v, void *o,
                             float *S, float *z, int B, int H, int N, int D, int Dv,
                             const float *gamma, float eps, la_dtype_t dtype,
                             void *stream) {
  la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return st;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  Gammas g;
  bool decay = false;
  if ((st = load_gammas(gamma, H, &g, &decay)) != LA_OK) return st;
  const int BH = B * H;
  if (BH == 0) return LA_OK;
  if (!S || !z || !aligned16(S) || !aligned16(z)) return LA_ERR_INVALID_ARG;
  const size_t nS = sizeof(float) * (size_t)BH * D * Dv, nz = sizeof(float) * (size_t)BH * D;
  if (overlaps(S, nS, z, nz)) return LA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    if (cudaMemsetAsync(S, 0, nS, s) != cudaSuccess || cudaMemsetAsync(z, 0, nz, s) != cudaSuccess)
      return LA_ERR_CUDA;
    return LA_OK;
  }
  if (!q || !k || !v || !o) return LA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return LA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t nqk = (size_t)BH * N * D * es, nv = (size_t)BH * N * Dv * es;
  const void *ins[4] = {q, k, v, o};
  const size_t insz[4] = {nqk, nqk, nv, nv};
  for (int i = 0; i < 4; ++i)
    if (overlaps(S, nS, ins[i], insz[i]) || overlaps(z, nz, ins[i], insz[i])) return LA_ERR_INVALID_ARG;
  if (overlaps(o, nv, q, nqk) || overlaps(o, nv, k, nqk) || overlaps(o, nv, v, nv))
    return LA_ERR_INVALID_ARG;
  Problem p{q, k, v, o, B, H, N, D, Dv, decay, eps, dtype == LA_F32 ? kF32 : kBF16};
  if (chunk128_supported(p, g)) {
    // one pass: the CTA of the last part writes the state
    const int P = chunk128_parts(BH, N);
    const size_t wsb = chunk128_workspace_bytes(BH, P);
    void *ws = nullptr;
    if (wsb && cudaMallocAsync(&ws, wsb, s) != cudaSuccess) return LA_ERR_CUDA;
    cudaError_t e = launch_causal_chunk128(p, g, ws, P, s, S, z);
    cudaError_t ef = ws ? cudaFreeAsync(ws, s) : cudaSuccess;
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(ef);
  }
  if ((st = la_forward(q, k, v, o, B, H, N, D, Dv, 1, gamma, eps, dtype, stream)) != LA_OK) return st;
  return la_prefill_state(k, v, S, z, B, H, N, D, Dv, gamma, dtype, stream);
}

la_status_t la_decode_step(const void *q, const void *k, const void *v,
                           float *S, float *z, void *o, int B, int H, int D,
                           int Dv, const float *gamma, float eps,
                           la_dtype_t dtype, void *stream) {
  la_status_t st = check_sizes(B, H, 1, D, Dv, dtype);
  if (st != LA_OK) return st;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  Gammas g;
  bool decay = false;
  if ((st = load_gammas(gamma, H, &g, &decay)) != LA_OK) return st;
  const int BH = B * H;
  if (BH == 0) return LA_OK;
  if (!q || !k || !v || !S || !z || !o) return LA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(S) ||
      !aligned16(z) || !aligned16(o))
    return LA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const void *ptr[6] = {q, k, v, S, z, o};
  const size_t len[6] = {(size_t)BH * D * es, (size_t)BH * D * es,
                         (size_t)BH * Dv * es, sizeof(float) * (size_t)BH * D * Dv,
                         sizeof(float) * (size_t)BH * D, (size_t)BH * Dv * es};
  // the written buffers (S, z, o) may overlap nothing
  for (int w = 3; w < 6; ++w)
    for (int i = 0; i < 6; ++i)
      if (i != w && overlaps(ptr[w], len[w], ptr[i], len[i])) return LA_ERR_INVALID_ARG;
  return from_cuda(launch_decode_step(q, k, v, S, z, o, B, H, D, Dv, decay, g,
                                      eps, dtype == LA_F32 ? kF32 : kBF16,
                                      static_cast<cudaStream_t>(stream)));
}

la_status_t la_forward_gated(const void *q, const void *k, const void *v, const float *a,
                             void *o, float *S, float *z, int B, int H, int N, int D, int Dv,
                             float eps, la_dtype_t dtype, void *stream) {
  la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return st;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  if ((S == nullptr) != (z == nullptr)) return LA_ERR_INVALID_ARG;
  const int BH = B * H;
  if (BH == 0) return LA_OK;
  const size_t nS = sizeof(float) * (size_t)BH * D * Dv, nz = sizeof(float) * (size_t)BH * D;
  if (S) {
    if (!aligned16(S) || !aligned16(z) || overlaps(S, nS, z, nz)) return LA_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    if (S && (cudaMemsetAsync(S, 0, nS, s) != cudaSuccess || cudaMemsetAsync(z, 0, nz, s) != cudaSuccess))
      return LA_ERR_CUDA;
    return LA_OK;
  }
  if (!q || !k || !v || !a || !o) return LA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || !aligned16(o))
    return LA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t nqk = (size_t)BH * N * D * es, nv = (size_t)BH * N * Dv * es;
  const size_t na = sizeof(float) * (size_t)BH * N * D;
  const void *ins[4] = {q, k, v, a};
  const size_t insz[4] = {nqk, nqk, nv, na};
  for (int i = 0; i < 4; ++i) {
    if (overlaps(o, nv, ins[i], insz[i])) return LA_ERR_INVALID_ARG;
    if (S && (overlaps(S, nS, ins[i], insz[i]) || overlaps(z, nz, ins[i], insz[i])))
      return LA_ERR_INVALID_ARG;
  }
  if (S && (overlaps(S, nS, o, nv) || overlaps(z, nz, o, nv))) return LA_ERR_INVALID_ARG;
  const Problem p{q, k, v, o, B, H, N, D, Dv, false, eps, dtype == LA_F32 ? kF32 : kBF16};
  const int P = gla_parts(BH, N, Dv);
  const size_t wsb_simt = (gla_workspace_bytes(BH, P, D, Dv) + 255) & ~(size_t)255;
  const bool tc = gla_tc_supported(p);
  const size_t wsb = wsb_simt + (tc ? gla_tc_workspace_bytes(BH, N) : 0);
  void *ws = nullptr;
  if (wsb && cudaMallocAsync(&ws, wsb, s) != cudaSuccess) return LA_ERR_CUDA;
  cudaError_t e = cudaSuccess;
  const int *hard = nullptr;
  if (tc) {
    // tensor cores; the CUDA-core form runs after it only if some chunk
    // forgot too hard for the scaled operands (a device flag decides)
    e = launch_gla_tc(p, a, static_cast<uint8_t *>(ws) + wsb_simt, s, &hard, S, z);
  }
  if (e == cudaSuccess) e = launch_gla_simt(p, a, ws, P, S, z, s, hard);
  cudaError_t ef = ws ? cudaFreeAsync(ws, s) : cudaSuccess;
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(ef);
}

int la_gated_kernel(int B, int H, int N, int D, int Dv, la_dtype_t dtype, int want_state) {
  const la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return -static_cast<int>(st);
  const Problem p{nullptr, nullptr, nullptr, nullptr, B, H, N, D, Dv, false, 0.f,
                  dtype == LA_F32 ? kF32 : kBF16};
  (void)want_state;  // the tensor-core form writes the final state as well
  return gla_tc_supported(p) ? 1 : 0;
}

la_status_t la_decode_gated(const void *q, const void *k, const void *v, const float *a,
                            float *S, float *z, void *o, int B, int H, int D, int Dv, float eps,
                            la_dtype_t dtype, void *stream) {
  la_status_t st = check_sizes(B, H, 1, D, Dv, dtype);
  if (st != LA_OK) return st;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  const int BH = B * H;
  if (BH == 0) return LA_OK;
  if (!q || !k || !v || !a || !S || !z || !o) return LA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || !aligned16(S) ||
      !aligned16(z) || !aligned16(o))
    return LA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const void *ptr[7] = {q, k, v, a, S, z, o};
  const size_t len[7] = {(size_t)BH * D * es, (size_t)BH * D * es, (size_t)BH * Dv * es,
                         sizeof(float) * (size_t)BH * D, sizeof(float) * (size_t)BH * D * Dv,
                         sizeof(float) * (size_t)BH * D, (size_t)BH * Dv * es};
  // the written buffers (S, z, o) may overlap nothing
  for (int w = 4; w < 7; ++w)
    for (int i = 0; i < 7; ++i)
      if (i != w && overlaps(ptr[w], len[w], ptr[i], len[i])) return LA_ERR_INVALID_ARG;
  return from_cuda(launch_decode_gated(q, k, v, a, S, z, o, B, H, D, Dv, eps,
                                       dtype == LA_F32 ? kF32 : kBF16,
                                       static_cast<cudaStream_t>(stream)));
}

la_status_t la_favor_features(const void *x, const void *W, void *phi, int rows, int D,
                              int r, la_dtype_t dtype, void *stream) {
  if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
  if (rows < 0 || D <= 0 || r <= 0) return LA_ERR_INVALID_ARG;
  if (!supported_dim(D) || !supported_dim(r)) return LA_ERR_UNSUPPORTED;
  if (rows == 0) return LA_OK;
  if (!x || !W || !phi || !aligned16(x) || !aligned16(W) || !aligned16(phi))
    return LA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t nx = (size_t)rows * D * es, nW = (size_t)r * D * es, nf = (size_t)rows * r * es;
  if (overlaps(phi, nf, x, nx) || overlaps(phi, nf, W, nW)) return LA_ERR_INVALID_ARG;
  return from_cuda(launch_favor_features(x, nullptr, W, phi, nullptr, rows, D, r,
                                         dtype == LA_F32 ? kF32 : kBF16,
                                         static_cast<cudaStream_t>(stream)));
}

la_status_t la_forward_favor(const void *q, const void *k, const void *v, const void *W, void *o,
                             int B, int H, int N, int D, int Dv, int r, int causal,
                             const float *gamma, float eps, la_dtype_t dtype, void *stream) {
  la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return st;
  if (r <= 0) return LA_ERR_INVALID_ARG;
  if (!supported_dim(r)) return LA_ERR_UNSUPPORTED;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  Gammas g;
  bool decay = false;
  if ((st = load_gammas(gamma, H, &g, &decay)) != LA_OK) return st;
  if (!causal && decay) return LA_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)B * H * N;
  if (rows == 0) return LA_OK;
  if (!q || !k || !v || !W || !o) return LA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(W) || !aligned16(o))
    return LA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t nqk = (size_t)rows * D * es, nv = (size_t)rows * Dv * es, nW = (size_t)r * D * es;
  if (overlaps(o, nv, q, nqk) || overlaps(o, nv, k, nqk) || overlaps(o, nv, v, nv) ||
      overlaps(o, nv, W, nW))
    return LA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dtype dt = dtype == LA_F32 ? kF32 : kBF16;
  // the features of q and k, [B][H][N][r] each, in a stream-ordered workspace
  const size_t nf = (((size_t)rows * r * es) + 255) & ~(size_t)255;
  void *ws = nullptr;
  if (cudaMallocAsync(&ws, 2 * nf, s) != cudaSuccess) return LA_ERR_CUDA;
  void *fq = ws, *fk = static_cast<uint8_t *>(ws) + nf;
  la_status_t out = from_cuda(launch_favor_features(q, k, W, fq, fk, rows, D, r, dt, s));
  if (out == LA_OK) {
    Problem p{fq, fk, v, o, B, H, N, r, Dv, decay, eps, dt};
    p.ident = true;
    out = run_forward(p, g, causal, s);
  }
  const cudaError_t ef = cudaFreeAsync(ws, s);
  if (out != LA_OK) return out;
  return from_cuda(ef);
}

la_status_t la_backward(const void *q, const void *k, const void *v, const void *dO, void *dq,
                        void *dk, void *dv, int B, int H, int N, int D, int Dv,
                        const float *gamma, float eps, la_dtype_t dtype, void *stream) {
  la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return st;
  if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
  Gammas g;
  bool decay = false;
  if ((st = load_gammas(gamma, H, &g, &decay)) != LA_OK) return st;
  const int64_t rows = (int64_t)B * H * N;
  if (rows == 0) return LA_OK;
  const void *ins[4] = {q, k, v, dO};
  void *outs[3] = {dq, dk, dv};
  for (const void *x : ins)
    if (!x || !aligned16(x)) return LA_ERR_INVALID_ARG;
  for (void *x : outs)
    if (!x || !aligned16(x)) return LA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t nqk = (size_t)rows * D * es, nv = (size_t)rows * Dv * es;
  const size_t insz[4] = {nqk, nqk, nv, nv};
  const size_t outsz[3] = {nqk, nqk, nv};
  // the gradients may overlap no input and no other gradient
  for (int w = 0; w < 3; ++w) {
    for (int i = 0; i < 4; ++i)
      if (overlaps(outs[w], outsz[w], ins[i], insz[i])) return LA_ERR_INVALID_ARG;
    for (int u = w + 1; u < 3; ++u)
      if (overlaps(outs[w], outsz[w], outs[u], outsz[u])) return LA_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Problem p{q, k, v, nullptr, B, H, N, D, Dv, decay, eps, dtype == LA_F32 ? kF32 : kBF16};
  // tensor cores for bf16 with Dv = 64 inside the chunk kernel's decay
  // envelope; the fp32 CUDA-core kernels otherwise
  const bool tc = backward_tc_supported(p, g);
  void *ws = nullptr;
  const size_t wsb = tc ? backward_tc_workspace_bytes(B * H, N, D) : backward_workspace_bytes(B * H, N, D, Dv);
  if (cudaMallocAsync(&ws, wsb, s) != cudaSuccess) return LA_ERR_CUDA;
  const cudaError_t e = tc ? launch_backward_tc(p, dO, dq, dk, dv, g, ws, s)
                           : launch_backward(p, dO, dq, dk, dv, g, ws, s);
  const cudaError_t ef = cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(ef);
}

int la_backward_kernel(int B, int H, int N, int D, int Dv, const float *gamma, la_dtype_t dtype) {
  la_status_t st = check_sizes(B, H, N, D, Dv, dtype);
  if (st != LA_OK) return -static_cast<int>(st);
  Gammas g;
  bool decay = false;
  if ((st = load_gammas(gamma, H, &g, &decay)) != LA_OK) return -static_cast<int>(st);
  const Problem p{nullptr, nullptr, nullptr, nullptr, B, H, N > 0 ? N : 1, D, Dv, decay, 0.f,
                  dtype == LA_F32 ? kF32 : kBF16};
  return backward_tc_supported(p, g) ? 1 : 0;
}

int la_backward_launches(int B, int H, int N, int D, int Dv, const float *gamma, la_dtype_t dtype) {
  const int path = la_backward_kernel(B, H, N, D, Dv, gamma, dtype);
  if (path < 0) return path;
  if ((int64_t)B * H * N == 0) return 0;
  return path == 1 ? backward_tc_launches() : backward_launches(B * H, N, D, Dv);
}

la_status_t la_wait_selftest(long long cycles, int *gave_up) {
  if (!gave_up || cycles <= 0 || cycles > 4000000000LL) return LA_ERR_INVALID_ARG;
  return from_cuda(wait_selftest(cycles, gave_up));
}

}  // extern "C"
