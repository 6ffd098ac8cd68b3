// Host-side launchers of the library's kernels (internal to the library).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace linattn {

constexpr int kMaxHeads = 256;

// Per-head decay values, passed to kernels by value.
struct Gammas {
  float g[kMaxHeads];
};

enum Dtype { kF32 = 0, kBF16 = 1 };

struct Problem {
  const void *q, *k, *v;
  void *o;
  int B, H, N, D, Dv;
  bool decay;  // any gamma != 1
  float eps;
  Dtype dtype;
  // q, k already are features (the Performer path computes them first): the
  // kernels use them as they are instead of applying phi = elu + 1
  bool ident = false;
};

// First chunk of part p when nch chunks split into P equal parts (the
// 128-token kernel's split; the gated form's gate tables follow it).
__host__ __device__ inline int chunk_part_begin(int p, int P, int nch) {
  if (p <= 0) return 0;
  if (p >= P) return nch;
  const int base = nch / P, rem = nch % P;
  return p * base + (p < rem ? p : rem);
}

// Causal forward on CUDA cores (fp32 FFMA): any dtype.
cudaError_t launch_causal_simt(const Problem &p, const Gammas &g,
                               cudaStream_t s);

// Sequence-parallel chunked kernels on tcgen05 tensor cores (bf16 operands,
// fp32 state).  chunk_tc_supported() gives the envelope (bf16, D and Dv in
// {64, 128}, every decay >= 0.35); chunk_parts() the number of parts per
// (batch, head); chunk_workspace_bytes() the fp32 per-part records for that
// many parts (prefill, non-causal) and chunk_causal_workspace_bytes() the
// causal launcher's workspace (flags and inclusive states; 0 for one part).
bool chunk_tc_supported(const Problem &p, const Gammas &g);
int chunk_parts(int BH, int N);        // causal
int chunk_state_parts(int BH, int N, int D, int Dv);  // prefill, non-causal
size_t chunk_workspace_bytes(int BH, int P, int D, int Dv);
size_t chunk_causal_workspace_bytes(int BH, int P, int D, int Dv);
Gammas log2_gammas(const Gammas &g, int H, bool decay);
cudaError_t launch_causal_chunk(const Problem &p, const Gammas &g, void *ws, int P,
                                cudaStream_t s);
// The causal chunk kernel with another epilogue in place of o = numerators /
// (normaliser + eps) (p.o unused): out_raw [B*H][N][Dv] and den_raw [B*H][N]
// fp32, the undivided numerators and normalisers; or grad_out [B*H][N][Dv]
// bf16, the numerators times phi'(grad_in) elementwise (factor 1 when
// grad_in is null), at row N - 1 - t for rev (a product over token-reversed
// operands stored back in token order).
struct ChunkEpilogue {
  float *out_raw, *den_raw;
  __nv_bfloat16 *grad_out;
  const __nv_bfloat16 *grad_in;
  int rev;
};
// Non-causal forward on tensor cores with persistent streaming kernels
// (noncausal_tc.cu): bf16, D and Dv in {64, 128}, no decay.  A reduce pass
// writes per-part [S | z] records (noncausal_tc_workspace_bytes()), a scan
// sums them, an apply pass writes o.
bool noncausal_tc_supported(const Problem &p);
size_t noncausal_tc_workspace_bytes(const Problem &p);
cudaError_t launch_noncausal_tc(const Problem &p, void *ws, cudaStream_t s);
cudaError_t launch_causal_chunk_epilogue(const Problem &p, const Gammas &g, void *ws, int P,
                                         cudaStream_t s, const ChunkEpilogue &ep);
// The causal kernel with 128-token chunks for D = Dv = 128 (chunk128.cu):
// bf16, every decay >= 0.61; workspace (flags and inclusive states) for P
// parts, 0 for one part.
bool chunk128_supported(const Problem &p, const Gammas &g);
int chunk128_parts(int BH, int N);
size_t chunk128_workspace_bytes(int BH, int P);
// S_out, z_out (optional, both or neither): the state after the last token,
// [B*H][D][Dv] and [B*H][D] fp32.
cudaError_t launch_causal_chunk128(const Problem &p, const Gammas &g, void *ws, int P,
                                   cudaStream_t s, float *S_out = nullptr,
                                   float *z_out = nullptr);
// Final state S [BH][D][Dv], z [BH][D] of the causal recurrence over N tokens.
cudaError_t launch_prefill_chunk(const void *k, const void *v, float *S, float *z, int B, int H,
                                 int N, int D, int Dv, bool decay, const Gammas &g, void *ws,
                                 int P, cudaStream_t s);

// Scan over per-part records [BH][P][D*Dv + D] (part_scan.cu): kScanStarts
// turns A_p into the state before part p in place; kScanFinal writes the
// state after all parts to S_out, z_out; kScanSum writes sum_p A_p to slot 0.
enum ScanMode { kScanStarts = 0, kScanFinal = 1, kScanSum = 2 };
cudaError_t launch_part_scan(float *rec, int BH, int H, int P, int N, int D, int Dv,
                             const Gammas &lg, int mode, float *S_out, float *z_out,
                             cudaStream_t s);

// Split-N reduction of S = sum_j w_j phi(k_j) v_j^T and z = sum_j w_j
// phi(k_j) with w_j = gamma^(N-1-j): partials [nsplit][BH][D*Dv + D] in
// `partials` (fp32) unless nsplit == 1, in which case S, z are written
// directly.  Then a fixed-order reduction into S [BH][D][Dv], z [BH][D].
int kv_state_num_splits(int BH, int N);
size_t kv_state_workspace_bytes(int BH, int N, int D, int Dv);
// ident: k already holds features (no phi).
cudaError_t launch_kv_state(const void *k, const void *v, float *S, float *z,
                            float *partials, int B, int H, int N, int D,
                            int Dv, bool decay, const Gammas &g, Dtype dt,
                            cudaStream_t s, bool ident = false);

// The same reduction (no decay) with a caller-chosen number of splits
// (partials [nsplit][BH][D*Dv + D] in `partials` when nsplit > 1).
cudaError_t launch_kv_state_splits(const void *k, const void *v, float *S, float *z,
                                   float *partials, int B, int H, int N, int D, int Dv,
                                   int nsplit, const Gammas &g, Dtype dt, cudaStream_t s);

// o = phi(q) S / (phi(q) . z + eps) for every row, S and z per (b, h).
cudaError_t launch_noncausal_apply(const void *q, const float *S,
                                   const float *z, void *o, int BH, int N,
                                   int D, int Dv, float eps, Dtype dt,
                                   cudaStream_t s, bool ident = false);

// One decode step in place on S, z.
cudaError_t launch_decode_step(const void *q, const void *k, const void *v,
                               float *S, float *z, void *o, int B, int H,
                               int D, int Dv, bool decay, const Gammas &g,
                               float eps, Dtype dt, cudaStream_t s);

// One gated decode step in place on S, z: row d of S and z[d] scaled by
// a[(b, h)][d] (fp32 gates in [0, 1]) before the update.
cudaError_t launch_decode_gated(const void *q, const void *k, const void *v, const float *a,
                                float *S, float *z, void *o, int B, int H, int D, int Dv,
                                float eps, Dtype dt, cudaStream_t s);

// Gated causal forward on CUDA cores (gla_simt.cu): gates a [B*H][N][D] fp32
// in [0, 1], one per key feature and token.  gla_parts() gives the number of
// sequence parts, gla_workspace_bytes() the per-part records (0 for one
// part).  S_out, z_out (optional, both or neither): the state after the last
// token, [B*H][D][Dv] and [B*H][D] fp32.
int gla_parts(int BH, int N, int Dv);
size_t gla_workspace_bytes(int BH, int P, int D, int Dv);
// only_if (optional): the kernels do nothing unless *only_if is nonzero
cudaError_t launch_gla_simt(const Problem &p, const float *a, void *ws, int P, float *S_out,
                            float *z_out, cudaStream_t s, const int *only_if = nullptr);
// The gated tensor-core form (bf16, D = Dv = 128, B*H >= 8; S_out, z_out
// optional, the state after the last token):
// a prep kernel scales q, k per 128-token chunk by gate suffix products,
// then the 128-token causal kernel runs with one part per (batch, head) and
// rescales its state by each chunk's gate products.  *hard_out receives a
// device flag that is nonzero when some chunk forgets too hard for this form
// (the causal kernel then does nothing and the caller runs the CUDA-core
// form with only_if = the flag).
bool gla_tc_supported(const Problem &p);
size_t gla_tc_workspace_bytes(int BH, int N);
cudaError_t launch_gla_tc(const Problem &p, const float *a, void *ws, cudaStream_t s,
                          const int **hard_out, float *S_out = nullptr, float *z_out = nullptr);
// gate_suf / gate_part: see gla_tc (P > 1); ws: chunk128_workspace_bytes(BH, P)
cudaError_t launch_gated_chunk128(const Problem &p, const float *gate_prod, const float *gate_suf,
                                  const float *gate_part, const int *skip, void *ws, int P,
                                  cudaStream_t s, float *S_out = nullptr, float *z_out = nullptr);

// Performer random-feature map (favor.cu): fq = phi(q), fk = phi(k) for
// `rows` rows of q and k [rows][D], directions W [R][D], outputs [rows][R],
// all of dtype dt; phi(x) = R^(-1/2) exp(W x - |x|^2 / 2).  D, R in {64, 128}.
// k = nullptr: q only (fk unused).
cudaError_t launch_favor_features(const void *q, const void *k, const void *W, void *fq,
                                  void *fk, long long rows, int D, int R, Dtype dt,
                                  cudaStream_t s);

// Backward of the causal form (backward_simt.cu): dq, dk, dv (dtype of p)
// from q, k, v of p and the upstream gradient dO [B*H][N][Dv]; fp32 on CUDA
// cores in a workspace of backward_workspace_bytes().
size_t backward_workspace_bytes(int BH, int N, int D, int Dv);
int backward_launches(int BH, int N, int D, int Dv);  // kernels one call launches
cudaError_t launch_backward(const Problem &p, const void *dO, void *dq, void *dk, void *dv,
                            const Gammas &g, void *ws, cudaStream_t s);
// The same on tensor cores (backward_tc.cu) for bf16, Dv = 64, D in {64,
// 128} and the 64-token chunk kernel's decay envelope: the forward's
// undivided n and d, a prep kernel, three gradient products.
bool backward_tc_supported(const Problem &p, const Gammas &g);
size_t backward_tc_workspace_bytes(int BH, int N, int D);
int backward_tc_launches();
cudaError_t launch_backward_tc(const Problem &p, const void *dO, void *dq, void *dk, void *dv,
                               const Gammas &g, void *ws, cudaStream_t s);

}  // namespace linattn
