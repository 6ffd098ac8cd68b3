// Causal linear attention with 128-token chunks, D = Dv = 128, on tcgen05
// tensor cores (sm_103a).
//
// Method: the recurrence of "Linear Attention Mechanisms" (dileepadev.github.io),
// "Recurrent Reformulation", S_i = gamma S_(i-1) + phi(k_i) v_i^T,
// z_i = gamma z_(i-1) + phi(k_i), o_i = phi(q_i)^T S_i / (phi(q_i) . z_i + eps),
// phi = elu + 1, with the fixed per-head decay gamma of its "Gating and
// Selective State Updates" (RetNet) on both S and z.
//
// The same chunkwise regrouping and sequence split as the 64-token kernel
// (chunk_tc.cu): parts of whole chunks per (batch, head), phase A (the
// part's own sum A_p), a chain of inclusive states between the CTAs of one
// (batch, head), then phase C over the part's chunks:
//   qh_t = gamma^(c0+t-E) phi(q_t),  kh_s = gamma^(E-c0-s) phi(k_s)
//   A'   = qh kh^T,  P = A' masked to s <= t
//   O    = qh [T | z] + P [V | 1],  T += kh^T [V | 1]
//   o_t  = O[t, :Dv] / (O[t, Dv] + eps)
// with T the state scaled to the end E of the current decay window.
//
// What differs: chunks of 128 tokens, so every product of phase C is an
// M = 128 MMA (twice the work per instruction of the M = 64 products, and
// half the hand-offs per token), and the A operands qh and P live in tensor
// memory: the feature-map warps write qh there (no shared-memory tile for
// the mapped q), and the P warps overwrite A' in place with bf16 P.  That
// leaves shared memory for double-buffered k and v tiles of 128 tokens.
//
// Warp roles (18 warps):
//   0-3   P: A' -> masked bf16 P in tensor memory
//   4-7   state and output: the chain, the bf16 copy of [T | z] for the MMA
//         and window rescaling (thread = row d of T), then O -> o rows
//         (divide by the normaliser; thread = token row)
//   8-15  feature map: kh in place, qh into tensor memory; warp 8 + j maps
//         the rows of TMEM lane quadrant j % 4, dims [64 (j / 4), + 64)
//   (warps 0-15 share the phase A feature map)
//   16    TMA: lane 0 the k ring, lane 1 the v ring, lane 2 the q tile
//   17    TMEM owner and MMA issuer
// Every wait is bounded; a CTA that gives up counts the failure in device
// memory, drains its in-flight copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace linattn {
namespace {

using namespace tc;

constexpr int kC = 128;      // tokens per chunk
constexpr int kD = 128;      // key / query width
constexpr int kDV = 128;     // value width
constexpr int kNA = kDV + 16;  // columns of [V | 1], [T | z] and O
constexpr int kThreads = 576;
constexpr int kWarpS = 4;
constexpr int kWarpPhi = 8;
constexpr int kWarpTma = 16;
constexpr int kWarpMma = 17;
constexpr float kGammaMin = 0.61f;       // gamma^128 stays above 1e-28
constexpr float kLog2Floor = -93.0139f;  // log2(1e-28): smallest factor in a window

// Shared memory, from a 1024-byte aligned base.
//   k ring: 2 slots x 2 boxes of 128 rows x 128 bytes (64 dims), 128-byte swizzle
//   v ring: 2 slots x 2 atoms of 128 rows x 128 bytes (64 columns), 128-byte
//           swizzle, and one ones atom (column 0 = 1) shared by both slots:
//           [V | 1] is MN-major with atom stride LBO, so slot 0 (atoms at
//           +64K, +80K, LBO 16 KB) and slot 1 (atoms at +0, +48K, LBO 48 KB)
//           both reach the ones atom at +96K; the q tile fills the gap
//   q tile: one slot, 2 boxes like k, at +16K in the v region
//   [T | z]: bf16, 5 atoms of 128 rows (d) x 64 bytes, 64-byte swizzle
//   output staging: per state/output warp 32 rows x 64 bytes (32 columns of
//           o), 64-byte swizzle, written back by TMA tile stores
constexpr int kKBox = 128 * 128;
constexpr int kVAtom = 128 * 128;  // 64 columns of v, 128-byte swizzle
constexpr int kKSlot = 2 * kKBox;

constexpr int kOffK = 0;
constexpr int kOffVR = kOffK + 2 * kKSlot;  // v slot 1 atom 0 | q | v slot 1 atom 1 | v slot 0 | ones
constexpr int kOffQ = kOffVR + kVAtom;
constexpr int kOffOnes = kOffVR + 6 * kVAtom;
__host__ __device__ constexpr int v_base(int sl) { return sl == 0 ? kOffVR + 4 * kVAtom : kOffVR; }
__host__ __device__ constexpr int v_lbo(int sl) { return sl == 0 ? kVAtom : 3 * kVAtom; }
constexpr int kSopAtom = kD * 64;
constexpr int kOffSop = kOffVR + 7 * kVAtom;
constexpr int kStgBytes = 32 * 64;
constexpr int kOffStg = kOffSop + 5 * kSopAtom;
constexpr int kNumBars = 24;
constexpr int kOffBar = kOffStg + 4 * kStgBytes;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kBytes = kOffMisc + 32;
constexpr int kAlloc = kBytes + 1024;  // slack for the 1024-byte alignment
static_assert(kAlloc <= 227 * 1024, "shared memory");
static_assert(kOffVR % 1024 == 0 && kOffQ % 1024 == 0 && kOffSop % 1024 == 0, "align");

// Tensor memory (512 columns): qh as bf16 pairs, A' (fp32; P as bf16 pairs
// in its first 64 columns), T = [S | z] (fp32), O (fp32).
constexpr uint32_t kColQ = 0;
constexpr uint32_t kColA = 64;
constexpr uint32_t kColT = 192;
constexpr uint32_t kColO = kColT + kNA;
static_assert(kColO + kNA <= 512, "tensor memory");

// barrier slots
enum Bar : int {
  kKFull = 0,      // [2] TMA k tile landed
  kKEmpty = 2,     // [2] k slot free (MMA commit)
  kVFull = 4,      // [2]
  kVEmpty = 6,     // [2]
  kQFull = 8,      // q tile landed
  kQEmpty = 9,     // q tile read by the feature-map warps
  kKMapped = 10,   // [2] kh in place
  kQReady = 12,    // qh in tensor memory
  kAFull = 13,     // A' computed
  kPFull = 14,     // P in tensor memory
  kTReady = 15,    // T updated
  kTFree = 16,     // T read (and rescaled) by the state warps
  kSFull = 17,     // bf16 [T | z] written
  kInterDone = 18, // O = qh [T | z] done: [T | z] and qh may be replaced
  kOFull = 19,     // O complete
  kOFree = 20,     // O read by the output warps
  kDrain = 21,
};

// Part boundaries (in chunks).  The CTA of part p > 0 runs phase A over
// part p - 1 and then, once every earlier part's sum is published, phase C
// over part p; part 0 runs phase C only.
//
// Relay split (n0 > 0): part 0 has n0 chunks and the later parts share the
// rest equally.  Part 0 starts phase C at once, so it can take more chunks
// than the others; to keep part 1 from paying a phase A over all of them,
// the CTA of part 0 publishes its running state after its first m0 chunks
// (a checkpoint), and part 1's phase A covers only chunks [m0, n0), the
// state before part 1 being gamma^(C (n0 - m0)) times the checkpoint plus
// that sum.  Sizes are chosen so that the checkpoint and part 1's phase A
// land together and all parts end together.  n0 = 0: equal parts, no
// checkpoint.
__host__ __device__ __forceinline__ int part_begin(int p, int P, int nch_all, int n0) {
  if (n0 <= 0 || P <= 1) return chunk_part_begin(p, P, nch_all);
  if (p <= 0) return 0;
  if (p >= P) return nch_all;
  return n0 + chunk_part_begin(p - 1, P - 1, nch_all - n0);
}

struct Chunk128Params {
  CUtensorMap tmQ, tmK, tmV, tmO;
  float *rec;      // P > 1: inclusive states [B*H][P][D*Dv + D]
  int *ws_flag;    // P > 1: [B*H][P], 1 once incl_p is published
  int *ws_ticket;  // P > 1: part-major work counter
  unsigned int *timeouts;
  // optional: the state after the last token, S [B*H][D][Dv] and z [B*H][D]
  // fp32, written by the CTA of the last part (nullptr: not written)
  float *S_out, *z_out;
  // gated mode: the state is rescaled row by row at every chunk boundary by
  // the chunk's gate products gate_prod [B*H][chunks][D] (q, k arrive
  // already scaled); nonzero *skip: some chunk forgets too hard for this
  // form, the launch does nothing
  const float *gate_prod;
  // gated, P > 1: gate_suf [B*H][chunks][D], the product of gate_prod over
  // the later chunks of the same part; gate_part [B*H][P][D], over a whole part
  const float *gate_suf, *gate_part;
  const int *skip;
  int BH, H, N, P;
  // relay split (see part_begin): chunks of part 0 and the checkpoint
  // position (0, 0: equal parts); the checkpoint is record P - 1 of its
  // (batch, head); flag P - 1 counts the state warps that have written it
  int n0, m0;
  float eps;
  Gammas lg;  // log2(gamma) per head
};

// phi and the row scale in place on one box row: 8 chunks of 16 bytes of
// row r of a 128-byte-swizzled box.
template <bool IDENT>
__device__ __forceinline__ void map_row(uint8_t *box, int r, uint32_t sc) {
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

// The same on chunks [c0, c0 + 4) of the row.
template <bool IDENT>
__device__ __forceinline__ void map_row4(uint8_t *box, int r, int c0, uint32_t sc) {
  uint4 x[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) x[c] = *reinterpret_cast<const uint4 *>(box + sw128_off(r, 16 * (c0 + c)));
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    x[c].x = feat_scale_bf16x2<IDENT>(x[c].x, sc);
    x[c].y = feat_scale_bf16x2<IDENT>(x[c].y, sc);
    x[c].z = feat_scale_bf16x2<IDENT>(x[c].z, sc);
    x[c].w = feat_scale_bf16x2<IDENT>(x[c].w, sc);
    *reinterpret_cast<uint4 *>(box + sw128_off(r, 16 * (c0 + c))) = x[c];
  }
}

// Per-feature factors on chunks [c0, c0 + 4) of row r of a box (features
// 8 (c0 + c) + j of the box, factor 8 c + j held by lane 8 c + j of the warp
// in f_lane); a row past the sequence end becomes 0.  All 32 lanes call it.
__device__ __forceinline__ void map_row4_feat(uint8_t *box, int r, int c0, float f_lane,
                                              bool valid) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 *ptr = reinterpret_cast<uint4 *>(box + sw128_off(r, 16 * (c0 + c)));
    uint4 x = *ptr;
    float f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = __shfl_sync(0xffffffffu, f_lane, 8 * c + j);
    if (valid) {
      x.x = feat_scale_bf16x2<true>(x.x, pack_bf16x2(f[0], f[1]));
      x.y = feat_scale_bf16x2<true>(x.y, pack_bf16x2(f[2], f[3]));
      x.z = feat_scale_bf16x2<true>(x.z, pack_bf16x2(f[4], f[5]));
      x.w = feat_scale_bf16x2<true>(x.w, pack_bf16x2(f[6], f[7]));
    } else {
      x = make_uint4(0u, 0u, 0u, 0u);
    }
    *ptr = x;
  }
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t *v) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
  tmem_st32(taddr, f);
}
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t *v) {
  float f[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
  tmem_st16(taddr, f);
}

template <bool DECAY, bool IDENT, bool GATED = false>
__global__ void __launch_bounds__(kThreads, 1) chunk128_kernel(const __grid_constant__ Chunk128Params p) {
  if (GATED && *p.skip) return;  // uniform: every thread reads the same flag
  constexpr size_t kRec = static_cast<size_t>(kD) * kDV + kD;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
  int *item = reinterpret_cast<int *>(sm + kOffMisc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.BH, N = p.N, P = p.P;

  // ---- set-up: work item, constant operand blocks, barriers, TMEM ----
  if (tid == 0) {
    int t = static_cast<int>(blockIdx.x);
    if (P > 1) t = atomicAdd(p.ws_ticket, 1);
    item[0] = t / BH;  // part (part-major order)
    item[1] = t % BH;  // batch * head
  }
  {
    // the ones atom (shared by both v slots) and the [T | z] operand: zero,
    // then column 0 of every ones row = 1
    for (int i = tid; i < kVAtom / 16; i += kThreads)
      reinterpret_cast<uint4 *>(sm + kOffOnes)[i] = make_uint4(0, 0, 0, 0);
    for (int i = tid; i < 5 * kSopAtom / 16; i += kThreads)
      reinterpret_cast<uint4 *>(sm + kOffSop)[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (tid < kC) {
    const int r = tid;
    *reinterpret_cast<__nv_bfloat16 *>(sm + kOffOnes + sw128_off(r, 0)) =
        __float2bfloat16_rn(1.f);
  }
  if (tid == 32 * kWarpTma) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[kKFull + s], 1);
      mbar_init(&bar[kKEmpty + s], 1);
      mbar_init(&bar[kVFull + s], 1);
      mbar_init(&bar[kVEmpty + s], 1);
      mbar_init(&bar[kKMapped + s], 16);
    }
    mbar_init(&bar[kQFull], 1);
    mbar_init(&bar[kQEmpty], 8);
    mbar_init(&bar[kQReady], 8);
    mbar_init(&bar[kAFull], 1);
    mbar_init(&bar[kPFull], 4);
    mbar_init(&bar[kTReady], 1);
    mbar_init(&bar[kTFree], 4);
    mbar_init(&bar[kSFull], 4);
    mbar_init(&bar[kInterDone], 1);
    mbar_init(&bar[kOFull], 1);
    mbar_init(&bar[kOFree], 4);
    mbar_init(&bar[kDrain], 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, 512);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int part = item[0], bh = item[1];
  // identity features without per-row decay (Performer features, gated
  // k-hat): the phase-C k map would multiply every row by one (rows past the
  // sequence end are already zero from the copy's bounds), so it is skipped,
  // in phase A too; the call stays for rows past the end (a no-op at run
  // time on full chunks: without it ptxas spilled in the per-chunk loops).
  constexpr bool kMapK = !(IDENT && !DECAY);

  // the part: chunks [cb, cb + nch) of this (batch, head); phase A runs
  // over the previous part, chunks [cbA, cbA + nA)
  const int nch_all = (N + kC - 1) / kC;
  const bool relay = P > 1 && p.n0 > 0 && p.m0 > 0;
  const int cb = part_begin(part, P, nch_all, p.n0);
  const int nch = part_begin(part + 1, P, nch_all, p.n0) - cb;
  const bool hasA = part > 0;
  // part 1 of a relay split sums only the chunks of part 0 after the checkpoint
  const int cbA = hasA ? (relay && part == 1 ? p.m0 : part_begin(part - 1, P, nch_all, p.n0)) : 0;
  const int nA = hasA ? cb - cbA : 0;
  const float lg = DECAY ? p.lg.g[bh % p.H] : 0.f;
  const bool final_state = p.S_out != nullptr && part == P - 1;
  int WC = 64;  // chunks per decay window
  if (DECAY && lg < 0.f) {
    const float c = kLog2Floor / lg / static_cast<float>(kC);
    WC = c < 1.f ? 1 : (c > 64.f ? 64 : static_cast<int>(c));
  }
  const int W = kC * WC;
  auto phase_a_chunk = [&](int i) { return part == 1 && !relay ? i : nA - 1 - i; };
  auto scale2 = [&](float e) -> uint32_t {  // gamma^e as a bf16 pair
    const float f = DECAY ? exp2f(e * lg) : 1.f;
    return pack_bf16x2(f, f);
  };

  // Phase A feature map over the previous part, kh_s = gamma^(E - 1 - s)
  // phi(k_s) with E the end of that part (a chunk boundary).  Phase A takes
  // the chunks of parts 1, 2, ... last first, so that the tiles the owner of
  // that part reads first in its phase C are the most recent in L2; part 0
  // (read in phase C from time zero) goes first chunk first, ahead of its
  // owner, unless a checkpoint cuts it (then last first, like the others).
  // All 16 compute warps share the map: warp u maps rows 32 (u % 4) + lane,
  // 16-byte chunks [4 (u / 4), + 4) of the row (box u / 8).
  auto phase_a_map = [&](int u) {
    const int r = 32 * (u & 3) + lane, quarter = u >> 2;
    // gated: k-hat already carries the gates up to its chunk's end; the
    // later chunks of the previous part add their products, feature by
    // feature.  Lane l holds factor l of this warp's 32 features, loaded one
    // chunk ahead so that the load is not on the chunk's critical path.
    auto gate_factor = [&](int i) {
      const int ia = phase_a_chunk(i);
      return __ldg(p.gate_suf + (static_cast<size_t>(bh) * ((N + kC - 1) / kC) + cbA + ia) * kD +
                   64 * (quarter >> 1) + 32 * (quarter & 1) + lane);
    };
    float f_next = GATED && nA > 0 ? gate_factor(0) : 0.f;
    for (int i = 0; i < nA; ++i) {
      const int sl = i & 1, ia = phase_a_chunk(i);
      const float f_lane = f_next;
      if (GATED && i + 1 < nA) f_next = gate_factor(i + 1);
      if (!warp_wait(&bar[kKFull + sl], (i >> 1) & 1, abort_flag, p.timeouts)) break;
      const int nv = min(kC, N - (cbA + ia) * kC);
      if (GATED) {
        map_row4_feat(sm + kOffK + sl * kKSlot + (quarter >> 1) * kKBox, r, 4 * (quarter & 1), f_lane,
                      r < nv);
      } else if (kMapK || r >= nv) {
        const uint32_t sc = r < nv ? scale2(static_cast<float>(kC * (nA - ia) - 1 - r)) : 0u;
        map_row4<IDENT>(sm + kOffK + sl * kKSlot + (quarter >> 1) * kKBox, r, 4 * (quarter & 1), sc);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kKMapped + sl]);
    }
  };

  // Before phase C, by the 16 compute warps (warp u: rows 32 (u % 4) +
  // lane, columns [32 (u / 4), + 32) of S; warps 0-3 also z): the state
  // before the part, S0 = sum_(j < part) gamma^(c0 - E_j) A_j (c0 = the
  // part's first token, E_j = the end of part j, A_j = part j's own sum
  // scaled to E_j).  A_(part-1) is this CTA's phase A, in tensor memory; it
  // is published for the later parts that need it.  A_j, j < part - 1, was
  // published by the CTA of part j + 1 (a flag per record, release/acquire
  // at GPU scope; parts are started in part-major order by an atomic ticket,
  // so every wait ends).  With a relay split, part 1 adds part 0's checkpoint
  // to its phase A before publishing A_0 (then the whole state before part
  // 1).  T = gamma^W S0 goes to tensor memory and, in bf16, to [T | z].
  auto look_back = [&](int u) {
    const int qd = u & 3, g4 = u >> 2;
    const int d = 32 * qd + lane;
    const bool zcol = g4 == 0;
    const uint32_t tS = tmem_addr(tmem, 32 * qd, kColT + 32 * g4);
    const uint32_t tZ = tmem_addr(tmem, 32 * qd, kColT + kDV);
    float acc[32], accz = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
    if (hasA) {
      warp_wait(&bar[kTReady], 0, abort_flag, p.timeouts);
      tc_fence_after();
      tmem_ld32(tS, acc);
      if (zcol) accz = tmem_ld1(tZ);
      tmem_wait_ld();
    }
    if (relay && part == 1) {
      // the state before part 1: the checkpoint of part 0 (the state after
      // its first m0 chunks, relative to token m0 C - 1), carried to token
      // cb C - 1, plus this CTA's phase A over chunks [m0, cb)
      if (tid == 0) {
        const long long t0 = clock64();
        const int *f = p.ws_flag + bh * P + P - 1;  // one count per state warp
        while (ld_acquire_gpu(f) < 4) {
          if (*abort_flag) break;
          if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            atomicAdd(p.timeouts, 1u);
            break;
          }
          __nanosleep(32);
        }
      }
      named_sync(1, 512);
      if (!*abort_flag) {
        const float wk = DECAY ? exp2f(static_cast<float>((cb - p.m0) * kC) * lg) : 1.f;
        const float *ck = p.rec + (static_cast<size_t>(bh) * P + P - 1) * kRec;
        float4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = __ldcg(reinterpret_cast<const float4 *>(ck) + (8 * g4 + q) * kD + d);
        const float vz = zcol ? __ldcg(ck + kD * kDV + d) : 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          acc[4 * q] = fmaf(wk, v[q].x, acc[4 * q]);
          acc[4 * q + 1] = fmaf(wk, v[q].y, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(wk, v[q].z, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(wk, v[q].w, acc[4 * q + 3]);
        }
        accz = fmaf(wk, vz, accz);
      }
    }
    if (hasA && part < P - 1) {  // A_(part-1) is read by the parts after this one
      float *rec = p.rec + (static_cast<size_t>(bh) * P + part - 1) * kRec;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        __stcg(reinterpret_cast<float4 *>(rec) + (8 * g4 + q) * kD + d,
               make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
      if (zcol) __stcg(rec + kD * kDV + d, accz);
      __threadfence();
    }
    named_sync(1, 512);
    if (hasA && part < P - 1 && tid == 0) st_release_gpu(p.ws_flag + bh * P + part - 1, 1);
    if (part >= 2) {
      if (tid == 0) {
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
      named_sync(1, 512);
      // gated: the weight of A_j is the product of the whole-part gate
      // products of parts j + 1 .. part - 1, built up from j = part - 2 down
      float wg = 1.f;
      for (int jj = 0; jj < part - 1 && !*abort_flag; ++jj) {
        const int j = GATED ? part - 2 - jj : jj;
        if (GATED) wg *= __ldg(p.gate_part + (static_cast<size_t>(bh) * P + j + 1) * kD + d);
        const float wj =
            GATED ? wg
                  : (DECAY ? exp2f(static_cast<float>((cb - part_begin(j + 1, P, nch_all, p.n0)) * kC) * lg)
                           : 1.f);
        const float *rec = p.rec + (static_cast<size_t>(bh) * P + j) * kRec;
        float4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = __ldcg(reinterpret_cast<const float4 *>(rec) + (8 * g4 + q) * kD + d);
        const float vz = zcol ? __ldcg(rec + kD * kDV + d) : 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          acc[4 * q] = fmaf(wj, v[q].x, acc[4 * q]);
          acc[4 * q + 1] = fmaf(wj, v[q].y, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(wj, v[q].z, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(wj, v[q].w, acc[4 * q + 3]);
        }
        accz = fmaf(wj, vz, accz);
      }
    }
    // to the end of the first window (decay) or of the first chunk (gated)
    const float gW = GATED ? __ldg(p.gate_prod + (static_cast<size_t>(bh) * ((N + kC - 1) / kC) + cb) * kD + d)
                           : (DECAY ? exp2f(static_cast<float>(W) * lg) : 1.f);
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] *= gW;
    tmem_st32(tS, acc);
    put_sop32(sm + kOffSop, kSopAtom, g4, d, acc);
    if (zcol) {
      float zz[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) zz[e] = 0.f;
      zz[0] = accz * gW;
      tmem_st16(tZ, zz);
      put_sop16(sm + kOffSop, kSopAtom, kDV / 32, d, zz);
    }
    tmem_wait_st();
    tc_fence_before();
    fence_async_smem();
    named_sync(1, 512);
  };

  if (warp == kWarpTma) {
    // ---------------- TMA: three independent rings, one lane each ----------------
    // lane 0: k tiles (phase A then phase C), lane 1: v tiles, lane 2: q tiles
    // (phase C).  Slot of ring chunk c: c % 2, phase (c / 2) & 1.
    if (lane < 3) {
      const CUtensorMap *map = lane == 0 ? &p.tmK : (lane == 1 ? &p.tmV : &p.tmQ);
      prefetch_tmap(map);
      const int n = lane == 2 ? nch : nA + nch;
      const int slots = lane == 2 ? 1 : 2;
      uint64_t *fullb = &bar[lane == 0 ? kKFull : (lane == 1 ? kVFull : kQFull)];
      uint64_t *emptyb = &bar[lane == 0 ? kKEmpty : (lane == 1 ? kVEmpty : kQEmpty)];
      // first token row of ring chunk c: phase A (previous part), then phase C
      auto ring_row = [&](int c) {
        return (lane == 2 ? cb + c : (c < nA ? cbA + phase_a_chunk(c) : cb + c - nA)) * kC;
      };
      int issued = 0;
      for (int c = 0; c < n; ++c) {
        const int sl = c % slots;
        const uint32_t ph = static_cast<uint32_t>((c / slots) & 1);
        if (!mbar_wait(&emptyb[sl], ph ^ 1, abort_flag, p.timeouts)) break;
        const int row = ring_row(c);
        mbar_arrive_expect_tx(&fullb[sl], lane == 1 ? 2 * kVAtom : kKSlot);
        if (lane == 1) {
          tma_load_3d(sm + v_base(sl), map, 0, row, bh, &fullb[sl]);
          tma_load_3d(sm + v_base(sl) + v_lbo(sl), map, 64, row, bh, &fullb[sl]);
        } else {
          uint8_t *dst = sm + (lane == 0 ? kOffK + sl * kKSlot : kOffQ);
          tma_load_3d(dst, map, 0, row, bh, &fullb[sl]);
          tma_load_3d(dst + kKBox, map, 64, row, bh, &fullb[sl]);
        }
        issued = c + 1;
        // During phase A, an L2 prefetch of the next ring chunk (its load
        // waits for a slot).  Phase C prefetches nothing: with every CTA
        // streaming, a prefetch only adds L2 traffic ahead of a load that is
        // already queued.
        const int cp = c + 1;
        if (lane != 2 && c < nA && cp < n) {
          const int rowp = ring_row(cp);
          tma_prefetch_3d(map, 0, rowp, bh);
          tma_prefetch_3d(map, 64, rowp, bh);
        }
      }
      if (*abort_flag) {  // let every issued copy land before the CTA exits
        for (int c = issued > slots ? issued - slots : 0; c < issued; ++c)
          mbar_wait_drain(&fullb[c % slots], (c / slots) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer (warp-wide loop, lane 0 issues) ----------------
    const bool leader = lane == 0;
    constexpr uint32_t ID_A = idesc_bf16(128, 128, false, false);  // qh (TMEM) kh^T
    constexpr uint32_t ID_DS = idesc_bf16(128, kNA, true, true);   // kh^T [V | 1]
    constexpr uint32_t ID_O = idesc_bf16(128, kNA, false, true);   // qh [T|z], P [V|1]
    const uint32_t base = smem_u32(sm);
    // kh as B of A' (K-major: rows s, K = d), kh^T as A of dS (MN-major: M = d
    // in two 64-wide atoms, K = tokens), [V | 1] and [T | z] as B (MN-major:
    // N in 32-wide atoms, K = tokens or d)
    auto dk = [&](int sl) { return smem_desc(base + kOffK + sl * kKSlot, 16, 1024, kSw128); };
    auto dkt = [&](int sl) { return smem_desc(base + kOffK + sl * kKSlot, kKBox, 1024, kSw128); };
    auto dv = [&](int sl) { return smem_desc(base + v_base(sl), v_lbo(sl), 1024, kSw128); };
    const uint64_t dsop = smem_desc(base + kOffSop, kSopAtom, 512, kSw64);
    const uint32_t tQ = tmem + kColQ, tA = tmem + kColA, tT = tmem + kColT, tO = tmem + kColO;
    bool ok = true;
    // phase A: T = kh^T [V | 1] over the part
    for (int i = 0; i < nA; ++i) {
      const int sl = i & 1;
      const uint32_t ph = static_cast<uint32_t>((i >> 1) & 1);
      if (!warp_wait(&bar[kKMapped + sl], ph, abort_flag, p.timeouts) ||
          !warp_wait(&bar[kVFull + sl], ph, abort_flag, p.timeouts)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (leader) {
        const uint64_t a = dkt(sl), b = dv(sl);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tT, a + kk * 128, b + kk * 128, ID_DS, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar[kKEmpty + sl]);
        mma_commit(&bar[kVEmpty + sl]);
      }
      __syncwarp();
    }
    if (ok && hasA) {
      if (leader) mma_commit(&bar[kTReady]);
      __syncwarp();
    }
    // phase C.  Iteration i: [dS_i], inter_i, intra_i, then A'_(i+1), so that
    // each consumer round trip (P, the [T | z] copy, the O read-out, qh) has
    // at least one group of 8 MMAs queued in front of the MMA that waits on it.
    auto issue_a = [&](int i) -> bool {  // A'_i = qh_i kh_i^T  (M 128 t, N 128 s, K = D)
      const int c = nA + i, sl = c & 1;
      if (!warp_wait(&bar[kKMapped + sl], (c >> 1) & 1, abort_flag, p.timeouts) ||
          !warp_wait(&bar[kQReady], i & 1, abort_flag, p.timeouts))
        return false;
      tc_fence_after();
      if (leader) {
        const uint64_t b = dk(sl);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ta(tA, tQ + 8 * kk, b + (kk >> 2) * (kKBox >> 4) + (kk & 3) * 2, ID_A,
                      kk > 0 ? 1u : 0u);
        mma_commit(&bar[kAFull]);
      }
      __syncwarp();
      return true;
    };
    if (ok && nch > 0 && !issue_a(0)) ok = false;
    for (int i = 0; ok && i < nch; ++i) {
      const int c = nA + i, sl = c & 1;
      const uint32_t ph = static_cast<uint32_t>((c >> 1) & 1);
      if (i + 1 < nch || final_state) {
        // T += kh^T [V | 1]: after the last chunk only for the final state
        if (!warp_wait(&bar[kTFree], i & 1, abort_flag, p.timeouts) ||
            !warp_wait(&bar[kVFull + sl], ph, abort_flag, p.timeouts))
          break;
        tc_fence_after();
        if (leader) {
          const uint64_t a = dkt(sl), b = dv(sl);
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk) mma_bf16(tT, a + kk * 128, b + kk * 128, ID_DS, 1u);
          mma_commit(&bar[kTReady]);
        }
      }
      if (leader) mma_commit(&bar[kKEmpty + sl]);
      __syncwarp();
      // O = qh [T | z]  (M 128, N Dv + 16, K = D)
      if (!warp_wait(&bar[kSFull], i & 1, abort_flag, p.timeouts)) break;
      if (i > 0 && !warp_wait(&bar[kOFree], (i - 1) & 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ta(tO, tQ + 8 * kk, dsop + kk * 64, ID_O, kk > 0 ? 1u : 0u);
        mma_commit(&bar[kInterDone]);
      }
      __syncwarp();
      // O += P [V | 1]  (M 128, N Dv + 16, K 128 tokens)
      if (!warp_wait(&bar[kPFull], i & 1, abort_flag, p.timeouts) ||
          !warp_wait(&bar[kVFull + sl], ph, abort_flag, p.timeouts))
        break;
      tc_fence_after();
      if (leader) {
        const uint64_t b = dv(sl);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) mma_bf16_ta(tO, tA + 8 * kk, b + kk * 128, ID_O, 1u);
        mma_commit(&bar[kOFull]);
        mma_commit(&bar[kVEmpty + sl]);
      }
      __syncwarp();
      if (i + 1 < nch && !issue_a(i + 1)) break;
    }
    // every MMA issued has completed before TMEM is released
    if (leader) {
      mma_commit(&bar[kDrain]);
      mbar_wait_drain(&bar[kDrain], 0);
    }
    __syncwarp();
  } else if (warp >= kWarpPhi) {
    // ---------------- feature map: kh in place, qh into tensor memory ----------------
    const int j = warp - kWarpPhi;
    const int qd = j & 3, h = j >> 2;  // TMEM lane quadrant, half of the dims
    const int r = 32 * qd + lane;      // token row of the chunk
    phase_a_map(warp);
    const uint32_t tq = tmem_addr(tmem, 32 * qd, kColQ + 32 * h);
    bool looked = false;  // the look-back runs once, after chunk 0 is mapped
    for (int i = 0; i < nch; ++i) {
      const int c = nA + i, sl = c & 1;
      const int nv = min(kC, N - (cb + i) * kC);
      const int jw = i % WC;  // chunk within its decay window
      // kh_s = gamma^(E - s) phi(k_s), rows past the sequence end zero
      if (!warp_wait(&bar[kKFull + sl], (c >> 1) & 1, abort_flag, p.timeouts)) break;
      if (kMapK || GATED && r >= nv)
        map_row<IDENT>(sm + kOffK + sl * kKSlot + h * kKBox, r,
                       r < nv ? scale2(static_cast<float>(W - 1 - kC * jw - r)) : 0u);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(&bar[kKMapped + sl], 2);
      // qh_t = gamma^(t - E) phi(q_t), as bf16 pairs (column m = dims 2m, 2m+1)
      if (!warp_wait(&bar[kQFull], i & 1, abort_flag, p.timeouts)) break;
      uint32_t qh[32];
      {
        const uint32_t sc = scale2(static_cast<float>(kC * jw - (W - 1) + r));
        uint4 x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          x[q] = *reinterpret_cast<const uint4 *>(sm + kOffQ + h * kKBox + sw128_off(r, 16 * q));
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          qh[4 * q + 0] = feat_scale_bf16x2<IDENT>(x[q].x, sc);
          qh[4 * q + 1] = feat_scale_bf16x2<IDENT>(x[q].y, sc);
          qh[4 * q + 2] = feat_scale_bf16x2<IDENT>(x[q].z, sc);
          qh[4 * q + 3] = feat_scale_bf16x2<IDENT>(x[q].w, sc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kQEmpty]);
      // qh_(i-1) is consumed once O = qh [T | z] of chunk i-1 is done
      if (i > 0 && !warp_wait(&bar[kInterDone], (i - 1) & 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      tmem_st32u(tq, qh);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kQReady]);
      if (i == 0) {
        look_back(warp);
        looked = true;
      }
    }
    if (!looked) look_back(warp);
  } else if (warp >= kWarpS) {
    // ---------------- state, then output rows ----------------
    const int w = warp - kWarpS;  // TMEM lane quadrant
    const int d = 32 * w + lane;  // row of T (state) and token row (output)
    const uint32_t tT = tmem_addr(tmem, 32 * w, kColT);
    const uint32_t to = tmem_addr(tmem, 32 * w, kColO);
    uint8_t *sop = sm + kOffSop;
    uint8_t *stg = sm + kOffStg + w * kStgBytes;
    if (lane == 0) prefetch_tmap(&p.tmO);
    phase_a_map(warp);
    look_back(warp);
    const float gW = DECAY ? exp2f(static_cast<float>(W) * lg) : 1.f;
    if (lane == 0) {  // the chain is done (chain_part ends with a barrier)
      mbar_arrive(&bar[kTFree]);
      mbar_arrive(&bar[kSFull]);
    }
    // gated: row d of T times the gate product of chunk i before chunk i;
    // each is loaded one chunk ahead, off the chunk's critical path
    auto gate_row = [&](int i) {
      return __ldg(p.gate_prod + (static_cast<size_t>(bh) * ((N + kC - 1) / kC) + cb + i) * kD + d);
    };
    float fr_next = GATED && nch > 1 ? gate_row(1) : gW;
    for (int i = 1; i <= nch; ++i) {
      // (1) after T += kh^T [V | 1] of chunk i-1 and once O = qh [T | z] of
      // chunk i-1 has read the old copy, publish bf16 [T | z] for chunk i
      // (rescaled when chunk i opens a new decay window)
      if (i < nch) {
        const float fr = fr_next;
        if (GATED && i + 1 < nch) fr_next = gate_row(i + 1);
        if (!warp_wait(&bar[kTReady], static_cast<uint32_t>((i - 1 + (hasA ? 1 : 0)) & 1), abort_flag,
                       p.timeouts) ||
            !warp_wait(&bar[kInterDone], static_cast<uint32_t>((i - 1) & 1), abort_flag, p.timeouts))
          break;
        tc_fence_after();
        const bool rebase = (DECAY && (i % WC == 0)) || GATED;
        if (relay && part == 0 && i == p.m0) {
          // relay split, part 0 after m0 chunks: the checkpoint, T carried
          // from the end of the window of chunk i - 1 back to token i C - 1;
          // this warp's rows are written and fenced, then counted
          float *ck = p.rec + (static_cast<size_t>(bh) * P + P - 1) * kRec;
          const float fk = DECAY ? exp2f(static_cast<float>(((i - 1) % WC + 1) * kC - W) * lg) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < kDV / 32; ++cc) {
            float x[32];
            tmem_ld32(tT + 32 * cc, x);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg(reinterpret_cast<float4 *>(ck) + (8 * cc + q) * kD + d,
                     make_float4(fk * x[4 * q], fk * x[4 * q + 1], fk * x[4 * q + 2], fk * x[4 * q + 3]));
          }
          const float zd = tmem_ld1(tT + kDV);
          tmem_wait_ld();
          __stcg(ck + kD * kDV + d, fk * zd);
          __threadfence();
          __syncwarp();
          if (lane == 0) atomicAdd(p.ws_flag + bh * P + P - 1, 1);
        }
        if (GATED) {
          // every chunk rebases: one 32-column tile at a time keeps the
          // scaled copy within the register budget
#pragma unroll 1
          for (int cc = 0; cc < kDV / 32; ++cc) {
            float x0[32];
            tmem_ld32(tT + 32 * cc, x0);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) x0[e] *= fr;
            tmem_st32(tT + 32 * cc, x0);
            put_sop32(sop, kSopAtom, cc, d, x0);
          }
        } else {
#pragma unroll 1
          for (int cc = 0; cc < kDV / 32; cc += 2) {
            float x0[32], x1[32];
            tmem_ld32(tT + 32 * cc, x0);
            tmem_ld32(tT + 32 * cc + 32, x1);
            tmem_wait_ld();
            if (rebase) {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                x0[e] *= fr;
                x1[e] *= fr;
              }
              tmem_st32(tT + 32 * cc, x0);
              tmem_st32(tT + 32 * cc + 32, x1);
            }
            put_sop32(sop, kSopAtom, cc, d, x0);
            put_sop32(sop, kSopAtom, cc + 1, d, x1);
          }
        }
        {
          float x0[16];
          tmem_ld16(tT + kDV, x0);
          tmem_wait_ld();
          if (rebase) {
#pragma unroll
            for (int e = 0; e < 16; ++e) x0[e] *= fr;
            tmem_st16(tT + kDV, x0);
          }
          put_sop16(sop, kSopAtom, kDV / 32, d, x0);
        }
        if (rebase) tmem_wait_st();
        tc_fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bar[kTFree]);
          mbar_arrive(&bar[kSFull]);
        }
      }
      // (2) output rows of chunk i-1: o_t = O[t, :Dv] / (O[t, Dv] + eps),
      // 32 columns at a time through this warp's staging tile and a TMA
      // store (rows past the sequence end are clipped by the tensor map)
      const int io = i - 1;
      if (!warp_wait(&bar[kOFull], io & 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      float inv = 0.f;
#pragma unroll 1
      for (int j = 0; j < kDV / 32; ++j) {
        float x[32], den = 0.f;
        tmem_ld32(to + 32 * j, x);
        if (j == 0) den = tmem_ld1(to + kDV);
        tmem_wait_ld();
        if (j == 0) inv = 1.f / (den + p.eps);
        if (j == kDV / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_relaxed(&bar[kOFree]);
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(x[2 * e] * inv, x[2 * e + 1] * inv);
        if (lane == 0) bulk_wait_group_read0();  // the previous store has read the tile
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4 *>(stg + sw64_off(lane, 16 * q)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&p.tmO, stg, 32 * j, (cb + io) * kC + 32 * w, bh);
          bulk_commit_group();
        }
      }
    }
    if (final_state && !*abort_flag) {
      // the state after the last token: T after the last chunk's update is
      // scaled to the end of its decay window, E; the state wants the last
      // token N - 1 as its reference, a factor gamma^((N - 1) - E)
      warp_wait(&bar[kTReady], static_cast<uint32_t>((nch - 1 + (hasA ? 1 : 0)) & 1), abort_flag,
                p.timeouts);
      tc_fence_after();
      const int jl = (nch - 1) % WC;
      const long long e_abs = static_cast<long long>(cb + nch - 1 - jl) * kC + W - 1;
      const float fs = DECAY ? exp2f(static_cast<float>(static_cast<long long>(N - 1) - e_abs) * lg) : 1.f;
      float *srow = p.S_out + (static_cast<size_t>(bh) * kD + d) * kDV;
#pragma unroll 1
      for (int cc = 0; cc < kDV / 32; ++cc) {
        float x[32];
        tmem_ld32(tT + 32 * cc, x);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          reinterpret_cast<float4 *>(srow + 32 * cc)[q] =
              make_float4(fs * x[4 * q], fs * x[4 * q + 1], fs * x[4 * q + 2], fs * x[4 * q + 3]);
      }
      const float zd = tmem_ld1(tT + kDV);
      tmem_wait_ld();
      p.z_out[static_cast<size_t>(bh) * kD + d] = fs * zd;
    }
    if (lane == 0) bulk_wait_group0();  // every store complete before the CTA exits
  } else {
    // ---------------- P = A' masked to s <= t, bf16 pairs in place ----------------
    const int w = warp;  // TMEM lane quadrant
    const int t = 32 * w + lane;
    const uint32_t ta = tmem_addr(tmem, 32 * w, kColA);
    phase_a_map(warp);
    look_back(warp);
    for (int i = 0; i < nch; ++i) {
      if (!warp_wait(&bar[kAFull], i & 1, abort_flag, p.timeouts)) break;
      tc_fence_after();
      // A' columns [32 g, 32 g + 32) -> P pair columns [16 g, 16 g + 16): a
      // block wholly above this warp's diagonal is zero without a load
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t pk[16];
        if (g <= w) {
          float a[32];
          tmem_ld32(ta + 32 * g, a);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int s0 = 32 * g + 2 * e;
            pk[e] = pack_bf16x2(s0 <= t ? a[2 * e] : 0.f, s0 + 1 <= t ? a[2 * e + 1] : 0.f);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = 0u;
        }
        tmem_st16u(ta + 16 * g, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kPFull]);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

int num_sms128() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    return 148;
  return v;
}

// Relay split (see part_begin) from a cost model in units of one phase-C
// chunk: a phase-A chunk costs kPhaseARatio of one (it maps and multiplies
// k and v only), and a part that waits for earlier sums starts kLookBack
// chunks after they are published.  Part 0 runs n0 chunks from time 0; part
// 1 sums n0 - m0 chunks of it while part 0 reaches its checkpoint m0; parts
// 2.. sum the whole part before them, which takes as long when every later
// part has n = n0 / (1 + ratio) - kLookBack chunks; all parts then end
// together.
constexpr double kPhaseARatio = 0.40;
constexpr double kLookBack = 1.5;

void relay_split(int P, int nch, int *n0, int *m0) {
  *n0 = 0;
  *m0 = 0;
  if (P < 2) return;
  const double r = kPhaseARatio;
  int a = static_cast<int>((nch + (P - 1) * kLookBack) / (1.0 + (P - 1) / (1.0 + r)) + 0.5);
  if (a > nch - (P - 1)) a = nch - (P - 1);  // every later part keeps a chunk
  int m = static_cast<int>(r * a / (1.0 + r) + 0.5);
  if (m > a - 1) m = a - 1;
  if (a < 2 || m < 1) return;  // too short to gain: equal parts
  *n0 = a;
  *m0 = m;
}

size_t flag_bytes(int BH, int P) {
  const size_t flags = (static_cast<size_t>(BH) * P + 1) * sizeof(int);
  return (flags + 255) & ~static_cast<size_t>(255);
}

}  // namespace

bool chunk128_supported(const Problem &p, const Gammas &g) {
  if (p.dtype != kBF16 || p.D != kD || p.Dv != kDV || p.N <= 0) return false;
  const long long rows = static_cast<long long>(p.B) * p.H;
  if (rows <= 0 || rows * chunk128_parts(static_cast<int>(rows), p.N) >= (1LL << 31)) return false;
  if (p.decay)
    for (int h = 0; h < p.H; ++h)
      if (!(g.g[h] >= kGammaMin)) return false;
  return true;
}

int chunk128_parts(int BH, int N) {
  // at most one wave of CTAs (one per SM); a part's CTA pays phase A and
  // the chain links before it, so no more parts than minimise phase C +
  // chain: P ~ sqrt(0.43 * (N / 64))
  const int nch = (N + kC - 1) / kC;
  if (BH <= 0 || nch <= 0) return 1;
  int P = num_sms128() / BH;
  const int pmax = static_cast<int>(sqrt(0.43 * ((N + 63) / 64)));
  if (P > pmax) P = pmax;
  if (P > nch) P = nch;
  return P < 1 ? 1 : P;
}

size_t chunk128_workspace_bytes(int BH, int P) {
  if (P <= 1) return 0;
  return flag_bytes(BH, P) +
         sizeof(float) * static_cast<size_t>(BH) * P * (static_cast<size_t>(kD) * kDV + kD);
}

cudaError_t launch_causal_chunk128(const Problem &p, const Gammas &g, void *ws, int P, cudaStream_t s,
                                   float *S_out, float *z_out) {
  if (!chunk128_supported(p, g) || P < 1) return cudaErrorNotSupported;
  const int BH = p.B * p.H;
  Chunk128Params prm = {};
  if (!make_tmap_3d_bf16(&prm.tmQ, p.q, kD, p.N, BH, 64, kC, 128) ||
      !make_tmap_3d_bf16(&prm.tmK, p.k, kD, p.N, BH, 64, kC, 128) ||
      !make_tmap_3d_bf16(&prm.tmV, p.v, kDV, p.N, BH, 64, kC, 128) ||
      !make_tmap_3d_bf16(&prm.tmO, p.o, kDV, p.N, BH, 32, 32, 64))
    return cudaErrorNotSupported;
  prm.timeouts = wait_timeout_counter();
  if (!prm.timeouts) return cudaErrorNotSupported;
  prm.BH = BH;
  prm.H = p.H;
  prm.N = p.N;
  prm.P = P;
  prm.eps = p.eps;
  prm.S_out = S_out;
  prm.z_out = z_out;
  prm.lg = log2_gammas(g, p.H, p.decay);
  relay_split(P, (p.N + kC - 1) / kC, &prm.n0, &prm.m0);
  if (P > 1) {
    if (!ws) return cudaErrorInvalidValue;
    // flags and ticket start at zero; the records need no initialisation
    prm.ws_flag = static_cast<int *>(ws);
    prm.ws_ticket = prm.ws_flag + static_cast<size_t>(BH) * P;
    prm.rec = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + flag_bytes(BH, P));
    cudaError_t e = cudaMemsetAsync(ws, 0, (static_cast<size_t>(BH) * P + 1) * sizeof(int), s);
    if (e != cudaSuccess) return e;
  }
  auto kern = p.ident ? (p.decay ? chunk128_kernel<true, true> : chunk128_kernel<false, true>)
                      : (p.decay ? chunk128_kernel<true, false> : chunk128_kernel<false, false>);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (err != cudaSuccess) return err;
  kern<<<BH * P, kThreads, kAlloc, s>>>(prm);
  return cudaGetLastError();
}

cudaError_t launch_gated_chunk128(const Problem &p, const float *gate_prod, const float *gate_suf,
                                  const float *gate_part, const int *skip, void *ws, int P,
                                  cudaStream_t s, float *S_out, float *z_out) {
  if (p.dtype != kBF16 || p.D != kD || p.Dv != kDV || p.N <= 0 || !p.ident || P < 1)
    return cudaErrorNotSupported;
  const int BH = p.B * p.H;
  Chunk128Params prm = {};
  if (!make_tmap_3d_bf16(&prm.tmQ, p.q, kD, p.N, BH, 64, kC, 128) ||
      !make_tmap_3d_bf16(&prm.tmK, p.k, kD, p.N, BH, 64, kC, 128) ||
      !make_tmap_3d_bf16(&prm.tmV, p.v, kDV, p.N, BH, 64, kC, 128) ||
      !make_tmap_3d_bf16(&prm.tmO, p.o, kDV, p.N, BH, 32, 32, 64))
    return cudaErrorNotSupported;
  prm.timeouts = wait_timeout_counter();
  if (!prm.timeouts) return cudaErrorNotSupported;
  prm.BH = BH;
  prm.H = p.H;
  prm.N = p.N;
  prm.P = P;
  prm.eps = p.eps;
  prm.gate_prod = gate_prod;
  prm.gate_suf = gate_suf;
  prm.gate_part = gate_part;
  prm.skip = skip;
  // the state after the last token: T after the last chunk is relative to
  // that chunk's last token, N - 1, so it is written as it is
  prm.S_out = S_out;
  prm.z_out = z_out;
  if (P > 1) {
    if (!ws || !gate_suf || !gate_part) return cudaErrorInvalidValue;
    // flags and ticket start at zero; the records need no initialisation
    prm.ws_flag = static_cast<int *>(ws);
    prm.ws_ticket = prm.ws_flag + static_cast<size_t>(BH) * P;
    prm.rec = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + flag_bytes(BH, P));
    cudaError_t e = cudaMemsetAsync(ws, 0, (static_cast<size_t>(BH) * P + 1) * sizeof(int), s);
    if (e != cudaSuccess) return e;
  }
  Gammas ones;
  for (int h = 0; h < kMaxHeads; ++h) ones.g[h] = 1.f;
  prm.lg = log2_gammas(ones, p.H, false);
  auto kern = chunk128_kernel<false, true, true>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (err != cudaSuccess) return err;
  kern<<<BH * P, kThreads, kAlloc, s>>>(prm);
  return cudaGetLastError();
}

}  // namespace linattn
