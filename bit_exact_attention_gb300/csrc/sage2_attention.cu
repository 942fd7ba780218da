// sage2_attention.cu -- the fused SageAttention2 attention kernels for sm_103a.
//
// Two kernels share the helpers below. attn_pp (further down) computes two 128-row Q tiles per
// CTA and runs the method's INT4 codes, and their debug dumps. attn_fwd, described first,
// computes one tile per CTA. It runs the INT8-code path, the debug unit whose producer issues
// nothing, and the INT4 codes when SAGE2_ATTN_PP=0.
//
// attn_fwd: one CTA per (sequence, q head, 128-row Q tile); twelve warps in three warpgroups:
//   warp 0      TMA producer (one lane): per KV tile the K codes, the transposed V codes,
//               128 DeltaS*c values and 4 K scales into an ST-stage ring.
//   warps 1, 2  MMA issuers (one lane each), tcgen05 kind::f8f6f4 (e4m3 x e4m3 -> f32), A from
//               tensor memory, B from shared memory: warp 1 issues S(j) = Qcode Kcode(j)^T as
//               soon as S is free, warp 2 issues R(j) = P~(j) V(j) into R[j%2] as soon as P~(j)
//               is written, so neither stream waits behind the other.
//   warp 3      idle (it only gives its registers away).
//   warps 4-7   softmax: thread t of warp 4+w owns accumulator row 32w+t (its TMEM lane). It
//               first stores its row's Q codes into tensor memory (the A operand of Q K^T).
//               Per 128-key tile it loads the S row into registers (freeing S for the next
//               Q K^T at once), dequantizes and adds DeltaS with one FMA per element, takes the
//               row maximum, computes P448 = 2^(S' - m + log2 448) in base 2, writes
//               P~ = e4m3(P448) into tensor memory (the A operand of the P~V MMA) and hands
//               alpha = 2^(m_old - m_new) to the fold. The load of S(j) is issued before the
//               other waits of tile j, and P~(j-1) is handed over after it, so their latencies
//               overlap.
//   warps 8-11  fold + epilogue: thread t of warp 8+w owns row 32w+t of the FP32 output in
//               registers and folds each fresh per-tile partial: O = alpha O + R. At the end it
//               divides by the row sum and writes the output row.
// setmaxnreg moves registers from the control warpgroup to the softmax and fold warpgroups.
// Method (SageAttention2 pages): INT4-grid Q and K codes with per-thread-group scales; P~ and
// V in e4m3; two-level accumulation of P~V ("SageAttention2: Efficient Attention with Thorough
// Outlier Smoothing and Per-thread INT4 Quantization" research note, components 2 and 3;
// "SageAttention2 and Fast Exact INT4 Attention" visual companion, Numerical Repair Stack).
//
// The integer products are exact: codes lie in [-7, 7], stored as e4m3 (exact), products are
// at most 49 and a 128-channel dot product at most 6272 < 2^24, so the FP32 accumulator holds
// the integer Q K^T exactly.
//
// Tensor memory (512 columns allocated): S [0,128) R0 [128, 128+Dp) R1 [256, 256+Dp)
// P~0 [384,416) P~1 [416,448) Q [448, 448+Dp/4).
// Ordering: QK(j+1) overwrites S once the softmax has read S(j) (s_free); PV(j) overwrites
// R[j%2] once the fold of tile j-2 has read it (r_free[j%2]); the softmax of tile j rewrites
// P~[j%2] only after PV(j-2) is complete (pv_done[j%2]). Every mbarrier is waited on at most
// one phase behind its next completion, so parity waits cannot alias. The alpha of tile j
// travels through a 4-deep shared ring; tile j+4 writes its slot only after PV(j+2), which needs
// the fold of tile j.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <mutex>

#include "sage2_device.cuh"
#include "sage2_internal.h"

namespace sage2 {
namespace {

#ifndef SAGE2_TMA_WARP
#define SAGE2_TMA_WARP 0
#endif
#ifndef SAGE2_QK_WARP
#define SAGE2_QK_WARP 1
#endif
#ifndef SAGE2_PV_WARP
#define SAGE2_PV_WARP 2
#endif
constexpr int kTmaWarp = SAGE2_TMA_WARP, kMmaWarp = SAGE2_QK_WARP, kPvWarp = SAGE2_PV_WARP,
              kSmWarp0 = 4, kFoldWarp0 = 8;
static_assert(kSmWarp0 == 4 && kFoldWarp0 == 8, "softmax warps 4-7, fold warps 8-11");
static_assert(kTmaWarp >= 0 && kTmaWarp < 4 && kMmaWarp >= 0 && kMmaWarp < 4 && kPvWarp >= 0 &&
                  kPvWarp < 4 && kTmaWarp != kMmaWarp && kTmaWarp != kPvWarp &&
                  kMmaWarp != kPvWarp,
              "the producer and the issuers are distinct warps of the control warpgroup");
constexpr int kNumWarps = 12, kThreads = 32 * kNumWarps;
// Registers per thread after the split (the launch gives every warpgroup 128; setmaxnreg.inc
// waits until the other warpgroups have released enough, so the sum must stay within 4 x 128).
constexpr int kRegsLaunch = 168;  // 65536 registers / 384 threads, in steps of 8
constexpr int kRegsCtl = 40, kRegsSoftmax = 232, kRegsFold = 200;
static_assert(kRegsCtl + kRegsSoftmax + kRegsFold <= 3 * kRegsLaunch,
              "register split above the launch budget");
// setmaxnreg.dec may only lower and setmaxnreg.inc only raise the current count
static_assert(kRegsCtl <= kRegsLaunch, "the control warpgroup releases");
static_assert(kRegsSoftmax >= kRegsLaunch && kRegsFold >= kRegsLaunch,
              "the softmax and fold warpgroups acquire");
constexpr uint32_t kColS = 0, kColR0 = 128, kColR1 = 256, kColP0 = 384, kColP1 = 416,
                   kColQ = 448;
constexpr uint32_t kTmemCols = 512;

// wait-site ids reported in the status word
enum : int {
  kSiteQ = 1, kSiteKvFull = 2, kSiteKvEmpty = 3, kSiteSFull = 4, kSitePFull = 5, kSiteRFull = 6,
  kSiteRFree = 7, kSiteKvFullSm = 8, kSiteAFull = 9, kSiteLFull = 10, kSiteSFree = 11,
  kSitePvDone = 12
};

struct AttnArgs {
  Geometry g;
  Layout L;
  const float *qscale, *kscale, *dsc, *vscale;
  const uint8_t *qcode;
  void *out;
  int out_dtype;
  int *status;
  const int *seq_order;  // varlen: the sequence each z index takes (two-tile kernel)
  int hq0, hq_n;         // the q heads [hq0, hq0 + hq_n) of this launch
  AttnDebug dbg;
};

template <int DP, int ST, bool I8>
struct SmemPlan {
  // K codes: e4m3 bytes, or fp16 values of the INT8-grid codes (I8) stored as DP / 64 blocks of
  // 64 channels (128-byte swizzled rows, 16 KB per block)
  static constexpr int kKStage = 128 * DP * (I8 ? 2 : 1);
  static constexpr int kK = 0;                           // [ST][128 keys][DP]     (swizzled)
  static constexpr int kV = kK + ST * kKStage;           // [ST][DP][128 keys]     (swizzled)
  static constexpr int kDsc = kV + ST * DP * 128;        // float [ST][128]
  static constexpr int kSk = kDsc + ST * 512;            // float [ST][4]
  static constexpr int kAlpha = kSk + ST * 16;           // float [4][128]
  static constexpr int kLsum = kAlpha + 4 * 128 * 4;     // float [128]
  static constexpr int kSv = kLsum + 128 * 4;            // float [4 fold warps][DP]
  static constexpr int kBar = kSv + 4 * DP * 4;
  // q, full[ST], empty[ST], s_full, s_free, p_full[2], pv_done[2], r_free[2], a[4], l, drain[2]
  static constexpr int kNumBars = 1 + 2 * ST + 1 + 1 + 2 + 2 + 2 + 4 + 1 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kEnd = kMisc + 16;
  static constexpr int kBytes = kEnd + 1024;  // + alignment slack
  static_assert(kBytes <= 227 * 1024, "shared memory plan too large");
};

// Waits that ignore the abort flag (used to drain copies and MMAs already in flight).
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > SAGE2_WAIT_NS) return false;
  return true;
}

__device__ __forceinline__ bool warp_all(bool ok) {
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// S' = A * (s_q c s_k) + DeltaS c for 64 keys (one FMA each), masked beyond `lim`, and their max.
// Without DeltaS (the INT8 path, no Q smoothing) the addend is +0, as in the definition.
template <bool DS>
__device__ __forceinline__ float logits64(float (&x)[64], const uint32_t (&v)[64], const float *dsc,
                                          const float *skv, float sqc, int lim) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const float mult = __fmul_rn(sqc, skv[c]);
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 d4 =
          DS ? *reinterpret_cast<const float4 *>(dsc + c * 32 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      const int k0 = c * 32 + e;
      fma2(x[k0], x[k0 + 1], __uint_as_float(v[k0]), __uint_as_float(v[k0 + 1]), mult, mult, d4.x,
           d4.y);
      fma2(x[k0 + 2], x[k0 + 3], __uint_as_float(v[k0 + 2]), __uint_as_float(v[k0 + 3]), mult,
           mult, d4.z, d4.w);
    }
  }
  if (lim < 63) {  // diagonal / ragged tile: keys beyond lim are not visible
#pragma unroll
    for (int e = 0; e < 64; ++e) x[e] = (e <= lim) ? x[e] : -INFINITY;
  }
  float mk[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) mk[k] = fmaxf(x[16 * k], x[16 * k + 1]);
#pragma unroll
  for (int e = 2; e < 16; e += 2)
#pragma unroll
    for (int k = 0; k < 4; ++k) mk[k] = max3(mk[k], x[16 * k + e], x[16 * k + e + 1]);
  return max3(mk[0], mk[1], fmaxf(mk[2], mk[3]));
}

// The logits of one 128-key tile of a softmax row, on packed FP32 pairs (key 2k in x[k].x, key
// 2k + 1 in x[k].y): S' = fma(A, fl32(sqc * s_K), DeltaS c), one K scale per 32 keys, -inf
// beyond key `lim`; returns the row maximum of the tile.
__device__ __forceinline__ float logits128(float2 (&x)[64], const uint32_t (&v)[128],
                                           const float *dsc, const float *skv, float sqc, int lim) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float mult = __fmul_rn(sqc, skv[c]);
    const float2 m2 = make_float2(mult, mult);
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 d4 = *reinterpret_cast<const float4 *>(dsc + c * 32 + e);
      const int k = (c * 32 + e) >> 1;
      x[k] = __ffma2_rn(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), m2,
                        make_float2(d4.x, d4.y));
      x[k + 1] =
          __ffma2_rn(make_float2(__uint_as_float(v[2 * k + 2]), __uint_as_float(v[2 * k + 3])), m2,
                     make_float2(d4.z, d4.w));
    }
  }
  if (lim < 127) {  // diagonal / ragged tile: keys beyond lim are not visible
#pragma unroll
    for (int k = 0; k < 64; ++k) {
      x[k].x = (2 * k <= lim) ? x[k].x : -INFINITY;
      x[k].y = (2 * k + 1 <= lim) ? x[k].y : -INFINITY;
    }
  }
  float mk[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) mk[q] = fmaxf(x[q].x, x[q].y);
#pragma unroll
  for (int k = 4; k < 64; ++k) mk[k & 3] = max3(mk[k & 3], x[k].x, x[k].y);
  return max3(mk[0], mk[1], fmaxf(mk[2], mk[3]));
}

// P448 = 2^(S' - m448) for the 128 keys of a row (masked keys give 0), their sum (pairs summed
// into four accumulators by pair index mod 4, then combined in a fixed order) and the e4m3 codes
// P~ = e4m3(P448), key 4e + i in byte i of pk[e]. The codes of each 32-key chunk are stored to
// the row's P~ buffer `prow` (16-byte piece c at position c ^ (row & 7), the 128-byte swizzle)
// as soon as they exist, so the stores drain while the next chunk's exponentials run.
__device__ __forceinline__ float probs128(float2 (&x)[64], float m448, uint32_t (&pk)[32],
                                          uint8_t *prow, int row) {
  const float2 nm = make_float2(-m448, -m448);
  float2 ps[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) ps[q] = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int k = 16 * c; k < 16 * c + 16; ++k) {
      x[k] = __fadd2_rn(x[k], nm);
      x[k].x = ex2_approx(x[k].x);
      x[k].y = ex2_approx(x[k].y);
    }
#pragma unroll
    for (int k = 16 * c; k < 16 * c + 16; ++k) ps[k & 3] = __fadd2_rn(ps[k & 3], x[k]);
#pragma unroll
    for (int e = 8 * c; e < 8 * c + 8; ++e)
      pk[e] = cvt_e4m3x4(x[2 * e].x, x[2 * e].y, x[2 * e + 1].x, x[2 * e + 1].y);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      *reinterpret_cast<uint4 *>(prow + (((2 * c + h) ^ (row & 7)) << 4)) =
          make_uint4(pk[8 * c + 4 * h], pk[8 * c + 4 * h + 1], pk[8 * c + 4 * h + 2],
                     pk[8 * c + 4 * h + 3]);
  }
  return __fadd_rn(__fadd_rn(__fadd_rn(ps[0].x, ps[0].y), __fadd_rn(ps[1].x, ps[1].y)),
                   __fadd_rn(__fadd_rn(ps[2].x, ps[2].y), __fadd_rn(ps[3].x, ps[3].y)));
}


// probs128 for P~ in tensor memory (D = 64): each 32-key chunk's 8 code words go to columns
// tP + 8c with one 32x32b.x8 store as soon as they exist; the caller waits for the stores
// before the hand-over.
__device__ __forceinline__ float probs128_tm(float2 (&x)[64], float m448, uint32_t (&pk)[32],
                                             uint32_t tP) {
  const float2 nm = make_float2(-m448, -m448);
  float2 ps[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) ps[q] = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int k = 16 * c; k < 16 * c + 16; ++k) {
      x[k] = __fadd2_rn(x[k], nm);
      x[k].x = ex2_approx(x[k].x);
      x[k].y = ex2_approx(x[k].y);
    }
#pragma unroll
    for (int k = 16 * c; k < 16 * c + 16; ++k) ps[k & 3] = __fadd2_rn(ps[k & 3], x[k]);
    uint32_t w8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      pk[8 * c + e] = cvt_e4m3x4(x[2 * (8 * c + e)].x, x[2 * (8 * c + e)].y,
                                 x[2 * (8 * c + e) + 1].x, x[2 * (8 * c + e) + 1].y);
      w8[e] = pk[8 * c + e];
    }
    tmem_st8(tP + 8 * c, w8);
  }
  return __fadd_rn(__fadd_rn(__fadd_rn(ps[0].x, ps[0].y), __fadd_rn(ps[1].x, ps[1].y)),
                   __fadd_rn(__fadd_rn(ps[2].x, ps[2].y), __fadd_rn(ps[3].x, ps[3].y)));
}

// End of every role branch: all 512 threads meet once more (each warp from its own branch, so
// the per-warpgroup register budgets never merge into one code path), then the MMA warp frees
// tensor memory.
__device__ __forceinline__ void cta_teardown(bool owner, uint32_t tbase) {
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (owner) tmem_dealloc(tbase, kTmemCols);
}

template <int DP, int ST, bool DBG, bool I8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
             const AttnArgs a) {
  using P = SmemPlan<DP, ST, I8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const Geometry &g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the code format recorded by the prepass (loaded together with the sequence bounds below)
  const int format = a.status[1];

  int b, hq, qt;
  if (DBG) {
    b = a.dbg.b;
    hq = a.dbg.h;
    qt = a.dbg.qt;
  } else {
    // launch order as in attn_pp: varlen sequences longest K/V first, then (tile x head) with
    // all heads of a tile index together, heaviest first under causal masks
    b = blockIdx.z;
    if (g.cu_kv) {
      const int ob = a.seq_order[blockIdx.z];
      if (ob >= 0 && ob < g.B) b = ob;
    }
    hq = a.hq0 + (int)blockIdx.x % a.hq_n;
    const int ntiles = (int)gridDim.x / a.hq_n, tidx = (int)blockIdx.x / a.hq_n;
    qt = g.causal ? ntiles - 1 - tidx : tidx;
  }
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (format != (I8 ? kFormatInt8 : kFormatInt4)) {  // a workspace of the other code format
    if (tid == 0) atomicCAS(a.status, 0, kStatusFormat);
    return;
  }
  if (!s.ok || qt * kBQ >= s.nq) return;
  const int hk = hq / (g.Hq / g.Hkv);
  const int T = kv_tiles_for(qt, s.nq, s.nkv, g.causal);
  const size_t out_row0 = (size_t)(s.q0 + qt * kBQ) * g.Hq + hq;  // in rows of D0 elements

  if (T == 0) {  // no visible key for any row of this tile: the output is 0
    if (tid < kBQ && qt * kBQ + tid < s.nq) {
      const size_t o = (out_row0 + (size_t)tid * g.Hq) * g.D0;
      for (int d = 0; d < g.D0; ++d) {
        if (a.out_dtype == SAGE2_FP32)
          static_cast<float *>(a.out)[o + d] = 0.f;
        else
          static_cast<uint16_t *>(a.out)[o + d] = 0;
      }
    }
    return;
  }

  float *alpha_ring = reinterpret_cast<float *>(smem + P::kAlpha);
  float *lsum = reinterpret_cast<float *>(smem + P::kLsum);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::kBar);
  uint64_t *q_full = bars;
  uint64_t *kv_full = bars + 1;
  uint64_t *kv_empty = kv_full + ST;
  uint64_t *s_full = kv_empty + ST;  // completed by QK(j), once per tile
  uint64_t *s_free = s_full + 1;     // completed when the softmax has read S(j)
  uint64_t *p_full = s_free + 1;     // [2]
  uint64_t *pv_done = p_full + 2;    // [2]
  uint64_t *r_free = pv_done + 2;    // [2]
  uint64_t *a_full = r_free + 2;     // [4]
  uint64_t *l_full = a_full + 4;
  uint64_t *drain = l_full + 1;     // [2]: one per MMA-issuing warp
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + P::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P::kMisc + 4);

  if (warp == kTmaWarp && lane == 0) {
    mbar_init(q_full, 4);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(s_free, 4);
    mbar_init(s_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
      mbar_init(&r_free[i], 4);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&a_full[i], 4);
    mbar_init(l_full, 4);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const AbortCtx ab{abort_flag, a.status};

  if (warp < 4) {
    regs_release<kRegsCtl>();
    if (warp == kTmaWarp && lane == 0) {
    // ------------------------------------------------------------ TMA producer (one lane)
      const int yk0 = hk * a.L.Tkv + s.kvpad0;
      const float *dsc_row =
          a.dsc + ((size_t)hq * a.L.nqblk + s.qpad0 / kBQ + qt) * a.L.nkv_pad;
      const float *sk_row = a.kscale + (size_t)hk * (a.L.Tkv / kGK) + s.kvpad0 / kGK;
      const bool skip = DBG && a.dbg.skip_loads;
      int issued = 0;
      for (int j = 0; j < T; ++j) {
        const int st = j % ST;
        if (j >= ST && !mbar_wait<true>(&kv_empty[st], ((j / ST) - 1) & 1, ab, kSiteKvEmpty)) break;
        if (skip) continue;
        mbar_arrive_expect_tx(&kv_full[st], P::kKStage + DP * 128 + (I8 ? 0 : 512) + 16);
        if (I8) {  // 64-channel blocks of fp16 codes: inner coordinate 64 h (128 bytes)
#pragma unroll
          for (int hb = 0; hb < DP / 64; ++hb)
            tma_load_2d(smem + P::kK + st * P::kKStage + hb * 16384, &tm_k, 64 * hb,
                        yk0 + j * kBKV, &kv_full[st]);
        } else {
          tma_load_2d(smem + P::kK + st * P::kKStage, &tm_k, 0, yk0 + j * kBKV, &kv_full[st]);
        }
        tma_load_2d(smem + P::kV + st * DP * 128, &tm_v, s.kvpad0 + j * kBKV, hk * DP,
                    &kv_full[st]);
        if (!I8)
          bulk_load(smem + P::kDsc + st * 512, dsc_row + (size_t)j * kBKV, 512, &kv_full[st]);
        bulk_load(smem + P::kSk + st * 16, sk_row + j * (kBKV / kGK), 16, &kv_full[st]);
        issued = j + 1;
      }
      if (*abort_flag) {  // let the copies already issued land before the CTA exits
        for (int n = issued > ST ? issued - ST : 0; n < issued; ++n)
          drain_wait(&kv_full[n % ST], (n / ST) & 1);
      }
    } else if (warp == kMmaWarp && lane == 0) {
    // ------------------------------------------------------------ Q K^T issuer (one lane)
      constexpr uint32_t idesc_qk = idesc_e4m3_f32(128, 128);
      bool ok = mbar_wait(q_full, 0, ab, kSiteQ);
      for (int j = 0; ok && j < T; ++j) {
        // S is free once the four warps of tile j-1 have read it
        ok = (j == 0 || mbar_wait<true>(s_free, (j - 1) & 1, ab, kSiteSFree)) &&
             mbar_wait<true>(&kv_full[j % ST], (j / ST) & 1, ab, kSiteKvFull);
        if (!ok) break;
        tc_fence_after();
        if (I8) {  // fp16 codes, 16 channels (32 bytes, 8 TMEM columns of A) per MMA
          const uint64_t kdesc = sdesc_kmajor(smem_u32(smem + P::kK + (j % ST) * P::kKStage), 128);
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk)
            mma_f16_ts(tbase + kColS, tbase + kColQ + kk * 8,
                       kdesc + (uint64_t)((kk & 3) * 2 + (kk >> 2) * (16384 >> 4)), idesc_qk,
                       kk > 0);
        } else {
          const uint64_t kdesc = sdesc_kmajor(smem_u32(smem + P::kK + (j % ST) * P::kKStage), DP);
#pragma unroll
          for (int kk = 0; kk < DP / 32; ++kk)  // A = the Q codes in tensor memory
            mma_e4m3_ts(tbase + kColS, tbase + kColQ + kk * 8, kdesc + (uint64_t)(kk * 2),
                        idesc_qk, kk > 0);
        }
        mma_commit(s_full);
      }
      mma_commit(&drain[0]);  // every MMA issued above completes before tensor memory is freed
      drain_wait(&drain[0], 0);
    } else if (warp == kPvWarp && lane == 0) {
    // ------------------------------------------------------------ P~ V issuer (one lane)
      constexpr uint32_t idesc_pv = idesc_e4m3_f32(128, DP);
      bool ok = true;
      for (int j = 0; ok && j < T; ++j) {
        // P~(j) V(j) once its P~ tile is written and the fold of tile j-2 has read R[j%2]
        ok = mbar_wait<true>(&p_full[j & 1], (j >> 1) & 1, ab, kSitePFull) &&
             (j < 2 || mbar_wait<true>(&r_free[j & 1], ((j - 2) >> 1) & 1, ab, kSiteRFree));
        if (!ok) break;
        tc_fence_after();
        const uint64_t vdesc = sdesc_kmajor(smem_u32(smem + P::kV + (j % ST) * DP * 128), 128);
        const uint32_t d = tbase + ((j & 1) ? kColR1 : kColR0);
        const uint32_t aP = tbase + ((j & 1) ? kColP1 : kColP0);  // P~(j) in tensor memory
#pragma unroll
        for (int kk = 0; kk < kBKV / 32; ++kk)
          mma_e4m3_ts(d, aP + kk * 8, vdesc + (uint64_t)(kk * 2), idesc_pv, kk > 0);
        mma_commit(&pv_done[j & 1]);
        // K(j) was read by QK(j), complete before the softmax of tile j began
        mma_commit(&kv_empty[j % ST]);
      }
      mma_commit(&drain[1]);
      drain_wait(&drain[1], 0);
    }
    cta_teardown(warp == kMmaWarp, tbase);
  } else if (warp < kFoldWarp0) {
    regs_acquire<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax (4 warps)
    // thread t of softmax warp w owns accumulator row 32w+t (its TMEM lane), all 128 keys
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    const int i = qt * kBQ + row;
    const bool row_ok = i < s.nq;
    const float c32 = g.c32;
    const float sqc =
        row_ok ? __fmul_rn(a.qscale[(size_t)hq * a.L.Tq + s.qpad0 + qt * kBQ + row], c32) : 0.f;
    const int last_key = g.causal ? min(i + (s.nkv - s.nq), s.nkv - 1) : s.nkv - 1;
    const float L32 = 8.8073549220576041f;  // fl32(log2(448))
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t tS = tbase + lane_base + kColS;
    {  // the row's Q codes into tensor memory: the A operand of Q K^T
      constexpr int kRowBytes = DP * (I8 ? 2 : 1);
      const uint4 *qrow = reinterpret_cast<const uint4 *>(
          a.qcode + ((size_t)hq * a.L.Tq + s.qpad0 + qt * kBQ + row) * kRowBytes);
#pragma unroll
      for (int c = 0; c < kRowBytes / 32; ++c) {  // 32 bytes = 8 words per store
        const uint4 u0 = __ldg(qrow + 2 * c), u1 = __ldg(qrow + 2 * c + 1);
        const uint32_t w8[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        tmem_st8(tbase + lane_base + kColQ + 8 * c, w8);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    float m = -INFINITY, l = 0.f;
    // Latency overlap without carrying S across tiles: the load of S(j) is issued first and this
    // tile's other waits are tried while it is in flight; tile j-1's P~ (stored at its end) is
    // handed over to the MMA after the load, by when the store has landed.
    float alpha_prev = 1.f;
    int jprev = -1;  // tile whose P~ store is still to be handed over
    auto hand_over = [&]() {
      tmem_st_wait();
      tc_fence_before();
      alpha_ring[(jprev & 3) * 128 + row] = alpha_prev;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&p_full[jprev & 1]);
        mbar_arrive(&a_full[jprev & 3]);
      }
      jprev = -1;
    };
#pragma unroll 1
    for (int j = 0; j < T; ++j) {
      const int st = j % ST;
      const int pb = j & 1;
      bool ok = warp_all(mbar_wait(s_full, j & 1, ab, kSiteSFull));
      uint32_t v[128];
      if (ok) {
        tc_fence_after();
        tmem_ld128_nowait(tS, v);
      }
      if (!ok) {
        if (jprev >= 0) hand_over();
        break;
      }
      // this tile's K scales and DeltaS, and the P~ tile [j%2] free (PV(j-2) complete): one
      // try each while the load is in flight, the bounded wait after it if needed (keep loops,
      // barriers and tcgen05 waits out of the span between a load and its wait: ptxas then
      // spills the 128 pending registers)
      const bool kv_ready = mbar_try_wait(&kv_full[st], (j / ST) & 1);
      const bool pv_ready = (j < 2) || mbar_try_wait(&pv_done[pb], ((j - 2) >> 1) & 1);
      tmem_wait_ld128(v);  // S(j) is in registers: QK(j+1) may overwrite S
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      if (jprev >= 0) hand_over();  // tile j-1's P~ store has long landed by now
      ok = warp_all((kv_ready || mbar_wait(&kv_full[st], (j / ST) & 1, ab, kSiteKvFullSm)) &&
                    (pv_ready || mbar_wait(&pv_done[pb], ((j - 2) >> 1) & 1, ab, kSitePvDone)));
      if (!ok) break;
      if (DBG && j == a.dbg.kt) {
#pragma unroll
        for (int e = 0; e < 128; ++e) a.dbg.s_out[row * 128 + e] = __uint_as_float(v[e]);
      }
      const float *dsc = reinterpret_cast<const float *>(smem + P::kDsc + st * 512);
      const float *skv = reinterpret_cast<const float *>(smem + P::kSk + st * 16);
      const int lim = last_key - j * kBKV;  // keys 0..lim of this tile are visible
      float x[128];
      float pmax = -INFINITY;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float xh[64];
        uint32_t vh[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) vh[e] = v[64 * h + e];
        pmax = fmaxf(pmax, logits64<!I8>(xh, vh, dsc + 64 * h, skv + 2 * h, sqc, lim - 64 * h));
#pragma unroll
        for (int e = 0; e < 64; ++e) x[64 * h + e] = xh[e];
      }
      const float m_new = fmaxf(m, pmax);
      const bool none = (m_new == -INFINITY);  // no visible key so far in this row
      const float alpha = none ? 1.f : ex2_approx(__fsub_rn(m, m_new));
      const float m448 = none ? 0.f : __fsub_rn(m_new, L32);
      // P448 = 2^(S' - m448); masked keys have S' = -inf and give 0
#pragma unroll
      for (int e = 0; e < 128; e += 2) add2(x[e], x[e + 1], x[e], x[e + 1], -m448, -m448);
#pragma unroll
      for (int e = 0; e < 128; ++e) x[e] = ex2_approx(x[e]);
      float ps[4][2];
#pragma unroll
      for (int k = 0; k < 4; ++k) ps[k][0] = ps[k][1] = 0.f;
#pragma unroll
      for (int e = 0; e < 128; e += 2)
        add2(ps[(e >> 1) & 3][0], ps[(e >> 1) & 3][1], ps[(e >> 1) & 3][0], ps[(e >> 1) & 3][1],
             x[e], x[e + 1]);
      const float rs = __fadd_rn(
          __fadd_rn(__fadd_rn(ps[0][0], ps[0][1]), __fadd_rn(ps[1][0], ps[1][1])),
          __fadd_rn(__fadd_rn(ps[2][0], ps[2][1]), __fadd_rn(ps[3][0], ps[3][1])));
      // P~ = e4m3(P448): 128 keys -> 32 words, into the P~ tile [j%2] in tensor memory; it is
      // handed over to the MMA at the top of the next tile (or after the last one)
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 32; ++e)
        pk[e] = cvt_e4m3x2(x[4 * e], x[4 * e + 1]) | (cvt_e4m3x2(x[4 * e + 2], x[4 * e + 3]) << 16);
      tmem_st32(tbase + lane_base + (pb ? kColP1 : kColP0), pk);
      if (DBG && j == a.dbg.kt) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          *reinterpret_cast<uint32_t *>(a.dbg.p_out + row * 128 + 4 * e) = pk[e];
      }
      alpha_prev = alpha;
      jprev = j;
      l = __fmaf_rn(alpha, l, rs);
      m = m_new;
    }
    if (jprev >= 0) hand_over();
    lsum[row] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(l_full);
    cta_teardown(false, tbase);
  } else {
    regs_acquire<kRegsFold>();
    // ------------------------------------------------------------ fold + epilogue (4 warps)
    // thread t of fold warp w folds row 32w+t: O = alpha O + R, O in registers
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    const int i = qt * kBQ + row;
    const bool row_ok = i < s.nq;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    // the V channel scales into this warp's own slice of shared memory now, so that the
    // epilogue does not wait on global loads
    float *sv_s = reinterpret_cast<float *>(smem + P::kSv) + qd * DP;
    {
      const float *svp = a.vscale + ((size_t)b * g.Hkv + hk) * DP;
      for (int c = lane; c < DP; c += 32) sv_s[c] = __ldg(svp + c);
    }
    float O[DP];
#pragma unroll
    for (int d = 0; d < DP; ++d) O[d] = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      ok = warp_all(mbar_wait<true>(&a_full[j & 3], (j >> 2) & 1, ab, kSiteAFull));
      if (!ok) break;
      const float alpha = alpha_ring[(j & 3) * 128 + row];
      ok = warp_all(mbar_wait<true>(&pv_done[j & 1], (j >> 1) & 1, ab, kSiteRFull));  // R(j) complete
      if (!ok) break;
      tc_fence_after();
      const uint32_t tR = tbase + lane_base + ((j & 1) ? kColR1 : kColR0);
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t r[32];
        tmem_ld32_wait(tR + 32 * c, r);
        if (c == DP / 32 - 1) {  // R[j%2] is read: PV(j+2) may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&r_free[j & 1]);
        }
        if (DBG && j == a.dbg.kt) {
#pragma unroll
          for (int e = 0; e < 32; ++e) a.dbg.r_out[row * DP + 32 * c + e] = __uint_as_float(r[e]);
        }
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          fma2(O[32 * c + e], O[32 * c + e + 1], alpha, alpha, O[32 * c + e], O[32 * c + e + 1],
               __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
      }
    }
    if (ok) ok = mbar_wait(l_full, 0, ab, kSiteLFull);
    ok = warp_all(ok);
    // ------------------------------------------------------------ epilogue
    if (warp_all(ok && !*abort_flag)) {
      const float l = lsum[row];
      const float inv_l = l > 0.f ? __frcp_rn(l) : 0.f;
      const size_t o = (out_row0 + (size_t)row * g.Hq) * g.D0;
      __syncwarp();  // the slice of channel scales is complete
#pragma unroll
      for (int c = 0; c < DP / 8; ++c) {
        const int d = 8 * c;
        if (row_ok && d < g.D0) {
          const float4 s0 = *reinterpret_cast<const float4 *>(sv_s + d);
          const float4 s1 = *reinterpret_cast<const float4 *>(sv_s + d + 4);
          const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(O[d + e], sv[e]), inv_l);
          if (a.out_dtype == SAGE2_FP32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + o + d);
            dst[0] = make_float4(y[0], y[1], y[2], y[3]);
            dst[1] = make_float4(y[4], y[5], y[6], y[7]);
          } else {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint16_t lo, hi;
              if (a.out_dtype == SAGE2_BF16) {
                lo = __bfloat16_as_ushort(__float2bfloat16_rn(y[2 * e]));
                hi = __bfloat16_as_ushort(__float2bfloat16_rn(y[2 * e + 1]));
              } else {
                lo = __half_as_ushort(__float2half_rn(y[2 * e]));
                hi = __half_as_ushort(__float2half_rn(y[2 * e + 1]));
              }
              w[e] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + o + d) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
    cta_teardown(false, tbase);
  }
}

// ---------------------------------------------------------------- two-tile kernel
// One CTA per (sequence, q head, pair of 128-row Q tiles); the two tiles share every K and V
// stage, so each K/V byte brought in feeds twice the tensor work. Warps: 0 loads Q, K and the
// DeltaS*c / K-scale ring, 1 Q K^T issuer, 2 P~V issuer, 3 stages the V channel scales and then
// loads V, 4-7 softmax + epilogue of tile 0, 8-11 of tile 1 (each SM sub-partition runs one
// softmax warp of each tile, so one tile's arithmetic fills the other's waits).
// Three rings with their own barriers: K stage n is free once QK_0(n) and QK_1(n) complete, so
// the next K tiles load well ahead; V stage n and DeltaS*c / K-scale stage n (read by the
// softmax) once PV_0(n) and PV_1(n) complete. With one ring for all of them a stage stayed
// held until the P~V products, and the K load of tile n + ST sat on the critical path.
// Per tile t: tensor memory S_t [256 t, 256 t + 128) and O_t [256 t + 128, 256 t + 128 + DP) (the
// FP32 output accumulator); Q_t codes in shared memory, and two P~_t buffers (128 x 128 e4m3, the
// A operand of P~V): in shared memory, 128-byte swizzled K-major, at D = 128; in the 64 free
// tensor-memory columns of the tile at D = 64 (no shared-memory stores, no proxy fence, and the
// P~V MMA reads only V from shared memory). Per KV tile j the softmax loads S_t(j) into
// registers and releases S_t at once, so QK_t(j+1) runs while it computes P~_t(j). If a row
// maximum of the warp moved, it waits for PV_t(j-1) and rescales O_t by alpha(j) in tensor memory.
// It writes P~_t(j) into buffer j % 2 (free: QK_t(j) is issued only after PV_t(j-2) completed)
// and hands it to the P~V issuer; PV_t(j) then adds the block partial P~(j) V(j) into O_t.
// The two issuers are separate threads: issuing a group of MMAs blocks the issuing thread while
// the tensor pipe is busy (a few hundred cycles per group), and with one thread for both
// products each P~V issue delayed the next Q K^T of both tiles by that much. Each follows a fixed
// order (n = 0, 1, ..., tile 0 then tile 1) with blocking waits: polling several barriers in turn
// kept the issuer's sub-partition busy and slowed the softmax warps sharing it, which paced the
// whole CTA. tcgen05.commit covers the MMAs of the issuing thread only, so each issuer signals its
// own products: s_full_t after QK_t(n), pv_done[t][n % 2] after PV_t(n), k_empty(n) after the
// two QK(n), v_empty(n) and d_empty(n) after the two PV(n).
template <int DP, int ST>
struct PPPlan {
  static constexpr int kQ = 0;                       // [2][128 rows][DP]   (swizzled)
  // [2 tiles][2][128][128] (128B swizzled); at D = 64 the P~ buffers live in tensor memory
  static constexpr int kP = kQ + 2 * 128 * DP;
  static constexpr int kK = kP + (DP == 128 ? 4 * 128 * 128 : 0);      // [ST][128 keys][DP]  (swizzled)
  static constexpr int kV = kK + ST * 128 * DP;      // [ST][DP][128 keys]  (swizzled)
  static constexpr int kDS = 4;                      // DeltaS*c / K-scale stages
  static constexpr int kDsc = kV + ST * DP * 128;    // float [kDS][2][128]
  static constexpr int kSk = kDsc + kDS * 2 * 512;   // float [kDS][4]
  static constexpr int kSv = kSk + kDS * 16;         // float [DP]
  static constexpr int kBar = kSv + DP * 4;
  // q, k_full[ST], k_empty[ST], v_full[ST], v_empty[ST], d_full[kDS], d_empty[kDS], s_full[2],
  // s_free[2], p_full[2][2], pv_done[2][2], drain[2]
  static constexpr int kNumBars = 1 + 4 * ST + 2 * kDS + 2 + 2 + 4 + 4 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kEnd = kMisc + 16;
  static constexpr int kBytes = kEnd + 1024;
  static_assert(kBytes <= 227 * 1024, "shared memory plan too large");
};
// register split: the control warpgroup keeps 56 (its loops spilled at 40), the two softmax
// warpgroups take 224 each (56 + 2 x 224 = 3 x 168, the launch budget)
constexpr int kPPRegsCtl = 56, kPPRegsSoftmax = 224;
// sleep between barrier tests of the producer and the two issuers (measured best on the long
// GQA workload; the producer's waits were the most sensitive: 1000 ns cost 7 %)
constexpr uint32_t kPollProducerNs = 64, kPollQkNs = 64, kPollPvNs = 100;
static_assert(kPPRegsCtl + 2 * kPPRegsSoftmax <= 3 * kRegsLaunch, "register split above budget");
static_assert(kPvWarp != 3, "warp 3 stages the V channel scales");
// tensor-memory columns of tile t: S at 256 t, O at 256 t + 128
__device__ __forceinline__ uint32_t pp_col_s(int t) { return (uint32_t)t * 256u; }
__device__ __forceinline__ uint32_t pp_col_o(int t) { return (uint32_t)t * 256u + 128u; }
// D = 64: P~ buffer b of tile t in the 64 tensor-memory columns after O_t
__device__ __forceinline__ uint32_t pp_col_p(int t, int b) {
  return (uint32_t)t * 256u + 192u + 32u * (uint32_t)b;
}

// One 128-row tile's output rows from the FP32 accumulator in tensor memory: O * vscale / l,
// rounded to the output type (row `row` of the tile, `o` its element offset in the output).
template <int DP>
__device__ __forceinline__ void store_out_row(const AttnArgs &a, uint32_t tO, const float *sv_s,
                                              float l, bool row_ok, size_t o) {
  const float inv_l = l > 0.f ? __frcp_rn(l) : 0.f;
#pragma unroll
  for (int c = 0; c < DP / 32; ++c) {
    uint32_t r[32];
    tmem_ld32_wait(tO + 32 * c, r);
#pragma unroll
    for (int e8 = 0; e8 < 32; e8 += 8) {
      const int d = 32 * c + e8;
      if (row_ok && d < a.g.D0) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          y[e] = __fmul_rn(__fmul_rn(__uint_as_float(r[e8 + e]), sv_s[d + e]), inv_l);
        if (a.out_dtype == SAGE2_FP32) {
          float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + o + d);
          dst[0] = make_float4(y[0], y[1], y[2], y[3]);
          dst[1] = make_float4(y[4], y[5], y[6], y[7]);
        } else {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint16_t lo, hi;
            if (a.out_dtype == SAGE2_BF16) {
              lo = __bfloat16_as_ushort(__float2bfloat16_rn(y[2 * e]));
              hi = __bfloat16_as_ushort(__float2bfloat16_rn(y[2 * e + 1]));
            } else {
              lo = __half_as_ushort(__float2half_rn(y[2 * e]));
              hi = __half_as_ushort(__float2half_rn(y[2 * e + 1]));
            }
            w[e] = (uint32_t)lo | ((uint32_t)hi << 16);
          }
          *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + o + d) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
}

// DBG: one CTA, the pair holding Q tile a.dbg.qt of (sequence a.dbg.b, head a.dbg.h); the
// softmax warps of that tile dump S(kt) (the raw integer accumulators) and P~(kt), and for
// kt = 0 the first block partial P~(0) V(0), which is O after PV(0).
template <int DP, int ST, bool DBG>
__global__ void __launch_bounds__(kThreads, 1)
    attn_pp(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using P = PPPlan<DP, ST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Geometry &g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int format = a.status[1];
  // Launch order (the order CTAs start in): z sequences, longest K/V first for varlen calls
  // (the prepass's order); within a sequence the pairs in x-major (pair index, q head) order,
  // heaviest pair first under causal masks, all heads of a pair index together. Starting the
  // longest CTAs first keeps them out of the tail.
  int b = (int)blockIdx.z;
  if (!DBG && g.cu_kv) {
    const int ob = a.seq_order[blockIdx.z];
    if (ob >= 0 && ob < g.B) b = ob;  // (a workspace of another prepass keeps the batch order)
  }
  if (DBG) b = a.dbg.b;
  const int npairs = (int)gridDim.x / a.hq_n, pidx = (int)blockIdx.x / a.hq_n;
  const int hq = DBG ? a.dbg.h : a.hq0 + (int)blockIdx.x % a.hq_n;
  const int pair = DBG ? a.dbg.qt / 2 : (g.causal ? npairs - 1 - pidx : pidx);
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (format != kFormatInt4) {
    if (tid == 0) atomicCAS(a.status, 0, kStatusFormat);
    return;
  }
  if (!s.ok || 2 * pair * kBQ >= s.nq) return;
  const int hk = hq / (g.Hq / g.Hkv);
  int qtt[2], Tt[2];
  bool valid[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    qtt[t] = 2 * pair + t;
    valid[t] = qtt[t] * kBQ < s.nq;
    Tt[t] = valid[t] ? kv_tiles_for(qtt[t], s.nq, s.nkv, g.causal) : 0;
  }
  const int Tmax = max(Tt[0], Tt[1]);
  if (Tmax == 0) {  // no visible key for any row of either tile: the output is 0
    for (int t = 0; t < 2; ++t)
      if (valid[t] && tid < kBQ && qtt[t] * kBQ + tid < s.nq) {
        const size_t o = ((size_t)(s.q0 + qtt[t] * kBQ + tid) * g.Hq + hq) * g.D0;
        for (int d = 0; d < g.D0; ++d) {
          if (a.out_dtype == SAGE2_FP32)
            static_cast<float *>(a.out)[o + d] = 0.f;
          else
            static_cast<uint16_t *>(a.out)[o + d] = 0;
        }
      }
    return;
  }

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::kBar);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + ST;      // QK_0(n), QK_1(n) complete
  uint64_t *v_full = k_empty + ST;
  uint64_t *v_empty = v_full + ST;      // PV_0(n), PV_1(n) complete
  uint64_t *d_full = v_empty + ST;      // DeltaS*c rows and K scales of tile n
  uint64_t *d_empty = d_full + P::kDS;  // PV_0(n), PV_1(n) complete
  uint64_t *s_full = d_empty + P::kDS;  // [2] QK_t(j) complete
  uint64_t *s_free = s_full + 2;      // [2] the softmax of tile t has read S_t(j)
  uint64_t *p_full = s_free + 2;      // [2][2] P~_t(j) written into buffer j % 2, O_t rescaled
  uint64_t *pv_done = p_full + 4;     // [2][2] PV_t(n) complete, by n % 2
  uint64_t *drain = pv_done + 4;      // [2] one per issuer
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + P::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P::kMisc + 4);
  float *sv_s = reinterpret_cast<float *>(smem + P::kSv);

  if (warp == kTmaWarp && lane == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < P::kDS; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], 4);
      for (int k = 0; k < 2; ++k) {
        mbar_init(&p_full[2 * t + k], 4);
        mbar_init(&pv_done[2 * t + k], 1);
      }
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 3) {  // the V channel scales for the epilogue
    const float *svp = a.vscale + ((size_t)b * g.Hkv + hk) * DP;
    for (int c = lane; c < DP; c += 32) sv_s[c] = __ldg(svp + c);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const AbortCtx ab{abort_flag, a.status};
  const int T0 = Tt[0], T1 = Tt[1];

  if (warp < 4) {
    regs_release<kPPRegsCtl>();
    if (warp == kTmaWarp && lane == 0) {
      // ---------------------------------------------------------- TMA producer (one lane)
      const int yk0 = hk * a.L.Tkv + s.kvpad0;
      const float *sk_row = a.kscale + (size_t)hk * (a.L.Tkv / kGK) + s.kvpad0 / kGK;
      const float *dsc0 = a.dsc + ((size_t)hq * a.L.nqblk + s.qpad0 / kBQ + qtt[0]) * a.L.nkv_pad;
      const float *dsc1 = dsc0 + a.L.nkv_pad;  // the next Q block's row
      mbar_arrive_expect_tx(q_full, (valid[1] ? 2 : 1) * 128 * DP);
      tma_load_2d(smem + P::kQ, &tm_q, 0, hq * a.L.Tq + s.qpad0 + qtt[0] * kBQ, q_full);
      if (valid[1])
        tma_load_2d(smem + P::kQ + 128 * DP, &tm_q, 0, hq * a.L.Tq + s.qpad0 + qtt[1] * kBQ,
                    q_full);
      int issued = 0;
      for (int j = 0; j < Tmax; ++j) {
        const int st = j % ST, sd = j % P::kDS;
        if (j >= ST && !mbar_wait_poll<kPollProducerNs>(&k_empty[st], ((j / ST) - 1) & 1, ab,
                                                         kSiteKvEmpty))
          break;
        mbar_arrive_expect_tx(&k_full[st], 128 * DP);
        tma_load_2d(smem + P::kK + st * 128 * DP, &tm_k, 0, yk0 + j * kBKV, &k_full[st]);
        if (j >= P::kDS && !mbar_wait_poll<kPollProducerNs>(&d_empty[sd], ((j / P::kDS) - 1) & 1,
                                                              ab, kSiteKvEmpty))
          break;
        const bool u0 = j < T0, u1 = j < T1;
        mbar_arrive_expect_tx(&d_full[sd], ((u0 ? 1 : 0) + (u1 ? 1 : 0)) * 512 + 16);
        if (u0) bulk_load(smem + P::kDsc + sd * 1024, dsc0 + (size_t)j * kBKV, 512, &d_full[sd]);
        if (u1)
          bulk_load(smem + P::kDsc + sd * 1024 + 512, dsc1 + (size_t)j * kBKV, 512, &d_full[sd]);
        bulk_load(smem + P::kSk + sd * 16, sk_row + j * (kBKV / kGK), 16, &d_full[sd]);
        issued = j + 1;
      }
      if (*abort_flag) {  // let the copies already issued land before the CTA exits
        for (int n = issued > ST ? issued - ST : 0; n < issued; ++n)
          drain_wait(&k_full[n % ST], (n / ST) & 1);
        for (int n = issued > P::kDS ? issued - P::kDS : 0; n < issued; ++n)
          drain_wait(&d_full[n % P::kDS], (n / P::kDS) & 1);
        drain_wait(q_full, 0);
      }
    } else if (warp == 3 && lane == 0) {
      // ---------------------------------------------------------- V producer (one lane)
      int issued = 0;
      for (int j = 0; j < Tmax; ++j) {
        const int st = j % ST;
        if (j >= ST && !mbar_wait_poll<kPollProducerNs>(&v_empty[st], ((j / ST) - 1) & 1, ab,
                                                         kSiteKvEmpty))
          break;
        mbar_arrive_expect_tx(&v_full[st], DP * 128);
        tma_load_2d(smem + P::kV + st * DP * 128, &tm_v, s.kvpad0 + j * kBKV, hk * DP, &v_full[st]);
        issued = j + 1;
      }
      if (*abort_flag)
        for (int n = issued > ST ? issued - ST : 0; n < issued; ++n)
          drain_wait(&v_full[n % ST], (n / ST) & 1);
    } else if (warp == kMmaWarp && lane == 0) {
      // ---------------------------------------------------------- Q K^T issuer (one lane)
      // In the fixed order n = 0, 1, ..., tile 0 then tile 1, each with blocking waits: QK_t(n)
      // once the softmax of tile t has read S_t(n-1), PV_t(n-2) is complete (so the softmax
      // knows from s_full_t(n) alone that P~ buffer n % 2 is free, and its own parity waits on
      // pv_done come at most one phase ahead of what has completed), K(n) and the DeltaS*c of
      // tile n have landed. K stage n is released once QK_0(n) and QK_1(n) complete.
      constexpr uint32_t idesc_qk = idesc_e4m3_f32(128, 128);
      bool ok = mbar_wait(q_full, 0, ab, kSiteQ);
      for (int n = 0; ok && n < Tmax; ++n) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || n >= (t ? T1 : T0)) continue;
          if (n > 0) ok = mbar_wait_poll<kPollQkNs>(&s_free[t], (n - 1) & 1, ab, kSiteSFree);
          if (ok && n >= 2)
            ok = mbar_wait_poll<kPollQkNs>(&pv_done[2 * t + (n & 1)], ((n - 2) >> 1) & 1, ab,
                                           kSitePvDone);
          if (ok) ok = mbar_wait(&k_full[n % ST], (n / ST) & 1, ab, kSiteKvFull);
          if (ok) ok = mbar_wait(&d_full[n % P::kDS], (n / P::kDS) & 1, ab, kSiteKvFull);
          if (!ok) break;
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor(smem_u32(smem + P::kQ + t * 128 * DP), DP);
          const uint64_t kdesc = sdesc_kmajor(smem_u32(smem + P::kK + (n % ST) * 128 * DP), DP);
#pragma unroll
          for (int kk = 0; kk < DP / 32; ++kk)
            mma_e4m3_ss(tbase + pp_col_s(t), adesc + (uint64_t)(kk * 2),
                        kdesc + (uint64_t)(kk * 2), idesc_qk, kk > 0);
          mma_commit(&s_full[t]);
        }
        if (ok) mma_commit(&k_empty[n % ST]);
      }
      mma_commit(&drain[0]);  // every MMA issued above completes before tensor memory is freed
      drain_wait(&drain[0], 0);
    } else if (warp == kPvWarp && lane == 0) {
      // ---------------------------------------------------------- P~V issuer (one lane)
      // Same order: PV_t(n) once P~_t(n) is written (after the rescale of O_t) and V(n) has
      // landed. V stage n and DeltaS*c stage n get this issuer's arrivals once PV_0(n) and PV_1(n)
      // complete.
      constexpr uint32_t idesc_pv = idesc_e4m3_f32(128, DP);
      bool ok = true;
      for (int n = 0; ok && n < Tmax; ++n) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || n >= (t ? T1 : T0)) continue;
          ok = mbar_wait_poll<kPollPvNs>(&p_full[2 * t + (n & 1)], (n >> 1) & 1, ab, kSitePFull);
          if (ok) ok = mbar_wait(&v_full[n % ST], (n / ST) & 1, ab, kSiteKvFull);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vdesc = sdesc_kmajor(smem_u32(smem + P::kV + (n % ST) * DP * 128), 128);
          if constexpr (DP == 64) {
#pragma unroll
            for (int kk = 0; kk < kBKV / 32; ++kk)
              mma_e4m3_ts(tbase + pp_col_o(t), tbase + pp_col_p(t, n & 1) + kk * 8,
                          vdesc + (uint64_t)(kk * 2), idesc_pv, (n > 0 || kk > 0) ? 1u : 0u);
          } else {
            const uint64_t pdesc =
                sdesc_kmajor(smem_u32(smem + P::kP + (2 * t + (n & 1)) * 16384), 128);
#pragma unroll
            for (int kk = 0; kk < kBKV / 32; ++kk)
              mma_e4m3_ss(tbase + pp_col_o(t), pdesc + (uint64_t)(kk * 2),
                          vdesc + (uint64_t)(kk * 2), idesc_pv, (n > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&pv_done[2 * t + (n & 1)]);
        }
        if (ok) {
          mma_commit(&v_empty[n % ST]);
          mma_commit(&d_empty[n % P::kDS]);
        }
      }
      mma_commit(&drain[1]);
      drain_wait(&drain[1], 0);
    }
    cta_teardown(warp == kMmaWarp, tbase);
  } else {
    regs_acquire<kPPRegsSoftmax>();
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp < kFoldWarp0 ? 0 : 1;  // warps 4-7: tile 0, warps 8-11: tile 1
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    const int qt = qtt[t];
    const int i = qt * kBQ + row;
    const bool row_ok = valid[t] && i < s.nq;
    const int T = Tt[t];
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const size_t o = ((size_t)(s.q0 + i) * g.Hq + hq) * g.D0;
    if (valid[t] && T == 0) {  // no visible key in this tile
      if (row_ok)
        for (int d = 0; d < g.D0; ++d) {
          if (a.out_dtype == SAGE2_FP32)
            static_cast<float *>(a.out)[o + d] = 0.f;
          else
            static_cast<uint16_t *>(a.out)[o + d] = 0;
        }
    }
    if (T > 0) {
      const float c32 = g.c32;
      const float sqc =
          row_ok ? __fmul_rn(a.qscale[(size_t)hq * a.L.Tq + s.qpad0 + qt * kBQ + row], c32) : 0.f;
      const int last_key = g.causal ? min(i + (s.nkv - s.nq), s.nkv - 1) : s.nkv - 1;
      const float L32 = 8.8073549220576041f;  // fl32(log2(448))
      const uint32_t tS = tbase + lane_base + pp_col_s(t);
      const uint32_t tO = tbase + lane_base + pp_col_o(t);
      // this thread's row of P~_t(j) in buffer j % 2: 8 chunks of 16 bytes, chunk c at position
      // c ^ (row & 7)
      uint8_t *prow0 = smem + P::kP + 2 * t * 16384 + row * 128;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      // Barrier phases are tested ahead of the blocking waits, at phase boundaries where the
      // test's shared-memory round trip overlaps arithmetic: S_t(j+1) right after the P~ stores
      // and their fence, PV_t(j-1) right after the logits. A wait then runs only if its test
      // failed.
      bool s_ready = false;
#pragma unroll 1
      for (int j = 0; j < T; ++j) {
        if (!__all_sync(0xffffffffu, s_ready)) {
          ok = warp_all(mbar_wait(&s_full[t], j & 1, ab, kSiteSFull));
          if (!ok) break;
        }
        tc_fence_after();
        uint32_t v[128];
        tmem_ld128_nowait(tS, v);
        tmem_wait_ld128(v);  // S_t(j) is in registers: QK_t(j+1) may overwrite S_t
        const bool dump = DBG && t == (a.dbg.qt & 1) && j == a.dbg.kt;
        if (dump) {
#pragma unroll
          for (int e = 0; e < 128; ++e) a.dbg.s_out[row * 128 + e] = __uint_as_float(v[e]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[t]);
        // DeltaS*c and the K scales of tile j: the copy completed d_full(j), which the Q K^T
        // issuer waited for before issuing QK_t(j), whose completion (s_full) this warp has seen
        const float *dsc =
            reinterpret_cast<const float *>(smem + P::kDsc + (j % P::kDS) * 1024 + t * 512);
        const float *skv = reinterpret_cast<const float *>(smem + P::kSk + (j % P::kDS) * 16);
        const int lim = last_key - j * kBKV;
        float2 x[64];
        const float pmax = logits128(x, v, dsc, skv, sqc, lim);
        const bool pv_ready =
            j == 0 || mbar_test_wait(&pv_done[2 * t + ((j - 1) & 1)], ((j - 1) >> 1) & 1);
        const float m_new = fmaxf(m, pmax);
        const bool none = (m_new == -INFINITY);
        const float alpha = none ? 1.f : ex2_approx(__fsub_rn(m, m_new));
        const float m448 = none ? 0.f : __fsub_rn(m_new, L32);
        // P~_t(j) into buffer j % 2, free: QK_t(j) was issued after PV_t(j-2) had completed
        uint32_t pk[32];
        float rs;
        if constexpr (DP == 64) {
          rs = probs128_tm(x, m448, pk, tbase + lane_base + pp_col_p(t, j & 1));
        } else {
          rs = probs128(x, m448, pk, prow0 + (j & 1) * 16384, row);
          fence_async_smem();  // the generic-proxy stores become visible to the MMA
        }
        s_ready = j + 1 < T && mbar_test_wait(&s_full[t], (j + 1) & 1);
        if (dump) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            *reinterpret_cast<uint32_t *>(a.dbg.p_out + row * 128 + 4 * e) = pk[e];
        }
        // O = alpha O once PV_t(j-1) is complete (with every alpha of the warp's rows equal to 1
        // there is nothing to do), while the P~ stores drain.
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!__all_sync(0xffffffffu, pv_ready)) {
            ok = warp_all(
                mbar_wait(&pv_done[2 * t + ((j - 1) & 1)], ((j - 1) >> 1) & 1, ab, kSitePvDone));
            if (!ok) break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < DP / 64; ++h) {  // 64 columns per load
            uint32_t ov[64];
            tmem_ld64(tO + 64 * h, ov);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t r[32];
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                const float2 y = __fmul2_rn(
                    make_float2(__uint_as_float(ov[32 * c + e]), __uint_as_float(ov[32 * c + e + 1])),
                    make_float2(alpha, alpha));
                r[e] = __float_as_uint(y.x);
                r[e + 1] = __float_as_uint(y.y);
              }
              tmem_st32(tO + 64 * h + 32 * c, r);
            }
          }
          tmem_st_wait();
        }
        if constexpr (DP == 64) tmem_st_wait();  // the P~ stores
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[2 * t + (j & 1)]);
        if (dump && j == 0) {  // O after PV(0) is the fresh partial P~(0) V(0)
          ok = warp_all(mbar_wait(&pv_done[2 * t], 0, ab, kSitePvDone));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DP / 32; ++c) {
            uint32_t r[32];
            tmem_ld32_wait(tO + 32 * c, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) a.dbg.r_out[row * DP + 32 * c + e] = __uint_as_float(r[e]);
          }
        }
        l = __fmaf_rn(alpha, l, rs);
        m = m_new;
      }
      // ---------------------------------------------------------- epilogue
      // PV_t(T-1) on its buffer's barrier, whose previous phase (PV_t(T-3)) the Q K^T issuer saw
      // complete before issuing QK_t(T-1)
      if (ok)
        ok = warp_all(
            mbar_wait(&pv_done[2 * t + ((T - 1) & 1)], ((T - 1) >> 1) & 1, ab, kSitePvDone));
      if (warp_all(ok && !*abort_flag)) {
        tc_fence_after();
        store_out_row<DP>(a, tO, sv_s, l, row_ok, o);
      }
    }
    cta_teardown(false, tbase);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D tensor map of 1- or 2-byte elements: inner extent `inner` elements, `rows` rows, box
// (box_inner x box_rows) elements.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
              uint32_t box_rows, CUtensorMapSwizzle sw, int elem_bytes = 1) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DP, int ST, bool DBG, bool I8>
cudaError_t launch_t(const CUtensorMap &mk, const CUtensorMap &mv, const AttnArgs &a, dim3 grid,
                     cudaStream_t st) {
  using P = SmemPlan<DP, ST, I8>;
  // at least 116 KB so that a single CTA occupies an SM (each allocates all 512 TMEM columns)
  constexpr int kSmem = P::kBytes > 116 * 1024 ? P::kBytes : 116 * 1024;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_fwd<DP, ST, DBG, I8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  attn_fwd<DP, ST, DBG, I8><<<grid, kThreads, kSmem, st>>>(mk, mv, a);
  return cudaGetLastError();
}

template <int DP, int ST, bool DBG>
cudaError_t launch_pp(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                      const AttnArgs &a, dim3 grid, cudaStream_t st) {
  using P = PPPlan<DP, ST>;
  constexpr int kSmem = P::kBytes > 116 * 1024 ? P::kBytes : 116 * 1024;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_pp<DP, ST, DBG>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  attn_pp<DP, ST, DBG><<<grid, kThreads, kSmem, st>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

// INT4 codes run on the two-tile kernel (the debug hook too, except the unit whose producer
// issues nothing); SAGE2_ATTN_PP=0 in the environment selects the one-tile kernel instead, which
// also serves the INT8 path. Read at every launch, so a process can compare the two.
bool use_pp() {
  const char *e = getenv("SAGE2_ATTN_PP");
  return !(e && e[0] == '0');
}

}  // namespace

cudaError_t launch_attention(void *out, int out_dtype, const Geometry &g, const Layout &L,
                             const void *ws, cudaStream_t st, const AttnDebug *dbg, bool int8_qk,
                             int hq0, int hq_n) {
  if (int8_qk != (L.code_bytes == 2)) return cudaErrorInvalidValue;
  const WsPtrs w = ws_ptrs(const_cast<void *>(ws), L);
  AttnArgs a;
  a.g = g;
  a.L = L;
  a.qscale = w.qscale;
  a.kscale = w.kscale;
  a.dsc = w.dsc;
  a.vscale = w.vscale;
  a.qcode = w.qcode;
  a.out = out;
  a.out_dtype = out_dtype;
  a.status = w.status;
  a.seq_order = w.status + kSeqOrderWord;
  a.dbg = dbg ? *dbg : AttnDebug{0, 0, 0, 0, nullptr, nullptr, nullptr, 0};
  if (hq0 < 0 || hq_n < 0 || hq0 + hq_n > g.Hq) return cudaErrorInvalidValue;
  a.hq0 = hq0;
  a.hq_n = hq_n > 0 ? hq_n : g.Hq - hq0;
  const CUtensorMapSwizzle qk_sw =
      g.Dp == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap mk, mv;
  // INT8 path: fp16 codes in 64-channel boxes (128-byte swizzled rows), DP / 64 per tile
  const bool mk_ok = int8_qk ? make_map(&mk, w.kcode, g.Dp, (uint64_t)g.Hkv * L.Tkv, 64, 128,
                                        CU_TENSOR_MAP_SWIZZLE_128B, 2)
                             : make_map(&mk, w.kcode, g.Dp, (uint64_t)g.Hkv * L.Tkv, g.Dp, 128, qk_sw);
  if (!mk_ok || !make_map(&mv, w.vcodeT, L.Tkv, (uint64_t)g.Hkv * g.Dp, 128, g.Dp,
                          CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int nqt = (g.max_nq + kBQ - 1) / kBQ;
  if (!int8_qk && !(dbg && dbg->skip_loads) && use_pp()) {
    CUtensorMap mq;
    if (!make_map(&mq, w.qcode, g.Dp, (uint64_t)g.Hq * L.Tq, g.Dp, 128, qk_sw))
      return cudaErrorInvalidValue;
    const dim3 grid2(a.hq_n * ((nqt + 1) / 2), 1, g.B);
    // K and V stages: 3 each at D = 128; 8 each at D = 64 (no P~ buffers in shared memory there;
    // 8 measured 1.5 % faster than 6 on the video DiT shape, 10 no better)
    if (dbg) {
      if (g.Dp == 128) return launch_pp<128, 3, true>(mq, mk, mv, a, dim3(1), st);
      return launch_pp<64, 8, true>(mq, mk, mv, a, dim3(1), st);
    }
    if (g.Dp == 128) return launch_pp<128, 3, false>(mq, mk, mv, a, grid2, st);
    return launch_pp<64, 8, false>(mq, mk, mv, a, grid2, st);
  }
  const dim3 grid = dbg ? dim3(1) : dim3(a.hq_n * nqt, 1, g.B);
  // pipeline depth: as many K/V stages as fit (a stage of fp16 K codes is twice as large)
  if (int8_qk) {
    if (dbg) {
      if (g.Dp == 128) return launch_t<128, 4, true, true>(mk, mv, a, grid, st);
      return launch_t<64, 8, true, true>(mk, mv, a, grid, st);
    }
    if (g.Dp == 128) return launch_t<128, 4, false, true>(mk, mv, a, grid, st);
    return launch_t<64, 8, false, true>(mk, mv, a, grid, st);
  }
  if (dbg) {
    if (g.Dp == 128) return launch_t<128, 6, true, false>(mk, mv, a, grid, st);
    return launch_t<64, 8, true, false>(mk, mv, a, grid, st);
  }
  if (g.Dp == 128) return launch_t<128, 6, false, false>(mk, mv, a, grid, st);
  return launch_t<64, 8, false, false>(mk, mv, a, grid, st);
}

}  // namespace sage2
