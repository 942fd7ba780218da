// sage2_attention.cu -- the fused SageAttention2 attention kernel for sm_103a.
//
// One CTA per (sequence, q head, 128-row Q tile); ten warps:
//   warps 0-3  softmax: thread t of warp w owns accumulator row 32w+t (its TMEM lane). It first
//              stores its row's Q codes into tensor memory (the A operand of Q K^T). Per 128-key
//              tile it loads the whole S row in one instruction, dequantizes and adds DeltaS
//              with one FMA per element, takes the row maximum, computes
//              P448 = 2^(S' - m + log2 448) in base 2, writes P~ = e4m3(P448) to tensor memory
//              (the A operand of the P~V MMA) and hands alpha = 2^(m_old - m_new) to the fold.
//              The arithmetic runs in long independent phases over the 128 values, in place.
//   warps 4-7  fold + epilogue: thread t of warp 4+w owns row 32w+t of the FP32 output in
//              registers and folds the fresh per-tile partial: O = alpha O + R. At the end it
//              divides by the row sum and writes the output row.
//   warp 8     TMA producer (one lane): per KV tile the K codes, the transposed V codes,
//              128 DeltaS*c values and 4 K scales into an ST-stage ring.
//   warp 9     MMA issuer (one lane), tcgen05 kind::f8f6f4 (e4m3 x e4m3 -> f32), A operands from
//              tensor memory, B from shared memory. Q K^T runs two tiles ahead of the softmax
//              (S is double-buffered); P~ V runs as soon as every row's P~ is written and the
//              previous partial is folded.
// Method (SageAttention2 pages): INT4-grid Q and K codes with per-thread-group scales; P~ and
// V in e4m3; two-level accumulation of P~V ("SageAttention2: Efficient Attention with Thorough
// Outlier Smoothing and Per-thread INT4 Quantization" research note, components 2 and 3;
// "SageAttention2 and Fast Exact INT4 Attention" visual companion, Numerical Repair Stack).
//
// The integer products are exact: codes lie in [-7, 7], stored as e4m3 (exact), products are
// at most 49 and a 128-channel dot product at most 6272 < 2^24, so the FP32 accumulator holds
// the integer Q K^T exactly.
//
// Tensor memory (512 columns allocated): S0 [0,128) S1 [128,256) R [256, 256+Dp)
// P~0 [384,416) P~1 [416,448) Q [448, 448+Dp/4).
// Ordering: QK(j+2) overwrites S[j%2] once every softmax warp has copied S(j) out (s_free);
// PV(j) overwrites R once the fold of tile j-1 is done (r_free); the softmax of tile j rewrites
// P~[j%2] only after PV(j-2) is complete (pv_done). Every barrier is waited on at most one phase
// behind its next completion, so parity waits cannot alias. The alpha of tile j travels through
// a 4-deep shared ring: tile j+4 first waits for PV(j+2), which needs the fold of tile j+1.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "sage2_device.cuh"
#include "sage2_internal.h"

namespace sage2 {
namespace {

// Warp roles: 0-3 softmax, 4-7 fold, then the TMA and MMA warps.
#ifndef SAGE2_TMA_WARP
#define SAGE2_TMA_WARP 8
#endif
#ifndef SAGE2_MMA_WARP
#define SAGE2_MMA_WARP 9
#endif
constexpr int kTmaWarp = SAGE2_TMA_WARP, kMmaWarp = SAGE2_MMA_WARP;
constexpr int kThreads = 32 * ((kTmaWarp > kMmaWarp ? kTmaWarp : kMmaWarp) + 1);
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColR = 256, kColP0 = 384, kColP1 = 416,
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
  AttnDebug dbg;
};

template <int DP, int ST>
struct SmemPlan {
  static constexpr int kK = 0;
  static constexpr int kV = kK + ST * 128 * DP;
  static constexpr int kDsc = kV + ST * DP * 128;
  static constexpr int kSk = kDsc + ST * 512;
  static constexpr int kAlpha = kSk + ST * 16;         // float [4][128]
  static constexpr int kLsum = kAlpha + 4 * 128 * 4;  // float [128]
  static constexpr int kBar = kLsum + 128 * 4;
  // q, full[ST], empty[ST], s_full[2], s_free[2], p[2], pv_done[2], r_free, a[4], l, drain
  static constexpr int kNumBars = 1 + 2 * ST + 2 + 2 + 2 + 2 + 1 + 4 + 1 + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kEnd = kMisc + 16;
  static constexpr int kBytes = kEnd + 1024;  // + alignment slack
};

// Waits that ignore the abort flag (used to drain copies and MMAs already in flight).
__device__ bool drain_wait(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > SAGE2_WAIT_NS) return false;
  return true;
}

template <int DP, int ST, bool DBG>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
             const AttnArgs a) {
  using P = SmemPlan<DP, ST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const Geometry &g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int b, hq, qt;
  if (DBG) {
    b = a.dbg.b;
    hq = a.dbg.h;
    qt = a.dbg.qt;
  } else {
    b = blockIdx.z;
    hq = blockIdx.y;
    qt = g.causal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
  }
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
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
  uint64_t *s_full = kv_empty + ST;  // [2]
  uint64_t *s_free = s_full + 2;     // [2]
  uint64_t *p_full = s_free + 2;     // [2]
  uint64_t *pv_done = p_full + 2;    // [2]
  uint64_t *r_free = pv_done + 2;
  uint64_t *a_full = r_free + 1;     // [4]
  uint64_t *l_full = a_full + 4;
  uint64_t *drain = l_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + P::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P::kMisc + 4);

  if (warp == kTmaWarp && lane == 0) {
    mbar_init(q_full, 4);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(r_free, 4);
    for (int i = 0; i < 4; ++i) mbar_init(&a_full[i], 4);
    mbar_init(l_full, 4);
    mbar_init(drain, 1);
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

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer (one lane)
    if (lane == 0) {
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
        mbar_arrive_expect_tx(&kv_full[st], 128 * DP + DP * 128 + 512 + 16);
        tma_load_2d(smem + P::kK + st * 128 * DP, &tm_k, 0, yk0 + j * kBKV, &kv_full[st]);
        tma_load_2d(smem + P::kV + st * DP * 128, &tm_v, s.kvpad0 + j * kBKV, hk * DP,
                    &kv_full[st]);
        bulk_load(smem + P::kDsc + st * 512, dsc_row + (size_t)j * kBKV, 512, &kv_full[st]);
        bulk_load(smem + P::kSk + st * 16, sk_row + j * (kBKV / kGK), 16, &kv_full[st]);
        issued = j + 1;
      }
      if (*abort_flag) {  // let the copies already issued land before the CTA exits
        for (int n = issued > ST ? issued - ST : 0; n < issued; ++n)
          drain_wait(&kv_full[n % ST], (n / ST) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_e4m3_f32(128, 128);
      constexpr uint32_t idesc_pv = idesc_e4m3_f32(128, DP);
      auto issue_qk = [&](int j) {  // S[j % 2] = Qcode Kcode(j)^T, A from tensor memory
        const uint64_t kdesc = sdesc_kmajor(smem_u32(smem + P::kK + (j % ST) * 128 * DP), DP);
        const uint32_t dS = tbase + ((j & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < DP / 32; ++kk)
          mma_e4m3_ts(dS, tbase + kColQ + kk * 8, kdesc + (uint64_t)(kk * 2), idesc_qk, kk > 0);
        mma_commit(&s_full[j & 1]);
      };
      bool ok = mbar_wait(q_full, 0, ab, kSiteQ);
      for (int j = 0; ok && j < 2 && j < T; ++j) {  // the first two tiles' Q K^T
        ok = mbar_wait(&kv_full[j], 0, ab, kSiteKvFull);
        if (ok) {
          tc_fence_after();
          issue_qk(j);
        }
      }
      for (int j = 0; ok && j < T; ++j) {
        const int sb = j & 1;
        // Q K^T two tiles ahead, into the S buffer the softmax of tile j has just copied out
        if (j + 2 < T) {
          ok = mbar_wait(&s_free[sb], (j >> 1) & 1, ab, kSiteSFree) &&
               mbar_wait(&kv_full[(j + 2) % ST], ((j + 2) / ST) & 1, ab, kSiteKvFull);
          if (!ok) break;
          tc_fence_after();
          issue_qk(j + 2);
        }
        // P~(j) V(j) once every row's P~ is written and R is folded
        ok = mbar_wait(&p_full[sb], (j >> 1) & 1, ab, kSitePFull);
        if (ok && j >= 1) ok = mbar_wait(r_free, (j - 1) & 1, ab, kSiteRFree);
        if (!ok) break;
        tc_fence_after();
        const uint64_t vdesc = sdesc_kmajor(smem_u32(smem + P::kV + (j % ST) * DP * 128), 128);
        const uint32_t aP = tbase + (sb ? kColP1 : kColP0);
#pragma unroll
        for (int kk = 0; kk < kBKV / 32; ++kk)
          mma_e4m3_ts(tbase + kColR, aP + kk * 8, vdesc + (uint64_t)(kk * 2), idesc_pv, kk > 0);
        mma_commit(&pv_done[sb]);
        mma_commit(&kv_empty[j % ST]);
      }
      mma_commit(drain);  // every MMA issued above completes before tensor memory is freed
      drain_wait(drain, 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int row = warp * 32 + lane;
    const int i = qt * kBQ + row;
    const bool row_ok = i < s.nq;
    const float c32 = g.c32;
    const float sqc =
        row_ok ? __fmul_rn(a.qscale[(size_t)hq * a.L.Tq + s.qpad0 + qt * kBQ + row], c32) : 0.f;
    const int last_key = g.causal ? min(i + (s.nkv - s.nq), s.nkv - 1) : s.nkv - 1;
    const float L32 = 8.8073549220576041f;  // fl32(log2(448))
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    {  // this row's Q codes (Dp bytes) into tensor memory: the A operand of Q K^T
      const uint4 *qrow = reinterpret_cast<const uint4 *>(
          a.qcode + ((size_t)hq * a.L.Tq + s.qpad0 + qt * kBQ + row) * DP);
      uint32_t qw[DP / 4];
#pragma unroll
      for (int c = 0; c < DP / 16; ++c) {
        const uint4 u = __ldg(qrow + c);
        qw[4 * c] = u.x;
        qw[4 * c + 1] = u.y;
        qw[4 * c + 2] = u.z;
        qw[4 * c + 3] = u.w;
      }
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t w8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w8[e] = qw[8 * c + e];
        tmem_st8(tbase + lane_base + kColQ + 8 * c, w8);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    // Every decision to continue is warp-uniform: after each wait the warp takes lane 0's result.
    bool ok = true;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; ok && j < T; ++j) {
      const int sb = j & 1, st = j % ST;
      // S(j) computed, its ring stage loaded, and P~[sb] no longer read by PV(j-2)
      ok = mbar_wait(&s_full[sb], (j >> 1) & 1, ab, kSiteSFull) &&
           mbar_wait(&kv_full[st], (j / ST) & 1, ab, kSiteKvFullSm) &&
           (j < 2 || mbar_wait(&pv_done[sb], ((j - 2) >> 1) & 1, ab, kSitePvDone));
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tbase + lane_base + (sb ? kColS1 : kColS0);
      const uint32_t tP = tbase + lane_base + (sb ? kColP1 : kColP0);
      uint32_t v[128];
      tmem_ld128(tS, v);
      // S(j) is in registers: the MMA warp may compute S(j+2) into this buffer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);
      if (DBG && j == a.dbg.kt) {
#pragma unroll
        for (int e = 0; e < 128; ++e) a.dbg.s_out[row * 128 + e] = __uint_as_float(v[e]);
      }
      const float *dsc = reinterpret_cast<const float *>(smem + P::kDsc + st * 512);
      const float *skv = reinterpret_cast<const float *>(smem + P::kSk + st * 16);
      const int lim = last_key - j * kBKV;  // columns 0..lim are visible to this row
      // The arithmetic below runs in long independent phases over the 128 values, in place,
      // so the scheduler can keep the FMA and MUFU pipes busy with one warp.
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // S' = A * (s_q c s_k) + DeltaS c
        const float mult = __fmul_rn(sqc, skv[c]);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 d4 = *reinterpret_cast<const float4 *>(dsc + c * 32 + e);
          const int k0 = c * 32 + e;
          fma2(x[k0], x[k0 + 1], __uint_as_float(v[k0]), __uint_as_float(v[k0 + 1]), mult, mult,
               d4.x, d4.y);
          fma2(x[k0 + 2], x[k0 + 3], __uint_as_float(v[k0 + 2]), __uint_as_float(v[k0 + 3]), mult,
               mult, d4.z, d4.w);
        }
      }
      if (lim < kBKV - 1) {  // diagonal / ragged tile: hide the keys this row does not see
#pragma unroll
        for (int e = 0; e < 128; ++e) x[e] = (e <= lim) ? x[e] : -INFINITY;
      }
      // row maximum: eight independent 3-input max chains, then a small tree
      float mk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mk[k] = fmaxf(x[16 * k], x[16 * k + 1]);
#pragma unroll
      for (int e = 2; e < 16; e += 2)
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = max3(mk[k], x[16 * k + e], x[16 * k + e + 1]);
      const float m_new = max3(max3(mk[0], mk[1], mk[2]), max3(mk[3], mk[4], mk[5]),
                               max3(mk[6], mk[7], m));
      const float m448 = (m_new == -INFINITY) ? 0.f : __fsub_rn(m_new, L32);
      const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(__fsub_rn(m, m_new));
      // P448 = 2^(S' - m448); masked keys have S' = -inf and give 0
#pragma unroll
      for (int e = 0; e < 128; e += 2) add2(x[e], x[e + 1], x[e], x[e + 1], -m448, -m448);
#pragma unroll
      for (int e = 0; e < 128; ++e) x[e] = ex2_approx(x[e]);
      float ps[8][2];  // row sum: eight independent packed accumulators
#pragma unroll
      for (int k = 0; k < 8; ++k) ps[k][0] = ps[k][1] = 0.f;
#pragma unroll
      for (int e = 0; e < 128; e += 2)
        add2(ps[(e >> 1) & 7][0], ps[(e >> 1) & 7][1], ps[(e >> 1) & 7][0], ps[(e >> 1) & 7][1],
             x[e], x[e + 1]);
      uint32_t pk[32];  // P~ = e4m3(P448), four keys per word
#pragma unroll
      for (int e = 0; e < 32; ++e)
        pk[e] = cvt_e4m3x2(x[4 * e], x[4 * e + 1]) | (cvt_e4m3x2(x[4 * e + 2], x[4 * e + 3]) << 16);
      tmem_st32(tP, pk);
      if (DBG && j == a.dbg.kt) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          *reinterpret_cast<uint32_t *>(a.dbg.p_out + row * 128 + e * 4) = pk[e];
      }
      tmem_st_wait();
      tc_fence_before();
      alpha_ring[(j & 3) * 128 + row] = alpha;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&p_full[sb]);
        mbar_arrive(&a_full[j & 3]);
      }
      float psum[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        psum[k] = __fadd_rn(__fadd_rn(ps[2 * k][0], ps[2 * k][1]), __fadd_rn(ps[2 * k + 1][0], ps[2 * k + 1][1]));
      l = __fmaf_rn(alpha, l, __fadd_rn(__fadd_rn(psum[0], psum[1]), __fadd_rn(psum[2], psum[3])));
      m = m_new;
    }
    lsum[row] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(l_full);
  } else if (warp < 8) {
    // ------------------------------------------------------------ fold + epilogue (warps 4-7)
    const int q4 = warp - 4;
    const int row = q4 * 32 + lane;
    const int i = qt * kBQ + row;
    const bool row_ok = i < s.nq;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    float O[DP];
#pragma unroll
    for (int d = 0; d < DP; ++d) O[d] = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      ok = mbar_wait(&a_full[j & 3], (j >> 2) & 1, ab, kSiteAFull);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const float alpha = alpha_ring[(j & 3) * 128 + row];
      ok = mbar_wait(&pv_done[j & 1], (j >> 1) & 1, ab, kSiteRFull);  // R(j) is complete
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const uint32_t tR = tbase + lane_base + kColR;
#pragma unroll
      for (int c = 0; c < DP / 16; ++c) {
        uint32_t v[16];
        tmem_ld16_wait(tR + c * 16, v);
        if (DBG && j == a.dbg.kt) {
#pragma unroll
          for (int e = 0; e < 16; ++e) a.dbg.r_out[row * DP + c * 16 + e] = __uint_as_float(v[e]);
        }
#pragma unroll
        for (int e = 0; e < 16; e += 2)
          fma2(O[c * 16 + e], O[c * 16 + e + 1], alpha, alpha, O[c * 16 + e], O[c * 16 + e + 1],
               __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(r_free);
    }
    if (ok) ok = mbar_wait(l_full, 0, ab, kSiteLFull);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    // ------------------------------------------------------------ epilogue
    if (ok && row_ok && !*abort_flag) {
      const float l = lsum[row];
      const float inv_l = l > 0.f ? __frcp_rn(l) : 0.f;
      const float *svp = a.vscale + ((size_t)b * g.Hkv + hk) * DP;
      const size_t o = (out_row0 + (size_t)row * g.Hq) * g.D0;
#pragma unroll
      for (int d = 0; d < DP; d += 8) {
        if (d < g.D0) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(O[d + e], svp[d + e]), inv_l);
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

  // ------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, kTmemCols);
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

// 2-D u8 tensor map: inner extent `inner` bytes, `rows` rows, box (box_inner x box_rows).
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
              uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DP, int ST, bool DBG>
cudaError_t launch_t(const CUtensorMap &mk, const CUtensorMap &mv, const AttnArgs &a, dim3 grid,
                     cudaStream_t st) {
  using P = SmemPlan<DP, ST>;
  // at least 116 KB so that a single CTA occupies an SM (each allocates all 512 TMEM columns)
  constexpr int kSmem = P::kBytes > 116 * 1024 ? P::kBytes : 116 * 1024;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_fwd<DP, ST, DBG>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  attn_fwd<DP, ST, DBG><<<grid, kThreads, kSmem, st>>>(mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(void *out, int out_dtype, const Geometry &g, const Layout &L,
                             const void *ws, cudaStream_t st, const AttnDebug *dbg) {
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
  a.dbg = dbg ? *dbg : AttnDebug{0, 0, 0, 0, nullptr, nullptr, nullptr, 0};
  const CUtensorMapSwizzle qk_sw =
      g.Dp == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap mk, mv;
  if (!make_map(&mk, w.kcode, g.Dp, (uint64_t)g.Hkv * L.Tkv, g.Dp, 128, qk_sw) ||
      !make_map(&mv, w.vcodeT, L.Tkv, (uint64_t)g.Hkv * g.Dp, 128, g.Dp,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int nqt = (g.max_nq + kBQ - 1) / kBQ;
  if (dbg) {
    if (g.Dp == 128) return launch_t<128, 6, true>(mk, mv, a, dim3(1), st);
    return launch_t<64, 8, true>(mk, mv, a, dim3(1), st);
  }
  const dim3 grid(nqt, g.Hq, g.B);
  if (g.Dp == 128) return launch_t<128, 6, false>(mk, mv, a, grid, st);
  return launch_t<64, 8, false>(mk, mv, a, grid, st);
}

}  // namespace sage2
