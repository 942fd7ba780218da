// sage2_attention.cu -- the fused SageAttention2 attention kernel for sm_103a.
//
// One CTA per (sequence, q head, 128-row Q tile); ten warps:
//   warps 0-3  softmax: thread t of warp w owns accumulator row 32w+t (its TMEM lane). Per
//              128-key tile it loads the whole S row from tensor memory in one instruction,
//              dequantizes and adds DeltaS with one FMA per element, takes the row maximum,
//              computes P448 = 2^(S' - m + log2 448) in base 2, writes P~ = e4m3(P448) back to
//              tensor memory (the A operand of the P~V MMA) and hands alpha = 2^(m_old - m_new)
//              to the fold warps.
//   warps 4-7  fold + epilogue: thread t of warp 4+w owns row 32w+t of the FP32 output in
//              registers and folds the fresh per-tile partial: O = alpha O + R. At the end it
//              divides by the row sum and writes the output row.
//   warp 8     TMA producer (one lane): Q codes once, then per KV tile the K codes, transposed
//              V codes, 128 DeltaS*c values and 4 K scales into an ST-stage ring.
//   warp 9     MMA issuer (one lane) and tensor-memory owner: S = Qcode Kcode^T
//              (tcgen05 kind::f8f6f4, e4m3 x e4m3 -> f32, both operands from shared memory),
//              R = P~ Vcode (A from tensor memory), into double-buffered S and R.
// Method (SageAttention2 pages): INT4-grid Q and K codes with per-thread-group scales; P~ and
// V in e4m3; two-level accumulation of P~V ("SageAttention2: Efficient Attention with Thorough
// Outlier Smoothing and Per-thread INT4 Quantization" research note, components 2 and 3;
// "SageAttention2 and Fast Exact INT4 Attention" visual companion, Numerical Repair Stack).
//
// The integer products are exact: codes lie in [-7, 7], stored as e4m3 (exact), products are
// at most 49 and a 128-channel dot product at most 6272 < 2^24, so the FP32 accumulator holds
// the integer Q K^T exactly.
//
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) R0 [256, 256+Dp) R1 [384, 384+Dp);
// P~ of tile j overwrites the first 32 columns of its S buffer once the softmax has read S.
//
// Pipeline per KV tile j (sb = j % 2): the MMA warp issues QK(j+1) as soon as PV(j-1) has
// finished reading P~(j-1) from S[(j+1)%2], so the tensor core computes the next S while the
// softmax works on this one; PV(j) waits for P~(j) and for the fold of R(j-2). The alpha of
// tile j travels through a 4-deep shared ring: the softmax cannot run more than three tiles
// ahead of the fold (tile j+4 needs PV(j+2), which needs the fold of tile j).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "sage2_device.cuh"
#include "sage2_internal.h"

namespace sage2 {
namespace {

constexpr int kThreads = 320;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColR0 = 256, kColR1 = 384;
constexpr uint32_t kTmemCols = 512;

// wait-site ids reported in the status word
enum : int {
  kSiteQ = 1, kSiteKvFull = 2, kSiteKvEmpty = 3, kSiteSFull = 4, kSitePFull = 5, kSiteRFull = 6,
  kSiteRFree = 7, kSiteKvFullSm = 8, kSiteAFull = 9, kSiteLFull = 10
};

struct AttnArgs {
  Geometry g;
  Layout L;
  const float *qscale, *kscale, *dsc, *vscale;
  void *out;
  int out_dtype;
  int *status;
  AttnDebug dbg;
};

template <int DP, int ST>
struct SmemPlan {
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 128 * DP;
  static constexpr int kV = kK + ST * 128 * DP;
  static constexpr int kDsc = kV + ST * DP * 128;
  static constexpr int kSk = kDsc + ST * 512;
  static constexpr int kAlpha = kSk + ST * 16;         // float [4][128]
  static constexpr int kLsum = kAlpha + 4 * 128 * 4;  // float [128]
  static constexpr int kBar = kLsum + 128 * 4;
  // q, full[ST], empty[ST], s[2], p[2], r_full[2], r_free[2], a[4], l, drain
  static constexpr int kNumBars = 1 + 2 * ST + 2 + 2 + 2 + 2 + 4 + 1 + 1;
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
    attn_fwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
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

  uint8_t *sQ = smem + P::kQ;
  float *alpha_ring = reinterpret_cast<float *>(smem + P::kAlpha);
  float *lsum = reinterpret_cast<float *>(smem + P::kLsum);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::kBar);
  uint64_t *q_full = bars;
  uint64_t *kv_full = bars + 1;
  uint64_t *kv_empty = kv_full + ST;
  uint64_t *s_full = kv_empty + ST;
  uint64_t *p_full = s_full + 2;
  uint64_t *r_full = p_full + 2;
  uint64_t *r_free = r_full + 2;
  uint64_t *a_full = r_free + 2;
  uint64_t *l_full = a_full + 4;
  uint64_t *drain = l_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + P::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P::kMisc + 4);

  if (warp == 8 && lane == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&r_full[i], 1);
      mbar_init(&r_free[i], 4);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&a_full[i], 4);
    mbar_init(l_full, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const AbortCtx ab{abort_flag, a.status};

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int yq = hq * a.L.Tq + s.qpad0 + qt * kBQ;
      const int yk0 = hk * a.L.Tkv + s.kvpad0;
      const int yv = hk * DP;
      const float *dsc_row =
          a.dsc + ((size_t)hq * a.L.nqblk + s.qpad0 / kBQ + qt) * a.L.nkv_pad;
      const float *sk_row = a.kscale + (size_t)hk * (a.L.Tkv / kGK) + s.kvpad0 / kGK;
      const bool skip = DBG && a.dbg.skip_loads;
      bool q_issued = false;
      int issued = 0;
      if (!skip) {
        mbar_arrive_expect_tx(q_full, 128 * DP);
        tma_load_2d(sQ, &tm_q, 0, yq, q_full);
        q_issued = true;
      }
      for (int j = 0; j < T; ++j) {
        const int st = j % ST;
        if (j >= ST && !mbar_wait(&kv_empty[st], ((j / ST) - 1) & 1, ab, kSiteKvEmpty)) break;
        if (skip) continue;
        uint8_t *sK = smem + P::kK + st * 128 * DP;
        uint8_t *sV = smem + P::kV + st * DP * 128;
        float *sD = reinterpret_cast<float *>(smem + P::kDsc + st * 512);
        float *sS = reinterpret_cast<float *>(smem + P::kSk + st * 16);
        mbar_arrive_expect_tx(&kv_full[st], 128 * DP + DP * 128 + 512 + 16);
        tma_load_2d(sK, &tm_k, 0, yk0 + j * kBKV, &kv_full[st]);
        tma_load_2d(sV, &tm_v, s.kvpad0 + j * kBKV, yv, &kv_full[st]);
        bulk_load(sD, dsc_row + (size_t)j * kBKV, 512, &kv_full[st]);
        bulk_load(sS, sk_row + j * (kBKV / kGK), 16, &kv_full[st]);
        issued = j + 1;
      }
      if (*abort_flag) {  // let the copies already issued land before the CTA exits
        if (q_issued) drain_wait(q_full, 0);
        for (int n = issued > ST ? issued - ST : 0; n < issued; ++n)
          drain_wait(&kv_full[n % ST], (n / ST) & 1);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_e4m3_f32(128, 128);
      constexpr uint32_t idesc_pv = idesc_e4m3_f32(128, DP);
      const uint64_t qdesc = sdesc_kmajor(smem_u32(sQ), DP);
      bool ok = mbar_wait(q_full, 0, ab, kSiteQ);
      auto issue_qk = [&](int j) {
        const int st = j % ST;
        const uint64_t kdesc = sdesc_kmajor(smem_u32(smem + P::kK + st * 128 * DP), DP);
        const uint32_t dS = tbase + ((j & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < DP / 32; ++kk)
          mma_e4m3_ss(dS, qdesc + (uint64_t)(kk * 2), kdesc + (uint64_t)(kk * 2), idesc_qk, kk > 0);
        mma_commit(&s_full[j & 1]);
      };
      if (ok) ok = mbar_wait(&kv_full[0], 0, ab, kSiteKvFull);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
      }
      for (int j = 0; ok && j < T; ++j) {
        if (j + 1 < T) {
          ok = mbar_wait(&kv_full[(j + 1) % ST], ((j + 1) / ST) & 1, ab, kSiteKvFull);
          // S[(j+1)%2] still holds P~(j-1): PV(j-1) must have finished reading it
          if (ok && j >= 1) ok = mbar_wait(&r_full[(j - 1) & 1], ((j - 1) >> 1) & 1, ab, kSiteRFull);
          if (!ok) break;
          tc_fence_after();
          issue_qk(j + 1);
        }
        ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1, ab, kSitePFull);
        if (ok && j >= 2) ok = mbar_wait(&r_free[j & 1], ((j - 2) >> 1) & 1, ab, kSiteRFree);
        if (!ok) break;
        tc_fence_after();
        const int st = j % ST;
        const uint64_t vdesc = sdesc_kmajor(smem_u32(smem + P::kV + st * DP * 128), 128);
        const uint32_t aP = tbase + ((j & 1) ? kColS1 : kColS0);
        const uint32_t dR = tbase + ((j & 1) ? kColR1 : kColR0);
#pragma unroll
        for (int kk = 0; kk < kBKV / 32; ++kk)
          mma_e4m3_ts(dR, aP + kk * 8, vdesc + (uint64_t)(kk * 2), idesc_pv, kk > 0);
        mma_commit(&r_full[j & 1]);
        mma_commit(&kv_empty[st]);
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
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < T; ++j) {
      const int sb = j & 1, st = j % ST;
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, ab, kSiteSFull)) break;
      if (!mbar_wait(&kv_full[st], (j / ST) & 1, ab, kSiteKvFullSm)) break;
      tc_fence_after();
      const float *dsc = reinterpret_cast<const float *>(smem + P::kDsc + st * 512);
      const float *skv = reinterpret_cast<const float *>(smem + P::kSk + st * 16);
      const int lim = last_key - j * kBKV;  // columns 0..lim are visible to this row
      const uint32_t tS = tbase + lane_base + (sb ? kColS1 : kColS0);
      uint32_t v[128];
      tmem_ld128(tS, v);
      if (DBG && j == a.dbg.kt) {
#pragma unroll
        for (int e = 0; e < 128; ++e) a.dbg.s_out[row * 128 + e] = __uint_as_float(v[e]);
      }
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
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
      float mx = m;
#pragma unroll
      for (int e = 0; e < 128; e += 2) mx = max3(mx, x[e], x[e + 1]);
      const float m_new = mx;
      const float m448 = (m_new == -INFINITY) ? 0.f : __fsub_rn(m_new, L32);
      const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(__fsub_rn(m, m_new));
      // P448 = 2^(S' - m448); masked keys have S' = -inf and give 0
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 32 keys -> 8 words of P~ per chunk
        uint32_t pk[8];
#pragma unroll
        for (int e = c * 32; e < c * 32 + 32; e += 4) {
          float t0, t1, t2, t3;
          add2(t0, t1, x[e], x[e + 1], -m448, -m448);
          add2(t2, t3, x[e + 2], x[e + 3], -m448, -m448);
          const float p0 = ex2_approx(t0), p1 = ex2_approx(t1), p2 = ex2_approx(t2),
                      p3 = ex2_approx(t3);
          add2(ps0, ps1, ps0, ps1, p0, p1);
          add2(ps0, ps1, ps0, ps1, p2, p3);
          pk[(e - c * 32) / 4] = cvt_e4m3x2(p0, p1) | (cvt_e4m3x2(p2, p3) << 16);
        }
        tmem_st8(tS + c * 8, pk);
        if (DBG && j == a.dbg.kt) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            *reinterpret_cast<uint32_t *>(a.dbg.p_out + row * 128 + c * 32 + e * 4) = pk[e];
        }
      }
      tmem_st_wait();
      tc_fence_before();
      alpha_ring[(j & 3) * 128 + row] = alpha;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&p_full[sb]);
        mbar_arrive(&a_full[j & 3]);
      }
      l = __fmaf_rn(alpha, l, __fadd_rn(ps0, ps1));
      m = m_new;
    }
    lsum[row] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(l_full);
  } else {
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
      const int sb = j & 1;
      ok = mbar_wait(&a_full[j & 3], (j >> 2) & 1, ab, kSiteAFull);
      if (!ok) break;
      const float alpha = alpha_ring[(j & 3) * 128 + row];
      ok = mbar_wait(&r_full[sb], (j >> 1) & 1, ab, kSiteRFull);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tR = tbase + lane_base + (sb ? kColR1 : kColR0);
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
      if (lane == 0) mbar_arrive(&r_free[sb]);
    }
    if (ok) ok = mbar_wait(l_full, 0, ab, kSiteLFull);
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
  if (warp == 9) tmem_dealloc(tbase, kTmemCols);
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
cudaError_t launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                     const AttnArgs &a, dim3 grid, cudaStream_t st) {
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
  attn_fwd<DP, ST, DBG><<<grid, kThreads, kSmem, st>>>(mq, mk, mv, a);
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
  a.out = out;
  a.out_dtype = out_dtype;
  a.status = w.status;
  a.dbg = dbg ? *dbg : AttnDebug{0, 0, 0, 0, nullptr, nullptr, nullptr, 0};
  const CUtensorMapSwizzle qk_sw =
      g.Dp == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, w.qcode, g.Dp, (uint64_t)g.Hq * L.Tq, g.Dp, 128, qk_sw) ||
      !make_map(&mk, w.kcode, g.Dp, (uint64_t)g.Hkv * L.Tkv, g.Dp, 128, qk_sw) ||
      !make_map(&mv, w.vcodeT, L.Tkv, (uint64_t)g.Hkv * g.Dp, 128, g.Dp,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int nqt = (g.max_nq + kBQ - 1) / kBQ;
  if (dbg) {
    if (g.Dp == 128) return launch_t<128, 3, true>(mq, mk, mv, a, dim3(1), st);
    return launch_t<64, 4, true>(mq, mk, mv, a, dim3(1), st);
  }
  const dim3 grid(nqt, g.Hq, g.B);
  if (g.Dp == 128) return launch_t<128, 3, false>(mq, mk, mv, a, grid, st);
  return launch_t<64, 4, false>(mq, mk, mv, a, grid, st);
}

}  // namespace sage2
