// sage2_prepass.cu -- the smoothing and quantization prepass (memory-bound kernels).
//
// Steps, in launch order (SageAttention2 pages: "SageAttention2: Efficient Attention with
// Thorough Outlier Smoothing and Per-thread INT4 Quantization" research note, components 1
// and 2; PMLR v267 zhang25ae, Abstract; "SageAttention2 and Fast Exact INT4 Attention"
// visual companion, Channel Outlier Smoothing and Per-Thread INT4 Geometry):
//   1. kv_stats_partial / kv_stats_final: per (sequence, kv head, channel) the mean of K
//      and the absolute maximum of V. The K sums are error-free double-float sums, rounded
//      once to FP32 after an FP64 division, so they equal an exact FP64 sum.
//   2. k_quant: K~ = fl32(K - kmean); one INT4 scale per 32 consecutive tokens over all
//      channels; codes in [-7, 7] stored as e4m3 bytes (integers up to 7 are exact).
//   3. v_quant: V codes = e4m3(fl32(V * fl32(448 / amax))), written transposed
//      [kv head][channel][token] so both operands of the P~V MMA are K-major.
//   4. q_quant: per block of 128 rows the mean qmean; Q~ = fl32(Q - qmean); one scale per
//      row; codes as for K.
//   5. delta_s: DeltaS = qmean . K~ in FP32, one fused multiply-add per channel in channel
//      order (register-blocked tiles), stored pre-multiplied by c = log2(e) * sm_scale.
// Every padded position (channels D0..Dp, tokens past a sequence end up to its 128-row
// boundary) is written with zero codes and zero scales.
// Ablation switches (sage2_quant_flags) change only what these kernels write: a zero K
// channel mean (kv_stats_final), a zero Q block mean (q_quant), or one INT4 scale per 128-key
// K tile (k_quant) and per 128-row Q block (q_quant), still stored per 32-key group and per
// row so that the attention kernel reads them unchanged.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sage2_device.cuh"
#include "sage2_internal.h"

namespace sage2 {
namespace {

struct PrepassArgs {
  const uint16_t *q, *k, *v;
  int bf16;
  int flags;  // sage2_quant_flags
  Geometry g;
  Layout L;
  WsPtrs w;
};

__device__ __forceinline__ float to_f32(uint16_t bits, int bf16) {
  if (bf16) return __uint_as_float(((uint32_t)bits) << 16);
  return __half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ void unpack8(const uint4 &u, int bf16, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = to_f32((uint16_t)(w[i] & 0xFFFFu), bf16);
    x[2 * i + 1] = to_f32((uint16_t)(w[i] >> 16), bf16);
  }
}

// INT4-grid code of x * inv, as an e4m3 byte (canonical +0 for zero).
__device__ __forceinline__ float int4_code(float x, float inv) {
  float r = rintf(__fmul_rn(x, inv));
  r = fminf(fmaxf(r, -7.f), 7.f);
  return __fadd_rn(r, 0.f);
}

__device__ __forceinline__ void flag_bad_seq(int *status) {
  atomicCAS(status, 0, kStatusSeqTooLong);
}

// ------------------------------------------------------------------ 1a. K/V statistics
// grid (nchunk, B), block = 32 * ceil(Hkv * D0 / 8 / 32) capped at 256. Each thread owns a
// run of 8 channels (one 16-byte vector of a token row) and walks kStatChunk tokens.
__global__ void __launch_bounds__(256) kv_stats_partial(PrepassArgs a) {
  const int b = blockIdx.y, chunk = blockIdx.x;
  const Geometry &g = a.g;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (!s.ok) {
    if (threadIdx.x == 0 && chunk == 0) flag_bad_seq(a.w.status);
    return;
  }
  const int t0 = chunk * kStatChunk;
  if (t0 >= s.nkv) return;
  const int t1 = min(t0 + kStatChunk, s.nkv);
  const int row_elems = g.Hkv * g.D0;
  const int nvec = row_elems / 8;
  for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
    float hi[8], lo[8], mx[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) hi[e] = lo[e] = mx[e] = 0.f;
    const uint4 *kp = reinterpret_cast<const uint4 *>(a.k + (size_t)(s.kv0 + t0) * row_elems) + vi;
    const uint4 *vp = reinterpret_cast<const uint4 *>(a.v + (size_t)(s.kv0 + t0) * row_elems) + vi;
    const int stride = nvec;
    int t = t0;
    for (; t + 4 <= t1; t += 4) {
      uint4 kk[4], vv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        kk[u] = __ldg(kp + (size_t)(t - t0 + u) * stride);
        vv[u] = __ldg(vp + (size_t)(t - t0 + u) * stride);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {  // tokens in order
        float xk[8], xv[8];
        unpack8(kk[u], a.bf16, xk);
        unpack8(vv[u], a.bf16, xv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          df_add(hi[e], lo[e], xk[e]);
          mx[e] = fmaxf(mx[e], fabsf(xv[e]));
        }
      }
    }
    for (; t < t1; ++t) {
      float xk[8], xv[8];
      unpack8(__ldg(kp + (size_t)(t - t0) * stride), a.bf16, xk);
      unpack8(__ldg(vp + (size_t)(t - t0) * stride), a.bf16, xv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        df_add(hi[e], lo[e], xk[e]);
        mx[e] = fmaxf(mx[e], fabsf(xv[e]));
      }
    }
    const size_t o = ((size_t)b * a.L.nchunk + chunk) * row_elems + (size_t)vi * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      a.w.kpart[o + e] = (double)hi[e] + (double)lo[e];
      a.w.vpart[o + e] = mx[e];
    }
  }
}

// grid (B * Hkv), block Dp.
__global__ void kv_stats_final(PrepassArgs a) {
  const Geometry &g = a.g;
  const int b = blockIdx.x / g.Hkv, h = blockIdx.x % g.Hkv, d = threadIdx.x;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  const size_t o = ((size_t)b * g.Hkv + h) * g.Dp + d;
  float mean = 0.f, amax = 0.f;
  if (s.ok && d < g.D0 && s.nkv > 0) {
    const int nch = (s.nkv + kStatChunk - 1) / kStatChunk;
    const int row_elems = g.Hkv * g.D0;
    double sum = 0.0;
    for (int c = 0; c < nch; ++c) {
      const size_t po = ((size_t)b * a.L.nchunk + c) * row_elems + (size_t)h * g.D0 + d;
      sum += a.w.kpart[po];
      amax = fmaxf(amax, a.w.vpart[po]);
    }
    mean = (a.flags & SAGE2_QUANT_NO_SMOOTH_K) ? 0.f : (float)(sum / (double)s.nkv);
  }
  a.w.kmean[o] = mean;
  a.w.vscale[o] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
  a.w.vinv[o] = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
}

// ------------------------------------------------------------------ 2. K codes
// grid (ceil(max_nkv / 128), Hkv, B), block 128: warp w quantizes the 32-token group
// 4 * tile + w; lane l holds channels [l * CPL, l * CPL + CPL). Per-block switch: the four
// warps share the tile's absolute maximum.
template <int DP>
__global__ void __launch_bounds__(128) k_quant(PrepassArgs a) {
  constexpr int CPL = DP / 32;
  const Geometry &g = a.g;
  const int b = blockIdx.z, h = blockIdx.y, tile = blockIdx.x;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (!s.ok || tile * kBKV >= ((s.nkv + kBKV - 1) / kBKV) * kBKV) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = lane * CPL;
  const bool chan_ok = c0 < g.D0;  // D0 % 8 == 0, so a lane's channels are all in or all out
  const int g0 = tile * kBKV + warp * kGK;  // first token of this group (sequence-local)
  float mu[CPL];
#pragma unroll
  for (int e = 0; e < CPL; ++e) mu[e] = a.w.kmean[((size_t)b * g.Hkv + h) * DP + c0 + e];
  float x[kGK][CPL];
  float amax = 0.f;
  const size_t row_elems = (size_t)g.Hkv * g.D0;
#pragma unroll
  for (int r = 0; r < kGK; ++r) {
    const int t = g0 + r;
    float val[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) val[e] = 0.f;
    if (t < s.nkv && chan_ok) {
      const uint16_t *src = a.k + (size_t)(s.kv0 + t) * row_elems + (size_t)h * g.D0 + c0;
      if (CPL == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(src));
        val[0] = to_f32((uint16_t)(u.x & 0xFFFFu), a.bf16);
        val[1] = to_f32((uint16_t)(u.x >> 16), a.bf16);
        val[2] = to_f32((uint16_t)(u.y & 0xFFFFu), a.bf16);
        val[3] = to_f32((uint16_t)(u.y >> 16), a.bf16);
      } else {
        const uint32_t u = __ldg(reinterpret_cast<const uint32_t *>(src));
        val[0] = to_f32((uint16_t)(u & 0xFFFFu), a.bf16);
        val[1] = to_f32((uint16_t)(u >> 16), a.bf16);
      }
#pragma unroll
      for (int e = 0; e < CPL; ++e) {
        val[e] = __fsub_rn(val[e], mu[e]);
        amax = fmaxf(amax, fabsf(val[e]));
      }
    }
#pragma unroll
    for (int e = 0; e < CPL; ++e) x[r][e] = val[e];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (a.flags & SAGE2_QUANT_PER_BLOCK) {  // block-uniform branch
    __shared__ float wmax[kBKV / kGK];
    if (lane == 0) wmax[warp] = amax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kBKV / kGK; ++w) amax = fmaxf(amax, wmax[w]);
  }
  const float inv = amax > 0.f ? __fdiv_rn(7.f, amax) : 0.f;
  const float scale = amax > 0.f ? __fdiv_rn(amax, 7.f) : 0.f;
  uint8_t *dst = a.w.kcode + ((size_t)h * a.L.Tkv + s.kvpad0 + g0) * DP + c0;
#pragma unroll
  for (int r = 0; r < kGK; ++r) {
    if (CPL == 4) {
      const uint32_t lo = cvt_e4m3x2(int4_code(x[r][0], inv), int4_code(x[r][1], inv));
      const uint32_t hi = cvt_e4m3x2(int4_code(x[r][2], inv), int4_code(x[r][3], inv));
      *reinterpret_cast<uint32_t *>(dst + (size_t)r * DP) = lo | (hi << 16);
    } else {
      *reinterpret_cast<uint16_t *>(dst + (size_t)r * DP) =
          (uint16_t)cvt_e4m3x2(int4_code(x[r][0], inv), int4_code(x[r][1], inv));
    }
  }
  if (lane == 0) a.w.kscale[(size_t)h * (a.L.Tkv / kGK) + (s.kvpad0 + g0) / kGK] = scale;
}

// ------------------------------------------------------------------ 3. V codes, transposed
// grid (ceil(max_nkv / 128), Hkv, B), block 256.
template <int DP>
__global__ void __launch_bounds__(256) v_quant(PrepassArgs a) {
  constexpr int TP = kBKV + 16;  // padded smem row (bytes)
  __shared__ __align__(16) uint8_t tb[DP * TP];
  __shared__ float vinv[DP];
  const Geometry &g = a.g;
  const int b = blockIdx.z, h = blockIdx.y, tile = blockIdx.x;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (!s.ok || tile * kBKV >= ((s.nkv + kBKV - 1) / kBKV) * kBKV) return;
  for (int d = threadIdx.x; d < DP; d += blockDim.x)
    vinv[d] = a.w.vinv[((size_t)b * g.Hkv + h) * DP + d];
  __syncthreads();
  const size_t row_elems = (size_t)g.Hkv * g.D0;
  constexpr int VPT = DP / 8;  // 8-channel vectors per token (padded dim)
  for (int i = threadIdx.x; i < kBKV * VPT; i += blockDim.x) {
    const int tok = i / VPT, c8 = (i % VPT) * 8;
    const int t = tile * kBKV + tok;
    float x[8];
    if (t < s.nkv && c8 < g.D0) {
      const uint4 u = __ldg(reinterpret_cast<const uint4 *>(a.v + (size_t)(s.kv0 + t) * row_elems +
                                                            (size_t)h * g.D0 + c8));
      unpack8(u, a.bf16, x);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const uint32_t two = cvt_e4m3x2(__fmul_rn(x[e], vinv[c8 + e]), __fmul_rn(x[e + 1], vinv[c8 + e + 1]));
      tb[(c8 + e) * TP + tok] = (uint8_t)(two & 0xFF);
      tb[(c8 + e + 1) * TP + tok] = (uint8_t)(two >> 8);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < DP * (kBKV / 16); i += blockDim.x) {
    const int c = i / (kBKV / 16), part = i % (kBKV / 16);
    const uint4 val = *reinterpret_cast<const uint4 *>(&tb[c * TP + part * 16]);
    *reinterpret_cast<uint4 *>(a.w.vcodeT + ((size_t)h * DP + c) * a.L.Tkv + s.kvpad0 +
                               tile * kBKV + part * 16) = val;
  }
}

// ------------------------------------------------------------------ 4. Q codes
// grid (ceil(max_nq / 128), Hq, B), block 256. The block's 128 x D0 input values are staged in
// shared memory with asynchronous 16-byte copies (few registers, so many CTAs per SM keep enough
// loads in flight). Channel sums: thread t sums channel t % DP over one half of the rows in
// double-float; the two halves are combined in double. The sums are exact for 16-bit inputs, so
// the mean is the definition's fl32(sum / n). Quantization: warp w owns rows 16w .. 16w + 15,
// lane l channels [l * CPL, l * CPL + CPL).
template <int DP>
__global__ void __launch_bounds__(256) q_quant(PrepassArgs a) {
  constexpr int CPL = DP / 32, RPW = 16;
  __shared__ __align__(16) uint16_t blk[kBQ][DP];  // rows past the end / channels past D0: 0
  __shared__ double colsum[2][DP];
  __shared__ float qbar[DP];
  const Geometry &g = a.g;
  const int b = blockIdx.z, h = blockIdx.y, qb = blockIdx.x;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (!s.ok) {
    if (threadIdx.x == 0 && qb == 0 && h == 0) flag_bad_seq(a.w.status);
    return;
  }
  if (qb * kBQ >= ((s.nq + kBQ - 1) / kBQ) * kBQ) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t row_elems = (size_t)g.Hq * g.D0;
  const int nvalid = min(kBQ, s.nq - qb * kBQ);
  // stage: 8-element (16-byte) chunks; D0 % 8 == 0, so a chunk is wholly inside or outside
  constexpr int kChunks = DP / 8;
  for (int c = tid; c < kBQ * kChunks; c += blockDim.x) {
    const int r = c / kChunks, ch = (c % kChunks) * 8;
    uint16_t *dst = &blk[r][ch];
    if (r < nvalid && ch < g.D0) {
      const uint16_t *src = a.q + (size_t)(s.q0 + qb * kBQ + r) * row_elems + (size_t)h * g.D0 + ch;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                   : "memory");
    } else {
      *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  {  // channel sums: thread t, channel t % DP, rows [half * 64, half * 64 + 64) (256 / DP halves)
    constexpr int kParts = 256 / DP, kRowsPer = kBQ / kParts;
    const int d = tid % DP, part = tid / DP;
    float hi = 0.f, lo = 0.f;
#pragma unroll 8
    for (int r = part * kRowsPer; r < (part + 1) * kRowsPer; ++r)
      df_add(hi, lo, to_f32(blk[r][d], a.bf16));  // staged zeros add nothing
    if (kParts == 2) {
      colsum[part][d] = (double)hi + (double)lo;
    } else {  // DP = 64: four parts, folded pairwise into the two slots
      __shared__ double part4[4][64];
      part4[part][d] = (double)hi + (double)lo;
      __syncthreads();
      if (part < 2) colsum[part][d] = part4[2 * part][d] + part4[2 * part + 1][d];
    }
  }
  __syncthreads();
  for (int d = tid; d < DP; d += blockDim.x) {
    const double sum = colsum[0][d] + colsum[1][d];
    const bool smooth = !(a.flags & SAGE2_QUANT_NO_SMOOTH_Q);
    const float m = (smooth && nvalid > 0 && d < g.D0) ? (float)(sum / (double)nvalid) : 0.f;
    qbar[d] = m;
    a.w.qmean[((size_t)h * a.L.nqblk + s.qpad0 / kBQ + qb) * DP + d] = m;
  }
  __syncthreads();
  // Q~ = fl32(Q - qbar); one scale per row (the row spans the warp's 32 lanes)
  const int c0 = lane * CPL;
  const bool chan_ok = c0 < g.D0;
  float mb[CPL];
#pragma unroll
  for (int e = 0; e < CPL; ++e) mb[e] = qbar[c0 + e];
  const int rbase = warp * RPW;  // row within the block
  float amax[RPW];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const bool rv = rbase + r < nvalid && chan_ok;
    amax[r] = 0.f;
#pragma unroll
    for (int e = 0; e < CPL; ++e)
      amax[r] = fmaxf(amax[r], fabsf(rv ? __fsub_rn(to_f32(blk[rbase + r][c0 + e], a.bf16), mb[e]) : 0.f));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int r = 0; r < RPW; ++r) amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], off));
  if (a.flags & SAGE2_QUANT_PER_BLOCK) {  // block-uniform branch: one scale for the valid rows
    __shared__ float wmax[kBQ / RPW];
    float m = 0.f;
#pragma unroll
    for (int r = 0; r < RPW; ++r) m = fmaxf(m, amax[r]);
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
    m = 0.f;
#pragma unroll
    for (int w = 0; w < kBQ / RPW; ++w) m = fmaxf(m, wmax[w]);
#pragma unroll
    for (int r = 0; r < RPW; ++r) amax[r] = rbase + r < nvalid ? m : 0.f;
  }
  const size_t row0 = (size_t)h * a.L.Tq + s.qpad0 + qb * kBQ + rbase;
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const bool rv = rbase + r < nvalid && chan_ok;
    float xt[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e)
      xt[e] = rv ? __fsub_rn(to_f32(blk[rbase + r][c0 + e], a.bf16), mb[e]) : 0.f;
    const float inv = amax[r] > 0.f ? __fdiv_rn(7.f, amax[r]) : 0.f;
    uint8_t *dst = a.w.qcode + (row0 + r) * DP + c0;
    if (CPL == 4) {
      const uint32_t lo2 = cvt_e4m3x2(int4_code(xt[0], inv), int4_code(xt[1], inv));
      const uint32_t hi2 = cvt_e4m3x2(int4_code(xt[2], inv), int4_code(xt[3], inv));
      *reinterpret_cast<uint32_t *>(dst) = lo2 | (hi2 << 16);
    } else {
      *reinterpret_cast<uint16_t *>(dst) =
          (uint16_t)cvt_e4m3x2(int4_code(xt[0], inv), int4_code(xt[1], inv));
    }
    if (lane == 0) a.w.qscale[row0 + r] = amax[r] > 0.f ? __fdiv_rn(amax[r], 7.f) : 0.f;
  }
}

// ------------------------------------------------------------------ 5. DeltaS
// A small FP32 GEMM per (sequence, kv head): rows are the (Q block, q head of the group)
// pairs, ordered Q-block-major (r = qb * g + head), columns the keys, inner dimension the
// channels. grid (key tiles of 128, row tiles of 128, B * Hkv), block 256. Thread (tr, tk)
// owns rows 8tr..8tr+7 and keys 8tk..8tk+7; channels are staged 32 at a time in shared memory,
// transposed, and every output is one FMA chain in increasing channel order (the same
// operation sequence as the definition, so the result is bit-identical to it). Causal: a
// (row tile, key tile) pair that no row of the tile visits is skipped; rows that do not visit
// the key tile are not written.
constexpr int kDsRows = 128, kDsKeys = 128, kDsChan = 32;

template <int DP>
__global__ void __launch_bounds__(256) delta_s(PrepassArgs a) {
  __shared__ __align__(16) float Qs[kDsChan][kDsRows];
  __shared__ __align__(16) float Ks[kDsChan][kDsKeys];
  const Geometry &g = a.g;
  const int kt = blockIdx.x, rt = blockIdx.y;
  const int b = blockIdx.z / g.Hkv, hk = blockIdx.z % g.Hkv;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (!s.ok || kt * kBKV >= s.nkv || s.nq == 0) return;
  const int grp = g.Hq / g.Hkv;
  const int nqb = (s.nq + kBQ - 1) / kBQ;
  const int nrows = grp * nqb;
  const int r0 = rt * kDsRows;
  if (r0 >= nrows) return;
  const int qb_last = min(nrows - 1, r0 + kDsRows - 1) / grp;
  if (g.causal && kv_tiles_for(qb_last, s.nq, s.nkv, 1) <= kt) return;

  const int tid = threadIdx.x;
  const int tr = tid >> 4, tk = tid & 15;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  // loader roles: row / key = tid / 2, channel half = (tid & 1) * 16 of the 32-channel chunk
  const int lr = tid >> 1, lh = (tid & 1) * 16;
  const int key = kt * kBKV + lr;
  const bool key_ok = key < s.nkv;
  const uint16_t *ksrc = a.k + (size_t)(s.kv0 + (key_ok ? key : 0)) * g.Hkv * g.D0 + (size_t)hk * g.D0;
  const float *mu = a.w.kmean + ((size_t)b * g.Hkv + hk) * DP;
  const int r = r0 + lr;
  const bool row_ok = r < nrows;
  const float *qsrc = nullptr;
  if (row_ok) {
    const int qb = r / grp, hq = hk * grp + r % grp;
    qsrc = a.w.qmean + ((size_t)hq * a.L.nqblk + s.qpad0 / kBQ + qb) * DP;
  }

#pragma unroll 1
  for (int c0 = 0; c0 < DP; c0 += kDsChan) {
    const int cb = c0 + lh;  // first channel this thread loads
    float kv[16], qv[16];
    if (key_ok && cb < g.D0) {
      float x[8];
      unpack8(__ldg(reinterpret_cast<const uint4 *>(ksrc + cb)), a.bf16, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) kv[e] = __fsub_rn(x[e], mu[cb + e]);
      unpack8(__ldg(reinterpret_cast<const uint4 *>(ksrc + cb + 8)), a.bf16, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) kv[8 + e] = __fsub_rn(x[e], mu[cb + 8 + e]);
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) kv[e] = 0.f;
    }
    if (row_ok) {
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        const float4 m4 = __ldg(reinterpret_cast<const float4 *>(qsrc + cb + e));
        qv[e] = m4.x;
        qv[e + 1] = m4.y;
        qv[e + 2] = m4.z;
        qv[e + 3] = m4.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) qv[e] = 0.f;
    }
    __syncthreads();  // the previous chunk's reads are done
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      Ks[lh + e][lr] = kv[e];
      Qs[lh + e][lr] = qv[e];
    }
    __syncthreads();
#pragma unroll 4
    for (int d = 0; d < kDsChan; ++d) {
      const float4 qa = *reinterpret_cast<const float4 *>(&Qs[d][tr * 8]);
      const float4 qc = *reinterpret_cast<const float4 *>(&Qs[d][tr * 8 + 4]);
      const float4 ka = *reinterpret_cast<const float4 *>(&Ks[d][tk * 8]);
      const float4 kc = *reinterpret_cast<const float4 *>(&Ks[d][tk * 8 + 4]);
      const float qq[8] = {qa.x, qa.y, qa.z, qa.w, qc.x, qc.y, qc.z, qc.w};
      const float kk[8] = {ka.x, ka.y, ka.z, ka.w, kc.x, kc.y, kc.z, kc.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; j += 2)  // packed: two independent, correctly rounded FMAs
          fma2(acc[i][j], acc[i][j + 1], qq[i], qq[i], kk[j], kk[j + 1], acc[i][j], acc[i][j + 1]);
    }
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = r0 + tr * 8 + i;
    if (rr >= nrows) break;
    const int qb = rr / grp, hq = hk * grp + rr % grp;
    if (g.causal && kv_tiles_for(qb, s.nq, s.nkv, 1) <= kt) continue;
    float *dst = a.w.dsc + ((size_t)hq * a.L.nqblk + s.qpad0 / kBQ + qb) * a.L.nkv_pad +
                 (size_t)kt * kBKV + tk * 8;
    float4 lo, hi;
    lo.x = __fmul_rn(acc[i][0], g.c32);
    lo.y = __fmul_rn(acc[i][1], g.c32);
    lo.z = __fmul_rn(acc[i][2], g.c32);
    lo.w = __fmul_rn(acc[i][3], g.c32);
    hi.x = __fmul_rn(acc[i][4], g.c32);
    hi.y = __fmul_rn(acc[i][5], g.c32);
    hi.z = __fmul_rn(acc[i][6], g.c32);
    hi.w = __fmul_rn(acc[i][7], g.c32);
    reinterpret_cast<float4 *>(dst)[0] = lo;
    reinterpret_cast<float4 *>(dst)[1] = hi;
  }
}

}  // namespace

cudaError_t launch_prepass(const void *q, const void *k, const void *v, int in_dtype,
                           int quant_flags, const Geometry &g, const Layout &L, void *ws,
                           cudaStream_t st) {
  PrepassArgs a;
  a.q = static_cast<const uint16_t *>(q);
  a.k = static_cast<const uint16_t *>(k);
  a.v = static_cast<const uint16_t *>(v);
  a.bf16 = in_dtype == SAGE2_BF16;
  a.flags = quant_flags;
  a.g = g;
  a.L = L;
  a.w = ws_ptrs(ws, L);
  cudaError_t e = cudaMemsetAsync(a.w.status, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;

  const int nvec = g.Hkv * g.D0 / 8;
  int threads = ((nvec + 31) / 32) * 32;
  threads = threads < 32 ? 32 : (threads > 256 ? 256 : threads);
  kv_stats_partial<<<dim3(L.nchunk, g.B), threads, 0, st>>>(a);
  kv_stats_final<<<g.B * g.Hkv, g.Dp, 0, st>>>(a);
  // every grid dimension at least 1 (a zero-length maximum is legal; the kernels bound-check)
  const int kv_tiles = max(1, (g.max_nkv + kBKV - 1) / kBKV);
  const int q_tiles = max(1, (g.max_nq + kBQ - 1) / kBQ);
  const dim3 kv_grid(kv_tiles, g.Hkv, g.B);
  const dim3 q_grid(q_tiles, g.Hq, g.B);
  const int max_rows = (g.Hq / g.Hkv) * q_tiles;
  const dim3 ds_grid(kv_tiles, (max_rows + kDsRows - 1) / kDsRows, g.B * g.Hkv);
  if (g.Dp == 128) {
    k_quant<128><<<kv_grid, 128, 0, st>>>(a);
    v_quant<128><<<kv_grid, 256, 0, st>>>(a);
    q_quant<128><<<q_grid, 256, 0, st>>>(a);
    delta_s<128><<<ds_grid, 256, 0, st>>>(a);
  } else {
    k_quant<64><<<kv_grid, 128, 0, st>>>(a);
    v_quant<64><<<kv_grid, 256, 0, st>>>(a);
    q_quant<64><<<q_grid, 256, 0, st>>>(a);
    delta_s<64><<<ds_grid, 256, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace sage2
