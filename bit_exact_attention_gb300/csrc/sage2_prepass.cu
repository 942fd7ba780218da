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
//   5. delta_s_tc: DeltaS = qmean . K~ on the tensor cores (both operands split exactly into
//      three bf16 pieces, the six leading piece products summed in FP32), stored multiplied by
//      c = log2(e) * sm_scale.
// Every padded position (channels D0..Dp, tokens past a sequence end up to its 128-row
// boundary) is written with zero codes and zero scales.
// Ablation switches (sage2_quant_flags) change only what these kernels write: a zero K
// channel mean (kv_stats_final), a zero Q block mean (q_quant), or one INT4 scale per 128-key
// K tile (k_quant) and per 128-row Q block (q_quant), still stored per 32-key group and per
// row so that the attention kernel reads them unchanged.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "sage2_device.cuh"
#include "sage2_internal.h"

namespace sage2 {
namespace {

struct PrepassArgs {
  const uint16_t *q, *k, *v;
  int flags;     // sage2_quant_flags
  int ds_chunk;  // delta_s_tc: key tiles per CTA
  Geometry g;
  Layout L;
  WsPtrs w;
};

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t bits) {
  if (BF16) return __uint_as_float(((uint32_t)bits) << 16);
  return __half2float(__ushort_as_half(bits));
}

// The two 16-bit values of a 32-bit word (low half first) as floats.
template <bool BF16>
__device__ __forceinline__ void unpack2(uint32_t w, float &x0, float &x1) {
  if (BF16) {
    x0 = __uint_as_float(w << 16);
    x1 = __uint_as_float(w & 0xFFFF0000u);
  } else {
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
    x0 = f.x;
    x1 = f.y;
  }
}

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4 &u, float (&x)[8]) {
  unpack2<BF16>(u.x, x[0], x[1]);
  unpack2<BF16>(u.y, x[2], x[3]);
  unpack2<BF16>(u.z, x[4], x[5]);
  unpack2<BF16>(u.w, x[6], x[7]);
}

// INT4-grid code of x * inv, as an e4m3 byte (canonical +0 for zero).
__device__ __forceinline__ float int4_code(float x, float inv) {
  float r = rintf(__fmul_rn(x, inv));
  r = fminf(fmaxf(r, -7.f), 7.f);
  return __fadd_rn(r, 0.f);
}

// Code of x * inv on the grid [-G, G] as a float (canonical +0 for zero).
__device__ __forceinline__ float grid_code(float x, float inv, float G) {
  float r = rintf(__fmul_rn(x, inv));
  r = fminf(fmaxf(r, -G), G);
  return __fadd_rn(r, 0.f);
}

__device__ __forceinline__ void flag_bad_seq(int *status) {
  atomicCAS(status, 0, kStatusSeqTooLong);
}

// ------------------------------------------------------------------ 1a. K/V statistics
// grid (nchunk, B, ceil(nvec / VPB)), block kStatThreads, nvec = Hkv * D0 / 8 vectors of 8
// channels per token. A block covers VPB = min(nvec, kStatThreads) vectors and splits the
// chunk's kStatChunk tokens over L = kStatThreads / VPB token lanes (a row of few vectors, as in
// a chunk of one kv head, still keeps the block busy); each thread walks its tokens with
// double-float sums, and the lanes' partials (each exact) are added in lane order in FP64.
constexpr int kStatThreads = 128;
template <bool BF16>
__global__ void __launch_bounds__(kStatThreads) kv_stats_partial(PrepassArgs a) {
  __shared__ double lane_sum[kStatThreads][8];
  __shared__ float lane_max[kStatThreads][8];
  const int b = blockIdx.y, chunk = blockIdx.x;
  const Geometry &g = a.g;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (!s.ok) {
    if (threadIdx.x == 0 && chunk == 0 && blockIdx.z == 0) flag_bad_seq(a.w.status);
    return;
  }
  const int t0 = chunk * kStatChunk;
  if (t0 >= s.nkv) return;
  const int t1 = min(t0 + kStatChunk, s.nkv);
  const int row_elems = g.Hkv * g.D0;
  const int nvec = row_elems / 8;
  const int vpb = min(nvec, kStatThreads), lanes = kStatThreads / vpb;
  const int vl = threadIdx.x % vpb, lane = threadIdx.x / vpb;
  const int vi = blockIdx.z * vpb + vl;
  const bool active = lane < lanes && vi < nvec;
  float hi[8], lo[8], mx[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) hi[e] = lo[e] = mx[e] = 0.f;
  if (active) {
    const uint4 *kp = reinterpret_cast<const uint4 *>(a.k + (size_t)(s.kv0 + t0) * row_elems) + vi;
    const uint4 *vp = reinterpret_cast<const uint4 *>(a.v + (size_t)(s.kv0 + t0) * row_elems) + vi;
    const int stride = nvec;
    constexpr int U = 8;  // tokens whose loads are all issued before any is used
#pragma unroll 1
    for (int t = t0 + lane; t < t1; t += U * lanes) {
      uint4 kk[U], vv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {  // tokens past the end read as 0 and add nothing
        const int tu = t + u * lanes;
        const bool ok = tu < t1;
        kk[u] = ok ? __ldg(kp + (size_t)(tu - t0) * stride) : make_uint4(0u, 0u, 0u, 0u);
        vv[u] = ok ? __ldg(vp + (size_t)(tu - t0) * stride) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float xk[8], xv[8];
        unpack8<BF16>(kk[u], xk);
        unpack8<BF16>(vv[u], xv);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          df_add2(hi[e], hi[e + 1], lo[e], lo[e + 1], xk[e], xk[e + 1]);
          mx[e] = fmaxf(mx[e], fabsf(xv[e]));
          mx[e + 1] = fmaxf(mx[e + 1], fabsf(xv[e + 1]));
        }
      }
    }
  }
  if (lanes > 1) {  // block-uniform: combine the token lanes of each vector
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      lane_sum[threadIdx.x][e] = (double)hi[e] + (double)lo[e];
      lane_max[threadIdx.x][e] = mx[e];
    }
    __syncthreads();
    if (lane != 0 || !active) return;
    double sum[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sum[e] = lane_sum[vl][e];
    for (int l = 1; l < lanes; ++l)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sum[e] += lane_sum[l * vpb + vl][e];
        mx[e] = fmaxf(mx[e], lane_max[l * vpb + vl][e]);
      }
    const size_t o = ((size_t)b * a.L.nchunk + chunk) * row_elems + (size_t)vi * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      a.w.kpart[o + e] = sum[e];
      a.w.vpart[o + e] = mx[e];
    }
    return;
  }
  if (!active) return;
  const size_t o = ((size_t)b * a.L.nchunk + chunk) * row_elems + (size_t)vi * 8;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    a.w.kpart[o + e] = (double)hi[e] + (double)lo[e];
    a.w.vpart[o + e] = mx[e];
  }
}

// grid (B * Hkv, Dp / CH), block 1024 = CH channels x 1024 / CH parts: part p sums chunks p,
// p + parts, ... in FP64, then the parts are added pairwise in a fixed tree. The chunk sums are
// exact (see above), and so is every FP64 sum of them for 16-bit inputs, so the order does not
// change the result. CH = 32 when the grid already has enough blocks; CH = 8 (128 parts, so
// each thread adds few chunks) when it has few, as for a single kv head, where this reduction
// is otherwise a chain of dependent loads on a handful of SMs.
constexpr int kFinalThreads = 1024;
template <int CH>
__global__ void __launch_bounds__(kFinalThreads) kv_stats_final(PrepassArgs a) {
  constexpr int kParts = kFinalThreads / CH;
  __shared__ double psum[kParts][CH];
  __shared__ float pmax[kParts][CH];
  const Geometry &g = a.g;
  const int b = blockIdx.x / g.Hkv, h = blockIdx.x % g.Hkv;
  const int dl = threadIdx.x % CH, part = threadIdx.x / CH;
  const int d = blockIdx.y * CH + dl;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  const bool live = s.ok && d < g.D0 && s.nkv > 0;
  double sum = 0.0;
  float amax = 0.f;
  if (live) {
    const int nch = (s.nkv + kStatChunk - 1) / kStatChunk;
    const int row_elems = g.Hkv * g.D0;
#pragma unroll 4
    for (int c = part; c < nch; c += kParts) {
      const size_t po = ((size_t)b * a.L.nchunk + c) * row_elems + (size_t)h * g.D0 + d;
      sum += a.w.kpart[po];
      amax = fmaxf(amax, a.w.vpart[po]);
    }
  }
  psum[part][dl] = sum;
  pmax[part][dl] = amax;
  __syncthreads();
#pragma unroll
  for (int n = kParts / 2; n >= 1; n >>= 1) {
    if (part < n) {
      psum[part][dl] += psum[part + n][dl];
      pmax[part][dl] = fmaxf(pmax[part][dl], pmax[part + n][dl]);
    }
    __syncthreads();
  }
  if (part != 0) return;
  sum = psum[0][dl];
  amax = pmax[0][dl];
  const size_t o = ((size_t)b * g.Hkv + h) * g.Dp + d;
  float mean = 0.f;
  if (live) mean = (a.flags & SAGE2_QUANT_NO_SMOOTH_K) ? 0.f : (float)(sum / (double)s.nkv);
  a.w.kmean[o] = mean;
  a.w.vscale[o] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
  a.w.vinv[o] = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
}

// ------------------------------------------------------------------ 2. K codes
// grid (ceil(max_nkv / 128), Hkv, B), block 256. The tile's 128 x D0 keys are staged in shared
// memory with asynchronous 16-byte copies (rows past the end and channels past D0 read as 0);
// warp w handles keys 16w .. 16w + 15, i.e. half of the 32-key scale group w / 2; lane l
// channels [l * CPL, l * CPL + CPL). Per-block switch: the eight warps share one maximum.
template <int DP, bool BF16, bool I8>
__global__ void __launch_bounds__(256) k_quant(PrepassArgs a) {
  constexpr int CPL = DP / 32, RPW = 16;
  constexpr float G = I8 ? 127.f : 7.f;  // the code grid [-G, G]
  __shared__ __align__(16) uint16_t blk[kBKV][DP];
  __shared__ float wmax[kBKV / RPW];
  const Geometry &g = a.g;
  const int b = blockIdx.z, h = blockIdx.y, tile = blockIdx.x;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (!s.ok || tile * kBKV >= ((s.nkv + kBKV - 1) / kBKV) * kBKV) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t row_elems = (size_t)g.Hkv * g.D0;
  const int nvalid = min(kBKV, s.nkv - tile * kBKV);
  constexpr int kChunks = DP / 8;
  for (int c = tid; c < kBKV * kChunks; c += blockDim.x) {
    const int r = c / kChunks, ch = (c % kChunks) * 8;
    uint16_t *dst = &blk[r][ch];
    if (r < nvalid && ch < g.D0) {
      const uint16_t *src = a.k + (size_t)(s.kv0 + tile * kBKV + r) * row_elems + (size_t)h * g.D0 + ch;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                   : "memory");
    } else {
      *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  const int c0 = lane * CPL;
  const bool chan_ok = c0 < g.D0;  // D0 % 8 == 0, so a lane's channels are all in or all out
  float mu[CPL];
#pragma unroll
  for (int e = 0; e < CPL; ++e) mu[e] = a.w.kmean[((size_t)b * g.Hkv + h) * DP + c0 + e];
  const int rbase = warp * RPW;
  auto smoothed = [&](int r, int e) {  // K~ = fl32(K - kmean); 0 outside the data
    return (rbase + r < nvalid && chan_ok) ? __fsub_rn(to_f32<BF16>(blk[rbase + r][c0 + e]), mu[e])
                                           : 0.f;
  };
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < RPW; ++r)
#pragma unroll
    for (int e = 0; e < CPL; ++e) amax = fmaxf(amax, fabsf(smoothed(r, e)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) wmax[warp] = amax;
  __syncthreads();
  if (a.flags & SAGE2_QUANT_PER_BLOCK) {
#pragma unroll
    for (int w = 0; w < kBKV / RPW; ++w) amax = fmaxf(amax, wmax[w]);
  } else {
    amax = fmaxf(wmax[warp & ~1], wmax[warp | 1]);  // the two halves of the 32-key group
  }
  const float inv = amax > 0.f ? __fdiv_rn(G, amax) : 0.f;
  const float scale = amax > 0.f ? __fdiv_rn(amax, G) : 0.f;
  const size_t e0 = ((size_t)h * a.L.Tkv + s.kvpad0 + tile * kBKV + rbase) * DP + c0;
  uint8_t *dst = a.w.kcode + e0;
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    if (I8) {  // INT8-grid codes as fp16 values (exact), two bytes each
      uint16_t hv[CPL];
#pragma unroll
      for (int e = 0; e < CPL; ++e)
        hv[e] = __half_as_ushort(__float2half_rn(grid_code(smoothed(r, e), inv, G)));
      uint16_t *d16 = reinterpret_cast<uint16_t *>(a.w.kcode) + e0 + (size_t)r * DP;
      if (CPL == 4)
        *reinterpret_cast<uint2 *>(d16) = make_uint2(hv[0] | ((uint32_t)hv[1] << 16),
                                                     hv[2] | ((uint32_t)hv[3] << 16));
      else
        *reinterpret_cast<uint32_t *>(d16) = hv[0] | ((uint32_t)hv[1] << 16);
    } else if (CPL == 4) {
      const uint32_t lo = cvt_e4m3x2(int4_code(smoothed(r, 0), inv), int4_code(smoothed(r, 1), inv));
      const uint32_t hi = cvt_e4m3x2(int4_code(smoothed(r, 2), inv), int4_code(smoothed(r, 3), inv));
      *reinterpret_cast<uint32_t *>(dst + (size_t)r * DP) = lo | (hi << 16);
    } else {
      *reinterpret_cast<uint16_t *>(dst + (size_t)r * DP) =
          (uint16_t)cvt_e4m3x2(int4_code(smoothed(r, 0), inv), int4_code(smoothed(r, 1), inv));
    }
  }
  if (lane == 0 && (warp & 1) == 0)
    a.w.kscale[(size_t)h * (a.L.Tkv / kGK) + (s.kvpad0 + tile * kBKV) / kGK + warp / 2] = scale;
}

// ------------------------------------------------------------------ 3. V codes, transposed
// grid (ceil(max_nkv / 128), Hkv, B), block 256. Warp w covers 64 channels (channel group
// w % CG, CG = DP / 64) of TPW = 128 / (8 / CG) consecutive tokens (token group w / CG); lane l
// owns channels 2l, 2l + 1 of the group. Each token row is one 128-byte load per warp; each
// lane writes TPW contiguous code bytes per channel (whole 16- or 32-byte pieces of the
// transposed rows), so no shared-memory transpose is needed.
template <int DP, bool BF16>
__global__ void __launch_bounds__(256) v_quant(PrepassArgs a) {
  constexpr int CG = DP / 64, TG = 8 / CG, TPW = kBKV / TG, WORDS = TPW / 4;
  const Geometry &g = a.g;
  const int b = blockIdx.z, h = blockIdx.y, tile = blockIdx.x;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (!s.ok || tile * kBKV >= ((s.nkv + kBKV - 1) / kBKV) * kBKV) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = 64 * (warp % CG) + 2 * lane;
  const int t0 = tile * kBKV + TPW * (warp / CG);  // sequence-local first token
  const bool chan_ok = c < g.D0;                  // D0 even: both channels in or out
  const size_t vo = ((size_t)b * g.Hkv + h) * DP + c;
  const float inv0 = a.w.vinv[vo], inv1 = a.w.vinv[vo + 1];
  const size_t row_elems = (size_t)g.Hkv * g.D0;
  const uint16_t *src = a.v + (size_t)(s.kv0 + t0) * row_elems + (size_t)h * g.D0 + c;
  uint32_t raw[TPW];
#pragma unroll
  for (int u = 0; u < TPW; ++u)
    raw[u] = (chan_ok && t0 + u < s.nkv) ? __ldg(reinterpret_cast<const uint32_t *>(src + (size_t)u * row_elems))
                                         : 0u;
  uint32_t w0[WORDS], w1[WORDS];
#pragma unroll
  for (int i = 0; i < WORDS; ++i) w0[i] = w1[i] = 0u;
#pragma unroll
  for (int u = 0; u < TPW; ++u) {
    float x0, x1;
    unpack2<BF16>(raw[u], x0, x1);
    const uint32_t two = cvt_e4m3x2(__fmul_rn(x0, inv0), __fmul_rn(x1, inv1));
    w0[u / 4] |= (two & 0xFFu) << (8 * (u % 4));
    w1[u / 4] |= ((two >> 8) & 0xFFu) << (8 * (u % 4));
  }
  uint8_t *d0 = a.w.vcodeT + ((size_t)h * DP + c) * a.L.Tkv + s.kvpad0 + t0;
  uint8_t *d1 = d0 + a.L.Tkv;
#pragma unroll
  for (int i = 0; i < WORDS; i += 4) {
    *reinterpret_cast<uint4 *>(d0 + 4 * i) = make_uint4(w0[i], w0[i + 1], w0[i + 2], w0[i + 3]);
    *reinterpret_cast<uint4 *>(d1 + 4 * i) = make_uint4(w1[i], w1[i + 1], w1[i + 2], w1[i + 3]);
  }
}

// fl32(sum / n) of an exact FP64 sum over n rows. A whole block (n = 128) divides by a power of
// two, so the quotient is exact and fl32(sum / 128) = fl32(sum) * 2^-7 whenever that is a normal
// float; this skips the FP64 division, which GB300's few FP64 units made the bottleneck of the Q
// codes kernel (one per channel of every block). Other n, and results outside the normal range,
// take the division.
__device__ __forceinline__ float block_mean(double sum, int n) {
  if (n == kBQ) {
    const float f = __double2float_rn(sum);
    const float af = fabsf(f);
    if (af == 0.f || (af >= 0x1p-119f && af <= 0x1p127f)) return __fmul_rn(f, 1.f / kBQ);
  }
  return __double2float_rn(sum / (double)n);
}

// ------------------------------------------------------------------ 4. Q codes
// grid (ceil(max_nq / 128), Hq, B), block 256. The block's 128 x D0 input values are staged in
// shared memory with asynchronous 16-byte copies (few registers, so many CTAs per SM keep enough
// loads in flight). Channel sums: thread t owns the channel pair 2 (t % (DP/2)) and one of
// 256 / (DP/2) row ranges, summed as two double-float accumulators; the ranges are combined in
// double. The sums are exact for 16-bit inputs, so the mean is the definition's fl32(sum / n).
// Quantization: warp w owns rows 16w .. 16w + 15, lane l channels [l * CPL, l * CPL + CPL), all
// elementwise steps on packed FP32 pairs (each lane of a pair rounds like the scalar form).
template <int DP, bool BF16, bool I8>
__global__ void __launch_bounds__(256) q_quant(PrepassArgs a) {
  constexpr int CPL = DP / 32, RPW = 16;
  constexpr float G = I8 ? 127.f : 7.f;  // the code grid [-G, G]
  constexpr int kPairs = DP / 2, kParts = 256 / kPairs, kRowsPer = kBQ / kParts;
  __shared__ __align__(16) uint16_t blk[kBQ][DP];  // rows past the end / channels past D0: 0
  __shared__ double colsum[kParts][DP];
  __shared__ float qbar[DP];
  __shared__ float wmax[kBQ / RPW];
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
  {  // channel sums (staged zeros add nothing)
    const int d = 2 * (tid % kPairs), part = tid / kPairs;
    float hi0 = 0.f, hi1 = 0.f, lo0 = 0.f, lo1 = 0.f;
#pragma unroll 8
    for (int r = part * kRowsPer; r < (part + 1) * kRowsPer; ++r) {
      float x0, x1;
      unpack2<BF16>(*reinterpret_cast<const uint32_t *>(&blk[r][d]), x0, x1);
      df_add2(hi0, hi1, lo0, lo1, x0, x1);
    }
    colsum[part][d] = (double)hi0 + (double)lo0;
    colsum[part][d + 1] = (double)hi1 + (double)lo1;
  }
  __syncthreads();
  for (int d = tid; d < DP; d += blockDim.x) {
    double sum = colsum[0][d];
#pragma unroll
    for (int p = 1; p < kParts; ++p) sum += colsum[p][d];
    const bool smooth = !(a.flags & SAGE2_QUANT_NO_SMOOTH_Q);
    const float m = (smooth && nvalid > 0 && d < g.D0) ? block_mean(sum, nvalid) : 0.f;
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
  auto smoothed = [&](int r, float (&x)[CPL]) {
    if (rbase + r < nvalid && chan_ok) {
      if (CPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(&blk[rbase + r][c0]);
        unpack2<BF16>(w.x, x[0], x[1]);
        unpack2<BF16>(w.y, x[2], x[3]);
      } else {
        unpack2<BF16>(*reinterpret_cast<const uint32_t *>(&blk[rbase + r][c0]), x[0], x[1]);
      }
#pragma unroll
      for (int e = 0; e < CPL; e += 2) sub2(x[e], x[e + 1], x[e], x[e + 1], mb[e], mb[e + 1]);
    } else {
#pragma unroll
      for (int e = 0; e < CPL; ++e) x[e] = 0.f;
    }
  };
  float amax[RPW];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    float x[CPL];
    smoothed(r, x);
    amax[r] = 0.f;
#pragma unroll
    for (int e = 0; e < CPL; ++e) amax[r] = fmaxf(amax[r], fabsf(x[e]));
  }
  // Transposing butterfly: after the steps over lane bits 4..1 lane l holds the maximum of row
  // l >> 1 over the lanes that agree with it in those bits; the last step (bit 0) completes it.
#pragma unroll
  for (int half = RPW / 2, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
    const bool upper = lane & bit;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? amax[i] : amax[i + half];
      const float keep = upper ? amax[i + half] : amax[i];
      amax[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, bit));
    }
  }
  float rmax = fmaxf(amax[0], __shfl_xor_sync(0xffffffffu, amax[0], 1));  // row lane >> 1
  if (a.flags & SAGE2_QUANT_PER_BLOCK) {  // block-uniform branch: one scale for the valid rows
    float m = rmax;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
    m = 0.f;
#pragma unroll
    for (int w = 0; w < kBQ / RPW; ++w) m = fmaxf(m, wmax[w]);
    rmax = rbase + (lane >> 1) < nvalid ? m : 0.f;
  }
  // one division per lane (row lane >> 1); rows past the end have rmax = 0: codes and scale 0
  const float inv_mine = rmax > 0.f ? __fdiv_rn(G, rmax) : 0.f;
  const size_t row0 = (size_t)h * a.L.Tq + s.qpad0 + qb * kBQ + rbase;
  if ((lane & 1) == 0) a.w.qscale[row0 + (lane >> 1)] = rmax > 0.f ? __fdiv_rn(rmax, G) : 0.f;
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    float x[CPL];
    smoothed(r, x);
    const float inv = __shfl_sync(0xffffffffu, inv_mine, 2 * r);
    float t[CPL];
#pragma unroll
    for (int e = 0; e < CPL; e += 2) mul2(t[e], t[e + 1], x[e], x[e + 1], inv, inv);
#pragma unroll
    for (int e = 0; e < CPL; ++e) t[e] = rintf(t[e]);
    // |x| <= rmax and inv = fl32(G / rmax) give |fl32(x * inv)| <= G whenever inv is finite
    // (G(1 + 2^-24) rounds to G for G = 7 and 127); only an overflowed inv (rmax below
    // G / FLT_MAX) needs the clamp to [-G, G]
    if (__builtin_expect(isinf(inv), 0)) {
#pragma unroll
      for (int e = 0; e < CPL; ++e) t[e] = fminf(fmaxf(t[e], -G), G);
    }
#pragma unroll
    for (int e = 0; e < CPL; e += 2) add2(t[e], t[e + 1], t[e], t[e + 1], 0.f, 0.f);  // +0 for -0
    uint8_t *dst = a.w.qcode + (row0 + r) * DP + c0;
    if (I8) {  // INT8-grid codes as fp16 values (exact), two bytes each
      uint16_t *d16 = reinterpret_cast<uint16_t *>(a.w.qcode) + (row0 + r) * DP + c0;
      uint16_t hv[CPL];
#pragma unroll
      for (int e = 0; e < CPL; ++e) hv[e] = __half_as_ushort(__float2half_rn(t[e]));
      if (CPL == 4)
        *reinterpret_cast<uint2 *>(d16) = make_uint2(hv[0] | ((uint32_t)hv[1] << 16),
                                                     hv[2] | ((uint32_t)hv[3] << 16));
      else
        *reinterpret_cast<uint32_t *>(d16) = hv[0] | ((uint32_t)hv[1] << 16);
    } else if (CPL == 4) {
      *reinterpret_cast<uint32_t *>(dst) = cvt_e4m3x2(t[0], t[1]) | (cvt_e4m3x2(t[2], t[3]) << 16);
    } else {
      *reinterpret_cast<uint16_t *>(dst) = (uint16_t)cvt_e4m3x2(t[0], t[1]);
    }
  }
}

// ------------------------------------------------------------------ 5. DeltaS
// DeltaS on the tensor cores. Per (sequence, kv head) a GEMM: rows are the (Q block, q head of
// the group) pairs, ordered Q-block-major (r = qb * grp + head), columns the keys, inner
// dimension the channels; out[r][j] = fl32(c * fl32(qmean_r . K~_j)), K~ = fl32(K - kmean).
// Each FP32 operand is split exactly into three bf16 pieces (x = x1 + x2 + x3 with truncation:
// x1 the top 8 significant bits, x2 the next 8, x3 the last 8, each exactly a bf16), and the
// six products xa_i * xb_j with i + j <= 4 (1-based) are summed by kind::f16 MMAs into one FP32
// accumulator in tensor memory, smallest first. Each piece product is exact; the three dropped
// ones are below 2^-23 of |qmean_d K~_jd|, and the accumulator rounds once per MMA step
// (6 x D / 16 steps), so the result lies within about 50 units of 2^-24 of
// sum_d |qmean_d K~_jd| of the exact dot product.
// One CTA per (128-row tile, chunk of ds_chunk key tiles, sequence x kv head); warps:
//   0-7  per key tile K~ of 32 keys x half the channels per warp: each load instruction reads
//        whole 128-byte row segments (DP / 16 lanes per segment), and each lane splits its
//        8 channels and stores the three 16-byte pieces straight into their swizzled places in
//        one of two shared buffers (the split is elementwise, so no lane needs another's
//        data); warps 0-3 first put the qmean pieces into tensor memory (thread = row = TMEM
//        lane, 16 channels at a time);
//   8-11 epilogue: one accumulator row per thread, 32 columns at a time times c, through a
//        small swizzled shared block so that the global stores are whole 128-byte segments,
//        for the key tiles each row's Q block visits;
//   12   MMA issuer (one lane); it also allocates tensor memory.
// Tensor memory: the qmean pieces at [0, 3 DP / 2), two 128-column accumulators at 256 and 384.
// key tiles per CTA: 16, 8 or 4, whichever gives the least waves x (key tiles per CTA + the
// per-CTA set-up, measured at about 3 key tiles' time; ties to the larger chunk). With few heads
// a grid of 16-tile CTAs can cover under half the SMs (causal rows see few key tiles), and a
// smaller chunk fills them; with many, the set-up of more CTAs outweighs the shorter tail.
constexpr int kDsChunkMax = 16, kDsChunkMin = 4, kDsCtaSetupTiles = 3;
constexpr int kDsThreads = 416, kDsLoadWarps = 8, kDsMmaWarp = 12;  // epilogue: warps 8-11

template <int DP>
struct DsPlan {
  static constexpr int kPiece = 128 * DP * 2;         // one bf16 piece of 128 keys x DP
  static constexpr int kBuf = 3 * kPiece;             // the three pieces
  static constexpr int kB = 0;                        // [2][3][DP / 64][128][128 B] (swizzled)
  static constexpr int kStage = kB + 2 * kBuf;        // float [4 warps][32][32] (swizzled)
  static constexpr int kMu = kStage + 4 * 32 * 32 * 4;  // float [DP]
  static constexpr int kBar = kMu + DP * 4;           // a_full, b_full[2], b_empty[2],
  static constexpr int kNumBars = 1 + 2 + 2 + 2 + 2 + 1;  // acc_full[2], acc_empty[2], drain
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16 + 1024;
  static_assert(kBytes <= 227 * 1024, "shared memory plan too large");
};

// Instruction descriptor, kind::f16 with A = B = bf16, D = f32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// x = p0 + p1 + p2 exactly, each a bf16 (as its 16 bits): truncation to the top 8 significant
// bits, twice, leaves at most 8 significant bits in the last remainder.
__device__ __forceinline__ void split3(float x, uint32_t &p0, uint32_t &p1, uint32_t &p2) {
  const uint32_t b0 = __float_as_uint(x) & 0xFFFF0000u;
  const float r1 = __fsub_rn(x, __uint_as_float(b0));
  const uint32_t b1 = __float_as_uint(r1) & 0xFFFF0000u;
  const float r2 = __fsub_rn(r1, __uint_as_float(b1));
  p0 = b0 >> 16;
  p1 = b1 >> 16;
  p2 = __float_as_uint(r2) >> 16;
}

__device__ __forceinline__ bool ds_wait(uint64_t *bar, uint32_t parity, const AbortCtx &ab,
                                        int site) {
  return __shfl_sync(0xffffffffu, mbar_wait(bar, parity, ab, site) ? 1 : 0, 0) != 0;
}

template <int DP, bool BF16>
__global__ void __launch_bounds__(kDsThreads, 1) delta_s_tc(PrepassArgs a) {
  using P = DsPlan<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Geometry &g = a.g;
  const int rt = blockIdx.y;
  const int b = blockIdx.z / g.Hkv, hk = blockIdx.z % g.Hkv;
  const Seq s = seq_info(g.cu_q, g.cu_kv, b, g.max_nq, g.max_nkv);
  if (!s.ok || s.nkv == 0 || s.nq == 0) return;
  const int grp = g.Hq / g.Hkv;
  const int nrows = grp * ((s.nq + kBQ - 1) / kBQ);
  const int r0 = rt * 128;
  if (r0 >= nrows) return;
  const int ntile_kv = (s.nkv + kBKV - 1) / kBKV;
  const int qb_last = min(nrows - 1, r0 + 127) / grp;
  const int t_end_all = g.causal ? kv_tiles_for(qb_last, s.nq, s.nkv, 1) : ntile_kv;
  const int t0 = blockIdx.x * a.ds_chunk, t1 = min(t_end_all, t0 + a.ds_chunk);
  if (t0 >= t1) return;
  const int nt = t1 - t0;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float *mu_s = reinterpret_cast<float *>(smem + P::kMu);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::kBar);
  uint64_t *a_full = bars, *b_full = bars + 1, *b_empty = bars + 3, *acc_full = bars + 5,
           *acc_empty = bars + 7, *drain = bars + 9;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + P::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P::kMisc + 4);
  for (int d = tid; d < DP; d += kDsThreads)
    mu_s[d] = a.w.kmean[((size_t)b * g.Hkv + hk) * DP + d];
  if (tid == 0) {
    mbar_init(a_full, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b_full[i], kDsLoadWarps);
      mbar_init(&b_empty[i], 1);
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kDsMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const AbortCtx ab{abort_flag, a.w.status};
  constexpr uint32_t kColA = 0, kColAcc = 256;

  if (warp < kDsLoadWarps) {
    // ------------------------------------------------------------ qmean pieces, then K~ tiles
    if (warp < 4) {
      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      const int r = r0 + warp * 32 + lane;
      const bool row_ok = r < nrows;
      const float4 *src = reinterpret_cast<const float4 *>(
          a.w.qmean + ((size_t)(hk * grp + (row_ok ? r % grp : 0)) * a.L.nqblk + s.qpad0 / kBQ +
                       (row_ok ? r / grp : 0)) * DP);
#pragma unroll 1
      for (int c = 0; c < DP / 16; ++c) {  // 16 channels = 8 columns per piece
        float qv[16];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 f = row_ok ? __ldg(src + 4 * c + e) : make_float4(0.f, 0.f, 0.f, 0.f);
          qv[4 * e] = f.x;
          qv[4 * e + 1] = f.y;
          qv[4 * e + 2] = f.z;
          qv[4 * e + 3] = f.w;
        }
        uint32_t w0[8], w1[8], w2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          uint32_t a0, a1, a2, b0, b1, b2;
          split3(qv[2 * e], a0, a1, a2);
          split3(qv[2 * e + 1], b0, b1, b2);
          w0[e] = a0 | (b0 << 16);
          w1[e] = a1 | (b1 << 16);
          w2[e] = a2 | (b2 << 16);
        }
        tmem_st8(tbase + lane_base + kColA + 8 * c, w0);
        tmem_st8(tbase + lane_base + kColA + DP / 2 + 8 * c, w1);
        tmem_st8(tbase + lane_base + kColA + DP + 8 * c, w2);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(a_full);
    }
    // warp w: keys 32 (w % 4) .. + 31, channel half w / 4. Lane l: chunk c8 = half * CPR +
    // l % CPR of the keys 32 (w % 4) + RPI i + l / CPR, i < CPR (CPR 8-channel chunks per half
    // row, RPI rows per instruction)
    constexpr int CPR = DP / 16, RPI = 32 / CPR;
    const int c8 = (warp >> 2) * CPR + lane % CPR;
    const int key0 = (warp & 3) * 32 + lane / CPR;
    const bool ch_live = c8 * 8 < g.D0;
    float mu8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mu8[e] = mu_s[c8 * 8 + e];
    const int off_blk = (c8 >> 3) * 16384;
    const size_t krow_stride = (size_t)g.Hkv * g.D0;
    bool ok = true;
#pragma unroll 1
    for (int t = 0; t < nt && ok; ++t) {
      const int buf = t & 1;
      const int kbase = (t0 + t) * kBKV;
      uint4 raw[CPR];
#pragma unroll
      for (int i = 0; i < CPR; ++i) {
        const int key = kbase + key0 + RPI * i;
        raw[i] = (key < s.nkv && ch_live)
                     ? __ldg(reinterpret_cast<const uint4 *>(
                           a.k + (size_t)(s.kv0 + key) * krow_stride + (size_t)hk * g.D0 + c8 * 8))
                     : make_uint4(0u, 0u, 0u, 0u);
      }
      if (t >= 2 && !(ok = ds_wait(&b_empty[buf], ((t - 2) >> 1) & 1, ab, 1))) break;
      uint8_t *bufp = smem + P::kB + buf * P::kBuf + off_blk;
#pragma unroll
      for (int i = 0; i < CPR; ++i) {
        const int n = key0 + RPI * i;  // key within the tile
        const bool live = kbase + n < s.nkv && ch_live;
        float x[8];
        unpack8<BF16>(raw[i], x);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = live ? __fsub_rn(x[e], mu8[e]) : 0.f;
        uint32_t w0[4], w1[4], w2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t a0, a1, a2, b0, b1, b2;
          split3(x[2 * e], a0, a1, a2);
          split3(x[2 * e + 1], b0, b1, b2);
          w0[e] = a0 | (b0 << 16);
          w1[e] = a1 | (b1 << 16);
          w2[e] = a2 | (b2 << 16);
        }
        // 64 channels per 128-byte row; 16-byte chunk j of row n at position j ^ (n & 7)
        uint8_t *dst = bufp + n * 128 + (((c8 & 7) ^ (n & 7)) << 4);
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
        *reinterpret_cast<uint4 *>(dst + P::kPiece) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
        *reinterpret_cast<uint4 *>(dst + 2 * P::kPiece) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
      }
      fence_async_smem();  // the generic-proxy stores become visible to the MMA
      __syncwarp();
      if (lane == 0) mbar_arrive(&b_full[buf]);
    }
  } else if (warp < kDsMmaWarp) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    // the warp's largest visited tile: its last valid row has the largest Q block
    const int r_last = min(nrows - 1, r0 + q * 32 + 31);
    const int vis_warp = (r0 + q * 32 < nrows)
                             ? (g.causal ? kv_tiles_for(r_last / grp, s.nq, s.nkv, 1) : ntile_kv)
                             : 0;
    // the staging block of this warp: 32 rows x 32 floats, 16-byte chunk j of row r at j ^ (r & 7)
    float *stage = reinterpret_cast<float *>(smem + P::kStage) + q * 32 * 32;
    // in the store phase lane l writes chunk l % 8 of rows 4 i + l / 8: their dsc rows
    float *orow[8];
    int ovis[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = r0 + q * 32 + 4 * i + lane / 8;
      const bool ok_r = rr < nrows;
      const int qb_r = ok_r ? rr / grp : 0, hq_r = hk * grp + (ok_r ? rr % grp : 0);
      orow[i] = a.w.dsc + ((size_t)hq_r * a.L.nqblk + s.qpad0 / kBQ + qb_r) * a.L.nkv_pad;
      ovis[i] = ok_r ? (g.causal ? kv_tiles_for(qb_r, s.nq, s.nkv, 1) : ntile_kv) : 0;
    }
    bool ok = true;
#pragma unroll 1
    for (int t = 0; t < nt && ok; ++t) {
      const int buf = t & 1;
      if (!(ok = ds_wait(&acc_full[buf], (t >> 1) & 1, ab, 2))) break;
      tc_fence_after();
      const int kt = t0 + t;
      if (kt < vis_warp) {
        const uint32_t tA = tbase + lane_base + kColAcc + buf * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32_wait(tA + 32 * c, v);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4 *>(stage + lane * 32 + ((j ^ (lane & 7)) << 2)) =
                make_float4(__fmul_rn(__uint_as_float(v[4 * j]), g.c32),
                            __fmul_rn(__uint_as_float(v[4 * j + 1]), g.c32),
                            __fmul_rn(__uint_as_float(v[4 * j + 2]), g.c32),
                            __fmul_rn(__uint_as_float(v[4 * j + 3]), g.c32));
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + lane / 8, j = lane & 7;
            const float4 f = *reinterpret_cast<const float4 *>(stage + r * 32 + ((j ^ (r & 7)) << 2));
            if (kt < ovis[i])
              *reinterpret_cast<float4 *>(orow[i] + kt * kBKV + 32 * c + 4 * j) = f;
          }
          __syncwarp();  // the block is read before the next chunk overwrites it
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  } else if (lane == 0) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
    // piece products, smallest first: (qmean piece, K~ piece), 0 = the leading piece
    constexpr int kPa[6] = {2, 1, 0, 1, 0, 0}, kPb[6] = {0, 1, 2, 0, 1, 0};
    bool ok = mbar_wait(a_full, 0, ab, 3);
#pragma unroll 1
    for (int t = 0; t < nt && ok; ++t) {
      const int buf = t & 1;
      ok = mbar_wait(&b_full[buf], (t >> 1) & 1, ab, 4) &&
           (t < 2 || mbar_wait(&acc_empty[buf], ((t - 2) >> 1) & 1, ab, 5));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tbase + kColAcc + buf * 128;
      const uint32_t bbase = smem_u32(smem + P::kB + buf * P::kBuf);
#pragma unroll
      for (int pp = 0; pp < 6; ++pp) {
        const uint64_t bdesc = sdesc_kmajor(bbase + kPb[pp] * P::kPiece, 128);
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk)  // 16 channels = 32 bytes per MMA
          mma_f16_ts(d, tbase + kColA + kPa[pp] * (DP / 2) + kk * 8,
                     bdesc + (uint64_t)((kk & 3) * 2 + (kk >> 2) * (16384 >> 4)), idesc,
                     (pp > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(&b_empty[buf]);
      mma_commit(&acc_full[buf]);
    }
    mma_commit(drain);  // every MMA issued above completes before tensor memory is freed
    const uint64_t t_drain = global_timer_ns();
    while (!mbar_try_wait(drain, 0))
      if (global_timer_ns() - t_drain > SAGE2_WAIT_NS) break;
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kDsMmaWarp) tmem_dealloc(tbase, 512);
}

// The order in which the two-tile attention kernel takes the sequences of a varlen call: by
// decreasing K/V length (the length of every CTA's loop), ties by index, so that the longest
// CTAs start first and the short ones fill the tail. One CTA; a rank count per sequence, for at
// most kSeqOrderMaxSort sequences (beyond that the batch keeps its order).
__global__ void __launch_bounds__(256) seq_order(const int *cu_kv, int B, int *order) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int rank = b;
    if (B <= kSeqOrderMaxSort) {
      const int n = cu_kv[b + 1] - cu_kv[b];
      rank = 0;
      for (int c = 0; c < B; ++c) {
        const int m = cu_kv[c + 1] - cu_kv[c];
        rank += (m > n || (m == n && c < b)) ? 1 : 0;
      }
    }
    order[rank] = b;  // ranks are a permutation of 0 .. B - 1 (a strict total order)
  }
}

// Two side streams per device on which the prepass runs the kernels that do not wait for the
// launches before them on the caller's stream (the Q codes from the start; the V and K codes
// next to DeltaS), forked from and joined back into the caller's stream with events. One mutex per device makes each call's record /
// wait sequence whole, so concurrent callers cannot wait on one another's events.
struct SideStreams {
  std::mutex mu;
  bool ready = false;
  cudaStream_t s[2] = {nullptr, nullptr};
  cudaEvent_t fork = nullptr, kv_done = nullptr, q_done = nullptr, v_done = nullptr;
};
constexpr int kMaxDevices = 64;
SideStreams g_side[kMaxDevices];

cudaError_t init_side(SideStreams &p) {  // with p.mu held
  if (p.ready) return cudaSuccess;
  const unsigned ef = cudaEventDisableTiming;
  cudaError_t e;
  for (int i = 0; i < 2; ++i)
    if ((e = cudaStreamCreateWithFlags(&p.s[i], cudaStreamNonBlocking)) != cudaSuccess) return e;
  if ((e = cudaEventCreateWithFlags(&p.fork, ef)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&p.kv_done, ef)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&p.q_done, ef)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&p.v_done, ef)) != cudaSuccess)
    return e;
  p.ready = true;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_prepass(const void *q, const void *k, const void *v, int in_dtype,
                           int quant_flags, const Geometry &g, const Layout &L, void *ws,
                           cudaStream_t st, cudaEvent_t q_ready) {
  PrepassArgs a;
  a.q = static_cast<const uint16_t *>(q);
  a.k = static_cast<const uint16_t *>(k);
  a.v = static_cast<const uint16_t *>(v);
  const bool bf16 = in_dtype == SAGE2_BF16;
  const bool int8 = (quant_flags & SAGE2_QUANT_SAGE1) != 0;
  a.flags = int8 ? (SAGE2_QUANT_NO_SMOOTH_Q | SAGE2_QUANT_PER_BLOCK) : quant_flags;
  a.g = g;
  a.L = L;
  a.w = ws_ptrs(ws, L);
  cudaError_t e = cudaMemsetAsync(a.w.status, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  // the code format, checked by the attention kernel
  e = cudaMemsetAsync(a.w.status + 1, int8 ? kFormatInt8Byte : kFormatInt4Byte, sizeof(int), st);
  if (e != cudaSuccess) return e;
  if (g.cu_kv) seq_order<<<1, 256, 0, st>>>(g.cu_kv, g.B, a.w.status + kSeqOrderWord);

  const int nvec = g.Hkv * g.D0 / 8;
  // every grid dimension at least 1 (a zero-length maximum is legal; the kernels bound-check)
  const int kv_tiles = max(1, (g.max_nkv + kBKV - 1) / kBKV);
  const int q_tiles = max(1, (g.max_nq + kBQ - 1) / kBQ);
  const int stat_vpb = min(nvec, kStatThreads);
  const dim3 stat_grid(L.nchunk, g.B, (nvec + stat_vpb - 1) / stat_vpb);
  const dim3 kv_grid(kv_tiles, g.Hkv, g.B);
  const dim3 q_grid(q_tiles, g.Hq, g.B);
  // DeltaS: 128-row tiles of (Q block, q head) pairs, a.ds_chunk key tiles per CTA
  const int max_rows = (g.Hq / g.Hkv) * q_tiles;
  const int row_tiles = (max_rows + 127) / 128;
  int nsm = 0, dev = -1;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) nsm = 0;
  a.ds_chunk = kDsChunkMax;
  if (nsm > 0) {
    // CTAs with work per chunk size: a dense call's row tile rt visits the key tiles of its last
    // Q block (all of them without a causal mask); a varlen call's lengths live on the device,
    // so every chunk of the longest sequence counts
    long long best = -1;
    for (int ch = kDsChunkMax; ch >= kDsChunkMin; ch /= 2) {
      long long active = 0;
      for (int rt = 0; rt < row_tiles; ++rt) {
        int t_end = kv_tiles;
        if (!g.cu_kv && g.causal) {
          const int qb_last = std::min(max_rows - 1, rt * 128 + 127) / (g.Hq / g.Hkv);
          t_end = kv_tiles_for(qb_last, g.max_nq, g.max_nkv, 1);
        }
        active += (t_end + ch - 1) / ch;
      }
      active *= (long long)g.B * g.Hkv;
      const long long cost = (active + nsm - 1) / nsm * (ch + kDsCtaSetupTiles);
      if (best < 0 || cost < best) {
        best = cost;
        a.ds_chunk = ch;
      }
    }
  }
  const dim3 ds_grid((kv_tiles + a.ds_chunk - 1) / a.ds_chunk, row_tiles, g.B * g.Hkv);
  // kernels instantiated per padded head dim and input type
  // kernels instantiated per padded head dim, input type and code grid. The INT8 path (the
  // SageAttention (v1) switch) has per-block scales, no Q smoothing and so no DeltaS: the
  // attention kernel for it reads none.
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  SideStreams &side = g_side[dev];
  std::lock_guard<std::mutex> lock(side.mu);
  if ((e = init_side(side)) != cudaSuccess) return e;
  cudaError_t err = cudaSuccess;
  // Q codes on side stream 0 from the start (after the status words; once q_ready has fired,
  // when given); the statistics on the caller's stream, then the V and K codes on side stream 1
  // while DeltaS (which needs the K means and the Q block means, not the K codes) runs on the
  // caller's stream; that stream finally waits for side stream 1.
  auto run = [&](auto dp_tag, auto bf_tag, auto i8_tag) {
    constexpr int DP = decltype(dp_tag)::value;
    constexpr bool BF = decltype(bf_tag)::value;
    constexpr bool I8 = decltype(i8_tag)::value;
    if ((err = cudaEventRecord(side.fork, st)) != cudaSuccess ||
        (err = cudaStreamWaitEvent(side.s[0], side.fork, 0)) != cudaSuccess ||
        (q_ready && (err = cudaStreamWaitEvent(side.s[0], q_ready, 0)) != cudaSuccess))
      return;
    q_quant<DP, BF, I8><<<q_grid, 256, 0, side.s[0]>>>(a);
    if ((err = cudaEventRecord(side.q_done, side.s[0])) != cudaSuccess) return;
    kv_stats_partial<BF><<<stat_grid, kStatThreads, 0, st>>>(a);
    if (g.B * g.Hkv * (g.Dp / 32) >= 64)
      kv_stats_final<32><<<dim3(g.B * g.Hkv, g.Dp / 32), kFinalThreads, 0, st>>>(a);
    else
      kv_stats_final<8><<<dim3(g.B * g.Hkv, g.Dp / 8), kFinalThreads, 0, st>>>(a);
    if ((err = cudaEventRecord(side.kv_done, st)) != cudaSuccess ||
        (err = cudaStreamWaitEvent(side.s[1], side.kv_done, 0)) != cudaSuccess)
      return;
    v_quant<DP, BF><<<kv_grid, 256, 0, side.s[1]>>>(a);
    k_quant<DP, BF, I8><<<kv_grid, 256, 0, side.s[1]>>>(a);
    if ((err = cudaEventRecord(side.v_done, side.s[1])) != cudaSuccess ||
        (err = cudaStreamWaitEvent(st, side.q_done, 0)) != cudaSuccess)
      return;
    if (I8) {
      err = cudaStreamWaitEvent(st, side.v_done, 0);
      return;
    }
    constexpr int kSmem = DsPlan<DP>::kBytes;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
      attr_err = cudaFuncSetAttribute(delta_s_tc<DP, BF>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    });
    if ((err = attr_err) != cudaSuccess) {
      cudaStreamWaitEvent(st, side.v_done, 0);  // still join the side stream
      return;
    }
    delta_s_tc<DP, BF><<<ds_grid, kDsThreads, kSmem, st>>>(a);
    err = cudaStreamWaitEvent(st, side.v_done, 0);
  };
  auto run_dp = [&](auto i8_tag) {
    using T128 = std::integral_constant<int, 128>;
    using T64 = std::integral_constant<int, 64>;
    if (g.Dp == 128) {
      if (bf16) run(T128(), std::true_type(), i8_tag);
      else run(T128(), std::false_type(), i8_tag);
    } else {
      if (bf16) run(T64(), std::true_type(), i8_tag);
      else run(T64(), std::false_type(), i8_tag);
    }
  };
  if (int8) run_dp(std::true_type());
  else run_dp(std::false_type());
  const cudaError_t last = cudaGetLastError();
  return err != cudaSuccess ? err : last;
}

}  // namespace sage2
