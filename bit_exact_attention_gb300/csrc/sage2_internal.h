// sage2_internal.h -- types shared by the library's translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sage2_attn.h"

namespace sage2 {

constexpr int kBQ = 128;        // Q tile rows = Q smoothing block
constexpr int kBKV = 128;       // KV tile keys = online-softmax step = two-level partial
constexpr int kGK = 32;         // K tokens per INT4 scale group
constexpr int kStatChunk = 32;  // tokens per partial in the K/V statistics pass

// Problem geometry. Dense calls have cu_q == cu_kv == nullptr and every sequence of length
// max_nq / max_nkv; varlen calls pass device prefix sums.
struct Geometry {
  int B, Hq, Hkv, max_nq, max_nkv, total_q, total_kv;
  int D0, Dp, causal;
  const int *cu_q;
  const int *cu_kv;
  float sm_scale;  // resolved (> 0)
  float c32;       // fl32(log2(e) * sm_scale)
};

struct Layout {
  size_t total;
  size_t qcode, kcode, vcodeT, qscale, kscale, qmean, kmean, vscale, vinv, dsc, kpart, vpart,
      status;
  int Tq, Tkv, nqblk, nkv_pad, nchunk;
  int code_bytes;  // bytes per Q / K code: 1 (INT4 grid as e4m3), 2 (INT8 grid as fp16)
};

// Computes the workspace layout; returns false on sizes that overflow or are invalid.
// code_bytes: 1 for the method's INT4-grid codes, 2 for the INT8-grid codes (fp16 values).
bool make_layout(int B, int Hq, int Hkv, int max_nq, int max_nkv, int Dp, int total_q,
                 int total_kv, int code_bytes, Layout *L);

// The workspace status area: word 0 the device status, word 1 the code format, words
// kSeqOrderWord .. + B - 1 the order in which the two-tile attention kernel takes the sequences
// of a varlen call (longest K/V first; written by the prepass).
constexpr int kSeqOrderWord = 64;
// The prepass sorts at most this many sequences (a rank count per sequence in one CTA); larger
// batches keep their own order.
constexpr int kSeqOrderMaxSort = 256;

// Code format a prepass leaves in word 1 of the workspace status area (every byte of the word
// the same), checked by the attention kernel before it reads anything else.
constexpr unsigned char kFormatInt4Byte = 0x34, kFormatInt8Byte = 0x38;
constexpr int kFormatInt4 = 0x34343434, kFormatInt8 = 0x38383838;

// Pointers into a workspace.
struct WsPtrs {
  uint8_t *qcode, *kcode, *vcodeT;
  float *qscale, *kscale, *qmean, *kmean, *vscale, *vinv, *dsc;
  double *kpart;
  float *vpart;
  int *status;
};
WsPtrs ws_ptrs(void *ws, const Layout &L);

// Per-sequence geometry on the device. Sequence b owns tokens [q0, q0 + nq) of Q and
// [kv0, kv0 + nkv) of K/V; its padded rows start at 128 * (q0 / 128 + b) (and likewise for
// K/V), which keeps every sequence on a tile boundary with room for its ragged tail.
struct Seq {
  int q0, nq, kv0, nkv, qpad0, kvpad0;
  bool ok;
};
__host__ __device__ inline Seq seq_info(const int *cu_q, const int *cu_kv, int b, int max_nq,
                                        int max_nkv) {
  Seq s;
  if (cu_q) {
    s.q0 = cu_q[b];
    s.nq = cu_q[b + 1] - s.q0;
  } else {
    s.q0 = b * max_nq;
    s.nq = max_nq;
  }
  if (cu_kv) {
    s.kv0 = cu_kv[b];
    s.nkv = cu_kv[b + 1] - s.kv0;
  } else {
    s.kv0 = b * max_nkv;
    s.nkv = max_nkv;
  }
  s.ok = s.q0 >= 0 && s.kv0 >= 0 && s.nq >= 0 && s.nkv >= 0 && s.nq <= max_nq &&
         s.nkv <= max_nkv;
  s.qpad0 = kBQ * (s.q0 / kBQ + b);
  s.kvpad0 = kBKV * (s.kv0 / kBKV + b);
  return s;
}

// Number of KV tiles Q tile `qt` of a sequence visits (causal: up to the last key visible to
// its last valid row, bottom-right aligned).
__host__ __device__ inline int kv_tiles_for(int qt, int nq, int nkv, int causal) {
  const int nt = (nkv + kBKV - 1) / kBKV;
  if (!causal) return nt;
  int i_last = qt * kBQ + kBQ - 1;
  if (i_last > nq - 1) i_last = nq - 1;
  const int j_max = i_last + (nkv - nq);
  if (j_max < 0) return 0;
  const int t = j_max / kBKV + 1;
  return t < nt ? t : nt;
}

// ---------------------------------------------------------------- checked entry points
// The prepass and attention calls behind the C ABI (argument checks, then the launches);
// cu_q / cu_kv nullptr for dense problems. Return sage2_status codes. q_ready: when not null,
// the prepass's Q kernels wait for this event (its K/V statistics and codes do not), so that a
// caller copying Q in after K and V can overlap the two.
int prepass_impl(const void *q, const void *k, const void *v, int in_dtype, const int *cu_q,
                 const int *cu_kv, int B, int Hq, int Hkv, int max_nq, int max_nkv, int total_q,
                 int total_kv, int D, int causal, float sm_scale, int quant_flags, void *ws,
                 size_t ws_bytes, void *stream, cudaEvent_t q_ready = nullptr);
// hq0, hq_n: attention for the q heads [hq0, hq0 + hq_n) only (hq_n = 0: through the last);
// the other heads' output rows are left as they are.
int attention_impl(void *out, int out_dtype, int quant_flags, const int *cu_q, const int *cu_kv,
                   int B, int Hq, int Hkv, int max_nq, int max_nkv, int total_q, int total_kv,
                   int D, int causal, float sm_scale, const void *ws, size_t ws_bytes,
                   void *stream, int hq0 = 0, int hq_n = 0);

// ---------------------------------------------------------------- launchers
cudaError_t launch_prepass(const void *q, const void *k, const void *v, int in_dtype,
                           int quant_flags, const Geometry &g, const Layout &L, void *ws,
                           cudaStream_t st, cudaEvent_t q_ready = nullptr);

struct AttnDebug {
  int b, h, qt, kt;        // the single work unit to run (debug launches only)
  float *s_out;            // [128][128]
  uint8_t *p_out;          // [128][128]
  float *r_out;            // [128][Dp]
  int skip_loads;          // producer issues nothing: every wait must time out
};
// int8_qk: the INT8-grid variant (Q K^T on fp16 codes); the workspace must come from a prepass
// with SAGE2_QUANT_SAGE1, and the other way round (checked on the device). hq0, hq_n: only the
// q heads [hq0, hq0 + hq_n) (hq_n = 0: through the last head).
cudaError_t launch_attention(void *out, int out_dtype, const Geometry &g, const Layout &L,
                             const void *ws, cudaStream_t st, const AttnDebug *dbg,
                             bool int8_qk = false, int hq0 = 0, int hq_n = 0);

}  // namespace sage2
