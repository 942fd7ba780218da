// sage2_api.cu -- the C ABI: argument checks, workspace layout, launches.
#include <math.h>
#include <string.h>

#include <mutex>

#include "sage2_device.cuh"
#include "sage2_internal.h"

namespace sage2 {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool make_layout(int B, int Hq, int Hkv, int max_nq, int max_nkv, int Dp, int total_q,
                 int total_kv, int code_bytes, Layout *L) {
  if (code_bytes != 1 && code_bytes != 2) return false;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || max_nq < 0 || max_nkv < 0 || total_q < 0 || total_kv < 0)
    return false;
  // padded rows: every sequence starts at 128 * (cu[b] / 128 + b) and occupies a whole
  // number of 128-row tiles, so total + 128 * B rows (rounded up) hold them all
  const long long tq = ((long long)total_q + 128LL * B + 127) / 128 * 128;
  const long long tkv = ((long long)total_kv + 128LL * B + 127) / 128 * 128;
  const long long nkv_pad = ((long long)max_nkv + 127) / 128 * 128;
  if ((long long)Hq * tq >= (1LL << 31) || (long long)Hkv * tkv >= (1LL << 31) ||
      (long long)Hkv * Dp >= (1LL << 31))
    return false;
  L->Tq = (int)tq;
  L->Tkv = (int)tkv;
  L->nqblk = (int)(tq / 128);
  L->nkv_pad = (int)(nkv_pad > 0 ? nkv_pad : 128);
  L->nchunk = (max_nkv + kStatChunk - 1) / kStatChunk;
  if (L->nchunk < 1) L->nchunk = 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 1024);
    return o;
  };
  L->code_bytes = code_bytes;
  L->status = take(4 * (kSeqOrderWord + (size_t)B));
  L->qcode = take((size_t)Hq * tq * Dp * code_bytes);
  L->kcode = take((size_t)Hkv * tkv * Dp * code_bytes);
  L->vcodeT = take((size_t)Hkv * Dp * tkv);
  L->qscale = take((size_t)Hq * tq * 4);
  L->kscale = take((size_t)Hkv * (tkv / kGK) * 4);
  L->qmean = take((size_t)Hq * (tq / 128) * Dp * 4);
  L->kmean = take((size_t)B * Hkv * Dp * 4);
  L->vscale = take((size_t)B * Hkv * Dp * 4);
  L->vinv = take((size_t)B * Hkv * Dp * 4);
  L->dsc = take((size_t)Hq * (tq / 128) * L->nkv_pad * 4);
  L->kpart = take((size_t)B * L->nchunk * Hkv * 128 * 8);
  L->vpart = take((size_t)B * L->nchunk * Hkv * 128 * 4);
  L->total = off + 1024;  // slack: the base is aligned up to 1024 bytes inside the call
  return true;
}

static uint8_t *ws_base(void *ws) {
  const uintptr_t p = reinterpret_cast<uintptr_t>(ws);
  return reinterpret_cast<uint8_t *>((p + 1023) & ~uintptr_t(1023));
}

WsPtrs ws_ptrs(void *ws, const Layout &L) {
  uint8_t *base = ws_base(ws);
  WsPtrs w;
  w.qcode = base + L.qcode;
  w.kcode = base + L.kcode;
  w.vcodeT = base + L.vcodeT;
  w.qscale = reinterpret_cast<float *>(base + L.qscale);
  w.kscale = reinterpret_cast<float *>(base + L.kscale);
  w.qmean = reinterpret_cast<float *>(base + L.qmean);
  w.kmean = reinterpret_cast<float *>(base + L.kmean);
  w.vscale = reinterpret_cast<float *>(base + L.vscale);
  w.vinv = reinterpret_cast<float *>(base + L.vinv);
  w.dsc = reinterpret_cast<float *>(base + L.dsc);
  w.kpart = reinterpret_cast<double *>(base + L.kpart);
  w.vpart = reinterpret_cast<float *>(base + L.vpart);
  w.status = reinterpret_cast<int *>(base + L.status);
  return w;
}

static int padded_dim(int D) { return D <= 64 ? 64 : 128; }

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// sm_103 check, cached per device.
static int check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SAGE2_ECUDA;
  static std::mutex mu;
  static int cached[64] = {0};  // 0 unknown, 1 ok, 2 unsupported
  if (dev < 0 || dev >= 64) return SAGE2_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SAGE2_ECUDA;
    cached[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return cached[dev] == 1 ? SAGE2_OK : SAGE2_EUNSUPPORTED;
}

// Shape checks shared by every entry point (no CUDA calls).
static int check_shapes(int B, int Hq, int Hkv, int max_nq, int max_nkv, int D, int total_q,
                        int total_kv, int causal) {
  if (D > 128 || D < 8 || (D % 8) != 0) return D > 0 ? SAGE2_EUNSUPPORTED : SAGE2_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || (Hq % Hkv) != 0) return SAGE2_EINVAL;
  if (max_nq < 0 || max_nkv < 0 || total_q < 0 || total_kv < 0) return SAGE2_EINVAL;
  if ((long long)max_nq * B < total_q && max_nq >= 0) return SAGE2_EINVAL;
  if ((long long)max_nkv * B < total_kv) return SAGE2_EINVAL;
  if (causal != 0 && causal != 1) return SAGE2_EINVAL;
  return SAGE2_OK;
}

static bool make_geometry(int B, int Hq, int Hkv, int max_nq, int max_nkv, int D, int total_q,
                          int total_kv, int causal, float sm_scale, const int *cu_q,
                          const int *cu_kv, int code_bytes, Geometry *g, Layout *L) {
  g->B = B;
  g->Hq = Hq;
  g->Hkv = Hkv;
  g->max_nq = max_nq;
  g->max_nkv = max_nkv;
  g->total_q = total_q;
  g->total_kv = total_kv;
  g->D0 = D;
  g->Dp = padded_dim(D);
  g->causal = causal;
  g->cu_q = cu_q;
  g->cu_kv = cu_kv;
  g->sm_scale = sm_scale > 0.f ? sm_scale : (float)(1.0 / sqrt((double)D));
  g->c32 = (float)(1.4426950408889634074 * (double)g->sm_scale);
  return make_layout(B, Hq, Hkv, max_nq, max_nkv, g->Dp, total_q, total_kv, code_bytes, L);
}

// Quantization switches: the ablation bits in any combination, or SAGE2_QUANT_SAGE1 alone.
static bool valid_quant_flags(int f) {
  const int ablations = SAGE2_QUANT_NO_SMOOTH_Q | SAGE2_QUANT_NO_SMOOTH_K | SAGE2_QUANT_PER_BLOCK;
  if (f & SAGE2_QUANT_SAGE1) return f == SAGE2_QUANT_SAGE1;
  return (f & ~ablations) == 0;
}
static int code_bytes_of(int quant_flags) { return (quant_flags & SAGE2_QUANT_SAGE1) ? 2 : 1; }

static int check_ws(const void *ws, size_t bytes, const Layout &L) {
  if (!ws || !aligned16(ws)) return SAGE2_EWORKSPACE;
  if (bytes < L.total) return SAGE2_EWORKSPACE;
  return SAGE2_OK;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? SAGE2_OK : SAGE2_ECUDA; }

// The one path behind the dense and varlen prepass entry points (also used by the
// host-streaming forward).
int prepass_impl(const void *q, const void *k, const void *v, int in_dtype, const int *cu_q,
                 const int *cu_kv, int B, int Hq, int Hkv, int max_nq, int max_nkv, int total_q,
                 int total_kv, int D, int causal, float sm_scale, int quant_flags, void *ws,
                 size_t ws_bytes, void *stream, cudaEvent_t q_ready) {
  int rc = check_shapes(B, Hq, Hkv, max_nq, max_nkv, D, total_q, total_kv, causal);
  if (rc) return rc;
  if (in_dtype != SAGE2_FP16 && in_dtype != SAGE2_BF16) return SAGE2_EINVAL;
  if (!valid_quant_flags(quant_flags)) return SAGE2_EINVAL;
  if ((total_q > 0 && (!q || !aligned16(q))) || (total_kv > 0 && (!k || !v || !aligned16(k) ||
                                                                  !aligned16(v))))
    return SAGE2_EINVAL;
  Geometry g;
  Layout L;
  if (!make_geometry(B, Hq, Hkv, max_nq, max_nkv, D, total_q, total_kv, causal, sm_scale, cu_q,
                     cu_kv, code_bytes_of(quant_flags), &g, &L))
    return SAGE2_EINVAL;
  if ((rc = check_ws(ws, ws_bytes, L))) return rc;
  if ((rc = check_device())) return rc;
  return cuda_status(
      launch_prepass(q, k, v, in_dtype, quant_flags, g, L, ws, (cudaStream_t)stream, q_ready));
}

int attention_impl(void *out, int out_dtype, int quant_flags, const int *cu_q, const int *cu_kv,
                   int B, int Hq, int Hkv, int max_nq, int max_nkv, int total_q, int total_kv,
                   int D, int causal, float sm_scale, const void *ws, size_t ws_bytes,
                   void *stream, int hq0, int hq_n) {
  int rc = check_shapes(B, Hq, Hkv, max_nq, max_nkv, D, total_q, total_kv, causal);
  if (rc) return rc;
  if (!valid_quant_flags(quant_flags)) return SAGE2_EINVAL;
  if (out_dtype != SAGE2_FP16 && out_dtype != SAGE2_BF16 && out_dtype != SAGE2_FP32)
    return SAGE2_EINVAL;
  if (hq0 < 0 || hq_n < 0 || hq0 + hq_n > Hq || (hq_n == 0 && hq0 >= Hq)) return SAGE2_EINVAL;
  if (total_q > 0 && (!out || !aligned16(out))) return SAGE2_EINVAL;
  Geometry g;
  Layout L;
  if (!make_geometry(B, Hq, Hkv, max_nq, max_nkv, D, total_q, total_kv, causal, sm_scale, cu_q,
                     cu_kv, code_bytes_of(quant_flags), &g, &L))
    return SAGE2_EINVAL;
  if ((rc = check_ws(ws, ws_bytes, L))) return rc;
  if ((rc = check_device())) return rc;
  if (total_q == 0 || max_nq == 0) return SAGE2_OK;
  return cuda_status(launch_attention(out, out_dtype, g, L, ws, (cudaStream_t)stream, nullptr,
                                      (quant_flags & SAGE2_QUANT_SAGE1) != 0, hq0, hq_n));
}

}  // namespace sage2

using namespace sage2;

extern "C" {

const char *sage2_status_str(int s) {
  switch (s) {
    case SAGE2_OK: return "ok";
    case SAGE2_EINVAL: return "invalid argument";
    case SAGE2_EUNSUPPORTED: return "unsupported (head dim or device)";
    case SAGE2_EWORKSPACE: return "workspace too small or misaligned";
    case SAGE2_ECUDA: return "CUDA error";
    case SAGE2_EDEVICE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int sage2_version(void) { return 100; }

size_t sage2_workspace_size_ex(int B, int Hq, int Hkv, int max_Nq, int max_Nkv, int D,
                               int total_q, int total_kv, int quant_flags) {
  if (check_shapes(B, Hq, Hkv, max_Nq, max_Nkv, D, total_q, total_kv, 0)) return 0;
  if (!valid_quant_flags(quant_flags)) return 0;
  Layout L;
  if (!make_layout(B, Hq, Hkv, max_Nq, max_Nkv, padded_dim(D), total_q, total_kv,
                   code_bytes_of(quant_flags), &L))
    return 0;
  return L.total;
}

size_t sage2_workspace_size(int B, int Hq, int Hkv, int max_Nq, int max_Nkv, int D, int total_q,
                            int total_kv) {
  return sage2_workspace_size_ex(B, Hq, Hkv, max_Nq, max_Nkv, D, total_q, total_kv, 0);
}

int sage2_workspace_layout(int B, int Hq, int Hkv, int max_Nq, int max_Nkv, int D, int total_q,
                           int total_kv, sage2_ws_layout *out) {
  return sage2_workspace_layout_ex(B, Hq, Hkv, max_Nq, max_Nkv, D, total_q, total_kv, 0, out);
}

int sage2_workspace_layout_ex(int B, int Hq, int Hkv, int max_Nq, int max_Nkv, int D,
                              int total_q, int total_kv, int quant_flags, sage2_ws_layout *out) {
  int rc = check_shapes(B, Hq, Hkv, max_Nq, max_Nkv, D, total_q, total_kv, 0);
  if (rc) return rc;
  if (!out || !valid_quant_flags(quant_flags)) return SAGE2_EINVAL;
  Layout L;
  if (!make_layout(B, Hq, Hkv, max_Nq, max_Nkv, padded_dim(D), total_q, total_kv,
                   code_bytes_of(quant_flags), &L))
    return SAGE2_EINVAL;
  out->total_bytes = L.total;
  out->qcode = L.qcode;
  out->kcode = L.kcode;
  out->vcodeT = L.vcodeT;
  out->qscale = L.qscale;
  out->kscale = L.kscale;
  out->qmean = L.qmean;
  out->kmean = L.kmean;
  out->vscale = L.vscale;
  out->vinv = L.vinv;
  out->dsc = L.dsc;
  out->kpart = L.kpart;
  out->vpart = L.vpart;
  out->status = L.status;
  out->Dp = padded_dim(D);
  out->Tq = L.Tq;
  out->Tkv = L.Tkv;
  out->nkv_pad = L.nkv_pad;
  out->nchunk = L.nchunk;
  out->code_bytes = L.code_bytes;
  return SAGE2_OK;
}

int sage2_prepass(const void *q, const void *k, const void *v, int in_dtype, int B, int Hq,
                  int Hkv, int Nq, int Nkv, int D, int causal, float sm_scale, void *workspace,
                  size_t workspace_bytes, void *stream) {
  if ((long long)B * Nq >= (1LL << 31) || (long long)B * Nkv >= (1LL << 31)) return SAGE2_EINVAL;
  return prepass_impl(q, k, v, in_dtype, nullptr, nullptr, B, Hq, Hkv, Nq, Nkv, B * Nq, B * Nkv,
                      D, causal, sm_scale, 0, workspace, workspace_bytes, stream);
}

int sage2_prepass_varlen(const void *q, const void *k, const void *v, int in_dtype,
                         const int *cu_seqlens_q, const int *cu_seqlens_kv, int B, int Hq,
                         int Hkv, int max_Nq, int max_Nkv, int total_q, int total_kv, int D,
                         int causal, float sm_scale, void *workspace, size_t workspace_bytes,
                         void *stream) {
  if (!cu_seqlens_q || !cu_seqlens_kv) return SAGE2_EINVAL;
  return prepass_impl(q, k, v, in_dtype, cu_seqlens_q, cu_seqlens_kv, B, Hq, Hkv, max_Nq,
                      max_Nkv, total_q, total_kv, D, causal, sm_scale, 0, workspace,
                      workspace_bytes, stream);
}

int sage2_prepass_varlen_ex(const void *q, const void *k, const void *v, int in_dtype,
                            const int *cu_seqlens_q, const int *cu_seqlens_kv, int B, int Hq,
                            int Hkv, int max_Nq, int max_Nkv, int total_q, int total_kv, int D,
                            int causal, float sm_scale, int quant_flags, void *workspace,
                            size_t workspace_bytes, void *stream) {
  if (!cu_seqlens_q || !cu_seqlens_kv) return SAGE2_EINVAL;
  return prepass_impl(q, k, v, in_dtype, cu_seqlens_q, cu_seqlens_kv, B, Hq, Hkv, max_Nq,
                      max_Nkv, total_q, total_kv, D, causal, sm_scale, quant_flags, workspace,
                      workspace_bytes, stream);
}

int sage2_attention(void *out, int out_dtype, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                    int causal, float sm_scale, const void *workspace, size_t workspace_bytes,
                    void *stream) {
  if ((long long)B * Nq >= (1LL << 31) || (long long)B * Nkv >= (1LL << 31)) return SAGE2_EINVAL;
  return attention_impl(out, out_dtype, 0, nullptr, nullptr, B, Hq, Hkv, Nq, Nkv, B * Nq,
                        B * Nkv, D, causal, sm_scale, workspace, workspace_bytes, stream);
}

int sage2_attention_varlen(void *out, int out_dtype, const int *cu_seqlens_q,
                           const int *cu_seqlens_kv, int B, int Hq, int Hkv, int max_Nq,
                           int max_Nkv, int total_q, int total_kv, int D, int causal,
                           float sm_scale, const void *workspace, size_t workspace_bytes,
                           void *stream) {
  if (!cu_seqlens_q || !cu_seqlens_kv) return SAGE2_EINVAL;
  return attention_impl(out, out_dtype, 0, cu_seqlens_q, cu_seqlens_kv, B, Hq, Hkv, max_Nq,
                        max_Nkv, total_q, total_kv, D, causal, sm_scale, workspace,
                        workspace_bytes, stream);
}

int sage2_attention_varlen_ex(void *out, int out_dtype, const int *cu_seqlens_q,
                              const int *cu_seqlens_kv, int B, int Hq, int Hkv, int max_Nq,
                              int max_Nkv, int total_q, int total_kv, int D, int causal,
                              float sm_scale, int quant_flags, const void *workspace,
                              size_t workspace_bytes, void *stream) {
  if (!cu_seqlens_q || !cu_seqlens_kv) return SAGE2_EINVAL;
  return attention_impl(out, out_dtype, quant_flags, cu_seqlens_q, cu_seqlens_kv, B, Hq, Hkv,
                        max_Nq, max_Nkv, total_q, total_kv, D, causal, sm_scale, workspace,
                        workspace_bytes, stream);
}

static int check_out_dtype(int in_dtype, int out_dtype) {
  if (in_dtype != SAGE2_FP16 && in_dtype != SAGE2_BF16) return SAGE2_EINVAL;
  if (out_dtype != in_dtype && out_dtype != SAGE2_FP32) return SAGE2_EINVAL;
  return SAGE2_OK;
}

int sage2_attn_fwd(const void *q, const void *k, const void *v, void *out, int in_dtype,
                   int out_dtype, int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal,
                   float sm_scale, void *workspace, size_t workspace_bytes, void *stream) {
  int rc = check_out_dtype(in_dtype, out_dtype);
  if (rc) return rc;
  rc = sage2_prepass(q, k, v, in_dtype, B, Hq, Hkv, Nq, Nkv, D, causal, sm_scale, workspace,
                     workspace_bytes, stream);
  if (rc) return rc;
  return sage2_attention(out, out_dtype, B, Hq, Hkv, Nq, Nkv, D, causal, sm_scale, workspace,
                         workspace_bytes, stream);
}

int sage2_attn_fwd_varlen(const void *q, const void *k, const void *v, void *out, int in_dtype,
                          int out_dtype, const int *cu_seqlens_q, const int *cu_seqlens_kv, int B,
                          int Hq, int Hkv, int max_Nq, int max_Nkv, int total_q, int total_kv,
                          int D, int causal, float sm_scale, void *workspace,
                          size_t workspace_bytes, void *stream) {
  int rc = check_out_dtype(in_dtype, out_dtype);
  if (rc) return rc;
  rc = sage2_prepass_varlen(q, k, v, in_dtype, cu_seqlens_q, cu_seqlens_kv, B, Hq, Hkv, max_Nq,
                            max_Nkv, total_q, total_kv, D, causal, sm_scale, workspace,
                            workspace_bytes, stream);
  if (rc) return rc;
  return sage2_attention_varlen(out, out_dtype, cu_seqlens_q, cu_seqlens_kv, B, Hq, Hkv, max_Nq,
                                max_Nkv, total_q, total_kv, D, causal, sm_scale, workspace,
                                workspace_bytes, stream);
}

int sage2_device_status(const void *workspace, void *stream, int *raw) {
  if (!workspace) return SAGE2_EINVAL;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SAGE2_ECUDA;
  int word = 0;
  // the status word sits at offset 0 of the 1024-aligned workspace base
  if (cudaMemcpy(&word, ws_base(const_cast<void *>(workspace)), sizeof(int),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return SAGE2_ECUDA;
  if (raw) *raw = word;
  if (word == 0) return SAGE2_OK;
  if (word == kStatusSeqTooLong || word == kStatusFormat) return SAGE2_EINVAL;
  return SAGE2_EDEVICE_TIMEOUT;
}

int sage2_debug_tile(const int *cu_seqlens_q, const int *cu_seqlens_kv, int B, int Hq, int Hkv,
                     int max_Nq, int max_Nkv, int total_q, int total_kv, int D, int causal,
                     float sm_scale, const void *workspace, size_t workspace_bytes, int b, int h,
                     int qt, int kt, float *s_out, uint8_t *p_out, float *r_out, void *stream) {
  return sage2_debug_tile_ex(cu_seqlens_q, cu_seqlens_kv, B, Hq, Hkv, max_Nq, max_Nkv, total_q,
                             total_kv, D, causal, sm_scale, 0, workspace, workspace_bytes, b, h,
                             qt, kt, s_out, p_out, r_out, stream);
}

int sage2_debug_tile_ex(const int *cu_seqlens_q, const int *cu_seqlens_kv, int B, int Hq,
                        int Hkv, int max_Nq, int max_Nkv, int total_q, int total_kv, int D,
                        int causal, float sm_scale, int quant_flags, const void *workspace,
                        size_t workspace_bytes, int b, int h, int qt, int kt, float *s_out,
                        uint8_t *p_out, float *r_out, void *stream) {
  int rc = check_shapes(B, Hq, Hkv, max_Nq, max_Nkv, D, total_q, total_kv, causal);
  if (rc) return rc;
  if (!valid_quant_flags(quant_flags)) return SAGE2_EINVAL;
  if ((cu_seqlens_q == nullptr) != (cu_seqlens_kv == nullptr)) return SAGE2_EINVAL;
  if (!s_out || !p_out || !r_out || b < 0 || b >= B || h < 0 || h >= Hq || qt < 0 || kt < 0)
    return SAGE2_EINVAL;
  Geometry g;
  Layout L;
  if (!make_geometry(B, Hq, Hkv, max_Nq, max_Nkv, D, total_q, total_kv, causal, sm_scale,
                     cu_seqlens_q, cu_seqlens_kv, code_bytes_of(quant_flags), &g, &L))
    return SAGE2_EINVAL;
  if ((rc = check_ws(workspace, workspace_bytes, L))) return rc;
  if ((rc = check_device())) return rc;
  if (qt * 128 >= max_Nq) return SAGE2_EINVAL;
  // the debug launch still runs its epilogue: give it a private FP32 output buffer
  void *scratch = nullptr;
  const size_t out_bytes = (size_t)(total_q > 0 ? total_q : 1) * Hq * D * sizeof(float);
  if (cudaMallocAsync(&scratch, out_bytes, (cudaStream_t)stream) != cudaSuccess) return SAGE2_ECUDA;
  AttnDebug dbg{b, h, qt, kt, s_out, p_out, r_out, 0};
  cudaError_t e = launch_attention(scratch, SAGE2_FP32, g, L, workspace, (cudaStream_t)stream, &dbg,
                                   (quant_flags & SAGE2_QUANT_SAGE1) != 0);
  cudaFreeAsync(scratch, (cudaStream_t)stream);
  return cuda_status(e);
}

int sage2_debug_timeout(int B, int Hq, int Hkv, int Nq, int Nkv, int D, const void *workspace,
                        size_t workspace_bytes, void *stream) {
  int rc = check_shapes(B, Hq, Hkv, Nq, Nkv, D, B * Nq, B * Nkv, 0);
  if (rc) return rc;
  if (Nq <= 0 || Nkv <= 0) return SAGE2_EINVAL;
  Geometry g;
  Layout L;
  if (!make_geometry(B, Hq, Hkv, Nq, Nkv, D, B * Nq, B * Nkv, 0, 0.f, nullptr, nullptr, 1, &g, &L))
    return SAGE2_EINVAL;
  if ((rc = check_ws(workspace, workspace_bytes, L))) return rc;
  if ((rc = check_device())) return rc;
  void *scratch = nullptr;
  const size_t out_bytes = (size_t)B * Nq * Hq * D * sizeof(float);
  if (cudaMallocAsync(&scratch, out_bytes, (cudaStream_t)stream) != cudaSuccess) return SAGE2_ECUDA;
  float *sbuf = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void **>(&sbuf), 128 * 128 * 4 * 3, (cudaStream_t)stream) !=
      cudaSuccess)
    return SAGE2_ECUDA;
  AttnDebug dbg{0, 0, 0, 0, sbuf, reinterpret_cast<uint8_t *>(sbuf + 128 * 128),
                sbuf + 2 * 128 * 128, 1};
  dbg.kt = 1 << 30;  // dump nothing
  cudaError_t e = launch_attention(scratch, SAGE2_FP32, g, L, workspace, (cudaStream_t)stream, &dbg);
  cudaFreeAsync(scratch, (cudaStream_t)stream);
  cudaFreeAsync(sbuf, (cudaStream_t)stream);
  return cuda_status(e);
}

}  // extern "C"
