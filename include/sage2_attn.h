/*
 * sage2_attn.h -- C ABI of the GB300 (sm_103a) SageAttention2 quantized attention forward.
 *
 * What it computes: exact attention O = softmax(Q K^T * sm_scale) V, evaluated the
 * SageAttention2 way (sources: the web pages "SageAttention2 and Fast Exact INT4
 * Attention" visual companion, sections Visual Thesis, Numerical Repair Stack and
 * Per-Thread INT4 Geometry; "SageAttention2: Efficient Attention with Thorough Outlier
 * Smoothing and Per-thread INT4 Quantization" research note, its three components;
 * PMLR v267 zhang25ae, Abstract):
 *   1. K is smoothed by its per-(sequence, kv head) channel mean; Q by the mean of each
 *      block of 128 rows, with the correction DeltaS = qmean . (K - kmean)^T added back
 *      to the logits.
 *   2. Smoothed Q and K are put on the INT4 grid [-7, 7]: one FP32 scale per Q row and
 *      one per 32 consecutive K tokens (the thread-owned groups of the tensor-memory
 *      accumulator layout). Q K^T of the codes is exact (integer valued).
 *   3. V is quantized per channel to FP8 e4m3 (scale amax/448); P~ = e4m3(448 P).
 *   4. Two-level accumulation of P~ V: each 128-key block's FP8 products are summed by the
 *      tensor core into an FP32 accumulator in tensor memory, and the running output stays
 *      FP32 across blocks. The default kernel (two Q tiles per CTA) rescales the FP32 output
 *      accumulator by alpha on the CUDA cores when a row maximum moves and lets the block's
 *      MMA add into it; with SAGE2_ATTN_PP=0 in the environment (and for SAGE2_QUANT_SAGE1),
 *      the one-tile kernel sums each block into a fresh FP32 partial and folds it into an FP32
 *      output held in registers (O = alpha O + R).
 * Interface envelope (visual companion, Per-Thread INT4 Geometry, implementation panel):
 * GQA, different q and kv lengths, packed variable-length batches, head dim padded to
 * 64 or 128, head dims above 128 rejected.
 *
 * Conventions shared by every entry point:
 *   - Tensors are token-major: dense calls take q [B, Nq, Hq, D], k and v [B, Nkv, Hkv, D],
 *     out [B, Nq, Hq, D]; varlen calls take the packed forms [total, H, D] with
 *     cu_seqlens (int32, B + 1 prefix sums). All row-major and contiguous.
 *   - q, k, v, out, workspace are DEVICE pointers owned by the caller; nothing is retained
 *     after a call returns (except by sage2_attn_fwd_noalloc, whose scratch array lives in the
 *     library and keeps the last call's contents). Pointers, the workspace included, must be
 *     16-byte aligned; the library aligns the workspace base up to 1024 bytes inside the call
 *     (sage2_workspace_size() includes that slack).
 *   - in_dtype: SAGE2_FP16 or SAGE2_BF16. out_dtype: the input dtype or SAGE2_FP32.
 *   - D (the head dim of the tensors, called D0 in the comments) must satisfy 8 <= D <= 128
 *     and D % 8 == 0; it is computed as 64 (D <= 64) or 128 (D <= 128) with zero channels.
 *   - Hq % Hkv == 0 (GQA: q head h reads kv head h / (Hq / Hkv)).
 *   - causal: key j is visible to query i of a sequence iff j <= i + Nkv - Nq (aligned at
 *     the bottom-right); a row with no visible key outputs 0.
 *   - sm_scale <= 0 selects 1/sqrt(D).
 *   - stream is a cudaStream_t (NULL = legacy default stream). Calls are asynchronous on it:
 *     the return code covers argument checks and launch errors only; a device-side wait
 *     that gave up is reported later by sage2_device_status().
 *   - Two calls that share a workspace must be ordered (same stream, or synchronized).
 *   - The device must be sm_103 (GB300); other devices return SAGE2_EUNSUPPORTED.
 */
#ifndef SAGE2_ATTN_H
#define SAGE2_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SAGE2_OK = 0,
  SAGE2_EINVAL = -1,          /* bad argument: null/misaligned pointer, bad size, Hq % Hkv */
  SAGE2_EUNSUPPORTED = -2,    /* head dim > 128 or not a multiple of 8, or not an sm_103 GPU */
  SAGE2_EWORKSPACE = -3,      /* workspace smaller than sage2_workspace_size() or misaligned */
  SAGE2_ECUDA = -4,           /* a CUDA call (launch, copy, tensor-map encode) failed */
  SAGE2_EDEVICE_TIMEOUT = -5  /* a bounded device-side wait expired (kernel returned early) */
} sage2_status;

typedef enum { SAGE2_FP16 = 0, SAGE2_BF16 = 1, SAGE2_FP32 = 2 } sage2_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *sage2_status_str(int status);

/* Library ABI version: 100 * major + minor. */
int sage2_version(void);

/* Bytes of device workspace a call with these sizes needs (0 on invalid sizes).
 * Dense calls: total_q = B * Nq, total_kv = B * Nkv, max_Nq = Nq, max_Nkv = Nkv. */
size_t sage2_workspace_size(int B, int Hq, int Hkv, int max_Nq, int max_Nkv, int D, int total_q,
                            int total_kv);

/* Full forward (prepass + attention) on dense [B, N, H, D] tensors. */
int sage2_attn_fwd(const void *q, const void *k, const void *v, void *out, int in_dtype,
                   int out_dtype, int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal,
                   float sm_scale, void *workspace, size_t workspace_bytes, void *stream);

/* Full forward on packed variable-length batches. cu_seqlens_q / cu_seqlens_kv are
 * DEVICE int32 arrays of B + 1 prefix sums whose last entries equal total_q / total_kv;
 * max_Nq / max_Nkv bound every sequence length (checked on the device: a sequence that
 * exceeds them is skipped and reported through sage2_device_status). */
int sage2_attn_fwd_varlen(const void *q, const void *k, const void *v, void *out, int in_dtype,
                          int out_dtype, const int *cu_seqlens_q, const int *cu_seqlens_kv, int B,
                          int Hq, int Hkv, int max_Nq, int max_Nkv, int total_q, int total_kv,
                          int D, int causal, float sm_scale, void *workspace,
                          size_t workspace_bytes, void *stream);

/* The two halves of the forward, for callers (and benchmarks) that time or schedule them
 * apart. sage2_prepass*: smoothing and quantization only (K/V statistics, Q/K INT4 codes
 * and scales, V e4m3 codes transposed, DeltaS), written into the workspace.
 * sage2_attention*: the fused attention kernel only, reading a workspace that a prepass
 * call with the same arguments filled.
 * Every prepass (these and the one inside the full forwards) runs its Q codes and V codes on
 * two library-owned streams, forked from `stream` and joined back into it with events before
 * the call's last kernel, so the call stays ordered on `stream` as a whole. The first prepass
 * on a device creates those streams and events (kept until the process exits): make it before
 * any stream capture. */
int sage2_prepass(const void *q, const void *k, const void *v, int in_dtype, int B, int Hq,
                  int Hkv, int Nq, int Nkv, int D, int causal, float sm_scale, void *workspace,
                  size_t workspace_bytes, void *stream);
int sage2_attention(void *out, int out_dtype, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                    int causal, float sm_scale, const void *workspace, size_t workspace_bytes,
                    void *stream);
int sage2_prepass_varlen(const void *q, const void *k, const void *v, int in_dtype,
                         const int *cu_seqlens_q, const int *cu_seqlens_kv, int B, int Hq,
                         int Hkv, int max_Nq, int max_Nkv, int total_q, int total_kv, int D,
                         int causal, float sm_scale, void *workspace, size_t workspace_bytes,
                         void *stream);
int sage2_attention_varlen(void *out, int out_dtype, const int *cu_seqlens_q,
                           const int *cu_seqlens_kv, int B, int Hq, int Hkv, int max_Nq,
                           int max_Nkv, int total_q, int total_kv, int D, int causal,
                           float sm_scale, const void *workspace, size_t workspace_bytes,
                           void *stream);

/* Quantization switches for sage2_prepass_varlen_ex: accuracy ablations of the method's
 * three repairs (SageAttention2 research note, components 1 and 2; PMLR v267 zhang25ae,
 * Abstract: smoothing Q, smoothing K, per-thread instead of per-block INT4 scales).
 * 0 is the method itself. The attention kernel is the same for every setting; only what the
 * prepass writes into the workspace changes. */
typedef enum {
  SAGE2_QUANT_NO_SMOOTH_Q = 1, /* Q block mean taken as 0: Q~ = Q and DeltaS = 0 */
  SAGE2_QUANT_NO_SMOOTH_K = 2, /* K channel mean taken as 0: K~ = K */
  SAGE2_QUANT_PER_BLOCK = 4,   /* one INT4 scale per 128-row Q block and per 128-key K block
                                  (instead of one per query row and per 32 keys) */
  SAGE2_QUANT_SAGE1 = 8        /* the SageAttention (v1) path the research note contrasts the
                                  method with (its opening paragraph): Q and K codes on the INT8
                                  grid [-127, 127], one scale per 128-row Q block and per 128-key
                                  K block, K smoothed, Q not (no DeltaS); P~ and V as in the
                                  method. Q K^T runs on 16-bit tensor-core operands holding the
                                  integer codes exactly. Must be used alone; it changes the
                                  workspace size (two bytes per Q and K code) and the attention
                                  kernel, so the workspace, prepass and attention calls must all
                                  be given it. */
} sage2_quant_flags;

/* Workspace size and layout for a quantization setting (sage2_quant_flags; 0 gives
 * sage2_workspace_size / sage2_workspace_layout). 0 / SAGE2_EINVAL on invalid arguments. */
size_t sage2_workspace_size_ex(int B, int Hq, int Hkv, int max_Nq, int max_Nkv, int D,
                               int total_q, int total_kv, int quant_flags);

/* sage2_prepass_varlen with quantization switches (sage2_quant_flags: the first three in any
 * combination, or SAGE2_QUANT_SAGE1 alone; anything else returns SAGE2_EINVAL). Same arguments,
 * workspace contents and errors otherwise; the workspace must hold
 * sage2_workspace_size_ex(..., quant_flags) bytes. Follow it with sage2_attention_varlen_ex
 * (same quant_flags) on the same workspace. The prepass records the code format in the
 * workspace; an attention call for the other format finds it there, writes nothing and makes
 * sage2_device_status return SAGE2_EINVAL. */
int sage2_prepass_varlen_ex(const void *q, const void *k, const void *v, int in_dtype,
                            const int *cu_seqlens_q, const int *cu_seqlens_kv, int B, int Hq,
                            int Hkv, int max_Nq, int max_Nkv, int total_q, int total_kv, int D,
                            int causal, float sm_scale, int quant_flags, void *workspace,
                            size_t workspace_bytes, void *stream);

/* sage2_attention_varlen for a workspace filled by sage2_prepass_varlen_ex with the same
 * quant_flags (only SAGE2_QUANT_SAGE1 selects another kernel; the other switches only change
 * what the prepass wrote). */
int sage2_attention_varlen_ex(void *out, int out_dtype, const int *cu_seqlens_q,
                              const int *cu_seqlens_kv, int B, int Hq, int Hkv, int max_Nq,
                              int max_Nkv, int total_q, int total_kv, int D, int causal,
                              float sm_scale, int quant_flags, const void *workspace,
                              size_t workspace_bytes, void *stream);

/* Synchronizes `stream`, then reads the workspace's device status word (cleared by every
 * prepass). Returns SAGE2_OK, SAGE2_EDEVICE_TIMEOUT (a bounded wait expired) or
 * SAGE2_EINVAL (a varlen sequence exceeded max_Nq/max_Nkv, or the attention call's code format
 * was not the one its prepass wrote); *raw (if not NULL) receives the word itself (0 when clean;
 * otherwise a code naming the wait that gave up). */
int sage2_device_status(const void *workspace, void *stream, int *raw);

/* The forward from host memory: q, k, v [B, Nq or Nkv, H, D] and out [B, Nq, Hq, D] are host
 * pointers (page-locked for the copies to overlap; pageable memory works but serializes), the
 * rest as sage2_attn_fwd, plus quant_flags (sage2_quant_flags, 0 for the method). The problem is
 * run in chunks of kv_heads_per_chunk kv heads (and their q heads; it must divide Hkv): the
 * copies in of one chunk and out of another overlap the computation of a third, on two copy
 * streams of the library's own and the given stream. Results are those of sage2_attn_fwd on the
 * whole problem. `scratch` is caller-owned device memory of at least sage2_host_scratch_size(...)
 * bytes (two chunk slots: inputs, output, workspace); calls that overlap in time must not share
 * it. The given stream completes after the last copy out. Device-side errors (bounded waits,
 * format) are kept for sage2_host_status. Returns SAGE2_EINVAL / SAGE2_EWORKSPACE / SAGE2_ECUDA
 * before or while queuing. */
size_t sage2_host_scratch_size(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int out_dtype,
                               int kv_heads_per_chunk, int quant_flags);
int sage2_attn_fwd_host(const void *q, const void *k, const void *v, void *out, int in_dtype,
                        int out_dtype, int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal,
                        float sm_scale, int quant_flags, int kv_heads_per_chunk, void *scratch,
                        size_t scratch_bytes, void *stream);
/* As sage2_device_status, for the chunks of the last sage2_attn_fwd_host call on `scratch`. */
int sage2_host_status(const void *scratch, void *stream, int *raw);

/* Byte offsets of the buffers inside a workspace, for tests and tools that read the
 * intermediate results. Layouts (Tq, Tkv = padded token counts; every sequence starts on a
 * 128-row boundary at row 128 * (cu_seqlens[b] / 128 + b)):
 *   qcode  u8 (e4m3 bytes holding integers in [-7,7]) [Hq][Tq][Dp]
 *   kcode  u8 (same)                                  [Hkv][Tkv][Dp]
 *   vcodeT u8 (e4m3)                                  [Hkv][Dp][Tkv]
 *   qscale f32 [Hq][Tq]        kscale f32 [Hkv][Tkv/32]
 *   qmean  f32 [Hq][Tq/128][Dp]
 *   kmean  f32 [B][Hkv][Dp]    vscale f32 [B][Hkv][Dp] (amax/448)
 *   dsc    f32 [Hq][Tq/128][Nkv_pad] = fl32(DeltaS * log2(e) * sm_scale) */
typedef struct {
  size_t total_bytes;
  size_t qcode, kcode, vcodeT, qscale, kscale, qmean, kmean, vscale, vinv, dsc;
  size_t kpart, vpart, status;
  int Dp, Tq, Tkv, nkv_pad, nchunk;
  int code_bytes; /* bytes per Q and K code: 1 (e4m3 byte), 2 (SAGE2_QUANT_SAGE1: fp16 value) */
} sage2_ws_layout;

int sage2_workspace_layout(int B, int Hq, int Hkv, int max_Nq, int max_Nkv, int D, int total_q,
                           int total_kv, sage2_ws_layout *layout);
int sage2_workspace_layout_ex(int B, int Hq, int Hkv, int max_Nq, int max_Nkv, int D,
                              int total_q, int total_kv, int quant_flags,
                              sage2_ws_layout *layout);

/* Test hook (unstable): reruns the attention kernel for the single (sequence b, q head h,
 * q tile qt) work unit on a prepared workspace and dumps, for its KV tile kt, the raw
 * integer Q K^T accumulators (s_out: f32 [128][128], exact integers), the P~ e4m3 bytes
 * (p_out: u8 [128][128]) and the fresh P~V partial (r_out: f32 [128][Dp]), all device
 * buffers. The two-tile kernel that runs the INT4 codes accumulates P~V straight into the
 * output accumulator, so there r_out is written for kt = 0 only (the first partial) and left
 * untouched otherwise; with SAGE2_ATTN_PP=0 in the environment, and for INT8 codes, the
 * one-tile kernel runs and r_out is written for every kt. Same size arguments as
 * sage2_attention_varlen (cu_seqlens may be NULL for dense inputs, then Nq = max_Nq and
 * Nkv = max_Nkv for every sequence). */
int sage2_debug_tile(const int *cu_seqlens_q, const int *cu_seqlens_kv, int B, int Hq, int Hkv,
                     int max_Nq, int max_Nkv, int total_q, int total_kv, int D, int causal,
                     float sm_scale, const void *workspace, size_t workspace_bytes, int b, int h,
                     int qt, int kt, float *s_out, uint8_t *p_out, float *r_out, void *stream);
/* sage2_debug_tile for a workspace prepared with quant_flags (see sage2_prepass_varlen_ex). */
int sage2_debug_tile_ex(const int *cu_seqlens_q, const int *cu_seqlens_kv, int B, int Hq,
                        int Hkv, int max_Nq, int max_Nkv, int total_q, int total_kv, int D,
                        int causal, float sm_scale, int quant_flags, const void *workspace,
                        size_t workspace_bytes, int b, int h, int qt, int kt, float *s_out,
                        uint8_t *p_out, float *r_out, void *stream);

/* Test hook (unstable): runs one attention work unit whose producer never issues its
 * loads, so every consumer wait must expire (about one second); the kernel must return on
 * its own and leave SAGE2_EDEVICE_TIMEOUT in the workspace status word. Needs a workspace
 * filled by a prepass with the same sizes. */
int sage2_debug_timeout(int B, int Hq, int Hkv, int Nq, int Nkv, int D, const void *workspace,
                        size_t workspace_bytes, void *stream);

/* Forward without any device allocation. No counterpart in the paper: this exists for
 * callers that cannot give the library a workspace -- runtimes that hand out device memory
 * only from their own pre-planned pools and forbid allocation calls from third-party code,
 * and latency-critical loops where an allocation call (which may synchronize the device) is
 * not allowed. Same arguments and results as sage2_attn_fwd, minus the workspace: the
 * library uses a fixed scratch array of SAGE2_NOALLOC_SCRATCH_BYTES that every GPU loading
 * the library holds until the process exits.
 *   - Returns SAGE2_EWORKSPACE, before queuing any work, when sage2_workspace_size() of the
 *     problem exceeds SAGE2_NOALLOC_SCRATCH_BYTES; other argument errors as sage2_attn_fwd.
 *   - The first call on a device looks up the scratch address with that device current;
 *     make that first call before any stream capture.
 *   - All calls share the scratch, which keeps the last call's contents (each call rewrites
 *     what it reads and clears its status word). Calls that overlap on the GPU race and
 *     corrupt each other; order them (one stream, or explicit synchronization).
 *   - Allocates nothing: no cudaMalloc/cudaFree, no allocating library routine. */
#define SAGE2_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int sage2_attn_fwd_noalloc(const void *q, const void *k, const void *v, void *out, int in_dtype,
                           int out_dtype, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                           int causal, float sm_scale, void *stream);

/* Device status of the noalloc scratch on the current device, the sage2_device_status of the
 * workspace that sage2_attn_fwd_noalloc uses: synchronizes `stream`, then reads the status word
 * of the last noalloc call. Returns SAGE2_OK, SAGE2_EINVAL (a sequence exceeded its bound, or
 * the code format was wrong) or SAGE2_EDEVICE_TIMEOUT (a device-side wait gave up; the wait
 * site is in the low byte of *raw); SAGE2_ECUDA if the scratch or the word cannot be read.
 * `raw` (may be NULL) receives the status word. */
int sage2_noalloc_status(void *stream, int *raw);

#ifdef __cplusplus
}
#endif

#endif /* SAGE2_ATTN_H */
