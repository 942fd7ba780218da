// sage2_host.cu -- the forward from host memory, with the transfers overlapped with compute.
//
// A caller whose q, k, v and output live in (page-locked) host memory would otherwise pay the
// copies in, the prepass and attention, and the copy out back to back. The problem splits
// exactly into groups of kv heads (every quantity the method computes -- K channel means, V
// scales, Q block means, DeltaS, the attention rows -- stays inside one kv head and its group
// of q heads), so sage2_attn_fwd_host runs it group chunk by group chunk: while chunk c is
// computed, the inputs of chunk c + 1 are copied in on a copy stream and the output of chunk
// c - 1 is copied out on another. Even chunks compute on the caller's stream and odd ones on a
// second compute stream, so the first CTAs of one chunk fill the SMs that the last CTAs of the
// previous one leave idle. Two device slots (inputs, output, workspace) alternate with the
// chunks; a slot's inputs are refilled as soon as the prepass of its previous chunk has read
// them, so that copy overlaps the previous chunk's attention. A chunk's K and V are copied
// before its Q, and its K/V statistics and codes start while Q is still coming in. Chunk
// results are those of the whole problem, bit for bit.
#include <mutex>

#include "sage2_device.cuh"
#include "sage2_internal.h"

namespace sage2 {
namespace {

size_t align1k(size_t x) { return (x + 1023) / 1024 * 1024; }

struct HostPlan {
  int chunks, hq_c, hk_c;
  size_t q, kv, o, ws;  // bytes of one slot's parts
  size_t slot;          // bytes of one slot
  size_t total;         // scratch bytes (status area + two slots + alignment slack)
};

bool make_plan(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int in_bytes, int out_bytes,
               int hk_c, int quant_flags, HostPlan *p) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || hk_c <= 0 || Hkv % hk_c != 0) return false;
  p->hk_c = hk_c;
  p->hq_c = hk_c * (Hq / Hkv);
  p->chunks = Hkv / hk_c;
  p->q = align1k((size_t)B * Nq * p->hq_c * D * in_bytes);
  p->kv = align1k((size_t)B * Nkv * p->hk_c * D * in_bytes);
  p->o = align1k((size_t)B * Nq * p->hq_c * D * out_bytes);
  p->ws = sage2_workspace_size_ex(B, p->hq_c, p->hk_c, Nq, Nkv, D, B * Nq, B * Nkv, quant_flags);
  if (p->ws == 0) return false;
  p->ws = align1k(p->ws);
  p->slot = p->q + 2 * p->kv + p->o + p->ws;
  p->total = 1024 + 2 * p->slot + 1024;
  return true;
}

uint8_t *base1k(void *p) {
  const uintptr_t u = reinterpret_cast<uintptr_t>(p);
  return reinterpret_cast<uint8_t *>((u + 1023) & ~uintptr_t(1023));
}

// The copy streams and the events of the pipeline, one set per device, created on first use.
// One mutex per device orders whole calls: every event a call waits on was recorded by that
// call.
struct DevPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp = nullptr;  // comp: the odd chunks
  cudaStream_t tail = nullptr;  // the second half of the last chunk's attention
  cudaEvent_t entry = nullptr, kv_in[2] = {}, in_done[2] = {}, pre_done[2] = {},
              comp_done[2] = {}, out_done[2] = {}, half_done = nullptr;
};
constexpr int kMaxDevices = 64;
DevPipe g_pipes[kMaxDevices];

int get_pipe(DevPipe **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAGE2_ECUDA;
  DevPipe &p = g_pipes[dev];
  *out = &p;
  return SAGE2_OK;
}

int init_pipe(DevPipe &p) {  // with p.mu held
  if (p.ready) return SAGE2_OK;
  const unsigned ef = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p.tail, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&p.entry, ef) != cudaSuccess ||
      cudaEventCreateWithFlags(&p.half_done, ef) != cudaSuccess)
    return SAGE2_ECUDA;
  for (int i = 0; i < 2; ++i)
    if (cudaEventCreateWithFlags(&p.kv_in[i], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.in_done[i], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.pre_done[i], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.comp_done[i], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.out_done[i], ef) != cudaSuccess)
      return SAGE2_ECUDA;
  p.ready = true;
  return SAGE2_OK;
}

// Keeps the first nonzero chunk status in the call's status word.
__global__ void merge_status(const int *chunk, int *total) {
  const int v = *chunk;
  if (v != 0) atomicCAS(total, 0, v);
}

int dtype_bytes(int dt) { return dt == SAGE2_FP32 ? 4 : 2; }

}  // namespace
}  // namespace sage2

using namespace sage2;

extern "C" size_t sage2_host_scratch_size(int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                                          int out_dtype, int kv_heads_per_chunk,
                                          int quant_flags) {
  HostPlan p;
  if (out_dtype != SAGE2_FP16 && out_dtype != SAGE2_BF16 && out_dtype != SAGE2_FP32) return 0;
  if (!make_plan(B, Hq, Hkv, Nq, Nkv, D, 2, dtype_bytes(out_dtype), kv_heads_per_chunk,
                 quant_flags, &p))
    return 0;
  return p.total;
}

extern "C" int sage2_attn_fwd_host(const void *q, const void *k, const void *v, void *out,
                                   int in_dtype, int out_dtype, int B, int Hq, int Hkv, int Nq,
                                   int Nkv, int D, int causal, float sm_scale, int quant_flags,
                                   int kv_heads_per_chunk, void *scratch, size_t scratch_bytes,
                                   void *stream) {
  if ((long long)B * Nq >= (1LL << 31) || (long long)B * Nkv >= (1LL << 31)) return SAGE2_EINVAL;
  if (in_dtype != SAGE2_FP16 && in_dtype != SAGE2_BF16) return SAGE2_EINVAL;
  if (out_dtype != in_dtype && out_dtype != SAGE2_FP32) return SAGE2_EINVAL;
  if (!q || !k || !v || !out || !scratch) return SAGE2_EINVAL;
  HostPlan p;
  if (!make_plan(B, Hq, Hkv, Nq, Nkv, D, 2, dtype_bytes(out_dtype), kv_heads_per_chunk,
                 quant_flags, &p))
    return SAGE2_EINVAL;
  if (scratch_bytes < p.total) return SAGE2_EWORKSPACE;
  if (Nq == 0) return SAGE2_OK;
  DevPipe *pipe = nullptr;
  int rc = get_pipe(&pipe);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(pipe->mu);
  if ((rc = init_pipe(*pipe))) return rc;

  const cudaStream_t s0 = (cudaStream_t)stream;
  uint8_t *base = base1k(scratch);
  int *status_total = reinterpret_cast<int *>(base);
  const size_t ib = 2, ob = dtype_bytes(out_dtype);
  const size_t rows_q = (size_t)B * Nq, rows_kv = (size_t)B * Nkv;
  const size_t qw = (size_t)p.hq_c * D * ib, kw = (size_t)p.hk_c * D * ib, ow = (size_t)p.hq_c * D * ob;
  const size_t qpitch = (size_t)Hq * D * ib, kpitch = (size_t)Hkv * D * ib, opitch = (size_t)Hq * D * ob;

  // On an error after work was queued, the given stream still waits for everything queued on
  // the copy and compute streams (a caller that synchronizes it may then reuse its buffers).
  auto join = [&]() {
    cudaEvent_t done[4] = {pipe->in_done[0], pipe->comp_done[0], pipe->out_done[0],
                           pipe->half_done};
    const cudaStream_t side[4] = {pipe->h2d, pipe->comp, pipe->d2h, pipe->tail};
    for (int i = 0; i < 4; ++i)
      if (cudaEventRecord(done[i], side[i]) == cudaSuccess) cudaStreamWaitEvent(s0, done[i], 0);
  };
#define SAGE2_CK(x)              \
  do {                           \
    if ((x) != cudaSuccess) {    \
      join();                    \
      return SAGE2_ECUDA;        \
    }                            \
  } while (0)
  SAGE2_CK(cudaMemsetAsync(status_total, 0, sizeof(int), s0));
  SAGE2_CK(cudaEventRecord(pipe->entry, s0));  // copies start after the caller's earlier work
  SAGE2_CK(cudaStreamWaitEvent(pipe->h2d, pipe->entry, 0));
  SAGE2_CK(cudaStreamWaitEvent(pipe->d2h, pipe->entry, 0));
  SAGE2_CK(cudaStreamWaitEvent(pipe->comp, pipe->entry, 0));
  SAGE2_CK(cudaStreamWaitEvent(pipe->tail, pipe->entry, 0));
  for (int c = 0; c < p.chunks; ++c) {
    const int sl = c & 1;
    const cudaStream_t cs = sl ? pipe->comp : s0;  // the slot's compute stream
    uint8_t *slot = base + 1024 + sl * p.slot;
    uint8_t *dq = slot, *dk = slot + p.q, *dv = dk + p.kv, *dout = dv + p.kv, *dws = dout + p.o;
    // inputs of chunk c, once the prepass of the slot's previous chunk, c - 2, has read its
    // inputs (its attention reads only the workspace, so the copy overlaps it); K and V first,
    // so that the chunk's K/V statistics and codes overlap the copy of Q
    if (c >= 2) SAGE2_CK(cudaStreamWaitEvent(pipe->h2d, pipe->pre_done[sl], 0));
    if (rows_kv) {
      SAGE2_CK(cudaMemcpy2DAsync(dk, kw, static_cast<const uint8_t *>(k) + c * kw, kpitch, kw,
                                 rows_kv, cudaMemcpyHostToDevice, pipe->h2d));
      SAGE2_CK(cudaMemcpy2DAsync(dv, kw, static_cast<const uint8_t *>(v) + c * kw, kpitch, kw,
                                 rows_kv, cudaMemcpyHostToDevice, pipe->h2d));
    }
    SAGE2_CK(cudaEventRecord(pipe->kv_in[sl], pipe->h2d));
    SAGE2_CK(cudaMemcpy2DAsync(dq, qw, static_cast<const uint8_t *>(q) + c * qw, qpitch, qw,
                               rows_q, cudaMemcpyHostToDevice, pipe->h2d));
    SAGE2_CK(cudaEventRecord(pipe->in_done[sl], pipe->h2d));
    // compute chunk c (its output slot has been copied out); the prepass's Q kernels wait for
    // the copy of Q
    SAGE2_CK(cudaStreamWaitEvent(cs, pipe->kv_in[sl], 0));
    if (c >= 2) SAGE2_CK(cudaStreamWaitEvent(cs, pipe->out_done[sl], 0));
    rc = prepass_impl(dq, dk, dv, in_dtype, nullptr, nullptr, B, p.hq_c, p.hk_c, Nq, Nkv, B * Nq,
                      B * Nkv, D, causal, sm_scale, quant_flags, dws, p.ws, cs,
                      pipe->in_done[sl]);
    if (rc == SAGE2_OK && cudaEventRecord(pipe->pre_done[sl], cs) != cudaSuccess) rc = SAGE2_ECUDA;
    // The last chunk's output copy has nothing left to overlap: its attention runs as two
    // launches over halves of its q heads (the second on its own stream, so its CTAs fill the
    // first one's tail), and the first half is copied out while the second computes.
    const int h1 = (c == p.chunks - 1) ? p.hq_c / 2 : 0;
    if (rc == SAGE2_OK)
      rc = attention_impl(dout, out_dtype, quant_flags, nullptr, nullptr, B, p.hq_c, p.hk_c, Nq,
                          Nkv, B * Nq, B * Nkv, D, causal, sm_scale, dws, p.ws, cs, 0, h1);
    if (rc == SAGE2_OK && h1 > 0) {
      if (cudaEventRecord(pipe->half_done, cs) != cudaSuccess ||
          cudaStreamWaitEvent(pipe->tail, pipe->pre_done[sl], 0) != cudaSuccess)
        rc = SAGE2_ECUDA;
      else
        rc = attention_impl(dout, out_dtype, quant_flags, nullptr, nullptr, B, p.hq_c, p.hk_c,
                            Nq, Nkv, B * Nq, B * Nkv, D, causal, sm_scale, dws, p.ws, pipe->tail,
                            h1, p.hq_c - h1);
    }
    if (rc) {
      join();
      return rc;
    }
    const cudaStream_t cs_end = h1 > 0 ? pipe->tail : cs;  // after both halves
    if (h1 > 0) SAGE2_CK(cudaStreamWaitEvent(pipe->tail, pipe->half_done, 0));
    merge_status<<<1, 1, 0, cs_end>>>(reinterpret_cast<const int *>(base1k(dws)), status_total);
    SAGE2_CK(cudaGetLastError());
    SAGE2_CK(cudaEventRecord(pipe->comp_done[sl], cs_end));
    // output of chunk c (the first half of the last chunk's heads as soon as it is done)
    uint8_t *hout = static_cast<uint8_t *>(out) + c * ow;
    const size_t hw = (size_t)h1 * D * ob;  // bytes of a row's first h1 heads
    if (h1 > 0) {
      SAGE2_CK(cudaStreamWaitEvent(pipe->d2h, pipe->half_done, 0));
      SAGE2_CK(cudaMemcpy2DAsync(hout, opitch, dout, ow, hw, rows_q, cudaMemcpyDeviceToHost,
                                 pipe->d2h));
    }
    SAGE2_CK(cudaStreamWaitEvent(pipe->d2h, pipe->comp_done[sl], 0));
    SAGE2_CK(cudaMemcpy2DAsync(hout + hw, opitch, dout + hw, ow, ow - hw, rows_q,
                               cudaMemcpyDeviceToHost, pipe->d2h));
    SAGE2_CK(cudaEventRecord(pipe->out_done[sl], pipe->d2h));
  }
  // the caller's stream completes only after the last copies out
  SAGE2_CK(cudaStreamWaitEvent(s0, pipe->out_done[(p.chunks - 1) & 1], 0));
  if (p.chunks > 1) SAGE2_CK(cudaStreamWaitEvent(s0, pipe->out_done[p.chunks & 1], 0));
#undef SAGE2_CK
  return SAGE2_OK;
}

extern "C" int sage2_host_status(const void *scratch, void *stream, int *raw) {
  if (!scratch) return SAGE2_EINVAL;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SAGE2_ECUDA;
  int word = 0;
  if (cudaMemcpy(&word, base1k(const_cast<void *>(scratch)), sizeof(int),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return SAGE2_ECUDA;
  if (raw) *raw = word;
  if (word == 0) return SAGE2_OK;
  if (word == kStatusSeqTooLong || word == kStatusFormat) return SAGE2_EINVAL;
  return SAGE2_EDEVICE_TIMEOUT;
}
