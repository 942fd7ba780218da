// sage2_noalloc.cu -- a forward entry point that allocates no device memory.
//
// Some callers cannot hand this library a workspace: runtimes that give out device memory only
// from their own pre-planned pools and forbid allocation calls from third-party code, or
// latency-critical loops where an allocation call (which may synchronize the device) is not
// allowed. For them, sage2_attn_fwd_noalloc uses a fixed scratch array that lives in the
// library's own device image instead of a caller workspace. The caller still provides q, k, v
// and out.
//
// Limits and behaviour:
//   - The scratch holds SAGE2_NOALLOC_SCRATCH_BYTES (64 MiB) on every GPU that loads this
//     library, until the process exits. Problems whose workspace (sage2_workspace_size) is
//     larger are rejected with SAGE2_EWORKSPACE before any work is queued.
//   - The first call on each device looks up the array's device address (with that device
//     current); make that first call before any stream capture.
//   - Every call shares the one array, which keeps the previous call's contents. Each call's
//     prepass clears the status word and rewrites every byte the attention kernel reads, so no
//     other clearing is needed; calls that overlap on the GPU (different streams, no ordering)
//     race on the array and corrupt each other's results.
#include <mutex>

#include "sage2_internal.h"

namespace {

constexpr size_t kScratchBytes = SAGE2_NOALLOC_SCRATCH_BYTES;

// In host code this name is only a host-side stand-in for the array; kernels must be given the
// device address obtained below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAGE2_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SAGE2_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SAGE2_OK;
}

}  // namespace

extern "C" int sage2_attn_fwd_noalloc(const void *q, const void *k, const void *v, void *out,
                                      int in_dtype, int out_dtype, int B, int Hq, int Hkv,
                                      int Nq, int Nkv, int D, int causal, float sm_scale,
                                      void *stream) {
  if ((long long)B * Nq >= (1LL << 31) || (long long)B * Nkv >= (1LL << 31) || B <= 0)
    return SAGE2_EINVAL;
  const size_t need = sage2_workspace_size(B, Hq, Hkv, Nq, Nkv, D, B * Nq, B * Nkv);
  if (need == 0)  // invalid sizes: let the regular checks name the problem (no CUDA call)
    return sage2_attn_fwd(q, k, v, out, in_dtype, out_dtype, B, Hq, Hkv, Nq, Nkv, D, causal,
                          sm_scale, nullptr, 0, stream);
  if (need > kScratchBytes) return SAGE2_EWORKSPACE;
  void *scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != SAGE2_OK) return rc;
  return sage2_attn_fwd(q, k, v, out, in_dtype, out_dtype, B, Hq, Hkv, Nq, Nkv, D, causal,
                        sm_scale, scratch, kScratchBytes, stream);
}

extern "C" int sage2_noalloc_status(void *stream, int *raw) {
  void *scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != SAGE2_OK) return rc;
  return sage2_device_status(scratch, stream, raw);
}
