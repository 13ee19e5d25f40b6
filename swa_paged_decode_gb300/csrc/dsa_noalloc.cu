// dsa_noalloc.cu -- dsa_decode_run_noalloc: one decode call (run + combine)
// whose workspace is the library's own file-scope device array instead of
// caller memory. Host code plus one __device__ array; the kernels are the
// ones dsa_decode_run / dsa_decode_combine launch, called unchanged.
//
// Per device, the first call made with that device current looks the array
// up with cudaGetSymbolAddress (loading this module if needed) and caches the
// pointer; later calls reuse it. Calls share the one array: two calls in
// flight at the same time on one device (other streams, other host threads)
// race on it.
#include <mutex>

#include "dsa_internal.cuh"

// The scratch: status word, selection records and split-KV partials of one
// call, laid out by the plan exactly as in a caller-owned workspace.
static __device__ __align__(256) unsigned char g_dsa_noalloc_scratch[DSA_NOALLOC_MAX_WORKSPACE];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (set up once).
dsa_status scratch_for_current_device(void **ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dsa_noalloc_scratch) != cudaSuccess || !p)
      return DSA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" {

dsa_status dsa_decode_run_noalloc(const dsa_decode_plan_t *plan, const void *q,
                                  int64_t q_stride_t, int64_t q_stride_h,
                                  const dsa_cache_desc *swa_cache, const int32_t *swa_idx,
                                  int64_t swa_idx_stride, const int32_t *swa_lens,
                                  const dsa_cache_desc *extra_cache, const int32_t *extra_idx,
                                  int64_t extra_idx_stride, const int32_t *extra_lens,
                                  const float *sink, const int64_t *positions,
                                  const float *cos_sin, int64_t cos_sin_rows, float scale,
                                  void *out, float *lse, int32_t *device_status,
                                  dsa_stream_t stream) {
  if (!plan || plan->magic != dsa::kPlanMagic || plan->abi_version != DSA_DECODE_ABI_VERSION)
    return DSA_ERR_PLAN;
  // Checked before any CUDA call: plans needing more than the array are refused.
  if (plan->workspace_bytes > (int64_t)DSA_NOALLOC_MAX_WORKSPACE) return DSA_ERR_WORKSPACE;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) % 4) != 0)
    return DSA_ERR_ALIGNMENT;
  if (plan->num_tokens == 0) {   // nothing to launch; the status word still says DSA_OK
    if (device_status &&
        cudaMemsetAsync(device_status, 0, 4, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return DSA_ERR_CUDA;
    return DSA_OK;
  }
  void *ws = nullptr;
  dsa_status s = scratch_for_current_device(&ws);
  if (s != DSA_OK) return s;
  const size_t ws_bytes = (size_t)DSA_NOALLOC_MAX_WORKSPACE;
  // dsa_decode_run zeroes the status block of the workspace before its
  // launch; the selection records and partials are written in full by the
  // kernels, so nothing else has to start at zero.
  s = dsa_decode_run(plan, ws, ws_bytes, q, q_stride_t, q_stride_h, swa_cache, swa_idx,
                     swa_idx_stride, swa_lens, extra_cache, extra_idx, extra_idx_stride,
                     extra_lens, sink, positions, cos_sin, cos_sin_rows, scale, out, lse, stream);
  if (s != DSA_OK) return s;
  s = dsa_decode_combine(plan, ws, ws_bytes, sink, out, lse, stream);
  if (s != DSA_OK) return s;
  if (device_status) {
    const cudaError_t e = cudaMemcpyAsync(device_status, ws, 4, cudaMemcpyDeviceToDevice,
                                          reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

}  // extern "C"
