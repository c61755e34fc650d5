/*
 * fa_noalloc.cu -- fa_fwd_splitkv_noalloc: the split-KV forward pass with its
 * workspace taken from a fixed buffer in the library's own device memory.
 *
 * The buffer is a file-scope __device__ array, so the CUDA runtime sets it
 * aside when this translation unit's module is loaded on a device; nothing
 * here calls cudaMalloc, cudaFree or any other allocating routine.  Its
 * address is looked up with the device current and cached per device for
 * the context it was found in.  This file is its own module so that callers
 * who never use the entry point never load the buffer (with the runtime's
 * lazy module loading).
 */
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fa_api.h"

namespace fa {
// Workspace size of a split run (defined beside the split entry point).
size_t split_workspace_bytes(int64_t B, int64_t H, int64_t S_q, int64_t D, int n_splits);
// The split entry point's host checks, apart from its workspace.
fa_status_t check_splitkv_args(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, int64_t B, int64_t H, int64_t H_kv, int64_t S_q,
                               int64_t S_kv, int64_t D, float scale, fa_layout_t layout,
                               fa_dtype_t dtype, const float* descale_q, const float* descale_k,
                               const float* descale_v, int n_splits);
// The calling thread's current context (made current if it has none), or null.
CUcontext current_context(int* dev_out);
}  // namespace fa

static_assert(FA_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte parts");

// The scratch: fp32 partial O and lse of one split run at a time per device.
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
struct Scratch {
  CUcontext ctx = nullptr;  // the context the address was looked up in
  void* addr = nullptr;
};
Scratch g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

// Address of the scratch in the calling thread's current context on the
// current device.  It is looked up (cudaGetSymbolAddress, with that device
// current) on the first call and again whenever the context differs from the
// one it was found in: a device reset, or a caller that switches contexts,
// loads the module anew at another address.
fa_status_t scratch_on_current_device(void** out) {
  int dev = 0;
  const CUcontext ctx = fa::current_context(&dev);
  if (!ctx || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  Scratch& s = g_scratch[dev];
  if (!s.addr || s.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
    s.ctx = ctx;
    s.addr = p;
  }
  *out = s.addr;
  return FA_OK;
}

}  // namespace

extern "C" fa_status_t fa_fwd_splitkv_noalloc(
    const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
    int64_t H_kv, int64_t S_q, int64_t S_kv, int64_t D, float scale, fa_layout_t layout,
    int causal, fa_dtype_t dtype, const float* descale_q, const float* descale_k,
    const float* descale_v, int n_splits, cudaStream_t stream) {
  // The host checks of fa_fwd_splitkv first (same statuses), then the
  // scratch's capacity; both before any CUDA call.
  const fa_status_t chk = fa::check_splitkv_args(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale,
                                                 layout, dtype, descale_q, descale_k, descale_v,
                                                 n_splits);
  if (chk != FA_OK) return chk;
  if (n_splits == 1)  // no partials: the whole pass writes o and lse directly
    return fa_fwd_splitkv(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout, causal, dtype,
                          descale_q, descale_k, descale_v, 1, nullptr, 0, stream);
  // Larger than the buffer: refused (the same problem runs through
  // fa_fwd_splitkv with a caller-owned workspace).
  const double rows = static_cast<double>(n_splits) * B * H * S_q;
  if (rows * (D + 1) * 4.0 > static_cast<double>(FA_NOALLOC_SCRATCH_BYTES) ||
      fa::split_workspace_bytes(B, H, S_q, D, n_splits) > FA_NOALLOC_SCRATCH_BYTES)
    return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const fa_status_t st = scratch_on_current_device(&scratch);
  if (st != FA_OK) return st;
  return fa_fwd_splitkv(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout, causal, dtype,
                        descale_q, descale_k, descale_v, n_splits, scratch,
                        FA_NOALLOC_SCRATCH_BYTES, stream);
}
