/*
 * fa_api.cu -- host side of libfa_b200 (see include/fa_api.h).
 *
 * Argument checks (all before any CUDA call), TMA descriptor encoding with
 * 64-bit strides and per-dimension bounds, schedule parameters, the launch,
 * and the device error word that bounded waits report into.
 *
 * The page "npu_flash_attention, from ATen down to the Cube unit" walks the
 * Ascend call through op registration, a tiling calculation that fails with
 * "UB overflow", allocation and task submission; here the whole of that is
 * one validation pass and one asynchronous kernel launch, and every failure
 * is a returned status.
 */
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <numeric>
#include <vector>

#include "../../include/fa_api.h"
#include "fa_bwd.cuh"
#include "fa_combine.cuh"
#include "fa_kernel.cuh"
#include "fa_seq_order.cuh"

// Explicit instantiations live in fa_inst_*.cu (compiled in parallel).
#define FA_FWD_EXTERN_ALL_MODES(D, DT)                    \
  FA_FWD_INSTANTIATE(extern, D, DT, fa::kModeDense)       \
  FA_FWD_INSTANTIATE(extern, D, DT, fa::kModeSplit)       \
  FA_FWD_INSTANTIATE(extern, D, DT, fa::kModeVarlen)      \
  FA_FWD_INSTANTIATE(extern, D, DT, fa::kModePaged)      \
  FA_FWD_INSTANTIATE(extern, D, DT, fa::kModePagedSplit)
FA_FWD_EXTERN_ALL_MODES(64, fa::kDtF16)
FA_FWD_EXTERN_ALL_MODES(128, fa::kDtF16)
FA_FWD_EXTERN_ALL_MODES(64, fa::kDtBF16)
FA_FWD_EXTERN_ALL_MODES(128, fa::kDtBF16)
FA_FWD_EXTERN_ALL_MODES(128, fa::kDtE4M3)
#undef FA_FWD_EXTERN_ALL_MODES

// Backward launchers live in fa_bwd_inst_*.cu.
FA_BWD_INSTANTIATE(extern, 64, fa::bwd::kF16)
FA_BWD_INSTANTIATE(extern, 128, fa::bwd::kF16)
FA_BWD_INSTANTIATE(extern, 64, fa::bwd::kBF16)
FA_BWD_INSTANTIATE(extern, 128, fa::bwd::kBF16)

// Device error word: bounded waits OR their error bits in here.
__device__ uint32_t g_fa_device_error = 0;

namespace {

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready = false;
  CUcontext ctx = nullptr;   // the context the facts below were looked up in
  int sm_count = 0;
  uint32_t* err_word = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

// cuCtxGetCurrent through the runtime's driver entry point (the library does
// not link libcuda directly).
PFN_cuCtxGetCurrent_v4000 ctx_get_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  return fn;
}

}  // namespace

namespace fa {
// The calling thread's current context, made current first if the thread has
// none.  Tensor-map encoding is a driver call that needs one, and a thread on
// which no CUDA runtime call has touched the device yet (a framework's worker
// thread, say) has none: the current device's primary context is then made
// current (cudaSetDevice on the device the thread already reports, which
// changes nothing the caller chose).  A context the caller made current --
// primary or not -- is left as it is.  Null if no context can be had.
CUcontext current_context(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  auto get = ctx_get_fn();
  if (!get) return nullptr;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return nullptr;
  if (!ctx) {
    if (cudaSetDevice(dev) != cudaSuccess || get(&ctx) != CUDA_SUCCESS) return nullptr;
  }
  if (dev_out) *dev_out = dev;
  return ctx;
}
}  // namespace fa

namespace {

// Per-device facts, looked up with that device current and kept until the
// thread's current context on that device changes (a device reset, or a
// caller that switches contexts, moves the module's symbols: the device
// error word is then looked up again).
fa_status_t device_info(DeviceInfo* out) {
  int dev = 0;
  const CUcontext ctx = fa::current_context(&dev);
  if (!ctx || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready || d.ctx != ctx) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FA_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_device_error) != cudaSuccess) return FA_ERR_CUDA;
    d.ctx = ctx;
    d.sm_count = sms;
    d.err_word = static_cast<uint32_t*>(p);
    d.ready = true;
  }
  *out = d;
  return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The last few tensor maps this thread encoded, by their arguments: a caller
// that runs the same shapes on the same buffers call after call (a training
// or decode loop) skips the encoding.  A map holds only the address, sizes
// and strides, so it stays valid for whatever the buffer holds.
struct MapKey {
  const void* ptr;
  int64_t B, H, S, D;
  int32_t dtype, layout;
  uint32_t box_rows, box_heads;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && B == o.B && H == o.H && S == o.S && D == o.D && dtype == o.dtype &&
           layout == o.layout && box_rows == o.box_rows && box_heads == o.box_heads;
  }
};
constexpr int kMapCache = 8;
struct MapCache {
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  bool used[kMapCache] = {};
  int next = 0;
};
thread_local MapCache t_maps;

bool make_map_encode(CUtensorMap* m, const void* ptr, fa_dtype_t dtype, fa_layout_t layout,
                     int64_t B, int64_t H, int64_t S, int64_t D, cuuint32_t box_rows,
                     cuuint32_t box_heads);

// 4-D tensor map over a [B,H,S,D] (BNSD) or [B,S,H,D] (BSND) tensor, boxes
// of 128 rows x 128 bytes, 128-byte swizzle, zero fill out of bounds.  The
// sequence dimension is its own map dimension, so rows >= S are never read
// (in BSND the bytes after row S-1 of batch b are batch b+1's rows).
bool make_map(CUtensorMap* m, const void* ptr, fa_dtype_t dtype, fa_layout_t layout, int64_t B,
              int64_t H, int64_t S, int64_t D, cuuint32_t box_rows = 128,
              cuuint32_t box_heads = 1) {
  const MapKey key{ptr, B, H, S, D, static_cast<int32_t>(dtype), static_cast<int32_t>(layout),
                   box_rows, box_heads};
  MapCache& c = t_maps;
  for (int i = 0; i < kMapCache; ++i) {
    if (c.used[i] && c.key[i] == key) {
      *m = c.map[i];
      return true;
    }
  }
  if (!make_map_encode(m, ptr, dtype, layout, B, H, S, D, box_rows, box_heads)) return false;
  c.key[c.next] = key;
  c.map[c.next] = *m;
  c.used[c.next] = true;
  c.next = (c.next + 1) % kMapCache;
  return true;
}

bool make_map_encode(CUtensorMap* m, const void* ptr, fa_dtype_t dtype, fa_layout_t layout,
                     int64_t B, int64_t H, int64_t S, int64_t D, cuuint32_t box_rows,
                     cuuint32_t box_heads) {
  auto enc = encode_fn();
  if (!enc) return false;
  const uint64_t eb = (dtype == FA_DTYPE_FP8E4M3) ? 1 : 2;
  const CUtensorMapDataType t = dtype == FA_DTYPE_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                : dtype == FA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  const cuuint32_t inner = static_cast<cuuint32_t>(128 / eb);
  if (layout == FA_LAYOUT_BNSD) {
    dims[0] = D; dims[1] = S; dims[2] = H; dims[3] = B;
    strides[0] = D * eb; strides[1] = S * D * eb; strides[2] = H * S * D * eb;
    box[0] = inner; box[1] = box_rows; box[2] = 1; box[3] = 1;
  } else {
    dims[0] = D; dims[1] = H; dims[2] = S; dims[3] = B;
    strides[0] = D * eb; strides[1] = H * D * eb; strides[2] = S * H * D * eb;
    box[0] = inner; box[1] = box_heads; box[2] = box_rows; box[3] = 1;
  }
  CUresult r = enc(m, t, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 partial-O map: [n, H, S, D] with n = n_splits * B, boxes of `box_rows`
// rows of `box_heads` heads x 32 columns (128 bytes), 128-byte swizzle.
bool make_map_f32(CUtensorMap* m, const void* ptr, int64_t n, int64_t H, int64_t S, int64_t D,
                  cuuint32_t box_rows = 32, cuuint32_t box_heads = 1) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(n)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D * 4), static_cast<cuuint64_t>(S * D * 4),
                           static_cast<cuuint64_t>(H * S * D * 4)};
  cuuint32_t box[4] = {32, box_rows, box_heads, 1}, estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Paged K/V cache [num_pages, page_size, H_kv, D]: map {D, H_kv, page_size,
// num_pages}, boxes of min(page_size, 128) rows x 128 bytes of one head of one
// page, 128-byte swizzle, zero fill out of bounds.
bool make_map_paged(CUtensorMap* m, const void* ptr, fa_dtype_t dtype, int64_t num_pages,
                    int64_t page_size, int64_t H_kv, int64_t D) {
  auto enc = encode_fn();
  if (!enc) return false;
  const uint64_t eb = (dtype == FA_DTYPE_FP8E4M3) ? 1 : 2;
  const CUtensorMapDataType t = dtype == FA_DTYPE_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                : dtype == FA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H_kv),
                        static_cast<cuuint64_t>(page_size), static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {D * eb, H_kv * D * eb, page_size * H_kv * D * eb};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), 1,
                       static_cast<cuuint32_t>(page_size < 128 ? page_size : 128), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, t, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A [B, H, S, D] tensor with element strides (batch, head, seq) and contiguous
// D, as a 4-D map {D, S, H, B} (the BNSD coordinate order whatever the memory
// order), boxes of `box_rows` rows x 128 bytes, 128-byte swizzle.
bool make_map_strided(CUtensorMap* m, const void* ptr, fa_dtype_t dtype, int64_t B, int64_t H,
                      int64_t S, int64_t D, const fa_strides_t& st, cuuint32_t box_rows = 128) {
  auto enc = encode_fn();
  if (!enc) return false;
  const uint64_t eb = (dtype == FA_DTYPE_FP8E4M3) ? 1 : 2;
  const CUtensorMapDataType t = dtype == FA_DTYPE_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                : dtype == FA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.seq) * eb, static_cast<cuuint64_t>(st.head) * eb,
                           static_cast<cuuint64_t>(st.batch) * eb};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, t, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The element strides of a dense tensor in one of the two layouts.
fa_strides_t dense_strides(fa_layout_t layout, int64_t H, int64_t S, int64_t D) {
  if (layout == FA_LAYOUT_BNSD) return fa_strides_t{H * S * D, S * D, D};
  return fa_strides_t{S * H * D, D, H * D};
}

// Strides a TMA map can use: positive, 16-byte multiples, below 2^40 bytes.
fa_status_t check_strides(const fa_strides_t* st, int n, fa_dtype_t dtype) {
  if (!st) return FA_ERR_INVALID_ARG;
  const int64_t eb = (dtype == FA_DTYPE_FP8E4M3) ? 1 : 2;
  for (int i = 0; i < n; ++i) {
    const int64_t v[3] = {st[i].batch, st[i].head, st[i].seq};
    for (int64_t x : v) {
      if (x < 1) return FA_ERR_INVALID_ARG;
      if ((x * eb) % 16 != 0) return FA_ERR_MISALIGNED;
      if (x > (int64_t(1) << 39) / eb) return FA_ERR_UNSUPPORTED;
    }
  }
  return FA_OK;
}

__global__ void fa_wait_probe_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t a = fa::smem_addr(&bar);
  if (threadIdx.x == 0) {
    fa::mbar_init(a, 1);
    abort_flag = 0;
    fa::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const fa::WaitCtl wc{limit_ns, err, &abort_flag};
    (void)fa::mbar_wait(a, 0u, wc);  // nothing ever arrives: must time out
  }
}

}  // namespace

extern "C" {

const char* fa_version(void) { return "0.1.0"; }

const char* fa_status_string(fa_status_t s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

void fa_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns ? ns : kDefaultWaitLimitNs);
}

}  // extern "C"

namespace fa {
// Workspace of a split run: fp32 partial O [n_splits, B, H, S_q, D], then fp32
// partial lse [n_splits, B, H, S_q]; each part 256-byte aligned.  (Also used
// by the no-allocation entry point in fa_noalloc.cu.)
size_t split_workspace_bytes(int64_t B, int64_t H, int64_t S_q, int64_t D, int n_splits) {
  const size_t rows = static_cast<size_t>(n_splits) * B * H * S_q;
  const size_t o_bytes = (rows * D * 4 + 255) / 256 * 256;
  return o_bytes + (rows * 4 + 255) / 256 * 256;
}
// fa_fwd_paged_split's workspace: the sequence order (int32 [n_seqs], when
// n_seqs <= kMaxOrderedSeqs), then the split partials (n_splits > 1); each
// part 256-byte aligned.
size_t order_bytes(int64_t n_seqs) {
  return n_seqs <= kMaxOrderedSeqs ? (static_cast<size_t>(n_seqs) * 4 + 255) / 256 * 256 : 0;
}
size_t paged_split_workspace_bytes(int64_t H, int64_t total_q, int64_t D, int n_splits,
                                   int64_t n_seqs) {
  return order_bytes(n_seqs) + (n_splits > 1 ? split_workspace_bytes(1, H, total_q, D, n_splits) : 0);
}
}  // namespace fa
using fa::split_workspace_bytes;

namespace {

// Checks shared by every forward entry point (all before any CUDA call).
fa_status_t check_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv, int64_t D,
                       float scale, fa_layout_t layout, fa_dtype_t dtype, const float* descale_q,
                       const float* descale_k, const float* descale_v) {
  // ---- host-side checks: nothing below touches the device until they pass
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S_q < 1 || S_kv < 1 || D < 1) return FA_ERR_INVALID_ARG;
  if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
  if (layout != FA_LAYOUT_BNSD && layout != FA_LAYOUT_BSND) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP8E4M3)
    return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP8E4M3 && (descale_q || descale_k || descale_v)) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_DTYPE_FP8E4M3 && D != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  if (dtype == FA_DTYPE_FP8E4M3 &&
      (!aligned(descale_q, 4) || !aligned(descale_k, 4) || !aligned(descale_v, 4)))
    return FA_ERR_MISALIGNED;
  // Limits: row coordinates are 32-bit in the TMA descriptors, the unit count
  // is a 32-bit index, and TMA strides must stay below 2^40 bytes.
  const int64_t kMaxSeq = (int64_t(1) << 31) - 256;
  if (S_q > kMaxSeq || S_kv > kMaxSeq || B > INT32_MAX || H > INT32_MAX) return FA_ERR_UNSUPPORTED;
  const int64_t eb = (dtype == FA_DTYPE_FP8E4M3) ? 1 : 2;
  const int64_t n_qtiles = (S_q + 127) / 128;
  const int64_t n_pairs = (n_qtiles + 1) / 2;
  if (B * H > INT32_MAX / n_pairs) return FA_ERR_UNSUPPORTED;
  const int64_t max_s = S_q > S_kv ? S_q : S_kv;
  if ((double)H * (double)max_s * (double)D * (double)eb >= 1099511627776.0)
    return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

constexpr int kMaxSplits = 32;

}  // namespace

namespace fa {
// Host checks of a split-KV call, apart from its workspace (all before any
// CUDA call); fa_fwd_splitkv and the no-allocation entry point share them.
fa_status_t check_splitkv_args(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, int64_t B, int64_t H, int64_t H_kv, int64_t S_q,
                               int64_t S_kv, int64_t D, float scale, fa_layout_t layout,
                               fa_dtype_t dtype, const float* descale_q, const float* descale_k,
                               const float* descale_v, int n_splits) {
  const fa_status_t st = check_args(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout,
                                    dtype, descale_q, descale_k, descale_v);
  if (st != FA_OK) return st;
  if (n_splits < 1) return FA_ERR_INVALID_ARG;
  if (n_splits > kMaxSplits) return FA_ERR_UNSUPPORTED;
  if (n_splits > 1 && static_cast<double>(n_splits) * B * H * S_q * ((S_q + 127) / 128) > 2e9)
    return FA_ERR_UNSUPPORTED;
  return FA_OK;
}
}  // namespace fa

namespace {

// The busiest CTA's load under the kernels' static schedule: units in groups
// of g heads, rank-major inside a group (heads vary fastest; rank r costs
// cost[r] key blocks -- or query tiles -- plus one for the unit's fixed
// cost), unit w * grid + b to CTA b in even rounds and to CTA grid - 1 - b in
// odd ones.
int64_t snake_makespan(int64_t n_heads, const std::vector<int64_t>& cost, int64_t g, int grid,
                       std::vector<int64_t>& load) {
  const int64_t n_ranks = static_cast<int64_t>(cost.size());
  load.assign(static_cast<size_t>(grid), 0);
  const int64_t per_group = g * n_ranks, units = n_heads * n_ranks;
  for (int64_t u = 0; u < units; ++u) {
    const int64_t gi = u / per_group, r = u - gi * per_group;
    const int64_t heads = std::min(g, n_heads - gi * g);
    const int64_t w = u / grid, b = u - w * grid;
    load[static_cast<size_t>((w & 1) ? grid - 1 - b : b)] += cost[static_cast<size_t>(r / heads)] + 1;
  }
  return *std::max_element(load.begin(), load.end());
}

// Heads per scheduling group of a causal pass (forward, or one of the
// backward's kernels).  The data the heads in flight together share should
// fit in L2: about 48 MB a group (bytes_per_head each).  The longest units
// come first inside each group, so a group whose units are not a whole
// number of snake round pairs (g * ranks a multiple of 2 * grid) leaves the
// rounds that straddle a group boundary uneven.  Such groups -- multiples of
// g0 = 2 * grid / gcd(2 * grid, ranks), up to 96 MB -- are weighed against
// the 48 MB group with the schedule above and taken when the busiest CTA is
// lighter (up to a million units).  Measured on bf16, D = 128 causal passes
// against the 48 MB rule:
// forward 4 x 32 x 4096 455 -> 414 us (19 heads), 2 x 32 x 8192 828 -> 761 us
// (19), 8 x 32 x 4096 851-864 -> 809-812 us (38); backward 4 x 32 x 4096
// 1542-1573 -> 1479-1499 us, 8 x 32 x 4096 3249-3340 -> 3028-3094 us (19).
// Choices are cached per shape.
int64_t balanced_group(int64_t n_heads, const std::vector<int64_t>& cost, int64_t bytes_per_head,
                       int grid, bool balance) {
  const int64_t per_head = bytes_per_head > 0 ? bytes_per_head : 1;
  int64_t group = std::min(std::max<int64_t>((48ll << 20) / per_head, 1), n_heads);
  const int64_t n_ranks = static_cast<int64_t>(cost.size());
  if (!balance || grid < 1 || n_ranks < 1) return group;
  const int64_t g_max = std::min(std::max<int64_t>((96ll << 20) / per_head, 1), n_heads);
  const int64_t g0 = 2 * grid / std::gcd<int64_t>(2 * grid, n_ranks);
  // (The model walks every unit: beyond a million units the first call of a
  // shape would spend milliseconds on it, so those keep the 48 MB group.)
  if (g0 > g_max || n_heads * n_ranks > (int64_t(1) << 20)) return group;
  static std::mutex mu;
  static std::map<std::vector<int64_t>, int64_t> cache;
  std::vector<int64_t> key = {n_heads, per_head, grid};
  key.insert(key.end(), cost.begin(), cost.end());
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  std::vector<int64_t> load;
  int64_t best = snake_makespan(n_heads, cost, group, grid, load);
  for (int64_t g = g0, tries = 0; g <= g_max && tries < 8; g += g0, ++tries) {
    const int64_t m = snake_makespan(n_heads, cost, g, grid, load);
    if (m < best) {
      best = m;
      group = g;
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() >= 1024) cache.clear();
  cache[key] = group;
  return group;
}

// Key blocks that query tile t needs under the top-left causal mask (0 for a
// tile past S_q).
int64_t causal_tile_blocks(int64_t t, int64_t S_q, int64_t S_kv) {
  if (t * 128 >= S_q) return 0;
  return std::min(std::min(t * 128 + 127, S_q - 1), S_kv - 1) / 128 + 1;
}

// The forward pass, whole (n_splits = 1: o / lse written directly) or split
// over the keys (n_splits > 1: partials in `workspace`, then the merge).
fa_status_t run_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                        int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv, int64_t D,
                        float scale, fa_layout_t layout, int causal, fa_dtype_t dtype,
                        const float* descale_q, const float* descale_k, const float* descale_v,
                        int n_splits, void* workspace, cudaStream_t stream,
                        const fa_strides_t* strides = nullptr) {
  const int64_t eb = (dtype == FA_DTYPE_FP8E4M3) ? 1 : 2;
  const int64_t n_pairs = ((S_q + 127) / 128 + 1) / 2;
  DeviceInfo dev;
  if (device_info(&dev) != FA_OK) return FA_ERR_CUDA;

  // O: the output dtype (16-bit; bf16 for fp8 inputs), boxes of 32 rows (one
  // warp's rows) x 128 bytes, written by TMA stores.
  CUtensorMap mq, mk, mv, mo;
  const fa_dtype_t odt = (dtype == FA_DTYPE_F16) ? FA_DTYPE_F16 : FA_DTYPE_BF16;
  if (strides) {  // q, k, v, o with their own strides: BNSD coordinate order
    if (!make_map_strided(&mq, q, dtype, B, H, S_q, D, strides[0]) ||
        !make_map_strided(&mk, k, dtype, B, H_kv, S_kv, D, strides[1]) ||
        !make_map_strided(&mv, v, dtype, B, H_kv, S_kv, D, strides[2]) ||
        !make_map_strided(&mo, o, odt, B, H, S_q, D, strides[3], 32))
      return FA_ERR_CUDA;
    layout = FA_LAYOUT_BNSD;
  } else if (!make_map(&mq, q, dtype, layout, B, H, S_q, D) ||
             !make_map(&mk, k, dtype, layout, B, H_kv, S_kv, D) ||
             !make_map(&mv, v, dtype, layout, B, H_kv, S_kv, D) ||
             !make_map(&mo, o, odt, layout, B, H, S_q, D, 32)) {
    return FA_ERR_CUDA;
  }
  // Split partials: fp32 [n_splits * B, H, S_q, D] (BNSD), boxes of 32 rows x
  // 32 fp32 columns.
  CUtensorMap mop = mo;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  if (n_splits > 1) {
    o_part = static_cast<float*>(workspace);
    const size_t rows = static_cast<size_t>(n_splits) * B * H * S_q;
    lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + (rows * D * 4 + 255) / 256 * 256);
    if (!make_map_f32(&mop, o_part, n_splits * B, H, S_q, D)) return FA_ERR_CUDA;
  }

  fa::KernelParams p = {};
  p.B = B; p.H = H; p.S_q = S_q; p.S_kv = S_kv;
  p.kv_group = static_cast<int32_t>(H / H_kv);
  p.n_kv_blocks = static_cast<int32_t>((S_kv + 127) / 128);
  p.n_pairs = static_cast<int32_t>(n_pairs);
  p.num_units = static_cast<int32_t>(B * H * n_pairs * n_splits);
  p.n_splits = n_splits;
  p.lse_part = lse_part;
  // Causal: heads in scheduling groups, longest pairs first inside each.
  // (K/V bytes one query head brings into L2: a key/value head is shared by
  // H / H_kv consecutive query heads.)
  // When the K/V of all heads is at most 192 MB (about the size of L2)
  // grouping buys little locality, and with few groups the longest-first
  // order that restarts in each group leaves CTAs unevenly loaded (1 x 32
  // heads x 8192 bf16: 429 us grouped by 12 heads, 382 us as one group): one
  // group then.  Split passes keep the 48 MB rule.
  int64_t group = 1;
  if (causal) {
    const int64_t kv_bytes = 2 * S_kv * D * eb * H_kv / H;
    if (B * H * kv_bytes <= (192ll << 20)) {
      group = B * H;
    } else {
      std::vector<int64_t> cost(static_cast<size_t>(n_pairs));
      for (int64_t r = 0; r < n_pairs; ++r) {
        const int64_t pair = n_pairs - 1 - r;
        cost[static_cast<size_t>(r)] = std::max(causal_tile_blocks(2 * pair, S_q, S_kv),
                                                causal_tile_blocks(2 * pair + 1, S_q, S_kv));
      }
      const int64_t sched_grid = std::min<int64_t>(B * H * n_pairs, dev.sm_count);
      group = balanced_group(B * H, cost, kv_bytes, static_cast<int>(sched_grid), n_splits == 1);
    }
  }
  p.group_heads = static_cast<int32_t>(group);
  p.layout = static_cast<int32_t>(layout);
  p.causal = causal ? 1 : 0;
  // A negative scale: the products give -Q K^T and the softmax takes |scale|.
  p.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.neg_scale = scale < 0.0f ? 1 : 0;
  p.descale_q = descale_q;
  p.descale_k = descale_k;
  p.descale_v = descale_v;
  p.o = o;
  p.lse = lse;
  p.err = dev.err_word;
  p.wait_limit_ns = g_wait_limit_ns.load();
  // Without a mask all units cost the same, and a last round of T < SMs / 2
  // units leaves the other SMs idle for a whole unit: its units become 2T
  // single-tile units whose key blocks are split over both tile slots, so
  // that round takes about half as long (4 x 32 x 4096: 2048 units, T = 72).
  p.solo_base = p.num_units;
  if (!causal && n_splits == 1) {
    const int64_t units = p.num_units, tail = units % dev.sm_count;
    if (tail > 0 && 2 * tail <= dev.sm_count && units + tail < INT32_MAX - 2 * dev.sm_count) {
      p.solo_base = static_cast<int32_t>(units - tail);
      p.num_units = static_cast<int32_t>(units + tail);
    }
  }

  const int grid = static_cast<int>(p.num_units < dev.sm_count ? p.num_units : dev.sm_count);
  const bool sp = n_splits > 1;
  cudaError_t e;
#define FA_LAUNCH(DD, DTY)                                                                     \
  (sp ? fa::launch_fa_fwd<DD, DTY, fa::kModeSplit>(mq, mk, mv, mo, mop, p, grid, stream)       \
      : fa::launch_fa_fwd<DD, DTY, fa::kModeDense>(mq, mk, mv, mo, mop, p, grid, stream))
  if (dtype == FA_DTYPE_F16)
    e = (D == 64) ? FA_LAUNCH(64, fa::kDtF16) : FA_LAUNCH(128, fa::kDtF16);
  else if (dtype == FA_DTYPE_BF16)
    e = (D == 64) ? FA_LAUNCH(64, fa::kDtBF16) : FA_LAUNCH(128, fa::kDtBF16);
  else
    e = FA_LAUNCH(128, fa::kDtE4M3);
#undef FA_LAUNCH
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (n_splits > 1) {
    fa::CombineParams c = {};
    c.o_part = o_part;
    c.lse_part = lse_part;
    c.o = o;
    c.lse = lse;
    c.B = B; c.H = H; c.S_q = S_q;
    c.D = static_cast<int32_t>(D);
    c.n_splits = n_splits;
    c.layout = static_cast<int32_t>(layout);
    c.out_f16 = dtype == FA_DTYPE_F16 ? 1 : 0;
    if (fa::launch_fa_combine(c, dev.sm_count, stream) != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status_t fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                       int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv, int64_t D,
                       float scale, fa_layout_t layout, int causal, fa_dtype_t dtype,
                       const float* descale_q, const float* descale_k, const float* descale_v,
                       cudaStream_t stream) {
  const fa_status_t st = check_args(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout,
                                    dtype, descale_q, descale_k, descale_v);
  if (st != FA_OK) return st;
  return run_forward(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout, causal, dtype,
                     descale_q, descale_k, descale_v, 1, nullptr, stream);
}

fa_status_t fa_fwd_splitkv_plan(int64_t B, int64_t H, int64_t S_q, int64_t S_kv, int64_t D,
                                int* n_splits, size_t* workspace_bytes) {
  if (!n_splits || !workspace_bytes) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S_q < 1 || S_kv < 1 || D < 1) return FA_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (device_info(&dev) != FA_OK) return FA_ERR_CUDA;
  const int64_t units = B * H * (((S_q + 127) / 128 + 1) / 2);
  const int64_t kv_blocks = (S_kv + 127) / 128;
  // Waves of work items times the blocks each item walks, plus about three
  // blocks' worth of fixed cost per item (Q load, pipeline fill, partial
  // write); the smallest estimate wins, ties to fewer splits.
  int64_t splits = 1, best = -1;
  for (int64_t sp = 1; sp <= kMaxSplits && sp <= (kv_blocks > 1 ? kv_blocks / 2 : 1); ++sp) {
    const int64_t waves = (units * sp + dev.sm_count - 1) / dev.sm_count;
    const int64_t cost = waves * ((kv_blocks + sp - 1) / sp + 3);
    if (best < 0 || cost < best) {
      best = cost;
      splits = sp;
    }
  }
  *n_splits = static_cast<int>(splits);
  *workspace_bytes = splits > 1 ? split_workspace_bytes(B, H, S_q, D, static_cast<int>(splits)) : 0;
  return FA_OK;
}

fa_status_t fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                           int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv,
                           int64_t D, float scale, fa_layout_t layout, int causal,
                           fa_dtype_t dtype, const float* descale_q, const float* descale_k,
                           const float* descale_v, int n_splits, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  const fa_status_t st = fa::check_splitkv_args(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale,
                                                layout, dtype, descale_q, descale_k, descale_v,
                                                n_splits);
  if (st != FA_OK) return st;
  if (n_splits > 1) {
    if (!workspace || workspace_bytes < split_workspace_bytes(B, H, S_q, D, n_splits))
      return FA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  }
  return run_forward(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout, causal, dtype,
                     descale_q, descale_k, descale_v, n_splits, workspace, stream);
}

fa_status_t fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                           int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv,
                           int64_t D, const fa_strides_t* strides, float scale, int causal,
                           fa_dtype_t dtype, const float* descale_q, const float* descale_k,
                           const float* descale_v, cudaStream_t stream) {
  fa_status_t st = check_args(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, FA_LAYOUT_BNSD,
                              dtype, descale_q, descale_k, descale_v);
  if (st != FA_OK) return st;
  st = check_strides(strides, 4, dtype);
  if (st != FA_OK) return st;
  return run_forward(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, FA_LAYOUT_BNSD, causal,
                     dtype, descale_q, descale_k, descale_v, 1, nullptr, stream, strides);
}

fa_status_t fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                   int64_t H, int64_t S_q, int64_t S_kv, int64_t D, float scale,
                   fa_layout_t layout, int causal, fa_dtype_t dtype, const float* descale_q,
                   const float* descale_k, const float* descale_v, cudaStream_t stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, S_q, S_kv, D, scale, layout, causal, dtype,
                    descale_q, descale_k, descale_v, stream);
}

fa_status_t fa_last_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  DeviceInfo dev;
  if (device_info(&dev) != FA_OK) return FA_ERR_CUDA;
  uint32_t word = 0, zero = 0;
  if (cudaMemcpy(&word, dev.err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  if (cudaMemcpy(dev.err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return FA_ERR_CUDA;
  if (word & fa::kErrTimeout) return FA_ERR_DEVICE_TIMEOUT;
  return word ? FA_ERR_CUDA : FA_OK;
}

fa_status_t fa_probe_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  DeviceInfo dev;
  if (device_info(&dev) != FA_OK) return FA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  if (cudaLaunchKernelEx(&cfg, fa_wait_probe_kernel, dev.err_word,
                         static_cast<uint64_t>(limit_ns ? limit_ns : 1000000ull)) != cudaSuccess)
    return FA_ERR_CUDA;
  return fa_last_device_error(stream);
}

}  // extern "C"

namespace {

// Backward workspace: lse * log2(e), then rowsum(dO * O), each fp32
// [B * H, S_q rounded up to 128], 256-byte aligned.
size_t bwd_workspace_bytes(int64_t B, int64_t H, int64_t S_q) {
  const size_t rows = static_cast<size_t>(B) * H * ((S_q + 127) / 128 * 128);
  return 2 * ((rows * 4 + 255) / 256 * 256);
}

}  // namespace

namespace {

// The backward pass; strides (q, k, v, o, dout, dq, dk, dv) or NULL for the
// dense layout.
fa_status_t run_backward(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv, int64_t D,
                         float scale, fa_layout_t layout, int causal, fa_dtype_t dtype,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream,
                         const fa_strides_t* strides) {
  fa_status_t st = check_args(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout, dtype,
                              nullptr, nullptr, nullptr);
  if (st != FA_OK) return st;
  if (!dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (dtype == FA_DTYPE_FP8E4M3) return FA_ERR_UNSUPPORTED;
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return FA_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < bwd_workspace_bytes(B, H, S_q)) return FA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  const int64_t n_q = (S_q + 127) / 128, n_kv = (S_kv + 127) / 128;
  if (B * H > INT32_MAX / n_q || B * H_kv > INT32_MAX / n_kv) return FA_ERR_UNSUPPORTED;

  DeviceInfo dev;
  if (device_info(&dev) != FA_OK) return FA_ERR_CUDA;
  CUtensorMap mq, mk, mv, mdo, mdk, mdv;
  fa_strides_t ts[8];  // q, k, v, o, dout, dq, dk, dv
  if (strides) {
    for (int i = 0; i < 8; ++i) ts[i] = strides[i];
    if (!make_map_strided(&mq, q, dtype, B, H, S_q, D, ts[0]) ||
        !make_map_strided(&mk, k, dtype, B, H_kv, S_kv, D, ts[1]) ||
        !make_map_strided(&mv, v, dtype, B, H_kv, S_kv, D, ts[2]) ||
        !make_map_strided(&mdo, dout, dtype, B, H, S_q, D, ts[4]) ||
        !make_map_strided(&mdk, dk, dtype, B, H_kv, S_kv, D, ts[6], 16) ||
        !make_map_strided(&mdv, dv, dtype, B, H_kv, S_kv, D, ts[7], 16))
      return FA_ERR_CUDA;
    layout = FA_LAYOUT_BNSD;  // the maps take BNSD coordinates
  } else {
    const fa_strides_t sq = dense_strides(layout, H, S_q, D), sk = dense_strides(layout, H_kv, S_kv, D);
    const fa_strides_t dense[8] = {sq, sk, sk, sq, sq, sq, sk, sk};
    for (int i = 0; i < 8; ++i) ts[i] = dense[i];
    if (!make_map(&mq, q, dtype, layout, B, H, S_q, D) ||
        !make_map(&mk, k, dtype, layout, B, H_kv, S_kv, D) ||
        !make_map(&mv, v, dtype, layout, B, H_kv, S_kv, D) ||
        !make_map(&mdo, dout, dtype, layout, B, H, S_q, D) ||
        !make_map(&mdk, dk, dtype, layout, B, H_kv, S_kv, D, 16) ||
        !make_map(&mdv, dv, dtype, layout, B, H_kv, S_kv, D, 16))
      return FA_ERR_CUDA;
  }

  const int64_t S_q_pad = n_q * 128;
  const size_t half_ws = bwd_workspace_bytes(B, H, S_q) / 2;
  float* lse2 = static_cast<float*>(workspace);
  float* dsum = reinterpret_cast<float*>(static_cast<char*>(workspace) + half_ws);

  fa::bwd::BwdParams p = {};
  p.B = B; p.H = H; p.H_kv = H_kv; p.S_q = S_q; p.S_kv = S_kv;
  p.S_q_pad = S_q_pad;
  p.kv_group = static_cast<int32_t>(H / H_kv);
  p.n_q_tiles = static_cast<int32_t>(n_q);
  p.n_kv_tiles = static_cast<int32_t>(n_kv);
  p.layout = static_cast<int32_t>(layout);
  p.causal = causal ? 1 : 0;
  // A negative scale: the products give -Q K^T and the softmax takes |scale|.
  p.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.neg_scale = scale < 0.0f ? 1 : 0;
  p.scale = scale;
  p.lse2 = lse2;
  p.dsum = dsum;
  p.err = dev.err_word;
  p.wait_limit_ns = g_wait_limit_ns.load();
  const fa_strides_t* sp3[3] = {&ts[3], &ts[4], &ts[5]};
  int64_t* dst3[3] = {p.o_st, p.do_st, p.dq_st};
  for (int i = 0; i < 3; ++i) {
    dst3[i][0] = sp3[i]->batch;
    dst3[i][1] = sp3[i]->head;
    dst3[i][2] = sp3[i]->seq;
  }

  // dQ: one unit per (query head, query tile); causal runs group heads so
  // that the K/V in flight fit in L2, at a size that keeps the static
  // schedule balanced (balanced_group, as the forward).
  fa::bwd::BwdParams pq = p;
  pq.num_units = static_cast<int32_t>(B * H * n_q);
  int64_t gq = 1;
  if (causal) {
    std::vector<int64_t> cost(static_cast<size_t>(n_q));
    for (int64_t r = 0; r < n_q; ++r)
      cost[static_cast<size_t>(r)] = causal_tile_blocks(n_q - 1 - r, S_q, S_kv);
    gq = balanced_group(B * H, cost, 2 * S_kv * D * 2 * H_kv / H,
                        static_cast<int>(std::min<int64_t>(B * H * n_q, dev.sm_count)), true);
  }
  pq.group_heads = static_cast<int32_t>(gq);
  // dK / dV: one unit per (key/value head, key tile); heads grouped so that
  // the Q / dO their query heads stream fit in L2 (balanced_group).
  fa::bwd::BwdParams pk = p;
  pk.num_units = static_cast<int32_t>(B * H_kv * n_kv);
  int64_t gk = 1;
  if (causal) {
    // key tile j is seen by query tiles j .. n_q - 1 of each of its query heads
    std::vector<int64_t> cost(static_cast<size_t>(n_kv));
    for (int64_t j = 0; j < n_kv; ++j)
      cost[static_cast<size_t>(j)] = std::max<int64_t>(0, n_q - j) * (H / H_kv);
    gk = balanced_group(B * H_kv, cost, 2 * S_q * D * 2 * (H / H_kv),
                        static_cast<int>(std::min<int64_t>(B * H_kv * n_kv, dev.sm_count)), true);
  }
  pk.group_heads = static_cast<int32_t>(gk);

  const int grid_q = static_cast<int>(pq.num_units < dev.sm_count ? pq.num_units : dev.sm_count);
  const int grid_k = static_cast<int>(pk.num_units < dev.sm_count ? pk.num_units : dev.sm_count);
  const int64_t prep_threads = B * H * S_q_pad * (D / 8);
  const int64_t prep_blocks = (prep_threads + 255) / 256;
  const int grid_p = static_cast<int>(prep_blocks < 8ll * dev.sm_count ? prep_blocks : 8ll * dev.sm_count);
  cudaError_t e;
  if (dtype == FA_DTYPE_F16)
    e = (D == 64) ? fa::bwd::launch_fa_bwd<64, fa::bwd::kF16>(mq, mk, mv, mdo, dq, mdk, mdv, o, dout,
                                                              lse, lse2, dsum, pq, pk, grid_q,
                                                              grid_k, grid_p, stream)
                  : fa::bwd::launch_fa_bwd<128, fa::bwd::kF16>(mq, mk, mv, mdo, dq, mdk, mdv, o,
                                                               dout, lse, lse2, dsum, pq, pk,
                                                               grid_q, grid_k, grid_p, stream);
  else
    e = (D == 64) ? fa::bwd::launch_fa_bwd<64, fa::bwd::kBF16>(mq, mk, mv, mdo, dq, mdk, mdv, o,
                                                               dout, lse, lse2, dsum, pq, pk,
                                                               grid_q, grid_k, grid_p, stream)
                  : fa::bwd::launch_fa_bwd<128, fa::bwd::kBF16>(mq, mk, mv, mdo, dq, mdk, mdv, o,
                                                                dout, lse, lse2, dsum, pq, pk,
                                                                grid_q, grid_k, grid_p, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

fa_status_t fa_bwd_workspace_size(int64_t B, int64_t H, int64_t S_q, size_t* workspace_bytes) {
  if (!workspace_bytes || B < 1 || H < 1 || S_q < 1) return FA_ERR_INVALID_ARG;
  *workspace_bytes = bwd_workspace_bytes(B, H, S_q);
  return FA_OK;
}

fa_status_t fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H,
                   int64_t H_kv, int64_t S_q, int64_t S_kv, int64_t D, float scale,
                   fa_layout_t layout, int causal, fa_dtype_t dtype, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  return run_backward(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S_q, S_kv, D, scale, layout,
                      causal, dtype, workspace, workspace_bytes, stream, nullptr);
}

fa_status_t fa_bwd_strided(const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv,
                           int64_t D, const fa_strides_t* strides, float scale, int causal,
                           fa_dtype_t dtype, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  const fa_status_t st = check_strides(strides, 8, dtype);
  if (st != FA_OK) return st;
  return run_backward(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S_q, S_kv, D, scale,
                      FA_LAYOUT_BNSD, causal, dtype, workspace, workspace_bytes, stream, strides);
}

}  // extern "C"

namespace {

// GQA packing: the query heads that share a key/value head fill one tile
// together (2^shift heads x 128 >> shift tokens), so a K/V block is read
// once for all of them -- what makes decoding (one token per sequence) use
// more than one row of the 128.
int q_pack_shift(int64_t H, int64_t H_kv) {
  const int64_t g = H / H_kv;
  int shift = 0;
  if (g > 1 && g <= 32 && (g & (g - 1)) == 0)
    while ((int64_t(1) << shift) < g) ++shift;
  return shift;
}

// Varlen and paged forward passes: packed queries [total_q, H, D], one unit
// per (sequence, head, pair of 128-row query tiles up to max_seqlen_q).
fa_status_t run_var(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int32_t* cu_q, const int32_t* cu_k, const int32_t* seqused_k,
                    const int32_t* block_table, int64_t n_seqs, int64_t max_pages,
                    int64_t page_size, int64_t num_pages, int64_t total_q, int64_t total_k,
                    int64_t max_seqlen_q, int64_t H, int64_t H_kv, int64_t D, float scale,
                    int causal, fa_dtype_t dtype, const float* descale_q, const float* descale_k,
                    const float* descale_v, cudaStream_t stream, int n_splits = 1,
                    void* workspace = nullptr, size_t workspace_bytes = 0) {
  const bool paged = block_table != nullptr;
  // ---- host-side checks: nothing below touches the device until they pass
  if (!q || !k || !v || !o || !lse || !cu_q) return FA_ERR_INVALID_ARG;
  if (paged ? !seqused_k : !cu_k) return FA_ERR_INVALID_ARG;
  if (n_seqs < 1 || total_q < 0 || max_seqlen_q < 1 || H < 1 || D < 1) return FA_ERR_INVALID_ARG;
  if (!paged && total_k < 0) return FA_ERR_INVALID_ARG;
  if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
  if (causal < 0 || causal > 2) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP8E4M3)
    return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP8E4M3 && (descale_q || descale_k || descale_v)) return FA_ERR_INVALID_ARG;
  if (paged) {
    if (max_pages < 1 || num_pages < 1 || page_size < 16) return FA_ERR_INVALID_ARG;
    if (!((page_size <= 128 && 128 % page_size == 0) || (page_size > 128 && page_size % 128 == 0)))
      return FA_ERR_UNSUPPORTED;
  }
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_DTYPE_FP8E4M3 && D != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(cu_q, 4) || !aligned(cu_k, 4) || !aligned(seqused_k, 4) || !aligned(block_table, 4))
    return FA_ERR_MISALIGNED;
  if (dtype == FA_DTYPE_FP8E4M3 &&
      (!aligned(descale_q, 4) || !aligned(descale_k, 4) || !aligned(descale_v, 4)))
    return FA_ERR_MISALIGNED;
  const int64_t kMaxRows = (int64_t(1) << 31) - 256;
  if (total_q > kMaxRows || total_k > kMaxRows || max_seqlen_q > kMaxRows || H > INT32_MAX ||
      n_seqs > INT32_MAX - 1 || max_pages > INT32_MAX || num_pages > INT32_MAX ||
      page_size > 65536 || max_pages * page_size > kMaxRows)
    return FA_ERR_UNSUPPORTED;
  const int shift = q_pack_shift(H, H_kv);
  const int64_t toks = 128 >> shift;
  const int64_t n_pairs = ((max_seqlen_q + toks - 1) / toks + 1) / 2;
  if (n_seqs * (H >> shift) > INT32_MAX / n_pairs) return FA_ERR_UNSUPPORTED;
  if (n_splits < 1) return FA_ERR_INVALID_ARG;
  if (n_splits > kMaxSplits) return FA_ERR_UNSUPPORTED;
  if (n_splits > 1 && !workspace) return FA_ERR_INVALID_ARG;
  if (workspace) {  // fa_fwd_paged_split: sequence order, then split partials
    if (workspace_bytes < fa::paged_split_workspace_bytes(H, total_q, D, n_splits, n_seqs))
      return FA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  }
  if (n_splits > 1 && static_cast<double>(n_splits) * n_seqs * (H >> shift) * n_pairs > 2e9)
    return FA_ERR_UNSUPPORTED;
  if (total_q == 0) return FA_OK;  // no query rows: nothing to compute or write

  DeviceInfo dev;
  if (device_info(&dev) != FA_OK) return FA_ERR_CUDA;
  const fa_dtype_t odt = (dtype == FA_DTYPE_F16) ? FA_DTYPE_F16 : FA_DTYPE_BF16;
  CUtensorMap mq, mk, mv, mo;
  bool ok = make_map(&mq, q, dtype, FA_LAYOUT_BSND, 1, H, total_q, D,
                     static_cast<cuuint32_t>(toks), static_cast<cuuint32_t>(1 << shift)) &&
            make_map(&mo, o, odt, FA_LAYOUT_BSND, 1, H, total_q, D,
                     static_cast<cuuint32_t>(32 >> shift), static_cast<cuuint32_t>(1 << shift));
  if (paged)
    ok = ok && make_map_paged(&mk, k, dtype, num_pages, page_size, H_kv, D) &&
         make_map_paged(&mv, v, dtype, num_pages, page_size, H_kv, D);
  else
    ok = ok && make_map(&mk, k, dtype, FA_LAYOUT_BSND, 1, H_kv, total_k > 0 ? total_k : 1, D) &&
         make_map(&mv, v, dtype, FA_LAYOUT_BSND, 1, H_kv, total_k > 0 ? total_k : 1, D);
  // Split partials: fp32 O [n_splits, H, total_q, D] then fp32 lse
  // [n_splits, H, total_q]; a partial box holds the packed tile's heads x
  // tokens.
  CUtensorMap mop = mo;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  int32_t* seq_order = nullptr;
  if (workspace && n_seqs <= fa::kMaxOrderedSeqs) seq_order = static_cast<int32_t*>(workspace);
  if (n_splits > 1) {
    o_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + fa::order_bytes(n_seqs));
    const size_t rows = static_cast<size_t>(n_splits) * H * total_q;
    lse_part = reinterpret_cast<float*>(reinterpret_cast<char*>(o_part) + (rows * D * 4 + 255) / 256 * 256);
    ok = ok && make_map_f32(&mop, o_part, n_splits, H, total_q, D,
                            static_cast<cuuint32_t>(32 >> shift), static_cast<cuuint32_t>(1 << shift));
  }
  if (!ok) return FA_ERR_CUDA;

  fa::KernelParams p = {};
  p.B = 1; p.H = H; p.S_q = total_q; p.S_kv = paged ? 0 : total_k;
  p.kv_group = static_cast<int32_t>(H / H_kv);
  p.n_kv_blocks = 0;
  p.n_pairs = static_cast<int32_t>(n_pairs);
  p.num_units = static_cast<int32_t>(n_seqs * (H >> shift) * n_pairs * n_splits);
  p.group_heads = 1;
  p.q_pack_log2 = shift;
  p.layout = 1;
  p.causal = causal != 0 ? 1 : 0;
  p.causal_br = causal == 2 ? 1 : 0;
  // A negative scale: the products give -Q K^T and the softmax takes |scale|.
  p.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.neg_scale = scale < 0.0f ? 1 : 0;
  p.descale_q = descale_q;
  p.descale_k = descale_k;
  p.descale_v = descale_v;
  p.o = o;
  p.lse = lse;
  p.err = dev.err_word;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.n_splits = n_splits;
  p.lse_part = lse_part;
  p.o_part = o_part;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.seqused_k = seqused_k;
  p.block_table = block_table;
  p.n_seqs = static_cast<int32_t>(n_seqs);
  p.max_pages = static_cast<int32_t>(paged ? max_pages : 0);
  p.page_size = static_cast<int32_t>(paged ? page_size : 0);
  p.seq_order = seq_order;
  if (seq_order &&
      fa::launch_seq_order(seqused_k, static_cast<int>(n_seqs), max_pages * page_size, seq_order,
                           stream) != cudaSuccess)
    return FA_ERR_CUDA;

  const int grid = static_cast<int>(p.num_units < dev.sm_count ? p.num_units : dev.sm_count);
  cudaError_t e;
#define FA_LAUNCH_VAR(DD, DTY)                                                                  \
  (n_splits > 1 ? fa::launch_fa_fwd<DD, DTY, fa::kModePagedSplit>(mq, mk, mv, mo, mop, p, grid, stream) \
   : paged      ? fa::launch_fa_fwd<DD, DTY, fa::kModePaged>(mq, mk, mv, mo, mo, p, grid, stream)    \
                : fa::launch_fa_fwd<DD, DTY, fa::kModeVarlen>(mq, mk, mv, mo, mo, p, grid, stream))
  if (dtype == FA_DTYPE_F16)
    e = (D == 64) ? FA_LAUNCH_VAR(64, fa::kDtF16) : FA_LAUNCH_VAR(128, fa::kDtF16);
  else if (dtype == FA_DTYPE_BF16)
    e = (D == 64) ? FA_LAUNCH_VAR(64, fa::kDtBF16) : FA_LAUNCH_VAR(128, fa::kDtBF16);
  else
    e = FA_LAUNCH_VAR(128, fa::kDtE4M3);
#undef FA_LAUNCH_VAR
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (n_splits > 1) {
    fa::CombineParams c = {};
    c.o_part = o_part;
    c.lse_part = lse_part;
    c.o = o;
    c.lse = lse;
    c.B = 1; c.H = H; c.S_q = total_q;
    c.D = static_cast<int32_t>(D);
    c.n_splits = n_splits;
    c.layout = 1;  // o is [total_q, H, D]: BSND with B = 1
    c.out_f16 = dtype == FA_DTYPE_F16 ? 1 : 0;
    if (fa::launch_fa_combine(c, dev.sm_count, stream) != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status_t fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                          int64_t n_seqs, int64_t total_q, int64_t total_k, int64_t max_seqlen_q,
                          int64_t H, int64_t H_kv, int64_t D, float scale, int causal,
                          fa_dtype_t dtype, const float* descale_q, const float* descale_k,
                          const float* descale_v, cudaStream_t stream) {
  return run_var(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, nullptr, nullptr, n_seqs, 0, 0, 0,
                 total_q, total_k, max_seqlen_q, H, H_kv, D, scale, causal, dtype, descale_q,
                 descale_k, descale_v, stream);
}

fa_status_t fa_fwd_paged(const void* q, const void* k_cache, const void* v_cache, void* o,
                         float* lse, const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                         const int32_t* block_table, int64_t n_seqs, int64_t max_pages_per_seq,
                         int64_t page_size, int64_t num_pages, int64_t total_q,
                         int64_t max_seqlen_q, int64_t H, int64_t H_kv, int64_t D, float scale,
                         int causal, fa_dtype_t dtype, const float* descale_q,
                         const float* descale_k, const float* descale_v, cudaStream_t stream) {
  if (!block_table) return FA_ERR_INVALID_ARG;
  return run_var(q, k_cache, v_cache, o, lse, cu_seqlens_q, nullptr, seqused_k, block_table,
                 n_seqs, max_pages_per_seq, page_size, num_pages, total_q, 0, max_seqlen_q, H,
                 H_kv, D, scale, causal, dtype, descale_q, descale_k, descale_v, stream);
}

}  // extern "C"

extern "C" {

fa_status_t fa_fwd_paged_split_workspace_size(int64_t H, int64_t total_q, int64_t D, int n_splits,
                                              int64_t n_seqs, size_t* workspace_bytes) {
  if (!workspace_bytes || H < 1 || total_q < 0 || D < 1 || n_splits < 1 || n_seqs < 1)
    return FA_ERR_INVALID_ARG;
  *workspace_bytes = fa::paged_split_workspace_bytes(H, total_q, D, n_splits, n_seqs);
  return FA_OK;
}

fa_status_t fa_fwd_paged_split_plan(int64_t n_seqs, int64_t total_q, int64_t max_seqlen_q,
                                    int64_t total_k, int64_t max_seqlen_k, int64_t H,
                                    int64_t H_kv, int64_t D, int sm_count, int* n_splits,
                                    size_t* workspace_bytes) {
  if (!n_splits || !workspace_bytes) return FA_ERR_INVALID_ARG;
  if (n_seqs < 1 || total_q < 0 || max_seqlen_q < 1 || total_k < 0 || max_seqlen_k < 0 ||
      max_seqlen_k > total_k || H < 1 || H_kv < 1 || H % H_kv != 0 || D < 1 || sm_count < 0)
    return FA_ERR_INVALID_ARG;
  if (sm_count == 0) {
    DeviceInfo dev;
    if (device_info(&dev) != FA_OK) return FA_ERR_CUDA;
    sm_count = dev.sm_count;
  }
  // Work in 128-key blocks per head group (the query heads packed into one
  // tile), times the query-tile pairs a sequence has on average.  Sequences
  // are taken longest first, so the static hand-out stays balanced while the
  // longest work item (a split of the longest sequence, plus about three
  // blocks of fixed cost) is at most half of one SM's share; measured on the
  // paged decode workloads (32 and 128 sequences, 1K-32K keys), that rule
  // picks the fastest count or one within 2 % of it.
  const int shift = q_pack_shift(H, H_kv);
  const int64_t toks = 128 >> shift;
  const int64_t groups = H >> shift;
  const int64_t pairs = std::max<int64_t>(1, (total_q + n_seqs * 2 * toks - 1) / (n_seqs * 2 * toks));
  const double share = (static_cast<double>(total_k) / 128.0 + 0.5 * static_cast<double>(n_seqs)) *
                       static_cast<double>(groups * pairs) / sm_count;
  const int64_t longest = (max_seqlen_k + 127) / 128;
  const int64_t cap = std::min<int64_t>(kMaxSplits, std::max<int64_t>(1, longest / 2));
  int64_t splits = 1;
  while (splits < cap && static_cast<double>((longest + splits - 1) / splits + 3) > 0.5 * share)
    ++splits;
  *n_splits = static_cast<int>(splits);
  *workspace_bytes = fa::paged_split_workspace_bytes(H, total_q, D, static_cast<int>(splits), n_seqs);
  return FA_OK;
}

fa_status_t fa_fwd_paged_split(const void* q, const void* k_cache, const void* v_cache, void* o,
                               float* lse, const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                               const int32_t* block_table, int64_t n_seqs,
                               int64_t max_pages_per_seq, int64_t page_size, int64_t num_pages,
                               int64_t total_q, int64_t max_seqlen_q, int64_t H, int64_t H_kv,
                               int64_t D, float scale, int causal, fa_dtype_t dtype,
                               const float* descale_q, const float* descale_k,
                               const float* descale_v, int n_splits, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  if (!block_table) return FA_ERR_INVALID_ARG;
  return run_var(q, k_cache, v_cache, o, lse, cu_seqlens_q, nullptr, seqused_k, block_table,
                 n_seqs, max_pages_per_seq, page_size, num_pages, total_q, 0, max_seqlen_q, H,
                 H_kv, D, scale, causal, dtype, descale_q, descale_k, descale_v, stream, n_splits,
                 workspace, workspace_bytes);
}

}  // extern "C"
