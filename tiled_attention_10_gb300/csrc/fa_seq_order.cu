// Longest-first sequence order for the paged forward (see fa_seq_order.cuh):
// thread i counts the sequences that rank before sequence i -- longer, or as
// long with a smaller index -- and writes i at that rank.
#include "fa_seq_order.cuh"

namespace fa {
namespace {

constexpr int kThreadsPerBlock = 256;

__device__ __forceinline__ int32_t clamped_len(const int32_t* len, int i, int64_t cap) {
  const int64_t l = len[i];
  return static_cast<int32_t>(l < 0 ? 0 : (l > cap ? cap : l));
}

__global__ void __launch_bounds__(kThreadsPerBlock)
    fa_seq_order_kernel(const int32_t* seqused_k, int n, int64_t cap, int32_t* order) {
  __shared__ int32_t tile[kThreadsPerBlock];
  const int i = blockIdx.x * kThreadsPerBlock + threadIdx.x;
  const int32_t li = i < n ? clamped_len(seqused_k, i, cap) : 0;
  int rank = 0;
  for (int base = 0; base < n; base += kThreadsPerBlock) {
    const int j = base + threadIdx.x;
    tile[threadIdx.x] = j < n ? clamped_len(seqused_k, j, cap) : -1;
    __syncthreads();
    const int m = min(kThreadsPerBlock, n - base);
    for (int t = 0; t < m; ++t) {
      const int32_t lj = tile[t];
      rank += (lj > li || (lj == li && base + t < i)) ? 1 : 0;
    }
    __syncthreads();
  }
  if (i < n) order[rank] = i;
}

}  // namespace

cudaError_t launch_seq_order(const int32_t* seqused_k, int n, int64_t cap, int32_t* order,
                             cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + kThreadsPerBlock - 1) / kThreadsPerBlock);
  cfg.blockDim = dim3(kThreadsPerBlock);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, fa_seq_order_kernel, seqused_k, n, cap, order);
}

}  // namespace fa
