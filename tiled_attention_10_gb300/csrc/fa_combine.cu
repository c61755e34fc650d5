// Split-KV merge kernel (see fa_combine.cuh): one warp per query row; lane s
// holds split s's lse, lane l accumulates head-dim elements [l*D/32, +D/32).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "fa_combine.cuh"

namespace fa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) fa_combine_kernel(const CombineParams c) {
  constexpr int kPer = D / 32;  // head-dim elements per lane
  const int lane = threadIdx.x & 31;
  // Launched as a programmatic dependent of the split forward pass: nothing
  // is read before that pass has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t rows = c.B * c.H * c.S_q;
  const int64_t split_stride = rows;  // rows per split
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); row < rows;
       row += static_cast<int64_t>(gridDim.x) * 8) {
    const float lp = lane < c.n_splits ? c.lse_part[lane * split_stride + row] : -CUDART_INF_F;
    float mx = lp;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float wgt = (lp == -CUDART_INF_F) ? 0.0f : expf(lp - mx);
    float sum = wgt;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.0f;
    for (int s = 0; s < c.n_splits; ++s) {
      const float ws = __shfl_sync(0xffffffffu, wgt, s);
      if (ws == 0.0f) continue;  // empty split: its partial O is not read
      const float* src = c.o_part + (s * split_stride + row) * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] += ws * src[e];
    }
    const float inv = (sum > 0.0f) ? 1.0f / sum : 0.0f;
    const int64_t bh = row / c.S_q, i = row - bh * c.S_q;
    const int64_t b = bh / c.H, h = bh - b * c.H;
    const int64_t orow = (c.layout == 0) ? row : ((b * c.S_q + i) * c.H + h);
    uint16_t* dst = reinterpret_cast<uint16_t*>(c.o) + orow * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
      const float x0 = acc[e] * inv, x1 = acc[e + 1] * inv;
      uint32_t pk;
      if (c.out_f16) {
        const __half2 hv = __floats2half2_rn(x0, x1);
        pk = *reinterpret_cast<const uint32_t*>(&hv);
      } else {
        const __nv_bfloat162 hv = __floats2bfloat162_rn(x0, x1);
        pk = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *reinterpret_cast<uint32_t*>(dst + e) = pk;
    }
    if (lane == 0) c.lse[row] = (sum > 0.0f) ? mx + logf(sum) : -CUDART_INF_F;
  }
}

}  // namespace

cudaError_t launch_fa_combine(const CombineParams& c, int sm_count, cudaStream_t stream) {
  const int64_t rows = c.B * c.H * c.S_q;
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sm_count) * 16;
  if (blocks > cap) blocks = cap;
  // cudaLaunchKernelEx reports this launch's own status (not an error left
  // pending by other code on the thread).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  // Programmatic dependent launch: the merge grid is scheduled while the
  // forward pass drains and waits on the device for it (griddepcontrol.wait)
  // instead of on the launch path.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (c.D == 64) return cudaLaunchKernelEx(&cfg, fa_combine_kernel<64>, c);
  return cudaLaunchKernelEx(&cfg, fa_combine_kernel<128>, c);
}

}  // namespace fa
