/*
 * fa_combine.cuh -- merge of split-KV partial results.
 *
 * A split s of a query row's keys yields the attention over that split alone,
 * O_s (normalised) and its log-sum-exp lse_s.  The attention over all keys is
 *     lse = log sum_s exp(lse_s),     O = sum_s exp(lse_s - lse) O_s,
 * the partition-and-reduce scheme of the paged-decode kernels in the Hygon
 * retrospective (defect 7: per-partition exp_sums / max_logits, then a
 * second kernel that reduces them).  A split with no visible key has
 * lse_s = -inf and weight 0; its O_s is never read.
 */
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace fa {

struct CombineParams {
  const float* o_part;    // fp32 [n_splits, B, H, S_q, D]
  const float* lse_part;  // fp32 [n_splits, B, H, S_q]
  void* o;                // output, caller's layout, f16 or bf16
  float* lse;             // fp32 [B, H, S_q]
  int64_t B, H, S_q;
  int32_t D, n_splits, layout, out_f16;
};

cudaError_t launch_fa_combine(const CombineParams& c, int sm_count, cudaStream_t stream);

}  // namespace fa
