// Kernel instantiations for bf16 inputs (one translation unit per element
// type so the library builds in parallel).
#include "fa_kernel.cuh"

namespace fa {
template cudaError_t launch_fa_fwd<64, kDtBF16, false>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const KernelParams&,
                                                       int, cudaStream_t);
template cudaError_t launch_fa_fwd<64, kDtBF16, true>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const KernelParams&,
                                                       int, cudaStream_t);
template cudaError_t launch_fa_fwd<128, kDtBF16, false>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const KernelParams&,
                                                       int, cudaStream_t);
template cudaError_t launch_fa_fwd<128, kDtBF16, true>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const KernelParams&,
                                                       int, cudaStream_t);
}  // namespace fa
