// Kernel instantiations for f16 inputs (one translation unit per element
// type so the library builds in parallel).
#include "fa_kernel.cuh"

namespace fa {
template cudaError_t launch_fa_fwd<64, kDtF16, false>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const KernelParams&,
                                                       int, cudaStream_t);
template cudaError_t launch_fa_fwd<64, kDtF16, true>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const KernelParams&,
                                                       int, cudaStream_t);
template cudaError_t launch_fa_fwd<128, kDtF16, false>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const KernelParams&,
                                                       int, cudaStream_t);
template cudaError_t launch_fa_fwd<128, kDtF16, true>(const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const CUtensorMap&,
                                                       const CUtensorMap&, const KernelParams&,
                                                       int, cudaStream_t);
}  // namespace fa
