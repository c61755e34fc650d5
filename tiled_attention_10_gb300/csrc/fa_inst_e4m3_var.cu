// Forward kernel instantiations for e4m3 inputs, varlen, paged-KV and paged split-KV modes.
#include "fa_kernel.cuh"

FA_FWD_INSTANTIATE(, 128, fa::kDtE4M3, fa::kModeVarlen)
FA_FWD_INSTANTIATE(, 128, fa::kDtE4M3, fa::kModePaged)
FA_FWD_INSTANTIATE(, 128, fa::kDtE4M3, fa::kModePagedSplit)
