// Forward kernel instantiations for f16 inputs, varlen, paged-KV and paged split-KV modes.
#include "fa_kernel.cuh"

FA_FWD_INSTANTIATE(, 64, fa::kDtF16, fa::kModeVarlen)
FA_FWD_INSTANTIATE(, 64, fa::kDtF16, fa::kModePaged)
FA_FWD_INSTANTIATE(, 64, fa::kDtF16, fa::kModePagedSplit)
FA_FWD_INSTANTIATE(, 128, fa::kDtF16, fa::kModeVarlen)
FA_FWD_INSTANTIATE(, 128, fa::kDtF16, fa::kModePaged)
FA_FWD_INSTANTIATE(, 128, fa::kDtF16, fa::kModePagedSplit)
