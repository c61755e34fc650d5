// Forward kernel instantiations for f16 inputs, dense and split-KV modes (one
// translation unit per element type and mode group so the library builds in parallel).
#include "fa_kernel.cuh"

FA_FWD_INSTANTIATE(, 64, fa::kDtF16, fa::kModeDense)
FA_FWD_INSTANTIATE(, 64, fa::kDtF16, fa::kModeSplit)
FA_FWD_INSTANTIATE(, 128, fa::kDtF16, fa::kModeDense)
FA_FWD_INSTANTIATE(, 128, fa::kDtF16, fa::kModeSplit)
