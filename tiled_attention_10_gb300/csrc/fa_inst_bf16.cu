// Forward kernel instantiations for bf16 inputs, dense and split-KV modes (one
// translation unit per element type and mode group so the library builds in parallel).
#include "fa_kernel.cuh"

FA_FWD_INSTANTIATE(, 64, fa::kDtBF16, fa::kModeDense)
FA_FWD_INSTANTIATE(, 64, fa::kDtBF16, fa::kModeSplit)
FA_FWD_INSTANTIATE(, 128, fa::kDtBF16, fa::kModeDense)
FA_FWD_INSTANTIATE(, 128, fa::kDtBF16, fa::kModeSplit)
