// Forward kernel instantiations for e4m3 inputs, dense and split-KV modes (one
// translation unit per element type and mode group so the library builds in parallel).
#include "fa_kernel.cuh"

FA_FWD_INSTANTIATE(, 128, fa::kDtE4M3, fa::kModeDense)
FA_FWD_INSTANTIATE(, 128, fa::kDtE4M3, fa::kModeSplit)
