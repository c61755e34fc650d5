// Backward-pass kernel instantiations for bf16 inputs (one translation unit per
// element type so the library builds in parallel).
#include "fa_bwd.cuh"

FA_BWD_INSTANTIATE(, 64, fa::bwd::kBF16)
FA_BWD_INSTANTIATE(, 128, fa::bwd::kBF16)
