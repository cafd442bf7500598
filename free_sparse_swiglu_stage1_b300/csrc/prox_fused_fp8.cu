// FP8-row instantiations of the fused single-token kernel (prox_fused_impl.cuh); the bf16
// ones and the launch code are in prox_fused.cu.
#include "prox_fused_impl.cuh"

namespace prox {
namespace fused_detail {

FusedFn fused_fn_fp8(const FusedShape& s) {
#define PROX_FUSED(run, cw, cpt) \
    if (s.RUN == run && s.CW == cw && s.CPTMAX == cpt) return fused_token_kernel<run, cw, cpt, true>;
    PROX_FUSED(4, 4, 2)
    PROX_FUSED(4, 8, 2)
    PROX_FUSED(4, 16, 2)
    PROX_FUSED(8, 4, 4)
    PROX_FUSED(8, 8, 4)
    PROX_FUSED(8, 16, 4)
    PROX_FUSED(16, 4, 4)
    PROX_FUSED(16, 8, 4)
    PROX_FUSED(16, 16, 4)
#undef PROX_FUSED
    return nullptr;
}

}  // namespace fused_detail
}  // namespace prox
