// Multi-pass launches with sub-rows of 4096 points, dense plans.
#include "mp_l4k.cuh"

namespace fftconv {

cudaError_t launch_mp_l4k(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated, cudaStream_t st) {
    return launch_l4k<false>(p, args, rows, gated, st);
}

cudaError_t launch_mp_l4k_2level(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
                                 cudaStream_t st) {
    return launch_l4k_2level<false>(p, args, rows, gated, st);
}

}  // namespace fftconv
