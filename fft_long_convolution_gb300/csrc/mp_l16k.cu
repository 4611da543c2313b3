// Multi-pass launches with sub-rows of 16384 points, dense plans.
#include "mp_l16k.cuh"

namespace fftconv {

cudaError_t launch_mp_l16k(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated, cudaStream_t st) {
    return launch_l16k<false>(p, args, rows, gated, st);
}

}  // namespace fftconv
