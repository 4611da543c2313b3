// Multi-pass launches with sub-rows of 16384 points, frequency-sparse plans.
#include "mp_l16k.cuh"

namespace fftconv {

cudaError_t launch_mp_l16k_sparse(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
                                  cudaStream_t st) {
    return launch_l16k<true>(p, args, rows, gated, st);
}

}  // namespace fftconv
