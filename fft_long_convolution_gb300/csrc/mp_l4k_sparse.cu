// Multi-pass launches with sub-rows of 4096 points, frequency-sparse plans
// (pairs of sub-rows whose spectrum is zero are skipped).
#include "mp_l4k.cuh"

namespace fftconv {

cudaError_t launch_mp_l4k_sparse(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
                                 cudaStream_t st) {
    return launch_l4k<true>(p, args, rows, gated, st);
}

cudaError_t launch_mp_l4k_2level_sparse(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
                                        cudaStream_t st) {
    return launch_l4k_2level<true>(p, args, rows, gated, st);
}

}  // namespace fftconv
