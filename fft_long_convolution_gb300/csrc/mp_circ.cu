// Multi-pass launches of the circular convolution (sub-rows of 4096 points).
#include "mp_l4k.cuh"

namespace fftconv {

cudaError_t launch_mp_l4k_circular(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
                                   cudaStream_t st) {
    return launch_circ(p, args, rows, gated, st);
}

}  // namespace fftconv
