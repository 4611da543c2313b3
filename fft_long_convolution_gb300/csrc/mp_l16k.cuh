// Multi-pass launches with sub-rows of 16384 points (pass B on warp-level
// MMAs).  SP selects the kernels of frequency-sparse plans; the dense and the
// sparse entry points are instantiated in units of their own.
#pragma once
#include "plan.h"

namespace fftconv {
namespace {

template <int DT, int R0, bool G, bool SP>
cudaError_t launch_t(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, cudaStream_t st) {
    constexpr int HALF = R0 / 2, L = kMpL;
    const size_t smem_a = mp_pass_a_smem<R0, G>(), smem_c = mp_pass_c_smem<R0, G>();
    static PerDevice ca, cb, cc;
    int na = 0, nb = 0, nc = 0;
    cudaError_t e;
    if ((e = prep_kernel(mp_pass_a<DT, R0, G, L, false, SP>, smem_a, 256, ca, &na)) != cudaSuccess) return e;
    if ((e = prep_kernel(mp_pass_b<DT, SP>, kMpBSmem, 512, cb, &nb)) != cudaSuccess) return e;
    if ((e = prep_kernel(mp_pass_c<DT, R0, G, L, false, false, SP>, smem_c, 32 * mp_pass_c_warps<R0>(), cc, &nc)) != cudaSuccess) return e;
    const int64_t items_ac = rows * (L / mp_tile<R0>()), items_b = rows * p->pairs_run;
    auto grid = [&](int64_t items, int per_sm) {
        int64_t gsz = int64_t(p->num_sms) * per_sm;
        return unsigned(gsz < items ? gsz : items);
    };
    mp_pass_a<DT, R0, G, L, false, SP><<<grid(items_ac, na), 256, smem_a, st>>>(args);
    if (items_b > 0) mp_pass_b<DT, SP><<<grid(items_b, nb), 512, kMpBSmem, st>>>(args);
    mp_pass_c<DT, R0, G, L, false, false, SP><<<grid(items_ac, nc), 32 * mp_pass_c_warps<R0>(), smem_c, st>>>(args);
    return cudaGetLastError();
}

template <int DT, bool G, bool SP>
cudaError_t launch_r(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, cudaStream_t st) {
    switch (p->R0) {
        case 2: return launch_t<DT, 2, G, SP>(p, args, rows, st);
        case 4: return launch_t<DT, 4, G, SP>(p, args, rows, st);
        case 8: return launch_t<DT, 8, G, SP>(p, args, rows, st);
        case 16: return launch_t<DT, 16, G, SP>(p, args, rows, st);
        case 32: return launch_t<DT, 32, G, SP>(p, args, rows, st);
        case 64: return launch_t<DT, 64, G, SP>(p, args, rows, st);
        case 128: return launch_t<DT, 128, G, SP>(p, args, rows, st);
    }
    return cudaErrorInvalidValue;
}

template <bool SP>
cudaError_t launch_l16k(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated, cudaStream_t st) {
    if (p->info.dtype == FFTCONV_F16)
        return gated ? launch_r<0, true, SP>(p, args, rows, st) : launch_r<0, false, SP>(p, args, rows, st);
    return gated ? launch_r<1, true, SP>(p, args, rows, st) : launch_r<1, false, SP>(p, args, rows, st);
}

}  // namespace
}  // namespace fftconv
