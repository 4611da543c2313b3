// Multi-pass launches with sub-rows of 4096 points (pass B on the
// fifth-generation tensor cores, tcpass.cuh).  SP selects the kernels of
// frequency-sparse plans (pairs of sub-rows skipped); the dense and the
// sparse entry points are instantiated in units of their own.
#pragma once
#include "plan.h"
#include "tcpass.cuh"

namespace fftconv {
namespace {

template <int DT, int R0, bool G, bool SP>
cudaError_t launch_t(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, cudaStream_t st) {
    constexpr int L = kMpLtc;
    static PerDevice cb;
    int nb = 0;
    cudaError_t e;
    if ((e = prep_kernel(mp_pass_b_tc<DT, SP>, TcB::SMEM, TcB::THREADS, cb, &nb)) != cudaSuccess) return e;
    // pass B: one CTA per SM (its tensor-memory allocation takes all 512
    // columns), two item pipelines per CTA
    const int64_t items_b = rows * p->pairs_run, need_b = (items_b + 1) / 2;
    if (items_b >= (int64_t(1) << 30)) return cudaErrorInvalidValue;  // pass B counts items in int
    const unsigned grid_b = unsigned(need_b < p->num_sms ? need_b : p->num_sms);
    TcBArgs b{args.T, args.kf, p->fmat, args.B, args.H, R0, args.err, 0, p->pairs_run, p->plist};
    // the outer passes on the tensor cores; frequency-sparse plans (SP) skip
    // the dead sub-rows there (not stored by pass A, not loaded by pass C)
    if ((e = launch_otc<DT, R0, 0, G, L, false, SP>(p, args, rows, p->otc_fa, st)) != cudaSuccess) return e;
    if (items_b > 0) mp_pass_b_tc<DT, SP><<<grid_b, TcB::THREADS, TcB::SMEM, st>>>(b);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_otc<DT, R0, 3, G, L, false, SP>(p, args, rows, p->otc_fc, st);
}

template <int DT, bool G, bool SP>
cudaError_t launch_r(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, cudaStream_t st) {
    switch (p->R0) {  // N = 32768 (R0 = 8) runs fused
        case 16: return launch_t<DT, 16, G, SP>(p, args, rows, st);
        case 32: return launch_t<DT, 32, G, SP>(p, args, rows, st);
        case 64: return launch_t<DT, 64, G, SP>(p, args, rows, st);
        case 128: return launch_t<DT, 128, G, SP>(p, args, rows, st);
    }
    return cudaErrorInvalidValue;
}

// Two-level outer factor R0 = RA * 64 (N = RA * 64 * 64 * 64): each outer
// direction is one tensor-core pass (otc2.cuh: the RA-point level in
// registers, the 64-point level as the contraction), pass B on sub-rows of
// 4096 (sub-row k0 = a + RA k at position 64 a + k).  Frequency-sparse plans
// (SP) skip the dead sub-rows in the outer passes and run only the live
// pairs in pass B.
template <int DT, int RA, bool G, bool SP>
cudaError_t launch_2l_t(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, cudaStream_t st) {
    constexpr int R0 = RA * 64;
    static PerDevice cb;
    int nb = 0;
    cudaError_t e;
    if ((e = prep_kernel(mp_pass_b_tc<DT, SP>, TcB::SMEM, TcB::THREADS, cb, &nb)) != cudaSuccess) return e;
    const int64_t items_b = rows * p->pairs_run, need_b = (items_b + 1) / 2;
    if (items_b >= (int64_t(1) << 30) || rows * RA >= (int64_t(1) << 30)) return cudaErrorInvalidValue;
    const unsigned grid_b = unsigned(need_b < p->num_sms ? need_b : p->num_sms);
    TcBArgs b{args.T, args.kf, p->fmat, args.B, args.H, R0, args.err, RA, p->pairs_run, p->plist};
    if ((e = launch_otc2<DT, RA, true, G, SP>(p, args, rows, st)) != cudaSuccess) return e;
    if (items_b > 0) mp_pass_b_tc<DT, SP><<<grid_b, TcB::THREADS, TcB::SMEM, st>>>(b);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_otc2<DT, RA, false, G, SP>(p, args, rows, st);
}

template <int DT, bool G, bool SP>
cudaError_t launch_2l_r(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, cudaStream_t st) {
    switch (p->R0 / 64) {
        case 4: return launch_2l_t<DT, 4, G, SP>(p, args, rows, st);
        case 8: return launch_2l_t<DT, 8, G, SP>(p, args, rows, st);
    }
    return cudaErrorInvalidValue;
}

template <bool SP>
cudaError_t launch_l4k_2level(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated, cudaStream_t st) {
    if (p->info.dtype == FFTCONV_F16)
        return gated ? launch_2l_r<0, true, SP>(p, args, rows, st) : launch_2l_r<0, false, SP>(p, args, rows, st);
    return gated ? launch_2l_r<1, true, SP>(p, args, rows, st) : launch_2l_r<1, false, SP>(p, args, rows, st);
}

// Circular convolution of length 2 M, M = R0 * 4096: pass A over all R0 rows
// of z, pass B unchanged, pass C writing all R0 output rows.
template <int DT, int R0, bool G>
cudaError_t launch_circ_t(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, cudaStream_t st) {
    constexpr int L = kMpLtc;
    static PerDevice cb;
    int nb = 0;
    cudaError_t e;
    if ((e = prep_kernel(mp_pass_b_tc<DT, false>, TcB::SMEM, TcB::THREADS, cb, &nb)) != cudaSuccess) return e;
    const int64_t items_b = rows * (R0 / 2), need_b = (items_b + 1) / 2;
    if (items_b >= (int64_t(1) << 30)) return cudaErrorInvalidValue;  // pass B counts items in int
    const unsigned grid_b = unsigned(need_b < p->num_sms ? need_b : p->num_sms);
    TcBArgs b{args.T, args.kf, p->fmat, args.B, args.H, R0, args.err, 0, R0 / 2, nullptr};
    if ((e = launch_otc<DT, R0, 0, G, L, true>(p, args, rows, p->otc_fa, st)) != cudaSuccess) return e;
    mp_pass_b_tc<DT, false><<<grid_b, TcB::THREADS, TcB::SMEM, st>>>(b);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_otc<DT, R0, 3, G, L, true>(p, args, rows, p->otc_fc, st);
}

template <int DT, bool G>
cudaError_t launch_circ_r(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, cudaStream_t st) {
    switch (p->R0) {
        case 2: return launch_circ_t<DT, 2, G>(p, args, rows, st);
        case 4: return launch_circ_t<DT, 4, G>(p, args, rows, st);
        case 8: return launch_circ_t<DT, 8, G>(p, args, rows, st);
        case 16: return launch_circ_t<DT, 16, G>(p, args, rows, st);
        case 32: return launch_circ_t<DT, 32, G>(p, args, rows, st);
        case 64: return launch_circ_t<DT, 64, G>(p, args, rows, st);
    }
    return cudaErrorInvalidValue;
}

inline cudaError_t launch_circ(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated, cudaStream_t st) {
    if (p->info.dtype == FFTCONV_F16)
        return gated ? launch_circ_r<0, true>(p, args, rows, st) : launch_circ_r<0, false>(p, args, rows, st);
    return gated ? launch_circ_r<1, true>(p, args, rows, st) : launch_circ_r<1, false>(p, args, rows, st);
}

template <bool SP>
cudaError_t launch_l4k(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated, cudaStream_t st) {
    if (p->info.dtype == FFTCONV_F16)
        return gated ? launch_r<0, true, SP>(p, args, rows, st) : launch_r<0, false, SP>(p, args, rows, st);
    return gated ? launch_r<1, true, SP>(p, args, rows, st) : launch_r<1, false, SP>(p, args, rows, st);
}

}  // namespace
}  // namespace fftconv
