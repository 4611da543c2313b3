// The plan object shared by the library's translation units, and the
// multi-pass launchers that live in their own units (compiled in parallel).
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/fftconv.h"
#include "multipass.cuh"

struct fftconv_plan_s {
    fftconv_plan_info_t info;
    int R1 = 0;
    void* dev = nullptr;  // one allocation: tables + error word
    int* dev_err = nullptr;
    fftconv::FusedTables tb{};
    fftconv::MPTables mp{};
    int R0 = 1;     // outer factor through HBM (1 on the fused path)
    int mpL = 0;    // multi-pass sub-row length: 16384 (warp-level pass B) or 4096 (tensor-core pass B)
    bool mp2 = false;  // sub-rows of 4096 with the outer factor R0 = RA * 64 in two levels (N >= 2^20)
    bool tc64 = false;               // N = 4096: order-2 64 x 64 product on tcgen05
    int ftc = 0;                     // N = 8192 / 16384 / 32768: the fused R0 x 64 x 64 kernel on tcgen05
    const float2* ftw_in = nullptr;  // its per-thread starting twiddles (device, inside dev)
    const float4* ftw_out = nullptr;
    const uint32_t* fmat = nullptr;  // the 64 x 64 DFT matrix rows (device), N = 4096 and mpL = 4096
    // frequency-sparse plan: a band per factor (every band >= M_j/2 + 1 on a
    // dense plan); on the multi-pass path the pass-B pairs that run and the
    // dead sub-rows of passes A and C (device tables inside dev)
    bool sparse = false;
    int32_t band[8] = {};
    int pairs_run = 0;                          // = R0 / 2 when nothing is skipped
    const uint16_t* plist = nullptr;            // [pairs_run]; null: every pair runs
    const unsigned long long* zbits = nullptr;  // [RA or 1][2] bit k0: sub-row k0 is dead; null: none
    int num_sms = 0;
    int device = 0;  // the device the plan's tables live on (current at creation)
    void* workspace = nullptr;
    size_t workspace_bytes = 0;
    // host-buffer forward: two copy streams and the events that order its
    // three device buffer sets (start, end, then per set: in, done, out),
    // created on first use
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev[11] = {};
};

namespace fftconv {

// Pass A, pass B, pass C of one forward call (args.T is the intermediate).
cudaError_t launch_mp_l16k(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated, cudaStream_t st);
cudaError_t launch_mp_l4k(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated, cudaStream_t st);
cudaError_t launch_mp_l4k_2level(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
                                 cudaStream_t st);
// The same for frequency-sparse plans (p->zbits and p->plist set).
cudaError_t launch_mp_l16k_sparse(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
                                  cudaStream_t st);
cudaError_t launch_mp_l4k_sparse(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
                                 cudaStream_t st);
cudaError_t launch_mp_l4k_2level_sparse(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
                                        cudaStream_t st);

// A value per device: kernel attribute opt-ins belong to the context of the
// device that is current when they are made, so launch preparations are kept
// per device ordinal (0: not prepared on that device yet).
constexpr int kDevSlots = 64;
struct PerDevice {
    int v[kDevSlots] = {};
    int* slot() {
        int d = 0;
        if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kDevSlots) return nullptr;
        return &v[d];
    }
};

// Dynamic shared memory opt-in and resident blocks per SM of a kernel, once
// per device; *per_sm receives the block count.
template <typename K>
cudaError_t prep_kernel(K fn, size_t smem, int threads, PerDevice& cache, int* per_sm) {
    int* s = cache.slot();
    if (!s) return cudaErrorInvalidDevice;
    if (*s == 0) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        int nb = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem);
        if (e != cudaSuccess) return e;
        *s = nb > 0 ? nb : 1;
    }
    *per_sm = *s;
    return cudaSuccess;
}

}  // namespace fftconv
