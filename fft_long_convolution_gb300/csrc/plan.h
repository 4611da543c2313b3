// The plan object shared by the library's translation units, and the
// multi-pass launchers that live in their own units (compiled in parallel).
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <cstring>

#include "../../include/fftconv.h"
#include "multipass.cuh"
#include "otc.cuh"
#include "otc2.cuh"

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
    // multi-pass outer passes on the tensor cores (otc.cuh): the DFT matrices of
    // pass A and pass C (the outermost factor) and of the in-place 64-point
    // stages of a two-level outer factor (device, inside dev)
    const uint8_t* otc_fa = nullptr;
    const uint8_t* otc_fc = nullptr;
    const uint8_t* otc_fa2 = nullptr;
    const uint8_t* otc_fc2 = nullptr;
    // two levels: W_(64 RA)^(n_b k_a) / sqrt(RA) as packed pairs, pass A's
    // table then pass C's (Otc2::TABB bytes each)
    const float4* otc_tw2 = nullptr;
    const uint32_t* fmat = nullptr;  // the 64 x 64 DFT matrix rows (device), N = 4096 and mpL = 4096
    // frequency-sparse plan: a band per factor (every band >= M_j/2 + 1 on a
    // dense plan); on the multi-pass path the pass-B pairs that run and the
    // dead sub-rows of passes A and C (device tables inside dev)
    bool sparse = false;
    int32_t band[8] = {};
    int pairs_run = 0;                          // = R0 / 2 when nothing is skipped
    const uint16_t* plist = nullptr;            // [pairs_run]; null: every pair runs
    const unsigned long long* zbits = nullptr;  // [RA or 1][2] bit k0: sub-row k0 is dead; null: none
    // one-level plans: the sub-rows whose bins are all dropped (a superset of
    // the skipped pairs' sub-rows, whose pass-B output is exactly zero), read
    // as zeros by the last pass: device copy and host copy
    const unsigned long long* zcbits = nullptr;
    unsigned long long zhost[2] = {0ull, 0ull};
    int num_sms = 0;
    bool circular = false;  // circular convolution of length 2 M (every input and output row of the outer passes)
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
// Circular convolution of length 2 M (p->circular): the outer passes over all
// R0 input and output rows, R0 = 2 .. 128.
cudaError_t launch_mp_l4k_circular(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, bool gated,
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

// cuTensorMapEncodeTiled, reached through the runtime (once per process;
// null if the driver does not provide it).
using TensorMapEncoder = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
inline TensorMapEncoder tensor_map_encoder() {
    static TensorMapEncoder fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return TensorMapEncoder(nullptr);
        }
        return reinterpret_cast<TensorMapEncoder>(ptr);
    }();
    return fn;
}

// A tensor map over rows of `nin` sub-rows of L 32-bit words (row stride
// row_bytes), read as boxes of box_cols words (default 128) x box_rows
// sub-rows (default: all nin) x 1 row.
inline bool encode_rows_map(CUtensorMap* m, const void* base, uint64_t L, uint64_t nin, uint64_t rows,
                            uint64_t row_bytes, uint32_t box_rows = 0, uint32_t box_cols = 128) {
    TensorMapEncoder enc = tensor_map_encoder();
    if (!enc || !base) return false;
    const cuuint64_t dims[3] = {L, nin, rows};
    const cuuint64_t strides[2] = {4 * L, row_bytes};
    const cuuint32_t box[3] = {box_cols, box_rows ? box_rows : cuuint32_t(nin), 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One outer pass on the tensor cores: rows x (L / 128) column tiles over the
// resident CTAs of the SM (their tensor-memory columns included).  FULL: the
// circular form (rows of u and y of 2 R L samples, every input and output row).
template <int DT, int R, int MODE, bool G, int L, bool FULL = false, bool SP = false>
cudaError_t launch_otc(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, const uint8_t* fmat,
                       cudaStream_t st) {
    using C = Otc<R, MODE, FULL>;
    auto fn = otc_pass<DT, R, MODE, G, L, FULL, SP>;
    // no more CTAs per SM than its 512 tensor-memory columns hold: the shared
    // memory request is raised until the SM's 228 KB (1 KB reserved per CTA)
    // fit no more of them
    constexpr int tmem_cap = int(512 / C::TMEM_COLS);
    constexpr size_t smem_need = otc_smem<R, MODE, G, FULL>();
    constexpr size_t smem_floor = size_t(233472 / (tmem_cap + 1)) - 1024 + 16;
    constexpr size_t smem = smem_need > smem_floor ? smem_need : smem_floor;
    static_assert(smem <= 232448, "shared memory");
    static PerDevice cache;  // per instantiation and device
    int per_sm = 0;
    cudaError_t e = prep_kernel(fn, smem, C::THREADS, cache, &per_sm);
    if (e != cudaSuccess) return e;
    // resident CTAs from the shared-memory and tensor-memory budgets
    per_sm = int(233472 / (smem + 1024));
    if (per_sm > tmem_cap) per_sm = tmem_cap;
    if (per_sm < 1) per_sm = 1;
    const int64_t items = rows * (L / C::TC);
    int64_t grid = int64_t(p->num_sms) * per_sm;
    if (grid > items) grid = items;
    if (grid < 1) return cudaSuccess;
    // the input rows: u (MODE 0: R/2 sub-rows of a row of R L / 2 words; FULL:
    // R sub-rows of R L words) or T (R sub-rows of a row of R L words); w_in in
    // u's shape
    CUtensorMap tin, tgate;
    std::memset(&tgate, 0, sizeof(tgate));
    constexpr uint64_t uin = FULL ? R : R / 2, urow = uint64_t(FULL ? 4 : 2) * R * L;
    // SP pass C copies the runs of live sub-rows (boxes of the longest run's height)
    uint32_t box = 0;
    if (SP && MODE == 3) {
        const OtcRuns r = otc_live_runs(p->zhost[0], p->zhost[1], R);
        box = uint32_t(r.box > 0 ? r.box : R);
    }
    const bool ok = MODE == 0 ? encode_rows_map(&tin, args.u, L, uin, uint64_t(rows), urow)
                              : encode_rows_map(&tin, args.T, L, R, uint64_t(rows), uint64_t(4) * R * L, box);
    if (!ok) return cudaErrorInvalidValue;
    if (G && MODE == 0 && !encode_rows_map(&tgate, args.w_in, L, uin, uint64_t(rows), urow))
        return cudaErrorInvalidValue;
    fn<<<unsigned(grid), C::THREADS, smem, st>>>(args, fmat, tin, tgate);
    return cudaGetLastError();
}

// The fused two-level outer pass (otc2.cuh): pass A (FWD, from u) or pass C
// (to y) over rows x (4096 / TC) column tiles, as many CTAs per SM as shared
// and tensor memory hold.  SP: a frequency-sparse plan's dead sub-rows
// (args.zbits, [RA][2] words) are not stored by pass A and read as zeros by
// pass C.
template <int DT, int RA, bool FWD, bool G, bool SP = false>
cudaError_t launch_otc2(const fftconv_plan_s* p, const MPArgs& args, int64_t rows, cudaStream_t st) {
    using C = Otc2<RA>;
    using P = Otc2Pass<RA, FWD, G>;
    auto fn = otc2_pass<DT, RA, FWD, G, SP>;
    constexpr size_t smem = P::SMEM;
    static_assert(smem <= 232448, "shared memory");
    static PerDevice cache;  // per instantiation and device
    int per_sm = 0;
    cudaError_t e = prep_kernel(fn, smem, C::THREADS, cache, &per_sm);
    if (e != cudaSuccess) return e;
    per_sm = int(233472 / (smem + 1024));
    if (per_sm > 512 / C::TMEM_COLS) per_sm = 512 / C::TMEM_COLS;
    if (per_sm < 1) per_sm = 1;
    const int64_t items = rows * C::TILES;
    int64_t grid = int64_t(p->num_sms) * per_sm;
    if (grid > items) grid = items;
    if (grid < 1) return cudaSuccess;
    if (!p->otc_fa2 || !p->otc_fc2 || !p->otc_tw2 || (SP && !args.zbits)) return cudaErrorInvalidValue;
    CUtensorMap tin, tgate;
    std::memset(&tgate, 0, sizeof(tgate));
    // pass A: u as RA/2 x 64 sub-rows of 4096 words per row (2 M bytes);
    // pass C: T as RA x 64 sub-rows per row (4 M bytes)
    const bool ok =
        FWD ? encode_rows_map(&tin, args.u, C::L, P::NIN, uint64_t(rows), uint64_t(2) * C::M, P::BOXR, C::TC)
            : encode_rows_map(&tin, args.T, C::L, P::NIN, uint64_t(rows), uint64_t(4) * C::M, P::BOXR, C::TC);
    if (!ok) return cudaErrorInvalidValue;
    if (G && FWD &&
        !encode_rows_map(&tgate, args.w_in, C::L, P::NIN, uint64_t(rows), uint64_t(2) * C::M, P::BOXR, C::TC))
        return cudaErrorInvalidValue;
    const float4* tab = p->otc_tw2 + (FWD ? 0 : C::TABB / 16);
    fn<<<unsigned(grid), C::THREADS, smem, st>>>(args, FWD ? p->otc_fa2 : p->otc_fc2, tab, tin, tgate);
    return cudaGetLastError();
}

}  // namespace fftconv
