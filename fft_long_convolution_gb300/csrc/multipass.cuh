// Multi-pass causal long convolution for N = M = R0 * L (32K..2M), with
// sub-rows of L = 16384 (pass B on warp-level MMAs, below) or L = 4096 (pass B
// on the fifth-generation tensor cores, tcpass.cuh).
//
// Partial fusion (FlashFFTConv page, section 3.4 "Kernel Fusion and
// Recomputation Strategies" and the order-4 Algorithm 4): the outermost
// Monarch factor R0 goes through HBM, everything inside it stays fused.
//   n = L*n0 + n',  k = k0 + R0*kappa
//   pass A:  T[k0][n'] = W_M^(n'*k0) * sum_{n0 < R0/2} z[L*n0 + n'] W_R0^(n0*k0) / sqrt(R0)
//            (implicit zero padding: z[n] = 0 for n >= M/2, i.e. n0 >= R0/2)
//   pass B:  per pair of sub-rows (k0, R0-k0): the L-point transform of each
//            sub-row, the decimation-in-time fold with the kernel spectrum
//            (bin k pairs with M-k, which lives in sub-row R0-k0), the same
//            stages back, then the W_M^(n'*k0) twiddle of the conjugate-trick
//            inverse -> T (in place).  L = 16384: R1 = 64 outer factor x 16 x
//            16 (the fused machinery with a full outer stage).  L = 4096: 64 x
//            64 on the tensor cores, and the twiddle moves into pass C.
//   pass C:  y_z[L*n0 + n'] = sum_{k0} W_R0^(n0*k0) T[k0][n'] / sqrt(R0), only
//            n0 < R0/2 (causal truncation), conjugated (and gated) -> y.
// T holds 16-bit complex words (the plan dtype); it is the caller's
// workspace of B*H*N*4 bytes.  Each pass reads its operands with bulk copies
// (TMA engine) into padded shared-memory segments and writes contiguous
// 32-byte runs per output row.
#pragma once
#include "fused.cuh"

namespace fftconv {

constexpr int kMpL = 16384;   // sub-row length of the warp-level pass B
constexpr int kMpLtc = 4096;  // sub-row length of the tensor-core pass B
constexpr int kMpR1 = 64;     // outer factor inside pass B
constexpr int kSeg = 264;     // staged 1 KB segment + 32 B pad (words)

struct MPTables {
    const uint4* lf;      // inner 16-point fragments (as the fused path)
    const uint4* rf;
    const float4* tw;
    const uint4* of_a;    // pass A: F_R0/sqrt(R0) A fragments, half input   [m][s][lane]
    const uint4* oi_c;    // pass C: F_R0/sqrt(R0) A fragments, half output  [m][s][lane]
    const uint4* ofull;   // pass B: F_64/8 A fragments, full               [8][8][lane]
    const float4* twf;    // pass B: W_L^(o*k1), outer-output order          [nt][m][lane]
    const float4* twi;    // pass B: W_L^(o*k1), inner-output order          [k1][nt][lane]
};

struct MPArgs {
    const uint16_t* u;
    const uint16_t* w_in;
    const uint16_t* w_out;
    const uint4* kf;
    uint16_t* y;
    uint32_t* T;  // [rows][R0][L] 16-bit complex words
    int B, H, R0;
    MPTables tb;
    int* err;
    // frequency-sparse plans: sub-rows whose pair of pass B is skipped (bit k0
    // of [row % zmod][2], k0 < 128) are not written by pass A and read as
    // zeros by pass C; pass B runs only the np pairs listed in plist
    const unsigned long long* zbits = nullptr;  // null: every sub-row is live
    int zmod = 1;
    int np = 0;                                 // pass-B pairs that run (R0 / 2 when plist is null)
    const uint16_t* plist = nullptr;
    // one-level frequency-sparse plans: sub-rows whose bins are all dropped
    // (bit k0 of [2]); the tensor-core last pass reads them as zeros
    const unsigned long long* zcbits = nullptr;
};

// Bit k0 (< 128) of a dead-sub-row pair of words.
__device__ __forceinline__ bool zbit(unsigned long long z0, unsigned long long z1, int k0) {
    return ((k0 < 64 ? z0 >> k0 : z1 >> (k0 - 64)) & 1ull) != 0;
}

// W_M^j for M a power of two (exact angle: j / M is exact in float).
__device__ __forceinline__ cpx twiddle_pow2(uint32_t j, uint32_t M) {
    float s, c;
    sincospif(-2.0f * (float(j) / float(M)), &s, &c);
    return {c, s};
}

// Thread 0 waits (bounded) on a barrier phase, the CTA learns the outcome.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, int* s_fail, int* err) {
    if (threadIdx.x == 0 && !mbar_wait_bounded(bar, parity, kWaitLimit)) {
        *s_fail = 1;
        atomicExch(err, 7);
    }
    __syncthreads();
    if (*s_fail) return false;
    mbar_wait_bounded(bar, parity, 4);
    return true;
}

// Columns per pass A / C item (wider where few segments are staged, so the
// per-item staging, barrier and twiddle set-up are amortized) and the padded
// staged segment in words (row stride = 8 banks, conflict free).
template <int R0>
__host__ __device__ constexpr int mp_tile() { return R0 <= 8 ? 2048 : 256; }
template <int R0>
__host__ __device__ constexpr int mp_seg() { return mp_tile<R0>() + 8; }

// Dynamic shared memory of pass A (half or full input rows, gated) and pass C.
template <int R0, bool GATED, bool FULL = false>
constexpr size_t mp_pass_a_smem() {
    return size_t(FULL ? R0 : R0 / 2) * mp_seg<R0>() * 4 * (GATED ? 2 : 1) + 32;
}
template <int R0, bool GATED>
constexpr size_t mp_pass_c_smem() {
    return size_t(R0) * mp_seg<R0>() * 4 + (GATED ? size_t(R0 / 2) * mp_seg<R0>() * 4 : 0) + 32;
}

// ------------------------------------------------------------------ pass A
// FULL: an inner outer stage of a two-level outer factor: all R0 input rows
// are nonzero and come from T itself (16-bit complex words, rows of length
// R0*L), the result overwrites them (each item stages its whole tile first).
// SP: frequency-sparse plan: outputs of dead sub-rows (a.zbits) are not stored.
template <int DT, int R0, bool GATED, int L, bool FULL = false, bool SP = false>
__global__ void __launch_bounds__(256, (R0 <= 64 && !FULL) ? 3 : 2) mp_pass_a(const MPArgs a) {
    using O = Op<DT>;
    static_assert(!(FULL && GATED), "the inner stage has no gates");
    constexpr int HALF = FULL ? R0 : R0 / 2, SEG = mp_seg<R0>(), TILE = mp_tile<R0>();  // input rows staged
    constexpr uint32_t M = uint32_t(R0) * L;
    constexpr bool K8 = !FULL && R0 <= 8;
    constexpr int KS = K8 ? 1 : HALF / 8, MT = (R0 + 7) / 8;
    const uint4* frag = FULL ? a.tb.ofull : a.tb.of_a;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t* su = reinterpret_cast<uint32_t*>(smem);  // [HALF][SEG]
    uint32_t* sw = su + HALF * SEG;                     // gated: w_in
    uint64_t* bar = reinterpret_cast<uint64_t*>(sw + (GATED ? HALF * SEG : 0));
    __shared__ int s_fail;
    __shared__ unsigned long long s_z[2];
    // the DFT fragments of the outer factor, staged once per CTA in shared
    // memory where that keeps the resident CTAs (else read through L1)
    constexpr bool FS = MT * KS * 32 * 16 <= (GATED ? 8192 : 32768);
    __shared__ uint4 s_frag[FS ? MT * KS * 32 : 1];
    if (FS)
        for (int i = threadIdx.x; i < MT * KS * 32; i += blockDim.x) s_frag[i] = frag[i];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    const long rows = long(a.B) * a.H, tiles = L / TILE, items = rows * tiles;
    if (threadIdx.x == 0) {
        s_fail = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    uint32_t par = 0;
    for (long item = blockIdx.x; item < items; item += gridDim.x, par ^= 1) {
        const long row = item / tiles;
        const int o_base = int(item % tiles) * TILE;
        const uint16_t* ur = a.u + row * long(M);
        if (threadIdx.x == 0) {
            mbar_expect_tx(bar, HALF * TILE * 4u * (GATED ? 2u : 1u));
            for (int n0 = 0; n0 < HALF; ++n0) {
                if (FULL)
                    bulk_g2s(su + n0 * SEG, a.T + row * long(M) + long(L) * n0 + o_base, TILE * 4, bar);
                else
                    bulk_g2s(su + n0 * SEG, ur + 2 * (long(L) * n0 + o_base), TILE * 4, bar);
                if (GATED) bulk_g2s(sw + n0 * SEG, a.w_in + row * long(M) + 2 * (long(L) * n0 + o_base), TILE * 4, bar);
            }
        }
        if constexpr (SP) {
            if (threadIdx.x == 32) {  // outputs k0 that nothing reads
                s_z[0] = a.zbits ? __ldg(a.zbits + 2 * (row % a.zmod)) : 0ull;
                s_z[1] = a.zbits ? __ldg(a.zbits + 2 * (row % a.zmod) + 1) : 0ull;
            }
        }
        if (!cta_wait(bar, par, &s_fail, a.err)) return;
        uint32_t* Trow = a.T + row * long(M);
        // SP: bit m of lm set when this thread's output k0 = 8m + g exists and
        // is read later; bit m of lt (the same in every thread) when some
        // output of the tile 8m .. 8m + 7 is, else the tile is not computed
        uint32_t lm = 0, lt = 0;
        if constexpr (SP) {
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                const int k0 = 8 * m + g, kc = 8 * m;
                if (k0 < R0 && !((s_z[k0 >> 6] >> (k0 & 63)) & 1ull)) lm |= 1u << m;
                if (((s_z[kc >> 6] >> (kc & 63)) & 0xffull) != 0xffull) lt |= 1u << m;
            }
        }
        // NT column groups of 8 per iteration share each DFT fragment load; the
        // twiddle of output (k0 = 8m + g, o) is W_M^(o g) * W_M^(8 o)^m, a
        // product chain over the output tiles m.  CHAIN (one output tile): the
        // columns advance by 64 NT per iteration, so W_M^(o g) is carried from
        // one iteration to the next by W_M^(64 NT g) instead of recomputed
        constexpr int NT = 2;
        constexpr bool CHAIN = MT == 1;
        cpx cb[NT][2], cstep;
        if constexpr (CHAIN) {
            #pragma unroll
            for (int j = 0; j < NT; ++j)
                #pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t o = uint32_t(o_base + 8 * (warp + 8 * j) + 2 * t + e);
                    cb[j][e] = twiddle_pow2((o * uint32_t(g)) & (M - 1), M);
                }
            cstep = twiddle_pow2((64u * NT * uint32_t(g)) & (M - 1), M);
        }
        #pragma unroll 1
        for (int i = 0; i < TILE / 64 / NT; ++i) {
            uint32_t bf[NT][KS][2];
            cpx tw[NT][2], ts[NT][2];
            #pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int nt = warp + 8 * (NT * i + j);
                #pragma unroll
                for (int s = 0; s < KS; ++s) {
                    const int na = 8 * s + t, nb = 8 * s + 4 + t;
                    uint32_t va = 0, vb = 0;
                    if (na < HALF) {
                        va = su[na * SEG + 8 * nt + g];
                        if (GATED) va = O::mul2(va, sw[na * SEG + 8 * nt + g]);
                    }
                    if (!K8 && nb < HALF) {
                        vb = su[nb * SEG + 8 * nt + g];
                        if (GATED) vb = O::mul2(vb, sw[nb * SEG + 8 * nt + g]);
                    }
                    bf[j][s][0] = va;
                    bf[j][s][1] = vb;
                }
                #pragma unroll
                for (int e = 0; e < 2; ++e) {
                    if constexpr (CHAIN) {
                        tw[j][e] = cb[j][e];
                        cb[j][e] = cmul(cb[j][e], cstep);
                    } else {
                        const uint32_t o = uint32_t(o_base + 8 * nt + 2 * t + e);
                        tw[j][e] = twiddle_pow2((o * uint32_t(g)) & (M - 1), M);
                        if (MT > 1) ts[j][e] = twiddle_pow2((8 * o) & (M - 1), M);
                    }
                }
            }
            #pragma unroll 2
            for (int m = 0; m < MT; ++m) {
                float acc[NT][4];
                #pragma unroll
                for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
                #pragma unroll
                for (int s = 0; s < KS; ++s) {
                    if (SP && !((lt >> m) & 1u)) break;  // no output of this tile is stored
                    const uint4 af = FS ? s_frag[(m * KS + s) * 32 + lane] : frag[(m * KS + s) * 32 + lane];
                    #pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        if (K8) {
                            O::mma8(acc[j], af.x, af.y, bf[j][0][0]);
                        } else {
                            const uint32_t a4[4] = {af.x, af.y, af.z, af.w};
                            O::mma16(acc[j], a4, bf[j][s][0], bf[j][s][1]);
                        }
                    }
                }
                // SP: outputs that nothing reads are not stored (their HBM writes
                // are the saving; the contraction itself stays branch free)
                const uint32_t k0 = uint32_t(8 * m + g);
                const bool live = SP ? ((lm >> m) & 1u) != 0 : k0 < uint32_t(R0);
                #pragma unroll
                for (int j = 0; j < NT; ++j) {
                    if (live) {
                        const uint32_t o = uint32_t(o_base + 8 * (warp + 8 * (NT * i + j)) + 2 * t);
                        const cpx v0 = cmul({acc[j][0], acc[j][2]}, tw[j][0]);
                        const cpx v1 = cmul({acc[j][1], acc[j][3]}, tw[j][1]);
                        *reinterpret_cast<uint2*>(Trow + long(k0) * L + o) =
                            make_uint2(O::pack(v0.r, v0.i), O::pack(v1.r, v1.i));
                    }
                    if (m + 1 < MT) {
                        tw[j][0] = cmul(tw[j][0], ts[j][0]);
                        tw[j][1] = cmul(tw[j][1], ts[j][1]);
                    }
                }
            }
        }
        __syncthreads();  // staging is reused by the next item
    }
}

// ------------------------------------------------------------------ pass C
// Warps per CTA: 16 when the staged segments leave room for one CTA per SM.
template <int R0>
__host__ __device__ constexpr int mp_pass_c_warps() { return R0 >= 128 ? 16 : 8; }

// TWID: T still lacks the W_M^(n'*k0) twiddle (tensor-core pass B); it is
// applied here to each element before the contraction, as the chain
// W_M^(n' t) * W_M^(8 n')^s (and * W_M^(4 n')) for k0 = 8s + t (+ 4).
// TOT: an inner outer stage of a two-level outer factor: all R0 outputs,
// neither conjugated nor gated, written back over the staged tile of T.
// SP: frequency-sparse plan: dead sub-rows (a.zbits) are not loaded and count
// as zeros; chunks of eight dead sub-rows are skipped.
template <int DT, int R0, bool GATED, int L, bool TWID, bool TOT = false, bool SP = false>
__global__ void __launch_bounds__(32 * mp_pass_c_warps<R0>(), (R0 <= 64 && !TOT) ? 3 : (R0 <= 64 ? 2 : 1))
    mp_pass_c(const MPArgs a) {
    using O = Op<DT>;
    static_assert(!(TOT && GATED), "the inner stage has no gates");
    constexpr int HALF = R0 / 2, SEG = mp_seg<R0>(), TILE = mp_tile<R0>();
    constexpr int NOUT = TOT ? R0 : HALF;  // outputs kept
    constexpr long M = long(R0) * L;
    constexpr bool K8 = R0 <= 4;
    constexpr int KS = K8 ? 1 : R0 / 8, MT = (NOUT + 7) / 8;
    const uint4* frag = TOT ? a.tb.ofull : a.tb.oi_c;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t* st = reinterpret_cast<uint32_t*>(smem);  // [R0][SEG]
    uint32_t* swo = st + R0 * SEG;                      // gated: w_out [HALF][SEG]
    uint64_t* bar = reinterpret_cast<uint64_t*>(swo + (GATED ? HALF * SEG : 0));
    __shared__ int s_fail;
    // the DFT fragments staged once per CTA in shared memory where that keeps
    // the resident CTAs (the in-place stage and R0 <= 32), else read through L1
    constexpr bool FS = (TOT || R0 <= 32) && MT * KS * 32 * 16 <= 32768;
    constexpr int UNR = FS ? 2 : MT;  // full unroll keeps the L1 fragment loads ahead
    __shared__ uint4 s_frag[FS ? MT * KS * 32 : 1];
    if (FS)
        for (int i = threadIdx.x; i < MT * KS * 32; i += blockDim.x) s_frag[i] = frag[i];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    const long rows = long(a.B) * a.H, tiles = L / TILE, items = rows * tiles;
    // SP, last pass: one set of dead sub-rows for the whole launch; their
    // staged segments are cleared once and never copied into.  SP, in-place
    // stage: the set depends on the row's group, so dead inputs are masked
    // per load instead.
    constexpr bool CLR = SP && !TOT, ROWP = SP && TOT;
    uint32_t lc_fixed = 0;  // CLR: bit s set when the chunk 8s .. 8s + 7 holds a live sub-row
    if constexpr (CLR) {
        const unsigned long long z0 = a.zbits ? __ldg(a.zbits) : 0ull, z1 = a.zbits ? __ldg(a.zbits + 1) : 0ull;
        for (int k0 = 0; k0 < R0; ++k0)
            if (zbit(z0, z1, k0))
                for (int c = threadIdx.x; c < TILE / 4; c += blockDim.x)
                    reinterpret_cast<uint4*>(st + k0 * SEG)[c] = make_uint4(0u, 0u, 0u, 0u);
        #pragma unroll
        for (int s = 0; s < KS; ++s) {
            const int kc = 8 * s;
            if ((((kc < 64 ? z0 >> kc : z1 >> (kc - 64))) & 0xffull) != 0xffull) lc_fixed |= 1u << s;
        }
    }
    if (threadIdx.x == 0) {
        s_fail = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    uint32_t par = 0;
    __shared__ unsigned long long s_z[2];  // ROWP: dead sub-rows of this item
    for (long item = blockIdx.x; item < items; item += gridDim.x, par ^= 1) {
        const long row = item / tiles;
        const int o_base = int(item % tiles) * TILE;
        if (threadIdx.x == 0) {
            if constexpr (!SP) {
                mbar_expect_tx(bar, (R0 + (GATED ? HALF : 0)) * TILE * 4u);
                for (int k0 = 0; k0 < R0; ++k0)
                    bulk_g2s(st + k0 * SEG, a.T + row * M + long(k0) * L + o_base, TILE * 4, bar);
            } else {  // dead sub-rows are not loaded; their inputs are taken as zeros
                const unsigned long long z0 = a.zbits ? __ldg(a.zbits + 2 * (row % a.zmod)) : 0ull;
                const unsigned long long z1 = a.zbits ? __ldg(a.zbits + 2 * (row % a.zmod) + 1) : 0ull;
                s_z[0] = z0;
                s_z[1] = z1;
                const int live = R0 - __popcll(z0) - __popcll(z1);  // bits exist for k0 < R0 only
                mbar_expect_tx(bar, (live + (GATED ? HALF : 0)) * TILE * 4u);
                for (int k0 = 0; k0 < R0; ++k0)
                    if (!zbit(z0, z1, k0))
                        bulk_g2s(st + k0 * SEG, a.T + row * M + long(k0) * L + o_base, TILE * 4, bar);
            }
            if (GATED)
                for (int n0 = 0; n0 < HALF; ++n0)
                    bulk_g2s(swo + n0 * SEG, a.w_out + row * M + 2 * (long(L) * n0 + o_base), TILE * 4, bar);
        }
        if (!cta_wait(bar, par, &s_fail, a.err)) return;
        // ROWP: bit s of la / lb: this thread's input row 8s + t / 8s + 4 + t
        // is live; bit s of lc (the same in every thread): some row of the chunk
        // 8s .. 8s + 7 is live, else the chunk's twiddles and products are skipped
        uint32_t la = 0, lb = 0, lc = lc_fixed;
        if constexpr (ROWP) {
            #pragma unroll
            for (int s = 0; s < KS; ++s) {
                const int ka = 8 * s + t, kb = 8 * s + 4 + t, kc = 8 * s;
                if (!((s_z[ka >> 6] >> (ka & 63)) & 1ull)) la |= 1u << s;
                if (!((s_z[kb >> 6] >> (kb & 63)) & 1ull)) lb |= 1u << s;
                if (((s_z[kc >> 6] >> (kc & 63)) & 0xffull) != 0xffull) lc |= 1u << s;
            }
        }
        // NT column groups of 8 per iteration share each DFT fragment load.
        // CHAIN (R0 <= 8): the columns advance by 8 NW NT per iteration, so the
        // input twiddles W_M^(n' t) and W_M^(4 n') are carried from one
        // iteration to the next by constant factors instead of recomputed
        constexpr int NT = KS <= 8 ? 2 : 1, NW = mp_pass_c_warps<R0>();
        constexpr bool CHAIN = TWID && R0 <= 8;
        constexpr uint32_t CSTEP = 8u * NW * NT;
        cpx ca[NT], c4[NT], sa, s4;
        if constexpr (CHAIN) {
            #pragma unroll
            for (int j = 0; j < NT; ++j) {
                const uint32_t np = uint32_t(o_base + 8 * (warp + NW * j) + g);
                ca[j] = twiddle_pow2((np * uint32_t(t)) & (uint32_t(M) - 1), uint32_t(M));
                c4[j] = twiddle_pow2((4 * np) & (uint32_t(M) - 1), uint32_t(M));
            }
            sa = twiddle_pow2((CSTEP * uint32_t(t)) & (uint32_t(M) - 1), uint32_t(M));
            s4 = twiddle_pow2((4 * CSTEP) & (uint32_t(M) - 1), uint32_t(M));
        }
        #pragma unroll 1
        for (int i = 0; i < TILE / 8 / NW / NT; ++i) {
            uint32_t bf[NT][KS][2];
            #pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int nt = warp + NW * (NT * i + j);
                #pragma unroll
                for (int s = 0; s < KS; ++s) {
                    const int ka = 8 * s + t, kb = 8 * s + 4 + t;
                    const bool va = ka < R0 && (!ROWP || ((la >> s) & 1u));
                    const bool vb = !K8 && kb < R0 && (!ROWP || ((lb >> s) & 1u));
                    bf[j][s][0] = va ? st[ka * SEG + 8 * nt + g] : 0u;
                    bf[j][s][1] = vb ? st[kb * SEG + 8 * nt + g] : 0u;
                }
                if constexpr (TWID && K8) {  // one input k0 = t per thread
                    const uint32_t np = uint32_t(o_base + 8 * nt + g);
                    cpx w;
                    if constexpr (CHAIN) {
                        w = ca[j];
                        ca[j] = cmul(ca[j], sa);
                    } else {
                        w = twiddle_pow2((np * uint32_t(t)) & (uint32_t(M) - 1), uint32_t(M));
                    }
                    const cpx xa = cmul(O::unpack(bf[j][0][0]), w);
                    bf[j][0][0] = O::pack(xa.r, xa.i);
                }
                if constexpr (TWID && !K8) {
                    static_assert(R0 % 8 == 0, "twiddled pass C needs R0 = 4 or a multiple of 8");
                    const uint32_t np = uint32_t(o_base + 8 * nt + g);
                    const uint32_t mask = uint32_t(M) - 1;
                    cpx wa, w4;
                    if constexpr (CHAIN) {
                        wa = ca[j];
                        w4 = c4[j];
                        ca[j] = cmul(ca[j], sa);
                        c4[j] = cmul(c4[j], s4);
                    } else {
                        wa = twiddle_pow2((np * uint32_t(t)) & mask, uint32_t(M));
                        w4 = twiddle_pow2((4 * np) & mask, uint32_t(M));
                    }
                    const cpx w8 = KS > 1 ? twiddle_pow2((8 * np) & mask, uint32_t(M)) : cpx{1.f, 0.f};
                    #pragma unroll
                    for (int s = 0; s < KS; ++s) {
                        if (!SP || ((lc >> s) & 1u)) {
                            const cpx xa = cmul(O::unpack(bf[j][s][0]), wa);
                            const cpx xb = cmul(O::unpack(bf[j][s][1]), cmul(wa, w4));
                            bf[j][s][0] = O::pack(xa.r, xa.i);
                            bf[j][s][1] = O::pack(xb.r, xb.i);
                        }
                        if (s + 1 < KS) wa = cmul(wa, w8);
                    }
                }
            }
            #pragma unroll UNR
            for (int m = 0; m < MT; ++m) {
                float acc[NT][4];
                #pragma unroll
                for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
                #pragma unroll
                for (int s = 0; s < KS; ++s) {
                    if (SP && !K8 && !((lc >> s) & 1u)) continue;  // all eight inputs are zero
                    const uint4 af = FS ? s_frag[(m * KS + s) * 32 + lane] : frag[(m * KS + s) * 32 + lane];
                    #pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        if (K8) {
                            O::mma8(acc[j], af.x, af.y, bf[j][0][0]);
                        } else {
                            const uint32_t a4[4] = {af.x, af.y, af.z, af.w};
                            O::mma16(acc[j], a4, bf[j][s][0], bf[j][s][1]);
                        }
                    }
                }
                const int n0 = 8 * m + g;
                if (TOT && n0 < NOUT) {
                    #pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const int nt = warp + NW * (NT * i + j);
                        *reinterpret_cast<uint2*>(a.T + row * M + long(L) * n0 + o_base + 8 * nt + 2 * t) =
                            make_uint2(O::pack(acc[j][0], acc[j][2]), O::pack(acc[j][1], acc[j][3]));
                    }
                } else if (!TOT && n0 < HALF) {
                    #pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const int nt = warp + NW * (NT * i + j);
                        const long p = long(L) * n0 + o_base + 8 * nt + 2 * t;  // reals 2p..2p+3
                        float r0 = acc[j][0], i0 = -acc[j][2], r1 = acc[j][1], i1 = -acc[j][3];
                        if (GATED) {
                            const uint2 wv = *reinterpret_cast<const uint2*>(swo + n0 * SEG + 8 * nt + 2 * t);
                            const cpx w0 = O::unpack(wv.x), w1 = O::unpack(wv.y);
                            r0 *= w0.r; i0 *= w0.i; r1 *= w1.r; i1 *= w1.i;
                        }
                        *reinterpret_cast<uint2*>(a.y + row * M + 2 * p) =
                            make_uint2(O::pack(r0, i0), O::pack(r1, i1));
                    }
                }
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ pass B
constexpr size_t kMpBFrag = size_t(8) * 8 * 32 * 16;  // F_64/8 A fragments, resident in shared memory
constexpr size_t kMpBSmem = size_t(2) * kMpR1 * kSeg * 4 + 256 * 8 + kMpBFrag + 32;

// SP: frequency-sparse plan: only the a.np pairs listed in a.plist run.
template <int DT, bool SP = false>
__global__ void __launch_bounds__(512, 1) mp_pass_b(const MPArgs a) {
    using O = Op<DT>;
    constexpr int L = kMpL, R1 = kMpR1, SEG = kSeg;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t* rbuf = reinterpret_cast<uint32_t*>(smem);                 // [2][R1][SEG]
    cpx* scratch = reinterpret_cast<cpx*>(rbuf + 2 * R1 * SEG);         // [256]
    uint4* ofull = reinterpret_cast<uint4*>(scratch + 256);             // [8][8][lane]
    uint64_t* bar = reinterpret_cast<uint64_t*>(ofull + 8 * 8 * 32);    // items, table
    __shared__ int s_fail;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    const int R0 = a.R0;
    const uint32_t M = uint32_t(R0) * L;
    const long rows = long(a.B) * a.H, np = SP ? a.np : R0 / 2, items = rows * np;
    if (threadIdx.x == 0) {
        s_fail = 0;
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        fence_mbar_init();
        mbar_expect_tx(bar + 1, uint32_t(kMpBFrag));
        bulk_g2s(ofull, a.tb.ofull, uint32_t(kMpBFrag), bar + 1);
    }
    __syncthreads();
    Inner<DT> in;
    in.load({a.tb.lf, a.tb.rf, a.tb.tw, nullptr, 0, 0, 0, 0}, lane);
    if (!cta_wait(bar + 1, 0, &s_fail, a.err)) return;
    uint32_t par = 0;
    for (long item = blockIdx.x; item < items; item += gridDim.x, par ^= 1) {
        // items channel-major with b fastest: the B rows of one channel use the
        // same k_f sub-rows at about the same time, so k_f is read from HBM once
        const long b = item % a.B, hp = item / a.B;
        const int p = SP ? int(__ldg(a.plist + hp % np)) : int(hp % np);
        const long h = hp / np, row = b * a.H + h;
        const int k0s[2] = {p == 0 ? 0 : p, p == 0 ? R0 / 2 : R0 - p};
        uint32_t* Trow = a.T + row * long(M);
        if (threadIdx.x == 0) {
            mbar_expect_tx(bar, 2u * R1 * 1024u);
            for (int side = 0; side < 2; ++side)
                for (int n1 = 0; n1 < R1; ++n1)
                    bulk_g2s(rbuf + (side * R1 + n1) * SEG, Trow + long(k0s[side]) * L + 256 * n1, 1024, bar);
        }
        if (!cta_wait(bar, par, &s_fail, a.err)) return;

        // full 64-point outer stage, in place (each warp owns 8 columns)
        #pragma unroll 1
        for (int job = warp; job < 64; job += 16) {
            uint32_t* rs = rbuf + (job >> 5) * R1 * SEG;
            const int nt = job & 31;
            uint32_t bf[8][2];
            #pragma unroll
            for (int s = 0; s < 8; ++s) {
                bf[s][0] = rs[(8 * s + t) * SEG + 8 * nt + g];
                bf[s][1] = rs[(8 * s + 4 + t) * SEG + 8 * nt + g];
            }
            #pragma unroll 1
            for (int m = 0; m < 8; ++m) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                #pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint4 af = ofull[(m * 8 + s) * 32 + lane];
                    const uint32_t a4[4] = {af.x, af.y, af.z, af.w};
                    O::mma16(acc, a4, bf[s][0], bf[s][1]);
                }
                const float4 v = cmul2_split(acc[0], acc[1], acc[2], acc[3], a.tb.twf[(nt * 8 + m) * 32 + lane]);
                *reinterpret_cast<uint2*>(rs + (8 * m + g) * SEG + 8 * nt + 2 * t) =
                    make_uint2(O::pack(v.x, v.z), O::pack(v.y, v.w));
            }
        }
        __syncthreads();

        // sub-problem pairs: 256-point transforms, fold, and back
        #pragma unroll 1
        for (int un = warp; un < 64; un += 16) {
            int sa, sb, ka, kb;
            bool fusedlike = false;
            if (p == 0 && un < 32) {  // sub-row 0 pairs with itself: kappa <-> L - kappa
                fusedlike = true;
                sa = sb = 0;
                ka = un;
                kb = un == 0 ? R1 / 2 : R1 - un;
            } else if (p == 0) {      // sub-row R0/2 pairs with itself: kappa <-> L-1-kappa
                sa = sb = 1;
                ka = un - 32;
                kb = R1 - 1 - ka;
            } else {                  // sub-rows k0 and R0-k0: kappa <-> L-1-kappa
                sa = 0;
                sb = 1;
                ka = un;
                kb = R1 - 1 - un;
            }
            uint32_t* ra = rbuf + sa * R1 * SEG + ka * SEG + 16 * t + g;
            uint32_t* rbp = rbuf + sb * R1 * SEG + kb * SEG + 16 * t + g;
            cpx za[8], zb[8], pp[8];
            in.forward_at(ra, ra + 8, za);
            in.forward_at(rbp, rbp + 8, zb);
            const uint4* fa = a.kf + (size_t((h * R0 + k0s[sa]) * R1 + ka) * 4) * 32 + lane;
            const uint4* fb = a.kf + (size_t((h * R0 + k0s[sb]) * R1 + kb) * 4) * 32 + lane;
            if (fusedlike && un == 0) {
                // sub-problem R1/2 with itself through lane ^ 31; sub-problem 0
                // pairs bin kappa' with (256 - kappa') mod 256 of itself
                #pragma unroll
                for (int i = 0; i < 8; ++i) pp[i] = shfl31(zb[7 - i]);
                #pragma unroll
                for (int i = 0; i < 8; ++i) scratch[(g + 8 * (i >> 2)) + 16 * (4 * (i & 3) + t)] = za[i];
                __syncwarp();
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = fa[q * 32];
                    #pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        const int i = 2 * q + sl;
                        const int kap = (g + 8 * (i >> 2)) + 16 * (4 * (i & 3) + t);
                        za[i] = dit_fold<DT>(sl ? v.z : v.x, sl ? v.w : v.y, za[i], scratch[(256 - kap) & 255]);
                    }
                }
                __syncwarp();
            } else {
                #pragma unroll
                for (int i = 0; i < 8; ++i) pp[i] = shfl31(za[7 - i]);
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = fa[q * 32];
                    #pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        const int i = 2 * q + sl;
                        za[i] = dit_fold<DT>(sl ? v.z : v.x, sl ? v.w : v.y, za[i], shfl31(zb[7 - i]));
                    }
                }
            }
            #pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 v = fb[q * 32];
                #pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const int i = 2 * q + sl;
                    zb[i] = dit_fold<DT>(sl ? v.z : v.x, sl ? v.w : v.y, zb[i], pp[i]);
                }
            }
            #pragma unroll
            for (int side = 0; side < 2; ++side) {
                const int k1 = side ? kb : ka;
                uint32_t* dst = side ? rbp : ra;  // (n2 = t, n3 = g) of sub-problem k1
                cpx w[8];
                in.inverse(side ? zb : za, w);
                #pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const float4 tv = a.tb.twi[(k1 * 4 + nt) * 32 + lane];
                    const cpx v0 = cmul(w[nt], {tv.x, tv.y});
                    const cpx v1 = cmul(w[4 + nt], {tv.z, tv.w});
                    dst[64 * nt] = O::pack(v0.r, v0.i);
                    dst[64 * nt + 8] = O::pack(v1.r, v1.i);
                }
            }
        }
        __syncthreads();

        // full 64-point inverse outer stage, pass-A twiddle, back to T
        #pragma unroll 1
        for (int job = warp; job < 64; job += 16) {
            const int side = job >> 5, nt = job & 31;
            const uint32_t* rs = rbuf + side * R1 * SEG;
            const uint32_t k0 = uint32_t(k0s[side]);
            uint32_t bf[8][2];
            #pragma unroll
            for (int s = 0; s < 8; ++s) {
                bf[s][0] = rs[(8 * s + t) * SEG + 8 * nt + g];
                bf[s][1] = rs[(8 * s + 4 + t) * SEG + 8 * nt + g];
            }
            uint32_t* To = Trow + long(k0) * L;
            #pragma unroll 1
            for (int m = 0; m < 8; ++m) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                #pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint4 af = ofull[(m * 8 + s) * 32 + lane];
                    const uint32_t a4[4] = {af.x, af.y, af.z, af.w};
                    O::mma16(acc, a4, bf[s][0], bf[s][1]);
                }
                const uint32_t np = uint32_t(256 * (8 * m + g) + 8 * nt + 2 * t);
                const cpx v0 = cmul({acc[0], acc[2]}, twiddle_pow2((np * k0) & (M - 1), M));
                const cpx v1 = cmul({acc[1], acc[3]}, twiddle_pow2(((np + 1) * k0) & (M - 1), M));
                *reinterpret_cast<uint2*>(To + np) = make_uint2(O::pack(v0.r, v0.i), O::pack(v1.r, v1.i));
            }
        }
        __syncthreads();  // the row buffers are refilled by the next item
    }
}

}  // namespace fftconv
