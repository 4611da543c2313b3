// The two-level outer factor of the multi-pass path (M = RA * 64 * 4096
// complex points, RA = 4 or 8) in one pass per direction on the
// fifth-generation tensor cores: the RA-point level in registers and the
// 64-point level as one contraction, so that the intermediate T crosses HBM
// once on the way in and once on the way out.
//
// FlashFFTConv page, section 3.4 "Kernel Fusion and Recomputation
// Strategies": the outer Monarch factors go through HBM, the inner ones stay
// on chip; "Higher-order decompositions": the order-p factorization.  With
// n = L1 n_a + 4096 n_b + n_c and k = k_a + RA k_b + 64 RA k_c (L1 = 64 *
// 4096), W_M^(nk) splits into W_RA^(n_a k_a) W_(64 RA)^(n_b k_a)
// W_64^(n_b k_b) W_M^(n_c (k_a + RA k_b)) W_4096^(n_c k_c), so
//   pass A  T[64 k_a + k_b][n_c] = W_M^(n_c k0) sum_(n_b) W_64^(n_b k_b)
//             W_(64 RA)^(n_b k_a) sum_(n_a < RA/2) W_RA^(n_a k_a) z[n_a][n_b][n_c]
//             / sqrt(64 RA),   k0 = k_a + RA k_b
//           (z: the packed row of u, times w_in; n_a >= RA/2 is the zero half)
//   pass C  out[n_a][n_b][n_c] = sum_(k_a) W_RA^(n_a k_a) W_(64 RA)^(n_b k_a)
//             sum_(k_b) W_64^(n_b k_b) W_M^(n_c k0) T[64 k_a + k_b][n_c] / sqrt(64 RA),
//           only n_a < RA/2 (the causal truncation), y_z = conj(out) (times w_out)
// and pass B transforms the 4096-point sub-rows at positions 64 k_a + k_b
// (the inverse transform is the forward one of the conjugate spectrum that
// pass B leaves in T, conjugated at the store).
//
// A tile is TC = 128 / RA columns n_c of one row.  Its staged rows arrive by
// the TMA engine (pass A: the RA/2 x 64 nonzero rows of z; pass C: all RA x
// 64 rows of T).  The contraction is D = X F with M = 128 rows (k_a, n_c) =
// (m / TC, m % TC), K = the 64 complex inputs real-embedded, N = the 64
// complex outputs (F: the 64-point DFT matrix / 8, both operands in shared
// memory, D float32 in tensor memory):
//   pass A  X[(k_a, n_c)][n_b] = W_(64 RA)^(n_b k_a) / sqrt(RA) x the RA-point
//           transform of the staged column (a radix-RA butterfly per thread)
//   pass C  X[(k_a, n_c)][k_b] = W_M^(n_c k0) T[64 k_a + k_b][n_c]
// In pass A's epilogue tensor-memory lane m is row (k_a, n_c): the thread
// applies W_M^(n_c k0) along k_b (a product chain) and writes T.  In pass
// C's, the thread applies W_(64 RA)^(n_b k_a) / sqrt(RA) and parks the
// results in shared memory (the A operand's space); a last phase reads the
// RA values of each (n_b, n_c), applies the radix-RA butterfly for the
// outputs n_a < RA/2 and writes y.
#pragma once
#include <cuda.h>

#include "multipass.cuh"
#include "tc.cuh"

namespace fftconv {

template <int RA>
struct Otc2 {
    static_assert(RA == 4 || RA == 8, "two-level outer factor: RA = 4 or 8");
    static constexpr int L = 4096, L1 = 64 * L, NA = RA / 2;
    static constexpr uint32_t M = uint32_t(RA) * L1;
    static constexpr int TC = 128 / RA;     // columns per tile
    static constexpr int TILES = L / TC;    // tiles per row
    static constexpr int THREADS = 256;
    static constexpr int TPC = THREADS / TC;  // threads per column
    static constexpr int NBT = 64 / TPC;      // sub-rows per thread in the reformat and the last phase
    // operands: 128 rows x K = 128 (16-bit), K-major without swizzle:
    // element (row, k) at (row/8) SBO + (k/8) LBO + (row%8) 16 + (k%8) 2 bytes
    static constexpr uint32_t LBO = 128, SBO = 16 * 128;
    static constexpr uint32_t ABYTES = 16 * SBO, BBYTES = 16 * SBO;
    // W_(64 RA)^(n_b k_a) / sqrt(RA) as pairs (re, re', im, im') for packed
    // f32x2 products: pass A pairs k_a with k_a + RA/2, [k_a < RA/2][n_b];
    // pass C pairs n_b with n_b + 1, [k_a][n_b / 2]
    static constexpr uint32_t TABB = uint32_t(RA) * 64 * 8;
    static constexpr int TMEM_COLS = 128;                    // one accumulator of 128 float32 columns
};

template <int RA, bool FWD, bool GATED>
struct Otc2Pass {
    using C = Otc2<RA>;
    static constexpr int NIN = FWD ? C::NA * 64 : RA * 64;           // staged rows
    static constexpr int BOXR = NIN < 256 ? NIN : 256;               // rows per tensor copy
    static constexpr int NBOX = NIN / BOXR;
    static constexpr uint32_t STAGE_WORDS = uint32_t(NIN) * C::TC;   // 16 KB (A) / 32 KB (C)
    static constexpr int NST = (FWD && !GATED) ? 2 : 1;              // staged tiles in flight
    static constexpr int NGATE = (FWD && GATED) ? NST : 0;           // pass A: w_in staged beside u
    static constexpr size_t OFF_B = C::ABYTES, OFF_ST = OFF_B + C::BBYTES;
    static constexpr size_t OFF_TAB = OFF_ST + size_t(NST + NGATE) * STAGE_WORDS * 4;
    static constexpr size_t OFF_BAR = OFF_TAB + C::TABB;
    static constexpr size_t SMEM = OFF_BAR + size_t(NST + 2) * 8 + 16;
};

// The RA-point transform of x[n_a], n_a < RA/2 (the rest zero):
// X[k] = sum_(n_a) W_RA^(n_a k) x[n_a].
template <int RA>
__device__ __forceinline__ void otc2_fwd_radix(const cpx (&x)[RA / 2], cpx (&X)[RA]) {
    if constexpr (RA == 4) {
        X[0] = {x[0].r + x[1].r, x[0].i + x[1].i};
        X[1] = {x[0].r + x[1].i, x[0].i - x[1].r};  // x0 - i x1
        X[2] = {x[0].r - x[1].r, x[0].i - x[1].i};
        X[3] = {x[0].r - x[1].i, x[0].i + x[1].r};  // x0 + i x1
    } else {
        // E[k] = x0 + W_4^k x2, P[k] = x1 + W_4^k x3, X[k] = E[k] + W_8^k P[k], X[k + 4] = E[k] - W_8^k P[k]
        const cpx E[4] = {{x[0].r + x[2].r, x[0].i + x[2].i},
                          {x[0].r + x[2].i, x[0].i - x[2].r},
                          {x[0].r - x[2].r, x[0].i - x[2].i},
                          {x[0].r - x[2].i, x[0].i + x[2].r}};
        const cpx P[4] = {{x[1].r + x[3].r, x[1].i + x[3].i},
                          {x[1].r + x[3].i, x[1].i - x[3].r},
                          {x[1].r - x[3].r, x[1].i - x[3].i},
                          {x[1].r - x[3].i, x[1].i + x[3].r}};
        constexpr float h = 0.70710678118654752f;
        const cpx O[4] = {P[0],
                          {h * (P[1].r + P[1].i), h * (P[1].i - P[1].r)},     // (1 - i)/sqrt2 P1
                          {P[2].i, -P[2].r},                                  // -i P2
                          {h * (P[3].i - P[3].r), -h * (P[3].r + P[3].i)}};   // (-1 - i)/sqrt2 P3
        #pragma unroll
        for (int k = 0; k < 4; ++k) {
            X[k] = {E[k].r + O[k].r, E[k].i + O[k].i};
            X[k + 4] = {E[k].r - O[k].r, E[k].i - O[k].i};
        }
    }
}

// The outputs n < RA/2 of the RA-point transform of v[k], k < RA:
// out[n] = sum_(k) W_RA^(n k) v[k].
template <int RA>
__device__ __forceinline__ void otc2_half_radix(const cpx (&v)[RA], cpx (&out)[RA / 2]) {
    if constexpr (RA == 4) {
        out[0] = {v[0].r + v[1].r + v[2].r + v[3].r, v[0].i + v[1].i + v[2].i + v[3].i};
        // v0 - i v1 - v2 + i v3
        out[1] = {v[0].r + v[1].i - v[2].r - v[3].i, v[0].i - v[1].r - v[2].i + v[3].r};
    } else {
        // E[n], O[n]: the 4-point transforms of the even and odd inputs;
        // out[n] = E[n] + W_8^n O[n], n < 4
        auto dft4 = [](cpx a, cpx b, cpx c, cpx d, cpx (&r)[4]) {
            const cpx s0 = {a.r + c.r, a.i + c.i}, s1 = {a.r - c.r, a.i - c.i};
            const cpx s2 = {b.r + d.r, b.i + d.i}, s3 = {b.r - d.r, b.i - d.i};
            r[0] = {s0.r + s2.r, s0.i + s2.i};
            r[1] = {s1.r + s3.i, s1.i - s3.r};  // s1 - i s3
            r[2] = {s0.r - s2.r, s0.i - s2.i};
            r[3] = {s1.r - s3.i, s1.i + s3.r};  // s1 + i s3
        };
        cpx E[4], O[4];
        dft4(v[0], v[2], v[4], v[6], E);
        dft4(v[1], v[3], v[5], v[7], O);
        constexpr float h = 0.70710678118654752f;
        out[0] = {E[0].r + O[0].r, E[0].i + O[0].i};
        out[1] = {E[1].r + h * (O[1].r + O[1].i), E[1].i + h * (O[1].i - O[1].r)};  // (1 - i)/sqrt2
        out[2] = {E[2].r + O[2].i, E[2].i - O[2].r};                               // -i
        out[3] = {E[3].r + h * (O[3].i - O[3].r), E[3].i - h * (O[3].r + O[3].i)};  // (-1 - i)/sqrt2
    }
}

// Word index of the parked value (k_a, n_b, column c) of pass C in the A
// space (RA x 64 x TC words).  RA = 8 (TC = 16): rows of 32 words hold k_a
// pairs, the half of a row swapped by bit 2 of n_b, so that the epilogue's
// warps (two k_a, 16 columns, one n_b) and the last phase's (one k_a, 16
// columns, n_b four apart) each touch 32 distinct banks.
template <int RA>
__device__ __forceinline__ int otc2_park(int ka, int nb, int c) {
    if constexpr (RA == 8)
        return (((ka >> 1) * 64 + nb) << 5) + ((((ka & 1) ^ (nb >> 2)) & 1) << 4) + c;
    else
        return ((ka * 64 + nb) << 5) + c;
}

// Frequency-sparse plans (SP): the sub-rows whose pass-B pair is skipped
// (bit k_b of zbits[2 k_a], never written by pass B) are not stored by pass
// A and read as zeros by pass C.  Pass C still copies every row of a tile:
// per-k_a boxes of only the live runs (a few rows of 64 bytes each) made the
// copies latency-bound (275 us against 102 us for all rows on gene-2m with
// band 5, 8, 33, 33).

// fmat: the 64-point DFT matrix / 8 as the B operand; tab: this pass's
// W_(64 RA)^(n_b k_a) / sqrt(RA) pairs (Otc2::TABB bytes); tin: pass A u as 32-bit words [rows][RA/2
// x 64][4096], pass C T [rows][RA x 64][4096]; tgate: w_in in u's shape.
template <int DT, int RA, bool FWD, bool GATED, bool SP = false>
__global__ void __launch_bounds__(256, 2) otc2_pass(const MPArgs a, const uint8_t* __restrict__ fmat,
                                                 const float4* __restrict__ tab,
                                                 const __grid_constant__ CUtensorMap tin,
                                                 const __grid_constant__ CUtensorMap tgate) {
    using O = Op<DT>;
    using C = Otc2<RA>;
    using P = Otc2Pass<RA, FWD, GATED>;
    constexpr int TC = C::TC, NBT = C::NBT;
    constexpr uint32_t M = C::M;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sa = smem;                                                  // A operand (pass C: then the parked outputs)
    uint8_t* sf = smem + P::OFF_B;                                       // DFT matrix
    uint32_t* st = reinterpret_cast<uint32_t*>(smem + P::OFF_ST);        // [NST][NIN][TC]
    uint32_t* sw = st + P::NST * P::STAGE_WORDS;                         // pass A gated: w_in
    const float4* s_tab = reinterpret_cast<const float4*>(smem + P::OFF_TAB);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + P::OFF_BAR);     // [NST]
    uint64_t* mbar = full + P::NST;                                      // contraction done
    uint64_t* fbar = mbar + 1;                                           // matrix and table arrived
    uint32_t& s_tmem = *reinterpret_cast<uint32_t*>(fbar + 1);

    const int t = threadIdx.x, wq = t >> 5;
    const long rows = long(a.B) * a.H;
    const long items = rows * C::TILES;
    const long first_item = blockIdx.x, stride = gridDim.x;

    auto stage = [&](long item, int s) {
        const int row = int(item / C::TILES);
        const int o_base = int(item % C::TILES) * TC;
        mbar_expect_tx(&full[s], P::STAGE_WORDS * 4u * (P::NGATE ? 2u : 1u));
        #pragma unroll
        for (int bx = 0; bx < P::NBOX; ++bx)
            tma_load_3d(st + s * P::STAGE_WORDS + bx * P::BOXR * TC, &tin, o_base, bx * P::BOXR, row, &full[s]);
        if constexpr (P::NGATE > 0) tma_load_3d(sw + s * P::STAGE_WORDS, &tgate, o_base, 0, row, &full[s]);
    };

    uint32_t issued = 0;
    bool mma_pending = false;
    if (t == 0) {
        for (int s = 0; s < P::NST + 2; ++s) mbar_init(full + s, 1);
        fence_mbar_init();
        mbar_expect_tx(fbar, C::BBYTES + C::TABB);
        bulk_g2s(sf, fmat, C::BBYTES, fbar);
        bulk_g2s(smem + P::OFF_TAB, tab, C::TABB, fbar);
        for (int s = 0; s < P::NST; ++s)
            if (first_item + s * stride < items) {
                stage(first_item + s * stride, s);
                issued |= 1u << s;
            }
    }
    if (wq == 0) tc::alloc(&s_tmem, C::TMEM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    bool failed = __syncthreads_or(!mbar_wait_bounded(fbar, 0, kWaitLimit));

    // reformat and last phase: column c of the tile, sub-rows [NBT g, NBT g + NBT)
    const int c = t % TC, g = t / TC, nb0 = NBT * g;
    // epilogue: tensor-memory lane 32 (warp % 4) + lane = row (k_a, column);
    // the warps of a lane quarter split the 64 outputs
    const int eq = wq & 3, eh = wq >> 2;
    const int em = 32 * eq + (t & 31), eka = em / TC, ec = em % TC;
    constexpr int EOUT = 64 / (C::THREADS / 128);  // outputs per thread in the epilogue

    uint32_t par = 0, mpar = 0;  // bit s: the phase of staging slot s
    long li = 0;
    for (long item = first_item; item < items && !failed; item += stride, ++li) {
        const int s = int(li % P::NST);
        const long row = item / C::TILES;
        const int o_base = int(item % C::TILES) * TC;
        bool bad = !mbar_wait_sleep(&full[s], (par >> s) & 1u, kWaitSleepLimit, kWaitHintNs);
        if (!bad) {
            par ^= 1u << s;
            issued &= ~(1u << s);
        }
        if (__syncthreads_or(bad)) { failed = true; break; }

        // ---------------- the staged column -> row (k_a, c) of the A operand
        {
            const uint32_t* sts = st + s * P::STAGE_WORDS + c;
            const uint32_t n_c = uint32_t(o_base + c);
            if constexpr (FWD) {
                const uint32_t* sws = sw + s * P::STAGE_WORDS + c;
                uint32_t w[RA][NBT];
                #pragma unroll
                for (int i = 0; i < NBT; ++i) {
                    const int nb = nb0 + i;
                    cpx x[C::NA];
                    #pragma unroll
                    for (int na = 0; na < C::NA; ++na) {
                        uint32_t v = sts[(na * 64 + nb) * TC];
                        if constexpr (GATED) v = O::mul2(v, sws[(na * 64 + nb) * TC]);
                        x[na] = O::unpack(v);
                    }
                    cpx X[RA];
                    otc2_fwd_radix<RA>(x, X);
                    #pragma unroll
                    for (int kp = 0; kp < C::NA; ++kp) {  // k_a = kp and kp + RA/2, packed
                        const float4 v = cmul2_split(X[kp].r, X[kp + C::NA].r, X[kp].i, X[kp + C::NA].i,
                                                     s_tab[kp * 64 + nb]);
                        w[kp][i] = O::pack(v.x, v.z);
                        w[kp + C::NA][i] = O::pack(v.y, v.w);
                    }
                }
                #pragma unroll
                for (int ka = 0; ka < RA; ++ka) {
                    const int m = ka * TC + c;
                    uint8_t* arow = sa + (m >> 3) * C::SBO + (m & 7) * 16;
                    #pragma unroll
                    for (int q = 0; q < NBT / 4; ++q)
                        *reinterpret_cast<uint4*>(arow + (nb0 / 4 + q) * C::LBO) =
                            make_uint4(w[ka][4 * q], w[ka][4 * q + 1], w[ka][4 * q + 2], w[ka][4 * q + 3]);
                }
            } else {
                // W_M^(n_c k0), k0 = k_a + RA k_b, for k_a = 2 kp and 2 kp + 1 as a
                // packed pair: steps W_M^(RA n_c) along k_b, W_M^(2 n_c) along kp
                const cpx a1 = twiddle_pow2(n_c, M);
                const cpx stp = twiddle_pow2((uint32_t(RA) * n_c) & (M - 1), M);
                const cpx t0 = twiddle_pow2((n_c * uint32_t(RA * nb0)) & (M - 1), M);
                const cpx t1 = cmul(t0, a1), a2 = cmul(a1, a1);
                float4 tp = make_float4(t0.r, t1.r, t0.i, t1.i);
                const float4 s4 = make_float4(stp.r, stp.r, stp.i, stp.i), a24 = make_float4(a2.r, a2.r, a2.i, a2.i);
                #pragma unroll 1
                for (int kp = 0; kp < RA / 2; ++kp) {
                    uint32_t w0[NBT], w1[NBT];
                    float4 tw = tp;
                    // SP: the dead sub-rows of this pair of k_a (never written by pass B) read as zero
                    const unsigned long long za = SP ? __ldg(a.zbits + 4 * kp) >> nb0 : 0ull;
                    const unsigned long long zc = SP ? __ldg(a.zbits + 4 * kp + 2) >> nb0 : 0ull;
                    #pragma unroll
                    for (int i = 0; i < NBT; ++i) {
                        const uint32_t r0 = ((za >> i) & 1ull) ? 0u : sts[(64 * (2 * kp) + nb0 + i) * TC];
                        const uint32_t r1 = ((zc >> i) & 1ull) ? 0u : sts[(64 * (2 * kp + 1) + nb0 + i) * TC];
                        const cpx x0 = O::unpack(r0), x1 = O::unpack(r1);
                        const float4 v = cmul2_split(x0.r, x1.r, x0.i, x1.i, tw);
                        w0[i] = O::pack(v.x, v.z);
                        w1[i] = O::pack(v.y, v.w);
                        if (i + 1 < NBT) tw = cmul2_split(tw.x, tw.y, tw.z, tw.w, s4);
                    }
                    tp = cmul2_split(tp.x, tp.y, tp.z, tp.w, a24);
                    #pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int m = (2 * kp + h) * TC + c;
                        uint8_t* arow = sa + (m >> 3) * C::SBO + (m & 7) * 16;
                        const uint32_t* wv = h ? w1 : w0;
                        #pragma unroll
                        for (int q = 0; q < NBT / 4; ++q)
                            *reinterpret_cast<uint4*>(arow + (nb0 / 4 + q) * C::LBO) =
                                make_uint4(wv[4 * q], wv[4 * q + 1], wv[4 * q + 2], wv[4 * q + 3]);
                    }
                }
            }
        }
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        if (t == 0) {
            // the staging slot is free: the tile NST ahead
            const long nxt = item + long(P::NST) * stride;
            if (nxt < items) {
                stage(nxt, s);
                issued |= 1u << s;
            }
            tc::fence_after();
            const uint32_t sam = smem_u32(sa), sfm = smem_u32(sf);
            constexpr uint32_t id = tc::idesc(DT, 128, 128);
            #pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_ss(tmem, tc::sdesc(sam + 2 * ks * C::LBO, C::LBO, C::SBO),
                           tc::sdesc(sfm + 2 * ks * C::LBO, C::LBO, C::SBO), id, ks > 0);
            tc::commit(mbar);
            mma_pending = true;
        }
        {
            const bool ok = mbar_wait_sleep(mbar, mpar, kWaitSleepLimit, kWaitHintNs);
            if (ok) {
                mpar ^= 1;
                mma_pending = false;
            }
            tc::fence_after();
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }

        // ---------------- epilogue: outputs [EOUT eh, EOUT eh + EOUT) of row (eka, ec)
        const uint32_t n_ce = uint32_t(o_base + ec);
        if constexpr (FWD) {
            // W_M^(n_c (k_a + RA k_b)) along k_b: in each chunk of 16 outputs,
            // outputs j and j + 8 as a packed pair of product chains
            const uint32_t k00 = uint32_t(eka + RA * EOUT * eh);
            const cpx ta = twiddle_pow2((n_ce * k00) & (M - 1), M);
            const cpx sp = twiddle_pow2((uint32_t(RA) * n_ce) & (M - 1), M);
            cpx s8 = cmul(sp, sp);
            s8 = cmul(s8, s8);
            s8 = cmul(s8, s8);  // W_M^(8 RA n_c)
            const cpx tb = cmul(ta, s8);
            float4 tw = make_float4(ta.r, tb.r, ta.i, tb.i);
            const float4 st4 = make_float4(sp.r, sp.r, sp.i, sp.i), s84 = make_float4(s8.r, s8.r, s8.i, s8.i);
            uint32_t* trow = a.T + row * long(M) + long(64 * eka + EOUT * eh) * C::L + n_ce;
            // SP: sub-rows of skipped pass-B pairs are not stored
            const uint32_t md = SP ? uint32_t(__ldg(a.zbits + 2 * eka) >> (EOUT * eh)) : 0u;
            #pragma unroll
            for (int c0 = 0; c0 < EOUT; c0 += 16) {
                uint32_t vv[32];
                tc::ld32x32b_x32(tmem + (uint32_t(32 * eq) << 16) + uint32_t(2 * (EOUT * eh + c0)), vv);
                tc::wait_ld();
                #pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 x = cmul2_split(__uint_as_float(vv[2 * j]), __uint_as_float(vv[2 * j + 16]),
                                                 __uint_as_float(vv[2 * j + 1]), __uint_as_float(vv[2 * j + 17]), tw);
                    tw = cmul2_split(tw.x, tw.y, tw.z, tw.w, st4);
                    if (!((md >> (c0 + j)) & 1u)) trow[long(c0 + j) * C::L] = O::pack(x.x, x.z);
                    if (!((md >> (c0 + j + 8)) & 1u)) trow[long(c0 + j + 8) * C::L] = O::pack(x.y, x.w);
                }
                // (outputs c0 + 8, c0 + 16) -> (c0 + 16, c0 + 24)
                if (c0 + 16 < EOUT) tw = cmul2_split(tw.x, tw.y, tw.z, tw.w, s84);
            }
        } else {
            // W_(64 RA)^(n_b k_a) / sqrt(RA) on pairs (n_b, n_b + 1), parked in the A space
            uint32_t* park = reinterpret_cast<uint32_t*>(sa);
            #pragma unroll
            for (int c0 = 0; c0 < EOUT; c0 += 16) {
                uint32_t vv[32];
                tc::ld32x32b_x32(tmem + (uint32_t(32 * eq) << 16) + uint32_t(2 * (EOUT * eh + c0)), vv);
                tc::wait_ld();
                #pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const int nb = EOUT * eh + c0 + j;
                    const float4 x = cmul2_split(__uint_as_float(vv[2 * j]), __uint_as_float(vv[2 * j + 2]),
                                                 __uint_as_float(vv[2 * j + 1]), __uint_as_float(vv[2 * j + 3]),
                                                 s_tab[eka * 32 + nb / 2]);
                    park[otc2_park<RA>(eka, nb, ec)] = O::pack(x.x, x.z);
                    park[otc2_park<RA>(eka, nb + 1, ec)] = O::pack(x.y, x.w);
                }
            }
        }
        tc::fence_before();
        if constexpr (!FWD) {
            __syncthreads();
            // ---------------- the RA-point stage, outputs n_a < RA/2 -> y
            const uint32_t* park = reinterpret_cast<const uint32_t*>(sa) + c;
            const uint32_t n_c = uint32_t(o_base + c);
            #pragma unroll 2
            for (int i = 0; i < NBT; ++i) {
                const int nb = nb0 + i;
                cpx v[RA];
                #pragma unroll
                for (int ka = 0; ka < RA; ++ka) v[ka] = O::unpack(park[otc2_park<RA>(ka, nb, 0)]);
                cpx out[C::NA];
                otc2_half_radix<RA>(v, out);
                #pragma unroll
                for (int na = 0; na < C::NA; ++na) {
                    // y_z = conj(out): y[2n] = Re, y[2n+1] = -Im
                    const long e = row * long(M) + 2 * (long(C::L1) * na + long(C::L) * nb + n_c);
                    float re = out[na].r, im = -out[na].i;
                    if constexpr (GATED) {
                        const cpx gv = O::unpack(__ldg(reinterpret_cast<const uint32_t*>(a.w_out + e)));
                        re *= gv.r;
                        im *= gv.i;
                    }
                    *reinterpret_cast<uint32_t*>(a.y + e) = O::pack(re, im);
                }
            }
        }
    }
    if (failed && t == 0) {
        // record the timeout, then wait (bounded) for the copies and the contraction in flight
        atomicExch(a.err, 7);
        for (int s = 0; s < P::NST; ++s)
            if ((issued >> s) & 1u) mbar_wait_bounded(&full[s], (par >> s) & 1u, kWaitLimit);
        if (mma_pending) mbar_wait_bounded(mbar, mpar, kWaitLimit);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (wq == 0) tc::dealloc(tmem, C::TMEM_COLS);
}

}  // namespace fftconv
