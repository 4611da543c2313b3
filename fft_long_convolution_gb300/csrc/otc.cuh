// Outer passes of the multi-pass path on the fifth-generation tensor cores
// (tcgen05): pass A (forward outer stage, from u or in place on T) and pass
// C (inverse outer stage, in place on T or to y).
//
// FlashFFTConv page, section 3.4 "Kernel Fusion and Recomputation
// Strategies": the outermost Monarch factor goes through HBM.  With the
// row of length M = R * L viewed as R sub-rows of L columns (n = L n0 + n',
// k = k0 + R kappa):
//   pass A  T[k0][n'] = W_M^(n' k0) sum_{n0 < NIN} x[n0][n'] W_R^(n0 k0) / sqrt(R)
//           MODE 0: x = z (the packed row of u, times w_in), NIN = R/2 (the
//           implicit zero padding); MODE 1: x = T itself, NIN = R (an inner
//           stage of a two-level outer factor), written back in place
//   pass C  out[n0][n'] = sum_{k0} W_R^(n0 k0) W_M^(n' k0) T[k0][n'] / sqrt(R)
//           MODE 2: all R outputs, in place; MODE 3: n0 < R/2 only (the
//           causal truncation), y_z = conj(out) (times w_out)
// FULL (circular convolution of length 2M): MODE 0 reads all R input rows
// of z (no zero half) and MODE 3 writes all R output rows; u and y rows hold
// 2M samples instead of M.
// SP (frequency-sparse plans, one-level outer factor): sub-rows k0 whose
// pass-B pair is skipped (bit k0 of a.zbits[0..1]) are not stored by MODE 0;
// MODE 3 reads as zeros every sub-row whose bins are all dropped (bit k0 of
// a.zcbits[0..1]: pass B leaves exact zeros there, or nothing for a skipped
// pair) and copies only the runs of the others (otc_live_runs) when there
// are at most two of them.
//
// One CTA of 128 threads walks tiles of 128 columns of one row; thread t
// owns column t of the tile.  A tile's input rows are staged by one tiled
// copy of the TMA engine (a box of 128 columns x all input rows of a
// three-dimensional tensor map: columns, input rows, rows) in a ring of NST
// buffers issued NST tiles ahead.  Each thread
// moves its column into the K-major A operand of the contraction (M = the
// 128 columns, K = the real-embedded inputs), multiplying by w_in (MODE 0)
// or by W_M^(n' k0) (MODE 2, 3: a product chain along k0); one thread issues
// D = X F on the tensor cores (F: the real-embedded DFT matrix as the B
// operand, N = the outputs, real and imaginary part adjacent, padded to a
// multiple of 16; both operands in shared memory; D float32 in tensor
// memory, double-buffered so that the contraction of a tile runs during the
// epilogue of the one before).  In the epilogue tensor-memory lane t is
// column t: the thread reads all outputs of its column, applies the output
// twiddle W_M^(n' k0) (pass A, a chain along k0) or the conjugation and
// gate (MODE 3), and every output row is written as 128-byte runs per warp.
#pragma once
#include <cuda.h>  // CUtensorMap (the encoder is reached through the runtime)

#include "multipass.cuh"
#include "tc.cuh"

namespace fftconv {

template <int R, int MODE, bool FULL = false>
struct Otc {
    static_assert(R >= (FULL ? 2 : 4) && R <= 128 && MODE >= 0 && MODE <= 3, "outer pass shape");
    static constexpr bool FWD = MODE <= 1;
    static constexpr int NIN = (MODE == 0 && !FULL) ? R / 2 : R;   // input rows
    static constexpr int NOUT = (MODE == 3 && !FULL) ? R / 2 : R;  // outputs kept
    static constexpr int TC = 128, THREADS = 128;                // columns per tile = threads = the MMA's M
    static constexpr int KP = 2 * NIN < 16 ? 16 : 2 * NIN;       // K of the contraction (real), padded
    static constexpr int NP = (2 * NOUT + 15) / 16 * 16;         // N (output re/im), padded
    static constexpr int NG = KP / 8;                            // groups of four complex inputs (16 bytes)
    // operand layouts (K-major, no swizzle): element (row, k) at
    // (row/8) SBO + (k/8) LBO + (row%8) 16 + (k%8) 2 bytes
    static constexpr uint32_t LBO = 128, SBO = (KP / 8) * 128;
    static constexpr uint32_t ABYTES = (TC / 8) * SBO;             // the data tile
    static constexpr uint32_t BBYTES = uint32_t(NP / 8) * SBO;     // the DFT matrix
    static constexpr int SEG = TC;                               // staged row segment (words)
    static constexpr uint32_t STAGE_WORDS = uint32_t(NIN) * SEG;
    // staged tiles in flight; the last pass at R = 64 keeps two stages of
    // 32 KB (its DFT matrix has only NOUT = 32 outputs, so two CTAs per SM
    // still fit, as its tensor memory allows)
    static constexpr int NST = NIN <= 16 ? 4 : (NIN <= 32 ? 2 : ((MODE == 3 && !FULL && R == 64) ? 2 : 1));
    static constexpr uint32_t DCOLS = NP;                            // tensor-memory columns per accumulator
    static constexpr uint32_t TMEM_COLS = 2 * DCOLS < 32 ? 32 : 2 * DCOLS;  // double-buffered (allocation >= 32)
};

// The live sub-rows of a frequency-sparse plan as at most two runs of
// consecutive rows, each copied as one box of `box` rows starting at
// start[i] (start[i] + box <= R; a box may cover dead rows, which are read
// as zeros).  n = 0: more than two runs, or boxes that would overlap: copy
// all R rows.  The host encodes the tensor map's box height with the same
// function.
struct OtcRuns {
    int n, box, start[2];
};
__host__ __device__ inline OtcRuns otc_live_runs(unsigned long long z0, unsigned long long z1, int R) {
    OtcRuns r{0, 0, {0, 0}};
    int len[2] = {0, 0}, runs = 0;
    bool prev = false;
    for (int k = 0; k < R; ++k) {
        const bool live = ((k < 64 ? z0 >> k : z1 >> (k - 64)) & 1ull) == 0;
        if (live && !prev) {
            if (runs == 2) return OtcRuns{0, R, {0, 0}};
            r.start[runs++] = k;
        }
        if (live) ++len[runs - 1];
        prev = live;
    }
    if (runs == 0) return OtcRuns{0, 0, {0, 0}};  // nothing live: nothing to copy
    r.n = runs;
    r.box = len[0] > len[1] ? len[0] : len[1];
    for (int i = 0; i < runs; ++i)
        if (r.start[i] + r.box > R) r.start[i] = R - r.box;
    if (runs == 2 && r.start[0] + r.box > r.start[1]) return OtcRuns{0, R, {0, 0}};
    return r;
}

template <int R, int MODE, bool GATED, bool FULL = false>
constexpr size_t otc_smem() {
    using C = Otc<R, MODE, FULL>;
    return size_t(C::ABYTES) + size_t(C::BBYTES) + size_t(C::NST) * C::STAGE_WORDS * 4 * ((GATED && MODE == 0) ? 2 : 1) +
           size_t(C::NST + 3) * 8 + 3 * 8 + 8;
}

// tin: the input rows (MODE 0: u as 32-bit words, [rows][R/2][L], FULL
// [rows][R][L]; else T, [rows][R][L]); tgate: w_in in u's shape (gated MODE 0).
template <int DT, int R, int MODE, bool GATED, int L, bool FULL = false, bool SP = false>
__global__ void __launch_bounds__(128) otc_pass(const MPArgs a, const uint8_t* __restrict__ fmat,
                                                const __grid_constant__ CUtensorMap tin,
                                                const __grid_constant__ CUtensorMap tgate) {
    using O = Op<DT>;
    using C = Otc<R, MODE, FULL>;
    static_assert(!SP || ((MODE == 0 || MODE == 3) && !FULL), "sparse outer passes: one level, causal");
    static_assert(!(GATED && (MODE == 1 || MODE == 2)), "the inner stages have no gates");
    constexpr uint32_t M = uint32_t(R) * L;  // the twiddle modulus (the row length of this pass)
    constexpr int TILES = L / C::TC;
    // all shared state is dynamic (no static shared memory, so the dynamic
    // region starts at the CTA's base without an alignment gap and two CTAs
    // of the R = 64 last pass fit an SM)
    extern __shared__ __align__(1024) uint8_t smem[];

    uint8_t* sa = smem;                                          // data tile (A operand)
    uint8_t* sf = sa + C::ABYTES;                                // DFT matrix (B operand)
    uint32_t* st = reinterpret_cast<uint32_t*>(sf + C::BBYTES);  // [NST][NIN][SEG]
    uint32_t* sw = st + C::NST * C::STAGE_WORDS;                 // gated pass A: w_in, same shape
    uint64_t* full = reinterpret_cast<uint64_t*>(sw + ((GATED && MODE == 0) ? C::NST * C::STAGE_WORDS : 0));  // [NST] staged tile arrived
    uint64_t* mbar = full + C::NST;                              // [2] contraction done, per accumulator
    uint64_t* fbar = mbar + 2;                                   // DFT matrix arrived
    // W_M^(o_base) of a tile, by local tile index mod 3: tile i's value is read
    // in its own reformat and epilogue (the next iteration), and rewritten
    // by tile i + 3 only after every thread has passed tile i + 1's barrier
    float2* s_pt = reinterpret_cast<float2*>(fbar + 1);
    uint32_t& s_tmem = *reinterpret_cast<uint32_t*>(s_pt + 3);

    const int t = threadIdx.x, wq = t >> 5;
    // SP: the dead sub-rows (every row of the plan shares them)
    const unsigned long long* zb = MODE == 3 ? a.zcbits : a.zbits;
    const unsigned long long z0 = (SP && zb) ? __ldg(zb) : 0ull;
    const unsigned long long z1 = (SP && zb) ? __ldg(zb + 1) : 0ull;
    uint32_t live_bytes = C::STAGE_WORDS * 4u;  // bytes one tile's staging receives
    OtcRuns runs{0, C::NIN, {0, 0}};
    uint32_t gmask = ~0u;  // SP pass C: groups of four input rows with a live row (the others stay zero in A)
    unsigned long long omask = ~0ull;  // SP pass A: chunks of outputs (CH/2 sub-rows) with a live sub-row
    if constexpr (SP && MODE == 0) {
        constexpr int OPC = (C::NP < 32 ? C::NP : 32) / 2;  // outputs per epilogue chunk
        omask = 0ull;
        for (int o = 0; o < C::NOUT; ++o)
            if (!zbit(z0, z1, o)) omask |= 1ull << (o / OPC);
    }
    if constexpr (SP && MODE == 3) {
        runs = otc_live_runs(z0, z1, C::NIN);
        live_bytes = uint32_t(runs.n ? runs.n * runs.box : runs.box) * C::SEG * 4u;
        gmask = 0u;
        for (int n0 = 0; n0 < C::NIN; ++n0)
            if (!zbit(z0, z1, n0)) gmask |= 1u << (n0 >> 2);
    }
    const long rows = long(a.B) * a.H;
    const long items = rows * TILES;
    const long first_item = blockIdx.x, stride = gridDim.x;

    auto stage = [&](long item, int s) {  // the tile's input rows into staging slot s
        const int row = int(item / TILES);
        const int o_base = int(item % TILES) * C::TC;
        mbar_expect_tx(&full[s], live_bytes * ((GATED && MODE == 0) ? 2u : 1u));
        if constexpr (SP && MODE == 3) {  // the runs of live rows (or all rows; none if nothing is live)
            if (runs.n == 0 && runs.box > 0) tma_load_3d(st + s * C::STAGE_WORDS, &tin, o_base, 0, row, &full[s]);
            for (int i = 0; i < runs.n; ++i)
                tma_load_3d(st + s * C::STAGE_WORDS + runs.start[i] * C::SEG, &tin, o_base, runs.start[i], row,
                            &full[s]);
        } else {
            tma_load_3d(st + s * C::STAGE_WORDS, &tin, o_base, 0, row, &full[s]);
        }
        if (GATED && MODE == 0) tma_load_3d(sw + s * C::STAGE_WORDS, &tgate, o_base, 0, row, &full[s]);
    };

    // ---------------- set-up
    // thread 0's record of what is in flight: staging slots with copies
    // issued and not yet consumed, and the contractions per accumulator
    uint32_t issued = 0, mma_pending = 0;
    if (t == 0) {
        for (int s = 0; s < C::NST + 3; ++s) mbar_init(full + s, 1);
        fence_mbar_init();
        mbar_expect_tx(fbar, C::BBYTES);
        bulk_g2s(sf, fmat, C::BBYTES, fbar);
        for (int s = 0; s < C::NST; ++s)
            if (first_item + s * stride < items) {
                stage(first_item + s * stride, s);
                issued |= 1u << s;
            }
    }
    if (wq == 0) tc::alloc(&s_tmem, C::TMEM_COLS);
    for (uint32_t i = t; i < C::ABYTES / 16; i += blockDim.x)  // K padding stays zero
        reinterpret_cast<uint4*>(sa)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    bool failed = __syncthreads_or(!mbar_wait_bounded(fbar, 0, kWaitLimit));
    float2 qt;  // W_M^t, this thread's column within a tile
    {
        const cpx v = twiddle_pow2(uint32_t(t) & (M - 1), M);
        qt = make_float2(v.r, v.i);
    }
    // this thread's row of the A operand (column t of the tile)
    uint8_t* arow = sa + (t >> 3) * C::SBO + (t & 7) * 16;

    // the epilogue of a tile (accumulator slot d): all outputs of column t
    auto epilogue = [&](long pitem, int d, int ps) {
        const long row = pitem / TILES;
        const int o_base = int(pitem % TILES) * C::TC;
        const int n1 = o_base + t;  // this thread's column
        const float2 pt = s_pt[ps];
        const cpx w1 = cmul({pt.x, pt.y}, {qt.x, qt.y});  // W_M^(n1)
        cpx tw = {1.f, 0.f};                                // W_M^(n1 k0), k0 = 0, 1, ...
        constexpr int CH = C::NP < 32 ? C::NP : 32;         // accumulator columns per load
        cpx wch = {1.f, 0.f};                               // SP pass A: W_M^(n1 CH/2), one chunk of outputs
        if constexpr (SP && MODE == 0) {
            wch = w1;
            #pragma unroll
            for (int e = 1; e < CH / 2; e <<= 1) wch = cmul(wch, wch);
        }
        #pragma unroll 1
        for (int c0 = 0; c0 < 2 * C::NOUT; c0 += CH) {
            if (SP && MODE == 0 && !((omask >> (c0 / CH)) & 1ull)) {  // a chunk of dead outputs: not stored
                tw = cmul(tw, wch);
                continue;
            }
            uint32_t vv[32];
            const uint32_t taddr = tmem + (uint32_t(32 * wq) << 16) + d * C::DCOLS + c0;
            if constexpr (CH == 16)
                tc::ld32x32b_x16(taddr, vv);
            else
                tc::ld32x32b_x32(taddr, vv);
            tc::wait_ld();
            #pragma unroll
            for (int j = 0; j < CH / 2; ++j) {
                const int o = c0 / 2 + j;
                if (o >= C::NOUT) break;
                cpx x = {__uint_as_float(vv[2 * j]), __uint_as_float(vv[2 * j + 1])};
                if constexpr (C::FWD) {
                    x = cmul(x, tw);
                    tw = cmul(tw, w1);
                }
                if constexpr (MODE <= 2) {
                    if (SP && zbit(z0, z1, o)) continue;  // a skipped pair's sub-row: never read
                    a.T[row * long(M) + long(L) * o + n1] = O::pack(x.r, x.i);
                } else {
                    // y_z = conj(out): y[2n] = Re, y[2n+1] = -Im
                    const long e = row * long(FULL ? 2 * M : M) + 2 * (long(L) * o + n1);
                    float re = x.r, im = -x.i;
                    if (GATED) {
                        const cpx g = O::unpack(__ldg(reinterpret_cast<const uint32_t*>(a.w_out + e)));
                        re *= g.r;
                        im *= g.i;
                    }
                    *reinterpret_cast<uint32_t*>(a.y + e) = O::pack(re, im);
                }
            }
        }
    };

    uint32_t par[C::NST] = {}, mpar[2] = {0, 0};
    long li = 0;     // local tile index
    long prev = -1;  // the tile whose epilogue is pending
    for (long item = first_item; item < items && !failed; item += stride, ++li) {
        const int s = int(li % C::NST), d = int(li & 1), ps = int(li % 3);
        const int o_base = int(item % TILES) * C::TC;
        if (t == 0) {
            const cpx v = twiddle_pow2(uint32_t(o_base) & (M - 1), M);
            s_pt[ps] = make_float2(v.r, v.i);
        }
        bool bad = !mbar_wait_sleep(&full[s], par[s], kWaitSleepLimit, kWaitHintNs);
        if (!bad) {
            par[s] ^= 1;
            issued &= ~(1u << s);
        }
        // the contraction of the tile before must be done reading the A operand
        if (prev >= 0) {
            const bool ok = mbar_wait_sleep(&mbar[d ^ 1], mpar[d ^ 1], kWaitSleepLimit, kWaitHintNs);
            bad |= !ok;
            if (ok) {
                mpar[d ^ 1] ^= 1;
                mma_pending &= ~(1u << (d ^ 1));
            }
        }
        tc::fence_after();
        if (__syncthreads_or(bad)) { failed = true; break; }

        // ---------------- column t of the staged rows -> row t of the A operand
        {
            const uint32_t* sts = st + s * C::STAGE_WORDS + t;
            const uint32_t* sws = sw + s * C::STAGE_WORDS + t;
            cpx tw = {1.f, 0.f}, w1 = {1.f, 0.f}, w4 = {1.f, 0.f};  // pass C: W_M^(n' k0) along k0
            if constexpr (!C::FWD) {
                const float2 pt = s_pt[ps];
                w1 = cmul({pt.x, pt.y}, {qt.x, qt.y});
                if constexpr (SP) w4 = cmul(cmul(w1, w1), cmul(w1, w1));
            }
            static_assert(C::NG <= 32, "group mask");
            #pragma unroll 4
            for (int g = 0; g < C::NG; ++g) {
                if (SP && MODE == 3 && !((gmask >> g) & 1u)) {  // four dead rows: A keeps its zeros
                    if constexpr (!C::FWD) tw = cmul(tw, w4);
                    continue;
                }
                uint32_t v[4];
                #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int n0 = 4 * g + i;
                    uint32_t x = 0u;
                    if (n0 < C::NIN) {
                        // SP, pass C: a skipped pair's sub-row was never written and reads as zero
                        if (!(SP && MODE == 3 && zbit(z0, z1, n0))) {
                            x = sts[n0 * C::SEG];
                            if (GATED && MODE == 0) x = O::mul2(x, sws[n0 * C::SEG]);
                            if constexpr (!C::FWD) {
                                const cpx xv = cmul(O::unpack(x), tw);
                                x = O::pack(xv.r, xv.i);
                            }
                        }
                        if constexpr (!C::FWD) tw = cmul(tw, w1);
                    }
                    v[i] = x;
                }
                *reinterpret_cast<uint4*>(arow + g * C::LBO) = make_uint4(v[0], v[1], v[2], v[3]);
            }
        }
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        if (t == 0) {
            // the staging slot is free: the tile NST ahead
            const long nxt = item + long(C::NST) * stride;
            if (nxt < items) {
                stage(nxt, s);
                issued |= 1u << s;
            }
            tc::fence_after();
            const uint32_t sam = smem_u32(sa), sfm = smem_u32(sf);
            constexpr uint32_t id = tc::idesc(DT, 128, C::NP);
            #pragma unroll
            for (int ks = 0; ks < C::KP / 16; ++ks)
                tc::mma_ss(tmem + d * C::DCOLS, tc::sdesc(sam + 2 * ks * C::LBO, C::LBO, C::SBO),
                           tc::sdesc(sfm + 2 * ks * C::LBO, C::LBO, C::SBO), id, ks > 0);
            tc::commit(&mbar[d]);
            mma_pending |= 1u << d;
        }

        // ---------------- the previous tile's epilogue, while this contraction runs
        if (prev >= 0) epilogue(prev, d ^ 1, int((li + 2) % 3));
        prev = item;
    }
    // the last tile's epilogue
    if (!failed && prev >= 0) {
        const int d = int((li - 1) & 1);
        const bool ok = mbar_wait_sleep(&mbar[d], mpar[d], kWaitSleepLimit, kWaitHintNs);
        if (ok) {
            mpar[d] ^= 1;
            mma_pending &= ~(1u << d);
        }
        tc::fence_after();
        failed = __syncthreads_or(!ok);
        if (!failed) epilogue(prev, d, int((li - 1) % 3));
    }
    if (failed && t == 0) {
        // record the timeout, then wait (bounded) for the copies and the contractions in flight
        atomicExch(a.err, 7);
        for (int s = 0; s < C::NST; ++s)
            if ((issued >> s) & 1u) mbar_wait_bounded(&full[s], par[s], kWaitLimit);
        for (int d = 0; d < 2; ++d)
            if ((mma_pending >> d) & 1u) mbar_wait_bounded(&mbar[d], mpar[d], kWaitLimit);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (wq == 0) tc::dealloc(tmem, C::TMEM_COLS);
}

}  // namespace fftconv
