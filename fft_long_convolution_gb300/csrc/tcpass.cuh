// Pass B of the multi-pass path for sub-rows of L = 4096 points on the
// fifth-generation tensor cores (tcgen05): per pair of sub-rows (k0, R0 - k0)
// of T, the 4096-point transform of each sub-row as 64 x 64, the
// decimation-in-time fold with the kernel spectrum, and the same stages
// back, written over the two sub-rows of T (without the W_M^(n' k0) twiddle,
// which pass C applies).
//
// Monarch factorization of a sub-row (FlashFFTConv page, "The Monarch FFT
// Decomposition"), decimation in frequency, n' = 64 n1 + o, kappa = k1 + 64 k2,
// global bin k = k0 + R0 kappa:
//   S1  X[k1][o]  = W_L^(o k1) * sum_{n1 < 64} T[k0][64 n1 + o] W_64^(n1 k1) / 8
//   S2  Z[k1 + 64 k2] = sum_o X[k1][o] W_64^(o k2) / 8
//   fold  C[k] = alpha~_k conj Z[k] + beta~_k Z[M - k]
//   S3  U[k1][o]  = W_L^(o k1) * sum_{k2} C[k1 + 64 k2] W_64^(k2 o) / 8
//   S4  T[k0][64 n1 + o] = sum_{k1} U[k1][o] W_64^(n1 k1) / 8   (all n1)
// The contractions, the row order of the DFT matrix in tensor memory, the
// B-operand layouts and the two-pipeline structure are those of the
// N = 4096 fused kernel (tcconv.cuh); S1 has the full K = 64 inputs and S4
// keeps all 64 outputs (M = 128).
//
// Fold pairing.  Bin k = k0 + R0 (k1 + 64 k2) pairs with M - k:
// - k0 > 0: sub-row R0 - k0, kappa' = L - 1 - kappa = (63 - k1) + 64 (63 - k2).
//   A work item holds sub-rows A = p and B = R0 - p; S2's columns put
//   sub-problem s of A (slot 2s) beside sub-problem 63 - s of B (slot
//   2(63 - s) + 1 = 2s + 1), so a thread holds both bins of every pair.
// - pair 0 holds sub-rows 0 and R0/2, each of which pairs with itself: sub-row
//   0 as the fused 4096-point kernel (kappa' = L - kappa: slots of
//   tcconv.cuh with the copies of sub-problems 0 and 32, 72 columns),
//   sub-row R0/2 as kappa' = L - 1 - kappa (sub-problem s < 32 beside
//   63 - s, at columns 72 + 2s and 72 + 2s + 1).  S2 then has N = 144.
// The fold's coefficients follow the layout of this kernel's columns:
// [h][pair][chunk 17][warp 4][half 2][lane 32] uint4, read through L2.
#pragma once
#include "multipass.cuh"
#include "tcconv.cuh"

namespace fftconv {

struct TcBArgs {
    uint32_t* T;            // [rows][R0][L] 16-bit complex words, in place
    const uint4* kf;        // [h][pair][chunk 17][warp 4][half 2][lane 32]
    const uint32_t* fmat;   // the three DFT matrices of the N = 4096 kernel
    int B, H, R0;
    int* err;
    int RA;                 // 0: sub-row k0 at position k0; else (two-level outer factor R0 = RA * 64)
                            // at position (k0 mod RA) * 64 + k0 / RA
    int np;                 // pairs that run (frequency-sparse plans skip pairs whose bins are all zero)
    const uint16_t* plist;  // [np] pair indices; null: all R0 / 2 pairs
};

struct TcB {
    static constexpr int L = 4096;
    static constexpr int THREADS = 512;   // two pipelines of 256
    // B operand layouts, two sub-rows side by side along N (LBO, SBO in
    // bytes).  B1: K = 128 (n1) x N = 128 (sub-row, o).  B2: K = 128 (o) x N =
    // 128 or 144 (slots).  B3: K = 128 (k2, order P3) x N = 128 (sub-row, k1)
    // plus a trash row group.  B4: K = 128 (k1, order P4) x N = 128 (sub-row, o).
    static constexpr uint32_t LBO1 = 128, SBO1 = 2048;
    static constexpr uint32_t LBO2 = 144, SBO2 = 2304;
    static constexpr uint32_t LBO3 = 144, SBO3 = 2304;
    static constexpr uint32_t LBO4 = 144, SBO4 = 2304;
    static constexpr uint32_t TRASH = 16 * SBO3;
    static constexpr uint32_t BBUF = 18 * SBO2;            // 41472 (B1 needs 32768)
    static constexpr uint32_t STG = 16384;                 // one staged sub-row (4096 words)
    static constexpr uint32_t OFF_B = 0, OFF_ST = BBUF;
    static constexpr uint32_t PIPE = OFF_ST + 2 * STG;     // 74240 per pipeline
    static constexpr uint32_t OFF_TW = 2 * PIPE;           // twiddles [b 2][jj 4][tg 256] float4
    static constexpr uint32_t TWB = 2 * 4 * 256 * 16;
    static constexpr uint32_t OFF_W64 = OFF_TW + TWB;      // W_64^o table (32 float4)
    static constexpr uint32_t OFF_BAR = OFF_W64 + 512;
    static constexpr uint32_t SMEM = OFF_BAR + 4 * 8;
    static constexpr int KF_CHUNKS = 17;
    static constexpr uint32_t KFP = KF_CHUNKS * 4 * 2 * 32;  // uint4 per pair of sub-rows
    static constexpr uint32_t TMEM_COLS = 512;
};
static_assert(TcB::SMEM <= 232448, "shared memory");
static_assert(TcB::BBUF >= 16 * TcB::SBO1, "B1 fits");

// SP: frequency-sparse plan: only the a.np pairs listed in a.plist run.
template <int DT, bool SP = false>
__global__ void __launch_bounds__(TcB::THREADS, 1) mp_pass_b_tc(const TcBArgs a) {
    using O = Op<DT>;
    using C = TcB;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint32_t s_tmem;

    const int g = threadIdx.x >> 8, tg = threadIdx.x & 255;
    const int hf = tg >> 7, w = (tg >> 5) & 3, lane = tg & 31, r = lane >> 2, q = lane & 3;
    uint8_t* pb = smem + g * C::PIPE;
    uint8_t* bbuf = pb + C::OFF_B;
    const float4* w64 = reinterpret_cast<const float4*>(smem + C::OFF_W64);
    const float4* tws = reinterpret_cast<const float4*>(smem + C::OFF_TW) + tg;
    const uint32_t* stg = reinterpret_cast<const uint32_t*>(pb + C::OFF_ST);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 2 * g;  // mma, in

    // items (row b*H + h, pair p): b fastest, then p, then h (the B rows of a
    // pair use the same k_f back to back); contiguous ranges per pipeline
    const int pairs = a.R0 >> 1;
    const int items = a.B * a.H * (SP ? a.np : pairs);  // the host guarantees < 2^30
    const int V = int(gridDim.x) * 2, v = int(blockIdx.x) * 2 + g;
    const int i0 = int(int64_t(v) * items / V), i1 = int(int64_t(v + 1) * items / V);
    const size_t M = size_t(a.R0) * C::L;

    struct Item {
        int p, h;
        uint32_t* TA;  // sub-row A (k0 = p), B (k0 = p ? R0 - p : R0/2)
        uint32_t* TB;
    };
    auto pos = [&](int k0) -> size_t { return a.RA ? size_t(k0 % a.RA) * 64 + size_t(k0 / a.RA) : size_t(k0); };
    auto decode = [&](int it) -> Item {
        int b, p, h;
        if constexpr (SP) {
            b = it % a.B;
            const int hp = it / a.B;
            p = int(__ldg(a.plist + hp % a.np));
            h = hp / a.np;
        } else {
            b = it % a.B;
            const int hp = it / a.B;
            p = hp % pairs;
            h = hp / pairs;
        }
        uint32_t* Trow = a.T + (size_t(b) * a.H + h) * M;
        return {p, h, Trow + pos(p) * C::L, Trow + pos(p ? a.R0 - p : pairs) * C::L};
    };
    auto stage_item = [&](int it, uint8_t* pbp, uint64_t* bp) {
        const Item x = decode(it);
        mbar_expect_tx(&bp[1], 2 * C::STG);
        bulk_g2s(pbp + C::OFF_ST, x.TA, C::STG, &bp[1]);
        bulk_g2s(pbp + C::OFF_ST + C::STG, x.TB, C::STG, &bp[1]);
    };

    // ---------------- set-up: barriers, TMEM, tables
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + i, 1);
        fence_mbar_init();
        for (int gp = 0; gp < 2; ++gp) {  // the first item of both pipelines, overlapping the set-up
            const int vp = int(blockIdx.x) * 2 + gp;
            const int j0 = int(int64_t(vp) * items / V), j1 = int(int64_t(vp + 1) * items / V);
            if (j0 < j1) {
                stage_item(j0, smem + gp * C::PIPE, reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 2 * gp);
                const Item x = decode(j0);
                bulk_prefetch_l2(a.kf + (size_t(x.h) * pairs + x.p) * C::KFP, C::KFP * 16);
            }
        }
    }
    if (threadIdx.x < 32) {
        tc::alloc(&s_tmem, C::TMEM_COLS);
        float s0, c0, s1, c1;
        sincospif(-float(2 * lane) / 32.f, &s0, &c0);
        sincospif(-float(2 * lane + 1) / 32.f, &s1, &c1);
        reinterpret_cast<float4*>(smem + C::OFF_W64)[lane] = make_float4(c0, c1, s0, s1);
    }
    const int kapA = 8 * w + r, kapB = 63 - kapA;
    if (g == 0) {
        // W_L^(kappa (8j + 2q + e)) for this thread's chunks j = 4 hf + jj: S1
        // (kappa = k1, columns o) and S3 (kappa = o, columns k1)
        #pragma unroll 1
        for (int bj = 0; bj < 8; ++bj) {
            const int kap = (bj >> 2) ? kapB : kapA, o0 = 8 * (4 * hf + (bj & 3)) + 2 * q;
            float s0, c0, s1, c1;
            sincospif(-float((kap * o0) & (C::L - 1)) / 2048.f, &s0, &c0);
            sincospif(-float((kap * (o0 + 1)) & (C::L - 1)) / 2048.f, &s1, &c1);
            reinterpret_cast<float4*>(smem + C::OFF_TW)[bj * 256 + tg] = make_float4(c0, c1, s0, s1);
        }
    }
    for (uint32_t i = threadIdx.x; i < 2 * C::BBUF / 16; i += blockDim.x) {  // padding columns start finite
        const uint32_t pi = i / (C::BBUF / 16), off = (i % (C::BBUF / 16)) * 16;
        *reinterpret_cast<uint4*>(smem + pi * C::PIPE + off) = make_uint4(0, 0, 0, 0);
    }
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t tD = tmem + 192 + 160 * g;
    const uint32_t laneA = uint32_t(32 * w) << 16, laneB = uint32_t(32 * w + 16) << 16;
    {  // the three DFT matrices, lane t <- row t; each warpgroup moves three of the twelve 16-column chunks
        const int grp = threadIdx.x >> 7, row = 32 * w + lane;
        uint32_t rr[3][16];
        #pragma unroll
        for (int c3 = 0; c3 < 3; ++c3) {
            const int c = 3 * grp + c3;
            const uint4* src = reinterpret_cast<const uint4*>(a.fmat + (c >> 2) * 128 * 64 + row * 64 + 16 * (c & 3));
            #pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 x = src[i];
                rr[c3][4 * i] = x.x; rr[c3][4 * i + 1] = x.y; rr[c3][4 * i + 2] = x.z; rr[c3][4 * i + 3] = x.w;
            }
        }
        #pragma unroll
        for (int c3 = 0; c3 < 3; ++c3) tc::st16(tmem + laneA + 16 * (3 * grp + c3), rr[c3]);
        tc::wait_st();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();

    auto rowoff = [](int s) -> uint32_t { return uint32_t(s >> 3) * C::SBO2 + uint32_t(s & 7) * 16; };
    const uint32_t kq2 = (q >> 1) * C::LBO2 + (q & 1) * 8 + 8 * hf * C::LBO2;
    const uint32_t kq4 = (4 * (q >> 1) + 8 * hf) * C::LBO4 + (q & 1) * 8;
    const bool is_k0 = kapA == 0, is_k32 = kapB == 32;
    auto koff3 = [](int k2) -> uint32_t {  // B3 K position of input k2
        const int pos = tc64_p3(k2);
        return uint32_t(pos >> 2) * C::LBO3 + uint32_t(pos & 3) * 4;
    };
    const uint32_t kAo = koff3(kapA), kBo = koff3(kapB);
    // input pass: sub-row hf, column o, inputs n1 = 32 in_g .. 32 in_g + 31
    const int in_o = tg & 63, in_g = (tg >> 6) & 1;
    const uint32_t in_dst = (8 * hf + (in_o >> 3)) * C::SBO1 + (in_o & 7) * 16 + 8 * in_g * C::LBO1;

    const uint32_t bsm = smem_u32(bbuf);
    constexpr uint32_t id128 = tc::idesc(DT, 128, 128), id144 = tc::idesc(DT, 128, 144);

    bool mma_pending = false, in_pending = i0 < i1;  // the first item's copies were issued in the set-up
    uint32_t mmapar = 0, inpar = 0;
    const uint32_t bar_id = 1 + g;
    bool failed = false;

    for (int it = i0; it < i1; ++it) {
        const Item x = decode(it);
        const bool sp = x.p == 0;
        const bool has_next = it + 1 < i1;
        if (tg == 32 && has_next) {  // the next item's k_f into L2 (read by the next fold)
            const Item xn = decode(it + 1);
            if (xn.p != x.p || xn.h != x.h)
                bulk_prefetch_l2(a.kf + (size_t(xn.h) * pairs + xn.p) * C::KFP, C::KFP * 16);
        }

        // ---------------- input: sub-row hf -> B1
        bool bad = !mbar_wait_sleep(&bars[1], inpar, kWaitSleepLimit, kWaitHintNs);
        if (!bad) {
            const uint32_t* ur = stg + hf * (C::STG / 4) + 32 * in_g * 64 + in_o;
            #pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t z[16];
                #pragma unroll
                for (int i = 0; i < 16; ++i) z[i] = ur[(16 * h2 + i) * 64];
                #pragma unroll
                for (int gq = 0; gq < 4; ++gq)
                    *reinterpret_cast<uint4*>(bbuf + in_dst + (4 * h2 + gq) * C::LBO1) =
                        make_uint4(z[4 * gq], z[4 * gq + 1], z[4 * gq + 2], z[4 * gq + 3]);
            }
        }
        tc::fence_proxy_async();
        tc::fence_before();
        if (tc::bar_vote(bar_id, 256, bad)) { failed = true; break; }
        in_pending = false;
        inpar ^= 1;
        if (tg == 0) {
            tc::fence_after();
            #pragma unroll
            for (int s = 0; s < 8; ++s)
                tc::mma(tD, tmem + 8 * s, tc::sdesc(bsm + 2 * s * C::LBO1, C::LBO1, C::SBO1), id128, s > 0);
            tc::commit(&bars[0]);
        }
        mma_pending = true;
        if (has_next) {  // the staging is free: fetch the next item
            if (tg == 64) stage_item(it + 1, pb, bars);
            in_pending = true;
        }

        // ---------------- S1 post: twiddle, -> B2 (slot rows)
        bad = !mbar_wait_sleep(&bars[0], mmapar, kWaitSleepLimit, kWaitHintNs);
        bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the collective TMEM loads
        tc::fence_after();
        if (!bad) {
            // [sub-row][block]: block b = 1's loads fly while block 0 of both
            // sub-rows is processed; each twiddle serves both sub-rows
            uint32_t vr[2][2][16];
            tc::ld16x256b_x4(tD + laneA + 32 * hf, vr[0][0]);
            tc::ld16x256b_x4(tD + laneA + 64 + 32 * hf, vr[1][0]);
            tc::wait_ld();
            tc::ld16x256b_x4(tD + laneB + 32 * hf, vr[0][1]);
            tc::ld16x256b_x4(tD + laneB + 64 + 32 * hf, vr[1][1]);
            float4 x0[4];   // sub-row 0, k1 = 0 (block a): kept for the pre-twiddled copy
            uint2 p32[4];   // sub-row 0, k1 = 32 (block b): kept for the duplicate
            #pragma unroll
            for (int b = 0; b < 2; ++b) {
                if (b == 1) tc::wait_ld();
                const int kap = b ? kapB : kapA;
                const int slot0 = sp ? tc64_slot(kap) : 2 * kap;                // sub-row 0 (R = 0)
                const int slot1 = sp ? 72 + 2 * kapA + b : 2 * (63 - kap) + 1;  // sub-row 1 (R = 1)
                uint8_t* dst0 = bbuf + rowoff(slot0) + kq2;
                uint8_t* dst1 = bbuf + rowoff(slot1) + kq2;
                #pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float4 tw = tws[(4 * b + jj) * 256];
                    const uint32_t* v0 = vr[0][b] + 4 * jj;
                    const uint32_t* v1 = vr[1][b] + 4 * jj;
                    const float4 xv = cmul2_twiddle(__uint_as_float(v0[0]), __uint_as_float(v0[1]),
                                                    __uint_as_float(v0[2]), __uint_as_float(v0[3]), tw);
                    const float4 xw = cmul2_twiddle(__uint_as_float(v1[0]), __uint_as_float(v1[1]),
                                                    __uint_as_float(v1[2]), __uint_as_float(v1[3]), tw);
                    const uint2 wd = make_uint2(O::pack(xv.x, xv.z), O::pack(xv.y, xv.w));
                    *reinterpret_cast<uint2*>(dst0 + 2 * jj * C::LBO2) = wd;
                    *reinterpret_cast<uint2*>(dst1 + 2 * jj * C::LBO2) = make_uint2(O::pack(xw.x, xw.z), O::pack(xw.y, xw.w));
                    if (b == 0) x0[jj] = xv;
                    else p32[jj] = wd;
                }
                if (b == 0 && sp && is_k0) {  // sub-problem 0 again, pre-twiddled by W_64^o (slot 1)
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float4 y0 = cmul2_twiddle(x0[jj].x, x0[jj].y, x0[jj].z, x0[jj].w, w64[4 * (4 * hf + jj) + q]);
                        *reinterpret_cast<uint2*>(bbuf + 16 + kq2 + 2 * jj * C::LBO2) =
                            make_uint2(O::pack(y0.x, y0.z), O::pack(y0.y, y0.w));
                    }
                }
                if (b == 1 && sp && is_k32) {  // sub-problem 32 again (slot 65)
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        *reinterpret_cast<uint2*>(bbuf + 8 * C::SBO2 + 16 + kq2 + 2 * jj * C::LBO2) = p32[jj];
                }
            }
        }
        // the fold's k_f of chunks 0..3 ([c][w][half][lane], this warpgroup's
        // first chunk), read from L2 while the vote, S2 and its wait run
        const uint4* kft = a.kf + (size_t(x.h) * pairs + x.p) * C::KFP + (sp ? 9 : 8) * hf * 256 + w * 64 + lane;
        uint4 kv[2][4][2];
        #pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            kv[0][jj][0] = __ldg(kft + jj * 256);
            kv[0][jj][1] = __ldg(kft + jj * 256 + 32);
        }
        tc::fence_proxy_async();
        tc::fence_before();
        if (tc::bar_vote(bar_id, 256, bad)) { failed = true; break; }
        mma_pending = false;
        mmapar ^= 1;
        if (tg == 0) {
            tc::fence_after();
            #pragma unroll
            for (int s = 0; s < 8; ++s)
                tc::mma(tD, tmem + 8 * s, tc::sdesc(bsm + 2 * s * C::LBO2, C::LBO2, C::SBO2), sp ? id144 : id128, s > 0);
            tc::commit(&bars[0]);
        }
        mma_pending = true;

        // ---------------- fold of this warpgroup's columns with the kernel spectrum -> B3
        bad = !mbar_wait_sleep(&bars[0], mmapar, kWaitSleepLimit, kWaitHintNs);
        bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the collective TMEM loads
        tc::fence_after();
        if (!bad) {
            auto fold4 = [&](const uint32_t* va, const uint32_t* vb, const uint4 (&k)[2], uint32_t r0, uint32_t r1) {
                const cpx za0 = {__uint_as_float(va[0]), __uint_as_float(va[2])};  // (s0, k2a)
                const cpx za1 = {__uint_as_float(va[1]), __uint_as_float(va[3])};  // (s1, k2a)
                const cpx zb0 = {__uint_as_float(vb[0]), __uint_as_float(vb[2])};  // (s0, k2b)
                const cpx zb1 = {__uint_as_float(vb[1]), __uint_as_float(vb[3])};  // (s1, k2b)
                const cpx c00 = dit_fold<DT>(k[0].x, k[0].y, za0, zb1);
                const cpx c11 = dit_fold<DT>(k[0].z, k[0].w, zb1, za0);
                const cpx c01 = dit_fold<DT>(k[1].x, k[1].y, zb0, za1);
                const cpx c10 = dit_fold<DT>(k[1].z, k[1].w, za1, zb0);
                *reinterpret_cast<uint32_t*>(bbuf + r0 + kAo) = O::pack(c00.r, c00.i);
                *reinterpret_cast<uint32_t*>(bbuf + r1 + kBo) = O::pack(c11.r, c11.i);
                *reinterpret_cast<uint32_t*>(bbuf + r0 + kBo) = O::pack(c01.r, c01.i);
                *reinterpret_cast<uint32_t*>(bbuf + r1 + kAo) = O::pack(c10.r, c10.i);
            };
            // B3 rows: sub-row A's sub-problem k1 at row k1, sub-row B's at 64 + k1.
            // Column pair (2q, 2q + 1) of chunk j holds s0 = 4j + q (row r0) and
            // s1 = its partner (row r1); both rows step by 4 per chunk.
            const uint32_t dcol = tD + (sp ? 72 : 64) * hf;
            const uint32_t r0b = (sp ? 8 : 4) * hf * C::SBO3 + 16 * q;
            const int X = sp ? (hf ? 127 : 64) : 127 - 32 * hf;   // row of s1 at chunk 0 (q = 0)
            const uint32_t r1p[2] = {rowoff(X - q), rowoff(X - 4 - q)};
            // pair 0, sub-row 0: s1 of column 1 is the copy of sub-problem 0 (no bin of its own)
            const uint32_t r1c0 = (sp && hf == 0 && q == 0) ? C::TRASH : r1p[0];
            #pragma unroll
            for (int gq = 0; gq < 2; ++gq) {  // chunks 4 gq .. 4 gq + 3
                uint32_t va[16], vb[16];
                tc::ld16x256b_x4(dcol + laneA + 32 * gq, va);
                tc::ld16x256b_x4(dcol + laneB + 32 * gq, vb);
                if (gq == 0) {
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        kv[1][jj][0] = __ldg(kft + (4 + jj) * 256);
                        kv[1][jj][1] = __ldg(kft + (4 + jj) * 256 + 32);
                    }
                }
                tc::wait_ld();
                #pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = 4 * gq + jj;
                    const uint32_t r0 = r0b + (j >> 1) * C::SBO3 + (j & 1) * 64;
                    const uint32_t r1 = j == 0 ? r1c0 : r1p[j & 1] - (j >> 1) * C::SBO3;
                    fold4(va + 4 * jj, vb + 4 * jj, kv[gq][jj], r0, r1);
                }
            }
            if (sp && hf == 0) {  // chunk 8 of sub-row 0: sub-problem 32 beside its copy, and padding
                uint32_t va[4], vb[4];
                uint4 k8[2];
                tc::ld16x256b_x1(dcol + laneA + 64, va);
                tc::ld16x256b_x1(dcol + laneB + 64, vb);
                k8[0] = __ldg(kft + 8 * 256);
                k8[1] = __ldg(kft + 8 * 256 + 32);
                tc::wait_ld();
                fold4(va, vb, k8, q == 0 ? 4 * C::SBO3 : C::TRASH, C::TRASH);
            }
        }
        tc::fence_proxy_async();
        tc::fence_before();
        if (tc::bar_vote(bar_id, 256, bad)) { failed = true; break; }
        mma_pending = false;
        mmapar ^= 1;
        if (tg == 0) {
            tc::fence_after();
            #pragma unroll
            for (int s = 0; s < 8; ++s)
                tc::mma(tD, tmem + 64 + 8 * s, tc::sdesc(bsm + 2 * s * C::LBO3, C::LBO3, C::SBO3), id128, s > 0);
            tc::commit(&bars[0]);
        }
        mma_pending = true;

        // ---------------- S3 post: twiddle, -> B4
        bad = !mbar_wait_sleep(&bars[0], mmapar, kWaitSleepLimit, kWaitHintNs);
        bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the collective TMEM loads
        tc::fence_after();
        if (!bad) {
            // as in S1 post: block 1's loads fly while block 0 of both sub-rows
            // is processed, one twiddle per column pair serving both
            uint32_t vr[2][2][16];
            tc::ld16x256b_x4(tD + laneA + 32 * hf, vr[0][0]);
            tc::ld16x256b_x4(tD + laneA + 64 + 32 * hf, vr[1][0]);
            tc::wait_ld();
            tc::ld16x256b_x4(tD + laneB + 32 * hf, vr[0][1]);
            tc::ld16x256b_x4(tD + laneB + 64 + 32 * hf, vr[1][1]);
            #pragma unroll
            for (int b = 0; b < 2; ++b) {
                if (b == 1) tc::wait_ld();
                uint8_t* dst = bbuf + rowoff(b ? kapB : kapA) + kq4;
                #pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float4 tw = tws[(4 * b + jj) * 256];
                    #pragma unroll
                    for (int R = 0; R < 2; ++R) {
                        const uint32_t* vv = vr[R][b] + 4 * jj;
                        const float4 xv = cmul2_twiddle(__uint_as_float(vv[0]), __uint_as_float(vv[1]),
                                                        __uint_as_float(vv[2]), __uint_as_float(vv[3]), tw);
                        *reinterpret_cast<uint2*>(dst + 8 * R * C::SBO4 + jj * C::LBO4) =
                            make_uint2(O::pack(xv.x, xv.z), O::pack(xv.y, xv.w));
                    }
                }
            }
        }
        tc::fence_proxy_async();
        tc::fence_before();
        if (tc::bar_vote(bar_id, 256, bad)) { failed = true; break; }
        mma_pending = false;
        mmapar ^= 1;
        if (tg == 0) {
            tc::fence_after();
            #pragma unroll
            for (int s = 0; s < 8; ++s)
                tc::mma(tD, tmem + 128 + 8 * s, tc::sdesc(bsm + 2 * s * C::LBO4, C::LBO4, C::SBO4), id128, s > 0);
            tc::commit(&bars[0]);
        }
        mma_pending = true;

        // ---------------- S4 post: all 64 outputs n1 of both sub-rows -> T
        bad = !mbar_wait_sleep(&bars[0], mmapar, kWaitSleepLimit, kWaitHintNs);
        bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the collective TMEM loads
        tc::fence_after();
        if (!bad) {
            uint32_t vr[2][2][16];
            tc::ld16x256b_x4(tD + laneA + 32 * hf, vr[0][0]);
            tc::ld16x256b_x4(tD + laneB + 32 * hf, vr[0][1]);
            tc::wait_ld();
            tc::ld16x256b_x4(tD + laneA + 64 + 32 * hf, vr[1][0]);
            tc::ld16x256b_x4(tD + laneB + 64 + 32 * hf, vr[1][1]);
            #pragma unroll
            for (int R = 0; R < 2; ++R) {
                if (R == 1) tc::wait_ld();
                #pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const uint32_t* vv = vr[R][b];
                    uint32_t* dst = (R ? x.TB : x.TA) + 64 * (b ? kapB : kapA) + 32 * hf + 2 * q;
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        *reinterpret_cast<uint2*>(dst + 8 * jj) =
                            make_uint2(O::pack(__uint_as_float(vv[4 * jj]), __uint_as_float(vv[4 * jj + 2])),
                                       O::pack(__uint_as_float(vv[4 * jj + 1]), __uint_as_float(vv[4 * jj + 3])));
                }
            }
        }
        tc::fence_before();
        if (tc::bar_vote(bar_id, 256, bad)) { failed = true; break; }
        mma_pending = false;
        mmapar ^= 1;
    }
    if (failed && tg == 0) {
        // record the timeout, then wait (bounded) for this pipeline's work in flight
        atomicExch(a.err, 7);
        if (mma_pending) mbar_wait_bounded(&bars[0], mmapar, kWaitLimit);
        if (in_pending) mbar_wait_bounded(&bars[1], inpar, kWaitLimit);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (threadIdx.x < 32) tc::dealloc(tmem, C::TMEM_COLS);
}

}  // namespace fftconv
