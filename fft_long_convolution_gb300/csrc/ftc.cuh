// Fused causal long convolution for N = M = R0 * 4096 (R0 = 2: N = 8192,
// R0 = 4: N = 16384, R0 = 8: N = 32768, i.e. 2N <= 64K) in one kernel on the
// fifth-generation tensor cores (tcgen05): the whole row stays on the SM.
//
// Monarch factorization (FlashFFTConv page, section 3.4, "The Monarch FFT
// Decomposition" and "Higher-order decompositions"), decimation in
// frequency with the outer factor R0 first, n = 4096 n0 + n',
// k = k0 + R0 kappa:
//   outer    X_k0[n'] = W_M^(n' k0) sum_{n0 < R0/2} z[4096 n0 + n'] W_R0^(n0 k0) / sqrt(R0)
//            (decimation-in-time packing z[n] = x[2n] + i x[2n+1] and the
//            implicit zero padding z[n] = 0 for n >= M/2: "The real-valued FFT
//            optimization", "Implicit zero-padding")
//   inner    per pair of sub-rows (k0, R0 - k0): the 4096-point transform of
//            each sub-row as 64 x 64 on the tensor cores, the
//            decimation-in-time fold with the kernel spectrum and the same
//            stages back -- the engine of the multi-pass pass B (tcpass.cuh),
//            with its slot layouts, fold pairing and k_f layout unchanged
//   outer^-1 y_z[4096 n0 + n'] = conj( sum_k0 W_R0^(n0 k0) W_M^(n' k0) T_k0[n'] / sqrt(R0) ),
//            n0 < R0/2 only (the causal truncation)
// The outer stage runs in the input phase of each pair, from the row of u
// staged in shared memory (the radix-R0 butterfly over the nonzero half and
// the twiddle, as product chains along each thread's column).  The inverse
// outer stage runs in the last phase of the row's last pair (pair 0):
// R0 = 2 combines the pair's two sub-rows; R0 = 4 first reduces pair (1, 3)
// to its two contributions S = V1 + V3 and D = -i (V1 - V3) (V_k0 =
// W_M^(n' k0) T_k0), kept per thread in shared memory in 16-bit, and pair
// (0, 2) adds them: y_z[n'] = (T0 + V2 + S) / 2, y_z[4096 + n'] =
// (T0 - V2 + D) / 2, conjugated.  R0 = 8 accumulates the four pairs'
// contributions c_p[n0] = W_8^(n0 kA) V_kA + W_8^(n0 kB) V_kB to the four
// output blocks n0 < 4 in a shared 16-bit accumulator, in the order pair
// (1, 7), (2, 6), (3, 5), (0, 4); the last one writes y.
//
// Each CTA runs two pipelines of eight warps (as tcpass.cuh).  For R0 = 2
// and 4 they are independent: a pipeline owns a contiguous range of rows
// taken channel-major (the B rows of a channel use the same k_f back to back
// through L2), and the row of u (and, for R0 = 2, w_in) is staged by a bulk
// copy (TMA engine) as soon as the previous row's last input phase has read
// its staging.  Gated R0 = 4 reads w_in through L2 in the row's first input
// phase and writes the gated row back into the staging for the second pair
// (each position of the staging is read and written by one thread only).
// For R0 = 8 a row (64 KB staged, 64 KB of accumulator) only fits once per
// SM, so both pipelines work on the same rows: pipeline 0 takes pairs
// (1, 7) and (3, 5), pipeline 1 pairs (2, 6) and (0, 4).  Two mbarriers pass
// the accumulator between them in the order above, a third one tells
// pipeline 1 that both have read the staged row, after which it stages the
// next; gated R0 = 8 reads w_in through L2 in every input phase.
#pragma once
#include "tcpass.cuh"

namespace fftconv {

struct FtcArgs {
    const uint16_t* u;
    const uint16_t* w_in;
    const uint16_t* w_out;
    const uint4* kf;        // [h][pair][chunk 17][warp 4][half 2][lane 32] uint4 (the pass-B layout)
    uint16_t* y;
    const uint32_t* fmat;   // the three 64 x 64 DFT matrices of tcconv.cuh
    // per-thread starting twiddles, built with the plan (ftc_twiddle_tables):
    // input phase  W_M^(k0 n') / sqrt(R0) at n' = 1024 (t / 64) + t % 64, [k0][t 256]
    // S4 post      W_M^(k0 n') at n' = 64 kappa_b + 32 hf + 2q + e, [k0][b][t 256] as
    //              (re e0, re e1, im e0, im e1)
    const float2* twin;
    const float4* twout;
    int B, H;
    int* err;
    int skip1;  // R0 = 4, frequency-sparse plan: pair (1, 3) holds no kept bin and is not run
};

// FULL: the circular convolution of length 2M (R0 = 2 only): the input
// stage sums both blocks of z (no zero half), the output stage writes both
// blocks, and rows of u and y hold 2M samples.
template <int R0, bool GATED, bool FULL = false>
struct Ftc {
    static_assert(R0 == 2 || R0 == 4 || R0 == 8, "fused tensor-core path: N = 8192, 16384 or 32768");
    static_assert(!FULL || R0 == 2, "circular fused rows: R0 = 2");
    static constexpr int L = 4096, M = R0 * L, NP = R0 / 2;  // sub-row length, row length, pairs per row
    static constexpr int NB = FULL ? R0 : R0 / 2;            // blocks of z in and of y_z out
    static constexpr bool SPLIT = R0 == 8;                   // both pipelines on one row
    static constexpr int THREADS = 512;                      // two pipelines of 256
    static constexpr uint32_t LBO1 = TcB::LBO1, SBO1 = TcB::SBO1;
    static constexpr uint32_t LBO2 = TcB::LBO2, SBO2 = TcB::SBO2;
    static constexpr uint32_t LBO3 = TcB::LBO3, SBO3 = TcB::SBO3;
    static constexpr uint32_t LBO4 = TcB::LBO4, SBO4 = TcB::SBO4;
    static constexpr uint32_t TRASH = TcB::TRASH, BBUF = TcB::BBUF;
    static constexpr uint32_t ZB = uint32_t(NB * L) * 4;             // a row of u: NB L complex words
    static constexpr uint32_t WIB = (GATED && R0 == 2 && !FULL) ? ZB : 0;  // staged w_in
    static constexpr uint32_t TOB = R0 == 4 ? 8u * 256u * 16u : 0;   // S, D of pair (1, 3): [8][tg] uint4
    static constexpr uint32_t ACCB = SPLIT ? 32u * 256u * 8u : 0;    // R0 = 8: [b 2][jj 4][n0 4][tg] uint2
    // per pipeline: the B buffer, and (unless SPLIT) the staging and the handed-over outputs
    static constexpr uint32_t OFF_B = 0, OFF_Z = BBUF, OFF_WI = OFF_Z + ZB, OFF_TO = OFF_WI + WIB;
    static constexpr uint32_t PIPE = SPLIT ? BBUF : OFF_TO + TOB;
    static constexpr uint32_t OFF_ZS = 2 * PIPE, OFF_ACC = OFF_ZS + (SPLIT ? ZB : 0);  // SPLIT: shared
    // twiddles W_L^(kappa o) of S1 / S3 post per thread, [b 2][jj 4][tg 256]:
    // float32 where that fits, else two 16-bit pairs (binary16)
    static constexpr uint32_t SHARED_END = OFF_ACC + ACCB;
    static constexpr bool TW16 = SHARED_END + 8u * 256u * 16u + 1024u > 232448u;
    static constexpr uint32_t TWB = TW16 ? 8u * 256u * 8u : 8u * 256u * 16u;
    static constexpr uint32_t OFF_TW = SHARED_END, OFF_W64 = OFF_TW + TWB;
    static constexpr uint32_t OFF_STEP = OFF_W64 + 512;              // W_M^(64 k0), W_M^(8 k0) per k0: float4
    // barriers: per pipeline (contraction, staging); SPLIT: staging read by both,
    // accumulator handed to pipeline 1, accumulator handed to pipeline 0
    static constexpr uint32_t OFF_BAR = OFF_STEP + R0 * 16;
    static constexpr uint32_t SMEM = OFF_BAR + 8 * 8;
    static constexpr uint32_t TMEM_COLS = 512;
};

template <int DT, int R0, bool GATED, bool FULL = false>
__global__ void __launch_bounds__(512, 1) ftc_conv_kernel(const FtcArgs a) {
    using O = Op<DT>;
    using C = Ftc<R0, GATED, FULL>;
    constexpr int NP = C::NP, NB = C::NB;
    constexpr size_t RS = size_t(FULL ? 2 : 1) * C::M;  // 16-bit samples per row of u and y
    constexpr uint32_t M = uint32_t(C::M);
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint32_t s_tmem;

    const int g = threadIdx.x >> 8, tg = threadIdx.x & 255;
    const int hf = tg >> 7, w = (tg >> 5) & 3, lane = tg & 31, r = lane >> 2, q = lane & 3;
    uint8_t* pb = smem + g * C::PIPE;
    uint8_t* bbuf = pb + C::OFF_B;
    uint32_t* zs = reinterpret_cast<uint32_t*>(C::SPLIT ? smem + C::OFF_ZS : pb + C::OFF_Z);
    uint2* accs = reinterpret_cast<uint2*>(smem + C::OFF_ACC) + tg;  // R0 = 8: [(b 4 + jj) 4 + n0] x 256 threads
    const uint32_t* wis = reinterpret_cast<const uint32_t*>(pb + C::OFF_WI);
    uint4* tout = reinterpret_cast<uint4*>(pb + C::OFF_TO) + tg;  // [b 2][jj 4] x 256 threads
    const float4* w64 = reinterpret_cast<const float4*>(smem + C::OFF_W64);
    const float4* steps = reinterpret_cast<const float4*>(smem + C::OFF_STEP);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 2 * g;  // mma, in
    uint64_t* zfree = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 4;      // R0 = 8 (count 2)
    uint64_t* accbar = zfree + 1;                                              // R0 = 8: [to pipeline 1, to 0]
    // R0 = 8: both pipelines stage from one barrier (pipeline 0's slot)
    uint64_t* zbar = C::SPLIT ? reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 1 : &bars[1];

    // twiddle (wr0, wr1, wi0, wi1) of this thread's chunk bj = 4 b + jj
    auto twl = [&](int bj) -> float4 {
        if constexpr (C::TW16) {
            const uint2 v = reinterpret_cast<const uint2*>(smem + C::OFF_TW)[bj * 256 + tg];
            const cpx c = Op<0>::unpack(v.x), s = Op<0>::unpack(v.y);
            return make_float4(c.r, c.i, s.r, s.i);
        } else {
            return reinterpret_cast<const float4*>(smem + C::OFF_TW)[bj * 256 + tg];
        }
    };

    // rows of this pipeline (R0 = 8: of this CTA): a contiguous range in
    // channel-major order (row index h*B + b, memory row b*H + h).  Items:
    // the row's pairs, NP - 1 .. 0 (R0 = 8: pipeline 0 pairs 1, 3, pipeline
    // 1 pairs 2, 0).
    const int rows = a.B * a.H;  // the host guarantees B*H < 2^30
    const int V = C::SPLIT ? int(gridDim.x) : int(gridDim.x) * 2;
    const int v = C::SPLIT ? int(blockIdx.x) : int(blockIdx.x) * 2 + g;
    const int IPR = C::SPLIT ? 2 : NP - a.skip1;  // items per row of one pipeline
    const int i0 = int(int64_t(v) * rows / V) * IPR, i1 = int(int64_t(v + 1) * rows / V) * IPR;
    auto item_row = [&](int it) -> int { return it / IPR; };
    auto item_pair = [&](int it) -> int {
        if constexpr (C::SPLIT) return g == 0 ? ((it & 1) ? 3 : 1) : ((it & 1) ? 0 : 2);
        return IPR - 1 - (it - (it / IPR) * IPR);
    };
    auto chan = [&](int ri) -> int { return int(unsigned(ri) / unsigned(a.B)); };
    auto mrow = [&](int ri) -> size_t {
        const int h = chan(ri), b = ri - h * a.B;
        return size_t(b) * a.H + h;
    };
    auto kf_of = [&](int h, int p) -> const uint4* { return a.kf + (size_t(h) * NP + p) * TcB::KFP; };
    // the row's u (and w_in) into the staging (one bulk copy each); the gates
    // that are read through L2 are prefetched there
    auto stage_row = [&](int ri, uint8_t* pbp, uint64_t* bp) {
        const size_t off = mrow(ri) * RS;
        mbar_expect_tx(&bp[1], C::ZB + C::WIB);
        bulk_g2s(C::SPLIT ? smem + C::OFF_ZS : pbp + C::OFF_Z, a.u + off, C::ZB, &bp[1]);
        if (GATED && C::WIB) bulk_g2s(pbp + C::OFF_WI, a.w_in + off, C::ZB, &bp[1]);
        if (GATED && (R0 == 4 || FULL)) bulk_prefetch_l2(a.w_in + off, C::ZB);
        if (GATED) bulk_prefetch_l2(a.w_out + off, C::ZB);
    };

    // ---------------- set-up: barriers, TMEM, tables
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + i, 1);
        fence_mbar_init();
        if (C::SPLIT) mbar_init(zfree, 2);
        if (C::SPLIT) mbar_init(accbar, 256);
        if (C::SPLIT) mbar_init(accbar + 1, 256);
        fence_mbar_init();
        for (int gp = 0; gp < (C::SPLIT ? 1 : 2); ++gp) {  // the first row of both pipelines, overlapping the set-up
            const int vp = C::SPLIT ? int(blockIdx.x) : int(blockIdx.x) * 2 + gp;
            const int j0 = int(int64_t(vp) * rows / V) * IPR, j1 = int(int64_t(vp + 1) * rows / V) * IPR;
            if (j0 < j1) {
                stage_row(j0 / IPR, smem + gp * C::PIPE, reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 2 * gp);
                for (int k = 0; k < (C::SPLIT ? 4 : 1); ++k)
                    bulk_prefetch_l2(kf_of(chan(j0 / IPR), C::SPLIT ? k : NP - 1), TcB::KFP * 16);
            }
        }
    }
    if (threadIdx.x < 32) {
        tc::alloc(&s_tmem, C::TMEM_COLS);
        float s0, c0, s1, c1;
        sincospif(-float(2 * lane) / 32.f, &s0, &c0);
        sincospif(-float(2 * lane + 1) / 32.f, &s1, &c1);
        reinterpret_cast<float4*>(smem + C::OFF_W64)[lane] = make_float4(c0, c1, s0, s1);
    } else if (threadIdx.x < 32 + R0) {  // per k0: W_M^(64 k0) and W_M^(8 k0)
        const int k0 = int(threadIdx.x) - 32;
        const cpx s64 = twiddle_pow2((64u * uint32_t(k0)) & (M - 1), M);
        const cpx s8 = twiddle_pow2((8u * uint32_t(k0)) & (M - 1), M);
        reinterpret_cast<float4*>(smem + C::OFF_STEP)[k0] = make_float4(s64.r, s64.i, s8.r, s8.i);
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
            if constexpr (C::TW16)
                reinterpret_cast<uint2*>(smem + C::OFF_TW)[bj * 256 + tg] =
                    make_uint2(Op<0>::pack(c0, c1), Op<0>::pack(s0, s1));
            else
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
    // input phase: column o, inputs n1 = 16 grp .. 16 grp + 15 of both sub-rows
    const int in_o = tg & 63, in_grp = tg >> 6;
    const uint32_t in_dst = (in_o >> 3) * C::SBO1 + (in_o & 7) * 16 + 4 * in_grp * C::LBO1;
    const uint32_t in_n = 1024u * uint32_t(in_grp) + uint32_t(in_o);  // n' of the first input

    const uint32_t bsm = smem_u32(bbuf);
    constexpr uint32_t id128 = tc::idesc(DT, 128, 128), id144 = tc::idesc(DT, 128, 144);
    const float scale = R0 == 2 ? 0.70710678118654752f : (R0 == 4 ? 0.5f : 0.35355339059327373f);  // 1 / sqrt(R0)

    bool mma_pending = false, in_pending = i0 < i1;  // the first row's copies were issued in the set-up
    uint32_t mmapar = 0, inpar = 0;
    uint32_t zfpar = 0, accpar = 0;  // R0 = 8: the staging-read and accumulator hand-over phases
    const uint32_t bar_id = 1 + g;
    bool failed = false;

    for (int it = i0; it < i1; ++it) {
        const int ri = item_row(it), p = item_pair(it);
        const int h = chan(ri);
        const bool sp = p == 0;
        // first / last: this pipeline's first and last input phase of the row;
        // fin: the row's output is written here
        const bool first = (it % IPR) == 0, last = (it % IPR) == IPR - 1, fin = p == 0;
        const int kA = p, kB = p ? R0 - p : R0 / 2;
        const size_t roff = mrow(ri) * RS;  // element offset of the row
        const bool has_next = it + 1 < i1;
        if (tg == 32 && has_next) {  // the next item's k_f into L2 (read by the next fold)
            const int rn = item_row(it + 1), pn = item_pair(it + 1), hn = chan(rn);
            if (pn != p || hn != h) bulk_prefetch_l2(kf_of(hn, pn), TcB::KFP * 16);
        }

        // ---------------- input: the outer stage for sub-rows kA, kB -> B1
        const float2 tin_a = __ldg(a.twin + kA * 256 + tg), tin_b = __ldg(a.twin + kB * 256 + tg);
        bool bad = false;
        if (first) bad = !mbar_wait_sleep(zbar, inpar, kWaitSleepLimit, kWaitHintNs);
        constexpr int NZW = NB;  // nonzero input blocks (n0 < R0/2; FULL: all)
        uint32_t zlo[16], zhi[16];
        if (!bad && R0 == 8) {
            // the radix-8 stage over the four nonzero blocks, with gating on the fly
            const cpx wa = twiddle_pow2(uint32_t(kA), 8), wb = twiddle_pow2(uint32_t(kB), 8);  // W_8^k0
            const float4 sa = steps[kA], sb = steps[kB];
            float4 tw = make_float4(tin_a.x, tin_b.x, tin_a.y, tin_b.y);
            const float4 st = make_float4(sa.x, sb.x, sa.y, sb.y);
            const uint32_t* wr = GATED ? reinterpret_cast<const uint32_t*>(a.w_in + roff) : nullptr;
            #pragma unroll 1
            for (int gq = 0; gq < 4; ++gq) {  // inputs n1 = 16 grp + 4 gq + 0..3
                uint32_t xa[4], xb[4];
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t n = in_n + 64 * uint32_t(4 * gq + e);
                    cpx zz[4];
                    #pragma unroll
                    for (int n0 = 0; n0 < 4; ++n0) {
                        uint32_t wd = zs[4096 * n0 + n];
                        if (GATED) wd = O::mul2(wd, __ldg(wr + 4096 * n0 + n));
                        zz[n0] = O::unpack(wd);
                    }
                    // sum_n0 W_8^(n0 k0) z_n0 by Horner's rule, for kA and kB
                    cpx xA = zz[3], xB = zz[3];
                    #pragma unroll
                    for (int n0 = 2; n0 >= 0; --n0) {
                        xA = cmul(xA, wa); xA.r += zz[n0].r; xA.i += zz[n0].i;
                        xB = cmul(xB, wb); xB.r += zz[n0].r; xB.i += zz[n0].i;
                    }
                    const float4 x = cmul2_split(xA.r, xB.r, xA.i, xB.i, tw);
                    xa[e] = O::pack(x.x, x.z);
                    xb[e] = O::pack(x.y, x.w);
                    tw = cmul2_split(tw.x, tw.y, tw.z, tw.w, st);
                }
                *reinterpret_cast<uint4*>(bbuf + in_dst + gq * C::LBO1) = make_uint4(xa[0], xa[1], xa[2], xa[3]);
                *reinterpret_cast<uint4*>(bbuf + in_dst + 8 * C::SBO1 + gq * C::LBO1) =
                    make_uint4(xb[0], xb[1], xb[2], xb[3]);
            }
        } else if (!bad) {
            #pragma unroll
            for (int i = 0; i < 16; ++i) {
                zlo[i] = zs[in_n + 64 * i];
                zhi[i] = NZW == 2 ? zs[4096 + in_n + 64 * i] : 0u;
            }
            if constexpr (GATED) {
                if (R0 == 2 && !FULL) {
                    #pragma unroll
                    for (int i = 0; i < 16; ++i) zlo[i] = O::mul2(zlo[i], wis[in_n + 64 * i]);
                } else if (first) {
                    const uint32_t* wr = reinterpret_cast<const uint32_t*>(a.w_in + roff);
                    uint32_t wl[16], wh[16];
                    #pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        wl[i] = __ldg(wr + in_n + 64 * i);
                        wh[i] = __ldg(wr + 4096 + in_n + 64 * i);
                    }
                    // the gated row for the row's next pair: every position is
                    // read and written by this thread only
                    #pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        zlo[i] = O::mul2(zlo[i], wl[i]);
                        zhi[i] = O::mul2(zhi[i], wh[i]);
                        zs[in_n + 64 * i] = zlo[i];
                        zs[4096 + in_n + 64 * i] = zhi[i];
                    }
                }
            }
            // twiddles W_M^(k0 n') / sqrt(R0) along n' = in_n + 64 i, both sub-rows
            // as the two halves of packed pairs: (A, B)
            const float4 sa = steps[kA], sb = steps[kB];
            float4 tw = make_float4(tin_a.x, tin_b.x, tin_a.y, tin_b.y);
            const float4 st = make_float4(sa.x, sb.x, sa.y, sb.y);
            const bool odd = (p & 1) != 0;  // R0 = 4, pair (1, 3): W_4^(kA) = -i, W_4^(kB) = i
            #pragma unroll
            for (int gq = 0; gq < 4; ++gq) {  // inputs n1 = 16 grp + 4 gq + 0..3: one 16-byte store per sub-row
                uint32_t xa[4], xb[4];
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 4 * gq + e;
                    const cpx l = O::unpack(zlo[i]);
                    cpx t = {0.f, 0.f};
                    if (R0 == 4 || FULL) {  // the second nonzero block
                        const cpx hh = O::unpack(zhi[i]);
                        t = odd ? cpx{hh.i, -hh.r} : hh;
                    }
                    const float4 x = cmul2_split(l.r + t.r, l.r - t.r, l.i + t.i, l.i - t.i, tw);
                    xa[e] = O::pack(x.x, x.z);
                    xb[e] = O::pack(x.y, x.w);
                    if (i + 1 < 16) tw = cmul2_split(tw.x, tw.y, tw.z, tw.w, st);
                }
                *reinterpret_cast<uint4*>(bbuf + in_dst + gq * C::LBO1) = make_uint4(xa[0], xa[1], xa[2], xa[3]);
                *reinterpret_cast<uint4*>(bbuf + in_dst + 8 * C::SBO1 + gq * C::LBO1) =
                    make_uint4(xb[0], xb[1], xb[2], xb[3]);
            }
        }
        tc::fence_proxy_async();
        tc::fence_before();
        if (tc::bar_vote(bar_id, 256, bad)) { failed = true; break; }
        if (first) {
            in_pending = false;
            inpar ^= 1;
        }
        if (tg == 0) {
            tc::fence_after();
            #pragma unroll
            for (int s = 0; s < 8; ++s)
                tc::mma(tD, tmem + 8 * s, tc::sdesc(bsm + 2 * s * C::LBO1, C::LBO1, C::SBO1), id128, s > 0);
            tc::commit(&bars[0]);
        }
        mma_pending = true;
        if (last && has_next) {  // the staging is free: fetch the next row
            if constexpr (C::SPLIT) {
                // both pipelines have to be done with it; pipeline 1 stages the next row
                if (tg == 64) {
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(zfree)) : "memory");
                    if (g == 1) {
                        if (mbar_wait_sleep(zfree, zfpar, kWaitSleepLimit, kWaitHintNs))
                            stage_row(ri + 1, smem, reinterpret_cast<uint64_t*>(smem + C::OFF_BAR));
                        else
                            atomicExch(a.err, 7);  // the next row's staging wait then gives up too
                    }
                }
                zfpar ^= 1;
            } else {
                if (tg == 64) stage_row(ri + 1, pb, bars);
            }
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
                    const float4 tw = twl(4 * b + jj);
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
        // the fold's k_f of chunks 0..3, read from L2 while the vote, S2 and its
        // wait run (chunks 4..7 follow during the fold's first half)
        const uint4* kft = kf_of(h, p) + (sp ? 9 : 8) * hf * 256 + w * 64 + lane;
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

        // ---------------- fold of this warpgroup's sub-row with the kernel spectrum -> B3
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
            const uint32_t dcol = tD + (sp ? 72 : 64) * hf;
            const uint32_t r0b = (sp ? 8 : 4) * hf * C::SBO3 + 16 * q;
            const int X = sp ? (hf ? 127 : 64) : 127 - 32 * hf;   // row of s1 at chunk 0 (q = 0)
            const uint32_t r1p[2] = {rowoff(X - q), rowoff(X - 4 - q)};
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
                    const float4 tw = twl(4 * b + jj);
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

        // ---------------- S4 post: the inverse outer stage.  This thread's
        // outputs n' = 64 kappa_b + 32 hf + 8 jj + 2q + e of both sub-rows.
        // gated, last pair: w_out at (b, jj, n0), read while the contraction
        // runs (R0 = 2; R0 = 4 and the circular rows read it at the store,
        // registers being short)
        constexpr bool WPRE = GATED && R0 == 2 && !FULL;
        uint2 wov[2][4][WPRE ? NB : 1];
        if constexpr (WPRE) {
          if (last) {
            #pragma unroll
            for (int b = 0; b < 2; ++b)
                #pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    #pragma unroll
                    for (int n0 = 0; n0 < NB; ++n0)
                        wov[b][jj][n0] = __ldg(reinterpret_cast<const uint2*>(
                            a.w_out + roff + 2 * size_t(4096 * n0 + 64 * (b ? kapB : kapA) + 32 * hf + 2 * q + 8 * jj)));
          }
        }
        // the starting twiddles of this thread's outputs, read while the contraction runs
        float4 tstart[2][2];  // [sub-row A, B][b]
        #pragma unroll
        for (int b = 0; b < 2; ++b) {
            tstart[0][b] = __ldg(a.twout + (kA * 2 + b) * 256 + tg);
            tstart[1][b] = __ldg(a.twout + (kB * 2 + b) * 256 + tg);
        }
        // R0 = 4, last pair: pair (1, 3)'s S and D of block 0, read while the
        // contraction runs (block 1's are read in the loop; all eight would spill)
        uint4 sdp[R0 == 4 ? 4 : 1];
        if constexpr (R0 == 4 && !C::SPLIT) {
            if (last) {
                #pragma unroll
                for (int c = 0; c < 4; ++c) sdp[c] = a.skip1 ? make_uint4(0, 0, 0, 0) : tout[c * 256];
            }
        }
        bad = !mbar_wait_sleep(&bars[0], mmapar, kWaitSleepLimit, kWaitHintNs);
        // R0 = 8: the accumulator's turn (pair 1 of the CTA's first row starts it)
        const bool acc_wait = C::SPLIT && !(p == 1 && it == i0);
        if (acc_wait) bad |= !mbar_wait_sleep(&accbar[g == 0 ? 1 : 0], accpar, kWaitSleepLimit, kWaitHintNs);
        bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the collective TMEM loads
        tc::fence_after();
        if (acc_wait) accpar ^= 1;
        if constexpr (C::SPLIT) {
          if (!bad) {
            uint32_t vr[2][2][16];
            tc::ld16x256b_x4(tD + laneA + 32 * hf, vr[0][0]);
            tc::ld16x256b_x4(tD + laneB + 32 * hf, vr[0][1]);
            tc::ld16x256b_x4(tD + laneA + 64 + 32 * hf, vr[1][0]);
            tc::ld16x256b_x4(tD + laneB + 64 + 32 * hf, vr[1][1]);
            // c[n0] = W_8^(n0 kA) V_A + W_8^(n0 kB) V_B, V = W_M^(k0 n') T, added
            // to the accumulator of the four output blocks n0 < 4
            const cpx wa = twiddle_pow2(uint32_t(kA), 8), wb = twiddle_pow2(uint32_t(kB), 8);
            const float4 sB = steps[kB], sA = steps[kA];
            const float4 stB = make_float4(sB.z, sB.z, sB.w, sB.w), stA = make_float4(sA.z, sA.z, sA.w, sA.w);
            tc::wait_ld();
            #pragma unroll
            for (int b = 0; b < 2; ++b) {
                const uint32_t n0p = uint32_t(64 * (b ? kapB : kapA) + 32 * hf + 2 * q);
                float4 twA = tstart[0][b], twB = tstart[1][b];
                #pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint32_t* va = vr[0][b] + 4 * jj;
                    const uint32_t* vb = vr[1][b] + 4 * jj;
                    const float4 vA = cmul2_split(__uint_as_float(va[0]), __uint_as_float(va[1]), __uint_as_float(va[2]),
                                                  __uint_as_float(va[3]), twA);
                    const float4 vB = cmul2_split(__uint_as_float(vb[0]), __uint_as_float(vb[1]), __uint_as_float(vb[2]),
                                                  __uint_as_float(vb[3]), twB);
                    if (jj + 1 < 4) {
                        twA = cmul2_split(twA.x, twA.y, twA.z, twA.w, stA);
                        twB = cmul2_split(twB.x, twB.y, twB.z, twB.w, stB);
                    }
                    cpx al = {1.f, 0.f}, be = {1.f, 0.f};  // W_8^(n0 kA), W_8^(n0 kB)
                    #pragma unroll
                    for (int n0 = 0; n0 < 4; ++n0) {
                        const float4 x = cmul2_split(vA.x, vA.y, vA.z, vA.w, make_float4(al.r, al.r, al.i, al.i));
                        const float4 yv = cmul2_split(vB.x, vB.y, vB.z, vB.w, make_float4(be.r, be.r, be.i, be.i));
                        float4 cc = make_float4(x.x + yv.x, x.y + yv.y, x.z + yv.z, x.w + yv.w);
                        uint2* ap = accs + ((4 * b + jj) * 4 + n0) * 256;
                        if (p != 1) {  // pairs 2, 3, 0 add to the accumulator
                            const uint2 old = *ap;
                            const cpx o0 = O::unpack(old.x), o1 = O::unpack(old.y);
                            cc.x += o0.r; cc.y += o1.r; cc.z += o0.i; cc.w += o1.i;
                        }
                        if (!fin) {
                            *ap = make_uint2(O::pack(cc.x, cc.z), O::pack(cc.y, cc.w));
                        } else {
                            // y_z = conj(sum / sqrt(8)): y[2n] = Re, y[2n+1] = -Im
                            const size_t yo = roff + 2 * size_t(n0p + 8 * jj + 4096 * n0);
                            float r0 = scale * cc.x, r1 = scale * cc.y, im0 = -scale * cc.z, im1 = -scale * cc.w;
                            if (GATED) {
                                const uint2 wv = __ldg(reinterpret_cast<const uint2*>(a.w_out + yo));
                                const cpx w0 = O::unpack(wv.x), w1 = O::unpack(wv.y);
                                r0 *= w0.r; im0 *= w0.i; r1 *= w1.r; im1 *= w1.i;
                            }
                            *reinterpret_cast<uint2*>(a.y + yo) = make_uint2(O::pack(r0, im0), O::pack(r1, im1));
                        }
                        al = cmul(al, wa);
                        be = cmul(be, wb);
                    }
                }
            }
            // the accumulator to the other pipeline (release of this thread's writes)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&accbar[g == 0 ? 0 : 1]))
                         : "memory");
          }
        } else if (!bad) {
            uint32_t vr[2][2][16];
            tc::ld16x256b_x4(tD + laneA + 32 * hf, vr[0][0]);
            tc::ld16x256b_x4(tD + laneB + 32 * hf, vr[0][1]);
            tc::ld16x256b_x4(tD + laneA + 64 + 32 * hf, vr[1][0]);
            tc::ld16x256b_x4(tD + laneB + 64 + 32 * hf, vr[1][1]);
            // twiddles W_M^(k0 n') for sub-row B (k0 = kB) and, on pair (1, 3),
            // sub-row A (k0 = kA = 1); e = 0, 1 as the two halves of packed pairs
            const float4 sB = steps[kB], sA = steps[kA];
            const float4 stB = make_float4(sB.z, sB.z, sB.w, sB.w), stA = make_float4(sA.z, sA.z, sA.w, sA.w);
            tc::wait_ld();
            #pragma unroll
            for (int b = 0; b < 2; ++b) {
                const uint32_t n0p = uint32_t(64 * (b ? kapB : kapA) + 32 * hf + 2 * q);
                float4 twB = tstart[1][b];
                float4 twA = tstart[0][b];  // k0 = kA = 1 on pair (1, 3)
                const uint32_t* va = vr[0][b];
                const uint32_t* vb = vr[1][b];
                #pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    // sub-row A (k0 = kA), sub-row B (k0 = kB): (re e0, re e1, im e0, im e1)
                    const float4 tA = make_float4(__uint_as_float(va[4 * jj]), __uint_as_float(va[4 * jj + 1]),
                                                  __uint_as_float(va[4 * jj + 2]), __uint_as_float(va[4 * jj + 3]));
                    const float4 vB = cmul2_split(__uint_as_float(vb[4 * jj]), __uint_as_float(vb[4 * jj + 1]),
                                                  __uint_as_float(vb[4 * jj + 2]), __uint_as_float(vb[4 * jj + 3]), twB);
                    if (jj + 1 < 4) twB = cmul2_split(twB.x, twB.y, twB.z, twB.w, stB);
                    if (!last) {
                        // pair (1, 3): S = V1 + V3, D = -i (V1 - V3)
                        const float4 vA = cmul2_split(tA.x, tA.y, tA.z, tA.w, twA);
                        if (jj + 1 < 4) twA = cmul2_split(twA.x, twA.y, twA.z, twA.w, stA);
                        const float4 S = make_float4(vA.x + vB.x, vA.y + vB.y, vA.z + vB.z, vA.w + vB.w);
                        const float4 D = make_float4(vA.z - vB.z, vA.w - vB.w, vB.x - vA.x, vB.y - vA.y);
                        tout[(4 * b + jj) * 256] = make_uint4(O::pack(S.x, S.z), O::pack(S.y, S.w),
                                                              O::pack(D.x, D.z), O::pack(D.y, D.w));
                    } else {
                        // (re e0, re e1, im e0, im e1) of each output block n0
                        float4 out[NB];
                        if constexpr (R0 == 2) {
                            out[0] = make_float4(scale * (tA.x + vB.x), scale * (tA.y + vB.y), scale * (tA.z + vB.z),
                                                 scale * (tA.w + vB.w));
                            if constexpr (FULL)  // block 1: W_2^(1 * 1) = -1 on sub-row 1
                                out[NB - 1] = make_float4(scale * (tA.x - vB.x), scale * (tA.y - vB.y),
                                                          scale * (tA.z - vB.z), scale * (tA.w - vB.w));
                        } else {
                            const uint4 sd = b == 0 ? sdp[R0 == 4 ? jj : 0]
                                                    : (a.skip1 ? make_uint4(0, 0, 0, 0) : tout[(4 * b + jj) * 256]);
                            const cpx s0 = O::unpack(sd.x), s1 = O::unpack(sd.y);
                            const cpx d0 = O::unpack(sd.z), d1 = O::unpack(sd.w);
                            out[0] = make_float4(scale * (tA.x + vB.x + s0.r), scale * (tA.y + vB.y + s1.r),
                                                 scale * (tA.z + vB.z + s0.i), scale * (tA.w + vB.w + s1.i));
                            out[NP - 1] = make_float4(scale * (tA.x - vB.x + d0.r), scale * (tA.y - vB.y + d1.r),
                                                      scale * (tA.z - vB.z + d0.i), scale * (tA.w - vB.w + d1.i));
                        }
                        uint16_t* yr = a.y + roff + 2 * size_t(n0p + 8 * jj);
                        #pragma unroll
                        for (int n0 = 0; n0 < NB; ++n0) {
                            // y_z = conj(out): y[2n] = Re, y[2n+1] = -Im
                            float r0 = out[n0].x, r1 = out[n0].y, im0 = -out[n0].z, im1 = -out[n0].w;
                            if (GATED) {
                                const uint2 wv = WPRE ? wov[b][jj][n0]
                                                      : __ldg(reinterpret_cast<const uint2*>(
                                                            a.w_out + roff + 2 * size_t(n0p + 8 * jj + 4096 * n0)));
                                const cpx w0 = O::unpack(wv.x), w1 = O::unpack(wv.y);
                                r0 *= w0.r; im0 *= w0.i; r1 *= w1.r; im1 *= w1.i;
                            }
                            *reinterpret_cast<uint2*>(yr + 2 * 4096 * n0) =
                                make_uint2(O::pack(r0, im0), O::pack(r1, im1));
                        }
                    }
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
        if (in_pending) mbar_wait_bounded(zbar, inpar, kWaitLimit);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (threadIdx.x < 32) tc::dealloc(tmem, C::TMEM_COLS);
}

}  // namespace fftconv
