// Fused causal long convolution for N = M = 4096 as an order-2 Monarch
// product, 4096 = 64 x 64, on the fifth-generation tensor cores (tcgen05).
//
// Decimation-in-time packing (FlashFFTConv page, section 3.4, "The
// real-valued FFT optimization"): z[n] = x[2n] + i x[2n+1], n < 2048, and
// z[n] = 0 above (implicit zero padding, "Implicit zero-padding").
// Monarch factorization ("The Monarch FFT Decomposition"), decimation in
// frequency, n = 64 n1 + o, k = k1 + 64 k2:
//   S1  X[k1][o]  = W_M^(o k1) * sum_{n1 < 32} z[64 n1 + o] W_64^(n1 k1) / 8
//   S2  Z[k1 + 64 k2] = sum_o X[k1][o] W_64^(o k2) / 8
//   fold  C[k] = conj(Z_y[k]) = alpha~_k conj Z[k] + beta~_k Z[M - k]
//   S3  T[k1][o]  = W_M^(o k1) * sum_{k2} C[k1 + 64 k2] W_64^(k2 o) / 8
//   S4  y_z[64 n1 + o] = conj( sum_{k1} T[k1][o] W_64^(n1 k1) / 8 ),  n1 < 32
// (the inverse as the conjugate of the forward transform of conj Z_y, in
// reverse stage order; the causal truncation keeps n1 < 32 only).
//
// Every stage is one dense contraction D = F64 x B on the tensor cores: the
// real-embedded 64-point DFT matrix F64 ([[Fr, -Fi], [Fi, Fr]] interleaved
// along K, scaled by 1/8) is the A operand and stays in tensor memory for
// the whole kernel; the data is the B operand (K = the contracted index, N =
// the independent vectors) in shared memory; the float32 accumulator D is in
// tensor memory.  The DFT matrix rows (outputs) are permuted so that, with
// 16x256b loads, a thread receives the real and imaginary parts of the same
// output, and -- for the fold -- outputs k2 and 63 - k2 together:
//   TMEM lane L = 32w + 16b + 8p + r  <->  output kappa = b ? 63 - 8w - r : 8w + r,
//   part p (0 real, 1 imaginary).
// The same row order serves all four stages; S4 runs with M = 64 on the
// b = 0 lanes, which hold exactly the outputs n1 < 32 that the truncation
// keeps.
//
// Fold pairing: bin (k1, k2) pairs with (64 - k1, 63 - k2) (k1 > 0).  S2's
// columns (N "slots") put sub-problems s and 64 - s in adjacent columns
// (s = 4m + q, m = 0..7, q = 0..3 at slots 8m + 2q and 8m + 2q + 1), so a
// thread holds both bins of every pair it needs.  Sub-problem 32 pairs with
// itself (bins k2 and 63 - k2) and sits beside a copy of itself; sub-problem
// 0 pairs bin k2 with 64 - k2 and sits beside a copy pre-twiddled by W_64^o,
// whose transform is Z[64 (k2 + 1)].  Columns 66..71 are padding; the second
// row's slots follow at 72.
//
// Rows shorter than 4096 (Nu = 1024, 2048) run as the same transform of the
// row zero-padded to 4096 (the staging beyond the copied Nu / 2 words stays
// zero), and only the outputs n < Nu / 2 are stored: a causal convolution's
// first Nu outputs do not depend on anything beyond position Nu.
//
// Work item = two rows of the same channel (b = 2p, 2p + 1): every
// contraction covers both rows (N = 128, 144 for S2), which halves the number
// of tensor-core instructions per row (each one costs about the same up to
// N = 128).  Each CTA runs two independent item pipelines that share the DFT
// matrix; while one pipeline waits for its contraction the other one does its
// register work.  A pipeline has eight warps: two warpgroups on the same 128
// TMEM lanes, each handling half of the columns of S1/S3/S4 and one row of
// the fold.  u and w_in of an item are staged by bulk copies (TMA engine)
// one item ahead, k_f of a channel when the channel changes; w_out is read
// through L2 (prefetched by the TMA engine at the start of the item).
#pragma once
#include "mma.cuh"
#include "tc.cuh"

namespace fftconv {

struct Tc64Args {
    const uint16_t* u;
    const uint16_t* w_in;
    const uint16_t* w_out;
    const uint8_t* kf;      // [h][chunk 9][warp 4][half 2][lane 32] uint4
    uint16_t* y;
    const uint32_t* fmat;   // [3][lane 128][64 words]: F64/8 with permuted rows; columns natural, P3, P4
    int B, H;
    int* err;
    int Nu;                 // row length of u, w_in, w_out and y: 4096, or 1024 / 2048 (the row zero-padded
                            // to 4096: the causal convolution's first Nu outputs are those of the padded rows)
};

struct Tc64 {
    static constexpr int M = 4096;
    static constexpr int THREADS = 512;   // two pipelines of 256
    // B operand layouts, two rows side by side along N: (LBO, SBO) in bytes.
    // B1: K = 64 (n1 < 32) x N = 128 (row, o).  B2: K = 128 (o) x N = 144
    // (row, slot).  B3: K = 128 (k2) x N = 128 (row, k1) plus a trash row
    // group at row 128.  B4: K = 128 (k1) x N = 128 (row, o).  The 16-byte
    // pad per core matrix makes the stores of S1 post and of the input pass
    // conflict free and those of the fold and S3 post at most 2-way.
    static constexpr uint32_t LBO1 = 128, SBO1 = 1024;
    static constexpr uint32_t LBO2 = 144, SBO2 = 2304;
    static constexpr uint32_t LBO3 = 144, SBO3 = 2304;
    static constexpr uint32_t LBO4 = 144, SBO4 = 2304;
    static constexpr uint32_t TRASH = 16 * SBO3;
    static constexpr uint32_t BBUF = 18 * SBO2;       // 41472: B2, and B3 with its trash group
    static constexpr uint32_t STG = 8192;             // one staged row of u or w_in (2048 words)
    static constexpr uint32_t KFB = 9 * 4 * 2 * 32 * 16;  // k_f of one channel: 36864
    static constexpr uint32_t OFF_B = 0, OFF_ST = BBUF, OFF_KF = OFF_ST + 4 * STG;  // staging: u A, u B, w_in A, w_in B
    static constexpr uint32_t PIPE = OFF_KF + KFB;    // 111104 per pipeline
    static constexpr uint32_t OFF_W64 = 2 * PIPE;     // W_64^o table (32 float4)
    static constexpr uint32_t OFF_BAR = OFF_W64 + 512;
    static constexpr uint32_t SMEM = OFF_BAR + 6 * 8;
    // TMEM columns: F64 at 0..63 (columns natural, for S1 and S2), 64..127
    // (columns in the order P3, for S3), 128..191 (order P4, for S4);
    // pipeline g's accumulator at 192 + 160 g (144 columns).
    static constexpr uint32_t TMEM_COLS = 512;
};

// K positions of the B3 and B4 operands (and columns of the matching F64
// copies): a permutation of the 64 inputs that makes the fold's and S3
// post's shared-memory stores free of bank conflicts under the 144-byte pad.
__host__ __device__ constexpr int tc64_p3(int k2) {
    return k2 < 32 ? 4 * (k2 >> 3) + (k2 & 3) + 16 * ((k2 >> 2) & 1) : 32 + tc64_p3(63 - k2);
}
__host__ __device__ constexpr int tc64_p4(int s) {
    return 4 * ((s >> 3) & 3) + 32 * (s >> 5) + 2 * ((s >> 1) & 1) + 16 * ((s >> 2) & 1) + (s & 1);
}

// Complex products of two values (real parts r0, r1, imaginary parts i0, i1)
// with two twiddles given as (wr0, wr1, wi0, wi1); returns (re0, re1, im0, im1).
__device__ __forceinline__ float4 cmul2_twiddle(float r0, float r1, float i0, float i1, float4 w) {
    return cmul2_split(r0, r1, i0, i1, w);
}

// Slot (S2 column) of sub-problem s.
__device__ __forceinline__ int tc64_slot(int s) {
    if (s <= 31) return 8 * (s >> 2) + 2 * (s & 3);
    if (s == 32) return 64;
    const int x = 64 - s;
    return 8 * (x >> 2) + 2 * (x & 3) + 1;
}

template <int DT, bool GATED>
__global__ void __launch_bounds__(Tc64::THREADS, 1) tc64_conv_kernel(const Tc64Args a) {
    using O = Op<DT>;
    using C = Tc64;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint32_t s_tmem;

    const int g = threadIdx.x >> 8, tg = threadIdx.x & 255;
    const int hf = tg >> 7, w = (tg >> 5) & 3, lane = tg & 31, r = lane >> 2, q = lane & 3;
    uint8_t* pb = smem + g * C::PIPE;
    uint8_t* bbuf = pb + C::OFF_B;
    const uint4* kfs = reinterpret_cast<const uint4*>(pb + C::OFF_KF);
    const float4* w64 = reinterpret_cast<const float4*>(smem + C::OFF_W64);
    const uint32_t* stg = reinterpret_cast<const uint32_t*>(pb + C::OFF_ST);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 3 * g;  // kf, mma, in

    // items: pairs of rows (b = 2p, 2p + 1) of one channel, channel-major
    const int P = (a.B + 1) >> 1, items = P * a.H;  // the host guarantees B*H < 2^30
    const int V = int(gridDim.x) * 2, v = int(blockIdx.x) * 2 + g;
    const int i0 = int(int64_t(v) * items / V), i1 = int(int64_t(v + 1) * items / V);

    // ---------------- set-up: barriers, TMEM, tables
    if (threadIdx.x == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + i, 1);
        fence_mbar_init();
        // the first item's inputs and k_f of both pipelines, overlapping the set-up below
        for (int gp = 0; gp < 2; ++gp) {
            const int vp = int(blockIdx.x) * 2 + gp;
            const int j0 = int(int64_t(vp) * items / V), j1 = int(int64_t(vp + 1) * items / V);
            if (j0 >= j1) continue;
            uint8_t* pbp = smem + gp * C::PIPE;
            uint64_t* bp = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + 3 * gp;
            const int h0 = int(unsigned(j0) / unsigned(P)), b0 = 2 * (j0 - h0 * P);
            const bool okB0 = b0 + 1 < a.B;
            const uint32_t stg = uint32_t(a.Nu) * 2u;  // bytes of a row
            const size_t bA = (size_t(b0) * a.H + h0) * a.Nu, bB = (size_t(okB0 ? b0 + 1 : 0) * a.H + h0) * a.Nu;
            mbar_expect_tx(&bp[2], stg * (okB0 ? 2u : 1u) * (GATED ? 2u : 1u));
            bulk_g2s(pbp + C::OFF_ST, a.u + bA, stg, &bp[2]);
            if (okB0) bulk_g2s(pbp + C::OFF_ST + C::STG, a.u + bB, stg, &bp[2]);
            if (GATED) {
                bulk_g2s(pbp + C::OFF_ST + 2 * C::STG, a.w_in + bA, stg, &bp[2]);
                if (okB0) bulk_g2s(pbp + C::OFF_ST + 3 * C::STG, a.w_in + bB, stg, &bp[2]);
            }
            mbar_expect_tx(&bp[0], C::KFB);
            bulk_g2s(pbp + C::OFF_KF, a.kf + size_t(h0) * C::KFB, C::KFB, &bp[0]);
        }
    }
    if (threadIdx.x < 32) {
        tc::alloc(&s_tmem, C::TMEM_COLS);
        // W_64^o, W_64^(o+1) for o = 2*lane: (wr0, wr1, wi0, wi1)
        float s0, c0, s1, c1;
        sincospif(-float(2 * lane) / 32.f, &s0, &c0);
        sincospif(-float(2 * lane + 1) / 32.f, &s1, &c1);
        reinterpret_cast<float4*>(smem + C::OFF_W64)[lane] = make_float4(c0, c1, s0, s1);
    }
    for (uint32_t i = threadIdx.x; i < 2 * C::BBUF / 16; i += blockDim.x) {  // padding columns start finite
        const uint32_t pi = i / (C::BBUF / 16), off = (i % (C::BBUF / 16)) * 16;
        *reinterpret_cast<uint4*>(smem + pi * C::PIPE + off) = make_uint4(0, 0, 0, 0);
    }
    if (a.Nu < C::M) {  // the zero padding beyond a short row: the staging tails that no copy writes
        const uint32_t head = uint32_t(a.Nu) * 2u, tail = (C::STG - head) / 16;
        for (uint32_t i = threadIdx.x; i < 8 * tail; i += blockDim.x) {
            const uint32_t slot = i / tail, off = head + (i % tail) * 16;  // 2 pipelines x 4 staged rows
            *reinterpret_cast<uint4*>(smem + (slot >> 2) * C::PIPE + C::OFF_ST + (slot & 3) * C::STG + off) =
                make_uint4(0, 0, 0, 0);
        }
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

    // Per-thread twiddles W_M^(kappa (8j + 2q + e)) for this warpgroup's
    // chunks j = 4 hf + jj: S1 (kappa = k1, columns o) and S3 (kappa = o,
    // columns k1) use the same values.
    const int kapA = 8 * w + r, kapB = 63 - kapA;
    float4 tw[2][4];
    #pragma unroll
    for (int b = 0; b < 2; ++b)
        #pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int kap = b ? kapB : kapA, o0 = 8 * (4 * hf + jj) + 2 * q;
            float s0, c0, s1, c1;
            sincospif(-float((kap * o0) & (C::M - 1)) / 2048.f, &s0, &c0);
            sincospif(-float((kap * (o0 + 1)) & (C::M - 1)) / 2048.f, &s1, &c1);
            tw[b][jj] = make_float4(c0, c1, s0, s1);
        }
    // per-thread shared-memory offsets (row R of the item adds 9R SBO2 / 8R SBO3 / 8R SBO4)
    const uint32_t kq2 = (q >> 1) * C::LBO2 + (q & 1) * 8 + 8 * hf * C::LBO2;
    // B4 K position of columns s = 8 (4 hf + jj) + 2q (+1): tc64_p4 = 4 jj + 32 hf + 2 (q&1) + 16 (q>>1)
    const uint32_t kq4 = (4 * (q >> 1) + 8 * hf) * C::LBO4 + (q & 1) * 8;
    uint32_t row2[2], row4[2];
    #pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int kap = b ? kapB : kapA, sl = tc64_slot(kap);
        row2[b] = (sl >> 3) * C::SBO2 + (sl & 7) * 16;
        row4[b] = (kap >> 3) * C::SBO4 + (kap & 7) * 16;
    }
    const bool is_k0 = kapA == 0, is_k32 = kapB == 32;
    auto rowoff3 = [](int s) -> uint32_t { return uint32_t(s >> 3) * C::SBO3 + uint32_t(s & 7) * 16; };
    // fold of row hf: B3 rows 64 hf + s
    const uint32_t r3q = uint32_t(q) * 16 + 8 * hf * C::SBO3;   // + (j/2) SBO3 + (j%2) 64: row of s = 4j + q
    const uint32_t r3p[2] = {rowoff3(64 - q) + 8 * hf * C::SBO3,   // - (j/2) SBO3: row of 64 - 4j - q
                             rowoff3(60 - q) + 8 * hf * C::SBO3};
    const uint32_t r3c0 = q == 0 ? C::TRASH : r3p[0];              // chunk 0: 64 - q, or the copy of 0
    const uint32_t r3s32 = q == 0 ? 4 * C::SBO3 + 8 * hf * C::SBO3 : C::TRASH;  // chunk 8: sub-problem 32
    auto koff3 = [](int k2) -> uint32_t {  // B3 K position of input k2
        const int pos = tc64_p3(k2);
        return uint32_t(pos >> 2) * C::LBO3 + uint32_t(pos & 3) * 4;
    };
    const uint32_t kAo = koff3(kapA), kBo = koff3(kapB);
    // input pass: row hf, column o, inputs n1 = 16 in_g .. 16 in_g + 15
    const int in_o = tg & 63, in_g = (tg >> 6) & 1;
    const uint32_t in_dst = (8 * hf + (in_o >> 3)) * C::SBO1 + (in_o & 7) * 16 + 4 * in_g * C::LBO1;

    const uint32_t bsm = smem_u32(bbuf);
    constexpr uint32_t id1 = tc::idesc(DT, 128, 128), id2 = tc::idesc(DT, 128, 144),
                       id3 = tc::idesc(DT, 128, 128), id4 = tc::idesc(DT, 64, 128);

    auto chan = [&](int it) -> int { return int(unsigned(it) / unsigned(P)); };
    auto row_of = [&](int it, int R, bool& valid) -> int {  // row b*H + h of row R of item it
        const int h = chan(it), b = 2 * (it - h * P) + R;
        valid = b < a.B;
        return (valid ? b : 0) * a.H + h;
    };
    // u and w_in of both rows into the staging buffers (one bulk copy each)
    auto stage_item = [&](int it) {
        bool okA, okB;
        const uint32_t stg = uint32_t(a.Nu) * 2u;  // bytes of a row
        const size_t bA = size_t(row_of(it, 0, okA)) * a.Nu, bB = size_t(row_of(it, 1, okB)) * a.Nu;
        mbar_expect_tx(&bars[2], stg * (okB ? 2u : 1u) * (GATED ? 2u : 1u));
        bulk_g2s(pb + C::OFF_ST, a.u + bA, stg, &bars[2]);
        if (okB) bulk_g2s(pb + C::OFF_ST + C::STG, a.u + bB, stg, &bars[2]);
        if (GATED) {
            bulk_g2s(pb + C::OFF_ST + 2 * C::STG, a.w_in + bA, stg, &bars[2]);
            if (okB) bulk_g2s(pb + C::OFF_ST + 3 * C::STG, a.w_in + bB, stg, &bars[2]);
        }
    };
    auto issue_kf = [&](int h) {
        mbar_expect_tx(&bars[0], C::KFB);
        bulk_g2s(pb + C::OFF_KF, a.kf + size_t(h) * C::KFB, C::KFB, &bars[0]);
    };

    // pending phases and the parity of the next phase to consume, per barrier
    bool kf_pending = false, mma_pending = false, in_pending = false;
    uint32_t kfpar = 0, mmapar = 0, inpar = 0;
    if (i0 < i1) {  // the first item's copies were issued during the set-up
        kf_pending = true;
        in_pending = true;
    }
    const uint32_t bar_id = 1 + g;
    bool failed = false;

    for (int it = i0; it < i1; ++it) {
        const int h = chan(it);
        const bool has_next = it + 1 < i1;
        bool okA, okB;
        const int rowA = row_of(it, 0, okA), rowB = row_of(it, 1, okB);
        if (GATED && tg == 32) {  // w_out of this item into L2 (read in S4 post)
            bulk_prefetch_l2(a.w_out + size_t(rowA) * a.Nu, uint32_t(a.Nu) * 2u);
            if (okB) bulk_prefetch_l2(a.w_out + size_t(rowB) * a.Nu, uint32_t(a.Nu) * 2u);
        }

        // ---------------- input: z (times w_in) of row hf -> B1
        bool bad = !mbar_wait_sleep(&bars[2], inpar, kWaitSleepLimit, kWaitHintNs);
        if (!bad) {
            const bool ok = hf ? okB : okA;
            const uint32_t* ur = stg + hf * (C::STG / 4);
            const uint32_t* wr = stg + (2 + hf) * (C::STG / 4);
            uint32_t z[16], zw[16];
            #pragma unroll
            for (int i = 0; i < 16; ++i) {
                z[i] = ok ? ur[(16 * in_g + i) * 64 + in_o] : 0u;
                if (GATED) zw[i] = ok ? wr[(16 * in_g + i) * 64 + in_o] : 0u;
            }
            #pragma unroll
            for (int i = 0; i < 16; ++i)
                if (GATED) z[i] = O::mul2(z[i], zw[i]);
            #pragma unroll
            for (int gq = 0; gq < 4; ++gq)
                *reinterpret_cast<uint4*>(bbuf + in_dst + gq * C::LBO1) =
                    make_uint4(z[4 * gq], z[4 * gq + 1], z[4 * gq + 2], z[4 * gq + 3]);
        }
        tc::fence_proxy_async();
        tc::fence_before();
        if (tc::bar_vote(bar_id, 256, bad)) { failed = true; break; }
        in_pending = false;
        inpar ^= 1;
        if (tg == 0) {
            tc::fence_after();
            #pragma unroll
            for (int s = 0; s < 4; ++s)
                tc::mma(tD, tmem + 8 * s, tc::sdesc(bsm + 2 * s * C::LBO1, C::LBO1, C::SBO1), id1, s > 0);
            tc::commit(&bars[1]);
        }
        mma_pending = true;
        if (has_next) {  // the staging is free: fetch the next item
            if (tg == 64) stage_item(it + 1);
            in_pending = true;
        }

        // ---------------- S1 post: twiddle, -> B2 (slot rows)
        bad = !mbar_wait_sleep(&bars[1], mmapar, kWaitSleepLimit, kWaitHintNs);
        bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the collective TMEM loads
        tc::fence_after();
        if (!bad) {
            uint32_t vr[2][2][16];  // [row][block]: row 1's loads fly while row 0 is processed
            tc::ld16x256b_x4(tD + laneA + 32 * hf, vr[0][0]);
            tc::ld16x256b_x4(tD + laneB + 32 * hf, vr[0][1]);
            tc::wait_ld();
            tc::ld16x256b_x4(tD + laneA + 64 + 32 * hf, vr[1][0]);
            tc::ld16x256b_x4(tD + laneB + 64 + 32 * hf, vr[1][1]);
            #pragma unroll
            for (int R = 0; R < 2; ++R) {
                float4 x0[4];   // k1 = 0 (block a): kept for the pre-twiddled copy
                uint2 p32[4];   // k1 = 32 (block b): kept for the duplicate
                if (R == 1) tc::wait_ld();
                #pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const uint32_t* vv = vr[R][b];
                    uint8_t* dst = bbuf + row2[b] + 9 * R * C::SBO2 + kq2;
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float4 x = cmul2_twiddle(__uint_as_float(vv[4 * jj]), __uint_as_float(vv[4 * jj + 1]),
                                                     __uint_as_float(vv[4 * jj + 2]), __uint_as_float(vv[4 * jj + 3]),
                                                     tw[b][jj]);
                        const uint2 wd = make_uint2(O::pack(x.x, x.z), O::pack(x.y, x.w));
                        *reinterpret_cast<uint2*>(dst + 2 * jj * C::LBO2) = wd;
                        if (b == 0) x0[jj] = x;
                        else p32[jj] = wd;
                    }
                }
                if (is_k0) {  // sub-problem 0 again, pre-twiddled by W_64^o (slot 1)
                    float4 wv[4];
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj) wv[jj] = w64[4 * (4 * hf + jj) + q];
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float4 y0 = cmul2_twiddle(x0[jj].x, x0[jj].y, x0[jj].z, x0[jj].w, wv[jj]);
                        *reinterpret_cast<uint2*>(bbuf + 9 * R * C::SBO2 + 16 + kq2 + 2 * jj * C::LBO2) =
                            make_uint2(O::pack(y0.x, y0.z), O::pack(y0.y, y0.w));
                    }
                }
                if (is_k32) {  // sub-problem 32 again (slot 65)
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        *reinterpret_cast<uint2*>(bbuf + (9 * R + 8) * C::SBO2 + 16 + kq2 + 2 * jj * C::LBO2) = p32[jj];
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
                tc::mma(tD, tmem + 8 * s, tc::sdesc(bsm + 2 * s * C::LBO2, C::LBO2, C::SBO2), id2, s > 0);
            tc::commit(&bars[1]);
        }
        mma_pending = true;

        // ---------------- fold of row hf with the kernel spectrum -> B3
        bad = !mbar_wait_sleep(&bars[1], mmapar, kWaitSleepLimit, kWaitHintNs);
        if (kf_pending) bad |= !mbar_wait_sleep(&bars[0], kfpar, kWaitSleepLimit, kWaitHintNs);
        bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the collective TMEM loads
        tc::fence_after();
        if (!bad) {
            auto fold4 = [&](int j, const uint32_t* va, const uint32_t* vb, const uint4 (&k)[2], uint32_t r0,
                             uint32_t r1) {
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
            const uint32_t dcol = tD + 72 * hf;  // this warpgroup's row in S2's columns
            #pragma unroll
            for (int gq = 0; gq < 2; ++gq) {  // chunks 4 gq .. 4 gq + 3
                uint32_t va[16], vb[16];
                uint4 kv[4][2];
                tc::ld16x256b_x4(dcol + laneA + 32 * gq, va);
                tc::ld16x256b_x4(dcol + laneB + 32 * gq, vb);
                #pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    kv[jj][0] = kfs[(((4 * gq + jj) * 4 + w) * 2 + 0) * 32 + lane];
                    kv[jj][1] = kfs[(((4 * gq + jj) * 4 + w) * 2 + 1) * 32 + lane];
                }
                tc::wait_ld();
                #pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = 4 * gq + jj;
                    const uint32_t r0 = r3q + (j >> 1) * C::SBO3 + (j & 1) * 64;
                    const uint32_t r1 = j == 0 ? r3c0 : r3p[j & 1] - (j >> 1) * C::SBO3;
                    fold4(j, va + 4 * jj, vb + 4 * jj, kv[jj], r0, r1);
                }
            }
            {  // chunk 8: sub-problem 32 beside its copy, and padding
                uint32_t va[4], vb[4];
                uint4 kv[2];
                tc::ld16x256b_x1(dcol + laneA + 64, va);
                tc::ld16x256b_x1(dcol + laneB + 64, vb);
                kv[0] = kfs[((8 * 4 + w) * 2 + 0) * 32 + lane];
                kv[1] = kfs[((8 * 4 + w) * 2 + 1) * 32 + lane];
                tc::wait_ld();
                fold4(8, va, vb, kv, r3s32, C::TRASH);
            }
        }
        tc::fence_proxy_async();
        tc::fence_before();
        if (tc::bar_vote(bar_id, 256, bad)) { failed = true; break; }
        mma_pending = false;
        mmapar ^= 1;
        if (kf_pending) {
            kfpar ^= 1;
            kf_pending = false;
        }
        const bool next_kf = has_next && chan(it + 1) != h;
        if (tg == 0) {
            tc::fence_after();
            #pragma unroll
            for (int s = 0; s < 8; ++s)
                tc::mma(tD, tmem + 64 + 8 * s, tc::sdesc(bsm + 2 * s * C::LBO3, C::LBO3, C::SBO3), id3, s > 0);
            tc::commit(&bars[1]);
            if (next_kf) issue_kf(chan(it + 1));  // the k_f buffer is free: next channel's
        }
        mma_pending = true;
        kf_pending = next_kf;

        // ---------------- S3 post: twiddle, -> B4
        bad = !mbar_wait_sleep(&bars[1], mmapar, kWaitSleepLimit, kWaitHintNs);
        bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the collective TMEM loads
        tc::fence_after();
        if (!bad) {
            uint32_t vr[2][2][16];  // [row][block]: row 1's loads fly while row 0 is processed
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
                    uint8_t* dst = bbuf + row4[b] + 8 * R * C::SBO4 + kq4;
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float4 x = cmul2_twiddle(__uint_as_float(vv[4 * jj]), __uint_as_float(vv[4 * jj + 1]),
                                                     __uint_as_float(vv[4 * jj + 2]), __uint_as_float(vv[4 * jj + 3]),
                                                     tw[b][jj]);
                        *reinterpret_cast<uint2*>(dst + jj * C::LBO4) =
                            make_uint2(O::pack(x.x, x.z), O::pack(x.y, x.w));
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
                tc::mma(tD, tmem + 128 + 8 * s, tc::sdesc(bsm + 2 * s * C::LBO4, C::LBO4, C::SBO4), id4, s > 0);
            tc::commit(&bars[1]);
        }
        mma_pending = true;

        // ---------------- S4 post: conjugate, gate, store y (outputs n1 < 32)
        const size_t yin = 2 * size_t(64 * kapA + 32 * hf + 2 * q);  // element offset inside a row
        // outputs n = yin / 2 + 8 jj (+1) exist for n < Nu / 2
        auto kept = [&](int jj) { return 64 * kapA + 32 * hf + 8 * jj + 2 * q + 1 < (a.Nu >> 1); };
        uint2 wov[2][4];
        if (GATED) {  // w_out of this thread's outputs, read while the contraction runs
            #pragma unroll
            for (int R = 0; R < 2; ++R)
                #pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    wov[R][jj] = ((R ? okB : okA) && kept(jj))
                                     ? __ldg(reinterpret_cast<const uint2*>(
                                           a.w_out + size_t(R ? rowB : rowA) * a.Nu + yin + 16 * jj))
                                     : make_uint2(0, 0);
        }
        bad = !mbar_wait_sleep(&bars[1], mmapar, kWaitSleepLimit, kWaitHintNs);
        bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the collective TMEM loads
        tc::fence_after();
        if (!bad) {
            #pragma unroll
            for (int R = 0; R < 2; ++R) {
                uint32_t vv[16];
                tc::ld16x256b_x4(tD + laneA + 64 * R + 32 * hf, vv);
                tc::wait_ld();
                if (R ? okB : okA) {
                    uint16_t* yr = a.y + size_t(R ? rowB : rowA) * a.Nu + yin;
                    #pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        float r0 = __uint_as_float(vv[4 * jj]), r1 = __uint_as_float(vv[4 * jj + 1]);
                        float i0 = -__uint_as_float(vv[4 * jj + 2]), i1 = -__uint_as_float(vv[4 * jj + 3]);
                        if (GATED) {
                            const cpx w0 = O::unpack(wov[R][jj].x), w1 = O::unpack(wov[R][jj].y);
                            r0 *= w0.r; i0 *= w0.i; r1 *= w1.r; i1 *= w1.i;
                        }
                        if (kept(jj))
                            *reinterpret_cast<uint2*>(yr + 16 * jj) = make_uint2(O::pack(r0, i0), O::pack(r1, i1));
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
        if (mma_pending) mbar_wait_bounded(&bars[1], mmapar, kWaitLimit);
        if (kf_pending) mbar_wait_bounded(&bars[0], kfpar, kWaitLimit);
        if (in_pending) mbar_wait_bounded(&bars[2], inpar, kWaitLimit);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (threadIdx.x < 32) tc::dealloc(tmem, C::TMEM_COLS);
}

}  // namespace fftconv
