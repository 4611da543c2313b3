// Fused causal long convolution for N = M = R1 * 256 (1K..16K): one CTA
// keeps whole (b,h) rows on chip and runs every stage of the pipeline
// (FlashFFTConv page, section 3.2 "Big-Picture Architecture"):
//
//   load u (+ gate)  ->  outer R1-point DFT  ->  twiddle  ->  two 16-point DFTs
//   (register-chained)  ->  decimation-in-time fold with the kernel spectrum
//   ->  the same stages back  ->  causal truncation (+ gate)  ->  store y.
//
// Monarch factorization (section 3.4, "The Monarch FFT Decomposition" and
// "Higher-order decompositions"), order 3, decimation in frequency:
//   n = 256*n1 + 16*n2 + n3,   k = k1 + R1*(k2 + 16*k3)
//   a_k1[o]    = W_M^(o*k1)   * sum_{n1} z[256*n1 + o] W_R1^(n1*k1)   (o = 16*n2+n3)
//   b[k2][n3]  = W_256^(k2*n3) * sum_{n2} a[16*n2 + n3] W_16^(n2*k2)
//   Z[k2][k3]  =                 sum_{n3} b[k2][n3]    W_16^(n3*k3)
// Every contraction is scaled by 1/sqrt(points) so magnitudes stay O(|y|)
// in 16-bit storage.  The spectrum stays in this permuted order; the kernel
// spectrum k_f is stored in the same order (Algorithm 1 applies K_f^T to the
// permuted data directly).
//
// Implicit zero padding (section 3.4, "Implicit zero-padding"): z[n] = 0 for
// n >= M/2, i.e. for n1 >= R1/2, so the forward outer contraction runs over
// half of its inputs; the inverse outer contraction produces only the n1 <
// R1/2 outputs that the causal truncation keeps.
//
// Real-valued input (section 3.4, "The real-valued FFT optimization"):
// z[n] = x[2n] + i x[2n+1] is the interleaved input itself.  The split
// X[k] = E[k] + W_2M^k O[k], the pointwise product with K = rfft(k, 2N) and
// the merge back to Z_y are folded into Z_y[k] = alpha_k Z[k] +
// beta_k conj(Z[M-k]).  The inverse is computed as conj(DFT(conj Z_y)), so
// it reuses the forward DFT factors and twiddles in reverse stage order; the
// kernel spectrum is stored pre-conjugated (alpha~ = conj alpha, beta~ =
// conj beta) and the final conjugation is a sign on the odd outputs.
//
// Tensor cores: each DFT factor is a dense real-embedded complex matrix
// ([[Fr,-Fi],[Fi,Fr]] interleaved) contracted with mma.sync (16-bit operands,
// float32 accumulators).  Left products keep the DFT matrix in the A operand
// and the data in B ("broadcast over the sequence", Figure 3); the outputs of
// a left product are, register for register, the A operand of the following
// right product (the accumulator-reuse of Appendix A.2), so the two 16-point
// stages and the decimation fold never leave registers.  Shared memory is
// touched only at the outer/inner boundary.
#pragma once
#include "mma.cuh"

namespace fftconv {

// Device tables of a fused plan (built on the host in double precision).
// The four "outer" tables are one contiguous block so a CTA can copy them to
// shared memory with a single bulk copy.
struct FusedTables {
    const uint4* lf;       // [lane][4]  left-product A fragments of F16/4: (m,s) -> uint4
    const uint4* rf;       // [lane][4]  right-product B fragments of F16/4: (s,nt) pairs
    const float4* tw;      // [lane][4]  W_256^(k2*n3) for (m,c,e)
    const uint8_t* outer;  // block: of | oi | twf | twi
    uint32_t outer_bytes;  // multiple of 16
    uint32_t off_oi, off_twf, off_twi;  // byte offsets inside the block (of at 0)
    // of : [m][s][lane] uint4   outer forward A fragments of F_R1/sqrt(R1)
    // oi : [m][s][lane] uint4   outer inverse A fragments
    // twf: [nt][m][lane] float4 W_M^(o*k1) in outer-output order
    // twi: [k1][nt][lane] float4 W_M^(o*k1) in inner-output order
};

template <int R1, bool GATED>
struct FusedCfg {
    static constexpr int M = R1 * 256;            // complex length = N
    static constexpr int N = M;                   // real samples per row
    static constexpr int RP = R1 >= 16 ? 1 : 16 / R1;  // rows per CTA
    static constexpr int HALF = R1 / 2;           // nonzero outer inputs
    static constexpr int UNITS = RP * (R1 / 2);   // sub-problem pairs per row group
    static constexpr int NTILES = RP * 32;        // 8-vector tiles of the outer stage
    static constexpr int NWARPS = 8;
    static constexpr int SEG = 264;               // staged segment: 256 words + 8 pad
    static constexpr bool K8F = R1 <= 8;          // forward outer uses K = 8
    static constexpr int KS_F = K8F ? 1 : R1 / 16;
    static constexpr int MT_F = (R1 + 7) / 8;
    static constexpr bool K8I = R1 <= 4;          // inverse outer uses K = 8
    static constexpr int KS_I = K8I ? 1 : R1 / 8;
    static constexpr int MT_I = (R1 + 15) / 16;
    static constexpr bool TSMEM = R1 <= 16;       // outer tables resident in shared memory
    static constexpr int NSPEC = RP > 1 ? NWARPS : 1;  // warps that own a self-paired sub-problem 0
    // shared-memory layout (bytes)
    static constexpr size_t TAB_BYTES = TSMEM ? (size_t(MT_F) * KS_F * 512 + size_t(MT_I) * KS_I * 512 +
                                                 size_t(MT_F) * 16384 + size_t(R1) * 2048 + 4 * 256)
                                              : 0;
    static constexpr size_t ROW_BYTES = size_t(RP) * M * 4;
    static constexpr size_t SEG_BYTES = size_t(RP) * HALF * SEG * 4;
    static constexpr size_t IN_BYTES = SEG_BYTES * (GATED ? 2 : 1);
    static constexpr size_t WO_BYTES = GATED ? SEG_BYTES : 0;
    static constexpr size_t SCR_BYTES = size_t(NSPEC) * 256 * 8;
    static constexpr size_t OFF_ROW = TAB_BYTES;
    static constexpr size_t OFF_IN = OFF_ROW + ROW_BYTES;
    static constexpr size_t OFF_WO = OFF_IN + IN_BYTES;
    static constexpr size_t OFF_SCR = OFF_WO + WO_BYTES;
    static constexpr size_t OFF_BAR = OFF_SCR + SCR_BYTES;
    static constexpr size_t SMEM_BYTES = OFF_BAR + 32;
};

// Row-buffer swizzle (complex-word index): XOR bits 3-4 with bits of the
// sub-problem index and bit 5, which keeps all four access patterns of the
// kernel free of bank conflicts.  The kernel applies it through hoisted,
// per-thread bases (the XOR term is constant along each access sequence).
__device__ __forceinline__ int swz(int p) {
    return p ^ ((((p >> 8) & 3) ^ ((p >> 5) & 1)) << 3);
}

__device__ __forceinline__ cpx shfl31(cpx v) {
    return {__shfl_xor_sync(0xffffffffu, v.r, 31), __shfl_xor_sync(0xffffffffu, v.i, 31)};
}

constexpr uint32_t kWaitLimit = 1u << 22;

template <int DT>
struct Inner {
    using O = Op<DT>;
    uint32_t lf[2][2][4];  // [m][s]
    uint32_t rf[2][4][2];  // [s][nt]
    cpx tw[2][2][2];       // [m][c][e]

    __device__ __forceinline__ void load(const FusedTables& tb, int lane) {
        #pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 v = tb.lf[lane * 4 + q];
            lf[q >> 1][q & 1][0] = v.x; lf[q >> 1][q & 1][1] = v.y;
            lf[q >> 1][q & 1][2] = v.z; lf[q >> 1][q & 1][3] = v.w;
            uint4 w = tb.rf[lane * 4 + q];  // (s, nt) = (q>>1, 2*(q&1)) and +1
            const int s = q >> 1, nt = 2 * (q & 1);
            rf[s][nt][0] = w.x; rf[s][nt][1] = w.y;
            rf[s][nt + 1][0] = w.z; rf[s][nt + 1][1] = w.w;
            float4 x = tb.tw[lane * 4 + q];  // (m, c) = (q>>1, q&1), e = 0, 1
            tw[q >> 1][q & 1][0] = {x.x, x.y};
            tw[q >> 1][q & 1][1] = {x.z, x.w};
        }
    }

    // Forward 256-point sub-transform of one sub-problem held in shared
    // memory: b0 / b1 point at the words of (n2 = t, n3 = g) and (n2 = t,
    // n3 = 8 + g); the other inputs sit at +128*s + 64*j (n2 = 8s + 4j + t).
    // Result: z[m*4+nt] = Z[k2 = g+8m][k3 = 4nt+t].
    __device__ __forceinline__ void forward_at(const uint32_t* b0, const uint32_t* b1, cpx (&z)[8]) const {
        uint32_t b[2][2][2];  // [s][c][reg]
        #pragma unroll
        for (int s = 0; s < 2; ++s) {
            b[s][0][0] = b0[128 * s];
            b[s][0][1] = b0[128 * s + 64];
            b[s][1][0] = b1[128 * s];
            b[s][1][1] = b1[128 * s + 64];
        }
        float d[2][2][4];
        #pragma unroll
        for (int m = 0; m < 2; ++m)
            #pragma unroll
            for (int c = 0; c < 2; ++c) {
                d[m][c][0] = d[m][c][1] = d[m][c][2] = d[m][c][3] = 0.f;
                #pragma unroll
                for (int s = 0; s < 2; ++s) O::mma16(d[m][c], lf[m][s], b[s][c][0], b[s][c][1]);
            }
        right_product(d, z);
    }

    // Same, sub-problem k1 of a swizzled row buffer (position 256*k1 + o).
    __device__ __forceinline__ void forward(const uint32_t* rb, int k1, int g, int t, cpx (&z)[8]) const {
        const int X = ((k1 & 3) ^ ((t >> 1) & 1)) << 3;
        forward_at(rb + 256 * k1 + (((16 * t) ^ X) + g), rb + 256 * k1 + (((16 * t + 8) ^ X) + g), z);
    }

    // Twiddle the output of a left product and contract it with F16 from the
    // right: d[m][c] holds (k2 or n3 = 8m+g) x (8c+2t+e); out[m*4+nt] holds
    // row (g + 8m), column 4nt+t.
    __device__ __forceinline__ void right_product(const float (&d)[2][2][4], cpx (&out)[8]) const {
        uint32_t a[2][4];
        #pragma unroll
        for (int s = 0; s < 2; ++s) {
            cpx x00 = cmul({d[0][s][0], d[0][s][2]}, tw[0][s][0]);
            cpx x10 = cmul({d[1][s][0], d[1][s][2]}, tw[1][s][0]);
            cpx x01 = cmul({d[0][s][1], d[0][s][3]}, tw[0][s][1]);
            cpx x11 = cmul({d[1][s][1], d[1][s][3]}, tw[1][s][1]);
            a[s][0] = O::pack(x00.r, x00.i);
            a[s][1] = O::pack(x10.r, x10.i);
            a[s][2] = O::pack(x01.r, x01.i);
            a[s][3] = O::pack(x11.r, x11.i);
        }
        #pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            float e[4] = {0.f, 0.f, 0.f, 0.f};
            #pragma unroll
            for (int s = 0; s < 2; ++s) O::mma16(e, a[s], rf[s][nt][0], rf[s][nt][1]);
            out[nt] = {e[0], e[1]};
            out[4 + nt] = {e[2], e[3]};
        }
    }

    // Inverse direction on c = conj(Z_y) (same layout as forward's z):
    // returns w[m*4+nt] = transform at (n3 = g+8m, n2 = 4nt+t).
    __device__ __forceinline__ void inverse(const cpx (&c)[8], cpx (&w)[8]) const {
        uint32_t p[8];
        #pragma unroll
        for (int i = 0; i < 8; ++i) p[i] = O::pack(c[i].r, c[i].i);
        float d[2][2][4];
        #pragma unroll
        for (int m = 0; m < 2; ++m)
            #pragma unroll
            for (int n = 0; n < 2; ++n) {
                d[m][n][0] = d[m][n][1] = d[m][n][2] = d[m][n][3] = 0.f;
                #pragma unroll
                for (int s = 0; s < 2; ++s)
                    O::mma16(d[m][n], lf[m][s], p[n * 4 + 2 * s], p[n * 4 + 2 * s + 1]);
            }
        right_product(d, w);
    }
};

// One bin of the decimation-in-time fold with the kernel spectrum:
// returns alpha~ conj(z) + beta~ zp, alpha~ and beta~ packed 16-bit complex.
template <int DT>
__device__ __forceinline__ cpx dit_fold(uint32_t alpha, uint32_t beta, cpx z, cpx zp) {
    const cpx al = Op<DT>::unpack(alpha), be = Op<DT>::unpack(beta);
    return {al.r * z.r + al.i * z.i + be.r * zp.r - be.i * zp.i,
            al.i * z.r - al.r * z.i + be.r * zp.i + be.i * zp.r};
}

struct FusedArgs {
    const uint16_t* u;
    const uint16_t* w_in;
    const uint16_t* w_out;
    const uint4* kf;
    uint16_t* y;
    int B, H;
    FusedTables tb;
    int* err;
};

// Persistent fused kernel: each CTA walks a contiguous range of row groups
// taken channel-major (row index h*B + b), so consecutive rows share k_f[h].
// The next group's input is fetched by the TMA engine while the current
// group runs its inner stages; w_out (gated) is fetched during the same
// window into its own buffer.
template <int DT, int R1, bool GATED>
__global__ void __launch_bounds__(256, 2) fused_conv_kernel(const FusedArgs a) {
    using C = FusedCfg<R1, GATED>;
    using O = Op<DT>;
    constexpr int M = C::M, N = C::N, RP = C::RP, HALF = C::HALF, SEG = C::SEG;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t* rowbuf = reinterpret_cast<uint32_t*>(smem + C::OFF_ROW);   // [RP][M]
    uint32_t* stage_u = reinterpret_cast<uint32_t*>(smem + C::OFF_IN);   // [RP][HALF][SEG]
    uint32_t* stage_w = stage_u + RP * HALF * SEG;                       // gated: w_in
    uint32_t* wobuf = reinterpret_cast<uint32_t*>(smem + C::OFF_WO);     // gated: w_out
    cpx* scratch = reinterpret_cast<cpx*>(smem + C::OFF_SCR);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);     // tab, in, wo
    __shared__ int s_fail;

    const FusedTables& tb = a.tb;
    const uint4* of_t = reinterpret_cast<const uint4*>(C::TSMEM ? smem : tb.outer);
    const uint4* oi_t = reinterpret_cast<const uint4*>((C::TSMEM ? smem : tb.outer) + tb.off_oi);
    const float4* twf_t = reinterpret_cast<const float4*>((C::TSMEM ? smem : tb.outer) + tb.off_twf);
    const float4* twi_t = reinterpret_cast<const float4*>((C::TSMEM ? smem : tb.outer) + tb.off_twi);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const long rows = long(a.B) * a.H;
    const long G = (rows + RP - 1) / RP;
    const long g0 = long(blockIdx.x) * G / gridDim.x, g1 = long(blockIdx.x + 1) * G / gridDim.x;
    if (g0 >= g1) return;

    auto row_of = [&](long idx) -> long {  // channel-major index -> row b*H + h
        const long h = idx / a.B, b = idx - h * a.B;
        return b * a.H + h;
    };
    auto issue_in = [&](long grp) {  // thread 0: u (+ w_in) of a row group
        uint32_t bytes = 0;
        for (int j = 0; j < RP; ++j)
            if (grp * RP + j < rows) bytes += HALF * 1024u * (GATED ? 2u : 1u);
        mbar_expect_tx(&bars[1], bytes);
        for (int j = 0; j < RP; ++j) {
            if (grp * RP + j >= rows) break;
            const long base = row_of(grp * RP + j) * N;
            for (int n1 = 0; n1 < HALF; ++n1) {
                bulk_g2s(stage_u + (j * HALF + n1) * SEG, a.u + base + 512 * n1, 1024, &bars[1]);
                if (GATED) bulk_g2s(stage_w + (j * HALF + n1) * SEG, a.w_in + base + 512 * n1, 1024, &bars[1]);
            }
        }
    };
    auto issue_wo = [&](long grp) {  // thread 0: w_out of a row group
        uint32_t bytes = 0;
        for (int j = 0; j < RP; ++j)
            if (grp * RP + j < rows) bytes += HALF * 1024u;
        mbar_expect_tx(&bars[2], bytes);
        for (int j = 0; j < RP; ++j) {
            if (grp * RP + j >= rows) break;
            const long base = row_of(grp * RP + j) * N;
            for (int n1 = 0; n1 < HALF; ++n1)
                bulk_g2s(wobuf + (j * HALF + n1) * SEG, a.w_out + base + 512 * n1, 1024, &bars[2]);
        }
    };
    // bounded wait by thread 0, broadcast of the outcome; false = give up
    auto wait_all = [&](int b, uint32_t parity) -> bool {
        if (threadIdx.x == 0 && !mbar_wait_bounded(&bars[b], parity, kWaitLimit)) {
            s_fail = 1;
            atomicExch(a.err, 7);
        }
        __syncthreads();
        if (s_fail) return false;
        mbar_wait_bounded(&bars[b], parity, 4);  // completed phase: orders the copied bytes
        return true;
    };

    if (threadIdx.x == 0) {
        s_fail = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (C::TSMEM) {
            mbar_expect_tx(&bars[0], tb.outer_bytes);
            bulk_g2s(smem, tb.outer, tb.outer_bytes, &bars[0]);
        }
        issue_in(g0);
    }
    Inner<DT> in;
    in.load(tb, lane);
    if (C::TSMEM && !wait_all(0, 0)) {
        if (threadIdx.x == 0) mbar_wait_bounded(&bars[1], 0, kWaitLimit);
        return;
    }

    // per-thread address bases (see swz): warp w owns n-tiles w + 8i
    const int xs = (warp >> 2) & 1;
    const int st_base = 256 * g + ((8 * warp + 2 * t) ^ (((g & 3) ^ xs) << 3));   // + 2048m + 64i
    const int oi_base = 256 * t + ((8 * warp + g) ^ (((t & 3) ^ xs) << 3));       // + 256(8s+4j) + 64i

    uint32_t it = 0;
    for (long grp = g0; grp < g1; ++grp, ++it) {
        const uint32_t par = it & 1;
        if (!wait_all(1, par)) {
            if (threadIdx.x == 0 && GATED) mbar_wait_bounded(&bars[2], par ^ 1, kWaitLimit);
            return;
        }
        const long rbase = grp * RP;

        // ---------------- outer forward stage: k1 outputs of 8 vectors per tile
        #pragma unroll 1
        for (int ntg = warp; ntg < C::NTILES; ntg += C::NWARPS) {
            const int j = ntg >> 5, nt = ntg & 31, i4 = (ntg >> 3) & 3;
            if (rbase + j >= rows) continue;
            const uint32_t* su = stage_u + j * HALF * SEG + t * SEG + 8 * nt + g;
            const uint32_t* sw = stage_w + j * HALF * SEG + t * SEG + 8 * nt + g;
            uint32_t bf[C::KS_F][2];
            #pragma unroll
            for (int s = 0; s < C::KS_F; ++s) {
                const int na = 8 * s + t, nb = 8 * s + 4 + t;
                uint32_t va = 0, vb = 0;
                if (na < HALF) {
                    va = su[8 * s * SEG];
                    if (GATED) va = O::mul2(va, sw[8 * s * SEG]);
                }
                if (!C::K8F && nb < HALF) {
                    vb = su[(8 * s + 4) * SEG];
                    if (GATED) vb = O::mul2(vb, sw[(8 * s + 4) * SEG]);
                }
                bf[s][0] = va;
                bf[s][1] = vb;
            }
            uint32_t* rb = rowbuf + j * M + st_base + 64 * i4;
            #pragma unroll
            for (int m = 0; m < C::MT_F; ++m) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                if (C::K8F) {
                    const uint4 af = of_t[m * 32 + lane];
                    O::mma8(acc, af.x, af.y, bf[0][0]);
                } else {
                    #pragma unroll
                    for (int s = 0; s < C::KS_F; ++s) {
                        const uint4 af = of_t[(m * C::KS_F + s) * 32 + lane];
                        const uint32_t a4[4] = {af.x, af.y, af.z, af.w};
                        O::mma16(acc, a4, bf[s][0], bf[s][1]);
                    }
                }
                if (8 * m + g < R1) {
                    const float4 w = twf_t[(nt * C::MT_F + m) * 32 + lane];
                    const cpx v0 = cmul({acc[0], acc[2]}, {w.x, w.y});
                    const cpx v1 = cmul({acc[1], acc[3]}, {w.z, w.w});
                    *reinterpret_cast<uint2*>(rb + 2048 * m) = make_uint2(O::pack(v0.r, v0.i), O::pack(v1.r, v1.i));
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {  // staging is free again: fetch ahead
            if (GATED) issue_wo(grp);
            if (grp + 1 < g1) issue_in(grp + 1);
        }

        // ---------------- inner stages + decimation fold, per sub-problem pair
        #pragma unroll 1
        for (int ug = warp; ug < C::UNITS; ug += C::NWARPS) {
            const int j = ug / (R1 / 2), jj = ug % (R1 / 2);
            if (rbase + j >= rows) continue;
            const long h = (rbase + j) / a.B;
            uint32_t* rb = rowbuf + j * M;
            const int ka = jj, kb = jj == 0 ? R1 / 2 : R1 - jj;
            cpx za[8], zb[8], pp[8];
            in.forward(rb, ka, g, t, za);
            in.forward(rb, kb, g, t, zb);
            // C = alpha~ conj(Z) + beta~ Z_partner  (= conj Z_y), in place.
            const uint4* fa = a.kf + (size_t(h * R1 + ka) * 4) * 32 + lane;
            const uint4* fb = a.kf + (size_t(h * R1 + kb) * 4) * 32 + lane;
            if (jj != 0) {
                // bins of sub-problem ka pair with sub-problem kb through lane ^ 31
                #pragma unroll
                for (int i = 0; i < 8; ++i) pp[i] = shfl31(za[7 - i]);  // partners of zb
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = fa[q * 32];
                    #pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        const int i = 2 * q + sl;
                        za[i] = dit_fold<DT>(sl ? v.z : v.x, sl ? v.w : v.y, za[i], shfl31(zb[7 - i]));
                    }
                }
            } else {
                // sub-problem R1/2 pairs with itself through lane ^ 31; sub-problem 0
                // pairs bin kappa with (256 - kappa) mod 256 of itself
                #pragma unroll
                for (int i = 0; i < 8; ++i) pp[i] = shfl31(zb[7 - i]);
                cpx* sc = scratch + (RP > 1 ? warp : 0) * 256;
                #pragma unroll
                for (int i = 0; i < 8; ++i) sc[(g + 8 * (i >> 2)) + 16 * (4 * (i & 3) + t)] = za[i];
                __syncwarp();
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = fa[q * 32];
                    #pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        const int i = 2 * q + sl;
                        const int kap = (g + 8 * (i >> 2)) + 16 * (4 * (i & 3) + t);
                        za[i] = dit_fold<DT>(sl ? v.z : v.x, sl ? v.w : v.y, za[i], sc[(256 - kap) & 255]);
                    }
                }
                __syncwarp();
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
            // inverse inner stages, then the outer twiddle, back to the row buffer
            #pragma unroll
            for (int side = 0; side < 2; ++side) {
                const int k1 = side ? kb : ka;
                cpx w[8];
                in.inverse(side ? zb : za, w);
                const int X = ((k1 & 3) ^ ((t >> 1) & 1)) << 3;
                uint32_t* s0 = rb + 256 * k1 + (((16 * t) ^ X) + g);
                uint32_t* s1 = rb + 256 * k1 + (((16 * t + 8) ^ X) + g);
                #pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const float4 tv = twi_t[(k1 * 4 + nt) * 32 + lane];
                    const cpx v0 = cmul(w[nt], {tv.x, tv.y});
                    const cpx v1 = cmul(w[4 + nt], {tv.z, tv.w});
                    s0[64 * nt] = O::pack(v0.r, v0.i);
                    s1[64 * nt] = O::pack(v1.r, v1.i);
                }
            }
        }
        if (GATED) {
            if (!wait_all(2, par)) {
                if (threadIdx.x == 0 && grp + 1 < g1) mbar_wait_bounded(&bars[1], par ^ 1, kWaitLimit);
                return;
            }
        } else {
            __syncthreads();
        }

        // ---------------- outer inverse stage (first R1/2 outputs only) and store
        #pragma unroll 1
        for (int ntg = warp; ntg < C::NTILES; ntg += C::NWARPS) {
            const int j = ntg >> 5, nt = ntg & 31, i4 = (ntg >> 3) & 3;
            if (rbase + j >= rows) continue;
            const uint32_t* rb = rowbuf + j * M + oi_base + 64 * i4;
            uint32_t bf[C::KS_I][2];
            #pragma unroll
            for (int s = 0; s < C::KS_I; ++s) {
                bf[s][0] = rb[256 * 8 * s];
                bf[s][1] = C::K8I ? 0u : rb[256 * (8 * s + 4)];
            }
            const long base = row_of(rbase + j) * N;
            #pragma unroll
            for (int m = 0; m < C::MT_I; ++m) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                if (C::K8I) {
                    const uint4 af = oi_t[m * 32 + lane];
                    O::mma8(acc, af.x, af.y, bf[0][0]);
                } else {
                    #pragma unroll
                    for (int s = 0; s < C::KS_I; ++s) {
                        const uint4 af = oi_t[(m * C::KS_I + s) * 32 + lane];
                        const uint32_t a4[4] = {af.x, af.y, af.z, af.w};
                        O::mma16(acc, a4, bf[s][0], bf[s][1]);
                    }
                }
                const int n1 = 8 * m + g;
                if (n1 < HALF) {
                    const int p = 256 * n1 + 8 * nt + 2 * t;  // complex index; reals 2p..2p+3
                    float r0 = acc[0], i0 = -acc[2], r1 = acc[1], i1 = -acc[3];
                    if (GATED) {
                        const uint2 wv = *reinterpret_cast<const uint2*>(wobuf + (j * HALF + n1) * SEG + 8 * nt + 2 * t);
                        const cpx w0 = O::unpack(wv.x), w1 = O::unpack(wv.y);
                        r0 *= w0.r; i0 *= w0.i; r1 *= w1.r; i1 *= w1.i;
                    }
                    *reinterpret_cast<uint2*>(a.y + base + 2 * p) = make_uint2(O::pack(r0, i0), O::pack(r1, i1));
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace fftconv
