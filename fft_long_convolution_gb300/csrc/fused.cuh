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
    static constexpr int RP = R1 >= 16 ? 1 : 16 / R1;  // rows per row group
    static constexpr int HALF = R1 / 2;           // nonzero outer inputs
    static constexpr int UNITS = RP * (R1 / 2);   // sub-problem pairs per row group
    static constexpr int NTILES = RP * 32;        // 8-vector tiles of the outer stage
    static constexpr int NWARPS = 8;              // warps per row pipeline
    static constexpr int SEG = 264;               // staged segment: 256 words + 8 pad
    static constexpr bool K8F = R1 <= 8;          // forward outer uses K = 8
    static constexpr int KS_F = K8F ? 1 : R1 / 16;
    static constexpr int MT_F = (R1 + 7) / 8;
    static constexpr bool K8I = R1 <= 4;          // inverse outer uses K = 8
    static constexpr int KS_I = K8I ? 1 : R1 / 8;
    static constexpr int MT_I = (R1 + 15) / 16;
    // Short rows: one CTA per SM runs two independent 8-warp row pipelines that
    // share one copy of the tables, and each pipeline keeps the k_f of its
    // current channel(s) in shared memory (loaded by the TMA engine only when
    // the channel changes).  Long rows: two pipelines per CTA when their row
    // buffers fit beside the outer DFT fragments (which are then resident; the
    // outer twiddles and k_f are read through L2), else 8-warp CTAs.
    static constexpr bool TSMEM = R1 <= 16;       // all outer tables resident in shared memory
    static constexpr int NSPEC = RP > 1 ? NWARPS : 1;  // warps that own a self-paired sub-problem 0
    static constexpr size_t FRAG_BYTES = size_t(MT_F) * KS_F * 512 + size_t(MT_I) * KS_I * 512;
    static constexpr size_t ROW_BYTES = size_t(RP) * M * 4;
    static constexpr size_t SEG_BYTES = size_t(RP) * HALF * SEG * 4;
    static constexpr size_t IN_BYTES = SEG_BYTES * (GATED ? 2 : 1);
    static constexpr size_t WO_BYTES = GATED ? SEG_BYTES : 0;
    static constexpr size_t SCR_BYTES = size_t(NSPEC) * 256 * 8;
    static constexpr bool KFS = R1 <= 16;
    static constexpr size_t KF_BYTES = KFS ? size_t(RP) * R1 * 2048 : 0;
    static constexpr size_t GROUP_BYTES = ROW_BYTES + IN_BYTES + WO_BYTES + SCR_BYTES + KF_BYTES;
    static constexpr bool PAIR_FITS = 2 * GROUP_BYTES + FRAG_BYTES + 64 <= 227 * 1024;
    static constexpr int GROUPS = (R1 <= 16 || PAIR_FITS) ? 2 : 1;
    static constexpr bool FSMEM = TSMEM || GROUPS == 2;  // outer DFT fragments resident
    static constexpr int THREADS = 256 * GROUPS;
    static constexpr int MINB = GROUPS == 2 ? 1 : 2;
    // shared-memory layout (bytes)
    static constexpr size_t TAB_BYTES = TSMEM ? (FRAG_BYTES + size_t(MT_F) * 16384 + size_t(R1) * 2048 + 4 * 256)
                                              : (FSMEM ? FRAG_BYTES + 256 : 0);
    static constexpr size_t G_ROW = 0;
    static constexpr size_t G_IN = G_ROW + ROW_BYTES;
    static constexpr size_t G_WO = G_IN + IN_BYTES;
    static constexpr size_t G_SCR = G_WO + WO_BYTES;
    static constexpr size_t G_KF = G_SCR + SCR_BYTES;
    static_assert(GROUP_BYTES == G_KF + KF_BYTES, "group layout");
    static constexpr size_t OFF_BAR = TAB_BYTES + GROUPS * GROUP_BYTES;
    static constexpr size_t SMEM_BYTES = OFF_BAR + 64;
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
    float4 tw[2][2];       // [m][c]: (wr e=0, wr e=1, wi e=0, wi e=1)

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
            tw[q >> 1][q & 1] = tb.tw[lane * 4 + q];  // (m, c) = (q>>1, q&1)
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
            const float4 x0 = cmul2_split(d[0][s][0], d[0][s][1], d[0][s][2], d[0][s][3], tw[0][s]);
            const float4 x1 = cmul2_split(d[1][s][0], d[1][s][1], d[1][s][2], d[1][s][3], tw[1][s]);
            a[s][0] = O::pack(x0.x, x0.z);
            a[s][1] = O::pack(x1.x, x1.z);
            a[s][2] = O::pack(x0.y, x0.w);
            a[s][3] = O::pack(x1.y, x1.w);
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

    // Two independent sub-problems at once (instruction-level parallelism:
    // both left products, then both twiddles, then both right products).
    // p0[side] / p1[side] as the b0 / b1 of forward_at.
    __device__ __forceinline__ void forward2(const uint32_t* const (&p0)[2], const uint32_t* const (&p1)[2],
                                             cpx (&za)[8], cpx (&zb)[8]) const {
        uint32_t b[2][2][2][2];  // [side][s][c][reg]
        #pragma unroll
        for (int sd = 0; sd < 2; ++sd)
            #pragma unroll
            for (int s = 0; s < 2; ++s) {
                b[sd][s][0][0] = p0[sd][128 * s];
                b[sd][s][0][1] = p0[sd][128 * s + 64];
                b[sd][s][1][0] = p1[sd][128 * s];
                b[sd][s][1][1] = p1[sd][128 * s + 64];
            }
        float d[2][2][2][4];  // [side][m][c]
        #pragma unroll
        for (int sd = 0; sd < 2; ++sd)
            #pragma unroll
            for (int m = 0; m < 2; ++m)
                #pragma unroll
                for (int c = 0; c < 2; ++c) {
                    d[sd][m][c][0] = d[sd][m][c][1] = d[sd][m][c][2] = d[sd][m][c][3] = 0.f;
                    #pragma unroll
                    for (int s = 0; s < 2; ++s) O::mma16(d[sd][m][c], lf[m][s], b[sd][s][c][0], b[sd][s][c][1]);
                }
        right_product2(d, za, zb);
    }

    __device__ __forceinline__ void right_product2(const float (&d)[2][2][2][4], cpx (&oa)[8], cpx (&ob)[8]) const {
        uint32_t a[2][2][4];  // [side][s]
        #pragma unroll
        for (int sd = 0; sd < 2; ++sd)
            #pragma unroll
            for (int s = 0; s < 2; ++s) {
                const float4 x0 = cmul2_split(d[sd][0][s][0], d[sd][0][s][1], d[sd][0][s][2], d[sd][0][s][3], tw[0][s]);
                const float4 x1 = cmul2_split(d[sd][1][s][0], d[sd][1][s][1], d[sd][1][s][2], d[sd][1][s][3], tw[1][s]);
                a[sd][s][0] = O::pack(x0.x, x0.z);
                a[sd][s][1] = O::pack(x1.x, x1.z);
                a[sd][s][2] = O::pack(x0.y, x0.w);
                a[sd][s][3] = O::pack(x1.y, x1.w);
            }
        #pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            float ea[4] = {0.f, 0.f, 0.f, 0.f}, eb[4] = {0.f, 0.f, 0.f, 0.f};
            #pragma unroll
            for (int s = 0; s < 2; ++s) {
                O::mma16(ea, a[0][s], rf[s][nt][0], rf[s][nt][1]);
                O::mma16(eb, a[1][s], rf[s][nt][0], rf[s][nt][1]);
            }
            oa[nt] = {ea[0], ea[1]};
            oa[4 + nt] = {ea[2], ea[3]};
            ob[nt] = {eb[0], eb[1]};
            ob[4 + nt] = {eb[2], eb[3]};
        }
    }

    __device__ __forceinline__ void inverse2(const cpx (&ca)[8], const cpx (&cb)[8], cpx (&wa)[8], cpx (&wb)[8]) const {
        uint32_t p[2][8];
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            p[0][i] = O::pack(ca[i].r, ca[i].i);
            p[1][i] = O::pack(cb[i].r, cb[i].i);
        }
        float d[2][2][2][4];
        #pragma unroll
        for (int sd = 0; sd < 2; ++sd)
            #pragma unroll
            for (int m = 0; m < 2; ++m)
                #pragma unroll
                for (int n = 0; n < 2; ++n) {
                    d[sd][m][n][0] = d[sd][m][n][1] = d[sd][m][n][2] = d[sd][m][n][3] = 0.f;
                    #pragma unroll
                    for (int s = 0; s < 2; ++s)
                        O::mma16(d[sd][m][n], lf[m][s], p[sd][n * 4 + 2 * s], p[sd][n * 4 + 2 * s + 1]);
                }
        right_product2(d, wa, wb);
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

// Persistent fused kernel.  Each row pipeline (8 warps) walks a contiguous
// range of row groups taken channel-major (row index h*B + b), so consecutive
// rows share k_f[h].  The next group's input and the current w_out are
// fetched by the TMA engine while the inner stages run.
template <int DT, int R1, bool GATED>
__global__ void __launch_bounds__(FusedCfg<R1, GATED>::THREADS, FusedCfg<R1, GATED>::MINB)
fused_conv_kernel(const FusedArgs a) {
    using C = FusedCfg<R1, GATED>;
    using O = Op<DT>;
    constexpr int M = C::M, N = C::N, RP = C::RP, HALF = C::HALF, SEG = C::SEG;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_fail[2];
    __shared__ long s_kfh[2][4];  // channel held by each k_f slot
    __shared__ int s_kfwait[2];   // 1 when the group's k_f barrier has a phase in flight
    __shared__ uint32_t s_kfpar[2];
    __shared__ int s_row[2][4];   // row index b*H + h of each row of the current group (-1: none)
    __shared__ int s_ch[2][4];    // its channel h

    const int gi = C::GROUPS > 1 ? int(threadIdx.x >> 8) : 0;
    const int tg = threadIdx.x & 255;
    const int lane = tg & 31, warp = tg >> 5;
    const int g = lane >> 2, t = lane & 3;
    uint8_t* gb = smem + C::TAB_BYTES + gi * C::GROUP_BYTES;
    uint32_t* rowbuf = reinterpret_cast<uint32_t*>(gb + C::G_ROW);   // [RP][M]
    uint32_t* stage_u = reinterpret_cast<uint32_t*>(gb + C::G_IN);   // [RP][HALF][SEG]
    uint32_t* stage_w = stage_u + RP * HALF * SEG;                   // gated: w_in
    uint32_t* wobuf = reinterpret_cast<uint32_t*>(gb + C::G_WO);     // gated: w_out
    cpx* scratch = reinterpret_cast<cpx*>(gb + C::G_SCR);
    uint4* kfbuf = reinterpret_cast<uint4*>(gb + C::G_KF);            // [RP][R1][4][32]
    uint64_t* bar_tab = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* bars = bar_tab + 1 + 3 * gi;                           // in, wo, kf

    const FusedTables& tb = a.tb;
    const uint4* of_t = reinterpret_cast<const uint4*>(C::FSMEM ? smem : tb.outer);
    const uint4* oi_t = reinterpret_cast<const uint4*>((C::FSMEM ? smem : tb.outer) + tb.off_oi);
    const float4* twf_t = reinterpret_cast<const float4*>((C::TSMEM ? smem : tb.outer) + tb.off_twf);
    const float4* twi_t = reinterpret_cast<const float4*>((C::TSMEM ? smem : tb.outer) + tb.off_twi);

    // Row bookkeeping in 32-bit: the host guarantees B*H < 2^30.
    const int rows = a.B * a.H;
    const int G = (rows + RP - 1) / RP;
    const int V = int(gridDim.x) * C::GROUPS, v = int(blockIdx.x) * C::GROUPS + gi;
    const int g0 = int(int64_t(v) * G / V), g1 = int(int64_t(v + 1) * G / V);

    auto gsync = [&]() {
        if (C::GROUPS == 1) __syncthreads();
        else asm volatile("bar.sync %0, 256;" ::"r"(1 + gi) : "memory");
    };
    auto row_of = [&](int idx) -> int {  // channel-major index -> row b*H + h
        const int h = int(unsigned(idx) / unsigned(a.B)), b = idx - h * a.B;
        return b * a.H + h;
    };
    // Bulk copies of a row group, issued by the lanes of warp 0 together: lane
    // 0 arms the barrier with the byte count, lane l issues copies l, l+32, ...
    auto issue_in = [&](int grp) {  // u (+ w_in)
        int nrows = 0;
        for (int j = 0; j < RP; ++j) nrows += grp * RP + j < rows;
        if (lane == 0) mbar_expect_tx(&bars[0], uint32_t(nrows) * HALF * 1024u * (GATED ? 2u : 1u));
        const int ncopy = nrows * HALF * (GATED ? 2 : 1);
        for (int c = lane; c < ncopy; c += 32) {
            const int tsel = GATED ? (c & 1) : 0, jn = GATED ? (c >> 1) : c;
            const int j = jn / HALF, n1 = jn - j * HALF;
            const size_t base = size_t(row_of(grp * RP + j)) * N + 512 * n1;
            bulk_g2s((tsel ? stage_w : stage_u) + (j * HALF + n1) * SEG, (tsel ? a.w_in : a.u) + base, 1024, &bars[0]);
        }
    };
    auto issue_wo = [&](int grp) {  // w_out
        int nrows = 0;
        for (int j = 0; j < RP; ++j) nrows += grp * RP + j < rows;
        if (lane == 0) mbar_expect_tx(&bars[1], uint32_t(nrows) * HALF * 1024u);
        for (int c = lane; c < nrows * HALF; c += 32) {
            const int j = c / HALF, n1 = c - j * HALF;
            bulk_g2s(wobuf + (j * HALF + n1) * SEG, a.w_out + size_t(row_of(grp * RP + j)) * N + 512 * n1, 1024,
                     &bars[1]);
        }
    };
    // k_f of the group's channels into the slots (one slot per row of the
    // group), skipping slots that already hold the right channel.  Warp 0.
    auto issue_kf = [&](int grp) {
        if (!C::KFS) return;
        uint32_t need = 0;
        for (int j = 0; j < RP; ++j) {
            const int idx = grp * RP + j;
            if (idx < rows && s_kfh[gi][j] != long(unsigned(idx) / unsigned(a.B))) need |= 1u << j;
        }
        __syncwarp();
        if (need) {
            if (lane == 0) mbar_expect_tx(&bars[2], uint32_t(__popc(need)) * R1 * 2048u);
            for (int j = 0; j < RP; ++j)
                if ((need >> j) & 1) {
                    const int hh = int(unsigned(grp * RP + j) / unsigned(a.B));
                    // R1 * 2 KB per channel, in 1 KB copies spread over the lanes
                    for (int c = lane; c < R1 * 2; c += 32)
                        bulk_g2s(reinterpret_cast<uint8_t*>(kfbuf) + size_t(j) * R1 * 2048 + 1024 * c,
                                 reinterpret_cast<const uint8_t*>(a.kf) + size_t(hh) * R1 * 2048 + 1024 * c, 1024,
                                 &bars[2]);
                }
            __syncwarp();
            if (lane == 0) {
                for (int j = 0; j < RP; ++j)
                    if ((need >> j) & 1) s_kfh[gi][j] = long(unsigned(grp * RP + j) / unsigned(a.B));
                s_kfwait[gi] = 1;
            }
        }
        __syncwarp();
    };
    // bounded wait by the group's first thread, broadcast of the outcome
    auto wait_grp = [&](int b, uint32_t parity) -> bool {
        if (tg == 0 && !mbar_wait_bounded(&bars[b], parity, kWaitLimit)) {
            s_fail[gi] = 1;
            atomicExch(a.err, 7);
        }
        gsync();
        if (s_fail[gi]) return false;
        mbar_wait_bounded(&bars[b], parity, 4);  // completed phase: orders the copied bytes
        return true;
    };
    // the group's k_f wait (if a load is in flight), folded into the next barrier
    auto kf_ready = [&]() {
        if (C::KFS && tg == 0 && s_kfwait[gi]) {
            if (!mbar_wait_bounded(&bars[2], s_kfpar[gi], kWaitLimit)) {
                s_fail[gi] = 1;
                atomicExch(a.err, 7);
            }
            s_kfpar[gi] ^= 1;
            s_kfwait[gi] = 0;
        }
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < 1 + 3 * C::GROUPS; ++i) mbar_init(&bar_tab[i], 1);
        fence_mbar_init();
    }
    if (tg == 0) {
        s_fail[gi] = 0;
        s_kfwait[gi] = 0;
        s_kfpar[gi] = 0;
        for (int j = 0; j < 4; ++j) s_kfh[gi][j] = -1;
    }
    __syncthreads();
    if (threadIdx.x == 0 && C::FSMEM) {  // resident tables: all (short rows) or the DFT fragments
        const uint32_t nb = C::TSMEM ? tb.outer_bytes : tb.off_twf;
        mbar_expect_tx(bar_tab, nb);
        bulk_g2s(smem, tb.outer, nb, bar_tab);
    }
    if (warp == 0 && g0 < g1) {
        issue_in(g0);
        issue_kf(g0);
    }
    Inner<DT> in;
    in.load(tb, lane);
    if (C::FSMEM) {  // every thread of the CTA reaches this barrier
        if (threadIdx.x == 0 && !mbar_wait_bounded(bar_tab, 0, kWaitLimit)) {
            s_fail[0] = s_fail[C::GROUPS - 1] = 1;
            atomicExch(a.err, 7);
        }
        __syncthreads();
        if (s_fail[gi]) {
            if (tg == 0) mbar_wait_bounded(&bars[0], 0, kWaitLimit);
            return;
        }
        mbar_wait_bounded(bar_tab, 0, 4);
    }
    if (g0 >= g1) return;

    // per-thread address bases (see swz): warp w owns n-tiles w + 8i
    const int xs = (warp >> 2) & 1;
    const int st_base = 256 * g + ((8 * warp + 2 * t) ^ (((g & 3) ^ xs) << 3));   // + 2048m + 64i
    const int oi_base = 256 * t + ((8 * warp + g) ^ (((t & 3) ^ xs) << 3));       // + 256(8s+4j) + 64i

    uint32_t it = 0;
    for (int grp = g0; grp < g1; ++grp, ++it) {
        const uint32_t par = it & 1;
        if (tg < RP) {  // this group's rows, once (read after the barrier below)
            const int idx = grp * RP + tg;
            const int hh = int(unsigned(idx) / unsigned(a.B));
            s_row[gi][tg] = idx < rows ? (idx - hh * a.B) * a.H + hh : -1;
            s_ch[gi][tg] = hh;
        }
        if (!wait_grp(0, par)) {
            if (tg == 0 && GATED) mbar_wait_bounded(&bars[1], par ^ 1, kWaitLimit);
            return;
        }
        const int rbase = grp * RP;

        // ---------------- outer forward stage: k1 outputs of 8 vectors per tile
        if constexpr (C::FSMEM) {
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
                        const float4 v = cmul2_split(acc[0], acc[1], acc[2], acc[3], twf_t[(nt * C::MT_F + m) * 32 + lane]);
                        *reinterpret_cast<uint2*>(rb + 2048 * m) = make_uint2(O::pack(v.x, v.z), O::pack(v.y, v.w));
                    }
                }
            }
        } else {
            // fragments through L2: each A fragment once per row (m outer),
            // the staged inputs re-read from shared memory per m
            #pragma unroll 1
            for (int m = 0; m < C::MT_F; ++m) {
                uint32_t a4s[C::KS_F][4];
                #pragma unroll
                for (int s = 0; s < C::KS_F; ++s) {
                    const uint4 af = of_t[(m * C::KS_F + s) * 32 + lane];
                    a4s[s][0] = af.x; a4s[s][1] = af.y; a4s[s][2] = af.z; a4s[s][3] = af.w;
                }
                #pragma unroll 1
                for (int ntg = warp; ntg < C::NTILES; ntg += C::NWARPS) {
                    const int j = ntg >> 5, nt = ntg & 31, i4 = (ntg >> 3) & 3;
                    if (rbase + j >= rows) continue;
                    const uint32_t* su = stage_u + j * HALF * SEG + t * SEG + 8 * nt + g;
                    const uint32_t* sw = stage_w + j * HALF * SEG + t * SEG + 8 * nt + g;
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    #pragma unroll
                    for (int s = 0; s < C::KS_F; ++s) {
                        const int na = 8 * s + t, nb = 8 * s + 4 + t;
                        uint32_t va = 0, vb = 0;
                        if (na < HALF) {
                            va = su[8 * s * SEG];
                            if (GATED) va = O::mul2(va, sw[8 * s * SEG]);
                        }
                        if (nb < HALF) {
                            vb = su[(8 * s + 4) * SEG];
                            if (GATED) vb = O::mul2(vb, sw[(8 * s + 4) * SEG]);
                        }
                        O::mma16(acc, a4s[s], va, vb);
                    }
                    if (8 * m + g < R1) {
                        uint32_t* rb = rowbuf + j * M + st_base + 64 * i4;
                        const float4 v = cmul2_split(acc[0], acc[1], acc[2], acc[3], twf_t[(nt * C::MT_F + m) * 32 + lane]);
                        *reinterpret_cast<uint2*>(rb + 2048 * m) = make_uint2(O::pack(v.x, v.z), O::pack(v.y, v.w));
                    }
                }
            }
        }
        kf_ready();
        gsync();
        if (s_fail[gi]) return;
        if (warp == 0) {  // staging is free again: fetch ahead
            if (GATED) issue_wo(grp);
            if (grp + 1 < g1) issue_in(grp + 1);
            if (!C::KFS && lane == 0 && grp + 1 < g1 &&
                unsigned(grp * RP + RP) / unsigned(a.B) != unsigned(grp * RP) / unsigned(a.B)) {
                const int hh = int(unsigned(grp * RP + RP) / unsigned(a.B));  // next channel's k_f into L2
                bulk_prefetch_l2(a.kf + size_t(hh) * R1 * 128, R1 * 2048u);
            }
        }

        // ---------------- inner stages + decimation fold, per sub-problem pair
        #pragma unroll 1
        for (int ug = C::NWARPS - 1 - warp; ug < C::UNITS; ug += C::NWARPS) {
            // (the self-paired sub-problem 0 of each row lands on a late warp,
            // away from warp 0, which issues the bulk copies)
            const int j = ug / (R1 / 2), jj = ug % (R1 / 2);
            if (rbase + j >= rows) continue;
            const int h = s_ch[gi][j];
            uint32_t* rb = rowbuf + j * M;
            const int ka = jj, kb = jj == 0 ? R1 / 2 : R1 - jj;
            cpx za[8], zb[8], pp[8];
            const uint4* kfb = C::KFS ? kfbuf + size_t(j) * R1 * 128 : a.kf + size_t(h) * R1 * 128;
            const uint4* fa = kfb + ka * 128 + lane;
            const uint4* fb = kfb + kb * 128 + lane;
            {
                const int Xa = ((ka & 3) ^ ((t >> 1) & 1)) << 3, Xb = ((kb & 3) ^ ((t >> 1) & 1)) << 3;
                const uint32_t* const p0[2] = {rb + 256 * ka + (((16 * t) ^ Xa) + g), rb + 256 * kb + (((16 * t) ^ Xb) + g)};
                const uint32_t* const p1[2] = {rb + 256 * ka + (((16 * t + 8) ^ Xa) + g),
                                               rb + 256 * kb + (((16 * t + 8) ^ Xb) + g)};
                in.forward2(p0, p1, za, zb);
            }
            // C = alpha~ conj(Z) + beta~ Z_partner  (= conj Z_y), in place.
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
            cpx wab[2][8];
            in.inverse2(za, zb, wab[0], wab[1]);
            float4 tvs[2][4];
            #pragma unroll
            for (int side = 0; side < 2; ++side)
                #pragma unroll
                for (int nt = 0; nt < 4; ++nt) tvs[side][nt] = twi_t[((side ? kb : ka) * 4 + nt) * 32 + lane];
            #pragma unroll
            for (int side = 0; side < 2; ++side) {
                const int k1 = side ? kb : ka;
                const cpx (&w)[8] = wab[side];
                const int X = ((k1 & 3) ^ ((t >> 1) & 1)) << 3;
                uint32_t* s0 = rb + 256 * k1 + (((16 * t) ^ X) + g);
                uint32_t* s1 = rb + 256 * k1 + (((16 * t + 8) ^ X) + g);
                #pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const float4 tv = tvs[side][nt];
                    const cpx v0 = cmul(w[nt], {tv.x, tv.y});
                    const cpx v1 = cmul(w[4 + nt], {tv.z, tv.w});
                    s0[64 * nt] = O::pack(v0.r, v0.i);
                    s1[64 * nt] = O::pack(v1.r, v1.i);
                }
            }
        }
        if (GATED) {
            if (!wait_grp(1, par)) {
                if (tg == 0 && grp + 1 < g1) mbar_wait_bounded(&bars[0], par ^ 1, kWaitLimit);
                return;
            }
        } else {
            gsync();
        }
        // k_f slots are free until the next inner phase: fetch the next group's
        if (warp == 0 && grp + 1 < g1) issue_kf(grp + 1);

        // ---------------- outer inverse stage (first R1/2 outputs only) and store
        if constexpr (C::FSMEM) {
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
                const size_t base = size_t(s_row[gi][j]) * N;
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
        } else {
            // fragments through L2: each A fragment once per row (m outer),
            // the row buffer re-read per m
            #pragma unroll 1
            for (int m = 0; m < C::MT_I; ++m) {
                uint32_t a4s[C::KS_I][4];
                #pragma unroll
                for (int s = 0; s < C::KS_I; ++s) {
                    const uint4 af = oi_t[(m * C::KS_I + s) * 32 + lane];
                    a4s[s][0] = af.x; a4s[s][1] = af.y; a4s[s][2] = af.z; a4s[s][3] = af.w;
                }
                #pragma unroll 1
                for (int ntg = warp; ntg < C::NTILES; ntg += C::NWARPS) {
                    const int j = ntg >> 5, nt = ntg & 31, i4 = (ntg >> 3) & 3;
                    if (rbase + j >= rows) continue;
                    const uint32_t* rb = rowbuf + j * M + oi_base + 64 * i4;
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    #pragma unroll
                    for (int s = 0; s < C::KS_I; ++s) O::mma16(acc, a4s[s], rb[256 * 8 * s], rb[256 * (8 * s + 4)]);
                    const int n1 = 8 * m + g;
                    if (n1 < HALF) {
                        const size_t base = size_t(s_row[gi][j]) * N;
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
        }
        gsync();
    }
    if (C::KFS && tg == 0 && s_kfwait[gi]) mbar_wait_bounded(&bars[2], s_kfpar[gi], kWaitLimit);
}

}  // namespace fftconv
