// Kernel gradient dk for 2N = L in 16384 .. 65536: the batch sum of the
// cross spectra G_b conj X_b of each channel, in float32 (FlashFFTConv page,
// section 3.4, "Kernel Fusion and Recomputation Strategies": the backward
// recomputes the transforms instead of storing them).
//
// For a row, z[n] = g[n] + i x[n] (g = dy (* w_out), x = u (* w_in), zero for
// n >= N) and its L-point spectrum Z; G[f] = (Z[f] + conj Z[-f]) / 2 and
// X[f] = (Z[f] - conj Z[-f]) / (2i) are the spectra of the real rows g and x.
// The L-point transform is split as L = L1 x L2, L2 = 2048 (four-step):
//   n = L2 n1 + n2, f = k1 + L1 k2
//   Z[k1 + L1 k2] = sum_n2 W_L2^(n2 k2) W_L^(n2 k1) sum_{n1 < L1/2} z[L2 n1 + n2] W_L1^(n1 k1)
// (n1 < L1/2 only: the upper half of z is zero).
// dk_rows: one CTA per channel h and pair of sub-rows (k1, L1 - k1) (pair 0:
//   the self-paired sub-rows 0 and L1/2).  For every batch row: the two
//   sub-rows' column sums and twiddles, straight from u and dy; their
//   L2-point transforms in shared memory; S[f] += G[f] conj X[f] on the
//   pair's bins (the partner bin -f of f = k1 + L1 k2 lies in sub-row
//   L1 - k1 at L2 - 1 - k2 for k1 > 0, in sub-row 0 at L2 - k2 for k1 = 0).
//   Then the inverse's first step on the pair: the L2-point transform of
//   conj S along k2 and the twiddle W_L^(k1 n2) -> R[h][k1][n2].
// dk_cols_inv: dk[h][n2 + L2 n1] = Re(sum_k1 R[h][k1][n2] W_L1^(k1 n1)) / L for
//   the outputs n < N (n1 < L1/2), i.e. Re(IDFT_L(S)) on the kept half.
#pragma once
#include "mma.cuh"

namespace fftconv {

constexpr int kDkRowThreads = 512, kDkL2 = 2048;

// W_n^e = exp(-2 pi i e / n) for a power of two n, e reduced mod n (exact angle).
__device__ __forceinline__ float2 dk_twiddle(uint32_t e, uint32_t n) {
    float s, c;
    sincospif(-2.f * float(e & (n - 1)) / float(n), &s, &c);
    return make_float2(c, s);
}

__device__ __forceinline__ float2 dk_cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

// Twiddles of the radix-4 passes of the 2048-point transforms: W_4Ns^kk for
// kk < Ns, pass p (Ns = 2 * 4^p) at offset 2 (4^p - 1) / 3, i.e. 0, 2, 10,
// 42, 170.
constexpr int kDkTwEntries = 2 + 8 + 32 + 128 + 512;
__device__ __forceinline__ int dk_tw_off(int p) { return (2 * ((1 << (2 * p)) - 1)) / 3; }

// The two sub-rows of a pair travel together: entry n of a transform buffer
// is one float4 (Re A, Re B, Im A, Im B), so every butterfly and twiddle of
// the transform works on both sub-rows with packed f32x2 arithmetic.
struct DkPair {
    unsigned long long re, im;  // (A, B) real parts, (A, B) imaginary parts
};

__device__ __forceinline__ unsigned long long dk_pk(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 dk_upk(unsigned long long r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ unsigned long long dk_add2(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long dk_sub2(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long dk_mul2(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long dk_fma2(unsigned long long a, unsigned long long b,
                                                      unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ DkPair dk_ld(const float4* p) {
    const float4 v = *p;
    return {dk_pk(v.x, v.y), dk_pk(v.z, v.w)};
}
__device__ __forceinline__ void dk_st(float4* p, DkPair v) {
    const float2 r = dk_upk(v.re), i = dk_upk(v.im);
    *p = make_float4(r.x, r.y, i.x, i.y);
}
__device__ __forceinline__ DkPair dk_padd(DkPair a, DkPair b) { return {dk_add2(a.re, b.re), dk_add2(a.im, b.im)}; }
__device__ __forceinline__ DkPair dk_psub(DkPair a, DkPair b) { return {dk_sub2(a.re, b.re), dk_sub2(a.im, b.im)}; }
// both sub-rows times the same twiddle c + i s
__device__ __forceinline__ DkPair dk_pmul(DkPair v, float c, float s) {
    const unsigned long long C = dk_pk(c, c), S = dk_pk(s, s), Sn = dk_pk(-s, -s);
    return {dk_fma2(v.im, Sn, dk_mul2(v.re, C)), dk_fma2(v.re, S, dk_mul2(v.im, C))};
}

// Entry e of a transform buffer sits at slot e ^ ((e >> 2) & 7) (a bijection
// within each block of 32 entries): the strided stores of the first passes
// then spread over the banks (about 7 % above conflict-free over one row,
// against 43 % without it, counted per quarter-warp of 16-byte accesses).
__device__ __forceinline__ int dk_sw(int e) { return e ^ ((e >> 2) & 7); }

// The radix-4 passes (span Ns = 2, 8, 32, 128, 512) of two 2048-point DFTs
// (exponent sign -1, Stockham, self-sorting) whose radix-2 pass has been
// done into b: b -> a -> b -> a -> b -> a, the result in a.  512 threads:
// thread t runs butterfly t with the twiddle W_4Ns^(t mod Ns) of the table.
__device__ __forceinline__ void dk_fft_r4(float4* a, float4* b, const float2* tw) {
    constexpr int Q = kDkL2 / 4;
    const int t = threadIdx.x;
    #pragma unroll
    for (int p = 0; p < 5; ++p) {
        const int lgNs = 1 + 2 * p, Ns = 1 << lgNs;
        const float4* x = (p & 1) ? a : b;
        float4* y0 = (p & 1) ? b : a;
        const int kk = t & (Ns - 1), jj = t >> lgNs;
        const float2 w1 = tw[dk_tw_off(p) + kk];
        const float c1 = w1.x, s1 = w1.y;
        const float c2 = c1 * c1 - s1 * s1, s2 = 2.f * c1 * s1;
        const float c3 = c2 * c1 - s2 * s1, s3 = c2 * s1 + s2 * c1;
        const DkPair v0 = dk_ld(x + dk_sw(t));
        const DkPair v1 = dk_pmul(dk_ld(x + dk_sw(t + Q)), c1, s1);
        const DkPair v2 = dk_pmul(dk_ld(x + dk_sw(t + 2 * Q)), c2, s2);
        const DkPair v3 = dk_pmul(dk_ld(x + dk_sw(t + 3 * Q)), c3, s3);
        const DkPair a0 = dk_padd(v0, v2), a1 = dk_psub(v0, v2), a2 = dk_padd(v1, v3);
        const DkPair a3 = {dk_sub2(v1.im, v3.im), dk_sub2(v3.re, v1.re)};  // -i (v1 - v3)
        const int o = kk + (jj << (lgNs + 2));
        dk_st(y0 + dk_sw(o), dk_padd(a0, a2));
        dk_st(y0 + dk_sw(o + Ns), dk_padd(a1, a3));
        dk_st(y0 + dk_sw(o + 2 * Ns), dk_psub(a0, a2));
        dk_st(y0 + dk_sw(o + 3 * Ns), dk_psub(a1, a3));
        __syncthreads();
    }
}

// G[f] conj X[f] from Z[f] = (ar, ai) and Z[-f] = (cr, ci)
__device__ __forceinline__ float2 dk_cross(float ar, float ai, float cr, float ci) {
    const float gr = 0.5f * (ar + cr), gi = 0.5f * (ai - ci);   // G = (Z[f] + conj Z[-f]) / 2
    const float xr = 0.5f * (ai + ci), xi = -0.5f * (ar - cr);  // X = (Z[f] - conj Z[-f]) / (2i)
    return make_float2(gr * xr + gi * xi, gi * xr - gr * xi);
}

// One CTA per (channel h, pair of sub-rows p), looping over the batch.  The
// CTAs of a channel run side by side (items are numbered channel-major), so
// each row of u and dy comes from DRAM about once and from L2 L1/2 times.
// Thread t computes the column sums of columns 2t, 2t + 1, 2t + 1024 and
// 2t + 1025 (4-byte loads of two 16-bit inputs, a few rows n1 in flight at
// once), which are the inputs of the transform's radix-2 butterflies 2t and
// 2t + 1: that pass runs in registers.  It owns bins t + 512 e of the batch
// sum.  Shared memory: two transform buffers of 2048 float4, the batch sum S
// of both sub-rows and the radix-4 twiddles (101.5 KB, two CTAs per SM).
//
// FA (2N = 128K .. 1M): the column transforms come precomputed and twiddled
// from dk_colfft_fwd in A[row][k1][n2] (float32), so the CTA loads its two
// sub-rows instead of forming column sums (u, dy and the gates are unused).
template <int DT, int L1, bool G, bool FA = false>
__global__ void __launch_bounds__(kDkRowThreads, 2) dk_rows(const uint16_t* __restrict__ u,
                                                            const uint16_t* __restrict__ dy,
                                                            const uint16_t* __restrict__ w_in,
                                                            const uint16_t* __restrict__ w_out,
                                                            float2* __restrict__ R, int64_t B, int64_t H,
                                                            const float2* __restrict__ A) {
    using O = Op<DT>;
    constexpr int L2 = kDkL2, T = kDkRowThreads, NE = L2 / T;  // 4 bins per thread per sub-row
    constexpr int NH = L1 / 2, CH = G ? 2 : 4;                 // input rows n1; rows loaded per round
    static_assert(NE == 4 && (FA || NH % CH == 0), "2048-point sub-rows, 512 threads");
    constexpr int64_t N = int64_t(L2) * NH;
    constexpr uint32_t L = uint32_t(L1) * uint32_t(L2);
    extern __shared__ __align__(16) float4 dsm4[];
    float4* bufA = dsm4;
    float4* bufB = dsm4 + L2;
    float2* acc = reinterpret_cast<float2*>(dsm4 + 2 * L2);  // S[sub-row][k2]
    float2* ftw = acc + 2 * L2;                              // radix-4 twiddles
    const int t = threadIdx.x;
    for (int i = t; i < kDkTwEntries; i += T) {
        int p = 0;
        while (p < 4 && i >= dk_tw_off(p + 1)) ++p;
        const int Ns = 2 << (2 * p), kk = i - dk_tw_off(p);
        float s1, c1;
        sincospif(-float(kk) / float(2 * Ns), &s1, &c1);
        ftw[i] = make_float2(c1, s1);
    }
    __syncthreads();
    const int64_t items = H * NH;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t h = it / NH;
        const int p = int(it - h * NH);
        const int kA = p, kB = p ? L1 - p : NH;
        // W_L^(n2 k1) of this thread's columns n2 = 2t + 1024 gc + c, both sub-rows
        // (FA: already applied to A)
        float2 ctw[4][2];
        #pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t n2 = uint32_t(2 * t + 1024 * (c >> 1) + (c & 1));
            ctw[c][0] = FA ? make_float2(1.f, 0.f) : dk_twiddle(n2 * uint32_t(kA), L);
            ctw[c][1] = FA ? make_float2(1.f, 0.f) : dk_twiddle(n2 * uint32_t(kB), L);
        }
        const float2 wst = dk_twiddle(uint32_t(kA), uint32_t(L1));  // W_L1^kA
        #pragma unroll
        for (int e = 0; e < 2 * NE; ++e) acc[t + T * e] = make_float2(0.f, 0.f);
        for (int64_t b = 0; b < B; ++b) {
          float2 sa[4], sb[4];  // column c = 2 gc + e of this thread, sub-rows A and B
          if constexpr (FA) {
            const float2* ra = A + ((b * H + h) * L1 + kA) * int64_t(L2) + 2 * t;
            const float2* rb = A + ((b * H + h) * L1 + kB) * int64_t(L2) + 2 * t;
            #pragma unroll
            for (int gc = 0; gc < 2; ++gc) {
                const float4 va = __ldg(reinterpret_cast<const float4*>(ra + 1024 * gc));
                const float4 vb = __ldg(reinterpret_cast<const float4*>(rb + 1024 * gc));
                sa[2 * gc] = make_float2(va.x, va.y);
                sa[2 * gc + 1] = make_float2(va.z, va.w);
                sb[2 * gc] = make_float2(vb.x, vb.y);
                sb[2 * gc + 1] = make_float2(vb.z, vb.w);
            }
          } else {
            const int64_t roff = (b * H + h) * N + 2 * t;
            // A_k1[n2] = W_L^(n2 k1) sum_{n1 < L1/2} z[L2 n1 + n2] W_L1^(n1 k1), with
            // W_L1^(n1 kB) = conj W_L1^(n1 kA) (kB = L1 - kA) or, on pair 0,
            // W_L1^0 = 1 and W_L1^(n1 L1/2) = (-1)^n1
            // accumulators as f32x2 pairs over the columns (2t, 2t + 1) of group gc
            unsigned long long are[2], aim[2], bre[2], bim[2];  // sub-row A / B, real / imaginary
            #pragma unroll
            for (int gc = 0; gc < 2; ++gc) are[gc] = aim[gc] = bre[gc] = bim[gc] = 0ull;
            float2 w = make_float2(1.f, 0.f);
            #pragma unroll
            for (int n0 = 0; n0 < NH; n0 += CH) {
                uint32_t vg[CH][2], vx[CH][2], vo[G ? CH : 1][2], vi[G ? CH : 1][2];
                #pragma unroll
                for (int m = 0; m < CH; ++m)
                    #pragma unroll
                    for (int gc = 0; gc < 2; ++gc) {
                        const int64_t j = roff + int64_t(L2) * (n0 + m) + 1024 * gc;
                        vg[m][gc] = __ldg(reinterpret_cast<const uint32_t*>(dy + j));
                        vx[m][gc] = __ldg(reinterpret_cast<const uint32_t*>(u + j));
                        if constexpr (G) {
                            vo[m][gc] = __ldg(reinterpret_cast<const uint32_t*>(w_out + j));
                            vi[m][gc] = __ldg(reinterpret_cast<const uint32_t*>(w_in + j));
                        }
                    }
                #pragma unroll
                for (int m = 0; m < CH; ++m) {
                    const int n1 = n0 + m;
                    const unsigned long long WX = dk_pk(w.x, w.x), WY = dk_pk(w.y, w.y), WYn = dk_pk(-w.y, -w.y);
                    #pragma unroll
                    for (int gc = 0; gc < 2; ++gc) {
                        cpx g2 = O::unpack(vg[m][gc]), x2 = O::unpack(vx[m][gc]);
                        if constexpr (G) {
                            const cpx o2 = O::unpack(vo[m][gc]), i2 = O::unpack(vi[m][gc]);
                            g2.r *= o2.r; g2.i *= o2.i;
                            x2.r *= i2.r; x2.i *= i2.i;
                        }
                        const unsigned long long g = dk_pk(g2.r, g2.i), x = dk_pk(x2.r, x2.i);
                        if (p == 0) {
                            are[gc] = dk_add2(are[gc], g);
                            aim[gc] = dk_add2(aim[gc], x);
                            bre[gc] = (n1 & 1) ? dk_sub2(bre[gc], g) : dk_add2(bre[gc], g);
                            bim[gc] = (n1 & 1) ? dk_sub2(bim[gc], x) : dk_add2(bim[gc], x);
                        } else {
                            are[gc] = dk_fma2(x, WYn, dk_fma2(g, WX, are[gc]));  // z W
                            aim[gc] = dk_fma2(x, WX, dk_fma2(g, WY, aim[gc]));
                            bre[gc] = dk_fma2(x, WY, dk_fma2(g, WX, bre[gc]));   // z conj W
                            bim[gc] = dk_fma2(g, WYn, dk_fma2(x, WX, bim[gc]));
                        }
                    }
                    w = dk_cmul(w, wst);
                }
            }
            #pragma unroll
            for (int gc = 0; gc < 2; ++gc) {
                const float2 ar = dk_upk(are[gc]), ai = dk_upk(aim[gc]), br = dk_upk(bre[gc]), bi = dk_upk(bim[gc]);
                sa[2 * gc] = make_float2(ar.x, ai.x);
                sa[2 * gc + 1] = make_float2(ar.y, ai.y);
                sb[2 * gc] = make_float2(br.x, bi.x);
                sb[2 * gc + 1] = make_float2(br.y, bi.y);
            }
          }
            // the radix-2 pass: butterfly j = 2t + e takes columns j and j + 1024
            #pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float2 a0 = dk_cmul(sa[e], ctw[e][0]), b0 = dk_cmul(sb[e], ctw[e][1]);
                const float2 a1 = dk_cmul(sa[2 + e], ctw[2 + e][0]), b1 = dk_cmul(sb[2 + e], ctw[2 + e][1]);
                const int j = 2 * t + e;
                bufB[dk_sw(2 * j)] = make_float4(a0.x + a1.x, b0.x + b1.x, a0.y + a1.y, b0.y + b1.y);
                bufB[dk_sw(2 * j + 1)] = make_float4(a0.x - a1.x, b0.x - b1.x, a0.y - a1.y, b0.y - b1.y);
            }
            __syncthreads();
            dk_fft_r4(bufA, bufB, ftw);
            // S += G conj X on this thread's bins; for k1 > 0 on sub-row A only,
            // since S[-f] = conj S[f] gives sub-row B's bins at the end
            #pragma unroll
            for (int e = 0; e < NE; ++e) {
                const int k2 = t + T * e;
                const float4 z = bufA[dk_sw(k2)];
                const float4 zb = bufA[dk_sw(L2 - 1 - k2)];  // partner of sub-row A (k1 > 0) or of sub-row B (pair 0)
                float2 sA;
                if (p == 0) {
                    const float4 za = bufA[dk_sw((L2 - k2) & (L2 - 1))];
                    sA = dk_cross(z.x, z.z, za.x, za.z);
                    const float2 sB = dk_cross(z.y, z.w, zb.y, zb.w);
                    float2 v = acc[L2 + k2];
                    acc[L2 + k2] = make_float2(v.x + sB.x, v.y + sB.y);
                } else {
                    sA = dk_cross(z.x, z.z, zb.y, zb.w);
                }
                float2 v = acc[k2];
                acc[k2] = make_float2(v.x + sA.x, v.y + sA.y);
            }
            __syncthreads();  // the buffers are refilled by the next row
        }
        // conj S (both sub-rows; conj S_B[k2] = S_A[L2 - 1 - k2] for k1 > 0),
        // transformed along k2; the twiddle W_L^(k1 n2) -> R[h][k1][n2]
        #pragma unroll
        for (int e = 0; e < NE; ++e) {
            const int k2 = t + T * e;
            const float2 sA = acc[k2];
            float2 cB;  // conj S_B[k2]
            if (p == 0) {
                const float2 v = acc[L2 + k2];
                cB = make_float2(v.x, -v.y);
            } else {
                cB = acc[L2 - 1 - k2];
            }
            bufA[dk_sw(k2)] = make_float4(sA.x, cB.x, -sA.y, cB.y);
        }
        __syncthreads();
        #pragma unroll
        for (int e = 0; e < 2; ++e) {  // radix-2 pass: butterflies t and t + 512
            const int j = t + T * e;
            const float4 c0 = bufA[dk_sw(j)], c1 = bufA[dk_sw(j + L2 / 2)];
            bufB[dk_sw(2 * j)] = make_float4(c0.x + c1.x, c0.y + c1.y, c0.z + c1.z, c0.w + c1.w);
            bufB[dk_sw(2 * j + 1)] = make_float4(c0.x - c1.x, c0.y - c1.y, c0.z - c1.z, c0.w - c1.w);
        }
        __syncthreads();
        dk_fft_r4(bufA, bufB, ftw);
        #pragma unroll
        for (int e = 0; e < NE; ++e) {
            const int n2 = t + T * e;
            const float4 v = bufA[dk_sw(n2)];
            R[(h * L1 + kA) * L2 + n2] = dk_cmul(make_float2(v.x, v.z), dk_twiddle(uint32_t(kA) * uint32_t(n2), L));
            R[(h * L1 + kB) * L2 + n2] = dk_cmul(make_float2(v.y, v.w), dk_twiddle(uint32_t(kB) * uint32_t(n2), L));
        }
        __syncthreads();  // the buffers are reused by the next item
    }
}

// 2N = 128K .. 4M: the column passes of the four-step form run as batched
// L1-point transforms in shared memory, L1 = L / 2048 = 64 .. 2048, on tiles
// of TC = 2^lgTC consecutive columns (element (n1, c) at n1 * TC + c; TC = 16
// up to L1 = 512, then 8 and 4, so that two buffers take at most 128 KB);
// Stockham radix-4 passes (one radix-2 pass first for odd log2 L1) between
// two buffers.  Returns the buffer holding the result.
constexpr int kDkColThreads = 256;
__host__ __device__ inline int dk_col_lgtc(int lgL1) { return lgL1 <= 9 ? 4 : (lgL1 == 10 ? 3 : 2); }

__device__ float2* dk_colfft(float2* a, float2* b, int lgL1, int lgTC) {
    const int TC = 1 << lgTC;
    const int L1 = 1 << lgL1;
    int lgNs = 0;
    if (lgL1 & 1) {
        for (int j = threadIdx.x; j < (L1 / 2) * TC; j += blockDim.x) {
            const int c = j & (TC - 1), jj = j >> lgTC;
            const float2 c0 = a[jj * TC + c], c1 = a[(jj + L1 / 2) * TC + c];
            b[(2 * jj) * TC + c] = make_float2(c0.x + c1.x, c0.y + c1.y);
            b[(2 * jj + 1) * TC + c] = make_float2(c0.x - c1.x, c0.y - c1.y);
        }
        __syncthreads();
        float2* x = a; a = b; b = x;
        lgNs = 1;
    }
    for (; lgNs < lgL1; lgNs += 2) {
        const int Ns = 1 << lgNs, Q = L1 >> 2;
        for (int j = threadIdx.x; j < Q * TC; j += blockDim.x) {
            const int c = j & (TC - 1), jq = j >> lgTC;
            const int kk = jq & (Ns - 1), jh = jq >> lgNs;
            float2 v0 = a[jq * TC + c], v1 = a[(jq + Q) * TC + c], v2 = a[(jq + 2 * Q) * TC + c],
                   v3 = a[(jq + 3 * Q) * TC + c];
            float s1, c1;  // W_{4 Ns}^kk
            sincospif(-float(kk) / float(2 * Ns), &s1, &c1);
            const float c2 = c1 * c1 - s1 * s1, s2 = 2.f * c1 * s1;
            const float c3 = c2 * c1 - s2 * s1, s3 = c2 * s1 + s2 * c1;
            v1 = make_float2(v1.x * c1 - v1.y * s1, v1.x * s1 + v1.y * c1);
            v2 = make_float2(v2.x * c2 - v2.y * s2, v2.x * s2 + v2.y * c2);
            v3 = make_float2(v3.x * c3 - v3.y * s3, v3.x * s3 + v3.y * c3);
            const float2 a0 = make_float2(v0.x + v2.x, v0.y + v2.y), a1 = make_float2(v0.x - v2.x, v0.y - v2.y);
            const float2 a2 = make_float2(v1.x + v3.x, v1.y + v3.y);
            const float2 a3 = make_float2(v1.y - v3.y, v3.x - v1.x);  // -i (v1 - v3)
            const int o = kk + (jh << (lgNs + 2));
            b[o * TC + c] = make_float2(a0.x + a2.x, a0.y + a2.y);
            b[(o + Ns) * TC + c] = make_float2(a1.x + a3.x, a1.y + a3.y);
            b[(o + 2 * Ns) * TC + c] = make_float2(a0.x - a2.x, a0.y - a2.y);
            b[(o + 3 * Ns) * TC + c] = make_float2(a1.x - a3.x, a1.y - a3.y);
        }
        __syncthreads();
        float2* x = a; a = b; b = x;
    }
    return a;
}

// A[r][k1][n2] = W_L^(n2 k1) sum_{n1 < L1/2} z_r[L2 n1 + n2] W_L1^(n1 k1), one CTA
// per tile of TC columns of a row; shared memory 2 L1 TC float2.
template <int DT, bool G>
__global__ void __launch_bounds__(kDkColThreads) dk_colfft_fwd(const uint16_t* __restrict__ u,
                                                               const uint16_t* __restrict__ dy,
                                                               const uint16_t* __restrict__ w_in,
                                                               const uint16_t* __restrict__ w_out,
                                                               float2* __restrict__ A, int64_t rows, int lgL1) {
    using O = Op<DT>;
    constexpr int L2 = kDkL2;
    extern __shared__ __align__(16) float2 csm[];
    const int L1 = 1 << lgL1, lgTC = dk_col_lgtc(lgL1), TC = 1 << lgTC;
    const int64_t N = int64_t(L1 / 2) * L2;
    const uint32_t L = uint32_t(L1) * uint32_t(L2);
    const int64_t tiles = rows * (L2 / TC);
    for (int64_t it = blockIdx.x; it < tiles; it += gridDim.x) {
        const int64_t r = it / (L2 / TC);
        const int c0 = int(it - r * (L2 / TC)) * TC;
        for (int i = threadIdx.x; i < L1 * TC; i += blockDim.x) {
            const int n1 = i >> lgTC, c = i & (TC - 1);
            float2 v = make_float2(0.f, 0.f);
            if (n1 < L1 / 2) {  // the upper half of z is zero
                const int64_t j = r * N + int64_t(L2) * n1 + c0 + c;
                float g = O::unpack(uint32_t(dy[j])).r, x = O::unpack(uint32_t(u[j])).r;
                if (G) {
                    g *= O::unpack(uint32_t(w_out[j])).r;
                    x *= O::unpack(uint32_t(w_in[j])).r;
                }
                v = make_float2(g, x);
            }
            csm[i] = v;
        }
        __syncthreads();
        const float2* z = dk_colfft(csm, csm + L1 * TC, lgL1, lgTC);
        for (int i = threadIdx.x; i < L1 * TC; i += blockDim.x) {
            const int k1 = i >> lgTC, c = i & (TC - 1);
            const uint32_t n2 = uint32_t(c0 + c);
            A[(r * L1 + k1) * int64_t(L2) + n2] = dk_cmul(z[i], dk_twiddle(n2 * uint32_t(k1), L));
        }
        __syncthreads();  // the buffers are refilled by the next tile
    }
}

// dk[h][n2 + L2 n1] = Re(sum_k1 R[h][k1][n2] W_L1^(k1 n1)) / L for n1 < L1/2,
// one CTA per tile of TC columns of a channel.
__global__ void __launch_bounds__(kDkColThreads) dk_colfft_inv(const float2* __restrict__ R, float* __restrict__ dk,
                                                               int64_t H, int lgL1) {
    constexpr int L2 = kDkL2;
    extern __shared__ __align__(16) float2 csm[];
    const int L1 = 1 << lgL1, lgTC = dk_col_lgtc(lgL1), TC = 1 << lgTC;
    const int64_t N = int64_t(L1 / 2) * L2;
    const float sc = 1.f / (float(L1) * float(L2));
    const int64_t tiles = H * (L2 / TC);
    for (int64_t it = blockIdx.x; it < tiles; it += gridDim.x) {
        const int64_t h = it / (L2 / TC);
        const int c0 = int(it - h * (L2 / TC)) * TC;
        for (int i = threadIdx.x; i < L1 * TC; i += blockDim.x) {
            const int k1 = i >> lgTC, c = i & (TC - 1);
            csm[i] = R[(h * L1 + k1) * int64_t(L2) + c0 + c];
        }
        __syncthreads();
        const float2* y = dk_colfft(csm, csm + L1 * TC, lgL1, lgTC);
        for (int i = threadIdx.x; i < (L1 / 2) * TC; i += blockDim.x) {
            const int n1 = i >> lgTC, c = i & (TC - 1);
            dk[h * N + int64_t(L2) * n1 + c0 + c] = y[i].x * sc;
        }
        __syncthreads();
    }
}

// dk[h][n2 + L2 n1] = Re(sum_k1 R[h][k1][n2] W_L1^(k1 n1)) / L, n1 < L1/2; one
// thread per column (h, n2).
template <int L1>
__global__ void __launch_bounds__(256) dk_cols_inv(const float2* __restrict__ R, float* __restrict__ dk, int64_t H) {
    constexpr int L2 = kDkL2;
    constexpr int64_t N = int64_t(L2) * (L1 / 2);
    const float sc = 1.f / float(L1 * L2);
    float2 wt[L1];
    #pragma unroll
    for (int m = 0; m < L1; ++m) wt[m] = dk_twiddle(uint32_t(m), uint32_t(L1));
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < H * L2;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t h = i / L2, n2 = i % L2;
        float2 v[L1];
        #pragma unroll
        for (int k1 = 0; k1 < L1; ++k1) v[k1] = R[(h * L1 + k1) * L2 + n2];
        #pragma unroll
        for (int n1 = 0; n1 < L1 / 2; ++n1) {
            float s = 0.f;
            #pragma unroll
            for (int k1 = 0; k1 < L1; ++k1) {
                const float2 w = wt[(k1 * n1) & (L1 - 1)];
                s += v[k1].x * w.x - v[k1].y * w.y;
            }
            dk[h * N + L2 * n1 + n2] = s * sc;
        }
    }
}

}  // namespace fftconv
