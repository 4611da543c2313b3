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

// Twiddles of the radix-4 passes of dk_fft2048x2: W_4Ns^kk for kk < Ns, pass
// p (Ns = 2 * 4^p) at offset 2 (4^p - 1) / 3, i.e. 0, 2, 10, 42, 170.
constexpr int kDkTwEntries = 2 + 8 + 32 + 128 + 512;
__device__ __forceinline__ int dk_tw_off(int p) { return (2 * ((1 << (2 * p)) - 1)) / 3; }

// Two 2048-point DFTs (exponent sign -1) of the sequences at a[0..2048) and
// a[2048..4096), Stockham: one radix-2 pass a -> b, then five radix-4 passes
// of span Ns = 2, 8, 32, 128, 512 alternating b -> a -> b ..., so the result
// lands back in a.  512 threads: thread t runs butterfly t of both sequences
// with the twiddle W_4Ns^(t mod Ns) from the table tw.
__device__ __forceinline__ void dk_fft2048x2(float2* a, float2* b, const float2* tw) {
    constexpr int L2 = kDkL2, Q = L2 / 4;
    const int t = threadIdx.x;
    #pragma unroll
    for (int s = 0; s < 2; ++s) {  // radix 2: 1024 butterflies per sequence, two per thread
        #pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int j = t + kDkRowThreads * hh;
            const float2 c0 = a[s * L2 + j], c1 = a[s * L2 + j + L2 / 2];
            b[s * L2 + 2 * j] = make_float2(c0.x + c1.x, c0.y + c1.y);
            b[s * L2 + 2 * j + 1] = make_float2(c0.x - c1.x, c0.y - c1.y);
        }
    }
    __syncthreads();
    #pragma unroll
    for (int p = 0; p < 5; ++p) {
        const int lgNs = 1 + 2 * p, Ns = 1 << lgNs;
        const float2* x0 = (p & 1) ? a : b;
        float2* y0 = (p & 1) ? b : a;
        const int kk = t & (Ns - 1), jj = t >> lgNs;
        const float2 w1 = tw[dk_tw_off(p) + kk];
        const float c1 = w1.x, s1 = w1.y;
        const float c2 = c1 * c1 - s1 * s1, s2 = 2.f * c1 * s1;
        const float c3 = c2 * c1 - s2 * s1, s3 = c2 * s1 + s2 * c1;
        #pragma unroll
        for (int s = 0; s < 2; ++s) {
            const float2* x = x0 + s * L2;
            float2 v0 = x[t], v1 = x[t + Q], v2 = x[t + 2 * Q], v3 = x[t + 3 * Q];
            v1 = make_float2(v1.x * c1 - v1.y * s1, v1.x * s1 + v1.y * c1);
            v2 = make_float2(v2.x * c2 - v2.y * s2, v2.x * s2 + v2.y * c2);
            v3 = make_float2(v3.x * c3 - v3.y * s3, v3.x * s3 + v3.y * c3);
            const float2 a0 = make_float2(v0.x + v2.x, v0.y + v2.y), a1 = make_float2(v0.x - v2.x, v0.y - v2.y);
            const float2 a2 = make_float2(v1.x + v3.x, v1.y + v3.y);
            const float2 a3 = make_float2(v1.y - v3.y, v3.x - v1.x);  // -i (v1 - v3)
            float2* y = y0 + s * L2 + kk + (jj << (lgNs + 2));
            y[0] = make_float2(a0.x + a2.x, a0.y + a2.y);
            y[Ns] = make_float2(a1.x + a3.x, a1.y + a3.y);
            y[2 * Ns] = make_float2(a0.x - a2.x, a0.y - a2.y);
            y[3 * Ns] = make_float2(a1.x - a3.x, a1.y - a3.y);
        }
        __syncthreads();
    }
}

// One CTA per (channel h, pair of sub-rows p), looping over the batch.  The
// CTAs of a channel run side by side (items are numbered channel-major), so
// each row of u and dy comes from DRAM about once and from L2 L1/2 times.
// Thread t computes the column sums of columns n2 = 4t .. 4t + 3 (8-byte
// loads of four 16-bit inputs, a few rows n1 in flight at once) and owns
// entries t + 512 e of the pair's 2 x 2048 bins in the batch sum.  Shared
// memory: two transform buffers and the batch sum S, 2 x 2048 entries each,
// and the transform's twiddles (101.5 KB, two CTAs per SM).
template <int DT, int L1, bool G>
__global__ void __launch_bounds__(kDkRowThreads, 2) dk_rows(const uint16_t* __restrict__ u,
                                                            const uint16_t* __restrict__ dy,
                                                            const uint16_t* __restrict__ w_in,
                                                            const uint16_t* __restrict__ w_out,
                                                            float2* __restrict__ R, int64_t B, int64_t H) {
    using O = Op<DT>;
    constexpr int L2 = kDkL2, T = kDkRowThreads, COLS = L2 / T, E = 2 * COLS;
    constexpr int NH = L1 / 2, CH = G ? 2 : 4;  // input rows n1; rows loaded per round
    static_assert(COLS == 4 && NH % CH == 0, "four columns per thread");
    constexpr int64_t N = int64_t(L2) * NH;
    constexpr uint32_t L = uint32_t(L1) * uint32_t(L2);
    extern __shared__ __align__(16) float2 dsm[];
    float2* buf0 = dsm;
    float2* buf1 = dsm + 2 * L2;
    float2* acc = dsm + 4 * L2;  // S, entry q = sub-row * L2 + k2
    float2* ftw = dsm + 6 * L2;  // radix-4 twiddles of the transforms
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
        // W_L^(n2 k1) of this thread's columns n2 = 4t + c, both sub-rows
        float2 ctw[COLS][2];
        #pragma unroll
        for (int c = 0; c < COLS; ++c) {
            const uint32_t n2 = uint32_t(4 * t + c);
            ctw[c][0] = dk_twiddle(n2 * uint32_t(kA), L);
            ctw[c][1] = dk_twiddle(n2 * uint32_t(kB), L);
        }
        const float2 wst = dk_twiddle(uint32_t(kA), uint32_t(L1));  // W_L1^kA
        #pragma unroll
        for (int e = 0; e < E; ++e) acc[t + T * e] = make_float2(0.f, 0.f);
        for (int64_t b = 0; b < B; ++b) {
            const int64_t roff = (b * H + h) * N + 4 * t;
            // A_k1[n2] = W_L^(n2 k1) sum_{n1 < L1/2} z[L2 n1 + n2] W_L1^(n1 k1), with
            // W_L1^(n1 kB) = conj W_L1^(n1 kA) (kB = L1 - kA) or, on pair 0,
            // W_L1^0 = 1 and W_L1^(n1 L1/2) = (-1)^n1
            float2 sa[COLS], sb[COLS];
            #pragma unroll
            for (int c = 0; c < COLS; ++c) sa[c] = sb[c] = make_float2(0.f, 0.f);
            float2 w = make_float2(1.f, 0.f);
            #pragma unroll
            for (int n0 = 0; n0 < NH; n0 += CH) {
                uint2 vg[CH], vx[CH], vo[G ? CH : 1], vi[G ? CH : 1];
                #pragma unroll
                for (int m = 0; m < CH; ++m) {
                    const int64_t j = roff + int64_t(L2) * (n0 + m);
                    vg[m] = __ldg(reinterpret_cast<const uint2*>(dy + j));
                    vx[m] = __ldg(reinterpret_cast<const uint2*>(u + j));
                    if constexpr (G) {
                        vo[m] = __ldg(reinterpret_cast<const uint2*>(w_out + j));
                        vi[m] = __ldg(reinterpret_cast<const uint2*>(w_in + j));
                    }
                }
                #pragma unroll
                for (int m = 0; m < CH; ++m) {
                    const int n1 = n0 + m;
                    const cpx g01 = O::unpack(vg[m].x), g23 = O::unpack(vg[m].y);
                    const cpx x01 = O::unpack(vx[m].x), x23 = O::unpack(vx[m].y);
                    float gg[4] = {g01.r, g01.i, g23.r, g23.i}, xx[4] = {x01.r, x01.i, x23.r, x23.i};
                    if constexpr (G) {
                        const cpx o01 = O::unpack(vo[m].x), o23 = O::unpack(vo[m].y);
                        const cpx i01 = O::unpack(vi[m].x), i23 = O::unpack(vi[m].y);
                        gg[0] *= o01.r; gg[1] *= o01.i; gg[2] *= o23.r; gg[3] *= o23.i;
                        xx[0] *= i01.r; xx[1] *= i01.i; xx[2] *= i23.r; xx[3] *= i23.i;
                    }
                    #pragma unroll
                    for (int c = 0; c < COLS; ++c) {
                        const float g = gg[c], x = xx[c];
                        if (p == 0) {
                            const float sg = (n1 & 1) ? -1.f : 1.f;
                            sa[c].x += g;
                            sa[c].y += x;
                            sb[c].x += sg * g;
                            sb[c].y += sg * x;
                        } else {
                            const float P1 = g * w.x, P2 = x * w.y, P3 = g * w.y, P4 = x * w.x;
                            sa[c].x += P1 - P2;  // z W
                            sa[c].y += P3 + P4;
                            sb[c].x += P1 + P2;  // z conj W
                            sb[c].y += P4 - P3;
                        }
                    }
                    w = dk_cmul(w, wst);
                }
            }
            #pragma unroll
            for (int c = 0; c < COLS; c += 2) {
                const float2 a0 = dk_cmul(sa[c], ctw[c][0]), a1 = dk_cmul(sa[c + 1], ctw[c + 1][0]);
                const float2 b0 = dk_cmul(sb[c], ctw[c][1]), b1 = dk_cmul(sb[c + 1], ctw[c + 1][1]);
                *reinterpret_cast<float4*>(buf0 + 4 * t + c) = make_float4(a0.x, a0.y, a1.x, a1.y);
                *reinterpret_cast<float4*>(buf0 + L2 + 4 * t + c) = make_float4(b0.x, b0.y, b1.x, b1.y);
            }
            __syncthreads();
            dk_fft2048x2(buf0, buf1, ftw);
            // S += G conj X on this thread's entries; for k1 > 0 on sub-row A only,
            // since S[-f] = conj S[f] gives sub-row B's bins at the end
            #pragma unroll
            for (int e = 0; e < E; ++e) {
                const int s = e / COLS, q = t + T * e, k2 = q - s * L2;  // sub-row s (T * COLS = L2)
                if (s == 1 && p != 0) break;
                int pq;  // the partner entry -f
                if (p == 0)
                    pq = s == 0 ? ((L2 - k2) & (L2 - 1)) : L2 + (L2 - 1 - k2);
                else
                    pq = (s == 0 ? L2 : 0) + (L2 - 1 - k2);
                const float2 a = buf0[q], cc = buf0[pq];  // Z[f], Z[-f]
                const float gr = 0.5f * (a.x + cc.x), gi = 0.5f * (a.y - cc.y);   // G
                const float xr = 0.5f * (a.y + cc.y), xi = -0.5f * (a.x - cc.x);  // X
                float2 v = acc[q];
                v.x += gr * xr + gi * xi;  // G conj X
                v.y += gi * xr - gr * xi;
                acc[q] = v;
            }
            __syncthreads();  // buf0 is refilled by the next row
        }
        // conj S, transformed along k2; the twiddle W_L^(k1 n2) -> R[h][k1][n2]
        if (p == 0) {
            #pragma unroll
            for (int e = 0; e < E; ++e) {
                const float2 v = acc[t + T * e];
                buf0[t + T * e] = make_float2(v.x, -v.y);
            }
        } else {  // conj S_B[L2 - 1 - k2] = S_A[k2]
            #pragma unroll
            for (int e = 0; e < COLS; ++e) {
                const int q = t + T * e;
                const float2 v = acc[q];
                buf0[q] = make_float2(v.x, -v.y);
                buf0[2 * L2 - 1 - q] = v;
            }
        }
        __syncthreads();
        dk_fft2048x2(buf0, buf1, ftw);
        #pragma unroll
        for (int e = 0; e < E; ++e) {
            const int s = e / COLS, q = t + T * e, n2 = q - s * L2;
            const int k1 = s ? kB : kA;
            R[(h * L1 + k1) * L2 + n2] = dk_cmul(buf0[q], dk_twiddle(uint32_t(k1) * uint32_t(n2), L));
        }
        __syncthreads();  // the buffers are reused by the next item
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
