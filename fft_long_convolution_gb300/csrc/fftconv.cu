// C-ABI implementation: plans, kernel spectrum, forward launches.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/fftconv.h"
#include "plan.h"
#include "dkgrad.cuh"
#include "ftc.cuh"
#include "tcconv.cuh"
#include "tcpass.cuh"

using namespace fftconv;

namespace {

constexpr double kPi = 3.14159265358979323846264338327950288;

struct cd {
    double r, i;
};

// exp(-2 pi i e / n), with e reduced mod n first so the angle is exact.
cd W(int64_t n, int64_t e) {
    e %= n;
    if (e < 0) e += n;
    double a = -2.0 * kPi * double(e) / double(n);
    return {std::cos(a), std::sin(a)};
}

// Element of the real embedding of a complex weight w: output part ro
// (0 = real, 1 = imaginary) from input part ri.
double embed(cd w, int ro, int ri) {
    if (ro == 0) return ri == 0 ? w.r : -w.i;
    return ri == 0 ? w.i : w.r;
}

uint16_t to_bits(double v, int dtype) {
    float f = static_cast<float>(v);
    if (dtype == FFTCONV_F16) {
        __half h = __float2half_rn(f);
        uint16_t b;
        std::memcpy(&b, &h, 2);
        return b;
    }
    uint32_t x;
    std::memcpy(&x, &f, 4);
    uint32_t bias = 0x7FFFu + ((x >> 16) & 1u);
    return static_cast<uint16_t>((x + bias) >> 16);
}

uint32_t pack2(double lo, double hi, int dtype) {
    return uint32_t(to_bits(lo, dtype)) | (uint32_t(to_bits(hi, dtype)) << 16);
}

bool is_pow2(int64_t n) { return n > 0 && (n & (n - 1)) == 0; }

// Row counts the kernels index with 32-bit integers: B, H and B*H each at
// most 2^30, tested without forming a product that could overflow.
constexpr int64_t kMaxRows = int64_t(1) << 30;
bool too_many_rows(int64_t B, int64_t H) {
    return B > kMaxRows || H > kMaxRows || (B > 0 && H > kMaxRows / B);
}

}  // namespace

// A plan's tables live on the device that was current when it was made; a
// call made with another device current is refused (FFTCONV_ERR_INVALID).
static bool wrong_device(const fftconv_plan_s* p) {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return d != p->device;
}

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace


// --------------------------------------------------------------- planning

extern "C" fftconv_status_t fftconv_plan_query(int64_t N, fftconv_dtype_t dtype, int order,
                                               fftconv_plan_info_t* info) {
    if (!info) return FFTCONV_ERR_INVALID;
    if (dtype != FFTCONV_F16 && dtype != FFTCONV_BF16) return FFTCONV_ERR_UNSUPPORTED;
    if (!is_pow2(N) || N < 1024 || N > (int64_t(1) << 21)) return FFTCONV_ERR_UNSUPPORTED;
    fftconv_plan_info_t q;
    std::memset(&q, 0, sizeof(q));
    q.N = N;
    q.M = N;
    q.dtype = dtype;
    if (N == 4096 || (N < 4096 && (order == 0 || order == 2))) {
        // fused on the fifth-generation tensor cores: M = 64 * 64; N = 1024 and
        // 2048 as rows zero-padded to 4096 (a causal convolution's first N
        // outputs are those of the padded rows)
        q.path = FFTCONV_PATH_FUSED;
        q.order = 2;
        q.factors[0] = 64;
        q.factors[1] = 64;
        q.M = 4096;
        q.workspace_bytes_per_row = 0;
    } else if (N == 8192 || N == 16384 || (N == 32768 && order != 4)) {
        // fused on the fifth-generation tensor cores: M = R0 * 64 * 64, the
        // outer factor R0 = 2, 4 or 8 in shared memory
        q.path = FFTCONV_PATH_FUSED;
        q.order = 3;
        q.factors[0] = int32_t(N / 4096);
        q.factors[1] = 64;
        q.factors[2] = 64;
        q.workspace_bytes_per_row = 0;
    } else if (N <= 16384) {
        // fused: M = R1 * 16 * 16
        q.path = FFTCONV_PATH_FUSED;
        q.order = 3;
        q.factors[0] = int32_t(N / 256);
        q.factors[1] = 16;
        q.factors[2] = 16;
        q.workspace_bytes_per_row = 0;
    } else if ((order == 0 || order == 4) && N >= (int64_t(1) << 20)) {
        // multi-pass: M = RA * 64 * 64 * 64, the outer factor R0 = RA * 64 through
        // HBM in two levels, sub-rows of 4096 on the tensor cores
        q.path = FFTCONV_PATH_MULTIPASS;
        q.order = 4;
        q.factors[0] = int32_t(N >> 18);
        q.factors[1] = 64;
        q.factors[2] = 64;
        q.factors[3] = 64;
        q.workspace_bytes_per_row = 4 * N;  // 16-bit complex intermediate
    } else if ((order == 0 || order == 3) && N <= (int64_t(1) << 19)) {
        // multi-pass: M = R0 * 64 * 64, outer factor R0 through HBM, sub-rows
        // of 4096 on the tensor cores (the default up to N = 512K)
        q.path = FFTCONV_PATH_MULTIPASS;
        q.order = 3;
        q.factors[0] = int32_t(N / 4096);
        q.factors[1] = 64;
        q.factors[2] = 64;
        q.workspace_bytes_per_row = 4 * N;  // 16-bit complex intermediate
    } else {
        // multi-pass: M = R0 * 64 * 16 * 16, outer factor R0 through HBM
        q.path = FFTCONV_PATH_MULTIPASS;
        q.order = 4;
        q.factors[0] = int32_t(N / 16384);
        q.factors[1] = 64;
        q.factors[2] = 16;
        q.factors[3] = 16;
        q.workspace_bytes_per_row = 4 * N;  // 16-bit complex intermediate
    }
    if (order != 0 && order != q.order) return FFTCONV_ERR_UNSUPPORTED;
    // two 16-bit complex coefficients per bin (plus zero padding bins on the
    // 64 x 64 paths, whose k_f follows the kernels' column layouts)
    if (q.order == 2)
        q.kf_bytes_per_channel = int64_t(Tc64::KFB);
    else if (q.order == 3 && q.factors[1] == 64)  // pairs of 4096-point sub-rows (fused or multi-pass)
        q.kf_bytes_per_channel = int64_t(q.factors[0] / 2) * TcB::KFP * 16;
    else if (q.path == FFTCONV_PATH_MULTIPASS && q.factors[3] == 64)  // two-level outer factor
        q.kf_bytes_per_channel = int64_t(q.factors[0] * 64 / 2) * TcB::KFP * 16;
    else
        q.kf_bytes_per_channel = q.M * 8;
    *info = q;
    return FFTCONV_OK;
}

namespace {

// Host tables of the fused path for M = R1 * 256 (layouts documented in
// fused.cuh, FusedTables).
struct HostTables {
    std::vector<uint32_t> lf, rf, of, oi;
    std::vector<float> tw, twf, twi;
};

HostTables build_fused_tables(int R1, int dtype) {
    HostTables T;
    const int64_t M = int64_t(R1) * 256;
    const double s16 = 0.25, sR = 1.0 / std::sqrt(double(R1));
    auto F16 = [&](int a, int b) { cd w = W(16, int64_t(a) * b); return cd{w.r * s16, w.i * s16}; };
    T.lf.assign(32 * 16, 0);
    T.rf.assign(32 * 16, 0);
    T.tw.assign(32 * 16, 0.f);
    for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3;
        // left product (A operand): rows (k, ro) = (8m + (r&7), r>>3), K (n, ri) = (8s + (q>>1), q&1)
        for (int m = 0; m < 2; ++m)
            for (int s = 0; s < 2; ++s) {
                auto el = [&](int r, int q) {
                    return embed(F16(8 * m + (r & 7), 8 * s + (q >> 1)), r >> 3, q & 1);
                };
                uint32_t* o = &T.lf[lane * 16 + (m * 2 + s) * 4];
                o[0] = pack2(el(g, 2 * t), el(g, 2 * t + 1), dtype);
                o[1] = pack2(el(g + 8, 2 * t), el(g + 8, 2 * t + 1), dtype);
                o[2] = pack2(el(g, 2 * t + 8), el(g, 2 * t + 9), dtype);
                o[3] = pack2(el(g + 8, 2 * t + 8), el(g + 8, 2 * t + 9), dtype);
            }
        // right product (B operand): K (n3, ri) = (8s + 2((q&7)>>1) + (q>>3), q&1),
        // columns (k3, ro) = (4nt + (c>>1), c&1)
        for (int s = 0; s < 2; ++s)
            for (int nt = 0; nt < 4; ++nt) {
                auto el = [&](int q, int c) {
                    int n3 = 8 * s + 2 * ((q & 7) >> 1) + (q >> 3);
                    int k3 = 4 * nt + (c >> 1);
                    return embed(F16(n3, k3), c & 1, q & 1);
                };
                const int q4 = s * 2 + (nt >> 1), slot = nt & 1;
                uint32_t* o = &T.rf[lane * 16 + q4 * 4 + slot * 2];
                o[0] = pack2(el(2 * t, g), el(2 * t + 1, g), dtype);
                o[1] = pack2(el(2 * t + 8, g), el(2 * t + 9, g), dtype);
            }
        for (int m = 0; m < 2; ++m)
            for (int c = 0; c < 2; ++c)
                for (int e = 0; e < 2; ++e) {
                    cd w = W(256, int64_t(8 * m + g) * (8 * c + 2 * t + e));
                    float* o = &T.tw[lane * 16 + (m * 2 + c) * 4];
                    o[e] = float(w.r);      // real parts of e = 0, 1
                    o[2 + e] = float(w.i);  // imaginary parts
                }
    }
    // outer stages
    const bool k8f = R1 <= 8, k8i = R1 <= 4;
    const int KS_F = k8f ? 1 : R1 / 16, MT_F = (R1 + 7) / 8;
    const int KS_I = k8i ? 1 : R1 / 8, MT_I = (R1 + 15) / 16;
    auto FR = [&](int a, int b) { cd w = W(R1, int64_t(a) * b); return cd{w.r * sR, w.i * sR}; };
    T.of.assign(size_t(MT_F) * KS_F * 32 * 4, 0);
    T.oi.assign(size_t(MT_I) * KS_I * 32 * 4, 0);
    for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3;
        for (int m = 0; m < MT_F; ++m)
            for (int s = 0; s < KS_F; ++s) {
                auto el = [&](int r, int q) -> double {
                    int k1 = 8 * m + (r & 7), n1 = 8 * s + (q >> 1);
                    if (k1 >= R1 || n1 >= R1 / 2) return 0.0;
                    return embed(FR(k1, n1), r >> 3, q & 1);
                };
                uint32_t* o = &T.of[((m * KS_F + s) * 32 + lane) * 4];
                o[0] = pack2(el(g, 2 * t), el(g, 2 * t + 1), dtype);
                o[1] = pack2(el(g + 8, 2 * t), el(g + 8, 2 * t + 1), dtype);
                if (!k8f) {
                    o[2] = pack2(el(g, 2 * t + 8), el(g, 2 * t + 9), dtype);
                    o[3] = pack2(el(g + 8, 2 * t + 8), el(g + 8, 2 * t + 9), dtype);
                }
            }
        for (int m = 0; m < MT_I; ++m)
            for (int s = 0; s < KS_I; ++s) {
                auto el = [&](int r, int q) -> double {
                    int n1 = 8 * m + (r & 7), k1 = 8 * s + (q >> 1);
                    if (n1 >= R1 / 2 || k1 >= R1) return 0.0;
                    return embed(FR(n1, k1), r >> 3, q & 1);
                };
                uint32_t* o = &T.oi[((m * KS_I + s) * 32 + lane) * 4];
                o[0] = pack2(el(g, 2 * t), el(g, 2 * t + 1), dtype);
                o[1] = pack2(el(g + 8, 2 * t), el(g + 8, 2 * t + 1), dtype);
                if (!k8i) {
                    o[2] = pack2(el(g, 2 * t + 8), el(g, 2 * t + 9), dtype);
                    o[3] = pack2(el(g + 8, 2 * t + 8), el(g + 8, 2 * t + 9), dtype);
                }
            }
    }
    // outer twiddles W_M^(o*k1)
    T.twf.assign(size_t(32) * MT_F * 32 * 4, 0.f);
    for (int nt = 0; nt < 32; ++nt)
        for (int m = 0; m < MT_F; ++m)
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, t = lane & 3, k1 = 8 * m + g;
                float* o = &T.twf[((nt * MT_F + m) * 32 + lane) * 4];
                if (k1 >= R1) continue;
                for (int e = 0; e < 2; ++e) {
                    cd w = W(M, int64_t(8 * nt + 2 * t + e) * k1);
                    o[e] = float(w.r);      // (wr e=0, wr e=1, wi e=0, wi e=1)
                    o[2 + e] = float(w.i);
                }
            }
    T.twi.assign(size_t(R1) * 4 * 32 * 4, 0.f);
    for (int k1 = 0; k1 < R1; ++k1)
        for (int nt = 0; nt < 4; ++nt)
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, t = lane & 3;
                const int o0 = 16 * (4 * nt + t) + g;
                float* o = &T.twi[((k1 * 4 + nt) * 32 + lane) * 4];
                for (int e = 0; e < 2; ++e) {
                    cd w = W(M, int64_t(o0 + 8 * e) * k1);
                    o[2 * e] = float(w.r);
                    o[2 * e + 1] = float(w.i);
                }
            }
    return T;
}

// A fragments of the full R-point DFT F_R/sqrt(R) (R a multiple of 16):
// rows (k, ro) = (8m + (r&7), r>>3), K (n, ri) = (8s + (q>>1), q&1).
std::vector<uint32_t> build_full_frags(int R, int dtype) {
    const int MT = R / 8, KS = R / 8;
    const double sc = 1.0 / std::sqrt(double(R));
    std::vector<uint32_t> v(size_t(MT) * KS * 32 * 4, 0);
    for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3;
        for (int m = 0; m < MT; ++m)
            for (int s = 0; s < KS; ++s) {
                auto el = [&](int r, int q) {
                    cd w = W(R, int64_t(8 * m + (r & 7)) * (8 * s + (q >> 1)));
                    return embed(cd{w.r * sc, w.i * sc}, r >> 3, q & 1);
                };
                uint32_t* o = &v[((m * KS + s) * 32 + lane) * 4];
                o[0] = pack2(el(g, 2 * t), el(g, 2 * t + 1), dtype);
                o[1] = pack2(el(g + 8, 2 * t), el(g + 8, 2 * t + 1), dtype);
                o[2] = pack2(el(g, 2 * t + 8), el(g, 2 * t + 9), dtype);
                o[3] = pack2(el(g + 8, 2 * t + 8), el(g + 8, 2 * t + 9), dtype);
            }
    }
    return v;
}

// Rows of F64/8 in the tensor-memory order of the 64 x 64 path (tcconv.cuh):
// lane L = 32w + 16b + 8p + r holds output kappa = b ? 63 - 8w - r : 8w + r,
// part p; word n holds the two K elements of input n (real, imaginary).
// Three copies: columns natural, then at positions tc64_p3(n), tc64_p4(n).
std::vector<uint32_t> build_tc64_fmat(int dtype) {
    std::vector<uint32_t> v(3 * 128 * 64, 0);
    for (int L = 0; L < 128; ++L) {
        const int w = L >> 5, b = (L >> 4) & 1, part = (L >> 3) & 1, r = L & 7;
        const int kap = b ? 63 - 8 * w - r : 8 * w + r;
        for (int n = 0; n < 64; ++n) {
            cd x = W(64, int64_t(kap) * n);
            x = {x.r / 8.0, x.i / 8.0};
            const uint32_t word = pack2(embed(x, part, 0), embed(x, part, 1), dtype);
            v[size_t(L) * 64 + n] = word;
            v[size_t(128 + L) * 64 + tc64_p3(n)] = word;
            v[size_t(256 + L) * 64 + tc64_p4(n)] = word;
        }
    }
    return v;
}

// Starting twiddles of the fused R0 x 64 x 64 kernel's threads (ftc.cuh):
// input phase W_M^(k0 n') / sqrt(R0) at n' = 1024 (t / 64) + t % 64, [k0][t];
// S4 post W_M^(k0 n') at n' = 64 kappa_b + 32 hf + 2q + e (thread t = 128 hf
// + 32 w + 4 r + q, kappa_0 = 8w + r, kappa_1 = 63 - kappa_0), [k0][b][t] x
// (re e0, re e1, im e0, im e1).  Built in double, rounded to float.
void ftc_twiddle_tables(int R0, std::vector<float>& tin, std::vector<float>& tout) {
    const int64_t M = int64_t(R0) * 4096;
    const double sc = 1.0 / std::sqrt(double(R0));
    tin.assign(size_t(R0) * 256 * 2, 0.f);
    tout.assign(size_t(R0) * 2 * 256 * 4, 0.f);
    for (int k0 = 0; k0 < R0; ++k0)
        for (int t = 0; t < 256; ++t) {
            const int64_t n = 1024 * (t >> 6) + (t & 63);
            const cd w = W(M, int64_t(k0) * n);
            tin[(size_t(k0) * 256 + t) * 2] = float(w.r * sc);
            tin[(size_t(k0) * 256 + t) * 2 + 1] = float(w.i * sc);
            const int hf = t >> 7, wq = (t >> 5) & 3, r = (t & 31) >> 2, q = t & 3;
            for (int b = 0; b < 2; ++b) {
                const int kap = b ? 63 - (8 * wq + r) : 8 * wq + r;
                const int64_t n0p = 64 * kap + 32 * hf + 2 * q;
                float* o = &tout[((size_t(k0) * 2 + b) * 256 + t) * 4];
                for (int e = 0; e < 2; ++e) {
                    const cd v = W(M, int64_t(k0) * (n0p + e));
                    o[e] = float(v.r);
                    o[2 + e] = float(v.i);
                }
            }
        }
}

// The real-embedded DFT matrix of an outer pass on the tensor cores
// (otc.cuh), F[o][n] = W_R^(o n) / sqrt(R) for the pass's outputs o and
// inputs n (pass A: o = k0, n = n0 < NIN; pass C: o = n0 < NOUT, n = k0), as
// the B operand of Otc<R, MODE>: row 2 o + part (0 real, 1 imaginary part of
// output o), K index 2 n + pin (0 real, 1 imaginary part of input n),
// K-major without swizzle; padding rows and K indices zero.
template <int R, int MODE, bool FULL = false>
std::vector<uint16_t> build_otc_fmat(int dtype) {
    using C = Otc<R, MODE, FULL>;
    std::vector<uint16_t> v(C::BBYTES / 2, 0);
    const double sc = 1.0 / std::sqrt(double(R));
    for (int o = 0; o < C::NOUT; ++o)
        for (int part = 0; part < 2; ++part) {
            const int row = 2 * o + part;
            for (int n = 0; n < C::NIN; ++n) {
                cd w = W(R, int64_t(o) * n);
                w = {w.r * sc, w.i * sc};
                for (int pin = 0; pin < 2; ++pin) {
                    const int k = 2 * n + pin;
                    const size_t off = size_t(row / 8) * C::SBO + size_t(k / 8) * C::LBO + size_t(row % 8) * 16 +
                                       size_t(k % 8) * 2;
                    v[off / 2] = to_bits(embed(w, part, pin), dtype);
                }
            }
        }
    return v;
}

// The outer-pass matrices a multi-pass plan with 4096-point sub-rows uses:
// pass A and pass C over the outermost factor (R0, or RA of a two-level
// factor) and, for two levels, the in-place 64-point stages.
struct OtcTables {
    std::vector<uint16_t> fa, fc, fa2, fc2;
    // two levels: W_(64 RA)^(n_b k_a) / sqrt(RA) as packed pairs (re, re', im,
    // im'): pass A's [k_a < RA/2][n_b] (pairs k_a, k_a + RA/2), then pass C's
    // [k_a][n_b / 2] (pairs n_b, n_b + 1)
    std::vector<float> tw2;
};

template <int R>
void otc_outer(OtcTables& t, int dtype) {
    t.fa = build_otc_fmat<R, 0>(dtype);
    t.fc = build_otc_fmat<R, 3>(dtype);
}

template <int R>
void otc_outer_full(OtcTables& t, int dtype) {
    t.fa = build_otc_fmat<R, 0, true>(dtype);
    t.fc = build_otc_fmat<R, 3, true>(dtype);
}

OtcTables build_otc_tables(int R, bool two_level, int dtype, bool full = false) {
    OtcTables t;
    if (full) {  // circular plans: every input and output row of the outer factor
        switch (R) {
            case 2: otc_outer_full<2>(t, dtype); break;
            case 4: otc_outer_full<4>(t, dtype); break;
            case 8: otc_outer_full<8>(t, dtype); break;
            case 16: otc_outer_full<16>(t, dtype); break;
            case 32: otc_outer_full<32>(t, dtype); break;
            case 64: otc_outer_full<64>(t, dtype); break;
        }
        return t;
    }
    switch (R) {
        case 4: otc_outer<4>(t, dtype); break;
        case 8: otc_outer<8>(t, dtype); break;
        case 16: otc_outer<16>(t, dtype); break;
        case 32: otc_outer<32>(t, dtype); break;
        case 64: otc_outer<64>(t, dtype); break;
        case 128: otc_outer<128>(t, dtype); break;
    }
    if (two_level) {
        t.fa2 = build_otc_fmat<64, 1>(dtype);
        t.fc2 = build_otc_fmat<64, 2>(dtype);
        const double sc = 1.0 / std::sqrt(double(R));
        auto tw = [&](int ka, int nb) {
            const cd w = W(64 * R, int64_t(nb) * ka);
            return cd{w.r * sc, w.i * sc};
        };
        auto put = [&](cd a, cd b) {
            t.tw2.push_back(float(a.r));
            t.tw2.push_back(float(b.r));
            t.tw2.push_back(float(a.i));
            t.tw2.push_back(float(b.i));
        };
        for (int kp = 0; kp < R / 2; ++kp)
            for (int nb = 0; nb < 64; ++nb) put(tw(kp, nb), tw(kp + R / 2, nb));
        for (int ka = 0; ka < R; ++ka)
            for (int nb = 0; nb < 64; nb += 2) put(tw(ka, nb), tw(ka, nb + 1));
    }
    return t;
}

template <typename T>
size_t append(std::vector<uint8_t>& blob, const std::vector<T>& v) {
    size_t off = (blob.size() + 255) & ~size_t(255);
    blob.resize(off + v.size() * sizeof(T));
    std::memcpy(blob.data() + off, v.data(), v.size() * sizeof(T));
    return off;
}

// ---- fused kernel dispatch
template <int DT, int R1, bool G>
cudaError_t launch_fused_t(const fftconv_plan_s* p, const void* u, const void* wi, const void* wo,
                           const void* kf, void* y, int64_t B, int64_t H, cudaStream_t st) {
    using C = FusedCfg<R1, G>;
    auto fn = fused_conv_kernel<DT, R1, G>;
    static PerDevice cache;  // per instantiation and device
    int blocks_per_sm = 0;
    cudaError_t e = prep_kernel(fn, C::SMEM_BYTES, C::THREADS, cache, &blocks_per_sm);
    if (e != cudaSuccess) return e;
    if (C::TSMEM && p->tb.outer_bytes > C::TAB_BYTES) return cudaErrorInvalidValue;
    if (C::FSMEM && p->tb.off_twf > C::TAB_BYTES) return cudaErrorInvalidValue;
    const int64_t groups = (B * H + C::RP - 1) / C::RP;
    int64_t grid = int64_t(p->num_sms) * blocks_per_sm;
    const int64_t need = (groups + C::GROUPS - 1) / C::GROUPS;
    if (grid > need) grid = need;
    FusedArgs args{static_cast<const uint16_t*>(u), static_cast<const uint16_t*>(wi),
                   static_cast<const uint16_t*>(wo), static_cast<const uint4*>(kf), static_cast<uint16_t*>(y),
                   int(B), int(H), p->tb, p->dev_err};
    fn<<<dim3(unsigned(grid)), dim3(C::THREADS), C::SMEM_BYTES, st>>>(args);
    return cudaGetLastError();
}

template <int DT, bool G>
cudaError_t launch_tc64_t(const fftconv_plan_s* p, const void* u, const void* wi, const void* wo,
                          const void* kf, void* y, int64_t B, int64_t H, cudaStream_t st) {
    auto fn = tc64_conv_kernel<DT, G>;
    static PerDevice cache;  // per instantiation and device
    int per_sm = 0;
    cudaError_t e = prep_kernel(fn, Tc64::SMEM, Tc64::THREADS, cache, &per_sm);
    if (e != cudaSuccess) return e;
    // one CTA per SM (its tensor-memory allocation takes all 512 columns);
    // work items are pairs of rows of one channel, two pipelines per CTA
    const int64_t items = (B + 1) / 2 * H;
    const int64_t need = (items + 1) / 2;
    const int64_t grid = need < p->num_sms ? need : p->num_sms;
    Tc64Args args{static_cast<const uint16_t*>(u), static_cast<const uint16_t*>(wi),
                  static_cast<const uint16_t*>(wo), static_cast<const uint8_t*>(kf), static_cast<uint16_t*>(y),
                  p->fmat, int(B), int(H), p->dev_err, int(p->info.N)};
    fn<<<dim3(unsigned(grid)), dim3(Tc64::THREADS), Tc64::SMEM, st>>>(args);
    return cudaGetLastError();
}

// N = R0 * 4096 (8192, 16384, 32768): the fused tensor-core kernel
// (ftc.cuh), one CTA per SM (all 512 tensor-memory columns).  FULL: the
// circular convolution of C = 16384 samples (R0 = 2, no zero half).
template <int DT, int R0, bool G, bool FULL = false>
cudaError_t launch_ftc_t(const fftconv_plan_s* p, const void* u, const void* wi, const void* wo,
                         const void* kf, void* y, int64_t B, int64_t H, cudaStream_t st) {
    using C = Ftc<R0, G, FULL>;
    auto fn = ftc_conv_kernel<DT, R0, G, FULL>;
    static PerDevice cache;  // per instantiation and device
    int per_sm = 0;
    cudaError_t e = prep_kernel(fn, C::SMEM, C::THREADS, cache, &per_sm);
    if (e != cudaSuccess) return e;
    // rows split over the two pipelines of a CTA; for R0 = 8 both work on each row
    const int64_t rows = B * H, need = C::SPLIT ? rows : (rows + 1) / 2;
    const int64_t grid = need < p->num_sms ? need : p->num_sms;
    FtcArgs args{static_cast<const uint16_t*>(u), static_cast<const uint16_t*>(wi),
                 static_cast<const uint16_t*>(wo), static_cast<const uint4*>(kf), static_cast<uint16_t*>(y),
                 p->fmat, p->ftw_in, p->ftw_out, int(B), int(H), p->dev_err,
                 (R0 == 4 && p->pairs_run == 1) ? 1 : 0};
    fn<<<dim3(unsigned(grid)), dim3(C::THREADS), C::SMEM, st>>>(args);
    return cudaGetLastError();
}

template <int DT, bool G>
cudaError_t launch_fused_r(const fftconv_plan_s* p, const void* u, const void* wi, const void* wo,
                           const void* kf, void* y, int64_t B, int64_t H, cudaStream_t st) {
    if (p->tc64) return launch_tc64_t<DT, G>(p, u, wi, wo, kf, y, B, H, st);
    switch (p->ftc) {
        case 2:
            return p->circular ? launch_ftc_t<DT, 2, G, true>(p, u, wi, wo, kf, y, B, H, st)
                               : launch_ftc_t<DT, 2, G>(p, u, wi, wo, kf, y, B, H, st);
        case 4: return launch_ftc_t<DT, 4, G>(p, u, wi, wo, kf, y, B, H, st);
        case 8: return launch_ftc_t<DT, 8, G>(p, u, wi, wo, kf, y, B, H, st);
    }
    switch (p->R1) {
        case 4: return launch_fused_t<DT, 4, G>(p, u, wi, wo, kf, y, B, H, st);
        case 8: return launch_fused_t<DT, 8, G>(p, u, wi, wo, kf, y, B, H, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fused(const fftconv_plan_s* p, const void* u, const void* wi, const void* wo,
                         const void* kf, void* y, int64_t B, int64_t H, cudaStream_t st) {
    const bool gated = wi != nullptr;
    if (p->info.dtype == FFTCONV_F16)
        return gated ? launch_fused_r<0, true>(p, u, wi, wo, kf, y, B, H, st)
                     : launch_fused_r<0, false>(p, u, wi, wo, kf, y, B, H, st);
    return gated ? launch_fused_r<1, true>(p, u, wi, wo, kf, y, B, H, st)
                 : launch_fused_r<1, false>(p, u, wi, wo, kf, y, B, H, st);
}

// ---- multi-pass dispatch (T: the intermediate, B*H*N*4 bytes)
cudaError_t launch_multipass(const fftconv_plan_s* p, const void* u, const void* wi, const void* wo,
                             const void* kf, void* y, void* T, int64_t B, int64_t H, cudaStream_t st) {
    MPArgs args{static_cast<const uint16_t*>(u), static_cast<const uint16_t*>(wi),
                static_cast<const uint16_t*>(wo), static_cast<const uint4*>(kf), static_cast<uint16_t*>(y),
                static_cast<uint32_t*>(T), int(B), int(H), p->R0, p->mp, p->dev_err,
                p->zbits, 1, p->pairs_run, p->plist, p->zcbits};
    const bool gated = wi != nullptr;
    if (p->circular) return launch_mp_l4k_circular(p, args, B * H, gated, st);
    if (p->zbits) {  // frequency-sparse plan with pairs of sub-rows to skip
        if (p->mp2) return launch_mp_l4k_2level_sparse(p, args, B * H, gated, st);
        return p->mpL == kMpLtc ? launch_mp_l4k_sparse(p, args, B * H, gated, st)
                                : launch_mp_l16k_sparse(p, args, B * H, gated, st);
    }
    if (p->mp2) return launch_mp_l4k_2level(p, args, B * H, gated, st);
    return p->mpL == kMpLtc ? launch_mp_l4k(p, args, B * H, gated, st) : launch_mp_l16k(p, args, B * H, gated, st);
}

}  // namespace

namespace {

// Frequency-sparse skipping on the multi-pass path.  Sub-row k0 of pass B
// holds the bins whose leading digits (r_1, or r_1 + RA r_2 for a two-level
// outer factor) make up k0; it is all zero when one of those digits is out of
// its band or an inner axis keeps nothing.  Pass B's pair (k0, R0 - k0) (pair
// 0: sub-rows 0 and R0/2) is skipped when both of its sub-rows are; then no
// pass reads or writes its sub-rows.  Outputs: the pairs that run, and the
// dead bits per sub-row ([RA][2] words for two levels, [1][2] otherwise).
struct SparseTables {
    std::vector<uint16_t> plist;
    std::vector<unsigned long long> zbits;
    unsigned long long zero[2] = {0ull, 0ull};  // bit k0 (one level): every bin of sub-row k0 is dropped
    bool any_skipped = false;
};

SparseTables sparse_tables(const fftconv_plan_info_t& info, const int32_t* band, int R0, bool two_level) {
    const int nlead = two_level ? 2 : 1;
    bool inner_empty = false;
    for (int j = nlead; j < info.order; ++j) inner_empty |= band[j] == 0;
    auto out_of_band = [&](int d, int j) {
        const int Mj = info.factors[j];
        return std::min(d, Mj - d) >= band[j];
    };
    std::vector<char> zero_sub(size_t(R0), 0);
    for (int k0 = 0; k0 < R0; ++k0) {
        bool z = inner_empty;
        if (two_level) {
            const int RA = info.factors[0];
            z |= out_of_band(k0 % RA, 0) || out_of_band(k0 / RA, 1);
        } else {
            z |= out_of_band(k0, 0);
        }
        zero_sub[size_t(k0)] = z;
    }
    SparseTables t;
    if (!two_level)
        for (int k0 = 0; k0 < R0; ++k0)
            if (zero_sub[size_t(k0)]) t.zero[k0 >> 6] |= 1ull << (k0 & 63);
    std::vector<char> dead(size_t(R0), 0);
    for (int pr = 0; pr < R0 / 2; ++pr) {
        const int a = pr, b = pr ? R0 - pr : R0 / 2;
        if (zero_sub[size_t(a)] && zero_sub[size_t(b)]) {
            dead[size_t(a)] = dead[size_t(b)] = 1;
            t.any_skipped = true;
        } else {
            t.plist.push_back(uint16_t(pr));
        }
    }
    const int groups = two_level ? info.factors[0] : 1;
    t.zbits.assign(size_t(groups) * 2, 0ull);
    for (int k0 = 0; k0 < R0; ++k0) {
        if (!dead[size_t(k0)]) continue;
        const int g = two_level ? k0 % groups : 0, bit = two_level ? k0 / groups : k0;  // bit < 128
        t.zbits[size_t(g) * 2 + size_t(bit >> 6)] |= 1ull << (bit & 63);
    }
    return t;
}

// The fused tensor-core kernel at N = 16384 (outer factor R0 = 4) runs its
// row as the sub-row pairs (1, 3) and (0, 2); pair (1, 3) is skipped when
// both of its sub-rows are dead, pair (0, 2) always runs (it writes the row).
// Returns the pairs that run out of R0 / 2 (R0 = 2 and 8: all of them).
int ftc_pairs_run(const fftconv_plan_info_t& info, const int32_t* band, bool sparse) {
    const int R0 = info.factors[0];
    if (!sparse || R0 != 4) return R0 / 2;
    const SparseTables t = sparse_tables(info, band, R0, false);
    const bool pair1 = std::find(t.plist.begin(), t.plist.end(), uint16_t(1)) != t.plist.end();
    return pair1 ? 2 : 1;
}

fftconv_status_t plan_create_impl(fftconv_plan_t* out, int64_t N, fftconv_dtype_t dtype, int order,
                                  const int32_t* band, int nband, bool circular = false) {
    if (!out) return FFTCONV_ERR_INVALID;
    *out = nullptr;
    // a band pattern is defined over the digits of an N-point transform: rows
    // shorter than 4096 keep their own factorization R1 x 16 x 16 then
    if (band && order == 0 && N < 4096) order = 3;
    fftconv_plan_info_t info;
    fftconv_status_t st = circular ? fftconv_circular_query(N, dtype, &info) : fftconv_plan_query(N, dtype, order, &info);
    if (st != FFTCONV_OK) return st;
    if (band) {
        if (nband != info.order) return FFTCONV_ERR_INVALID;
        for (int j = 0; j < nband; ++j)
            if (band[j] < 0) return FFTCONV_ERR_INVALID;
    }
    fftconv_plan_s* p = new (std::nothrow) fftconv_plan_s();
    if (!p) return FFTCONV_ERR_ALLOC;
    p->info = info;
    p->circular = circular;
    for (int j = 0; j < info.order; ++j) {
        const int32_t full = info.factors[j] / 2 + 1;  // keeps every digit value
        p->band[j] = band ? std::min(band[j], full) : full;
        p->sparse |= p->band[j] < full;
    }
    p->R1 = info.factors[0];
    const bool multi = info.path == FFTCONV_PATH_MULTIPASS;
    p->R0 = multi ? info.factors[0] : 1;
    p->R1 = multi ? kMpR1 : info.factors[0];
    p->tc64 = info.order == 2;  // 4096 = 64 x 64 (N = 1024, 2048 zero-padded to it)
    p->ftc = (info.path == FFTCONV_PATH_FUSED && info.order == 3 && info.factors[1] == 64) ? info.factors[0] : 0;
    p->mp2 = multi && info.order == 4 && info.factors[3] == 64;
    if (p->mp2) p->R0 = info.factors[0] * 64;  // the sub-row count of pass B
    p->mpL = multi ? ((info.order == 3 || p->mp2) ? kMpLtc : kMpL) : 0;
    const bool need_fmat = p->tc64 || p->ftc || p->mpL == kMpLtc;
    HostTables T = (p->tc64 || p->ftc) ? HostTables{} : build_fused_tables(p->R1, dtype);
    std::vector<uint32_t> fmat;
    if (need_fmat) fmat = build_tc64_fmat(dtype);
    HostTables T0;
    std::vector<uint32_t> ofull;
    if (multi && !circular) {  // the warp-level outer passes (frequency-sparse and order-4 plans)
        T0 = build_fused_tables(p->mp2 ? info.factors[0] : p->R0, dtype);  // fragments of the outermost factor
        ofull = build_full_frags(kMpR1, dtype);
    }
    std::vector<uint8_t> blob;
    const size_t o_err = append(blob, std::vector<int>(64, 0));
    const size_t o_lf = append(blob, T.lf), o_rf = append(blob, T.rf), o_tw = append(blob, T.tw);
    const size_t o_of = append(blob, T.of), o_oi = append(blob, T.oi);
    const size_t o_twf = append(blob, T.twf), o_twi = append(blob, T.twi);
    const size_t outer_end = o_twi + T.twi.size() * sizeof(float);
    const size_t o_fmat = need_fmat ? append(blob, fmat) : 0;
    std::vector<float> ftin, ftout;
    if (p->ftc) ftc_twiddle_tables(p->ftc, ftin, ftout);
    const size_t o_ftin = p->ftc ? append(blob, ftin) : 0, o_ftout = p->ftc ? append(blob, ftout) : 0;
    const bool otc = p->mpL == kMpLtc;
    OtcTables ot;
    if (otc) ot = build_otc_tables(p->mp2 ? info.factors[0] : p->R0, p->mp2, dtype, circular);
    const size_t o_tfa = otc ? append(blob, ot.fa) : 0, o_tfc = otc ? append(blob, ot.fc) : 0;
    const size_t o_tfa2 = (otc && p->mp2) ? append(blob, ot.fa2) : 0, o_tfc2 = (otc && p->mp2) ? append(blob, ot.fc2) : 0;
    const size_t o_ttw2 = (otc && p->mp2) ? append(blob, ot.tw2) : 0;
    size_t o_ofa = 0, o_oic = 0, o_ofull = 0;
    if (multi && !circular) {
        o_ofa = append(blob, T0.of);
        o_oic = append(blob, T0.oi);
        o_ofull = append(blob, ofull);
    }
    SparseTables sp;
    size_t o_plist = 0, o_zbits = 0, o_zc = 0;
    p->pairs_run = multi ? p->R0 / 2 : (p->ftc ? ftc_pairs_run(info, p->band, p->sparse) : 0);
    if (multi && p->sparse) {
        sp = sparse_tables(info, p->band, p->R0, p->mp2);
        if (sp.any_skipped) {
            p->pairs_run = int(sp.plist.size());
            if (sp.plist.empty()) sp.plist.push_back(0);  // nothing runs; keep the table non-empty
            o_plist = append(blob, sp.plist);
            o_zbits = append(blob, sp.zbits);
            if (!p->mp2) {  // the last pass reads zeros for every sub-row whose bins are all dropped
                p->zhost[0] = sp.zero[0];
                p->zhost[1] = sp.zero[1];
                o_zc = append(blob, std::vector<unsigned long long>{sp.zero[0], sp.zero[1]});
            }
        }
    }
    blob.resize((blob.size() + 255) & ~size_t(255));
    if (cudaMalloc(&p->dev, blob.size()) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return FFTCONV_ERR_ALLOC;
    }
    if (cudaMemcpy(p->dev, blob.data(), blob.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p->dev);
        delete p;
        return FFTCONV_ERR_CUDA;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p->dev);
        delete p;
        return FFTCONV_ERR_CUDA;
    }
    p->device = dev;
    uint8_t* d = static_cast<uint8_t*>(p->dev);
    p->dev_err = reinterpret_cast<int*>(d + o_err);
    if (need_fmat) p->fmat = reinterpret_cast<const uint32_t*>(d + o_fmat);
    if (p->ftc) {
        p->ftw_in = reinterpret_cast<const float2*>(d + o_ftin);
        p->ftw_out = reinterpret_cast<const float4*>(d + o_ftout);
    }
    if (otc) {
        p->otc_fa = d + o_tfa;
        p->otc_fc = d + o_tfc;
        if (p->mp2) {
            p->otc_fa2 = d + o_tfa2;
            p->otc_fc2 = d + o_tfc2;
            p->otc_tw2 = reinterpret_cast<const float4*>(d + o_ttw2);
        }
    }
    p->tb.lf = reinterpret_cast<const uint4*>(d + o_lf);
    p->tb.rf = reinterpret_cast<const uint4*>(d + o_rf);
    p->tb.tw = reinterpret_cast<const float4*>(d + o_tw);
    p->tb.outer = d + o_of;
    p->tb.outer_bytes = uint32_t(((outer_end - o_of) + 15) & ~size_t(15));
    p->tb.off_oi = uint32_t(o_oi - o_of);
    p->tb.off_twf = uint32_t(o_twf - o_of);
    p->tb.off_twi = uint32_t(o_twi - o_of);
    if (multi && !circular) {
        p->mp.lf = p->tb.lf;
        p->mp.rf = p->tb.rf;
        p->mp.tw = p->tb.tw;
        p->mp.of_a = reinterpret_cast<const uint4*>(d + o_ofa);
        p->mp.oi_c = reinterpret_cast<const uint4*>(d + o_oic);
        p->mp.ofull = reinterpret_cast<const uint4*>(d + o_ofull);
        p->mp.twf = reinterpret_cast<const float4*>(d + o_twf);
        p->mp.twi = reinterpret_cast<const float4*>(d + o_twi);
    }
    if (sp.any_skipped) {
        p->plist = reinterpret_cast<const uint16_t*>(d + o_plist);
        p->zbits = reinterpret_cast<const unsigned long long*>(d + o_zbits);
        if (o_zc) p->zcbits = reinterpret_cast<const unsigned long long*>(d + o_zc);
    }
    *out = p;
    return FFTCONV_OK;
}

}  // namespace

extern "C" fftconv_status_t fftconv_plan_create(fftconv_plan_t* out, int64_t N, fftconv_dtype_t dtype,
                                                int order) {
    return plan_create_impl(out, N, dtype, order, nullptr, 0);
}

extern "C" fftconv_status_t fftconv_plan_create_sparse(fftconv_plan_t* out, int64_t N, fftconv_dtype_t dtype,
                                                       int order, const int32_t* band, int nband) {
    if (!band) return FFTCONV_ERR_INVALID;
    return plan_create_impl(out, N, dtype, order, band, nband);
}

extern "C" fftconv_status_t fftconv_circular_query(int64_t C, fftconv_dtype_t dtype, fftconv_plan_info_t* info) {
    if (!info) return FFTCONV_ERR_INVALID;
    if (dtype != FFTCONV_F16 && dtype != FFTCONV_BF16) return FFTCONV_ERR_UNSUPPORTED;
    // M = C / 2 = R0 * 4096 with R0 = 2 .. 64, factored R0 x 64 x 64: C = 16384
    // on the fused tensor-core kernel (both blocks of the row in shared
    // memory), longer rows multi-pass with the outer passes over every row
    if (!is_pow2(C) || C < 16384 || C > (int64_t(1) << 19)) return FFTCONV_ERR_UNSUPPORTED;
    fftconv_plan_info_t q;
    std::memset(&q, 0, sizeof(q));
    q.N = C;
    q.M = C / 2;
    q.order = 3;
    q.factors[0] = int32_t(C / 8192);
    q.factors[1] = 64;
    q.factors[2] = 64;
    q.path = C == 16384 ? FFTCONV_PATH_FUSED : FFTCONV_PATH_MULTIPASS;
    q.dtype = dtype;
    q.kf_bytes_per_channel = int64_t(q.factors[0] / 2) * TcB::KFP * 16;
    q.workspace_bytes_per_row = C == 16384 ? 0 : 4 * q.M;  // 16-bit complex intermediate
    *info = q;
    return FFTCONV_OK;
}

extern "C" fftconv_status_t fftconv_plan_create_circular(fftconv_plan_t* out, int64_t C, fftconv_dtype_t dtype) {
    return plan_create_impl(out, C, dtype, 0, nullptr, 0, true);
}

extern "C" fftconv_status_t fftconv_sparse_query(int64_t N, fftconv_dtype_t dtype, int order, const int32_t* band,
                                                 int nband, int32_t* pairs_run, int32_t* pairs_total) {
    if (order == 0 && N < 4096) order = 3;  // as fftconv_plan_create_sparse
    fftconv_plan_info_t info;
    fftconv_status_t st = fftconv_plan_query(N, dtype, order, &info);
    if (st != FFTCONV_OK) return st;
    if (!band || nband != info.order) return FFTCONV_ERR_INVALID;
    int32_t b[8] = {};
    bool sparse = false;
    for (int j = 0; j < nband; ++j) {
        if (band[j] < 0) return FFTCONV_ERR_INVALID;
        const int32_t full = info.factors[j] / 2 + 1;
        b[j] = std::min(band[j], full);
        sparse |= b[j] < full;
    }
    int run = 0, total = 0;
    if (info.path == FFTCONV_PATH_MULTIPASS) {
        const bool two_level = info.order == 4 && info.factors[3] == 64;
        const int R0 = two_level ? info.factors[0] * 64 : info.factors[0];
        total = run = R0 / 2;
        if (sparse) run = int(sparse_tables(info, b, R0, two_level).plist.size());
    } else if (info.order == 3 && info.factors[1] == 64) {  // the fused tensor-core kernel
        total = info.factors[0] / 2;
        run = ftc_pairs_run(info, b, sparse);
    }
    if (pairs_run) *pairs_run = run;
    if (pairs_total) *pairs_total = total;
    return FFTCONV_OK;
}

extern "C" fftconv_status_t fftconv_plan_get_band(fftconv_plan_t plan, int32_t* band, int32_t* pairs_run,
                                                  int32_t* pairs_total) {
    if (!plan) return FFTCONV_ERR_INVALID;
    if (band)
        for (int j = 0; j < 8; ++j) band[j] = j < plan->info.order ? plan->band[j] : 0;
    const bool multi = plan->info.path == FFTCONV_PATH_MULTIPASS;
    const int total = multi ? plan->R0 / 2 : (plan->ftc ? plan->ftc / 2 : 0);
    if (pairs_run) *pairs_run = (multi || plan->ftc) ? plan->pairs_run : 0;
    if (pairs_total) *pairs_total = total;
    return FFTCONV_OK;
}

extern "C" fftconv_status_t fftconv_plan_destroy(fftconv_plan_t plan) {
    if (!plan) return FFTCONV_OK;
    cudaError_t e = cudaSuccess;
    for (cudaEvent_t& ev : plan->ev)
        if (ev) cudaEventDestroy(ev);
    if (plan->s_in) cudaStreamDestroy(plan->s_in);
    if (plan->s_out) cudaStreamDestroy(plan->s_out);
    if (plan->dev) e = cudaFree(plan->dev);
    delete plan;
    return e == cudaSuccess ? FFTCONV_OK : FFTCONV_ERR_CUDA;
}

extern "C" fftconv_status_t fftconv_plan_get_info(fftconv_plan_t plan, fftconv_plan_info_t* info) {
    if (!plan || !info) return FFTCONV_ERR_INVALID;
    *info = plan->info;
    return FFTCONV_OK;
}

extern "C" size_t fftconv_kf_bytes(fftconv_plan_t plan, int64_t H) {
    if (!plan || H < 0) return 0;
    return size_t(H) * size_t(plan->info.kf_bytes_per_channel);
}

extern "C" size_t fftconv_workspace_bytes(fftconv_plan_t plan, int64_t B, int64_t H) {
    if (!plan || B < 0 || H < 0) return 0;
    return size_t(B) * size_t(H) * size_t(plan->info.workspace_bytes_per_row);
}

extern "C" fftconv_status_t fftconv_set_workspace(fftconv_plan_t plan, void* dev_ptr, size_t bytes) {
    if (!plan) return FFTCONV_ERR_INVALID;
    if (dev_ptr && (reinterpret_cast<uintptr_t>(dev_ptr) & 15)) return FFTCONV_ERR_ALIGN;
    plan->workspace = dev_ptr;
    plan->workspace_bytes = dev_ptr ? bytes : 0;
    return FFTCONV_OK;
}

// --------------------------------------------------------------- kernel spectrum

namespace {

// buf[h][n] = k[h][n] for n < Nk, 0 up to 2N (Nk <= N: a kernel shorter than
// the transform, as for rows zero-padded to the transform length)
__global__ void kfft_init(const float* __restrict__ k, float2* __restrict__ buf, int64_t H, int64_t N,
                          int64_t Nk) {
    const int64_t L = 2 * N;
    int lgL = 0;
    while ((int64_t(1) << lgL) < L) ++lgL;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < H * L;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t h = i >> lgL, n = i & (L - 1);
        buf[i] = make_float2(n < Nk ? k[h * Nk + n] : 0.f, 0.f);
    }
}

// Stockham passes (self-sorting, out of place) of length-L DFTs with exponent
// sign -1, one per row, L = 2^lgL.  A pass of radix R with current span Ns
// (the product of the radices before it): element j = kk + Ns jj of the
// R-way split reads x[j + r L/R] (r < R), multiplies by W_{R Ns}^(kk r), takes
// the R-point DFT and writes y[kk + R Ns jj + q Ns] (q < R).  Powers of two
// throughout, so every index is a shift or a mask.
__global__ void kfft_pass2(const float2* __restrict__ x, float2* __restrict__ yv, int64_t H, int lgL, int lgNs) {
    const int64_t L = int64_t(1) << lgL, n = H << (lgL - 1);
    const int64_t Ns = int64_t(1) << lgNs;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t h = i >> (lgL - 1), j = i & ((L >> 1) - 1);
        const int64_t kk = j & (Ns - 1), jj = j >> lgNs;
        float wi, wr;  // kk / Ns is exact in float
        sincospif(-float(kk) / float(Ns), &wi, &wr);
        const float2* xr = x + (h << lgL);
        const float2 c0 = xr[j], c1 = xr[j + (L >> 1)];
        const float tr = c1.x * wr - c1.y * wi, ti = c1.x * wi + c1.y * wr;
        float2* yr = yv + (h << lgL) + kk + (jj << (lgNs + 1));
        yr[0] = make_float2(c0.x + tr, c0.y + ti);
        yr[Ns] = make_float2(c0.x - tr, c0.y - ti);
    }
}

__global__ void kfft_pass4(const float2* __restrict__ x, float2* __restrict__ yv, int64_t H, int lgL, int lgNs) {
    const int64_t L = int64_t(1) << lgL, Q = L >> 2, n = H << (lgL - 2);
    const int64_t Ns = int64_t(1) << lgNs;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t h = i >> (lgL - 2), j = i & (Q - 1);
        const int64_t kk = j & (Ns - 1), jj = j >> lgNs;
        const float2* xr = x + (h << lgL);
        float2 v0 = xr[j], v1 = xr[j + Q], v2 = xr[j + 2 * Q], v3 = xr[j + 3 * Q];
        float s1, c1;  // W_{4 Ns}^kk; kk / (2 Ns) is exact in float
        sincospif(-float(kk) / float(2 * Ns), &s1, &c1);
        const float c2 = c1 * c1 - s1 * s1, s2 = 2.f * c1 * s1;
        const float c3 = c2 * c1 - s2 * s1, s3 = c2 * s1 + s2 * c1;
        v1 = make_float2(v1.x * c1 - v1.y * s1, v1.x * s1 + v1.y * c1);
        v2 = make_float2(v2.x * c2 - v2.y * s2, v2.x * s2 + v2.y * c2);
        v3 = make_float2(v3.x * c3 - v3.y * s3, v3.x * s3 + v3.y * c3);
        const float2 a0 = make_float2(v0.x + v2.x, v0.y + v2.y), a1 = make_float2(v0.x - v2.x, v0.y - v2.y);
        const float2 a2 = make_float2(v1.x + v3.x, v1.y + v3.y);
        const float2 a3 = make_float2(v1.y - v3.y, v3.x - v1.x);  // -i (v1 - v3)
        float2* yr = yv + (h << lgL) + kk + (jj << (lgNs + 2));
        yr[0] = make_float2(a0.x + a2.x, a0.y + a2.y);
        yr[Ns] = make_float2(a1.x + a3.x, a1.y + a3.y);
        yr[2 * Ns] = make_float2(a0.x - a2.x, a0.y - a2.y);
        yr[3 * Ns] = make_float2(a1.x - a3.x, a1.y - a3.y);
    }
}

int ilog2(int64_t v) {
    int l = 0;
    while ((int64_t(1) << l) < v) ++l;
    return l;
}

int grid_for(int64_t work);

// DFT of every row of a [H][L] (L a power of two >= 2), ping-ponging between
// a and b; returns the buffer that holds the result.
float2* fft_rows(float2* a, float2* b, int64_t H, int64_t L, cudaStream_t st) {
    const int lgL = ilog2(L);
    int lgNs = 0;
    if (lgL & 1) {
        kfft_pass2<<<grid_for(H * L / 2), 256, 0, st>>>(a, b, H, lgL, 0);
        std::swap(a, b);
        lgNs = 1;
    }
    for (; lgNs < lgL; lgNs += 2) {
        kfft_pass4<<<grid_for(H * L / 4), 256, 0, st>>>(a, b, H, lgL, lgNs);
        std::swap(a, b);
    }
    return a;
}

__device__ __forceinline__ uint32_t pack_dt(float lo, float hi, int dtype) {
    return dtype == FFTCONV_F16 ? Op<0>::pack(lo, hi) : Op<1>::pack(lo, hi);
}

// The two coefficients of bin k of the decimation fold Z_y[k] = alpha Z[k] +
// beta conj Z[M-k], stored conjugated (alpha~, beta~) as 16-bit complex words,
// from the 2M-point spectrum K of the channel.
__device__ void fold_coeffs(const float2* __restrict__ Kh, int64_t k, int64_t M, int dtype, uint32_t* wa,
                            uint32_t* wb) {
    const float2 A = Kh[k], Bm = Kh[M - k];
    float st, ct;
    sincospif(float(k) / float(M), &st, &ct);  // theta = pi k / M (M a power of two: exact)
    const float Pr = 0.5f * (1.f - st), Pi = 0.5f * ct;
    const float Qr = 0.5f * (1.f + st), Qi = -0.5f * ct;
    const float Ar = A.x, Ai = A.y, Br = Bm.x, Bi = -Bm.y;  // B = conj K[M-k]
    const float PAr = Pr * Ar - Pi * Ai, PAi = Pr * Ai + Pi * Ar;
    const float QBr = Qr * Br - Qi * Bi, QBi = Qr * Bi + Qi * Br;
    const float Sr = PAr + QBr, Si = PAi + QBi, Dr = PAr - QBr, Di = PAi - QBi;
    // (i/2) W^k D with W^k = (cos, -sin)
    const float WDr = ct * Dr + st * Di, WDi = ct * Di - st * Dr;
    const float Xr = -0.5f * WDi, Xi = 0.5f * WDr;
    const float ar = 0.5f * Sr - Xr, ai = 0.5f * Si - Xi;
    const float br = 0.5f * Sr + Xr, bi = 0.5f * Si + Xi;
    *wa = pack_dt(ar, -ai, dtype);
    *wb = pack_dt(br, -bi, dtype);
}

// k_f: per (h, k0, k1, q, lane) two bins, each with alpha~ = conj(alpha)
// and beta~ = conj(beta) of the decimation fold, in the order the forward
// kernels hold the bins: thread (g, t) of the warp that transforms
// sub-problem k1 of sub-row k0 holds kappa' = (g + 8m) + 16(4nt + t), i.e.
// frequency k = k0 + R0*(k1 + R1*kappa').  R0 = 1 on the fused path.
__global__ void kfft_finalize(const float2* __restrict__ K, uint4* __restrict__ kf, int64_t H, int R0,
                              int R1, int dtype) {
    const int64_t M = int64_t(R0) * R1 * 256, L = 2 * M;
    const int64_t total = H * R0 * R1 * 4 * 32;
    for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
         idx += int64_t(gridDim.x) * blockDim.x) {
        const int lane = int(idx & 31);
        const int q = int((idx >> 5) & 3);
        const int64_t hk = idx >> 7;
        const int k1 = int(hk % R1);
        const int64_t hk0 = hk / R1;
        const int k0 = int(hk0 % R0);
        const int64_t h = hk0 / R0;
        const int g = lane >> 2, t = lane & 3;
        uint32_t words[4];
        for (int sl = 0; sl < 2; ++sl) {
            const int i = 2 * q + sl, m = i >> 2, nt = i & 3;
            const int64_t kap = (g + 8 * m) + 16 * (4 * nt + t);
            const int64_t k = k0 + int64_t(R0) * (k1 + int64_t(R1) * kap);
            fold_coeffs(K + h * L, k, M, dtype, &words[2 * sl], &words[2 * sl + 1]);
        }
        kf[idx] = make_uint4(words[0], words[1], words[2], words[3]);
    }
}

// k_f of the 64 x 64 path: per (h, chunk j < 9, warp w, half, lane) four
// words, in the order the fold of tc64_conv_kernel consumes them: half 0 =
// bins (s0, k2a), (s1, k2b); half 1 = bins (s0, k2b), (s1, k2a), where lane =
// 4r + q, k2a = 8w + r, k2b = 63 - k2a, s0 = 4j + q and s1 = 64 - s0 (j < 8),
// s0 = 32 for j = 8, q = 0.  Bin (s, k2) is k = s + 64 k2; padding bins
// (the copies of sub-problems 0 and 32, unused columns) are zero.
__global__ void kfft_finalize_tc64(const float2* __restrict__ K, uint4* __restrict__ kf, int64_t H, int dtype) {
    const int64_t M = 4096, L = 2 * M;
    const int64_t total = H * 9 * 4 * 2 * 32;
    for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
         idx += int64_t(gridDim.x) * blockDim.x) {
        const int lane = int(idx & 31), half = int((idx >> 5) & 1), w = int((idx >> 6) & 3);
        const int64_t hj = idx >> 8;
        const int j = int(hj % 9);
        const int64_t h = hj / 9;
        const int r = lane >> 2, q = lane & 3, k2a = 8 * w + r, k2b = 63 - k2a;
        int s0, s1;
        if (j < 8) {
            s0 = 4 * j + q;
            s1 = s0 == 0 ? -1 : 64 - s0;
        } else {
            s0 = q == 0 ? 32 : -1;
            s1 = -1;
        }
        const int sa[2] = {s0, s1}, ka[2] = {half ? k2b : k2a, half ? k2a : k2b};
        uint32_t words[4] = {0, 0, 0, 0};
        for (int i = 0; i < 2; ++i)
            if (sa[i] >= 0) fold_coeffs(K + h * L, sa[i] + 64 * int64_t(ka[i]), M, dtype, &words[2 * i], &words[2 * i + 1]);
        kf[idx] = make_uint4(words[0], words[1], words[2], words[3]);
    }
}

// k_f of the multi-pass path with 4096-point sub-rows (tcpass.cuh): per (h,
// pair p, chunk c < 17, warp w, half, lane) four words, in the order the fold
// of mp_pass_b_tc consumes them.  lane = 4r + q, k2a = 8w + r, k2b = 63 - k2a;
// half 0 = bins (s0, k2a), (s1, k2b), half 1 = bins (s0, k2b), (s1, k2a);
// bin (sub-row k0, s, k2) is k = k0 + R0 (s + 64 k2).
// - p > 0, c < 16: s0 = 4c + q of sub-row p, s1 = 63 - s0 of sub-row R0 - p.
// - p = 0, c < 9: sub-row 0 as the N = 4096 kernel (s0 = 4c + q, s1 = 64 - s0,
//   c = 8: s0 = 32 for q = 0); c >= 9: s0 = 4(c - 9) + q and s1 = 63 - s0,
//   both of sub-row R0/2.
// Bins that do not exist (copies, padding, chunk 16 of p > 0) are zero.
__global__ void kfft_finalize_tcmp(const float2* __restrict__ K, uint4* __restrict__ kf, int64_t H, int R0,
                                   int dtype) {
    const int64_t M = int64_t(R0) * 4096, L2 = 2 * M;
    const int pairs = R0 / 2;
    const int64_t total = H * pairs * TcB::KFP;
    for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
         idx += int64_t(gridDim.x) * blockDim.x) {
        const int lane = int(idx & 31), half = int((idx >> 5) & 1), w = int((idx >> 6) & 3);
        const int64_t hpc = idx >> 8;
        const int c = int(hpc % TcB::KF_CHUNKS);
        const int64_t hp = hpc / TcB::KF_CHUNKS;
        const int p = int(hp % pairs);
        const int64_t h = hp / pairs;
        const int r = lane >> 2, q = lane & 3, k2a = 8 * w + r, k2b = 63 - k2a;
        int s0 = -1, s1 = -1, kr0 = 0, kr1 = 0;  // sub-problems and their sub-rows
        if (p > 0) {
            if (c < 16) {
                s0 = 4 * c + q;
                s1 = 63 - s0;
                kr0 = p;
                kr1 = R0 - p;
            }
        } else if (c < 8) {
            s0 = 4 * c + q;
            s1 = s0 == 0 ? -1 : 64 - s0;
        } else if (c == 8) {
            s0 = q == 0 ? 32 : -1;
        } else {
            s0 = 4 * (c - 9) + q;
            s1 = 63 - s0;
            kr0 = kr1 = pairs;
        }
        const int sa[2] = {s0, s1}, ra[2] = {kr0, kr1}, ka[2] = {half ? k2b : k2a, half ? k2a : k2b};
        uint32_t words[4] = {0, 0, 0, 0};
        for (int i = 0; i < 2; ++i)
            if (sa[i] >= 0)
                fold_coeffs(K + h * L2, ra[i] + int64_t(R0) * (sa[i] + 64 * int64_t(ka[i])), M, dtype, &words[2 * i],
                            &words[2 * i + 1]);
        kf[idx] = make_uint4(words[0], words[1], words[2], words[3]);
    }
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int grid_for(int64_t work) {
    int64_t g = (work + 255) / 256;
    return int(g < 1 ? 1 : (g > 65535 * 16 ? 65535 * 16 : g));
}

}  // namespace

namespace {

// The band pattern of a frequency-sparse plan (factors outer first).
struct BandSpec {
    int n;
    int f[4];
    int b[4];
};

// Zero the bins f = 0..M of every channel's 2M-point spectrum that the band
// pattern drops: r = f mod M in mixed radix over the factors (outer digit
// first) keeps bin f when min(r_j, M_j - r_j) < band_j for every j.  Only
// these bins feed the decimation fold.
__global__ void kfft_band(float2* __restrict__ K, int64_t H, int64_t M, BandSpec bs) {
    const int64_t bins = M + 1;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < H * bins;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t h = i / bins, f = i % bins;
        int64_t r = f & (M - 1);
        bool keep = true;
        for (int j = 0; j < bs.n; ++j) {
            const int d = int(r % bs.f[j]);
            r /= bs.f[j];
            keep &= min(d, bs.f[j] - d) < bs.b[j];
        }
        if (!keep) K[h * 2 * M + f] = make_float2(0.f, 0.f);
    }
}

// conj of every spectrum value (the adjoint k_f: correlation instead of convolution)
__global__ void kfft_conj(float2* __restrict__ x, int64_t n) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
        x[i].y = -x[i].y;
}

fftconv_status_t kernel_fft_impl(fftconv_plan_t plan, const float* k, void* k_f, int64_t H,
                                 fftconv_stream_t stream, bool adjoint);

}  // namespace

extern "C" fftconv_status_t fftconv_kernel_fft(fftconv_plan_t plan, const float* k, void* k_f, int64_t H,
                                               fftconv_stream_t stream) {
    return kernel_fft_impl(plan, k, k_f, H, stream, false);
}

extern "C" fftconv_status_t fftconv_kernel_fft_adjoint(fftconv_plan_t plan, const float* k, void* k_f, int64_t H,
                                                       fftconv_stream_t stream) {
    return kernel_fft_impl(plan, k, k_f, H, stream, true);
}

namespace {

fftconv_status_t kernel_fft_impl(fftconv_plan_t plan, const float* k, void* k_f, int64_t H,
                                 fftconv_stream_t stream, bool adjoint) {
    if (!plan || H < 0 || wrong_device(plan)) return FFTCONV_ERR_INVALID;
    if (H == 0) return FFTCONV_OK;
    if (!k || !k_f) return FFTCONV_ERR_INVALID;
    if (misaligned(k) || misaligned(k_f)) return FFTCONV_ERR_ALIGN;
    // the transform length (4096 for rows of 1024 / 2048 zero-padded to it) and the kernel's length
    const int64_t N = plan->info.M, Nk = plan->info.N, L = 2 * N;
    if (overlap(k, size_t(H * Nk) * 4, k_f, fftconv_kf_bytes(plan, H))) return FFTCONV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float2* buf = nullptr;
    const size_t bytes = size_t(H) * size_t(L) * sizeof(float2);
    if (cudaMallocAsync(reinterpret_cast<void**>(&buf), 2 * bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return FFTCONV_ERR_ALLOC;
    }
    float2* a = buf;
    float2* b = buf + H * L;
    kfft_init<<<grid_for(H * L), 256, 0, st>>>(k, a, H, N, Nk);
    a = fft_rows(a, b, H, L, st);
    if (adjoint) kfft_conj<<<grid_for(H * L), 256, 0, st>>>(a, H * L);
    if (plan->sparse) {
        BandSpec bs{plan->info.order, {1, 1, 1, 1}, {1, 1, 1, 1}};
        for (int j = 0; j < plan->info.order && j < 4; ++j) {
            bs.f[j] = plan->info.factors[j];
            bs.b[j] = plan->band[j];
        }
        kfft_band<<<grid_for(H * (N + 1)), 256, 0, st>>>(a, H, N, bs);
    }
    if (plan->tc64)
        kfft_finalize_tc64<<<grid_for(H * 9 * 4 * 2 * 32), 256, 0, st>>>(a, static_cast<uint4*>(k_f), H,
                                                                           plan->info.dtype);
    else if (plan->mpL == kMpLtc || plan->ftc) {
        const int R0 = plan->ftc ? plan->ftc : plan->R0;
        kfft_finalize_tcmp<<<grid_for(H * (R0 / 2) * TcB::KFP), 256, 0, st>>>(a, static_cast<uint4*>(k_f), H, R0,
                                                                             plan->info.dtype);
    }
    else
        kfft_finalize<<<grid_for(H * plan->R0 * plan->R1 * 128), 256, 0, st>>>(
            a, static_cast<uint4*>(k_f), H, plan->R0, plan->R1, plan->info.dtype);
    cudaError_t e = cudaGetLastError();
    cudaFreeAsync(buf, st);
    return e == cudaSuccess ? FFTCONV_OK : FFTCONV_ERR_CUDA;
}

}  // namespace

// --------------------------------------------------------------- forward

static fftconv_status_t forward_impl(fftconv_plan_t plan, const void* u, const void* w_in,
                                     const void* w_out, const void* k_f, void* y, int64_t B, int64_t H,
                                     fftconv_stream_t stream, bool gated) {
    if (!plan || B < 0 || H < 0 || wrong_device(plan)) return FFTCONV_ERR_INVALID;
    if (B == 0 || H == 0) return FFTCONV_OK;
    if (!u || !k_f || !y || (gated && (!w_in || !w_out))) return FFTCONV_ERR_INVALID;
    if (misaligned(u) || misaligned(k_f) || misaligned(y) || (gated && (misaligned(w_in) || misaligned(w_out))))
        return FFTCONV_ERR_ALIGN;
    if (too_many_rows(B, H)) return FFTCONV_ERR_UNSUPPORTED;
    const size_t nb = size_t(B) * size_t(H) * size_t(plan->info.N) * 2;
    const size_t kb = fftconv_kf_bytes(plan, H);
    if (overlap(y, nb, u, nb) || overlap(y, nb, k_f, kb) ||
        (gated && (overlap(y, nb, w_in, nb) || overlap(y, nb, w_out, nb))))
        return FFTCONV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (plan->info.path == FFTCONV_PATH_MULTIPASS) {
        const size_t need = fftconv_workspace_bytes(plan, B, H);
        if (!plan->workspace || plan->workspace_bytes < need) return FFTCONV_ERR_WORKSPACE;
        const size_t nbw = need;
        if (overlap(plan->workspace, nbw, u, nb) || overlap(plan->workspace, nbw, y, nb) ||
            overlap(plan->workspace, nbw, k_f, kb) ||
            (gated && (overlap(plan->workspace, nbw, w_in, nb) || overlap(plan->workspace, nbw, w_out, nb))))
            return FFTCONV_ERR_INVALID;
        e = launch_multipass(plan, u, gated ? w_in : nullptr, gated ? w_out : nullptr, k_f, y, plan->workspace, B,
                             H, st);
    } else {
        e = launch_fused(plan, u, gated ? w_in : nullptr, gated ? w_out : nullptr, k_f, y, B, H, st);
    }
    if (e != cudaSuccess) return FFTCONV_ERR_CUDA;
    return FFTCONV_OK;
}

extern "C" fftconv_status_t fftconv_forward(fftconv_plan_t plan, const void* u, const void* k_f, void* y,
                                            int64_t B, int64_t H, fftconv_stream_t stream) {
    return forward_impl(plan, u, nullptr, nullptr, k_f, y, B, H, stream, false);
}

extern "C" fftconv_status_t fftconv_forward_gated(fftconv_plan_t plan, const void* u, const void* w_in,
                                                  const void* w_out, const void* k_f, void* y, int64_t B,
                                                  int64_t H, fftconv_stream_t stream) {
    return forward_impl(plan, u, w_in, w_out, k_f, y, B, H, stream, true);
}

extern "C" fftconv_status_t fftconv_device_status(fftconv_plan_t plan, fftconv_stream_t stream, int* out) {
    if (!plan || !out || wrong_device(plan)) return FFTCONV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, plan->dev_err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemsetAsync(plan->dev_err, 0, sizeof(int), st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return FFTCONV_ERR_CUDA;
    }
    *out = v;
    return FFTCONV_OK;
}

// --------------------------------------------------------------- failure-detection self-test
//
// One CTA waits, with the library's own bounded waits, on an mbarrier phase
// that nothing ever completes (no arrival, no copy): the wait must give up,
// record FFTCONV_ERR_TIMEOUT in the plan's error word and return, leaving the
// context usable.  No fault, trap or unbounded loop is involved.

namespace {

__global__ void selftest_wait_kernel(int* err, int sleep) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool done = sleep ? mbar_wait_sleep(&bar, 0, kWaitSleepLimit, kWaitHintNs)
                                : mbar_wait_bounded(&bar, 0, kWaitLimit);
        if (!done) atomicExch(err, FFTCONV_ERR_TIMEOUT);
    }
}

}  // namespace

extern "C" fftconv_status_t fftconv_selftest_wait(fftconv_plan_t plan, int sleep, fftconv_stream_t stream) {
    if (!plan || wrong_device(plan)) return FFTCONV_ERR_INVALID;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(plan->dev_err, sleep);
    return cudaGetLastError() == cudaSuccess ? FFTCONV_OK : FFTCONV_ERR_CUDA;
}

// --------------------------------------------------------------- backward
//
// Gradients of the convolution (FlashFFTConv page, section 3.4, "Kernel
// Fusion and Recomputation Strategies": the backward pass recomputes the
// transforms instead of storing them).  For y = conv(u, k) and the output
// gradient dy: du[j] = sum_{t>=j} dy[t] k[t-j] is the causal convolution
// machinery run with conj(rfft(k, 2N)) (fftconv_kernel_fft_adjoint); dk[h] =
// sum_b sum_{t>=i} dy_b[t] u_b[t-i] is the batch sum of the cross spectra
// DY_b conj(U_b), transformed back.

extern "C" fftconv_status_t fftconv_backward_du(fftconv_plan_t plan, const void* dy, const void* k_f_adj, void* du,
                                                int64_t B, int64_t H, fftconv_stream_t stream) {
    return forward_impl(plan, dy, nullptr, nullptr, k_f_adj, du, B, H, stream, false);
}

extern "C" fftconv_status_t fftconv_backward_du_gated(fftconv_plan_t plan, const void* dy, const void* w_in,
                                                      const void* w_out, const void* k_f_adj, void* du, int64_t B,
                                                      int64_t H, fftconv_stream_t stream) {
    // du = w_in * corr(w_out * dy, k): the gated kernels with the gates swapped
    return forward_impl(plan, dy, w_out, w_in, k_f_adj, du, B, H, stream, true);
}

namespace {

// The kernel gradient of whole channels for 2N <= 8192, in shared memory: one
// CTA per channel transforms each batch row g + i x (Stockham radix-4 /
// radix-2 passes between two shared buffers), adds the row's cross spectrum
// G conj X to per-thread accumulators (bins f = tid + 512 m), and after the
// batch transforms conj P once more and writes dk.  Only u, dy (and the gates)
// are read and dk written.
constexpr int kDkThreads = 512, kDkMaxL = 8192;

__device__ void smem_fft(float2* a, float2* b, int lgL, float2** out) {
    const int L = 1 << lgL;
    int lgNs = 0;
    if (lgL & 1) {  // radix-2 pass
        for (int j = threadIdx.x; j < L / 2; j += blockDim.x) {
            const float2 c0 = a[j], c1 = a[j + L / 2];
            b[2 * j] = make_float2(c0.x + c1.x, c0.y + c1.y);
            b[2 * j + 1] = make_float2(c0.x - c1.x, c0.y - c1.y);
        }
        __syncthreads();
        float2* t = a; a = b; b = t;
        lgNs = 1;
    }
    for (; lgNs < lgL; lgNs += 2) {
        const int Ns = 1 << lgNs, Q = L >> 2;
        for (int j = threadIdx.x; j < Q; j += blockDim.x) {
            const int kk = j & (Ns - 1), jj = j >> lgNs;
            float2 v0 = a[j], v1 = a[j + Q], v2 = a[j + 2 * Q], v3 = a[j + 3 * Q];
            float s1, c1;
            sincospif(-float(kk) / float(2 * Ns), &s1, &c1);
            const float c2 = c1 * c1 - s1 * s1, s2 = 2.f * c1 * s1;
            const float c3 = c2 * c1 - s2 * s1, s3 = c2 * s1 + s2 * c1;
            v1 = make_float2(v1.x * c1 - v1.y * s1, v1.x * s1 + v1.y * c1);
            v2 = make_float2(v2.x * c2 - v2.y * s2, v2.x * s2 + v2.y * c2);
            v3 = make_float2(v3.x * c3 - v3.y * s3, v3.x * s3 + v3.y * c3);
            const float2 a0 = make_float2(v0.x + v2.x, v0.y + v2.y), a1 = make_float2(v0.x - v2.x, v0.y - v2.y);
            const float2 a2 = make_float2(v1.x + v3.x, v1.y + v3.y);
            const float2 a3 = make_float2(v1.y - v3.y, v3.x - v1.x);
            float2* y = b + kk + (jj << (lgNs + 2));
            y[0] = make_float2(a0.x + a2.x, a0.y + a2.y);
            y[Ns] = make_float2(a1.x + a3.x, a1.y + a3.y);
            y[2 * Ns] = make_float2(a0.x - a2.x, a0.y - a2.y);
            y[3 * Ns] = make_float2(a1.x - a3.x, a1.y - a3.y);
        }
        __syncthreads();
        float2* t = a; a = b; b = t;
    }
    *out = a;
}

template <int DT>
__global__ void __launch_bounds__(kDkThreads, 1) dk_channel_smem(const uint16_t* __restrict__ u, const uint16_t* __restrict__ dy,
                                                                 const uint16_t* __restrict__ w_in,
                                                                 const uint16_t* __restrict__ w_out,
                                                                 float* __restrict__ dk, int64_t B, int64_t H, int lgN) {
    using O = Op<DT>;
    extern __shared__ __align__(16) float2 sbuf[];
    const int N = 1 << lgN, L = 2 * N, lgL = lgN + 1;
    constexpr int PER = kDkMaxL / kDkThreads;  // accumulated bins per thread (at most)
    for (int64_t h = blockIdx.x; h < H; h += gridDim.x) {
        float pr[PER], pi[PER];
        #pragma unroll
        for (int m = 0; m < PER; ++m) pr[m] = pi[m] = 0.f;
        for (int64_t b = 0; b < B; ++b) {
            const int64_t r = b * H + h;
            for (int n = threadIdx.x; n < L; n += blockDim.x) {
                float g = 0.f, x = 0.f;
                if (n < N) {
                    const int64_t j = r * N + n;
                    g = O::unpack(uint32_t(dy[j])).r;
                    x = O::unpack(uint32_t(u[j])).r;
                    if (w_out) g *= O::unpack(uint32_t(w_out[j])).r;
                    if (w_in) x *= O::unpack(uint32_t(w_in[j])).r;
                }
                sbuf[n] = make_float2(g, x);
            }
            __syncthreads();
            float2* z;
            smem_fft(sbuf, sbuf + L, lgL, &z);
            #pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int f = threadIdx.x + kDkThreads * m;
                if (f < L) {
                    const float2 a = z[f], c = z[(L - f) & (L - 1)];
                    const float gr = 0.5f * (a.x + c.x), gi = 0.5f * (a.y - c.y);
                    const float xr = 0.5f * (a.y + c.y), xi = -0.5f * (a.x - c.x);
                    pr[m] += gr * xr + gi * xi;
                    pi[m] += gi * xr - gr * xi;
                }
            }
            __syncthreads();  // the buffers are refilled by the next row
        }
        #pragma unroll
        for (int m = 0; m < PER; ++m) {
            const int f = threadIdx.x + kDkThreads * m;
            if (f < L) sbuf[f] = make_float2(pr[m], -pi[m]);
        }
        __syncthreads();
        float2* y;
        smem_fft(sbuf, sbuf + L, lgL, &y);
        const float sc = 1.f / float(L);
        for (int n = threadIdx.x; n < N; n += blockDim.x) dk[h * N + n] = y[n].x * sc;
        __syncthreads();
    }
}

// 2N in (8192, 65536]: the four-step form of dkgrad.cuh, L = L1 x 2048
constexpr int64_t kDk4MaxL = 65536;

template <int DT, int L1, bool G>
cudaError_t launch_dk4_t(const void* u, const void* dy, const void* w_in, const void* w_out, float* dk, int64_t B,
                         int64_t H, float2* R, cudaStream_t st) {
    const size_t smem = size_t(2) * kDkL2 * sizeof(float4) + (size_t(2) * kDkL2 + kDkTwEntries) * sizeof(float2);
    static PerDevice ready;  // per instantiation and device
    auto fn = dk_rows<DT, L1, G>;
    int* rd = ready.slot();
    if (!rd) return cudaErrorInvalidDevice;
    if (!*rd) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        *rd = 1;
    }
    const int64_t items = H * (L1 / 2);
    fn<<<unsigned(items < 65535 * 16 ? items : 65535 * 16), kDkRowThreads, smem, st>>>(
        static_cast<const uint16_t*>(u), static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(w_in),
        static_cast<const uint16_t*>(w_out), R, B, H, nullptr);
    dk_cols_inv<L1><<<grid_for(H * kDkL2), 256, 0, st>>>(R, dk, H);
    return cudaGetLastError();
}

// 2N in (64K, 4M]: the four-step form with the column transforms through HBM
// (A: rows x L float2, then R: H x L float2), L = L1 x 2048, L1 = 64 .. 2048
constexpr int64_t kDk4FaMaxL = int64_t(1) << 22;

template <int L1>
cudaError_t launch_dk4_rows_fa(const float2* A, float2* R, int64_t B, int64_t H, cudaStream_t st) {
    const size_t smem = size_t(2) * kDkL2 * sizeof(float4) + (size_t(2) * kDkL2 + kDkTwEntries) * sizeof(float2);
    static PerDevice ready;
    auto fn = dk_rows<0, L1, false, true>;
    int* rd = ready.slot();
    if (!rd) return cudaErrorInvalidDevice;
    if (!*rd) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        *rd = 1;
    }
    const int64_t items = H * (L1 / 2);
    fn<<<unsigned(items < 65535 * 16 ? items : 65535 * 16), kDkRowThreads, smem, st>>>(nullptr, nullptr, nullptr,
                                                                                          nullptr, R, B, H, A);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dk4_fa(const void* u, const void* dy, const void* w_in, const void* w_out, float* dk, int64_t B,
                          int64_t H, int64_t L, void* scratch, cudaStream_t st) {
    const int L1 = int(L / kDkL2), lgL1 = ilog2(L1);
    const int64_t rows = B * H;
    float2* A = static_cast<float2*>(scratch);
    float2* R = A + rows * L;
    const int lgTC = dk_col_lgtc(lgL1);
    const size_t csmem = size_t(2) * L1 * (size_t(1) << lgTC) * sizeof(float2);  // at most 128 KB
    static PerDevice ready[2];  // per gating and device (the column kernels' shared-memory opt-in)
    auto fwd = w_in ? dk_colfft_fwd<DT, true> : dk_colfft_fwd<DT, false>;
    int* rd = ready[w_in ? 1 : 0].slot();
    if (!rd) return cudaErrorInvalidDevice;
    if (!*rd) {
        cudaError_t e = cudaFuncSetAttribute(fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(dk_colfft_inv, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024);
        if (e != cudaSuccess) return e;
        *rd = 1;
    }
    const int64_t tiles_f = rows * (kDkL2 >> lgTC), tiles_i = H * (kDkL2 >> lgTC);
    fwd<<<unsigned(tiles_f < 65535 * 16 ? tiles_f : 65535 * 16), kDkColThreads, csmem, st>>>(
        static_cast<const uint16_t*>(u), static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(w_in),
        static_cast<const uint16_t*>(w_out), A, rows, lgL1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    switch (L1) {
        case 64: e = launch_dk4_rows_fa<64>(A, R, B, H, st); break;
        case 128: e = launch_dk4_rows_fa<128>(A, R, B, H, st); break;
        case 256: e = launch_dk4_rows_fa<256>(A, R, B, H, st); break;
        case 512: e = launch_dk4_rows_fa<512>(A, R, B, H, st); break;
        case 1024: e = launch_dk4_rows_fa<1024>(A, R, B, H, st); break;
        case 2048: e = launch_dk4_rows_fa<2048>(A, R, B, H, st); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    dk_colfft_inv<<<unsigned(tiles_i < 65535 * 16 ? tiles_i : 65535 * 16), kDkColThreads, csmem, st>>>(R, dk, H, lgL1);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dk4(const void* u, const void* dy, const void* w_in, const void* w_out, float* dk, int64_t B,
                       int64_t H, int64_t L, void* scratch, cudaStream_t st) {
    float2* R = static_cast<float2*>(scratch);
    const bool g = w_in != nullptr;
    switch (L / kDkL2) {
        case 8: return g ? launch_dk4_t<DT, 8, true>(u, dy, w_in, w_out, dk, B, H, R, st)
                         : launch_dk4_t<DT, 8, false>(u, dy, w_in, w_out, dk, B, H, R, st);
        case 16: return g ? launch_dk4_t<DT, 16, true>(u, dy, w_in, w_out, dk, B, H, R, st)
                          : launch_dk4_t<DT, 16, false>(u, dy, w_in, w_out, dk, B, H, R, st);
        case 32: return g ? launch_dk4_t<DT, 32, true>(u, dy, w_in, w_out, dk, B, H, R, st)
                          : launch_dk4_t<DT, 32, false>(u, dy, w_in, w_out, dk, B, H, R, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

extern "C" size_t fftconv_backward_dk_scratch_bytes(fftconv_plan_t plan, int64_t B, int64_t H) {
    if (!plan || B <= 0 || H <= 0) return 0;
    const int64_t L = 2 * plan->info.N;
    if (L <= kDkMaxL) return 0;  // whole channels in shared memory
    if (L <= kDk4MaxL) return size_t(H) * size_t(L) * sizeof(float2);
    return (size_t(B) * size_t(H) + size_t(H)) * size_t(L) * sizeof(float2);  // L <= kDk4FaMaxL (N <= 2^21)
}

extern "C" fftconv_status_t fftconv_backward_dk(fftconv_plan_t plan, const void* u, const void* dy, const void* w_in,
                                                const void* w_out, float* dk, int64_t B, int64_t H, void* scratch,
                                                size_t scratch_bytes, fftconv_stream_t stream) {
    if (!plan || B < 0 || H < 0 || wrong_device(plan)) return FFTCONV_ERR_INVALID;
    if (plan->sparse) return FFTCONV_ERR_UNSUPPORTED;  // the kernel gradient is not band-limited here
    if (plan->circular) return FFTCONV_ERR_UNSUPPORTED;  // the batch sum assumes causal (zero-padded) rows
    if (H == 0) return FFTCONV_OK;
    if (!dk || (w_in == nullptr) != (w_out == nullptr)) return FFTCONV_ERR_INVALID;
    const int64_t N = plan->info.N, L = 2 * N;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (misaligned(dk)) return FFTCONV_ERR_ALIGN;
    if (B == 0) {  // no rows: the gradient is zero
        return cudaMemsetAsync(dk, 0, size_t(H) * size_t(N) * 4, st) == cudaSuccess ? FFTCONV_OK : FFTCONV_ERR_CUDA;
    }
    if (!u || !dy) return FFTCONV_ERR_INVALID;
    if (too_many_rows(B, H)) return FFTCONV_ERR_UNSUPPORTED;
    if (misaligned(u) || misaligned(dy) || (w_in && (misaligned(w_in) || misaligned(w_out)))) return FFTCONV_ERR_ALIGN;
    const size_t nb = size_t(B) * size_t(H) * size_t(N) * 2, kb = size_t(H) * size_t(N) * 4;
    if (overlap(dk, kb, u, nb) || overlap(dk, kb, dy, nb) || (w_in && (overlap(dk, kb, w_in, nb) || overlap(dk, kb, w_out, nb))))
        return FFTCONV_ERR_INVALID;
    const size_t need = fftconv_backward_dk_scratch_bytes(plan, B, H);
    if (L <= kDkMaxL) {
        const size_t smem = size_t(2) * L * sizeof(float2);
        static PerDevice ready[2];  // per dtype and device
        auto fn = plan->info.dtype == FFTCONV_F16 ? dk_channel_smem<0> : dk_channel_smem<1>;
        const int di = plan->info.dtype == FFTCONV_F16 ? 0 : 1;
        int* rd = ready[di].slot();
        if (!rd) return FFTCONV_ERR_CUDA;
        if (!*rd) {
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(2 * kDkMaxL * sizeof(float2))) !=
                cudaSuccess) {
                cudaGetLastError();
                return FFTCONV_ERR_CUDA;
            }
            *rd = 1;
        }
        const int64_t grid = H < 65535 ? H : 65535;
        fn<<<unsigned(grid), kDkThreads, smem, st>>>(static_cast<const uint16_t*>(u), static_cast<const uint16_t*>(dy),
                                                     static_cast<const uint16_t*>(w_in),
                                                     static_cast<const uint16_t*>(w_out), dk, B, H, ilog2(N));
        return cudaGetLastError() == cudaSuccess ? FFTCONV_OK : FFTCONV_ERR_CUDA;
    }
    if (!scratch || scratch_bytes < need) return FFTCONV_ERR_WORKSPACE;
    if (misaligned(scratch)) return FFTCONV_ERR_ALIGN;
    if (L <= kDk4MaxL) {
        const cudaError_t e = plan->info.dtype == FFTCONV_F16
                                  ? launch_dk4<0>(u, dy, w_in, w_out, dk, B, H, L, scratch, st)
                                  : launch_dk4<1>(u, dy, w_in, w_out, dk, B, H, L, scratch, st);
        return e == cudaSuccess ? FFTCONV_OK : FFTCONV_ERR_CUDA;
    }
    // every plan length (2N <= 4M): the four-step form with the column transforms through HBM
    const cudaError_t e = plan->info.dtype == FFTCONV_F16
                              ? launch_dk4_fa<0>(u, dy, w_in, w_out, dk, B, H, L, scratch, st)
                              : launch_dk4_fa<1>(u, dy, w_in, w_out, dk, B, H, L, scratch, st);
    return e == cudaSuccess ? FFTCONV_OK : FFTCONV_ERR_CUDA;
}

// --------------------------------------------------------------- partial convolution
//
// Kernels with at most C = W/2 taps (FlashFFTConv page, "Architectural
// Extensions: Partial and Frequency-Sparse Convolutions"): the sequence of
// any length N (a multiple of C) runs as overlapping windows of W = 2C
// inputs, window w covering inputs [(w-1)C, (w+1)C) (zeros before the
// start); its causal convolution with the kernel is exact on window
// positions [C, 2C), i.e. outputs [wC, (w+1)C), which are kept.

namespace {

// windows of one [B][H][N] tensor: out[(b*nwin + w)*H + h][j] = in[b][h][(w-1)C + j] (0 before the start)
// (wrap: the part before the start is taken from the end of the row instead)
__global__ void partial_gather(const uint4* __restrict__ in, uint4* __restrict__ out, int64_t B, int64_t H,
                               int64_t N, int64_t C, int64_t nwin, bool wrap) {
    const int64_t W8 = (2 * C) / 8, C8 = C / 8, N8 = N / 8;  // 16-byte units (8 values)
    const int64_t total = B * nwin * H * W8;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t j = i % W8, r = i / W8, h = r % H, bw = r / H, w = bw % nwin, b = bw / nwin;
        const int64_t src = (w - 1) * C8 + j;  // 16-byte unit inside the row
        out[i] = src >= 0 ? in[(b * H + h) * N8 + src]
                          : (wrap ? in[(b * H + h) * N8 + src + N8] : make_uint4(0, 0, 0, 0));
    }
}

// kept outputs: y[b][h][wC + i] = yw[(b*nwin + w)*H + h][C + i]
__global__ void partial_scatter(const uint4* __restrict__ yw, uint4* __restrict__ y, int64_t B, int64_t H,
                                int64_t N, int64_t C, int64_t nwin) {
    const int64_t W8 = (2 * C) / 8, C8 = C / 8, N8 = N / 8;
    const int64_t total = B * H * N8;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t n = i % N8, r = i / N8, h = r % H, b = r / H, w = n / C8, c = n - w * C8;
        y[i] = yw[((b * nwin + w) * H + h) * W8 + C8 + c];
    }
}

struct PartialLayout {
    int64_t C, nwin;
    size_t buf, ws, total;  // one windowed tensor, the multi-pass intermediate, all
};

PartialLayout partial_layout(const fftconv_plan_s* p, int64_t B, int64_t H, int64_t N, bool gated) {
    PartialLayout l{};
    const int64_t W = p->info.N;
    l.C = W / 2;
    l.nwin = N / l.C;
    const size_t rows = size_t(B) * size_t(l.nwin) * size_t(H);
    l.buf = align256(rows * size_t(W) * 2);
    l.ws = p->info.path == FFTCONV_PATH_MULTIPASS ? align256(rows * size_t(W) * 4) : 0;
    l.total = l.buf * (gated ? 4 : 2) + l.ws;
    return l;
}

}  // namespace

extern "C" size_t fftconv_partial_scratch_bytes(fftconv_plan_t plan, int64_t B, int64_t H, int64_t N, int gated) {
    if (!plan || B <= 0 || H <= 0 || N <= 0) return 0;
    const int64_t C = plan->info.N / 2;
    if (N % C != 0) return 0;
    return partial_layout(plan, B, H, N, gated != 0).total;
}

namespace {

fftconv_status_t windowed_forward(fftconv_plan_t plan, const void* u, const void* w_in, const void* w_out,
                                  const void* k_f, void* y, int64_t B, int64_t H, int64_t N, void* scratch,
                                  size_t scratch_bytes, fftconv_stream_t stream, bool wrap);

}  // namespace

extern "C" fftconv_status_t fftconv_forward_partial(fftconv_plan_t plan, const void* u, const void* w_in,
                                                    const void* w_out, const void* k_f, void* y, int64_t B,
                                                    int64_t H, int64_t N, void* scratch, size_t scratch_bytes,
                                                    fftconv_stream_t stream) {
    return windowed_forward(plan, u, w_in, w_out, k_f, y, B, H, N, scratch, scratch_bytes, stream, false);
}

// Circular convolution of length C = W/2: y[t] = sum_j u[j] k[(t - j) mod C]
// equals outputs [C, 2C) of the causal convolution of [u, u] with [k, 0]
// (the first copy supplies the wrapped-around terms): one window of the
// partial form whose first half wraps instead of being zero.
extern "C" size_t fftconv_circular_scratch_bytes(fftconv_plan_t plan, int64_t B, int64_t H, int gated) {
    if (!plan) return 0;
    return fftconv_partial_scratch_bytes(plan, B, H, plan->info.N / 2, gated);
}

extern "C" fftconv_status_t fftconv_forward_circular(fftconv_plan_t plan, const void* u, const void* w_in,
                                                     const void* w_out, const void* k_f, void* y, int64_t B,
                                                     int64_t H, void* scratch, size_t scratch_bytes,
                                                     fftconv_stream_t stream) {
    if (!plan) return FFTCONV_ERR_INVALID;
    return windowed_forward(plan, u, w_in, w_out, k_f, y, B, H, plan->info.N / 2, scratch, scratch_bytes, stream,
                            true);
}

namespace {

fftconv_status_t windowed_forward(fftconv_plan_t plan, const void* u, const void* w_in, const void* w_out,
                                  const void* k_f, void* y, int64_t B, int64_t H, int64_t N, void* scratch,
                                  size_t scratch_bytes, fftconv_stream_t stream, bool wrap) {
    if (!plan || B < 0 || H < 0 || N < 0 || wrong_device(plan)) return FFTCONV_ERR_INVALID;
    if (plan->sparse) return FFTCONV_ERR_UNSUPPORTED;  // windows of a band-limited kernel are not defined here
    if (plan->circular) return FFTCONV_ERR_UNSUPPORTED;  // windows are causal convolutions
    if (B == 0 || H == 0 || N == 0) return FFTCONV_OK;
    if (!u || !k_f || !y || (w_in == nullptr) != (w_out == nullptr)) return FFTCONV_ERR_INVALID;
    const bool gated = w_in != nullptr;
    const int64_t C = plan->info.N / 2;
    if (N % C != 0) return FFTCONV_ERR_UNSUPPORTED;
    if (misaligned(u) || misaligned(k_f) || misaligned(y) || (gated && (misaligned(w_in) || misaligned(w_out))))
        return FFTCONV_ERR_ALIGN;
    const PartialLayout lay = partial_layout(plan, B, H, N, gated);
    if (too_many_rows(B, lay.nwin) || too_many_rows(B * lay.nwin, H)) return FFTCONV_ERR_UNSUPPORTED;
    const size_t nb = size_t(B) * size_t(H) * size_t(N) * 2;
    if (overlap(y, nb, u, nb) || (gated && (overlap(y, nb, w_in, nb) || overlap(y, nb, w_out, nb))))
        return FFTCONV_ERR_INVALID;
    if (!scratch || scratch_bytes < lay.total) return FFTCONV_ERR_WORKSPACE;
    if (misaligned(scratch)) return FFTCONV_ERR_ALIGN;
    if (overlap(scratch, lay.total, u, nb) || overlap(scratch, lay.total, y, nb)) return FFTCONV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* sb = static_cast<uint8_t*>(scratch);
    uint4* uw = reinterpret_cast<uint4*>(sb);
    uint4* yw = reinterpret_cast<uint4*>(sb + lay.buf);
    uint4* wiw = gated ? reinterpret_cast<uint4*>(sb + 2 * lay.buf) : nullptr;
    uint4* wow = gated ? reinterpret_cast<uint4*>(sb + 3 * lay.buf) : nullptr;
    void* ws = sb + lay.buf * (gated ? 4 : 2);
    const int64_t Bw = B * lay.nwin, units = Bw * H * (2 * C) / 8;
    partial_gather<<<grid_for(units), 256, 0, st>>>(static_cast<const uint4*>(u), uw, B, H, N, C, lay.nwin, wrap);
    if (gated) {
        partial_gather<<<grid_for(units), 256, 0, st>>>(static_cast<const uint4*>(w_in), wiw, B, H, N, C, lay.nwin,
                                                        wrap);
        partial_gather<<<grid_for(units), 256, 0, st>>>(static_cast<const uint4*>(w_out), wow, B, H, N, C, lay.nwin,
                                                        wrap);
    }
    cudaError_t e = plan->info.path == FFTCONV_PATH_MULTIPASS
                        ? launch_multipass(plan, uw, wiw, wow, k_f, yw, ws, Bw, H, st)
                        : launch_fused(plan, uw, wiw, wow, k_f, yw, Bw, H, st);
    if (e == cudaSuccess) {
        partial_scatter<<<grid_for(B * H * N / 8), 256, 0, st>>>(yw, static_cast<uint4*>(y), B, H, N, C, lay.nwin);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FFTCONV_ERR_CUDA;
    }
    return FFTCONV_OK;
}

}  // namespace

extern "C" const char* fftconv_status_string(fftconv_status_t s) {
    switch (s) {
        case FFTCONV_OK: return "ok";
        case FFTCONV_ERR_INVALID: return "invalid argument";
        case FFTCONV_ERR_UNSUPPORTED: return "unsupported length, order or dtype";
        case FFTCONV_ERR_ALIGN: return "pointer not 16-byte aligned";
        case FFTCONV_ERR_WORKSPACE: return "workspace missing or too small";
        case FFTCONV_ERR_CUDA: return "CUDA runtime error";
        case FFTCONV_ERR_ALLOC: return "device allocation failed";
        case FFTCONV_ERR_TIMEOUT: return "bounded on-device wait gave up";
    }
    return "unknown status";
}

extern "C" const char* fftconv_version(void) { return "0.1.0"; }

// --------------------------------------------------------------- no-allocation forward
//
// For callers that cannot allocate device memory: the multi-pass
// intermediate lives in this file-scope array instead of a caller workspace.
// Host code must not use the array's name as a pointer (it is a host-side
// stand-in); the device address is looked up once per device below.

static __device__ __align__(256) uint8_t g_static_scratch[FFTCONV_STATIC_SCRATCH_BYTES];

#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up the
// first time each device asks; nullptr on failure).
void* static_scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" fftconv_status_t fftconv_forward_noalloc(fftconv_plan_t plan, const void* u, const void* k_f,
                                                    void* y, int64_t B, int64_t H, fftconv_stream_t stream) {
    if (!plan || B < 0 || H < 0 || wrong_device(plan)) return FFTCONV_ERR_INVALID;
    if (B == 0 || H == 0) return FFTCONV_OK;
    if (!u || !k_f || !y) return FFTCONV_ERR_INVALID;
    if (misaligned(u) || misaligned(k_f) || misaligned(y)) return FFTCONV_ERR_ALIGN;
    if (too_many_rows(B, H)) return FFTCONV_ERR_UNSUPPORTED;
    const size_t nb = size_t(B) * size_t(H) * size_t(plan->info.N) * 2;
    const size_t kb = fftconv_kf_bytes(plan, H);
    if (overlap(y, nb, u, nb) || overlap(y, nb, k_f, kb)) return FFTCONV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (plan->info.path == FFTCONV_PATH_MULTIPASS) {
        if (fftconv_workspace_bytes(plan, B, H) > FFTCONV_STATIC_SCRATCH_BYTES) return FFTCONV_ERR_WORKSPACE;
        void* scratch = static_scratch_for_current_device();
        if (!scratch) return FFTCONV_ERR_CUDA;
        e = launch_multipass(plan, u, nullptr, nullptr, k_f, y, scratch, B, H, st);
    } else {
        e = launch_fused(plan, u, nullptr, nullptr, k_f, y, B, H, st);
    }
    return e == cudaSuccess ? FFTCONV_OK : FFTCONV_ERR_CUDA;
}

// --------------------------------------------------------------- host-buffer forward
//
// Rows that live in host memory pass through three device buffer sets in
// chunks; the copy of chunk c to the device (stream s_in), the convolution of
// chunk c - 1 (the caller's stream) and the copy back of chunk c - 2 (stream
// s_out) overlap.  Events order each buffer set's reuse: its inputs are
// overwritten only after the convolution that read them, its output only
// after the copy that drained it.

namespace {

constexpr int kHostSets = 3;
constexpr int64_t kHostChunks = 8;  // target number of chunks per call

struct HostChunks {
    bool by_b;       // chunks of whole batch entries; else (B = 1) ranges of channels
    int64_t per, n;  // batch entries (or channels) per chunk, number of chunks
    int64_t rows;    // rows of the largest chunk
};

HostChunks host_chunks(int64_t B, int64_t H) {
    HostChunks c{};
    c.by_b = B >= 2;
    const int64_t ext = c.by_b ? B : H;
    c.per = (ext + kHostChunks - 1) / kHostChunks;
    c.n = (ext + c.per - 1) / c.per;
    c.rows = c.by_b ? c.per * H : c.per;
    return c;
}

struct HostLayout {
    size_t buf, set, ws, total;  // one chunk buffer, one set, the multi-pass intermediate, all
};

HostLayout host_layout(const fftconv_plan_s* p, int64_t B, int64_t H, bool gated) {
    const HostChunks c = host_chunks(B, H);
    HostLayout l{};
    l.buf = align256(size_t(c.rows) * size_t(p->info.N) * 2);
    l.set = l.buf * (gated ? 4 : 2);
    l.ws = p->info.path == FFTCONV_PATH_MULTIPASS ? align256(size_t(c.rows) * size_t(p->info.N) * 4) : 0;
    l.total = kHostSets * l.set + l.ws;
    return l;
}

cudaError_t host_pipeline_init(fftconv_plan_s* p) {
    if (p->s_in) return cudaSuccess;
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    for (cudaEvent_t& ev : p->ev)
        if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

extern "C" size_t fftconv_host_scratch_bytes(fftconv_plan_t plan, int64_t B, int64_t H, int gated) {
    if (!plan || B <= 0 || H <= 0) return 0;
    return host_layout(plan, B, H, gated != 0).total;
}

extern "C" fftconv_status_t fftconv_forward_host(fftconv_plan_t plan, const void* u, const void* w_in,
                                                 const void* w_out, const void* k_f, void* y, int64_t B,
                                                 int64_t H, void* scratch, size_t scratch_bytes,
                                                 fftconv_stream_t stream) {
    if (!plan || B < 0 || H < 0 || wrong_device(plan)) return FFTCONV_ERR_INVALID;
    if (B == 0 || H == 0) return FFTCONV_OK;
    if (!u || !k_f || !y || (w_in == nullptr) != (w_out == nullptr)) return FFTCONV_ERR_INVALID;
    const bool gated = w_in != nullptr;
    if (misaligned(k_f)) return FFTCONV_ERR_ALIGN;
    if (too_many_rows(B, H)) return FFTCONV_ERR_UNSUPPORTED;
    const size_t nb = size_t(B) * size_t(H) * size_t(plan->info.N) * 2;
    if (overlap(y, nb, u, nb) || (gated && (overlap(y, nb, w_in, nb) || overlap(y, nb, w_out, nb))))
        return FFTCONV_ERR_INVALID;
    const HostLayout lay = host_layout(plan, B, H, gated);
    if (!scratch || scratch_bytes < lay.total) return FFTCONV_ERR_WORKSPACE;
    if (misaligned(scratch)) return FFTCONV_ERR_ALIGN;
    if (host_pipeline_init(plan) != cudaSuccess) {
        cudaGetLastError();
        return FFTCONV_ERR_CUDA;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaEvent_t ev_start = plan->ev[0], ev_end = plan->ev[1];
    cudaEvent_t* ev_in = plan->ev + 2;
    cudaEvent_t* ev_done = plan->ev + 2 + kHostSets;
    cudaEvent_t* ev_out = plan->ev + 2 + 2 * kHostSets;
    uint8_t* sb = static_cast<uint8_t*>(scratch);
    void* ws = sb + kHostSets * lay.set;
    const HostChunks c = host_chunks(B, H);
    const size_t row_bytes = size_t(plan->info.N) * 2;
    const size_t kfc = size_t(plan->info.kf_bytes_per_channel);
    auto hptr = [](const void* base, size_t off) { return static_cast<const uint8_t*>(base) + off; };
    cudaError_t e = cudaEventRecord(ev_start, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->s_in, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->s_out, ev_start, 0);
    for (int64_t ci = 0; ci < c.n && e == cudaSuccess; ++ci) {
        const int s = int(ci % kHostSets);
        // the chunk's rows are contiguous: batch entries [b0, b0 + nbc) x all
        // channels, or (B = 1) channels [h0, h0 + nhc)
        const int64_t b0 = c.by_b ? ci * c.per : 0, h0 = c.by_b ? 0 : ci * c.per;
        const int64_t nbc = c.by_b ? std::min(c.per, B - b0) : 1;
        const int64_t nhc = c.by_b ? H : std::min(c.per, H - h0);
        const size_t off = size_t(b0 * H + h0) * row_bytes, bytes = size_t(nbc * nhc) * row_bytes;
        uint8_t* du = sb + size_t(s) * lay.set;
        uint8_t* dy = du + lay.buf;
        uint8_t* dwi = gated ? dy + lay.buf : nullptr;
        uint8_t* dwo = gated ? dwi + lay.buf : nullptr;
        if (ci >= kHostSets) e = cudaStreamWaitEvent(plan->s_in, ev_done[s], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(du, hptr(u, off), bytes, cudaMemcpyHostToDevice, plan->s_in);
        if (gated && e == cudaSuccess)
            e = cudaMemcpyAsync(dwi, hptr(w_in, off), bytes, cudaMemcpyHostToDevice, plan->s_in);
        if (gated && e == cudaSuccess)
            e = cudaMemcpyAsync(dwo, hptr(w_out, off), bytes, cudaMemcpyHostToDevice, plan->s_in);
        if (e == cudaSuccess) e = cudaEventRecord(ev_in[s], plan->s_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_in[s], 0);
        if (e == cudaSuccess && ci >= kHostSets) e = cudaStreamWaitEvent(st, ev_out[s], 0);
        if (e != cudaSuccess) break;
        const void* kfp = hptr(k_f, size_t(h0) * kfc);
        e = plan->info.path == FFTCONV_PATH_MULTIPASS
                ? launch_multipass(plan, du, dwi, dwo, kfp, dy, ws, nbc, nhc, st)
                : launch_fused(plan, du, dwi, dwo, kfp, dy, nbc, nhc, st);
        if (e == cudaSuccess) e = cudaEventRecord(ev_done[s], st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->s_out, ev_done[s], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<uint8_t*>(y) + off, dy, bytes, cudaMemcpyDeviceToHost, plan->s_out);
        if (e == cudaSuccess) e = cudaEventRecord(ev_out[s], plan->s_out);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev_end, plan->s_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_end, 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FFTCONV_ERR_CUDA;
    }
    return FFTCONV_OK;
}
