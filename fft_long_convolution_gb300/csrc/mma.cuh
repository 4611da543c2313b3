// Warp-level tensor-core contractions and 16-bit complex packing.
//
// A complex number travels as one 32-bit word: the real part in the low
// 16 bits, the imaginary part in the high 16 bits (the order in which an
// interleaved real sequence x[2n], x[2n+1] sits in memory).  The same word is
// a pair of consecutive K-elements of an mma.sync operand fragment, which is
// how complex data enters the real-embedded DFT contractions.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace fftconv {

struct cpx {
    float r, i;
};

__device__ __forceinline__ cpx cmul(cpx a, cpx b) {
    return {a.r * b.r - a.i * b.i, a.r * b.i + a.i * b.r};
}

// Two complex numbers held as a real pair (r0, r1) and an imaginary pair
// (i0, i1) -- the layout of an mma accumulator's (c0, c1) and (c2, c3) --
// times two twiddles given as (wr0, wr1, wi0, wi1), with packed f32x2
// arithmetic.  Returns (re0, re1) in out.x/out.y and (im0, im1) in out.z/out.w.
__device__ __forceinline__ float4 cmul2_split(float r0, float r1, float i0, float i1, float4 w) {
    unsigned long long R, I, Wr, Wi, t, u, v, re, im;
    asm("mov.b64 %0, {%1, %2};" : "=l"(R) : "f"(r0), "f"(r1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(I) : "f"(i0), "f"(i1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(Wr) : "f"(w.x), "f"(w.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(Wi) : "f"(w.z), "f"(w.w));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(R), "l"(Wr));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(u) : "l"(I), "l"(Wi));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(re) : "l"(t), "l"(u));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(v) : "l"(R), "l"(Wi));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(im) : "l"(I), "l"(Wr), "l"(v));
    float4 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(re));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.z), "=f"(o.w) : "l"(im));
    return o;
}

// Operand-type traits: 16-bit packing, unpacking, packed product and the
// m16n8k16 / m16n8k8 contractions with float32 accumulation.
template <int DTYPE> struct Op;

// DTYPE 0: IEEE binary16
template <> struct Op<0> {
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    static __device__ __forceinline__ cpx unpack(uint32_t v) {
        float lo, hi;
        asm("{.reg .f16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;}"
            : "=f"(lo), "=f"(hi) : "r"(v));
        return {lo, hi};
    }
    static __device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
    static __device__ __forceinline__ void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                 uint32_t b1) {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ void mma8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
        asm(
            "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(b0));
    }
};

// DTYPE 1: bfloat16
template <> struct Op<1> {
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    static __device__ __forceinline__ cpx unpack(uint32_t v) {
        return {__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u)};
    }
    static __device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
    static __device__ __forceinline__ void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                 uint32_t b1) {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ void mma8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
        asm(
            "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(b0));
    }
};

// ---- shared-memory / async-copy helpers -----------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Wall-clock bound of every on-device wait: about one second (a poll can
// suspend for a system-dependent time, so a poll count alone does not bound
// the time).
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until phase `parity` of the barrier completes; gives up after `limit`
// polls or about kWaitNs, whichever comes first.  Returns true when the phase
// completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
    uint32_t addr = smem_u32(bar);
    uint64_t t0 = 0;
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{.reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, "
            "1, 0, p;}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
        if ((it & 63) == 0) {
            const uint64_t t = globaltimer_ns();
            if (it == 0) t0 = t;
            else if (t - t0 > kWaitNs) return false;
        }
    }
    return false;
}

// Bounded waits of the tensor-core kernels: polls that may each suspend for
// up to 2 us (at most about 2 s in total before the kernel reports a timeout).
constexpr uint32_t kWaitSleepLimit = 1u << 20, kWaitHintNs = 2000;

// Same, but each poll may suspend the thread for up to `hint_ns` nanoseconds
// until the phase completes, so waiting warps do not compete for issue slots.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t limit, uint32_t hint_ns) {
    uint32_t addr = smem_u32(bar);
    uint64_t t0 = 0;
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{.reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, "
            "1, 0, p;}"
            : "=r"(done)
            : "r"(addr), "r"(parity), "r"(hint_ns)
            : "memory");
        if (done) return true;
        if ((it & 63) == 0) {
            const uint64_t t = globaltimer_ns();
            if (it == 0) t0 = t;
            else if (t - t0 > kWaitNs) return false;
        }
    }
    return false;
}

// One-dimensional bulk copy global -> shared through the TMA engine,
// completing on `bar` with its byte count.  Addresses 16-byte aligned, size a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Three-dimensional tiled copy global -> shared through the TMA engine (the
// box of the tensor map at coordinates x, y, z, innermost first), completing
// on `bar` with its byte count.  x times the element size must be a multiple
// of 16 bytes; the destination is 128-byte aligned.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Hint the TMA engine to pull a contiguous range into L2 (no completion).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

}  // namespace fftconv
