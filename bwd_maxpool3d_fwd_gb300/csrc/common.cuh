// Device-side helpers shared by the pooling kernels: element types, the
// max/argmax comparison rule, window geometry and launch bookkeeping.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace mp3d {

// ---------------------------------------------------------------- types

enum Dtype { F32 = 0, F16 = 1, BF16 = 2 };

// Exact widening to float and round-to-nearest-even narrowing.
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// "v beats the running maximum m": larger, or a NaN against a number.
// Equal values (including +0 against -0) do not beat, so the first
// occurrence in scan order is kept.
__device__ __forceinline__ bool beats(float v, float m) {
    return (v != v) ? (m == m) : (v > m);
}

// ---------------------------------------------------------------- geometry

// Problem geometry as the kernels see it. Per-plane volumes are < 2^31, so
// in-plane offsets are 32-bit; plane counts and global offsets are 64-bit.
struct Geo {
    long long P;          // planes N*C
    int D, H, W;          // input extent
    int OD, OH, OW;       // output extent
    int kd, kh, kw;       // fixed window (unused when adaptive)
    int sd, sh, sw;
    int adaptive;         // 1: adaptive windows
    int vol;              // D*H*W
    int ovol;             // OD*OH*OW
    int pd, ph, pw;       // fixed windows: padding (0 unless padded)
    int dd, dh, dw;       // fixed windows: dilation (1 unless dilated)
};

// Window i along one axis: [start, end).
__device__ __forceinline__ int win_start(int i, int I, int O, int K, int S, bool adaptive) {
    return adaptive ? (int)(((long long)i * I) / O) : i * S;
}
__device__ __forceinline__ int win_end(int i, int I, int O, int K, int S, bool adaptive) {
    return adaptive ? (int)(((long long)(i + 1) * I + O - 1) / O) : i * S + K;
}

// Range [lo, hi] of windows along one axis that contain position x
// (empty when lo > hi).
__device__ __forceinline__ int cover_lo(int x, int I, int O, int K, int S, bool adaptive) {
    if (adaptive) return (int)(((long long)x * O) / I);
    return x < K ? 0 : (x - K) / S + 1;
}
__device__ __forceinline__ int cover_hi(int x, int I, int O, int K, int S, bool adaptive) {
    if (adaptive) return (int)(((long long)(x + 1) * O - 1) / I);
    int h = x / S;
    return h < O - 1 ? h : O - 1;
}

// ---------------------------------------------------------------- division
// Division of a non-negative int below 2^31 by a fixed divisor d >= 1 as a
// multiply-high and a shift (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994): with l = ceil(log2 d) and
// m = floor(2^32 * (2^l - d) / d) + 1, n / d = (mulhi(n, m) + n) >> l; the
// sum cannot overflow because mulhi(n, m) <= n < 2^31.
struct FastDiv {
    uint32_t d, m, l;
    FastDiv() : d(1), m(1), l(0) {}
    explicit FastDiv(uint32_t div) : d(div) {
        l = 0;
        while ((1ull << l) < div) ++l;
        m = (uint32_t)((((1ull << l) - div) << 32) / div + 1);
    }
    __host__ __device__ __forceinline__ int div(int n) const {
#ifdef __CUDA_ARCH__
        const uint32_t t = __umulhi((uint32_t)n, m);
#else
        const uint32_t t = (uint32_t)(((uint64_t)(uint32_t)n * m) >> 32);
#endif
        return (int)((t + (uint32_t)n) >> l);
    }
    __host__ __device__ __forceinline__ int mod(int n, int q) const { return n - q * (int)d; }
};

// ---------------------------------------------------------------- windows per axis
// Windows along one axis, fixed (K, S) or adaptive (I -> O), with the
// divisions done by multiply-shift. Adaptive products (o + 1) * I and
// (x + 1) * O must stay below 2^31 (checked by the launchers).
struct AxisMap {
    int I, O, K, S;
    int adaptive;
    int pad;      // fixed windows: padding before the first position (window o starts at o*S - pad)
    FastDiv fS;   // fixed: divide by S
    FastDiv fI;   // adaptive: divide by I
    FastDiv fO;   // adaptive: divide by O
    // Window o along this axis: [start(o), end(o)).
    __device__ __forceinline__ int start(int o) const { return adaptive ? fO.div(o * I) : o * S; }
    __device__ __forceinline__ int end(int o) const {
        return adaptive ? fO.div((o + 1) * I + O - 1) : o * S + K;
    }
    __device__ __forceinline__ int len(int o) const {
        return adaptive ? fO.div((o + 1) * I + O - 1) - fO.div(o * I) : K;
    }
    __device__ __forceinline__ int lo(int x) const {
        if (adaptive) return fI.div(x * O);
        return x < K ? 0 : fS.div(x - K) + 1;
    }
    __device__ __forceinline__ int hi(int x) const {
        if (adaptive) return fI.div((x + 1) * O - 1);
        const int h = fS.div(x);
        return h < O - 1 ? h : O - 1;
    }
    // Windows before o that also cover position start(o) + rel.
    __device__ __forceinline__ int earlier(int o, int rel) const {
        if (adaptive) return o - lo(start(o) + rel);
        const int e = fS.div(K - 1 - rel);
        return e < o ? e : o;
    }
};

// Host-side construction of an AxisMap.
inline AxisMap axis_map(int I, int O, int K, int S, bool adaptive, int pad = 0) {
    AxisMap a;
    a.I = I; a.O = O; a.K = K; a.S = S; a.adaptive = adaptive ? 1 : 0;
    a.pad = adaptive ? 0 : pad;
    a.fS = FastDiv((uint32_t)(S > 0 ? S : 1));
    a.fI = FastDiv((uint32_t)I);
    a.fO = FastDiv((uint32_t)O);
    return a;
}


// ---------------------------------------------------------------- vectors

// Element-wise access to a 16-byte vector of T.
template <typename T> struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
    union { uint4 u; T e[N]; };
};

// ------------------------------------------------------ order keys (16-bit)
// An order key of a 16-bit float: an unsigned 16-bit number whose order is
// the forward scan's preference among values: +0 and -0 share a key,
// negative values rank below positive ones by magnitude, and every NaN
// ranks above +inf (all NaNs one key).
// Two 16-bit values (one per half of w) -> their order keys, half by half.
// NANADD = 0x7FFF - (largest non-NaN magnitude): bit 15 of mag + NANADD is
// set exactly for NaN magnitudes.
template <unsigned NANADD>
__device__ __forceinline__ unsigned order_keys2(unsigned w) {
    const unsigned mag = w & 0x7FFF7FFFu;
    unsigned neg, nan;
    // prmt with selector nibbles 9 / B: each result byte is the sign of
    // byte 1 (low half) or byte 3 (high half), replicated
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(neg) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(nan) : "r"(mag + NANADD * 0x10001u));
    const unsigned up = 0x80008000u + mag, down = 0x80008000u - mag;   // no carry between halves
    return (down & neg) | (up & ~neg) | nan;
}

template <typename T> struct KeyConst;
template <> struct KeyConst<__half> { static constexpr unsigned nanadd = 0x7FFFu - 0x7C00u; };
template <> struct KeyConst<__nv_bfloat16> { static constexpr unsigned nanadd = 0x7FFFu - 0x7F80u; };

// ------------------------------------------------ packed pairs (16-bit)
// Two 16-bit values in one 32-bit word, compared lane by lane with set.gt on
// f16x2 / bf16x2 (a mask of 0xFFFF per lane where the first is greater).
// NaN never compares greater, so packed scans track NaN and infinities with
// a running x*0 + acc, which turns NaN once either was seen; the caller then
// recomputes with the exact scalar rule.
template <typename T> struct Pair;
template <> struct Pair<__half> {
    static __device__ __forceinline__ uint32_t gt(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("set.gt.u32.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
    static __device__ __forceinline__ uint32_t poison(uint32_t acc, uint32_t v) {
        uint32_t r;
        asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(0u), "r"(acc));
        return r;
    }
    static __device__ __forceinline__ bool is_poisoned(uint32_t acc) {
        return ((acc & 0x7FFFu) > 0x7C00u) || (((acc >> 16) & 0x7FFFu) > 0x7C00u);
    }
};
template <> struct Pair<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t gt(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
    static __device__ __forceinline__ uint32_t poison(uint32_t acc, uint32_t v) {
        uint32_t r;
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(0u), "r"(acc));
        return r;
    }
    static __device__ __forceinline__ bool is_poisoned(uint32_t acc) {
        return ((acc & 0x7FFFu) > 0x7F80u) || (((acc >> 16) & 0x7FFFu) > 0x7F80u);
    }
};

// Replace (mv, mc) lane by lane where v is strictly greater.
template <typename T>
__device__ __forceinline__ void merge2(uint32_t& mv, uint32_t& mc, uint32_t v, uint32_t c) {
    const uint32_t m = Pair<T>::gt(v, mv);
    mv = (v & m) | (mv & ~m);
    mc = (c & m) | (mc & ~m);
}

// Exact scalar max/argmax over a fixed window (the fallback).
template <typename T>
__device__ __noinline__ void exact_window(const T* __restrict__ xp, int ds, int de, int hs, int he,
                                          int ws, int we, int W, int HW, T* yo, int64_t* io) {
    int best = ds * HW + hs * W + ws;
    float m = Elem<T>::to_f(xp[best]);
    for (int d = ds; d < de; ++d)
        for (int h = hs; h < he; ++h)
            for (int w = ws; w < we; ++w) {
                const int off = d * HW + h * W + w;
                const float v = Elem<T>::to_f(xp[off]);
                if (beats(v, m)) {
                    m = v;
                    best = off;
                }
            }
    *yo = xp[best];
    *io = best;
}

// ---- bulk-copy pipeline helpers (mbarrier + cp.async.bulk, sm_90+) ----

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}
// Bounded wait: gives up after `limit` polls (each poll may itself suspend
// for a short, hardware-defined time) and reports failure.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int limit) {
    for (int i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Flag bit of a pipeline wait that gave up, and the polls a wait makes first.
constexpr unsigned int kErrPipelineTimeout = 1u;
constexpr int kWaitLimit = 1 << 22;

// The one window length along an axis (fixed windows: K; adaptive windows
// [floor(i*I/O), ceil((i+1)*I/O)): their common length), or 0 when the
// lengths differ. Host side, for choosing compiled window shapes.
inline int uniform_window_len(int I, int O, int K, bool adaptive) {
    if (!adaptive) return K;
    int len = -1;
    for (int i = 0; i < O; ++i) {
        const int l = (int)((((long long)(i + 1) * I + O - 1) / O) - ((long long)i * I / O));
        if (len >= 0 && l != len) return 0;
        len = l;
    }
    return len;
}

}  // namespace mp3d
