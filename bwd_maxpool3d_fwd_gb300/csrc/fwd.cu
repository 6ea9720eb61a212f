// Forward kernels: max and argmax over fixed or adaptive 3-D windows.
//
// Definition followed (teenygrad docs "Struct Maxpool3dForward",
// description and Constraints): y[p,od,oh,ow] is the maximum of x over the
// window box of that output; no padding. The index written is the in-plane
// flat offset d*H*W + h*W + w of the first element (in d, h, w row-major
// order) that attains the maximum; a NaN beats every number.
#include <cfloat>
#include <climits>

#include "internal.h"

namespace mp3d {

// ------------------------------------------------------------------ generic
// One thread per output; scans its window from global memory (read-only
// path, L1-cached). Any window shape, fixed or adaptive.
template <typename T, bool ADAPTIVE>
__global__ void __launch_bounds__(256)
k_fwd_generic(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g) {
    const long long total = g.P * (long long)g.ovol;
    const int HW = g.H * g.W;
    for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
         o += (long long)gridDim.x * blockDim.x) {
        const int ow = (int)(o % g.OW);
        long long t = o / g.OW;
        const int oh = (int)(t % g.OH);
        t /= g.OH;
        const int od = (int)(t % g.OD);
        const long long p = t / g.OD;
        const int ds = win_start(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int de = win_end(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int hs = win_start(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int he = win_end(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int ws = win_start(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        const int we = win_end(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        const T* xp = x + p * g.vol;
        int best = ds * HW + hs * g.W + ws;
        float m = Elem<T>::to_f(xp[best]);
        for (int d = ds; d < de; ++d)
            for (int h = hs; h < he; ++h) {
                const int row = d * HW + h * g.W;
                for (int w = ws; w < we; ++w) {
                    const float v = Elem<T>::to_f(xp[row + w]);
                    if (beats(v, m)) {
                        m = v;
                        best = row + w;
                    }
                }
            }
        y[o] = xp[best];
        idx[o] = best;
    }
}

// ------------------------------------------------------------------ global
// One window per plane (output 1x1x1). One warp per plane: each lane scans
// a strided share of the plane with 16-byte loads when every plane starts
// on a 16-byte boundary, then the warp combines (value, offset) pairs.
// The combine takes the pair that beats, and among equal values (or two
// NaNs) the smaller offset, so the result is the first occurrence.
__device__ __forceinline__ void take_better(float v, int i, float& m, int& best) {
    if (beats(v, m) || (!beats(m, v) && i < best)) {
        m = v;
        best = i;
    }
}

template <typename T, int VEC>
__global__ void __launch_bounds__(256)
k_fwd_global(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx,
             long long P, int vol) {
    const int lane = threadIdx.x & 31;
    const long long warp0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const int nvec = vol / VEC;
    for (long long p = warp0; p < P; p += nwarps) {
        const T* xp = x + p * vol;
        float m = -INFINITY;
        int best = INT_MAX;
        if (VEC > 1) {
            const uint4* xv = reinterpret_cast<const uint4*>(xp);
#pragma unroll 4
            for (int v = lane; v < nvec; v += 32) {
                Vec16<T> c;
                c.u = __ldg(xv + v);
#pragma unroll
                for (int j = 0; j < VEC; ++j) take_better(Elem<T>::to_f(c.e[j]), v * VEC + j, m, best);
            }
        }
        for (int e = nvec * VEC + lane; e < vol; e += 32) take_better(Elem<T>::to_f(xp[e]), e, m, best);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const int b2 = __shfl_xor_sync(0xffffffffu, best, off);
            take_better(m2, b2, m, best);
        }
        if (lane == 0) {
            y[p] = xp[best];
            idx[p] = best;
        }
    }
}

// ------------------------------------------------------------------ launch

static int grid_for(long long work, int per_block, int sms, int blocks_per_sm) {
    long long b = (work + per_block - 1) / per_block;
    long long cap = (long long)sms * blocks_per_sm;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

template <typename T>
static cudaError_t fwd_generic_t(const void* x, void* y, int64_t* idx, const Geo& g, int sms,
                                 cudaStream_t s) {
    const long long total = g.P * (long long)g.ovol;
    const int grid = grid_for(total, 256, sms, 8);
    if (g.adaptive)
        k_fwd_generic<T, true><<<grid, 256, 0, s>>>((const T*)x, (T*)y, idx, g);
    else
        k_fwd_generic<T, false><<<grid, 256, 0, s>>>((const T*)x, (T*)y, idx, g);
    return cudaGetLastError();
}

cudaError_t launch_fwd_generic(const void* x, void* y, int64_t* idx, const Geo& g, int dtype,
                               int sms, cudaStream_t s) {
    switch (dtype) {
    case F32: return fwd_generic_t<float>(x, y, idx, g, sms, s);
    case F16: return fwd_generic_t<__half>(x, y, idx, g, sms, s);
    default: return fwd_generic_t<__nv_bfloat16>(x, y, idx, g, sms, s);
    }
}

template <typename T>
static cudaError_t fwd_global_t(const void* x, void* y, int64_t* idx, const Geo& g, int sms,
                                cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    const bool vec_ok = ((uintptr_t)x % 16 == 0) && (((long long)g.vol * sizeof(T)) % 16 == 0);
    const int grid = grid_for(g.P * 32, 256, sms, 8);
    if (vec_ok)
        k_fwd_global<T, VEC><<<grid, 256, 0, s>>>((const T*)x, (T*)y, idx, g.P, g.vol);
    else
        k_fwd_global<T, 1><<<grid, 256, 0, s>>>((const T*)x, (T*)y, idx, g.P, g.vol);
    return cudaGetLastError();
}

cudaError_t launch_fwd_global(const void* x, void* y, int64_t* idx, const Geo& g, int dtype,
                              int sms, cudaStream_t s) {
    switch (dtype) {
    case F32: return fwd_global_t<float>(x, y, idx, g, sms, s);
    case F16: return fwd_global_t<__half>(x, y, idx, g, sms, s);
    default: return fwd_global_t<__nv_bfloat16>(x, y, idx, g, sms, s);
    }
}

// ------------------------------------------------------------------ stride 2
bool fwd_s2_supported(const Geo&, int) { return false; }

cudaError_t launch_fwd_s2(const void*, void*, int64_t*, const Geo&, int, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace mp3d
