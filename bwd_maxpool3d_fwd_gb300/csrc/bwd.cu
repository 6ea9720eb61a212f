// Backward kernels: route each output gradient to its argmax input
// (FlagGems-Experimental PR #308, "Add adaptive_max_pool3d_backward Moore
// Threads specialized operator", Summary).
//
// grad_in[p, j] = sum, in ascending (od, oh, ow) order, of grad_out[p, o]
// over the outputs o whose index is j; binary32 accumulation starting from
// the first term, one rounding to the type; +0 where nothing is routed.
//
// Paths:
//  - disjoint gather: every input lies in at most one window; each thread
//    owns a run of inputs, finds each one's window, compares the stored
//    index with its own offset and writes the gradient or zero. One pass,
//    no zero fill, no atomics, coalesced vector stores.
//  - overlapping gather, direct: each input enumerates its covering
//    windows in ascending order and sums the matching gradients.
//  - atomic ablation: zero fill, atomicAdd scatter in binary32, and a
//    rounding pass for 16-bit types (the page's non-divisible path).
#include "internal.h"

namespace mp3d {

static int grid_for(long long work, int per_block, int sms, int blocks_per_sm) {
    long long b = (work + per_block - 1) / per_block;
    long long cap = (long long)sms * blocks_per_sm;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

// Position of a flat input element, advanced one element at a time so that
// a thread decodes its run with a single set of divisions. For each axis it
// also tracks the (only) window that can hold the position when windows
// are disjoint: window o = x / S, at relative offset x - o*S.
struct RunPos {
    long long p;
    int r;                 // in-plane offset
    int d, h, w;
    int od, oh, ow;        // candidate window per axis
    int dr, hr, wr;        // offset inside the candidate window

    __device__ __forceinline__ void init(long long e, const Geo& g) {
        p = e / g.vol;
        r = (int)(e - p * g.vol);
        const int HW = g.H * g.W;
        d = r / HW;
        const int r2 = r - d * HW;
        h = r2 / g.W;
        w = r2 - h * g.W;
        od = d / g.sd; dr = d - od * g.sd;
        oh = h / g.sh; hr = h - oh * g.sh;
        ow = w / g.sw; wr = w - ow * g.sw;
    }
    __device__ __forceinline__ void next(const Geo& g) {
        ++r;
        ++w;
        if (++wr == g.sw) { wr = 0; ++ow; }
        if (w == g.W) {
            w = 0; ow = 0; wr = 0;
            ++h;
            if (++hr == g.sh) { hr = 0; ++oh; }
            if (h == g.H) {
                h = 0; oh = 0; hr = 0;
                ++d;
                if (++dr == g.sd) { dr = 0; ++od; }
                if (d == g.D) {
                    d = 0; od = 0; dr = 0; r = 0;
                    ++p;
                }
            }
        }
    }
    __device__ __forceinline__ bool covered(const Geo& g) const {
        return od < g.OD && dr < g.kd && oh < g.OH && hr < g.kh && ow < g.OW && wr < g.kw;
    }
    __device__ __forceinline__ long long window(const Geo& g) const {
        return ((p * g.OD + od) * g.OH + oh) * (long long)g.OW + ow;
    }
};

// ------------------------------------------------------------------ disjoint
template <typename T, int VEC>
__global__ void __launch_bounds__(256)
k_bwd_disjoint(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi,
               Geo g) {
    const long long total = g.P * (long long)g.vol;
    const long long nchunks = (total + VEC - 1) / VEC;
    const T zero = Elem<T>::from_f(0.0f);
    for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < nchunks;
         c += (long long)gridDim.x * blockDim.x) {
        const long long e0 = c * VEC;
        RunPos pos;
        pos.init(e0, g);
        long long last_o = -1;
        int64_t li = -1;
        T lg = zero;
        Vec16<T> out;
        T outs[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            T val = zero;
            if (e0 + i < total && pos.covered(g)) {
                const long long o = pos.window(g);
                if (o != last_o) {
                    last_o = o;
                    li = __ldg(idx + o);
                    lg = go[o];
                }
                if (li == pos.r) val = lg;
            }
            outs[i] = val;
            pos.next(g);
        }
        if (VEC * sizeof(T) == 16 && e0 + VEC <= total) {
#pragma unroll
            for (int i = 0; i < VEC; ++i) out.e[i] = outs[i];
            *reinterpret_cast<uint4*>(gi + e0) = out.u;
        } else {
#pragma unroll
            for (int i = 0; i < VEC; ++i)
                if (e0 + i < total) gi[e0 + i] = outs[i];
        }
    }
}

template <typename T>
static cudaError_t bwd_disjoint_t(const void* go, const int64_t* idx, void* gi, const Geo& g,
                                  int sms, cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    const long long total = g.P * (long long)g.vol;
    if ((uintptr_t)gi % 16 == 0) {
        const int grid = grid_for((total + VEC - 1) / VEC, 256, sms, 8);
        k_bwd_disjoint<T, VEC><<<grid, 256, 0, s>>>((const T*)go, idx, (T*)gi, g);
    } else {
        const int grid = grid_for(total, 256, sms, 8);
        k_bwd_disjoint<T, 1><<<grid, 256, 0, s>>>((const T*)go, idx, (T*)gi, g);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_disjoint(const void* go, const int64_t* idx, void* gi, const Geo& g,
                                int dtype, int sms, cudaStream_t s) {
    switch (dtype) {
    case F32: return bwd_disjoint_t<float>(go, idx, gi, g, sms, s);
    case F16: return bwd_disjoint_t<__half>(go, idx, gi, g, sms, s);
    default: return bwd_disjoint_t<__nv_bfloat16>(go, idx, gi, g, sms, s);
    }
}

// ------------------------------------------------------------------ overlap, direct
// One thread per input element: enumerate the covering windows in
// ascending (od, oh, ow) order, read each one's stored index, and sum the
// gradients of those that selected this element.
template <typename T, bool ADAPTIVE>
__global__ void __launch_bounds__(256)
k_bwd_overlap_direct(const T* __restrict__ go, const int64_t* __restrict__ idx,
                     T* __restrict__ gi, Geo g) {
    const long long total = g.P * (long long)g.vol;
    const int HW = g.H * g.W;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long p = e / g.vol;
        const int r = (int)(e - p * g.vol);
        const int d = r / HW;
        const int h = (r - d * HW) / g.W;
        const int w = r - d * HW - h * g.W;
        const int d0 = cover_lo(d, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int d1 = cover_hi(d, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int h0 = cover_lo(h, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int h1 = cover_hi(h, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int w0 = cover_lo(w, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        const int w1 = cover_hi(w, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        float acc = 0.0f;
        bool any = false;
        for (int od = d0; od <= d1; ++od)
            for (int oh = h0; oh <= h1; ++oh) {
                const long long row = ((p * g.OD + od) * g.OH + oh) * (long long)g.OW;
                for (int ow = w0; ow <= w1; ++ow) {
                    if (__ldg(idx + row + ow) == r) {
                        const float v = Elem<T>::to_f(go[row + ow]);
                        acc = any ? acc + v : v;
                        any = true;
                    }
                }
            }
        gi[e] = any ? Elem<T>::from_f(acc) : Elem<T>::from_f(0.0f);
    }
}

template <typename T>
static cudaError_t bwd_direct_t(const void* go, const int64_t* idx, void* gi, const Geo& g,
                                int sms, cudaStream_t s) {
    const long long total = g.P * (long long)g.vol;
    const int grid = grid_for(total, 256, sms, 8);
    if (g.adaptive)
        k_bwd_overlap_direct<T, true><<<grid, 256, 0, s>>>((const T*)go, idx, (T*)gi, g);
    else
        k_bwd_overlap_direct<T, false><<<grid, 256, 0, s>>>((const T*)go, idx, (T*)gi, g);
    return cudaGetLastError();
}

cudaError_t launch_bwd_overlap_direct(const void* go, const int64_t* idx, void* gi,
                                      const Geo& g, int dtype, int sms, cudaStream_t s) {
    switch (dtype) {
    case F32: return bwd_direct_t<float>(go, idx, gi, g, sms, s);
    case F16: return bwd_direct_t<__half>(go, idx, gi, g, sms, s);
    default: return bwd_direct_t<__nv_bfloat16>(go, idx, gi, g, sms, s);
    }
}

// ------------------------------------------------------------------ atomic ablation
// Zero n floats; 16-byte stores when the buffer starts on a 16-byte boundary.
__global__ void __launch_bounds__(256) k_zero_f32(float* __restrict__ a, long long n) {
    const long long n4 = ((uintptr_t)a % 16 == 0) ? n / 4 : 0;
    float4* a4 = reinterpret_cast<float4*>(a);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
         i += (long long)gridDim.x * blockDim.x)
        a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = n4 * 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        a[i] = 0.f;
}

// One thread per output: add its gradient into the accumulator of the
// input its index names. Indices outside [0, D*H*W) are dropped.
template <typename T>
__global__ void __launch_bounds__(256)
k_bwd_atomic_scatter(const T* __restrict__ go, const int64_t* __restrict__ idx,
                     float* __restrict__ acc, Geo g) {
    const long long total = g.P * (long long)g.ovol;
    for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
         o += (long long)gridDim.x * blockDim.x) {
        const long long p = o / g.ovol;
        const int64_t j = __ldg(idx + o);
        if (j >= 0 && j < g.vol) atomicAdd(acc + p * g.vol + j, Elem<T>::to_f(go[o]));
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
k_round_from_f32(const float* __restrict__ acc, T* __restrict__ out, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        out[i] = Elem<T>::from_f(acc[i]);
}

template <typename T>
static cudaError_t bwd_atomic_t(const void* go, const int64_t* idx, void* gi, float* ws,
                                const Geo& g, int sms, cudaStream_t s) {
    const long long n = g.P * (long long)g.vol;
    const long long nout = g.P * (long long)g.ovol;
    float* acc = (sizeof(T) == 4) ? (float*)gi : ws;
    k_zero_f32<<<grid_for(n / 4 + 1, 256, sms, 8), 256, 0, s>>>(acc, n);
    k_bwd_atomic_scatter<T><<<grid_for(nout, 256, sms, 8), 256, 0, s>>>((const T*)go, idx, acc, g);
    if (sizeof(T) != 4)
        k_round_from_f32<T><<<grid_for(n, 256, sms, 8), 256, 0, s>>>(acc, (T*)gi, n);
    return cudaGetLastError();
}

cudaError_t launch_bwd_atomic(const void* go, const int64_t* idx, void* gi, float* ws,
                              const Geo& g, int dtype, int sms, cudaStream_t s) {
    switch (dtype) {
    case F32: return bwd_atomic_t<float>(go, idx, gi, ws, g, sms, s);
    case F16: return bwd_atomic_t<__half>(go, idx, gi, ws, g, sms, s);
    default: return bwd_atomic_t<__nv_bfloat16>(go, idx, gi, ws, g, sms, s);
    }
}

// ------------------------------------------------------------------ overlap, shared masks
bool bwd_mask_supported(const Geo&) { return false; }

cudaError_t launch_bwd_overlap_mask(const void*, const int64_t*, void*, const Geo&, int, int,
                                    cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace mp3d
