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

// ------------------------------------------------------------------ padded / dilated, direct
// Fixed windows with padding and dilation. One thread per input position:
// along each axis the windows that contain position x are the o with
// x = o*S - p + k*dl for some k in [0, K); stepping k downwards gives them
// in ascending o. The gradients of those that selected the input are
// summed in ascending (od, oh, ow) order (first term as the initial value).
template <typename T>
__global__ void __launch_bounds__(256)
k_bwd_ex_direct(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi,
                Geo g) {
    const long long total = g.P * (long long)g.vol;
    const int HW = g.H * g.W;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long p = e / g.vol;
        const int r = (int)(e - p * g.vol);
        const int d = r / HW;
        const int h = (r - d * HW) / g.W;
        const int w = r - d * HW - h * g.W;
        float acc = 0.0f;
        bool any = false;
        for (int a = g.kd - 1; a >= 0; --a) {
            const int td = d + g.pd - a * g.dd;
            if (td < 0 || td % g.sd != 0 || td / g.sd >= g.OD) continue;
            const int od = td / g.sd;
            for (int b = g.kh - 1; b >= 0; --b) {
                const int th = h + g.ph - b * g.dh;
                if (th < 0 || th % g.sh != 0 || th / g.sh >= g.OH) continue;
                const long long row = ((p * g.OD + od) * g.OH + th / g.sh) * (long long)g.OW;
                for (int c = g.kw - 1; c >= 0; --c) {
                    const int tw = w + g.pw - c * g.dw;
                    if (tw < 0 || tw % g.sw != 0 || tw / g.sw >= g.OW) continue;
                    const long long o = row + tw / g.sw;
                    if (__ldg(idx + o) == r) {
                        const float v = Elem<T>::to_f(go[o]);
                        acc = any ? acc + v : v;
                        any = true;
                    }
                }
            }
        }
        gi[e] = any ? Elem<T>::from_f(acc) : Elem<T>::from_f(0.0f);
    }
}

cudaError_t launch_bwd_ex_direct(const void* go, const int64_t* idx, void* gi, const Geo& g,
                                 int dtype, int sms, cudaStream_t s) {
    const long long total = g.P * (long long)g.vol;
    const int grid = grid_for(total, 256, sms, 8);
    switch (dtype) {
    case F32: k_bwd_ex_direct<float><<<grid, 256, 0, s>>>((const float*)go, idx, (float*)gi, g); break;
    case F16: k_bwd_ex_direct<__half><<<grid, 256, 0, s>>>((const __half*)go, idx, (__half*)gi, g); break;
    default:
        k_bwd_ex_direct<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)go, idx,
                                                            (__nv_bfloat16*)gi, g);
        break;
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------------ recompute (no stored index)
// Backward without stored indices: each window's argmax is recomputed from
// the input x with the forward's rule (scan d, then h, then w; replace only
// on "beats"), so the result equals the backward through the forward's
// indices bit for bit.

// Argmax (in-plane offset) of window (od, oh, ow) of plane xp.
template <typename T, bool ADAPTIVE>
__device__ __forceinline__ int window_argmax(const T* __restrict__ xp, int od, int oh, int ow,
                                             const Geo& g) {
    const int HW = g.H * g.W;
    const int ds = win_start(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
    const int de = win_end(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
    const int hs = win_start(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
    const int he = win_end(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
    const int ws = win_start(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
    const int we = win_end(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
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
    return best;
}

// Any geometry: one thread per input position enumerates its covering
// windows in ascending (od, oh, ow) order, recomputes each one's argmax and
// sums the gradients of those that chose it (first term as initial value).
template <typename T, bool ADAPTIVE>
__global__ void __launch_bounds__(256)
k_bwd_recompute_direct(const T* __restrict__ x, const T* __restrict__ go, T* __restrict__ gi,
                       Geo g) {
    const long long total = g.P * (long long)g.vol;
    const int HW = g.H * g.W;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long p = e / g.vol;
        const int r = (int)(e - p * g.vol);
        const int d = r / HW;
        const int h = (r - d * HW) / g.W;
        const int w = r - d * HW - h * g.W;
        const T* xp = x + p * g.vol;
        float acc = 0.0f;
        bool any = false;
        const int d1 = cover_hi(d, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int h1 = cover_hi(h, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int w1 = cover_hi(w, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        for (int od = cover_lo(d, g.D, g.OD, g.kd, g.sd, ADAPTIVE); od <= d1; ++od)
            for (int oh = cover_lo(h, g.H, g.OH, g.kh, g.sh, ADAPTIVE); oh <= h1; ++oh)
                for (int ow = cover_lo(w, g.W, g.OW, g.kw, g.sw, ADAPTIVE); ow <= w1; ++ow) {
                    if (window_argmax<T, ADAPTIVE>(xp, od, oh, ow, g) != r) continue;
                    const float v = Elem<T>::to_f(go[((p * g.OD + od) * g.OH + oh) * (long long)g.OW + ow]);
                    acc = any ? acc + v : v;
                    any = true;
                }
        gi[e] = any ? Elem<T>::from_f(acc) : Elem<T>::from_f(0.0f);
    }
}

// 2x2x2 windows, stride 2, tiling the input, rows of 16-byte chunks: one
// thread per run of VEC/2 windows of one window row loads the two-by-two
// input rows of the run (16-byte loads), finds each window's argmax with
// the exact scalar rule, loads the gradients and writes the run's 2x2 rows
// of gradient chunks (the gradient at the argmax, zero elsewhere).
template <typename T>
__global__ void __launch_bounds__(256)
k_bwd_recompute_k2s2(const T* __restrict__ x, const T* __restrict__ go, T* __restrict__ gi, Geo g,
                     FastDiv fSpr, FastDiv fOH) {
    constexpr int VEC = 16 / sizeof(T);
    constexpr int NW = VEC / 2;
    const int HW = g.H * g.W;
    const int spr = g.OW / NW;
    const int nseg = g.ovol / NW;
    const T zero = Elem<T>::from_f(0.0f);
    for (long long p = blockIdx.y; p < g.P; p += gridDim.y) {
        const T* xp = x + p * g.vol;
        for (int sg = blockIdx.x * blockDim.x + threadIdx.x; sg < nseg; sg += gridDim.x * blockDim.x) {
            const int row = fSpr.div(sg);
            const int ow0 = (sg - row * spr) * NW;
            const int od = fOH.div(row);
            const int oh = row - od * g.OH;
            const int base = 2 * od * HW + 2 * oh * g.W + 2 * ow0;
            Vec16<T> r[4];
#pragma unroll
            for (int dh = 0; dh < 4; ++dh)
                r[dh].u = __ldg(reinterpret_cast<const uint4*>(xp + base + (dh >> 1) * HW + (dh & 1) * g.W));
            // code of each window's argmax: dh * 2 + ww (scan d, h, then w)
            int code[NW];
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                float m = Elem<T>::to_f(r[0].e[2 * k]);
                int c = 0;
#pragma unroll
                for (int q = 1; q < 8; ++q) {
                    const float v = Elem<T>::to_f(r[q >> 1].e[2 * k + (q & 1)]);
                    if (beats(v, m)) {
                        m = v;
                        c = q;
                    }
                }
                code[k] = c;
            }
            const long long o0 = p * (long long)g.ovol + (long long)sg * NW;
            T gv[NW];
#pragma unroll
            for (int k = 0; k < NW; ++k) gv[k] = go[o0 + k];
            T* out = gi + p * (long long)g.vol + base;
#pragma unroll
            for (int dh = 0; dh < 4; ++dh) {
                Vec16<T> c;
#pragma unroll
                for (int k = 0; k < NW; ++k)
#pragma unroll
                    for (int t = 0; t < 2; ++t) c.e[2 * k + t] = code[k] == dh * 2 + t ? gv[k] : zero;
                *reinterpret_cast<uint4*>(out + (dh >> 1) * HW + (dh & 1) * g.W) = c.u;
            }
        }
    }
}

template <typename T>
static cudaError_t bwd_recompute_t(const void* x, const void* go, void* gi, const Geo& g, int sms,
                                   cudaStream_t s, int* kind) {
    constexpr int VEC = 16 / sizeof(T);
    const bool tiles = !g.adaptive && g.kd == 2 && g.kh == 2 && g.kw == 2 && g.sd == 2 && g.sh == 2 &&
                       g.sw == 2 && g.D == 2 * g.OD && g.H == 2 * g.OH && g.W == 2 * g.OW &&
                       g.W % VEC == 0 && (uintptr_t)x % 16 == 0 && (uintptr_t)gi % 16 == 0;
    if (tiles) {
        *kind = 0;
        const int nseg = g.ovol / (VEC / 2);
        dim3 grid((unsigned)((nseg + 255) / 256), (unsigned)(g.P < 65535 ? g.P : 65535));
        k_bwd_recompute_k2s2<T><<<grid, 256, 0, s>>>((const T*)x, (const T*)go, (T*)gi, g,
                                                     FastDiv((uint32_t)(g.OW / (VEC / 2))),
                                                     FastDiv((uint32_t)g.OH));
        return cudaGetLastError();
    }
    *kind = 1;
    const int grid = grid_for(g.P * (long long)g.vol, 256, sms, 8);
    if (g.adaptive)
        k_bwd_recompute_direct<T, true><<<grid, 256, 0, s>>>((const T*)x, (const T*)go, (T*)gi, g);
    else
        k_bwd_recompute_direct<T, false><<<grid, 256, 0, s>>>((const T*)x, (const T*)go, (T*)gi, g);
    return cudaGetLastError();
}

cudaError_t launch_bwd_recompute(const void* x, const void* go, void* gi, const Geo& g, int dtype,
                                 int sms, cudaStream_t s, int* kind) {
    switch (dtype) {
    case F32: return bwd_recompute_t<float>(x, go, gi, g, sms, s, kind);
    case F16: return bwd_recompute_t<__half>(x, go, gi, g, sms, s, kind);
    default: return bwd_recompute_t<__nv_bfloat16>(x, go, gi, g, sms, s, kind);
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

// ------------------------------------------------------------------ global
// Disjoint special case where one window covers each whole plane (output
// 1x1x1): one warp per plane writes the plane with 16-byte stores, the
// gradient at the stored index and zero elsewhere.
template <typename T, int VEC>
__global__ void __launch_bounds__(256)
k_bwd_global(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi,
             long long P, int vol) {
    const int lane = threadIdx.x & 31;
    const long long warp0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const T zero = Elem<T>::from_f(0.0f);
    const int nvec = vol / VEC;
    for (long long p = warp0; p < P; p += nwarps) {
        const int64_t best = __ldg(idx + p);
        const T gv = go[p];
        T* out = gi + p * vol;
        if (VEC > 1) {
            uint4* ov = reinterpret_cast<uint4*>(out);
            for (int v = lane; v < nvec; v += 32) {
                Vec16<T> c;
#pragma unroll
                for (int j = 0; j < VEC; ++j) c.e[j] = (v * VEC + j == best) ? gv : zero;
                ov[v] = c.u;
            }
        }
        for (int e = nvec * VEC + lane; e < vol; e += 32) out[e] = (e == best) ? gv : zero;
    }
}

// ------------------------------------------------------------------ disjoint, row chunks
// Disjoint windows, rows of W elements that split into 16-byte chunks.
// Block y walks planes; threads walk the chunks of a plane. A chunk lies in
// one row (d, h), so its row window (od, oh) is found once; with SW a
// divisor of VEC the chunk's element i falls in window ow0 + i / SW at
// offset i % SW. The indices and gradients of those VEC / SW windows are
// loaded together, then each element takes its window's gradient if the
// stored index is its own offset, else zero.
template <typename T, int VEC, int SW>
__global__ void __launch_bounds__(256)
k_bwd_disjoint_rows(const T* __restrict__ go, const int64_t* __restrict__ idx,
                    T* __restrict__ gi, Geo g, FastDiv fHW, FastDiv fW, FastDiv fSD, FastDiv fSH) {
    constexpr int NWIN = VEC / SW;
    constexpr int UNR = 4;                       // chunks per thread, loads issued together
    const int nchunks = g.vol / VEC;
    const T zero = Elem<T>::from_f(0.0f);
    for (long long p = blockIdx.y; p < g.P; p += gridDim.y) {
        for (int cb = blockIdx.x * blockDim.x * UNR + threadIdx.x; cb < nchunks;
             cb += gridDim.x * blockDim.x * UNR) {
            int64_t li[UNR][NWIN];
            T lg[UNR][NWIN];
            bool cov[UNR];
            int r0[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int c = cb + u * blockDim.x;
                r0[u] = c * VEC;
                cov[u] = false;
#pragma unroll
                for (int j = 0; j < NWIN; ++j) {
                    li[u][j] = -1;
                    lg[u][j] = zero;
                }
                if (c >= nchunks) continue;
                const int d = fHW.div(r0[u]);
                const int rr = r0[u] - d * g.H * g.W;
                const int h = fW.div(rr);
                const int w0 = rr - h * g.W;
                const int od = fSD.div(d), dr = d - od * g.sd;
                const int oh = fSH.div(h), hr = h - oh * g.sh;
                cov[u] = od < g.OD && dr < g.kd && oh < g.OH && hr < g.kh;
                if (!cov[u]) continue;
                const int ow0 = w0 / SW;
                const long long rowo = ((p * g.OD + od) * g.OH + oh) * (long long)g.OW;
#pragma unroll
                for (int j = 0; j < NWIN; ++j) {
                    if (ow0 + j < g.OW) {
                        li[u][j] = __ldg(idx + rowo + ow0 + j);
                        lg[u][j] = go[rowo + ow0 + j];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int c = cb + u * blockDim.x;
                if (c >= nchunks) continue;
                Vec16<T> out;
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const bool hit = cov[u] && (i % SW) < g.kw && li[u][i / SW] == (int64_t)(r0[u] + i);
                    out.e[i] = hit ? lg[u][i / SW] : zero;
                }
                *reinterpret_cast<uint4*>(gi + p * g.vol + r0[u]) = out.u;
            }
        }
    }
}

// ------------------------------------------------------------------ disjoint, window blocks
// Windows that tile the input exactly (kernel == stride on every axis, the
// input a whole number of windows, rows that split into 16-byte chunks).
// One thread owns NW = VEC / KW consecutive windows of one window row
// (od, oh): it loads their indices and gradients once (vector loads) and
// writes every input they cover, KD * KH output chunks of VEC elements, each
// element the gradient of its window when the stored index names it and
// zero otherwise.
template <typename T, int KD, int KH, int KW>
__global__ void __launch_bounds__(256)
k_bwd_disjoint_blocks(const T* __restrict__ go, const int64_t* __restrict__ idx,
                      T* __restrict__ gi, Geo g, FastDiv fSpr, FastDiv fOH) {
    constexpr int VEC = 16 / sizeof(T);
    constexpr int NW = VEC / KW;
    static_assert(NW * KW == VEC, "windows fill a chunk");
    const int HW = g.H * g.W;
    const int spr = g.OW / NW;                      // segments per window row
    const int nseg = g.ovol / NW;                   // segments per plane
    const T zero = Elem<T>::from_f(0.0f);
    for (long long p = blockIdx.y; p < g.P; p += gridDim.y) {
        for (int sg = blockIdx.x * blockDim.x + threadIdx.x; sg < nseg; sg += gridDim.x * blockDim.x) {
            const int row = fSpr.div(sg);
            const int ow0 = (sg - row * spr) * NW;
            const int od = fOH.div(row);
            const int oh = row - od * g.OH;
            const long long o0 = p * (long long)g.ovol + (long long)sg * NW;
            int64_t j[NW];
            T gv[NW];
            {
                const uint4* ip = reinterpret_cast<const uint4*>(idx + o0);
#pragma unroll
                for (int v = 0; v < NW / 2; ++v) {
                    const uint4 q = __ldg(ip + v);
                    j[2 * v] = (int64_t)((uint64_t)q.y << 32 | q.x);
                    j[2 * v + 1] = (int64_t)((uint64_t)q.w << 32 | q.z);
                }
                if (NW == 1) j[0] = __ldg(idx + o0);
#pragma unroll
                for (int k = 0; k < NW; ++k) gv[k] = go[o0 + k];
            }
            // place of each window's winner: row code dd * KH + hh (or -1), column ww
            const int base = (od * KD) * HW + (oh * KH) * g.W + ow0 * KW;
            int code[NW], ww[NW];
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                const int rel = (int)j[k] - (base + k * KW);
                int dd = 0, hh = 0;
#pragma unroll
                for (int i = 1; i < KD; ++i) dd += rel >= i * HW;
                const int r1 = rel - dd * HW;
#pragma unroll
                for (int i = 1; i < KH; ++i) hh += r1 >= i * g.W;
                ww[k] = r1 - hh * g.W;
                const bool ok = (uint64_t)j[k] < (uint64_t)g.vol && rel >= 0 && rel < KD * HW &&
                                r1 < KH * g.W && ww[k] < KW;
                code[k] = ok ? dd * KH + hh : -1;
            }
            T* out = gi + p * (long long)g.vol + base;
#pragma unroll
            for (int dd = 0; dd < KD; ++dd)
#pragma unroll
                for (int hh = 0; hh < KH; ++hh) {
                    Vec16<T> c;
#pragma unroll
                    for (int k = 0; k < NW; ++k)
#pragma unroll
                        for (int t = 0; t < KW; ++t)
                            c.e[k * KW + t] = (code[k] == dd * KH + hh && ww[k] == t) ? gv[k] : zero;
                    *reinterpret_cast<uint4*>(out + dd * HW + hh * g.W) = c.u;
                }
        }
    }
}

// ------------------------------------------------------------------ overlap, tiles
// Overlapping windows, deterministic gather. One CTA owns a tile of TD
// depth slices of one plane and every input in it:
//  1. It zero-fills the tile with 16-byte stores. Each window that can
//     cover the tile reads its stored index j; if j lies in the tile and in
//     the window, the window sets one bit in a per-input byte in shared
//     memory: its slot, the rank of the window among the windows covering
//     j in ascending (od, oh, ow) order, packed as (jd, jh, jw) with
//     power-of-two radices. It records (j, slot) and stages its gradient.
//  2. After a barrier (which also orders the zero stores before what
//     follows) each window checks whether its slot is the lowest bit set on
//     its j. That owner sums, in ascending bit order (= ascending
//     (od, oh, ow)), its own gradient and those of the windows whose bits
//     follow (found by slot offsets), in binary32, rounds once and stores.
// Per input the work is a share of one vector store; per window, a few
// integer operations, one shared atomic and, for owners, the sum.
struct TileGeo {
    int TD, ntiles;
    int rows;             // window rows (od values) staged per tile, at most
    int lch, lcw;         // log2 of the slot radix along h and w
    AxisMap ad, ah, aw;
    FastDiv fHW, fW, fOW, fOHOW;
};

template <typename T, int VEC>
__global__ void __launch_bounds__(256)
k_bwd_overlap_tile(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi,
                   Geo g, TileGeo tg) {
    constexpr int UNR = 8;                       // window loads in flight per thread
    extern __shared__ __align__(16) unsigned char smem[];
    const int HW = g.H * g.W;
    const int d0 = blockIdx.x * tg.TD;
    const int d1 = min(d0 + tg.TD, g.D);
    const int n = (d1 - d0) * HW;
    const int ohow = g.OH * g.OW;
    const int od_lo = tg.ad.lo(d0), od_hi = tg.ad.hi(d1 - 1);
    const int wbeg = od_lo * ohow;
    const int wend = (od_hi + 1) * ohow;          // empty when od_lo > od_hi
    const int mask_bytes = (tg.TD * HW + 15) / 16 * 16;
    uint32_t* mask32 = reinterpret_cast<uint32_t*>(smem);
    int* wrec = reinterpret_cast<int*>(smem + mask_bytes);
    T* gt = reinterpret_cast<T*>(smem + mask_bytes + (size_t)tg.rows * ohow * sizeof(int));
    const T zero = Elem<T>::from_f(0.0f);
    const int lo_j = d0 * HW, hi_j = d1 * HW;     // the tile's in-plane offsets
    const int lhw = tg.lch + tg.lcw;
    for (long long p = blockIdx.y; p < g.P; p += gridDim.y) {
        T* out = gi + p * (long long)g.vol + (long long)d0 * HW;
        const long long obase = p * (long long)g.ovol;
        uint4* m16 = reinterpret_cast<uint4*>(smem);
        for (int i = threadIdx.x; i < mask_bytes / 16; i += blockDim.x) m16[i] = make_uint4(0, 0, 0, 0);
        if (VEC > 1) {
            uint4* o4 = reinterpret_cast<uint4*>(out);
            for (int c = threadIdx.x; c < n / VEC; c += blockDim.x) o4[c] = make_uint4(0, 0, 0, 0);
            for (int e = (n / VEC) * VEC + threadIdx.x; e < n; e += blockDim.x) out[e] = zero;
        } else {
            for (int e = threadIdx.x; e < n; e += blockDim.x) out[e] = zero;
        }
        __syncthreads();
        // 1. claims
        for (int wb = wbeg; wb < wend; wb += UNR * blockDim.x) {
            int64_t j[UNR];
            T gv[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int wi = wb + u * blockDim.x + threadIdx.x;
                const bool ok = wi < wend;
                j[u] = ok ? __ldg(idx + obase + wi) : -1;
                gv[u] = ok ? go[obase + wi] : zero;
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int wi = wb + u * blockDim.x + threadIdx.x;
                if (wi >= wend) continue;
                const int me = wi - wbeg;
                gt[me] = gv[u];
                int rec = -1;
                if (j[u] >= lo_j && j[u] < hi_j) {
                    const int jj = (int)j[u];
                    const int od = tg.fOHOW.div(wi);
                    const int rem = wi - od * ohow;
                    const int oh = tg.fOW.div(rem);
                    const int ow = rem - oh * g.OW;
                    const int ds = tg.ad.start(od), hs = tg.ah.start(oh), ws = tg.aw.start(ow);
                    const int rel = jj - (ds * HW + hs * g.W + ws);
                    if (rel >= 0) {
                        const int dl = tg.fHW.div(rel);
                        const int r2 = rel - dl * HW;
                        const int hl = tg.fW.div(r2);
                        const int wl = r2 - hl * g.W;
                        if (dl < tg.ad.len(od) && hl < tg.ah.len(oh) && wl < tg.aw.len(ow)) {
                            const int slot = (tg.ad.earlier(od, dl) << lhw) |
                                             (tg.ah.earlier(oh, hl) << tg.lcw) | tg.aw.earlier(ow, wl);
                            const int local = jj - lo_j;
                            atomicOr(&mask32[local >> 2], 1u << ((local & 3) * 8 + slot));
                            rec = local << 3 | slot;
                        }
                    }
                }
                wrec[me] = rec;
            }
        }
        __syncthreads();
        // 2. owners
        for (int me = threadIdx.x; me < wend - wbeg; me += blockDim.x) {
            const int rec = wrec[me];
            if (rec < 0) continue;
            const int local = rec >> 3, slot = rec & 7;
            uint32_t m = (mask32[local >> 2] >> ((local & 3) * 8)) & 0xFFu;
            if (__ffs(m) - 1 != slot) continue;
            float acc = Elem<T>::to_f(gt[me]);
            m &= m - 1;
            const int sd = slot >> lhw, sh = (slot >> tg.lcw) & ((1 << tg.lch) - 1),
                      sw = slot & ((1 << tg.lcw) - 1);
            while (m) {
                const int b = __ffs(m) - 1;
                m &= m - 1;
                const int bd = b >> lhw, bh = (b >> tg.lcw) & ((1 << tg.lch) - 1),
                          bw = b & ((1 << tg.lcw) - 1);
                const int k = me + (bd - sd) * ohow + (bh - sh) * g.OW + (bw - sw);
                acc += Elem<T>::to_f(gt[k]);
            }
            out[local] = Elem<T>::from_f(acc);
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ overlap, chunk gather
// Overlapping fixed windows with kernel <= 2 * stride on every axis (so at
// most two windows cover an input along each axis), window shape known at
// compile time. One CTA owns a tile of TD depth slices of one plane:
//  1. stage, for every window that can cover the tile, one 8-byte word: its
//     winner as a tile-local index held in a float (exact below 2^24; a
//     large negative value when outside the tile) and its gradient widened
//     to binary32 (exact);
//  2. each thread computes VEC consecutive inputs of one row (d, h), a
//     chunk starting on a window boundary along w: it walks the at most
//     2 x 2 window rows (od, oh) that cover the row, in ascending order, and
//     in each the windows ow that overlap the chunk, in ascending order; a
//     window can only have chosen one of the at most KW inputs it covers, so
//     its winner is compared against those fixed chunk positions and, on a
//     match, its gradient is added to that input's binary32 sum. Every
//     input therefore sums the windows that chose it in ascending (od, oh,
//     ow) order and is rounded once;
//  3. the chunk leaves as one coalesced 16-byte store (element stores when
//     rows are not 16-byte multiples); inputs no window chose get +0.
// Two forms of step 2, chosen per tile:
//  - when every staged gradient is finite and none is -0, a match is taken
//    arithmetically: with x = winner - position (an integer held exactly),
//    h = sat(1 - x*x) is 1 for x == 0 and 0 otherwise, and acc = fma(g, h,
//    acc) equals acc + g or acc exactly (a sum that starts from +0 and has
//    no -0 term is never -0, so adding a signed zero leaves it unchanged);
//    this keeps the selection on the floating-point pipe;
//  - otherwise sums start from -0, matches are taken by comparison and
//    per-input "touched" bits turn inputs no window chose into +0.
// Staged window rows are interleaved: window ow of a row sits at
// ((ow + R) % R) * Q + (ow + R) / R with R = VEC / SW and Q = chunks + 1, so
// the lanes of a warp, whose chunks start R windows apart, read consecutive
// words; the places of the missing windows ow = -1 and ow >= OW hold a
// sentinel that matches nothing. Rows of a tile are visited with all even h
// before all odd h when the stride along h is 2, so the lanes of a warp
// mostly have the same number of covering window rows.
static constexpr float kNoWinner = -16777216.0f;   // never within 2^24 of a chunk

// 1 when the integer x (held exactly in a float) is 0, else 0: the
// saturated 1 - x*x, as one fused multiply-add with saturation.
__device__ __forceinline__ float hit_weight(float x) {
    float h;
    asm("fma.rn.sat.f32 %0, %1, %2, 0f3F800000;" : "=f"(h) : "f"(-x), "f"(x));
    return h;
}

// Sums, rounds and stores one chunk of VEC inputs (see the kernel below).
// row0 points at the first covering window row; off[i] is the place of the
// chunk's window ow = c * R + DMIN + i within a staged window row.
template <typename T, int VEC, int KW, int SW, bool EXACT>
__device__ __forceinline__ void gather_chunk(const float2* __restrict__ row0, const int (&off)[(VEC - 1) / SW + (KW - 1) / SW + 1],
                                             int nod, int noh, int rowsp, int RQ, float basef,
                                             T* __restrict__ dst, bool vstore, int nt) {
    constexpr int DMIN = -((KW - 1) / SW), DMAX = (VEC - 1) / SW;
    float acc[VEC];
    unsigned touched = 0;
#pragma unroll
    for (int t = 0; t < VEC; ++t) acc[t] = EXACT ? -0.0f : 0.0f;
#pragma unroll
    for (int a = 0; a < 2; ++a) {
        if (a >= nod) break;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            if (b >= noh) break;
            const float2* row = row0 + (a * rowsp + b * RQ);
#pragma unroll
            for (int dl = DMIN; dl <= DMAX; ++dl) {
                const float2 e = row[off[dl - DMIN]];
                const float u = e.x - basef;     // winner relative to the chunk start
#pragma unroll
                for (int q = 0; q < KW; ++q) {
                    const int t = SW * dl + q;
                    if (t < 0 || t >= VEC) continue;
                    if (EXACT) {
                        if (u == (float)t) {
                            acc[t] += e.y;
                            touched |= 1u << t;
                        }
                    } else {
                        acc[t] = fmaf(e.y, hit_weight(u - (float)t), acc[t]);
                    }
                }
            }
        }
    }
    Vec16<T> v;
#pragma unroll
    for (int t = 0; t < VEC; ++t)
        v.e[t] = Elem<T>::from_f((EXACT && !((touched >> t) & 1u)) ? 0.0f : acc[t]);
    if (vstore) {
        *reinterpret_cast<uint4*>(dst) = v.u;
    } else {
        for (int t = 0; t < nt; ++t) dst[t] = v.e[t];
    }
}

template <typename T, int VEC, int KD, int SD, int KH, int SH, int KW, int SW>
__global__ void __launch_bounds__(512)
k_bwd_overlap_gather(const T* __restrict__ go, const int64_t* __restrict__ idx,
                     T* __restrict__ gi, Geo g, int TD, int rows_max, int nchunk, bool vstore,
                     FastDiv fOW) {
    static_assert(KD <= 2 * SD && KH <= 2 * SH && KW <= 2 * SW, "at most two covering windows per axis");
    static_assert(VEC % SW == 0, "chunks start on a window boundary along w");
    static_assert(SH == 1 || SH == 2, "row order handles strides 1 and 2 along h");
    static_assert((KW - 1) / SW <= VEC / SW, "one sentinel column before the first chunk suffices");
    constexpr int R = VEC / SW;
    constexpr int DMIN = -((KW - 1) / SW), DMAX = (VEC - 1) / SW, NDL = DMAX - DMIN + 1;
    extern __shared__ __align__(16) unsigned char smem[];
    const int HW = g.H * g.W;
    const int d0 = blockIdx.x * TD;
    const int d1 = min(d0 + TD, g.D);
    const int od_lo = d0 < KD ? 0 : (d0 - KD) / SD + 1;
    const int od_hi = min((d1 - 1) / SD, g.OD - 1);
    const int ohow = g.OH * g.OW;
    const int nwin = (od_hi >= od_lo) ? (od_hi - od_lo + 1) * ohow : 0;
    const long long lo_j = (long long)d0 * HW, hi_j = (long long)d1 * HW;
    const int Q = nchunk + 1, RQ = R * Q, rowsp = g.OH * RQ;
    float2* wt = reinterpret_cast<float2*>(smem);
    int2* rinfo = reinterpret_cast<int2*>(smem + (size_t)rows_max * rowsp * sizeof(float2));
    const int nrows_t = (d1 - d0) * g.H;
    const int h_even = (g.H + 1) / 2;
    // sentinels everywhere once (the staging below overwrites the places of
    // real windows only) and, per input row of the tile, {row offset in the
    // tile, first covering window row | #covering along d << 28 | along h << 30}
    for (int e = threadIdx.x; e < rows_max * rowsp; e += blockDim.x) wt[e] = make_float2(kNoWinner, 0.0f);
    for (int ri = threadIdx.x; ri < nrows_t; ri += blockDim.x) {
        const int dr = ri / g.H, r = ri - dr * g.H;
        const int h = (SH == 2) ? (r < h_even ? 2 * r : 2 * (r - h_even) + 1) : r;
        const int d = d0 + dr;
        const int odl = d < KD ? 0 : (d - KD) / SD + 1, odh = min(d / SD, g.OD - 1);
        const int ohl = h < KH ? 0 : (h - KH) / SH + 1, ohh = min(h / SH, g.OH - 1);
        const int nod = max(0, odh - odl + 1), noh = max(0, ohh - ohl + 1);
        const int wrow = (nod > 0 && noh > 0) ? (odl - od_lo) * rowsp + ohl * RQ : 0;
        rinfo[ri] = make_int2(dr * HW + h * g.W,
                              (int)((unsigned)wrow | ((unsigned)nod << 28) | ((unsigned)noh << 30)));
    }
    // this thread's chunk column and the places of its windows in a row
    const int rstep = blockDim.x / nchunk;
    const int c = threadIdx.x % nchunk, r0 = threadIdx.x / nchunk;
    int off[NDL];
#pragma unroll
    for (int dl = DMIN; dl <= DMAX; ++dl) {
        const int slot = ((dl % R) + R) % R, cadd = (dl - slot) / R;
        off[dl - DMIN] = slot * Q + c + 1 + cadd;
    }
    const int nt = min(VEC, g.W - c * VEC);
    __syncthreads();
    for (long long p = blockIdx.y; p < g.P; p += gridDim.y) {
        const long long obase = p * (long long)g.ovol + (long long)od_lo * ohow;
        // 1. stage the windows
        constexpr int UNR = 4;
        bool special = false;
        for (int wb = 0; wb < nwin; wb += UNR * blockDim.x) {
            int64_t j[UNR];
            T gv[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int me = wb + u * blockDim.x + threadIdx.x;
                const bool ok = me < nwin;
                j[u] = ok ? __ldg(idx + obase + me) : -1;
                gv[u] = ok ? go[obase + me] : Elem<T>::from_f(0.0f);
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int me = wb + u * blockDim.x + threadIdx.x;
                if (me >= nwin) continue;
                const float gf = Elem<T>::to_f(gv[u]);
                const unsigned gb = __float_as_uint(gf);
                special |= gb == 0x80000000u || (gb & 0x7f800000u) == 0x7f800000u;
                const int row = fOW.div(me);
                const int ow = me - row * g.OW + R;
                const bool in = j[u] >= lo_j && j[u] < hi_j;
                wt[row * RQ + (ow % R) * Q + ow / R] =
                    make_float2(in ? (float)(int)(j[u] - lo_j) : kNoWinner, gf);
            }
        }
        const bool exact = __syncthreads_or(special) != 0;
        // 2. this thread's chunk in rows r0, r0 + rstep, ...
        T* out = gi + p * (long long)g.vol + lo_j + c * VEC;
        if (r0 < rstep) {
            for (int ri = r0; ri < nrows_t; ri += rstep) {
                const int2 info = rinfo[ri];
                const int base = info.x + c * VEC;
                const float2* row0 = wt + (info.y & 0x0FFFFFFF);
                const int nod = (info.y >> 28) & 3, noh = (int)((unsigned)info.y >> 30);
                if (!exact)
                    gather_chunk<T, VEC, KW, SW, false>(row0, off, nod, noh, rowsp, RQ, (float)base,
                                                        out + info.x, vstore, nt);
                else
                    gather_chunk<T, VEC, KW, SW, true>(row0, off, nod, noh, rowsp, RQ, (float)base,
                                                       out + info.x, vstore, nt);
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ launch: disjoint

template <typename T, int SW>
static cudaError_t bwd_rows_t(const void* go, const int64_t* idx, void* gi, const Geo& g,
                              cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    const int nchunks = g.vol / VEC;
    dim3 grid((unsigned)((nchunks + 1023) / 1024), (unsigned)(g.P < 65535 ? g.P : 65535));
    k_bwd_disjoint_rows<T, VEC, SW><<<grid, 256, 0, s>>>(
        (const T*)go, idx, (T*)gi, g, FastDiv((uint32_t)(g.H * g.W)), FastDiv((uint32_t)g.W),
        FastDiv((uint32_t)g.sd), FastDiv((uint32_t)g.sh));
    return cudaGetLastError();
}

template <typename T>
static cudaError_t bwd_disjoint_t(const void* go, const int64_t* idx, void* gi, const Geo& g,
                                  int sms, cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    const long long total = g.P * (long long)g.vol;
    const bool aligned = (uintptr_t)gi % 16 == 0;
    const bool plane_vec = aligned && ((long long)g.vol * sizeof(T)) % 16 == 0;
    if (g.ovol == 1 && g.kd == g.D && g.kh == g.H && g.kw == g.W) {
        const int grid = grid_for(g.P * 32, 256, sms, kGlobalCtasPerSm);
        if (plane_vec)
            k_bwd_global<T, VEC><<<grid, 256, 0, s>>>((const T*)go, idx, (T*)gi, g.P, g.vol);
        else
            k_bwd_global<T, 1><<<grid, 256, 0, s>>>((const T*)go, idx, (T*)gi, g.P, g.vol);
        return cudaGetLastError();
    }
    // exact tiling by 2x2x2 windows: one thread per run of windows
    if (aligned && (uintptr_t)idx % 16 == 0 && g.kd == 2 && g.kh == 2 && g.kw == 2 && g.sd == 2 &&
        g.sh == 2 && g.sw == 2 && g.D == 2 * g.OD && g.H == 2 * g.OH && g.W == 2 * g.OW &&
        g.W % VEC == 0) {
        constexpr int NW = VEC / 2;
        const int nseg = g.ovol / NW;
        dim3 grid((unsigned)((nseg + 255) / 256), (unsigned)(g.P < 65535 ? g.P : 65535));
        k_bwd_disjoint_blocks<T, 2, 2, 2><<<grid, 256, 0, s>>>(
            (const T*)go, idx, (T*)gi, g, FastDiv((uint32_t)(g.OW / NW)), FastDiv((uint32_t)g.OH));
        return cudaGetLastError();
    }
    if (aligned && g.W % VEC == 0) {
        switch (g.sw) {
        case 1: return bwd_rows_t<T, 1>(go, idx, gi, g, s);
        case 2: return bwd_rows_t<T, 2>(go, idx, gi, g, s);
        case 4: return bwd_rows_t<T, 4>(go, idx, gi, g, s);
        case 8: if (VEC == 8) return bwd_rows_t<T, VEC>(go, idx, gi, g, s); break;
        default: break;
        }
    }
    if (aligned) {
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

// ------------------------------------------------------------------ launch: tiles

static constexpr int kTileBytes = 110 * 1024;   // shared bytes per tile (two CTAs per SM)

// Most windows that can cover one position along an axis.
static int max_cover(int I, int O, int K, int S, bool adaptive) {
    int c;
    if (adaptive) c = (O + I - 1) / I + 1;
    else c = K <= S ? 1 : (K + S - 1) / S;
    return c < O ? c : O;
}

static int pow2_at_least(int c) {
    int p = 1;
    while (p < c) p <<= 1;
    return p;
}

static int log2_exact(int p) {
    int l = 0;
    while ((1 << l) < p) ++l;
    return l;
}


// Window rows (od values) that can cover one tile of td slices, at most.
static int max_window_rows(const Geo& g, int td) {
    int best = 0;
    for (int d0 = 0; d0 < g.D; d0 += td) {
        const int d1 = (d0 + td < g.D ? d0 + td : g.D) - 1;
        int lo, hi;
        if (g.adaptive) {
            lo = (int)(((long long)d0 * g.OD) / g.D);
            hi = (int)(((long long)(d1 + 1) * g.OD - 1) / g.D);
        } else {
            lo = d0 < g.kd ? 0 : (d0 - g.kd) / g.sd + 1;
            hi = d1 / g.sd < g.OD - 1 ? d1 / g.sd : g.OD - 1;
        }
        if (hi - lo + 1 > best) best = hi - lo + 1;
    }
    return best;
}

static size_t tile_smem_bytes(const Geo& g, int td, int es) {
    const size_t masks = ((size_t)td * g.H * g.W + 15) / 16 * 16;
    const size_t wins = (size_t)max_window_rows(g, td) * g.OH * g.OW;
    return masks + wins * sizeof(int) + (wins * es + 15) / 16 * 16;
}

bool bwd_tile_supported(const Geo& g) {
    const bool a = g.adaptive != 0;
    const long long slots = (long long)pow2_at_least(max_cover(g.D, g.OD, g.kd, g.sd, a)) *
                            pow2_at_least(max_cover(g.H, g.OH, g.kh, g.sh, a)) *
                            pow2_at_least(max_cover(g.W, g.OW, g.kw, g.sw, a));
    if (slots > 8) return false;
    if (tile_smem_bytes(g, 1, 4) > (size_t)kTileBytes) return false;
    // local offsets in a tile are packed with a 3-bit slot into an int
    if ((long long)g.H * g.W * g.D >= (1LL << 28)) return false;
    if (a) {   // products used by the adaptive window arithmetic stay below 2^31
        const long long lim = (1LL << 31) - 1;
        if ((long long)g.D * g.OD + g.OD > lim || (long long)g.H * g.OH + g.OH > lim ||
            (long long)g.W * g.OW + g.OW > lim)
            return false;
    }
    return true;
}

template <typename T, int VEC>
static cudaError_t bwd_tile_launch(const void* go, const int64_t* idx, void* gi, const Geo& g,
                                   const TileGeo& tg, size_t smem, cudaStream_t s) {
    auto kern = k_bwd_overlap_tile<T, VEC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)tg.ntiles, (unsigned)(g.P < 65535 ? g.P : 65535));
    kern<<<grid, 256, smem, s>>>((const T*)go, idx, (T*)gi, g, tg);
    return cudaGetLastError();
}

// Window shapes with a compiled fixed-window overlap kernel.
static int fixed_variant(const Geo& g) {
    if (g.adaptive) return -1;
    if (g.kd == 3 && g.sd == 2 && g.kh == 3 && g.sh == 2 && g.kw == 3 && g.sw == 2) return 0;
    if (g.kd == 2 && g.sd == 1 && g.kh == 2 && g.sh == 1 && g.kw == 2 && g.sw == 1) return 1;
    return -1;
}

static constexpr int kFixedTileBytes = 113 * 1024;   // shared bytes per tile (two CTAs per SM)

// Staged window rows: R = (16 / element size) / stride_w slots of
// (chunks per row + 1) columns each.
static int fixed_row_words(const Geo& g, int es) {
    const int vec = 16 / es;
    return (vec / g.sw) * ((g.W + vec - 1) / vec + 1);
}

// Staged window rows plus one int2 per input row of the tile.
static size_t fixed_smem_bytes(const Geo& g, int td, int es) {
    return (size_t)max_window_rows(g, td) * g.OH * fixed_row_words(g, es) * sizeof(float2) +
           (size_t)td * g.H * sizeof(int2);
}

template <typename T, int KD, int SD, int KH, int SH, int KW, int SW>
static cudaError_t bwd_fixed_launch(const void* go, const int64_t* idx, void* gi, const Geo& g,
                                    int td, cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    const size_t smem = fixed_smem_bytes(g, td, sizeof(T));
    auto kern = k_bwd_overlap_gather<T, VEC, KD, SD, KH, SH, KW, SW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int nchunk = (g.W + VEC - 1) / VEC;
    const bool vstore = g.W % VEC == 0 && (uintptr_t)gi % 16 == 0;
    dim3 grid((unsigned)((g.D + td - 1) / td), (unsigned)(g.P < 65535 ? g.P : 65535));
    kern<<<grid, 512, smem, s>>>((const T*)go, idx, (T*)gi, g, td, max_window_rows(g, td), nchunk,
                                 vstore, FastDiv((uint32_t)g.OW));
    return cudaGetLastError();
}

// The fixed-window kernel when the shape has a variant and the tile fits;
// cudaErrorNotSupported otherwise.
template <typename T>
static cudaError_t bwd_fixed_t(const void* go, const int64_t* idx, void* gi, const Geo& g,
                               cudaStream_t s) {
    const int v = fixed_variant(g);
    if (v < 0) return cudaErrorNotSupported;
    const int HW = g.H * g.W;
    int td = g.D;
    while (td > 1 && fixed_smem_bytes(g, td, sizeof(T)) > (size_t)kFixedTileBytes) --td;
    if (fixed_smem_bytes(g, td, sizeof(T)) > (size_t)kFixedTileBytes) return cudaErrorNotSupported;
    if ((long long)td * HW >= (1LL << 24)) return cudaErrorNotSupported;   // exact in a float
    if ((g.W + 16 / (int)sizeof(T) - 1) / (16 / (int)sizeof(T)) > 512) return cudaErrorNotSupported;
    if (v == 0) return bwd_fixed_launch<T, 3, 2, 3, 2, 3, 2>(go, idx, gi, g, td, s);
    return bwd_fixed_launch<T, 2, 1, 2, 1, 2, 1>(go, idx, gi, g, td, s);
}

template <typename T>
static cudaError_t bwd_tile_t(const void* go, const int64_t* idx, void* gi, const Geo& g,
                              cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    {
        const cudaError_t ef = bwd_fixed_t<T>(go, idx, gi, g, s);
        if (ef != cudaErrorNotSupported) return ef;
    }
    const bool a = g.adaptive != 0;
    const int HW = g.H * g.W;
    TileGeo tg;
    tg.lch = log2_exact(pow2_at_least(max_cover(g.H, g.OH, g.kh, g.sh, a)));
    tg.lcw = log2_exact(pow2_at_least(max_cover(g.W, g.OW, g.kw, g.sw, a)));
    tg.ad = axis_map(g.D, g.OD, g.kd, g.sd, a);
    tg.ah = axis_map(g.H, g.OH, g.kh, g.sh, a);
    tg.aw = axis_map(g.W, g.OW, g.kw, g.sw, a);
    tg.fHW = FastDiv((uint32_t)HW);
    tg.fW = FastDiv((uint32_t)g.W);
    tg.fOW = FastDiv((uint32_t)g.OW);
    tg.fOHOW = FastDiv((uint32_t)(g.OH * g.OW));
    // Deepest tile whose masks and staged windows fit the shared budget.
    int td = g.D;
    while (td > 1 && tile_smem_bytes(g, td, sizeof(T)) > (size_t)kTileBytes) --td;
    // 16-byte fill stores need every tile (and plane) on a 16-byte boundary.
    bool vec = (uintptr_t)gi % 16 == 0 && ((long long)g.vol * sizeof(T)) % 16 == 0;
    if (vec && td < g.D) {
        int t = td;
        while (t > 0 && ((long long)t * HW * sizeof(T)) % 16 != 0) --t;
        if (t > 0) td = t;
        else vec = false;
    }
    tg.TD = td;
    tg.ntiles = (g.D + td - 1) / td;
    tg.rows = max_window_rows(g, td);
    const size_t smem = tile_smem_bytes(g, td, sizeof(T));
    if (vec) return bwd_tile_launch<T, VEC>(go, idx, gi, g, tg, smem, s);
    return bwd_tile_launch<T, 1>(go, idx, gi, g, tg, smem, s);
}

cudaError_t launch_bwd_overlap_tile(const void* go, const int64_t* idx, void* gi, const Geo& g,
                                    int dtype, int, cudaStream_t s) {
    switch (dtype) {
    case F32: return bwd_tile_t<float>(go, idx, gi, g, s);
    case F16: return bwd_tile_t<__half>(go, idx, gi, g, s);
    default: return bwd_tile_t<__nv_bfloat16>(go, idx, gi, g, s);
    }
}

}  // namespace mp3d
