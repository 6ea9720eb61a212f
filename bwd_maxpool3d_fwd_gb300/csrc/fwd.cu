// Forward kernels: max and argmax over fixed or adaptive 3-D windows.
//
// Definition followed (teenygrad docs "Struct Maxpool3dForward",
// description and Constraints): y[p,od,oh,ow] is the maximum of x over the
// window box of that output; no padding. The index written is the in-plane
// flat offset d*H*W + h*W + w of the first element (in d, h, w row-major
// order) that attains the maximum; a NaN beats every number.
#include <atomic>
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
        if (idx) idx[o] = best;
    }
}

// ------------------------------------------------------------------ padded / dilated
// Fixed windows with padding and dilation: the window of output o along an
// axis takes the positions o*S - p + k*dl, k = 0 .. K-1, inside the input
// (padding is never chosen). One thread per output scans them in ascending
// (d, h, w) order with the exact rule.
template <typename T>
__global__ void __launch_bounds__(256)
k_fwd_ex(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g) {
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
        const T* xp = x + p * g.vol;
        int best = -1;
        float m = 0.0f;
        for (int a = 0; a < g.kd; ++a) {
            const int d = od * g.sd - g.pd + a * g.dd;
            if (d < 0 || d >= g.D) continue;
            for (int b = 0; b < g.kh; ++b) {
                const int h = oh * g.sh - g.ph + b * g.dh;
                if (h < 0 || h >= g.H) continue;
                const int row = d * HW + h * g.W;
                for (int c = 0; c < g.kw; ++c) {
                    const int w = ow * g.sw - g.pw + c * g.dw;
                    if (w < 0 || w >= g.W) continue;
                    const float v = Elem<T>::to_f(xp[row + w]);
                    if (best < 0 || beats(v, m)) {
                        m = v;
                        best = row + w;
                    }
                }
            }
        }
        // the host rejects geometries with an empty window, so best >= 0
        y[o] = xp[best];
        if (idx) idx[o] = best;
    }
}

// ------------------------------------------------------------------ global
// One window per plane (output 1x1x1). One warp per plane: each lane scans
// a strided share of the plane with 16-byte loads when every plane starts
// on a 16-byte boundary, then the warp combines (value, offset) pairs. A
// lane meets its elements in ascending offset order, so inside a lane an
// element replaces the running best only when it beats it; the combine
// across lanes takes the pair that beats, and among equal values (or two
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
            // U loads per lane in flight together, then their elements in order
            constexpr int U = 8;
            const uint4* xv = reinterpret_cast<const uint4*>(xp);
            for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
                Vec16<T> c[U];
#pragma unroll
                for (int i = 0; i < U; ++i)
                    if (v0 + 32 * i < nvec) c[i].u = __ldg(xv + v0 + 32 * i);
#pragma unroll
                for (int i = 0; i < U; ++i) {
                    const int v = v0 + 32 * i;
                    if (v >= nvec) break;
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const float f = Elem<T>::to_f(c[i].e[j]);
                        if (beats(f, m) || best == INT_MAX) {
                            m = f;
                            best = v * VEC + j;
                        }
                    }
                }
            }
        }
        for (int e = nvec * VEC + lane; e < vol; e += 32) {
            const float f = Elem<T>::to_f(xp[e]);
            if (beats(f, m) || best == INT_MAX) {
                m = f;
                best = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const int b2 = __shfl_xor_sync(0xffffffffu, best, off);
            take_better(m2, b2, m, best);
        }
        if (lane == 0) {
            y[p] = xp[best];
            if (idx) idx[p] = best;
        }
    }
}

// ------------------------------------------------------------------ slab
// Any window shape (fixed or adaptive) whose depth slab fits in shared
// memory. One CTA per (plane, output depth od): the slices [ds, de) of the
// window depth are one contiguous span of the plane; the CTA copies it into
// shared memory with 16-byte loads (the span is placed at the same offset
// modulo 16 bytes, so both sides stay aligned; the ragged ends are copied
// element by element), then each thread scans whole windows of that depth
// from shared memory, d then h then w ascending, with the exact rule
// (strict "beats", NaN beats numbers, first occurrence kept).
template <typename T, bool ADAPTIVE>
__global__ void __launch_bounds__(256)
k_fwd_slab(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int VEC = 16 / sizeof(T);
    const int od = blockIdx.x;
    const int HW = g.H * g.W;
    const int ds = win_start(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
    const int de = win_end(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
    const int n = (de - ds) * HW;
    for (long long p = blockIdx.y; p < g.P; p += gridDim.y) {
        const T* src = x + p * g.vol + (long long)ds * HW;
        const int mis = (int)(((uintptr_t)src % 16) / sizeof(T));   // elements before a 16-byte boundary
        T* sl = reinterpret_cast<T*>(smem) + mis;                    // sl[i] = src[i]
        const int head = mis ? min(VEC - mis, n) : 0;
        const int nvec = (n - head) / VEC;
        const uint4* gv = reinterpret_cast<const uint4*>(src + head);
        uint4* sv = reinterpret_cast<uint4*>(sl + head);
        for (int c = threadIdx.x; c < nvec; c += blockDim.x) sv[c] = __ldg(gv + c);
        for (int e = threadIdx.x; e < head; e += blockDim.x) sl[e] = src[e];
        for (int e = head + nvec * VEC + threadIdx.x; e < n; e += blockDim.x) sl[e] = src[e];
        __syncthreads();
        const long long obase = ((p * g.OD + od) * (long long)g.OH) * g.OW;
        for (int t = threadIdx.x; t < g.OH * g.OW; t += blockDim.x) {
            const int oh = t / g.OW, ow = t - (t / g.OW) * g.OW;
            const int hs = win_start(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
            const int he = win_end(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
            const int ws = win_start(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
            const int we = win_end(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
            int best = hs * g.W + ws;
            float m = Elem<T>::to_f(sl[best]);
            for (int d = 0; d < de - ds; ++d)
                for (int h = hs; h < he; ++h) {
                    const int row = d * HW + h * g.W;
                    for (int w = ws; w < we; ++w) {
                        const float v = Elem<T>::to_f(sl[row + w]);
                        if (beats(v, m)) {
                            m = v;
                            best = row + w;
                        }
                    }
                }
            y[obase + t] = sl[best];
            if (idx) idx[obase + t] = (int64_t)ds * HW + best;
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ keyed slab
// 16-bit types: the slab of one (plane, od) is staged as one 32-bit word
// per element whose unsigned order is the scan's preference, so that the
// winner of a window is the plain unsigned maximum of its words.
//   high half: an order key of the value: +0 and -0 the same key, negative
//              values below positive ones by magnitude, every NaN above
//              +inf (all NaNs one key);
//   low half:  0xFFFF minus the element's offset in the slab, so that among
//              equal keys (equal values, or NaNs) the earliest in (d, h, w)
//              order is the largest word.
// This is the rule of the scan ("beats": strictly greater, or a NaN over a
// number; the first occurrence kept) as one total order. The value written
// to y is re-read from x at the winning offset, so its bits (sign of zero,
// NaN payload) are the input element's.

template <typename T>
__device__ __forceinline__ unsigned order_word(unsigned short b, int e) {
    const unsigned k = order_keys2<KeyConst<T>::nanadd>(b) & 0xFFFFu;
    return k << 16 | (0xFFFFu - (unsigned)e);
}

constexpr int KS_NT = 256;

// KH, KW > 0: every window along h (w) is exactly KH (KW) long, and the
// window scan unrolls; 0: lengths read from the tables.
template <typename T, bool ADAPTIVE, int KH, int KW>
__global__ void __launch_bounds__(KS_NT)
k_fwd_keyslab(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g,
              int nwords, FastDiv fnout, FastDiv fOW) {
    // shared: the slab words (nwords, a multiple of 32), the winning word of
    // each output of the plane-depth, the window rows of each oh and the
    // window columns of each ow
    extern __shared__ __align__(128) unsigned smem_ks[];
    constexpr int VEC = 8;                       // 16-bit elements per 16-byte load
    constexpr unsigned NANADD = KeyConst<T>::nanadd;
    const int od = blockIdx.x;
    const int tid = threadIdx.x;
    const int HW = g.H * g.W;
    const int nout = g.OH * g.OW;
    unsigned* words = smem_ks;                                // [nwords]
    unsigned* win = words + nwords;                           // [OH*OW]
    int2* htab = reinterpret_cast<int2*>(win + ((nout + 1) & ~1));   // [OH] (hs, he)
    int2* wtab = htab + g.OH;                                 // [OW] (ws, we)
    for (int i = tid; i < g.OH; i += KS_NT)
        htab[i] = make_int2(win_start(i, g.H, g.OH, g.kh, g.sh, ADAPTIVE),
                            win_end(i, g.H, g.OH, g.kh, g.sh, ADAPTIVE));
    for (int i = tid; i < g.OW; i += KS_NT)
        wtab[i] = make_int2(win_start(i, g.W, g.OW, g.kw, g.sw, ADAPTIVE),
                            win_end(i, g.W, g.OW, g.kw, g.sw, ADAPTIVE));
    for (int i = tid; i < nout; i += KS_NT) win[i] = 0u;
    const int ds = win_start(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
    const int de = win_end(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
    const int nd = de - ds;
    const int n = nd * HW;                       // slab elements (<= 65536)
    for (long long p = blockIdx.y; p < g.P; p += gridDim.y) {
        const T* src = x + p * g.vol + (long long)ds * HW;
        const unsigned short* sb = reinterpret_cast<const unsigned short*>(src);
        const int mis = (int)(((uintptr_t)src % 16) / sizeof(T));   // elements before a 16-byte boundary
        unsigned* wl = words + mis;              // wl[e] = word of slab element e
        const int head = mis ? min(VEC - mis, n) : 0;
        const int nvec = (n - head) / VEC;
        const uint4* gv = reinterpret_cast<const uint4*>(src + head);
        // U loads per thread in flight together, then their words
        constexpr int U = 8;
        for (int c0 = tid; c0 < nvec; c0 += U * KS_NT) {
            uint4 u[U];
#pragma unroll
            for (int i = 0; i < U; ++i)
                if (c0 + i * KS_NT < nvec) u[i] = __ldg(gv + c0 + i * KS_NT);
#pragma unroll
            for (int i = 0; i < U; ++i) {
                const int c = c0 + i * KS_NT;
                if (c >= nvec) break;
                const unsigned k0 = order_keys2<NANADD>(u[i].x), k1 = order_keys2<NANADD>(u[i].y);
                const unsigned k2 = order_keys2<NANADD>(u[i].z), k3 = order_keys2<NANADD>(u[i].w);
                const unsigned inv = 0xFFFFu - (unsigned)(head + c * VEC);   // low half of element 0
                // word of element j: key j in the high half, inv - j in the low half
                const uint4 lo = make_uint4(__byte_perm(k0, inv, 0x1054), __byte_perm(k0, inv - 1, 0x3254),
                                            __byte_perm(k1, inv - 2, 0x1054), __byte_perm(k1, inv - 3, 0x3254));
                const uint4 hi = make_uint4(__byte_perm(k2, inv - 4, 0x1054), __byte_perm(k2, inv - 5, 0x3254),
                                            __byte_perm(k3, inv - 6, 0x1054), __byte_perm(k3, inv - 7, 0x3254));
                uint4* dst = reinterpret_cast<uint4*>(wl + head + c * VEC);   // 16-byte aligned
                dst[0] = lo;
                dst[1] = hi;
            }
        }
        for (int e = tid; e < head; e += KS_NT) wl[e] = order_word<T>(sb[e], e);
        for (int e = head + nvec * VEC + tid; e < n; e += KS_NT) wl[e] = order_word<T>(sb[e], e);
        __syncthreads();
        // one item per (d, oh, ow): the best word of that depth row of the
        // window; the items of a window meet in an unsigned max (the word
        // order does not depend on the order they arrive in)
        for (int t = tid; t < nd * nout; t += KS_NT) {
            const int d = fnout.div(t);
            const int o = t - d * nout;
            const int oh = fOW.div(o), ow = o - oh * g.OW;
            const int2 hr = htab[oh], wr = wtab[ow];
            unsigned best = 0u;                  // every word is above 0 (keys are at least 0x80)
            const unsigned* base = wl + d * HW + hr.x * g.W + wr.x;
            if constexpr (KH > 0 && KW > 0) {
#pragma unroll
                for (int h = 0; h < KH; ++h)
#pragma unroll
                    for (int w = 0; w < KW; ++w) best = max(best, base[h * g.W + w]);
            } else {
                for (int h = 0; h < hr.y - hr.x; ++h)
                    for (int w = 0; w < wr.y - wr.x; ++w) best = max(best, base[h * g.W + w]);
            }
            atomicMax(win + o, best);
        }
        __syncthreads();
        const long long obase = ((p * g.OD + od) * (long long)g.OH) * g.OW;
        for (int t = tid; t < nout; t += KS_NT) {
            const unsigned best = win[t];
            win[t] = 0u;                         // ready for the next plane
            const int off = (int)(0xFFFFu - (best & 0xFFFFu));
            y[obase + t] = src[off];
            if (idx) idx[obase + t] = (int64_t)ds * HW + off;
        }
        __syncthreads();
    }
}

static constexpr int kSlabBytes = 96 * 1024;

// Deepest window along D (slices the slab must hold).
static int max_depth(const Geo& g) {
    if (!g.adaptive) return g.kd;
    int best = 0;
    for (int i = 0; i < g.OD; ++i) {
        const int s = (int)(((long long)i * g.D) / g.OD);
        const int e = (int)(((long long)(i + 1) * g.D + g.OD - 1) / g.OD);
        if (e - s > best) best = e - s;
    }
    return best;
}

bool fwd_slab_supported(const Geo& g, int dtype) {
    const int es = dtype == F32 ? 4 : 2;
    return (long long)max_depth(g) * g.H * g.W * es + 16 <= kSlabBytes;
}

// The keyed form: 16-bit types, slab offsets that fit the low half of a
// word, and four bytes per slab element in shared memory.
static constexpr int kKeySlabBytes = 100 * 1024;
// Slab words: the deepest slab plus up to 7 elements before a 16-byte
// boundary, rounded up to 32.
static int keyslab_words(const Geo& g) {
    return (int)(((long long)max_depth(g) * g.H * g.W + 7 + 31) / 32 * 32);
}
static size_t keyslab_smem(const Geo& g) {
    const long long nout = (long long)g.OH * g.OW;
    return (size_t)(4LL * keyslab_words(g) + 4 * ((nout + 1) / 2 * 2) + 8LL * (g.OH + g.OW));
}
static bool keyslab_fits(const Geo& g) {
    const long long n = (long long)max_depth(g) * g.H * g.W;
    return n <= 65536 && (long long)g.OH + g.OW <= 4096 && (long long)g.OH * g.OW <= 8192 &&
           keyslab_smem(g) <= (size_t)kKeySlabBytes;
}

template <typename T, bool AD>
static auto keyslab_kernel(int kh, int kw) {
    if (kh == kw) {
        switch (kh) {
        case 2: return k_fwd_keyslab<T, AD, 2, 2>;
        case 3: return k_fwd_keyslab<T, AD, 3, 3>;
        case 4: return k_fwd_keyslab<T, AD, 4, 4>;
        case 5: return k_fwd_keyslab<T, AD, 5, 5>;
        default: break;
        }
    }
    return k_fwd_keyslab<T, AD, 0, 0>;
}

template <typename T>
static cudaError_t keyslab_t(const void* x, void* y, int64_t* idx, const Geo& g, cudaStream_t s) {
    const size_t smem = keyslab_smem(g);
    dim3 grid((unsigned)g.OD, (unsigned)(g.P < 65535 ? g.P : 65535));
    const int kh = uniform_window_len(g.H, g.OH, g.kh, g.adaptive), kw = uniform_window_len(g.W, g.OW, g.kw, g.adaptive);
    auto kern = g.adaptive ? keyslab_kernel<T, true>(kh, kw) : keyslab_kernel<T, false>(kh, kw);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, KS_NT, smem, s>>>((const T*)x, (T*)y, idx, g, keyslab_words(g),
                                   FastDiv((uint32_t)(g.OH * g.OW)), FastDiv((uint32_t)g.OW));
    return cudaGetLastError();
}

template <typename T>
static cudaError_t fwd_slab_t(const void* x, void* y, int64_t* idx, const Geo& g, cudaStream_t s) {
    if constexpr (sizeof(T) == 2)
        if (keyslab_fits(g)) return keyslab_t<T>(x, y, idx, g, s);
    const size_t smem = (size_t)max_depth(g) * g.H * g.W * sizeof(T) + 16;
    dim3 grid((unsigned)g.OD, (unsigned)(g.P < 65535 ? g.P : 65535));
    if (g.adaptive) {
        cudaError_t e = cudaFuncSetAttribute(k_fwd_slab<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_fwd_slab<T, true><<<grid, 256, smem, s>>>((const T*)x, (T*)y, idx, g);
    } else {
        cudaError_t e = cudaFuncSetAttribute(k_fwd_slab<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_fwd_slab<T, false><<<grid, 256, smem, s>>>((const T*)x, (T*)y, idx, g);
    }
    return cudaGetLastError();
}

cudaError_t launch_fwd_slab(const void* x, void* y, int64_t* idx, const Geo& g, int dtype, int,
                            cudaStream_t s) {
    switch (dtype) {
    case F32: return fwd_slab_t<float>(x, y, idx, g, s);
    case F16: return fwd_slab_t<__half>(x, y, idx, g, s);
    default: return fwd_slab_t<__nv_bfloat16>(x, y, idx, g, s);
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

template <typename T>
static cudaError_t fwd_ex_t(const void* x, void* y, int64_t* idx, const Geo& g, int sms,
                            cudaStream_t s) {
    const long long total = g.P * (long long)g.ovol;
    k_fwd_ex<T><<<grid_for(total, 256, sms, 8), 256, 0, s>>>((const T*)x, (T*)y, idx, g);
    return cudaGetLastError();
}

cudaError_t launch_fwd_ex(const void* x, void* y, int64_t* idx, const Geo& g, int dtype, int sms,
                          cudaStream_t s) {
    switch (dtype) {
    case F32: return fwd_ex_t<float>(x, y, idx, g, sms, s);
    case F16: return fwd_ex_t<__half>(x, y, idx, g, sms, s);
    default: return fwd_ex_t<__nv_bfloat16>(x, y, idx, g, sms, s);
    }
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
    const int grid = grid_for(g.P * 32, 256, sms, kGlobalCtasPerSm);
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
// Fast fixed-window forward for 16-bit types with stride 2 along W.
//
// Each thread owns one 16-byte chunk of a row (8 elements, so the 4 outputs
// whose windows start in it), an oh-tile of TOH output rows and a range of
// output depths. It walks the depth once: for every slice d it loads the
// tile's rows of its chunk (plus the one element past the chunk that a
// size-3 window needs), reduces along W, then H, then folds the slice into
// the accumulators of the (at most two) output depths whose windows contain
// d. Values travel as packed pairs (two adjacent outputs per 32-bit word)
// and are compared two at a time with set.gt on f16x2/bf16x2; each lane
// carries a small code of its winner's (dl, hl, wl) position in the window.
//
// Tie rule: reductions run W first, then H, then D, and replace only on a
// strictly greater value, so the winner is the smallest d, then h, then w
// among equal maxima: the first occurrence in (d, h, w) row-major order.
// +0 and -0 compare equal. NaN and infinities are not handled by packed
// compares; a running x*0 + acc over every loaded word turns NaN once any
// NaN or infinity was seen, and then the thread recomputes the affected
// outputs with the exact scalar scan (same rule as the generic kernel).

constexpr uint32_t kLanes = 0x00010001u;   // a constant in both 16-bit lanes

// Set when a pipeline wait gave up (never expected); read and cleared by
// mp3d_device_error_flags().
__device__ unsigned int g_mp3d_device_error = 0;

// Polls the main pipeline waits make before giving up (host side; lowered
// only by tests of the give-up path).
static std::atomic<int> g_wait_limit{kWaitLimit};

int pipeline_wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

int set_pipeline_wait_limit(int polls) {
    return g_wait_limit.exchange(polls < 0 ? kWaitLimit : polls, std::memory_order_relaxed);
}

// One CTA = (plane p, output-depth group, band of G oh-tiles of TOH rows).
// Threads = nc chunks x G tiles. Each depth slice's band of input rows is
// one contiguous span of memory; thread 0 streams slice after slice into a
// ring of NS shared-memory stages with cp.async.bulk, completion counted by
// an mbarrier per stage; every thread reduces its chunk's rows from shared
// memory. Each thread writes its outputs straight from registers (the two
// pair words of an output row are its four values). Blocks of at most 128
// threads at five CTAs per SM: with the outputs no longer staged in shared
// memory (and no barriers around their flush), 466 -> 412 us on the
// 32x128x16x112x112 fp16 forward.
//
// PADC: windows padded by pd = bit 0, ph = bit 1, pw = bit 2 of PADC (one
// position per side at most; 3x3x3 windows, stride 2, floor output sizes),
// compiled per combination, at four CTAs per SM (the padded forms' extra
// state spills at five: 788 -> 430 us on the 32x128x16x112x112 fp16
// forward with padding 1): window o starts at 2o - p. A position outside the
// input is read as its nearest position inside (the clamped slice, row or
// column) carrying that position's own offset in the window as its code:
// such a duplicate is either the same element as a candidate met earlier,
// or comes first and bears the code of the real element that follows it,
// so ties still go to the first real occurrence and padding is never chosen.
template <typename T, int KD, int SD, int KH, int SH, int KW, int TOH, int NS, int PADC = 0,
          bool VO = false>
__global__ void __launch_bounds__(128, PADC ? 4 : 5)
k_fwd_s2(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g, int odg,
         int nq, int G, int nbands, int nc, int wait_limit) {
    static_assert(KD <= 2 * SD && KD <= 4 && KH <= 4 && KW >= 2 && KW <= 3, "shape");
    constexpr bool PAD = PADC != 0;
    static_assert(!PAD || (KD == 3 && SD == 2 && KH == 3 && SH == 2 && KW == 3), "padded shape");
    constexpr int pd = PADC & 1, ph = (PADC >> 1) & 1, pw = (PADC >> 2) & 1;
    extern __shared__ __align__(128) unsigned char smem[];
    const int band = (int)(blockIdx.x % nbands);
    long long rest = blockIdx.x / nbands;
    const int q = (int)(rest % nq);
    const long long p = rest / nq;

    const int tid = threadIdx.x;
    const int c = tid % nc;
    const int tl = tid / nc;                       // tile inside the band
    const int ow0 = 4 * c, w0 = 8 * c;
    const int oh_band = band * G * TOH;            // first output row of the band
    const int oh_band_end = min(g.OH, oh_band + G * TOH);
    const int oh0 = oh_band + tl * TOH;
    const int nh = max(0, min(TOH, oh_band_end - oh0));
    const int od0 = q * odg;
    const int nd = min(odg, g.OD - od0);
    const int HW = g.H * g.W;
    const bool has_extra = (KW > 2) && (w0 + 8 < g.W);
    // input rows of the band that exist: [r0, r1)
    const int r0 = max(oh_band * SH - ph, 0);
    const int r1 = min((oh_band_end - 1) * SH - ph + KH, g.H);
    const int band_rows = r1 - r0;
    const uint32_t span_bytes = (uint32_t)band_rows * g.W * sizeof(T);
    const uint32_t stage_stride = (span_bytes + 127) / 128 * 128;
    // shared layout: [NS stages][NS mbarriers]
    unsigned char* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * stage_stride);

    const T* xp = x + p * g.vol;
    const T* band_src = xp + (long long)r0 * g.W;
    const int nslices = (KD >= SD) ? nd * SD + KD - SD : nd * KD;
    // nominal slice of step k (before the first or past the last slice when
    // padded) and the slice it is read from
    auto slice_nom = [&](int k) { return (KD >= SD) ? od0 * SD - pd + k : (od0 + k / KD) * SD + k % KD; };
    auto slice_d = [&](int k) { return PAD ? min(max(slice_nom(k), 0), g.D - 1) : slice_nom(k); };

    // Bounded waits. Each thread waits for a slice itself and, once a wait
    // gives up, stops waiting (its outputs are then incomplete; the error
    // flag says so). Only thread 0 issues copies, and it waits for every
    // slice it issued until its own wait gives up, at slice s_fail_at; it
    // refills nothing after that, so at most the copies of slices
    // [s_fail_at, s_fail_at + NS) are in flight, and it lets them land
    // before the CTA exits. (Agreeing on a failure CTA-wide at the slice
    // barrier cost 2-4% on the full-size forwards and adds no safety: a
    // wait that gives up in another thread leaves no copy in flight.)
    __shared__ int s_fail_at;
    if (tid == 0) {
        for (int st = 0; st < NS; ++st) mbar_init(smem_addr(&bars[st]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0) {
        for (int k = 0; k < NS && k < nslices; ++k) {
            const uint32_t bar = smem_addr(&bars[k]);
            mbar_expect_tx(bar, span_bytes);
            bulk_g2s(smem_addr(stages + k * stage_stride), band_src + (long long)slice_d(k) * HW,
                     span_bytes, bar);
        }
    }

    uint32_t poison = 0;
    bool failed = false;
    uint32_t cv[TOH][2], cc[TOH][2], pv[TOH][2], pc[TOH][2];
#pragma unroll
    for (int j = 0; j < TOH; ++j)
#pragma unroll
        for (int k = 0; k < 2; ++k) cv[j][k] = cc[j][k] = pv[j][k] = pc[j][k] = 0;

    // Write this thread's outputs of depth od (four consecutive ow per
    // output row) straight from registers: a row's four values are the two
    // pair words, its four indices 32 bytes; 16-byte (8-byte for y) stores
    // where the row's address allows, element stores otherwise.
    auto write_out = [&](int od, uint32_t (&v)[TOH][2], uint32_t (&cd)[TOH][2]) {
        const bool exact = Pair<T>::is_poisoned(poison);
#pragma unroll
        for (int j = 0; j < TOH; ++j) {
            if (j >= nh) break;
            const int oh = oh0 + j;
            const long long o0 = ((p * g.OD + od) * g.OH + oh) * (long long)g.OW + ow0;
            uint16_t* yo = reinterpret_cast<uint16_t*>(y) + o0;
            int64_t* io = !VO && idx ? idx + o0 : nullptr;   // VO: values only
            // in-plane offsets (below 2^31) of the four winners
            int off[4];
            uint32_t yw[2] = {v[j][0], v[j][1]};
            const int base = (od * SD - pd) * HW + (oh * SH - ph) * g.W + ow0 * 2 - pw;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t code = (cd[j][e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
                off[e] = base + (int)(code >> 4) * HW + (int)((code >> 2) & 3) * g.W + 2 * e + (int)(code & 3);
            }
            if (exact) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (ow0 + e >= g.OW) break;
                    T yv;
                    int64_t iv;
                    const int ow = ow0 + e;
                    if constexpr (PAD)
                        exact_window<T>(xp, max(od * SD - pd, 0), min(od * SD - pd + KD, g.D),
                                        max(oh * SH - ph, 0), min(oh * SH - ph + KH, g.H),
                                        max(ow * 2 - pw, 0), min(ow * 2 - pw + KW, g.W), g.W, HW, &yv, &iv);
                    else
                        exact_window<T>(xp, od * SD, od * SD + KD, oh * SH, oh * SH + KH, ow * 2,
                                        ow * 2 + KW, g.W, HW, &yv, &iv);
                    yo[e] = *reinterpret_cast<uint16_t*>(&yv);
                    if (io) io[e] = iv;
                }
                continue;
            }
            if (ow0 + 4 <= g.OW) {
                const uintptr_t ya = (uintptr_t)yo;
                if (ya % 8 == 0) {
                    *reinterpret_cast<uint2*>(yo) = make_uint2(yw[0], yw[1]);
                } else if (ya % 4 == 0) {
                    reinterpret_cast<uint32_t*>(yo)[0] = yw[0];
                    reinterpret_cast<uint32_t*>(yo)[1] = yw[1];
                } else {
                    yo[0] = (uint16_t)(yw[0] & 0xFFFFu);
                    *reinterpret_cast<uint32_t*>(yo + 1) = __byte_perm(yw[0], yw[1], 0x5432);
                    yo[3] = (uint16_t)(yw[1] >> 16);
                }
                if (io) {
                    if ((uintptr_t)io % 16 == 0) {
                        reinterpret_cast<int4*>(io)[0] = make_int4(off[0], 0, off[1], 0);
                        reinterpret_cast<int4*>(io)[1] = make_int4(off[2], 0, off[3], 0);
                    } else {
                        io[0] = off[0];
                        *reinterpret_cast<int4*>(io + 1) = make_int4(off[1], 0, off[2], 0);
                        io[3] = off[3];
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (ow0 + e >= g.OW) break;
                    yo[e] = (uint16_t)((yw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
                    if (io) io[e] = off[e];
                }
            }
        }
    };

    int sl = 0;   // slices consumed so far
    for (int od = od0; od <= od0 + nd; ++od) {
#pragma unroll
        for (int i = 0; i < SD; ++i) {
            const bool role_cur = (od < od0 + nd) && (i < KD);
            const bool role_prev = (od > od0) && (SD + i < KD);
            if (!role_cur && !role_prev) continue;
            const int stage = sl % NS;
            const uint32_t parity = (uint32_t)((sl / NS) & 1);
            if (!failed && !mbar_wait(smem_addr(&bars[stage]), parity, wait_limit)) {
                failed = true;
                if (tid == 0) s_fail_at = sl;
                atomicOr(&g_mp3d_device_error, kErrPipelineTimeout);
            }
            const unsigned char* buf = stages + stage * stage_stride;
            // a clamped slice: its code offset from the nominal one
            const int ddelta = PAD ? slice_d(sl) - slice_nom(sl) : 0;
            uint32_t hv[TOH][2], hc[TOH][2];
#pragma unroll
            for (int j = 0; j < TOH; ++j) hv[j][0] = hv[j][1] = hc[j][0] = hc[j][1] = 0;
            if (nh > 0) {
                const int nrows = (nh - 1) * SH + KH;
                const int rbase = tl * TOH * SH;
#pragma unroll
                for (int r = 0; r < (TOH - 1) * SH + KH; ++r) {
                    if (r >= nrows) break;
                    // nominal input row oh0*SH - ph + r, read from the nearest row that exists
                    int srow = rbase + r, hdelta = 0;
                    if constexpr (PAD) {
                        const int hn = oh0 * SH - ph + r;
                        const int hs = min(max(hn, 0), g.H - 1);
                        hdelta = hs - hn;
                        srow = hs - r0;
                    }
                    const unsigned char* row = buf + (srow * g.W + w0) * sizeof(T);
                    const uint4 raw = *reinterpret_cast<const uint4*>(row);
                    uint32_t e8 = 0;
                    if (PAD && pw) {
                        // the element before the chunk (window 4c starts at 8c - 1);
                        // at the left edge, element 8c itself
                        e8 = c > 0 ? *reinterpret_cast<const unsigned short*>(row - 2) : raw.x;
                    } else if (KW > 2 && has_extra) {
                        // the element after the chunk (with floor output sizes the
                        // window that needs it past the last column is never written)
                        e8 = *reinterpret_cast<const unsigned short*>(row + 16);
                    }
                    poison = Pair<T>::poison(poison, raw.x);
                    poison = Pair<T>::poison(poison, raw.y);
                    poison = Pair<T>::poison(poison, raw.z);
                    poison = Pair<T>::poison(poison, raw.w);
                    if (KW > 2) poison = Pair<T>::poison(poison, e8);
                    uint32_t wv[2], wc[2];
                    if (PAD && pw) {
                        // windows 4c..4c+3 over elements 8c-1..8c+7: lanes
                        // (e-1, e1), (e0, e2), (e1, e3) and (e3, e5), (e4, e6), (e5, e7);
                        // at the left edge e-1 is e0 with e0's code
                        wv[0] = __byte_perm(e8, raw.x, 0x7610);
                        wc[0] = c > 0 ? 0u : 1u;
                        merge2<T>(wv[0], wc[0], __byte_perm(raw.x, raw.y, 0x5410), 1u * kLanes);
                        merge2<T>(wv[0], wc[0], __byte_perm(raw.x, raw.y, 0x7632), 2u * kLanes);
                        wv[1] = __byte_perm(raw.y, raw.z, 0x7632);
                        wc[1] = 0;
                        merge2<T>(wv[1], wc[1], __byte_perm(raw.z, raw.w, 0x5410), 1u * kLanes);
                        merge2<T>(wv[1], wc[1], __byte_perm(raw.z, raw.w, 0x7632), 2u * kLanes);
                    } else {
                        wv[0] = __byte_perm(raw.x, raw.y, 0x5410);
                        wc[0] = 0;
                        merge2<T>(wv[0], wc[0], __byte_perm(raw.x, raw.y, 0x7632), 1u * kLanes);
                        wv[1] = __byte_perm(raw.z, raw.w, 0x5410);
                        wc[1] = 0;
                        merge2<T>(wv[1], wc[1], __byte_perm(raw.z, raw.w, 0x7632), 1u * kLanes);
                        if (KW > 2) {
                            merge2<T>(wv[0], wc[0], __byte_perm(raw.y, raw.z, 0x5410), 2u * kLanes);
                            merge2<T>(wv[1], wc[1], __byte_perm(raw.w, e8, 0x5410), 2u * kLanes);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < TOH; ++j) {
                        const int hl = r - j * SH;
                        if (hl < 0 || hl >= KH) continue;
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            if (hl == 0) {
                                hv[j][k] = wv[k];
                                hc[j][k] = wc[k] | ((uint32_t)hdelta << 2) * kLanes;
                            } else {
                                merge2<T>(hv[j][k], hc[j][k], wv[k], wc[k] | ((uint32_t)(hl + hdelta) << 2) * kLanes);
                            }
                        }
                    }
                }
            }
            // Every thread is done reading this stage: refill it.
            __syncthreads();
            if (tid == 0 && sl + NS < nslices && !failed) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                const uint32_t bar = smem_addr(&bars[stage]);
                mbar_expect_tx(bar, span_bytes);
                bulk_g2s(smem_addr(stages + stage * stage_stride),
                         band_src + (long long)slice_d(sl + NS) * HW, span_bytes, bar);
            }
            ++sl;
#pragma unroll
            for (int j = 0; j < TOH; ++j)
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    if (role_prev)
                        merge2<T>(pv[j][k], pc[j][k], hv[j][k], hc[j][k] | ((uint32_t)(SD + i + ddelta) << 4) * kLanes);
                    if (role_cur) {
                        if (i == 0) {
                            cv[j][k] = hv[j][k];
                            cc[j][k] = hc[j][k] | ((uint32_t)ddelta << 4) * kLanes;
                        } else {
                            merge2<T>(cv[j][k], cc[j][k], hv[j][k], hc[j][k] | ((uint32_t)(i + ddelta) << 4) * kLanes);
                        }
                    }
                }
            if (role_prev && SD + i == KD - 1 && !failed) write_out(od - 1, pv, pc);
            if (role_cur && i == KD - 1 && !failed) write_out(od, cv, cc);
        }
#pragma unroll
        for (int j = 0; j < TOH; ++j)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                pv[j][k] = cv[j][k];
                pc[j][k] = cc[j][k];
            }
    }
    // After thread 0's wait gave up, let the copies still in flight land
    // before the CTA exits (these waits keep the normal bound).
    if (failed && tid == 0) {
        for (int k = s_fail_at; k < s_fail_at + NS && k < nslices; ++k)
            mbar_wait(smem_addr(&bars[k % NS]), (uint32_t)((k / NS) & 1), kWaitLimit);
    }
}

// ------------------------------------------------------------------ 2x2x2 tiling
// Windows 2x2x2 with stride 2 that tile the input exactly, rows that split
// into 16-byte chunks. One thread per run of four windows of one window row
// (od, oh): four 16-byte loads (input rows (dd, hh) of the run, straight
// from global memory), packed two-window compares (W, then H, then D; a
// strictly greater value replaces, so the first occurrence wins), one 8-byte
// store of the four maxima and two 16-byte stores of their indices. When a
// NaN or an infinity was loaded, the four windows are rescanned exactly from
// the loaded rows with the scalar rule.
template <typename T, bool VO = false>
__global__ void __launch_bounds__(256)
k_fwd_k2s2(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g,
           FastDiv fSpr, FastDiv fOH) {
    constexpr int NW = 4;
    const int HW = g.H * g.W;
    const int spr = g.OW / NW;
    const int nseg = g.ovol / NW;
    for (long long p = blockIdx.y; p < g.P; p += gridDim.y) {
        const T* xp = x + p * g.vol;
        for (int sg = blockIdx.x * blockDim.x + threadIdx.x; sg < nseg; sg += gridDim.x * blockDim.x) {
            const int row = fSpr.div(sg);
            const int ow0 = (sg - row * spr) * NW;
            const int od = fOH.div(row);
            const int oh = row - od * g.OH;
            const int base = 2 * od * HW + 2 * oh * g.W + 2 * ow0;
            uint4 r[4];
#pragma unroll
            for (int dh = 0; dh < 4; ++dh)
                r[dh] = __ldg(reinterpret_cast<const uint4*>(xp + base + (dh >> 1) * HW + (dh & 1) * g.W));
            uint32_t poison = 0;
#pragma unroll
            for (int dh = 0; dh < 4; ++dh) {
                poison = Pair<T>::poison(poison, r[dh].x);
                poison = Pair<T>::poison(poison, r[dh].y);
                poison = Pair<T>::poison(poison, r[dh].z);
                poison = Pair<T>::poison(poison, r[dh].w);
            }
            // per row: lanes (window 2k, window 2k+1), code wl | hl << 1 | dl << 2
            uint32_t mv[4][2], mc[4][2];
#pragma unroll
            for (int dh = 0; dh < 4; ++dh) {
                const uint32_t cb = (uint32_t)(((dh >> 1) << 2) | ((dh & 1) << 1)) * kLanes;
                mv[dh][0] = __byte_perm(r[dh].x, r[dh].y, 0x5410);
                mc[dh][0] = cb;
                merge2<T>(mv[dh][0], mc[dh][0], __byte_perm(r[dh].x, r[dh].y, 0x7632), cb | kLanes);
                mv[dh][1] = __byte_perm(r[dh].z, r[dh].w, 0x5410);
                mc[dh][1] = cb;
                merge2<T>(mv[dh][1], mc[dh][1], __byte_perm(r[dh].z, r[dh].w, 0x7632), cb | kLanes);
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                merge2<T>(mv[0][k], mc[0][k], mv[1][k], mc[1][k]);   // h within d = 0
                merge2<T>(mv[2][k], mc[2][k], mv[3][k], mc[3][k]);   // h within d = 1
                merge2<T>(mv[0][k], mc[0][k], mv[2][k], mc[2][k]);   // d
            }
            const long long o0 = p * (long long)g.ovol + (long long)sg * NW;
            int64_t iv[NW];
            uint2 yv = make_uint2(mv[0][0], mv[0][1]);
            if (Pair<T>::is_poisoned(poison)) {
                // exact scan of each window from the loaded rows (d, h, w order)
                uint32_t yb[NW];
#pragma unroll
                for (int k = 0; k < NW; ++k) {
                    uint32_t bb = 0, bc = 0;
                    float m = 0.0f;
#pragma unroll
                    for (int dh = 0; dh < 4; ++dh) {
                        const uint32_t wd = k == 0 ? r[dh].x : k == 1 ? r[dh].y : k == 2 ? r[dh].z : r[dh].w;
#pragma unroll
                        for (int ww = 0; ww < 2; ++ww) {
                            const uint32_t b = (wd >> (16 * ww)) & 0xFFFFu;
                            const uint16_t b16 = (uint16_t)b;
                            const float v = Elem<T>::to_f(*reinterpret_cast<const T*>(&b16));
                            if ((dh == 0 && ww == 0) || beats(v, m)) {
                                m = v;
                                bb = b;
                                bc = (uint32_t)(((dh >> 1) << 2) | ((dh & 1) << 1) | ww);
                            }
                        }
                    }
                    yb[k] = bb;
                    iv[k] = base + (int)(bc >> 2) * HW + (int)((bc >> 1) & 1) * g.W + 2 * k + (int)(bc & 1);
                }
                yv = make_uint2(yb[0] | yb[1] << 16, yb[2] | yb[3] << 16);
            } else {
#pragma unroll
                for (int k = 0; k < NW; ++k) {
                    const uint32_t code = (mc[0][k >> 1] >> (16 * (k & 1))) & 7u;
                    iv[k] = base + (int)(code >> 2) * HW + (int)((code >> 1) & 1) * g.W + 2 * k +
                            (int)(code & 1);
                }
            }
            *reinterpret_cast<uint2*>(y + o0) = yv;
            if (!VO && idx) {   // VO: values only, the codes are never used
                int4* id = reinterpret_cast<int4*>(idx + o0);
                id[0] = make_int4((int)iv[0], (int)(iv[0] >> 32), (int)iv[1], (int)(iv[1] >> 32));
                id[1] = make_int4((int)iv[2], (int)(iv[2] >> 32), (int)iv[3], (int)(iv[3] >> 32));
            }
        }
    }
}

// Window shapes with a compiled stride-2 kernel: (kd, sd, kh, sh, kw), sw = 2.
static int s2_variant(const Geo& g) {
    if (g.adaptive || g.sw != 2) return -1;
    if (g.kd == 2 && g.sd == 2 && g.kh == 2 && g.sh == 2 && g.kw == 2) return 0;
    if (g.kd == 3 && g.sd == 2 && g.kh == 3 && g.sh == 2 && g.kw == 3) return 1;
    return -1;
}

bool fwd_s2_supported(const Geo& g, int dtype, bool aligned16) {
    if (!((dtype == F16 || dtype == BF16) && s2_variant(g) >= 0 && g.W % 8 == 0 && g.W <= 1024 && aligned16))
        return false;
    if (g.dd != 1 || g.dh != 1 || g.dw != 1) return false;
    // floor output sizes (no ceil-mode window past the input)
    if (g.OD != (g.D + 2 * g.pd - g.kd) / g.sd + 1 || g.OH != (g.H + 2 * g.ph - g.kh) / g.sh + 1 ||
        g.OW != (g.W + 2 * g.pw - g.kw) / g.sw + 1)
        return false;
    // padding: 3x3x3 windows with stride 2, at most one position per side
    if (g.pd || g.ph || g.pw) return s2_variant(g) == 1 && g.pd <= 1 && g.ph <= 1 && g.pw <= 1;
    return true;
}

template <typename T, int KD, int SD, int KH, int SH, int KW, int PADC = 0, bool VO = false>
static cudaError_t fwd_s2_t(const void* x, void* y, int64_t* idx, const Geo& g, int sms,
                            cudaStream_t s) {
    constexpr int TOH = 4, NS = 2;
    const int nc = g.W / 8;
    const int nt = (g.OH + TOH - 1) / TOH;
    // Band of G tiles: at most 128 threads and 16 KB of input rows per stage.
    int G = 128 / nc;
    if (G > nt) G = nt;
    while (G > 1 && ((long long)((G * TOH - 1) * SH + KH) * g.W * sizeof(T)) > 16384) --G;
    const int nbands = (nt + G - 1) / G;
    // Split output depths into groups until there are about 4 CTAs per SM
    // (the groups re-read the slices their windows share; on the padded
    // 8x64x16x56x56 fp16 forward: 8 per SM 26.6 us, 4 per SM 24.6 us).
    const long long base = g.P * nbands;
    const long long target = (long long)sms * 4;
    long long want = (target + base - 1) / base;
    if (want < 1) want = 1;
    if (want > g.OD) want = g.OD;
    const int odg = (int)((g.OD + want - 1) / want);
    const int nq = (g.OD + odg - 1) / odg;
    const int band_rows = (G * TOH - 1) * SH + KH;
    const size_t stage = ((size_t)band_rows * g.W * sizeof(T) + 127) / 128 * 128;
    const size_t smem = NS * stage + NS * 8;
    auto kern = k_fwd_s2<T, KD, SD, KH, SH, KW, TOH, NS, PADC, VO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long blocks = g.P * nq * nbands;
    kern<<<(unsigned)blocks, nc * G, smem, s>>>((const T*)x, (T*)y, idx, g, odg, nq, G, nbands, nc,
                                                 pipeline_wait_limit());
    return cudaGetLastError();
}

template <typename T>
static cudaError_t fwd_s2_dispatch(const void* x, void* y, int64_t* idx, const Geo& g, int sms,
                                   cudaStream_t s) {
    switch (g.pd | g.ph << 1 | g.pw << 2) {
    case 0: break;
    case 1: return fwd_s2_t<T, 3, 2, 3, 2, 3, 1>(x, y, idx, g, sms, s);
    case 2: return fwd_s2_t<T, 3, 2, 3, 2, 3, 2>(x, y, idx, g, sms, s);
    case 3: return fwd_s2_t<T, 3, 2, 3, 2, 3, 3>(x, y, idx, g, sms, s);
    case 4: return fwd_s2_t<T, 3, 2, 3, 2, 3, 4>(x, y, idx, g, sms, s);
    case 5: return fwd_s2_t<T, 3, 2, 3, 2, 3, 5>(x, y, idx, g, sms, s);
    case 6: return fwd_s2_t<T, 3, 2, 3, 2, 3, 6>(x, y, idx, g, sms, s);
    default: return fwd_s2_t<T, 3, 2, 3, 2, 3, 7>(x, y, idx, g, sms, s);
    }
    // 2x2x2 windows tiling the input: direct loads, one thread per four windows
    if (s2_variant(g) == 0 && g.D == 2 * g.OD && g.H == 2 * g.OH && g.W == 2 * g.OW &&
        g.OW % 4 == 0 && (uintptr_t)y % 8 == 0 && (uintptr_t)idx % 16 == 0) {
        const int nseg = g.ovol / 4;
        dim3 grid((unsigned)((nseg + 255) / 256), (unsigned)(g.P < 65535 ? g.P : 65535));
        auto kern = idx ? k_fwd_k2s2<T, false> : k_fwd_k2s2<T, true>;
        kern<<<grid, 256, 0, s>>>((const T*)x, (T*)y, idx, g, FastDiv((uint32_t)(g.OW / 4)),
                                  FastDiv((uint32_t)g.OH));
        return cudaGetLastError();
    }
    // values only (no index output): compiled without the winners' codes,
    // which the packed merges otherwise carry in a second word
    const int v = s2_variant(g);
    if (v < 0) return cudaErrorNotSupported;
    switch (v + (idx ? 0 : 2)) {
    case 0: return fwd_s2_t<T, 2, 2, 2, 2, 2>(x, y, idx, g, sms, s);
    case 1: return fwd_s2_t<T, 3, 2, 3, 2, 3>(x, y, idx, g, sms, s);
    case 2: return fwd_s2_t<T, 2, 2, 2, 2, 2, 0, true>(x, y, idx, g, sms, s);
    case 3: return fwd_s2_t<T, 3, 2, 3, 2, 3, 0, true>(x, y, idx, g, sms, s);
    default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_fwd_s2(const void* x, void* y, int64_t* idx, const Geo& g, int dtype, int sms,
                          cudaStream_t s) {
    if (dtype == F16) return fwd_s2_dispatch<__half>(x, y, idx, g, sms, s);
    if (dtype == BF16) return fwd_s2_dispatch<__nv_bfloat16>(x, y, idx, g, sms, s);
    return cudaErrorNotSupported;
}

}  // namespace mp3d

namespace mp3d {

cudaError_t read_device_error(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_mp3d_device_error, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    unsigned int more = 0;
    e = read_roll_fwd_error(&more, clear);      // the flag of the kernels in fwd_roll.cu
    if (e != cudaSuccess) return e;
    *flags |= more;
    if (!clear) return cudaSuccess;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_mp3d_device_error, &zero, sizeof(unsigned int));
}

}  // namespace mp3d
