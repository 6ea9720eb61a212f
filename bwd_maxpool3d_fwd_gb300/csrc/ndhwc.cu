// Channels-last (NDHWC) layout: x [N, D, H, W, C], y and idx
// [N, OD, OH, OW, C], grad_in like x. Windows, ties, NaN rule, index form
// (the spatial offset d*H*W + h*W + w of the winner in its own (n, c)
// volume) and the backward's summation order are those of the NCDHW entry
// points (teenygrad docs "Struct Maxpool3dForward"; FlagGems-Experimental
// PR #308 Summary), so the results are the NCDHW results permuted.
//
// Channels are the innermost axis, so a thread handles one 16-byte chunk
// of VEC channels at one spatial position: every window position is one
// 16-byte load across channels, and neighbouring threads read neighbouring
// chunks (coalesced). Channel counts that are not a multiple of VEC, or
// buffers off a 16-byte boundary, take the same kernels with VEC = 1.
#include "internal.h"

namespace mp3d {

// Forward: one thread per (n, od, oh, ow, channel chunk); scans the window
// positions in ascending (d, h, w) order, per channel keeping the first
// element that beats the running maximum.
template <typename T, int VEC, bool ADAPTIVE>
__global__ void __launch_bounds__(256)
k_fwd_ndhwc(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g, int C) {
    const int nch = C / VEC;                         // chunks per position
    const long long total = (long long)g.P * g.ovol * nch;   // g.P = N here
    const int HW = g.H * g.W;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int ch = (int)(t % nch);
        long long r = t / nch;
        const int ow = (int)(r % g.OW);
        r /= g.OW;
        const int oh = (int)(r % g.OH);
        r /= g.OH;
        const int od = (int)(r % g.OD);
        const long long n = r / g.OD;
        const int ds = win_start(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int de = win_end(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int hs = win_start(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int he = win_end(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int ws = win_start(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        const int we = win_end(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        const T* xn = x + n * (long long)g.vol * C + ch * VEC;
        float m[VEC];
        T bv[VEC];
        int best[VEC];
        bool first = true;
        for (int d = ds; d < de; ++d)
            for (int h = hs; h < he; ++h)
                for (int w = ws; w < we; ++w) {
                    const int s = d * HW + h * g.W + w;
                    T v[VEC];
                    if constexpr (VEC * sizeof(T) == 16) {
                        Vec16<T> c;
                        c.u = __ldg(reinterpret_cast<const uint4*>(xn + (long long)s * C));
#pragma unroll
                        for (int k = 0; k < VEC; ++k) v[k] = c.e[k];
                    } else {
#pragma unroll
                        for (int k = 0; k < VEC; ++k) v[k] = xn[(long long)s * C + k];
                    }
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        const float f = Elem<T>::to_f(v[k]);
                        if (first || beats(f, m[k])) {
                            m[k] = f;
                            bv[k] = v[k];
                            best[k] = s;
                        }
                    }
                    first = false;
                }
        const long long o = (((n * g.OD + od) * g.OH + oh) * (long long)g.OW + ow) * C + ch * VEC;
        if constexpr (VEC * sizeof(T) == 16) {
            Vec16<T> c;
#pragma unroll
            for (int k = 0; k < VEC; ++k) c.e[k] = bv[k];
            *reinterpret_cast<uint4*>(y + o) = c.u;
        } else {
#pragma unroll
            for (int k = 0; k < VEC; ++k) y[o + k] = bv[k];
        }
        if (idx) {
            if constexpr (VEC * sizeof(T) == 16) {
                int4* id = reinterpret_cast<int4*>(idx + o);
#pragma unroll
                for (int q = 0; q < VEC / 2; ++q) id[q] = make_int4(best[2 * q], 0, best[2 * q + 1], 0);
            } else {
#pragma unroll
                for (int k = 0; k < VEC; ++k) idx[o + k] = best[k];
            }
        }
    }
}

// Forward for 16-bit types, packed: one thread per (n, od, oh, ow, 16-byte
// chunk of 8 channels). The chunk is four words of two channels each; the
// window is scanned in (d, h, w) order and each word is merged with set.gt on
// f16x2 / bf16x2 (a later element replaces only when strictly greater, so
// the first occurrence is kept and +0 / -0 tie). Each lane carries the
// winner's offset from the window's first element, d_l*H*W + h_l*W + w_l
// (below 65536, checked by the launcher). NaN and infinities: a running
// x*0 + acc turns NaN once either was seen, and the chunk is then recomputed
// with the exact scalar scan.
template <typename T, bool ADAPTIVE>
__global__ void __launch_bounds__(256)
k_fwd_ndhwc_pk(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g, int C) {
    constexpr int VEC = 8;
    const int nch = C / VEC;
    const long long total = (long long)g.P * g.ovol * nch;
    const int HW = g.H * g.W;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int ch = (int)(t % nch);
        long long r = t / nch;
        const int ow = (int)(r % g.OW);
        r /= g.OW;
        const int oh = (int)(r % g.OH);
        r /= g.OH;
        const int od = (int)(r % g.OD);
        const long long n = r / g.OD;
        const int ds = win_start(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int de = win_end(od, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int hs = win_start(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int he = win_end(oh, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int ws = win_start(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        const int we = win_end(ow, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        const T* xn = x + n * (long long)g.vol * C + ch * VEC;
        const int origin = ds * HW + hs * g.W + ws;
        uint32_t mv[4], mc[4] = {0u, 0u, 0u, 0u}, pz = 0u;
        {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(xn + (long long)origin * C));
            mv[0] = u.x; mv[1] = u.y; mv[2] = u.z; mv[3] = u.w;
        }
        for (int d = ds; d < de; ++d)
            for (int h = hs; h < he; ++h) {
                const int rowoff = (d - ds) * HW + (h - hs) * g.W;
                const T* row = xn + ((long long)d * HW + h * g.W) * C;
                for (int w = ws; w < we; ++w) {
                    const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + (long long)w * C));
                    const uint32_t code = (uint32_t)(rowoff + w - ws) * 0x00010001u;
                    merge2<T>(mv[0], mc[0], u.x, code);
                    merge2<T>(mv[1], mc[1], u.y, code);
                    merge2<T>(mv[2], mc[2], u.z, code);
                    merge2<T>(mv[3], mc[3], u.w, code);
                    pz = Pair<T>::poison(pz, u.x);
                    pz = Pair<T>::poison(pz, u.y);
                    pz = Pair<T>::poison(pz, u.z);
                    pz = Pair<T>::poison(pz, u.w);
                }
            }
        const long long o = (((n * g.OD + od) * g.OH + oh) * (long long)g.OW + ow) * C + ch * VEC;
        if (Pair<T>::is_poisoned(pz)) {
            // exact scalar scan of the chunk's eight channels
            for (int k = 0; k < VEC; ++k) {
                int best = origin;
                float m = Elem<T>::to_f(xn[(long long)origin * C + k]);
                for (int d = ds; d < de; ++d)
                    for (int h = hs; h < he; ++h)
                        for (int w = ws; w < we; ++w) {
                            const int sidx = d * HW + h * g.W + w;
                            const float f = Elem<T>::to_f(xn[(long long)sidx * C + k]);
                            if (beats(f, m)) {
                                m = f;
                                best = sidx;
                            }
                        }
                y[o + k] = xn[(long long)best * C + k];
                if (idx) idx[o + k] = best;
            }
            continue;
        }
        *reinterpret_cast<uint4*>(y + o) = make_uint4(mv[0], mv[1], mv[2], mv[3]);
        if (idx) {
            int4* id = reinterpret_cast<int4*>(idx + o);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                id[q] = make_int4(origin + (int)(mc[q] & 0xFFFFu), 0, origin + (int)(mc[q] >> 16), 0);
        }
    }
}

// Backward: one thread per (n, d, h, w, channel chunk); walks the covering
// windows in ascending (od, oh, ow) order and, per channel, sums the
// gradients of the windows whose stored index is this position (first
// term as the initial value, binary32, one rounding; +0 if none).
template <typename T, int VEC, bool ADAPTIVE>
__global__ void __launch_bounds__(256)
k_bwd_ndhwc(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi, Geo g,
            int C) {
    const int nch = C / VEC;
    const long long total = (long long)g.P * g.vol * nch;
    const int HW = g.H * g.W;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int ch = (int)(t % nch);
        const long long r = t / nch;
        const long long n = r / g.vol;
        const int s = (int)(r - n * g.vol);
        const int d = s / HW;
        const int h = (s - d * HW) / g.W;
        const int w = s - d * HW - h * g.W;
        float acc[VEC];
        bool any[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
            acc[k] = 0.0f;
            any[k] = false;
        }
        const int d1 = cover_hi(d, g.D, g.OD, g.kd, g.sd, ADAPTIVE);
        const int h1 = cover_hi(h, g.H, g.OH, g.kh, g.sh, ADAPTIVE);
        const int w1 = cover_hi(w, g.W, g.OW, g.kw, g.sw, ADAPTIVE);
        for (int od = cover_lo(d, g.D, g.OD, g.kd, g.sd, ADAPTIVE); od <= d1; ++od)
            for (int oh = cover_lo(h, g.H, g.OH, g.kh, g.sh, ADAPTIVE); oh <= h1; ++oh)
                for (int ow = cover_lo(w, g.W, g.OW, g.kw, g.sw, ADAPTIVE); ow <= w1; ++ow) {
                    const long long o =
                        (((n * g.OD + od) * g.OH + oh) * (long long)g.OW + ow) * C + ch * VEC;
                    int64_t j[VEC];
                    T gv[VEC];
                    if constexpr (VEC * sizeof(T) == 16) {
                        const uint4* ip = reinterpret_cast<const uint4*>(idx + o);
#pragma unroll
                        for (int q = 0; q < VEC / 2; ++q) {
                            const uint4 u = __ldg(ip + q);
                            j[2 * q] = (int64_t)((uint64_t)u.y << 32 | u.x);
                            j[2 * q + 1] = (int64_t)((uint64_t)u.w << 32 | u.z);
                        }
                        Vec16<T> c;
                        c.u = *reinterpret_cast<const uint4*>(go + o);
#pragma unroll
                        for (int k = 0; k < VEC; ++k) gv[k] = c.e[k];
                    } else {
#pragma unroll
                        for (int k = 0; k < VEC; ++k) {
                            j[k] = __ldg(idx + o + k);
                            gv[k] = go[o + k];
                        }
                    }
#pragma unroll
                    for (int k = 0; k < VEC; ++k)
                        if (j[k] == s) {
                            const float v = Elem<T>::to_f(gv[k]);
                            acc[k] = any[k] ? acc[k] + v : v;
                            any[k] = true;
                        }
                }
        const long long e = r * C + ch * VEC;
        T out[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) out[k] = Elem<T>::from_f(any[k] ? acc[k] : 0.0f);
        if constexpr (VEC * sizeof(T) == 16) {
            Vec16<T> c;
#pragma unroll
            for (int k = 0; k < VEC; ++k) c.e[k] = out[k];
            *reinterpret_cast<uint4*>(gi + e) = c.u;
        } else {
#pragma unroll
            for (int k = 0; k < VEC; ++k) gi[e + k] = out[k];
        }
    }
}

namespace {

int grid_of(long long work, int sms) {
    long long b = (work + 255) / 256;
    const long long cap = (long long)sms * 8;
    return (int)(b < 1 ? 1 : b > cap ? cap : b);
}

// 16-byte chunks when C holds whole chunks and every buffer is aligned.
bool chunked(int C, int es, std::initializer_list<const void*> ptrs) {
    if (C % (16 / es) != 0) return false;
    for (const void* p : ptrs)
        if (p && (uintptr_t)p % 16 != 0) return false;
    return true;
}

template <typename T, int VEC>
cudaError_t fwd_t(const void* x, void* y, int64_t* idx, const Geo& g, int C, int sms, cudaStream_t s) {
    const long long work = (long long)g.P * g.ovol * (C / VEC);
    if (g.adaptive)
        k_fwd_ndhwc<T, VEC, true><<<grid_of(work, sms), 256, 0, s>>>((const T*)x, (T*)y, idx, g, C);
    else
        k_fwd_ndhwc<T, VEC, false><<<grid_of(work, sms), 256, 0, s>>>((const T*)x, (T*)y, idx, g, C);
    return cudaGetLastError();
}

template <typename T, int VEC>
cudaError_t bwd_t(const void* go, const int64_t* idx, void* gi, const Geo& g, int C, int sms,
                  cudaStream_t s) {
    const long long work = (long long)g.P * g.vol * (C / VEC);
    if (g.adaptive)
        k_bwd_ndhwc<T, VEC, true><<<grid_of(work, sms), 256, 0, s>>>((const T*)go, idx, (T*)gi, g, C);
    else
        k_bwd_ndhwc<T, VEC, false><<<grid_of(work, sms), 256, 0, s>>>((const T*)go, idx, (T*)gi, g, C);
    return cudaGetLastError();
}

// The winner's offset from its window's first element fits a 16-bit lane
// for every window of the geometry.
bool rel_fits(const Geo& g) {
    long long kd = g.kd, kh = g.kh, kw = g.kw;
    if (g.adaptive) {
        auto longest = [](int I, int O) {
            long long m = 0;
            for (int i = 0; i < O; ++i) {
                const long long l = ((long long)(i + 1) * I + O - 1) / O - (long long)i * I / O;
                m = l > m ? l : m;
            }
            return m;
        };
        kd = longest(g.D, g.OD);
        kh = longest(g.H, g.OH);
        kw = longest(g.W, g.OW);
    }
    return (kd - 1) * g.H * g.W + (kh - 1) * g.W + (kw - 1) < 65536;
}

template <typename T>
cudaError_t fwd_dispatch(const void* x, void* y, int64_t* idx, const Geo& g, int C, int sms,
                         cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    if (chunked(C, sizeof(T), {x, y, idx})) {
        if constexpr (sizeof(T) == 2) {
            if (rel_fits(g)) {
                const long long work = (long long)g.P * g.ovol * (C / VEC);
                if (g.adaptive)
                    k_fwd_ndhwc_pk<T, true><<<grid_of(work, sms), 256, 0, s>>>((const T*)x, (T*)y, idx, g, C);
                else
                    k_fwd_ndhwc_pk<T, false><<<grid_of(work, sms), 256, 0, s>>>((const T*)x, (T*)y, idx, g, C);
                return cudaGetLastError();
            }
        }
        return fwd_t<T, VEC>(x, y, idx, g, C, sms, s);
    }
    return fwd_t<T, 1>(x, y, idx, g, C, sms, s);
}

template <typename T>
cudaError_t bwd_dispatch(const void* go, const int64_t* idx, void* gi, const Geo& g, int C, int sms,
                         cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    if (chunked(C, sizeof(T), {go, idx, gi})) return bwd_t<T, VEC>(go, idx, gi, g, C, sms, s);
    return bwd_t<T, 1>(go, idx, gi, g, C, sms, s);
}

}  // namespace

cudaError_t launch_fwd_ndhwc(const void* x, void* y, int64_t* idx, const Geo& g, int C, int dtype,
                             int sms, cudaStream_t s) {
    switch (dtype) {
    case F32: return fwd_dispatch<float>(x, y, idx, g, C, sms, s);
    case F16: return fwd_dispatch<__half>(x, y, idx, g, C, sms, s);
    default: return fwd_dispatch<__nv_bfloat16>(x, y, idx, g, C, sms, s);
    }
}

cudaError_t launch_bwd_ndhwc(const void* go, const int64_t* idx, void* gi, const Geo& g, int C,
                             int dtype, int sms, cudaStream_t s) {
    switch (dtype) {
    case F32: return bwd_dispatch<float>(go, idx, gi, g, C, sms, s);
    case F16: return bwd_dispatch<__half>(go, idx, gi, g, C, sms, s);
    default: return bwd_dispatch<__nv_bfloat16>(go, idx, gi, g, C, sms, s);
    }
}

}  // namespace mp3d
