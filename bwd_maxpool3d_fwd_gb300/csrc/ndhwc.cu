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
#include <climits>
#include <cstring>

#include "internal.h"
#include "mp3d.h"

namespace mp3d {

// Divisors of a work index t = (((n * OD + od) * OH + oh) * OW + ow) * nch + ch
// (multiply-shift division; the launchers keep t below 2^31).
struct NdDecomp {
    FastDiv fc, fw, fh, fd;
};

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
// KH, KW > 0: every window is KH x KW in (h, w); each depth's KH * KW loads
// are issued together before they are merged (in order).
template <typename T, bool ADAPTIVE, int KH, int KW>
__global__ void __launch_bounds__(256, 4)
k_fwd_ndhwc_pk(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g, int C,
               NdDecomp dc) {
    constexpr int VEC = 8;
    const int nch = C / VEC;
    const int total = (int)(g.P * g.ovol * nch);
    const int HW = g.H * g.W;
    for (long long tt = blockIdx.x * (long long)blockDim.x + threadIdx.x; tt < total;
         tt += (long long)gridDim.x * blockDim.x) {
        const int t = (int)tt;
        int r = dc.fc.div(t);
        const int ch = t - r * nch;
        int r2 = dc.fw.div(r);
        const int ow = r - r2 * g.OW;
        r = dc.fh.div(r2);
        const int oh = r2 - r * g.OH;
        const int nn = dc.fd.div(r);
        const int od = r - nn * g.OD;
        const long long n = nn;
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
        auto take = [&](const uint4& u, uint32_t code) {
            merge2<T>(mv[0], mc[0], u.x, code);
            merge2<T>(mv[1], mc[1], u.y, code);
            merge2<T>(mv[2], mc[2], u.z, code);
            merge2<T>(mv[3], mc[3], u.w, code);
            pz = Pair<T>::poison(pz, u.x);
            pz = Pair<T>::poison(pz, u.y);
            pz = Pair<T>::poison(pz, u.z);
            pz = Pair<T>::poison(pz, u.w);
        };
        if constexpr (KH > 0 && KW > 0) {
            for (int d = ds; d < de; ++d) {
                const T* plane = xn + ((long long)d * HW + hs * g.W + ws) * C;
                uint4 u[KH * KW];
#pragma unroll
                for (int k = 0; k < KH * KW; ++k)
                    u[k] = __ldg(reinterpret_cast<const uint4*>(plane + ((long long)(k / KW) * g.W + k % KW) * C));
                const int dofs = (d - ds) * HW;
#pragma unroll
                for (int k = 0; k < KH * KW; ++k)
                    take(u[k], (uint32_t)(dofs + (k / KW) * g.W + k % KW) * 0x00010001u);
            }
        } else {
            for (int d = ds; d < de; ++d)
                for (int h = hs; h < he; ++h) {
                    const int rowoff = (d - ds) * HW + (h - hs) * g.W;
                    const T* row = xn + ((long long)d * HW + h * g.W) * C;
                    for (int w = ws; w < we; ++w) {
                        const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + (long long)w * C));
                        take(u, (uint32_t)(rowoff + w - ws) * 0x00010001u);
                    }
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

// Forward for 16-bit types, packed, fixed windows whose consecutive depth
// windows share one slice (KD = SD + 1; 3x3x3 with stride 2, for one): one
// thread per (n, oh, ow, 16-byte chunk of 8 channels) walks the output
// depths. Each slice's KH x KW box is reduced once, in (h, w) order, to a
// best element and its (h, w) offset per lane (a later element replaces only
// when strictly greater); the slices of a window are then merged in depth
// order the same way, so the winner is the first maximum in (d, h, w) order.
// The slice a window shares with the next is reduced once and carried, which
// saves a third of the loads and one round of load latency per output. NaN
// and infinities: a running x*0 + acc per window; such chunks are recomputed
// with the exact scalar scan.
template <typename T, int KD, int SD, int KH, int KW>
__global__ void __launch_bounds__(256, 3)
k_fwd_ndhwc_dw(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g, int C) {
    static_assert(KD == SD + 1, "consecutive depth windows share one slice");
    constexpr int VEC = 8;
    const int nch = C / VEC;
    const long long total = (long long)g.P * g.OH * g.OW * nch;
    const int HW = g.H * g.W;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int ch = (int)(t % nch);
        long long r = t / nch;
        const int ow = (int)(r % g.OW);
        r /= g.OW;
        const int oh = (int)(r % g.OH);
        const long long n = r / g.OH;
        const int hs = oh * g.sh, ws = ow * g.sw;
        const T* xn = x + n * (long long)g.vol * C + ch * VEC;
        // slice d's box: best element and its (h, w) offset per lane, and a
        // running x*0 + acc
        auto slice = [&](int d, uint32_t (&sv)[4], uint32_t (&sc)[4], uint32_t& sp) {
            const T* plane = xn + ((long long)d * HW + hs * g.W + ws) * C;
            uint4 u[KH * KW];
#pragma unroll
            for (int k = 0; k < KH * KW; ++k)
                u[k] = __ldg(reinterpret_cast<const uint4*>(plane + ((long long)(k / KW) * g.W + k % KW) * C));
            sv[0] = u[0].x; sv[1] = u[0].y; sv[2] = u[0].z; sv[3] = u[0].w;
            sc[0] = sc[1] = sc[2] = sc[3] = 0u;
            sp = 0u;
#pragma unroll
            for (int k = 0; k < KH * KW; ++k) {
                if (k > 0) {
                    const uint32_t code = (uint32_t)((k / KW) * g.W + k % KW) * 0x00010001u;
                    merge2<T>(sv[0], sc[0], u[k].x, code);
                    merge2<T>(sv[1], sc[1], u[k].y, code);
                    merge2<T>(sv[2], sc[2], u[k].z, code);
                    merge2<T>(sv[3], sc[3], u[k].w, code);
                }
                sp = Pair<T>::poison(sp, u[k].x);
                sp = Pair<T>::poison(sp, u[k].y);
                sp = Pair<T>::poison(sp, u[k].z);
                sp = Pair<T>::poison(sp, u[k].w);
            }
        };
        uint32_t cv[4], cc[4], cp;           // the carried slice: first slice of window od
        slice(0, cv, cc, cp);
        for (int od = 0; od < g.OD; ++od) {
            const int d0 = od * SD;
            uint32_t mv[4] = {cv[0], cv[1], cv[2], cv[3]};
            uint32_t mc[4] = {cc[0], cc[1], cc[2], cc[3]};
            uint32_t pz = cp;
#pragma unroll
            for (int j = 1; j < KD; ++j) {
                uint32_t sv[4], sc[4], sp;
                slice(d0 + j, sv, sc, sp);
                const uint32_t dcode = (uint32_t)(j * HW) * 0x00010001u;
#pragma unroll
                for (int q = 0; q < 4; ++q) merge2<T>(mv[q], mc[q], sv[q], sc[q] + dcode);
                pz = Pair<T>::poison(pz, sp);
                if (j == KD - 1) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        cv[q] = sv[q];
                        cc[q] = sc[q];
                    }
                    cp = sp;
                }
            }
            const int origin = d0 * HW + hs * g.W + ws;
            const long long o = (((n * g.OD + od) * g.OH + oh) * (long long)g.OW + ow) * C + ch * VEC;
            if (Pair<T>::is_poisoned(pz)) {
                // exact scalar scan of the chunk's eight channels
                for (int k = 0; k < VEC; ++k) {
                    int best = origin;
                    float m = Elem<T>::to_f(xn[(long long)origin * C + k]);
                    for (int d = d0; d < d0 + KD; ++d)
                        for (int h = hs; h < hs + KH; ++h)
                            for (int w = ws; w < ws + KW; ++w) {
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
}

// Backward for fixed windows that tile the input exactly (K = S on every
// axis, each size a multiple of its window): every input lies in exactly
// one window, so its gradient is that window's gradient where the stored
// index names it and +0 elsewhere (a sum of one term is the term, -0
// included). One thread per (window, 16-byte chunk of channels) loads the
// chunk's gradients and indices once and writes the window's KD*KH*KW
// positions of the chunk with 16-byte stores.
template <typename T, int KD, int KH, int KW>
__global__ void __launch_bounds__(256)
k_bwd_ndhwc_tile(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi, Geo g,
                 int C, NdDecomp dc) {
    constexpr int VEC = 16 / sizeof(T);
    const int nch = C / VEC;
    const int total = (int)(g.P * g.ovol * nch);   // g.P = N here
    const int HW = g.H * g.W;
    for (long long tt = blockIdx.x * (long long)blockDim.x + threadIdx.x; tt < total;
         tt += (long long)gridDim.x * blockDim.x) {
        const int t = (int)tt;
        int r = dc.fc.div(t);
        const int ch = t - r * nch;
        int r2 = dc.fw.div(r);
        const int ow = r - r2 * g.OW;
        r = dc.fh.div(r2);
        const int oh = r2 - r * g.OH;
        const int nn = dc.fd.div(r);
        const int od = r - nn * g.OD;
        const long long n = nn;
        const long long o = (((n * g.OD + od) * g.OH + oh) * (long long)g.OW + ow) * C + ch * VEC;
        Vec16<T> gv;
        gv.u = *reinterpret_cast<const uint4*>(go + o);
        // the indices' low words; an index with a nonzero high word names no
        // position (all ones never equals an in-plane offset)
        unsigned lo[VEC];
#pragma unroll
        for (int q = 0; q < VEC / 2; ++q) {
            const uint4 iv = __ldg(reinterpret_cast<const uint4*>(idx + o + 2 * q));
            lo[2 * q] = iv.y == 0u ? iv.x : 0xFFFFFFFFu;
            lo[2 * q + 1] = iv.w == 0u ? iv.z : 0xFFFFFFFFu;
        }
        const int origin = (od * KD) * HW + (oh * KH) * g.W + ow * KW;
        T* gn = gi + n * (long long)g.vol * C + ch * VEC;
#pragma unroll
        for (int p = 0; p < KD * KH * KW; ++p) {
            const int off = origin + (p / (KH * KW)) * HW + ((p / KW) % KH) * g.W + p % KW;
            Vec16<T> out;
#pragma unroll
            for (int k = 0; k < VEC; ++k) out.e[k] = lo[k] == (unsigned)off ? gv.e[k] : Elem<T>::from_f(0.0f);
            *reinterpret_cast<uint4*>(gn + (long long)off * C) = out.u;
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

// Backward for fixed windows of stride 2 on every axis and length at most 4
// (so at most two windows cover a position along each axis: windows a - 1
// and a for the positions 2a, 2a + 1): one thread per (n, 2x2x2 block of
// input positions, CH channels). The thread streams the covering windows of
// its block, at most 8, in ascending (od, oh, ow) order, loading each
// window's CH indices and CH gradients once for all 8 positions, and sums for
// each position and channel the gradients of the windows whose index is
// that position (binary32, first term as the initial value, one rounding;
// +0 where none). Accumulators start at -0, the identity of binary32
// addition (x + -0 is x for every x, +0 and -0 included), so adding the
// first term to it gives the first term; a bit per position and channel
// records whether any term arrived.
// K > 0: every window is K long on every axis (the covering pairs of window
// and position are then known at compile time); 0: lengths from g. Four
// CTAs per SM for K = 3 (it spills a few registers there and is still
// faster: 1124 -> 1055 us on the 32x128x16x112x112 fp16 backward), three
// otherwise.
template <typename T, int CH, int K>
__global__ void __launch_bounds__(256, K == 3 ? 4 : 3)
k_bwd_ndhwc_blk(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi, Geo g,
                int C) {
    static_assert(CH == 2 || CH == 4, "2 or 4 channels per thread");
    const int nch = C / CH;
    const int BD = (g.D + 1) / 2, BH = (g.H + 1) / 2, BW = (g.W + 1) / 2;
    // blocks are taken in groups of 2x2x2 (neighbours share most of their
    // covering windows, so the group's loads of a window after the first
    // are served by L1): work index = ((n, group) * 8 + block in group) * nch + chunk
    const int GD = (BD + 1) / 2, GH = (BH + 1) / 2, GW = (BW + 1) / 2;
    const long long total = (long long)g.P * GD * GH * GW * 8 * nch;
    const int HW = g.H * g.W;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int ch = (int)(t % nch);
        long long r = t / nch;
        const int sub = (int)(r % 8);
        r /= 8;
        const int gw = (int)(r % GW);
        r /= GW;
        const int gh = (int)(r % GH);
        r /= GH;
        const int gd = (int)(r % GD);
        const long long n = r / GD;
        const int bd = 2 * gd + (sub >> 2), bh = 2 * gh + ((sub >> 1) & 1), bw = 2 * gw + (sub & 1);
        if (bd >= BD || bh >= BH || bw >= BW) continue;
        float acc[8][CH];
        unsigned any = 0u;                       // bit p * CH + k: position p, channel k has a term
#pragma unroll
        for (int p = 0; p < 8; ++p)
#pragma unroll
            for (int k = 0; k < CH; ++k) acc[p][k] = -0.0f;
        const int d0 = 2 * bd, h0 = 2 * bh, w0 = 2 * bw;
        const int s0 = d0 * HW + h0 * g.W + w0;  // in-plane offset of position 0
#pragma unroll
        for (int a = 0; a < 2; ++a) {
            const int od = bd - 1 + a;
            if (od < 0 || od >= g.OD) continue;
            // positions 2bd + i inside window od along d (window bd - 1 + a
            // covers position i when 2 - 2a + i < K)
            const int dm = K > 0 ? ((2 - 2 * a < K ? 1 : 0) | (3 - 2 * a < K && d0 + 1 < g.D ? 2 : 0))
                                 : ((d0 >= od * 2 && d0 < od * 2 + g.kd ? 1 : 0) |
                                    (d0 + 1 < g.D && d0 + 1 < od * 2 + g.kd ? 2 : 0));
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int oh = bh - 1 + b;
                if (oh < 0 || oh >= g.OH) continue;
                const int hm = K > 0 ? ((2 - 2 * b < K ? 1 : 0) | (3 - 2 * b < K && h0 + 1 < g.H ? 2 : 0))
                                     : ((h0 >= oh * 2 && h0 < oh * 2 + g.kh ? 1 : 0) |
                                        (h0 + 1 < g.H && h0 + 1 < oh * 2 + g.kh ? 2 : 0));
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int ow = bw - 1 + c;
                    if (ow < 0 || ow >= g.OW) continue;
                    const int wm = K > 0 ? ((2 - 2 * c < K ? 1 : 0) | (3 - 2 * c < K && w0 + 1 < g.W ? 2 : 0))
                                         : ((w0 >= ow * 2 && w0 < ow * 2 + g.kw ? 1 : 0) |
                                            (w0 + 1 < g.W && w0 + 1 < ow * 2 + g.kw ? 2 : 0));
                    if (!dm || !hm || !wm) continue;
                    const long long o = ((((n * g.OD + od) * g.OH + oh) * (long long)g.OW + ow) * C) + ch * CH;
                    // low words of the indices; an index with a nonzero high word
                    // names no position (all ones never equals an in-plane offset)
                    unsigned lo[CH];
#pragma unroll
                    for (int q = 0; q < CH / 2; ++q) {
                        const uint4 iv = __ldg(reinterpret_cast<const uint4*>(idx + o + 2 * q));
                        lo[2 * q] = iv.y == 0u ? iv.x : 0xFFFFFFFFu;
                        lo[2 * q + 1] = iv.w == 0u ? iv.z : 0xFFFFFFFFu;
                    }
                    float gv[CH];
                    {
                        T e[CH];
                        if constexpr (sizeof(T) * CH == 4) {
                            const unsigned u = *reinterpret_cast<const unsigned*>(go + o);
                            memcpy(e, &u, sizeof(u));
                        } else if constexpr (sizeof(T) * CH == 8) {
                            const uint2 u = *reinterpret_cast<const uint2*>(go + o);
                            memcpy(e, &u, sizeof(u));
                        } else {
                            const uint4 u = *reinterpret_cast<const uint4*>(go + o);
                            memcpy(e, &u, sizeof(u));
                        }
#pragma unroll
                        for (int k = 0; k < CH; ++k) gv[k] = Elem<T>::to_f(e[k]);
                    }
#pragma unroll
                    for (int p = 0; p < 8; ++p) {
                        const int i = p >> 2, j = (p >> 1) & 1, kk = p & 1;
                        if (!((dm >> i) & (hm >> j) & (wm >> kk) & 1)) continue;
                        const unsigned sp = (unsigned)(s0 + i * HW + j * g.W + kk);
#pragma unroll
                        for (int k = 0; k < CH; ++k) {
                            if (lo[k] == sp) {
                                acc[p][k] += gv[k];
                                any |= 1u << (p * CH + k);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int i = p >> 2, j = (p >> 1) & 1, kk = p & 1;
            if (d0 + i >= g.D || h0 + j >= g.H || w0 + kk >= g.W) continue;
            const long long e = (n * (long long)g.vol + s0 + i * HW + j * g.W + kk) * C + ch * CH;
            T out[CH];
#pragma unroll
            for (int k = 0; k < CH; ++k)
                out[k] = Elem<T>::from_f(((any >> (p * CH + k)) & 1u) ? acc[p][k] : 0.0f);
            if constexpr (sizeof(T) * CH == 4) {
                unsigned u;
                memcpy(&u, out, sizeof(u));
                *reinterpret_cast<unsigned*>(gi + e) = u;
            } else if constexpr (sizeof(T) * CH == 8) {
                uint2 u;
                memcpy(&u, out, sizeof(u));
                *reinterpret_cast<uint2*>(gi + e) = u;
            } else {
                uint4 u;
                memcpy(&u, out, sizeof(u));
                *reinterpret_cast<uint4*>(gi + e) = u;
            }
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

NdDecomp nd_decomp(const Geo& g, int nch) {
    NdDecomp d;
    d.fc = FastDiv((uint32_t)nch);
    d.fw = FastDiv((uint32_t)g.OW);
    d.fh = FastDiv((uint32_t)g.OH);
    d.fd = FastDiv((uint32_t)g.OD);
    return d;
}

template <typename T>
cudaError_t fwd_dispatch(const void* x, void* y, int64_t* idx, const Geo& g, int C, int sms,
                         cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    if (chunked(C, sizeof(T), {x, y, idx})) {
        if constexpr (sizeof(T) == 2) {
            if (rel_fits(g) && (long long)g.P * g.ovol * (C / VEC) < INT_MAX) {
                const NdDecomp dc = nd_decomp(g, C / VEC);
                const long long work = (long long)g.P * g.ovol * (C / VEC);
                // uniform (h, w) window extents 2 or 3: the unrolled form
                const int kh = uniform_window_len(g.H, g.OH, g.kh, g.adaptive);
                const int kw = uniform_window_len(g.W, g.OW, g.kw, g.adaptive);
                const int k = kh == kw && (kh == 2 || kh == 3) ? kh : 0;
                // 3x3x3 windows of stride 2 along d: walk the output depths
                if (!g.adaptive && g.kd == 3 && g.sd == 2 && k == 3) {
                    // one wave of resident CTAs (three per SM at 80 registers):
                    // with eight CTAs' worth per SM, the partial last wave cost
                    // 6% (384 -> 362 us on the 32x128x16x112x112 fp16 forward)
                    const long long walkers = (long long)g.P * g.OH * g.OW * (C / VEC);
                    auto kdw = k_fwd_ndhwc_dw<T, 3, 2, 3, 3>;
                    kdw<<<stride_grid(kdw, walkers, sms), 256, 0, s>>>((const T*)x, (T*)y, idx, g, C);
                    return cudaGetLastError();
                }
                auto kern = g.adaptive ? (k == 2 ? k_fwd_ndhwc_pk<T, true, 2, 2>
                                          : k == 3 ? k_fwd_ndhwc_pk<T, true, 3, 3> : k_fwd_ndhwc_pk<T, true, 0, 0>)
                                       : (k == 2 ? k_fwd_ndhwc_pk<T, false, 2, 2>
                                          : k == 3 ? k_fwd_ndhwc_pk<T, false, 3, 3> : k_fwd_ndhwc_pk<T, false, 0, 0>);
                kern<<<grid_of(work, sms), 256, 0, s>>>((const T*)x, (T*)y, idx, g, C, dc);
                return cudaGetLastError();
            }
        }
        return fwd_t<T, VEC>(x, y, idx, g, C, sms, s);
    }
    return fwd_t<T, 1>(x, y, idx, g, C, sms, s);
}

// The block form: fixed windows, stride 2 and length at most 4 on every
// axis, BLK_CH channels per thread with aligned vector access.
constexpr int BLK_CH = 4;
bool blk_ok(const Geo& g, int C, int es, const void* go, const int64_t* idx, const void* gi) {
    if (g.adaptive || g.sd != 2 || g.sh != 2 || g.sw != 2) return false;
    if (g.kd > 4 || g.kh > 4 || g.kw > 4 || C % BLK_CH != 0) return false;
    const uintptr_t a = BLK_CH * (uintptr_t)es;   // bytes of the thread's channels
    return (uintptr_t)idx % 16 == 0 && (uintptr_t)go % a == 0 && (uintptr_t)gi % a == 0;
}

template <typename T>
cudaError_t bwd_dispatch(const void* go, const int64_t* idx, void* gi, const Geo& g, int C, int sms,
                         cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    // 2x2x2 windows tiling the input: each input in exactly one window
    if (!g.adaptive && g.kd == 2 && g.kh == 2 && g.kw == 2 && g.sd == 2 && g.sh == 2 && g.sw == 2 &&
        g.D == 2 * g.OD && g.H == 2 * g.OH && g.W == 2 * g.OW && chunked(C, sizeof(T), {go, idx, gi}) &&
        (long long)g.P * g.ovol * (C / VEC) < INT_MAX) {
        const long long work = (long long)g.P * g.ovol * (C / VEC);
        k_bwd_ndhwc_tile<T, 2, 2, 2><<<grid_of(work, sms), 256, 0, s>>>((const T*)go, idx, (T*)gi, g, C,
                                                                     nd_decomp(g, C / VEC));
        return cudaGetLastError();
    }
    if (blk_ok(g, C, sizeof(T), go, idx, gi)) {
        const long long work = (long long)g.P * ((g.D + 3) / 4) * ((g.H + 3) / 4) * ((g.W + 3) / 4) * 8 *
                               (C / BLK_CH);
        const int k = g.kd == g.kh && g.kd == g.kw && (g.kd == 2 || g.kd == 3) ? g.kd : 0;
        auto kern = k == 2 ? k_bwd_ndhwc_blk<T, BLK_CH, 2>
                           : k == 3 ? k_bwd_ndhwc_blk<T, BLK_CH, 3> : k_bwd_ndhwc_blk<T, BLK_CH, 0>;
        kern<<<grid_of(work, sms), 256, 0, s>>>((const T*)go, idx, (T*)gi, g, C);
        return cudaGetLastError();
    }
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

// The rolling scatter for adaptive windows and for fixed windows that
// overlap along some axis; fixed windows that tile the input take the
// gather (for 2x2x2 stride-2 windows on the 8x32x64x64x64 bf16 backward:
// gather 53.3 us, rolling scatter 64-76 us).
int bwd_ndhwc_path(const Geo& g, int C, int dtype, bool aligned16) {
    const bool overlap = g.adaptive || g.kd > g.sd || g.kh > g.sh || g.kw > g.sw;
    return aligned16 && overlap && bwd_ndhwc_roll_supported(g, C, dtype) ? MP3D_PATH_BWD_NDHWC_ROLL
                                                                         : MP3D_PATH_BWD_NDHWC;
}

cudaError_t launch_bwd_ndhwc(const void* go, const int64_t* idx, void* gi, const Geo& g, int C,
                             int dtype, int sms, cudaStream_t s) {
    if (bwd_ndhwc_path(g, C, dtype, (uintptr_t)gi % 16 == 0) == MP3D_PATH_BWD_NDHWC_ROLL)
        return launch_bwd_ndhwc_roll(go, idx, gi, g, C, dtype, s);
    switch (dtype) {
    case F32: return bwd_dispatch<float>(go, idx, gi, g, C, sms, s);
    case F16: return bwd_dispatch<__half>(go, idx, gi, g, C, sms, s);
    default: return bwd_dispatch<__nv_bfloat16>(go, idx, gi, g, C, sms, s);
    }
}

}  // namespace mp3d
