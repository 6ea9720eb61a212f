// Channels-last (NDHWC) backward as an ordered scatter: grad_in[n, j, c] =
// sum of grad_out[n, o, c] over the outputs o whose stored index idx[n, o, c]
// is j, in ascending (od, oh, ow) order, binary32, one rounding
// (FlagGems-Experimental PR #308 Summary, the adaptive_max_pool3d_backward
// operator; teenygrad docs "Struct Maxpool3dForward" for the index form).
// Every channel is an independent problem, so this is the rolling scatter
// of the NCDHW layout run on CG channels at once, with the channel the
// fastest axis everywhere:
//  - a CTA takes one sample n, one group of CG channels and one tile of
//    TH x TW input positions (rows x columns), and walks the window rows od
//    in order. Its items are (window, channel) pairs: the windows that
//    cover the tile (the tile's own and, along h and w, the neighbours whose
//    last row or column reaches into it), each with CG channels, so a warp
//    reads CG consecutive indices and gradients per window;
//  - a ring of RS depth slices of binary32 accumulators in shared memory,
//    laid out [slot][row][column][channel], holds the tile's inputs; the
//    item's stored index is decoded to its input and the term goes to that
//    accumulator, or nowhere when the input lies outside the tile (another
//    tile takes it) or outside the window (an index the forward could not
//    have stored);
//  - four passes separated by barriers add the terms, pass (rh, rw) taking
//    the items whose input the next window along h (rh) and w (rw) also
//    covers, in the order (1,1), (1,0), (0,1), (0,0): with at most two
//    windows covering any input along each axis, the lower one has role 1
//    and the upper role 0, so every input receives its terms of a row in
//    ascending (oh, ow) order, and no pass holds two items on one
//    accumulator. Channels never share an accumulator. Earlier rows were
//    added in earlier iterations;
//  - the slices no later row reaches are rounded and written: one 16-byte
//    store per chunk of 16/sizeof(T) channels of a position, and their
//    accumulators cleared.
// Signed zeros follow the NCDHW rolling kernel: accumulators start at +0,
// so a sum differs from the first-term sum only when every term is -0; a
// -0 gradient sets a bit for its input, and before the store an input whose
// accumulator is +0 and whose bit is set re-reads its covering windows and
// becomes -0 when every window that chose it has a -0 gradient.
#include <climits>

#include "internal.h"

namespace mp3d {

namespace {

struct NRollGeo {
    int TH, TW;          // input rows and columns per tile
    int nht, nwt;        // tiles per plane along h and w
    int ncg;             // channel groups, C / CG
    int C;               // channels
    int RS;              // ring slots (depth slices)
    int SSTR;            // floats per slot: TH*TW*CG rounded up to a multiple of 32
    int NWH, NWW;        // most windows covering a tile along h and w (items: NWH x NWW x CG)
    int units;           // N * ncg * nht * nwt
    AxisMap ad, ah, aw;
    FastDiv fHW, fW, fTW, fNWW, fncg, fnwt, fnht;
};

template <bool AD>
__device__ __forceinline__ int nr_start(const AxisMap& a, int o) {
    if constexpr (AD) return a.fO.div(o * a.I);
    else return o * a.S;
}
template <bool AD>
__device__ __forceinline__ int nr_end(const AxisMap& a, int o) {
    if constexpr (AD) return a.fO.div((o + 1) * a.I + a.O - 1);
    else return o * a.S + a.K;
}
template <bool AD>
__device__ __forceinline__ int nr_lo(const AxisMap& a, int x) {
    if constexpr (AD) return a.fI.div(x * a.O);
    else return x < a.K ? 0 : a.fS.div(x - a.K) + 1;
}
template <bool AD>
__device__ __forceinline__ int nr_hi(const AxisMap& a, int x) {
    if constexpr (AD) return a.fI.div((x + 1) * a.O - 1);
    else return min(a.fS.div(x), a.O - 1);
}

// Whether every window that chose input j (in-plane offset) of sample n,
// channel c has a -0 gradient (the input is known to be chosen by at least
// one window).
template <typename T, bool AD>
__device__ __forceinline__ bool nroll_all_negzero(const T* __restrict__ go, const int64_t* __restrict__ idx,
                                                  long long n, int c, int j, const Geo& g,
                                                  const NRollGeo& rg) {
    const int HW = g.H * g.W;
    const int jd = rg.fHW.div(j);
    const int rem = j - jd * HW;
    const int jh = rg.fW.div(rem);
    const int jw = rem - jh * g.W;
    const long long C = rg.C;
    for (int od = nr_lo<AD>(rg.ad, jd); od <= nr_hi<AD>(rg.ad, jd); ++od)
        for (int oh = nr_lo<AD>(rg.ah, jh); oh <= nr_hi<AD>(rg.ah, jh); ++oh)
            for (int ow = nr_lo<AD>(rg.aw, jw); ow <= nr_hi<AD>(rg.aw, jw); ++ow) {
                const long long o = (((n * g.OD + od) * g.OH + oh) * (long long)g.OW + ow) * C + c;
                if (idx[o] == j && __float_as_uint(Elem<T>::to_f(go[o])) != 0x80000000u) return false;
            }
    return true;
}

template <typename T> __device__ __forceinline__ unsigned nr_pack2(float a, float b);
template <> __device__ __forceinline__ unsigned nr_pack2<__half>(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const unsigned*>(&h);
}
template <> __device__ __forceinline__ unsigned nr_pack2<__nv_bfloat16>(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const unsigned*>(&h);
}

// Accumulator x of a slot (floats from the slot's start) sits at nr_swz(x):
// for 16-bit types the two 16-byte halves of 32-byte chunk c = x / 8 trade
// places when bit 2 of c is set (the map is its own inverse). A thread's
// store chunks all have that bit equal to f = bit 2 of its lane, so it reads
// its lower halves at float offset 4 * f of each chunk and gets the halves
// in output order, while the eight chunks of a quarter-warp meet each of the
// eight 16-byte bank groups once per access.
template <typename T>
__device__ __forceinline__ int nr_swz(int x) {
    if constexpr (sizeof(T) == 2) return x ^ ((x >> 3) & 4);
    else return x;
}

// One 16-byte output chunk from its accumulators (chunk base src, lane bit
// f as above), which are reset to +0.
template <typename T>
__device__ __forceinline__ uint4 nr_take(float* src, int f) {
    if constexpr (sizeof(T) == 4) {
        float4* s4 = reinterpret_cast<float4*>(src);
        const float4 a = s4[0];
        s4[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        return make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(a.z),
                          __float_as_uint(a.w));
    } else {
        float4* lo = reinterpret_cast<float4*>(src + 4 * f);
        float4* hi = reinterpret_cast<float4*>(src + 4 * (f ^ 1));
        const float4 a = *lo, b = *hi;
        *lo = make_float4(0.f, 0.f, 0.f, 0.f);
        *hi = make_float4(0.f, 0.f, 0.f, 0.f);
        return make_uint4(nr_pack2<T>(a.x, a.y), nr_pack2<T>(a.z, a.w), nr_pack2<T>(b.x, b.y),
                          nr_pack2<T>(b.z, b.w));
    }
}

// Store chunks (16 bytes of output) per thread and slice, at most.
constexpr int kNRollSpt = 2;

// AD: adaptive windows. K3: fixed 3x3x3 windows of stride 2, the stored
// index decoded by compares against the window's slice and row strides.
// CG: channels per CTA (a whole number of 16-byte chunks of T); with 32 or
// more bytes of channels, neighbouring lanes store the 16-byte halves of one
// 32-byte sector.
template <typename T, bool AD, int NT, int WPT, int MINB, int CG, bool K3>
__global__ void __launch_bounds__(NT, MINB)
k_bwd_ndhwc_roll(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi, Geo g,
                 NRollGeo rg) {
    constexpr int VEC = 16 / sizeof(T);
    constexpr int NCH = CG / VEC;          // 16-byte output chunks per position
    static_assert(CG % VEC == 0 && (CG & (CG - 1)) == 0, "whole chunks, power-of-two group");
    static_assert(NT % 32 == 0, "the store's half order uses lane bits");
    extern __shared__ __align__(16) float ring[];
    const int RS = K3 ? 3 : rg.RS, SSTR = rg.SSTR;
    const int nacc = RS * SSTR;
    unsigned* negbits = reinterpret_cast<unsigned*>(ring + nacc);   // one bit per accumulator
    int* slotmask = reinterpret_cast<int*>(negbits + nacc / 32);    // slots holding a set bit
    const int tid = threadIdx.x;
    const int fh = (tid >> 2) & 1;
    const int W = g.W, HW = g.H * g.W, OD = g.OD, TH = rg.TH, TW = rg.TW;
    const long long C = rg.C;
    {
        float4* r4 = reinterpret_cast<float4*>(ring);
        for (int i = tid; i < nacc / 4; i += NT) r4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = tid; i < nacc / 32; i += NT) negbits[i] = 0u;
        if (tid == 0) *slotmask = 0;
    }
    for (int u = blockIdx.x; u < rg.units; u += gridDim.x) {
        int r = rg.fncg.div(u);
        const int cgi = u - r * rg.ncg;
        int r2 = rg.fnwt.div(r);
        const int wt = r - r2 * rg.nwt;
        const int n = rg.fnht.div(r2);
        const int ht = r2 - n * rg.nht;
        const int h0 = ht * TH, h1 = min(h0 + TH, g.H);
        const int w0 = wt * TW, w1 = min(w0 + TW, W);
        const int THv = h1 - h0, TWv = w1 - w0;
        const int ohl = nr_lo<AD>(rg.ah, h0), ohh = nr_hi<AD>(rg.ah, h1 - 1);
        const int owl = nr_lo<AD>(rg.aw, w0), owh = nr_hi<AD>(rg.aw, w1 - 1);
        const int c0 = cgi * CG;
        // this thread's items me = tid + k * NT: channel me % CG of window
        // (row, col) = divmod(me / CG, NWW) of the tile's windows; items
        // outside the tile's windows stay idle (ioff < 0)
        int hw0[WPT];     // window's first row and column relative to the tile, packed
        int wsh[WPT];     // adaptive: kh | kw << 8 | sh << 16 | sw << 24 (each < 256)
        int ioff[WPT];    // offset of the item in a row of grad_out / idx, or -1
#pragma unroll
        for (int k = 0; k < WPT; ++k) {
            const int me = tid + k * NT;
            const int wi = me / CG, ch = me & (CG - 1);
            const int row = rg.fNWW.div(wi), col = wi - row * rg.NWW;
            const bool in = ohl + row <= ohh && owl + col <= owh && row < rg.NWH;
            const int oh = min(ohl + row, g.OH - 1), ow = min(owl + col, g.OW - 1);
            const int hs = nr_start<AD>(rg.ah, oh), ws = nr_start<AD>(rg.aw, ow);
            hw0[k] = ((hs - h0) & 0xFFFF) | ((ws - w0) << 16);
            ioff[k] = in ? (oh * g.OW + ow) * rg.C + c0 + ch : -1;
            if constexpr (AD) {
                const int kh = nr_end<AD>(rg.ah, oh) - hs, kw = nr_end<AD>(rg.aw, ow) - ws;
                const int sh = oh + 1 < g.OH ? nr_start<AD>(rg.ah, oh + 1) - hs : 255;
                const int sw = ow + 1 < g.OW ? nr_start<AD>(rg.aw, ow + 1) - ws : 255;
                wsh[k] = kh | kw << 8 | sh << 16 | sw << 24;
            } else {
                wsh[k] = 0;
            }
        }
        const long long rstride = (long long)g.OH * g.OW * C;
        const int64_t* ip = idx + n * OD * rstride;
        const T* gp = go + n * OD * rstride;
        int64_t rj[WPT];
        T rgd[WPT];
#pragma unroll
        for (int k = 0; k < WPT; ++k) {
            const bool in = ioff[k] >= 0;
            rj[k] = in ? __ldg(ip + ioff[k]) : -1;
            rgd[k] = in ? gp[ioff[k]] : Elem<T>::from_f(0.0f);
        }
        // the tile's first position, channel c0, of sample n
        T* gbase = gi + ((long long)n * g.vol + (long long)h0 * W + w0) * C + c0;
        // this thread's store chunks c = tid + i * NT of a slice: position
        // c / NCH of the tile (row-major, TW wide), chunk c % NCH of its
        // channels; offset from the tile's first element, or -1 (outside)
        int soff[kNRollSpt];
#pragma unroll
        for (int i = 0; i < kNRollSpt; ++i) {
            const int c = tid + i * NT;
            const int pos = c / NCH, q = c - pos * NCH;
            const int lr = rg.fTW.div(pos), lc = pos - lr * TW;
            soff[i] = lr < THv && lc < TWv ? (lr * W + lc) * rg.C + q * VEC : -1;
        }
        const int tile0 = h0 * W + w0;  // in-plane offset of the tile's first position
        int cs = 0, sbc = 0;            // first slice the row completes and its ring slot
        __syncthreads();   // the ring is clear before any pass
        for (int od = 0; od < OD; ++od) {
            const int ods = K3 ? 2 * od : nr_start<AD>(rg.ad, od);
            const int oe = K3 ? ods + 3 : nr_end<AD>(rg.ad, od);
            const int kd = oe - ods;
            const int de = min(oe, g.D);
            int sbo = ods % RS;          // ring slot of the window's first slice
            const int dsHW = ods * HW;
            int a3[3];                   // K3: float offsets of the window's three slots
            if constexpr (K3) {
#pragma unroll
                for (int t = 0; t < 3; ++t) a3[t] = (sbo + t >= 3 ? sbo + t - 3 : sbo + t) * SSTR;
            }
            // 1. decode this row: the item's pass q and accumulator, as
            //    q << 20 plus the accumulator's byte offset in the ring
            //    (below 2^18), or -1 (adds nothing); items with a -0
            //    gradient are marked in negm
            int kf[WPT];
            float gv[WPT];
            unsigned negm = 0u;
#pragma unroll
            for (int k = 0; k < WPT; ++k) {
                const int64_t j = rj[k];
                gv[k] = Elem<T>::to_f(rgd[k]);
                const int hr0 = (int)(short)(hw0[k] & 0xFFFF), wc0 = hw0[k] >> 16;
                const int ch = (tid + k * NT) & (CG - 1);
                const int rel = (int)j - dsHW - (tile0 + hr0 * W + wc0);
                int offd, offh, offw;
                bool ok;
                if constexpr (K3) {
                    const bool d1 = rel >= HW, d2 = rel >= 2 * HW;
                    const int rem = rel - (d1 ? HW : 0) - (d2 ? HW : 0);
                    const bool e1 = rem >= W, e2 = rem >= 2 * W;
                    offd = (int)d1 + (int)d2;
                    offh = (int)e1 + (int)e2;
                    offw = rem - (e1 ? W : 0) - (e2 ? W : 0);
                    ok = (int)(j >> 32) == 0 && (unsigned)rel < (unsigned)(3 * HW) &&
                         (unsigned)rem < (unsigned)(3 * W) && (unsigned)offw < 3u;
                } else {
                    offd = rg.fHW.div(rel);
                    const int rem = rel - offd * HW;
                    offh = rg.fW.div(rem);
                    offw = rem - offh * W;
                    int kh, kw;
                    if constexpr (AD) {
                        kh = wsh[k] & 255;
                        kw = (wsh[k] >> 8) & 255;
                    } else {
                        kh = g.kh;
                        kw = g.kw;
                    }
                    ok = (uint64_t)j < (uint64_t)g.vol && rel >= 0 && offd < kd && offh < kh && offw < kw;
                }
                const int lr = hr0 + offh, lc = wc0 + offw;   // place in the tile
                ok = ok && (unsigned)lr < (unsigned)THv && (unsigned)lc < (unsigned)TWv;
                int sh, sw;
                if constexpr (AD) {
                    sh = (wsh[k] >> 16) & 255;
                    sw = (unsigned)wsh[k] >> 24;
                } else if constexpr (K3) {
                    sh = 2;
                    sw = 2;
                } else {
                    sh = g.sh;
                    sw = g.sw;
                }
                int slot;
                if constexpr (K3) {
                    slot = offd == 2 ? a3[2] : offd == 1 ? a3[1] : a3[0];
                } else {
                    slot = sbo + offd;
                    slot = (slot >= RS ? slot - RS : slot) * SSTR;
                }
                const int off = slot + nr_swz<T>((lr * TW + lc) * CG + ch);
                kf[k] = ok ? off * 4 + (((offh >= sh ? 0 : 2) | (offw >= sw ? 0 : 1)) << 20) : -1;
                negm |= (ok && __float_as_uint(gv[k]) == 0x80000000u) ? 1u << k : 0u;
            }
            if (negm) {
#pragma unroll
                for (int k = 0; k < WPT; ++k) {
                    if ((negm >> k) & 1u) {
                        const int off = (kf[k] & 0xFFFFF) >> 2;
                        atomicOr(&negbits[off >> 5], 1u << (off & 31));
                        atomicOr(slotmask, 1 << (off / SSTR));
                    }
                }
            }
            // the next row's loads are in flight during the passes and the store
            if (od + 1 < OD) {
                ip += rstride;
                gp += rstride;
#pragma unroll
                for (int k = 0; k < WPT; ++k) {
                    if (ioff[k] >= 0) {
                        rj[k] = __ldg(ip + ioff[k]);
                        rgd[k] = gp[ioff[k]];
                    }
                }
            }
            // 2. four ordered passes
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int k = 0; k < WPT; ++k) {
                    const unsigned t = (unsigned)kf[k] - ((unsigned)q << 20);
                    if (t < (1u << 20)) {
                        float* a = reinterpret_cast<float*>(reinterpret_cast<char*>(ring) + t);
                        *a += gv[k];
                    }
                }
                __syncthreads();
            }
            // 3. round and store the completed slices [cs, dn), clear their accumulators
            const int dn = od + 1 < OD ? (K3 ? 2 * od + 2 : nr_start<AD>(rg.ad, od + 1)) : g.D;
            const int nring = min(dn, de) - cs;        // completed slices held in the ring
            const int stored = ((1 << nring) - 1) << sbc | ((1 << nring) - 1) >> (RS - sbc);
            const int marked = *slotmask & stored;
            if (marked) {
                // inputs chosen only by -0 gradients: accumulator +0 -> -0
                for (int s = 0; s < nring; ++s) {
                    int slot = sbc + s;
                    slot -= slot >= RS ? RS : 0;
                    if (!((marked >> slot) & 1)) continue;
                    for (int i = tid; i < SSTR / 32; i += NT) {
                        unsigned m = negbits[slot * (SSTR / 32) + i];
                        negbits[slot * (SSTR / 32) + i] = 0u;
                        while (m) {
                            const int b = __ffs(m) - 1;
                            m &= m - 1;
                            float* acc = ring + slot * SSTR + i * 32 + b;
                            const int x = nr_swz<T>(i * 32 + b);   // its place in the slot's order
                            const int pos = x / CG;
                            const int lr = rg.fTW.div(pos), lc = pos - lr * TW;
                            const int jj = (cs + s) * HW + (h0 + lr) * W + w0 + lc;
                            if (__float_as_uint(*acc) == 0u &&
                                nroll_all_negzero<T, AD>(go, idx, n, c0 + (x & (CG - 1)), jj, g, rg))
                                *acc = -0.0f;
                        }
                    }
                }
                __syncthreads();
                if (tid == 0) *slotmask &= ~stored;
            }
            for (int s = 0; s < dn - cs; ++s) {
                int slot = sbc + s;
                slot -= slot >= RS ? RS : 0;
                float* src = ring + slot * SSTR + tid * VEC;
                T* dst = gbase + (long long)(cs + s) * HW * C;
                if (s < nring) {
#pragma unroll
                    for (int i = 0; i < kNRollSpt; ++i) {
                        if (soff[i] < 0) continue;
                        *reinterpret_cast<uint4*>(dst + soff[i]) = nr_take<T>(src + i * NT * VEC, fh);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < kNRollSpt; ++i)
                        if (soff[i] >= 0) *reinterpret_cast<uint4*>(dst + soff[i]) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // the next row completes from dn; its slot follows
            sbc += dn - cs;
            while (sbc >= RS) sbc -= RS;
            cs = dn;
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------- host side

struct NAxis {
    int I, O, K, S;
    bool adaptive;
    long long start(int o) const { return adaptive ? (long long)o * I / O : (long long)o * S; }
    long long end(int o) const { return adaptive ? ((long long)(o + 1) * I + O - 1) / O : (long long)o * S + K; }
    int lo(int x) const {
        if (adaptive) return (int)((long long)x * O / I);
        return x < K ? 0 : (x - K) / S + 1;
    }
    int hi(int x) const {
        if (adaptive) return (int)(((long long)(x + 1) * O - 1) / I);
        const int h = x / S;
        return h < O - 1 ? h : O - 1;
    }
    bool two_cover() const {
        if (!adaptive) return K <= 2 * S;
        for (int i = 0; i + 2 < O; ++i)
            if (end(i) > start(i + 2)) return false;
        return true;
    }
    int longest() const {
        if (!adaptive) return K;
        long long m = 0;
        for (int i = 0; i < O; ++i) m = end(i) - start(i) > m ? end(i) - start(i) : m;
        return (int)m;
    }
    // The most windows covering one tile of t positions, over the tiles.
    int most(int t) const {
        int m = 0;
        for (int x0 = 0; x0 < I; x0 += t) {
            const int x1 = x0 + t < I ? x0 + t : I;
            const int l = lo(x0), h = hi(x1 - 1);
            m = h - l + 1 > m ? h - l + 1 : m;
        }
        return m;
    }
};

struct NRollCfg {
    int nt, wpt, minb;
    size_t budget;       // shared bytes per CTA
};

// 256 threads holding up to four items each at four CTAs per SM.
constexpr NRollCfg kNRollCfg = {256, 4, 4, 54 * 1024};

// Channels per CTA: 32 bytes of each position (whole 32-byte sectors per
// pair of lanes) when C allows, else 16 bytes; 0 when C holds no whole
// 16-byte chunk.
int nroll_cg(int C, int es) {
    if (C % (32 / es) == 0) return 32 / es;
    if (C % (16 / es) == 0) return 16 / es;
    return 0;
}

size_t nroll_smem(int RS, int SSTR) {
    const size_t nacc = (size_t)RS * SSTR;
    return nacc * sizeof(float) + nacc / 8 + sizeof(int);
}

// Fills rg and the shared bytes, or returns false when the kernel does not
// apply. Tiles: the TH x TW (at most 64 x 64) whose windows fit the CTA's
// items and whose accumulators fit its shared memory, with the most tile
// positions per window taken (the fewest windows read twice), then the
// largest tile.
bool nroll_plan(const Geo& g, int C, int es, const NRollCfg& cfg, NRollGeo* rg, size_t* smem, int* wpt) {
    const bool a = g.adaptive != 0;
    if (g.P == 0 || g.vol == 0 || g.ovol == 0) return false;
    const int CG = nroll_cg(C, es);
    if (CG == 0) return false;
    // item offsets within a sample's windows and store offsets within a
    // slice are int
    if ((long long)g.OH * g.OW * C > INT_MAX || (long long)g.H * g.W * C > INT_MAX) return false;
    if (a) {
        const long long lim = (1LL << 31) - 1;
        if ((long long)g.D * g.OD + g.OD > lim || (long long)g.H * g.OH + g.OH > lim ||
            (long long)g.W * g.OW + g.OW > lim)
            return false;
    }
    if (!a && (g.pd || g.ph || g.pw || g.dd != 1 || g.dh != 1 || g.dw != 1)) return false;
    const NAxis ad = {g.D, g.OD, g.kd, g.sd, a}, ah = {g.H, g.OH, g.kh, g.sh, a},
                aw = {g.W, g.OW, g.kw, g.sw, a};
    if (!ad.two_cover() || !ah.two_cover() || !aw.two_cover()) return false;
    const int RS = ad.longest();
    if (RS > 30) return false;
    if (a && (ah.longest() > 254 || aw.longest() > 254)) return false;
    const int maxt = 64;
    const int tH = g.H < maxt ? g.H : maxt, tW = g.W < maxt ? g.W : maxt;
    int mh[65], mw[65];
    for (int t = 1; t <= tH; ++t) mh[t] = ah.most(t);
    for (int t = 1; t <= tW; ++t) mw[t] = aw.most(t);
    const long long cap = (long long)cfg.nt * cfg.wpt;
    double best = -1.0;
    int bh = 0, bw = 0;
    for (int th = 1; th <= tH; ++th) {
        for (int tw = 1; tw <= tW; ++tw) {
            const long long items = (long long)mh[th] * mw[tw] * CG;
            if (items > cap) break;                      // more columns only add windows
            const long long sstr = ((long long)th * tw * CG + 31) / 32 * 32;
            if (nroll_smem(RS, (int)sstr) > cfg.budget || sstr * RS >= (1 << 16) ||
                (long long)th * tw * CG > (long long)kNRollSpt * cfg.nt * (16 / es))
                break;
            const double score = (double)th * tw / ((double)mh[th] * mw[tw]);
            if (score > best + 1e-9 || (score > best - 1e-9 && th * tw > bh * bw)) {
                best = score;
                bh = th;
                bw = tw;
            }
        }
    }
    if (!bh) return false;
    const long long items = (long long)mh[bh] * mw[bw] * CG;
    *wpt = items <= cfg.nt ? 1 : items <= 2 * cfg.nt ? 2 : 4;
    rg->TH = bh;
    rg->TW = bw;
    rg->nht = (g.H + bh - 1) / bh;
    rg->nwt = (g.W + bw - 1) / bw;
    rg->ncg = C / CG;
    rg->C = C;
    rg->RS = RS;
    rg->SSTR = (bh * bw * CG + 31) / 32 * 32;
    rg->ad = axis_map(g.D, g.OD, g.kd, g.sd, a);
    rg->ah = axis_map(g.H, g.OH, g.kh, g.sh, a);
    rg->aw = axis_map(g.W, g.OW, g.kw, g.sw, a);
    rg->fHW = FastDiv((uint32_t)(g.H * g.W));
    rg->fW = FastDiv((uint32_t)g.W);
    rg->fTW = FastDiv((uint32_t)bw);
    rg->NWH = mh[bh];
    rg->NWW = mw[bw];
    rg->fNWW = FastDiv((uint32_t)rg->NWW);
    rg->fncg = FastDiv((uint32_t)rg->ncg);
    rg->fnwt = FastDiv((uint32_t)rg->nwt);
    rg->fnht = FastDiv((uint32_t)rg->nht);
    const long long units = g.P * rg->ncg * rg->nht * rg->nwt;
    if (units >= INT_MAX) return false;
    rg->units = (int)units;
    *smem = nroll_smem(RS, rg->SSTR);
    return true;
}

template <typename T, bool AD, int WPT, bool K3>
cudaError_t nroll_launch(const void* go, const int64_t* idx, void* gi, const Geo& g, const NRollGeo& rg,
                         size_t smem, cudaStream_t s) {
    constexpr NRollCfg cfg = kNRollCfg;
    constexpr int VEC = 16 / sizeof(T);
    auto kern = rg.C % (2 * VEC) == 0 ? k_bwd_ndhwc_roll<T, AD, cfg.nt, WPT, cfg.minb, 2 * VEC, K3>
                                      : k_bwd_ndhwc_roll<T, AD, cfg.nt, WPT, cfg.minb, VEC, K3>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)rg.units, cfg.nt, smem, s>>>((const T*)go, idx, (T*)gi, g, rg);
    return cudaGetLastError();
}

template <typename T>
cudaError_t nroll_t(const void* go, const int64_t* idx, void* gi, const Geo& g, int C, cudaStream_t s) {
    NRollGeo rg;
    size_t smem = 0;
    int wpt = 0;
    if (!nroll_plan(g, C, sizeof(T), kNRollCfg, &rg, &smem, &wpt)) return cudaErrorNotSupported;
    const bool k3 = !g.adaptive && g.kd == 3 && g.kh == 3 && g.kw == 3 && g.sd == 2 && g.sh == 2 && g.sw == 2;
    if (k3) {
        if (wpt == 1) return nroll_launch<T, false, 1, true>(go, idx, gi, g, rg, smem, s);
        if (wpt == 2) return nroll_launch<T, false, 2, true>(go, idx, gi, g, rg, smem, s);
        return nroll_launch<T, false, 4, true>(go, idx, gi, g, rg, smem, s);
    }
    if (g.adaptive) {
        if (wpt == 1) return nroll_launch<T, true, 1, false>(go, idx, gi, g, rg, smem, s);
        if (wpt == 2) return nroll_launch<T, true, 2, false>(go, idx, gi, g, rg, smem, s);
        return nroll_launch<T, true, 4, false>(go, idx, gi, g, rg, smem, s);
    }
    if (wpt == 1) return nroll_launch<T, false, 1, false>(go, idx, gi, g, rg, smem, s);
    if (wpt == 2) return nroll_launch<T, false, 2, false>(go, idx, gi, g, rg, smem, s);
    return nroll_launch<T, false, 4, false>(go, idx, gi, g, rg, smem, s);
}

}  // namespace

bool bwd_ndhwc_roll_supported(const Geo& g, int C, int dtype) {
    NRollGeo rg;
    size_t smem = 0;
    int wpt = 0;
    return nroll_plan(g, C, dtype == F32 ? 4 : 2, kNRollCfg, &rg, &smem, &wpt);
}

cudaError_t launch_bwd_ndhwc_roll(const void* go, const int64_t* idx, void* gi, const Geo& g, int C,
                                  int dtype, cudaStream_t s) {
    switch (dtype) {
    case F32: return nroll_t<float>(go, idx, gi, g, C, s);
    case F16: return nroll_t<__half>(go, idx, gi, g, C, s);
    default: return nroll_t<__nv_bfloat16>(go, idx, gi, g, C, s);
    }
}

}  // namespace mp3d
