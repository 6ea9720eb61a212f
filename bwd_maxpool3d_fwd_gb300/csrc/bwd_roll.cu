// Overlapping backward as an ordered scatter into a rolling ring of depth
// slices held in shared memory (FlagGems-Experimental PR #308, "Add
// adaptive_max_pool3d_backward Moore Threads specialized operator",
// Summary: when the axes do not divide evenly, windows overlap and the
// gradients of the windows that chose one input are summed).
//
// grad_in[p, j] is the binary32 sum of the gradients of the windows whose
// stored index is j, taken in ascending (od, oh, ow) order and starting from
// the first term, rounded once to the type; +0 where no window chose j.
//
// Scope: at most two windows cover any position along each axis (fixed
// windows with kernel <= 2 * stride; adaptive windows with
// end(i) <= start(i + 2)). One CTA owns the inputs of one plane in the rows
// [h0, h1) (an h-tile) and walks the window rows od = 0 .. OD-1 in order.
// For each row:
//  1. Every thread decodes its windows of the row (the (oh, ow) whose rows
//     meet [h0, h1)). The stored index must name an input inside the window
//     and inside the h-tile, else the window adds nothing here (as in every
//     gather path). The input's binary32 accumulator lives in a ring of RS
//     depth slices in shared memory, slot jd mod RS, RS being the longest
//     window along d; the slices one row reaches never share a slot.
//  2. Four passes, separated by barriers, add the gradients. Pass (rh, rw)
//     takes the windows whose input is also covered by the next window
//     along h (rh = 0) or not (rh = 1), and likewise along w. Two windows
//     of one row that choose the same input differ in oh or ow; on such an
//     axis the lower window has role 0 and the upper role 1, so they fall in
//     different passes with the lower first, and no pass has two windows on
//     one accumulator (plain shared loads and stores, no atomics). Earlier
//     rows were added in earlier iterations, so every input receives its
//     terms in ascending (od, oh, ow) order.
//  3. The slices no later row reaches, [start(od), start(od + 1)) (up to D
//     after the last row), are rounded and written with coalesced 16-byte
//     stores, and their accumulators are reset.
// Accumulators start at +0. Adding the first term t to +0 gives t, except
// that +0 + (-0) is +0, so the sum differs from the first-term sum only when
// every term is -0 (the first-term sum is then -0); and an accumulator never
// holds -0. Windows with a -0 gradient therefore set a bit for their input;
// before the store, an input whose accumulator is +0 and whose bit is set
// re-reads its covering windows in global memory, and its accumulator is set
// to -0 when every window that chose it has a -0 gradient. Inputs no window
// chose leave as +0.
#include <climits>

#include "internal.h"

namespace mp3d {

struct RollGeo {
    int TH, nht;        // input rows per h-tile, h-tiles per plane
    int RS;             // ring slots (depth slices)
    int SSTR;           // floats per slot: a multiple of 32 holding TH*W + alignment
    AxisMap ad, ah, aw;
    FastDiv fHW, fW, fOW;
};

// Window arithmetic along one axis with the window kind known at compile
// time (fixed: [o*S, o*S + K); adaptive: [floor(o*I/O), ceil((o+1)*I/O))).
// Fixed windows may be padded: window o starts at o*S - pad (possibly
// before the first position; only positions inside the input are ever
// chosen).
template <bool AD>
__device__ __forceinline__ int ax_start(const AxisMap& a, int o) {
    if constexpr (AD) return a.fO.div(o * a.I);
    else return o * a.S - a.pad;
}
template <bool AD>
__device__ __forceinline__ int ax_end(const AxisMap& a, int o) {
    if constexpr (AD) return a.fO.div((o + 1) * a.I + a.O - 1);
    else return o * a.S - a.pad + a.K;
}
template <bool AD>
__device__ __forceinline__ int ax_lo(const AxisMap& a, int x) {
    if constexpr (AD) return a.fI.div(x * a.O);
    else return x + a.pad < a.K ? 0 : a.fS.div(x + a.pad - a.K) + 1;
}
template <bool AD>
__device__ __forceinline__ int ax_hi(const AxisMap& a, int x) {
    if constexpr (AD) return a.fI.div((x + 1) * a.O - 1);
    else return min(a.fS.div(x + a.pad), a.O - 1);
}

// Whether every window that chose input j of plane p has a -0 gradient
// (the input is known to be chosen by at least one). Windows are visited
// through their stored indices in global memory.
template <typename T, bool AD>
__device__ __forceinline__ bool roll_all_negzero(const T* __restrict__ go,
                                                 const int64_t* __restrict__ idx, long long p, int j,
                                                 const Geo& g, const RollGeo& rg) {
    const int HW = g.H * g.W;
    const int jd = rg.fHW.div(j);
    const int rem = j - jd * HW;
    const int jh = rg.fW.div(rem);
    const int jw = rem - jh * g.W;
    const long long ob = p * (long long)g.ovol;
    for (int od = ax_lo<AD>(rg.ad, jd); od <= ax_hi<AD>(rg.ad, jd); ++od)
        for (int oh = ax_lo<AD>(rg.ah, jh); oh <= ax_hi<AD>(rg.ah, jh); ++oh)
            for (int ow = ax_lo<AD>(rg.aw, jw); ow <= ax_hi<AD>(rg.aw, jw); ++ow) {
                const long long o = ob + ((long long)od * g.OH + oh) * g.OW + ow;
                if (idx[o] == j && __float_as_uint(Elem<T>::to_f(go[o])) != 0x80000000u) return false;
            }
    return true;
}

// Two binary32 values rounded to T and packed into 32 bits (low = first).
template <typename T> __device__ __forceinline__ unsigned pack2(float a, float b);
template <> __device__ __forceinline__ unsigned pack2<__half>(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const unsigned*>(&h);
}
template <> __device__ __forceinline__ unsigned pack2<__nv_bfloat16>(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const unsigned*>(&h);
}

// Place of accumulator x of a slice (x counted in floats from the slot's
// start) in the swizzled order: the two 16-byte halves of 32-byte chunk
// c = x / 8 trade places when bit 2 of c is set. A thread whose store chunks
// all have that bit equal to fh then reads its lower halves at float offset
// 4 * fh of each chunk: the eight chunks of a quarter-warp meet every
// 16-byte bank group once per access, and the halves arrive in output
// order. The map is its own inverse.
__device__ __forceinline__ int roll_swz(int x) { return x ^ ((x >> 3) & 4); }

// One 16-byte output chunk from its accumulators at src (reset to +0).
// For 16-bit types a chunk is 32 bytes of accumulators, read and cleared as
// two 16-byte halves. Taken in the same order by every thread, eight
// neighbouring chunks would put their halves two to a bank group; with
// f = bit 2 of the chunk's place in its warp (lanes 4-7 of each
// quarter-warp take the upper half first), each quarter-warp's accesses
// cover all eight 16-byte bank groups once.
template <typename T>
__device__ __forceinline__ uint4 roll_take(float* src, int f) {
    float4* s4 = reinterpret_cast<float4*>(src);
    uint4 out;
    if constexpr (sizeof(T) == 4) {
        const float4 a = s4[0];
        s4[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        out = make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(a.z),
                         __float_as_uint(a.w));
    } else {
        const float4 a = s4[f], b = s4[f ^ 1];
        s4[f] = make_float4(0.f, 0.f, 0.f, 0.f);
        s4[f ^ 1] = make_float4(0.f, 0.f, 0.f, 0.f);
        const unsigned a0 = pack2<T>(a.x, a.y), a1 = pack2<T>(a.z, a.w);
        const unsigned b0 = pack2<T>(b.x, b.y), b1 = pack2<T>(b.z, b.w);
        out = f ? make_uint4(b0, b1, a0, a1) : make_uint4(a0, a1, b0, b1);
    }
    return out;
}

// K3 (a specialization): fixed 3x3x3 windows with stride 2, sizes known at
// compile time; the stored index is decoded with compares instead of
// divisions (496 -> 484 us on the 32x128x16x112x112 fp16 backward). KP:
// K3 windows padded by at most one position per side (window o starts at
// 2o - p); the decode also checks that the index lies in the plane and its
// column inside the input, so an index outside its window still adds
// nothing. AL:
// every row span starts on a 16-byte boundary and holds a whole number of
// 16-byte chunks (W and D*H*W multiples of the vector width), so the store
// has no ragged ends.
template <typename T, bool AD, int NT, int WPT, int MINB, bool K3 = false, bool AL = false,
          bool KP = false>
__global__ void __launch_bounds__(NT, MINB)
k_bwd_roll(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi, Geo g,
           RollGeo rg) {
    constexpr int VEC = 16 / sizeof(T);
    // SW: the compiled 3x3x3 form for 16-bit types keeps its accumulators
    // in the swizzled order of roll_swz
    constexpr bool SW = K3 && sizeof(T) == 2;
    static_assert(NT % 32 == 0, "the store's chunk c and its thread share lane bits");
    extern __shared__ __align__(16) float ring[];
    const int RS = K3 ? 3 : rg.RS, SSTR = rg.SSTR;
    const int nacc = RS * SSTR;
    unsigned* negbits = reinterpret_cast<unsigned*>(ring + nacc);   // one bit per accumulator
    int* slotmask = reinterpret_cast<int*>(negbits + nacc / 32);    // slots holding a set bit
    const int tid = threadIdx.x;
    const int fh = (tid >> 2) & 1;       // half order of this thread's store chunks
    const int W = g.W, HW = g.H * g.W, OW = g.OW, OD = g.OD;
    {
        float4* r4 = reinterpret_cast<float4*>(ring);
        for (int i = tid; i < nacc / 4; i += NT) r4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = tid; i < nacc / 32; i += NT) negbits[i] = 0u;
        if (tid == 0) *slotmask = 0;
    }
    const long long units = g.P * rg.nht;
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
        const long long p = u / rg.nht;
        const int h0 = (int)(u - p * rg.nht) * rg.TH;
        const int h1 = min(h0 + rg.TH, g.H);
        const int h0W = h0 * W;
        const int L = (h1 - h0) * W;
        const int ohl = ax_lo<AD>(rg.ah, h0), ohh = ax_hi<AD>(rg.ah, h1 - 1);
        const int nw = ohh >= ohl ? (ohh - ohl + 1) * OW : 0;
        const long long pbase = p * (long long)g.vol;
        const int pv = (int)(pbase & (VEC - 1));
        T* gplane = gi + pbase;
        // this thread's windows me = tid + k * NT: first (h, w) offset of each,
        // and (adaptive) its lengths and the distances to the next windows
        int wo[WPT];
        int wsh[WPT];    // adaptive: kh | kw << 8 | sh << 16 | sw << 24 (each < 256)
        int wcol[WPT];   // KP: the window's first column (-1 when padded)
#pragma unroll
        for (int k = 0; k < WPT; ++k) {
            const int me = tid + k * NT;
            const int row = rg.fOW.div(me);
            const int oh = min(ohl + row, g.OH - 1), ow = me - row * OW;   // slots past nw stay idle
            const int hs = ax_start<AD>(rg.ah, oh), ws = ax_start<AD>(rg.aw, ow);
            wo[k] = hs * W + ws;
            wcol[k] = ws;
            if constexpr (AD) {
                const int kh = ax_end<AD>(rg.ah, oh) - hs, kw = ax_end<AD>(rg.aw, ow) - ws;
                const int sh = oh + 1 < g.OH ? ax_start<AD>(rg.ah, oh + 1) - hs : 255;
                const int sw = ow + 1 < OW ? ax_start<AD>(rg.aw, ow + 1) - ws : 255;
                wsh[k] = kh | kw << 8 | sh << 16 | sw << 24;
            } else {
                wsh[k] = 0;
            }
        }
        const long long rstride = (long long)g.OH * OW;
        const int64_t* ip = idx + p * (long long)g.ovol + (long long)ohl * OW + tid;
        const T* gp = go + p * (long long)g.ovol + (long long)ohl * OW + tid;
        int64_t rj[WPT];
        T rgd[WPT];
#pragma unroll
        for (int k = 0; k < WPT; ++k) {
            const bool in = tid + k * NT < nw;
            rj[k] = in ? __ldg(ip + k * NT) : -1;
            rgd[k] = in ? gp[k * NT] : Elem<T>::from_f(0.0f);
        }
        int cs = 0, sbc = 0;            // first slice the row completes and its ring slot
        __syncthreads();   // the ring is clear (first unit: initialised) before any pass
        for (int od = 0; od < OD; ++od) {
            const int pdk = KP ? g.pd : 0;
            const int ods = K3 ? 2 * od - pdk : ax_start<AD>(rg.ad, od);   // window origin (before 0 when padded)
            const int oe = K3 ? ods + 3 : ax_end<AD>(rg.ad, od);
            const int kd = oe - ods;                   // window length along d
            const int de = min(oe, g.D);               // slices at or beyond de are in no window
            int sbo = ods % RS;                        // ring slot of the origin
            sbo += sbo < 0 ? RS : 0;
            const int dsHW = ods * HW;
            const int pvt = pv + dsHW + h0W;
            // K3: byte offsets of the ring slots of the window's three slices,
            // less the slice offset a decoded index carries
            int a3[3];
            if constexpr (K3) {
#pragma unroll
                for (int t = 0; t < 3; ++t) {
                    const int sl = sbo + t >= 3 ? sbo + t - 3 : sbo + t;
                    a3[t] = SW ? sl * SSTR * (int)sizeof(float)
                               : (sl * SSTR - t * HW - h0W) * (int)sizeof(float);
                }
            }
            // 1. decode this row (key 4: the window adds nothing here);
            //    mark inputs reached by -0 gradients
            int key[WPT], off[WPT];
            float gv[WPT];
#pragma unroll
            for (int k = 0; k < WPT; ++k) {
                const int64_t j = rj[k];
                gv[k] = Elem<T>::to_f(rgd[k]);
                if constexpr (K3) {
                    // the index relative to the window's first element is
                    // offd*HW + offh*W + offw with each offset in [0, 3):
                    // compares instead of divisions
                    const int rel = (int)j - dsHW - wo[k];
                    const bool d1 = rel >= HW, d2 = rel >= 2 * HW;
                    const int rem = rel - (d1 ? HW : 0) - (d2 ? HW : 0);
                    const bool h1 = rem >= W, h2 = rem >= 2 * W;
                    const int offw = rem - (h1 ? W : 0) - (h2 ? W : 0);
                    const int loc = wo[k] + rem - h0W;        // place inside the h-tile's rows
                    bool ok = (int)(j >> 32) == 0 && (unsigned)rel < (unsigned)(3 * HW) &&
                              (unsigned)rem < (unsigned)(3 * W) && (unsigned)offw < 3u &&
                              (unsigned)loc < (unsigned)L;
                    if constexpr (KP)
                        ok = ok && (unsigned)(int)j < (unsigned)g.vol && (unsigned)(wcol[k] + offw) < (unsigned)W;
                    if constexpr (SW)
                        off[k] = (d2 ? a3[2] : d1 ? a3[1] : a3[0]) + roll_swz(loc) * (int)sizeof(float);
                    else
                        off[k] = (d2 ? a3[2] : d1 ? a3[1] : a3[0]) + (wo[k] + rel) * (int)sizeof(float);
                    key[k] = ok ? ((h2 ? 0 : 2) | (offw >= 2 ? 0 : 1)) : 4;
                    if (ok && __float_as_uint(gv[k]) == 0x80000000u) {
                        const int a = off[k] >> 2;
                        atomicOr(&negbits[a >> 5], 1u << (a & 31));
                        atomicOr(slotmask, 1 << (a / SSTR));
                    }
                    continue;
                }
                const int rel = (int)j - dsHW - wo[k];
                const int offd = rg.fHW.div(rel);
                const int rem = rel - offd * HW;
                const int offh = rg.fW.div(rem);
                const int offw = rem - offh * W;
                int kh, kw, sh, sw;
                if constexpr (AD) {
                    kh = wsh[k] & 255; kw = (wsh[k] >> 8) & 255;
                    sh = (wsh[k] >> 16) & 255; sw = (unsigned)wsh[k] >> 24;
                } else if constexpr (K3) {
                    kh = 3; kw = 3; sh = 2; sw = 2;
                } else {
                    kh = g.kh; kw = g.kw; sh = g.sh; sw = g.sw;
                }
                const int loc = wo[k] - h0W + rem;      // place inside the h-tile's rows
                const bool ok = (uint64_t)j < (uint64_t)g.vol && rel >= 0 && offd < kd && offh < kh &&
                                offw < kw && (unsigned)loc < (unsigned)L;
                int slot = sbo + offd;
                slot -= slot >= RS ? RS : 0;
                const int ph = AL ? 0 : (pvt + offd * HW) & (VEC - 1);
                off[k] = (slot * SSTR + ph + loc) * (int)sizeof(float);
                key[k] = ok ? ((offh >= sh ? 0 : 2) | (offw >= sw ? 0 : 1)) : 4;
                if (ok && __float_as_uint(gv[k]) == 0x80000000u) {
                    const int a = off[k] >> 2;
                    atomicOr(&negbits[a >> 5], 1u << (a & 31));
                    atomicOr(slotmask, 1 << slot);
                }
            }
            // the next row's loads are in flight during the passes and the store
            if (od + 1 < OD) {
                ip += rstride;
                gp += rstride;
#pragma unroll
                for (int k = 0; k < WPT; ++k) {
                    if (tid + k * NT < nw) {
                        rj[k] = __ldg(ip + k * NT);
                        rgd[k] = gp[k * NT];
                    }
                }
            }
            // 2. four ordered passes
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int k = 0; k < WPT; ++k)
                    if (key[k] == q) {
                        float* a = reinterpret_cast<float*>(reinterpret_cast<char*>(ring) + off[k]);
                        *a += gv[k];
                    }
                __syncthreads();
            }
            // 3. round and store the completed slices [cs, dn), clear their accumulators
            const int dn = od + 1 < OD ? (K3 ? max(2 * od + 2 - pdk, 0) : max(ax_start<AD>(rg.ad, od + 1), 0)) : g.D;
            const int nring = min(dn, de) - cs;        // completed slices held in the ring
            const int stored = ((1 << nring) - 1) << sbc | ((1 << nring) - 1) >> (RS - sbc);
            const int marked = *slotmask & stored;
            if (marked) {
                // inputs chosen only by -0 gradients: accumulator +0 -> -0
                for (int s = 0; s < nring; ++s) {
                    int slot = sbc + s;
                    slot -= slot >= RS ? RS : 0;
                    if (!((marked >> slot) & 1)) continue;
                    const int off0 = (cs + s) * HW + h0W;
                    const int ph = AL ? 0 : (pv + off0) & (VEC - 1);
                    for (int i = tid; i < SSTR / 32; i += NT) {
                        unsigned m = negbits[slot * (SSTR / 32) + i];
                        negbits[slot * (SSTR / 32) + i] = 0u;
                        while (m) {
                            const int b = __ffs(m) - 1;
                            m &= m - 1;
                            float* acc = ring + slot * SSTR + i * 32 + b;
                            const int x = SW ? roll_swz(i * 32 + b) : i * 32 + b;   // its place in the slice
                            if (__float_as_uint(*acc) == 0u &&
                                roll_all_negzero<T, AD>(go, idx, p, off0 + x - ph, g, rg))
                                *acc = -0.0f;
                        }
                    }
                }
                __syncthreads();
                if (tid == 0) *slotmask &= ~stored;
            }
            if constexpr (SW) {
                // chunk c's lower half sits at float offset 4 * fh (fh is bit 2
                // of c for every chunk of this thread), its upper half beside it
                const int nc = L / VEC;
                for (int s = 0; s < dn - cs; ++s) {
                    T* dst = gplane + (cs + s) * HW + h0W;     // on a 16-byte boundary
                    int slot = sbc + s;
                    slot -= slot >= RS ? RS : 0;
                    float* src = ring + slot * SSTR;
                    const int fo = 4 * fh;
                    if (s < nring) {
                        for (int c = tid; c < nc; c += NT) {
                            float4* lo = reinterpret_cast<float4*>(src + c * VEC + fo);
                            float4* hi = reinterpret_cast<float4*>(src + c * VEC + (fo ^ 4));
                            const float4 a = *lo, b = *hi;
                            *lo = make_float4(0.f, 0.f, 0.f, 0.f);
                            *hi = make_float4(0.f, 0.f, 0.f, 0.f);
                            *reinterpret_cast<uint4*>(dst + c * VEC) =
                                make_uint4(pack2<T>(a.x, a.y), pack2<T>(a.z, a.w), pack2<T>(b.x, b.y),
                                           pack2<T>(b.z, b.w));
                        }
                    } else {
                        for (int c = tid; c < nc; c += NT)
                            *reinterpret_cast<uint4*>(dst + c * VEC) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            } else if constexpr (AL) {
                for (int s = 0; s < dn - cs; ++s) {
                    T* dst = gplane + (cs + s) * HW + h0W;     // on a 16-byte boundary
                    const bool cov = s < nring;
                    int slot = sbc + s;
                    slot -= slot >= RS ? RS : 0;
                    float* src = ring + slot * SSTR;
                    for (int c = tid; c < L / VEC; c += NT) {
                        uint4 out = make_uint4(0u, 0u, 0u, 0u);
                        if (cov) out = roll_take<T>(src + c * VEC, fh);
                        *reinterpret_cast<uint4*>(dst + c * VEC) = out;
                    }
                }
            }
            for (int s = 0; !AL && s < dn - cs; ++s) {
                const int off0 = (cs + s) * HW + h0W;
                const int ph = (pv + off0) & (VEC - 1);
                T* dst = gplane + (off0 - ph);          // on a 16-byte boundary
                const int nch = (ph + L + VEC - 1) / VEC;
                const bool cov = s < nring;
                int slot = sbc + s;
                slot -= slot >= RS ? RS : 0;
                float* src = ring + slot * SSTR;
                for (int c = tid; c < nch; c += NT) {
                    const int e0 = c * VEC - ph;
                    Vec16<T> out;
                    if (cov) out.u = roll_take<T>(src + c * VEC, fh);
                    else out.u = make_uint4(0u, 0u, 0u, 0u);
                    if (e0 >= 0 && e0 + VEC <= L) {
                        *reinterpret_cast<uint4*>(dst + c * VEC) = out.u;
                    } else {
#pragma unroll
                        for (int t = 0; t < VEC; ++t)
                            if (e0 + t >= 0 && e0 + t < L) dst[c * VEC + t] = out.e[t];
                    }
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

// ------------------------------------------------------------------ exchange store
// Adaptive windows whose inputs outnumber them many times over (most of
// grad_in is zeros): the same decode, ring and ordered passes as k_bwd_roll,
// but the slices a window row completes are written without reading their
// accumulators. Every element of those slices is first stored as +0 with
// 16-byte stores; then each window whose chosen input lies in them takes
// that input's accumulator with a shared atomicExch(acc, 0), which reads the
// sum and clears the accumulator in one step, and stores the rounded sum
// when it is not +0. Several windows of one input: the first exchange gets
// the sum and the others +0, so which is first does not matter. An input
// whose terms are all -0 keeps +0 in its accumulator; a window with a -0
// gradient that gets +0 re-reads the input's covering windows and stores -0
// when every term is -0. A window whose input lies in a slice the next row
// also covers takes it when the next row completes that slice.
template <typename T, int NT, int WPT, int MINB>
__global__ void __launch_bounds__(NT, MINB)
k_bwd_xroll(const T* __restrict__ go, const int64_t* __restrict__ idx, T* __restrict__ gi, Geo g,
            RollGeo rg) {
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ __align__(16) float ring[];
    const int RS = rg.RS, SSTR = rg.SSTR;
    const int nacc = RS * SSTR;
    const int tid = threadIdx.x;
    const int W = g.W, HW = g.H * g.W, OW = g.OW, OD = g.OD;
    {
        float4* r4 = reinterpret_cast<float4*>(ring);
        for (int i = tid; i < nacc / 4; i += NT) r4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const long long units = g.P * rg.nht;
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
        const long long p = u / rg.nht;
        const int h0 = (int)(u - p * rg.nht) * rg.TH;
        const int h1 = min(h0 + rg.TH, g.H);
        const int h0W = h0 * W;
        const int L = (h1 - h0) * W;
        const int ohl = ax_lo<true>(rg.ah, h0), ohh = ax_hi<true>(rg.ah, h1 - 1);
        const int nw = ohh >= ohl ? (ohh - ohl + 1) * OW : 0;
        T* gplane = gi + p * (long long)g.vol;
        int wo[WPT], wsh[WPT];
#pragma unroll
        for (int k = 0; k < WPT; ++k) {
            const int me = tid + k * NT;
            const int row = rg.fOW.div(me);
            const int oh = min(ohl + row, g.OH - 1), ow = me - row * OW;
            const int hs = ax_start<true>(rg.ah, oh), ws = ax_start<true>(rg.aw, ow);
            wo[k] = hs * W + ws;
            const int kh = ax_end<true>(rg.ah, oh) - hs, kw = ax_end<true>(rg.aw, ow) - ws;
            const int sh = oh + 1 < g.OH ? ax_start<true>(rg.ah, oh + 1) - hs : 255;
            const int sw = ow + 1 < OW ? ax_start<true>(rg.aw, ow + 1) - ws : 255;
            wsh[k] = kh | kw << 8 | sh << 16 | sw << 24;
        }
        const long long rstride = (long long)g.OH * OW;
        const int64_t* ip = idx + p * (long long)g.ovol + (long long)ohl * OW + tid;
        const T* gp = go + p * (long long)g.ovol + (long long)ohl * OW + tid;
        int64_t rj[WPT];
        T rgd[WPT];
#pragma unroll
        for (int k = 0; k < WPT; ++k) {
            const bool in = tid + k * NT < nw;
            rj[k] = in ? __ldg(ip + k * NT) : -1;
            rgd[k] = in ? gp[k * NT] : Elem<T>::from_f(0.0f);
        }
        int pj[WPT], poff[WPT];        // windows of the previous row to take in this row
        unsigned pneg = 0u;
#pragma unroll
        for (int k = 0; k < WPT; ++k) pj[k] = poff[k] = -1;
        int cs = 0;                    // first slice not yet written
        __syncthreads();
        for (int od = 0; od < OD; ++od) {
            const int ods = ax_start<true>(rg.ad, od);
            const int kd = ax_end<true>(rg.ad, od) - ods;
            const int sbo = ods % RS;
            const int dsHW = ods * HW;
            const int dn = od + 1 < OD ? ax_start<true>(rg.ad, od + 1) : g.D;   // [cs, dn) complete
            int key[WPT], off[WPT], jl[WPT];
            float gv[WPT];
            unsigned cneg = 0u;
#pragma unroll
            for (int k = 0; k < WPT; ++k) {
                const int64_t j = rj[k];
                gv[k] = Elem<T>::to_f(rgd[k]);
                jl[k] = (int)j;
                const int rel = (int)j - dsHW - wo[k];
                const int offd = rg.fHW.div(rel);
                const int rem = rel - offd * HW;
                const int offh = rg.fW.div(rem);
                const int offw = rem - offh * W;
                const int kh = wsh[k] & 255, kw = (wsh[k] >> 8) & 255;
                const int sh = (wsh[k] >> 16) & 255, sw = (unsigned)wsh[k] >> 24;
                const int loc = wo[k] - h0W + rem;
                const bool ok = (uint64_t)j < (uint64_t)g.vol && rel >= 0 && offd < kd && offh < kh &&
                                offw < kw && (unsigned)loc < (unsigned)L;
                int slot = sbo + offd;
                slot -= slot >= RS ? RS : 0;
                off[k] = (slot * SSTR + loc) * (int)sizeof(float);
                // 0-3: pass; 4: nothing; bit 3: the next row completes the input's slice
                key[k] = ok ? ((offh >= sh ? 0 : 2) | (offw >= sw ? 0 : 1) | (ods + offd >= dn ? 8 : 0)) : 4;
                if (ok && __float_as_uint(gv[k]) == 0x80000000u) cneg |= 1u << k;
            }
            if (od + 1 < OD) {
                ip += rstride;
                gp += rstride;
#pragma unroll
                for (int k = 0; k < WPT; ++k) {
                    if (tid + k * NT < nw) {
                        rj[k] = __ldg(ip + k * NT);
                        rgd[k] = gp[k * NT];
                    }
                }
            }
            // zeros into the tile's rows of the slices this row completes
            for (int s = cs; s < dn; ++s) {
                T* base = gplane + s * HW + h0W;
                const int head = (int)(((16 - ((uintptr_t)base & 15)) & 15) / sizeof(T));
                const int hd = head < L ? head : L;
                const int nv = (L - hd) / VEC;
                for (int e = tid; e < hd; e += NT) base[e] = Elem<T>::from_f(0.0f);
                uint4* v4 = reinterpret_cast<uint4*>(base + hd);
                for (int c = tid; c < nv; c += NT) v4[c] = make_uint4(0u, 0u, 0u, 0u);
                for (int e = hd + nv * VEC + tid; e < L; e += NT) base[e] = Elem<T>::from_f(0.0f);
            }
            // four ordered passes
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int k = 0; k < WPT; ++k)
                    if ((key[k] & 7) == q) {
                        float* a = reinterpret_cast<float*>(reinterpret_cast<char*>(ring) + off[k]);
                        *a += gv[k];
                    }
                __syncthreads();
            }
            auto take = [&](int aoff, int jj, bool neg) {
                unsigned* a = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(ring) + aoff);
                const unsigned v = atomicExch(a, 0u);
                if (v != 0u)
                    gplane[jj] = Elem<T>::from_f(__uint_as_float(v));
                else if (neg && roll_all_negzero<T, true>(go, idx, p, jj, g, rg))
                    gplane[jj] = Elem<T>::from_f(-0.0f);
            };
#pragma unroll
            for (int k = 0; k < WPT; ++k)
                if (pj[k] >= 0) take(poff[k], pj[k], (pneg >> k) & 1u);
#pragma unroll
            for (int k = 0; k < WPT; ++k)
                if (key[k] < 4) take(off[k], jl[k], (cneg >> k) & 1u);
#pragma unroll
            for (int k = 0; k < WPT; ++k) {
                const bool later = key[k] != 4 && (key[k] & 8);
                pj[k] = later ? jl[k] : -1;
                poff[k] = off[k];
            }
            pneg = cneg;
            cs = dn;
            __syncthreads();   // exchanges done before the next row's passes
        }
    }
}

// ------------------------------------------------------------------ host side

namespace {

// Windows along one axis as the host sees them.
struct HostAxis {
    int I, O, K, S;
    bool adaptive;
    int pad;      // fixed windows: window o starts at o*S - pad
    long long start(int o) const { return adaptive ? (long long)o * I / O : (long long)o * S - pad; }
    long long end(int o) const {
        return adaptive ? ((long long)(o + 1) * I + O - 1) / O : (long long)o * S - pad + K;
    }
    int lo(int x) const {
        if (adaptive) return (int)((long long)x * O / I);
        return x + pad < K ? 0 : (x + pad - K) / S + 1;
    }
    int hi(int x) const {
        if (adaptive) return (int)(((long long)(x + 1) * O - 1) / I);
        const int h = (x + pad) / S;
        return h < O - 1 ? h : O - 1;
    }
    // At most two windows cover any position.
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
};

HostAxis host_axis(int I, int O, int K, int S, bool adaptive, int pad = 0) {
    HostAxis a;
    a.I = I; a.O = O; a.K = K; a.S = S; a.adaptive = adaptive; a.pad = adaptive ? 0 : pad;
    return a;
}

struct RollCfg {
    int nt, wpt;     // threads, and windows per thread at most (1, 2 or 4)
    int minb;        // CTAs per SM the registers are sized for
    size_t budget;   // shared bytes per CTA
};

// 256 threads holding up to 4 windows each (64 registers), at most 54 KB of
// shared memory, so that four CTAs fit on an SM. A launch compiles for the
// fewest windows per thread that its h-tiles need. The compiled 3x3x3
// stride-2 form runs 128 threads at eight CTAs per SM: smaller h-tiles
// (512 windows each) and more CTAs in flight hide the shared-memory latency
// of the ordered passes better (on the 32x128x16x112x112 fp16 backward:
// 224 threads x 4 CTAs 523 us, 192 x 5 514 us, 160 x 6 517 us, 128 x 8
// 496 us, 96 x 10 558 us, 64 x 16 595 us).
constexpr RollCfg kRollCfg = {256, 4, 4, 54 * 1024};
constexpr RollCfg kRollCfgK3 = {128, 4, 8, 27 * 1024};

size_t roll_smem(int RS, int SSTR) {
    const size_t nacc = (size_t)RS * SSTR;
    return nacc * sizeof(float) + nacc / 8 + sizeof(int);
}

// Fills rg (h-tiling, ring size), the shared bytes and the windows per
// thread for geometry g, or returns false when the kernel does not apply.
// The planes are split into the fewest h-tiles that fit, and into more when
// that gives fewer than min_units CTAs (rows of at least 8 per h-tile).
bool roll_plan(const Geo& g, int es, long long min_units, const RollCfg& cfg, RollGeo* rg,
               size_t* smem, int* wpt) {
    const bool a = g.adaptive != 0;
    if (g.P == 0) return false;
    if (a) {   // products used by the adaptive window arithmetic stay below 2^31
        const long long lim = (1LL << 31) - 1;
        if ((long long)g.D * g.OD + g.OD > lim || (long long)g.H * g.OH + g.OH > lim ||
            (long long)g.W * g.OW + g.OW > lim)
            return false;
        if (g.OD > (1 << 20) || g.OH > (1 << 20) || g.OW > (1 << 20)) return false;
    }
    if (!a && (g.dd != 1 || g.dh != 1 || g.dw != 1)) return false;      // no dilation
    if (!a && (g.pd || g.ph || g.pw) && (g.kd > g.D || g.kh > g.H || g.kw > g.W))
        return false;      // padded windows no longer than the input (offsets decode per axis)
    const HostAxis ad = host_axis(g.D, g.OD, g.kd, g.sd, a, g.pd);
    const HostAxis ah = host_axis(g.H, g.OH, g.kh, g.sh, a, g.ph);
    const HostAxis aw = host_axis(g.W, g.OW, g.kw, g.sw, a, g.pw);
    if (!ad.two_cover() || !ah.two_cover() || !aw.two_cover()) return false;
    const int vec = 16 / es;
    const int RS = ad.longest();
    if (RS > 30) return false;                                  // slots fit a bit mask
    if (a && (ah.longest() > 254 || aw.longest() > 254)) return false;   // packed in bytes
    for (int nht = 1; nht <= g.H; ++nht) {
        const int TH = (g.H + nht - 1) / nht;
        if ((g.H + TH - 1) / TH != nht) continue;
        const long long span = (long long)TH * g.W + vec - 1;
        const long long SSTR = (span + 31) / 32 * 32;
        if (SSTR * RS > (1LL << 24)) continue;
        if (roll_smem(RS, (int)SSTR) > cfg.budget) continue;
        long long most = 0;
        for (int h0 = 0; h0 < g.H; h0 += TH) {
            const int h1 = h0 + TH < g.H ? h0 + TH : g.H;
            const int lo = ah.lo(h0), hi = ah.hi(h1 - 1);
            const long long n = hi >= lo ? (long long)(hi - lo + 1) * g.OW : 0;
            most = n > most ? n : most;
        }
        if (most > (long long)cfg.nt * cfg.wpt) continue;
        if (g.P * nht < min_units && TH > 8) {
            // more h-tiles for more CTAs, as long as each keeps 8 rows
            long long want = (min_units + g.P - 1) / g.P;
            long long cap = (g.H + 7) / 8;
            const int n2 = (int)(want < cap ? want : cap);
            if (n2 > nht) {
                nht = n2 - 1;   // the loop's increment tries n2 next
                continue;
            }
        }
        *wpt = most <= cfg.nt ? 1 : most <= 2 * cfg.nt ? 2 : 4;
        rg->TH = TH;
        rg->nht = nht;
        rg->RS = RS;
        rg->SSTR = (int)SSTR;
        rg->ad = axis_map(g.D, g.OD, g.kd, g.sd, a, g.pd);
        rg->ah = axis_map(g.H, g.OH, g.kh, g.sh, a, g.ph);
        rg->aw = axis_map(g.W, g.OW, g.kw, g.sw, a, g.pw);
        rg->fHW = FastDiv((uint32_t)(g.H * g.W));
        rg->fW = FastDiv((uint32_t)g.W);
        rg->fOW = FastDiv((uint32_t)g.OW);
        *smem = roll_smem(RS, (int)SSTR);
        return true;
    }
    return false;
}

template <typename T, bool AD, int WPT, bool K3 = false, bool AL = false, bool KP = false>
cudaError_t roll_launch(const void* go, const int64_t* idx, void* gi, const Geo& g,
                        const RollGeo& rg, size_t smem, cudaStream_t s) {
    constexpr RollCfg cfg = K3 ? kRollCfgK3 : kRollCfg;
    auto kern = k_bwd_roll<T, AD, cfg.nt, WPT, cfg.minb, K3, AL, KP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long units = g.P * rg.nht;
    const unsigned grid = (unsigned)(units < INT_MAX ? units : INT_MAX);
    kern<<<grid, cfg.nt, smem, s>>>((const T*)go, idx, (T*)gi, g, rg);
    return cudaGetLastError();
}

template <typename T>
cudaError_t roll_t(const void* go, const int64_t* idx, void* gi, const Geo& g, int sms,
                   cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    RollGeo rg;
    size_t smem = 0;
    int wpt = 0;
    // h-tiles split further only while the planes give fewer than half a
    // wave of CTAs at minb per SM: splitting to reach a whole wave left a
    // partial second one (the padded 8x64x16x56x56 fp16 backward: 1536
    // CTAs 34.8 us, 1024 CTAs 26.6 us, 2560 CTAs 45.1 us)
    const bool k3 = !g.adaptive && g.kd == 3 && g.kh == 3 && g.kw == 3 && g.sd == 2 && g.sh == 2 &&
                    g.sw == 2 && g.pd <= 1 && g.ph <= 1 && g.pw <= 1 && g.W % VEC == 0 &&
                    g.vol % VEC == 0;
    // padded, or ceil-mode sizes: windows reach past the input
    const bool reach = g.pd || g.ph || g.pw || g.OD != (g.D - 3) / 2 + 1 || g.OH != (g.H - 3) / 2 + 1 ||
                       g.OW != (g.W - 3) / 2 + 1;
    if (k3 && roll_plan(g, sizeof(T), 1LL * sms * kRollCfgK3.minb / 2, kRollCfgK3, &rg, &smem, &wpt) &&
        wpt == 4)
        return reach ? roll_launch<T, false, 4, true, true, true>(go, idx, gi, g, rg, smem, s)
                     : roll_launch<T, false, 4, true, true, false>(go, idx, gi, g, rg, smem, s);
    if (!roll_plan(g, sizeof(T), 1LL * sms * kRollCfg.minb / 2, kRollCfg, &rg, &smem, &wpt))
        return cudaErrorNotSupported;
    if (g.adaptive && g.vol >= 16LL * g.ovol) {
        // adaptive windows with many inputs each: the exchange store (the
        // 16x64x30x50x50 -> 8x12x12 fp16 backward 47.1 -> 41.0 us; on 3x3x3
        // stride-2 windows, 9.5 inputs each, it measured 565 against 481 us)
        auto kern = wpt == 1 ? k_bwd_xroll<T, kRollCfg.nt, 1, kRollCfg.minb>
                  : wpt == 2 ? k_bwd_xroll<T, kRollCfg.nt, 2, kRollCfg.minb>
                             : k_bwd_xroll<T, kRollCfg.nt, 4, kRollCfg.minb>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const long long units = g.P * rg.nht;
        kern<<<(unsigned)(units < INT_MAX ? units : INT_MAX), kRollCfg.nt, smem, s>>>((const T*)go, idx,
                                                                                     (T*)gi, g, rg);
        return cudaGetLastError();
    }
    if (g.adaptive) {
        if (wpt == 1) return roll_launch<T, true, 1>(go, idx, gi, g, rg, smem, s);
        if (wpt == 2) return roll_launch<T, true, 2>(go, idx, gi, g, rg, smem, s);
        return roll_launch<T, true, 4>(go, idx, gi, g, rg, smem, s);
    }
    if (wpt == 1) return roll_launch<T, false, 1>(go, idx, gi, g, rg, smem, s);
    if (wpt == 2) return roll_launch<T, false, 2>(go, idx, gi, g, rg, smem, s);
    return roll_launch<T, false, 4>(go, idx, gi, g, rg, smem, s);
}

int elem_bytes(int dtype) { return dtype == F32 ? 4 : 2; }

}  // namespace

bool bwd_roll_supported(const Geo& g, int dtype, bool aligned16) {
    RollGeo rg;
    size_t smem = 0;
    int wpt = 0;
    return aligned16 && roll_plan(g, elem_bytes(dtype), 0, kRollCfg, &rg, &smem, &wpt);
}

cudaError_t launch_bwd_roll(const void* go, const int64_t* idx, void* gi, const Geo& g, int dtype,
                            int sms, cudaStream_t s) {
    switch (dtype) {
    case F32: return roll_t<float>(go, idx, gi, g, sms, s);
    case F16: return roll_t<__half>(go, idx, gi, g, sms, s);
    default: return roll_t<__nv_bfloat16>(go, idx, gi, g, sms, s);
    }
}

}  // namespace mp3d
