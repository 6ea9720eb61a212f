// Forward for 16-bit types as a walk along depth: a CTA takes one plane (or
// two, in the plane-pair form further down, which the launcher prefers) and
// a group of consecutive output depths, and streams the depth slices its
// windows cover, in ascending order, through shared memory. This first form
// (order words, one plane) serves plane volumes that are not a multiple of
// 8 elements.
//
// Definition followed (teenygrad docs "Struct Maxpool3dForward",
// description and Constraints; adaptive windows
// [floor(i*I/O), ceil((i+1)*I/O)) per axis): y is the maximum of the window
// and idx the in-plane offset d*H*W + h*W + w of the first element, in
// (d, h, w) order, that attains it; a NaN beats every number.
//
// Per slice:
//  1. its bytes arrive by 16-byte asynchronous copies issued NS - 1 slices
//     ahead (cp.async groups, one per slice), so loads overlap the work on
//     earlier slices;
//  2. every element becomes one 32-bit word: the value's order key in the
//     high half (+0 and -0 one key, NaN above everything, all NaNs one key),
//     0xFFFF minus the element's in-slice offset h*W + w in the low half;
//     the unsigned maximum of a window's words is then the slice's winner
//     of that window (the earliest (h, w) among equal keys);
//  3. thread t owns output (oh, ow) = t: it takes the maximum word over its
//     (h, w) window in the slice and folds it into the accumulators of the
//     (at most two) depth windows that contain the slice, replacing an
//     accumulator only for a strictly larger key, so an earlier slice keeps
//     a tie. When the last slice of a depth window has been folded in, the
//     output is written: idx from the slice and the in-slice offset, y
//     re-read from x at that offset (the element's own bits).
// Scope of this form: 16-bit types, no padding or dilation, every window
// inside the input, at most two windows over any slice along d (fixed
// K <= 2 * S, or adaptive end(i) <= start(i + 2)), H * W <= 65536 (in-slice
// offsets fit 16 bits), OH * OW <= threads, x on a 16-byte boundary.
#include <climits>
#include <cstring>
#include <vector>

#include "internal.h"

namespace mp3d {

namespace {

constexpr int RF_NT = 256;      // threads per CTA (and the most outputs per plane-depth)
constexpr int RF_NS = 4;        // slices in flight: the current one plus NS - 1 ahead

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct RollFwdGeo {
    int odg, ngrp;      // output depths per CTA, groups per plane
    int bh, nband;      // output rows per band, bands per plane (the pair form)
    int wstr;           // words per slice buffer (multiple of 32)
    int rstr;           // bytes per raw stage (multiple of 128)
    int wait_limit;     // polls a pipeline wait makes before giving up
};

// The output (oh * OW + ow) each thread owns, 0xFFFF for none. Outputs are
// dealt to warps so that the first words of the windows of one warp lie in
// different shared-memory banks wherever the geometry allows: every lane
// then adds the same offsets as the scan proceeds, so every load of the
// window scan is one wavefront.
struct OutMap {
    uint16_t t[RF_NT];
};

}  // namespace

template <typename T, bool AD, int KH, int KW>
__global__ void __launch_bounds__(RF_NT)
k_fwd_roll(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g,
           RollFwdGeo rg, const unsigned char* __restrict__ x_end, const __grid_constant__ OutMap om) {
    extern __shared__ __align__(128) unsigned char smem_rf[];
    constexpr unsigned NANADD = KeyConst<T>::nanadd;
    unsigned* words = reinterpret_cast<unsigned*>(smem_rf);                  // [2][wstr]
    unsigned char* raw = smem_rf + 2 * rg.wstr * sizeof(unsigned);          // [NS][rstr]
    const int tid = threadIdx.x;
    const int fh = (tid >> 2) & 1;          // half order of this thread's 32-byte word stores
    const int HW = g.H * g.W;
    const long long p = blockIdx.x / rg.ngrp;
    const int grp = (int)(blockIdx.x - p * rg.ngrp);
    const int od0 = grp * rg.odg;
    const int od1 = min(od0 + rg.odg, g.OD);          // output depths [od0, od1)
    const int d_first = win_start(od0, g.D, g.OD, g.kd, g.sd, AD);
    const int d_last = win_end(od1 - 1, g.D, g.OD, g.kd, g.sd, AD);   // exclusive
    const int ns = d_last - d_first;

    // this thread's output and its (h, w) window
    const int mine = om.t[tid];
    const bool owner = mine != 0xFFFF;
    const int oh = owner ? mine / g.OW : 0;
    const int ow = owner ? mine - oh * g.OW : 0;
    const int hs = win_start(oh, g.H, g.OH, g.kh, g.sh, AD);
    const int he = win_end(oh, g.H, g.OH, g.kh, g.sh, AD);
    const int ws = win_start(ow, g.W, g.OW, g.kw, g.sw, AD);
    const int we = win_end(ow, g.W, g.OW, g.kw, g.sw, AD);
    const int woff = hs * g.W + ws;

    const unsigned char* xb = reinterpret_cast<const unsigned char*>(x + p * g.vol);
    // slice i of this CTA: global bytes [a, a + HW*2) copied from the 16-byte
    // boundary at or below a
    auto issue = [&](int i) {
        if (i < ns) {
            const unsigned char* sa = xb + (size_t)(d_first + i) * HW * sizeof(T);
            const unsigned char* a0 = reinterpret_cast<const unsigned char*>((uintptr_t)sa & ~(uintptr_t)15);
            const int nvec = (int)((sa + HW * sizeof(T) - a0 + 15) / 16);
            unsigned char* st = raw + (i % RF_NS) * rg.rstr;
            for (int v = tid; v < nvec; v += RF_NT) {
                const unsigned char* src = a0 + 16 * v;
                if (src + 16 <= x_end) {
                    cp_async16((uint32_t)__cvta_generic_to_shared(st + 16 * v), src);
                } else {
                    // the last vector of the tensor: only its bytes inside x
                    for (int b = 0; b < 16; b += 2)
                        *reinterpret_cast<unsigned short*>(st + 16 * v + b) =
                            src + b < x_end ? *reinterpret_cast<const unsigned short*>(src + b) : 0;
                }
            }
        }
        cp_async_commit();   // one group per slice, empty past the end
    };
#pragma unroll
    for (int i = 0; i < RF_NS - 1; ++i) issue(i);

    unsigned acc0 = 0u, acc1 = 0u;     // best words of depth windows a and a + 1 (key 0: none yet)
    int dd0 = 0, dd1 = 0;              // their slices
    int a = od0;                       // lowest depth window not yet written
    int a_start = d_first;             // its slices [a_start, a_end)
    int a_end = win_end(a, g.D, g.OD, g.kd, g.sd, AD);
    int b_start = a + 1 < od1 ? win_start(a + 1, g.D, g.OD, g.kd, g.sd, AD) : INT_MAX;
    for (int i = 0; i < ns; ++i) {
        cp_async_wait<RF_NS - 2>();    // this thread's copies of slice i have landed
        __syncthreads();               // everyone's have; slice i - 1's stage is free again
        issue(i + RF_NS - 1);
        // 2. order words of slice i
        const unsigned char* a_ptr = xb + (size_t)(d_first + i) * HW * sizeof(T);
        const int mis = (int)(((uintptr_t)a_ptr & 15) / sizeof(T));   // elements before the slice
        const int nvec = (int)((mis * sizeof(T) + HW * sizeof(T) + 15) / 16);
        const uint4* st = reinterpret_cast<const uint4*>(raw + (i % RF_NS) * rg.rstr);
        unsigned* wb = words + (i & 1) * rg.wstr;
        for (int v = tid; v < nvec; v += RF_NT) {
            const uint4 u = st[v];
            const unsigned k0 = order_keys2<NANADD>(u.x), k1 = order_keys2<NANADD>(u.y);
            const unsigned k2 = order_keys2<NANADD>(u.z), k3 = order_keys2<NANADD>(u.w);
            const unsigned inv = 0xFFFFu - (unsigned)(8 * v - mis);   // element 8v sits at offset 8v - mis
            const uint4 lo = make_uint4(__byte_perm(k0, inv, 0x1054), __byte_perm(k0, inv - 1, 0x3254),
                                        __byte_perm(k1, inv - 2, 0x1054), __byte_perm(k1, inv - 3, 0x3254));
            const uint4 hi = make_uint4(__byte_perm(k2, inv - 4, 0x1054), __byte_perm(k2, inv - 5, 0x3254),
                                        __byte_perm(k3, inv - 6, 0x1054), __byte_perm(k3, inv - 7, 0x3254));
            // lanes 4-7 of each quarter-warp store their upper 16 bytes first, so a
            // quarter-warp's stores meet all eight 16-byte bank groups once
            uint4* dst = reinterpret_cast<uint4*>(wb + 8 * v);
            dst[fh] = fh ? hi : lo;
            dst[fh ^ 1] = fh ? lo : hi;
        }
        __syncthreads();
        // 3. this slice's winner of the (h, w) window, folded into depth windows
        if (owner) {
            const unsigned* base = wb + mis + woff;
            unsigned best = 0u;
            if constexpr (KH > 0 && KW > 0) {
#pragma unroll
                for (int h = 0; h < KH; ++h)
#pragma unroll
                    for (int w = 0; w < KW; ++w) best = max(best, base[h * g.W + w]);
            } else {
                for (int h = 0; h < he - hs; ++h)
                    for (int w = 0; w < we - ws; ++w) best = max(best, base[h * g.W + w]);
            }
            const int d = d_first + i;
            if (d >= a_start && d < a_end && (best >> 16) > (acc0 >> 16)) { acc0 = best; dd0 = d; }
            if (d >= b_start && (best >> 16) > (acc1 >> 16)) { acc1 = best; dd1 = d; }
            // windows whose last slice this is (two adjacent windows may end together)
            while (d == a_end - 1) {
                const int off = dd0 * HW + (int)(0xFFFFu - (acc0 & 0xFFFFu));
                const long long o = ((p * g.OD + a) * (long long)g.OH) * g.OW + mine;
                y[o] = x[p * g.vol + off];
                if (idx) idx[o] = off;
                acc0 = acc1; dd0 = dd1;
                acc1 = 0u;
                ++a;
                a_start = b_start;
                a_end = a < od1 ? win_end(a, g.D, g.OD, g.kd, g.sd, AD) : INT_MAX;
                b_start = a + 1 < od1 ? win_start(a + 1, g.D, g.OD, g.kd, g.sd, AD) : INT_MAX;
            }
        }
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------ plane pairs
// The same walk with two planes per CTA, carried as the two 16-bit lanes of
// every word: a slice of each plane is staged, the two are interleaved into
// pair words, and each owner scans its (h, w) window once for both planes
// with packed compares (set.gt on f16x2 / bf16x2: strictly greater replaces,
// so the first occurrence in (h, w) order is kept, and +0 / -0 tie). The
// winner's step in the window travels in the lanes of a second word. Slices
// fold into the depth windows lane by lane with the same strict compare (an
// earlier slice keeps a tie). NaN and infinities: a running x*0 + acc turns
// NaN once either was seen in a window; those outputs are recomputed with
// the exact scalar scan. Needs both planes' slices at the same offset
// modulo 16 bytes (plane volume a multiple of 8 elements).
//
// A CTA covers a band of output rows [oh0, oh1) (at most RF_NT outputs);
// its input rows [r0, r1) are one contiguous span of each slice. Fixed
// windows may be padded (dilation 1): window o covers [o*S - p, o*S - p + K)
// clipped to the input; padding is never chosen. Windows of full size take
// the unrolled scan, clipped ones the general loop.
constexpr int PF_NS = 3;

// Set when a pipeline wait of the kernels in this file gave up (never
// expected); folded into mp3d_device_error_flags().
__device__ unsigned int g_mp3d_roll_error = 0;

// Clipped window bounds along one axis (fixed windows with padding p, or
// adaptive windows; the planner keeps (O + 1) * I below 2^31, so 32-bit
// division is exact).
template <bool AD>
__device__ __forceinline__ int cw_start(int o, int I, int O, int K, int S, int p) {
    if constexpr (AD) return (o * I) / O;
    else return max(o * S - p, 0);
}
template <bool AD>
__device__ __forceinline__ int cw_end(int o, int I, int O, int K, int S, int p) {
    if constexpr (AD) return ((o + 1) * I + O - 1) / O;
    else return min(o * S - p + K, I);
}

template <typename T>
__device__ __noinline__ void exact_output(const T* __restrict__ xp, int ds, int de, int hs, int he,
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
    if (io) *io = best;
}

template <typename T>
__device__ __forceinline__ T lane_value(uint32_t word, int lane) {
    const unsigned short b = (unsigned short)(lane ? word >> 16 : word & 0xFFFFu);
    T v;
    memcpy(&v, &b, sizeof(T));
    return v;
}

// KH, KW > 0: windows are KH x KW where not clipped; CLIP: some windows are
// clipped by the input's edges (padding or ceil mode) and take the general
// scan; KH = KW = 0: every window takes the general scan.
template <typename T, bool AD, int KH, int KW, bool CLIP>
__global__ void __launch_bounds__(RF_NT, CLIP ? 3 : 4)
k_fwd_pair(const T* __restrict__ x, T* __restrict__ y, int64_t* __restrict__ idx, Geo g,
           RollFwdGeo rg, const unsigned char* __restrict__ x_end, const __grid_constant__ OutMap om) {
    extern __shared__ __align__(128) unsigned char smem_rf[];
    uint32_t* words = reinterpret_cast<uint32_t*>(smem_rf);                 // [2][wstr] pair words
    unsigned char* raw = smem_rf + 2 * rg.wstr * sizeof(uint32_t);         // [NS][2][rstr]
    const int tid = threadIdx.x;
    const int HW = g.H * g.W;
    const int band = (int)(blockIdx.x % rg.nband);
    const long long rest = blockIdx.x / rg.nband;
    const long long pp = rest / rg.ngrp;
    const int grp = (int)(rest - pp * rg.ngrp);
    const long long p0 = 2 * pp;
    const bool has1 = p0 + 1 < g.P;
    const long long p1 = has1 ? p0 + 1 : p0;   // a lone last plane runs in both lanes
    const int od0 = grp * rg.odg;
    const int od1 = min(od0 + rg.odg, g.OD);
    const int d_first = cw_start<AD>(od0, g.D, g.OD, g.kd, g.sd, g.pd);
    const int d_last = cw_end<AD>(od1 - 1, g.D, g.OD, g.kd, g.sd, g.pd);
    const int ns = d_last - d_first;
    const int oh0 = band * rg.bh;
    const int oh1 = min(oh0 + rg.bh, g.OH);
    const int r0 = cw_start<AD>(oh0, g.H, g.OH, g.kh, g.sh, g.ph);     // input rows of the band
    const int r1 = cw_end<AD>(oh1 - 1, g.H, g.OH, g.kh, g.sh, g.ph);
    const int span = (r1 - r0) * g.W;                                  // elements per slice

    const int mine = om.t[tid];                   // output of the band, (oh - oh0) * OW + ow
    const bool owner = mine < (oh1 - oh0) * g.OW;   // 0xFFFF: none
    const int oh = owner ? oh0 + mine / g.OW : oh0;
    const int ow = owner ? mine % g.OW : 0;
    const int hs = cw_start<AD>(oh, g.H, g.OH, g.kh, g.sh, g.ph);
    const int he = cw_end<AD>(oh, g.H, g.OH, g.kh, g.sh, g.ph);
    const int ws = cw_start<AD>(ow, g.W, g.OW, g.kw, g.sw, g.pw);
    const int we = cw_end<AD>(ow, g.W, g.OW, g.kw, g.sw, g.pw);
    const int wabs = hs * g.W + ws;              // in-slice offset of the window's first element
    const int woff = (hs - r0) * g.W + ws;       // the same inside the band's span
    // clipped windows scan the full KH x KW box with rows and columns clamped
    // into the window: a clamped position repeats an element already seen
    // earlier in the scan, which never replaces the running best (strictly
    // greater only), so the first occurrence is kept
    constexpr int KH1 = KH > 0 ? KH : 1, KW1 = KW > 0 ? KW : 1;
    int crow[KH1], ccol[KW1];                    // CLIP: clamped row (span-relative, times W) and column
    if constexpr (CLIP) {
        const int nh = oh * g.sh - g.ph, nw = ow * g.sw - g.pw;   // nominal window origin
#pragma unroll
        for (int h = 0; h < KH1; ++h) crow[h] = (min(max(nh + h, hs), he - 1) - r0) * g.W;
#pragma unroll
        for (int w = 0; w < KW1; ++w) ccol[w] = min(max(nw + w, ws), we - 1);
    }
    const bool full = KH > 0 && KW > 0;

    const unsigned char* xb0 = reinterpret_cast<const unsigned char*>(x + p0 * g.vol + (long long)r0 * g.W);
    const unsigned char* xb1 = reinterpret_cast<const unsigned char*>(x + p1 * g.vol + (long long)r0 * g.W);
    uint64_t* bars = reinterpret_cast<uint64_t*>(raw + PF_NS * 2 * rg.rstr);   // one per stage
    const unsigned char* x_last = reinterpret_cast<const unsigned char*>((uintptr_t)x_end & ~(uintptr_t)15);
    // (thread 0) slice i's band span of both planes into stage i % NS: one
    // bulk copy per plane from the 16-byte boundary at or below the span up
    // to the one at or above its end (bytes of x past its last 16-byte
    // boundary, if any, by plain loads), counted by the stage's mbarrier
    auto issue = [&](int i) {
        uint32_t total = 0;
        const unsigned char* src[2];
        uint32_t bytes[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const unsigned char* sa = (q ? xb1 : xb0) + (size_t)(d_first + i) * HW * sizeof(T);
            const unsigned char* a0 = reinterpret_cast<const unsigned char*>((uintptr_t)sa & ~(uintptr_t)15);
            const unsigned char* a1 = reinterpret_cast<const unsigned char*>(
                ((uintptr_t)(sa + span * sizeof(T)) + 15) & ~(uintptr_t)15);
            const unsigned char* bend = a1 < x_last ? a1 : x_last;
            unsigned char* st = raw + ((i % PF_NS) * 2 + q) * rg.rstr;
            for (const unsigned char* t = bend; t < a1 && t < x_end; t += 2)
                *reinterpret_cast<unsigned short*>(st + (t - a0)) = *reinterpret_cast<const unsigned short*>(t);
            src[q] = a0;
            bytes[q] = bend > a0 ? (uint32_t)(bend - a0) : 0u;
            total += bytes[q];
        }
        const uint32_t bar = smem_addr(&bars[i % PF_NS]);
        mbar_expect_tx(bar, total);
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (bytes[q]) bulk_g2s(smem_addr(raw + ((i % PF_NS) * 2 + q) * rg.rstr), src[q], bytes[q], bar);
    };
    if (tid == 0) {
        for (int st = 0; st < PF_NS; ++st) mbar_init(smem_addr(&bars[st]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0)
        for (int i = 0; i < PF_NS && i < ns; ++i) issue(i);

    // depth windows a (lowest not yet written) and a + 1: best pair word,
    // the in-plane offsets of its two lanes, whether anything was folded in,
    // whether a NaN or infinity was seen
    uint32_t av0 = 0u, av1 = 0u;
    int ao0[2] = {0, 0}, ao1[2] = {0, 0};
    bool fresh0 = true, fresh1 = true, bad0 = false, bad1 = false;
    // bounded waits: a thread whose wait gives up stops waiting (its outputs
    // are then incomplete; the error flag says so); thread 0 alone issues
    // copies, waits for every slice it issued until its own wait gives up
    // (at fail_at) and refills nothing after that
    bool failed = false;
    __shared__ int fail_at;                    // (thread 0) the slice whose wait gave up
    unsigned redo = 0u;                        // depth windows (bit a - od0) seen with NaN or inf
    int a = od0;
    int a_start = d_first;
    int a_end = cw_end<AD>(a, g.D, g.OD, g.kd, g.sd, g.pd);
    int b_start = a + 1 < od1 ? cw_start<AD>(a + 1, g.D, g.OD, g.kd, g.sd, g.pd) : INT_MAX;
    for (int i = 0; i < ns; ++i) {
        if (!failed && !mbar_wait(smem_addr(&bars[i % PF_NS]), (uint32_t)((i / PF_NS) & 1), rg.wait_limit)) {
            failed = true;
            if (tid == 0) fail_at = i;
            atomicOr(&g_mp3d_roll_error, kErrPipelineTimeout);
        }
        const unsigned char* sa = xb0 + (size_t)(d_first + i) * HW * sizeof(T);
        const int mis = (int)(((uintptr_t)sa & 15) / sizeof(T));
        const int nvec = (int)((mis * sizeof(T) + span * sizeof(T) + 15) / 16);
        const uint4* s0 = reinterpret_cast<const uint4*>(raw + ((i % PF_NS) * 2) * rg.rstr);
        const uint4* s1 = reinterpret_cast<const uint4*>(raw + ((i % PF_NS) * 2 + 1) * rg.rstr);
        uint32_t* wb = words + (i & 1) * rg.wstr;
        for (int v = tid; v < nvec; v += RF_NT) {
            const uint4 A = s0[v], B = s1[v];
            // word j: element j of plane p0 in the low lane, of plane p1 in the high lane
            const uint4 lo = make_uint4(__byte_perm(A.x, B.x, 0x5410), __byte_perm(A.x, B.x, 0x7632),
                                        __byte_perm(A.y, B.y, 0x5410), __byte_perm(A.y, B.y, 0x7632));
            const uint4 hi = make_uint4(__byte_perm(A.z, B.z, 0x5410), __byte_perm(A.z, B.z, 0x7632),
                                        __byte_perm(A.w, B.w, 0x5410), __byte_perm(A.w, B.w, 0x7632));
            uint4* dst = reinterpret_cast<uint4*>(wb + 8 * v);
            dst[0] = lo;
            dst[1] = hi;
        }
        // every thread is done with stage i % NS (refilled below) and with
        // the words of slice i - 1 (overwritten next iteration)
        __syncthreads();
        if (tid == 0 && i + PF_NS < ns && !failed) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(i + PF_NS);
        }
        if (owner) {
            const uint32_t* base = wb + mis + woff;
            uint32_t mv = base[0], mk = 0u;
            uint32_t pz = Pair<T>::poison(0u, mv);
            int o_lane[2];
            if (full) {
                // each row along w on its own (independent chains), then the
                // rows in ascending order; a later candidate replaces only
                // when strictly greater, so ties keep the earlier element
                const uint32_t* cbase = wb + mis;
                auto at = [&](int h, int w) {
                    if constexpr (CLIP) return cbase[crow[h] + ccol[w]];
                    else return base[h * g.W + w];
                };
                uint32_t rv[KH1], rk[KH1], rp[KH1];
#pragma unroll
                for (int h = 0; h < KH1; ++h) {
                    rv[h] = at(h, 0);
                    rk[h] = (uint32_t)(h * KW1) * 0x00010001u;
                    rp[h] = Pair<T>::poison(0u, rv[h]);
#pragma unroll
                    for (int w = 1; w < KW1; ++w) {
                        const uint32_t v = at(h, w);
                        merge2<T>(rv[h], rk[h], v, (uint32_t)(h * KW1 + w) * 0x00010001u);
                        rp[h] = Pair<T>::poison(rp[h], v);
                    }
                }
                mv = rv[0];
                mk = rk[0];
                pz = rp[0];
#pragma unroll
                for (int h = 1; h < KH1; ++h) {
                    merge2<T>(mv, mk, rv[h], rk[h]);
                    pz = Pair<T>::poison(pz, rp[h]);
                }
#pragma unroll
                for (int l = 0; l < 2; ++l) {
                    const int k = (int)(l ? mk >> 16 : mk & 0xFFFFu);
                    if constexpr (CLIP) {
                        const int nh = oh * g.sh - g.ph, nw = ow * g.sw - g.pw;
                        o_lane[l] = min(max(nh + k / KW1, hs), he - 1) * g.W + min(max(nw + k % KW1, ws), we - 1);
                    } else {
                        o_lane[l] = wabs + (k / KW1) * g.W + k % KW1;
                    }
                }
            } else {
                // general lengths: the lanes carry the winner's offset h * W + w
                // inside the window box (below H * W <= 65536)
                for (int h = 0; h < he - hs; ++h)
                    for (int w = 0; w < we - ws; ++w) {
                        if ((h | w) == 0) continue;
                        const uint32_t v = base[h * g.W + w];
                        merge2<T>(mv, mk, v, (uint32_t)(h * g.W + w) * 0x00010001u);
                        pz = Pair<T>::poison(pz, v);
                    }
#pragma unroll
                for (int l = 0; l < 2; ++l) o_lane[l] = wabs + (int)(l ? mk >> 16 : mk & 0xFFFFu);
            }
            const bool bad = Pair<T>::is_poisoned(pz);
            const int d = d_first + i;
            const int dHW = d * HW;
            if (d >= a_start && d < a_end) {
                const uint32_t m = fresh0 ? 0xFFFFFFFFu : Pair<T>::gt(mv, av0);
                av0 = (mv & m) | (av0 & ~m);
                if (m & 0xFFFFu) ao0[0] = dHW + o_lane[0];
                if (m >> 16) ao0[1] = dHW + o_lane[1];
                fresh0 = false;
                bad0 |= bad;
            }
            if (d >= b_start) {
                const uint32_t m = fresh1 ? 0xFFFFFFFFu : Pair<T>::gt(mv, av1);
                av1 = (mv & m) | (av1 & ~m);
                if (m & 0xFFFFu) ao1[0] = dHW + o_lane[0];
                if (m >> 16) ao1[1] = dHW + o_lane[1];
                fresh1 = false;
                bad1 |= bad;
            }
            // windows whose last slice this is (two adjacent windows may end together)
            while (d == a_end - 1) {
#pragma unroll
                for (int l = 0; l < 2; ++l) {
                    if (l == 1 && !has1) break;
                    const long long o = (((l ? p1 : p0) * g.OD + a) * (long long)g.OH + oh) * g.OW + ow;
                    y[o] = lane_value<T>(av0, l);
                    if (idx) idx[o] = ao0[l];
                }
                if (bad0) redo |= 1u << (a - od0);      // recomputed after the walk
                av0 = av1; ao0[0] = ao1[0]; ao0[1] = ao1[1];
                fresh0 = fresh1; bad0 = bad1;
                fresh1 = true; bad1 = false;
                ++a;
                a_start = b_start;
                a_end = a < od1 ? cw_end<AD>(a, g.D, g.OD, g.kd, g.sd, g.pd) : INT_MAX;
                b_start = a + 1 < od1 ? cw_start<AD>(a + 1, g.D, g.OD, g.kd, g.sd, g.pd) : INT_MAX;
            }
        }
    }
    // after thread 0's wait gave up at slice f, let the copies still in
    // flight land before the CTA exits: thread 0 issued nothing after that
    // wait, so they are among slices [f, f + NS)
    if (failed && tid == 0)
        for (int k = fail_at; k < fail_at + PF_NS && k < ns; ++k)
            mbar_wait(smem_addr(&bars[k % PF_NS]), (uint32_t)((k / PF_NS) & 1), kWaitLimit);
    // outputs whose windows held a NaN or an infinity: the exact scalar scan
    while (redo) {
        const int r = od0 + __ffs(redo) - 1;
        redo &= redo - 1;
        const int ds = cw_start<AD>(r, g.D, g.OD, g.kd, g.sd, g.pd);
        const int de = cw_end<AD>(r, g.D, g.OD, g.kd, g.sd, g.pd);
        for (int l = 0; l < (has1 ? 2 : 1); ++l) {
            const long long pl = l ? p1 : p0;
            const long long o = ((pl * g.OD + r) * (long long)g.OH + oh) * g.OW + ow;
            exact_output<T>(x + pl * g.vol, ds, de, hs, he, ws, we, g.W, HW, y + o, idx ? idx + o : nullptr);
        }
    }
}

namespace {


// Depth windows: at most two over any slice.
bool depth_two_cover(const Geo& g) {
    if (!g.adaptive) return g.kd <= 2 * g.sd;
    for (int i = 0; i + 2 < g.OD; ++i) {
        const long long e = ((long long)(i + 1) * g.D + g.OD - 1) / g.OD;
        const long long s2 = (long long)(i + 2) * g.D / g.OD;
        if (e > s2) return false;
    }
    return true;
}

// Clipped window bounds along one axis, as the kernels compute them.
long long h_start(int o, int I, int O, int K, int S, int p, bool ad) {
    if (ad) return (long long)o * I / O;
    const long long v = (long long)o * S - p;
    return v > 0 ? v : 0;
}
long long h_end(int o, int I, int O, int K, int S, int p, bool ad) {
    if (ad) return ((long long)(o + 1) * I + O - 1) / O;
    const long long v = (long long)o * S - p + K;
    return v < I ? v : I;
}

// pair: two planes per CTA (the packed form, bands of output rows, padded
// windows allowed); else one plane per CTA (order words, no padding, one
// band).
bool plan_rf(const Geo& g, int sms, bool pair, RollFwdGeo* rg, size_t* smem) {
    const bool ad = g.adaptive != 0;
    const long long HW = (long long)g.H * g.W;
    if (HW > 65536 || g.OW > RF_NT) return false;
    if (g.dd != 1 || g.dh != 1 || g.dw != 1) return false;
    if (ad && ((long long)(g.OD + 1) * g.D >= (1LL << 31) || (long long)(g.OH + 1) * g.H >= (1LL << 31) ||
               (long long)(g.OW + 1) * g.W >= (1LL << 31)))
        return false;     // adaptive window arithmetic in 32 bits
    if (!pair && (g.pd || g.ph || g.pw || (long long)g.OH * g.OW > RF_NT)) return false;
    // the order-word form does not clip windows: every fixed window must lie
    // inside the input (ceil mode can place the last one partly outside)
    if (!pair && !ad &&
        ((long long)(g.OD - 1) * g.sd + g.kd > g.D || (long long)(g.OH - 1) * g.sh + g.kh > g.H ||
         (long long)(g.OW - 1) * g.sw + g.kw > g.W))
        return false;
    if (!depth_two_cover(g)) return false;
    if (pair && g.vol % 8 != 0) return false;
    int bh = g.OH, nband = 1;
    if (pair) {
        const long long nb = ((long long)g.OH * g.OW + RF_NT - 1) / RF_NT;
        bh = (int)((g.OH + nb - 1) / nb);
        if (bh * g.OW > RF_NT) bh = RF_NT / g.OW;
        nband = (g.OH + bh - 1) / bh;
    }
    long long rows = 0;      // input rows of the widest band
    for (int b = 0; b < nband; ++b) {
        const int o0 = b * bh, o1 = o0 + bh < g.OH ? o0 + bh : g.OH;
        const long long r = h_end(o1 - 1, g.H, g.OH, g.kh, g.sh, g.ph, ad) -
                            h_start(o0, g.H, g.OH, g.kh, g.sh, g.ph, ad);
        rows = r > rows ? r : rows;
    }
    if (!pair) rows = g.H;   // the order-word form stages whole slices
    rg->bh = bh;
    rg->nband = nband;
    // a span reaches up to 7 elements before and after it
    rg->wstr = (int)((rows * g.W + 16 + 31) / 32 * 32);
    rg->rstr = (int)((rows * g.W * 2 + 32 + 127) / 128 * 128);
    *smem = 2 * (size_t)rg->wstr * 4 + (size_t)(pair ? 2 * PF_NS : RF_NS) * rg->rstr +
            (pair ? PF_NS * sizeof(uint64_t) : 0);
    if (*smem > 96 * 1024) return false;
    // groups of output depths: enough CTAs for a few waves (one wave of
    // four per SM for the pair form: longer walks load fewer slices twice;
    // measured 58 -> 54 us on the 16x64x30x50x50 adaptive forward)
    const long long units = (pair ? (g.P + 1) / 2 : g.P) * nband;
    const long long want = (pair ? 1LL : 4LL) * sms * 4;
    int odg = g.OD;
    while (odg > 1 && (units * ((g.OD + odg - 1) / odg) < want || (pair && odg > 32)))
        odg = (odg + 1) / 2;
    rg->odg = odg;
    rg->ngrp = (g.OD + odg - 1) / odg;
    return units * rg->ngrp <= INT_MAX;
}

// Deal the outputs of one band (local index (oh - oh0) * OW + ow, with the
// window pattern of a band inside the plane, where padding clips nothing)
// to threads: warp by warp, at most one output per bank of its window's
// first word (offset in the band's span modulo 32 words); outputs left over
// take any free thread.
void deal_outputs(const Geo& g, int bh, OutMap* om) {
    const bool ad = g.adaptive != 0;
    const int nloc = bh * g.OW;
    const int nband = (g.OH + bh - 1) / bh;
    const int oh0 = (nband > 2 ? 1 : 0) * bh;      // a band inside the plane, where windows are whole
    const long long r0 = h_start(oh0, g.H, g.OH, g.kh, g.sh, g.ph, ad);
    std::vector<std::vector<int>> by_bank(32);
    for (int o = nloc - 1; o >= 0; --o) {   // reversed: popped from the back in ascending order
        const int oh = oh0 + o / g.OW, ow = o - (o / g.OW) * g.OW;
        const long long hs = h_start(oh < g.OH ? oh : g.OH - 1, g.H, g.OH, g.kh, g.sh, g.ph, ad);
        const long long ws = h_start(ow, g.W, g.OW, g.kw, g.sw, g.pw, ad);
        by_bank[(int)(((hs - r0) * g.W + ws) % 32)].push_back(o);
    }
    for (int i = 0; i < RF_NT; ++i) om->t[i] = 0xFFFF;
    std::vector<int> spare;
    for (int w = 0; w < RF_NT / 32; ++w) {
        int lane = 0;
        for (int b = 0; b < 32; ++b)
            if (!by_bank[b].empty()) {
                om->t[w * 32 + lane++] = (uint16_t)by_bank[b].back();
                by_bank[b].pop_back();
            }
    }
    for (auto& v : by_bank)
        for (int o : v) spare.push_back(o);
    size_t k = 0;
    for (int i = 0; i < RF_NT && k < spare.size(); ++i)
        if (om->t[i] == 0xFFFF) om->t[i] = (uint16_t)spare[k++];
}

template <typename T, bool AD>
auto rf_kernel(int kh, int kw) {
    if (kh == kw) {
        switch (kh) {
        case 2: return k_fwd_roll<T, AD, 2, 2>;
        case 3: return k_fwd_roll<T, AD, 3, 3>;
        case 4: return k_fwd_roll<T, AD, 4, 4>;
        case 5: return k_fwd_roll<T, AD, 5, 5>;
        default: break;
        }
    }
    return k_fwd_roll<T, AD, 0, 0>;
}

template <typename T, bool AD, bool CLIP>
auto pf_kernel(int kh, int kw) {
    if (kh == kw) {
        switch (kh) {
        case 2: return k_fwd_pair<T, AD, 2, 2, CLIP>;
        case 3: return k_fwd_pair<T, AD, 3, 3, CLIP>;
        case 4: return k_fwd_pair<T, AD, 4, 4, CLIP>;
        case 5: return k_fwd_pair<T, AD, 5, 5, CLIP>;
        default: break;
        }
    }
    return k_fwd_pair<T, AD, 0, 0, false>;
}

// Whether a fixed-window geometry clips any window at the input's edges
// (padding, or ceil mode placing the last window partly outside).
bool clips(const Geo& g) {
    if (g.adaptive) return false;
    return g.pd || g.ph || g.pw || (long long)(g.OD - 1) * g.sd + g.kd > g.D ||
           (long long)(g.OH - 1) * g.sh + g.kh > g.H || (long long)(g.OW - 1) * g.sw + g.kw > g.W;
}

template <typename T>
cudaError_t rf_t(const void* x, void* y, int64_t* idx, const Geo& g, int sms, cudaStream_t s) {
    RollFwdGeo rg;
    size_t smem = 0;
    const bool pair = plan_rf(g, sms, true, &rg, &smem);
    if (!pair && !plan_rf(g, sms, false, &rg, &smem)) return cudaErrorNotSupported;
    const int kh = uniform_window_len(g.H, g.OH, g.kh, g.adaptive);
    const int kw = uniform_window_len(g.W, g.OW, g.kw, g.adaptive);
    auto kern = pair ? (g.adaptive ? pf_kernel<T, true, false>(kh, kw)
                                   : clips(g) ? pf_kernel<T, false, true>(kh, kw)
                                              : pf_kernel<T, false, false>(kh, kw))
                     : (g.adaptive ? rf_kernel<T, true>(kh, kw) : rf_kernel<T, false>(kh, kw));
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long ctas = (pair ? (g.P + 1) / 2 : g.P) * rg.ngrp * rg.nband;
    if (ctas > INT_MAX) return cudaErrorNotSupported;
    const unsigned char* x_end = static_cast<const unsigned char*>(x) + (size_t)g.P * g.vol * sizeof(T);
    OutMap om;
    deal_outputs(g, rg.bh, &om);
    rg.wait_limit = pipeline_wait_limit();
    kern<<<(unsigned)ctas, RF_NT, smem, s>>>((const T*)x, (T*)y, idx, g, rg, x_end, om);
    return cudaGetLastError();
}

}  // namespace

cudaError_t read_roll_fwd_error(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_mp3d_roll_error, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_mp3d_roll_error, &zero, sizeof(unsigned int));
}

bool fwd_roll_supported(const Geo& g, int dtype, bool aligned16) {
    RollFwdGeo rg;
    size_t smem = 0;
    return dtype != F32 && aligned16 &&
           (plan_rf(g, 1, true, &rg, &smem) || plan_rf(g, 1, false, &rg, &smem));
}

cudaError_t launch_fwd_roll(const void* x, void* y, int64_t* idx, const Geo& g, int dtype, int sms,
                            cudaStream_t s) {
    switch (dtype) {
    case F16: return rf_t<__half>(x, y, idx, g, sms, s);
    case BF16: return rf_t<__nv_bfloat16>(x, y, idx, g, sms, s);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace mp3d
