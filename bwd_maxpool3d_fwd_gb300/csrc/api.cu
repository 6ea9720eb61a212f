// C ABI of libmp3d.so: argument checks, shape math, path choice, launch.
//
// Every argument error is reported before the first CUDA call, so a bad
// call touches neither the device nor the buffers. The library allocates
// nothing and never synchronises; it enqueues on the caller's stream.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "internal.h"
#include "mp3d.h"

using namespace mp3d;

namespace {

constexpr long long kMaxVol = (1LL << 31) - 1;   // per-plane volumes stay int32

int elem_size(int dtype) {
    switch (dtype) {
    case MP3D_F32: return 4;
    case MP3D_F16: return 2;
    case MP3D_BF16: return 2;
    default: return 0;
    }
}

bool log_enabled() {
    static int on = -1;
    if (on < 0) {
        const char* v = std::getenv("MP3D_LOG");
        on = (v && *v && std::strcmp(v, "0") != 0) ? 1 : 0;
    }
    return on == 1;
}

const char* path_name(int path) {
    switch (path) {
    case MP3D_PATH_NOOP: return "noop";
    case MP3D_PATH_FWD_GENERIC: return "fwd_generic";
    case MP3D_PATH_FWD_S2: return "fwd_s2";
    case MP3D_PATH_FWD_GLOBAL: return "fwd_global";
    case MP3D_PATH_FWD_SLAB: return "fwd_slab";
    case MP3D_PATH_FWD_ROLL: return "fwd_roll";
    case MP3D_PATH_BWD_DISJOINT: return "bwd_disjoint";
    case MP3D_PATH_BWD_OVERLAP_TILE: return "bwd_overlap_tile";
    case MP3D_PATH_BWD_OVERLAP_DIRECT: return "bwd_overlap_direct";
    case MP3D_PATH_BWD_ATOMIC: return "bwd_atomic";
    case MP3D_PATH_BWD_OVERLAP_ROLL: return "bwd_overlap_roll";
    case MP3D_PATH_FWD_PADDED: return "fwd_padded";
    case MP3D_PATH_BWD_PADDED: return "bwd_padded";
    case MP3D_PATH_BWD_RECOMPUTE_TILES: return "bwd_recompute_k2s2";
    case MP3D_PATH_BWD_RECOMPUTE: return "bwd_recompute_direct";
    case MP3D_PATH_FWD_NDHWC: return "fwd_ndhwc";
    case MP3D_PATH_BWD_NDHWC: return "bwd_ndhwc";
    case MP3D_PATH_BWD_NDHWC_ROLL: return "bwd_ndhwc_roll";
    default: return "?";
    }
}

void log_path(const char* op, int path, const Geo& g, int dtype) {
    if (!log_enabled()) return;
    std::fprintf(stderr,
                 "mp3d: %s path=%s dtype=%d P=%lld in=%dx%dx%d out=%dx%dx%d %s k=%d,%d,%d s=%d,%d,%d\n",
                 op, path_name(path), dtype, g.P, g.D, g.H, g.W, g.OD, g.OH, g.OW,
                 g.adaptive ? "adaptive" : "fixed", g.kd, g.kh, g.kw, g.sd, g.sh, g.sw);
}

// Number of SMs of the current device (cached per device).
cudaError_t sm_count(int* out) {
    static int cache[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) {
        *out = cache[dev];
        return cudaSuccess;
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    *out = n;
    return cudaSuccess;
}

int check_dims(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, Geo* g) {
    if (N < 0 || C < 0 || D < 1 || H < 1 || W < 1) return MP3D_ERR_SHAPE;
    if (D > kMaxVol || H > kMaxVol || W > kMaxVol) return MP3D_ERR_SHAPE;
    if (D * H > kMaxVol || D * H * W > kMaxVol) return MP3D_ERR_SHAPE;
    const long long vol = D * H * W;
    if (C > 0 && N > (1LL << 62) / C) return MP3D_ERR_SHAPE;
    const long long P = N * C;
    if (P > 0 && P > (1LL << 62) / vol) return MP3D_ERR_SHAPE;
    std::memset(g, 0, sizeof(*g));
    g->dd = g->dh = g->dw = 1;
    g->P = P;
    g->D = (int)D; g->H = (int)H; g->W = (int)W;
    g->vol = (int)vol;
    return MP3D_OK;
}

int set_out(Geo* g, long long od, long long oh, long long ow) {
    if (od < 1 || oh < 1 || ow < 1) return MP3D_ERR_SHAPE;
    if (od > kMaxVol || oh > kMaxVol || ow > kMaxVol) return MP3D_ERR_SHAPE;
    if (od * oh > kMaxVol || od * oh * ow > kMaxVol) return MP3D_ERR_SHAPE;
    if (g->P > 0 && g->P > (1LL << 62) / (od * oh * ow)) return MP3D_ERR_SHAPE;
    g->OD = (int)od; g->OH = (int)oh; g->OW = (int)ow;
    g->ovol = (int)(od * oh * ow);
    return MP3D_OK;
}

int fixed_geo(Geo* g, int kd, int kh, int kw, int sd, int sh, int sw) {
    if (kd < 1 || kh < 1 || kw < 1 || sd < 1 || sh < 1 || sw < 1) return MP3D_ERR_WINDOW;
    if (kd > g->D || kh > g->H || kw > g->W) return MP3D_ERR_WINDOW;
    g->adaptive = 0;
    g->kd = kd; g->kh = kh; g->kw = kw;
    g->sd = sd; g->sh = sh; g->sw = sw;
    return set_out(g, (g->D - kd) / sd + 1, (g->H - kh) / sh + 1, (g->W - kw) / sw + 1);
}

int adaptive_geo(Geo* g, int od, int oh, int ow) {
    g->adaptive = 1;
    return set_out(g, od, oh, ow);
}

// Output length along one axis with padding p (both sides), dilation dl
// and ceil mode, as the usual max_pool3d defines it: padding at most half
// the kernel, floor (ceil) of (I + 2p - dl*(K-1) - 1)/S plus 1, and in ceil
// mode a last window wholly in the right padding dropped. 0 when invalid.
long long ex_out_len(long long I, long long K, long long S, long long p, long long dl, int ceil_mode) {
    if (I < 1 || K < 1 || S < 1 || dl < 1 || p < 0 || 2 * p > K) return 0;
    long long num = I + 2 * p - dl * (K - 1) - 1;
    if (ceil_mode) num += S - 1;
    long long O = (num >= 0 ? num / S : -((-num + S - 1) / S)) + 1;   // floor division
    if (ceil_mode && (O - 1) * S >= I + p) --O;
    return O < 1 ? 0 : O;
}

// Every window o < O along the axis has a position o*S - p + k*dl inside
// [0, I). Always true without dilation (padding is at most half the kernel
// and the last window starts before I); checked window by window otherwise.
bool ex_windows_nonempty(long long I, long long O, long long K, long long S, long long p,
                         long long dl) {
    if (dl == 1) return true;
    for (long long o = 0; o < O; ++o) {
        bool any = false;
        for (long long k = 0; k < K && !any; ++k) {
            const long long x = o * S - p + k * dl;
            any = x >= 0 && x < I;
        }
        if (!any) return false;
    }
    return true;
}

// Fixed windows with padding, dilation and ceil mode.
int ex_geo(Geo* g, int kd, int kh, int kw, int sd, int sh, int sw, int pd, int ph, int pw, int dd,
           int dh, int dw, int ceil_mode) {
    if (kd < 1 || kh < 1 || kw < 1 || sd < 1 || sh < 1 || sw < 1) return MP3D_ERR_WINDOW;
    if (dd < 1 || dh < 1 || dw < 1 || pd < 0 || ph < 0 || pw < 0) return MP3D_ERR_WINDOW;
    if (ceil_mode != 0 && ceil_mode != 1) return MP3D_ERR_WINDOW;
    const long long od = ex_out_len(g->D, kd, sd, pd, dd, ceil_mode);
    const long long oh = ex_out_len(g->H, kh, sh, ph, dh, ceil_mode);
    const long long ow = ex_out_len(g->W, kw, sw, pw, dw, ceil_mode);
    if (od < 1 || oh < 1 || ow < 1) return MP3D_ERR_WINDOW;
    if (!ex_windows_nonempty(g->D, od, kd, sd, pd, dd) || !ex_windows_nonempty(g->H, oh, kh, sh, ph, dh) ||
        !ex_windows_nonempty(g->W, ow, kw, sw, pw, dw))
        return MP3D_ERR_WINDOW;
    g->adaptive = 0;
    g->kd = kd; g->kh = kh; g->kw = kw;
    g->sd = sd; g->sh = sh; g->sw = sw;
    g->pd = pd; g->ph = ph; g->pw = pw;
    g->dd = dd; g->dh = dh; g->dw = dw;
    return set_out(g, od, oh, ow);
}

// No padding, no dilation, and the output the unpadded formula gives: the
// plain fixed-window geometry with its own fast paths.
bool ex_is_plain(const Geo& g) {
    return g.pd == 0 && g.ph == 0 && g.pw == 0 && g.dd == 1 && g.dh == 1 && g.dw == 1 &&
           g.OD == (g.D - g.kd) / g.sd + 1 && g.OH == (g.H - g.kh) / g.sh + 1 &&
           g.OW == (g.W - g.kw) / g.sw + 1;
}

// [a, a+na) and [b, b+nb) (bytes) overlap?
bool overlaps(const void* a, long long na, const void* b, long long nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return na > 0 && nb > 0 && pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

bool misaligned(const void* p, int bytes) { return ((uintptr_t)p % (uintptr_t)bytes) != 0; }

// Every window covers the whole plane: a global reduction per plane.
bool is_global(const Geo& g) {
    if (g.ovol != 1) return false;
    if (g.adaptive) return true;
    return g.kd == g.D && g.kh == g.H && g.kw == g.W;
}

// Disjoint windows: each input lies in at most one window.
bool is_disjoint(const Geo& g) {
    if (g.adaptive) return g.D % g.OD == 0 && g.H % g.OH == 0 && g.W % g.OW == 0;
    return g.kd <= g.sd && g.kh <= g.sh && g.kw <= g.sw;
}

// The disjoint gather works on fixed windows: divisible adaptive windows
// are fixed windows with kernel = stride = input / output.
Geo as_fixed(const Geo& g) {
    Geo f = g;
    if (g.adaptive) {
        f.adaptive = 0;
        f.kd = f.sd = g.D / g.OD;
        f.kh = f.sh = g.H / g.OH;
        f.kw = f.sw = g.W / g.OW;
    }
    return f;
}

int fwd_path(const Geo& g, int dtype, bool aligned16 = true) {
    if (g.P == 0) return MP3D_PATH_NOOP;
    if (is_global(g)) return MP3D_PATH_FWD_GLOBAL;
    if (fwd_s2_supported(g, dtype, aligned16)) return MP3D_PATH_FWD_S2;
    if (fwd_roll_supported(g, dtype, aligned16)) return MP3D_PATH_FWD_ROLL;
    if (fwd_slab_supported(g, dtype)) return MP3D_PATH_FWD_SLAB;
    return MP3D_PATH_FWD_GENERIC;
}

int bwd_path(const Geo& g, int dtype, int algo, bool aligned16 = true) {
    if (g.P == 0) return MP3D_PATH_NOOP;
    if (algo == MP3D_BWD_ATOMIC) return MP3D_PATH_BWD_ATOMIC;
    if (is_disjoint(g)) return MP3D_PATH_BWD_DISJOINT;
    if (bwd_roll_supported(g, dtype, aligned16)) return MP3D_PATH_BWD_OVERLAP_ROLL;
    if (bwd_tile_supported(g)) return MP3D_PATH_BWD_OVERLAP_TILE;
    return MP3D_PATH_BWD_OVERLAP_DIRECT;
}

int run_fwd(const void* x, void* y, int64_t* idx, const Geo& g, int dtype, cudaStream_t s) {
    const int path = fwd_path(g, dtype, (uintptr_t)x % 16 == 0);
    log_path("fwd", path, g, dtype);
    if (path == MP3D_PATH_NOOP) return MP3D_OK;
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return MP3D_ERR_CUDA;
    cudaError_t e;
    switch (path) {
    case MP3D_PATH_FWD_GLOBAL: e = launch_fwd_global(x, y, idx, g, dtype, sms, s); break;
    case MP3D_PATH_FWD_S2: e = launch_fwd_s2(x, y, idx, g, dtype, sms, s); break;
    case MP3D_PATH_FWD_SLAB: e = launch_fwd_slab(x, y, idx, g, dtype, sms, s); break;
    case MP3D_PATH_FWD_ROLL: e = launch_fwd_roll(x, y, idx, g, dtype, sms, s); break;
    default: e = launch_fwd_generic(x, y, idx, g, dtype, sms, s); break;
    }
    return e == cudaSuccess ? MP3D_OK : MP3D_ERR_CUDA;
}

// Checks shared by both forward entry points once the geometry is known.
int check_fwd_buffers(const void* x, const void* y, const int64_t* idx, const Geo& g, int dtype) {
    const int es = elem_size(dtype);
    if (es == 0) return MP3D_ERR_DTYPE;
    if (g.P == 0) return MP3D_OK;
    if (!x || !y) return MP3D_ERR_NULLPTR;                 // idx NULL: values only
    if (misaligned(x, es) || misaligned(y, es) || (idx && misaligned(idx, 8))) return MP3D_ERR_ALIGN;
    const long long nx = g.P * g.vol * es, ny = g.P * g.ovol * es, ni = idx ? g.P * g.ovol * 8 : 0;
    if (overlaps(x, nx, y, ny) || overlaps(x, nx, idx, ni) || overlaps(y, ny, idx, ni))
        return MP3D_ERR_ALIAS;
    return MP3D_OK;
}

size_t workspace_needed(const Geo& g, int dtype, int algo) {
    if (algo != MP3D_BWD_ATOMIC || dtype == MP3D_F32) return 0;
    return (size_t)(g.P * (long long)g.vol) * sizeof(float);
}

// Path choice and launch of a checked backward call on the plain (unpadded)
// geometry.
int run_bwd(const void* grad_out, const int64_t* idx, void* grad_in, void* workspace, const Geo& g,
            int dtype, int algo, cudaStream_t stream) {
    const int path = bwd_path(g, dtype, algo, (uintptr_t)grad_in % 16 == 0);
    const Geo gk = (path == MP3D_PATH_BWD_DISJOINT) ? as_fixed(g) : g;
    log_path("bwd", path, gk, dtype);
    if (path == MP3D_PATH_NOOP) return MP3D_OK;
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return MP3D_ERR_CUDA;
    cudaError_t e;
    switch (path) {
    case MP3D_PATH_BWD_ATOMIC:
        e = launch_bwd_atomic(grad_out, idx, grad_in, (float*)workspace, gk, dtype, sms, stream);
        break;
    case MP3D_PATH_BWD_DISJOINT:
        e = launch_bwd_disjoint(grad_out, idx, grad_in, gk, dtype, sms, stream);
        break;
    case MP3D_PATH_BWD_OVERLAP_ROLL:
        e = launch_bwd_roll(grad_out, idx, grad_in, gk, dtype, sms, stream);
        break;
    case MP3D_PATH_BWD_OVERLAP_TILE:
        e = launch_bwd_overlap_tile(grad_out, idx, grad_in, gk, dtype, sms, stream);
        break;
    default:
        e = launch_bwd_overlap_direct(grad_out, idx, grad_in, gk, dtype, sms, stream);
        break;
    }
    return e == cudaSuccess ? MP3D_OK : MP3D_ERR_CUDA;
}

// Path of a padded / dilated backward: ATOMIC on request; the rolling
// ordered scatter when it takes the geometry (no dilation, at most two
// windows over any position); else the direct gather.
// Padded / dilated / ceil-mode forward: the depth walk for 16-bit types
// (dilation 1), else the thread-per-output kernel.
int ex_fwd_path(const Geo& g, int dtype, bool aligned16 = true) {
    if (g.P == 0) return MP3D_PATH_NOOP;
    if (fwd_s2_supported(g, dtype, aligned16)) return MP3D_PATH_FWD_S2;
    if (fwd_roll_supported(g, dtype, aligned16)) return MP3D_PATH_FWD_ROLL;
    return MP3D_PATH_FWD_PADDED;
}

int bwd_ex_path(const Geo& g, int dtype, int algo, bool aligned16 = true) {
    if (g.P == 0) return MP3D_PATH_NOOP;
    if (algo == MP3D_BWD_ATOMIC) return MP3D_PATH_BWD_ATOMIC;
    if (bwd_roll_supported(g, dtype, aligned16)) return MP3D_PATH_BWD_OVERLAP_ROLL;
    return MP3D_PATH_BWD_PADDED;
}

// Geometry of a padded / dilated backward call: the given output sizes must
// be the ones the window yields.
int bwd_ex_geo(Geo* g, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int od, int oh, int ow,
               int kd, int kh, int kw, int sd, int sh, int sw, int pd, int ph, int pw, int dd, int dh,
               int dw, int ceil_mode, int dtype, int algo) {
    int st = check_dims(N, C, D, H, W, g);
    if (!st) st = ex_geo(g, kd, kh, kw, sd, sh, sw, pd, ph, pw, dd, dh, dw, ceil_mode);
    if (!st && (g->OD != od || g->OH != oh || g->OW != ow)) st = MP3D_ERR_WINDOW;
    if (st) return st;
    if (elem_size(dtype) == 0) return MP3D_ERR_DTYPE;
    if (algo < MP3D_BWD_AUTO || algo > MP3D_BWD_ATOMIC) return MP3D_ERR_ALGO;
    return MP3D_OK;
}

}  // namespace

namespace mp3d {

int resident_ctas(const void* kern, int block, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    const auto key = std::make_tuple(dev, kern, block, smem);
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, block, smem) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();   // the launch reports its own errors
        n = 1;
    }
    cache.emplace(key, n);
    return n;
}

// Geometry of a backward call (maxpool3d_bwd's checks of sizes, window,
// dtype and algorithm).
int bwd_geo(Geo* g, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int od, int oh,
            int ow, int kd, int kh, int kw, int sd, int sh, int sw, int dtype, int algo) {
    int st = check_dims(N, C, D, H, W, g);
    if (st) return st;
    const bool all_zero = !kd && !kh && !kw && !sd && !sh && !sw;
    if (all_zero) {
        st = adaptive_geo(g, od, oh, ow);
    } else {
        st = fixed_geo(g, kd, kh, kw, sd, sh, sw);
        if (!st && (g->OD != od || g->OH != oh || g->OW != ow)) st = MP3D_ERR_WINDOW;
    }
    if (st) return st;
    if (elem_size(dtype) == 0) return MP3D_ERR_DTYPE;
    if (algo < MP3D_BWD_AUTO || algo > MP3D_BWD_ATOMIC) return MP3D_ERR_ALGO;
    return MP3D_OK;
}

// Buffer checks of a backward call (before any CUDA call).
int check_bwd_buffers(const void* grad_out, const int64_t* idx, const void* grad_in,
                      const void* workspace, size_t workspace_bytes, const Geo& g, int dtype,
                      int algo) {
    const int es = elem_size(dtype);
    const size_t need = workspace_needed(g, dtype, algo);
    if (g.P == 0) return MP3D_OK;
    if (!grad_out || !idx || !grad_in) return MP3D_ERR_NULLPTR;
    if (misaligned(grad_out, es) || misaligned(idx, 8) || misaligned(grad_in, es))
        return MP3D_ERR_ALIGN;
    const long long ng = g.P * g.ovol * es, ni = g.P * g.ovol * 8, nin = g.P * g.vol * es;
    if (overlaps(grad_in, nin, grad_out, ng) || overlaps(grad_in, nin, idx, ni))
        return MP3D_ERR_ALIAS;
    if (need > 0) {
        if (!workspace || workspace_bytes < need || misaligned(workspace, 16))
            return MP3D_ERR_WORKSPACE;
        if (overlaps(workspace, (long long)need, grad_in, nin) ||
            overlaps(workspace, (long long)need, grad_out, ng) ||
            overlaps(workspace, (long long)need, idx, ni))
            return MP3D_ERR_ALIAS;
    }
    return MP3D_OK;
}

}  // namespace mp3d

// ==================================================================== C ABI

extern "C" {

int maxpool3d_out_size(int64_t D, int64_t H, int64_t W, int kd, int kh, int kw, int sd, int sh,
                       int sw, int* od, int* oh, int* ow) {
    if (!od || !oh || !ow) return MP3D_ERR_NULLPTR;
    Geo g;
    int st = check_dims(1, 1, D, H, W, &g);
    if (!st) st = fixed_geo(&g, kd, kh, kw, sd, sh, sw);
    if (st) return st;
    *od = g.OD; *oh = g.OH; *ow = g.OW;
    return MP3D_OK;
}

int maxpool3d_ex_out_size(int64_t D, int64_t H, int64_t W, int kd, int kh, int kw, int sd, int sh,
                          int sw, int pd, int ph, int pw, int dd, int dh, int dw, int ceil_mode,
                          int* od, int* oh, int* ow) {
    if (!od || !oh || !ow) return MP3D_ERR_NULLPTR;
    Geo g;
    int st = check_dims(1, 1, D, H, W, &g);
    if (!st) st = ex_geo(&g, kd, kh, kw, sd, sh, sw, pd, ph, pw, dd, dh, dw, ceil_mode);
    if (st) return st;
    *od = g.OD; *oh = g.OH; *ow = g.OW;
    return MP3D_OK;
}

int maxpool3d_fwd_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int kd, int kh,
                       int kw, int sd, int sh, int sw, int dtype, int* path) {
    Geo g;
    int st = check_dims(N, C, D, H, W, &g);
    if (!st) st = fixed_geo(&g, kd, kh, kw, sd, sh, sw);
    if (!st && elem_size(dtype) == 0) st = MP3D_ERR_DTYPE;
    if (!st && path) *path = fwd_path(g, dtype);
    return st;
}

int adaptive_maxpool3d_fwd_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int od,
                                int oh, int ow, int dtype, int* path) {
    Geo g;
    int st = check_dims(N, C, D, H, W, &g);
    if (!st) st = adaptive_geo(&g, od, oh, ow);
    if (!st && elem_size(dtype) == 0) st = MP3D_ERR_DTYPE;
    if (!st && path) *path = fwd_path(g, dtype);
    return st;
}

int maxpool3d_bwd_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int od, int oh,
                       int ow, int kd, int kh, int kw, int sd, int sh, int sw, int dtype,
                       int algo, int* path) {
    Geo g;
    int st = bwd_geo(&g, N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, dtype, algo);
    if (!st && path) *path = bwd_path(g, dtype, algo);
    return st;
}

int maxpool3d_fwd(const void* x, void* y, int64_t* idx, int64_t N, int64_t C, int64_t D,
                  int64_t H, int64_t W, int kd, int kh, int kw, int sd, int sh, int sw,
                  int dtype, cudaStream_t stream) {
    Geo g;
    int st = check_dims(N, C, D, H, W, &g);
    if (!st) st = fixed_geo(&g, kd, kh, kw, sd, sh, sw);
    if (!st) st = check_fwd_buffers(x, y, idx, g, dtype);
    if (st) return st;
    return run_fwd(x, y, idx, g, dtype, stream);
}

int adaptive_maxpool3d_fwd(const void* x, void* y, int64_t* idx, int64_t N, int64_t C,
                           int64_t D, int64_t H, int64_t W, int od, int oh, int ow, int dtype,
                           cudaStream_t stream) {
    Geo g;
    int st = check_dims(N, C, D, H, W, &g);
    if (!st) st = adaptive_geo(&g, od, oh, ow);
    if (!st) st = check_fwd_buffers(x, y, idx, g, dtype);
    if (st) return st;
    return run_fwd(x, y, idx, g, dtype, stream);
}

size_t maxpool3d_bwd_workspace_bytes(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                                     int dtype, int algo) {
    Geo g;
    if (check_dims(N, C, D, H, W, &g)) return 0;
    if (elem_size(dtype) == 0 || algo < MP3D_BWD_AUTO || algo > MP3D_BWD_ATOMIC) return 0;
    return workspace_needed(g, dtype, algo);
}

int maxpool3d_bwd(const void* grad_out, const int64_t* idx, void* grad_in, int64_t N, int64_t C,
                  int64_t D, int64_t H, int64_t W, int od, int oh, int ow, int kd, int kh,
                  int kw, int sd, int sh, int sw, int dtype, int algo, void* workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
    Geo g;
    int st = bwd_geo(&g, N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, dtype, algo);
    if (!st) st = check_bwd_buffers(grad_out, idx, grad_in, workspace, workspace_bytes, g, dtype, algo);
    if (st) return st;
    return run_bwd(grad_out, idx, grad_in, workspace, g, dtype, algo, stream);
}

int maxpool3d_fwd_ex(const void* x, void* y, int64_t* idx, int64_t N, int64_t C, int64_t D,
                     int64_t H, int64_t W, int kd, int kh, int kw, int sd, int sh, int sw, int pd,
                     int ph, int pw, int dd, int dh, int dw, int ceil_mode, int dtype,
                     cudaStream_t stream) {
    Geo g;
    int st = check_dims(N, C, D, H, W, &g);
    if (!st) st = ex_geo(&g, kd, kh, kw, sd, sh, sw, pd, ph, pw, dd, dh, dw, ceil_mode);
    if (!st) st = check_fwd_buffers(x, y, idx, g, dtype);
    if (st) return st;
    if (ex_is_plain(g)) return run_fwd(x, y, idx, g, dtype, stream);
    const int path = ex_fwd_path(g, dtype, (uintptr_t)x % 16 == 0);
    log_path("fwd", path, g, dtype);
    if (path == MP3D_PATH_NOOP) return MP3D_OK;
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return MP3D_ERR_CUDA;
    const cudaError_t e = path == MP3D_PATH_FWD_S2     ? launch_fwd_s2(x, y, idx, g, dtype, sms, stream)
                          : path == MP3D_PATH_FWD_ROLL ? launch_fwd_roll(x, y, idx, g, dtype, sms, stream)
                                                       : launch_fwd_ex(x, y, idx, g, dtype, sms, stream);
    return e == cudaSuccess ? MP3D_OK : MP3D_ERR_CUDA;
}

int maxpool3d_fwd_ex_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int kd, int kh,
                          int kw, int sd, int sh, int sw, int pd, int ph, int pw, int dd, int dh,
                          int dw, int ceil_mode, int dtype, int* path) {
    Geo g;
    int st = check_dims(N, C, D, H, W, &g);
    if (!st) st = ex_geo(&g, kd, kh, kw, sd, sh, sw, pd, ph, pw, dd, dh, dw, ceil_mode);
    if (!st && elem_size(dtype) == 0) st = MP3D_ERR_DTYPE;
    if (!st && path)
        *path = ex_is_plain(g) ? fwd_path(g, dtype) : ex_fwd_path(g, dtype);
    return st;
}

int maxpool3d_bwd_ex(const void* grad_out, const int64_t* idx, void* grad_in, int64_t N, int64_t C,
                     int64_t D, int64_t H, int64_t W, int od, int oh, int ow, int kd, int kh,
                     int kw, int sd, int sh, int sw, int pd, int ph, int pw, int dd, int dh, int dw,
                     int ceil_mode, int dtype, int algo, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
    Geo g;
    int st = bwd_ex_geo(&g, N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, pd, ph, pw, dd, dh, dw,
                        ceil_mode, dtype, algo);
    if (!st) st = check_bwd_buffers(grad_out, idx, grad_in, workspace, workspace_bytes, g, dtype, algo);
    if (st) return st;
    if (ex_is_plain(g)) return run_bwd(grad_out, idx, grad_in, workspace, g, dtype, algo, stream);
    const int path = bwd_ex_path(g, dtype, algo, (uintptr_t)grad_in % 16 == 0);
    log_path("bwd", path, g, dtype);
    if (path == MP3D_PATH_NOOP) return MP3D_OK;
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return MP3D_ERR_CUDA;
    cudaError_t e;
    if (path == MP3D_PATH_BWD_ATOMIC)
        e = launch_bwd_atomic(grad_out, idx, grad_in, (float*)workspace, g, dtype, sms, stream);
    else if (path == MP3D_PATH_BWD_OVERLAP_ROLL)
        e = launch_bwd_roll(grad_out, idx, grad_in, g, dtype, sms, stream);
    else
        e = launch_bwd_ex_direct(grad_out, idx, grad_in, g, dtype, sms, stream);
    return e == cudaSuccess ? MP3D_OK : MP3D_ERR_CUDA;
}

int maxpool3d_bwd_ex_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int od, int oh,
                          int ow, int kd, int kh, int kw, int sd, int sh, int sw, int pd, int ph,
                          int pw, int dd, int dh, int dw, int ceil_mode, int dtype, int algo,
                          int* path) {
    Geo g;
    int st = bwd_ex_geo(&g, N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, pd, ph, pw, dd, dh, dw,
                        ceil_mode, dtype, algo);
    if (!st && path) {
        if (ex_is_plain(g)) *path = bwd_path(g, dtype, algo);
        else *path = bwd_ex_path(g, dtype, algo);
    }
    return st;
}

int maxpool3d_bwd_recompute(const void* x, const void* grad_out, void* grad_in, int64_t N,
                            int64_t C, int64_t D, int64_t H, int64_t W, int od, int oh, int ow,
                            int kd, int kh, int kw, int sd, int sh, int sw, int dtype,
                            cudaStream_t stream) {
    Geo g;
    int st = bwd_geo(&g, N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, dtype, MP3D_BWD_AUTO);
    if (st) return st;
    if (g.P == 0) return MP3D_OK;
    const int es = elem_size(dtype);
    if (!x || !grad_out || !grad_in) return MP3D_ERR_NULLPTR;
    if (misaligned(x, es) || misaligned(grad_out, es) || misaligned(grad_in, es)) return MP3D_ERR_ALIGN;
    const long long nx = g.P * g.vol * es, ng = g.P * g.ovol * es;
    if (overlaps(grad_in, nx, x, nx) || overlaps(grad_in, nx, grad_out, ng)) return MP3D_ERR_ALIAS;
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return MP3D_ERR_CUDA;
    int kind = 1;
    const cudaError_t e = launch_bwd_recompute(x, grad_out, grad_in, g, dtype, sms, stream, &kind);
    log_path("bwd", kind == 0 ? MP3D_PATH_BWD_RECOMPUTE_TILES : MP3D_PATH_BWD_RECOMPUTE, g, dtype);
    return e == cudaSuccess ? MP3D_OK : MP3D_ERR_CUDA;
}

int maxpool3d_bwd_recompute_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int od,
                                 int oh, int ow, int kd, int kh, int kw, int sd, int sh, int sw,
                                 int dtype, int* path) {
    Geo g;
    int st = bwd_geo(&g, N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, dtype, MP3D_BWD_AUTO);
    if (!st && path) {
        const int vec = 16 / elem_size(dtype);
        const bool tiles = !g.adaptive && g.kd == 2 && g.kh == 2 && g.kw == 2 && g.sd == 2 &&
                           g.sh == 2 && g.sw == 2 && g.D == 2 * g.OD && g.H == 2 * g.OH &&
                           g.W == 2 * g.OW && g.W % vec == 0;
        *path = g.P == 0 ? MP3D_PATH_NOOP : tiles ? MP3D_PATH_BWD_RECOMPUTE_TILES : MP3D_PATH_BWD_RECOMPUTE;
    }
    return st;
}

// Channels-last entry points: the checks of the NCDHW ones (same byte
// counts), then the channels-last kernels with the batch as the plane count.
static int run_fwd_ndhwc(const void* x, void* y, int64_t* idx, Geo g, int64_t C, int dtype,
                         cudaStream_t stream) {
    if (g.P == 0) return MP3D_OK;
    if (C > INT32_MAX) return MP3D_ERR_SHAPE;
    g.P /= C;                                   // planes -> batch
    log_path("fwd", MP3D_PATH_FWD_NDHWC, g, dtype);
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return MP3D_ERR_CUDA;
    return launch_fwd_ndhwc(x, y, idx, g, (int)C, dtype, sms, stream) == cudaSuccess ? MP3D_OK
                                                                                     : MP3D_ERR_CUDA;
}

int maxpool3d_fwd_ndhwc(const void* x, void* y, int64_t* idx, int64_t N, int64_t C, int64_t D,
                        int64_t H, int64_t W, int kd, int kh, int kw, int sd, int sh, int sw,
                        int dtype, cudaStream_t stream) {
    Geo g;
    int st = check_dims(N, C, D, H, W, &g);
    if (!st) st = fixed_geo(&g, kd, kh, kw, sd, sh, sw);
    if (!st) st = check_fwd_buffers(x, y, idx, g, dtype);
    if (st) return st;
    return run_fwd_ndhwc(x, y, idx, g, C, dtype, stream);
}

int adaptive_maxpool3d_fwd_ndhwc(const void* x, void* y, int64_t* idx, int64_t N, int64_t C,
                                 int64_t D, int64_t H, int64_t W, int od, int oh, int ow, int dtype,
                                 cudaStream_t stream) {
    Geo g;
    int st = check_dims(N, C, D, H, W, &g);
    if (!st) st = adaptive_geo(&g, od, oh, ow);
    if (!st) st = check_fwd_buffers(x, y, idx, g, dtype);
    if (st) return st;
    return run_fwd_ndhwc(x, y, idx, g, C, dtype, stream);
}

int maxpool3d_bwd_ndhwc(const void* grad_out, const int64_t* idx, void* grad_in, int64_t N,
                        int64_t C, int64_t D, int64_t H, int64_t W, int od, int oh, int ow, int kd,
                        int kh, int kw, int sd, int sh, int sw, int dtype, cudaStream_t stream) {
    Geo g;
    int st = bwd_geo(&g, N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, dtype, MP3D_BWD_AUTO);
    if (!st) st = check_bwd_buffers(grad_out, idx, grad_in, nullptr, 0, g, dtype, MP3D_BWD_AUTO);
    if (st) return st;
    if (g.P == 0) return MP3D_OK;
    if (C > INT32_MAX) return MP3D_ERR_SHAPE;
    g.P /= C;
    log_path("bwd", bwd_ndhwc_path(g, (int)C, dtype, (uintptr_t)grad_in % 16 == 0), g, dtype);
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return MP3D_ERR_CUDA;
    return launch_bwd_ndhwc(grad_out, idx, grad_in, g, (int)C, dtype, sms, stream) == cudaSuccess
               ? MP3D_OK : MP3D_ERR_CUDA;
}

int maxpool3d_bwd_ndhwc_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int od, int oh,
                             int ow, int kd, int kh, int kw, int sd, int sh, int sw, int dtype,
                             int* path) {
    Geo g;
    int st = bwd_geo(&g, N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, dtype, MP3D_BWD_AUTO);
    if (st) return st;
    if (g.P > 0 && C > INT32_MAX) return MP3D_ERR_SHAPE;
    if (g.P > 0) g.P /= C;
    if (path) *path = g.P == 0 ? MP3D_PATH_NOOP : bwd_ndhwc_path(g, (int)C, dtype, true);
    return MP3D_OK;
}

int mp3d_device_error_flags(unsigned int* flags, int clear) {
    if (!flags) return MP3D_ERR_NULLPTR;
    return read_device_error(flags, clear != 0) == cudaSuccess ? MP3D_OK : MP3D_ERR_CUDA;
}

int mp3d_set_pipeline_wait_limit(int polls) { return set_pipeline_wait_limit(polls); }

const char* mp3d_status_string(int status) {
    switch (status) {
    case MP3D_OK: return "ok";
    case MP3D_ERR_NULLPTR: return "a required pointer is NULL";
    case MP3D_ERR_SHAPE: return "invalid size (dimension < 1, N or C < 0, or a volume >= 2^31)";
    case MP3D_ERR_WINDOW: return "invalid window (kernel or stride < 1, kernel larger than the "
                                 "input, or output sizes that do not match the window)";
    case MP3D_ERR_DTYPE: return "unsupported dtype (f32, f16, bf16 only)";
    case MP3D_ERR_WORKSPACE: return "workspace missing, too small or not 16-byte aligned";
    case MP3D_ERR_CUDA: return "CUDA launch or device query failed";
    case MP3D_ERR_ALGO: return "unknown backward algorithm";
    case MP3D_ERR_ALIGN: return "pointer not aligned to its element size";
    case MP3D_ERR_ALIAS: return "an output buffer overlaps another buffer";
    case MP3D_ERR_SCRATCH: return "problem larger than the built-in scratch of maxpool3d_bwd_noalloc "
                                  "(8 Mi binary32 accumulators for f16/bf16)";
    default: return "unknown status";
    }
}

}  // extern "C"
