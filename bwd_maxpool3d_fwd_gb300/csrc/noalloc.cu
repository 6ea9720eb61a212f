// maxpool3d_bwd_noalloc: the atomic-form backward for callers that cannot
// allocate device memory while they run (for example a plugin inside an
// engine that owns all device memory, or a deployment with a fixed memory
// budget). Instead of a caller-provided workspace, the binary32
// accumulators live in a fixed array built into this library.
#include <mutex>

#include "internal.h"
#include "mp3d.h"

// 8 Mi binary32 accumulators (32 MiB). Every GPU that loads the library
// holds this array until the process exits. In host code the name below is
// only a host-side stand-in for the symbol, not a device address: the
// device address is looked up with cudaGetSymbolAddress (per device) and
// passed to the kernels.
static constexpr long long kNoallocScratchFloats = 8LL << 20;
static __device__ __align__(256) float mp3d_noalloc_scratch[kNoallocScratchFloats];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on
// the first call per device (with that device current) and cached.
int scratch_on_current_device(float** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MP3D_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, mp3d_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return MP3D_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return MP3D_OK;
}

bool ranges_overlap(const void* a, long long na, const void* b, long long nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return na > 0 && nb > 0 && pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

}  // namespace

extern "C" int maxpool3d_bwd_noalloc(const void* grad_out, const int64_t* idx, void* grad_in,
                                     int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                                     int od, int oh, int ow, int kd, int kh, int kw, int sd,
                                     int sh, int sw, int dtype, cudaStream_t stream) {
    // Shapes, window, dtype: checked exactly as maxpool3d_bwd checks them.
    int path = MP3D_PATH_NOOP;
    int st = maxpool3d_bwd_plan(N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, dtype,
                                MP3D_BWD_ATOMIC, &path);
    if (st != MP3D_OK) return st;
    if (path == MP3D_PATH_NOOP) return MP3D_OK;

    const int es = (dtype == MP3D_F32) ? 4 : 2;
    const long long P = N * C, vol = D * H * W, ovol = (long long)od * oh * ow;
    if (!grad_out || !idx || !grad_in) return MP3D_ERR_NULLPTR;
    if ((uintptr_t)grad_out % es || (uintptr_t)idx % 8 || (uintptr_t)grad_in % es)
        return MP3D_ERR_ALIGN;
    if (ranges_overlap(grad_in, P * vol * es, grad_out, P * ovol * es) ||
        ranges_overlap(grad_in, P * vol * es, idx, P * ovol * 8))
        return MP3D_ERR_ALIAS;

    float* scratch = nullptr;
    if (dtype != MP3D_F32) {
        if (P * vol > kNoallocScratchFloats) return MP3D_ERR_SCRATCH;
        st = scratch_on_current_device(&scratch);
        if (st != MP3D_OK) return st;
    }

    mp3d::Geo g{};
    g.P = P;
    g.D = (int)D; g.H = (int)H; g.W = (int)W;
    g.OD = od; g.OH = oh; g.OW = ow;
    g.kd = kd; g.kh = kh; g.kw = kw;
    g.sd = sd; g.sh = sh; g.sw = sw;
    g.adaptive = (kd == 0) ? 1 : 0;
    g.vol = (int)vol;
    g.ovol = (int)ovol;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MP3D_ERR_CUDA;
    // The zero-fill kernel of the atomic path clears the accumulators this
    // call uses before the scatter, so earlier calls leave no trace.
    const cudaError_t e = mp3d::launch_bwd_atomic(grad_out, idx, grad_in, scratch, g, dtype, sms,
                                                  stream);
    return e == cudaSuccess ? MP3D_OK : MP3D_ERR_CUDA;
}
