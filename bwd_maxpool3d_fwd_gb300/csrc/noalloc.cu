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
// the first call per device (with that device current) and cached for the
// life of the process. The cache is keyed by device ordinal: after
// cudaDeviceReset, or under a context other than the device's primary one,
// the cached address no longer names the array (documented in mp3d.h).
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

}  // namespace

extern "C" int maxpool3d_bwd_noalloc(const void* grad_out, const int64_t* idx, void* grad_in,
                                     int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                                     int od, int oh, int ow, int kd, int kh, int kw, int sd,
                                     int sh, int sw, int dtype, cudaStream_t stream) {
    // Sizes, window, dtype and buffers: maxpool3d_bwd's own checks, made
    // before any CUDA call (the workspace is checked below, once its
    // address is known).
    mp3d::Geo g;
    int st = mp3d::bwd_geo(&g, N, C, D, H, W, od, oh, ow, kd, kh, kw, sd, sh, sw, dtype,
                           MP3D_BWD_ATOMIC);
    if (st == MP3D_OK)
        st = mp3d::check_bwd_buffers(grad_out, idx, grad_in, nullptr, 0, g, dtype, MP3D_BWD_AUTO);
    if (st != MP3D_OK) return st;
    if (g.P == 0) return MP3D_OK;

    float* scratch = nullptr;
    if (dtype != MP3D_F32) {
        if (g.P * (long long)g.vol > kNoallocScratchFloats) return MP3D_ERR_SCRATCH;
        st = scratch_on_current_device(&scratch);
        if (st != MP3D_OK) return st;
        // the array as the atomic form's workspace: size, alignment, overlap
        st = mp3d::check_bwd_buffers(grad_out, idx, grad_in, scratch,
                                     (size_t)kNoallocScratchFloats * sizeof(float), g, dtype,
                                     MP3D_BWD_ATOMIC);
        if (st != MP3D_OK) return st;
    }

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
