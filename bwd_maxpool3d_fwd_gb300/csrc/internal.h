// Launchers shared between the C-ABI layer (api.cu) and the kernel files.
// Every launcher enqueues on `stream`, returns the cudaError_t of the launch
// and never synchronises.
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

#include "common.cuh"

namespace mp3d {

// CTAs of `block` threads with `smem` bytes of dynamic shared memory that one
// SM of the current device keeps resident for kernel `kern` (api.cu; the
// occupancy query is made once per device and kernel; 1 if it fails).
int resident_ctas(const void* kern, int block, size_t smem);

// Blocks of 256 threads for a grid-stride loop over `work` threads: at most
// one wave of the CTAs that kern keeps resident on each SM. Not a general
// rule (the warp-per-plane global-window kernels run fastest with a CTA per
// eight planes and no stride, kGlobalCtasPerSm below), so each launch takes
// the grid measured best for it.
template <typename K>
inline int stride_grid(K kern, long long work, int sms) {
    long long b = (work + 255) / 256;
    const long long cap = (long long)sms * resident_ctas(reinterpret_cast<const void*>(kern), 256, 0);
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

// Grid cap of the warp-per-plane global-window kernels (k_fwd_global,
// k_bwd_global), in 256-thread CTAs per SM: high enough that each warp
// takes one plane (a CTA starts as another ends, so the planes' first loads
// overlap other planes' work), where a stride of eight CTAs per SM made each
// warp's planes wait on their loads one after another (on the
// 64x512x8x14x14 fp32 global pool: forward 45.1 -> 43.0 us, backward
// 32.8 -> 30.7 us); a grid-stride loop only for more planes than that.
constexpr int kGlobalCtasPerSm = 4096;

// Argument checks of a backward call (api.cu), before any CUDA call:
// sizes, window, dtype and algorithm into *g; then the buffers (NULL,
// alignment, overlap, and the workspace when algo needs one).
int bwd_geo(Geo* g, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int od, int oh,
            int ow, int kd, int kh, int kw, int sd, int sh, int sw, int dtype, int algo);
int check_bwd_buffers(const void* grad_out, const int64_t* idx, const void* grad_in,
                      const void* workspace, size_t workspace_bytes, const Geo& g, int dtype,
                      int algo);

// Forward paths (fwd.cu).
cudaError_t launch_fwd_generic(const void* x, void* y, int64_t* idx, const Geo& g,
                               int dtype, int sms, cudaStream_t s);
cudaError_t launch_fwd_global(const void* x, void* y, int64_t* idx, const Geo& g,
                              int dtype, int sms, cudaStream_t s);
cudaError_t launch_fwd_s2(const void* x, void* y, int64_t* idx, const Geo& g,
                          int dtype, int sms, cudaStream_t s);
cudaError_t launch_fwd_slab(const void* x, void* y, int64_t* idx, const Geo& g,
                            int dtype, int sms, cudaStream_t s);
// Fixed windows with padding and dilation (g.pd..g.dw): one thread per output.
cudaError_t launch_fwd_ex(const void* x, void* y, int64_t* idx, const Geo& g, int dtype, int sms,
                          cudaStream_t s);
// Whether a window-depth slab of this geometry fits the slab kernel's shared memory.
bool fwd_slab_supported(const Geo& g, int dtype);
// Whether the stride-2 kernel handles this geometry and type (it needs the
// input on a 16-byte boundary; plan queries assume an aligned buffer).
bool fwd_s2_supported(const Geo& g, int dtype, bool aligned16);
// 16-bit types, walking the depth slices of a plane in order (fwd_roll.cu):
// at most two windows over any slice along d, no padding or dilation, small
// planes of outputs, and the input on a 16-byte boundary.
bool fwd_roll_supported(const Geo& g, int dtype, bool aligned16);
cudaError_t launch_fwd_roll(const void* x, void* y, int64_t* idx, const Geo& g, int dtype, int sms,
                            cudaStream_t s);

// Channels-last layout (ndhwc.cu): g.P is the batch N, C the channel count.
cudaError_t launch_fwd_ndhwc(const void* x, void* y, int64_t* idx, const Geo& g, int C, int dtype,
                             int sms, cudaStream_t s);
cudaError_t launch_bwd_ndhwc(const void* go, const int64_t* idx, void* gi, const Geo& g, int C,
                             int dtype, int sms, cudaStream_t s);
// The channels-last backward's kernel (MP3D_PATH_BWD_NDHWC_ROLL or
// MP3D_PATH_BWD_NDHWC); aligned16: grad_in starts on a 16-byte boundary.
int bwd_ndhwc_path(const Geo& g, int C, int dtype, bool aligned16);
// The rolling channels-last backward (ndhwc_roll.cu): windows with at most
// two over any input per axis, C a multiple of its channel group, grad_in
// 16-byte aligned.
bool bwd_ndhwc_roll_supported(const Geo& g, int C, int dtype);
cudaError_t launch_bwd_ndhwc_roll(const void* go, const int64_t* idx, void* gi, const Geo& g, int C,
                                  int dtype, cudaStream_t s);

// Polls the main pipeline waits of the forward kernels make before giving
// up (fwd.cu; kWaitLimit unless a test set another value), and its setter
// (a negative value restores kWaitLimit; returns the previous value).
int pipeline_wait_limit();
int set_pipeline_wait_limit(int polls);

// Error flags set by kernels whose bounded waits gave up (fwd.cu, with the
// flag of fwd_roll.cu folded in).
cudaError_t read_device_error(unsigned int* flags, bool clear);
cudaError_t read_roll_fwd_error(unsigned int* flags, bool clear);

// Backward paths (bwd.cu). For the disjoint gather, g.kd..g.sw hold the
// fixed window (adaptive divisible shapes are passed as kernel = stride =
// input / output).
cudaError_t launch_bwd_disjoint(const void* go, const int64_t* idx, void* gi,
                                const Geo& g, int dtype, int sms, cudaStream_t s);
cudaError_t launch_bwd_overlap_direct(const void* go, const int64_t* idx, void* gi,
                                      const Geo& g, int dtype, int sms, cudaStream_t s);
cudaError_t launch_bwd_overlap_tile(const void* go, const int64_t* idx, void* gi,
                                    const Geo& g, int dtype, int sms, cudaStream_t s);
// Whether the tiled owner gather handles this geometry (its staged windows fit
// in shared memory).
bool bwd_tile_supported(const Geo& g);
// Ordered scatter into a rolling ring of shared depth slices (bwd_roll.cu):
// at most two windows cover any position along each axis, the ring fits in
// shared memory, and grad_in starts on a 16-byte boundary.
bool bwd_roll_supported(const Geo& g, int dtype, bool aligned16);
cudaError_t launch_bwd_roll(const void* go, const int64_t* idx, void* gi, const Geo& g,
                            int dtype, int sms, cudaStream_t s);
// Fixed windows with padding and dilation: direct gather in ascending order.
cudaError_t launch_bwd_ex_direct(const void* go, const int64_t* idx, void* gi, const Geo& g,
                                 int dtype, int sms, cudaStream_t s);
// Backward without stored indices (argmax recomputed from x). *kind is set
// to 0 for the fused 2x2x2 tiling kernel, 1 for the direct form.
cudaError_t launch_bwd_recompute(const void* x, const void* go, void* gi, const Geo& g, int dtype,
                                 int sms, cudaStream_t s, int* kind);
cudaError_t launch_bwd_atomic(const void* go, const int64_t* idx, void* gi, float* ws,
                              const Geo& g, int dtype, int sms, cudaStream_t s);

}  // namespace mp3d
