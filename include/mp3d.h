/*
 * mp3d.h: C ABI of libmp3d.so, 3-D max pooling over NCDHW tensors on
 * NVIDIA GB300 (sm_103a): forward with argmax indices (fixed and adaptive
 * windows) and the backward that routes each output gradient to its argmax
 * input.
 *
 * Sources (web pages on the subject):
 *  [MPF]  teenygrad API docs, "Struct Maxpool3dForward": a 3-D max-pooling
 *         forward pass; Constraints: no padding, OD = (D - KD)/STRIDE_D + 1,
 *         likewise OH, OW. Its launch-argument tuple (input pointer, output
 *         pointer, eight i32) is the model for passing plain pointers and
 *         integer sizes here.
 *  [AMPB] FlagGems-Experimental PR #308, "Add adaptive_max_pool3d_backward
 *         Moore Threads specialized operator", Summary: the backward
 *         scatters each output window's gradient back to its argmax input;
 *         when every axis divides evenly the windows tile the input and one
 *         gather launch suffices (no zero pass, no atomics); otherwise
 *         windows overlap and contributions to one input accumulate (the
 *         page uses a zero fill and an atomic scatter, kept here as an
 *         ablation).
 *
 * Conventions shared by every entry point
 *  - Layout: every tensor is dense, contiguous NCDHW. A "plane" is one
 *    (n, c) slice of D*H*W elements. Outputs are dense [N, C, OD, OH, OW].
 *  - Indices: int64 flat offsets d*H*W + h*W + w inside the element's own
 *    plane (not global offsets).
 *  - Ties: the first occurrence in (d, h, w) row-major order wins; +0 and
 *    -0 compare equal; a NaN beats every number and the first NaN wins.
 *    The output value is a bit copy of the winning input element.
 *  - Ownership: the caller allocates and owns every buffer, including the
 *    workspace. The library allocates nothing on the device, frees
 *    nothing, and never synchronises.
 *  - Pointers: device pointers (or managed memory), aligned to their
 *    element size. Inputs and outputs must not overlap.
 *  - Asynchrony: work is enqueued on `stream` (0 = the legacy default
 *    stream); the call returns after the launch.
 *  - Errors: argument errors return a nonzero status before any CUDA call,
 *    with nothing written. A launch failure returns MP3D_ERR_CUDA.
 *  - Empty input: N*C == 0 is a no-op returning MP3D_OK (other arguments are
 *    still checked).
 *  - Limits: D*H*W and OD*OH*OW must each be below 2^31.
 *  - Types: f32, f16, bf16 only; any other code returns MP3D_ERR_DTYPE
 *    (there is no fallback).
 */
#ifndef MP3D_H
#define MP3D_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { MP3D_F32 = 0, MP3D_F16 = 1, MP3D_BF16 = 2 } mp3d_dtype;

/* Backward algorithm. AUTO and GATHER both pick a deterministic form (a
 * gather, or the ordered rolling scatter, from the shape) whose sums are
 * bit-identical to the ordered definition; ATOMIC runs the
 * ablation of [AMPB]'s non-divisible path: zero fill, atomicAdd scatter in
 * binary32 and, for f16/bf16, a final rounding pass. */
typedef enum { MP3D_BWD_AUTO = 0, MP3D_BWD_GATHER = 1, MP3D_BWD_ATOMIC = 2 } mp3d_bwd_algo;

typedef enum {
    MP3D_OK = 0,
    MP3D_ERR_NULLPTR = 1,    /* a required pointer is NULL                 */
    MP3D_ERR_SHAPE = 2,      /* a size < 1 (or N, C < 0), or a volume >= 2^31 */
    MP3D_ERR_WINDOW = 3,     /* kernel/stride < 1, kernel > input, or output
                                sizes that do not match the window          */
    MP3D_ERR_DTYPE = 4,      /* dtype not in mp3d_dtype                     */
    MP3D_ERR_WORKSPACE = 5,  /* workspace missing or too small              */
    MP3D_ERR_CUDA = 6,       /* a CUDA launch or query failed               */
    MP3D_ERR_ALGO = 7,       /* algo not in mp3d_bwd_algo                   */
    MP3D_ERR_ALIGN = 8,      /* a pointer not aligned to its element size   */
    MP3D_ERR_ALIAS = 9,      /* an output overlaps an input or another output */
    MP3D_ERR_SCRATCH = 10    /* too large for maxpool3d_bwd_noalloc's built-in scratch */
} mp3d_status;

/* Kernel paths reported by the *_plan queries (for logging and tests). */
typedef enum {
    MP3D_PATH_NOOP = 0,              /* N*C == 0                              */
    MP3D_PATH_FWD_GENERIC = 1,       /* one thread per output, any window     */
    MP3D_PATH_FWD_S2 = 2,            /* stride-2 register-column kernel       */
    MP3D_PATH_FWD_GLOBAL = 3,        /* one window per plane (global pool)    */
    MP3D_PATH_FWD_SLAB = 4,          /* window-depth slab staged in shared memory */
    MP3D_PATH_FWD_PADDED = 5,        /* padded / dilated windows, thread per output */
    MP3D_PATH_FWD_NDHWC = 6,         /* channels-last layout                  */
    MP3D_PATH_BWD_DISJOINT = 10,     /* single-pass gather, disjoint windows  */
    MP3D_PATH_BWD_OVERLAP_TILE = 11, /* overlapping gather, staged tile + owner sums */
    MP3D_PATH_BWD_OVERLAP_DIRECT = 12, /* overlapping gather, direct reads    */
    MP3D_PATH_BWD_ATOMIC = 13,       /* zero fill + atomic scatter ablation   */
    MP3D_PATH_BWD_OVERLAP_ROLL = 14, /* overlapping, ordered scatter into a
                                        rolling ring of shared depth slices  */
    MP3D_PATH_BWD_PADDED = 15,       /* padded / dilated windows, direct gather */
    MP3D_PATH_BWD_RECOMPUTE_TILES = 16, /* no stored index, 2x2x2 tiling, fused */
    MP3D_PATH_BWD_RECOMPUTE = 17,    /* no stored index, direct form          */
    MP3D_PATH_BWD_NDHWC = 18,        /* channels-last layout                  */
    MP3D_PATH_FWD_ROLL = 19,         /* 16-bit, depth slices streamed in order,
                                        windows as unsigned maxima of order
                                        words                                 */
    MP3D_PATH_BWD_NDHWC_ROLL = 20    /* channels-last, ordered scatter into a
                                        rolling ring of shared depth slices  */
} mp3d_path;

/*
 * Output sizes of the fixed-window forward [MPF] (Constraints: no padding,
 * OD = (D - KD)/STRIDE_D + 1, likewise OH and OW): the sizes maxpool3d_fwd
 * writes and maxpool3d_bwd expects for this input and window. Checks the
 * arguments as maxpool3d_fwd does (sizes >= 1 with D*H*W below 2^31;
 * 1 <= k <= input size and s >= 1 on every axis). On MP3D_OK stores the
 * sizes in *od, *oh, *ow; otherwise returns MP3D_ERR_SHAPE or
 * MP3D_ERR_WINDOW (MP3D_ERR_NULLPTR for a NULL result pointer) and stores
 * nothing. Host only: no CUDA call.
 */
int maxpool3d_out_size(int64_t D, int64_t H, int64_t W, int kd, int kh, int kw,
                       int sd, int sh, int sw, int* od, int* oh, int* ow);

/*
 * Fixed-window forward [MPF]. x: [N, C, D, H, W]; y: [N, C, OD, OH, OW] of
 * the same type; idx: int64 [N, C, OD, OH, OW], with
 * OD = (D - kd)/sd + 1, OH = (H - kh)/sh + 1, OW = (W - kw)/sw + 1
 * (no padding). y[n,c,od,oh,ow] is the maximum of x over
 * d in [od*sd, od*sd + kd), h in [oh*sh, oh*sh + kh), w in [ow*sw, ow*sw + kw).
 * Requires 1 <= k <= input size and s >= 1 on every axis.
 * idx may be NULL: the values-only forward ([MPF]'s launch tuple has an
 * input and an output pointer and no index output). y is written exactly as
 * with an index buffer and no index is stored, which saves the 8-byte
 * index of every output (a backward then needs an index from another call).
 */
int maxpool3d_fwd(const void* x, void* y, int64_t* idx,
                  int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                  int kd, int kh, int kw, int sd, int sh, int sw,
                  int dtype, cudaStream_t stream);

/*
 * Adaptive-window forward (the forward of [AMPB]'s operator). Output size
 * (od, oh, ow) is given, each >= 1 (an output larger than the input is
 * accepted). Window i along an axis of input size I and output size O is
 * [floor(i*I/O), ceil((i+1)*I/O)). Buffers as for maxpool3d_fwd (idx may
 * be NULL: values only).
 */
int adaptive_maxpool3d_fwd(const void* x, void* y, int64_t* idx,
                           int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                           int od, int oh, int ow, int dtype, cudaStream_t stream);

/*
 * Backward [AMPB]: grad_in[n, c, j] = sum of grad_out[n, c, o] over the
 * outputs o of that plane whose idx[n, c, o] == j, summed in ascending
 * (od, oh, ow) order in binary32 (first term as the initial value) and
 * rounded once to the type; +0 where no output selects j. Every element of
 * grad_in is written.
 *
 * grad_out, idx: [N, C, od, oh, ow]; grad_in: [N, C, D, H, W].
 * Window: either fixed (kd..sw all >= 1, and (od, oh, ow) must equal the
 * fixed output sizes) or adaptive (kd..sw all 0; windows derived from
 * (D, H, W) -> (od, oh, ow)).
 * Precondition: idx comes from the matching forward (each index lies in its
 * own window). The gather paths only look at windows that cover an input,
 * so an index outside its window is ignored; the ATOMIC path drops indices
 * outside [0, D*H*W).
 * algo: mp3d_bwd_algo. ATOMIC with f16/bf16 needs a workspace of
 * maxpool3d_bwd_workspace_bytes(...) bytes (binary32 accumulators, 16-byte
 * aligned); every other case needs none (workspace may be NULL).
 */
int maxpool3d_bwd(const void* grad_out, const int64_t* idx, void* grad_in,
                  int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                  int od, int oh, int ow,
                  int kd, int kh, int kw, int sd, int sh, int sw,
                  int dtype, int algo, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream);

/* Workspace bytes maxpool3d_bwd needs: 4*N*C*D*H*W for ATOMIC with f16 or
 * bf16, else 0. Returns 0 for invalid arguments as well. */
size_t maxpool3d_bwd_workspace_bytes(int64_t N, int64_t C, int64_t D, int64_t H,
                                     int64_t W, int dtype, int algo);

/* Dispatch queries: validate exactly like the matching entry point, make
 * no CUDA call, and store the mp3d_path that the call would launch in
 * *path. Return the status the call would return for its arguments. */
int maxpool3d_fwd_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                       int kd, int kh, int kw, int sd, int sh, int sw,
                       int dtype, int* path);
int adaptive_maxpool3d_fwd_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                                int od, int oh, int ow, int dtype, int* path);
int maxpool3d_bwd_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                       int od, int oh, int ow,
                       int kd, int kh, int kw, int sd, int sh, int sw,
                       int dtype, int algo, int* path);

/*
 * Channels-last (NDHWC) layout: x [N, D, H, W, C], y and idx
 * [N, OD, OH, OW, C], grad_out like y, grad_in like x, all dense. Windows,
 * ties, NaN rule, index form (the spatial offset d*H*W + h*W + w of the
 * winner inside its own (n, c) volume) and the backward's order are those
 * of maxpool3d_fwd / adaptive_maxpool3d_fwd / maxpool3d_bwd: the results
 * are theirs with the channel axis moved last. Arguments and checks as for
 * those entry points (idx may be NULL in the forwards); the backward takes
 * no algorithm or workspace. Channel counts that are a
 * multiple of 16 bytes' worth of elements, on 16-byte aligned buffers, use
 * 16-byte accesses across channels; others take element accesses.
 */
int maxpool3d_fwd_ndhwc(const void* x, void* y, int64_t* idx,
                        int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                        int kd, int kh, int kw, int sd, int sh, int sw,
                        int dtype, cudaStream_t stream);
int adaptive_maxpool3d_fwd_ndhwc(const void* x, void* y, int64_t* idx,
                                 int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                                 int od, int oh, int ow, int dtype, cudaStream_t stream);
int maxpool3d_bwd_ndhwc(const void* grad_out, const int64_t* idx, void* grad_in,
                        int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                        int od, int oh, int ow,
                        int kd, int kh, int kw, int sd, int sh, int sw,
                        int dtype, cudaStream_t stream);
/* The kernel maxpool3d_bwd_ndhwc takes for these sizes with 16-byte
 * aligned buffers: MP3D_PATH_BWD_NDHWC_ROLL (adaptive windows, or fixed
 * windows overlapping along some axis, with at most two over any input per
 * axis and C * sizeof(element) a multiple of 16 bytes) or
 * MP3D_PATH_BWD_NDHWC (the rest: direct writes for 2x2x2 windows that tile
 * the input, gathers otherwise). Arguments as for maxpool3d_bwd_ndhwc;
 * *path is written on success. */
int maxpool3d_bwd_ndhwc_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                             int od, int oh, int ow,
                             int kd, int kh, int kw, int sd, int sh, int sw,
                             int dtype, int* path);

/*
 * Backward without stored indices [AMPB]: the same grad_in as
 * maxpool3d_bwd(grad_out, idx, ...) with idx the indices maxpool3d_fwd (or
 * adaptive_maxpool3d_fwd) would store for x, bit for bit: each window's
 * argmax is recomputed from x with the forward's rule. For callers that
 * keep the input but not the int64 indices (8 bytes per output). x:
 * [N, C, D, H, W] as given to the forward; grad_out [N, C, od, oh, ow];
 * grad_in like x, every element written. Window arguments as for
 * maxpool3d_bwd (kd..sw all 0: adaptive). No workspace.
 */
int maxpool3d_bwd_recompute(const void* x, const void* grad_out, void* grad_in,
                            int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                            int od, int oh, int ow,
                            int kd, int kh, int kw, int sd, int sh, int sw,
                            int dtype, cudaStream_t stream);
int maxpool3d_bwd_recompute_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                                 int od, int oh, int ow,
                                 int kd, int kh, int kw, int sd, int sh, int sw,
                                 int dtype, int* path);

/*
 * Padding, dilation and ceil-mode output sizes: the fixed-window forward
 * and backward beyond [MPF]'s "no padding" constraint, with the usual
 * max_pool3d definition (the pages fix only the unpadded case). Along each
 * axis (input I, kernel k, stride s, padding p on both sides, dilation dl):
 *  - the window of output o takes the positions o*s - p + j*dl, j < k, that
 *    lie inside [0, I) (padding is never chosen);
 *  - O = floor((I + 2p - dl*(k-1) - 1) / s) + 1, or with ceil in place of
 *    floor when ceil_mode = 1, where a last window starting at or past
 *    I + p is dropped;
 *  - requires k, s, dl >= 1, 0 <= 2p <= k, O >= 1, ceil_mode 0 or 1, and
 *    every window holding at least one input position (dilation with
 *    padding can leave a window empty): else MP3D_ERR_WINDOW.
 * Ties, NaN, index form and the backward's summation order are those of
 * maxpool3d_fwd / maxpool3d_bwd. Without padding or dilation, and with the
 * output size the unpadded formula gives, the calls take the same paths as
 * maxpool3d_fwd / maxpool3d_bwd. idx may be NULL in the forward (values
 * only). The backward's (od, oh, ow) must equal the forward's output sizes;
 * algo and workspace as for maxpool3d_bwd.
 */
int maxpool3d_fwd_ex(const void* x, void* y, int64_t* idx,
                     int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                     int kd, int kh, int kw, int sd, int sh, int sw,
                     int pd, int ph, int pw, int dd, int dh, int dw, int ceil_mode,
                     int dtype, cudaStream_t stream);
int maxpool3d_bwd_ex(const void* grad_out, const int64_t* idx, void* grad_in,
                     int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                     int od, int oh, int ow,
                     int kd, int kh, int kw, int sd, int sh, int sw,
                     int pd, int ph, int pw, int dd, int dh, int dw, int ceil_mode,
                     int dtype, int algo, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream);
/* Output sizes of maxpool3d_fwd_ex (the rule above), with its checks: on
 * MP3D_OK stores them in *od, *oh, *ow; an invalid geometry (including one
 * with a window that holds no input position) returns MP3D_ERR_WINDOW, bad
 * sizes MP3D_ERR_SHAPE, and nothing is stored. Host only: no CUDA call. */
int maxpool3d_ex_out_size(int64_t D, int64_t H, int64_t W,
                          int kd, int kh, int kw, int sd, int sh, int sw,
                          int pd, int ph, int pw, int dd, int dh, int dw, int ceil_mode,
                          int* od, int* oh, int* ow);
/* Path the padded calls take (mp3d_path), with the same checks. */
int maxpool3d_fwd_ex_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                          int kd, int kh, int kw, int sd, int sh, int sw,
                          int pd, int ph, int pw, int dd, int dh, int dw, int ceil_mode,
                          int dtype, int* path);
int maxpool3d_bwd_ex_plan(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                          int od, int oh, int ow, int kd, int kh, int kw, int sd, int sh, int sw,
                          int pd, int ph, int pw, int dd, int dh, int dw, int ceil_mode,
                          int dtype, int algo, int* path);

/*
 * Backward without any device allocation (atomic form). The pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory when they run, such as a plugin inside an engine
 * that owns all device memory and forbids cudaMalloc while executing, or a
 * deployment with a fixed memory budget. Those callers cannot provide the
 * binary32 workspace that maxpool3d_bwd needs for algo ATOMIC with f16/bf16.
 *
 * Computes what maxpool3d_bwd computes with algo = MP3D_BWD_ATOMIC (zero
 * fill, binary32 atomicAdd scatter, one rounding for f16/bf16), but keeps
 * the binary32 accumulators in an array built into the library: 8 Mi
 * floats (32 MiB), held on every GPU that loads the library until the
 * process exits. Same arguments as maxpool3d_bwd minus algo and workspace.
 *  - f16/bf16: N*C*D*H*W must be at most 8,388,608 (8 Mi); larger problems
 *    return MP3D_ERR_SCRATCH before any launch. f32 accumulates in grad_in
 *    directly, uses no scratch and has no such limit.
 *  - The first call on each device looks up the array's device address
 *    (with that device current) and caches it for the life of the
 *    process; make that first call before any stream capture. The cached
 *    address belongs to the device's primary context as it was at that
 *    first call: do not use this entry point after cudaDeviceReset on that
 *    device, or from a context created with the driver API.
 *  - Every call on a device shares the one array. Each call clears the part
 *    it uses before accumulating, so calls in sequence are independent, but
 *    calls that can overlap on the GPU (different streams without ordering,
 *    or several host threads) race on the array and give wrong results.
 *  - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *    call.
 */
int maxpool3d_bwd_noalloc(const void* grad_out, const int64_t* idx, void* grad_in,
                          int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                          int od, int oh, int ow,
                          int kd, int kh, int kw, int sd, int sh, int sw,
                          int dtype, cudaStream_t stream);

/* Error flags raised on the device by a kernel whose bounded wait for an
 * asynchronous copy gave up (bit 0: the copy pipeline of a forward kernel,
 * the stride-2 one or the depth walk, timed out; that call's outputs are
 * then incomplete and must not be used). Not expected in normal operation. Reads the current device's flags into *flags (clearing
 * them if clear != 0); this call waits for the device to finish prior work.
 * No counterpart on the pages: it exists because the library's kernels
 * never trap or spin without limit. */
int mp3d_device_error_flags(unsigned int* flags, int clear);

/* Sets how many times the forward kernels' copy pipelines poll a pending
 * copy before their wait gives up (bit 0 of mp3d_device_error_flags), for
 * launches made after the call, process-wide; returns the previous value.
 * A negative value restores the default (2^22 polls). Only for tests of the
 * give-up path: with 0 every pipeline wait gives up at once, the kernels
 * still let their copies in flight land before they exit (those waits keep
 * the default bound), and their outputs are incomplete. No counterpart on
 * the pages. */
int mp3d_set_pipeline_wait_limit(int polls);

/* Static description of a status code (never NULL). */
const char* mp3d_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MP3D_H */
