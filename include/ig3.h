/*
 * ig3 -- fused 3x3(x3) convolutions for NVIDIA GB300 (sm_103a): stride-1 valid conv3d
 * and depthwise 3x3 -> pointwise 1x1 conv2d with fused epilogues, plus zero-padded and
 * stride-2 conv3d (conv3d_fused_pad, conv3d_fused_ex) and K x K depthwise stages
 * (dwsep_conv2d_ex).
 *
 * A plain C ABI: raw pointers, sizes and a CUDA stream passed as `void*`
 * (a cudaStream_t; NULL = the legacy default stream).  No C++ or framework
 * types cross this boundary.
 *
 * Sources (web pages, cited by title and passage):
 *   [P47] "Kimi-K2.6__l2_p47": Conv3d(32->64, k=3, valid) followed by Mish and Tanh.
 *   [P8]  "Kimi-K2.6__l2_p8":  Conv3d(8->16, k=3, valid), divide by 2,
 *         MaxPool3d(2), AdaptiveAvgPool3d(1), + bias[c], sum over channels.
 *   [P86] "Kimi-K2.6__l1_p86": depthwise 3x3 conv (stride 1, pad 1) followed by
 *         a pointwise 1x1 conv, with the depthwise result kept on chip.
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer to dense, row-major float32 data
 *     owned by the caller, on the device that is current for the calling thread.
 *     The library never frees, keeps or allocates device memory.
 *   - Calls are asynchronous on `stream`.  Argument errors are detected on the
 *     host before anything is launched and returned as a negative status; the
 *     library never aborts the process.  A launch failure returns IG3_ERR_CUDA.
 *   - Outputs must not alias inputs or the workspace.
 *   - Kernels never spin forever: every wait inside a kernel is bounded in time
 *     (default 1 s, see ig3_set_wait_timeout_ns).  A wait that runs out makes
 *     the kernel stop early and records IG3_ERR_TIMEOUT in a per-device status
 *     word, which ig3_last_device_status() reports.
 *   - The message of the last failed call on the calling thread is available
 *     from ig3_last_error().
 */
#ifndef IG3_H
#define IG3_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  IG3_OK = 0,
  IG3_ERR_INVALID_ARG = -1,  /* NULL pointer, non-positive size, size overflow, bad enum */
  IG3_ERR_UNSUPPORTED = -2,  /* valid arguments outside what this library computes       */
  IG3_ERR_CUDA = -3,         /* a CUDA runtime call or a kernel launch failed             */
  IG3_ERR_TIMEOUT = -4,      /* a bounded wait inside a kernel ran out                    */
  IG3_ERR_WORKSPACE = -5     /* workspace missing or smaller than the size query returns  */
} ig3_status;

typedef enum {
  IG3_EPI_NONE = 0,        /* y = conv3d(x, w) + b                                      */
  IG3_EPI_TANH_MISH = 1,   /* y = tanh(mish(conv3d(x, w) + b))                  [P47]   */
  IG3_EPI_POOL_REDUCE = 2  /* y[n] = sum_c(mean(maxpool((conv + b) / divisor)) + bias2[c]) [P8] */
} ig3_epilogue;

typedef enum {
  IG3_PATH_AUTO = 0,  /* the library chooses (tensor cores where the shape allows)        */
  IG3_PATH_TC = 1,    /* tcgen05 implicit GEMM with split-TF32 (3xTF32) operands          */
  IG3_PATH_FMA = 2    /* register-blocked FP32 FMA direct convolution                     */
} ig3_path;

/* Parameters of IG3_EPI_POOL_REDUCE ([P8], its list of the model's operations). */
typedef struct {
  float divisor;        /* the conv output (with bias) is divided by this; must be nonzero */
  int pool;             /* max-pool window = stride = pool in every spatial dim; only 2   */
  const float* bias2;   /* [Cout] device pointer, added to each channel's mean            */
} ig3_epi_params;

/*
 * Workspace bytes conv3d_fused needs for this shape, epilogue and path (0 if
 * none).  Returns 0 as well for arguments conv3d_fused would reject.
 */
size_t conv3d_fused_workspace_size(int N, int Cin, int D, int H, int W, int Cout,
                                   int epilogue, int path);

/*
 * Valid (no padding), stride-1, 3x3x3 cross-correlation with a fused epilogue.
 * Definition ([P47], the per-output loop and its NCDHW index check):
 *   conv[n,k,od,oh,ow] = b[k] + sum_{c<Cin, kd,kh,kw<3} w[k,c,kd,kh,kw] * x[n,c,od+kd,oh+kh,ow+kw]
 * for od < D-2, oh < H-2, ow < W-2.
 *
 *   x   [N][Cin][D][H][W]                 input
 *   w   [Cout][Cin][3][3][3]              weights
 *   b   [Cout] or NULL                    conv bias (NULL = zero)
 *   epilogue / params                     see ig3_epilogue; params is read only for
 *                                         IG3_EPI_POOL_REDUCE (may be NULL otherwise)
 *   y   NONE, TANH_MISH: [N][Cout][D-2][H-2][W-2]
 *       POOL_REDUCE:     [N]  (one scalar per batch item; the pooled grid is
 *                        floor((D-2)/2) x floor((H-2)/2) x floor((W-2)/2), [P8] with
 *                        ceil_mode=False; it must be non-empty)
 *   workspace / workspace_bytes           device scratch of at least
 *                                         conv3d_fused_workspace_size(...) bytes,
 *                                         256-byte aligned; may be NULL when that is 0.
 *                                         Its contents are overwritten; calls that run
 *                                         concurrently need separate workspaces.
 *   path                                  see ig3_path
 * Requires D, H, W >= 3; N, Cin, Cout >= 1; every tensor below 2^31 elements.
 * IG3_PATH_TC additionally requires Cout to be a multiple of 16 and <= 128, and
 * for POOL_REDUCE that 128 is a multiple of 2*W (else IG3_ERR_UNSUPPORTED).
 */
int conv3d_fused(const float* x, int N, int Cin, int D, int H, int W,
                 const float* w, int Cout, const float* b,
                 int epilogue, const ig3_epi_params* params,
                 float* y, void* workspace, size_t workspace_bytes,
                 int path, void* stream);

/*
 * Zero-padded stride-1 3x3x3 cross-correlation with a fused epilogue ([P47], the
 * padding discussion: the input coordinate of an output is shifted by -pad, reads
 * outside the tensor give zero, the output size is D + 2*pad - 2):
 *   conv[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw] * x[n,c,od+kd-pad,oh+kh-pad,ow+kw-pad]
 * for od < D+2*pad-2, oh < H+2*pad-2, ow < W+2*pad-2 (pad = 1 keeps D, H, W).
 *
 * Arguments are those of conv3d_fused plus pad (0..16; 0 is conv3d_fused itself),
 * with every output size read as D+2*pad-2 etc. (POOL_REDUCE pools that grid).  The
 * zero border is never written to memory: the kernels read x at the shifted
 * coordinates and use zeros outside it.  The path (and its requirements) is the one
 * conv3d_fused takes for the padded dimensions D+2*pad, H+2*pad, W+2*pad, and so is
 * the workspace: conv3d_fused_pad_workspace_size bytes (0 when none is needed),
 * 256-byte aligned.  Requires D, H, W >= 1 and the padded volume below 2^31
 * elements; there is no no-allocation variant.
 */
size_t conv3d_fused_pad_workspace_size(int N, int Cin, int D, int H, int W, int pad, int Cout,
                                       int epilogue, int path);
int conv3d_fused_pad(const float* x, int N, int Cin, int D, int H, int W, int pad,
                     const float* w, int Cout, const float* b,
                     int epilogue, const ig3_epi_params* params,
                     float* y, void* workspace, size_t workspace_bytes,
                     int path, void* stream);

/*
 * 3x3x3 cross-correlation with zero padding `pad` and stride `stride`, fused epilogue
 * ([P47], the stride and padding discussion: the input window of output od starts at
 * od*stride - pad, reads outside the tensor give zero, the output size is
 * (D + 2*pad - 3)/stride + 1 in integer division):
 *   conv[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw]
 *                               * x[n,c,od*stride+kd-pad, oh*stride+kh-pad, ow*stride+kw-pad]
 *   y   [N][Cout][OD][OH][OW] with OD = (D + 2*pad - 3)/stride + 1 etc.
 * stride 1: exactly conv3d_fused_pad (every epilogue and path, its workspace).
 * stride 2: pad 0..16, the NONE and TANH_MISH epilogues (POOL_REDUCE returns
 *           IG3_ERR_UNSUPPORTED).  IG3_PATH_TC (and IG3_PATH_AUTO wherever it applies)
 *           runs a tensor-core kernel that gathers each tap's operand on chip; it needs
 *           Cout a multiple of 16 and <= 128, W a multiple of 4, x 16-byte aligned and
 *           ((W+2*pad-3)/2)*2 + 7 staged columns <= 256, and a 256-byte aligned
 *           workspace of conv3d_fused_ex_workspace_size bytes (the split weights;
 *           IG3_ERR_WORKSPACE if smaller).  The size query answers for a 16-byte
 *           aligned x.  Otherwise AUTO and IG3_PATH_FMA run the FP32-FMA kernel (no
 *           workspace; the size query returns 0 for IG3_PATH_FMA), which needs
 *           N * ceil(Cout/32) and OD at most 65535.
 * Other strides return IG3_ERR_UNSUPPORTED.  Other arguments as conv3d_fused.
 */
size_t conv3d_fused_ex_workspace_size(int N, int Cin, int D, int H, int W, int pad, int stride,
                                      int Cout, int epilogue, int path);
int conv3d_fused_ex(const float* x, int N, int Cin, int D, int H, int W, int pad, int stride,
                    const float* w, int Cout, const float* b,
                    int epilogue, const ig3_epi_params* params,
                    float* y, void* workspace, size_t workspace_bytes,
                    int path, void* stream);

/* Size of the library's own scratch buffer used by conv3d_fused_noalloc (4 MiB). */
#define IG3_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)

/*
 * conv3d_fused without a workspace argument, for callers that cannot allocate
 * device memory: for instance a host runtime that has reserved the whole device
 * memory budget and forbids further allocations, a latency-critical path that
 * cannot afford cudaMalloc's implicit device-wide synchronisation, or code with no
 * allocator at hand.  The source pages have no counterpart to this entry point; it
 * is an addition of this library.
 *
 * Arguments, layouts, results and error codes are those of conv3d_fused; the
 * caller still passes (and owns) x, w, b, params->bias2 and y.  The scratch comes
 * from a static buffer of IG3_NOALLOC_SCRATCH_BYTES inside the library, which every
 * device that loads the library keeps until the process exits; nothing is
 * allocated by this call.
 *   - Shapes whose scratch (conv3d_fused_workspace_size) exceeds the buffer are
 *     rejected with IG3_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device looks up the buffer's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is valid in the context it was
 *     looked up in: after a cudaDeviceReset (a new context) the next call looks it
 *     up again, so make that call before any capture too.
 *   - Every call on a device shares the one buffer, and it keeps the last call's
 *     contents.  No part of it needs to start at zero (each call rewrites all it
 *     reads), but calls whose work overlaps on the GPU (different streams, or
 *     host threads without ordering between them) race on it: order them.
 */
int conv3d_fused_noalloc(const float* x, int N, int Cin, int D, int H, int W,
                         const float* w, int Cout, const float* b,
                         int epilogue, const ig3_epi_params* params,
                         float* y, int path, void* stream);

/*
 * Depthwise-separable conv2d ([P86], the per-output pseudo-code with stride 1,
 * padding 1, dilation 1):
 *   dw[n,c,h,w]  = sum_{kh,kw<3} w_dw[c,0,kh,kw] * x[n,c,h+kh-1,w+kw-1]   (zero outside)
 *   y[n,o,h,w]   = sum_c w_pw[o,c,0,0] * dw[n,c,h,w] + (b ? b[o] : 0)
 * The depthwise result never leaves the chip.
 *
 *   x    [N][C][H][W]      w_dw [C][1][3][3]      w_pw [Cout][C][1][1]
 *   b    [Cout] or NULL    (a combined bias, sum_c w_pw[o,c] * b_dw[c] + b_pw[o])
 *   y    [N][Cout][H][W]
 * IG3_PATH_TC requires C a multiple of 16 and <= 64, Cout a multiple of 16 and <= 128,
 * W a multiple of 4 and x 16-byte aligned (else IG3_ERR_UNSUPPORTED); with
 * IG3_PATH_AUTO a misaligned x takes the FMA path.
 */
int dwsep_conv2d(const float* x, int N, int C, int H, int W,
                 const float* w_dw, const float* w_pw, int Cout, const float* b,
                 float* y, int path, void* stream);

/*
 * dwsep_conv2d with a K x K depthwise stage, K in {1, 3, 5, 7} ([P86], the discussion of
 * kernel sizes other than 3: a kernel templated on K, dispatched for the common sizes),
 * stride 1, dilation 1 and "same" padding P = (K-1)/2 (K = 3: P = 1, dwsep_conv2d itself):
 *   dw[n,c,h,w] = sum_{kh,kw<K} w_dw[c,0,kh,kw] * x[n,c,h+kh-P,w+kw-P]   (zero outside)
 *   y[n,o,h,w]  = sum_c w_pw[o,c,0,0] * dw[n,c,h,w] + (b ? b[o] : 0)
 *   w_dw [C][1][K][K]; other arguments as dwsep_conv2d.
 * K = 3 takes every path of dwsep_conv2d.  K = 5 has a tensor-core kernel too (the
 * depthwise window on the FMA pipe, the pointwise stage on tensor cores, the depthwise
 * result kept on chip) under the conditions of dwsep_conv2d's IG3_PATH_TC; IG3_PATH_AUTO
 * takes it wherever they hold.  K = 1 and 7 run on the FP32-FMA path (IG3_PATH_TC
 * returns IG3_ERR_UNSUPPORTED); other K return IG3_ERR_UNSUPPORTED.
 */
int dwsep_conv2d_ex(const float* x, int N, int C, int H, int W, int K,
                    const float* w_dw, const float* w_pw, int Cout, const float* b,
                    float* y, int path, void* stream);

/* Which path conv3d_fused / dwsep_conv2d would take for these arguments (IG3_PATH_TC or
 * IG3_PATH_FMA), or a negative status if they would be rejected. */
int conv3d_fused_select_path(int N, int Cin, int D, int H, int W, int Cout, int epilogue, int path);
int dwsep_conv2d_select_path(int N, int C, int H, int W, int Cout, int path);
/* The same for dwsep_conv2d_ex with a K x K depthwise stage. */
int dwsep_conv2d_ex_select_path(int N, int C, int H, int W, int K, int Cout, int path);

/* A static string naming a status code. */
const char* ig3_status_string(int status);

/* The message of the last call that failed on this host thread ("" if none). */
const char* ig3_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the current device's status word:
 * IG3_ERR_TIMEOUT if any kernel since the last call gave up on a bounded wait,
 * IG3_ERR_CUDA if the synchronisation itself failed, else IG3_OK.
 */
int ig3_last_device_status(void* stream);

/* Upper bound on any single wait inside a kernel, in nanoseconds, for launches made
 * after this call (process-wide; 0 restores the default of 1 s). */
void ig3_set_wait_timeout_ns(unsigned long long ns);

/*
 * Self-test of the bounded-wait machinery: launches one block that waits on a
 * shared-memory barrier nothing ever completes, with a limit of `timeout_ns`.
 * The kernel gives up, records IG3_ERR_TIMEOUT in the status word and returns;
 * the context stays usable.  Returns the launch status (IG3_OK if launched).
 */
int ig3_selftest_bounded_wait(unsigned long long timeout_ns, void* stream);

/* Number of kernels this library has launched in this process (all devices). */
unsigned long long ig3_kernel_launches(void);

/* Library version, "major.minor.patch". */
const char* ig3_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IG3_H */
