// Host-side internals of the ig3 library: argument bundles, error reporting and
// the kernel launchers each .cu file provides to the C ABI in ig3_api.cu.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ig3.h"
#include "ig3_device.cuh"

namespace ig3 {

struct Conv3dArgs {
  const float* x;
  int N, Cin, D, H, W;  // x's own dimensions
  int pad = 0;          // zero padding on every side (0: the valid convolution)
  const float* w;
  int Cout;
  const float* b;
  int epi;
  float divisor;
  int pool;
  const float* bias2;
  float* y;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  int OD() const { return D + 2 * pad - 2; }
  int OH() const { return H + 2 * pad - 2; }
  int OW() const { return W + 2 * pad - 2; }
};

struct DwsepArgs {
  const float* x;
  int N, C, H, W;
  const float* w_dw;
  const float* w_pw;
  int Cout;
  const float* b;
  float* y;
  cudaStream_t stream;
  int K = 3;  // depthwise size (the FMA path also takes 1, 5, 7)
};

// Records a message for ig3_last_error() (thread-local) and returns `status`.
int fail(int status, const char* fmt, ...);
// Converts a CUDA error into IG3_ERR_CUDA with a message; IG3_OK for cudaSuccess.
int cuda_status(cudaError_t e, const char* what);
// Counts one successful kernel launch (reported by ig3_kernel_launches) and
// returns `status` unchanged.
int count_launch(int status);
// Bounded-wait settings for a launch on the current device.
WaitCtl wait_ctl();
// Number of SMs of the current device (cached).
int num_sms();
// The calling thread's current CUDA context (through the driver entry point), or
// nullptr if none is current yet.  Device addresses of the library's __device__
// variables are valid within one context.
void* current_context();
// The driver's tensor-map encoder, looked up once through the runtime (no link-time
// dependency on the driver library); nullptr if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// conv3d_fused_select_path without touching ig3_last_error() (for size queries).
int conv3d_select_quiet(int N, int Cin, int D, int H, int W, int Cout, int epi, int path);

// The zero-padded (pad >= 0) stride-1 conv3d: argument checks, path choice on the
// padded volume, workspace check and launch (conv3d_fused, conv3d_fused_pad).
// `who` names the entry point in error messages.
int conv3d_run(const float* x, int N, int Cin, int D, int H, int W, int pad, const float* w, int Cout,
               const float* b, int epilogue, const ig3_epi_params* params, float* y, void* workspace,
               size_t workspace_bytes, int path, void* stream, const char* who);
// Workspace bytes conv3d_run needs (0 if none, or if the arguments are invalid).
size_t conv3d_workspace(int N, int Cin, int D, int H, int W, int pad, int Cout, int epi, int path);

// ---- FMA path (conv3d_fma.cu)
size_t conv3d_fma_workspace(const Conv3dArgs& a);
int conv3d_fma_launch(const Conv3dArgs& a);

// ---- tensor-core path (conv3d_tc.cu)
// Empty string if the TC path handles this shape, else the reason it does not.
const char* conv3d_tc_unsupported_reason(int N, int Cin, int D, int H, int W, int Cout, int epi);
size_t conv3d_tc_workspace(const Conv3dArgs& a);
int conv3d_tc_launch(const Conv3dArgs& a);

// ---- tensor-core path for 16 output channels with A in tensor memory (conv3d_tc16.cu);
// conv3d_tc_launch takes it wherever it applies and x is 16-byte aligned.
bool conv3d_tc16_applies(const Conv3dArgs& a, const char** why);
size_t conv3d_tc16_workspace(const Conv3dArgs& a);
int conv3d_tc16_launch(const Conv3dArgs& a);

// ---- stride-2 tensor-core path (conv3d_strided_tc.cu): A gathered into tensor memory.
// Empty string if it handles this shape (x alignment aside), else the reason it does not.
const char* conv3d_strided_tc_unsupported_reason(int N, int Cin, int D, int H, int W, int pad, int Cout, int epi);
size_t conv3d_strided_tc_workspace(int Cin, int Cout);
int conv3d_strided_tc_launch(const Conv3dArgs& a);

// ---- depthwise-separable (dwsep.cu)
// K: the depthwise size (3 or 5 on tensor cores).
const char* dwsep_tc_unsupported_reason(int N, int C, int H, int W, int Cout, int K = 3);
int dwsep_fma_launch(const DwsepArgs& a);
int dwsep_tc_launch(const DwsepArgs& a);

// ---- pool-reduce finalisation shared by both conv3d paths (conv3d_fma.cu):
// out[n] = scale * sum_{i < per_n} partial[n * per_n + i] + sum_c bias2[c], in a
// fixed order (deterministic).
int pool_reduce_finalize(const float* partial, int N, int per_n, float scale, const float* bias2,
                         int C, float* out, cudaStream_t stream);

// ---- bounded-wait self-test (ig3_api.cu)
int selftest_bounded_wait(unsigned long long timeout_ns, cudaStream_t stream);

}  // namespace ig3
