// The C ABI of the ig3 library: argument checks, path selection, workspace
// sizing, error reporting and the per-device status word.  Every compute step
// runs in the kernels of conv3d_fma.cu, conv3d_tc.cu and dwsep.cu.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "ig3_internal.h"

// One status word per device (each device holds its own copy of a __device__
// variable).  Kernels atomicOr error bits into it; ig3_last_device_status reads
// and clears it.
__device__ unsigned int g_ig3_device_status;

namespace ig3 {
namespace {

constexpr unsigned long long kDefaultWaitNs = 1000000000ull;  // 1 s
constexpr long long kMaxElems = 0x7fffffffLL;

thread_local char t_last_error[512] = "";
std::atomic<unsigned long long> g_wait_ns{0};
std::atomic<unsigned long long> g_launches{0};

struct DeviceInfo {
  bool ready = false;
  void* ctx = nullptr;  // the context the address below belongs to
  unsigned int* status = nullptr;
  int sms = 0;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

// Set-up of the current device: the status word's device address and the SM count,
// looked up once per context (a cudaDeviceReset makes a new context, in which the
// module's variables may sit at other addresses).
DeviceInfo* current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_devices_mu);
  DeviceInfo& d = g_devices[dev];
  void* ctx = current_context();
  if (!d.ready || ctx == nullptr || ctx != d.ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ig3_device_status) != cudaSuccess) return nullptr;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    d.status = static_cast<unsigned int*>(p);
    d.sms = sms;
    d.ctx = current_context();  // now initialised by the lookup
    d.ready = true;
  }
  return &d;
}

__global__ void selftest_wait_kernel(WaitCtl ctl) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`, so its phase 0 never completes.
  mbar_wait_bounded(&bar, 0, ctl, &abort_flag);
  __syncthreads();
}

long long prod(std::initializer_list<long long> v) {
  long long p = 1;
  for (long long e : v) {
    if (e <= 0) return -1;
    if (p > kMaxElems / e) return kMaxElems + 1;
    p *= e;
  }
  return p;
}

// Checks the shape arguments of conv3d_fused and chooses a path.  Returns the path
// (IG3_PATH_TC / IG3_PATH_FMA) or a negative status (with ig3_last_error set).
int conv3d_select(int N, int Cin, int D, int H, int W, int Cout, int epi, int path) {
  if (N < 1 || Cin < 1 || Cout < 1 || D < 1 || H < 1 || W < 1)
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused: sizes must be positive (N=%d Cin=%d Cout=%d D=%d H=%d W=%d)", N,
                Cin, Cout, D, H, W);
  if (D < 3 || H < 3 || W < 3)
    return fail(IG3_ERR_UNSUPPORTED, "conv3d_fused: a valid 3x3x3 conv needs D, H, W >= 3 (got %d, %d, %d)", D, H,
                W);
  if (epi < IG3_EPI_NONE || epi > IG3_EPI_POOL_REDUCE)
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused: unknown epilogue %d", epi);
  if (path < IG3_PATH_AUTO || path > IG3_PATH_FMA)
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused: unknown path %d", path);
  if (prod({N, Cin, D, H, W}) > kMaxElems || prod({N, Cout, D - 2, H - 2, W - 2}) > kMaxElems ||
      prod({Cout, Cin, 27}) > kMaxElems)
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused: a tensor has 2^31 or more elements");
  if (epi == IG3_EPI_POOL_REDUCE && ((D - 2) < 2 || (H - 2) < 2 || (W - 2) < 2))
    return fail(IG3_ERR_UNSUPPORTED, "conv3d_fused: the 2x2x2 pooled grid is empty");
  const char* why = conv3d_tc_unsupported_reason(N, Cin, D, H, W, Cout, epi);
  const bool tc_ok = (why[0] == '\0');
  if (path == IG3_PATH_TC) {
    if (!tc_ok) return fail(IG3_ERR_UNSUPPORTED, "conv3d_fused: tensor-core path: %s", why);
    return IG3_PATH_TC;
  }
  if (path == IG3_PATH_FMA) return IG3_PATH_FMA;
  // Automatic choice: the tensor-core kernels wherever they apply.  Measured over 42
  // shapes from x[1,1,3,3,4] to the full workloads (device time per call, one GB300),
  // they beat the FMA kernel on every one, by 1.5x on the smallest and 6.6x at full
  // size (the FMA kernel's fixed cost grows with Cin: each CTA walks the input
  // channels serially); the FMA kernel takes the shapes they do not cover.
  return tc_ok ? IG3_PATH_TC : IG3_PATH_FMA;
}

int dwsep_select(int N, int C, int H, int W, int Cout, int path) {
  if (N < 1 || C < 1 || H < 1 || W < 1 || Cout < 1)
    return fail(IG3_ERR_INVALID_ARG, "dwsep_conv2d: sizes must be positive (N=%d C=%d Cout=%d H=%d W=%d)", N, C,
                Cout, H, W);
  if (path < IG3_PATH_AUTO || path > IG3_PATH_FMA)
    return fail(IG3_ERR_INVALID_ARG, "dwsep_conv2d: unknown path %d", path);
  if (prod({N, C, H, W}) > kMaxElems || prod({N, Cout, H, W}) > kMaxElems || prod({Cout, C}) > kMaxElems)
    return fail(IG3_ERR_INVALID_ARG, "dwsep_conv2d: a tensor has 2^31 or more elements");
  const char* why = dwsep_tc_unsupported_reason(N, C, H, W, Cout);
  const bool tc_ok = (why[0] == '\0');
  if (path == IG3_PATH_TC) {
    if (!tc_ok) return fail(IG3_ERR_UNSUPPORTED, "dwsep_conv2d: tensor-core path: %s", why);
    return IG3_PATH_TC;
  }
  if (path == IG3_PATH_FMA) return IG3_PATH_FMA;
  if (!tc_ok) return IG3_PATH_FMA;
  // Per-call cost models (microseconds) fitted to the measured crossover of the two
  // paths (N 1..4, H = W 32..256, C 16..64, Cout 16..128; one GB300): a fixed part
  // that grows with the channel counts (both paths are latency-bound at these sizes)
  // plus the work at each path's large-size rate.
  const double gflop = 2e-9 * (double)N * H * W * (double)C * (9.0 + Cout);
  const double t_tc = 8.5 + 0.23 * C + 0.075 * Cout + 6.0 * gflop;
  const double t_fma = 6.6 + 0.39 * C + 93.0 * gflop;
  return t_tc < t_fma ? IG3_PATH_TC : IG3_PATH_FMA;
}

}  // namespace

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return IG3_OK;
  return fail(IG3_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

int count_launch(int status) {
  if (status == IG3_OK) g_launches.fetch_add(1);
  return status;
}

WaitCtl wait_ctl() {
  WaitCtl c;
  const unsigned long long ns = g_wait_ns.load();
  c.limit_ns = ns ? ns : kDefaultWaitNs;
  DeviceInfo* d = current_device();
  c.status = d ? d->status : nullptr;
  return c;
}

void* current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static std::once_flag once;
  static Fn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(ptr);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

int num_sms() {
  DeviceInfo* d = current_device();
  return d ? d->sms : 0;
}

int conv3d_select_quiet(int N, int Cin, int D, int H, int W, int Cout, int epi, int path) {
  char saved[sizeof(t_last_error)];
  snprintf(saved, sizeof(saved), "%s", t_last_error);
  const int p = conv3d_select(N, Cin, D, H, W, Cout, epi, path);
  snprintf(t_last_error, sizeof(t_last_error), "%s", saved);
  return p;
}

int selftest_bounded_wait(unsigned long long timeout_ns, cudaStream_t stream) {
  DeviceInfo* d = current_device();
  if (!d) return fail(IG3_ERR_CUDA, "ig3_selftest_bounded_wait: device set-up failed");
  WaitCtl c{timeout_ns ? timeout_ns : 1000000ull, d->status};
  selftest_wait_kernel<<<1, 32, 0, stream>>>(c);
  return count_launch(cuda_status(cudaGetLastError(), "bounded-wait self-test launch"));
}

size_t conv3d_workspace(int N, int Cin, int D, int H, int W, int pad, int Cout, int epi, int path) {
  const int p = conv3d_select_quiet(N, Cin, D + 2 * pad, H + 2 * pad, W + 2 * pad, Cout, epi, path);
  if (p < 0) return 0;
  Conv3dArgs a{};
  a.N = N; a.Cin = Cin; a.D = D; a.H = H; a.W = W; a.pad = pad; a.Cout = Cout; a.epi = epi;
  return p == IG3_PATH_TC ? conv3d_tc_workspace(a) : conv3d_fma_workspace(a);
}

int conv3d_run(const float* x, int N, int Cin, int D, int H, int W, int pad, const float* w, int Cout,
               const float* b, int epilogue, const ig3_epi_params* params, float* y, void* workspace,
               size_t workspace_bytes, int path, void* stream, const char* who) {
  // Path choice and shape checks on the convolution's (padded) input volume.
  const int p = conv3d_select(N, Cin, D + 2 * pad, H + 2 * pad, W + 2 * pad, Cout, epilogue, path);
  if (p < 0) return p;
  if (!x || !w || !y) return fail(IG3_ERR_INVALID_ARG, "%s: x, w and y must not be NULL", who);
  Conv3dArgs a{};
  a.x = x; a.N = N; a.Cin = Cin; a.D = D; a.H = H; a.W = W; a.pad = pad; a.w = w; a.Cout = Cout; a.b = b;
  a.epi = epilogue; a.divisor = 1.0f; a.pool = 2; a.bias2 = nullptr; a.y = y;
  a.ws = workspace; a.ws_bytes = workspace_bytes; a.stream = static_cast<cudaStream_t>(stream);
  if (epilogue == IG3_EPI_POOL_REDUCE) {
    if (!params || !params->bias2)
      return fail(IG3_ERR_INVALID_ARG, "%s: POOL_REDUCE needs params with a bias2 pointer", who);
    if (params->pool != 2) return fail(IG3_ERR_UNSUPPORTED, "%s: only pool = 2 is supported", who);
    if (!std::isfinite(params->divisor) || params->divisor == 0.0f)
      return fail(IG3_ERR_INVALID_ARG, "%s: divisor must be finite and nonzero", who);
    a.divisor = params->divisor;
    a.pool = params->pool;
    a.bias2 = params->bias2;
  }
  const size_t need = (p == IG3_PATH_TC) ? conv3d_tc_workspace(a) : conv3d_fma_workspace(a);
  if (need > 0) {
    if (!workspace || workspace_bytes < need)
      return fail(IG3_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", who, need,
                  workspace ? workspace_bytes : (size_t)0);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
      return fail(IG3_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", who);
  }
  if (!current_device()) return fail(IG3_ERR_CUDA, "%s: device set-up failed", who);
  return p == IG3_PATH_TC ? conv3d_tc_launch(a) : conv3d_fma_launch(a);
}

}  // namespace ig3

using namespace ig3;

extern "C" {

size_t conv3d_fused_workspace_size(int N, int Cin, int D, int H, int W, int Cout, int epilogue, int path) {
  return conv3d_workspace(N, Cin, D, H, W, 0, Cout, epilogue, path);
}

int conv3d_fused_select_path(int N, int Cin, int D, int H, int W, int Cout, int epilogue, int path) {
  return conv3d_select(N, Cin, D, H, W, Cout, epilogue, path);
}

int dwsep_conv2d_select_path(int N, int C, int H, int W, int Cout, int path) {
  return dwsep_select(N, C, H, W, Cout, path);
}

int conv3d_fused(const float* x, int N, int Cin, int D, int H, int W, const float* w, int Cout, const float* b,
                 int epilogue, const ig3_epi_params* params, float* y, void* workspace, size_t workspace_bytes,
                 int path, void* stream) {
  return conv3d_run(x, N, Cin, D, H, W, 0, w, Cout, b, epilogue, params, y, workspace, workspace_bytes, path, stream,
                    "conv3d_fused");
}

int dwsep_conv2d(const float* x, int N, int C, int H, int W, const float* w_dw, const float* w_pw, int Cout,
                 const float* b, float* y, int path, void* stream) {
  const int p = dwsep_select(N, C, H, W, Cout, path);
  if (p < 0) return p;
  if (!x || !w_dw || !w_pw || !y)
    return fail(IG3_ERR_INVALID_ARG, "dwsep_conv2d: x, w_dw, w_pw and y must not be NULL");
  if (!current_device()) return fail(IG3_ERR_CUDA, "dwsep_conv2d: device set-up failed");
  DwsepArgs a{x, N, C, H, W, w_dw, w_pw, Cout, b, y, static_cast<cudaStream_t>(stream)};
  // The tensor-core kernel copies 16-byte aligned row segments; a misaligned x goes to
  // the FMA kernel when the caller left the choice to the library.
  if (p == IG3_PATH_TC && path == IG3_PATH_AUTO && reinterpret_cast<uintptr_t>(x) % 16 != 0)
    return dwsep_fma_launch(a);
  return p == IG3_PATH_TC ? dwsep_tc_launch(a) : dwsep_fma_launch(a);
}

// Path of dwsep_conv2d_ex for K != 3 (IG3_PATH_TC or IG3_PATH_FMA), or a negative status.
// K = 5 has a tensor-core kernel (the depthwise window on the FMA pipe, the pointwise
// stage on tensor cores); AUTO takes it wherever it applies (x alignment is checked at
// the call).  The 3x3 cost model does not apply to other K.
int dwsep_ex_select(int N, int C, int H, int W, int K, int Cout, int path) {
  if (K != 1 && K != 5 && K != 7)
    return fail(IG3_ERR_UNSUPPORTED, "dwsep_conv2d_ex: depthwise size %d (1, 3, 5 or 7 are supported)", K);
  if (path < IG3_PATH_AUTO || path > IG3_PATH_FMA)
    return fail(IG3_ERR_INVALID_ARG, "dwsep_conv2d_ex: unknown path %d", path);
  // The shape and element-count checks of the 3x3 entry point.
  const int p0 = dwsep_select(N, C, H, W, Cout, IG3_PATH_FMA);
  if (p0 < 0) return p0;
  if ((long long)C * K * K >= (1ll << 31)) return fail(IG3_ERR_INVALID_ARG, "dwsep_conv2d_ex: w_dw too large");
  const char* why = (K == 5) ? dwsep_tc_unsupported_reason(N, C, H, W, Cout, K) : "runs on the FMA path only";
  const bool tc_ok = why[0] == '\0';
  if (path == IG3_PATH_TC && !tc_ok)
    return fail(IG3_ERR_UNSUPPORTED, "dwsep_conv2d_ex: depthwise size %d on the tensor-core path: %s", K, why);
  return (path != IG3_PATH_FMA && tc_ok) ? IG3_PATH_TC : IG3_PATH_FMA;
}

int dwsep_conv2d_ex_select_path(int N, int C, int H, int W, int K, int Cout, int path) {
  if (K == 3) return dwsep_select(N, C, H, W, Cout, path);
  return dwsep_ex_select(N, C, H, W, K, Cout, path);
}

int dwsep_conv2d_ex(const float* x, int N, int C, int H, int W, int K, const float* w_dw, const float* w_pw, int Cout,
                    const float* b, float* y, int path, void* stream) {
  if (K == 3) return dwsep_conv2d(x, N, C, H, W, w_dw, w_pw, Cout, b, y, path, stream);
  const int sel = dwsep_ex_select(N, C, H, W, K, Cout, path);
  if (sel < 0) return sel;
  if (!x || !w_dw || !w_pw || !y)
    return fail(IG3_ERR_INVALID_ARG, "dwsep_conv2d_ex: x, w_dw, w_pw and y must not be NULL");
  if (!current_device()) return fail(IG3_ERR_CUDA, "dwsep_conv2d_ex: device set-up failed");
  DwsepArgs a{x, N, C, H, W, w_dw, w_pw, Cout, b, y, static_cast<cudaStream_t>(stream)};
  a.K = K;
  // A misaligned x goes to the FMA kernel when the caller left the choice to the library.
  if (sel == IG3_PATH_TC && (path == IG3_PATH_TC || reinterpret_cast<uintptr_t>(x) % 16 == 0))
    return dwsep_tc_launch(a);
  return dwsep_fma_launch(a);
}

const char* ig3_status_string(int status) {
  switch (status) {
    case IG3_OK: return "IG3_OK";
    case IG3_ERR_INVALID_ARG: return "IG3_ERR_INVALID_ARG";
    case IG3_ERR_UNSUPPORTED: return "IG3_ERR_UNSUPPORTED";
    case IG3_ERR_CUDA: return "IG3_ERR_CUDA";
    case IG3_ERR_TIMEOUT: return "IG3_ERR_TIMEOUT";
    case IG3_ERR_WORKSPACE: return "IG3_ERR_WORKSPACE";
    default: return "IG3_ERR_UNKNOWN";
  }
}

const char* ig3_last_error(void) { return t_last_error; }

int ig3_last_device_status(void* stream) {
  int st = cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "ig3_last_device_status: sync");
  if (st != IG3_OK) return st;
  DeviceInfo* d = current_device();
  if (!d) return fail(IG3_ERR_CUDA, "ig3_last_device_status: device set-up failed");
  unsigned int v = 0;
  st = cuda_status(cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost), "ig3_last_device_status: read");
  if (st != IG3_OK) return st;
  if (v != 0) {
    const unsigned int zero = 0;
    st = cuda_status(cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice),
                     "ig3_last_device_status: clear");
    if (st != IG3_OK) return st;
    if (v & kDevStatusTimeout) return fail(IG3_ERR_TIMEOUT, "a bounded wait inside a kernel ran out");
  }
  return IG3_OK;
}

void ig3_set_wait_timeout_ns(unsigned long long ns) { g_wait_ns.store(ns); }

int ig3_selftest_bounded_wait(unsigned long long timeout_ns, void* stream) {
  return selftest_bounded_wait(timeout_ns, static_cast<cudaStream_t>(stream));
}

unsigned long long ig3_kernel_launches(void) { return g_launches.load(); }

const char* ig3_version(void) { return "0.1.0"; }

}  // extern "C"
