// conv3d_fused_noalloc: conv3d_fused for callers that cannot allocate device memory.
//
// conv3d_fused needs a scratch workspace on some paths (the split weights of the
// tensor-core path, the per-block partial sums of the pool-reduce epilogue), which
// its caller normally allocates.  Some callers cannot do that: a host runtime that
// has reserved the whole device memory budget up front and forbids other
// allocations, a latency-critical path where cudaMalloc's implicit device-wide
// synchronisation is not acceptable, or code with no allocator at hand.  This entry
// point gives them the same computation with the scratch taken from a fixed buffer
// that lives in the library itself, so nothing is allocated per call.
//
// The buffer is a file-scope __device__ array of IG3_NOALLOC_SCRATCH_BYTES; every
// device that loads the library holds it until the process exits.  Host code may
// not pass the array's name to a kernel (in host code it names a host-side stand-in,
// not device memory), so the first call on each device looks up the array's device
// address with cudaGetSymbolAddress while that device is current, and later calls
// reuse it.  The address belongs to the context it was looked up in: when the
// current context is another one (after a cudaDeviceReset, say), the next call
// looks it up again.
#include <mutex>

#include "ig3_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[IG3_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
void* g_scratch_ctx[kMaxDevices];  // the context each address was looked up in
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device (looked up once per
// device), or nullptr with the error recorded.
void* scratch_on_current_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    ig3::cuda_status(e, "conv3d_fused_noalloc: cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    ig3::fail(IG3_ERR_UNSUPPORTED, "conv3d_fused_noalloc: device ordinal %d out of range", dev);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  void* ctx = ig3::current_context();
  if (g_scratch_addr[dev] == nullptr || ctx == nullptr || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      g_scratch_addr[dev] = nullptr;
      ig3::cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                       "conv3d_fused_noalloc: cudaGetSymbolAddress of the static scratch");
      return nullptr;
    }
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = ig3::current_context();  // now initialised by the lookup
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int conv3d_fused_noalloc(const float* x, int N, int Cin, int D, int H, int W, const float* w, int Cout,
                                    const float* b, int epilogue, const ig3_epi_params* params, float* y, int path,
                                    void* stream) {
  // Shape and argument errors first, with the same codes conv3d_fused returns.
  const int chosen = conv3d_fused_select_path(N, Cin, D, H, W, Cout, epilogue, path);
  if (chosen < 0) return chosen;
  const size_t need = conv3d_fused_workspace_size(N, Cin, D, H, W, Cout, epilogue, path);
  if (need > (size_t)IG3_NOALLOC_SCRATCH_BYTES)
    return ig3::fail(IG3_ERR_WORKSPACE,
                     "conv3d_fused_noalloc: this shape needs %zu bytes of scratch, more than the %zu-byte static "
                     "buffer; use conv3d_fused with a caller-provided workspace",
                     need, (size_t)IG3_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_on_current_device();
    if (scratch == nullptr) return IG3_ERR_CUDA;
  }
  // Nothing in the scratch has to start at zero: each call rewrites the split
  // weights and every partial sum it later reads.
  return conv3d_fused(x, N, Cin, D, H, W, w, Cout, b, epilogue, params, y, scratch,
                      need > 0 ? (size_t)IG3_NOALLOC_SCRATCH_BYTES : 0, path, stream);
}
