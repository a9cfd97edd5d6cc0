// conv3d_fused_pad: the zero-padded stride-1 3x3x3 convolution with a fused epilogue.
//
// Definition ("Kimi-K2.6__l2_p47", the padding discussion): the input coordinate of
// output od is od + kd - P, read as zero outside the tensor, and the output size is
// D + 2P - 2.  That is the valid convolution of the input with a P-wide zero border,
// so this entry point writes the bordered copy xp[N][Cin][D+2P][H+2P][W+2P] into the
// caller's workspace (one HBM-bound pass: x read once, xp written once) and runs
// conv3d_fused on it; every kernel, tiling and epilogue of the valid path applies
// unchanged.  The copy costs (|x| + |xp|) of memory traffic, a few percent of the
// convolution for the channel counts the tensor-core path targets.
#include <cstdint>

#include "ig3_internal.h"

namespace {

constexpr int kMaxPad = 16;

// One CTA per bordered plane (n, c, dp) at a time, 32 x 8 threads walking its rows
// and columns: consecutive threads take consecutive columns (coalesced on both
// sides), and no index needs a per-element division.
__global__ void __launch_bounds__(256) conv3d_pad_kernel(const float* __restrict__ x, float* __restrict__ xp,
                                                         int planes, int D, int H, int W, int P) {
  const int Dp = D + 2 * P, Hp = H + 2 * P, Wp = W + 2 * P;
  for (int pl = blockIdx.x; pl < planes; pl += gridDim.x) {
    const int nc = pl / Dp, dp = pl - nc * Dp;
    const int d = dp - P;
    const bool d_in = d >= 0 && d < D;
    const float* src = x + ((size_t)nc * D + (d_in ? d : 0)) * H * W;
    float* dst = xp + (size_t)pl * Hp * Wp;
    for (int hp = threadIdx.y; hp < Hp; hp += 8) {
      const int h = hp - P;
      const bool row_in = d_in && h >= 0 && h < H;
      for (int wp = threadIdx.x; wp < Wp; wp += 32) {
        const int w = wp - P;
        dst[(size_t)hp * Wp + wp] = (row_in && w >= 0 && w < W) ? __ldg(src + (size_t)h * W + w) : 0.0f;
      }
    }
  }
}

// Bytes of the bordered copy, or 0 if the arguments are out of range.
size_t padded_bytes(int N, int Cin, int D, int H, int W, int P) {
  if (N < 1 || Cin < 1 || D < 1 || H < 1 || W < 1 || P < 1 || P > kMaxPad) return 0;
  const long long e = (long long)N * Cin * (D + 2 * P) * (H + 2 * P) * (W + 2 * P);
  if (e >= (1ll << 31)) return 0;
  return ig3::align_up((size_t)e * sizeof(float), 256);
}

}  // namespace

extern "C" {

size_t conv3d_fused_pad_workspace_size(int N, int Cin, int D, int H, int W, int pad, int Cout, int epilogue,
                                       int path) {
  if (pad == 0) return conv3d_fused_workspace_size(N, Cin, D, H, W, Cout, epilogue, path);
  const size_t xp = padded_bytes(N, Cin, D, H, W, pad);
  if (xp == 0) return 0;
  const int Dp = D + 2 * pad, Hp = H + 2 * pad, Wp = W + 2 * pad;
  if (ig3::conv3d_select_quiet(N, Cin, Dp, Hp, Wp, Cout, epilogue, path) < 0) return 0;
  return xp + conv3d_fused_workspace_size(N, Cin, Dp, Hp, Wp, Cout, epilogue, path);
}

int conv3d_fused_pad(const float* x, int N, int Cin, int D, int H, int W, int pad, const float* w, int Cout,
                     const float* b, int epilogue, const ig3_epi_params* params, float* y, void* workspace,
                     size_t workspace_bytes, int path, void* stream) {
  using namespace ig3;
  if (pad == 0)
    return conv3d_fused(x, N, Cin, D, H, W, w, Cout, b, epilogue, params, y, workspace, workspace_bytes, path,
                        stream);
  if (pad < 0 || pad > kMaxPad) return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_pad: pad must be in [0, %d]", kMaxPad);
  if (N < 1 || Cin < 1 || D < 1 || H < 1 || W < 1 || Cout < 1)
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_pad: N, Cin, D, H, W and Cout must be positive");
  const size_t xp_bytes = padded_bytes(N, Cin, D, H, W, pad);
  if (xp_bytes == 0) return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_pad: padded input exceeds 2^31 elements");
  const int Dp = D + 2 * pad, Hp = H + 2 * pad, Wp = W + 2 * pad;
  const int p = conv3d_fused_select_path(N, Cin, Dp, Hp, Wp, Cout, epilogue, path);
  if (p < 0) return p;
  if (!x || !w || !y) return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_pad: x, w and y must not be NULL");
  const size_t need = xp_bytes + conv3d_fused_workspace_size(N, Cin, Dp, Hp, Wp, Cout, epilogue, path);
  if (!workspace || workspace_bytes < need)
    return fail(IG3_ERR_WORKSPACE, "conv3d_fused_pad: workspace of %zu bytes needed, %zu given", need,
                workspace ? workspace_bytes : (size_t)0);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(IG3_ERR_WORKSPACE, "conv3d_fused_pad: workspace must be 256-byte aligned");
  if (epilogue == IG3_EPI_POOL_REDUCE && (!params || !params->bias2))
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_pad: POOL_REDUCE needs params with a bias2 pointer");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* xp = static_cast<float*>(workspace);
  const int planes = N * Cin * Dp;
  const int grid = planes < 8 * 1024 ? planes : 8 * 1024;
  conv3d_pad_kernel<<<grid, dim3(32, 8), 0, st>>>(x, xp, planes, D, H, W, pad);
  const int s = count_launch(cuda_status(cudaGetLastError(), "conv3d_fused_pad: border copy launch"));
  if (s != IG3_OK) return s;
  return conv3d_fused(xp, N, Cin, Dp, Hp, Wp, w, Cout, b, epilogue, params, y,
                      static_cast<unsigned char*>(workspace) + xp_bytes, workspace_bytes - xp_bytes, path, stream);
}

}  // extern "C"
