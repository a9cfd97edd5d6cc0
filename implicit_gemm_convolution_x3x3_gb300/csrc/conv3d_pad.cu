// conv3d_fused_pad: the zero-padded stride-1 3x3x3 convolution with a fused epilogue.
//
// Definition ("Kimi-K2.6__l2_p47", the padding discussion): the input coordinate of
// output od is od + kd - P, read as zero outside the tensor, and the output size is
// D + 2P - 2.  That is the valid convolution of the input with a P-wide zero border.
// The border is never written to memory: the tensor-core kernel's convert warps
// read x at the shifted coordinates of a virtual padded volume and write zeros into
// the MMA operand where the volume lies outside x (conv3d_tc.cu), and the FMA
// kernel's staging does the same for its halo (conv3d_fma.cu).  So the padded
// convolution costs what the valid one on the padded volume costs, with no extra
// pass over HBM and no workspace beyond the valid path's.
#include "ig3_internal.h"

namespace {

constexpr int kMaxPad = 16;

}  // namespace

extern "C" {

size_t conv3d_fused_pad_workspace_size(int N, int Cin, int D, int H, int W, int pad, int Cout, int epilogue,
                                       int path) {
  if (pad < 0 || pad > kMaxPad) return 0;
  return ig3::conv3d_workspace(N, Cin, D, H, W, pad, Cout, epilogue, path);
}

int conv3d_fused_pad(const float* x, int N, int Cin, int D, int H, int W, int pad, const float* w, int Cout,
                     const float* b, int epilogue, const ig3_epi_params* params, float* y, void* workspace,
                     size_t workspace_bytes, int path, void* stream) {
  using namespace ig3;
  if (pad < 0 || pad > kMaxPad) return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_pad: pad must be in [0, %d]", kMaxPad);
  if (N < 1 || Cin < 1 || D < 1 || H < 1 || W < 1 || Cout < 1)
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_pad: N, Cin, D, H, W and Cout must be positive");
  return conv3d_run(x, N, Cin, D, H, W, pad, w, Cout, b, epilogue, params, y, workspace, workspace_bytes, path,
                    stream, "conv3d_fused_pad");
}

}  // extern "C"
