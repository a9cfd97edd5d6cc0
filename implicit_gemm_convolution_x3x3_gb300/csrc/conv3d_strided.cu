// conv3d_fused_ex: the 3x3x3 convolution with zero padding P and stride S, fused
// epilogue.  Stride 1 is conv3d_fused_pad (every path); stride 2 runs the tensor-core
// kernel of conv3d_strided_tc.cu where it applies, else the FP32-FMA kernel below.
//
// Definition ("Kimi-K2.6__l2_p47", the stride and padding discussion): the input
// window of output od starts at od*S - P, reads outside the tensor are zero, and the
// output size is (D + 2P - 3)/S + 1:
//   conv[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw] * x[n,c,od*S+kd-P,oh*S+kh-P,ow*S+kw-P].
//
// Stride 2 breaks the stride-1 tensor-core kernels' addressing (the tap shift is a
// descriptor offset into one tile of consecutive positions; strided positions are
// not); the strided tensor-core kernel gathers its A tiles instead and needs Cout a
// multiple of 16 (<= 128), W a multiple of 4 and x 16-byte aligned.  Other shapes run
// on the FMA pipe: a CTA computes 16 x 32 outputs of one plane for 32 output
// channels, two rows per thread (64 accumulators).  Each input channel's strided halo,
// 3 x ((16-1)S+3) x ((32-1)S+3), and its weights for the 32 outputs are staged in
// shared memory by 4-byte cp.async copies whose zero-fill is the padding, two stages
// deep: the next channel's copies fly while this one is computed.  The kernel is
// bound by instruction issue, so each staged input feeds as many FMAs as the
// registers allow (32 output channels: per tap two input reads and eight broadcast
// float4 weight rows, the same for the whole CTA, for 64 FMAs).
#include <cstdint>

#include "ig3_internal.h"

namespace {

// CTA: 16 x 32 outputs of one plane x 32 output channels; thread (ty, tx) takes rows
// ty and ty + 8 of column tx (64 accumulators).
constexpr int kTH = 16, kTW = 32, kTCO = 32, kThreads = 256;
constexpr int kMaxPad = 16;

// One stage = one input channel: its 3 x H x W strided halo, then its weights for the
// CTA's 32 output channels.  Two stages: the copies of channel c+1 fly while channel c
// is computed.
template <int S>
struct Halo {
  static constexpr int H = (kTH - 1) * S + 3, W = (kTW - 1) * S + 3;
  // The weights follow the halo and are read as float4: keep their start 16-byte aligned.
  static constexpr int in_floats = (3 * H * W + 3) / 4 * 4;
  static constexpr int stage_floats = in_floats + 27 * kTCO;
  static constexpr size_t smem_bytes = 2 * (size_t)stage_floats * sizeof(float);
  static_assert(in_floats % 4 == 0 && stage_floats % 4 == 0 && (kTCO % 4) == 0,
                "float4 weight rows must stay 16-byte aligned");
};

using ig3::cp_async4;

template <int S, int EPI>
__global__ void __launch_bounds__(kThreads) conv3d_strided_fma_kernel(
    const float* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias, float* __restrict__ y,
    int Cin, int D, int H, int W, int Cout, int P, int OD, int OH, int OW) {
  constexpr int HH = Halo<S>::H, HW = Halo<S>::W, kRows = 3 * HH;
  extern __shared__ __align__(16) float smem[];   // [2 stages][halo | weights]

  const int tiles_w = (OW + kTW - 1) / kTW;
  const int ow0 = (blockIdx.x % tiles_w) * kTW, oh0 = (blockIdx.x / tiles_w) * kTH;
  const int od = blockIdx.y;
  const int cgroups = (Cout + kTCO - 1) / kTCO;
  const int n = blockIdx.z / cgroups, co0 = (blockIdx.z % cgroups) * kTCO;
  const int tid = threadIdx.x;
  const int ty = tid >> 5, tx = tid & 31;
  // Input origin of the tile (may be negative: the zero border).
  const int d0 = od * S - P, h0 = oh0 * S - P, w0 = ow0 * S - P;
  const size_t plane = (size_t)H * W;

  // Copies of channel c into stage st: halo rows (one index decomposition per row, a
  // warp across its columns) and the channel's weights.
  auto stage_in = [&](int c, int st) {
    float* s_in = smem + st * Halo<S>::stage_floats;
    float* s_w = s_in + Halo<S>::in_floats;
    for (int row = ty; row < kRows; row += kThreads / 32) {
      const int kd = row / HH, r = row % HH;
      const int d = d0 + kd, h = h0 + r;
      const bool row_in = d >= 0 && d < D && h >= 0 && h < H;
      const float* src = row_in ? x + (((size_t)n * Cin + c) * D + d) * plane + (size_t)h * W : x;
      float* dst = s_in + row * HW;
      for (int q = tx; q < HW; q += 32) {
        const int ww = w0 + q;
        const bool ok = row_in && ww >= 0 && ww < W;
        cp_async4(dst + q, ok ? src + ww : x, ok);
      }
    }
    for (int i = tid; i < 27 * kTCO; i += kThreads) {
      const int j = i % kTCO, tap = i / kTCO, co = co0 + j;
      const bool ok = co < Cout;
      cp_async4(s_w + i, ok ? w + ((size_t)co * Cin + c) * 27 + tap : w, ok);
    }
    ig3::cp_async_commit();
  };

  float acc[2][kTCO];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int j = 0; j < kTCO; ++j) acc[r][j] = 0.0f;

  stage_in(0, 0);
  for (int c = 0; c < Cin; ++c) {
    const int st = c & 1;
    if (c + 1 < Cin) {
      stage_in(c + 1, st ^ 1);   // that stage was last read before the barrier ending c - 1
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const float* s_in = smem + st * Halo<S>::stage_floats;
    const float* s_w = s_in + Halo<S>::in_floats;
#pragma unroll
    for (int kd = 0; kd < 3; ++kd)
#pragma unroll
      for (int kh = 0; kh < 3; ++kh)
#pragma unroll
        for (int kw = 0; kw < 3; ++kw) {
          const float* xr = s_in + (kd * HH + ty * S + kh) * HW + tx * S + kw;
          const float xv0 = xr[0], xv1 = xr[8 * S * HW];
          const float4* wr = reinterpret_cast<const float4*>(s_w + ((kd * 3 + kh) * 3 + kw) * kTCO);
#pragma unroll
          for (int q4 = 0; q4 < kTCO / 4; ++q4) {
            const float4 wv = wr[q4];
            acc[0][4 * q4 + 0] = fmaf(wv.x, xv0, acc[0][4 * q4 + 0]);
            acc[0][4 * q4 + 1] = fmaf(wv.y, xv0, acc[0][4 * q4 + 1]);
            acc[0][4 * q4 + 2] = fmaf(wv.z, xv0, acc[0][4 * q4 + 2]);
            acc[0][4 * q4 + 3] = fmaf(wv.w, xv0, acc[0][4 * q4 + 3]);
            acc[1][4 * q4 + 0] = fmaf(wv.x, xv1, acc[1][4 * q4 + 0]);
            acc[1][4 * q4 + 1] = fmaf(wv.y, xv1, acc[1][4 * q4 + 1]);
            acc[1][4 * q4 + 2] = fmaf(wv.z, xv1, acc[1][4 * q4 + 2]);
            acc[1][4 * q4 + 3] = fmaf(wv.w, xv1, acc[1][4 * q4 + 3]);
          }
        }
    __syncthreads();   // stage st is refilled two channels on
  }

  const int ow = ow0 + tx;
  if (ow >= OW) return;
  const size_t ohw = (size_t)OH * OW;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int oh = oh0 + ty + 8 * rr;
    if (oh >= OH) break;
#pragma unroll
    for (int j = 0; j < kTCO; ++j) {
      const int co = co0 + j;
      if (co >= Cout) break;
      float v = acc[rr][j] + (bias ? __ldg(bias + co) : 0.0f);
      if (EPI == IG3_EPI_TANH_MISH) v = ig3::tanh_mish(v);
      y[(((size_t)n * Cout + co) * OD + od) * ohw + (size_t)oh * OW + ow] = v;
    }
  }
}

// Output size of one dimension, or 0 if there is none.
int out_dim(int s, int P, int S) { return s + 2 * P < 3 ? 0 : (s + 2 * P - 3) / S + 1; }

// Which stride-2 path a call takes (IG3_PATH_TC or IG3_PATH_FMA), or a negative status.
// Automatic choice: the tensor-core kernel wherever it applies (x alignment is checked
// at the call).
int strided_select(int N, int Cin, int D, int H, int W, int pad, int Cout, int epilogue, int path) {
  using namespace ig3;
  if (path != IG3_PATH_AUTO && path != IG3_PATH_FMA && path != IG3_PATH_TC)
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_ex: unknown path %d", path);
  const char* why = conv3d_strided_tc_unsupported_reason(N, Cin, D, H, W, pad, Cout, epilogue);
  const bool tc_ok = why[0] == '\0';
  if (path == IG3_PATH_TC && !tc_ok) return fail(IG3_ERR_UNSUPPORTED, "conv3d_fused_ex: stride-2 tensor-core path: %s", why);
  if (path == IG3_PATH_FMA) return IG3_PATH_FMA;
  return tc_ok ? IG3_PATH_TC : IG3_PATH_FMA;
}

}  // namespace

extern "C" {

size_t conv3d_fused_ex_workspace_size(int N, int Cin, int D, int H, int W, int pad, int stride, int Cout,
                                      int epilogue, int path) {
  if (stride == 1) return conv3d_fused_pad_workspace_size(N, Cin, D, H, W, pad, Cout, epilogue, path);
  if (stride != 2 || N < 1 || Cin < 1 || D < 1 || H < 1 || W < 1 || Cout < 1 || pad < 0 || pad > kMaxPad) return 0;
  if (epilogue != IG3_EPI_NONE && epilogue != IG3_EPI_TANH_MISH) return 0;
  if (path != IG3_PATH_AUTO && path != IG3_PATH_TC) return 0;
  // The size query has no x pointer: it answers for a 16-byte aligned x.
  if (ig3::conv3d_strided_tc_unsupported_reason(N, Cin, D, H, W, pad, Cout, epilogue)[0] != '\0') return 0;
  return ig3::conv3d_strided_tc_workspace(Cin, Cout);
}

int conv3d_fused_ex(const float* x, int N, int Cin, int D, int H, int W, int pad, int stride, const float* w,
                    int Cout, const float* b, int epilogue, const ig3_epi_params* params, float* y, void* workspace,
                    size_t workspace_bytes, int path, void* stream) {
  using namespace ig3;
  if (stride == 1)
    return conv3d_fused_pad(x, N, Cin, D, H, W, pad, w, Cout, b, epilogue, params, y, workspace, workspace_bytes,
                            path, stream);
  if (stride != 2) return fail(IG3_ERR_UNSUPPORTED, "conv3d_fused_ex: stride %d (1 or 2 are supported)", stride);
  if (pad < 0 || pad > kMaxPad) return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_ex: pad must be in [0, %d]", kMaxPad);
  if (N < 1 || Cin < 1 || D < 1 || H < 1 || W < 1 || Cout < 1)
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_ex: N, Cin, D, H, W and Cout must be positive");
  if (epilogue != IG3_EPI_NONE && epilogue != IG3_EPI_TANH_MISH)
    return fail(epilogue == IG3_EPI_POOL_REDUCE ? IG3_ERR_UNSUPPORTED : IG3_ERR_INVALID_ARG,
                "conv3d_fused_ex: stride 2 supports the NONE and TANH_MISH epilogues");
  const int OD = out_dim(D, pad, 2), OH = out_dim(H, pad, 2), OW = out_dim(W, pad, 2);
  if (OD < 1 || OH < 1 || OW < 1) return fail(IG3_ERR_UNSUPPORTED, "conv3d_fused_ex: no output for these sizes");
  const long long nx = (long long)N * Cin * D * H * W, ny = (long long)N * Cout * OD * OH * OW;
  if (nx >= (1ll << 31) || ny >= (1ll << 31) || (long long)Cout * Cin * 27 >= (1ll << 31))
    return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_ex: a tensor has 2^31 or more elements");
  int pth = strided_select(N, Cin, D, H, W, pad, Cout, epilogue, path);
  if (pth < 0) return pth;
  if (!x || !w || !y) return fail(IG3_ERR_INVALID_ARG, "conv3d_fused_ex: x, w and y must not be NULL");
  if (pth == IG3_PATH_TC && reinterpret_cast<uintptr_t>(x) % 16 != 0) {
    if (path == IG3_PATH_TC)
      return fail(IG3_ERR_UNSUPPORTED, "conv3d_fused_ex: the stride-2 tensor-core path needs x 16-byte aligned");
    pth = IG3_PATH_FMA;
  }
  if (pth == IG3_PATH_TC) {
    Conv3dArgs a{};
    a.x = x; a.N = N; a.Cin = Cin; a.D = D; a.H = H; a.W = W; a.pad = pad;
    a.w = w; a.Cout = Cout; a.b = b; a.epi = epilogue; a.divisor = 1.0f; a.pool = 0; a.bias2 = nullptr;
    a.y = y; a.ws = workspace; a.ws_bytes = workspace_bytes; a.stream = static_cast<cudaStream_t>(stream);
    return conv3d_strided_tc_launch(a);
  }
  const long long gz = (long long)N * ((Cout + kTCO - 1) / kTCO);
  const long long gx = (long long)((OW + kTW - 1) / kTW) * ((OH + kTH - 1) / kTH);
  if (gz > 65535 || OD > 65535 || gx >= (1ll << 31))
    return fail(IG3_ERR_UNSUPPORTED, "conv3d_fused_ex: grid too large for these sizes");
  (void)params; (void)workspace; (void)workspace_bytes;
  const dim3 grid((unsigned)gx, (unsigned)OD, (unsigned)gz);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t smem = Halo<2>::smem_bytes;
  auto go = [&](auto kernel) -> int {
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_status(e, "conv3d_fused_ex: set shared memory size");
    kernel<<<grid, kThreads, smem, st>>>(x, w, b, y, Cin, D, H, W, Cout, pad, OD, OH, OW);
    return count_launch(cuda_status(cudaGetLastError(), "conv3d_fused_ex: stride-2 kernel launch"));
  };
  return epilogue == IG3_EPI_TANH_MISH ? go(conv3d_strided_fma_kernel<2, IG3_EPI_TANH_MISH>)
                                       : go(conv3d_strided_fma_kernel<2, IG3_EPI_NONE>);
}

}  // extern "C"
