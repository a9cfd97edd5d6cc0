// Depthwise 3x3 (stride 1, pad 1) followed by pointwise 1x1, fused so the
// depthwise result stays on chip ("Kimi-K2.6__l1_p86": the per-output pseudo-code
// and the note that fusing avoids writing and re-reading the intermediate).
//
// FP32-FMA path: a CTA owns a 64 x 4 pixel tile and 32 output channels; each
// thread owns one pixel and 32 accumulators.  Input channels are staged 8 at a
// time as a zero-padded (4+K-1) x (64+K-1) halo (4-byte cp.async copies, the
// zero-fill is the padding); each thread forms its depthwise
// value for a channel in registers (K*K FMAs) and immediately feeds the 32
// pointwise FMAs, so the depthwise tensor never exists in memory.  The pointwise
// work is done once per output channel (no repeated pointwise products per tap).
// The depthwise size K (1, 3, 5, 7; "same" padding (K-1)/2) is a template
// parameter, the dispatch on the common sizes the same page discusses.
#include "ig3_internal.h"

namespace ig3 {
namespace {

constexpr int kTW = 64, kTH = 4, kCO = 32, kCC = 8, kThreads = 256;

template <int K>
__global__ void __launch_bounds__(kThreads) dwsep_fma_kernel(const float* __restrict__ x,
                                                             const float* __restrict__ w_dw,
                                                             const float* __restrict__ w_pw,
                                                             const float* __restrict__ bias, float* __restrict__ y,
                                                             int N, int C, int H, int W, int Cout) {
  constexpr int P = (K - 1) / 2;
  constexpr int kXW = kTW + K - 1, kXWPad = (kXW + 3) / 4 * 4, kXH = kTH + K - 1;
  __shared__ float s_x[kCC][kXH][kXWPad];
  __shared__ float s_dw[kCC][K * K];
  __shared__ __align__(16) float s_pw[kCC][kCO];

  const int tiles_w = (W + kTW - 1) / kTW;
  const int w0 = (blockIdx.x % tiles_w) * kTW;
  const int h0 = (blockIdx.x / tiles_w) * kTH;
  const int cgroups = (Cout + kCO - 1) / kCO;
  const int n = blockIdx.y / cgroups;
  const int co0 = (blockIdx.y % cgroups) * kCO;
  const int tid = threadIdx.x;
  const int px = tid % kTW, py = tid / kTW;

  float acc[kCO];
#pragma unroll
  for (int j = 0; j < kCO; ++j) acc[j] = 0.0f;

  const size_t plane = (size_t)H * W;
  for (int c0 = 0; c0 < C; c0 += kCC) {
    __syncthreads();
    // Halo rows (one index decomposition per row, a warp across its columns) and the
    // chunk's weights, as 4-byte asynchronous copies whose zero-fill is the padding;
    // all in flight before the one wait.
    for (int row = tid / 32; row < kCC * kXH; row += kThreads / 32) {
      const int c = row / kXH, yy = row % kXH;
      const int gc = c0 + c, gh = h0 + yy - P;
      const bool row_in = gc < C && gh >= 0 && gh < H;
      const float* src = row_in ? x + ((size_t)n * C + gc) * plane + (size_t)gh * W : x;
      for (int xx = tid % 32; xx < kXW; xx += 32) {
        const int gw = w0 + xx - P;
        const bool ok = row_in && gw >= 0 && gw < W;
        cp_async4(&s_x[c][yy][xx], ok ? src + gw : x, ok);
      }
    }
    for (int i = tid; i < kCC * K * K; i += kThreads) {
      const int c = i / (K * K), t = i % (K * K);
      const bool ok = c0 + c < C;
      cp_async4(&s_dw[c][t], ok ? &w_dw[(size_t)(c0 + c) * (K * K) + t] : w_dw, ok);
    }
    for (int i = tid; i < kCC * kCO; i += kThreads) {
      const int c = i / kCO, co = i % kCO;
      const bool ok = c0 + c < C && co0 + co < Cout;
      cp_async4(&s_pw[c][co], ok ? &w_pw[(size_t)(co0 + co) * C + c0 + c] : w_pw, ok);
    }
    cp_async_wait_all();
    __syncthreads();
#pragma unroll 2
    for (int c = 0; c < kCC; ++c) {
      float d = 0.0f;
#pragma unroll
      for (int kh = 0; kh < K; ++kh)
#pragma unroll
        for (int kw = 0; kw < K; ++kw) d = fmaf(s_x[c][py + kh][px + kw], s_dw[c][kh * K + kw], d);
#pragma unroll
      for (int j = 0; j < kCO; j += 4) {
        const float4 p = *reinterpret_cast<const float4*>(&s_pw[c][j]);
        acc[j] = fmaf(d, p.x, acc[j]);
        acc[j + 1] = fmaf(d, p.y, acc[j + 1]);
        acc[j + 2] = fmaf(d, p.z, acc[j + 2]);
        acc[j + 3] = fmaf(d, p.w, acc[j + 3]);
      }
    }
  }

  const int h = h0 + py, w = w0 + px;
  if (h >= H || w >= W) return;
#pragma unroll
  for (int j = 0; j < kCO; ++j) {
    const int co = co0 + j;
    if (co < Cout) y[((size_t)n * Cout + co) * plane + (size_t)h * W + w] = acc[j] + (bias ? __ldg(&bias[co]) : 0.0f);
  }
}

}  // namespace

int dwsep_fma_launch(const DwsepArgs& a) {
  const long long tiles = (long long)((a.W + kTW - 1) / kTW) * ((a.H + kTH - 1) / kTH);
  const long long zy = (long long)a.N * ((a.Cout + kCO - 1) / kCO);
  if (tiles > 0x7fffffffLL || zy > 65535) return fail(IG3_ERR_UNSUPPORTED, "dwsep FMA path: grid too large");
  const dim3 grid((unsigned)tiles, (unsigned)zy);
  switch (a.K) {
    case 1: dwsep_fma_kernel<1><<<grid, kThreads, 0, a.stream>>>(a.x, a.w_dw, a.w_pw, a.b, a.y, a.N, a.C, a.H, a.W, a.Cout); break;
    case 3: dwsep_fma_kernel<3><<<grid, kThreads, 0, a.stream>>>(a.x, a.w_dw, a.w_pw, a.b, a.y, a.N, a.C, a.H, a.W, a.Cout); break;
    case 5: dwsep_fma_kernel<5><<<grid, kThreads, 0, a.stream>>>(a.x, a.w_dw, a.w_pw, a.b, a.y, a.N, a.C, a.H, a.W, a.Cout); break;
    case 7: dwsep_fma_kernel<7><<<grid, kThreads, 0, a.stream>>>(a.x, a.w_dw, a.w_pw, a.b, a.y, a.N, a.C, a.H, a.W, a.Cout); break;
    default: return fail(IG3_ERR_UNSUPPORTED, "dwsep FMA path: depthwise size %d (1, 3, 5 or 7)", a.K);
  }
  return count_launch(cuda_status(cudaGetLastError(), "dwsep FMA kernel launch"));
}

}  // namespace ig3
