// Depthwise 3x3 (stride 1, pad 1) followed by pointwise 1x1, fused so the
// depthwise result stays on chip ("Kimi-K2.6__l1_p86": the per-output pseudo-code
// and the note that fusing avoids writing and re-reading the intermediate).
//
// FP32-FMA path: a CTA owns a 64 x 4 pixel tile and 32 output channels; each
// thread owns one pixel and 32 accumulators.  Input channels are staged 8 at a
// time as a zero-padded (4+2) x (64+2) halo; each thread forms its depthwise value
// for a channel in registers (9 FMAs) and immediately feeds the 32 pointwise FMAs,
// so the depthwise tensor never exists in memory.  The pointwise work is done
// once per output channel (no repeated pointwise products per tap).
#include "ig3_internal.h"

namespace ig3 {
namespace {

constexpr int kTW = 64, kTH = 4, kCO = 32, kCC = 8, kThreads = 256;
constexpr int kXW = kTW + 2, kXWPad = 68, kXH = kTH + 2;

__global__ void __launch_bounds__(kThreads) dwsep_fma_kernel(const float* __restrict__ x,
                                                             const float* __restrict__ w_dw,
                                                             const float* __restrict__ w_pw,
                                                             const float* __restrict__ bias, float* __restrict__ y,
                                                             int N, int C, int H, int W, int Cout) {
  __shared__ float s_x[kCC][kXH][kXWPad];
  __shared__ float s_dw[kCC][9];
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
    for (int i = tid; i < kCC * kXH * kXW; i += kThreads) {
      const int xx = i % kXW;
      const int r = i / kXW;
      const int yy = r % kXH;
      const int c = r / kXH;
      const int gc = c0 + c, gh = h0 + yy - 1, gw = w0 + xx - 1;
      float v = 0.0f;
      if (gc < C && gh >= 0 && gh < H && gw >= 0 && gw < W)
        v = __ldg(&x[((size_t)n * C + gc) * plane + (size_t)gh * W + gw]);
      s_x[c][yy][xx] = v;
    }
    for (int i = tid; i < kCC * 9; i += kThreads) {
      const int c = i / 9, t = i % 9;
      s_dw[c][t] = (c0 + c < C) ? __ldg(&w_dw[(size_t)(c0 + c) * 9 + t]) : 0.0f;
    }
    for (int i = tid; i < kCC * kCO; i += kThreads) {
      const int c = i / kCO, co = i % kCO;
      s_pw[c][co] = (c0 + c < C && co0 + co < Cout) ? __ldg(&w_pw[(size_t)(co0 + co) * C + c0 + c]) : 0.0f;
    }
    __syncthreads();
#pragma unroll 2
    for (int c = 0; c < kCC; ++c) {
      float d = 0.0f;
#pragma unroll
      for (int kh = 0; kh < 3; ++kh)
#pragma unroll
        for (int kw = 0; kw < 3; ++kw) d = fmaf(s_x[c][py + kh][px + kw], s_dw[c][kh * 3 + kw], d);
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
  dwsep_fma_kernel<<<dim3((unsigned)tiles, (unsigned)zy), kThreads, 0, a.stream>>>(a.x, a.w_dw, a.w_pw, a.b, a.y,
                                                                                   a.N, a.C, a.H, a.W, a.Cout);
  return count_launch(cuda_status(cudaGetLastError(), "dwsep FMA kernel launch"));
}

}  // namespace ig3
