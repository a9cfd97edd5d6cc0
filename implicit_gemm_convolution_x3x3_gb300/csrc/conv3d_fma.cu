// Register-blocked FP32-FMA direct conv3d (valid, stride 1, 3x3x3) with the fused
// epilogues.  This is the small-channel path and the reference point for the
// tensor-core path.
//
// Definition followed ("Kimi-K2.6__l2_p47", the per-output loop and its NCDHW index
// check):  conv[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw] x[n,c,od+kd,oh+kh,ow+kw].
//
// CTA tile: 2 output planes x 8 rows x 32 columns x 16 output channels, 128 threads.
// Thread (tx, ty, cg): columns 4tx..4tx+3, rows 2ty..2ty+1, both planes, channels
// 4cg..4cg+3 -> 64 accumulators.  A warp is one channel group, so its weight reads
// are shared-memory broadcasts; its input reads are float4 rows (conflict free).
// Input channels are staged 4 at a time: a (2+2) x (8+2) x (32+2) halo per channel.
// With zero padding P (the padding discussion of the same page: input coordinate
// od + kd - P, zero outside x, output D + 2P - 2) the staging reads the halo at the
// shifted coordinates and writes zeros outside x; nothing else changes.
//
// The 2x2x2 output block of a thread is exactly one pooling window per column pair,
// so the pool-reduce epilogue ("Kimi-K2.6__l2_p8": /2, MaxPool3d(2), global mean,
// +bias, sum over channels) needs no data exchange before the block-level sum.
#include <cstdio>

#include "ig3_internal.h"

namespace ig3 {
namespace {

constexpr int kTW = 32, kTH = 8, kTD = 2, kTCO = 16, kCC = 4, kThreads = 128;
constexpr int kInW = kTW + 2, kInWPad = 36, kInH = kTH + 2, kInD = kTD + 2;

template <int EPI>
__global__ void __launch_bounds__(kThreads) conv3d_fma_kernel(
    const float* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
    float* __restrict__ y, float* __restrict__ partial, int N, int Cin, int D, int H, int W, int P, int Cout,
    float inv_div) {
  __shared__ __align__(16) float s_in[kCC][kInD][kInH][kInWPad];
  __shared__ __align__(16) float s_w[kCC][27][kTCO];

  // Zero padding P: output od reads input planes od + kd - P (zero outside x).
  const int OD = D + 2 * P - 2, OH = H + 2 * P - 2, OW = W + 2 * P - 2;
  const int tiles_w = (OW + kTW - 1) / kTW;
  const int ow0 = (blockIdx.x % tiles_w) * kTW;
  const int oh0 = (blockIdx.x / tiles_w) * kTH;
  const int od0 = blockIdx.y * kTD;
  const int cgroups = (Cout + kTCO - 1) / kTCO;
  const int n = blockIdx.z / cgroups;
  const int co0 = (blockIdx.z % cgroups) * kTCO;
  const int tid = threadIdx.x;
  const int tx = tid & 7, ty = (tid >> 3) & 3, cg = tid >> 5;

  float acc[kTD][2][4][4];
#pragma unroll
  for (int p = 0; p < kTD; ++p)
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[p][q][i][j] = 0.0f;

  const size_t plane = (size_t)H * W;
  for (int c0 = 0; c0 < Cin; c0 += kCC) {
    __syncthreads();
    for (int i = tid; i < kCC * kInD * kInH * kInW; i += kThreads) {
      const int xw = i % kInW;
      int r = i / kInW;
      const int xh = r % kInH;
      r /= kInH;
      const int xd = r % kInD;
      const int c = r / kInD;
      const int gc = c0 + c, gd = od0 + xd - P, gh = oh0 + xh - P, gw = ow0 + xw - P;
      float v = 0.0f;
      if (gc < Cin && (unsigned)gd < (unsigned)D && (unsigned)gh < (unsigned)H && (unsigned)gw < (unsigned)W)
        v = __ldg(&x[((size_t)n * Cin + gc) * D * plane + (size_t)gd * plane + (size_t)gh * W + gw]);
      s_in[c][xd][xh][xw] = v;
    }
    for (int i = tid; i < kCC * 27 * kTCO; i += kThreads) {
      const int co = i % kTCO;
      const int r = i / kTCO;
      const int tap = r % 27;
      const int c = r / 27;
      const int gco = co0 + co, gc = c0 + c;
      s_w[c][tap][co] = (gco < Cout && gc < Cin) ? __ldg(&w[((size_t)gco * Cin + gc) * 27 + tap]) : 0.0f;
    }
    __syncthreads();

#pragma unroll 1
    for (int c = 0; c < kCC; ++c) {
#pragma unroll
      for (int dz = 0; dz < kInD; ++dz) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float* src = &s_in[c][dz][ty * 2 + r][tx * 4];
          const float4 v03 = *reinterpret_cast<const float4*>(src);
          const float2 v45 = *reinterpret_cast<const float2*>(src + 4);
          const float v[6] = {v03.x, v03.y, v03.z, v03.w, v45.x, v45.y};
#pragma unroll
          for (int p = 0; p < kTD; ++p) {
            const int kd = dz - p;
            if (kd < 0 || kd > 2) continue;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int kh = r - q;
              if (kh < 0 || kh > 2) continue;
#pragma unroll
              for (int kw = 0; kw < 3; ++kw) {
                const float4 wv = *reinterpret_cast<const float4*>(&s_w[c][(kd * 3 + kh) * 3 + kw][cg * 4]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  acc[p][q][i][0] = fmaf(v[i + kw], wv.x, acc[p][q][i][0]);
                  acc[p][q][i][1] = fmaf(v[i + kw], wv.y, acc[p][q][i][1]);
                  acc[p][q][i][2] = fmaf(v[i + kw], wv.z, acc[p][q][i][2]);
                  acc[p][q][i][3] = fmaf(v[i + kw], wv.w, acc[p][q][i][3]);
                }
              }
            }
          }
        }
      }
    }
  }

  if constexpr (EPI == IG3_EPI_POOL_REDUCE) {
    // One window per (channel, column pair): planes od0..od0+1, rows oh..oh+1, 2 columns.
    const int PD = OD / 2, PH = OH / 2, PW = OW / 2;
    const int pd = od0 / 2, ph = (oh0 + 2 * ty) / 2;
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int co = co0 + cg * 4 + j;
      if (co >= Cout) continue;
      const float bj = bias ? __ldg(&bias[co]) : 0.0f;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int pw = (ow0 + 4 * tx) / 2 + k;
        if (pd < PD && ph < PH && pw < PW) {
          float m = -INFINITY;
#pragma unroll
          for (int p = 0; p < 2; ++p)
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
              for (int e = 0; e < 2; ++e) m = fmaxf(m, (acc[p][q][2 * k + e][j] + bj) * inv_div);
          s += m;
        }
      }
    }
    // Fixed-order block reduction: warp butterfly, then warps 0..3 in order.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    __shared__ float s_red[kThreads / 32];
    if ((tid & 31) == 0) s_red[tid >> 5] = s;
    __syncthreads();
    if (tid == 0) {
      float t = 0.0f;
      for (int i = 0; i < kThreads / 32; ++i) t += s_red[i];
      partial[((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x] = t;
    }
  } else {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int co = co0 + cg * 4 + j;
    if (co >= Cout) continue;
    const float bj = bias ? __ldg(&bias[co]) : 0.0f;
#pragma unroll
    for (int p = 0; p < kTD; ++p) {
      const int od = od0 + p;
      if (od >= OD) continue;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int oh = oh0 + 2 * ty + q;
        if (oh >= OH) continue;
        float* dst = y + (((size_t)n * Cout + co) * OD + od) * ((size_t)OH * OW) + (size_t)oh * OW;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ow = ow0 + 4 * tx + i;
          if (ow >= OW) continue;
          float v = acc[p][q][i][j] + bj;
          if (EPI == IG3_EPI_TANH_MISH) v = tanh_mish(v);
          dst[ow] = v;
        }
      }
    }
  }
  }
}

// out[n] = scale * sum(partial[n*per_n ..]) + sum_c bias2[c], fixed order.
__global__ void __launch_bounds__(256) pool_reduce_finalize_kernel(const float* __restrict__ partial, int per_n,
                                                                   float scale, const float* __restrict__ bias2,
                                                                   int C, float* __restrict__ out) {
  __shared__ float s_red[256];
  const int n = blockIdx.x;
  float s = 0.0f;
  for (int i = threadIdx.x; i < per_n; i += 256) s += partial[(size_t)n * per_n + i];
  s_red[threadIdx.x] = s;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) s_red[threadIdx.x] += s_red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    float bs = 0.0f;
    for (int c = 0; c < C; ++c) bs += bias2[c];
    out[n] = s_red[0] * scale + bs;
  }
}

dim3 fma_grid(const Conv3dArgs& a) {
  const int tiles = ((a.OW() + kTW - 1) / kTW) * ((a.OH() + kTH - 1) / kTH);
  const int planes = (a.OD() + kTD - 1) / kTD;
  const int cgroups = (a.Cout + kTCO - 1) / kTCO;
  return dim3(tiles, planes, a.N * cgroups);
}

}  // namespace

size_t conv3d_fma_workspace(const Conv3dArgs& a) {
  if (a.epi != IG3_EPI_POOL_REDUCE) return 0;
  const dim3 g = fma_grid(a);
  return align_up((size_t)g.x * g.y * g.z * sizeof(float), 256);
}

int conv3d_fma_launch(const Conv3dArgs& a) {
  const dim3 g = fma_grid(a);
  if (g.y > 65535u || g.z > 65535u) return fail(IG3_ERR_UNSUPPORTED, "conv3d FMA path: grid too large");
  const float inv_div = (a.epi == IG3_EPI_POOL_REDUCE) ? 1.0f / a.divisor : 1.0f;
  float* partial = static_cast<float*>(a.ws);
  switch (a.epi) {
    case IG3_EPI_NONE:
      conv3d_fma_kernel<IG3_EPI_NONE><<<g, kThreads, 0, a.stream>>>(a.x, a.w, a.b, a.y, nullptr, a.N, a.Cin, a.D,
                                                                    a.H, a.W, a.pad, a.Cout, inv_div);
      break;
    case IG3_EPI_TANH_MISH:
      conv3d_fma_kernel<IG3_EPI_TANH_MISH><<<g, kThreads, 0, a.stream>>>(a.x, a.w, a.b, a.y, nullptr, a.N, a.Cin,
                                                                         a.D, a.H, a.W, a.pad, a.Cout, inv_div);
      break;
    default:
      conv3d_fma_kernel<IG3_EPI_POOL_REDUCE><<<g, kThreads, 0, a.stream>>>(a.x, a.w, a.b, nullptr, partial, a.N,
                                                                           a.Cin, a.D, a.H, a.W, a.pad, a.Cout, inv_div);
      break;
  }
  int st = count_launch(cuda_status(cudaGetLastError(), "conv3d FMA kernel launch"));
  if (st != IG3_OK || a.epi != IG3_EPI_POOL_REDUCE) return st;
  const int per_n = (int)(g.x * g.y * (g.z / a.N));
  const long long cells = (long long)(a.OD() / 2) * (a.OH() / 2) * (a.OW() / 2);
  return pool_reduce_finalize(partial, a.N, per_n, (float)(1.0 / (double)cells), a.bias2, a.Cout, a.y, a.stream);
}

int pool_reduce_finalize(const float* partial, int N, int per_n, float scale, const float* bias2, int C, float* out,
                         cudaStream_t stream) {
  pool_reduce_finalize_kernel<<<N, 256, 0, stream>>>(partial, per_n, scale, bias2, C, out);
  return count_launch(cuda_status(cudaGetLastError(), "pool-reduce finalize launch"));
}

}  // namespace ig3
