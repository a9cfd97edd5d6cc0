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

// Two-phase form for the larger depthwise sizes (K = 5, 7), where recomputing the K*K
// depthwise sum for every group of output channels and reading it tap by tap from
// shared memory would cost more than the pointwise work: per channel chunk the CTA
// first forms the depthwise values of its 64 x 4 pixels once (a thread: 4 adjacent
// pixels of one row for 2 channels, the input row read as float4 and slid across the
// K taps) into shared memory, then each thread takes one pixel for 64 output channels
// (one depthwise read and sixteen broadcast float4 weight reads per channel for 64 FMAs).
// Two stages of copies: the next chunk's fly while this one is computed.
constexpr int k2CO = 64;

// Shared-memory layout of the two-phase kernel: two stages (input halo, depthwise
// weights, pointwise weights of one channel chunk), then the depthwise results.
template <int K>
struct Fma2Smem {
  static constexpr int XW = kTW + K - 1;
  static constexpr int RowV = (K + 3 + 3) / 4;  // float4 reads per input row (4 pixels + K - 1)
  static constexpr int XWPad = (XW + 3) / 4 * 4 + (4 * RowV > K + 3 ? 4 : 0);
  static constexpr int XH = kTH + K - 1;
  static constexpr int x_floats = kCC * XH * XWPad;
  static constexpr int dw_floats = (kCC * K * K + 3) / 4 * 4;
  static constexpr int pw_floats = kCC * k2CO;
  static constexpr int stage_floats = x_floats + dw_floats + pw_floats;
  static constexpr int d_floats = kCC * kTH * kTW;
  static constexpr size_t bytes = (size_t)(2 * stage_floats + d_floats) * sizeof(float);
  static_assert(x_floats % 4 == 0 && stage_floats % 4 == 0, "float4 reads stay 16-byte aligned");
  static_assert(4 * (kTW / 4 - 1) + 4 * RowV <= XWPad, "row reads stay inside the padded halo row");
};

template <int K>
__global__ void __launch_bounds__(kThreads) dwsep_fma2_kernel(const float* __restrict__ x,
                                                              const float* __restrict__ w_dw,
                                                              const float* __restrict__ w_pw,
                                                              const float* __restrict__ bias, float* __restrict__ y,
                                                              int N, int C, int H, int W, int Cout) {
  using L = Fma2Smem<K>;
  constexpr int P = (K - 1) / 2;
  extern __shared__ __align__(16) float smem[];
  float* s_d = smem + 2 * L::stage_floats;  // [kCC][kTH][kTW]

  const int tiles_w = (W + kTW - 1) / kTW;
  const int w0 = (blockIdx.x % tiles_w) * kTW;
  const int h0 = (blockIdx.x / tiles_w) * kTH;
  const int cgroups = (Cout + k2CO - 1) / k2CO;
  const int n = blockIdx.y / cgroups;
  const int co0 = (blockIdx.y % cgroups) * k2CO;
  const int tid = threadIdx.x;
  const int px = tid % kTW, py = tid / kTW;                               // phase 2
  const int g = tid % 16, r1 = (tid / 16) % kTH, cp = tid / (16 * kTH);   // phase 1
  const size_t plane = (size_t)H * W;

  // Copies of the chunk starting at channel c0 into stage st (zero-fill = padding).
  auto stage_in = [&](int c0, int st) {
    float* s_x = smem + st * L::stage_floats;
    float* s_dw = s_x + L::x_floats;
    float* s_pw = s_dw + L::dw_floats;
    for (int row = tid / 32; row < kCC * L::XH; row += kThreads / 32) {
      const int c = row / L::XH, yy = row % L::XH;
      const int gc = c0 + c, gh = h0 + yy - P;
      const bool row_in = gc < C && gh >= 0 && gh < H;
      const float* src = row_in ? x + ((size_t)n * C + gc) * plane + (size_t)gh * W : x;
      for (int xx = tid % 32; xx < L::XW; xx += 32) {
        const int gw = w0 + xx - P;
        const bool ok = row_in && gw >= 0 && gw < W;
        cp_async4(s_x + row * L::XWPad + xx, ok ? src + gw : x, ok);
      }
    }
    for (int i = tid; i < kCC * K * K; i += kThreads) {
      const int c = i / (K * K), t = i % (K * K);
      const bool ok = c0 + c < C;
      cp_async4(s_dw + i, ok ? &w_dw[(size_t)(c0 + c) * (K * K) + t] : w_dw, ok);
    }
    for (int i = tid; i < kCC * k2CO; i += kThreads) {
      const int c = i / k2CO, co = i % k2CO;
      const bool ok = c0 + c < C && co0 + co < Cout;
      cp_async4(s_pw + i, ok ? &w_pw[(size_t)(co0 + co) * C + c0 + c] : w_pw, ok);
    }
    cp_async_commit();
  };

  float acc[k2CO];
#pragma unroll
  for (int j = 0; j < k2CO; ++j) acc[j] = 0.0f;

  stage_in(0, 0);
  for (int c0 = 0, st = 0; c0 < C; c0 += kCC, st ^= 1) {
    if (c0 + kCC < C) {
      stage_in(c0 + kCC, st ^ 1);  // that stage was last read before the barrier ending c0 - kCC
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const float* s_x = smem + st * L::stage_floats;
    const float* s_dw = s_x + L::x_floats;
    const float* s_pw = s_dw + L::dw_floats;
    // Phase 1: depthwise values of 4 adjacent pixels, channels 2cp and 2cp + 1.
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * cp + cc;
      float dv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kh = 0; kh < K; ++kh) {
        float row[4 * L::RowV];
        const float* xr = s_x + (c * L::XH + r1 + kh) * L::XWPad + 4 * g;
#pragma unroll
        for (int v = 0; v < L::RowV; ++v) {
          const float4 q = *reinterpret_cast<const float4*>(xr + 4 * v);
          row[4 * v] = q.x; row[4 * v + 1] = q.y; row[4 * v + 2] = q.z; row[4 * v + 3] = q.w;
        }
#pragma unroll
        for (int kw = 0; kw < K; ++kw) {
          const float wv = s_dw[c * K * K + kh * K + kw];
#pragma unroll
          for (int j = 0; j < 4; ++j) dv[j] = fmaf(row[j + kw], wv, dv[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) s_d[(c * kTH + r1) * kTW + 4 * g + j] = dv[j];
    }
    __syncthreads();
    // Phase 2: the pointwise products of this thread's pixel.
#pragma unroll 2
    for (int c = 0; c < kCC; ++c) {
      const float d = s_d[(c * kTH + py) * kTW + px];
#pragma unroll
      for (int j = 0; j < k2CO; j += 4) {
        const float4 p = *reinterpret_cast<const float4*>(s_pw + c * k2CO + j);
        acc[j] = fmaf(d, p.x, acc[j]);
        acc[j + 1] = fmaf(d, p.y, acc[j + 1]);
        acc[j + 2] = fmaf(d, p.z, acc[j + 2]);
        acc[j + 3] = fmaf(d, p.w, acc[j + 3]);
      }
    }
    __syncthreads();  // stage st and s_d are rewritten on the next iterations
  }

  const int h = h0 + py, w = w0 + px;
  if (h >= H || w >= W) return;
#pragma unroll
  for (int j = 0; j < k2CO; ++j) {
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
  const long long zy2 = (long long)a.N * ((a.Cout + k2CO - 1) / k2CO);
  const dim3 grid2((unsigned)tiles, (unsigned)zy2);
  switch (a.K) {
    case 1: dwsep_fma_kernel<1><<<grid, kThreads, 0, a.stream>>>(a.x, a.w_dw, a.w_pw, a.b, a.y, a.N, a.C, a.H, a.W, a.Cout); break;
    case 3: dwsep_fma_kernel<3><<<grid, kThreads, 0, a.stream>>>(a.x, a.w_dw, a.w_pw, a.b, a.y, a.N, a.C, a.H, a.W, a.Cout); break;
    case 5:
    case 7: {
      auto go = [&](auto kernel, size_t smem) -> int {
        const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_status(e, "dwsep FMA path: set shared memory size");
        kernel<<<grid2, kThreads, smem, a.stream>>>(a.x, a.w_dw, a.w_pw, a.b, a.y, a.N, a.C, a.H, a.W, a.Cout);
        return IG3_OK;
      };
      const int st = a.K == 5 ? go(dwsep_fma2_kernel<5>, Fma2Smem<5>::bytes) : go(dwsep_fma2_kernel<7>, Fma2Smem<7>::bytes);
      if (st != IG3_OK) return st;
      break;
    }
    default: return fail(IG3_ERR_UNSUPPORTED, "dwsep FMA path: depthwise size %d (1, 3, 5 or 7)", a.K);
  }
  return count_launch(cuda_status(cudaGetLastError(), "dwsep FMA kernel launch"));
}

}  // namespace ig3
