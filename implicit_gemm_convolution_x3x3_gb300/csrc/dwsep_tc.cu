// Depthwise 3x3 (stride 1, pad 1) -> pointwise 1x1 on sm_103a, fused in one kernel:
// the depthwise result goes from registers to shared memory and straight into a
// tcgen05 GEMM; it never reaches HBM ("Kimi-K2.6__l1_p86": the per-output
// pseudo-code, and the note that fusing removes the intermediate's write and read).
//
//   dw[n,c,h,w] = sum_{kh,kw<3} w_dw[c,kh,kw] * x[n,c,h+kh-1,w+kw-1]   (zero outside)
//   y[n,o,h,w]  = sum_c w_pw[o,c] * dw[n,c,h,w] (+ b[o])
//
// Tile = 128 consecutive pixels of one image row (GEMM M = 128, N = Cout, K = C).
// Persistent CTAs (one per SM, 416 threads) walk strips of rows, so the rows above
// and below a tile were read for the previous tile and come from L2, not HBM.
//   warp 0      TMEM owner and MMA issuer (one thread);
//   warps 1-8   depthwise: lane l owns pixels l, l+32, l+64, l+96 of 4 channels;
//               each input row is one coalesced load per 32 pixels, the left and
//               right neighbours come by warp shuffle; the 3x3 sums are split into
//               tf32 hi/lo and stored K-major [channel group][pixel][4], with
//               consecutive lanes writing consecutive 16-byte rows (no bank conflicts);
//   warps 9-12  epilogue: tcgen05.ld from a double-buffered TMEM accumulator,
//               + bias, one full 128-byte line per warp store.
// The pointwise weights are split into [hi ; lo] rows once per CTA and stay in
// shared memory; acc = A_hi*[B_hi|B_lo] + A_lo*B_hi (3xTF32, as in conv3d_tc.cu).
// With tensor cores doing the pointwise sums the kernel is bound by HBM traffic
// (read x once, write y once).  Every wait is bounded.
#include <algorithm>
#include <cstdio>
#include <cstring>

#include "ig3_internal.h"

namespace ig3 {
namespace {

constexpr int kThreads = 416;
constexpr int kDwWarp0 = 1, kDwThreads = 256;
constexpr int kEpiWarp0 = 9, kEpiThreads = 128;
constexpr int kRows = 8;        // image rows per work unit
constexpr int kTile = 128;      // pixels per tile
constexpr int kTmemCols = 512;

struct DwParams {
  const float* x;
  const float* w_dw;
  const float* w_pw;
  const float* bias;
  float* y;
  int N, C, H, W, Cout;
  int WB;         // tiles per image row
  int HR;         // row strips per image
  int units;
  int prefetch;   // rows start on 16-byte boundaries, so bulk L2 prefetches are legal
  uint32_t a_half_bytes, a_stage_bytes, off_b, off_wdw, off_bar;
  WaitCtl ctl;
};

struct Ring {
  uint32_t idx = 0, phase = 0;
  __device__ void next(uint32_t n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

__device__ __forceinline__ bool test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool wait_fast(uint64_t* bar, uint32_t parity, const WaitCtl& ctl, volatile int* abort) {
  if (test_wait(bar, parity)) return true;
  return mbar_wait_bounded(bar, parity, ctl, abort);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl, volatile int* abort) {
  const bool ok = wait_fast(bar, parity, ctl, abort);
  return __all_sync(0xffffffffu, ok) != 0;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) dwsep_tc_kernel(const DwParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + p.off_b;
  float* s_wdw = reinterpret_cast<float*>(smem + p.off_wdw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* a_full = bars;        // [2]
  uint64_t* a_empty = bars + 2;   // [2]
  uint64_t* acc_full = bars + 4;  // [2]
  uint64_t* acc_empty = bars + 6; // [2]
  uint64_t* mma_done = bars + 8;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &s_abort;
  const int C = p.C, Cout = p.Cout;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], kDwThreads);
      mbar_init(&a_empty[i], 1);
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiThreads);
    }
    mbar_init(mma_done, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  // Pointwise weights -> [K-step][k-half][2*Cout rows: hi, lo][4]; depthwise weights.
  {
    const int ks_n = C >> 3;
    const int total = ks_n * 2 * (2 * Cout) * 4;
    float* sb = reinterpret_cast<float*>(smem_b);
    for (int i = tid; i < total; i += kThreads) {
      const int j = i & 3;
      int r = i >> 2;
      const int row = r % (2 * Cout);
      r /= 2 * Cout;
      const int kh = r & 1;
      const int ks = r >> 1;
      const int c = ks * 8 + kh * 4 + j;
      const int co = row % Cout;
      float hi, lo;
      split_tf32(__ldg(&p.w_pw[(size_t)co * C + c]), hi, lo);
      sb[i] = (row < Cout) ? hi : lo;
    }
    for (int i = tid; i < C * 9; i += kThreads) s_wdw[i] = __ldg(&p.w_dw[i]);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  const int HW = p.H * p.W;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_cat = umma_idesc_tf32(128, 2 * Cout);
      const uint32_t idesc_one = umma_idesc_tf32(128, Cout);
      const uint64_t a_desc0 = umma_desc_noswizzle(smem_addr(smem_a), (uint32_t)kTile * 16u, 128);
      const uint64_t b_desc0 = umma_desc_noswizzle(smem_addr(smem_b), (uint32_t)(2 * Cout) * 16u, 128);
      const uint32_t a_stage_u = p.a_stage_bytes >> 4, a_half_u = p.a_half_bytes >> 4;
      const uint32_t ks_a_u = 2u * kTile;            // two channel groups of 128 rows
      const uint32_t ks_b_u = (uint32_t)(4 * Cout);  // one B block: 2 halves x 2*Cout rows x 16 B
      const int ks_n = C >> 3;
      Ring ra, racc;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        const int hr = u % p.HR;
        const int h0 = hr * kRows, h1 = min(p.H, h0 + kRows);
        for (int h = h0; ok && h < h1; ++h) {
          if (!(ok = wait_fast(&a_full[ra.idx], ra.phase, p.ctl, abort_flag))) break;
          if (!(ok = wait_fast(&acc_empty[racc.idx], racc.phase ^ 1u, p.ctl, abort_flag))) break;
          tc_fence_after();
          const uint64_t ah = a_desc0 + (uint64_t)(ra.idx * a_stage_u);
          const uint64_t al = ah + a_half_u;
          const uint32_t d = tmem_base + racc.idx * (uint32_t)(2 * Cout);
          for (int ks = 0; ks < ks_n; ++ks) {
            const uint64_t ko = (uint64_t)((uint32_t)ks * ks_a_u);
            const uint64_t bh = b_desc0 + (uint64_t)((uint32_t)ks * ks_b_u);
            umma_tf32(d, ah + ko, bh, idesc_cat, ks > 0 ? 1u : 0u);
            umma_tf32(d, al + ko, bh, idesc_one, 1u);
          }
          umma_commit(&a_empty[ra.idx]);
          umma_commit(&acc_full[racc.idx]);
          ra.next(2);
          racc.next(2);
        }
      }
      umma_commit(mma_done);
      int never = 0;
      mbar_wait_bounded(mma_done, 0, p.ctl, &never);
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ depthwise
    const int wd = warp - kDwWarp0;  // 0..7
    const int groups = C >> 2;
    Ring ra;
    for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
      const int hr = u % p.HR;
      const int wb = (u / p.HR) % p.WB;
      const int n = u / (p.HR * p.WB);
      const int w0 = wb * kTile;
      const int h0 = hr * kRows, h1 = min(p.H, h0 + kRows);
      for (int h = h0; h < h1; ++h) {
        if (!warp_wait(&a_empty[ra.idx], ra.phase ^ 1u, p.ctl, abort_flag)) goto dw_done;
        const uint32_t hi_base = smem_addr(smem_a) + ra.idx * p.a_stage_bytes;
        const uint32_t lo_base = hi_base + p.a_half_bytes;
        // Ask L2 now for the row the next tile reads first (h + 2), so its loads hit
        // L2 instead of waiting on HBM: one 512-byte bulk prefetch per channel.
        if (p.prefetch && h + 2 < p.H && lane < 8 && w0 + kTile <= p.W) {
          const int g = wd + 8 * (lane >> 2);
          if (g < groups) {
            const float* src = p.x + ((size_t)n * C + g * 4 + (lane & 3)) * HW + (size_t)(h + 2) * p.W + w0;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"((uint32_t)kTile * 4u)
                         : "memory");
          }
        }
        for (int g = wd; g < groups; g += 8) {
          // All 12 rows (4 channels x 3 image rows) of the group are loaded first so
          // their latencies overlap; rows outside the image read as zeros (padding).
          // edge[c][dr]: lane 0 holds pixel w0 - 1 and lane 31 pixel w0 + 128 (one load
          // instruction for both ends of the row segment; other lanes hold zero).
          float v[4][3][4], edge[4][3];
          const bool edge_lane = (lane == 0) ? (w0 > 0) : (lane == 31 && w0 + kTile < p.W);
          const int edge_off = (lane == 0) ? -1 : kTile;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float* xc = p.x + ((size_t)n * C + g * 4 + c) * HW;
#pragma unroll
            for (int dr = 0; dr < 3; ++dr) {
              const int hh = h + dr - 1;
              const bool rv = (hh >= 0 && hh < p.H);
              const float* row = xc + (size_t)(rv ? hh : 0) * p.W + w0;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                v[c][dr][k] = (rv && w0 + lane + 32 * k < p.W) ? __ldg(row + lane + 32 * k) : 0.0f;
              edge[c][dr] = (rv && edge_lane) ? __ldg(row + edge_off) : 0.0f;
            }
          }
          float acc[4][4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[k][c] = 0.0f;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int ch = g * 4 + c;
#pragma unroll
            for (int dr = 0; dr < 3; ++dr) {
              const float k0 = s_wdw[ch * 9 + dr * 3 + 0];
              const float k1 = s_wdw[ch * 9 + dr * 3 + 1];
              const float k2 = s_wdw[ch * 9 + dr * 3 + 2];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                // One rotate per direction: lane 31 offers the last pixel of the previous
                // 32-pixel chunk (or the left edge) for lane 0's left neighbour, and lane 0
                // offers the first pixel of the next chunk (or the right edge) for lane 31.
                const float x0 = v[c][dr][k];
                // Edge pixels: lane 0's left end (held by lane 0) and lane 31's right end
                // (held by lane 31) are used by the same lane, so they bypass the shuffle.
                const float lsrc = (lane == 31) ? (k > 0 ? v[c][dr][k > 0 ? k - 1 : 0] : 0.0f) : x0;
                const float rsrc = (lane == 0) ? (k < 3 ? v[c][dr][k < 3 ? k + 1 : 3] : 0.0f) : x0;
                float left = __shfl_sync(0xffffffffu, lsrc, (lane + 31) & 31);
                float right = __shfl_sync(0xffffffffu, rsrc, (lane + 1) & 31);
                if (k == 0 && lane == 0) left = edge[c][dr];
                if (k == 3 && lane == 31) right = edge[c][dr];
                acc[k][c] = fmaf(k0, left, fmaf(k1, x0, fmaf(k2, right, acc[k][c])));
              }
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t off = (uint32_t)(g * kTile + lane + 32 * k) * 16u;
            float hi[4], lo[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) split_tf32(acc[k][c], hi[c], lo[c]);
            st_shared_v4(hi_base + off, hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(lo_base + off, lo[0], lo[1], lo[2], lo[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&a_full[ra.idx]);
        ra.next(2);
      }
    }
  dw_done:;
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant
    const int px = q * 32 + lane;
    Ring racc;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      const int hr = u % p.HR;
      const int wb = (u / p.HR) % p.WB;
      const int n = u / (p.HR * p.WB);
      const int w = wb * kTile + px;
      const int h0 = hr * kRows, h1 = min(p.H, h0 + kRows);
      for (int h = h0; h < h1; ++h) {
        if (!(ok = warp_wait(&acc_full[racc.idx], racc.phase, p.ctl, abort_flag))) break;
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + racc.idx * (uint32_t)(2 * Cout);
        float* yb = p.y + (size_t)n * Cout * HW + (size_t)h * p.W + w;
        for (int c0 = 0; c0 < Cout; c0 += 16) {
          float v[16], v2[16];
          tmem_ld16(tb + c0, v);
          tmem_ld16(tb + Cout + c0, v2);
          tmem_wait_ld();
          if (w < p.W) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              yb[(size_t)(c0 + j) * HW] = v[j] + v2[j] + (p.bias ? __ldg(&p.bias[c0 + j]) : 0.0f);
          }
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[racc.idx]);
        racc.next(2);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

struct DwPlan {
  bool ok = false;
  const char* why = "";
  DwParams prm;
  size_t smem = 0;
};

DwPlan make_dw_plan(int N, int C, int H, int W, int Cout) {
  DwPlan pl;
  DwParams& p = pl.prm;
  std::memset(&p, 0, sizeof(p));
  if (C % 8 != 0 || C > 64) {
    pl.why = "C must be a multiple of 8 and at most 64";
    return pl;
  }
  if (Cout % 16 != 0 || Cout > 128) {
    pl.why = "Cout must be a multiple of 16 and at most 128";
    return pl;
  }
  p.N = N; p.C = C; p.H = H; p.W = W; p.Cout = Cout;
  p.WB = (W + kTile - 1) / kTile;
  p.HR = (H + kRows - 1) / kRows;
  const long long units = (long long)N * p.WB * p.HR;
  if (units > 0x7fffffffLL) {
    pl.why = "too many tiles";
    return pl;
  }
  p.units = (int)units;
  p.a_half_bytes = (uint32_t)(C / 4) * kTile * 16u;
  p.a_stage_bytes = 2 * p.a_half_bytes;
  p.off_b = 2 * p.a_stage_bytes;
  const uint32_t b_bytes = (uint32_t)(C / 8) * 2u * (2u * Cout) * 16u;
  p.off_wdw = p.off_b + b_bytes;
  p.off_bar = (p.off_wdw + (uint32_t)C * 9u * 4u + 127) / 128 * 128;
  pl.smem = p.off_bar + 16 * 8;
  if (pl.smem + 2048 > (size_t)(227 * 1024)) {
    pl.why = "does not fit in shared memory";
    return pl;
  }
  pl.smem = std::max(pl.smem, (size_t)(116 * 1024));  // one CTA (one TMEM owner) per SM
  pl.ok = true;
  return pl;
}

}  // namespace

const char* dwsep_tc_unsupported_reason(int N, int C, int H, int W, int Cout) {
  static thread_local char buf[128];
  DwPlan pl = make_dw_plan(N, C, H, W, Cout);
  if (pl.ok) return "";
  snprintf(buf, sizeof(buf), "%s", pl.why);
  return buf;
}

int dwsep_tc_launch(const DwsepArgs& a) {
  const int sms = num_sms();
  if (sms <= 0) return fail(IG3_ERR_CUDA, "dwsep TC path: cannot query the SM count");
  DwPlan pl = make_dw_plan(a.N, a.C, a.H, a.W, a.Cout);
  if (!pl.ok) return fail(IG3_ERR_UNSUPPORTED, "dwsep TC path: %s", pl.why);
  DwParams p = pl.prm;
  p.x = a.x;
  p.w_dw = a.w_dw;
  p.w_pw = a.w_pw;
  p.bias = a.b;
  p.y = a.y;
  p.prefetch = (a.W % 4 == 0) && (reinterpret_cast<uintptr_t>(a.x) % 16 == 0);
  p.ctl = wait_ctl();
  if (!p.ctl.status) return fail(IG3_ERR_CUDA, "dwsep TC path: device status word unavailable");
  cudaError_t e = cudaFuncSetAttribute(dwsep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return cuda_status(e, "dwsep TC: set shared memory size");
  const int grid = std::min(p.units, sms);
  dwsep_tc_kernel<<<grid, kThreads, pl.smem, a.stream>>>(p);
  return count_launch(cuda_status(cudaGetLastError(), "dwsep TC kernel launch"));
}

}  // namespace ig3
