// Depthwise 3x3 (stride 1, pad 1) -> pointwise 1x1 on sm_103a, fused in one kernel:
// the depthwise result goes from registers into tensor memory and straight into a
// tcgen05 GEMM; it never reaches HBM ("Kimi-K2.6__l1_p86": the per-output
// pseudo-code, and the note that fusing removes the intermediate's write and read).
//
//   dw[n,c,h,w] = sum_{kh,kw<3} w_dw[c,kh,kw] * x[n,c,h+kh-1,w+kw-1]   (zero outside)
//   y[n,o,h,w]  = sum_c w_pw[o,c] * dw[n,c,h,w] (+ b[o])
//
// Tile = 128 consecutive pixels of one image row (GEMM M = 128, N = Cout, K = C).
// A work unit is a strip of R rows of one 128-pixel column segment; persistent CTAs
// (one per SM, 448 threads) walk units.
//   warp 0      TMEM owner and MMA issuer (one thread);
//   warp 1      row loader (one thread): each input row the strip needs (rows h0-1 ..
//               h0+R) as one tensor-map bulk copy of [C channels][136 pixels]
//               (pixels w0-4 .. w0+131) into a ring of four shared-memory row slots;
//               rows or pixels outside the image come back as zeros, which is the
//               padding;
//   warps 2-9   depthwise: lane = pixel (TMEM lane = GEMM row), two warps per TMEM
//               lane quadrant, each taking half of the channels.  A sliding
//               window over rows: each staged input row is read once (three values
//               per pixel and channel) and feeds the three output rows it belongs to
//               (kernel rows 2, 1, 0 of output rows r-1, r, r+1), whose partial sums
//               the lane keeps in registers; when row r arrives output row r-1 is
//               complete, split into tf32 hi/lo and written to tensor memory as the
//               GEMM's A operand;
//   warps 10-13 epilogue: tcgen05.ld of a double-buffered accumulator, + bias, one
//               128-byte line per warp store.
// Tensor memory: accumulators at columns [0, 2*Cout), A tiles (hi | lo, C columns
// each, double-buffered) at [256, 256 + 4*C).  The pointwise weights are split into
// [hi ; lo] rows once per CTA and stay in shared memory; the GEMM takes A from tensor
// memory and B from shared memory: acc = A_hi*B_hi + A_hi*B_lo + A_lo*B_hi (3xTF32, as
// in conv3d_tc.cu), three MMAs of N = Cout per 8 channels.  The kernel is meant to be
// bound by HBM traffic (read x once, write y once).  Every wait is bounded.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "ig3_internal.h"

namespace ig3 {
namespace {

constexpr int kMmaWarp = 0, kLoadWarp = 1;
constexpr int kEpiThreads = 128;
constexpr int kTile = 128;      // pixels per tile
constexpr int kHalo = 4;        // staged columns on each side (keeps the copy 16-byte aligned)
constexpr int kBoxW = kTile + 2 * kHalo;
constexpr int kRowSlots = 4;
constexpr int kTmemCols = 512;
constexpr int kACol0 = 256;     // first TMEM column of the A tiles

// Role layout per depthwise size K.  K = 3: an MMA warp, a loader warp, two depthwise
// warps per TMEM lane quadrant (each holding two open output rows for up to 32 channels:
// 64 partial sums) and four epilogue warps.  K = 5: four depthwise warps per quadrant
// (four open rows for up to 16 channels, again 64 partial sums) and four epilogue
// warps, the first of which also runs the row loads and the MMA issue (kMerged): 20
// warps, five per SM sub-partition, leave 96 registers per thread (22 would leave 80,
// and the partial sums would spill).
template <int K>
struct DwCfg {
  static constexpr int P = (K - 1) / 2;                 // "same" padding
  static constexpr bool kMerged = (K != 3);
  static constexpr int kPerQ = (K == 3) ? 2 : 4;        // depthwise warps per quadrant
  static constexpr int kDwWarps = 4 * kPerQ;
  static constexpr int kCMax = 64 / kPerQ;              // channels per depthwise warp, at most
  static constexpr int kWRow = (K <= 4) ? 4 : 8;        // floats per kernel row of w_dw in smem
  static constexpr int kDwWarp0 = kMerged ? 0 : 2;
  static constexpr int kEpiWarp0 = kDwWarp0 + kDwWarps;
  static constexpr int kOwnerWarp = kMerged ? kEpiWarp0 : kMmaWarp;  // allocates TMEM
  static constexpr int kThreads = 32 * kEpiWarp0 + kEpiThreads;
};
static_assert(DwCfg<5>::P <= kHalo, "the staged halo must cover the depthwise window");

struct DwParams {
  const float* w_dw;
  const float* w_pw;
  const float* bias;
  float* y;
  int N, C, H, W, Cout;
  int WB;         // 128-pixel segments per image row
  int R;          // rows per strip
  int HR;         // strips per image column
  int units;
  uint32_t row_bytes;                       // one staged row: C x kBoxW floats
  uint32_t off_wdw, off_rows, off_bar;      // shared-memory offsets (B at 0)
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

// 3-D tiled bulk copy (TMA) global -> shared, completion counted in bytes on `bar`.
// Coordinates are in elements, innermost first; parts of the box outside the tensor
// read as zeros.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread (A: 128 lanes x 8 columns).
__device__ __forceinline__ void umma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 4 consecutive columns from registers (thread i -> lane 32*(warp%4) + i).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, float a, float b, float c, float d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// Kernel row kr of a K x K depthwise kernel (padded to kWRow floats, 16-byte aligned)
// dotted with the K inputs of the window: init + sum over kw, folded from the last tap.
template <int K, int kWRow>
__device__ __forceinline__ float row_dot(const float* kr, const float (&xv)[K], float init, bool has_init) {
  float k[K];
#pragma unroll
  for (int i = 0; i < K; i += 4) {
    if (i + 4 <= kWRow && i + 1 < K) {
      const float4 q4 = *reinterpret_cast<const float4*>(kr + i);
      k[i] = q4.x;
      if (i + 1 < K) k[i + 1] = q4.y;
      if (i + 2 < K) k[i + 2] = q4.z;
      if (i + 3 < K) k[i + 3] = q4.w;
    } else {
      k[i] = kr[i];
    }
  }
  float v = has_init ? fmaf(k[K - 1], xv[K - 1], init) : k[K - 1] * xv[K - 1];
#pragma unroll
  for (int kw = K - 2; kw >= 0; --kw) v = fmaf(k[kw], xv[kw], v);
  return v;
}

// Row loads and MMA issue run by one thread as a state machine that never blocks
// (K = 5: the first epilogue warp's lane 0 calls it while it waits for accumulators).
struct CtlState {
  int lu, ln, lwb, lr, lr1;  // loader: unit, image, segment, next input row, end row
  bool lmore;
  int mu, mh, mh1;           // MMA: unit, next output row, end row
  bool mmore;
  Ring rr, ra, rm;           // row slots, A tiles, accumulators
  uint32_t issued;           // row copies issued
};

__device__ __forceinline__ void ctl_unit_rows(const DwParams& p, int u, int P, int& n, int& wb, int& r0, int& r1,
                                              int& h0, int& h1) {
  const int hr = u % p.HR;
  wb = (u / p.HR) % p.WB;
  n = u / (p.HR * p.WB);
  h0 = hr * p.R;
  h1 = min(p.H, h0 + p.R);
  r0 = h0 - P;
  r1 = h1 + P;
}

__device__ __forceinline__ void ctl_init(const DwParams& p, int P, CtlState& cs) {
  cs = CtlState{};
  cs.lu = cs.mu = blockIdx.x;
  cs.lmore = cs.mmore = blockIdx.x < p.units;
  if (cs.lmore) {
    int h0, h1;
    ctl_unit_rows(p, cs.lu, P, cs.ln, cs.lwb, cs.lr, cs.lr1, h0, h1);
    cs.mh = h0;
    cs.mh1 = h1;
  }
}

// One round: as many row copies as there are free slots, and the MMAs of one output
// row if its A tile and an accumulator are ready.
__device__ __forceinline__ void ctl_progress(const DwParams& p, const CUtensorMap* xmap, int P, CtlState& cs,
                                             uint8_t* smem_b, uint8_t* smem_rows, uint64_t* row_full,
                                             uint64_t* row_empty, uint64_t* a_full, uint64_t* a_empty,
                                             uint64_t* acc_full, uint64_t* acc_empty, uint32_t tmem_base) {
  for (int k = 0; k < kRowSlots && cs.lmore; ++k) {
    if (!test_wait(&row_empty[cs.rr.idx], cs.rr.phase ^ 1u)) break;
    mbar_arrive_expect_tx(&row_full[cs.rr.idx], p.row_bytes);
    tma_load_3d(smem_rows + (size_t)cs.rr.idx * p.row_bytes, xmap, cs.lwb * kTile - kHalo, cs.lr, cs.ln * p.C,
                &row_full[cs.rr.idx]);
    cs.rr.next(kRowSlots);
    ++cs.issued;
    if (++cs.lr == cs.lr1) {
      cs.lu += gridDim.x;
      cs.lmore = cs.lu < p.units;
      if (cs.lmore) {
        int h0, h1;
        ctl_unit_rows(p, cs.lu, P, cs.ln, cs.lwb, cs.lr, cs.lr1, h0, h1);
      }
    }
  }
  if (cs.mmore && test_wait(&a_full[cs.ra.idx], cs.ra.phase) && test_wait(&acc_empty[cs.rm.idx], cs.rm.phase ^ 1u)) {
    tc_fence_after();
    const int Cout = p.Cout;
    const uint32_t idesc = umma_idesc_tf32(128, Cout);
    const uint64_t b_desc0 = umma_desc_noswizzle(smem_addr(smem_b), (uint32_t)(2 * Cout) * 16u, 128);
    const uint32_t ks_b_u = (uint32_t)(4 * Cout);
    const uint32_t lo_u = (uint32_t)Cout;
    const uint32_t a_hi = tmem_base + (uint32_t)kACol0 + cs.ra.idx * (uint32_t)(2 * p.C);
    const uint32_t a_lo = a_hi + (uint32_t)p.C;
    const uint32_t d = tmem_base + cs.rm.idx * (uint32_t)Cout;
    for (int ks = 0; ks < (p.C >> 3); ++ks) {
      const uint64_t bh = b_desc0 + (uint64_t)((uint32_t)ks * ks_b_u);
      umma_tf32_ts(d, a_hi + 8u * ks, bh, idesc, ks > 0 ? 1u : 0u);
      umma_tf32_ts(d, a_hi + 8u * ks, bh + lo_u, idesc, 1u);
      umma_tf32_ts(d, a_lo + 8u * ks, bh, idesc, 1u);
    }
    umma_commit(&a_empty[cs.ra.idx]);
    umma_commit(&acc_full[cs.rm.idx]);
    cs.ra.next(2);
    cs.rm.next(2);
    if (++cs.mh == cs.mh1) {
      cs.mu += gridDim.x;
      cs.mmore = cs.mu < p.units;
      if (cs.mmore) {
        int n, wb, r0, r1;
        ctl_unit_rows(p, cs.mu, P, n, wb, r0, r1, cs.mh, cs.mh1);
      }
    }
  }
}

// Epilogue warps of the merged layout: each drains its TMEM lane quadrant of every
// output row (16-column chunks, the next load in flight while one is stored); while a
// warp waits for an accumulator, the first one also runs ctl_progress.  Every wait is
// bounded by the time limit; on a timeout or an abort the control thread lets its
// copies in flight land and waits for its MMAs before the CTA exits.
template <class Cfg>
__device__ __forceinline__ void merged_epilogue(const DwParams& p, const CUtensorMap& xmap, uint8_t* smem_b,
                                                uint8_t* smem_rows, uint64_t* row_full, uint64_t* row_empty,
                                                uint64_t* a_full, uint64_t* a_empty, uint64_t* acc_full,
                                                uint64_t* acc_empty, uint64_t* mma_done, uint32_t tmem_base,
                                                volatile int* abort_flag, int warp, int lane) {
  constexpr int P = Cfg::P;
  const bool ctl = (warp == Cfg::kEpiWarp0);
  const int q = warp & 3;
  const int px = q * 32 + lane;
  const int HW = p.H * p.W;
  const int Cout = p.Cout;
  CtlState cs;
  if (ctl && lane == 0) ctl_init(p, P, cs);
  Ring racc;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
    const int hr = u % p.HR;
    const int wb = (u / p.HR) % p.WB;
    const int n = u / (p.HR * p.WB);
    const int w = wb * kTile + px;
    const int h0 = hr * p.R, h1 = min(p.H, h0 + p.R);
    for (int h = h0; h < h1; ++h) {
      // Wait for the accumulator (the control thread keeps the pipeline moving).
      uint64_t t0 = 0;
      if (lane == 0) t0 = globaltimer_ns();
      for (uint32_t it = 0;; ++it) {
        if (ctl) {
          if (lane == 0)
            ctl_progress(p, &xmap, P, cs, smem_b, smem_rows, row_full, row_empty, a_full, a_empty, acc_full,
                         acc_empty, tmem_base);
          __syncwarp();
        }
        uint32_t st = 0;  // 1: ready, 2: give up
        if (lane == 0) {
          if (test_wait(&acc_full[racc.idx], racc.phase)) {
            st = 1;
          } else if (*abort_flag) {
            st = 2;
          } else if ((it & 15u) == 15u && globaltimer_ns() - t0 > p.ctl.limit_ns) {
            *abort_flag = 1;
            atomicOr(p.ctl.status, kDevStatusTimeout);
            st = 2;
          }
        }
        st = __shfl_sync(0xffffffffu, st, 0);
        if (st == 1) break;
        if (st == 2) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + racc.idx * (uint32_t)Cout;
      float* yb = p.y + (size_t)n * Cout * HW + (size_t)h * p.W + w;
      float va[16], vb[16];
      tmem_ld16(tb, va);
      tmem_wait_ld();
      for (int c0 = 0; c0 < Cout; c0 += 32) {
        if (c0 + 16 < Cout) tmem_ld16(tb + (uint32_t)(c0 + 16), vb);
        if (w < p.W) {
#pragma unroll
          for (int j = 0; j < 16; ++j) yb[(size_t)(c0 + j) * HW] = va[j] + (p.bias ? __ldg(&p.bias[c0 + j]) : 0.0f);
        }
        tmem_wait_ld();
        if (c0 + 16 < Cout) {
          if (c0 + 32 < Cout) tmem_ld16(tb + (uint32_t)(c0 + 32), va);
          if (w < p.W) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              yb[(size_t)(c0 + 16 + j) * HW] = vb[j] + (p.bias ? __ldg(&p.bias[c0 + 16 + j]) : 0.0f);
          }
          tmem_wait_ld();
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[racc.idx]);
      racc.next(2);
    }
  }
  if (ctl && lane == 0) {
    if (!ok || *abort_flag) {
      // Every copy still in flight lands before the CTA can exit (the copies before the
      // last kRowSlots were consumed, hence complete).
      Ring back = cs.rr;
      const uint32_t outstanding = min(cs.issued, (uint32_t)kRowSlots);
      for (uint32_t i = 0; i < outstanding; ++i) {
        if (back.idx == 0) {
          back.idx = kRowSlots - 1;
          back.phase ^= 1u;
        } else {
          --back.idx;
        }
        drain_wait(&row_full[back.idx], back.phase, p.ctl);
      }
    }
    umma_commit(mma_done);
    drain_wait(mma_done, 0, p.ctl);
  }
  __syncwarp();
}

template <int K>
__global__ void __launch_bounds__(DwCfg<K>::kThreads, 1)
    dwsep_tc_kernel(const DwParams p, const __grid_constant__ CUtensorMap xmap) {
  using Cfg = DwCfg<K>;
  constexpr int P = Cfg::P;
  constexpr int kThreads = Cfg::kThreads, kDwWarps = Cfg::kDwWarps, kEpiWarp0 = Cfg::kEpiWarp0;
  constexpr int kDwWarp0 = Cfg::kDwWarp0;
  constexpr int kWRow = Cfg::kWRow, kCMax = Cfg::kCMax;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  uint8_t* smem_b = smem;
  float* s_wdw = reinterpret_cast<float*>(smem + p.off_wdw);
  uint8_t* smem_rows = smem + p.off_rows;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* row_full = bars;                 // [kRowSlots]
  uint64_t* row_empty = bars + kRowSlots;    // [kRowSlots]
  uint64_t* a_full = bars + 2 * kRowSlots;   // [2]
  uint64_t* a_empty = a_full + 2;            // [2]
  uint64_t* acc_full = a_full + 4;           // [2]
  uint64_t* acc_empty = a_full + 6;          // [2]
  uint64_t* mma_done = a_full + 8;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &s_abort;
  const int C = p.C, Cout = p.Cout;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < kRowSlots; ++i) {
      mbar_init(&row_full[i], 1);
      mbar_init(&row_empty[i], kDwWarps);  // each depthwise warp releases a row once read
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], kDwWarps);
      mbar_init(&a_empty[i], 1);
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiThreads);
    }
    mbar_init(mma_done, 1);
    fence_mbarrier_init();
  }
  if (warp == Cfg::kOwnerWarp) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  // Pointwise weights -> [K-step][k-half][2*Cout rows: hi, lo][4]; depthwise weights
  // padded to [C][K rows][kWRow] so that 16-byte loads yield a row of the K x K kernel.
  {
    const int total = (C >> 3) * 2 * (2 * Cout) * 4;
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
    for (int i = tid; i < C * K * kWRow; i += kThreads) {
      const int c = i / (K * kWRow), r = (i / kWRow) % K, k = i % kWRow;
      s_wdw[i] = (k < K) ? __ldg(&p.w_dw[(c * K + r) * K + k]) : 0.0f;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  if (!Cfg::kMerged && warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_tf32(128, Cout);
      const uint64_t b_desc0 = umma_desc_noswizzle(smem_addr(smem_b), (uint32_t)(2 * Cout) * 16u, 128);
      const uint32_t ks_b_u = (uint32_t)(4 * Cout);  // one B block: 2 halves x 2*Cout rows x 16 B
      const uint32_t lo_u = (uint32_t)Cout;          // lo rows follow the hi rows
      const int ks_n = C >> 3;
      Ring ra, racc;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        const int hr = u % p.HR;
        const int h0 = hr * p.R, h1 = min(p.H, h0 + p.R);
        for (int h = h0; ok && h < h1; ++h) {
          if (!(ok = wait_fast(&a_full[ra.idx], ra.phase, p.ctl, abort_flag))) break;
          if (!(ok = wait_fast(&acc_empty[racc.idx], racc.phase ^ 1u, p.ctl, abort_flag))) break;
          tc_fence_after();
          const uint32_t a_hi = tmem_base + (uint32_t)kACol0 + ra.idx * (uint32_t)(2 * C);
          const uint32_t a_lo = a_hi + (uint32_t)C;
          const uint32_t d = tmem_base + racc.idx * (uint32_t)Cout;
          for (int ks = 0; ks < ks_n; ++ks) {
            const uint64_t bh = b_desc0 + (uint64_t)((uint32_t)ks * ks_b_u);
            umma_tf32_ts(d, a_hi + 8u * ks, bh, idesc, ks > 0 ? 1u : 0u);
            umma_tf32_ts(d, a_hi + 8u * ks, bh + lo_u, idesc, 1u);
            umma_tf32_ts(d, a_lo + 8u * ks, bh, idesc, 1u);
          }
          umma_commit(&a_empty[ra.idx]);
          umma_commit(&acc_full[racc.idx]);
          ra.next(2);
          racc.next(2);
        }
      }
      umma_commit(mma_done);
      drain_wait(mma_done, 0, p.ctl);
    }
  } else if (!Cfg::kMerged && warp == kLoadWarp) {
    // ------------------------------------------------------------ row loader
    if (lane == 0) {
      Ring rr;
      uint32_t issued = 0;
      for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
        const int hr = u % p.HR;
        const int wb = (u / p.HR) % p.WB;
        const int n = u / (p.HR * p.WB);
        const int h0 = hr * p.R, h1 = min(p.H, h0 + p.R);
        for (int r = h0 - P; r < h1 + P; ++r) {
          if (!wait_fast(&row_empty[rr.idx], rr.phase ^ 1u, p.ctl, abort_flag)) goto loader_done;
          mbar_arrive_expect_tx(&row_full[rr.idx], p.row_bytes);
          tma_load_3d(smem_rows + (size_t)rr.idx * p.row_bytes, &xmap, wb * kTile - kHalo, r, n * C, &row_full[rr.idx]);
          rr.next(kRowSlots);
          ++issued;
        }
      }
    loader_done:
      if (*abort_flag) {
        // Let every copy still in flight land before the CTA can exit.
        Ring back = rr;
        const uint32_t outstanding = min(issued, (uint32_t)kRowSlots);
        for (uint32_t i = 0; i < outstanding; ++i) {
          if (back.idx == 0) {
            back.idx = kRowSlots - 1;
            back.phase ^= 1u;
          } else {
            --back.idx;
          }
          drain_wait(&row_full[back.idx], back.phase, p.ctl);
        }
      }
    }
  } else if (warp >= kDwWarp0 && warp < kEpiWarp0) {
    // ------------------------------------------------------------ depthwise
    const int q = warp & 3;                        // TMEM lane quadrant = pixels 32q .. 32q+31
    const int grp = (warp - kDwWarp0) >> 2;        // which group of channels
    const int px = q * 32 + lane;
    const int cper = C / Cfg::kPerQ;               // channels per warp (a multiple of 4, <= kCMax)
    const int cbeg = grp * cper;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    Ring ra;
    uint32_t rseq = 0;                             // rows consumed before this unit
    for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
      const int hr = u % p.HR;
      const int h0 = hr * p.R, h1 = min(p.H, h0 + p.R);
      // acc[t][c]: output row r - P + 1 + t so far (its kernel rows 0 .. K - 2 - t; the
      // rows above the image are zeros).  Input row r completes output row r - P.
      float acc[K - 1][kCMax];
#pragma unroll
      for (int t = 0; t < K - 1; ++t)
#pragma unroll
        for (int c = 0; c < kCMax; ++c) acc[t][c] = 0.0f;
      for (int r = h0 - P; r < h1 + P; ++r) {
        const uint32_t sr = rseq + (uint32_t)(r - (h0 - P));
        if (!warp_wait(&row_full[sr % kRowSlots], (sr / kRowSlots) & 1u, p.ctl, abort_flag)) goto dw_done;
        const bool emit = (r - P >= h0);           // output row r - P completes with this row
        if (emit) {
          if (!warp_wait(&a_empty[ra.idx], ra.phase ^ 1u, p.ctl, abort_flag)) goto dw_done;
          tc_fence_after();
        }
        const float* row = reinterpret_cast<const float*>(smem_rows + (size_t)(sr % kRowSlots) * p.row_bytes) +
                           (size_t)cbeg * kBoxW + px + kHalo;
        const uint32_t a_hi = tmem_base + lane_off + (uint32_t)kACol0 + ra.idx * (uint32_t)(2 * C);
#pragma unroll
        for (int cg = 0; cg < kCMax; cg += 4) {
          if (cg < cper) {
            float fin[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = cg + j;
              const float* rw = row + c * kBoxW;
              float xv[K];
#pragma unroll
              for (int kw = 0; kw < K; ++kw) xv[kw] = rw[kw - P];
              const float* kp = s_wdw + (cbeg + c) * (K * kWRow);
              // Kernel row K-1 closes the oldest open row; row kr feeds the row opened
              // K-1-kr input rows ago; row 0 opens output row r + P.
              fin[j] = row_dot<K, kWRow>(kp + (K - 1) * kWRow, xv, acc[0][c], true);
#pragma unroll
              for (int t = 0; t < K - 2; ++t)
                acc[t][c] = row_dot<K, kWRow>(kp + (K - 2 - t) * kWRow, xv, acc[t + 1][c], true);
              acc[K - 2][c] = row_dot<K, kWRow>(kp, xv, 0.0f, false);
            }
            if (emit) {
              float hi[4], lo[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) split_tf32(fin[j], hi[j], lo[j]);
              tmem_st4(a_hi + (uint32_t)(cbeg + cg), hi[0], hi[1], hi[2], hi[3]);
              tmem_st4(a_hi + (uint32_t)(C + cbeg + cg), lo[0], lo[1], lo[2], lo[3]);
            }
          }
        }
        if (emit) {
          tmem_wait_st();
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&row_empty[sr % kRowSlots]);  // this row is not read again
          if (emit) mbar_arrive(&a_full[ra.idx]);
        }
        if (emit) ra.next(2);
      }
      rseq += (uint32_t)(h1 - h0 + 2 * P);
    }
  dw_done:;
  } else if (Cfg::kMerged) {
    // ------------------------------------------------------------ epilogue + control
    merged_epilogue<Cfg>(p, xmap, smem_b, smem_rows, row_full, row_empty, a_full, a_empty, acc_full, acc_empty,
                         mma_done, tmem_base, abort_flag, warp, lane);
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant
    const int px = q * 32 + lane;
    const int HW = p.H * p.W;
    Ring racc;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      const int hr = u % p.HR;
      const int wb = (u / p.HR) % p.WB;
      const int n = u / (p.HR * p.WB);
      const int w = wb * kTile + px;
      const int h0 = hr * p.R, h1 = min(p.H, h0 + p.R);
      for (int h = h0; h < h1; ++h) {
        if (!(ok = warp_wait(&acc_full[racc.idx], racc.phase, p.ctl, abort_flag))) break;
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + racc.idx * (uint32_t)Cout;
        float* yb = p.y + (size_t)n * Cout * HW + (size_t)h * p.W + w;
        // 32-column chunks, two register buffers: the load of chunk k+1 is in flight
        // while chunk k is stored.  When Cout is an odd multiple of 16 the last load
        // also reads 16 columns past the accumulator (inside the allocation); those
        // values are not stored.
        float va[32], vb[32];
        tmem_ld32(tb, va);
        tmem_wait_ld();
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 64) {
          if (c0 < Cout) {
            if (c0 + 32 < Cout) tmem_ld32(tb + (uint32_t)(c0 + 32), vb);
            if (w < p.W) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < 16 || c0 + 32 <= Cout)
                  yb[(size_t)(c0 + j) * HW] = va[j] + (p.bias ? __ldg(&p.bias[c0 + j]) : 0.0f);
            }
            tmem_wait_ld();
          }
          if (c0 + 32 < Cout) {
            if (c0 + 64 < Cout) tmem_ld32(tb + (uint32_t)(c0 + 64), va);
            if (w < p.W) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < 16 || c0 + 64 <= Cout)
                  yb[(size_t)(c0 + 32 + j) * HW] = vb[j] + (p.bias ? __ldg(&p.bias[c0 + 32 + j]) : 0.0f);
            }
            tmem_wait_ld();
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
  if (warp == Cfg::kOwnerWarp) {
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

DwPlan make_dw_plan(int N, int C, int H, int W, int Cout, int K, int sms = 148) {
  DwPlan pl;
  DwParams& p = pl.prm;
  std::memset(&p, 0, sizeof(p));
  if (K != 3 && K != 5) {
    pl.why = "the tensor-core kernel takes depthwise sizes 3 and 5";
    return pl;
  }
  const int P = (K - 1) / 2;
  const int w_row = (K <= 4) ? 4 : 8;
  if (C % 16 != 0 || C > 64) {
    pl.why = "C must be a multiple of 16 and at most 64";
    return pl;
  }
  if (Cout % 16 != 0 || Cout > 128) {
    pl.why = "Cout must be a multiple of 16 and at most 128";
    return pl;
  }
  if (W % 4 != 0) {
    pl.why = "W must be a multiple of 4 (rows are copied as 16-byte aligned segments)";
    return pl;
  }
  if ((long long)N * C > 0x7fffffffLL || (long long)H * W > 0x7fffffffLL) {
    pl.why = "tensor too large";
    return pl;
  }
  p.N = N; p.C = C; p.H = H; p.W = W; p.Cout = Cout;
  p.WB = (W + kTile - 1) / kTile;
  // Strips of R rows: each strip reads R + 2P rows, and the persistent grid takes
  // ceil(units / SMs) rounds of strips; pick R minimising rounds x (R + 2P).
  long long best = -1;
  for (int R : {8, 16, 32, 64}) {
    const int r = std::min(H, R);
    const long long u = (long long)N * p.WB * ((H + r - 1) / r);
    const long long cost = (u + sms - 1) / sms * (r + 2 * P);
    if (best < 0 || cost < best) {
      best = cost;
      p.R = r;
    }
    if (r == H) break;
  }
  p.HR = (H + p.R - 1) / p.R;
  const long long units = (long long)N * p.WB * p.HR;
  if (units > 0x7fffffffLL) {
    pl.why = "too many tiles";
    return pl;
  }
  p.units = (int)units;
  p.row_bytes = (uint32_t)C * kBoxW * 4u;
  const uint32_t b_bytes = (uint32_t)(C / 8) * 2u * (2u * Cout) * 16u;
  p.off_wdw = b_bytes;
  p.off_rows = (p.off_wdw + (uint32_t)(C * K * w_row) * 4u + 1023) / 1024 * 1024;
  p.off_bar = p.off_rows + kRowSlots * p.row_bytes;
  pl.smem = p.off_bar + 32 * 8;
  if (pl.smem + 2048 > (size_t)(227 * 1024)) {
    pl.why = "does not fit in shared memory";
    return pl;
  }
  pl.smem = std::max(pl.smem, (size_t)(116 * 1024));  // one CTA (one TMEM owner) per SM
  pl.ok = true;
  return pl;
}

}  // namespace

const char* dwsep_tc_unsupported_reason(int N, int C, int H, int W, int Cout, int K) {
  static thread_local char buf[160];
  DwPlan pl = make_dw_plan(N, C, H, W, Cout, K);
  if (pl.ok) return "";
  snprintf(buf, sizeof(buf), "%s", pl.why);
  return buf;
}

int dwsep_tc_launch(const DwsepArgs& a) {
  const int sms = num_sms();
  if (sms <= 0) return fail(IG3_ERR_CUDA, "dwsep TC path: cannot query the SM count");
  DwPlan pl = make_dw_plan(a.N, a.C, a.H, a.W, a.Cout, a.K, sms);
  if (!pl.ok) return fail(IG3_ERR_UNSUPPORTED, "dwsep TC path: %s", pl.why);
  if (reinterpret_cast<uintptr_t>(a.x) % 16 != 0)
    return fail(IG3_ERR_UNSUPPORTED, "dwsep TC path: x must be 16-byte aligned");
  DwParams p = pl.prm;
  p.w_dw = a.w_dw;
  p.w_pw = a.w_pw;
  p.bias = a.b;
  p.y = a.y;
  p.ctl = wait_ctl();
  if (!p.ctl.status) return fail(IG3_ERR_CUDA, "dwsep TC path: device status word unavailable");

  // x as a 3-D tensor [N*C][H][W] of floats; the box is one row of kBoxW pixels of all
  // C channels of one image.
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(IG3_ERR_CUDA, "dwsep TC path: cuTensorMapEncodeTiled is not available");
  CUtensorMap xmap;
  const cuuint64_t dims[3] = {(cuuint64_t)a.W, (cuuint64_t)a.H, (cuuint64_t)a.N * (cuuint64_t)a.C};
  const cuuint64_t strides[2] = {(cuuint64_t)a.W * 4u, (cuuint64_t)a.H * (cuuint64_t)a.W * 4u};
  const cuuint32_t box[3] = {(cuuint32_t)kBoxW, 1u, (cuuint32_t)a.C};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.x), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IG3_ERR_CUDA, "dwsep TC path: tensor map encoding failed (%d)", (int)r);

  const int grid = std::min(p.units, sms);
  auto go = [&](auto kernel, int threads) -> int {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return cuda_status(e, "dwsep TC: set shared memory size");
    kernel<<<grid, threads, pl.smem, a.stream>>>(p, xmap);
    return count_launch(cuda_status(cudaGetLastError(), "dwsep TC kernel launch"));
  };
  return a.K == 5 ? go(dwsep_tc_kernel<5>, DwCfg<5>::kThreads) : go(dwsep_tc_kernel<3>, DwCfg<3>::kThreads);
}

}  // namespace ig3
