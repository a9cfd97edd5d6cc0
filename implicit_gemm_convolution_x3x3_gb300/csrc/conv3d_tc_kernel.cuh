// Device side of the tensor-core conv3d: parameters, the warp-specialised kernel
// template and the launch switch over its compile-time variants.  The design is
// described at the top of conv3d_tc.cu.
#pragma once

#include <cstdint>

#include "ig3_internal.h"

namespace ig3 {
namespace tc {

constexpr int kThreads = 512;
constexpr int kConvWarp0 = 2, kConvThreads = 192;
constexpr int kEpiWarp0 = 8, kEpiThreads = 256;  // two warps per TMEM lane quadrant
constexpr int kAStages = 2;
constexpr int kTmemCols = 512;
constexpr int kMaxSlots = 32;  // accumulator slots per position tile (one parity bit each)
constexpr int kMaxStages = 8;  // weight ring stages
constexpr int kMaxXStages = 4; // raw input stages
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMinSmem = 116 * 1024;  // keeps one CTA (one TMEM owner) per SM

struct TcParams {
  const float* x;
  const float* wblob;  // pre-split weight blocks, layout set by KDM (see conv3d_tc.cu)
  const float* bias;
  float* y;
  float* partial;
  int N, Cin, D, H, W, Cout, OD, OH, OW;
  int KS;        // K-steps of 8 channels over the padded Cin (a multiple of KSS)
  int KSS;       // K-steps per channel chunk (= per weight stage)
  int nchunks;   // KS / KSS
  int T;         // position tiles of 128 per unit
  int NPOS;      // positions held per A stage
  int KDM;       // 3: one MMA spans the kd = 2, 1, 0 accumulators; 1: one MMA per kd;
                 // 9: one MMA spans kd and kw (slot = [kw=0 | kw=1 | kw=2] x Cout, summed
                 // with a one- and two-position shift in the epilogue)
  int HL;        // KDM 3 only: hi and lo products in separate columns (slot = 2*Cout)
  int NSLOT;     // accumulator slots per tile, Cout (HL: 2*Cout; KDM 9: 3*Cout) columns each
  int G, S, P;   // tile groups per plane, plane splits, output planes per split
  int units;
  int resident;  // weights loaded once
  int SB;        // weight ring stages (streaming)
  int TPS;       // streamed KDM 3 and 1: taps per ring stage (1, 2 or 3; with 2 the
                 // ninth tap of a chunk sits alone in its stage); KDM 9 and resident: 1
  int XS;        // raw input stages of the bulk-copy loader (0: convert warps load x)
  int epi;
  int vec;       // convert with 16-byte loads (aligned quads of positions)
  // Zero padding on chip.  With pad > 0 the kernel runs the valid convolution over a
  // virtual padded volume of D x H x W (W the virtual row pitch) whose position
  // (plane d, row h, column v) holds x[d - pad][h - pad][v - col0] of the real
  // Dr x Hr x Wr input, zero outside it; the convert warps fill the zeros.  Output
  // column v of a virtual row is stored at column v - ow_off (OW stored columns).
  int pad, Dr, Hr, Wr, col0, ow_off;
  float inv_div;
  uint32_t a_half_bytes;   // one of hi / lo in an A stage
  uint32_t a_stage_bytes;  // hi + lo
  uint32_t b_block_bytes;  // one K-step block of B
  uint32_t blob_bytes;     // all blocks (resident weights)
  uint32_t x_stage_bytes;  // one raw input stage: [CC channels][NPOS positions] floats
  uint32_t off_b, off_epi, off_x, off_bar;  // shared-memory offsets
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

struct Unit {
  int n, g, od0, od1;
};

static __host__ __device__ __forceinline__ Unit decode_unit(const TcParams& p, int u) {
  Unit r;
  const int s = u % p.S;
  const int g = (u / p.S) % p.G;
  r.n = u / (p.S * p.G);
  r.g = g;
  r.od0 = s * p.P;
  r.od1 = min(p.OD, r.od0 + p.P);
  return r;
}

// First accumulator slot of a unit: with KDM 3 and 9 every unit starts at slot 0 (its
// P planes fit in the slots, so a window of adjacent planes never wraps); with KDM 1
// the slots form a ring that runs on across units.
static __host__ __device__ __forceinline__ uint32_t unit_slot0(const TcParams& p, uint32_t plane_seq) {
  return p.KDM != 1 ? 0u : plane_seq % (uint32_t)p.NSLOT;
}

// Slot of the unit's k-th output plane (k >= 0; with KDM 1, k may exceed NSLOT).
static __host__ __device__ __forceinline__ uint32_t slot_add(const TcParams& p, uint32_t s0, int k) {
  return (s0 + (uint32_t)k) % (uint32_t)p.NSLOT;
}

// A bounded wait taken by every lane of a warp, returning one verdict for the whole
// warp (and leaving it converged): warp-collective tcgen05 instructions follow.
static __device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, ctl, abort);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Address of virtual position pos (= h * W + v) of virtual input plane d, channel 0 of
// batch item n, in the real input; nullptr where the position lies in the zero
// border (or past the virtual plane).  The division by the pitch is exact for
// pos < 2^24.
// What the padded convert needs of the parameters, passed by value: a reference to the
// kernel's parameters in an out-of-line function makes the compiler copy them to local
// memory and read every field from there inside the convert loops.
struct PadGeom {
  const float* x;
  int W, pad, col0, Dr, Hr, Wr, Cin, NPOS, vec;
};

static __device__ __forceinline__ const float* padded_src(const PadGeom& p, int n, int d, int pos) {
  int h = __float2int_rz(__fdividef((float)pos, (float)p.W));
  int v = pos - h * p.W;
  if (v < 0) { --h; v += p.W; }
  else if (v >= p.W) { ++h; v -= p.W; }
  const int dr = d - p.pad, hr = h - p.pad, wr = v - p.col0;
  if ((unsigned)dr >= (unsigned)p.Dr || (unsigned)hr >= (unsigned)p.Hr || (unsigned)wr >= (unsigned)p.Wr)
    return nullptr;
  return p.x + (((size_t)n * p.Cin * p.Dr + dr) * p.Hr + hr) * (size_t)p.Wr + wr;
}

// Non-blocking test of a barrier phase.
static __device__ __forceinline__ bool mbar_test_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return done != 0;
}

// The bounded wait of the MMA-issuing thread for its per-chunk hand-offs with resident
// weights, entirely inline: with MMAs in flight, a function call in the issue loop
// (even one never taken) slows every tcgen05.mma issue (measured: ~135 cycles more per
// wait than this form at N = 128; pool-reduce 0.547 -> 0.506 ms).  With streamed
// weights the loop also holds the per-tap weight-stage waits, and there the inline
// form measured 1-2% slower (and 13% slower as the per-tap wait): those keep
// wait_fast.
// Same contract as mbar_wait_bounded: the abort flag is polled, and past the time
// limit the wait sets it, records the timeout and returns false.
static __device__ __forceinline__ bool wait_issue(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                                  volatile int* abort) {
  const uint32_t a = smem_addr(bar);
  if (mbar_test_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_wait(a, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > ctl.limit_ns) {
        *abort = 1;
        atomicOr(ctl.status, kDevStatusTimeout);
        return false;
      }
    }
  }
}

// The common case inline (phase already complete), the bounded loop out of line.
static __device__ __forceinline__ bool wait_fast(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                                 volatile int* abort) {
  if (mbar_test_wait(smem_addr(bar), parity)) return true;
  return mbar_wait_bounded(bar, parity, ctl, abort);
}

// The MMA issuer's per-chunk wait: inline with resident weights, wait_fast otherwise.
template <bool INLINE>
static __device__ __forceinline__ bool wait_mma(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                                volatile int* abort) {
  if constexpr (INLINE) return wait_issue(bar, parity, ctl, abort);
  else return wait_fast(bar, parity, ctl, abort);
}

// The MMAs of one weight stage (KSS K-steps x T position tiles), fully unrolled so
// the issue is a straight run of adds and tcgen05.mma.  The accumulators start from
// the bias, so every MMA accumulates.
//   HL = false: each product of the split (A_hi B_hi, A_hi B_lo, A_lo B_hi) is one MMA
//               into the same columns; bl = bh + lo_u holds the B_lo rows.
//   HL = true:  two MMAs, A_hi x [B_hi | B_lo] and A_lo x [B_hi | 0], the B rows
//               interleaved per kd so that the hi and lo products land in the hh and
//               hl halves of each slot; bh + lo_u holds the [B_hi | 0] rows.
//   dcol      first accumulator column of tile 0
//   ah0, al0  A descriptors (hi, lo) of this A stage, tap offset included
//   bh0       B descriptor of the stage's first K-step, first row of the window
template <int T, int KSS, bool HL>
static __device__ __forceinline__ void issue_stage(uint32_t dcol, uint32_t tile_cols, uint64_t ah0, uint64_t al0,
                                                   uint64_t bh0, uint32_t lo_u, uint32_t ks_u, uint32_t blk_u,
                                                   uint32_t idesc) {
#pragma unroll
  for (int j = 0; j < KSS; ++j) {
    const uint64_t bh = bh0 + (uint64_t)(j * blk_u);
    const uint64_t bl = bh + lo_u;
    const uint64_t koff = (uint64_t)((uint32_t)j * ks_u);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const uint32_t dt = dcol + (uint32_t)t * tile_cols;
      const uint64_t ah = ah0 + koff + (uint64_t)(t * 128), al = al0 + koff + (uint64_t)(t * 128);
      if constexpr (HL) {
        umma_tf32(dt, ah, bh, idesc, 1u);
        umma_tf32(dt, al, bl, idesc, 1u);
      } else {
        umma_tf32(dt, ah, bh, idesc, 1u);
        umma_tf32(dt, ah, bl, idesc, 1u);
        umma_tf32(dt, al, bh, idesc, 1u);
      }
    }
  }
}

// All (kh, kw) taps of one A chunk against one set of accumulator columns: nine, or
// with NKW = 1 (kw inside the MMA's N) the three kh.  Streaming weights: one ring
// stage per TPS taps (NKW = 3) or per kh (NKW = 1, TPS = 1), waited for, used and
// released; the next stage's barrier is tested before this stage's MMAs are issued and
// its result read only after them, so the test's shared-memory latency (long while
// MMAs read their operands) overlaps the issue (`next_ready` carries the result across
// calls).  Resident weights: block
// (tap_base + kh * NKW + kw) * KS + blk0.  Returns false if a wait gave up (the MMAs
// are still issued, on whatever the buffers hold; the caller stops).
template <int T, int KSS, bool RES, bool HL, int NKW, int TPS>
static __device__ __forceinline__ bool issue_taps(const TcParams& p, uint32_t dcol, uint32_t tile_cols,
                                                  uint64_t ah0, uint64_t al0, uint64_t bwin, uint32_t lo_u,
                                                  uint32_t ks_u, uint32_t blk_u, uint32_t row_u, uint32_t idesc,
                                                  int tap_base, int blk0, uint64_t* b_full, uint64_t* b_empty,
                                                  Ring& rb, bool& next_ready, volatile int* abort_flag) {
  bool good = true;
  static_assert(TPS >= 1 && TPS <= 3 && (NKW == 3 || TPS == 1), "taps per stage");
  const uint32_t b_tap_u = blk_u * (uint32_t)KSS;
  uint64_t b_stage = 0;
  bool ahead = false;
#pragma unroll
  for (int kh = 0; kh < 3; ++kh) {
#pragma unroll
    for (int kw = 0; kw < NKW; ++kw) {
      const int i = kh * NKW + kw;
      const uint64_t tap_u = (uint64_t)((uint32_t)kh * row_u + (uint32_t)kw);
      uint64_t bst;
      if constexpr (RES) {
        bst = bwin + (uint64_t)((uint32_t)((tap_base + i) * p.KS + blk0) * blk_u);
      } else {
        if (i % TPS == 0) {
          if (!next_ready && !wait_fast(&b_full[rb.idx], rb.phase, p.ctl, abort_flag)) good = false;
          tc_fence_after();
          b_stage = bwin + (uint64_t)(rb.idx * (uint32_t)TPS * b_tap_u);
          // The next stage's barrier, tested now and read after this stage's MMAs.  (A
          // stage not yet refilled reads as not ready, and is then waited for.)
          uint32_t i1 = rb.idx + 1, ph1 = rb.phase;
          if (i1 == (uint32_t)p.SB) { i1 = 0; ph1 ^= 1u; }
          ahead = mbar_test_wait(smem_addr(&b_full[i1]), ph1);
        }
        bst = b_stage + (uint64_t)((uint32_t)(i % TPS) * b_tap_u);
      }
      issue_stage<T, KSS, HL>(dcol, tile_cols, ah0 + tap_u, al0 + tap_u, bst, lo_u, ks_u, blk_u, idesc);
      if constexpr (!RES) {
        if (i % TPS == TPS - 1 || i == 3 * NKW - 1) {
          umma_commit(&b_empty[rb.idx]);
          rb.next((uint32_t)p.SB);
          next_ready = ahead;
        }
      }
    }
  }
  return good;
}

// 16 consecutive floats from shared memory (16-byte aligned), the same for every lane.
static __device__ __forceinline__ void load_bias16(const float* src, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 q = reinterpret_cast<const float4*>(src)[i];
    v[4 * i] = q.x;
    v[4 * i + 1] = q.y;
    v[4 * i + 2] = q.z;
    v[4 * i + 3] = q.w;
  }
}

static __device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// bar.sync that also returns the AND of v over the participating threads.
static __device__ __forceinline__ bool named_bar_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

static __device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// The convert of one A stage over the virtual padded volume (zero padding on chip):
// the same items as the unpadded loops, with each position's source looked up in the
// real input (padded_src) and zeros for the border.  Out of line, so that the
// unpadded loops compile as they would without it.
template <int KSS>
static __device__ __noinline__ void convert_padded(const PadGeom p, int n, int d, int p0, int c0, int ct,
                                                   uint32_t hi_base, uint32_t lo_base) {
  constexpr int CC = KSS * 8;
  const size_t cstride = (size_t)p.Dr * p.Hr * p.Wr;
  if (p.vec) {
    // A quad of virtual positions is wholly inside x's row or wholly in the zero
    // border (the pitch and the first column are multiples of 4).
    const int quads = p.NPOS >> 2;
    const int vitems = (CC / 4) * quads;
    for (int i0 = ct; i0 < vitems; i0 += 2 * kConvThreads) {
      float4 v[2][4];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = i0 + k * kConvThreads;
        const int grp = i / quads, qd = i - grp * quads;
        const float* src = padded_src(p, n, d, p0 + 4 * qd);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = c0 + grp * 4 + j;
          v[k][j] = (i < vitems && src != nullptr && c < p.Cin)
                        ? __ldg(reinterpret_cast<const float4*>(src + (size_t)c * cstride))
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = i0 + k * kConvThreads;
        if (i < vitems) {
          const int grp = i / quads, qd = i - grp * quads;
          const uint32_t off = (uint32_t)(grp * p.NPOS + 4 * qd) * 16u;
          float h[4][4], l[4][4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            split_tf32(v[k][j].x, h[0][j], l[0][j]);
            split_tf32(v[k][j].y, h[1][j], l[1][j]);
            split_tf32(v[k][j].z, h[2][j], l[2][j]);
            split_tf32(v[k][j].w, h[3][j], l[3][j]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            st_shared_v4(hi_base + off + 16u * e, h[e][0], h[e][1], h[e][2], h[e][3]);
            st_shared_v4(lo_base + off + 16u * e, l[e][0], l[e][1], l[e][2], l[e][3]);
          }
        }
      }
    }
  } else {
    const int items = (CC / 4) * p.NPOS;
    for (int i0 = ct; i0 < items; i0 += 2 * kConvThreads) {
      float v[2][4];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = i0 + k * kConvThreads;
        const int grp = i / p.NPOS, pp = i - grp * p.NPOS;
        const float* src = padded_src(p, n, d, p0 + pp);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = c0 + grp * 4 + j;
          v[k][j] = (i < items && src != nullptr && c < p.Cin) ? __ldg(src + (size_t)c * cstride) : 0.0f;
        }
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = i0 + k * kConvThreads;
        if (i < items) {
          const uint32_t off = (uint32_t)i * 16u;  // [group][position][4]
          float h[4], l[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) split_tf32(v[k][j], h[j], l[j]);
          st_shared_v4(hi_base + off, h[0], h[1], h[2], h[3]);
          st_shared_v4(lo_base + off, l[0], l[1], l[2], l[3]);
        }
      }
    }
  }
}

template <int EPI, int KDM, int T, int KSS, bool RES, bool HL, int TPS>
__global__ void __launch_bounds__(kThreads, 1) conv3d_tc_kernel(const TcParams p) {
  static_assert((KDM == 9 || RES) ? TPS == 1 : (TPS >= 1 && TPS <= 3), "taps per weight stage");
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_red[kEpiThreads / 32];
  __shared__ __align__(16) float s_bias[128];

  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + p.off_b;
  float* s_epi = reinterpret_cast<float*>(smem + p.off_epi);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* a_full = bars;                     // [2]
  uint64_t* a_empty = bars + 2;                // [2]
  uint64_t* w_full = bars + 4;                 // resident weights
  uint64_t* mma_done = bars + 5;               // final drain of the MMA pipe
  uint64_t* acc_full = bars + 6;               // [NSLOT]
  uint64_t* acc_empty = acc_full + p.NSLOT;    // [NSLOT]
  uint64_t* b_full = acc_empty + p.NSLOT;      // [SB]
  uint64_t* b_empty = b_full + p.SB;           // [SB]
  uint64_t* x_full = b_empty + p.SB;           // [XS]
  uint64_t* x_empty = x_full + p.XS;           // [XS]
  // With the bulk-copy loader, the first convert warp issues the copies and the other
  // five transform; otherwise all six load and transform.
  const int conv_threads = kConvThreads - (p.XS > 0 ? 32 : 0);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &s_abort;
  const uint32_t slot_w = (uint32_t)((KDM == 9 ? 3 : HL ? 2 : 1) * p.Cout);  // accumulator columns per slot
  const uint32_t tile_cols = (uint32_t)p.NSLOT * slot_w;

  if (tid < p.Cout) s_bias[tid] = p.bias ? p.bias[tid] : 0.0f;
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&a_full[i], conv_threads);
      mbar_init(&a_empty[i], 1);
    }
    mbar_init(w_full, 1);
    mbar_init(mma_done, 1);
    for (int i = 0; i < p.NSLOT; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiThreads);
    }
    for (int i = 0; i < p.SB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < p.XS; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], conv_threads);
    }
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  if (warp >= kEpiWarp0) {
    // Every MMA accumulates, so each accumulator starts as the conv bias of its
    // column's channel (and the epilogue writes the bias back after reading a slot).
    const int grp = (warp - kEpiWarp0) >> 2;
    const uint32_t lane_base = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    for (uint32_t c = (uint32_t)grp * 16u; c < (uint32_t)T * tile_cols; c += 32u) {
      const uint32_t r = c % slot_w;  // column within its slot (HL: hh half, then hl half)
      float bv[16];
      if (r < (uint32_t)p.Cout) {
        load_bias16(s_bias + r, bv);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) bv[j] = 0.0f;
      }
      tmem_st16(lane_base + c, bv);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      if constexpr (RES) {
        const uint32_t total = p.blob_bytes;
        mbar_arrive_expect_tx(w_full, total);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.wblob);
        for (uint32_t off = 0; off < total;) {
          const uint32_t n = min(total - off, 32768u);
          bulk_copy_g2s(smem_b + off, src + off, n, w_full);
          off += n;
        }
        drain_wait(w_full, 0, p.ctl);
      } else {
        Ring rb;
        uint32_t issued = 0;
        const uint32_t tap_bytes = (uint32_t)KSS * p.b_block_bytes;
        const uint32_t stage_bytes = (uint32_t)TPS * tap_bytes;
        for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
          const Unit un = decode_unit(p, u);
          for (int d = un.od0; d < un.od1 + 2 && !*abort_flag; ++d) {
            const int kd_hi = min(2, d - un.od0), kd_lo = max(0, d - un.od1 + 1);
            for (int ch = 0; ch < p.nchunks; ++ch) {
              // The stages in the order the MMA issuer consumes them: KDM 3, the nine
              // taps (each block holds all three kd); KDM 9, the three kh (each block
              // holds all kd and kw); KDM 1, the valid kd from 2 down, nine taps each.
              const int nkd = (KDM != 1) ? 1 : kd_hi - kd_lo + 1;
              for (int k = 0; k < nkd; ++k) {
                const int tap_base = (KDM != 1) ? 0 : (kd_hi - k) * 9;
                for (int khw = 0; khw < (KDM == 9 ? 3 : 9); khw += TPS) {
                  const int nt = min(TPS, (KDM == 9 ? 3 : 9) - khw);
                  if (!wait_fast(&b_empty[rb.idx], rb.phase ^ 1u, p.ctl, abort_flag)) goto producer_done;
                  mbar_arrive_expect_tx(&b_full[rb.idx], (uint32_t)nt * tap_bytes);
                  for (int t = 0; t < nt; ++t) {
                    const int blk = (tap_base + khw + t) * p.KS + ch * KSS;
                    bulk_copy_g2s(smem_b + (size_t)rb.idx * stage_bytes + (size_t)t * tap_bytes,
                                  reinterpret_cast<const uint8_t*>(p.wblob) + (size_t)blk * p.b_block_bytes,
                                  tap_bytes, &b_full[rb.idx]);
                  }
                  rb.next((uint32_t)p.SB);
                  ++issued;
                }
              }
            }
          }
        }
      producer_done:
        if (*abort_flag) {
          // Let every copy still in flight land before the CTA can exit.
          Ring back = rb;
          const uint32_t outstanding = min(issued, (uint32_t)p.SB);
          for (uint32_t i = 0; i < outstanding; ++i) {
            if (back.idx == 0) {
              back.idx = p.SB - 1;
              back.phase ^= 1u;
            } else {
              --back.idx;
            }
            drain_wait(&b_full[back.idx], back.phase, p.ctl);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Descriptors are formed once and advanced by plain adds in 16-byte units (the
      // start-address field is the low 14 bits), so the issue loop stays a short
      // chain of adds and tcgen05.mma.
      const uint32_t b_rows = (uint32_t)((KDM == 9 ? 18 : KDM == 3 ? (HL ? 12 : 6) : 2) * p.Cout);
      const uint64_t a_desc0 = umma_desc_noswizzle(smem_addr(smem_a), (uint32_t)p.NPOS * 16u, 128);
      const uint64_t b_desc0 = umma_desc_noswizzle(smem_addr(smem_b), b_rows * 16u, 128);
      const uint32_t a_stage_u = p.a_stage_bytes >> 4, a_half_u = p.a_half_bytes >> 4;
      const uint32_t ks_u = 2u * (uint32_t)p.NPOS;  // next K-step: two channel groups on
      const uint32_t blk_u = p.b_block_bytes >> 4;
      const uint32_t lo_u = b_rows >> 1;             // the second half of the rows (lo, or [hi | 0])
      const uint32_t row_u = (uint32_t)p.W;          // one input row (kh step)
      const uint32_t cout = (uint32_t)p.Cout;
      const uint32_t idesc1 = umma_idesc_tf32(128, p.Cout);
      bool ok = true;
      if constexpr (RES) ok = wait_issue(w_full, 0, p.ctl, abort_flag);
      Ring ra, rb;
      bool b_next_ready = false;  // the next weight stage's barrier, tested one stage ahead
      uint32_t empty_par = 0;  // per slot: uses so far, mod 2
      uint32_t plane_seq = 0;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        const Unit un = decode_unit(p, u);
        const uint32_t s0 = unit_slot0(p, plane_seq);
        for (int d = un.od0; ok && d < un.od1 + 2; ++d) {
          // Output planes fed by input plane d: od = d - kd for kd in [kd_lo, kd_hi].
          const int kd_hi = min(2, d - un.od0), kd_lo = max(0, d - un.od1 + 1);
          for (int ch = 0; ok && ch < p.nchunks; ++ch) {
            if (!(ok = wait_mma<RES>(&a_full[ra.idx], ra.phase, p.ctl, abort_flag))) break;
            tc_fence_after();
            if (ch == 0 && kd_lo == 0) {
              // Plane d opens output plane od = d: its slot must have been drained.
              const uint32_t s = slot_add(p, s0, d - un.od0);
              if (!(ok = wait_mma<RES>(&acc_empty[s], ((empty_par >> s) & 1u) ^ 1u, p.ctl, abort_flag))) break;
              empty_par ^= 1u << s;
              tc_fence_after();
            }
            const uint64_t ah0 = a_desc0 + (uint64_t)(ra.idx * a_stage_u);
            const uint64_t al0 = ah0 + a_half_u;
            if constexpr (KDM != 1) {
              // One window: the accumulators of od = d - kd_hi .. d - kd_lo are adjacent
              // (slots ascend with od), the B rows of kd = kd_hi .. kd_lo too.
              const uint32_t nkd = (uint32_t)(kd_hi - kd_lo + 1);
              const uint32_t dcol = tmem_base + (s0 + (uint32_t)(d - kd_hi - un.od0)) * slot_w;
              const uint32_t idesc = umma_idesc_tf32(128, (int)(nkd * slot_w));
              const uint64_t bwin = b_desc0 + (uint64_t)((uint32_t)(2 - kd_hi) * slot_w);
              ok = issue_taps<T, KSS, RES, HL, (KDM == 9 ? 1 : 3), TPS>(p, dcol, tile_cols, ah0, al0, bwin, lo_u, ks_u, blk_u,
                                                                   row_u, idesc, 0, ch * KSS, b_full, b_empty, rb,
                                                                   b_next_ready, abort_flag);
            } else {
              for (int kd = kd_hi; ok && kd >= kd_lo; --kd) {
                const uint32_t dcol = tmem_base + slot_add(p, s0, d - kd - un.od0) * cout;
                ok = issue_taps<T, KSS, RES, false, 3, TPS>(p, dcol, tile_cols, ah0, al0, b_desc0, lo_u, ks_u, blk_u, row_u,
                                                idesc1, kd * 9, ch * KSS, b_full, b_empty, rb, b_next_ready,
                                                abort_flag);
                if (ok && kd == 2 && ch == p.nchunks - 1) umma_commit(&acc_full[slot_add(p, s0, d - 2 - un.od0)]);
              }
            }
            umma_commit(&a_empty[ra.idx]);
            ra.next(kAStages);
          }
          // KDM 3, 9: output plane d - 2 received its last contribution with this plane.
          if (KDM != 1 && ok && kd_hi == 2) umma_commit(&acc_full[s0 + (uint32_t)(d - 2 - un.od0)]);
        }
        plane_seq += (uint32_t)(un.od1 - un.od0);
      }
      // Wait until every MMA issued above has finished reading shared memory and
      // writing TMEM, whatever the path out of the loop.
      umma_commit(mma_done);
      drain_wait(mma_done, 0, p.ctl);
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ input convert
    const size_t HW = (size_t)p.H * p.W;
    const int plane_pos = p.H * p.W;
    const int CC = KSS * 8;
    if (p.XS > 0 && warp == kConvWarp0) {
      // Input loader (one thread): for each (plane, chunk) the CC channel rows of the
      // NPOS positions the unit needs, each a contiguous run of x, by 1-D bulk copy
      // into a ring of raw stages [CC][NPOS], up to XS chunks ahead of the transform.
      // Rows end at the plane's last position; channels past Cin are not copied.
      if (lane == 0) {
        Ring rx;
        uint32_t issued = 0;
        uint8_t* smem_x = smem + p.off_x;
        for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
          const Unit un = decode_unit(p, u);
          const int p0 = un.g * T * 128;
          const uint32_t row_bytes = (uint32_t)min(p.NPOS, plane_pos - p0) * 4u;
          for (int d = un.od0; d < un.od1 + 2; ++d) {
            for (int ch = 0; ch < p.nchunks; ++ch) {
              if (!wait_fast(&x_empty[rx.idx], rx.phase ^ 1u, p.ctl, abort_flag)) goto loader_done;
              const int c0 = ch * CC;
              const int nvalid = min(CC, p.Cin - c0);
              mbar_arrive_expect_tx(&x_full[rx.idx], (uint32_t)nvalid * row_bytes);
              const float* src = p.x + (((size_t)un.n * p.Cin + c0) * p.D + d) * HW + p0;
              uint8_t* dst = smem_x + (size_t)rx.idx * p.x_stage_bytes;
              for (int c = 0; c < nvalid; ++c)
                bulk_copy_g2s(dst + (size_t)c * p.NPOS * 4, src + (size_t)c * p.D * HW, row_bytes, &x_full[rx.idx]);
              rx.next((uint32_t)p.XS);
              ++issued;
            }
          }
        }
      loader_done:
        if (*abort_flag) {
          // Let every copy still in flight land before the CTA can exit.
          Ring back = rx;
          const uint32_t outstanding = min(issued, (uint32_t)p.XS);
          for (uint32_t i = 0; i < outstanding; ++i) {
            if (back.idx == 0) {
              back.idx = p.XS - 1;
              back.phase ^= 1u;
            } else {
              --back.idx;
            }
            drain_wait(&x_full[back.idx], back.phase, p.ctl);
          }
        }
      }
      goto convert_done;
    }
    {
    const int ct = tid - (kConvWarp0 + (p.XS > 0 ? 1 : 0)) * 32;
    Ring ra, rx;
    for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
      const Unit un = decode_unit(p, u);
      const int p0 = un.g * T * 128;
      for (int d = un.od0; d < un.od1 + 2; ++d) {
        for (int ch = 0; ch < p.nchunks; ++ch) {
          if (!warp_wait(&a_empty[ra.idx], ra.phase ^ 1u, p.ctl, abort_flag)) goto convert_done;
          const int c0 = ch * CC;
          const int items = (CC / 4) * p.NPOS;
          const uint32_t hi_base = smem_addr(smem_a) + ra.idx * p.a_stage_bytes;
          const uint32_t lo_base = hi_base + p.a_half_bytes;
          const float* xplane = p.x + ((size_t)un.n * p.Cin) * p.D * HW + (size_t)d * HW;
          if (p.XS > 0) {
            // Transform a raw stage: item = (channel group, 4 consecutive positions),
            // four 16-byte shared loads (one per channel), split, transposed to four
            // [position][4 channels] entries.  Positions past the plane and channels
            // past Cin read as zero.
            if (!warp_wait(&x_full[rx.idx], rx.phase, p.ctl, abort_flag)) goto convert_done;
            const float* raw = reinterpret_cast<const float*>(smem + p.off_x + (size_t)rx.idx * p.x_stage_bytes);
            const int quads = p.NPOS >> 2;
            const int vitems = (CC / 4) * quads;
            for (int i = ct; i < vitems; i += conv_threads) {
              const int grp = i / quads, qd = i - grp * quads;
              const bool in_plane = p0 + 4 * qd < plane_pos;
              float4 v[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int cl = grp * 4 + j;
                v[j] = (in_plane && c0 + cl < p.Cin) ? *reinterpret_cast<const float4*>(raw + cl * p.NPOS + 4 * qd)
                                                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
              }
              const uint32_t off = (uint32_t)(grp * p.NPOS + 4 * qd) * 16u;
              float h[4][4], l[4][4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                split_tf32(v[j].x, h[0][j], l[0][j]);
                split_tf32(v[j].y, h[1][j], l[1][j]);
                split_tf32(v[j].z, h[2][j], l[2][j]);
                split_tf32(v[j].w, h[3][j], l[3][j]);
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                st_shared_v4(hi_base + off + 16u * e, h[e][0], h[e][1], h[e][2], h[e][3]);
                st_shared_v4(lo_base + off + 16u * e, l[e][0], l[e][1], l[e][2], l[e][3]);
              }
            }
            mbar_arrive(&x_empty[rx.idx]);
            rx.next((uint32_t)p.XS);
          } else if (p.pad != 0) {
            const PadGeom g{p.x, p.W, p.pad, p.col0, p.Dr, p.Hr, p.Wr, p.Cin, p.NPOS, p.vec};
            convert_padded<KSS>(g, un.n, d, p0, c0, ct, hi_base, lo_base);
          } else if (p.vec) {
            // Item = (channel group, 4 consecutive positions): four 16-byte loads (one
            // per channel, coalesced along positions), transposed in registers to four
            // [position][4 channels] entries.  H*W % 4 == 0, so a quad lies wholly inside
            // or wholly past the plane.
            const int quads = p.NPOS >> 2;
            const int vitems = (CC / 4) * quads;
            for (int i0 = ct; i0 < vitems; i0 += 2 * kConvThreads) {
              float4 v[2][4];
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const int i = i0 + k * kConvThreads;
                const int grp = i / quads, qd = i - grp * quads;
                const int pos = p0 + 4 * qd;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int c = c0 + grp * 4 + j;
                  v[k][j] = (i < vitems && pos < plane_pos && c < p.Cin)
                                ? __ldg(reinterpret_cast<const float4*>(xplane + (size_t)c * p.D * HW + pos))
                                : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                }
              }
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const int i = i0 + k * kConvThreads;
                if (i < vitems) {
                  const int grp = i / quads, qd = i - grp * quads;
                  const uint32_t off = (uint32_t)(grp * p.NPOS + 4 * qd) * 16u;
                  float h[4][4], l[4][4];
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    split_tf32(v[k][j].x, h[0][j], l[0][j]);
                    split_tf32(v[k][j].y, h[1][j], l[1][j]);
                    split_tf32(v[k][j].z, h[2][j], l[2][j]);
                    split_tf32(v[k][j].w, h[3][j], l[3][j]);
                  }
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    st_shared_v4(hi_base + off + 16u * e, h[e][0], h[e][1], h[e][2], h[e][3]);
                    st_shared_v4(lo_base + off + 16u * e, l[e][0], l[e][1], l[e][2], l[e][3]);
                  }
                }
              }
            }
          } else
          for (int i0 = ct; i0 < items; i0 += 2 * kConvThreads) {
            float v[2][4];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int i = i0 + k * kConvThreads;
              const int grp = i / p.NPOS, pp = i - grp * p.NPOS;
              const int pos = p0 + pp;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int c = c0 + grp * 4 + j;
                v[k][j] = (i < items && pos < plane_pos && c < p.Cin)
                              ? __ldg(xplane + (size_t)c * p.D * HW + pos)
                              : 0.0f;
              }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int i = i0 + k * kConvThreads;
              if (i < items) {
                const uint32_t off = (uint32_t)i * 16u;  // [group][position][4]
                float h[4], l[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) split_tf32(v[k][j], h[j], l[j]);
                st_shared_v4(hi_base + off, h[0], h[1], h[2], h[3]);
                st_shared_v4(lo_base + off, l[0], l[1], l[2], l[3]);
              }
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&a_full[ra.idx]);
          ra.next(kAStages);
        }
      }
    }
    }
  convert_done:;
  } else {
    // ------------------------------------------------------------ epilogue
    // Two groups of four warps; each group covers all four TMEM lane quadrants and
    // takes every other (tile, 16-channel chunk) item of a plane (KDM 9: its half of
    // the 16 channels, every tile, in one pass).
    constexpr int CW = 16;
    const int et = tid - kEpiWarp0 * 32;
    const int q = warp & 3;                        // TMEM lane quadrant this warp may access
    const int grp = (warp - kEpiWarp0) >> 2;       // 0 or 1
    const size_t OHW = (size_t)p.OH * p.OW;
    const int PH = p.OH / 2, PW = p.OW / 2;
    const int cchunks = p.Cout / CW;
    const int items = T * cchunks;
    float* s_x = s_epi + grp * (16 * 32);          // pool: h-pair exchange [16][32] per group
    float* s_prev = s_epi + 2 * (16 * 32);         // pool: even-plane maxima [T][Cout][32]
    // KDM 9: the kw = 1, 2 columns of the first lanes of each quadrant, for the last
    // lanes of the quadrant before it; [group][2 buffers][T tiles][4 quadrants][24].
    float* s_kx = s_epi + grp * (2 * T * 4 * 24);
    uint32_t kx_buf = 0;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    uint32_t full_par = 0;  // per slot: completions seen so far, mod 2
    uint32_t plane_seq = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      const Unit un = decode_unit(p, u);
      const uint32_t s0 = unit_slot0(p, plane_seq);
      const int p0 = un.g * T * 128;
      float psum = 0.0f;
      for (int od = un.od0; od < un.od1; ++od) {
        const uint32_t slot = slot_add(p, s0, od - un.od0);
        // Every epilogue thread takes the same verdict, so that none is left waiting
        // at a named barrier below for a warp that gave up.
        ok = named_bar_and(6, kEpiThreads, mbar_wait_bounded(&acc_full[slot], (full_par >> slot) & 1u, p.ctl,
                                                             abort_flag));
        if (!ok) break;
        full_par ^= 1u << slot;
        tc_fence_after();
        const bool pool_plane = (EPI == IG3_EPI_POOL_REDUCE) && (od / 2 < p.OD / 2);
        if constexpr (KDM == 9) {
          static_assert(EPI != IG3_EPI_POOL_REDUCE, "KDM 9 has no pool-reduce epilogue");
          // Group g takes channels 8g .. 8g + 7 of every position tile in one pass.
          // Column block kw holds the sum over kd, kh and channels of the taps with
          // that kw, at the position of its INPUT pixel: output position o takes
          // block 0 at o, block 1 at o + 1 and block 2 at o + 2.
          const int c0 = grp * 8;
          float v[T][8], a1[T][8], a2[T][8];
#pragma unroll
          for (int t = 0; t < T; ++t) {
            const uint32_t taddr = lane_base + (uint32_t)t * tile_cols + slot * slot_w + (uint32_t)c0;
            tmem_ld8(taddr, v[t]);
            tmem_ld8(taddr + (uint32_t)p.Cout, a1[t]);
            tmem_ld8(taddr + 2u * (uint32_t)p.Cout, a2[t]);
          }
          tmem_wait_ld();
          {
            float bv[8], zv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              bv[j] = s_bias[c0 + j];
              zv[j] = 0.0f;
            }
#pragma unroll
            for (int t = 0; t < T; ++t) {
              const uint32_t taddr = lane_base + (uint32_t)t * tile_cols + slot * slot_w + (uint32_t)c0;
              tmem_st8(taddr, bv);  // the slot's next use starts from the bias again
              tmem_st8(taddr + (uint32_t)p.Cout, zv);
              tmem_st8(taddr + 2u * (uint32_t)p.Cout, zv);
            }
          }
          float s1[T][8], s2[T][8];
#pragma unroll
          for (int t = 0; t < T; ++t)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              s1[t][j] = __shfl_down_sync(0xffffffffu, a1[t][j], 1);
              s2[t][j] = __shfl_down_sync(0xffffffffu, a2[t][j], 2);
            }
          if (p.W > 32) {
            // A row crosses quadrants: lanes 30 and 31 take the neighbours from the
            // next quadrant's lanes 0 and 1 (the last quadrant ends a row, where the
            // two positions are wrap-around columns).  Two buffers alternate, so one
            // barrier per plane suffices.
            float* xb = s_kx + kx_buf * (T * 4 * 24);
            kx_buf ^= 1u;
            if (q > 0 && lane < 2) {
#pragma unroll
              for (int t = 0; t < T; ++t)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  if (lane == 0) {
                    xb[(t * 4 + q) * 24 + j] = a1[t][j];
                    xb[(t * 4 + q) * 24 + 8 + j] = a2[t][j];
                  } else {
                    xb[(t * 4 + q) * 24 + 16 + j] = a2[t][j];
                  }
                }
            }
            named_bar_sync(4 + grp, 128);
            if (q < 3 && lane >= 30) {
#pragma unroll
              for (int t = 0; t < T; ++t)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  if (lane == 31) {
                    s1[t][j] = xb[(t * 4 + q + 1) * 24 + j];
                    s2[t][j] = xb[(t * 4 + q + 1) * 24 + 16 + j];
                  } else {
                    s2[t][j] = xb[(t * 4 + q + 1) * 24 + 8 + j];
                  }
                }
            }
          }
#pragma unroll
          for (int t = 0; t < T; ++t)
#pragma unroll
            for (int j = 0; j < 8; ++j) v[t][j] += s1[t][j] + s2[t][j];
          // Tiles hold whole rows, so a lane has the same column in every tile.
          const int lq = q * 32 + lane;
          const int ow = (p0 + lq) % p.W - p.ow_off;
#pragma unroll
          for (int t = 0; t < T; ++t) {
            const int oh = (p0 + t * 128 + lq) / p.W;
            if (oh < p.OH && ow >= 0 && ow < p.OW) {
              float* yb = p.y + (((size_t)un.n * p.Cout + c0) * p.OD + od) * OHW + (size_t)oh * p.OW + ow;
#pragma unroll
              for (int j = 0; j < 8; j += 2) {
                float v0 = v[t][j], v1 = v[t][j + 1];
                if (EPI == IG3_EPI_TANH_MISH) tanh_mish2(v0, v1, v0, v1);
                yb[(size_t)j * p.OD * OHW] = v0;
                yb[(size_t)(j + 1) * p.OD * OHW] = v1;
              }
            }
          }
        }
        if constexpr (KDM != 9)
        for (int it = grp; it < items; it += 2) {
          const int t = it / cchunks;
          const int c0 = (it - t * cchunks) * CW;
          const int lp = t * 128 + q * 32 + lane;  // position within the unit
          const int pos = p0 + lp;
          const int oh = pos / p.W, ow = pos - oh * p.W - p.ow_off;
          const bool valid = (oh < p.OH) && (ow >= 0) && (ow < p.OW);
          const uint32_t taddr = lane_base + (uint32_t)t * tile_cols + slot * slot_w + (uint32_t)c0;
          float v[CW];
          float bv[16];
          tmem_ld16(taddr, v);
          if constexpr (HL) {
            float v2[16];
            tmem_ld16(taddr + (uint32_t)p.Cout, v2);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              v[j] += v2[j];
              v2[j] = 0.0f;
            }
            tmem_st16(taddr + (uint32_t)p.Cout, v2);
          } else {
            tmem_wait_ld();
          }
          load_bias16(s_bias + c0, bv);
          tmem_st16(taddr, bv);  // the slot's next use starts from the bias again
          if constexpr (EPI != IG3_EPI_POOL_REDUCE) {
            float* yb = p.y + (((size_t)un.n * p.Cout + c0) * p.OD + od) * OHW + (size_t)oh * p.OW + ow;
#pragma unroll
            for (int j = 0; j < CW; j += 2) {
              float v0 = v[j], v1 = v[j + 1];
              if (EPI == IG3_EPI_TANH_MISH) tanh_mish2(v0, v1, v0, v1);
              if (valid) {
                yb[(size_t)j * p.OD * OHW] = v0;
                yb[(size_t)(j + 1) * p.OD * OHW] = v1;
              }
            }
          } else {
            if (!pool_plane) continue;
            // w-pair: neighbouring lanes; h-pair: position + W.
            const int r = (q * 32 + lane) / p.W;          // row within the tile (tile rows start even)
            const int cw = ow >> 1;
            const int cell = (r >> 1) * (p.W >> 1) + cw;  // pooled cell within the tile, < 32
            const bool even_w = (ow & 1) == 0, even_r = (r & 1) == 0;
            float hm[CW];
#pragma unroll
            for (int j = 0; j < CW; ++j) {
              const float z = v[j] * p.inv_div;
              hm[j] = fmaxf(z, __shfl_xor_sync(0xffffffffu, z, 1));
            }
            if (p.W <= 16) {
#pragma unroll
              for (int j = 0; j < CW; ++j) hm[j] = fmaxf(hm[j], __shfl_xor_sync(0xffffffffu, hm[j], p.W));
            } else {
              if (!even_r && even_w) {
#pragma unroll
                for (int j = 0; j < CW; ++j) s_x[j * 32 + cell] = hm[j];
              }
              named_bar_sync(1 + grp, 128);
              if (even_r && even_w) {
#pragma unroll
                for (int j = 0; j < CW; ++j) hm[j] = fmaxf(hm[j], s_x[j * 32 + cell]);
              }
              named_bar_sync(1 + grp, 128);
            }
            if (even_r && even_w) {
              float* prev = s_prev + ((size_t)t * p.Cout + c0) * 32 + cell;
              if ((od & 1) == 0) {
#pragma unroll
                for (int j = 0; j < CW; ++j) prev[j * 32] = hm[j];
              } else if ((oh >> 1) < PH && cw < PW) {
#pragma unroll
                for (int j = 0; j < CW; ++j) psum += fmaxf(prev[j * 32], hm[j]);
              }
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&acc_empty[slot]);
      }
      if (!ok) break;
      if constexpr (EPI == IG3_EPI_POOL_REDUCE) {
        // Fixed-order reduction of the unit's partial: lanes, then warps in order.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
        if (lane == 0) s_red[warp - kEpiWarp0] = psum;
        named_bar_sync(3, kEpiThreads);
        if (et == 0) {
          float s = 0.0f;
          for (int i = 0; i < kEpiThreads / 32; ++i) s += s_red[i];
          p.partial[u] = s;
        }
        named_bar_sync(3, kEpiThreads);
      }
      plane_seq += (uint32_t)(un.od1 - un.od0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Kernel variants: (KDM, HL, T, KSS, resident, taps per weight stage).  The planner
// only produces these.
struct Variant {
  int kdm, hl, t, kss, res, tps;
};
constexpr Variant kVariants[] = {
    // one MMA per split product spans the kd window (Cout 48..80)
    {3, 0, 1, 2, 0, 3}, {3, 0, 2, 2, 0, 3}, {3, 0, 1, 2, 0, 2}, {3, 0, 2, 2, 0, 2}, {3, 0, 1, 2, 0, 1}, {3, 0, 2, 2, 0, 1},
    {3, 0, 1, 1, 1, 1}, {3, 0, 1, 2, 1, 1}, {3, 0, 2, 1, 1, 1}, {3, 0, 2, 2, 1, 1},
    // hi and lo products in separate columns: two MMAs span the window (Cout 16, 32)
    {3, 1, 1, 2, 0, 3}, {3, 1, 2, 2, 0, 3}, {3, 1, 1, 2, 0, 2}, {3, 1, 2, 2, 0, 2}, {3, 1, 1, 2, 0, 1}, {3, 1, 2, 2, 0, 1},
    {3, 1, 1, 1, 1, 1}, {3, 1, 1, 2, 1, 1}, {3, 1, 2, 1, 1, 1}, {3, 1, 2, 2, 1, 1},
    // one MMA per split product spans the kd and kw window (Cout 16, W dividing 128;
    // not pool-reduce)
    {9, 0, 1, 1, 1, 1}, {9, 0, 1, 2, 1, 1}, {9, 0, 2, 1, 1, 1}, {9, 0, 2, 2, 1, 1}, {9, 0, 1, 2, 0, 1}, {9, 0, 2, 2, 0, 1},
    // one MMA per kd (Cout 96..128)
    {1, 0, 1, 2, 0, 3}, {1, 0, 1, 1, 0, 3}, {1, 0, 1, 2, 0, 2}, {1, 0, 1, 1, 0, 2}, {1, 0, 1, 2, 0, 1}, {1, 0, 1, 1, 0, 1},
};

// Launches the kernel variant matching p.  Returns an ig3 status.
template <int EPI>
int launch_kernel(const TcParams& p, size_t smem, int grid, cudaStream_t stream) {
  auto go = [&](auto kernel) -> int {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_status(e, "conv3d TC: set shared memory size");
    kernel<<<grid, kThreads, smem, stream>>>(p);
    return count_launch(cuda_status(cudaGetLastError(), "conv3d TC kernel launch"));
  };
  const int key = p.KDM * 100000 + p.HL * 10000 + p.T * 1000 + p.KSS * 100 + p.resident * 10 + p.TPS;
  switch (key) {
    case 301203: return go(conv3d_tc_kernel<EPI, 3, 1, 2, false, false, 3>);
    case 302203: return go(conv3d_tc_kernel<EPI, 3, 2, 2, false, false, 3>);
    case 301202: return go(conv3d_tc_kernel<EPI, 3, 1, 2, false, false, 2>);
    case 302202: return go(conv3d_tc_kernel<EPI, 3, 2, 2, false, false, 2>);
    case 301201: return go(conv3d_tc_kernel<EPI, 3, 1, 2, false, false, 1>);
    case 302201: return go(conv3d_tc_kernel<EPI, 3, 2, 2, false, false, 1>);
    case 301111: return go(conv3d_tc_kernel<EPI, 3, 1, 1, true, false, 1>);
    case 301211: return go(conv3d_tc_kernel<EPI, 3, 1, 2, true, false, 1>);
    case 302111: return go(conv3d_tc_kernel<EPI, 3, 2, 1, true, false, 1>);
    case 302211: return go(conv3d_tc_kernel<EPI, 3, 2, 2, true, false, 1>);
    case 311203: return go(conv3d_tc_kernel<EPI, 3, 1, 2, false, true, 3>);
    case 312203: return go(conv3d_tc_kernel<EPI, 3, 2, 2, false, true, 3>);
    case 311202: return go(conv3d_tc_kernel<EPI, 3, 1, 2, false, true, 2>);
    case 312202: return go(conv3d_tc_kernel<EPI, 3, 2, 2, false, true, 2>);
    case 311201: return go(conv3d_tc_kernel<EPI, 3, 1, 2, false, true, 1>);
    case 312201: return go(conv3d_tc_kernel<EPI, 3, 2, 2, false, true, 1>);
    case 311111: return go(conv3d_tc_kernel<EPI, 3, 1, 1, true, true, 1>);
    case 311211: return go(conv3d_tc_kernel<EPI, 3, 1, 2, true, true, 1>);
    case 312111: return go(conv3d_tc_kernel<EPI, 3, 2, 1, true, true, 1>);
    case 312211: return go(conv3d_tc_kernel<EPI, 3, 2, 2, true, true, 1>);
    case 101203: return go(conv3d_tc_kernel<EPI, 1, 1, 2, false, false, 3>);
    case 101103: return go(conv3d_tc_kernel<EPI, 1, 1, 1, false, false, 3>);
    case 101202: return go(conv3d_tc_kernel<EPI, 1, 1, 2, false, false, 2>);
    case 101102: return go(conv3d_tc_kernel<EPI, 1, 1, 1, false, false, 2>);
    case 101201: return go(conv3d_tc_kernel<EPI, 1, 1, 2, false, false, 1>);
    case 101101: return go(conv3d_tc_kernel<EPI, 1, 1, 1, false, false, 1>);
    default:
      break;
  }
  if constexpr (EPI != IG3_EPI_POOL_REDUCE) {
    switch (key) {
      case 901111: return go(conv3d_tc_kernel<EPI, 9, 1, 1, true, false, 1>);
      case 901211: return go(conv3d_tc_kernel<EPI, 9, 1, 2, true, false, 1>);
      case 902111: return go(conv3d_tc_kernel<EPI, 9, 2, 1, true, false, 1>);
      case 902211: return go(conv3d_tc_kernel<EPI, 9, 2, 2, true, false, 1>);
      case 901201: return go(conv3d_tc_kernel<EPI, 9, 1, 2, false, false, 1>);
      case 902201: return go(conv3d_tc_kernel<EPI, 9, 2, 2, false, false, 1>);
      default: break;
    }
  }
  return fail(IG3_ERR_UNSUPPORTED,
              "conv3d TC: no kernel variant for KDM %d, HL %d, T %d, %d K-steps, resident %d, %d taps per stage", p.KDM,
              p.HL, p.T, p.KSS, p.resident, p.TPS);
}

extern template int launch_kernel<IG3_EPI_NONE>(const TcParams&, size_t, int, cudaStream_t);
extern template int launch_kernel<IG3_EPI_TANH_MISH>(const TcParams&, size_t, int, cudaStream_t);
extern template int launch_kernel<IG3_EPI_POOL_REDUCE>(const TcParams&, size_t, int, cudaStream_t);

}  // namespace tc
}  // namespace ig3
