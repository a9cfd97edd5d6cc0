// Tensor-core conv3d with stride 2 and any zero padding: the A operand of every tap is
// gathered into tensor memory.
//
// Definition followed ("Kimi-K2.6__l2_p47", the stride and padding discussion: the
// input window of output od starts at od*S - P, reads outside the tensor are zero, the
// output size is (D + 2P - 3)/S + 1):
//   conv[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw] * x[n,c,od*S+kd-P,oh*S+kh-P,ow*S+kw-P]
// with the NONE or tanh(mish) epilogue.
//
// Why a gathering kernel.  The stride-1 kernels shift a tap by offsetting the matrix
// descriptor of one tile of consecutive input positions.  With stride 2 the inputs of
// consecutive outputs are two apart, so no such tile exists.  Here producer warps read,
// for every output position of the tile and every tap, its input value from a raw box
// staged in shared memory, split it into tf32 hi / lo and write the tap's A tile to
// tensor memory (tcgen05.st); the MMAs take A from tensor memory and only the weights
// from shared memory.  The gather is a per-lane address, so stride and padding cost
// nothing on the tensor core.
//
// GEMM mapping.  M = 128 output positions p = oh*OW + ow of one output plane (one work
// unit = batch item, output plane od, 128 positions; the plan's T is 1);
// N = Cout; K = Cin*27 walked as (kd, K-step of 8 channels, kh, kw).  Input planes
// od*S + kd - P outside x are skipped (their taps read zeros).
//
// Per (kd, K-step), in one ring stage of shared memory: a tensor-map copy of the input
// box the unit's positions read, 8 channels x BY rows x BX columns of plane
// od*S + kd - P (rows from oh_lo*S - P, columns from a 16-byte aligned start left of
// -P; whatever lies outside x arrives as zeros, which is the padding), and a bulk copy
// of the pre-split weight block: 9 taps x [k-half 0 | k-half 1] x [hi | lo] x Cout
// rows x 4 channels.  The ring stage is released by the MMA commit.
//
// Tensor memory (512 columns): the accumulator [D_a | D_b] of 2*Cout columns, then AST
// A stages.  An A stage holds KHG kernel rows of one (kd, K-step): KHG x 3 kw taps x
// [hi 8 | lo 8] columns.  3xTF32 as in conv3d_tc.cu (A_hi*B_hi + A_hi*B_lo + A_lo*B_hi)
// in two MMAs per tap: A_hi x [B_hi | B_lo] (N = 2*Cout) into [D_a | D_b] and
// A_lo x B_hi (N = Cout) into D_a; the result is D_a + D_b.
//
// Roles (persistent CTAs, one per SM, 512 threads):
//   warp 0      loader (one thread): per (unit, kd, K-step) the box and the weight block;
//   warp 1      TMEM owner and MMA issuer (one thread);
//   warps 4-7   A producers, one per TMEM lane quadrant: thread = position m of each tile;
//   warps 8-15  epilogue, two teams of four, each half of the output channels: tcgen05.ld
//               of D_a and D_b, release, + bias, activation, store (lanes = consecutive
//               positions: coalesced rows).
// Every wait is bounded; on a timeout all roles stop, in-flight copies and MMAs are
// drained and TMEM is freed.
#include <algorithm>
#include <array>
#include <cstring>
#include <map>
#include <mutex>

#include "ig3_internal.h"

namespace ig3 {
namespace s2tc {

constexpr int kThreads = 512;
constexpr int kLoadWarp = 0, kMmaWarp = 1;
constexpr int kProdWarp0 = 4, kProdWarps = 4;  // warp % 4 is the TMEM lane quadrant it may access
constexpr int kEpiWarp0 = 8, kEpiWarps = 8;
constexpr int kTmemCols = 512;
constexpr int kMaxXS = 6, kMaxAST = 4;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kStaticSmem = 2048;              // s_bias, s_tmem, s_abort and alignment
constexpr int kMinSmem = 116 * 1024;           // keeps one CTA (one TMEM owner) per SM
constexpr int kStride = 2;
constexpr int kMaxCout = 128;
constexpr uint32_t kBulkChunk = 32768;         // bytes per 1-D bulk copy of a weight block

struct Params {
  const float* x;
  const float* wblob;  // [kd][KS][tap 9][khalf 2][2*Cout rows: hi | lo][4], split tf32
  const float* bias;
  float* y;
  int N, Cin, D, H, W, Cout, P, OD, OH, OW;
  int KS;          // K-steps of 8 channels
  int TP;          // output positions per unit (T * 128)
  int G;           // units per output plane
  int units;
  int BX, BY;      // staged box: columns, rows (per channel)
  int col0;        // first staged column (a multiple of 4, <= -P)
  int XS, AST;     // ring stages in shared memory, A stages in tensor memory
  uint32_t x_tx;         // bytes one box copy delivers (BX * BY * 8 * 4)
  uint32_t x_bytes;      // the box's share of a ring stage (x_tx rounded up to 1 KB)
  uint32_t b_bytes;      // one weight block (9 taps): 576 * Cout
  uint32_t stage_bytes;  // x_bytes + b_bytes
  uint32_t off_bar;
  uint32_t a_col0;       // first TMEM column of the A stages (2 * Cout: the accumulator)
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
  int n, od, p_lo, row0, kd_lo, kd_hi;
};

// Unit u -> batch item, output plane, first position; row0 = the box's first input row;
// [kd_lo, kd_hi] = the kernel planes whose input plane lies inside x (empty if none).
__host__ __device__ __forceinline__ Unit decode_unit(const Params& p, int u) {
  Unit r;
  const int gs = u % p.G;
  r.od = (u / p.G) % p.OD;
  r.n = u / (p.G * p.OD);
  r.p_lo = gs * p.TP;
  r.row0 = (r.p_lo / p.OW) * kStride - p.P;
  const int d0 = r.od * kStride - p.P;
  r.kd_lo = max(0, -d0);
  r.kd_hi = min(2, p.D - 1 - d0);
  return r;
}

__device__ __forceinline__ bool test_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool try_wait_suspend(uint32_t bar_addr, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Bounded wait for the roles off the tensor core's critical path: the thread sleeps in
// the barrier (up to ~20 us at a time, then looks at the abort flag and the time
// limit), leaving issue slots to the MMA-issuing thread.  Same contract as
// mbar_wait_bounded.
__device__ __noinline__ bool wait_relaxed(uint64_t* bar, uint32_t parity, const WaitCtl& ctl, volatile int* abort) {
  const uint32_t a = smem_addr(bar);
  if (test_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (try_wait_suspend(a, parity, 20000u)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > ctl.limit_ns) {
      *abort = 1;
      atomicOr(ctl.status, kDevStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool warp_wait_relaxed(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                                  volatile int* abort) {
  const bool ok = wait_relaxed(bar, parity, ctl, abort);
  return __all_sync(0xffffffffu, ok) != 0;
}

// The issuing thread's wait, inline (a call in the issue loop slows every MMA issue).
// Same contract as mbar_wait_bounded.
__device__ __forceinline__ bool wait_issue(uint64_t* bar, uint32_t parity, const WaitCtl& ctl, volatile int* abort) {
  const uint32_t a = smem_addr(bar);
  if (test_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (test_wait(a, parity)) return true;
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

// D[tmem] (+)= A[tmem] * B[smem]^T (A: 128 lanes x 8 columns), issued by one thread.
__device__ __forceinline__ void umma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 5-D tiled bulk copy (TMA) global -> shared, completion counted in bytes on `bar`.
// Coordinates in elements, innermost first; parts of the box outside the tensor read
// as zeros.
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, "
      "%6}], [%7];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_addr(bar))
      : "memory");
}

template <int EPI, int T, int KHG>
__global__ void __launch_bounds__(kThreads, 1)
    conv3d_strided_tc_kernel(const Params p, const __grid_constant__ CUtensorMap xmap) {
  static_assert(T == 1, "the accumulator and the epilogue hold one 128-position tile per unit");
  constexpr int NG = 3 / KHG;                 // A stages per (kd, K-step)
  constexpr int kAStageCols = T * KHG * 3 * 16;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_bias[kMaxCout];

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* mma_done = bars;
  uint64_t* in_full = bars + 1;               // [XS]
  uint64_t* in_empty = in_full + p.XS;        // [XS]
  uint64_t* a_full = in_empty + p.XS;         // [AST]
  uint64_t* a_empty = a_full + p.AST;         // [AST]
  uint64_t* acc_full = a_empty + p.AST;       // [1]
  uint64_t* acc_empty = acc_full + 1;         // [1]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &s_abort;
  const int Cout = p.Cout;

  for (int i = tid; i < Cout; i += kThreads) s_bias[i] = p.bias ? p.bias[i] : 0.0f;
  if (tid == 0) {
    s_abort = 0;
    mbar_init(mma_done, 1);
    for (int i = 0; i < p.XS; ++i) {
      mbar_init(&in_full[i], 1);
      mbar_init(&in_empty[i], 1);
    }
    for (int i = 0; i < p.AST; ++i) {
      mbar_init(&a_full[i], kProdWarps);
      mbar_init(&a_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);  // every epilogue warp, once it has read its part
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      Ring r;
      uint32_t issued = 0;
      const uint8_t* blob = reinterpret_cast<const uint8_t*>(p.wblob);
      for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
        const Unit un = decode_unit(p, u);
        for (int kd = un.kd_lo; kd <= un.kd_hi; ++kd) {
          const int id = un.od * kStride - p.P + kd;
          for (int ks = 0; ks < p.KS; ++ks) {
            if (!wait_relaxed(&in_empty[r.idx], r.phase ^ 1u, p.ctl, abort_flag)) goto loader_done;
            uint8_t* st = smem + (size_t)r.idx * p.stage_bytes;
            mbar_arrive_expect_tx(&in_full[r.idx], p.x_tx + p.b_bytes);
            tma_load_5d(st, &xmap, p.col0, un.row0, id, ks * 8, un.n, &in_full[r.idx]);
            const uint8_t* src = blob + (size_t)(kd * p.KS + ks) * p.b_bytes;
            for (uint32_t off = 0; off < p.b_bytes;) {
              const uint32_t nb = min(p.b_bytes - off, kBulkChunk);
              bulk_copy_g2s(st + p.x_bytes + off, src + off, nb, &in_full[r.idx]);
              off += nb;
            }
            r.next((uint32_t)p.XS);
            ++issued;
          }
        }
      }
    loader_done:
      if (*abort_flag) {
        // Every copy still in flight lands before the CTA can exit (the stages before
        // the last XS were consumed, hence complete).
        Ring back = r;
        const uint32_t outstanding = min(issued, (uint32_t)p.XS);
        for (uint32_t i = 0; i < outstanding; ++i) {
          if (back.idx == 0) {
            back.idx = p.XS - 1;
            back.phase ^= 1u;
          } else {
            --back.idx;
          }
          drain_wait(&in_full[back.idx], back.phase, p.ctl);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Per tap two MMAs: A_hi x [B_hi | B_lo] (N = 2 Cout) into [D_a | D_b], then
      // A_lo x B_hi (N = Cout) into D_a; the epilogue adds D_a + D_b.  Two instructions
      // instead of three per tap: a single thread issues an M = 128 tf32 MMA no faster
      // than one per ~50 cycles whatever N is up to ~96, and N = 128 runs in ~76.
      const uint32_t idesc1 = umma_idesc_tf32(128, Cout), idesc2 = umma_idesc_tf32(128, 2 * Cout);
      const uint32_t tap_u = (uint32_t)(4 * Cout);  // one tap's block in 16-byte units: 2 halves x 2*Cout rows
      const uint32_t lbo = (uint32_t)(2 * Cout) * 16u;
      Ring r, ra;
      uint32_t i = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x, ++i) {
        const Unit un = decode_unit(p, u);
        if (!(ok = wait_issue(acc_empty, (i & 1u) ^ 1u, p.ctl, abort_flag))) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base;
        bool first = true;
        for (int kd = un.kd_lo; ok && kd <= un.kd_hi; ++kd) {
          for (int ks = 0; ks < p.KS; ++ks) {
            // No wait on in_full here: the producers waited for this stage's copies (the
            // box and the weight block) before arriving on a_full, and this thread's wait
            // on a_full below orders its MMAs after both (measured 3% faster than testing
            // in_full too).
            const uint64_t b0 =
                umma_desc_noswizzle(smem_addr(smem + (size_t)r.idx * p.stage_bytes + p.x_bytes), lbo, 128);
#pragma unroll 1
            for (int g = 0; g < NG; ++g) {
              if (!(ok = wait_issue(&a_full[ra.idx], ra.phase, p.ctl, abort_flag))) break;
              tc_fence_after();
              const uint32_t a0 = tmem_base + p.a_col0 + ra.idx * (uint32_t)kAStageCols;
#pragma unroll
              for (int tt = 0; tt < T; ++tt) {
                const uint32_t d = d0 + (uint32_t)(tt * 2 * Cout);
#pragma unroll
                for (int khl = 0; khl < KHG; ++khl) {
#pragma unroll
                  for (int kw = 0; kw < 3; ++kw) {
                    const uint32_t tap = (uint32_t)((g * KHG + khl) * 3 + kw);
                    const uint32_t ac = a0 + (uint32_t)(((tt * KHG + khl) * 3 + kw) * 16);
                    const uint64_t bt = b0 + (uint64_t)(tap * tap_u);
                    umma_tf32_ts(d, ac, bt, idesc2, (first && khl == 0 && kw == 0) ? 0u : 1u);
                    umma_tf32_ts(d, ac + 8u, bt, idesc1, 1u);
                  }
                }
              }
              first = false;
              umma_commit(&a_empty[ra.idx]);
              ra.next((uint32_t)p.AST);
            }
            if (!ok) break;
            umma_commit(&in_empty[r.idx]);
            r.next((uint32_t)p.XS);
          }
        }
        if (!ok) break;
        umma_commit(acc_full);
      }
      // Wait until every MMA issued above has finished reading its operands and
      // writing TMEM, whatever the path out of the loop.
      umma_commit(mma_done);
      drain_wait(mma_done, 0, p.ctl);
    }
  } else if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps) {
    // ------------------------------------------------------------ A producers
    const int q = warp & 3;
    const int m = q * 32 + lane;  // TMEM lane = position within each tile
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int OHW = p.OH * p.OW;
    const int plane_floats = p.BX * p.BY;  // one channel of the box
    Ring r, ra;
    for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
      const Unit un = decode_unit(p, u);
      const int oh_lo = un.p_lo / p.OW;
      // Per tile: the box offset of this position's (kh, kw) = (0, 0) input.  Positions
      // past the plane read the unit's first position instead (their rows of the
      // accumulator are never stored).
      int off[T];
#pragma unroll
      for (int tt = 0; tt < T; ++tt) {
        int pp = un.p_lo + tt * 128 + m;
        if (pp >= OHW) pp = un.p_lo;
        const int oh = pp / p.OW, ow = pp - oh * p.OW;
        off[tt] = (oh - oh_lo) * kStride * p.BX + ow * kStride - p.P - p.col0;
      }
      for (int kd = un.kd_lo; kd <= un.kd_hi; ++kd) {
        for (int ks = 0; ks < p.KS; ++ks) {
          if (!warp_wait_relaxed(&in_full[r.idx], r.phase, p.ctl, abort_flag)) goto producer_done;
          const float* box = reinterpret_cast<const float*>(smem + (size_t)r.idx * p.stage_bytes);
#pragma unroll 1
          for (int g = 0; g < NG; ++g) {
            if (!warp_wait_relaxed(&a_empty[ra.idx], ra.phase ^ 1u, p.ctl, abort_flag)) goto producer_done;
            tc_fence_after();
            const uint32_t acol = tmem_base + lane_off + p.a_col0 + ra.idx * (uint32_t)kAStageCols;
#pragma unroll
            for (int tt = 0; tt < T; ++tt) {
#pragma unroll
              for (int khl = 0; khl < KHG; ++khl) {
                const float* row = box + off[tt] + (g * KHG + khl) * p.BX;
#pragma unroll
                for (int kw = 0; kw < 3; ++kw) {
                  float v[16];
#pragma unroll
                  for (int c = 0; c < 8; ++c) split_tf32(row[c * plane_floats + kw], v[c], v[8 + c]);
                  tmem_st16(acol + (uint32_t)(((tt * KHG + khl) * 3 + kw) * 16), v);
                }
              }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[ra.idx]);
            ra.next((uint32_t)p.AST);
          }
          r.next((uint32_t)p.XS);
        }
      }
    }
  producer_done:;
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    // Eight warps: team t (four warps, one per TMEM lane quadrant) takes output channels
    // [t * Cout/2, (t + 1) * Cout/2).  Each thread first reads its D_a + D_b sums into
    // registers and releases the accumulator, then applies bias and activation and
    // stores, so the next unit's MMAs start while the stores run.
    constexpr int kHalfMax = kMaxCout / 2;
    const int q = warp & 3;
    const int team = (warp - kEpiWarp0) >> 2;
    const int m = q * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    const int OHW = p.OH * p.OW;
    const int half = Cout >> 1;
    const int c0 = team * half;
    uint32_t i = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
      const Unit un = decode_unit(p, u);
      if (!warp_wait_relaxed(acc_full, i & 1u, p.ctl, abort_flag)) break;
      tc_fence_after();
      // No input plane inside x: the accumulator was never written, the output is the bias.
      const bool has = un.kd_lo <= un.kd_hi;
      float v[kHalfMax];
#pragma unroll
      for (int cc = 0; cc < kHalfMax; cc += 8) {
        if (cc < half) {
          float va[8], vb[8];
          tmem_ld8(lane_base + (uint32_t)(c0 + cc), va);
          tmem_ld8(lane_base + (uint32_t)(Cout + c0 + cc), vb);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 8; ++j) v[cc + j] = has ? va[j] + vb[j] : 0.0f;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      const int pp = un.p_lo + m;
      if (pp < OHW) {
        float* yb = p.y + ((size_t)un.n * Cout * p.OD + un.od) * (size_t)OHW + pp;
#pragma unroll
        for (int cc = 0; cc < kHalfMax; ++cc) {
          if (cc < half) {
            float val = v[cc] + s_bias[c0 + cc];
            if (EPI == IG3_EPI_TANH_MISH) val = tanh_mish(val);
            yb[(size_t)(c0 + cc) * p.OD * OHW] = val;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Weights [Cout][Cin][3][3][3] -> blocks (kd, ks), each [tap = kh*3 + kw][khalf][2*Cout
// rows: hi | lo][4]: channel ks*8 + khalf*4 + j of output channel row % Cout, zero past Cin.
__global__ void strided_tc_prep_weights(const float* __restrict__ w, float* __restrict__ blob, int Cin, int Cout,
                                        int KS, int total) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int j = i & 3;
    int t = i >> 2;
    const int row = t % (2 * Cout);
    t /= 2 * Cout;
    const int khalf = t & 1;
    t >>= 1;
    const int tap = t % 9;
    t /= 9;
    const int ks = t % KS;
    const int kd = t / KS;
    const int c = ks * 8 + khalf * 4 + j;
    const int co = row % Cout;
    const float v = (c < Cin) ? w[(((size_t)co * Cin + c) * 3 + kd) * 9 + tap] : 0.0f;
    float h, l;
    split_tf32(v, h, l);
    blob[i] = (row < Cout) ? h : l;
  }
}

// ------------------------------------------------------------------ host-side plan
struct Plan {
  bool ok = false;
  const char* why = "";
  Params prm;
  int T = 1, KHG = 3;
  size_t smem = 0;
};

size_t blob_bytes_for(int KS, int Cout) { return (size_t)3 * KS * 576u * (size_t)Cout; }

inline int out_dim(int s, int P) { return s + 2 * P < 3 ? 0 : (s + 2 * P - 3) / kStride + 1; }

// Most output rows that TP consecutive positions of an OH x OW plane, starting at a
// multiple of TP, touch.
int rows_spanned(int OH, int OW, int TP) {
  const long long ohw = (long long)OH * OW;
  int rs = 1;
  // The start's column repeats with a period of at most OW tiles.
  for (long long g = 0; g < std::min<long long>((ohw + TP - 1) / TP, OW + 1); ++g) {
    const long long lo = g * TP, hi = std::min(ohw, lo + TP) - 1;
    rs = std::max(rs, (int)(hi / OW - lo / OW + 1));
  }
  return rs;
}

// Tile shapes the kernel is instantiated for, in order of preference: (tiles per unit,
// kernel rows per A stage).  27 MMAs per A stage measured best (fewer hand-overs of the
// issuing thread per MMA): two tiles of one kernel row per stage (18 MMAs, half the
// weight and halo traffic per output) ran the stride-2 workload 7% slower, one tile of
// one row 36% slower.  Where two A stages of three rows do not fit beside the
// accumulators (Cout 128) the one-row stages take over.
constexpr int kShapes[][2] = {{1, 3}, {1, 1}};

Plan make_plan_uncached(int N, int Cin, int D, int H, int W, int P, int Cout, int epi, int sms) {
  Plan pl;
  if (epi != IG3_EPI_NONE && epi != IG3_EPI_TANH_MISH) {
    pl.why = "the strided tensor-core kernel has the NONE and TANH_MISH epilogues";
    return pl;
  }
  if (Cout % 16 != 0 || Cout < 16 || Cout > kMaxCout) {
    pl.why = "Cout must be a multiple of 16 and at most 128";
    return pl;
  }
  if (W % 4 != 0) {
    pl.why = "W must be a multiple of 4 (16-byte rows for the tensor-map copy)";
    return pl;
  }
  if (P < 0 || P > 16) {
    pl.why = "pad must be in [0, 16]";
    return pl;
  }
  const int OD = out_dim(D, P), OH = out_dim(H, P), OW = out_dim(W, P);
  if (OD < 1 || OH < 1 || OW < 1) {
    pl.why = "no output for these sizes";
    return pl;
  }
  const int KS = (Cin + 7) / 8;
  const int col0 = -((P + 3) / 4) * 4;
  const int BX = ((OW - 1) * kStride - P + 3 - col0 + 3) / 4 * 4;
  if (BX > 256) {
    pl.why = "an output row needs more than 256 staged input columns";
    return pl;
  }
  const uint32_t b_bytes = 576u * (uint32_t)Cout;
  for (const auto& sh : kShapes) {
    const int T = sh[0], KHG = sh[1];
    const int TP = 128 * T;
    const int acc_cols = 2 * T * Cout;
    const int ast = std::min(kMaxAST, (kTmemCols - acc_cols) / (T * KHG * 48));
    if (ast < 2) continue;
    const int RS = rows_spanned(OH, OW, TP);
    const int BY = (RS - 1) * kStride + 3;
    if (BY > 256) continue;
    const uint32_t x_tx = (uint32_t)(BX * BY * 8 * 4);
    const uint32_t x_bytes = (x_tx + 1023u) / 1024u * 1024u;
    const uint32_t stage = x_bytes + b_bytes;
    const long long avail = (long long)kSmemLimit - kStaticSmem - (1 + 2 * kMaxXS + 2 * kMaxAST + 4) * 8;
    const int xs = (int)std::min<long long>(kMaxXS, avail / (long long)stage);
    if (xs < 2) continue;
    const long long G = ((long long)OH * OW + TP - 1) / TP;
    const long long units = (long long)N * OD * G;
    if (units > 0x7fffffffLL) continue;
    Params& p = pl.prm;
    std::memset(&p, 0, sizeof(p));
    p.N = N; p.Cin = Cin; p.D = D; p.H = H; p.W = W; p.Cout = Cout; p.P = P;
    p.OD = OD; p.OH = OH; p.OW = OW;
    p.KS = KS;
    p.TP = TP;
    p.G = (int)G;
    p.units = (int)units;
    p.BX = BX;
    p.BY = BY;
    p.col0 = col0;
    p.XS = xs;
    p.AST = ast;
    p.x_tx = x_tx;
    p.x_bytes = x_bytes;
    p.b_bytes = b_bytes;
    p.stage_bytes = stage;
    p.off_bar = (uint32_t)xs * stage;
    p.a_col0 = (uint32_t)acc_cols;
    pl.T = T;
    pl.KHG = KHG;
    pl.smem = std::max<size_t>(p.off_bar + (size_t)(1 + 2 * xs + 2 * ast + 4) * 8, kMinSmem);
    pl.ok = true;
    (void)sms;
    return pl;
  }
  pl.why = "no tile shape fits (the staged box or the weight block is too large)";
  return pl;
}

Plan make_plan(int N, int Cin, int D, int H, int W, int P, int Cout, int epi, int sms) {
  using Key = std::array<int, 9>;
  static std::mutex mu;
  static std::map<Key, Plan> cache;
  const Key key{N, Cin, D, H, W, P, Cout, epi, sms};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  Plan pl = make_plan_uncached(N, Cin, D, H, W, P, Cout, epi, sms);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 256) cache.clear();
  cache.emplace(key, pl);
  return pl;
}

template <int EPI, int T, int KHG>
int launch(const Params& p, const CUtensorMap& xmap, size_t smem, int grid, cudaStream_t stream) {
  auto kernel = conv3d_strided_tc_kernel<EPI, T, KHG>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e, "conv3d stride-2 TC: set shared memory size");
  kernel<<<grid, kThreads, smem, stream>>>(p, xmap);
  return count_launch(cuda_status(cudaGetLastError(), "conv3d stride-2 TC kernel launch"));
}

template <int EPI>
int launch_epi(const Plan& pl, const Params& p, const CUtensorMap& xmap, int grid, cudaStream_t stream) {
  if (pl.T == 1 && pl.KHG == 3) return launch<EPI, 1, 3>(p, xmap, pl.smem, grid, stream);
  if (pl.T == 1 && pl.KHG == 1) return launch<EPI, 1, 1>(p, xmap, pl.smem, grid, stream);
  return fail(IG3_ERR_UNSUPPORTED, "conv3d stride-2 TC: no kernel variant for %d tiles x %d rows", pl.T, pl.KHG);
}

}  // namespace s2tc

const char* conv3d_strided_tc_unsupported_reason(int N, int Cin, int D, int H, int W, int pad, int Cout, int epi) {
  const s2tc::Plan pl = s2tc::make_plan(N, Cin, D, H, W, pad, Cout, epi, 148);
  return pl.ok ? "" : pl.why;
}

size_t conv3d_strided_tc_workspace(int Cin, int Cout) {
  return align_up(s2tc::blob_bytes_for((Cin + 7) / 8, Cout), 256);
}

int conv3d_strided_tc_launch(const Conv3dArgs& a) {
  using namespace s2tc;
  const int sms = num_sms();
  if (sms <= 0) return fail(IG3_ERR_CUDA, "conv3d stride-2 TC: cannot query the SM count");
  if (reinterpret_cast<uintptr_t>(a.x) % 16 != 0)
    return fail(IG3_ERR_UNSUPPORTED, "conv3d stride-2 TC: x must be 16-byte aligned");
  Plan pl = make_plan(a.N, a.Cin, a.D, a.H, a.W, a.pad, a.Cout, a.epi, sms);
  if (!pl.ok) return fail(IG3_ERR_UNSUPPORTED, "conv3d stride-2 TC: %s", pl.why);
  const size_t need = conv3d_strided_tc_workspace(a.Cin, a.Cout);
  if (!a.ws || a.ws_bytes < need)
    return fail(IG3_ERR_WORKSPACE, "conv3d stride-2 TC: workspace of %zu bytes needed, %zu given", need, a.ws_bytes);
  if (reinterpret_cast<uintptr_t>(a.ws) % 256 != 0)
    return fail(IG3_ERR_WORKSPACE, "conv3d stride-2 TC: workspace must be 256-byte aligned");
  Params p = pl.prm;
  p.x = a.x;
  p.wblob = static_cast<const float*>(a.ws);
  p.bias = a.b;
  p.y = a.y;
  p.ctl = wait_ctl();
  if (!p.ctl.status) return fail(IG3_ERR_CUDA, "conv3d stride-2 TC: device status word unavailable");

  const int total = (int)(blob_bytes_for(p.KS, p.Cout) / 4);
  strided_tc_prep_weights<<<std::min((total + 255) / 256, 4 * sms), 256, 0, a.stream>>>(
      a.w, const_cast<float*>(p.wblob), a.Cin, a.Cout, p.KS, total);
  int st = count_launch(cuda_status(cudaGetLastError(), "conv3d stride-2 TC weight prep launch"));
  if (st != IG3_OK) return st;

  // x as a 5-D tensor [N][Cin][D][H][W] of floats; the box is [1][8][1][BY][BX].
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(IG3_ERR_CUDA, "conv3d stride-2 TC: cuTensorMapEncodeTiled is not available");
  CUtensorMap xmap;
  const cuuint64_t W = (cuuint64_t)a.W, HW = W * (cuuint64_t)a.H, DHW = HW * (cuuint64_t)a.D;
  const cuuint64_t dims[5] = {W, (cuuint64_t)a.H, (cuuint64_t)a.D, (cuuint64_t)a.Cin, (cuuint64_t)a.N};
  const cuuint64_t strides[4] = {W * 4u, HW * 4u, DHW * 4u, DHW * (cuuint64_t)a.Cin * 4u};
  const cuuint32_t box[5] = {(cuuint32_t)p.BX, (cuuint32_t)p.BY, 1u, 8u, 1u};
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  const CUresult r = encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<float*>(a.x), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IG3_ERR_CUDA, "conv3d stride-2 TC: tensor map encoding failed (%d)", (int)r);

  const int grid = std::min(p.units, sms);
  return a.epi == IG3_EPI_TANH_MISH ? launch_epi<IG3_EPI_TANH_MISH>(pl, p, xmap, grid, a.stream)
                                    : launch_epi<IG3_EPI_NONE>(pl, p, xmap, grid, a.stream);
}

}  // namespace ig3
