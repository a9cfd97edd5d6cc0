// Tensor-core conv3d for 16 output channels with the A operand in tensor memory.
//
// Definition followed ("Kimi-K2.6__l2_p47", the per-output loop and its NCDHW index
// check; the implicit-GEMM view M = output positions, N = Cout, K = Cin*27):
//   conv[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw] * x[n,c,od+kd,oh+kh,ow+kw]
// with the tanh(mish) epilogue of that page or the pool-reduce epilogue of
// "Kimi-K2.6__l2_p8" (/divisor, MaxPool3d(2) floor mode, global mean, +bias2,
// sum over channels).
//
// Why a separate kernel.  With 16 output channels every MMA is narrow.  When both
// operands come from shared memory, an M = 128, K = 8 tf32 MMA reads a 4 KB A tile
// plus 32 B per B column, and at ~128 B per cycle the A read alone costs 32 cycles:
// for N <= 144 the operand reads, not the tensor core, set the pace, and they also
// delay every mbarrier test of the issuing thread.  Here the A tiles live in tensor
// memory (tcgen05.mma with A in TMEM), so an MMA reads only its B rows (4.6 KB at
// N = 144) from shared memory and runs at its execution rate (N/2 cycles).
//
// GEMM mapping.  A position tile is 128 consecutive positions p = h*W + w of one
// input plane, holding whole input rows (W divides 64).  For an input plane d and
// a K-step of 8 channels, three A tiles are formed, one per kh: A_kh[m][c] =
// x[c, p0 + m + kh*W] (TMEM lane m, 8 columns; hi and lo halves of the split).
// One MMA per (kh, split product) has N = nkd * 48: B rows [kd][kw][16 channels] for
// the kd of the output planes this input plane feeds (od = d - kd), so the
// accumulator of output plane od holds, per position o, three column blocks kw =
// 0, 1, 2, each the sum over kd, kh and c of the taps with that kw at INPUT
// position o.  The epilogue adds block kw at o + kw into output o (lane shuffles,
// and a shared-memory hand-over where a row crosses a 32-lane quadrant).
//
// Tensor memory (512 columns): accumulator slots of 48 columns ([kw=0 | kw=1 | kw=2]
// x 16) in a ring that runs across work units; the kd window of an input plane is
// one MMA, or two where it wraps the ring's end.  Then two A stages, each PP input
// planes x KSS K-steps (PP * KSS <= 2), each K-step three kh tiles of [hi 8 | lo 8]
// columns.  Every MMA accumulates: a slot starts as [bias | 0 | 0] and the epilogue
// writes that back after reading it.
//
// Precision: 3xTF32 as in conv3d_tc.cu (hi = fp32 with the low 13 bits cleared, lo =
// x - hi; acc += A_hi*B_hi + A_hi*B_lo + A_lo*B_hi in fp32).
//
// Data flow (persistent CTAs, one per SM, 512 threads):
//   warp 0      loader (one thread): the pre-split weights once (1-D bulk copy, they
//               stay resident), then for each (group of PP input planes, channel
//               chunk) one tensor-map copy of the 128 + 2W positions the tile needs
//               from each plane and channel of the chunk, into a ring of raw stages
//               (what lies outside x arrives as zeros);
//   warp 1      TMEM owner and MMA issuer (one thread, fully unrolled chunks);
//   warps 4-7   A producers, one per TMEM lane quadrant: thread = position m reads
//               x at m, m + W, m + 2W of each channel from the raw stage, splits it
//               and writes the three A tiles with tcgen05.st;
//   warps 8-15  epilogue, two teams of four taking alternating output planes (pool-
//               reduce: plane pairs), 16 channels each: tcgen05.ld of the three kw
//               blocks, the shifted sum, + activation and the store, or the 2x2x2 max
//               and the partial sum of the pooled cells.
// A work unit is (batch item, position tile, range of P output planes); input
// planes od0 .. od1 + 1 stream through it.  Every wait is bounded; on a timeout all
// roles stop, in-flight copies and MMAs are drained and TMEM is freed.
#include <algorithm>
#include <array>
#include <cstring>
#include <map>
#include <mutex>

#include "ig3_internal.h"

namespace ig3 {
namespace tc16 {

constexpr int kThreads = 512;
constexpr int kLoadWarp = 0, kMmaWarp = 1;
constexpr int kProdWarp0 = 4, kProdWarps = 4;  // warp % 4 is the TMEM lane quadrant it may access
constexpr int kEpiWarp0 = 8, kEpiWarps = 8, kEpiThreads = 32 * kEpiWarps;
constexpr int kCout = 16;
constexpr int kSlotCols = 3 * kCout;           // [kw=0 | kw=1 | kw=2] x 16
constexpr int kKStepCols = 3 * 16;             // three kh tiles of [hi 8 | lo 8]
constexpr int kMaxAStages = 4;
constexpr int kTmemCols = 512;
constexpr int kMaxXStages = 6;
constexpr int kBRows = 18 * kCout;             // [hi: kd 2,1,0 x kw 0,1,2 | lo: the same] x 16
constexpr uint32_t kBBlockBytes = 2u * kBRows * 16u;  // one (kh, K-step) block: two K halves
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMinSmem = 116 * 1024;           // keeps one CTA (one TMEM owner) per SM

struct Params {
  const float* x;
  const float* wblob;  // [kh][KS][khalf][kBRows][4], split tf32 hi / lo
  const float* bias;
  float* y;
  float* partial;
  int N, Cin, D, H, W, OD, OH, OW;
  int KS;       // K-steps of 8 channels (a multiple of KSS)
  int nchunks;  // KS / KSS (channel chunks per group of PP input planes)
  int NSLOT;    // accumulator slots in the ring
  int G, S, P;  // position tiles per plane, plane splits, output planes per split
  int units;
  int NPOS;     // positions per raw channel row: 128 + 2W
  int XS;       // raw stages
  int AST;      // A stages in tensor memory
  float inv_div;
  uint32_t blob_bytes;
  uint32_t x_stage_bytes;  // [8 * KSS channels][PP planes][NPOS positions] floats
  uint32_t off_x, off_bar;
  uint32_t a_col0;         // first TMEM column of the A stages
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

__host__ __device__ __forceinline__ Unit decode_unit(const Params& p, int u) {
  Unit r;
  const int s = u % p.S;
  r.g = (u / p.S) % p.G;
  r.n = u / (p.S * p.G);
  r.od0 = s * p.P;
  r.od1 = min(p.OD, r.od0 + p.P);
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

__device__ __forceinline__ bool wait_fast(uint64_t* bar, uint32_t parity, const WaitCtl& ctl, volatile int* abort) {
  if (test_wait(smem_addr(bar), parity)) return true;
  return mbar_wait_bounded(bar, parity, ctl, abort);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl, volatile int* abort) {
  const bool ok = wait_fast(bar, parity, ctl, abort);
  return __all_sync(0xffffffffu, ok) != 0;
}

// mbarrier.try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about `hint_ns` pass, so a waiting warp takes no issue slots.
__device__ __forceinline__ bool try_wait_suspend(uint32_t bar_addr, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// A bounded wait for the roles off the tensor core's critical path (loader,
// producers, epilogue): the thread is suspended in the barrier until the phase
// completes (re-checking the abort flag and the time limit every ~20 us), leaving
// issue slots to the MMA-issuing thread, whose bookkeeping between two chunks is not
// hidden by the short MMA queue.  Same contract as mbar_wait_bounded.
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

// Tests of PP + 1 barrier phases in one asm block, so that their shared-memory
// latencies overlap: r[i] = phase par[i] of bar[i] completed (i < PP), r[PP] = phase
// last_par of last_bar completed.
template <int PP>
__device__ __forceinline__ void test_wait_n(const uint32_t (&bar)[PP], const uint32_t (&par)[PP], uint32_t last_bar,
                                            uint32_t last_par, bool (&r)[PP + 1]) {
  uint32_t d0, d1 = 1, d2;
  if constexpr (PP == 1) {
    asm volatile(
        "{\n\t.reg .pred p0, p2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p0, [%2], %3;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p2, [%4], %5;\n\t"
        "selp.u32 %0, 1, 0, p0;\n\tselp.u32 %1, 1, 0, p2;\n\t}"
        : "=r"(d0), "=r"(d2)
        : "r"(bar[0]), "r"(par[0]), "r"(last_bar), "r"(last_par)
        : "memory");
    r[0] = d0 != 0;
    r[1] = d2 != 0;
  } else {
    asm volatile(
        "{\n\t.reg .pred p0, p1, p2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p0, [%3], %4;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p1, [%5], %6;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p2, [%7], %8;\n\t"
        "selp.u32 %0, 1, 0, p0;\n\tselp.u32 %1, 1, 0, p1;\n\tselp.u32 %2, 1, 0, p2;\n\t}"
        : "=r"(d0), "=r"(d1), "=r"(d2)
        : "r"(bar[0]), "r"(par[0]), "r"(bar[PP - 1]), "r"(par[PP - 1]), "r"(last_bar), "r"(last_par)
        : "memory");
    r[0] = d0 != 0;
    r[PP - 1] = d1 != 0;
    r[PP] = d2 != 0;
  }
}

// The issuing thread's wait, inline (a call in the issue loop slows every
// tcgen05.mma issue).  Same contract as mbar_wait_bounded.
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
// 16 consecutive floats from shared memory (16-byte aligned), the same for every lane.
__device__ __forceinline__ void load_bias16(const float* src, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 q4 = reinterpret_cast<const float4*>(src)[i];
    v[4 * i] = q4.x;
    v[4 * i + 1] = q4.y;
    v[4 * i + 2] = q4.z;
    v[4 * i + 3] = q4.w;
  }
}

// Every MMA here accumulates (the slots start from the bias).
__device__ __forceinline__ void umma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(1u)
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// The 16 channels of one output position: + activation, stored (NCDHW, 16 channels).
template <int EPI>
__device__ __forceinline__ void store_position(const Params& p, int n, int od, int oh, int ow, const float (&v)[kCout]) {
  const size_t OHW = (size_t)p.OH * p.OW;
  float* yb = p.y + ((size_t)n * kCout * p.OD + od) * OHW + (size_t)oh * p.OW + ow;
#pragma unroll
  for (int j = 0; j < kCout; j += 2) {
    float v0 = v[j], v1 = v[j + 1];
    if (EPI == IG3_EPI_TANH_MISH) tanh_mish2(v0, v1, v0, v1);
    yb[(size_t)j * p.OD * OHW] = v0;
    yb[(size_t)(j + 1) * p.OD * OHW] = v1;
  }
}

// bar.sync that also returns the AND of v over the participating threads.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// The MMAs of one channel chunk against one run of adjacent accumulator slots:
// KSS K-steps x three kh x three split products.  d: first slot's column; nw: slots
// in the run (N = 48 * nw); brow_u: the run's first B row (16-byte units).
template <int KSS>
__device__ __forceinline__ void issue_chunk(uint32_t d, uint32_t a0, uint64_t b0, uint32_t idesc, uint32_t ks_blk_u) {
  constexpr uint32_t kLoU = 9u * kCout;  // lo rows follow the nine hi row blocks
#pragma unroll
  for (int ks = 0; ks < KSS; ++ks) {
#pragma unroll
    for (int kh = 0; kh < 3; ++kh) {
      const uint32_t ah = a0 + (uint32_t)((ks * 3 + kh) * 16);
      const uint64_t bh = b0 + (uint64_t)((uint32_t)kh * ks_blk_u + (uint32_t)ks * (kBBlockBytes >> 4));
      umma_tf32_ts(d, ah, bh, idesc);
      umma_tf32_ts(d, ah, bh + kLoU, idesc);
      umma_tf32_ts(d, ah + 8u, bh, idesc);
    }
  }
}

// One chunk of the MMA issue sequence (PP input planes x one channel chunk), with
// what the issuing thread needs precomputed.  Per plane: the window's first run of
// slots (accumulator column dc1, descriptor id1, B descriptor b) and, where it wraps
// the ring, a second run from slot 0 (B rows n2off further, descriptor id2); the slot
// the plane opens (its first contribution: wait until drained) and the slot it
// closes (its last contribution: commit for the epilogue).
template <int PP>
struct Chunk {
  uint32_t dc1[PP], id1[PP], id2[PP], n2off[PP], open_slot[PP], close_slot[PP];
  uint64_t b[PP];
  bool valid[PP], run2[PP], opens[PP], closes[PP];
};

// Position of the issue sequence: unit u, its planes [od0, od1), the next group of
// input planes d0 and channel chunk ch; s_d is the slot of output plane od = d0, and
// s_unit the slot of the unit's first output plane (the ring runs on across units).
struct ChunkIter {
  int u, od0, od1, d0, ch;
  uint32_t s_d, s_unit;
};

__device__ __forceinline__ void chunk_iter_init(const Params& p, ChunkIter& it) {
  it.u = blockIdx.x;
  it.ch = 0;
  it.s_d = it.s_unit = 0;
  if (it.u < p.units) {
    const Unit un = decode_unit(p, it.u);
    it.od0 = un.od0;
    it.od1 = un.od1;
    it.d0 = un.od0;
  }
}

template <int PP, int KSS>
__device__ __forceinline__ bool next_chunk(const Params& p, ChunkIter& it, Chunk<PP>& c, uint32_t tmem_base,
                                           uint64_t b_desc0, uint32_t idesc0, uint32_t idesc_slot) {
  const uint32_t nslot = (uint32_t)p.NSLOT;
  if (it.u >= p.units) return false;
  if (it.ch == p.nchunks) {
    it.ch = 0;
    it.d0 += PP;
    it.s_d += PP;
    if (it.s_d >= nslot) it.s_d -= nslot;
    if (it.d0 >= it.od1 + 2) {
      it.s_unit = (it.s_unit + (uint32_t)(it.od1 - it.od0)) % nslot;
      it.u += gridDim.x;
      if (it.u >= p.units) return false;
      const Unit un = decode_unit(p, it.u);
      it.od0 = un.od0;
      it.od1 = un.od1;
      it.d0 = un.od0;
      it.s_d = it.s_unit;
    }
  }
  const int npl = min(PP, it.od1 + 2 - it.d0);
  const bool first = it.ch == 0, last = it.ch == p.nchunks - 1;
  const uint32_t boff = (uint32_t)(it.ch * KSS) * (kBBlockBytes >> 4);
  uint32_t sl = it.s_d;
#pragma unroll
  for (int pi = 0; pi < PP; ++pi) {
    // Input plane d feeds output planes od = d - kd for kd in [kd_lo, kd_hi]: slots
    // s_first .. in ascending order, wrapping the ring's end at most once.
    const int d = it.d0 + pi;
    const int kd_hi = min(2, d - it.od0), kd_lo = max(0, d - it.od1 + 1);
    const bool valid = pi < npl;
    const uint32_t nkd = valid ? (uint32_t)(kd_hi - kd_lo + 1) : 0u;
    const uint32_t s_first = (sl >= (uint32_t)kd_hi) ? sl - (uint32_t)kd_hi : sl + nslot - (uint32_t)kd_hi;
    const uint32_t n1 = min(nkd, nslot - s_first), n2 = nkd - n1;
    c.valid[pi] = valid;
    c.opens[pi] = valid && first && kd_lo == 0;
    c.open_slot[pi] = sl;
    c.closes[pi] = valid && last && kd_hi == 2;  // output plane d - 2 completes here
    c.close_slot[pi] = s_first;
    c.dc1[pi] = tmem_base + s_first * (uint32_t)kSlotCols;
    c.id1[pi] = idesc0 + n1 * idesc_slot;
    c.id2[pi] = idesc0 + n2 * idesc_slot;
    // B rows of kd = kd_hi .. kd_lo: [kd=2 | kd=1 | kd=0] blocks of 48 rows.
    c.b[pi] = b_desc0 + (uint64_t)((uint32_t)(2 - kd_hi) * kSlotCols + boff);
    c.run2[pi] = n2 > 0;
    c.n2off[pi] = n1 * (uint32_t)kSlotCols;
    sl = (sl + 1u == nslot) ? 0u : sl + 1u;
  }
  ++it.ch;
  return true;
}

// 4-D tiled bulk copy (TMA) global -> shared, completion counted in bytes on `bar`.
// Coordinates in elements, innermost first; parts of the box outside the tensor read
// as zeros.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}

template <int EPI, int KSS, int PP>
__global__ void __launch_bounds__(kThreads, 1) conv3d_tc16_kernel(const Params p, const __grid_constant__ CUtensorMap xmap) {
  constexpr int kCC = 8 * KSS;                         // channels per chunk
  constexpr int kAStageCols = PP * KSS * kKStepCols;   // one A stage: PP planes x KSS K-steps
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_red[kEpiWarps];
  __shared__ __align__(16) float s_bias[kCout];
  // kw hand-over across quadrants: [team][buffer][quadrant][lane 0: block 1, block 2 |
  // lane 1: block 2] x 16 channels
  __shared__ __align__(16) float s_kx[2][2][4][48];
  // h-pair hand-over of the pooled maxima: [team][buffer][cell][16 channels], the four
  // 16-byte granules of a cell rotated by (cell >> 1) & 3 so that the 16 cells a warp
  // writes or reads at once spread over all banks
  __shared__ __align__(16) float s_h[2][2][32][kCout];

  uint8_t* smem_b = smem;
  uint8_t* smem_x = smem + p.off_x;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* w_full = bars;
  uint64_t* mma_done = bars + 1;
  uint64_t* a_full = bars + 2;                 // [AST]
  uint64_t* a_empty = a_full + p.AST;          // [AST]
  uint64_t* x_full = a_empty + p.AST;          // [XS]
  uint64_t* x_empty = x_full + p.XS;           // [XS]
  uint64_t* acc_full = x_empty + p.XS;         // [NSLOT]
  uint64_t* acc_empty = acc_full + p.NSLOT;    // [NSLOT]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &s_abort;

  if (tid < kCout) s_bias[tid] = p.bias ? p.bias[tid] : 0.0f;
  if (tid == 0) {
    s_abort = 0;
    mbar_init(w_full, 1);
    mbar_init(mma_done, 1);
    for (int i = 0; i < p.AST; ++i) {
      mbar_init(&a_full[i], kProdWarps);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < p.XS; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], kProdWarps);
    }
    for (int i = 0; i < p.NSLOT; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps / 2);  // the four warps of the team that drained it
    }
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
  if (warp >= kEpiWarp0) {
    // Every slot starts as [bias | 0 | 0]: team t writes the slots s with s % 2 == t.
    const int team = (warp - kEpiWarp0) >> 2;
    const uint32_t lane_base = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    float bv[kCout], zv[kCout];
    load_bias16(s_bias, bv);
#pragma unroll
    for (int j = 0; j < kCout; ++j) zv[j] = 0.0f;
    for (int sl = team; sl < p.NSLOT; sl += 2) {
      const uint32_t col = lane_base + (uint32_t)(sl * kSlotCols);
      tmem_st16(col, bv);
      tmem_st16(col + 16u, zv);
      tmem_st16(col + 32u, zv);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      // The weight blocks come from the split kernel launched just before this one;
      // with a programmatic dependent launch this CTA may already run beside it, so
      // wait for that grid's completion (and its writes) here.  Without one it is a
      // no-op.
      asm volatile("griddepcontrol.wait;" ::: "memory");
      mbar_arrive_expect_tx(w_full, p.blob_bytes);
      const uint8_t* wsrc = reinterpret_cast<const uint8_t*>(p.wblob);
      for (uint32_t off = 0; off < p.blob_bytes;) {
        const uint32_t n = min(p.blob_bytes - off, 32768u);
        bulk_copy_g2s(smem_b + off, wsrc + off, n, w_full);
        off += n;
      }
      // One tensor-map copy per chunk: box [CC channels][PP planes][NPOS positions]
      // of x viewed as [N][Cin][D][H*W]; positions past the plane, planes past D and
      // channels past Cin come back as zeros.
      Ring rx;
      uint32_t issued = 0;
      for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
        const Unit un = decode_unit(p, u);
        const int p0 = un.g * 128;
        for (int d0 = un.od0; d0 < un.od1 + 2; d0 += PP) {
          for (int ch = 0; ch < p.nchunks; ++ch) {
            if (!wait_relaxed(&x_empty[rx.idx], rx.phase ^ 1u, p.ctl, abort_flag)) goto loader_done;
            mbar_arrive_expect_tx(&x_full[rx.idx], p.x_stage_bytes);
            tma_load_4d(smem_x + (size_t)rx.idx * p.x_stage_bytes, &xmap, p0, d0, ch * kCC, un.n, &x_full[rx.idx]);
            rx.next((uint32_t)p.XS);
            ++issued;
          }
        }
      }
    loader_done:
      // Every copy this thread issued lands before the CTA can exit: the weights and
      // the last XS raw stages (the earlier ones were consumed, hence complete).
      drain_wait(w_full, 0, p.ctl);
      if (*abort_flag) {
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
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t b_desc0 = umma_desc_noswizzle(smem_addr(smem_b), (uint32_t)kBRows * 16u, 128);
      const uint32_t ks_blk_u = (uint32_t)p.KS * (kBBlockBytes >> 4);  // next kh block
      const uint32_t idesc0 = umma_idesc_tf32(128, 0), idesc_slot = umma_idesc_tf32(128, kSlotCols) - idesc0;
      bool ok = wait_issue(w_full, 0, p.ctl, abort_flag);
      // The issue queue holds only ~8 MMAs, and every instruction of this thread runs
      // slowly beside the other roles, so the hand-over between two chunks is kept off
      // the tensor core's critical path: the next chunk is computed and its barriers
      // tested while the current chunk's last plane of MMAs is still queued, and the
      // blocking waits that remain are only for what was not ready then.
      ChunkIter it;
      chunk_iter_init(p, it);
      Chunk<PP> cur, nxt;
      bool have = ok && next_chunk<PP, KSS>(p, it, cur, tmem_base, b_desc0, idesc0, idesc_slot);
      Ring ra;
      uint32_t empty_par = 0;  // per slot: uses so far, mod 2
      if (have) {
#pragma unroll
        for (int pi = 0; pi < PP; ++pi) {
          if (ok && cur.opens[pi]) {
            const uint32_t sl = cur.open_slot[pi];
            ok = wait_issue(&acc_empty[sl], ((empty_par >> sl) & 1u) ^ 1u, p.ctl, abort_flag);
            empty_par ^= 1u << sl;
          }
        }
        ok = ok && wait_issue(&a_full[ra.idx], ra.phase, p.ctl, abort_flag);
        tc_fence_after();
      }
      while (have && ok) {
        const uint32_t a0 = tmem_base + p.a_col0 + ra.idx * (uint32_t)kAStageCols;
        // The first plane of the chunk.
        issue_chunk<KSS>(cur.dc1[0], a0, cur.b[0], cur.id1[0], ks_blk_u);
        if (cur.run2[0]) issue_chunk<KSS>(tmem_base, a0, cur.b[0] + cur.n2off[0], cur.id2[0], ks_blk_u);
        if (cur.closes[0]) umma_commit(&acc_full[cur.close_slot[0]]);
        // Look ahead while those MMAs execute.
        const bool have_n = next_chunk<PP, KSS>(p, it, nxt, tmem_base, b_desc0, idesc0, idesc_slot);
        Ring ra_n = ra;
        ra_n.next((uint32_t)p.AST);
        // The next chunk's barriers, tested in one go (the tests' latencies overlap):
        // the slots its planes open (an unused test reads a completed phase of the
        // A barrier instead) and its A stage.
        bool rdy[PP + 1];
        {
          const uint32_t a_bar = smem_addr(&a_full[ra_n.idx]);
          uint32_t bar[PP], par[PP];
#pragma unroll
          for (int pi = 0; pi < PP; ++pi) {
            const bool t = have_n && nxt.opens[pi];
            bar[pi] = t ? smem_addr(&acc_empty[nxt.open_slot[pi]]) : a_bar;
            par[pi] = t ? (((empty_par >> nxt.open_slot[pi]) & 1u) ^ 1u) : (ra_n.phase ^ 1u);
          }
          test_wait_n<PP>(bar, par, a_bar, ra_n.phase, rdy);
#pragma unroll
          for (int pi = 0; pi < PP; ++pi) rdy[pi] = rdy[pi] || !(have_n && nxt.opens[pi]);
          rdy[PP] = rdy[PP] || !have_n;
        }
        // Orders the next chunk's MMAs after the syncs just observed (the fence costs
        // the issuing thread a few hundred cycles: taken here, the queue covers it).
        tc_fence_after();
        // The chunk's other planes.
#pragma unroll
        for (int pi = 1; pi < PP; ++pi) {
          if (cur.valid[pi]) {
            const uint32_t ap = a0 + (uint32_t)(pi * KSS * kKStepCols);
            issue_chunk<KSS>(cur.dc1[pi], ap, cur.b[pi], cur.id1[pi], ks_blk_u);
            if (cur.run2[pi]) issue_chunk<KSS>(tmem_base, ap, cur.b[pi] + cur.n2off[pi], cur.id2[pi], ks_blk_u);
            if (cur.closes[pi]) umma_commit(&acc_full[cur.close_slot[pi]]);
          }
        }
        umma_commit(&a_empty[ra.idx]);
        if (!have_n) break;
        // What the look-ahead found not ready yet.
#pragma unroll
        for (int pi = 0; pi < PP; ++pi) {
          if (nxt.opens[pi]) {
            const uint32_t sl = nxt.open_slot[pi];
            if (!rdy[pi] && !(ok = wait_issue(&acc_empty[sl], ((empty_par >> sl) & 1u) ^ 1u, p.ctl, abort_flag)))
              break;
            empty_par ^= 1u << sl;
          }
        }
        if (!ok) break;
        if (!rdy[PP] && !(ok = wait_issue(&a_full[ra_n.idx], ra_n.phase, p.ctl, abort_flag))) break;
        bool all_ready = rdy[PP];
#pragma unroll
        for (int pi = 0; pi < PP; ++pi) all_ready = all_ready && rdy[pi];
        if (!all_ready) tc_fence_after();
        cur = nxt;
        ra = ra_n;
      }
      // Wait until every MMA issued above has finished reading its operands and
      // writing TMEM, whatever the path out of the loop.
      umma_commit(mma_done);
      drain_wait(mma_done, 0, p.ctl);
    }
  } else if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps) {
    // ------------------------------------------------------------ A producers
    const int q = warp & 3;
    const int m = q * 32 + lane;  // TMEM lane = position within the tile
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    Ring ra, rx;
    for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
      const Unit un = decode_unit(p, u);
      for (int d0 = un.od0; d0 < un.od1 + 2; d0 += PP) {
        const int npl = min(PP, un.od1 + 2 - d0);
        for (int ch = 0; ch < p.nchunks; ++ch) {
          if (!warp_wait_relaxed(&x_full[rx.idx], rx.phase, p.ctl, abort_flag)) goto producer_done;
          if (!warp_wait_relaxed(&a_empty[ra.idx], ra.phase ^ 1u, p.ctl, abort_flag)) goto producer_done;
          tc_fence_after();
          const float* raw = reinterpret_cast<const float*>(smem_x + (size_t)rx.idx * p.x_stage_bytes);
          const uint32_t acol = tmem_base + lane_off + p.a_col0 + ra.idx * (uint32_t)kAStageCols;
#pragma unroll
          for (int pi = 0; pi < PP; ++pi) {
            if (pi < npl) {
#pragma unroll
              for (int ks = 0; ks < KSS; ++ks) {
#pragma unroll
                for (int kh = 0; kh < 3; ++kh) {
                  float v[16];
#pragma unroll
                  for (int c = 0; c < 8; ++c) {
                    const int cl = ks * 8 + c;
                    split_tf32(raw[(cl * PP + pi) * p.NPOS + m + kh * p.W], v[c], v[8 + c]);
                  }
                  tmem_st16(acol + (uint32_t)(((pi * KSS + ks) * 3 + kh) * 16), v);
                }
              }
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&x_empty[rx.idx]);
            mbar_arrive(&a_full[ra.idx]);
          }
          rx.next((uint32_t)p.XS);
          ra.next((uint32_t)p.AST);
        }
      }
    }
  producer_done:;
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    // Two teams of four warps (one per TMEM lane quadrant) take alternating output
    // planes (pool-reduce: alternating plane pairs), all 16 channels each, so two
    // planes drain at once: a plane's epilogue is a chain of TMEM loads, shuffles
    // and hand-overs that takes longer than the plane's MMAs.
    const int q = warp & 3;                    // TMEM lane quadrant
    const int team = (warp - kEpiWarp0) >> 2;
    const int m = q * 32 + lane;
    const int et = tid - kEpiWarp0 * 32;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    const int PH = p.OH / 2, PW = p.OW / 2, PD = p.OD / 2;
    const uint32_t nslot = (uint32_t)p.NSLOT;
    // Tiles hold whole rows, so a lane has the same column in every tile.
    const int ow = m % p.W;
    const int r = m / p.W;  // row within the tile (tiles start on an even row)
    uint32_t kx_buf = 0, h_buf = 0;
    uint32_t gseq = 0, gpair = 0;  // output planes and plane pairs of this CTA's earlier units
    bool ok = true;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      const Unit un = decode_unit(p, u);
      const int p0 = un.g * 128;
      const int oh = (p0 + m) / p.W;
      const int planes = un.od1 - un.od0;
      float psum = 0.0f;
      float prev[kCout];  // the even plane of the pair: this position's scaled values
#pragma unroll
      for (int j = 0; j < kCout; ++j) prev[j] = 0.0f;
      for (int k = 0; k < planes; ++k) {
        const int od = un.od0 + k;
        const uint32_t i = gseq + (uint32_t)k;  // the plane's place in the slot ring
        const int owner = (EPI == IG3_EPI_POOL_REDUCE) ? (int)((gpair + (uint32_t)(k >> 1)) & 1u) : (int)(i & 1u);
        if (owner != team) continue;
        const uint32_t slot = i % nslot;
        // Every thread of the team takes the same verdict, so that none is left
        // waiting at a named barrier below for a warp that gave up.
        ok = named_bar_and(6 + team, 128, wait_relaxed(&acc_full[slot], (i / nslot) & 1u, p.ctl, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t taddr = lane_base + slot * (uint32_t)kSlotCols;
        float v[kCout], a1[kCout], a2[kCout];
        tmem_ld16(taddr, v);
        tmem_ld16(taddr + 16u, a1);
        tmem_ld16(taddr + 32u, a2);
        tmem_wait_ld();
        {
          // The slot's next use starts from [bias | 0 | 0] again.
          float bz[kCout];
          load_bias16(s_bias, bz);
          tmem_st16(taddr, bz);
#pragma unroll
          for (int j = 0; j < kCout; ++j) bz[j] = 0.0f;
          tmem_st16(taddr + 16u, bz);
          tmem_st16(taddr + 32u, bz);
        }
        // The slot goes back to the MMAs now: everything below works on registers and
        // shared memory (holding it through the exchanges and the pooling made the
        // issuing thread wait for slots: pool-reduce 363 -> 332 us).
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[slot]);
        // Output o takes block 0 at o, block 1 at o + 1 and block 2 at o + 2.
        float* xb = &s_kx[team][kx_buf][0][0];
        if (p.W > 32) {
          // A row crosses quadrants: lanes 30 and 31 take their neighbours from the
          // next quadrant's lanes 0 and 1 (in the last quadrant they are the row's
          // two wrap-around columns).  Two buffers alternate, one barrier per plane.
          kx_buf ^= 1u;
          if (q > 0 && lane < 2) {
            float4* d = reinterpret_cast<float4*>(xb + q * 48);
            if (lane == 0) {
#pragma unroll
              for (int i = 0; i < 4; ++i) d[i] = make_float4(a1[4 * i], a1[4 * i + 1], a1[4 * i + 2], a1[4 * i + 3]);
            }
            d += (lane == 0) ? 4 : 8;
#pragma unroll
            for (int i = 0; i < 4; ++i) d[i] = make_float4(a2[4 * i], a2[4 * i + 1], a2[4 * i + 2], a2[4 * i + 3]);
          }
          named_bar_sync(4 + team, 128);
        }
#pragma unroll
        for (int j = 0; j < kCout; ++j) {
          a1[j] = __shfl_down_sync(0xffffffffu, a1[j], 1);
          a2[j] = __shfl_down_sync(0xffffffffu, a2[j], 2);
        }
        if (p.W > 32 && q < 3 && lane >= 30) {
          // Lane 31 takes blocks 1 and 2 of the next quadrant's lane 0 and 1, lane 30
          // block 2 of its lane 0.
          const float4* src = reinterpret_cast<const float4*>(xb + (q + 1) * 48);
          const float4* s2 = src + ((lane == 31) ? 8 : 4);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 t = s2[i];
            a2[4 * i] = t.x; a2[4 * i + 1] = t.y; a2[4 * i + 2] = t.z; a2[4 * i + 3] = t.w;
          }
          if (lane == 31) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 t = src[i];
              a1[4 * i] = t.x; a1[4 * i + 1] = t.y; a1[4 * i + 2] = t.z; a1[4 * i + 3] = t.w;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kCout; ++j) v[j] += a1[j] + a2[j];
        if constexpr (EPI != IG3_EPI_POOL_REDUCE) {
          if (oh < p.OH && ow < p.OW) {
            store_position<EPI>(p, un.n, od, oh, ow, v);
          }
        } else if (od / 2 < PD && (od & 1) == 0) {
          // The 2x2x2 max is taken d-pair first: the even plane only keeps its scaled
          // values, so the shuffles and the exchange below run once per plane pair.
          // (The max of a set does not depend on the order, so this is exact.)
#pragma unroll
          for (int j = 0; j < kCout; ++j) prev[j] = v[j] * p.inv_div;
        } else if (od / 2 < PD) {
          // d-pair with the even plane, w-pair by lane shuffle, h-pair by shuffle
          // (W <= 16) or through shared memory (W = 32, 64).
#pragma unroll
          for (int j = 0; j < kCout; ++j) {
            const float z = fmaxf(prev[j], v[j] * p.inv_div);
            v[j] = fmaxf(z, __shfl_xor_sync(0xffffffffu, z, 1));
          }
          const bool even_w = (ow & 1) == 0, even_r = (r & 1) == 0;
          const int cell = (r >> 1) * (p.W >> 1) + (ow >> 1);  // pooled cell within the tile, < 32
          if (p.W <= 16) {
#pragma unroll
            for (int j = 0; j < kCout; ++j) v[j] = fmaxf(v[j], __shfl_xor_sync(0xffffffffu, v[j], p.W));
          } else {
            float4* hc = reinterpret_cast<float4*>(&s_h[team][h_buf][cell][0]);
            const int rot = (cell >> 1) & 3;
            h_buf ^= 1u;
            if (!even_r && even_w) {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                hc[i ^ rot] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
            named_bar_sync(1 + team, 128);
            if (even_r && even_w) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 t = hc[i ^ rot];
                v[4 * i] = fmaxf(v[4 * i], t.x);
                v[4 * i + 1] = fmaxf(v[4 * i + 1], t.y);
                v[4 * i + 2] = fmaxf(v[4 * i + 2], t.z);
                v[4 * i + 3] = fmaxf(v[4 * i + 3], t.w);
              }
            }
          }
          if (even_r && even_w && (oh >> 1) < PH && (ow >> 1) < PW) {
#pragma unroll
            for (int j = 0; j < kCout; ++j) psum += v[j];
          }
        }
      }
      if constexpr (EPI == IG3_EPI_POOL_REDUCE) {
        // Fixed-order reduction of the unit's partial: lanes, then warps in order.
        // Both teams pass this barrier once per unit, also after a failed wait.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
        if (lane == 0) s_red[warp - kEpiWarp0] = psum;
        ok = named_bar_and(3, kEpiThreads, ok);
        if (ok && et == 0) {
          float s = 0.0f;
          for (int w = 0; w < kEpiWarps; ++w) s += s_red[w];
          p.partial[u] = s;
        }
        named_bar_sync(3, kEpiThreads);
      }
      if (!ok) break;
      gseq += (uint32_t)planes;
      gpair += (uint32_t)((planes + 1) >> 1);
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

// Weights [16][Cin][27] -> blocks (kh, ks), each [khalf][kBRows][4]: rows [hi kd=2 kw=0 |
// hi kd=2 kw=1 | hi kd=2 kw=2 | hi kd=1 kw=0 | ... | hi kd=0 kw=2 | lo, the same nine]
// x 16 channels; channel ks*8 + khalf*4 + j of the row, zero past Cin.
__global__ void tc16_prep_weights(const float* __restrict__ w, float* __restrict__ blob, int Cin, int KS,
                                  int total) {
  // The conv kernel that follows may start now (programmatic dependent launch): only
  // its copy of these blocks waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int j = i & 3;
    int t = i >> 2;
    const int row = t % kBRows;
    t /= kBRows;
    const int khalf = t & 1;
    t >>= 1;
    const int ks = t % KS;
    const int kh = t / KS;
    const bool hi = row < 9 * kCout;
    const int rr = hi ? row : row - 9 * kCout;
    const int kd = 2 - rr / (3 * kCout);
    const int kw = (rr / kCout) % 3;
    const int co = rr % kCout;
    const int c = ks * 8 + khalf * 4 + j;
    const float v = (c < Cin) ? w[((size_t)co * Cin + c) * 27 + kd * 9 + kh * 3 + kw] : 0.0f;
    float h, l;
    split_tf32(v, h, l);
    blob[i] = hi ? h : l;
  }
}

// ------------------------------------------------------------------ host-side plan
struct Plan {
  bool ok = false;
  const char* why = "";
  Params prm;
  int kss = 1, pp = 1;
  size_t smem = 0;
};

size_t blob_bytes_for(int KS) { return (size_t)3 * KS * kBBlockBytes; }

// Chunk shapes the kernel is instantiated for: (K-steps, input planes) per A stage,
// and the number of A stages.  18 MMAs per chunk measured best: one plane of one
// K-step with three A stages ran pool-reduce at the same speed and the 16-channel
// sweep 17% slower than two K-steps of one plane with two stages.
constexpr int kShapes[][3] = {{2, 1, 2}, {1, 2, 2}, {1, 1, 2}};

// Cycles of one work unit of `planes` output planes: per input plane and K-step,
// nine MMAs (three kh x three split products) of N = 48 * nkd, about
// max(50, N/2 + 4) cycles each (measured: M = 128, K = 8 tf32 MMAs cost at least
// ~50 cycles whatever N is), plus ~900 cycles per chunk that the issuing thread
// spends between chunks without MMAs in flight (its waits, fences, commits and
// bookkeeping run at a fraction of an issue slot beside the other roles, and the
// MMA queue holds only ~8 MMAs).
double unit_cycles(int planes, int KS, int kss, int pp) {
  double mma = 0.0;
  for (int d = 0; d < planes + 2; ++d) {
    const int kd_hi = std::min(2, d), kd_lo = std::max(0, d - planes + 1);
    mma += 9.0 * KS * std::max(50.0, 24.0 * (kd_hi - kd_lo + 1) + 4.0);
  }
  const double chunks = (double)((planes + 2 + pp - 1) / pp) * (KS / kss);
  return mma + 900.0 * chunks;
}

Plan make_plan_uncached(int N, int Cin, int D, int H, int W, int Cout, int epi, int sms) {
  Plan pl;
  if (Cout != kCout) {
    pl.why = "the A-in-tensor-memory kernel takes 16 output channels";
    return pl;
  }
  if (W > 64 || 64 % W != 0) {
    pl.why = "W must divide 64 (tiles of whole input rows; a staged row of 128 + 2W positions is one copy box)";
    return pl;
  }
  if (epi == IG3_EPI_POOL_REDUCE && 64 % W != 0) {
    pl.why = "pool-reduce needs W to divide 64";
    return pl;
  }
  if ((H * W) % 4 != 0) {
    pl.why = "H*W must be a multiple of 4 (16-byte channel rows)";
    return pl;
  }
  const int OD = D - 2, OH = H - 2;
  const int ks0 = (Cin + 7) / 8;
  const int npos = 128 + 2 * W;
  const int G = (OH * W + 127) / 128;
  const int step = (epi == IG3_EPI_POOL_REDUCE) ? 2 : 1;
  double best = 1e300;
  for (const auto& shape : kShapes) {
    const int kss = shape[0], pp = shape[1], ast = shape[2];
    if (ast > kMaxAStages) continue;
    if (kss == 2 && ks0 == 1) continue;
    const int KS = (ks0 + kss - 1) / kss * kss;
    const int nchunks = KS / kss;
    const uint32_t blob = (uint32_t)blob_bytes_for(KS);
    const uint32_t x_stage = (uint32_t)(pp * 8 * kss) * npos * 4u;
    const int a_cols = ast * pp * kss * kKStepCols;
    const int nslot = (kTmemCols - a_cols) / kSlotCols;
    // A chunk's windows span pp + 2 slots; at least one more lets the MMAs run ahead.
    if (nslot < pp + 3) continue;
    const uint32_t off_x = (blob + 1023u) / 1024u * 1024u;
    // static shared memory (~11.3 KB), alignment and barriers
    const long long avail =
        (long long)kSmemLimit - off_x - 12 * 1024 - (2 + 2 * ast + 2 * kMaxXStages + 2 * nslot) * 8;
    const int xs = (int)std::min<long long>(kMaxXStages, avail / (long long)x_stage);
    if (xs < 2) continue;
    for (int P = OD - (OD % step); P >= step; P -= step) {
      const int S = (OD + P - 1) / P;
      const int last = OD - (S - 1) * P;
      const long long units = (long long)N * G * S;
      if (units > 0x7fffffffLL) continue;
      const int grid = (int)std::min<long long>(units, sms);
      const double c_full = unit_cycles(P, KS, kss, pp), c_last = unit_cycles(last, KS, kss, pp);
      // Round-robin over the grid: CTA c takes units c, c + grid, ...; a unit is the
      // last split iff u % S == S - 1.  Exact up to 65536 units, bounded past that.
      double worst = 0.0;
      if (units <= 65536) {
        for (int c = 0; c < grid; ++c) {
          double t = 0.0;
          for (long long u = c; u < units; u += grid) t += (u % S == S - 1) ? c_last : c_full;
          worst = std::max(worst, t);
        }
      } else {
        worst = (double)((units + grid - 1) / grid) * std::max(c_full, c_last);
      }
      if (worst < best * (1.0 - 1e-9)) {
        best = worst;
        Params& p = pl.prm;
        std::memset(&p, 0, sizeof(p));
        p.N = N; p.Cin = Cin; p.D = D; p.H = H; p.W = W;
        p.OD = OD; p.OH = OH; p.OW = W - 2;
        p.KS = KS;
        p.nchunks = nchunks;
        p.NSLOT = nslot;
        p.G = G;
        p.S = S;
        p.P = P;
        p.units = (int)units;
        p.NPOS = npos;
        p.XS = xs;
        p.blob_bytes = blob;
        p.x_stage_bytes = x_stage;
        p.off_x = off_x;
        p.off_bar = off_x + (uint32_t)xs * x_stage;
        p.a_col0 = (uint32_t)(nslot * kSlotCols);
        pl.kss = kss;
        pl.pp = pp;
        p.AST = ast;
        pl.smem = std::max<size_t>(p.off_bar + (size_t)(2 + 2 * ast + 2 * xs + 2 * nslot) * 8, kMinSmem);
        pl.ok = true;
      }
    }
  }
  if (!pl.ok) pl.why = "the resident weights and two raw stages do not fit in shared memory";
  return pl;
}

Plan make_plan(int N, int Cin, int D, int H, int W, int Cout, int epi, int sms) {
  using Key = std::array<int, 8>;
  static std::mutex mu;
  static std::map<Key, Plan> cache;
  const Key key{N, Cin, D, H, W, Cout, epi, sms};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  Plan pl = make_plan_uncached(N, Cin, D, H, W, Cout, epi, sms);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 256) cache.clear();
  cache.emplace(key, pl);
  return pl;
}

template <int EPI, int KSS, int PP>
int launch(const Params& p, const CUtensorMap& xmap, size_t smem, int grid, cudaStream_t stream) {
  auto kernel = conv3d_tc16_kernel<EPI, KSS, PP>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e, "conv3d TC16: set shared memory size");
  // Programmatic dependent launch: the kernel's set-up overlaps the weight split.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, p, xmap);
  return count_launch(cuda_status(e, "conv3d TC16 kernel launch"));
}

template <int EPI>
int launch_epi(const Plan& pl, const Params& p, const CUtensorMap& xmap, int grid, cudaStream_t stream) {
  if (pl.kss == 1 && pl.pp == 2) return launch<EPI, 1, 2>(p, xmap, pl.smem, grid, stream);
  if (pl.kss == 2 && pl.pp == 1) return launch<EPI, 2, 1>(p, xmap, pl.smem, grid, stream);
  if (pl.kss == 1 && pl.pp == 1) return launch<EPI, 1, 1>(p, xmap, pl.smem, grid, stream);
  return fail(IG3_ERR_UNSUPPORTED, "conv3d TC16 path: no kernel variant for %d K-steps x %d planes", pl.kss, pl.pp);
}

}  // namespace tc16

// Sizes that do not depend on the plan or the device: the weight blocks for an even
// number of K-steps, partial sums for the finest plane split.
size_t conv3d_tc16_workspace(const Conv3dArgs& a) {
  const int ks2 = ((a.Cin + 7) / 8 + 1) / 2 * 2;
  const int G = (a.OH() * a.W + 127) / 128;
  const size_t partial = (a.epi == IG3_EPI_POOL_REDUCE) ? align_up((size_t)a.N * G * a.OD() * sizeof(float), 256) : 0;
  return align_up(tc16::blob_bytes_for(ks2), 256) + partial;
}

bool conv3d_tc16_applies(const Conv3dArgs& a, const char** why) {
  tc16::Plan pl = tc16::make_plan(a.N, a.Cin, a.D, a.H, a.W, a.Cout, a.epi, 148);
  if (why) *why = pl.why;
  return pl.ok;
}

int conv3d_tc16_launch(const Conv3dArgs& a) {
  using namespace tc16;
  const int sms = num_sms();
  if (sms <= 0) return fail(IG3_ERR_CUDA, "conv3d TC16 path: cannot query the SM count");
  if (reinterpret_cast<uintptr_t>(a.x) % 16 != 0)
    return fail(IG3_ERR_UNSUPPORTED, "conv3d TC16 path: x must be 16-byte aligned");
  Plan pl = make_plan(a.N, a.Cin, a.D, a.H, a.W, a.Cout, a.epi, sms);
  if (!pl.ok) return fail(IG3_ERR_UNSUPPORTED, "conv3d TC16 path: %s", pl.why);
  Params p = pl.prm;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int ks2 = ((a.Cin + 7) / 8 + 1) / 2 * 2;
  p.x = a.x;
  p.wblob = reinterpret_cast<const float*>(ws);
  p.bias = a.b;
  p.y = a.y;
  p.partial = reinterpret_cast<float*>(ws + align_up(blob_bytes_for(ks2), 256));
  p.inv_div = (a.epi == IG3_EPI_POOL_REDUCE) ? 1.0f / a.divisor : 1.0f;
  p.ctl = wait_ctl();
  if (!p.ctl.status) return fail(IG3_ERR_CUDA, "conv3d TC16 path: device status word unavailable");

  const int total = (int)(blob_bytes_for(p.KS) / 4);
  tc16_prep_weights<<<std::min((total + 255) / 256, 4 * sms), 256, 0, a.stream>>>(a.w, const_cast<float*>(p.wblob),
                                                                                   a.Cin, p.KS, total);
  int st = count_launch(cuda_status(cudaGetLastError(), "conv3d TC16 weight prep launch"));
  if (st != IG3_OK) return st;

  // x as a 4-D tensor [N][Cin][D][H*W] of floats; the box is [8*KSS][PP][NPOS].
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(IG3_ERR_CUDA, "conv3d TC16 path: cuTensorMapEncodeTiled is not available");
  CUtensorMap xmap;
  const cuuint64_t HW = (cuuint64_t)a.H * (cuuint64_t)a.W;
  const cuuint64_t dims[4] = {HW, (cuuint64_t)a.D, (cuuint64_t)a.Cin, (cuuint64_t)a.N};
  const cuuint64_t strides[3] = {HW * 4u, HW * (cuuint64_t)a.D * 4u, HW * (cuuint64_t)a.D * (cuuint64_t)a.Cin * 4u};
  const cuuint32_t box[4] = {(cuuint32_t)p.NPOS, (cuuint32_t)pl.pp, (cuuint32_t)(8 * pl.kss), 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(a.x), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IG3_ERR_CUDA, "conv3d TC16 path: tensor map encoding failed (%d)", (int)r);

  const int grid = std::min(p.units, sms);
  switch (a.epi) {
    case IG3_EPI_NONE: st = launch_epi<IG3_EPI_NONE>(pl, p, xmap, grid, a.stream); break;
    case IG3_EPI_TANH_MISH: st = launch_epi<IG3_EPI_TANH_MISH>(pl, p, xmap, grid, a.stream); break;
    default: st = launch_epi<IG3_EPI_POOL_REDUCE>(pl, p, xmap, grid, a.stream); break;
  }
  if (st != IG3_OK || a.epi != IG3_EPI_POOL_REDUCE) return st;
  const long long cells = (long long)(p.OD / 2) * (p.OH / 2) * (p.OW / 2);
  return pool_reduce_finalize(p.partial, a.N, p.G * p.S, (float)(1.0 / (double)cells), a.bias2, kCout, a.y,
                              a.stream);
}

}  // namespace ig3
