// Tensor-core conv3d (valid, stride 1, 3x3x3) on sm_103a: an implicit GEMM on
// tcgen05 with split-TF32 operands and the epilogue fused into the same kernel.
//
// Definition followed ("Kimi-K2.6__l2_p47", the per-output loop and its NCDHW index
// check; the implicit-GEMM view M = output positions, N = Cout, K = Cin*27 is the
// page's own framing):
//   conv[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw] * x[n,c,od+kd,oh+kh,ow+kw]
//
// GEMM mapping.  M = 128 consecutive positions p = h*W + w of one input plane (the
// row length is the INPUT width W, so a tile may include the two wrap-around
// columns w = W-2, W-1, which are computed and discarded).  For tap (kd, kh, kw)
// the A operand of output position p is the input at position p + kh*W + kw of
// plane od + kd, so every tap of an input plane reads the SAME shared-memory tile
// with the descriptor's start address moved by (kh*W + kw) * 16 bytes: no im2col.
// A is stored K-major as [channel group of 4][position][4 channels] (16 B per
// position per group: the canonical no-swizzle core-matrix layout with SBO = 128 B
// and LBO = positions * 16 B).
//
// Precision.  fp32 operands are split into hi (tf32-exact, low 13 bits cleared) and
// lo = x - hi; the tensor core truncates operands to tf32, so hi is exact and
//   acc += A_hi*B_hi + A_hi*B_lo + A_lo*B_hi
// keeps the product to about 2^-21 relative with fp32 accumulation.  Each of the
// three products is one MMA into the same accumulator columns.
//
// Window MMAs.  Input plane d feeds output planes d-2, d-1, d through the kd = 2, 1, 0
// weights.  An M = 128, K = 8 tf32 MMA reads its whole A tile (4 KB) and its B rows
// (32 B per column) from shared memory at ~128 B per cycle, so below N ~ 128 the
// operand reads, not the arithmetic, set its cost (measured alone: 48 cycles at
// N = 48, 58 at 96, 66 at 128, 98 at 192).  Small MMAs are therefore merged: the
// accumulators of consecutive output planes sit in adjacent TMEM slots (Cout columns
// each) and the weights of one (kh, kw) tap are stored with rows [kd=2 | kd=1 |
// kd=0], so ONE MMA with N = 3*Cout applies all three kd of an input plane (KDM 3,
// Cout <= 80).  A unit's P output planes use slots 0..P-1, so the window never wraps;
// planes at the ends of a unit use the sub-window of the kd that fall inside it.
// Every MMA accumulates: the slots start at the bias and the epilogue writes the
// bias back after reading a slot.  For Cout > 80 (3*Cout > 256, the largest N) each
// kd is its own MMA (KDM 1) and the slots form a ring.
//
// Window over kd and kw (KDM 9, Cout 16, not pool-reduce).  The A tile is shifted by
// kh*W only, and one MMA with N = 9*Cout (three kd x three kw) applies an input
// plane to three output planes: slot = [kw=0 | kw=1 | kw=2] x Cout, and the
// epilogue adds block kw of position o + kw into output o (a lane shuffle; across a
// quadrant boundary, a shared-memory hand-over).  Tiles must hold whole input rows
// (W divides 128), so the shift never leaves the tile.
//
// Data flow (persistent CTAs, one per SM, 512 threads, warp-specialised):
//   warp 0      weight producer: 1-D bulk copies (TMA) of pre-split K-step blocks from
//               the workspace into a ring of stages (one stage = the K-steps of one
//               channel chunk for two consecutive taps; KDM 9: for one kh), or all
//               blocks once when they fit (resident);
//   warp 1      TMEM owner and MMA issuer (one thread; descriptors are formed once
//               and advanced by adds; the nine taps are unrolled);
//   warps 2-7   input convert: coalesced loads of x, hi/lo split, K-major stores;
//   warps 8-15  epilogue, two groups of four (one warp per TMEM lane quadrant each):
//               tcgen05.ld, zeroing tcgen05.st, bias, activation or pool-reduce, stores.
// A work unit is (batch item n, group of T position tiles, range of P output planes).
// Input planes stream through a 2-stage A buffer (one channel chunk per stage), so
// the convert of the next chunk and the epilogue of finished planes overlap the MMAs.
// The plan (T, chunk size, resident or streamed weights, P) comes from a cycle model
// of the issue and execution rates above and of the persistent schedule.
//
// Pool-reduce ("Kimi-K2.6__l2_p8": /divisor, MaxPool3d(2) floor mode, global mean,
// +bias2, sum over channels): TMEM lane = position, so the w-pair max is a lane
// shuffle, the h-pair max a shuffle (W <= 16) or a shared-memory exchange between
// warps (W = 32, 64), and the d-pair max combines consecutive planes.  Each unit
// writes one partial sum; a second, fixed-order kernel forms out[n]
// (deterministic).
//
// Every wait is bounded (ig3_device.cuh); on a timeout all roles stop, in-flight
// copies and MMAs are drained and TMEM is freed before the CTA exits.
#include <algorithm>
#include <array>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>

#include "conv3d_tc_kernel.cuh"

namespace ig3 {
namespace {

using namespace tc;

// Weights [Cout][Cin][27] -> pre-split K-step blocks, each [khalf][rows][4] (rows
// of 4 consecutive channels, the two channel halves of the K-step one after the
// other), channels past Cin zero:
//   KDM 3:       block (khw * KS + ks), rows [hi kd=2 | hi kd=1 | hi kd=0 | lo kd=2 |
//                lo kd=1 | lo kd=0] x Cout, so any run of adjacent kd is a contiguous
//                row range;
//   KDM 3, HL:   block (khw * KS + ks), rows [hi kd=2 | lo kd=2 | hi kd=1 | lo kd=1 |
//                hi kd=0 | lo kd=0 | hi kd=2 | 0 | hi kd=1 | 0 | hi kd=0 | 0] x Cout;
//   KDM 9:       block (kh * KS + ks), rows [hi kd=2 kw=0 | hi kd=2 kw=1 | hi kd=2 kw=2 |
//                hi kd=1 kw=0 | ... | hi kd=0 kw=2 | lo, the same nine] x Cout;
//   KDM 1:       block ((kd * 9 + khw) * KS + ks), rows [hi | lo] x Cout.
// khw = kh * 3 + kw.
__host__ __device__ int blob_rows(int kdm, int hl, int Cout) {
  return (kdm == 9 ? 18 : kdm == 3 ? (hl ? 12 : 6) : 2) * Cout;
}
size_t blob_floats(int kdm, int hl, int KS, int Cout) {
  return (size_t)(kdm == 9 ? 3 : kdm == 3 ? 9 : 27) * KS * 2 * blob_rows(kdm, hl, Cout) * 4;
}

__global__ void conv3d_tc_prep_weights(const float* __restrict__ w, float* __restrict__ blob, int Cin, int Cout,
                                       int KS, int kdm, int hl, int total) {
  const int rows = blob_rows(kdm, hl, Cout);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int j = i & 3;
    int r = i >> 2;
    const int row = r % rows;
    r /= rows;
    const int khalf = r & 1;
    r >>= 1;
    const int ks = r % KS;
    const int blk = r / KS;
    int tap, co;
    bool hi, zero = false;
    if (kdm == 3 && hl) {
      const int half = row / (6 * Cout);  // 0: [hi | lo] per kd, 1: [hi | 0] per kd
      const int rr = row % (6 * Cout);
      const int kd = 2 - rr / (2 * Cout);
      hi = (rr % (2 * Cout)) < Cout;
      zero = (half == 1) && !hi;
      co = rr % Cout;
      tap = kd * 9 + blk;  // blk = khw
    } else if (kdm == 9) {
      hi = row < 9 * Cout;
      const int rr = hi ? row : row - 9 * Cout;
      const int kd = 2 - rr / (3 * Cout);
      const int kw = (rr / Cout) % 3;
      co = rr % Cout;
      tap = kd * 9 + blk * 3 + kw;  // blk = kh
    } else if (kdm == 3) {
      hi = row < 3 * Cout;
      const int rr = hi ? row : row - 3 * Cout;
      const int kd = 2 - rr / Cout;
      co = rr % Cout;
      tap = kd * 9 + blk;  // blk = khw
    } else {
      hi = row < Cout;
      co = hi ? row : row - Cout;
      tap = blk;           // blk = kd * 9 + khw
    }
    const int c = ks * 8 + khalf * 4 + j;
    const float v = (c < Cin) ? w[((size_t)co * Cin + c) * 27 + tap] : 0.0f;
    float h, l;
    split_tf32(v, h, l);
    blob[i] = zero ? 0.0f : (hi ? h : l);
  }
}

// ------------------------------------------------------------------ host-side plan
struct Plan {
  bool ok = false;
  const char* why = "";
  TcParams prm;
  size_t smem = 0;
  size_t blob_bytes = 0, partial_bytes = 0;
};

int positions_tiles(int OH, int W, int T) { return ((OH * W) + T * 128 - 1) / (T * 128); }

// Cycle estimate of one input plane (per SM): nkd output planes fed; per (tap, K-step,
// tile) three MMAs (two with HL).  Measured inside the kernel, an MMA costs about
// max(70, N/2 + 5) cycles (one thread issues them; N/2 is the M = 128, K = 8 execution
// time) and every streamed weight stage ~250 more.  The chunk's input convert runs
// alongside: ~0.9 cycles per value when the convert warps load x themselves (latency
// bound), ~0.35 when a bulk-copy loader stages it ahead.  Each A chunk also costs
// the issuing thread ~900 cycles of hand-over (mbarrier tests, which queue behind the
// MMAs' shared-memory operand reads, and commits), not hidden by the shallow MMA queue.
//
// KDM 9: three MMAs (one per split product) per (kh, K-step, tile) with N = 3 * nkd *
// Cout.  At this N an MMA is bound as much by shared-memory reads (A 4 KB + B 32 B
// per column, at 128 B per cycle) as by its execution, and the input convert's
// traffic (raw copy in, raw read, hi and lo out) shares the same port.
double plane_cycles(int kdm, int hl, int nkd, int Cout, int KS, int nchunks, int T, bool res, int tps, int npos,
                    bool xstage) {
  if (kdm == 9) {
    const double n = 3.0 * nkd * Cout;
    const double mmas = 3.0 * KS * T * 3.0;
    const double exec = mmas * (0.5 * n + 5.0) + (res ? 0.0 : 250.0 * 3.0 * nchunks);
    const double port = (mmas * (4096.0 + 32.0 * n) + npos * 8.0 * KS * 16.0) / 128.0;
    const double conv = (xstage ? 0.35 : 0.9) * npos * (8.0 * KS);
    return 1.1 * std::max(std::max(exec, port), conv) + 900.0 * nchunks;
  }
  const int mmas_per_step = (kdm == 3) ? (hl ? 2 : 3) : 3 * nkd;
  const int n = (kdm == 3) ? nkd * Cout * (hl ? 2 : 1) : Cout;
  const double mmas = 9.0 * KS * T * mmas_per_step;
  const double stages = res ? 0.0 : (double)((9 + tps - 1) / tps) * nchunks * (kdm == 3 ? 1 : nkd);
  const double mma = mmas * std::max(70.0, 0.5 * n + 5.0) + 250.0 * stages;
  const double conv = (xstage ? 0.35 : 0.9) * npos * (8.0 * KS);
  return std::max(mma, conv) + 900.0 * nchunks;  // A hand-over per chunk (mbarrier tests, commits)
}

double unit_cycles(int kdm, int hl, int planes, int Cout, int KS, int nchunks, int T, bool res, int tps, int npos,
                   bool xstage) {
  double c = 0.0;
  for (int d = 0; d < planes + 2; ++d) {
    const int kd_hi = std::min(2, d), kd_lo = std::max(0, d - planes + 1);
    c += plane_cycles(kdm, hl, kd_hi - kd_lo + 1, Cout, KS, nchunks, T, res, tps, npos, xstage);
  }
  return c;
}

// flags: kNoKwWindow keeps the kd x kw window (KDM 9) out of the plan.  Its epilogue
// takes the kw = 1, 2 blocks of a row's last two positions from outside the tile, so
// it relies on those two columns being the discarded wrap-around columns of a valid
// convolution; with zero padding on chip the stored columns are shifted and can
// include them.
enum : int { kNoKwWindow = 1 };

Plan make_plan_uncached(int N, int Cin, int D, int H, int W, int Cout, int epi, int sms, int flags) {
  Plan pl;
  if (Cout % 16 != 0 || Cout > 128) {
    pl.why = "Cout must be a multiple of 16 and at most 128";
    return pl;
  }
  if (epi == IG3_EPI_POOL_REDUCE && (W > 64 || 64 % W != 0)) {
    pl.why = "pool-reduce on tensor cores needs W to divide 64";
    return pl;
  }
  if (W > 1024) {
    pl.why = "W above 1024";
    return pl;
  }
  const int OD = D - 2, OH = H - 2;
  // Cout 16 with tiles of whole input rows (W divides 128): kw joins kd inside the
  // MMA's N (the epilogue's shifted sum never crosses a tile).  Not for pool-reduce:
  // its epilogue, not the MMAs, bounds it, and the shift exchange adds to it.
  const int kdm = (epi != IG3_EPI_POOL_REDUCE && Cout == 16 && W <= 128 && 128 % W == 0 && !(flags & kNoKwWindow)) ? 9
                  : (3 * Cout <= 256)                                                      ? 3
                                                                                           : 1;
  const int hl = (kdm == 3 && 6 * Cout <= 256) ? 1 : 0;
  const int ks0 = (Cin + 7) / 8;
  const int step = (epi == IG3_EPI_POOL_REDUCE) ? 2 : 1;
  double best = 1e300;
  for (const Variant& v : kVariants) {
    if (v.kdm != kdm || v.hl != hl) continue;
    const int T = v.t, kss = v.kss, tps = v.tps;
    const bool res = v.res != 0;
    const int KS = (ks0 + kss - 1) / kss * kss;
    const int nchunks = KS / kss;
    const int nslot = std::min(kMaxSlots, kTmemCols / (T * Cout * (kdm == 9 ? 3 : hl ? 2 : 1)));
    if (nslot < (kdm != 1 ? step : 4)) continue;
    const int npos = ((T * 128 + 2 * W + 2) + 7) / 8 * 8;
    const uint32_t a_half = (uint32_t)(2 * kss) * npos * 16u;
    const uint32_t a_stage = 2 * a_half;
    const uint32_t blk = (uint32_t)(2 * blob_rows(kdm, hl, Cout) * 16);
    const uint32_t blob = (uint32_t)(blob_floats(kdm, hl, KS, Cout) * 4);
    const uint32_t epi_bytes = ((epi == IG3_EPI_POOL_REDUCE) ? (uint32_t)(2 * 16 * 32 + T * Cout * 32) * 4u : 0u) +
                               (kdm == 9 ? 2u * 2u * (uint32_t)T * 4u * 24u * 4u : 0u);
    const uint32_t off_b = kAStages * a_stage;
    // 2 KB for static shared memory and alignment; barriers for the largest ring.
    const long long avail = (long long)kSmemLimit - off_b - epi_bytes - 2048 - 128 - 128 -
                            (6 + 2 * nslot + 2 * kMaxStages + 2 * kMaxXStages) * 8;
    if (avail <= 0) continue;
    int sb = 0;
    if (res) {
      if ((long long)blob > avail) continue;
    } else {
      sb = (int)std::min<long long>(kMaxStages, avail / ((long long)tps * kss * blk));
      // At least two stages (one fills while the other is read) and three taps in flight.
      if (sb < 2 || sb * tps < 3) continue;
    }
    // Raw input stages for the bulk-copy loader in what is left (at least two).
    const uint32_t x_stage = (uint32_t)(8 * kss) * npos * 4u;
    const long long left = avail - (res ? (long long)blob : (long long)sb * tps * kss * blk);
    int xs = (int)std::min<long long>(kMaxXStages, left / x_stage);
    if (xs < 2) xs = 0;
    // Planes per unit: with KDM 3 and 9 a unit's planes must fit the slots.
    const int pmax = (kdm != 1) ? std::min(OD, nslot) : OD;
    const int G = positions_tiles(OH, W, T);
    for (int P = pmax - (pmax % step == 0 ? 0 : 1); P >= step; P -= step) {
      const int S = (OD + P - 1) / P;
      const int last = OD - (S - 1) * P;
      const long long units = (long long)N * G * S;
      const int grid = (int)std::min<long long>(units, sms);
      const double c_full = unit_cycles(kdm, hl, P, Cout, KS, nchunks, T, res, tps, npos, xs > 0);
      const double c_last = unit_cycles(kdm, hl, last, Cout, KS, nchunks, T, res, tps, npos, xs > 0);
      // Round-robin over the grid: CTA c takes units c, c + grid, ...; a unit is
      // the last split iff u % S == S - 1.  Simulated exactly up to 65536 units; past
      // that, bounded by the rounds times the dearer unit (the difference is small
      // once every CTA takes many units).
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
        TcParams& p = pl.prm;
        std::memset(&p, 0, sizeof(p));
        p.N = N; p.Cin = Cin; p.D = D; p.H = H; p.W = W; p.Cout = Cout;
        p.OD = OD; p.OH = OH; p.OW = W - 2;
        p.epi = epi;
        p.KS = KS;
        p.KSS = kss;
        p.nchunks = nchunks;
        p.T = T;
        p.NPOS = npos;
        p.KDM = kdm;
        p.HL = hl;
        p.NSLOT = nslot;
        p.G = G;
        p.S = S;
        p.P = P;
        p.units = (int)units;
        p.resident = res ? 1 : 0;
        p.SB = sb;
        p.TPS = tps;
        p.a_half_bytes = a_half;
        p.a_stage_bytes = a_stage;
        p.b_block_bytes = blk;
        p.blob_bytes = blob;
        p.off_b = off_b;
        p.XS = xs;
        p.x_stage_bytes = x_stage;
        p.off_epi = off_b + (res ? blob : (uint32_t)(sb * tps * kss) * blk);
        p.off_x = (p.off_epi + epi_bytes + 127) / 128 * 128;
        p.off_bar = p.off_x + (uint32_t)xs * x_stage;
        pl.smem = std::max<size_t>(p.off_bar + (6 + 2 * (size_t)nslot + 2 * (size_t)sb + 2 * (size_t)xs) * 8, kMinSmem);
        pl.ok = true;
      }
    }
  }
  if (!pl.ok) {
    pl.why = "no tiling fits in shared memory";
    return pl;
  }
  // Sizes that do not depend on the plan (nor on the device): the blob padded to a
  // multiple of 4 K-steps, partials for the finest possible split.
  pl.blob_bytes = align_up(blob_floats(kdm, hl, (ks0 + 3) / 4 * 4, Cout) * 4, 256);
  pl.partial_bytes =
      (epi == IG3_EPI_POOL_REDUCE) ? align_up((size_t)N * positions_tiles(OH, W, 1) * OD * sizeof(float), 256) : 0;
  return pl;
}

// Plans are cached per (shape, epilogue, SM count): the search above simulates the
// persistent schedule and is not free.
Plan make_plan(int N, int Cin, int D, int H, int W, int Cout, int epi, int sms, int flags = 0) {
  using Key = std::array<int, 9>;
  static std::mutex mu;
  static std::map<Key, Plan> cache;
  const Key key{N, Cin, D, H, W, Cout, epi, sms, flags};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  Plan pl = make_plan_uncached(N, Cin, D, H, W, Cout, epi, sms, flags);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 256) cache.clear();
  cache.emplace(key, pl);
  return pl;
}

}  // namespace

const char* conv3d_tc_unsupported_reason(int N, int Cin, int D, int H, int W, int Cout, int epi) {
  static thread_local char buf[128];
  Plan pl = make_plan(N, Cin, D, H, W, Cout, epi, 148);
  if (pl.ok) return "";
  snprintf(buf, sizeof(buf), "%s", pl.why);
  return buf;
}

// Zero padding on chip: the kernel runs the valid convolution over a virtual padded
// volume.  When the convert can load aligned quads (W % 4 == 0, x 16-byte aligned,
// pad <= 4, and not pool-reduce, whose 2x2 pairs need stored and virtual columns of
// the same parity) virtual column 0 is real column -4 and the row pitch W plus
// pad + 2 rounded up to 4 (so that the last stored output, at virtual column
// W + pad + 1, lies inside the row); else column 0 is real column -pad and the pitch
// W + 2*pad.  Either way every position a stored output reads beyond the real row
// (the right border) is inside the row or the next virtual row's left border, which
// is zero.
struct VirtualDims {
  int D, H, W, col0;
  bool vec;
};
VirtualDims virtual_dims(const Conv3dArgs& a, bool x_aligned) {
  VirtualDims v{a.D + 2 * a.pad, a.H + 2 * a.pad, a.W + 2 * a.pad, a.pad, false};
  if (a.pad > 0 && x_aligned && a.W % 4 == 0 && a.pad <= 4 && a.epi != IG3_EPI_POOL_REDUCE) {
    v.W = a.W + (a.pad + 2 + 3) / 4 * 4;
    v.col0 = 4;
    v.vec = true;
  }
  return v;
}

size_t conv3d_tc_workspace(const Conv3dArgs& a) {
  if (a.pad > 0) {
    // Sized for either virtual pitch (the choice depends on x's alignment at the call).
    size_t ws = 0;
    for (bool aligned : {false, true}) {
      const VirtualDims v = virtual_dims(a, aligned);
      Plan pl = make_plan(a.N, a.Cin, v.D, v.H, v.W, a.Cout, a.epi, 148, kNoKwWindow);
      if (pl.ok) ws = std::max(ws, pl.blob_bytes + pl.partial_bytes);
    }
    return ws;
  }
  Plan pl = make_plan(a.N, a.Cin, a.D, a.H, a.W, a.Cout, a.epi, 148);
  const size_t own = pl.ok ? pl.blob_bytes + pl.partial_bytes : 0;
  // Either kernel may run (the A-in-tensor-memory one needs x 16-byte aligned).
  return conv3d_tc16_applies(a, nullptr) ? std::max(own, conv3d_tc16_workspace(a)) : own;
}

int conv3d_tc_launch(const Conv3dArgs& a) {
  const bool x_aligned = reinterpret_cast<uintptr_t>(a.x) % 16 == 0;
  if (a.pad == 0 && x_aligned && conv3d_tc16_applies(a, nullptr)) return conv3d_tc16_launch(a);
  const int sms = num_sms();
  if (sms <= 0) return fail(IG3_ERR_CUDA, "conv3d TC path: cannot query the SM count");
  const VirtualDims vd = virtual_dims(a, x_aligned);
  Plan pl = make_plan(a.N, a.Cin, vd.D, vd.H, vd.W, a.Cout, a.epi, sms, a.pad > 0 ? kNoKwWindow : 0);
  if (!pl.ok) return fail(IG3_ERR_UNSUPPORTED, "conv3d TC path: %s", pl.why);
  TcParams p = pl.prm;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  p.x = a.x;
  p.wblob = reinterpret_cast<const float*>(ws);
  p.bias = a.b;
  p.y = a.y;
  p.partial = reinterpret_cast<float*>(ws + pl.blob_bytes);
  p.inv_div = (a.epi == IG3_EPI_POOL_REDUCE) ? 1.0f / a.divisor : 1.0f;
  if (a.pad == 0) {
    p.vec = ((size_t)a.H * a.W % 4 == 0 && x_aligned) ? 1 : 0;
    if (!p.vec) p.XS = 0;  // bulk copies need 16-byte aligned rows
  } else {
    p.pad = a.pad;
    p.Dr = a.D;
    p.Hr = a.H;
    p.Wr = a.W;
    p.col0 = vd.col0;
    p.ow_off = vd.col0 - a.pad;
    p.OW = a.OW();
    p.vec = vd.vec ? 1 : 0;
    p.XS = 0;  // the convert warps load x themselves and fill the border
  }
  p.ctl = wait_ctl();
  if (!p.ctl.status) return fail(IG3_ERR_CUDA, "conv3d TC path: device status word unavailable");

  const int total = (int)blob_floats(p.KDM, p.HL, p.KS, p.Cout);
  conv3d_tc_prep_weights<<<std::min((total + 255) / 256, 4 * sms), 256, 0, a.stream>>>(
      a.w, const_cast<float*>(p.wblob), a.Cin, a.Cout, p.KS, p.KDM, p.HL, total);
  int st = count_launch(cuda_status(cudaGetLastError(), "conv3d TC weight prep launch"));
  if (st != IG3_OK) return st;

  const int grid = std::min(p.units, sms);
  switch (a.epi) {
    case IG3_EPI_NONE: st = launch_kernel<IG3_EPI_NONE>(p, pl.smem, grid, a.stream); break;
    case IG3_EPI_TANH_MISH: st = launch_kernel<IG3_EPI_TANH_MISH>(p, pl.smem, grid, a.stream); break;
    default: st = launch_kernel<IG3_EPI_POOL_REDUCE>(p, pl.smem, grid, a.stream); break;
  }
  if (st != IG3_OK || a.epi != IG3_EPI_POOL_REDUCE) return st;
  const long long cells = (long long)(p.OD / 2) * (p.OH / 2) * (p.OW / 2);
  return pool_reduce_finalize(p.partial, a.N, p.G * p.S, (float)(1.0 / (double)cells), a.bias2, a.Cout, a.y,
                              a.stream);
}

}  // namespace ig3
