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
// keeps the product to about 2^-21 relative with fp32 accumulation.  For
// Cout <= 64 the first two terms are one MMA with B = [B_hi ; B_lo] (N = 2*Cout)
// into 2*Cout accumulator columns (summed in the epilogue) and the third is a
// second MMA into the first Cout columns; for Cout > 64 three MMAs of N = Cout.
//
// Data flow (persistent CTAs, one per SM, 512 threads, warp-specialised):
//   warp 0      weight producer: 1-D bulk copies (TMA) of pre-split K-step blocks
//               [hi rows ; lo rows] from the workspace into a ring of stages (one
//               stage = the K-steps of one tap, up to 16 KB), or all blocks once
//               when they fit (resident weights);
//   warp 1      TMEM owner and MMA issuer (one thread; descriptors are formed once
//               and advanced by adds, which keeps issue at the tensor pipe's rate);
//   warps 2-7   input convert: coalesced loads of x, hi/lo split, K-major stores;
//   warps 8-15  epilogue, two groups of four (one warp per TMEM lane quadrant each):
//               tcgen05.ld, bias, activation or pool-reduce, stores.
// A work unit is (batch item n, group of T position tiles, range of output
// planes).  Input planes stream through a 2-stage A buffer; each input plane d
// feeds output planes d, d-1, d-2 (kd = 0, 1, 2), whose accumulators live in a
// 4-slot TMEM ring, so the epilogue of one plane overlaps the MMAs of the next.
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
#include <cmath>
#include <cstdio>
#include <cstring>

#include "conv3d_tc_kernel.cuh"

namespace ig3 {
namespace {

using namespace tc;

// Weights [Cout][Cin][27] -> K-step blocks [tap][KS][khalf][2*Cout rows][4]:
// rows 0..Cout-1 hold the tf32 hi part, rows Cout..2*Cout-1 the lo part; channels
// past Cin are zero.
__global__ void conv3d_tc_prep_weights(const float* __restrict__ w, float* __restrict__ blob, int Cin, int Cout,
                                       int KS) {
  const int total = 27 * KS * 2 * (2 * Cout) * 4;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int j = i & 3;
    int r = i >> 2;
    const int row = r % (2 * Cout);
    r /= 2 * Cout;
    const int kh = r & 1;
    r >>= 1;
    const int ks = r % KS;
    const int tap = r / KS;
    const int c = ks * 8 + kh * 4 + j;
    const int co = row % Cout;
    float v = (c < Cin) ? w[((size_t)co * Cin + c) * 27 + tap] : 0.0f;
    float hi, lo;
    split_tf32(v, hi, lo);
    blob[i] = (row < Cout) ? hi : lo;
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

Plan make_plan(int N, int Cin, int D, int H, int W, int Cout, int epi, int grid) {
  Plan pl;
  TcParams& p = pl.prm;
  std::memset(&p, 0, sizeof(p));
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
  p.N = N; p.Cin = Cin; p.D = D; p.H = H; p.W = W; p.Cout = Cout;
  p.OD = D - 2; p.OH = H - 2; p.OW = W - 2;
  p.epi = epi;
  p.scheme = (Cout <= 64) ? 0 : 1;
  p.NACC = (p.scheme == 0) ? 2 * Cout : Cout;
  p.KS = (Cin + 7) / 8;
  const int tmax = std::max(1, std::min(4, kTmemCols / (kSlots * p.NACC)));
  const uint32_t bblock = 64u * (uint32_t)Cout;
  const int nblocks = 27 * p.KS;
  bool found = false;
  for (int T = tmax; T >= 1 && !found; --T) {
    const int npos = ((T * 128 + 2 * W + 2) + 7) / 8 * 8;
    for (int cc : {32, 24, 16, 8}) {
      if (cc > p.KS * 8) continue;
      const uint32_t a_half = (uint32_t)(cc / 4) * npos * 16u;
      const uint32_t a_stage = 2 * a_half;
      const uint32_t epi_bytes =
          (epi == IG3_EPI_POOL_REDUCE) ? (uint32_t)(2 * 16 * 32 + T * Cout * 32) * 4u : 0u;
      const uint32_t off_b = kAStages * a_stage;
      // Reserve 2 KB for static shared memory and alignment.
      const long long avail = (long long)kSmemLimit - off_b - epi_bytes - 16 * 8 - 2048;
      if (avail <= 0) continue;
      int resident = 0, sb = 0;
      // K-steps per weight stage: a power of two (1, 2 or 4) within kStageTarget
      // bytes that divides the K-steps of every channel chunk (the last may be short).
      const int last_ks = (p.KS * 8 - ((p.KS * 8 + cc - 1) / cc - 1) * cc) / 8;
      int kss = 4;
      while (kss > 1 && (kss * (int)bblock > kStageTarget || (cc / 8) % kss != 0 || last_ks % kss != 0)) kss >>= 1;
      const uint32_t stage_bytes = (uint32_t)kss * bblock;
      if ((long long)nblocks * bblock <= avail) {
        resident = 1;
      } else {
        sb = (int)(avail / (stage_bytes + 16));
        if (sb < 4) continue;
        sb = std::min(sb, 64);
      }
      const uint32_t b_bytes = resident ? nblocks * bblock : (uint32_t)sb * stage_bytes;
      p.KSS = kss;
      p.T = T;
      p.NPOS = npos;
      p.CC = cc;
      p.nchunks = (p.KS * 8 + cc - 1) / cc;
      p.a_half_bytes = a_half;
      p.a_stage_bytes = a_stage;
      p.b_block_bytes = bblock;
      p.resident = resident;
      p.SB = sb;
      p.off_b = off_b;
      p.off_epi = off_b + b_bytes;
      p.off_bar = (p.off_epi + epi_bytes + 127) / 128 * 128;
      pl.smem = p.off_bar + (16 + 2 * (size_t)sb) * 8;
      if (pl.smem > (size_t)kSmemLimit) continue;
      found = true;
      break;
    }
  }
  if (!found) {
    pl.why = "no tiling fits in shared memory";
    return pl;
  }
  p.G = positions_tiles(p.OH, W, p.T);
  // Split the output planes so the units fill the grid evenly; each extra split
  // costs about 2 input planes of conversion and pipeline fill (weight 0.3 each).
  const int step = (epi == IG3_EPI_POOL_REDUCE) ? 2 : 1;
  double best = 1e30;
  int bestS = 1, bestP = p.OD;
  for (int P = p.OD + (p.OD % step); P >= step; P -= step) {
    const int S = (p.OD + P - 1) / P;
    const long long units = (long long)N * p.G * S;
    const long long waves = (units + grid - 1) / grid;
    const double cost = (double)waves * (P + 0.6);
    if (cost < best - 1e-9) {
      best = cost;
      bestS = S;
      bestP = P;
    }
  }
  p.S = bestS;
  p.P = bestP;
  p.units = N * p.G * p.S;
  pl.blob_bytes = align_up((size_t)nblocks * bblock, 256);
  // Upper bound over any split, so the size query does not depend on the device.
  pl.partial_bytes = (epi == IG3_EPI_POOL_REDUCE)
                         ? align_up((size_t)N * positions_tiles(p.OH, W, p.T) * p.OD * sizeof(float), 256)
                         : 0;
  pl.smem = std::max(pl.smem, (size_t)kMinSmem);
  pl.ok = true;
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

size_t conv3d_tc_workspace(const Conv3dArgs& a) {
  Plan pl = make_plan(a.N, a.Cin, a.D, a.H, a.W, a.Cout, a.epi, 148);
  return pl.ok ? pl.blob_bytes + pl.partial_bytes : 0;
}

int conv3d_tc_launch(const Conv3dArgs& a) {
  const int sms = num_sms();
  if (sms <= 0) return fail(IG3_ERR_CUDA, "conv3d TC path: cannot query the SM count");
  Plan pl = make_plan(a.N, a.Cin, a.D, a.H, a.W, a.Cout, a.epi, sms);
  if (!pl.ok) return fail(IG3_ERR_UNSUPPORTED, "conv3d TC path: %s", pl.why);
  TcParams p = pl.prm;
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  p.x = a.x;
  p.wblob = reinterpret_cast<const float*>(ws);
  p.bias = a.b;
  p.y = a.y;
  p.partial = reinterpret_cast<float*>(ws + pl.blob_bytes);
  p.inv_div = (a.epi == IG3_EPI_POOL_REDUCE) ? 1.0f / a.divisor : 1.0f;
  p.ctl = wait_ctl();
  if (!p.ctl.status) return fail(IG3_ERR_CUDA, "conv3d TC path: device status word unavailable");

  const int total = 27 * p.KS * 2 * (2 * p.Cout) * 4;
  conv3d_tc_prep_weights<<<std::min((total + 255) / 256, 4 * sms), 256, 0, a.stream>>>(
      a.w, const_cast<float*>(p.wblob), a.Cin, a.Cout, p.KS);
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
