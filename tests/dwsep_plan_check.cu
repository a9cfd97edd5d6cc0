// Host-side check of the tensor-core depthwise-separable planner (make_dw_plan) and of
// the addresses its kernel and tensor map derive from a plan: strip length and unit
// count, the shared-memory layout (row slots aligned for the tensor-map copies), the
// TMEM column ranges, the tensor map's box and strides, and the x coordinate of every
// row copy (a multiple of 16 bytes), the rows a strip reads and the channels each
// depthwise warp owns, for the 3x3 and 5x5 depthwise sizes.  Shapes: a grid over the
// supported channel counts and seeded random images, on several SM counts.  Prints the failures and "fails: N".
// Built by tests/test_planner_cpu.py (host code only).
#include "../implicit_gemm_convolution_x3x3_gb300/csrc/dwsep_tc.cu"
#include <cstdio>
#include <cstdlib>
using namespace ig3;
static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { if (fails++ < 20) { printf("FAIL %s: ", #c); printf(__VA_ARGS__); printf("\n"); } } } while (0)

template <int K>
static void check_k(int N, int C, int H, int W, int Cout, int sms) {
  using Cfg = DwCfg<K>;
  constexpr int P = Cfg::P;
  DwPlan pl = make_dw_plan(N, C, H, W, Cout, K, sms);
  const bool supported = C % 16 == 0 && C <= 64 && Cout % 16 == 0 && Cout <= 128 && W % 4 == 0;
  CHECK(pl.ok == supported, "N%d C%d H%d W%d Cout%d: ok=%d (%s)", N, C, H, W, Cout, (int)pl.ok, pl.why);
  if (!pl.ok) return;
  const DwParams& p = pl.prm;
  // strips
  CHECK(p.R >= 1 && p.R <= H && (p.R == H || p.R == 8 || p.R == 16 || p.R == 32 || p.R == 64), "R %d H %d", p.R, H);
  CHECK((long long)p.HR * p.R >= H && (long long)(p.HR - 1) * p.R < H, "HR %d R %d H %d", p.HR, p.R, H);
  CHECK(p.WB == (W + kTile - 1) / kTile, "WB");
  CHECK((long long)p.units == (long long)N * p.WB * p.HR, "units");
  // shared memory
  const uint32_t b_bytes = (uint32_t)(C / 8) * 2u * (2u * Cout) * 16u;
  CHECK(p.off_wdw >= b_bytes, "B region");
  CHECK(p.off_rows >= p.off_wdw + (uint32_t)(C * K * Cfg::kWRow) * 4u, "w_dw region");
  CHECK(p.off_wdw % 16 == 0 && (K * Cfg::kWRow * 4) % 16 == 0 && Cfg::kWRow >= K, "w_dw rows 16-byte aligned");
  // depthwise warps: kPerQ per quadrant, C / kPerQ channels each, groups of 4 (tcgen05.st x4)
  CHECK(C % Cfg::kPerQ == 0 && (C / Cfg::kPerQ) % 4 == 0 && C / Cfg::kPerQ <= Cfg::kCMax, "channels per warp");
  CHECK(Cfg::kThreads <= 1024 && Cfg::kEpiWarp0 + 4 == Cfg::kThreads / 32, "roles");
  CHECK(P <= kHalo, "halo");
  CHECK(p.off_rows % 1024 == 0 && p.row_bytes % 16 == 0 && p.row_bytes == (uint32_t)C * kBoxW * 4u, "row slots");
  CHECK(p.off_bar >= p.off_rows + kRowSlots * p.row_bytes && p.off_bar % 8 == 0, "barriers");
  CHECK(pl.smem >= p.off_bar + 32 * 8 && pl.smem + 2048 <= (size_t)(227 * 1024), "smem %zu", pl.smem);
  // tensor memory: accumulators [0, 2 Cout), A tiles [kACol0, kACol0 + 2 * 2C)
  CHECK(2 * Cout <= kACol0 && kACol0 + 4 * C <= kTmemCols, "TMEM columns");
  // tensor map: box {kBoxW, 1, C} within limits, 16-byte inner box and strides
  CHECK(kBoxW <= 256 && C <= 256 && (kBoxW * 4) % 16 == 0, "box");
  CHECK(((long long)W * 4) % 16 == 0 && ((long long)H * W * 4) % 16 == 0, "strides");
  // every row copy of every unit: x coordinate 16-byte aligned, rows within [-1, H],
  // channel block inside [0, N*C)
  for (long long u = 0; u < p.units; u += (p.units > 4096 ? p.units / 4096 : 1)) {
    const int hr = (int)(u % p.HR), wb = (int)((u / p.HR) % p.WB), n = (int)(u / ((long long)p.HR * p.WB));
    const int h0 = hr * p.R, h1 = std::min(p.H, h0 + p.R);
    const long long xcoord = (long long)wb * kTile - kHalo;
    CHECK((xcoord * 4) % 16 == 0, "x coordinate %lld", xcoord);
    CHECK(h0 - P >= -P && h1 + P - 1 <= H - 1 + P && h0 < h1, "rows");
    // the depthwise warps consume rows h0-P .. h1+P-1 in the loader's order: R + 2P rows
    CHECK((h1 + P) - (h0 - P) == (h1 - h0) + 2 * P, "rows per strip");
    // pixels px - P .. px + P of the tile lie inside the staged row [w0 - kHalo, w0 + 128 + kHalo)
    CHECK(kHalo - P >= 0 && kTile - 1 + kHalo + P < kBoxW, "staged columns");
    CHECK((long long)n * C + C <= (long long)N * C, "channel block");
  }
}

static void check(int N, int C, int H, int W, int Cout, int sms) {
  check_k<3>(N, C, H, W, Cout, sms);
  check_k<5>(N, C, H, W, Cout, sms);
}

int main() {
  for (int sms : {148, 152, 7})
    for (int C = 16; C <= 80; C += 16)
      for (int Cout = 16; Cout <= 144; Cout += 16)
        for (int W : {4, 64, 128, 132, 260, 512, 1000})
          for (int H : {1, 2, 7, 8, 33, 70, 512})
            check(1 + (C + Cout + W + H) % 3, C, H, W, Cout, sms);
  check(16, 64, 512, 512, 128, 152);  // the benchmark workload
  check(1, 24, 8, 8, 16, 152);        // unsupported: C not a multiple of 16
  check(1, 16, 8, 10, 16, 152);       // unsupported: W not a multiple of 4
  srand(7);
  for (int i = 0; i < 3000; ++i) {
    const int N = 1 + rand() % 8, C = 16 * (1 + rand() % 4), Cout = 16 * (1 + rand() % 8);
    const int W = 4 * (1 + rand() % 400), H = 1 + rand() % 700;
    check(N, C, H, W, Cout, 1 + rand() % 160);
  }
  printf("fails: %d\n", fails);
  return fails != 0;
}
