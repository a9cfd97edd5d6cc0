// Host-side bounds check of the stride-2 tensor-core planner (csrc/conv3d_strided_tc.cu)
// and of the index arithmetic its kernel performs: for every work unit, tile position
// and tap, the box element a producer reads (inside the staged box, and holding the
// input coordinate the definition names), the tensor-map copy coordinates, the weight
// block offsets, tensor-memory columns, the shared-memory layout, and that the stored
// outputs cover every output position exactly once.  Shapes: the workload, the GPU test
// cases, edge shapes and 2000 seeded random shapes.  Prints the failures and "fails: N".
// Built by tests/test_planner_cpu.py (host code only: no kernel is instantiated here).
#include "../implicit_gemm_convolution_x3x3_gb300/csrc/conv3d_strided_tc.cu"
#include <cstdio>
#include <cstdlib>
#include <vector>
using namespace ig3;
using namespace ig3::s2tc;
static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { if (fails++ < 20) { printf("FAIL %s: ", #c); printf(__VA_ARGS__); printf("\n"); } } } while (0)

void check(int N, int Cin, int D, int H, int W, int P, int Cout, int epi, bool verbose) {
  Plan pl = make_plan(N, Cin, D, H, W, P, Cout, epi, 152);
  if (!pl.ok) {
    if (verbose) printf("NO plan N%d Cin%d D%d H%d W%d P%d Cout%d: %s\n", N, Cin, D, H, W, P, Cout, pl.why);
    return;
  }
  const Params& p = pl.prm;
  const int T = pl.T, KHG = pl.KHG;
  if (verbose)
    printf("N%d Cin%d D%d H%d W%d P%d Cout%d: T=%d KHG=%d KS=%d G=%d units=%d BX=%d BY=%d col0=%d XS=%d AST=%d "
           "stage=%u smem=%zu\n",
           N, Cin, D, H, W, P, Cout, T, KHG, p.KS, p.G, p.units, p.BX, p.BY, p.col0, p.XS, p.AST, p.stage_bytes,
           pl.smem);
  const int OD = (D + 2 * P - 3) / 2 + 1, OH = (H + 2 * P - 3) / 2 + 1, OW = (W + 2 * P - 3) / 2 + 1;
  CHECK(p.OD == OD && p.OH == OH && p.OW == OW, "output dims");
  CHECK(p.TP == 128 * T, "TP");
  CHECK(p.KS * 8 >= Cin && (p.KS - 1) * 8 < Cin, "K-steps");
  // Tensor memory.
  const int a_stage_cols = T * KHG * 48;
  CHECK(T == 1 && p.a_col0 == (uint32_t)(2 * Cout), "a_col0: the accumulator [D_a | D_b]");
  CHECK(2 * Cout <= 256, "N of the A_hi x [B_hi | B_lo] MMA");
  CHECK(p.a_col0 + (uint32_t)(p.AST * a_stage_cols) <= (uint32_t)kTmemCols, "tmem columns");
  CHECK(p.AST >= 2 && p.AST <= kMaxAST, "A stages");
  CHECK(Cout % 16 == 0 && Cout >= 16 && Cout <= 256, "MMA N");
  // Shared memory.
  CHECK(p.BX % 4 == 0 && p.BX <= 256 && p.BY <= 256 && p.BY >= 3, "box dims");
  CHECK(p.col0 % 4 == 0 && p.col0 <= -P && p.col0 > -P - 4, "col0");
  CHECK(p.x_tx == (uint32_t)(p.BX * p.BY * 32) && p.x_tx <= p.x_bytes && p.x_bytes % 1024 == 0, "x bytes");
  CHECK(p.b_bytes == 576u * (uint32_t)Cout && p.b_bytes % 1024 == 0, "b bytes");
  CHECK(p.stage_bytes == p.x_bytes + p.b_bytes, "stage");
  CHECK(p.XS >= 2 && p.XS <= kMaxXS, "XS");
  CHECK(p.off_bar == (uint32_t)p.XS * p.stage_bytes && p.off_bar % 8 == 0, "bars");
  CHECK(p.off_bar + (size_t)(1 + 2 * p.XS + 2 * p.AST + 4) * 8 <= pl.smem, "bars beyond smem");
  CHECK(pl.smem + 1024 <= (size_t)kSmemLimit, "dynamic + static shared memory %zu", pl.smem);
  // B operand: 9 taps of 64 * Cout bytes inside the stage's weight block.
  CHECK(9u * 64u * (uint32_t)Cout == p.b_bytes, "taps");
  CHECK((2u * Cout * 16u) >> 4 < 16384u, "LBO field");
  // Workspace.
  CHECK(conv3d_strided_tc_workspace(Cin, Cout) >= blob_bytes_for(p.KS, Cout), "workspace");
  CHECK(blob_bytes_for(p.KS, Cout) == (size_t)3 * p.KS * p.b_bytes, "blob");
  // Units: tile positions, box reads and the coverage of the outputs.
  const long long OHW = (long long)OH * OW;
  CHECK(p.G == (OHW + p.TP - 1) / p.TP && p.units == (long long)N * OD * p.G, "units");
  std::vector<unsigned char> seen((size_t)N * OD * OHW, 0);
  const int plane = p.BX * p.BY;
  for (int u = 0; u < p.units; ++u) {
    const Unit un = decode_unit(p, u);
    CHECK(un.n >= 0 && un.n < N && un.od >= 0 && un.od < OD && un.p_lo < OHW, "unit %d", u);
    const int oh_lo = un.p_lo / OW;
    CHECK(un.row0 == oh_lo * 2 - P, "row0");
    for (int kd = 0; kd < 3; ++kd) {
      const int id = un.od * 2 - P + kd;
      const bool inside = id >= 0 && id < D;
      CHECK(inside == (kd >= un.kd_lo && kd <= un.kd_hi), "kd range unit %d kd %d", u, kd);
      if (inside)
        for (int ks = 0; ks < p.KS; ++ks) {
          CHECK(ks * 8 < Cin, "channel coordinate");
          CHECK((size_t)(kd * p.KS + ks + 1) * p.b_bytes <= blob_bytes_for(p.KS, Cout), "weight block");
        }
    }
    for (int tt = 0; tt < T; ++tt)
      for (int m = 0; m < 128; ++m) {
        const long long pp = (long long)un.p_lo + tt * 128 + m;
        const bool valid = pp < OHW;
        const long long pc = valid ? pp : un.p_lo;
        const int oh = (int)(pc / OW), ow = (int)(pc % OW);
        const int off = (oh - oh_lo) * 2 * p.BX + ow * 2 - P - p.col0;
        for (int kh = 0; kh < 3; ++kh)
          for (int kw = 0; kw < 3; ++kw) {
            const int e = off + kh * p.BX + kw;  // channel 0; channel c adds c * plane
            CHECK(e >= 0 && e + 7 * plane < 8 * plane, "box read u%d tt%d m%d", u, tt, m);
            const int by = e / p.BX, bx = e % p.BX;
            CHECK(by >= 0 && by < p.BY && bx >= 0 && bx < p.BX, "box coords");
            CHECK(un.row0 + by == oh * 2 - P + kh && p.col0 + bx == ow * 2 - P + kw,
                  "gathered input coordinate u%d m%d kh%d kw%d", u, m, kh, kw);
          }
        if (valid) {
          unsigned char& s = seen[((size_t)un.n * OD + un.od) * OHW + pp];
          CHECK(s == 0, "output stored twice");
          s = 1;
        }
        // epilogue: team t reads D_a and D_b columns of its channel half, 8 at a time
        for (int team = 0; team < 2; ++team)
          for (int cc = 0; cc < Cout / 2; cc += 8)
            CHECK((uint32_t)(Cout + team * (Cout / 2) + cc + 8) <= p.a_col0 && (Cout / 2) % 8 == 0,
                  "epilogue columns");
      }
    for (int g = 0; g < 3 / KHG; ++g)
      for (int tt = 0; tt < T; ++tt)
        for (int khl = 0; khl < KHG; ++khl)
          for (int kw = 0; kw < 3; ++kw) {
            const int tap = (g * KHG + khl) * 3 + kw;
            CHECK(tap >= 0 && tap < 9, "tap");
            CHECK(((tt * KHG + khl) * 3 + kw) * 16 + 16 <= a_stage_cols, "A columns");
          }
  }
  for (size_t i = 0; i < seen.size(); ++i)
    if (!seen[i]) {
      CHECK(false, "output %zu never stored", i);
      break;
    }
}

int main() {
  // {N, Cin, D, H, W, P, Cout}
  int shapes[][7] = {{16, 32, 32, 64, 64, 1, 64}, {1, 3, 5, 6, 8, 1, 16},    {2, 8, 7, 9, 12, 1, 32},
                     {1, 16, 6, 10, 20, 0, 16},   {1, 8, 9, 16, 16, 2, 48},  {2, 5, 5, 8, 4, 1, 16},
                     {1, 40, 6, 12, 36, 1, 128},  {1, 8, 3, 3, 4, 0, 16},    {1, 8, 4, 4, 4, 3, 16},
                     {1, 8, 5, 5, 8, 5, 16},      {3, 12, 8, 30, 60, 1, 64}, {1, 8, 4, 130, 124, 1, 16},
                     {1, 8, 4, 6, 248, 1, 16},    {1, 17, 11, 13, 28, 2, 80}, {1, 8, 5, 6, 8, 5, 16},
                     {1, 16, 7, 10, 24, 2, 112},  {1, 8, 5, 8, 16, 1, 96},   {1, 12, 9, 33, 36, 1, 64},
                     {2, 24, 16, 64, 64, 1, 64},  {1, 3, 7, 9, 12, 0, 16},   {2, 8, 8, 20, 68, 1, 32},
                     {1, 5, 5, 6, 8, 2, 48}};
  for (auto& s : shapes)
    for (int epi : {0, 1}) check(s[0], s[1], s[2], s[3], s[4], s[5], s[6], epi, epi == 1);
  srand(11);
  for (int i = 0; i < 2000; ++i) {
    const int N = 1 + rand() % 3, Cin = 1 + rand() % 40, D = 1 + rand() % 12, H = 1 + rand() % 40;
    const int W = 4 * (1 + rand() % 40), P = rand() % 5, Cout = 16 * (1 + rand() % 8);
    check(N, Cin, D, H, W, P, Cout, rand() % 2, false);
  }
  printf("fails: %d\n", fails);
  return fails != 0;
}
