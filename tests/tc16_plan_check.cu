// Host-side bounds check of the 16-output-channel tensor-core planner (csrc/conv3d_tc16.cu)
// and of the index arithmetic its kernel performs for every work unit a CTA processes:
// tensor-memory columns of the slots and A stages, the slot ring and its wrapped runs,
// B rows and blocks, the raw input copies (bounds and 16-byte alignment) and the
// stage reads, the shared-memory layout, the partial sums and the workspace sizes.
// Shapes: the workloads, the GPU test cases and edge shapes on several SM counts, and
// 3000 seeded random shapes.  Prints the failures and "fails: N".
// Built by tests/test_planner_cpu.py (host code only: no kernel is instantiated here).
#include "../implicit_gemm_convolution_x3x3_gb300/csrc/conv3d_tc16.cu"
#include <cstdio>
#include <cstdlib>
using namespace ig3;
using namespace ig3::tc16;
static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { if (fails++ < 20) { printf("FAIL %s: ", #c); printf(__VA_ARGS__); printf("\n"); } } } while (0)

void check(int N, int Cin, int D, int H, int W, int epi, int sms, bool verbose) {
  Plan pl = make_plan(N, Cin, D, H, W, 16, epi, sms);
  if (!pl.ok) {
    if (verbose) printf("NO plan %d %d %d %d %d epi%d: %s\n", N, Cin, D, H, W, epi, pl.why);
    return;
  }
  const Params& p = pl.prm;
  const int KSS = pl.kss, PP = pl.pp;
  if (verbose)
    printf("AST=%d ", p.AST);
  if (verbose)
    printf("N%d Cin%d D%d H%d W%d epi%d: KSS=%d PP=%d KS=%d nch=%d NSLOT=%d G=%d S=%d P=%d units=%d NPOS=%d XS=%d smem=%zu\n",
           N, Cin, D, H, W, epi, KSS, PP, p.KS, p.nchunks, p.NSLOT, p.G, p.S, p.P, p.units, p.NPOS, p.XS, pl.smem);
  CHECK((KSS == 1 && PP == 2) || (KSS == 2 && PP == 1) || (KSS == 1 && PP == 1), "chunk shape");
  // Layout.
  CHECK(64 % W == 0, "W %d", W);
  CHECK((H * W) % 4 == 0, "HW %% 4");
  CHECK(p.KS % KSS == 0 && p.nchunks * KSS == p.KS, "chunks");
  CHECK(8 * p.KS >= Cin && 8 * (p.KS - KSS) < Cin, "K-steps cover Cin without an empty chunk");
  CHECK(p.a_col0 == (uint32_t)(p.NSLOT * kSlotCols), "a_col0");
  CHECK(p.AST >= 2 && p.AST <= kMaxAStages, "A stages");
  CHECK(p.a_col0 + (uint32_t)(p.AST * PP * KSS * kKStepCols) <= (uint32_t)kTmemCols, "tmem cols");
  CHECK(p.NSLOT >= PP + 3 && p.NSLOT <= 32, "nslot %d", p.NSLOT);
  CHECK(p.blob_bytes == blob_bytes_for(p.KS), "blob bytes");
  CHECK(p.off_x % 1024 == 0 && p.off_x >= p.blob_bytes, "x ring start");
  CHECK(p.x_stage_bytes == (uint32_t)(PP * 8 * KSS) * p.NPOS * 4 && p.x_stage_bytes % 16 == 0, "x stage");
  CHECK(p.off_bar == p.off_x + (uint32_t)p.XS * p.x_stage_bytes && p.off_bar % 8 == 0, "bars");
  CHECK(p.XS >= 2 && p.XS <= kMaxXStages, "xs");
  CHECK(p.off_bar + (size_t)(2 + 2 * p.AST + 2 * p.XS + 2 * p.NSLOT) * 8 <= pl.smem, "bars beyond smem");
  CHECK(pl.smem + 12288 <= (size_t)kSmemLimit, "dynamic + static shared memory %zu", pl.smem);
  CHECK(p.NPOS == 128 + 2 * W && (p.NPOS * 4) % 16 == 0, "npos");
  CHECK(p.G * 128 >= p.OH * W && (p.G - 1) * 128 < p.OH * W, "tiles cover");
  if (epi == 2) CHECK(p.P % 2 == 0, "pool P even");
  // Workspace of the public size query.
  Conv3dArgs a{};
  a.N = N; a.Cin = Cin; a.D = D; a.H = H; a.W = W; a.Cout = 16; a.epi = epi;
  const int ks2 = ((Cin + 7) / 8 + 1) / 2 * 2;
  CHECK(blob_bytes_for(p.KS) <= align_up(blob_bytes_for(ks2), 256), "blob beyond workspace");
  CHECK(conv3d_tc16_workspace(a) >= align_up(blob_bytes_for(ks2), 256) + (epi == 2 ? (size_t)p.units * 4 : 0),
        "partials beyond workspace");
  const long long HW = (long long)H * W;
  const int grid = std::min(p.units, sms);
  for (int cta = 0; cta < grid; ++cta) {
    uint32_t plane_seq = 0;
    for (int u = cta; u < p.units; u += grid) {
      const Unit un = decode_unit(p, u);
      CHECK(un.n < p.N && un.g < p.G && un.od0 < un.od1 && un.od1 - un.od0 <= p.P, "unit %d", u);
      if (epi == 2) CHECK(un.od0 % 2 == 0, "pool unit starts on an odd plane");
      CHECK(((long long)un.n * p.G + un.g) * p.S + (un.od0 / p.P) == u, "partial index");
      const long long p0 = (long long)un.g * 128;
      // Producer reads: position m + kh*W of the staged row, m < 128.
      CHECK(127 + 2 * W < p.NPOS, "A rows beyond the staged row");
      uint32_t s_d = plane_seq % p.NSLOT;
      for (int d0 = un.od0; d0 < un.od1 + 2; d0 += PP) {
        const int npl = std::min(PP, un.od1 + 2 - d0);
        CHECK(npl >= 1 && d0 + npl - 1 < D, "input planes %d..%d, D %d", d0, d0 + npl - 1, D);
        // One tensor-map copy per chunk: box [8*KSS][PP][NPOS] at (p0, d0, ch*8*KSS, n)
        // of x as [N][Cin][D][H*W]; the box start lies inside the tensor, its far
        // side may leave it (zero fill), the innermost start is 16-byte aligned.
        for (int ch = 0; ch < p.nchunks; ++ch) {
          const int c0 = ch * 8 * KSS;
          CHECK(c0 < Cin && d0 < D && p0 < HW && un.n < N, "box start outside x");
          CHECK((p0 * 4) % 16 == 0, "box x alignment");
        }
        CHECK(p.NPOS <= 256 && PP <= 256 && 8 * KSS <= 256, "box dims");
        CHECK((long long)p.x_stage_bytes < (1 << 20), "tx count");
        for (int pi = 0; pi < npl; ++pi)
          CHECK(p.a_col0 + (uint32_t)(p.AST - 1) * PP * KSS * kKStepCols + (uint32_t)((pi * KSS + KSS) * kKStepCols) <=
                    (uint32_t)kTmemCols, "A cols");
        // producer reads: rows (c * PP + pi) of NPOS, positions m + kh*W < 128 + 2W
        CHECK((8 * KSS - 1) * PP + (PP - 1) < 8 * KSS * PP && 127 + 2 * W < p.NPOS, "producer reads");
        for (int pi = 0; pi < npl; ++pi) {
          const int d = d0 + pi;
          const int kd_hi = std::min(2, d - un.od0), kd_lo = std::max(0, d - un.od1 + 1);
          CHECK(kd_lo <= kd_hi, "kd range");
          const uint32_t nkd = kd_hi - kd_lo + 1;
          const uint32_t s_first = (s_d >= (uint32_t)kd_hi) ? s_d - kd_hi : s_d + p.NSLOT - kd_hi;
          CHECK(s_first == (plane_seq + (uint32_t)(d - kd_hi - un.od0)) % p.NSLOT, "incremental slot");
          const uint32_t n1 = std::min(nkd, (uint32_t)p.NSLOT - s_first), n2 = nkd - n1;
          CHECK(n1 >= 1 && s_first + n1 <= (uint32_t)p.NSLOT && n2 <= (uint32_t)p.NSLOT, "run");
          CHECK(n1 * kSlotCols <= 256 && n2 * kSlotCols <= 256, "N");
          // B rows of the runs: [kd=2 | kd=1 | kd=0] x 48 within the hi half (144 rows).
          CHECK((2 - kd_hi) * kSlotCols + (n1 + n2) * kSlotCols <= 9 * 16, "B rows");
          for (int ch = 0; ch < p.nchunks; ++ch)
            for (int kh = 0; kh < 3; ++kh)
              for (int ks = 0; ks < KSS; ++ks) {
                const size_t blk = (size_t)kh * p.KS + ch * KSS + ks;
                CHECK((blk + 1) * kBBlockBytes <= p.blob_bytes, "B block");
              }
          s_d = (s_d + 1 == (uint32_t)p.NSLOT) ? 0 : s_d + 1;
        }
      }
      for (int od = un.od0; od < un.od1; ++od) {
        const uint32_t slot = (plane_seq + (uint32_t)(od - un.od0)) % p.NSLOT;
        CHECK((slot + 1) * kSlotCols <= p.a_col0, "epi slot cols");
      }
      plane_seq += un.od1 - un.od0;
    }
  }
}

int main() {
  int shapes[][6] = {{128, 8, 16, 64, 64, 2}, {8, 16, 32, 64, 64, 1}, {8, 16, 32, 64, 64, 0},
                     {1, 8, 5, 11, 64, 1},    {2, 16, 4, 9, 8, 1},    {1, 8, 5, 6, 4, 1},
                     {2, 8, 6, 12, 32, 1},    {1, 8, 6, 12, 128, 1},  {2, 8, 10, 64, 64, 1},
                     {1, 40, 5, 6, 64, 1},    {1, 136, 5, 6, 64, 1},  {3, 8, 6, 10, 64, 2},
                     {2, 8, 6, 8, 8, 2},      {2, 8, 6, 10, 16, 2},   {2, 8, 6, 10, 32, 2},
                     {1, 8, 6, 12, 4, 2},     {2, 8, 8, 64, 64, 2},   {1, 12, 9, 7, 64, 1},
                     {2, 3, 7, 5, 32, 2},     {1, 24, 40, 6, 16, 1},  {4, 8, 33, 10, 64, 2},
                     {1, 32, 12, 6, 128, 1},  {1, 48, 6, 6, 64, 1},   {2, 8, 16, 64, 64, 2}};
  for (auto& s : shapes)
    for (int sms : {152, 148, 132, 7, 1}) check(s[0], s[1], s[2], s[3], s[4], s[5], sms, sms == 152);
  srand(3);
  for (int i = 0; i < 3000; ++i) {
    const int ws[] = {4, 8, 16, 32, 64, 128};
    int epi = rand() % 3;
    int W = ws[rand() % 5];
    int N = 1 + rand() % 4, Cin = 1 + rand() % 48, D = 3 + rand() % 40, H = 3 + rand() % 40;
    if (epi == 2) { if (D < 4) D = 4; if (H < 4) H = 4; }
    check(N, Cin, D, H, W, epi, 1 + rand() % 160, false);
  }
  printf("fails: %d\n", fails);
  return fails != 0;
}
