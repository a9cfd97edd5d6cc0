// Host-side bounds check of the tensor-core conv3d planner and of the index arithmetic
// the kernel performs for every work unit a CTA processes: TMEM columns, accumulator
// slots, A rows, B blocks and stages, the shared-memory layout and the input copies.
// Shapes: a fixed list (the workloads, the GPU test cases, edge shapes) on several SM
// counts, and 3000 seeded random shapes.  Prints the failures and "fails: N".
// Built by tests/test_planner_cpu.py (host code only: no kernel is instantiated here).
#include "../implicit_gemm_convolution_x3x3_gb300/csrc/conv3d_tc.cu"
#include <cstdio>
#include <cstdlib>
using namespace ig3; using namespace ig3::tc;
static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { if (fails++ < 20) { printf("FAIL %s: ", #c); printf(__VA_ARGS__); printf("\n"); } } } while (0)
void check(int N, int Cin, int D, int H, int W, int Cout, int epi, int sms, bool verbose, int flags = 0) {
  Plan pl = make_plan(N, Cin, D, H, W, Cout, epi, sms, flags);
  if (flags & kNoKwWindow) CHECK(!pl.ok || pl.prm.KDM != 9, "kd x kw window in a padded plan");
  if (!pl.ok) { if (verbose) printf("NO plan %d %d %d %d %d %d epi%d: %s\n", N, Cin, D, H, W, Cout, epi, pl.why); return; }
  TcParams p = pl.prm;
  if (verbose) printf("N%d Cin%d D%d H%d W%d Cout%d epi%d: KDM=%d HL=%d T=%d KSS=%d KS=%d nch=%d res=%d SB=%d TPS=%d NSLOT=%d S=%d P=%d units=%d NPOS=%d XS=%d smem=%zu\n",
      N,Cin,D,H,W,Cout,epi,p.KDM,p.HL,p.T,p.KSS,p.KS,p.nchunks,p.resident,p.SB,p.TPS,p.NSLOT,p.S,p.P,p.units,p.NPOS,p.XS,pl.smem);
  const int T = p.T, KSS = p.KSS;
  const uint32_t sw = (p.KDM == 9 ? 3 : p.HL ? 2 : 1) * p.Cout; const uint32_t tile_cols = p.NSLOT * sw;
  CHECK(!p.HL || p.KDM == 3, "HL needs KDM3");
  if (p.KDM == 9) {
    CHECK(p.Cout == 16 && W <= 128 && 128 % W == 0, "KDM9 shape");
    const size_t epi_floats = (epi == 2 ? 2 * 512 + T * p.Cout * 32 : 0) + 2 * 2 * T * 96;
    CHECK(p.off_epi + epi_floats * 4 <= p.off_x, "s_kx beyond epi region");
  }
  CHECK(T * tile_cols <= 512, "tmem cols %u", T * tile_cols);
  CHECK(p.NSLOT <= kMaxSlots, "nslot");
  CHECK(p.SB <= kMaxStages, "sb");
  CHECK(pl.smem <= (size_t)kSmemLimit - 1024, "smem %zu", pl.smem);
  const size_t blob_need = (size_t)27 * p.KS * 64 * p.Cout * (p.HL ? 2 : 1);
  CHECK(blob_need == p.blob_bytes, "blob bytes %zu vs %u", blob_need, p.blob_bytes);
  CHECK(blob_need <= pl.blob_bytes, "blob %zu > ws %zu", blob_need, pl.blob_bytes);
  const uint32_t stage_bytes = p.TPS * KSS * p.b_block_bytes;
  if (p.resident) CHECK(p.off_b + blob_need <= p.off_epi, "resident blob overlaps");
  else CHECK(p.off_b + (size_t)p.SB * stage_bytes <= p.off_epi, "ring overlaps");
  CHECK(p.resident || (p.SB >= 2 && p.SB * p.TPS >= 3), "weight ring depth");
  CHECK((p.KDM == 9 || p.resident) ? p.TPS == 1 : (p.TPS >= 1 && p.TPS <= 3), "taps per stage");
  if (!p.resident) {
    // The loader's stages (taps khw .. khw + nt - 1 copied into one stage) and the MMA
    // issuer's (tap i read at stage offset (i % TPS) * tap bytes, the stage released
    // after tap TPS - 1 of it or after the last tap) must agree.
    const int ntaps = (p.KDM == 9) ? 3 : 9;
    const uint32_t tap_bytes = KSS * p.b_block_bytes;
    int loader_stages = 0, mma_stages = 0, copied = 0;
    for (int khw = 0; khw < ntaps; khw += p.TPS) {
      const int nt = std::min(p.TPS, ntaps - khw);
      CHECK(nt * tap_bytes <= stage_bytes, "stage copy");
      copied += nt;
      ++loader_stages;
    }
    for (int i = 0; i < ntaps; ++i) {
      CHECK((uint32_t)(i % p.TPS + 1) * tap_bytes <= stage_bytes, "tap %d beyond its stage", i);
      if (i % p.TPS == p.TPS - 1 || i == ntaps - 1) ++mma_stages;
    }
    CHECK(copied == ntaps && loader_stages == mma_stages, "stages per chunk: loader %d, MMA %d", loader_stages,
          mma_stages);
  }
  CHECK(p.off_b >= 2 * p.a_stage_bytes, "A overlaps B");
  CHECK(p.off_bar + (6 + 2 * p.NSLOT + 2 * p.SB + 2 * p.XS) * 8 <= pl.smem, "bars beyond smem");
  CHECK(p.XS == 0 || (p.XS >= 2 && p.XS <= kMaxXStages), "xs");
  CHECK(p.off_x >= p.off_epi && p.off_x % 16 == 0 && p.off_x + (size_t)p.XS * p.x_stage_bytes <= p.off_bar, "x ring");
  CHECK(p.x_stage_bytes == (uint32_t)(8 * KSS) * p.NPOS * 4, "x stage");
  CHECK(p.a_half_bytes == (uint32_t)(2 * KSS) * p.NPOS * 16, "a_half");
  CHECK(p.KS % KSS == 0 && p.nchunks * KSS == p.KS, "chunks");
  CHECK(p.NPOS >= T * 128 + 2 * W + 2, "npos %d", p.NPOS);
  const int nblocks_total = (p.KDM == 3 ? 9 : 27) * p.KS;
  const int grid = std::min(p.units, sms);
  CHECK(p.G * T * 128 >= p.OH * p.W, "tiles cover");
  for (int cta = 0; cta < grid; ++cta) {
    uint32_t plane_seq = 0;
    for (int u = cta; u < p.units; u += grid) {
      Unit un = decode_unit(p, u);
      CHECK(un.od1 > un.od0 && un.od1 - un.od0 <= p.P, "unit planes");
      CHECK(un.n < p.N && un.g < p.G, "unit idx");
      if (p.KDM != 1) CHECK(p.P <= p.NSLOT, "P > NSLOT for KDM3/9");
      if (epi == 2) CHECK(un.od0 % 2 == 0, "pool unit start odd");
      const uint32_t s0 = unit_slot0(p, plane_seq);
      if (p.XS) {
        const long long HW = (long long)p.H * p.W, p0 = (long long)un.g * T * 128;
        const long long row_elems = std::min<long long>(p.NPOS, HW - p0);
        CHECK(row_elems > 0 && (row_elems * 4) % 16 == 0 || (HW % 4 != 0), "row bytes %lld", row_elems * 4);
        for (int ch = 0; ch < p.nchunks; ++ch) {
          const int c0 = ch * KSS * 8; const int nvalid = std::min(KSS * 8, p.Cin - c0);
          CHECK(nvalid >= 1, "nvalid");
          const long long last = (((long long)un.n * p.Cin + c0 + nvalid - 1) * p.D + (un.od1 + 1)) * HW + p0 + row_elems;
          CHECK(last <= (long long)p.N * p.Cin * p.D * HW, "x read beyond tensor");
          CHECK((size_t)(nvalid - 1) * p.NPOS * 4 + row_elems * 4 <= p.x_stage_bytes, "x stage overflow");
        }
      }
      for (int d = un.od0; d < un.od1 + 2; ++d) {
        CHECK(d < p.D, "input plane %d >= D", d);
        const int kd_hi = std::min(2, d - un.od0), kd_lo = std::max(0, d - un.od1 + 1);
        CHECK(kd_lo <= kd_hi, "kd range");
        for (int ch = 0; ch < p.nchunks; ++ch) {
          if (ch == 0 && kd_lo == 0) CHECK(slot_add(p, s0, d - un.od0) < (uint32_t)p.NSLOT, "new slot");
          if (p.KDM == 9) {
            const uint32_t c0 = (s0 + (uint32_t)(d - kd_hi - un.od0)) * sw;
            const uint32_t n = (kd_hi - kd_lo + 1) * sw;
            CHECK(n <= 256 && n % 16 == 0, "N %u", n);
            CHECK(c0 + n <= tile_cols, "window cols %u+%u > %u", c0, n, tile_cols);
            CHECK((uint32_t)(2 - kd_hi) * sw + n <= 3u * sw, "B rows");
            CHECK(p.b_block_bytes == 2u * 18 * p.Cout * 16, "blk bytes9");
            for (int kh = 0; kh < 3; ++kh) CHECK(kh * p.KS + ch * KSS + KSS <= 3 * p.KS, "blk9");
          } else if (p.KDM == 3) {
            const uint32_t c0 = (s0 + (uint32_t)(d - kd_hi - un.od0)) * sw;
            const uint32_t n = (kd_hi - kd_lo + 1) * sw;
            CHECK(n <= 256 && n % 16 == 0, "N %u", n);
            CHECK(c0 + n <= tile_cols, "window cols %u+%u > %u", c0, n, tile_cols);
            CHECK((uint32_t)(2 - kd_hi) * sw + n <= 3u * sw, "B rows");
            CHECK(p.b_block_bytes == 2u * (p.HL ? 12 : 6) * p.Cout * 16, "blk bytes");
            for (int khw = 0; khw < 9; ++khw) CHECK(khw * p.KS + ch * KSS + KSS <= nblocks_total, "blk");
          } else {
            for (int kd = kd_hi; kd >= kd_lo; --kd) {
              const uint32_t sl = slot_add(p, s0, d - kd - un.od0);
              CHECK(sl < (uint32_t)p.NSLOT, "slot %u", sl);
              CHECK(sl * p.Cout + p.Cout <= tile_cols, "kd cols");
              for (int khw = 0; khw < 9; ++khw) CHECK((kd * 9 + khw) * p.KS + ch * KSS + KSS <= nblocks_total, "blk1");
              if (kd == 2) CHECK(slot_add(p, s0, d - 2 - un.od0) < (uint32_t)p.NSLOT, "full slot");
            }
          }
          // A reads: rows t*128 + 127 + 2W + 2, groups < 2*KSS
          CHECK((T - 1) * 128 + 127 + 2 * p.W + 2 < p.NPOS, "A rows");
        }
        if (p.KDM != 1 && kd_hi == 2) CHECK(s0 + (uint32_t)(d - 2 - un.od0) < (uint32_t)p.NSLOT, "full slot3");
      }
      for (int od = un.od0; od < un.od1; ++od) {
        const uint32_t slot = slot_add(p, s0, od - un.od0);
        CHECK(slot < (uint32_t)p.NSLOT, "epi slot");
        CHECK((T - 1) * tile_cols + slot * sw + sw <= 512, "epi cols");
      }
      plane_seq += un.od1 - un.od0;
    }
  }
}
int main() {
  int shapes[][7] = {{16,32,32,64,64,64,1},{128,8,16,64,64,16,2},{8,16,32,64,64,16,1},{8,64,32,64,64,64,1},{8,128,32,64,64,128,1},
    {2,32,6,20,70,64,1},{1,8,5,11,64,16,1},{2,16,4,9,8,16,1},{1,16,4,6,64,128,1},{1,24,3,7,33,48,1},{2,3,5,7,9,5,1},{1,1,3,3,3,1,1},
    {2,4,8,8,8,8,1},{1,16,4,8,64,32,1},{1,8,4,6,64,16,1},{3,8,6,10,64,16,2},{2,8,6,8,8,16,2},{2,4,7,9,13,16,2},{1,5,4,4,4,3,2},
    {2,16,5,12,32,32,2},{1,8,5,9,64,16,1},{2,16,5,10,64,32,1},{2,8,6,10,64,16,2},{1,5,9,11,13,80,1},{1,3,5,6,7,96,0},{2,4,8,8,8,16,1},
    {1,128,40,20,30,112,0},{1,40,5,10,32,32,1},{1,32,5,6,64,64,1},{1,16,4,6,64,32,1},{1,5,4,11,13,80,1},{1,12,5,8,20,96,1},{1,8,6,9,16,112,1},{2,72,4,6,24,64,1},{1,8,6,10,64,16,2},{1,32,5,8,64,64,1},{1,16,5,9,16,32,1},{3,40,34,17,19,96,1},{2,72,12,33,40,80,0},{4,8,20,18,16,32,2},
    {1,8,5,6,4,16,1},{2,8,5,9,8,16,1},{1,16,5,9,16,16,1},{2,8,6,12,32,16,1},{1,8,6,12,128,16,1},{1,40,5,6,64,16,1},{1,136,5,6,64,16,1},
    {2,8,6,10,16,16,2},{2,8,6,10,32,16,2},{1,8,6,12,8,16,2},{1,8,6,12,4,16,2},{1,8,7,9,128,16,0},
    {2,5,3,3,3,16,1},{1,4,7,7,7,16,1},{1,8,6,11,64,16,1},{2,16,7,9,32,32,1},{1,24,5,7,22,64,1},{2,8,8,10,64,16,2},
    {1,4,7,7,7,16,2},{16,32,34,66,66,64,1}};
  for (auto& s : shapes)
    for (int sms : {152, 148, 132, 7, 1})
      for (int epi : {s[6]})
        check(s[0],s[1],s[2],s[3],s[4],s[5],epi,sms, sms == 152);
  // zero padding on chip: the virtual volumes (pitch W + roundup(pad + 2, 4) or W + 2 * pad) without the
  // kd x kw window
  int padded[][8] = {{16, 32, 32, 64, 64, 64, 1, 1}, {1, 16, 5, 7, 60, 16, 2, 1}, {1, 8, 4, 6, 32, 96, 3, 1},
                     {1, 8, 5, 5, 16, 32, 4, 1}, {1, 8, 4, 5, 8, 48, 5, 1}, {2, 12, 5, 6, 13, 64, 1, 1},
                     {2, 8, 7, 6, 28, 32, 2, 2}, {1, 8, 6, 9, 30, 16, 1, 2}, {2, 32, 6, 10, 64, 64, 1, 1}};
  for (auto& s : padded)
    for (int sms : {152, 148, 7}) {
      const int P = s[6];
      check(s[0], s[1], s[2] + 2 * P, s[3] + 2 * P, s[4] + 2 * P, s[5], s[7], sms, sms == 152, kNoKwWindow);
      if (s[4] % 4 == 0 && P <= 4 && s[7] != 2)
        check(s[0], s[1], s[2] + 2 * P, s[3] + 2 * P, s[4] + (P + 5) / 4 * 4, s[5], s[7], sms, sms == 152, kNoKwWindow);
    }
  // The GPU tests' streamed-weight variant cases (tests/test_conv3d_gpu.py STAGE_CASES):
  // each shape must still map to the variant it stands for.  {N, Cin, D, H, W, Cout, epi,
  // KDM, HL, T, KSS, TPS}
  int stage_cases[][12] = {
      {1, 9, 5, 4, 280, 96, 1, 1, 0, 1, 1, 1},  {1, 9, 5, 4, 184, 96, 1, 1, 0, 1, 1, 2},
      {1, 17, 5, 48, 8, 96, 1, 1, 0, 1, 1, 3},  {1, 17, 5, 48, 8, 96, 2, 1, 0, 1, 1, 3},
      {8, 9, 6, 4, 288, 96, 0, 1, 0, 1, 2, 1},  {1, 9, 5, 4, 192, 128, 1, 1, 0, 1, 2, 2},
      {1, 9, 5, 48, 8, 96, 2, 1, 0, 1, 2, 3},   {1, 9, 5, 4, 240, 48, 1, 3, 0, 1, 2, 1},
      {1, 9, 5, 4, 168, 48, 1, 3, 0, 1, 2, 2},  {1, 9, 5, 48, 8, 80, 2, 3, 0, 1, 2, 2},
      {1, 9, 5, 4, 152, 48, 0, 3, 0, 1, 2, 3},  {1, 9, 5, 48, 8, 64, 2, 3, 0, 1, 2, 3},
      {4, 9, 12, 4, 200, 48, 1, 3, 0, 2, 2, 1}, {8, 9, 5, 48, 32, 80, 2, 3, 0, 2, 2, 1},
      {4, 9, 6, 9, 168, 48, 1, 3, 0, 2, 2, 2},  {8, 9, 5, 48, 32, 64, 2, 3, 0, 2, 2, 2},
      {4, 9, 5, 33, 96, 48, 1, 3, 0, 2, 2, 3},  {8, 9, 5, 48, 32, 48, 2, 3, 0, 2, 2, 3},
      {1, 9, 5, 4, 288, 16, 1, 3, 1, 1, 2, 1},  {1, 9, 5, 4, 248, 16, 0, 3, 1, 1, 2, 2},
      {1, 9, 5, 48, 8, 32, 1, 3, 1, 1, 2, 3},   {1, 9, 5, 48, 8, 32, 2, 3, 1, 1, 2, 3},
      {4, 17, 12, 4, 224, 16, 1, 3, 1, 2, 2, 1}, {4, 17, 12, 4, 200, 16, 1, 3, 1, 2, 2, 2},
      {8, 9, 5, 48, 32, 32, 2, 3, 1, 2, 2, 2},  {8, 17, 5, 9, 168, 16, 1, 3, 1, 2, 2, 3},
      {1, 57, 5, 6, 128, 16, 1, 9, 0, 1, 2, 1}, {4, 57, 12, 6, 128, 16, 1, 9, 0, 2, 2, 1}};
  for (auto& c : stage_cases) {
    const Plan pl = make_plan(c[0], c[1], c[2], c[3], c[4], c[5], c[6], 152, 0);
    const TcParams& p = pl.prm;
    CHECK(pl.ok && !p.resident && p.KDM == c[7] && p.HL == c[8] && p.T == c[9] && p.KSS == c[10] && p.TPS == c[11],
          "stage case %d %d %d %d %d %d epi%d: KDM %d HL %d T %d KSS %d res %d TPS %d", c[0], c[1], c[2], c[3], c[4],
          c[5], c[6], p.KDM, p.HL, p.T, p.KSS, p.resident, p.TPS);
    for (int sms : {152, 148, 7}) check(c[0], c[1], c[2], c[3], c[4], c[5], c[6], sms, false);
  }
  // random sweep
  srand(1);
  for (int i = 0; i < 3000; ++i) {
    int N = 1 + rand() % 4, Cin = 1 + rand() % 130, D = 3 + rand() % 40, H = 3 + rand() % 40, W = 3 + rand() % (i % 4 == 0 ? 320 : 100), Cout = 16 * (1 + rand() % 8), epi = rand() % 3;
    if (epi == 2) { int ws[] = {4, 8, 16, 32, 64}; W = ws[rand() % 5]; if (D < 4) D = 4; if (H < 4) H = 4; }
    check(N, Cin, D, H, W, Cout, epi, 1 + rand() % 160, false);
  }
  printf("fails: %d\n", fails);
  return fails != 0;
}
