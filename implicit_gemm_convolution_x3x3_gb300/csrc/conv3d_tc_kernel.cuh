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
constexpr int kStageTarget = 16 * 1024;           // bytes of weights per ring stage
constexpr int kSlots = 4;
constexpr int kAStages = 2;
constexpr int kTmemCols = 512;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMinSmem = 116 * 1024;  // keeps one CTA (one TMEM owner) per SM

struct TcParams {
  const float* x;
  const float* wblob;  // [27 taps][KS K-steps][2 k-halves][2*Cout rows][4]
  const float* bias;
  float* y;
  float* partial;
  int N, Cin, D, H, W, Cout, OD, OH, OW;
  int KS;        // K-steps of 8 channels over the padded Cin
  int CC;        // channels per A chunk (multiple of 8)
  int nchunks;
  int T;         // position tiles of 128 per unit
  int NPOS;      // positions held per A stage
  int NACC;      // accumulator columns per tile
  int scheme;    // 0: [hi;lo] B + 1 MMA for lo (Cout <= 64); 1: three MMAs
  int G, S, P;   // tile groups per plane, plane splits, planes per split
  int units;
  int resident;  // weights loaded once
  int SB;        // weight ring stages (streaming)
  int KSS;       // K-step blocks per ring stage (all of one tap, up to kStageTarget bytes)
  int epi;
  float inv_div;
  uint32_t a_half_bytes;   // one of hi / lo in an A stage
  uint32_t a_stage_bytes;  // hi + lo
  uint32_t b_block_bytes;  // one K-step block of B
  uint32_t off_b, off_epi, off_bar;  // shared-memory offsets
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

static __device__ __forceinline__ Unit decode_unit(const TcParams& p, int u) {
  Unit r;
  const int s = u % p.S;
  const int g = (u / p.S) % p.G;
  r.n = u / (p.S * p.G);
  r.g = g;
  r.od0 = s * p.P;
  r.od1 = min(p.OD, r.od0 + p.P);
  return r;
}

static __device__ __forceinline__ int chunk_channels(const TcParams& p, int ch) {
  return min(p.CC, p.KS * 8 - ch * p.CC);
}

// A bounded wait used while shutting down: ignores the abort flag.
static __device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
  int never = 0;
  return mbar_wait_bounded(bar, parity, ctl, &never);
}

// A bounded wait taken by every lane of a warp, returning one verdict for the whole
// warp (and leaving it converged): warp-collective tcgen05 instructions follow.
static __device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, ctl, abort);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Non-blocking test of a barrier phase (try_wait may suspend the thread for a while
// even when it returns true at once; test_wait never does).
static __device__ __forceinline__ bool mbar_test_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return done != 0;
}

// The common case inline (phase already complete), the bounded loop out of line.
static __device__ __forceinline__ bool wait_fast(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                                 volatile int* abort) {
  if (mbar_test_wait(smem_addr(bar), parity)) return true;
  return mbar_wait_bounded(bar, parity, ctl, abort);
}

// The MMAs of one weight stage: KSS K-steps x T position tiles, fully unrolled so the
// issue is a straight run of adds and tcgen05.mma.  `acc` is 0 only for the first
// K-step of a plane (it overwrites the accumulator) and 1 afterwards.
template <int SCHEME, int T, int KSS>
static __device__ __forceinline__ void issue_stage(uint32_t d0, uint64_t ah0, uint64_t al0, uint64_t bst,
                                                   uint32_t koff0, uint32_t ks_u, uint32_t b_block_u,
                                                   uint32_t b_lo_u, uint32_t nacc, uint32_t idesc_cat,
                                                   uint32_t idesc_one, uint32_t& acc) {
#pragma unroll
  for (int j = 0; j < KSS; ++j) {
    const uint64_t bh = bst + (uint64_t)(j * b_block_u);
    const uint64_t koff = (uint64_t)(koff0 + (uint32_t)j * ks_u);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const uint32_t dt = d0 + (uint32_t)t * nacc;
      const uint64_t ah = ah0 + koff + (uint64_t)(t * 128), al = al0 + koff + (uint64_t)(t * 128);
      if constexpr (SCHEME == 0) {
        umma_tf32(dt, ah, bh, idesc_cat, acc);
        umma_tf32(dt, al, bh, idesc_one, 1u);
      } else {
        umma_tf32(dt, ah, bh, idesc_one, acc);
        umma_tf32(dt, ah, bh + b_lo_u, idesc_one, 1u);
        umma_tf32(dt, al, bh, idesc_one, 1u);
      }
    }
    acc = 1u;
  }
}

static __device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

static __device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

template <int EPI, int SCHEME, int T, int KSS>
__global__ void __launch_bounds__(kThreads, 1) conv3d_tc_kernel(const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_red[kEpiThreads / 32];

  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + p.off_b;
  float* s_epi = reinterpret_cast<float*>(smem + p.off_epi);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* a_full = bars;                   // [2]
  uint64_t* a_empty = bars + 2;              // [2]
  uint64_t* acc_full = bars + 4;             // [4]
  uint64_t* acc_empty = bars + 8;            // [4]
  uint64_t* w_full = bars + 12;              // resident weights
  uint64_t* mma_done = bars + 13;            // final drain of the MMA pipe
  uint64_t* b_full = bars + 16;              // [SB]
  uint64_t* b_empty = bars + 16 + p.SB;      // [SB]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &s_abort;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&a_full[i], kConvThreads);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiThreads);
    }
    mbar_init(w_full, 1);
    mbar_init(mma_done, 1);
    for (int i = 0; i < p.SB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
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
  const int nblocks = 27 * p.KS;

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      if (p.resident) {
        const uint32_t total = (uint32_t)nblocks * p.b_block_bytes;
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
        for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
          const Unit un = decode_unit(p, u);
          for (int d = un.od0; d < un.od1 + 2 && !*abort_flag; ++d) {
            for (int ch = 0; ch < p.nchunks; ++ch) {
              const int ks_n = chunk_channels(p, ch) >> 3;
              for (int kd = 2; kd >= 0; --kd) {
                const int od = d - kd;
                if (od < un.od0 || od >= un.od1) continue;
                for (int khw = 0; khw < 9; ++khw) {
                  // One stage = up to KSS consecutive K-step blocks of this tap (contiguous
                  // in the blob), fetched with one bulk copy.
                  for (int s0 = 0; s0 < ks_n; s0 += p.KSS) {
                    const int nb = min(p.KSS, ks_n - s0);
                    if (!wait_fast(&b_empty[rb.idx], rb.phase ^ 1u, p.ctl, abort_flag)) goto producer_done;
                    const int blk = (kd * 9 + khw) * p.KS + ch * (p.CC >> 3) + s0;
                    const uint32_t bytes = (uint32_t)nb * p.b_block_bytes;
                    mbar_arrive_expect_tx(&b_full[rb.idx], bytes);
                    bulk_copy_g2s(smem_b + (size_t)rb.idx * p.KSS * p.b_block_bytes,
                                  reinterpret_cast<const uint8_t*>(p.wblob) + (size_t)blk * p.b_block_bytes, bytes,
                                  &b_full[rb.idx]);
                    rb.next(p.SB);
                    ++issued;
                  }
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
      // start-address field is the low 14 bits): the issue loop must stay a short
      // chain of adds for tcgen05.mma to issue at the tensor pipe's rate.
      const uint32_t idesc_cat = umma_idesc_tf32(128, SCHEME == 0 ? 2 * p.Cout : p.Cout);
      const uint32_t idesc_one = umma_idesc_tf32(128, p.Cout);
      const uint64_t a_desc0 = umma_desc_noswizzle(smem_addr(smem_a), (uint32_t)p.NPOS * 16u, 128);
      const uint64_t b_desc0 = umma_desc_noswizzle(smem_addr(smem_b), (uint32_t)(2 * p.Cout) * 16u, 128);
      const uint32_t a_stage_u = p.a_stage_bytes >> 4, a_half_u = p.a_half_bytes >> 4;
      const uint32_t ks_u = 2u * (uint32_t)p.NPOS;       // next K-step: two channel groups on
      const uint32_t b_block_u = p.b_block_bytes >> 4;
      const uint32_t b_stage_u = b_block_u * (uint32_t)p.KSS;
      const uint32_t b_lo_u = (uint32_t)p.Cout;           // lo rows start Cout rows further
      const uint32_t row_u = (uint32_t)p.W;               // one input row (kh step)
      const uint32_t slot_cols = (uint32_t)(p.T * p.NACC);
      const uint32_t nacc = (uint32_t)p.NACC;
      const int CC8 = p.CC >> 3;
      bool ok = true;
      if (p.resident) ok = mbar_wait_bounded(w_full, 0, p.ctl, abort_flag);
      Ring ra, rb;
      uint32_t plane_seq = 0;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        const Unit un = decode_unit(p, u);
        for (int d = un.od0; ok && d < un.od1 + 2; ++d) {
          for (int ch = 0; ok && ch < p.nchunks; ++ch) {
            const int ks_n = chunk_channels(p, ch) >> 3;
            if (!(ok = wait_fast(&a_full[ra.idx], ra.phase, p.ctl, abort_flag))) break;
            tc_fence_after();
            const uint64_t ah0 = a_desc0 + (uint64_t)(ra.idx * a_stage_u);
            const uint64_t al0 = ah0 + a_half_u;
            for (int kd = 2; ok && kd >= 0; --kd) {
              const int od = d - kd;
              if (od < un.od0 || od >= un.od1) continue;
              const uint32_t pseq = plane_seq + (uint32_t)(od - un.od0);
              const uint32_t slot = pseq & (kSlots - 1);
              if (kd == 0 && ch == 0) {
                if (!(ok = wait_fast(&acc_empty[slot], ((pseq >> 2) & 1u) ^ 1u, p.ctl, abort_flag))) break;
                tc_fence_after();
              }
              const uint32_t d0 = tmem_base + slot * slot_cols;
              // The first MMA of a plane (kd = 0, first chunk, first tap, first K-step)
              // overwrites the accumulator; every later one adds to it.
              uint32_t acc = (kd == 0 && ch == 0) ? 0u : 1u;
#pragma unroll
              for (int kh = 0; kh < 3; ++kh) {
#pragma unroll
                for (int kw = 0; kw < 3; ++kw) {
                  const uint32_t tap_u = (uint32_t)kh * row_u + (uint32_t)kw;
                  const int tap = (kd * 3 + kh) * 3 + kw;
                  for (int s0 = 0; s0 < ks_n; s0 += KSS) {
                    uint64_t bst;
                    if (p.resident) {
                      bst = b_desc0 + (uint64_t)((uint32_t)(tap * p.KS + ch * CC8 + s0) * b_block_u);
                    } else {
                      if (!(ok = wait_fast(&b_full[rb.idx], rb.phase, p.ctl, abort_flag))) break;
                      tc_fence_after();
                      bst = b_desc0 + (uint64_t)(rb.idx * b_stage_u);
                    }
                    issue_stage<SCHEME, T, KSS>(d0, ah0, al0, bst, (uint32_t)s0 * ks_u + tap_u, ks_u, b_block_u,
                                                b_lo_u, nacc, idesc_cat, idesc_one, acc);
                    if (!p.resident) {
                      umma_commit(&b_empty[rb.idx]);
                      rb.next(p.SB);
                    }
                  }
                  if (!ok) break;
                }
                if (!ok) break;
              }
              if (ok && kd == 2 && ch == p.nchunks - 1) umma_commit(&acc_full[slot]);
            }
            umma_commit(&a_empty[ra.idx]);
            ra.next(kAStages);
          }
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
    const int ct = tid - kConvWarp0 * 32;
    const size_t HW = (size_t)p.H * p.W;
    const int plane_pos = p.H * p.W;
    Ring ra;
    for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
      const Unit un = decode_unit(p, u);
      const int p0 = un.g * p.T * 128;
      for (int d = un.od0; d < un.od1 + 2; ++d) {
        for (int ch = 0; ch < p.nchunks; ++ch) {
          if (!warp_wait(&a_empty[ra.idx], ra.phase ^ 1u, p.ctl, abort_flag)) goto convert_done;
          const int c0 = ch * p.CC;
          const int groups = chunk_channels(p, ch) >> 2;
          const int items = groups * p.NPOS;
          const uint32_t hi_base = smem_addr(smem_a) + ra.idx * p.a_stage_bytes;
          const uint32_t lo_base = hi_base + p.a_half_bytes;
          const float* xplane = p.x + ((size_t)un.n * p.Cin) * p.D * HW + (size_t)d * HW;
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
                const int grp = i / p.NPOS, pp = i - grp * p.NPOS;
                const uint32_t off = (uint32_t)(grp * p.NPOS + pp) * 16u;
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
  convert_done:;
  } else {
    // ------------------------------------------------------------ epilogue
    // Two groups of four warps; each group covers all four TMEM lane quadrants and
    // takes every other (tile, 16-channel) item of a plane.
    const int et = tid - kEpiWarp0 * 32;
    const int q = warp & 3;                        // TMEM lane quadrant this warp may access
    const int grp = (warp - kEpiWarp0) >> 2;       // 0 or 1
    const size_t OHW = (size_t)p.OH * p.OW;
    const int PH = p.OH / 2, PW = p.OW / 2;
    const int cchunks = p.Cout >> 4;
    const int items = p.T * cchunks;
    float* s_x = s_epi + grp * (16 * 32);          // pool: h-pair exchange [16][32] per group
    float* s_prev = s_epi + 2 * (16 * 32);         // pool: even-plane maxima [T][Cout][32]
    uint32_t plane_seq = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      const Unit un = decode_unit(p, u);
      const int p0 = un.g * p.T * 128;
      float psum = 0.0f;
      for (int od = un.od0; od < un.od1; ++od) {
        const uint32_t pseq = plane_seq + (uint32_t)(od - un.od0);
        const uint32_t slot = pseq & (kSlots - 1);
        if (!(ok = warp_wait(&acc_full[slot], (pseq >> 2) & 1u, p.ctl, abort_flag))) break;
        tc_fence_after();
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) + slot * (uint32_t)(p.T * p.NACC);
        const bool pool_plane = (EPI == IG3_EPI_POOL_REDUCE) && (od / 2 < p.OD / 2);
        for (int it = grp; it < items; it += 2) {
          const int t = it / cchunks;
          const int c0 = (it - t * cchunks) << 4;
          const int lp = t * 128 + q * 32 + lane;  // position within the unit
          const int pos = p0 + lp;
          const int oh = pos / p.W, ow = pos - oh * p.W;
          const bool valid = (oh < p.OH) && (ow < p.OW);
          const uint32_t tcol = lane_base + (uint32_t)(t * p.NACC);
          float v[16];
          tmem_ld16(tcol + c0, v);
          if constexpr (SCHEME == 0) {
            float w2[16];
            tmem_ld16(tcol + p.Cout + c0, w2);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += w2[j];
          } else {
            tmem_wait_ld();
          }
          if constexpr (EPI != IG3_EPI_POOL_REDUCE) {
            float* yb = p.y + (((size_t)un.n * p.Cout + c0) * p.OD + od) * OHW + (size_t)oh * p.OW + ow;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float val = v[j] + (p.bias ? __ldg(&p.bias[c0 + j]) : 0.0f);
              if (EPI == IG3_EPI_TANH_MISH) val = tanh_mish(val);
              if (valid) yb[(size_t)j * p.OD * OHW] = val;
            }
          } else {
            if (!pool_plane) continue;
            // w-pair: neighbouring lanes; h-pair: position + W.
            const int r = (q * 32 + lane) / p.W;          // row within the tile (tile rows start even)
            const int cw = ow >> 1;
            const int cell = (r >> 1) * (p.W >> 1) + cw;  // pooled cell within the tile, < 32
            const bool even_w = (ow & 1) == 0, even_r = (r & 1) == 0;
            float hm[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float z = (v[j] + (p.bias ? __ldg(&p.bias[c0 + j]) : 0.0f)) * p.inv_div;
              hm[j] = fmaxf(z, __shfl_xor_sync(0xffffffffu, z, 1));
            }
            if (p.W <= 16) {
#pragma unroll
              for (int j = 0; j < 16; ++j) hm[j] = fmaxf(hm[j], __shfl_xor_sync(0xffffffffu, hm[j], p.W));
            } else {
              if (!even_r && even_w) {
#pragma unroll
                for (int j = 0; j < 16; ++j) s_x[j * 32 + cell] = hm[j];
              }
              named_bar_sync(1 + grp, 128);
              if (even_r && even_w) {
#pragma unroll
                for (int j = 0; j < 16; ++j) hm[j] = fmaxf(hm[j], s_x[j * 32 + cell]);
              }
              named_bar_sync(1 + grp, 128);
            }
            if (even_r && even_w) {
              float* prev = s_prev + ((size_t)t * p.Cout + c0) * 32 + cell;
              if ((od & 1) == 0) {
#pragma unroll
                for (int j = 0; j < 16; ++j) prev[j * 32] = hm[j];
              } else if ((oh >> 1) < PH && cw < PW) {
#pragma unroll
                for (int j = 0; j < 16; ++j) psum += fmaxf(prev[j * 32], hm[j]);
              }
            }
          }
        }
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


// Launches the kernel variant matching p.scheme, p.T and p.KSS (the planner only
// produces the combinations listed here).  Returns an ig3 status.
template <int EPI>
int launch_kernel(const TcParams& p, size_t smem, int grid, cudaStream_t stream) {
  auto go = [&](auto kernel) -> int {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_status(e, "conv3d TC: set shared memory size");
    kernel<<<grid, kThreads, smem, stream>>>(p);
    return count_launch(cuda_status(cudaGetLastError(), "conv3d TC kernel launch"));
  };
  const int key = p.scheme * 100 + p.T * 10 + p.KSS;
  switch (key) {
    case 11: return go(conv3d_tc_kernel<EPI, 0, 1, 1>);
    case 12: return go(conv3d_tc_kernel<EPI, 0, 1, 2>);
    case 14: return go(conv3d_tc_kernel<EPI, 0, 1, 4>);
    case 21: return go(conv3d_tc_kernel<EPI, 0, 2, 1>);
    case 22: return go(conv3d_tc_kernel<EPI, 0, 2, 2>);
    case 24: return go(conv3d_tc_kernel<EPI, 0, 2, 4>);
    case 41: return go(conv3d_tc_kernel<EPI, 0, 4, 1>);
    case 42: return go(conv3d_tc_kernel<EPI, 0, 4, 2>);
    case 44: return go(conv3d_tc_kernel<EPI, 0, 4, 4>);
    case 111: return go(conv3d_tc_kernel<EPI, 1, 1, 1>);
    case 112: return go(conv3d_tc_kernel<EPI, 1, 1, 2>);
    default: return fail(IG3_ERR_UNSUPPORTED, "conv3d TC: no kernel variant for scheme %d, T %d, %d K-steps per stage",
                         p.scheme, p.T, p.KSS);
  }
}

extern template int launch_kernel<IG3_EPI_NONE>(const TcParams&, size_t, int, cudaStream_t);
extern template int launch_kernel<IG3_EPI_TANH_MISH>(const TcParams&, size_t, int, cudaStream_t);
extern template int launch_kernel<IG3_EPI_POOL_REDUCE>(const TcParams&, size_t, int, cudaStream_t);

}  // namespace tc
}  // namespace ig3
