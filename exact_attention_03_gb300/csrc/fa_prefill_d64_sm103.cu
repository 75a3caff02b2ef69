// fa_prefill_d64_sm103.cu - attention forward for head dimension 64 on sm_103a
// with dropout on the weights (the plain forward at D = 64 runs on
// fa_prefill_d64x1_sm103.cu, one query tile per CTA).
//
// Two 128-row query tiles per CTA,
// S = Q K^T and O += P V on the tensor cores, the online-softmax recurrence of
// "NTU Hung-yi Lee ML 2026 Guide: Faster Generation, Part 1: Flash Attention"
// (quidproquo.cc), "Expand: why multiplying by exp(d1 - d2) fixes it" and
// "Expand: the correction for the output O", in base 2 with a lazily applied
// rescale), but scheduled for D = 64, where one 128-key tile costs the softmax
// (MUFU exponentials) about as much time as the tensor core:
//
//  * P has its own TMEM columns instead of overwriting S, so the next scores
//    S(j+1) are computed while the softmax still works on tile j: the softmax
//    releases S as soon as it has loaded it into registers.
//  * Each query tile has its own pipeline: its own MMA-issuing thread (warp 1
//    for tile 0, warp 3 for tile 1), barriers, S, P and O.  The two pipelines
//    share only the K/V ring and the tensor core, and their softmax groups run
//    about half an iteration apart (the second starts once the first has its
//    first half tile of weights), so that one group's TMEM loads, barrier waits
//    and the drain of its exponentials overlap the other's exponentials.
//  * Without dropout, exponentials would be taken against the running
//    maximum and checked afterwards, the row maximum computed only when the
//    check fails; with dropout (the only form this file now runs) every tile
//    takes its row maximum first, since a recomputed tile would draw its
//    random bits twice.
//  * K_j and V_j share one ring slot and one "full" barrier (two producer
//    warps, one TMA box each).
//
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384)
//                     P0 [384,448) P1 [448,512)  (P: bf16 pairs, 128 keys)
// Warps: 0 = TMA producer for Q and K, 1 = TMEM allocation + MMA issue for Q0,
// 2 = TMA producer for V, 3 = MMA issue for Q1, 4-7 = softmax of Q0,
// 8-11 = softmax of Q1.
#include "fa_internal.h"
#include "philox.cuh"
#include "sm103_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

constexpr int kThreads = 384;
// 128 threads x 80 + 256 threads x 208 = 63488 <= 384 x 168 registers at launch
constexpr uint32_t kRegsCtl = 80;
constexpr uint32_t kRegsSoftmax = 208;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleBound = 256.0f;        // 2^kRescaleLog2
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kD = 64;
constexpr int kTileBytes = 128 * kD * 2;       // one 128-row tile, one TMA box (16 KB)
constexpr int kStages = 5;                     // K/V slot pairs
constexpr int kQOff = 0;
constexpr int kKVOff = 2 * kTileBytes;         // slot s: K at +2s tiles, V at +2s+1 tiles
constexpr int kBarOff = kKVOff + kStages * 2 * kTileBytes;
constexpr int kBarQ = 0;
constexpr int kBarKVFull = 16;
constexpr int kBarKVEmpty = kBarKVFull + 8 * kStages;
constexpr int kBarS = kBarKVEmpty + 8 * kStages;   // [t] S_t(j) written
constexpr int kBarSFree = kBarS + 16;              // [t] softmax group t loaded S_t(j)
constexpr int kBarP = kBarSFree + 16;              // [t] P_t(j) written (O_t rescaled)
constexpr int kBarPV = kBarP + 16;                 // [t] PV_t(j) completed
constexpr int kBarGo = kBarPV + 16;                // group 0 is half a tile ahead
constexpr int kBarDone = kBarGo + 8;               // [t] all MMAs of issuer t completed
constexpr int kTmemHolder = kBarDone + 16;
constexpr int kAbort = kTmemHolder + 4;
constexpr int kMiscBytes = 256;
static_assert(kAbort + 4 <= kMiscBytes, "barrier area overflow");
constexpr int kSmemBytes = kBarOff + kMiscBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;

struct Params {
  __nv_bfloat16* o;
  float* lse;
  int* err;
  int BH, Lq, Lk;
  int n_qblk;  // ceil(Lq / 256)
  int group;   // heads per group of the grid order (K/V of a group stay in L2)
  int causal;
  float scale_log2;
  // dropout on the weights (the DROP instantiation only): bits from
  // philox.cuh's contract, key kept iff its byte >= t, O scaled by keep_scale
  uint32_t seed_lo, seed_hi, offset;
  uint32_t drop_tl4, drop_hsel;   // (t mod 128) * 0x01010101; all ones iff t >= 128
  PhiloxKeys keys;                 // round keys 3..10 of the seed
  float keep_scale;
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > 50000000ull) return;  // 50 ms
  }
}

// maximum of a 128-key score row (3-input max tree)
__device__ __forceinline__ float row_max128(const float (&s)[128]) {
  float pm[16];
#pragma unroll
  for (int g2 = 0; g2 < 16; ++g2) {
    float a = fmax3(s[8 * g2], s[8 * g2 + 1], s[8 * g2 + 2]);
    a = fmax3(a, s[8 * g2 + 3], s[8 * g2 + 4]);
    a = fmax3(a, s[8 * g2 + 5], s[8 * g2 + 6]);
    pm[g2] = fmaxf(a, s[8 * g2 + 7]);
  }
  return fmax3(fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmax3(pm[6], pm[7], pm[8])),
               fmax3(pm[9], pm[10], pm[11]), fmax3(fmax3(pm[12], pm[13], pm[14]), pm[15], -INFINITY));
}

template <bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fa_prefill_d64_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base + kQOff;
  const uint32_t sKV = base + kKVOff;
  const uint32_t sBar = base + kBarOff;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + kBarOff + kTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kBarOff + kAbort);

  auto bar_q = [&](int t) { return sBar + kBarQ + 8 * t; };
  auto bar_kvfull = [&](int s) { return sBar + kBarKVFull + 8 * s; };
  auto bar_kvempty = [&](int s) { return sBar + kBarKVEmpty + 8 * s; };
  auto bar_s = [&](int t) { return sBar + kBarS + 8 * t; };
  auto bar_sfree = [&](int t) { return sBar + kBarSFree + 8 * t; };
  auto bar_p = [&](int t) { return sBar + kBarP + 8 * t; };
  auto bar_pv = [&](int t) { return sBar + kBarPV + 8 * t; };
  const uint32_t bar_go = sBar + kBarGo;
  const uint32_t bar_done = sBar + kBarDone;
  auto slot_k = [&](int s) { return sKV + (2 * s) * kTileBytes; };
  auto slot_v = [&](int s) { return sKV + (2 * s + 1) * kTileBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which query tiles this CTA owns (heads in groups whose K/V stay in
  // L2; within a group the heaviest query blocks first)
  const TileOrder to = grouped_tile_order(blockIdx.x, p.BH, p.n_qblk, p.group);
  const int qblk = p.n_qblk - 1 - to.rank;
  const int bh = to.bh;
  const int q0 = qblk * 256;
  const int nk_all = (p.Lk + 127) / 128;
  // key tiles of query tile 0 and 1; nt0 >= 1, and nt1 is 0 (tile 1 past the
  // end of the sequence) or nt1 >= nt0
  const int nt0 = p.causal ? min(nk_all, min(q0 + 127, p.Lq - 1) / 128 + 1) : nk_all;
  const int nt1 = (q0 + 128 >= p.Lq) ? 0
                  : (p.causal ? min(nk_all, min(q0 + 255, p.Lq - 1) / 128 + 1) : nk_all);
  const int nkv = max(nt0, nt1);

  if (threadIdx.x == 0) {
    mbar_init(bar_q(0), 1);
    mbar_init(bar_q(1), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_kvfull(s), 2);  // the K and the V producer each arrive (with bytes)
      mbar_init(bar_kvempty(s), nt1 > 0 ? 2 : 1);  // each MMA issuer commits once per key tile
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s(t), 1);
      mbar_init(bar_sfree(t), 128);
      mbar_init(bar_p(t), 128);
      mbar_init(bar_pv(t), 1);
    }
    mbar_init(bar_go, 128);
    mbar_init(bar_done, 1);
    mbar_init(bar_done + 8, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int wgrp = __shfl_sync(0xffffffffu, int(threadIdx.x) / 128, 0);

  if (wgrp == 0) {
    setmaxnreg_dec<kRegsCtl>();
    if (warp == 0 || warp == 2) {
      // =================== TMA producers (warp 0: Q and K, warp 2: V) ===================
      if (lane == 0) {
        const bool is_k = (warp == 0);
        if (is_k) {
          mbar_arrive_expect_tx(bar_q(0), kTileBytes);
          tma_load_tile(sQ, &tmQ, bar_q(0), q0, bh);
          if (nt1 > 0) {
            mbar_arrive_expect_tx(bar_q(1), kTileBytes);
            tma_load_tile(sQ + kTileBytes, &tmQ, bar_q(1), q0 + 128, bh);
          }
        }
        int issued = 0;
        for (int j = 0; j < nkv; ++j) {
          const int s = j % kStages;
          const int use = j / kStages;
          if (!mbar_wait(bar_kvempty(s), (use & 1) ^ 1, abort_flag, p.err, kSiteProducerEmpty)) break;
          mbar_arrive_expect_tx(bar_kvfull(s), kTileBytes);
          tma_load_tile(is_k ? slot_k(s) : slot_v(s), is_k ? &tmK : &tmV, bar_kvfull(s), j * 128, bh);
          ++issued;
        }
        if (is_k) {
          drain_wait(bar_q(0), 0);
          if (nt1 > 0) drain_wait(bar_q(1), 0);
        }
        for (int s = 0; s < kStages && s < issued; ++s) {
          const int last = s + kStages * ((issued - 1 - s) / kStages);
          drain_wait(bar_kvfull(s), (last / kStages) & 1);
        }
      }
    } else if (warp == 1 || (warp == 3 && nt1 > 0)) {
      // =================== MMA issuers: warp 1 for query tile 0, warp 3 for tile 1 ===================
      if (lane == 0) {
        const int t = (warp == 1) ? 0 : 1;
        const int n = t ? nt1 : nt0;
        constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t kIdPV = idesc_bf16_f32(128, kD, false, true);
        constexpr uint64_t kDescK = sdesc_sw128(0, 16, 1024);      // Q, K: K-major
        constexpr uint64_t kDescMN = sdesc_sw128(0, 16, 1024);     // V: MN-major, one 64-col block
        bool ok = true;
        auto wait = [&](uint32_t b, uint32_t ph, int site) {
          if (ok && !mbar_wait(b, ph, abort_flag, p.err, site)) ok = false;
          return ok;
        };
        const uint32_t a0 = sQ + t * kTileBytes;
        wait(bar_q(t), 0, kSiteMmaQ);
        for (int j = 0; j <= nkv && ok; ++j) {
          const int sc = j % kStages;
          if (j < nkv && !wait(bar_kvfull(sc), (j / kStages) & 1, kSiteMmaK)) break;
          // S_t(j) once the softmax group holds S_t(j-1) in registers
          if (j < n) {
            if (j > 0 && !wait(bar_sfree(t), (j - 1) & 1, kSiteMmaS)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              umma_ss(tmem + t * 128, sdesc_at(kDescK, a0 + kk * 32), sdesc_at(kDescK, slot_k(sc) + kk * 32),
                      kIdQK, kk > 0 ? 1u : 0u);
            umma_commit(bar_s(t));
          }
          // PV_t(j-1) once P_t(j-1) is written; then this issuer is done with slot j-1
          if (j > 0) {
            const int sp = (j - 1) % kStages;
            if (j - 1 < n) {
              if (!wait(bar_p(t), (j - 1) & 1, kSiteMmaP)) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_ts(tmem + kColO + t * kD, tmem + kColP + t * 64 + kk * 8,
                        sdesc_at(kDescMN, slot_v(sp) + kk * 16 * 128), kIdPV, (j - 1 > 0 || kk > 0) ? 1u : 0u);
              umma_commit(bar_pv(t));
            }
            umma_commit(bar_kvempty(sp));
          }
        }
        umma_commit(bar_done + 8 * t);
        drain_wait(bar_done + 8 * t, 0);
      }
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // =================== softmax + epilogue (one query row per thread) ===================
    const int t = (warp - 4) >> 2;
    const int g = warp & 3;
    const int r = g * 32 + lane;
    const int qt = q0 + 128 * t;
    const int qrow = qt + r;
    const uint32_t lane_off = uint32_t(g * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tP = tmem + lane_off + kColP + t * 64;
    const uint32_t tO = tmem + lane_off + kColO + t * kD;
    const float c = p.scale_log2;
    const int n = t ? nt1 : nt0;
    // the parts of the Philox rounds shared by all of this row's calls
    PhiloxRow prow;
    if constexpr (DROP) prow = philox_row(uint32_t(qrow), uint32_t(bh), p.offset, p.seed_lo, p.seed_hi);
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    // first key tile with masked keys (past Lk, or above the causal diagonal)
    const int j_edge = min(p.Lk / 128, p.causal ? qt / 128 : (1 << 30));

    // group 1 starts once group 0 has its first half tile of weights
    if (t == 1 && n > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bar_go, 0, abort_flag, p.err, kSiteSoftmaxGo));

#pragma unroll 2
    for (int j = 0; j < n && ok; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_s(t), j & 1, abort_flag, p.err, kSiteSoftmaxS));
      if (!ok) break;
      float s[128];
      tc_fence_after();
      tmem_ld128_sync(tS, s);
      tc_fence_before();
      mbar_arrive(bar_sfree(t));  // S_t(j) is in registers: S_t may be overwritten

      float alpha = 1.f;
      bool resc = false;    // warp-uniform: O_t is multiplied by alpha before PV(j)
      float2 acc[4];
      const float2 c2 = make_float2(c, c);
      float2 nm2 = make_float2(0.f, 0.f);
      // 16 pairs of weights of keys 32cb .. 32cb+31, packed to bf16, summed into acc
      auto exp_block = [&](int cb, uint32_t (&w)[16]) {
        uint4 dw;          // dropout bits of the current 16 keys
        uint32_t keep4;    // keep bits (byte top bits) of the current 4 keys
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = 32 * cb + 2 * i;
          if constexpr (DROP)
            if ((i & 7) == 0)
              dw = philox4x32_10_row(uint32_t(j * 128 + e) >> 4, prow, p.keys);
          const float2 x = __ffma2_rn(make_float2(s[e], s[e + 1]), c2, nm2);
          const float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          acc[i & 3] = __fadd2_rn(acc[i & 3], pr);   // the row sum keeps the undropped weights
          w[i] = pack_bf16x2(pr.x, pr.y);
          if constexpr (DROP) {
            if ((i & 1) == 0) {
              const uint32_t wsel = ((i >> 1) & 3) == 0 ? dw.x : ((i >> 1) & 3) == 1 ? dw.y
                                  : ((i >> 1) & 3) == 2 ? dw.z : dw.w;
              keep4 = dropout_keep_msb(wsel, p.drop_tl4, p.drop_hsel);
            }
            w[i] &= dropout_pair_mask(keep4, i & 1);
          }
        }
      };
      auto rescale_o = [&]() {
#pragma unroll 1
        for (int cc = 0; cc < kD; cc += 16) {
          float ov[16];
          tmem_ld16_sync(tO + cc, ov);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(ov[i] * alpha);
          tmem_st16(tO + cc, w);
        }
      };
      uint32_t pk[2][16];   // P of keys 0-63, computed before PV(j-1) has freed P_t
      const int k0 = j * 128;
      const bool edge = j >= j_edge;
      if (edge) {
        const int lim = min(p.Lk - k0, p.causal ? qrow - k0 + 1 : 128);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) s[i] = -INFINITY;
      }
      // Until a row has a finite running maximum its first tile takes the
      // maximum before exponentiating; later tiles exponentiate against the
      // running maximum and check the result afterwards (below).  With dropout
      // every tile takes the maximum first: the random bits already dominate
      // the loop, and a recomputed tile would draw them twice.
      const bool exact = DROP || __any_sync(0xffffffffu, m_run == -INFINITY);
      if (exact) {
        const float m_cand = fmaxf(m_run, row_max128(s) * c);
        resc = __any_sync(0xffffffffu, m_cand > m_run + kRescaleLog2);
        if (resc) {
          alpha = ex2_approx(m_run - ((m_cand == -INFINITY) ? 0.f : m_cand));
          m_run = m_cand;
        }
      }
      {
        const float m_safe = (m_run == -INFINITY) ? 0.f : m_run;
        nm2 = make_float2(-m_safe, -m_safe);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) acc[a] = make_float2(0.f, 0.f);
      exp_block(0, pk[0]);
      exp_block(1, pk[1]);
      if (t == 0 && j == 0) mbar_arrive(bar_go);

      // PV_t(j-1) has completed: O_t is stable and P_t is free
      if (j > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_pv(t), (j - 1) & 1, abort_flag, p.err, kSiteSoftmaxO));
        if (!ok) break;
      }
      tc_fence_after();
      if (resc && j > 0) rescale_o();
      tmem_st16(tP, pk[0]);
      tmem_st16(tP + 16, pk[1]);
      // keys 64-127: computed and stored now that P_t is free
#pragma unroll
      for (int cb = 2; cb < 4; ++cb) {
        uint32_t w[16];
        exp_block(cb, w);
        tmem_st16(tP + 16 * cb, w);
      }
      float2 a03 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
      if (!exact) {
        // Every weight 2^(c s - m_run) is at most the tile's row sum, so a sum
        // up to 2^kRescaleLog2 means the maximum grew by at most kRescaleLog2
        // and the weights stand (the lazy rescale rule).  Otherwise take the
        // maximum, and where it grew further, rescale and recompute the tile.
        const bool check = !(a03.x + a03.y <= kRescaleBound);
        if (__any_sync(0xffffffffu, check)) {
          const float m_cand = fmaxf(m_run, row_max128(s) * c);
          if (__any_sync(0xffffffffu, m_cand > m_run + kRescaleLog2)) {
            alpha = ex2_approx(m_run - m_cand);
            m_run = m_cand;
            nm2 = make_float2(-m_cand, -m_cand);
#pragma unroll
            for (int a = 0; a < 4; ++a) acc[a] = make_float2(0.f, 0.f);
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
              uint32_t w[16];
              exp_block(cb, w);
              tmem_st16(tP + 16 * cb, w);
            }
            a03 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
            if (j > 0) rescale_o();
          }
        }
      }
      l_run = l_run * alpha + (a03.x + a03.y);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p(t));
    }

    // epilogue: wait for the last PV, then O / l -> bf16, LSE
    if (ok && n > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bar_pv(t), (n - 1) & 1, abort_flag, p.err, kSiteSoftmaxO));
    if (ok && n > 0) {
      tc_fence_after();
      const float inv_l = DROP ? p.keep_scale / l_run : 1.f / l_run;
      const bool valid = qrow < p.Lq;
      __nv_bfloat16* orow = p.o + (size_t(bh) * p.Lq + (valid ? qrow : 0)) * kD;
#pragma unroll 1
      for (int cc = 0; cc < kD; cc += 32) {
        float ov[32];
        tmem_ld32_sync(tO + cc, ov);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(ov[2 * i] * inv_l, ov[2 * i + 1] * inv_l);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
          dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
        }
      }
      if (valid && p.lse != nullptr) p.lse[size_t(bh) * p.Lq + qrow] = (m_run + __log2f(l_run)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_prefill_d64(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int Lq, int Lk, float scale, int causal, cudaStream_t stream,
                       int* err, const Dropout& dr) {
  // Without dropout, one query tile per CTA and two CTAs per SM
  // (fa_prefill_d64x1_sm103.cu) measured faster at every length (L = 64 ...
  // 8192, causal 8K and 32K); it does the same arithmetic in the same order,
  // so the outputs are bit-identical.  With dropout this kernel measured
  // faster (L = 8192: 1055 against 1138 us; L = 2048: 86 against 95 us).
  if (!dr.on) return launch_prefill_d64x1(q, k, v, o, lse, B, H, Lq, Lk, scale, causal, stream, err, dr);
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  int st = make_tensor_map_bf16(&mq, q, BH, Lq, kD);
  if (st == 0) st = make_tensor_map_bf16(&mk, k, BH, Lk, kD);
  if (st == 0) st = make_tensor_map_bf16(&mv, v, BH, Lk, kD);
  if (st != 0) return st;
  Params p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err = err;
  p.BH = BH;
  p.Lq = Lq;
  p.Lk = Lk;
  p.n_qblk = (Lq + 255) / 256;
  p.group = l2_head_group(BH, 2ll * Lk * 64 * 2);   // K and V of a head
  p.causal = causal;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.seed_lo = dr.seed_lo;
  p.seed_hi = dr.seed_hi;
  p.offset = dr.offset;
  p.drop_tl4 = (dr.t & 0x7fu) * 0x01010101u;
  p.drop_hsel = dr.t >= 128u ? 0xffffffffu : 0u;
  p.keys = philox_round_keys(dr.seed_lo, dr.seed_hi);
  p.keep_scale = dr.keep_scale;
  const long long nblk = (long long)p.n_qblk * BH;
  if (nblk > 0x7fffffffLL) return -2;
  auto kernel = fa_prefill_d64_kernel<true>;   // dr.on: the plain forward returned above
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return -4;
  kernel<<<dim3(unsigned(nblk)), dim3(kThreads), kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace fa
