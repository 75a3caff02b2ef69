// fa_prefill_sm103.cu - attention forward with dropout on the weights, head
// dimension 128, on sm_103a (launch_prefill also dispatches: the plain
// forward at D = 128 runs on fa_prefill_d128_sm103.cu, and D = 64 on
// fa_prefill_d64x1_sm103.cu / fa_prefill_d64_sm103.cu).
//
// One CTA owns two 128-row query tiles (Q0, Q1) of one (batch, head) and
// streams that head's K/V in 128-key tiles through a shared-memory ring.
// Both matrix products run on the 5th-generation tensor cores:
//   S_t = Q_t K_j^T   tcgen05.mma, A = Q_t (smem), B = K_j (smem), fp32 in TMEM
//   O_t += P_t V_j    tcgen05.mma, A = P_t (smem, bf16), B = V_j (smem), fp32 in TMEM
// and the softmax runs in between on CUDA cores, one thread per query row.
//
// The per-row update is the online-softmax recurrence of "NTU Hung-yi Lee ML
// 2026 Guide: Faster Generation, Part 1: Flash Attention" (quidproquo.cc),
// "Expand: why multiplying by exp(d1 - d2) fixes it" and "Expand: the
// correction for the output O": with d the running max and s the running
// denominator, a new tile moves d to max(d, tile max), multiplies s and O by
// exp(d_old - d_new) and adds the tile's terms.  The kernel keeps O
// unnormalised (the guide's O_k multiplied through by s_k) and divides by s
// once at the end, which is the same quantity.  It works in base 2:
// x = score * scale * log2(e), exp(a - d) = 2^(x - m).  A rescale is only
// applied when the running max grows by more than kRescaleLog2 (2^8): for
// any common reference value the ratio O/s is unchanged (the guide's rescale
// identity holds for any d2), and bounding the growth keeps 2^(x - m) <= 2^8.
//
// Warp roles (12 warps, 384 threads, one CTA per SM):
//   warp 0        TMA producer: Q0, Q1 once; then K_0, K_1, ... into the K ring
//   warp 1        TMEM allocation; lane 0 issues the MMAs of query tile 0
//   warp 2        TMA producer: V_0, V_1, ... into the V ring
//   warp 3        lane 0 issues the MMAs of query tile 1
//   warps 4-7     softmax + epilogue for Q0 (TMEM lanes 0-127 = its 128 rows)
//   warps 8-11    softmax + epilogue for Q1
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D).
// P_t goes to shared memory (128 x 128 bf16 in the 128-byte-swizzled K-major
// layout of a TMA tile), so S_t(j+1) no longer waits for P_t(j) V: each
// issuer computes S_t(j) as soon as its softmax group holds S_t(j-1) in
// registers, and P_t(j-1) V_(j-1) once P_t(j-1) is in shared memory; the
// softmax computes all 128 weights of a row in registers, then waits for the
// previous P V (O stable, P buffer free), rescales O if needed and stores P.
// With P read from shared memory both products stream two operands from it,
// and its bandwidth bounds the iteration (measured: the P stores wait behind
// the tensor core's operand reads); against P in TMEM overwriting S, where the
// next S waited for the P V of the same tile, this runs 3-5 % faster.
// Shared memory: Q0, Q1, the K ring (2 stages), V (1 stage), P0, P1: 224 KB.
#include "fa_internal.h"
#include "philox.cuh"
#include "sm103_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

constexpr int kThreads = 384;
// Registers per thread after the role split: 128 threads x kRegsCtl + 256 x
// kRegsSoftmax = 63488 <= 384 x 168 (the launch allocation).
constexpr uint32_t kRegsCtl = 80;
constexpr uint32_t kRegsSoftmax = 208;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kSubBytes = 128 * 128;  // one 128-row x 64-column bf16 sub-block (16 KB)

template <int D>
struct Cfg {
  static constexpr int kTileBytes = 128 * D * 2;   // one 128-row tile (one TMA box)
  static constexpr int kKStages = (D == 128) ? 2 : 4;   // K ring
  static constexpr int kVStages = (D == 128) ? 1 : 4;   // V ring
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kPOff = kVOff + kVStages * kTileBytes;   // P_t: 128 x 128 bf16, K-major SW128
  static constexpr int kPBytes = 128 * 128 * 2;
  static constexpr int kBarOff = kPOff + 2 * kPBytes;
  // barriers: q_full[2] kfull[SK] kempty[SK] vfull[SV] vempty[SV] s_full[2] p_full[2] o_full[2] mma_done
  static constexpr int kBarQ = 0;
  static constexpr int kBarKFull = 16;
  static constexpr int kBarKEmpty = kBarKFull + 8 * kKStages;
  static constexpr int kBarVFull = kBarKEmpty + 8 * kKStages;
  static constexpr int kBarVEmpty = kBarVFull + 8 * kVStages;
  static constexpr int kBarS = kBarVEmpty + 8 * kVStages;
  static constexpr int kBarP = kBarS + 16;
  static constexpr int kBarO = kBarP + 16;
  static constexpr int kBarSFree = kBarO + 16;
  static constexpr int kBarPV = kBarSFree + 16;
  static constexpr int kBarDone = kBarPV + 16;
  static constexpr int kTmemHolder = kBarDone + 16;   // after the two issuers' done barriers
  static constexpr int kAbort = kTmemHolder + 4;
  static constexpr int kMiscBytes = 256;
  static_assert(kAbort + 4 <= kMiscBytes, "barrier area overflow");
  static constexpr int kSmemBytes = kBarOff + kMiscBytes + 1024;  // + alignment slack
};

struct Params {
  __nv_bfloat16* o;
  float* lse;
  int* err;
  int BH, Lq, Lk;
  int n_qblk;       // ceil(Lq / 256)
  int group;   // heads per group of the grid order (K/V of a group stay in L2)
  int causal;
  float scale_log2;  // scale * log2(e)
  // dropout on the weights (the DROP instantiation only): bits from
  // philox.cuh's contract, key kept iff its byte >= t, O scaled by keep_scale
  uint32_t seed_lo, seed_hi, offset, drop_t4;   // drop_t4 = t * 0x01010101
  float keep_scale;
};

// Bounded wait that ignores the abort flag: used only to drain this CTA's own
// asynchronous operations before exit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > 50000000ull) return;  // 50 ms
  }
}

// Two counters under one key, their rounds interleaved so that the two
// independent multiply chains overlap; the same bits as two philox4x32_10
// calls (philox.cuh).
__device__ __forceinline__ void philox4x32_10_x2(uint4& a, uint4& b, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t ahi0 = __umulhi(0xD2511F53u, a.x), alo0 = 0xD2511F53u * a.x;
    const uint32_t bhi0 = __umulhi(0xD2511F53u, b.x), blo0 = 0xD2511F53u * b.x;
    const uint32_t ahi1 = __umulhi(0xCD9E8D57u, a.z), alo1 = 0xCD9E8D57u * a.z;
    const uint32_t bhi1 = __umulhi(0xCD9E8D57u, b.z), blo1 = 0xCD9E8D57u * b.z;
    a = make_uint4(ahi1 ^ a.y ^ k0, alo1, ahi0 ^ a.w ^ k1, alo0);
    b = make_uint4(bhi1 ^ b.y ^ k0, blo1, bhi0 ^ b.w ^ k1, blo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

template <int D, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fa_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base + C::kQOff;
  const uint32_t sK = base + C::kKOff;
  const uint32_t sV = base + C::kVOff;
  const uint32_t sBar = base + C::kBarOff;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + C::kBarOff + C::kTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBarOff + C::kAbort);

  auto bar_q = [&](int t) { return sBar + C::kBarQ + 8 * t; };
  auto bar_kfull = [&](int s) { return sBar + C::kBarKFull + 8 * s; };
  auto bar_kempty = [&](int s) { return sBar + C::kBarKEmpty + 8 * s; };
  auto bar_vfull = [&](int s) { return sBar + C::kBarVFull + 8 * s; };
  auto bar_vempty = [&](int s) { return sBar + C::kBarVEmpty + 8 * s; };
  auto bar_s = [&](int t) { return sBar + C::kBarS + 8 * t; };
  auto bar_p = [&](int t) { return sBar + C::kBarP + 8 * t; };
  auto bar_o = [&](int t) { return sBar + C::kBarO + 8 * t; };
  auto bar_sfree = [&](int t) { return sBar + C::kBarSFree + 8 * t; };
  auto bar_pv = [&](int t) { return sBar + C::kBarPV + 8 * t; };
  const uint32_t bar_done = sBar + C::kBarDone;
  const uint32_t sP = base + C::kPOff;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which query tiles this CTA owns (heads in groups whose K/V stay in
  // L2; within a group the heaviest query blocks first)
  const TileOrder to = grouped_tile_order(blockIdx.x, p.BH, p.n_qblk, p.group);
  const int qblk = p.n_qblk - 1 - to.rank;
  const int bh = to.bh;
  const int q0 = qblk * 256;
  const int nk_all = (p.Lk + 127) / 128;
  int nt[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = q0 + 128 * t;
    if (qt >= p.Lq) {
      nt[t] = 0;
    } else if (p.causal) {
      const int last_row = min(qt + 127, p.Lq - 1);
      nt[t] = min(nk_all, last_row / 128 + 1);
    } else {
      nt[t] = nk_all;
    }
  }
  const int nkv = max(nt[0], nt[1]);

  // ---- setup: barriers, TMEM
  if (threadIdx.x == 0) {
    mbar_init(bar_q(0), 1);
    mbar_init(bar_q(1), 1);
    // each MMA issuer releases every ring stage once (count 2 when both query
    // tiles have work)
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bar_kfull(s), 1);
      mbar_init(bar_kempty(s), nt[1] > 0 ? 2 : 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bar_vfull(s), 1);
      mbar_init(bar_vempty(s), nt[1] > 0 ? 2 : 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s(t), 1);
      mbar_init(bar_p(t), 128);
      mbar_init(bar_o(t), 1);
      mbar_init(bar_sfree(t), 128);
      mbar_init(bar_pv(t), 1);
    }
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
  // warp-uniform warpgroup index (the shuffle makes the uniformity explicit)
  const int wgrp = __shfl_sync(0xffffffffu, int(threadIdx.x) / 128, 0);

  if (wgrp == 0) {
    setmaxnreg_dec<kRegsCtl>();
  if (warp == 0 || warp == 2) {
    // =================== TMA producers ===================
    // Warp 0 streams Q and K, warp 2 streams V: TMA boxes issued by one thread
    // are processed one after the other, so two issuing threads double the
    // load rate.  One box = one 128-row tile (all D columns, D/64 swizzled
    // 128-byte column blocks).
    if (lane == 0) {
      const bool is_k = (warp == 0);
      const int NS = is_k ? C::kKStages : C::kVStages;
      const uint32_t ring = is_k ? sK : sV;
      const CUtensorMap* map = is_k ? &tmK : &tmV;
      if (is_k) {
        mbar_arrive_expect_tx(bar_q(0), C::kTileBytes);
        tma_load_tile(sQ, &tmQ, bar_q(0), q0, bh);
        if (nt[1] > 0) {
          mbar_arrive_expect_tx(bar_q(1), C::kTileBytes);
          tma_load_tile(sQ + C::kTileBytes, &tmQ, bar_q(1), q0 + 128, bh);
        }
      }
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int s = j % NS;
        const int use = j / NS;
        const uint32_t empty = is_k ? bar_kempty(s) : bar_vempty(s);
        const uint32_t full = is_k ? bar_kfull(s) : bar_vfull(s);
        if (!mbar_wait(empty, (use & 1) ^ 1, abort_flag, p.err, kSiteProducerEmpty)) break;
        mbar_arrive_expect_tx(full, C::kTileBytes);
        tma_load_tile(ring + s * C::kTileBytes, map, full, j * 128, bh);
        ++issued;
      }
      // drain: every copy this thread started has landed before the CTA exits
      if (is_k) {
        drain_wait(bar_q(0), 0);
        if (nt[1] > 0) drain_wait(bar_q(1), 0);
      }
      for (int s = 0; s < NS && s < issued; ++s) {
        const int last = s + NS * ((issued - 1 - s) / NS);
        drain_wait(is_k ? bar_kfull(s) : bar_vfull(s), (last / NS) & 1);
      }
    }
  } else if (warp == 1 || (warp == 3 && nt[1] > 0)) {
    // =================== MMA issuers: warp 1 for query tile 0, warp 3 for tile 1 ===================
    if (lane == 0) {
      const int t = (warp == 1) ? 0 : 1;
      const int n = nt[t];
      constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, false, true);
      constexpr uint64_t kDescK = sdesc_sw128(0, 16, 1024);
      constexpr uint64_t kDescMN = sdesc_sw128(0, kSubBytes, 1024);
      bool ok = true;
      auto wait = [&](uint32_t b, uint32_t ph, int site) {
        if (ok && !mbar_wait(b, ph, abort_flag, p.err, site)) ok = false;
        return ok;
      };
      const uint32_t a0 = sQ + t * C::kTileBytes;
      const uint32_t pt = sP + t * C::kPBytes;
      wait(bar_q(t), 0, kSiteMmaQ);
      // j: S_t(j) once K_j is in and the softmax holds S_t(j-1) in registers;
      // then P_t(j-1) V_(j-1) once P_t(j-1) is in shared memory.  Every key
      // tile's K and V stages are released by this issuer too.
      for (int j = 0; j <= nkv && ok; ++j) {
        if (j < nkv) {
          const int ks = j % C::kKStages;
          if (!wait(bar_kfull(ks), (j / C::kKStages) & 1, kSiteMmaK)) break;
          if (j < n) {
            if (j > 0 && !wait(bar_sfree(t), (j - 1) & 1, kSiteMmaS)) break;
            tc_fence_after();
            const uint32_t kaddr = sK + ks * C::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kSubBytes + (kk & 3) * 32;
              umma_ss(tmem + t * 128, sdesc_at(kDescK, a0 + off), sdesc_at(kDescK, kaddr + off), kIdQK,
                      kk > 0 ? 1u : 0u);
            }
            umma_commit(bar_s(t));
          }
          umma_commit(bar_kempty(ks));
        }
        if (j > 0) {
          const int vs = (j - 1) % C::kVStages;
          if (!wait(bar_vfull(vs), ((j - 1) / C::kVStages) & 1, kSiteMmaV)) break;
          if (j - 1 < n) {
            if (!wait(bar_p(t), (j - 1) & 1, kSiteMmaP)) break;
            tc_fence_after();
            const uint32_t vaddr = sV + vs * C::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * kSubBytes + (kk & 3) * 32;
              umma_ss(tmem + 256 + t * D, sdesc_at(kDescK, pt + off),
                      sdesc_at(kDescMN, vaddr + kk * 16 * 128), kIdPV, (j - 1 > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(bar_pv(t));
            if (j - 1 == n - 1) umma_commit(bar_o(t));
          }
          umma_commit(bar_vempty(vs));
        }
      }
      // every MMA issued above has completed before TMEM is released
      umma_commit(bar_done + 8 * t);
      drain_wait(bar_done + 8 * t, 0);
    }
  }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // =================== softmax + epilogue ===================
    const int t = (warp - 4) >> 2;
    const int g = warp & 3;                      // TMEM lane quarter of this warp
    const int r = g * 32 + lane;                 // row within the query tile
    const int qt = q0 + 128 * t;
    const int qrow = qt + r;
    const uint32_t lane_off = uint32_t(g * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t sPt = sP + t * C::kPBytes;
    const uint32_t tO = tmem + lane_off + 256 + t * D;
    const float c = p.scale_log2;
    float m_run = -INFINITY;  // running max, log2 units
    float l_run = 0.f;        // running denominator relative to m_run
    bool ok = true;
    const int n = t ? nt[1] : nt[0];

    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_s(t), j & 1, abort_flag, p.err, kSiteSoftmaxS));
      if (!ok) break;
      tc_fence_after();
      float s[128];
      tmem_ld128_sync(tS, s);
      tc_fence_before();
      mbar_arrive(bar_sfree(t));   // S_t is in registers: the next S_t may be computed

      const int k0 = j * 128;
      const bool edge = (k0 + 128 > p.Lk) || (p.causal && k0 + 127 > qt);
      if (edge) {
        // keys k0 + i with i < lim are visible: i < Lk - k0, and i <= qrow - k0 when causal
        const int lim = min(p.Lk - k0, p.causal ? qrow - k0 + 1 : 128);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) s[i] = -INFINITY;
      }
      // row max: 16 independent partial maxima (3-input max), then a short tree
      float pm[16];
#pragma unroll
      for (int g2 = 0; g2 < 16; ++g2) {
        float a = fmax3(s[8 * g2], s[8 * g2 + 1], s[8 * g2 + 2]);
        a = fmax3(a, s[8 * g2 + 3], s[8 * g2 + 4]);
        a = fmax3(a, s[8 * g2 + 5], s[8 * g2 + 6]);
        pm[g2] = fmaxf(a, s[8 * g2 + 7]);
      }
      const float mx = fmax3(fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]),
                                   fmax3(pm[6], pm[7], pm[8])),
                             fmax3(pm[9], pm[10], pm[11]),
                             fmax3(fmax3(pm[12], pm[13], pm[14]), pm[15], -INFINITY));
      const float m_cand = fmaxf(m_run, mx * c);
      const bool need = (m_cand - m_run) > kRescaleLog2;  // true on the first tile
      const bool any = __any_sync(0xffffffffu, need);
      const float m_use = any ? m_cand : m_run;
      const float m_safe = (m_use == -INFINITY) ? 0.f : m_use;
      const float alpha = ex2_approx(m_run - m_safe);    // 0 on the first tile
      m_run = m_use;

      // P = 2^(x - m) in bf16 pairs, all 128 keys in registers first;
      // x - m = s * c - m as packed fp32x2 FMAs, row sum in 8 independent chains
      const float2 c2 = make_float2(c, c);
      const float2 nm2 = make_float2(-m_safe, -m_safe);
      float2 acc[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) acc[a] = make_float2(0.f, 0.f);
      uint32_t pk[4][16];
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint4 dw;          // dropout bits of the current 16 keys
        uint32_t keep4;    // keep bytes of the current 4 keys
        uint4 dw2;         // bits of the block's second 16 keys (both drawn up front)
        if constexpr (DROP) {
          const uint32_t g16 = uint32_t(k0 + 32 * cb) >> 4;
          dw = make_uint4(g16, uint32_t(qrow), uint32_t(bh), p.offset);
          dw2 = make_uint4(g16 + 1u, uint32_t(qrow), uint32_t(bh), p.offset);
          philox4x32_10_x2(dw, dw2, p.seed_lo, p.seed_hi);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if constexpr (DROP)
            if (i == 8) dw = dw2;
          const float2 x = __ffma2_rn(make_float2(s[32 * cb + 2 * i], s[32 * cb + 2 * i + 1]), c2, nm2);
          const float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          acc[i & 3] = __fadd2_rn(acc[i & 3], pr);   // the row sum keeps the undropped weights
          pk[cb][i] = pack_bf16x2(pr.x, pr.y);
          if constexpr (DROP) {
            if ((i & 1) == 0) {
              const uint32_t wsel = ((i >> 1) & 3) == 0 ? dw.x : ((i >> 1) & 3) == 1 ? dw.y
                                  : ((i >> 1) & 3) == 2 ? dw.z : dw.w;
              keep4 = __vcmpgeu4(wsel, p.drop_t4);
            }
            pk[cb][i] &= dropout_pair_mask(keep4, i & 1);
          }
        }
      }
      const float2 a01 = __fadd2_rn(acc[0], acc[1]);
      const float2 a23 = __fadd2_rn(acc[2], acc[3]);
      const float2 a03 = __fadd2_rn(a01, a23);
      l_run = l_run * alpha + (a03.x + a03.y);

      // P_t(j-1) V has completed: O_t is stable and the P_t buffer is free
      if (j > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_pv(t), (j - 1) & 1, abort_flag, p.err, kSiteSoftmaxO));
        if (!ok) break;
        tc_fence_after();
      }
      if (any && j > 0) {
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float ov[32];
          tmem_ld32_sync(tO + cc, ov);
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(ov[i] * alpha);
          tmem_st32(tO + cc, w);
        }
      }
      // P row r into the K-major 128-byte-swizzled tile: keys 8c .. 8c+7 are
      // 16-byte chunk c, in block c / 8 (16 KB apart), at row r's chunk
      // position (c mod 8) xor (r mod 8)
#pragma unroll
      for (int cb = 0; cb < 4; ++cb)
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          const int ch = 4 * cb + m4;
          const uint32_t addr = sPt + (ch >> 3) * kSubBytes + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[cb][4 * m4]),
                       "r"(pk[cb][4 * m4 + 1]), "r"(pk[cb][4 * m4 + 2]), "r"(pk[cb][4 * m4 + 3])
                       : "memory");
        }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p(t));
    }

    // epilogue: O / l -> bf16, LSE = (m + log2 l) * ln 2
    if (ok && n > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bar_o(t), 0, abort_flag, p.err, kSiteSoftmaxO));
    if (ok && n > 0) {
      tc_fence_after();
      const float inv_l = DROP ? p.keep_scale / l_run : 1.f / l_run;
      const bool valid = qrow < p.Lq;
      __nv_bfloat16* orow = p.o + (size_t(bh) * p.Lq + (valid ? qrow : 0)) * D;
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 32) {
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

  // ---- teardown: all TMEM traffic of this CTA is finished
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

namespace {
template <int D, bool DROP>
int launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Lq,
           int Lk, float scale, int causal, const Dropout& dr, cudaStream_t stream, int* err) {
  using C = Cfg<D>;
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  int st = make_tensor_map_bf16(&mq, q, BH, Lq, D);
  if (st == 0) st = make_tensor_map_bf16(&mk, k, BH, Lk, D);
  if (st == 0) st = make_tensor_map_bf16(&mv, v, BH, Lk, D);
  if (st != 0) return st;

  Params p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err = err;
  p.BH = BH;
  p.Lq = Lq;
  p.Lk = Lk;
  p.n_qblk = (Lq + 255) / 256;
  p.group = l2_head_group(BH, 2ll * Lk * D * 2);   // K and V of a head
  p.causal = causal;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.seed_lo = dr.seed_lo;
  p.seed_hi = dr.seed_hi;
  p.offset = dr.offset;
  p.drop_t4 = dr.t * 0x01010101u;
  p.keep_scale = dr.keep_scale;

  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  if (cudaFuncSetAttribute(fa_prefill_kernel<D, DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess)
    return -4;
  const long long nblk = (long long)p.n_qblk * BH;
  if (nblk > 0x7fffffffLL) return -2;
  fa_prefill_kernel<D, DROP><<<dim3(unsigned(nblk)), dim3(kThreads), C::kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
}  // namespace

int launch_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int Lq, int Lk, int D, float scale, int causal, cudaStream_t stream, int* err,
                   const Dropout& dr) {
  if (D == 64) return launch_prefill_d64(q, k, v, o, lse, B, H, Lq, Lk, scale, causal, stream, err, dr);
  if (D == 128)
    return dr.on ? launch<128, true>(q, k, v, o, lse, B, H, Lq, Lk, scale, causal, dr, stream, err)
                 : launch_prefill_d128(q, k, v, o, lse, B, H, Lq, Lk, scale, causal, stream, err);
  return -2;
}

}  // namespace fa
