// fa_prefill_d128_sm103.cu - attention forward for head dimension 128 on
// sm_103a (plain, and with dropout on the weights).
//
// Two 128-row query tiles (Q0, Q1) of one (batch, head) per CTA; S = Q K^T
// and O += P V on the 5th-generation tensor cores, the weights computed in
// between on CUDA cores (one query row per thread) with the online-softmax
// recurrence of "NTU Hung-yi Lee ML 2026 Guide: Faster Generation, Part 1:
// Flash Attention" (quidproquo.cc), "Expand: why multiplying by exp(d1 - d2)
// fixes it" and "Expand: the correction for the output O": with d the
// running max and s the running denominator, a new tile moves d to max(d,
// tile max), multiplies s and O by exp(d_old - d_new) and adds the tile's
// terms.  O is kept unnormalised (the guide's O_k multiplied through by s_k)
// and divided by s once at the end; everything runs in base 2 (x = score *
// scale * log2 e) and the running maximum moves only when it grows by more
// than 2^8 (the guide's rescale identity holds for any common reference
// value, and the bound keeps every weight <= 2^8).  Data placement and the
// order of the products:
//
//  * TMEM (512 columns): S [0,128) shared by the two query tiles, P0
//    [128,192) and P1 [192,256) (bf16 pairs, 128 keys each), O0 [256,384),
//    O1 [384,512).  P V reads P from TMEM and only V from shared memory, and
//    the softmax stores P with tcgen05.st (an earlier design kept P in
//    shared memory, with one S buffer per query tile: 7 % slower on the
//    causal 8K workload, as both products streamed two operands from shared
//    memory and every P store waited for the previous P V).
//  * Each query tile has its own MMA-issuing thread, which issues S_t(j) and
//    then P_t(j-1) V(j-1).  S_t(j) overwrites the S of the other query tile
//    once that tile's softmax holds it in registers (S0(0), S1(0), S0(1),
//    ...), and P_t(j-1) V runs while the softmax of tile t loads S_t(j) and
//    takes its first exponentials: each softmax has about a whole iteration
//    to produce P_t(j), and waits for P_t(j-1) V only before overwriting P_t.
//    Two issuing threads keep the tensor core busy where one alone would
//    leave gaps between its products (each issue costs the thread about as
//    long as an N = 128 product runs).
//  * Shared memory: Q0, Q1 (32 KB each), a K ring of 3 slots and a V ring of
//    2 slots (32 KB each): 224 KB.
//
// Warps: 0 = TMA producer for Q0, Q1 and K (thread 0 issues Q and K(0)
// right after setting up the barriers), 1 = TMEM allocation + MMA issue for
// Q0, 2 = TMA producer for V, 3 = MMA issue for Q1, 4-7 = softmax + epilogue
// of Q0, 8-11 =
// softmax + epilogue of Q1 (one query row per thread; TMEM lane quarter =
// warp % 4).
#include "fa_internal.h"
#include "philox.cuh"
#include "sm103_ptx.cuh"

#include <cmath>
#include <type_traits>

namespace fa {
namespace {

constexpr int kThreads = 384;
// 128 threads x 80 + 256 threads x 208 = 63488 <= 384 x 168 registers at launch
constexpr uint32_t kRegsCtl = 80;
constexpr uint32_t kRegsSoftmax = 208;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleBound = 256.0f;        // 2^kRescaleLog2
constexpr float kLn2 = 0.69314718055994530942f;
// after a tile had to be recomputed, the rest of the warp's tiles take the
// maximum first: with sharp logits the maximum of some row of a warp keeps
// growing past the bound again and again, and a recomputed tile costs a
// second pass of exponentials
constexpr int kExactAfterRedo = 1 << 30;
constexpr int kD = 128;
constexpr int kTileBytes = 128 * kD * 2;       // one 128-row tile, one TMA box (32 KB)
constexpr int kSubBytes = 128 * 128;           // one 128-row x 64-column block (16 KB)
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kQOff = 0;
constexpr int kKOff = 2 * kTileBytes;
constexpr int kVOff = kKOff + kKStages * kTileBytes;
constexpr int kBarOff = kVOff + kVStages * kTileBytes;
constexpr int kBarQ = 0;                             // [t] Q_t landed
constexpr int kBarKFull = kBarQ + 16;
constexpr int kBarKEmpty = kBarKFull + 8 * kKStages;
constexpr int kBarVFull = kBarKEmpty + 8 * kKStages;
constexpr int kBarVEmpty = kBarVFull + 8 * kVStages;
constexpr int kBarS = kBarVEmpty + 8 * kVStages;     // [t] S_t(j) written
constexpr int kBarSFree = kBarS + 16;                // [t] softmax t loaded S_t(j)
constexpr int kBarP = kBarSFree + 16;                // [t] P_t(j) written (O_t rescaled)
constexpr int kBarPV = kBarP + 16;                   // [t] P_t(j) V completed
constexpr int kBarO = kBarPV + 16;                   // [t] the last P_t V completed
constexpr int kBarDone = kBarO + 16;                 // [t] every product of issuer t completed
constexpr int kTmemHolder = kBarDone + 16;
constexpr int kAbort = kTmemHolder + 4;
constexpr int kMiscBytes = 256;
static_assert(kAbort + 4 <= kMiscBytes, "barrier area overflow");
constexpr int kSmemBytes = kBarOff + kMiscBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kColP = 128;
constexpr uint32_t kColO = 256;

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

// Bounded wait that ignores the abort flag: used only to drain this CTA's own
// asynchronous operations before exit.
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
    fa_prefill_d128_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base + kQOff;
  const uint32_t sK = base + kKOff;
  const uint32_t sV = base + kVOff;
  const uint32_t sBar = base + kBarOff;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + kBarOff + kTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kBarOff + kAbort);

  auto bar_q = [&](int t) { return sBar + kBarQ + 8 * t; };
  auto bar_kfull = [&](int s) { return sBar + kBarKFull + 8 * s; };
  auto bar_kempty = [&](int s) { return sBar + kBarKEmpty + 8 * s; };
  auto bar_vfull = [&](int s) { return sBar + kBarVFull + 8 * s; };
  auto bar_vempty = [&](int s) { return sBar + kBarVEmpty + 8 * s; };
  auto bar_s = [&](int t) { return sBar + kBarS + 8 * t; };
  auto bar_sfree = [&](int t) { return sBar + kBarSFree + 8 * t; };
  auto bar_p = [&](int t) { return sBar + kBarP + 8 * t; };
  auto bar_pv = [&](int t) { return sBar + kBarPV + 8 * t; };
  auto bar_o = [&](int t) { return sBar + kBarO + 8 * t; };
  const uint32_t bar_done = sBar + kBarDone;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which query tiles this CTA owns (heads in groups whose K/V stay in
  // L2; within a group the heaviest query blocks first)
  const TileOrder to = grouped_tile_order(blockIdx.x, p.BH, p.n_qblk, p.group);
  const int qblk = p.n_qblk - 1 - to.rank;
  const int bh = to.bh;
  const int q0 = qblk * 256;
  const int nk_all = (p.Lk + 127) / 128;
  // key tiles of query tile 0 and 1: nt0 >= 1; nt1 is 0 (tile 1 past the end
  // of the sequence) or nt1 >= nt0
  const int nt0 = p.causal ? min(nk_all, min(q0 + 127, p.Lq - 1) / 128 + 1) : nk_all;
  const int nt1 = (q0 + 128 >= p.Lq) ? 0
                  : (p.causal ? min(nk_all, min(q0 + 255, p.Lq - 1) / 128 + 1) : nk_all);
  const int nkv = max(nt0, nt1);

  if (threadIdx.x == 0) {
    mbar_init(bar_q(0), 1);
    mbar_init(bar_q(1), 1);
    // each MMA issuer releases every ring slot once (count 2 when both query
    // tiles have work)
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar_kfull(s), 1);
      mbar_init(bar_kempty(s), nt1 > 0 ? 2 : 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar_vfull(s), 1);
      mbar_init(bar_vempty(s), nt1 > 0 ? 2 : 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s(t), 1);
      mbar_init(bar_sfree(t), 128);
      mbar_init(bar_p(t), 128);
      mbar_init(bar_pv(t), 1);
      mbar_init(bar_o(t), 1);
    }
    mbar_init(bar_done, 1);
    mbar_init(bar_done + 8, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // thread 0 is the K producer: Q and K(0) start loading before the CTA-wide
    // synchronisation (slot 0 of the K ring is free at the start)
    mbar_arrive_expect_tx(bar_q(0), kTileBytes);
    tma_load_tile(sQ, &tmQ, bar_q(0), q0, bh);
    if (nt1 > 0) {
      mbar_arrive_expect_tx(bar_q(1), kTileBytes);
      tma_load_tile(sQ + kTileBytes, &tmQ, bar_q(1), q0 + 128, bh);
    }
    mbar_arrive_expect_tx(bar_kfull(0), kTileBytes);
    tma_load_tile(sK, &tmK, bar_kfull(0), 0, bh);
  }
  if (warp == 2 && lane == 0) tma_prefetch_desc(&tmV);
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
      // One box = one 128-row tile (both 64-column blocks, 128-byte swizzle).
      if (lane == 0) {
        const bool is_k = (warp == 0);
        const int stages = is_k ? kKStages : kVStages;
        // Q and K(0) were issued by this thread before the CTA-wide sync
        const int j0 = is_k ? 1 : 0;
        int issued = j0;
        for (int j = j0; j < nkv; ++j) {
          const int s = j % stages;
          const int use = j / stages;
          const uint32_t empty = is_k ? bar_kempty(s) : bar_vempty(s);
          const uint32_t full = is_k ? bar_kfull(s) : bar_vfull(s);
          if (!mbar_wait(empty, (use & 1) ^ 1, abort_flag, p.err, kSiteProducerEmpty)) break;
          mbar_arrive_expect_tx(full, kTileBytes);
          tma_load_tile(is_k ? sK + s * kTileBytes : sV + s * kTileBytes, is_k ? &tmK : &tmV, full,
                        j * 128, bh);
          ++issued;
        }
        // every copy this thread issued has landed before the CTA can exit
        if (is_k) {
          drain_wait(bar_q(0), 0);
          if (nt1 > 0) drain_wait(bar_q(1), 0);
        }
        for (int s = 0; s < stages && s < issued; ++s) {
          const int last = s + stages * ((issued - 1 - s) / stages);
          drain_wait(is_k ? bar_kfull(s) : bar_vfull(s), (last / stages) & 1);
        }
      }
    } else if (warp == 1 || (warp == 3 && nt1 > 0)) {
      // =================== MMA issuers: warp 1 for query tile 0, warp 3 for tile 1 ===================
      if (lane == 0) {
        const int t = (warp == 1) ? 0 : 1;
        const int n = t ? nt1 : nt0;
        constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t kIdPV = idesc_bf16_f32(128, kD, false, true);
        constexpr uint64_t kDescK = sdesc_sw128(0, 16, 1024);          // Q, K: K-major
        constexpr uint64_t kDescMN = sdesc_sw128(0, kSubBytes, 1024);  // V: MN-major, two 64-col blocks
        bool ok = true;
        auto wait = [&](uint32_t b, uint32_t ph, int site) {
          if (ok && !mbar_wait(b, ph, abort_flag, p.err, site)) ok = false;
          return ok;
        };
        const uint32_t a0 = sQ + t * kTileBytes;
        const uint32_t tD = tmem + kColO + t * kD;
        const uint32_t tA = tmem + kColP + t * 64;
        wait(bar_q(t), 0, kSiteMmaQ);
        // Every issuer walks all key tiles and releases every K and V slot once
        // (the ring barriers count one release per issuer).
        for (int j = 0; j <= nkv && ok; ++j) {
          if (j < nkv) {
            const int ks = j % kKStages;
            if (!wait(bar_kfull(ks), (j / kKStages) & 1, kSiteMmaK)) break;
            if (j < n) {
              // the S buffer's previous owner (S0(0), S1(0), S0(1), S1(1), ...;
              // query tile 0 ends first when causal) must have loaded it
              if (t == 0) {
                if (j > 0 && !wait(bar_sfree(nt1 > 0 ? 1 : 0), (j - 1) & 1, kSiteMmaS)) break;
              } else {
                if (j < nt0 ? !wait(bar_sfree(0), j & 1, kSiteMmaS)
                            : !wait(bar_sfree(1), (j - 1) & 1, kSiteMmaS))
                  break;
              }
              tc_fence_after();
              const uint32_t kaddr = sK + ks * kTileBytes;
#pragma unroll
              for (int kk = 0; kk < kD / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kSubBytes + (kk & 3) * 32;
                umma_ss(tmem, sdesc_at(kDescK, a0 + off), sdesc_at(kDescK, kaddr + off), kIdQK, kk > 0 ? 1u : 0u);
              }
              umma_commit(bar_s(t));
            }
            umma_commit(bar_kempty(ks));
          }
          // P_t(j-1) V(j-1) once P_t(j-1) is written
          if (j > 0) {
            const int vs = (j - 1) % kVStages;
            if (!wait(bar_vfull(vs), ((j - 1) / kVStages) & 1, kSiteMmaV)) break;
            if (j - 1 < n) {
              if (!wait(bar_p(t), (j - 1) & 1, kSiteMmaP)) break;
              tc_fence_after();
              const uint32_t vaddr = sV + vs * kTileBytes;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_ts(tD, tA + kk * 8, sdesc_at(kDescMN, vaddr + kk * 16 * 128), kIdPV,
                        (j - 1 > 0 || kk > 0) ? 1u : 0u);
              umma_commit(bar_pv(t));
              if (j - 1 == n - 1) umma_commit(bar_o(t));
            }
            umma_commit(bar_vempty(vs));
          }
        }
        // every product this thread issued has completed before TMEM is released
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
    const uint32_t tS = tmem + lane_off;
    const uint32_t tP = tmem + lane_off + kColP + t * 64;
    const uint32_t tO = tmem + lane_off + kColO + t * kD;
    const float c = p.scale_log2;
    const int n = t ? nt1 : nt0;
    // the parts of the Philox rounds shared by all of this row's calls
    PhiloxRow prow;
    if constexpr (DROP) prow = philox_row(uint32_t(qrow), uint32_t(bh), p.offset, p.seed_lo, p.seed_hi);
    float m_run = -INFINITY;
    float l_run = 0.f;
    int exact_left = 0;   // tiles that take the maximum first (warp-uniform)
    bool ok = true;
    // first key tile with masked keys (past Lk, or above the causal diagonal);
    // they are the last tiles of the row, so the hot loop below has no mask code
    const int j_edge = min(p.Lk / 128, p.causal ? qt / 128 : (1 << 30));

    // One key tile: S -> weights P (bf16, TMEM) and the row statistics.  The
    // exponentials are taken against the running maximum m_run; afterwards
    // the tile's row sum is checked: every weight is at most that sum, so a
    // sum up to 2^kRescaleLog2 means the maximum grew by at most the lazy
    // rescale bound and the weights stand.  Otherwise (rare) the row maximum
    // is taken, and where it grew by more, O is rescaled and the same code
    // runs a second pass over the tile.  A row's first tile, and every tile
    // after a second pass, take the maximum before exponentiating.  Keys 0-63 are exponentiated before the
    // wait for P_t(j-1) V (P_t free, O_t stable).
    auto tile = [&](int j, auto masked_tag) -> bool {
      constexpr bool kMasked = decltype(masked_tag)::value;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_s(t), j & 1, abort_flag, p.err, kSiteSoftmaxS))) return false;
      float s[128];
      tc_fence_after();
      tmem_ld128_sync(tS, s);
      tc_fence_before();
      mbar_arrive(bar_sfree(t));  // S is in registers: the other tile's S may overwrite it
      if constexpr (kMasked) {
        const int k0 = j * 128;
        const int lim = min(p.Lk - k0, p.causal ? qrow - k0 + 1 : 128);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) s[i] = -INFINITY;
      }
      float alpha = 1.f;    // O and l are multiplied by alpha (the maximum moved)
      bool resc = false;    // warp-uniform
      // with dropout every tile takes the maximum first: a recomputed tile
      // would draw its random bits twice
      bool take_max = DROP || exact_left > 0 || __any_sync(0xffffffffu, m_run == -INFINITY);
      if (exact_left > 0) --exact_left;
      bool redo = false;
      bool waited = (j == 0);   // P_t(j-1) V has completed: O_t is stable, P_t is free
      float2 acc[4];
      float2 a03;
      const float2 c2 = make_float2(c, c);
      float2 nm2;
      // 16 pairs of weights of keys 32cb .. 32cb+31, packed to bf16, summed into acc
      auto exp_block = [&](int cb, uint32_t (&w)[16]) {
        [[maybe_unused]] uint4 dw, dw2;   // dropout bits of the block's two groups of 16 keys
        [[maybe_unused]] uint32_t keep4;  // keep bits (byte top bits) of the current 4 keys
        if constexpr (DROP) {
          const uint32_t g16 = uint32_t(j * 128 + 32 * cb) >> 4;
          philox4x32_10_row_x2(g16, g16 + 1u, prow, p.keys, dw, dw2);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if constexpr (DROP)
            if (i == 8) dw = dw2;
          const int e = 32 * cb + 2 * i;
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
      for (;;) {
        if (take_max) {
          const float m_cand = fmaxf(m_run, row_max128(s) * c);
          if (__any_sync(0xffffffffu, m_cand > m_run + kRescaleLog2)) {
            alpha = ex2_approx(m_run - ((m_cand == -INFINITY) ? 0.f : m_cand));
            m_run = m_cand;
            resc = true;
          } else if (redo) {
            break;   // the maximum grew by at most the bound: the first pass stands
          }
          if (redo) exact_left = kExactAfterRedo;
        }
        {
          const float m_safe = (m_run == -INFINITY) ? 0.f : m_run;
          nm2 = make_float2(-m_safe, -m_safe);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = make_float2(0.f, 0.f);
        uint32_t pk[2][16];   // P of keys 0-63, computed before P_t(j-1) V has freed P_t
        exp_block(0, pk[0]);
        exp_block(1, pk[1]);
        if (!waited) {
          if (!__all_sync(0xffffffffu, mbar_wait(bar_pv(t), (j - 1) & 1, abort_flag, p.err, kSiteSoftmaxO)))
            return false;
          waited = true;
        }
        tc_fence_after();
        if (resc && j > 0) {
          // 16 columns at a time: the scores and P of keys 0-63 are still live
#pragma unroll 1
          for (int cc = 0; cc < kD; cc += 16) {
            float ov[16];
            tmem_ld16_sync(tO + cc, ov);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(ov[i] * alpha);
            tmem_st16(tO + cc, w);
          }
        }
        tmem_st16(tP, pk[0]);
        tmem_st16(tP + 16, pk[1]);
        // keys 64-127: computed and stored now that P_t is free
#pragma unroll
        for (int cb = 2; cb < 4; ++cb) {
          uint32_t w[16];
          exp_block(cb, w);
          tmem_st16(tP + 16 * cb, w);
        }
        a03 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
        if (take_max) break;
        if (!__any_sync(0xffffffffu, !(a03.x + a03.y <= kRescaleBound))) break;
        take_max = true;
        redo = true;
      }
      l_run = l_run * alpha + (a03.x + a03.y);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p(t));
      return true;
    };
    const int j_hot = min(n, j_edge);
#pragma unroll 1
    for (int j = 0; j < j_hot && ok; ++j) ok = tile(j, std::false_type{});
#pragma unroll 1
    for (int j = j_hot; j < n && ok; ++j) ok = tile(j, std::true_type{});

    // epilogue: wait for the last P_t V, then O / l -> bf16, LSE
    if (ok && n > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bar_o(t), 0, abort_flag, p.err, kSiteSoftmaxO));
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

  // ---- teardown: all TMEM traffic of this CTA is finished
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_prefill_d128(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int Lq, int Lk, float scale, int causal, cudaStream_t stream,
                        int* err, const Dropout& dr) {
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
  p.group = l2_head_group(BH, 2ll * Lk * kD * 2);   // K and V of a head
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
  auto kernel = dr.on ? fa_prefill_d128_kernel<true> : fa_prefill_d128_kernel<false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return -4;
  kernel<<<dim3(unsigned(nblk)), dim3(kThreads), kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace fa
