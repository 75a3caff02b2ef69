// fa_prefill_d64x1_sm103.cu - attention forward for head dimension 64 on
// sm_103a, one 128-row query tile per CTA and two CTAs resident per SM.
//
// The computation is that of fa_prefill_d64_sm103.cu (S = Q K^T and O += P V
// on the tensor cores, the online-softmax recurrence of "NTU Hung-yi Lee ML
// 2026 Guide: Faster Generation, Part 1: Flash Attention" (quidproquo.cc),
// "Expand: why multiplying by exp(d1 - d2) fixes it" and "Expand: the
// correction for the output O", in base 2 with the same lazily applied
// rescale and the same check of the weights against the running maximum),
// for one query tile per CTA instead of two.  Each CTA takes half of the
// SM's TMEM and a little under half of its shared memory, so two CTAs share
// an SM; the hardware then overlaps one CTA's start (barrier set-up, TMEM
// allocation, the first Q and K loads) and end (the O store) with the other
// CTA's steady state, and a grid has twice as many work units of half the
// size: the chip fills at half the sequence length, and the last wave ends
// more evenly.
//
// TMEM (256 columns per CTA): S [0,128)  O [128,192)  P [192,256) (bf16 pairs).
// Shared memory: Q (16 KB), a K ring of 3 slots and a V ring of 2 slots
// (16 KB each): 96 KB + barriers.  A K slot is free once S of its tile has
// been computed, a V slot once P V has.
// Warps: 0 = TMA producer for Q and K (thread 0 issues Q and K(0) right
// after setting up the barriers), 1 = TMEM allocation + MMA issue,
// 2 = TMA producer for V, 3 = idle, 4-7 = softmax + epilogue (one query row
// per thread; TMEM lane quarter = warp % 4).
#include "fa_internal.h"
#include "sm103_ptx.cuh"

#include <cmath>
#include <type_traits>

namespace fa {
namespace {

constexpr int kThreads = 256;
// 128 threads x 48 + 128 threads x 208 = 32768 = 256 x 128 registers at launch
// (two CTAs per SM: 65536 / 512 threads)
constexpr uint32_t kRegsCtl = 48;
constexpr uint32_t kRegsSoftmax = 208;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleBound = 256.0f;        // 2^kRescaleLog2
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kD = 64;
constexpr int kTileBytes = 128 * kD * 2;       // one 128-row tile, one TMA box (16 KB)
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kQOff = 0;
constexpr int kKOff = kTileBytes;
constexpr int kVOff = kKOff + kKStages * kTileBytes;
constexpr int kBarOff = kVOff + kVStages * kTileBytes;
constexpr int kBarQ = 0;
constexpr int kBarKFull = 8;
constexpr int kBarKEmpty = kBarKFull + 8 * kKStages;
constexpr int kBarVFull = kBarKEmpty + 8 * kKStages;
constexpr int kBarVEmpty = kBarVFull + 8 * kVStages;
constexpr int kBarS = kBarVEmpty + 8 * kVStages;   // S(j) written
constexpr int kBarSFree = kBarS + 8;               // the softmax loaded S(j)
constexpr int kBarP = kBarSFree + 8;               // P(j) written (O rescaled)
constexpr int kBarPV = kBarP + 8;                  // PV(j) completed
constexpr int kBarDone = kBarPV + 8;               // all MMAs completed
constexpr int kTmemHolder = kBarDone + 8;
constexpr int kAbort = kTmemHolder + 4;
constexpr int kMiscBytes = 256;
static_assert(kAbort + 4 <= kMiscBytes, "barrier area overflow");
constexpr int kSmemBytes = kBarOff + kMiscBytes + 1024;  // + alignment slack
// two CTAs per SM: 2 x (dynamic + 1 KB reserved per CTA) <= 228 KB
static_assert(2 * (kSmemBytes + 1024) <= 233472, "shared memory budget for two CTAs per SM");
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 128;
constexpr uint32_t kColP = 192;

struct Params {
  __nv_bfloat16* o;
  float* lse;
  int* err;
  int BH, Lq, Lk;
  int n_qblk;  // ceil(Lq / 128)
  int group;   // heads per group of the grid order (K/V of a group stay in L2)
  int causal;
  float scale_log2;
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > 50000000ull) return;  // 50 ms
  }
}

// A full 128-column S row as two 64-column TMEM loads and one wait: no
// single instruction may name more registers than a thread has at launch
// (128 here).
__device__ __forceinline__ void tmem_ld128_2x64_sync(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
      "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%129];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]),
        "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]),
        "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]),
        "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]),
        "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]),
        "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
        "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]),
        "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]),
        "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]),
        "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr), "r"(taddr + 64u)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
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

__global__ void __launch_bounds__(kThreads, 2)
    fa_prefill_d64x1_kernel(const __grid_constant__ CUtensorMap tmQ,
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

  const uint32_t bar_q = sBar + kBarQ;
  auto bar_kfull = [&](int s) { return sBar + kBarKFull + 8 * s; };
  auto bar_kempty = [&](int s) { return sBar + kBarKEmpty + 8 * s; };
  auto bar_vfull = [&](int s) { return sBar + kBarVFull + 8 * s; };
  auto bar_vempty = [&](int s) { return sBar + kBarVEmpty + 8 * s; };
  const uint32_t bar_s = sBar + kBarS;
  const uint32_t bar_sfree = sBar + kBarSFree;
  const uint32_t bar_p = sBar + kBarP;
  const uint32_t bar_pv = sBar + kBarPV;
  const uint32_t bar_done = sBar + kBarDone;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which query tile this CTA owns (heads in groups whose K/V stay in
  // L2; within a group the heaviest query tiles first)
  const TileOrder to = grouped_tile_order(blockIdx.x, p.BH, p.n_qblk, p.group);
  const int qblk = p.n_qblk - 1 - to.rank;
  const int bh = to.bh;
  const int q0 = qblk * 128;
  const int nk_all = (p.Lk + 127) / 128;
  // key tiles of this query tile (>= 1)
  const int n = p.causal ? min(nk_all, min(q0 + 127, p.Lq - 1) / 128 + 1) : nk_all;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar_kfull(s), 1);
      mbar_init(bar_kempty(s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar_vfull(s), 1);
      mbar_init(bar_vempty(s), 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_sfree, 128);
    mbar_init(bar_p, 128);
    mbar_init(bar_pv, 1);
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // thread 0 is the K producer: Q and K(0) start loading before the CTA-wide
    // synchronisation (slot 0 of the K ring is free at the start)
    mbar_arrive_expect_tx(bar_q, kTileBytes);
    tma_load_tile(sQ, &tmQ, bar_q, q0, bh);
    mbar_arrive_expect_tx(bar_kfull(0), kTileBytes);
    tma_load_tile(sK, &tmK, bar_kfull(0), 0, bh);
  }
  if (warp == 2 && lane == 0) tma_prefetch_desc(&tmV);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
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
        const int stages = is_k ? kKStages : kVStages;
        // Q and K(0) were issued by this thread before the CTA-wide sync
        const int j0 = is_k ? 1 : 0;
        int issued = j0;
        for (int j = j0; j < n; ++j) {
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
        if (is_k) drain_wait(bar_q, 0);
        for (int s = 0; s < stages && s < issued; ++s) {
          const int last = s + stages * ((issued - 1 - s) / stages);
          drain_wait(is_k ? bar_kfull(s) : bar_vfull(s), (last / stages) & 1);
        }
      }
    } else if (warp == 1) {
      // =================== MMA issuer ===================
      if (lane == 0) {
        constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t kIdPV = idesc_bf16_f32(128, kD, false, true);
        constexpr uint64_t kDescK = sdesc_sw128(0, 16, 1024);      // Q, K: K-major
        constexpr uint64_t kDescMN = sdesc_sw128(0, 16, 1024);     // V: MN-major, one 64-col block
        bool ok = true;
        auto wait = [&](uint32_t b, uint32_t ph, int site) {
          if (ok && !mbar_wait(b, ph, abort_flag, p.err, site)) ok = false;
          return ok;
        };
        wait(bar_q, 0, kSiteMmaQ);
        for (int j = 0; j <= n && ok; ++j) {
          // S(j) once K(j) has landed and the softmax holds S(j-1) in registers
          if (j < n) {
            const int sk = j % kKStages;
            if (!wait(bar_kfull(sk), (j / kKStages) & 1, kSiteMmaK)) break;
            if (j > 0 && !wait(bar_sfree, (j - 1) & 1, kSiteMmaS)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              umma_ss(tmem, sdesc_at(kDescK, sQ + kk * 32), sdesc_at(kDescK, sK + sk * kTileBytes + kk * 32),
                      kIdQK, kk > 0 ? 1u : 0u);
            umma_commit(bar_s);
            umma_commit(bar_kempty(sk));   // K slot free once S(j) is computed
          }
          // PV(j-1) once V(j-1) has landed and P(j-1) is written
          if (j > 0) {
            const int sv = (j - 1) % kVStages;
            if (!wait(bar_vfull(sv), ((j - 1) / kVStages) & 1, kSiteMmaV)) break;
            if (!wait(bar_p, (j - 1) & 1, kSiteMmaP)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_ts(tmem + kColO, tmem + kColP + kk * 8, sdesc_at(kDescMN, sV + sv * kTileBytes + kk * 16 * 128),
                      kIdPV, (j - 1 > 0 || kk > 0) ? 1u : 0u);
            umma_commit(bar_pv);
            umma_commit(bar_vempty(sv));   // V slot free once PV(j-1) is computed
          }
        }
        umma_commit(bar_done);
        drain_wait(bar_done, 0);
      }
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // =================== softmax + epilogue (one query row per thread) ===================
    const int g = warp & 3;
    const int r = g * 32 + lane;
    const int qrow = q0 + r;
    const uint32_t lane_off = uint32_t(g * 32) << 16;
    const uint32_t tS = tmem + lane_off;
    const uint32_t tP = tmem + lane_off + kColP;
    const uint32_t tO = tmem + lane_off + kColO;
    const float c = p.scale_log2;
    float m_run = -INFINITY;
    float l_run = 0.f;
    // after a tile had to be recomputed, the warp's remaining tiles take the
    // maximum first (sharp logits keep moving the maximum of some row past
    // the bound, and a recomputed tile costs a second pass of exponentials)
    bool exact_rest = false;
    bool ok = true;
    // first key tile with masked keys (past Lk, or above the causal diagonal);
    // they are the last tiles of the row, so the hot loop below has no mask code
    const int j_edge = min(p.Lk / 128, p.causal ? q0 / 128 : (1 << 30));

    // One key tile: S -> weights P (bf16, TMEM) and the row statistics.  The
    // exponentials are taken against the running maximum m_run; afterwards
    // the tile's row sum is checked: every weight is at most that sum, so a
    // sum up to 2^kRescaleLog2 means the maximum grew by at most the lazy
    // rescale bound and the weights stand.  Otherwise (rare) the row maximum
    // is taken, and where it grew by more, O is rescaled and the same code
    // runs a second pass over the tile.  A row's first tile, and every tile
    // after a second pass, take the maximum before exponentiating.
    auto tile = [&](int j, auto masked_tag) -> bool {
      constexpr bool kMasked = decltype(masked_tag)::value;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_s, j & 1, abort_flag, p.err, kSiteSoftmaxS))) return false;
      float s[128];
      tc_fence_after();
      tmem_ld128_2x64_sync(tS, s);
      tc_fence_before();
      mbar_arrive(bar_sfree);  // S(j) is in registers: S may be overwritten
      if constexpr (kMasked) {
        const int k0 = j * 128;
        const int lim = min(p.Lk - k0, p.causal ? qrow - k0 + 1 : 128);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) s[i] = -INFINITY;
      }
      float alpha = 1.f;    // O and l are multiplied by alpha (the maximum moved)
      bool resc = false;    // warp-uniform
      bool take_max = exact_rest || __any_sync(0xffffffffu, m_run == -INFINITY);
      bool redo = false;
      bool waited = (j == 0);   // PV(j-1) has completed: O is stable, P is free
      float2 acc[4];
      float2 a03;
      const float2 c2 = make_float2(c, c);
      float2 nm2;
      // 16 pairs of weights of keys 32cb .. 32cb+31, packed to bf16, summed into acc
      auto exp_block = [&](int cb, uint32_t (&w)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = 32 * cb + 2 * i;
          const float2 x = __ffma2_rn(make_float2(s[e], s[e + 1]), c2, nm2);
          const float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          acc[i & 3] = __fadd2_rn(acc[i & 3], pr);
          w[i] = pack_bf16x2(pr.x, pr.y);
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
          if (redo) exact_rest = true;
        }
        {
          const float m_safe = (m_run == -INFINITY) ? 0.f : m_run;
          nm2 = make_float2(-m_safe, -m_safe);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = make_float2(0.f, 0.f);
        uint32_t pk[32];   // P of keys 0-63, computed before PV(j-1) has freed P
        exp_block(0, *reinterpret_cast<uint32_t(*)[16]>(pk));
        exp_block(1, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
        if (!waited) {
          if (!__all_sync(0xffffffffu, mbar_wait(bar_pv, (j - 1) & 1, abort_flag, p.err, kSiteSoftmaxO)))
            return false;
          waited = true;
        }
        tc_fence_after();
        if (resc && j > 0) {
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
        // each half of P in one 32-column store (fewer TMEM accesses beside the products)
        tmem_st32(tP, pk);
        // keys 64-127: computed and stored now that P is free
        {
          uint32_t w[32];
          exp_block(2, *reinterpret_cast<uint32_t(*)[16]>(w));
          exp_block(3, *reinterpret_cast<uint32_t(*)[16]>(w + 16));
          tmem_st32(tP + 32, w);
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
      mbar_arrive(bar_p);
      return true;
    };
    // (the loop body unrolled by two measured 2-3 % slower, with more stalls
    // on instruction fetch)
    const int j_hot = min(n, j_edge);
#pragma unroll 1
    for (int j = 0; j < j_hot && ok; ++j) ok = tile(j, std::false_type{});
#pragma unroll 1
    for (int j = j_hot; j < n && ok; ++j) ok = tile(j, std::true_type{});

    // epilogue: wait for the last PV, then O / l -> bf16, LSE
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(bar_pv, (n - 1) & 1, abort_flag, p.err, kSiteSoftmaxO));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
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
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int launch_prefill_d64x1(const void* q, const void* k, const void* v, void* o, float* lse, int B,
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
  p.n_qblk = (Lq + 127) / 128;
  p.group = l2_head_group(BH, 2ll * Lk * 64 * 2);   // K and V of a head
  p.causal = causal;
  p.scale_log2 = scale * 1.44269504088896340736f;
  const long long nblk = (long long)p.n_qblk * BH;
  if (nblk > 0x7fffffffLL) return -2;
  if (dr.on) return -2;   // the dropout forward runs on fa_prefill_d64_sm103.cu
  auto kernel = fa_prefill_d64x1_kernel;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return -4;
  kernel<<<dim3(unsigned(nblk)), dim3(kThreads), kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace fa
