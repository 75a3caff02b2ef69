// fa_backward_sm103.cu - attention backward pass (dQ, dK, dV) on sm_103a.
//
// "6.3 FlashAttention" (comfyai.app), "A simple implementation w/ C++" and
// "Computation and GPU Memory": for training, the forward pass keeps no
// attention weights; the backward pass recomputes them.  Given q, k, v, the
// forward's output O and log-sum-exp (natural log) per query row, and the
// output gradient dO, the gradients of <dO, O> are
//     P  = exp(scale q k^T - LSE)           (the weights, recomputed)
//     dV = P^T dO,   dP = dO V^T,   Dr = rowsum(dO * O) = rowsum(P * dP)
//     dS = P * (dP - Dr),   dQ = scale dS K,   dK = scale dS^T Q.
// Three kernels:
//   fa_bwd_prep_kernel   Dr per query row, and LSE in base 2, into a workspace
//                        padded to whole 128-row tiles (rows past Lq: Dr = 0,
//                        LSE = +inf, so their weights are 0);
//   fa_bwd_dkdv_kernel   one CTA per 128-key tile: walks the query tiles,
//                        S^T = K Q^T and dP^T = V dO^T on the tensor cores into
//                        TMEM, P^T and dS^T (bf16) written back over them by
//                        the element-wise warps (one key row per thread), then
//                        dV += P^T dO and dK += dS^T Q accumulate in TMEM;
//   fa_bwd_dq_kernel     one CTA per 128-query tile: walks the key tiles,
//                        S = Q K^T and dP = dO V^T, dS (bf16) over dP, then
//                        dQ += dS K in TMEM.
// S and dP are computed twice (once per kernel): no atomics, deterministic
// results.
// With dropout (the DROP instantiations, the backward of the forward with
// dropout on the weights): with z the keep mask of philox.cuh's contract and
// s = 256 / (256 - t), dV = s (P z)^T dO, the weights' gradient is
// s z dP, and dS = P (s z dP - Dr) (Dr = rowsum(dO * O) with the dropout
// O); no mask is stored: each kernel draws the bits again.  The dQ kernel's
// threads own query rows and use the row form of the generator, as the
// forward does; the dK/dV kernel's threads own keys, so the 16 lanes of a
// 16-key block draw the block's words for 4 query rows each (the column
// form) and hand each lane its key's bytes through a per-warp shared-memory
// transpose.  s multiplies dV once, in the epilogue.  TMEM (512 columns): dK/dV kernel S^T [0,128) dP^T [128,256)
// dV [256,256+D) dK [256+D,256+2D); dQ kernel S [0,128) dP [128,256)
// dQ [256,256+D).
// The element-wise work runs in two phases per tile, each hidden behind two
// products of the tensor core: P from S while dP is computed, dS from dP while
// the first gradient product runs.  Issue order of the MMA thread:
//   dK/dV:  S dP | dV S' dK dP' | dV' S'' dK' dP'' | ...
//   dQ:     S dP | S' dQ dP' | S'' dQ' dP'' | ...
// (' = the next tile; dV waits for P, dK and dQ for dS, the dQ kernel's S'
// for the element-wise warps to have read S).  The next tile's S (dP) is
// issued after the product that reads the bf16 data packed over S (dP):
// tcgen05.mma operations from one thread execute in order.  Each row's 128
// columns are split between two warps: warps 2-5 take columns 0-63 and warps
// 6-9 columns 64-127 (TMEM lane quarter = warp % 4), so each SM sub-partition
// runs two element-wise warps; half h's bf16 results are packed into columns
// [64h, 64h+32) of the S and dP regions, inside the columns it consumed.
// Warp 0 = TMA producer of the fixed tiles' first and ring A (Q tiles with
// their LSE2 / Dr slices in dK/dV, K tiles in dQ), warp 10 = TMA producer of
// the fixed tiles' second and ring B (dO or V tiles): two issuing threads
// double the TMA rate.  Warp 1 = TMEM allocation + MMA issue.
// Every wait is bounded (the same routine as the forward kernels).
#include "fa_internal.h"
#include "philox.cuh"
#include "sm103_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

constexpr int kThreads = 352;   // 11 warps
constexpr float kLog2e = 1.44269504088896340736f;

constexpr int kSubBytes = 128 * 128;   // one 64-column block of a 128-row tile

template <int D, bool DQ, bool DROP = false>
struct BwCfg {
  static constexpr int kTileBytes = 128 * D * 2;        // one 128-row tile (one TMA box)
  // ring A: Q tiles (dK/dV kernel) or K tiles (dQ kernel); ring B: dO or V tiles
  static constexpr int kStagesA = D == 64 ? 4 : (DQ ? 3 : 2);
  static constexpr int kStagesB = D == 64 ? 4 : 2;
  static constexpr int kFixedOff = 0;                   // the CTA's own two tiles
  static constexpr int kRingAOff = 2 * kTileBytes;
  static constexpr int kRingBOff = kRingAOff + kStagesA * kTileBytes;
  static constexpr int kVecOff = kRingBOff + kStagesB * kTileBytes;  // dK/dV: per A stage 128 LSE2 + 128 Dr
  static constexpr int kBarOff = kVecOff + (DQ ? 0 : kStagesA * 1024);
  // dK/dV with dropout: per element-wise warp, the Philox words of its two
  // 16-key groups for 64 query rows, [group][word][row], rows padded to 68
  // words so that the eight rows a warp reads at once fall on different banks
  static constexpr int kTransRow = 68;
  static constexpr int kTransWarpBytes = 2 * 4 * kTransRow * 4;
  static constexpr int kTransOff = kBarOff + 256;
  static constexpr int kSmemBytes = kTransOff + (DROP && !DQ ? 8 * kTransWarpBytes : 0) + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct BwParams {
  __nv_bfloat16* out_a;   // dK (dkdv kernel) or dQ (dq kernel)
  __nv_bfloat16* out_b;   // dV (dkdv kernel)
  const float* lse2;      // [BH][Lq_pad]: LSE * log2(e), +inf past Lq
  const float* drow;      // [BH][Lq_pad]: rowsum(dO * O), 0 past Lq
  int* err;
  int BH, Lq, Lk, Lq_pad;
  int group;              // heads per group of the grid order
  int causal;
  float scale, scale_log2;
  // dropout (the DROP instantiations): philox.cuh's contract, as in the
  // forward; keep_scale = 256 / (256 - t)
  uint32_t seed_lo, seed_hi, offset, drop_tl4, drop_hsel;
  PhiloxKeys keys;
  float keep_scale;
};

// 1-D bulk copy global -> shared, completing `bytes` on `bar` (16-byte aligned, multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > 50000000ull) return;  // 50 ms
  }
}

// before exit: wait (bounded) for the last copies into each used stage of a ring
__device__ __forceinline__ void drain_ring(uint32_t full0, int stages, int issued) {
  for (int s = 0; s < stages && s < issued; ++s) {
    const int last = s + stages * ((issued - 1 - s) / stages);
    drain(full0 + 8 * s, (last / stages) & 1);
  }
}

// ---------------------------------------------------------------- preparation

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __nv_bfloat16* o,
                                                          const __nv_bfloat16* dout,
                                                          const float* lse, float* lse2,
                                                          float* drow, int BH, int Lq,
                                                          int Lq_pad) {
  // D/8 lanes per row, 16 bytes of O and dO per lane
  constexpr int G = D / 8;
  const long long n = (long long)BH * Lq_pad;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gid / G;
  const int li = int(gid % G);
  const bool in = row < n;   // every lane stays for the shuffles below
  const int bh = in ? int(row / Lq_pad) : 0;
  const int r = in ? int(row % Lq_pad) : Lq;
  float acc = 0.f;
  if (r < Lq) {
    const size_t base = (size_t(bh) * Lq + r) * D + 8 * li;
    const uint4 a = *reinterpret_cast<const uint4*>(o + base);
    const uint4 b = *reinterpret_cast<const uint4*>(dout + base);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(wa[e] << 16), __uint_as_float(wb[e] << 16), acc);
      acc = fmaf(__uint_as_float(wa[e] & 0xffff0000u), __uint_as_float(wb[e] & 0xffff0000u), acc);
    }
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (in && li == 0) {
    drow[row] = acc;
    lse2[row] = r < Lq ? lse[size_t(bh) * Lq + r] * kLog2e : INFINITY;
  }
}

// ---------------------------------------------------------------- shared pieces

// operand descriptors: a [128 x D] tile as the K-major operand of a product
// over D, or as the MN-major operand (K = its 128 rows, N = D) of a product
// over its rows
template <int D>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
  constexpr uint64_t kDesc = sdesc_sw128(0, 16, 1024);
  return sdesc_at(kDesc, tile + (kk >> 2) * kSubBytes + (kk & 3) * 32);
}
template <int D>
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk) {
  constexpr uint64_t kDesc = sdesc_sw128(0, kSubBytes, 1024);
  return sdesc_at(kDesc, tile + kk * 16 * 128);
}

// TMEM column of the bf16 operand for K-step kk (16 rows of the K dimension) of
// a gradient product: half kk/4's data sits at [64 (kk/4), 64 (kk/4) + 32)
__device__ __forceinline__ uint32_t packed_col(int kk) { return uint32_t(64 * (kk >> 2) + 8 * (kk & 3)); }

// phase 1 of the element-wise step on half h of one 128-wide TMEM row: the
// 64 scores of columns 64h .. 64h+63 (loaded from S into pv) become the
// weights p = 2^(c s - lse2).  `l2(i)` gives column 64h+i's log2-domain LSE;
// with MASK, `valid(i)` gives its mask and a masked column's exponent argument
// becomes -inf (a select, not a branch around the exponential).
template <bool MASK, class L2, class Valid>
__device__ __forceinline__ void weights_p(float (&pv)[64], float c, L2 l2, Valid valid) {
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const float x = fmaf(pv[i], c, -l2(i));
    pv[i] = ex2_approx(!MASK || valid(i) ? x : -INFINITY);
  }
}

// bf16 pairs of 64 values into 32 TMEM columns at taddr
__device__ __forceinline__ void store_packed64(uint32_t taddr, const float (&v)[64]) {
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  tmem_st32(taddr, w);
}

// phase 2: dS = p (dP - Dr) for the same 64 columns, dP read from tdP, packed
// to bf16 into [64h, 64h+32) of the dP region.  `dr(i)` gives column
// 64h+i's Dr (the dK/dV kernel) or the row's (the dQ kernel).
template <class Dr>
__device__ __forceinline__ void weights_ds(uint32_t tdP, int h, const float (&pv)[64], Dr dr) {
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    float dp[32];
    tmem_ld32_sync(tdP + 64 * h + 32 * ch, dp);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = 32 * ch + 2 * i;
      w[i] = pack_bf16x2(pv[e] * (dp[2 * i] - dr(e)), pv[e + 1] * (dp[2 * i + 1] - dr(e + 1)));
    }
    tmem_st16(tdP + 64 * h + 16 * ch, w);
  }
}

// With dropout, the weights dV's product takes: p z (the rescale s is
// applied to dV once, in the epilogue), bf16 pairs into 32 TMEM columns.
// kw: the 16 keep words of the 64 values (dropout_keep_msb's form).
__device__ __forceinline__ void store_packed64_drop(uint32_t taddr, const float (&v)[64], const uint32_t (&kw)[16]) {
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]) & dropout_pair_mask(kw[i >> 1], i & 1);
  tmem_st32(taddr, w);
}

// dS of one value with dropout: p (s dP - Dr) if kept, else -p Dr, where dP is
// the gradient of the dropped weight (the product dO V^T gives it).  Written
// as -p sel(m, Dr - s dP, Dr) with m the key's 32-bit keep mask.
__device__ __forceinline__ float ds_drop(float p, float dp, float dr, uint32_t m, float s) {
  const float a = fmaf(-dp, s, dr);
  return -p * __uint_as_float((__float_as_uint(a) & m) | (__float_as_uint(dr) & ~m));
}

// phase 2 with dropout: weights_ds with ds_drop per value
template <class Dr>
__device__ __forceinline__ void weights_ds_drop(uint32_t tdP, int h, const float (&pv)[64], Dr dr,
                                                const uint32_t (&kw)[16], float s) {
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    float dp[32];
    tmem_ld32_sync(tdP + 64 * h + 32 * ch, dp);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = 32 * ch + 2 * i;
      const uint32_t kq = kw[e >> 2];
      w[i] = pack_bf16x2(ds_drop(pv[e], dp[2 * i], dr(e), dropout_byte_mask(kq, e & 3), s),
                         ds_drop(pv[e + 1], dp[2 * i + 1], dr(e + 1), dropout_byte_mask(kq, (e + 1) & 3), s));
    }
    tmem_st16(tdP + 64 * h + 16 * ch, w);
  }
}

// signal an mbarrier with one arrival per warp once the warp's TMEM stores
// have completed
__device__ __forceinline__ void warp_arrive_after_st(uint32_t bar, int lane) {
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// bf16 store of 32 fp32 values times `mul` to 16-byte aligned global memory
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float (&v)[32], float mul) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q8 = 0; q8 < 4; ++q8)
    d4[q8] = make_uint4(pack_bf16x2(v[8 * q8] * mul, v[8 * q8 + 1] * mul),
                        pack_bf16x2(v[8 * q8 + 2] * mul, v[8 * q8 + 3] * mul),
                        pack_bf16x2(v[8 * q8 + 4] * mul, v[8 * q8 + 5] * mul),
                        pack_bf16x2(v[8 * q8 + 6] * mul, v[8 * q8 + 7] * mul));
}

// ---------------------------------------------------------------- dK, dV

template <int D, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwParams p) {
  using C = BwCfg<D, false, DROP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sK = base + C::kFixedOff, sV = sK + C::kTileBytes;
  auto st_q = [&](int s) { return base + C::kRingAOff + s * C::kTileBytes; };
  auto st_do = [&](int s) { return base + C::kRingBOff + s * C::kTileBytes; };
  auto st_vec = [&](int s) { return base + C::kVecOff + s * 1024; };
  const uint32_t sBar = base + C::kBarOff;
  auto full_a = [&](int s) { return sBar + 8 * s; };
  auto full_b = [&](int s) { return sBar + 32 + 8 * s; };
  auto empty_a = [&](int s) { return sBar + 64 + 8 * s; };
  auto empty_b = [&](int s) { return sBar + 96 + 8 * s; };
  const uint32_t bar_kv = sBar + 128, bar_S = sBar + 136, bar_dP = sBar + 144, bar_P = sBar + 152,
                 bar_dS = sBar + 160, bar_done = sBar + 168;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + C::kBarOff + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBarOff + 196);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TileOrder to = grouped_tile_order(blockIdx.x, p.BH, (p.Lk + 127) / 128, p.group);
  const int jt = to.rank;      // key tile (the most query tiles first when causal)
  const int bh = to.bh;
  const int nq_all = (p.Lq + 127) / 128;
  const int i0 = p.causal ? jt : 0;           // causal: queries q >= key, so query tiles >= jt
  const int n = nq_all - i0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(full_a(s), 1);
      mbar_init(full_b(s), 1);
      mbar_init(empty_a(s), 1);
      mbar_init(empty_b(s), 1);
    }
    mbar_init(bar_kv, 2);   // one arrival (with its bytes) from each producer
    mbar_init(bar_S, 1);
    mbar_init(bar_dP, 1);
    mbar_init(bar_P, 8);    // one arrival per element-wise warp
    mbar_init(bar_dS, 8);
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0 || warp == 10) {
    if (lane == 0) {
      const bool ra = warp == 0;
      const int stages = ra ? C::kStagesA : C::kStagesB;
      mbar_arrive_expect_tx(bar_kv, C::kTileBytes);
      tma_load_tile(ra ? sK : sV, ra ? &tmK : &tmV, bar_kv, jt * 128, bh);
      int issued = 0;
      for (int it = 0; it < n; ++it) {
        const int s = it % stages, use = it / stages;
        if (!mbar_wait(ra ? empty_a(s) : empty_b(s), (use & 1) ^ 1, abort_flag, p.err, kSiteProducerEmpty))
          break;
        if (ra) {
          mbar_arrive_expect_tx(full_a(s), C::kTileBytes + 1024);
          tma_load_tile(st_q(s), &tmQ, full_a(s), (i0 + it) * 128, bh);
          const size_t voff = size_t(bh) * p.Lq_pad + size_t(i0 + it) * 128;
          bulk_load(st_vec(s), p.lse2 + voff, 512, full_a(s));
          bulk_load(st_vec(s) + 512, p.drow + voff, 512, full_a(s));
        } else {
          mbar_arrive_expect_tx(full_b(s), C::kTileBytes);
          tma_load_tile(st_do(s), &tmDO, full_b(s), (i0 + it) * 128, bh);
        }
        ++issued;
      }
      drain(bar_kv, 0);
      drain_ring(ra ? full_a(0) : full_b(0), stages, issued);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdSS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdTS = idesc_bf16_f32(128, D, false, true);
      // S^T = K Q^T, dP^T = V dO^T (M = 128 keys, N = 128 queries, K = D)
      auto issue_s = [&](int sa) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem, desc_kmajor<D>(sK, kk), desc_kmajor<D>(st_q(sa), kk), kIdSS, kk > 0 ? 1u : 0u);
        umma_commit(bar_S);
      };
      auto issue_dp = [&](int sb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + 128, desc_kmajor<D>(sV, kk), desc_kmajor<D>(st_do(sb), kk), kIdSS, kk > 0 ? 1u : 0u);
        umma_commit(bar_dP);
      };
      bool ok = mbar_wait(bar_kv, 0, abort_flag, p.err, kSiteMmaK) &&
                mbar_wait(full_a(0), 0, abort_flag, p.err, kSiteMmaQ) &&
                mbar_wait(full_b(0), 0, abort_flag, p.err, kSiteMmaQ);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int it = 0; it < n && ok; ++it) {
        const int sa = it % C::kStagesA, sb = it % C::kStagesB;
        const int sa2 = (it + 1) % C::kStagesA, sb2 = (it + 1) % C::kStagesB;
        const bool more = it + 1 < n;
        // the next dO stage (released a phase earlier than Q's), while the
        // element-wise warps still work on P
        if (more && !(ok = mbar_wait(full_b(sb2), ((it + 1) / C::kStagesB) & 1, abort_flag, p.err, kSiteMmaQ)))
          break;
        if (!(ok = mbar_wait(bar_P, it & 1, abort_flag, p.err, kSiteMmaP))) break;
        tc_fence_after();
        // dV += P^T dO (M = 128 keys, N = D, K = 128 queries); the last use of dO
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + 256, tmem + packed_col(kk), desc_mnmajor<D>(st_do(sb), kk), kIdTS,
                  (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit(empty_b(sb));
        if (more) {
          if (!(ok = mbar_wait(full_a(sa2), ((it + 1) / C::kStagesA) & 1, abort_flag, p.err, kSiteMmaQ))) break;
          tc_fence_after();
          issue_s(sa2);
        }
        if (!(ok = mbar_wait(bar_dS, it & 1, abort_flag, p.err, kSiteMmaP))) break;
        tc_fence_after();
        // dK += dS^T Q (M = 128 keys, N = D, K = 128 queries); the last use of Q
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + 256 + D, tmem + 128 + packed_col(kk), desc_mnmajor<D>(st_q(sa), kk), kIdTS,
                  (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit(empty_a(sa));
        if (more) issue_dp(sb2);
      }
      umma_commit(bar_done);
      drain(bar_done, 0);
    }
  } else {
    // element-wise: one key row per thread, queries 64h .. 64h+63 of each tile
    const int g = warp & 3, h = (warp - 2) >> 2;
    const int r = g * 32 + lane;
    const int key = jt * 128 + r;
    const uint32_t lane_off = uint32_t(g * 32) << 16;
    const uint32_t tS = tmem + lane_off, tdP = tmem + lane_off + 128;
    const bool key_ok = key < p.Lk;
    // dropout: this lane's 16-key group (counter word 0) and its transpose
    // buffer; the lanes of a group draw the group's words for 4 query rows
    // each, then each lane reads its key's byte for all 64 rows of the half
    PhiloxCol pcol;
    uint32_t* tb = nullptr;
    if constexpr (DROP) {
      pcol = philox_col(uint32_t(jt * 8 + g * 2 + (lane >> 4)), uint32_t(bh), p.offset, p.seed_lo, p.seed_hi);
      tb = reinterpret_cast<uint32_t*>(gbase + C::kTransOff + (warp - 2) * C::kTransWarpBytes);
    }
    bool ok = true;
    for (int it = 0; it < n && ok; ++it) {
      const int q0 = (i0 + it) * 128 + 64 * h;
      const bool diag = p.causal && (i0 + it) == jt;
      uint32_t kw[16];   // dropout: keep bits of this key for the half's 64 query rows
      if constexpr (DROP) {
        __syncwarp();    // the previous tile's reads of the buffer are done
        uint32_t* grp = tb + (lane >> 4) * 4 * C::kTransRow;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int e = (lane & 15) + 16 * t;
          const uint4 wv = philox4x32_10_col(uint32_t(q0 + e), pcol, p.keys);
          grp[e] = wv.x;
          grp[C::kTransRow + e] = wv.y;
          grp[2 * C::kTransRow + e] = wv.z;
          grp[3 * C::kTransRow + e] = wv.w;
        }
        __syncwarp();
        // this key's word (j div 4) mod 4 of every row, byte j mod 4 of each
        const uint4* row = reinterpret_cast<const uint4*>(grp + ((lane & 15) >> 2) * C::kTransRow);
        const uint32_t sel = uint32_t(lane & 3) | (uint32_t((lane & 3) + 4) << 4);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const uint4 w4 = row[m];
          const uint32_t lo = __byte_perm(w4.x, w4.y, sel), hi = __byte_perm(w4.z, w4.w, sel);
          kw[m] = dropout_keep_msb(__byte_perm(lo, hi, 0x5410u), p.drop_tl4, p.drop_hsel);
        }
      }
      // the stage's LSE2 / Dr slices landed with its Q, dO tiles: wait on that
      // barrier too (already complete; it cannot move on before this tile's
      // products are done) so that the copied values are visible here
      ok = __all_sync(0xffffffffu, mbar_wait(bar_S, it & 1, abort_flag, p.err, kSiteSoftmaxS) &&
                                       mbar_wait(full_a(it % C::kStagesA), (it / C::kStagesA) & 1,
                                                 abort_flag, p.err, kSiteSoftmaxS));
      if (!ok) break;
      tc_fence_after();
      const float* vl2 = reinterpret_cast<const float*>(gbase + (st_vec(it % C::kStagesA) - base)) + 64 * h;
      const float* vdr = vl2 + 128;
      float pv[64];
      // masked entries: keys past Lk (last key tile) and the causal diagonal
      // tile; query rows past Lq carry LSE2 = +inf and come out 0 either way
      auto l2 = [&](int i) { return vl2[i]; };
      auto valid = [&](int i) { return key_ok && (!diag || key <= q0 + i); };
      tmem_ld64_sync(tS + 64 * h, pv);
      if (__all_sync(0xffffffffu, key_ok && !diag))
        weights_p<false>(pv, p.scale_log2, l2, valid);
      else
        weights_p<true>(pv, p.scale_log2, l2, valid);
      // dV's operand: the weights as the forward applied them (dropped; the
      // rescale comes in the epilogue)
      if constexpr (DROP)
        store_packed64_drop(tS + 64 * h, pv, kw);
      else
        store_packed64(tS + 64 * h, pv);
      warp_arrive_after_st(bar_P, lane);
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dP, it & 1, abort_flag, p.err, kSiteSoftmaxS));
      if (!ok) break;
      tc_fence_after();
      if constexpr (DROP)
        weights_ds_drop(tdP, h, pv, [&](int i) { return vdr[i]; }, kw, p.keep_scale);
      else
        weights_ds(tdP, h, pv, [&](int i) { return vdr[i]; });
      warp_arrive_after_st(bar_dS, lane);
    }
    // epilogue: group 0 writes the dV row of this key (times the dropout
    // rescale s with dropout), group 1 scale * dK.
    // The TMEM loads are warp-collective: every lane takes part, only the
    // stores are predicated.
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_done, 0, abort_flag, p.err, kSiteSoftmaxO));
    if (ok) {
      tc_fence_after();
      const bool valid = key < p.Lk;
      const size_t orow = (size_t(bh) * p.Lk + (valid ? key : 0)) * D;
      __nv_bfloat16* dst = (h == 0 ? p.out_b : p.out_a) + orow;
      const float mul = h == 0 ? (DROP ? p.keep_scale : 1.f) : p.scale;
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 32) {
        float v[32];
        tmem_ld32_sync(tmem + lane_off + 256 + h * D + cc, v);
        if (valid) store_row32(dst + cc, v, mul);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- dQ

template <int D, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                     const BwParams p) {
  using C = BwCfg<D, true, DROP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + C::kFixedOff, sDO = sQ + C::kTileBytes;
  auto st_k = [&](int s) { return base + C::kRingAOff + s * C::kTileBytes; };
  auto st_v = [&](int s) { return base + C::kRingBOff + s * C::kTileBytes; };
  const uint32_t sBar = base + C::kBarOff;
  // ready(j): K_j and V_j have landed and the element-wise warps have read
  // S_(j-1) out of TMEM, so S_j may be computed (four slots by j mod 4)
  auto ready = [&](int j) { return sBar + 8 * (j & 3); };
  auto empty_a = [&](int s) { return sBar + 64 + 8 * s; };
  auto empty_b = [&](int s) { return sBar + 96 + 8 * s; };
  const uint32_t bar_q = sBar + 128, bar_S = sBar + 136, bar_dP = sBar + 144, bar_dS = sBar + 160,
                 bar_done = sBar + 168;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + C::kBarOff + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBarOff + 196);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq_all = (p.Lq + 127) / 128;
  const TileOrder to = grouped_tile_order(blockIdx.x, p.BH, nq_all, p.group);
  const int itile = nq_all - 1 - to.rank;  // the most key tiles first when causal
  const int bh = to.bh;
  const int nk_all = (p.Lk + 127) / 128;
  const int n = p.causal ? min(nk_all, itile + 1) : nk_all;   // causal: keys <= query

  if (threadIdx.x == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(ready(s), 2 + 8);   // each producer (with its bytes) + each element-wise warp
      mbar_init(empty_a(s), 1);
      mbar_init(empty_b(s), 1);
    }
    mbar_init(bar_q, 2);       // one arrival (with its bytes) from each producer
    mbar_init(bar_S, 1);
    mbar_init(bar_dP, 1);
    mbar_init(bar_dS, 8);
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0 || warp == 10) {
    if (lane == 0) {
      const bool ra = warp == 0;
      const int stages = ra ? C::kStagesA : C::kStagesB;
      mbar_arrive_expect_tx(bar_q, C::kTileBytes);
      tma_load_tile(ra ? sQ : sDO, ra ? &tmQ : &tmDO, bar_q, itile * 128, bh);
      int issued = 0;
      // no party runs four tiles ahead of the issuer's waits on ready(), so a
      // slot's previous phase has completed before anyone arrives on it again
      for (int it = 0; it < n; ++it) {
        const int s = it % stages, use = it / stages;
        if (!mbar_wait(ra ? empty_a(s) : empty_b(s), (use & 1) ^ 1, abort_flag, p.err, kSiteProducerEmpty))
          break;
        mbar_arrive_expect_tx(ready(it), C::kTileBytes);
        tma_load_tile(ra ? st_k(s) : st_v(s), ra ? &tmK : &tmV, ready(it), it * 128, bh);
        ++issued;
      }
      drain(bar_q, 0);
      for (int j = max(0, issued - 4); j < issued; ++j) drain(ready(j), (j >> 2) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdSS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdTS = idesc_bf16_f32(128, D, false, true);
      // S = Q K^T, dP = dO V^T (M = 128 queries, N = 128 keys, K = D)
      auto issue_s = [&](int sa) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem, desc_kmajor<D>(sQ, kk), desc_kmajor<D>(st_k(sa), kk), kIdSS, kk > 0 ? 1u : 0u);
        umma_commit(bar_S);
      };
      // dP's commit also releases its V stage (V has no other use)
      auto issue_dp = [&](int sb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + 128, desc_kmajor<D>(sDO, kk), desc_kmajor<D>(st_v(sb), kk), kIdSS, kk > 0 ? 1u : 0u);
        umma_commit(bar_dP);
        umma_commit(empty_b(sb));
      };
      bool ok = mbar_wait(bar_q, 0, abort_flag, p.err, kSiteMmaQ) &&
                mbar_wait(ready(0), 0, abort_flag, p.err, kSiteMmaK);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int it = 0; it < n && ok; ++it) {
        const int sa = it % C::kStagesA;
        const int sa2 = (it + 1) % C::kStagesA, sb2 = (it + 1) % C::kStagesB;
        const bool more = it + 1 < n;
        if (more) {
          if (!(ok = mbar_wait(ready(it + 1), ((it + 1) >> 2) & 1, abort_flag, p.err, kSiteMmaK))) break;
          tc_fence_after();
          issue_s(sa2);
        }
        if (!(ok = mbar_wait(bar_dS, it & 1, abort_flag, p.err, kSiteMmaP))) break;
        tc_fence_after();
        // dQ += dS K (M = 128 queries, N = D, K = 128 keys); dS sits in dP's
        // columns; the last use of K
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + 256, tmem + 128 + packed_col(kk), desc_mnmajor<D>(st_k(sa), kk), kIdTS,
                  (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit(empty_a(sa));
        if (more) issue_dp(sb2);
      }
      umma_commit(bar_done);
      drain(bar_done, 0);
    }
  } else {
    // element-wise: one query row per thread, keys 64h .. 64h+63 of each tile
    const int g = warp & 3, h = (warp - 2) >> 2;
    const int r = g * 32 + lane;
    const int qrow = itile * 128 + r;
    const uint32_t lane_off = uint32_t(g * 32) << 16;
    const uint32_t tS = tmem + lane_off, tdP = tmem + lane_off + 128;
    const float l2 = p.lse2[size_t(bh) * p.Lq_pad + qrow];
    const float dr = p.drow[size_t(bh) * p.Lq_pad + qrow];
    // dropout: the parts of the Philox rounds shared by this row's calls
    PhiloxRow prow;
    if constexpr (DROP) prow = philox_row(uint32_t(qrow), uint32_t(bh), p.offset, p.seed_lo, p.seed_hi);
    if (lane == 0) mbar_arrive(ready(0));   // nothing to read before the first tile
    bool ok = true;
    for (int it = 0; it < n && ok; ++it) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_S, it & 1, abort_flag, p.err, kSiteSoftmaxS));
      if (!ok) break;
      tc_fence_after();
      const int k0 = it * 128 + 64 * h;
      float pv[64];
      // masked entries: keys past Lk (last key tile) and keys above the
      // causal diagonal; the whole tile is checked once (uniform for the CTA)
      auto l2f = [&](int) { return l2; };
      auto valid = [&](int i) { return k0 + i < p.Lk && (!p.causal || k0 + i <= qrow); };
      tmem_ld64_sync(tS + 64 * h, pv);
      // S is in registers: the next tile's S may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ready(it + 1));
      if (it * 128 + 128 <= p.Lk && (!p.causal || it * 128 + 127 <= itile * 128))
        weights_p<false>(pv, p.scale_log2, l2f, valid);
      else
        weights_p<true>(pv, p.scale_log2, l2f, valid);
      uint32_t kw[16];   // dropout: keep bits of the half's 64 keys for this row
      if constexpr (DROP) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 wv = philox4x32_10_row(uint32_t(k0 >> 4) + uint32_t(c), prow, p.keys);
          kw[4 * c] = dropout_keep_msb(wv.x, p.drop_tl4, p.drop_hsel);
          kw[4 * c + 1] = dropout_keep_msb(wv.y, p.drop_tl4, p.drop_hsel);
          kw[4 * c + 2] = dropout_keep_msb(wv.z, p.drop_tl4, p.drop_hsel);
          kw[4 * c + 3] = dropout_keep_msb(wv.w, p.drop_tl4, p.drop_hsel);
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dP, it & 1, abort_flag, p.err, kSiteSoftmaxS));
      if (!ok) break;
      tc_fence_after();
      if constexpr (DROP)
        weights_ds_drop(tdP, h, pv, [&](int) { return dr; }, kw, p.keep_scale);
      else
        weights_ds(tdP, h, pv, [&](int) { return dr; });
      warp_arrive_after_st(bar_dS, lane);
    }
    // epilogue: scale * dQ, columns [h D/2, (h+1) D/2) of this query's row
    // (warp-collective TMEM loads, predicated stores)
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_done, 0, abort_flag, p.err, kSiteSoftmaxO));
    if (ok) {
      tc_fence_after();
      const bool valid = qrow < p.Lq;
      const size_t orow = (size_t(bh) * p.Lq + (valid ? qrow : 0)) * D;
#pragma unroll 1
      for (int cc = h * D / 2; cc < (h + 1) * D / 2; cc += 32) {
        float v[32];
        tmem_ld32_sync(tmem + lane_off + 256 + cc, v);
        if (valid) store_row32(p.out_a + orow + cc, v, p.scale);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool DROP>
int launch_bwd_d(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int BH, int Lq, int Lk, float scale,
                 int causal, float* ws, int* err, cudaStream_t stream, const Dropout& dr) {
  using CK = BwCfg<D, false, DROP>;
  using CQ = BwCfg<D, true, DROP>;
  CUtensorMap mq, mk, mv, mdo;
  int st = make_tensor_map_bf16(&mq, q, BH, Lq, D);
  if (st == 0) st = make_tensor_map_bf16(&mk, k, BH, Lk, D);
  if (st == 0) st = make_tensor_map_bf16(&mv, v, BH, Lk, D);
  if (st == 0) st = make_tensor_map_bf16(&mdo, dout, BH, Lq, D);
  if (st != 0) return st;
  BwParams p;
  p.BH = BH;
  p.Lq = Lq;
  p.Lk = Lk;
  p.Lq_pad = (Lq + 127) / 128 * 128;
  p.causal = causal;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.err = err;
  p.seed_lo = dr.seed_lo;
  p.seed_hi = dr.seed_hi;
  p.offset = dr.offset;
  p.drop_tl4 = (dr.t & 0x7fu) * 0x01010101u;
  p.drop_hsel = dr.t >= 128u ? 0xffffffffu : 0u;
  p.keys = philox_round_keys(dr.seed_lo, dr.seed_hi);
  p.keep_scale = dr.keep_scale;
  float* lse2 = ws;
  float* drow = ws + size_t(BH) * p.Lq_pad;
  p.lse2 = lse2;
  p.drow = drow;
  {
    const long long threads = (long long)BH * p.Lq_pad * (D / 8);
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return -2;
    fa_bwd_prep_kernel<D><<<dim3(unsigned(blocks)), dim3(256), 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, lse2, drow,
        BH, Lq, p.Lq_pad);
    if (cudaGetLastError() != cudaSuccess) return -4;
  }
  if (cudaFuncSetAttribute(fa_bwd_dkdv_kernel<D, DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           CK::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(fa_bwd_dq_kernel<D, DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           CQ::kSmemBytes) != cudaSuccess)
    return -4;
  const long long nk = (long long)((Lk + 127) / 128) * BH;
  const long long nq = (long long)((Lq + 127) / 128) * BH;
  if (nk > 0x7fffffffLL || nq > 0x7fffffffLL) return -2;
  p.out_a = static_cast<__nv_bfloat16*>(dk);
  p.out_b = static_cast<__nv_bfloat16*>(dv);
  p.group = l2_head_group(BH, 2ll * Lq * D * 2);   // Q and dO of a head
  fa_bwd_dkdv_kernel<D, DROP><<<dim3(unsigned(nk)), dim3(kThreads), CK::kSmemBytes, stream>>>(mq, mk, mv, mdo, p);
  if (cudaGetLastError() != cudaSuccess) return -4;
  p.out_a = static_cast<__nv_bfloat16*>(dq);
  p.out_b = nullptr;
  p.group = l2_head_group(BH, 2ll * Lk * D * 2);   // K and V of a head
  fa_bwd_dq_kernel<D, DROP><<<dim3(unsigned(nq)), dim3(kThreads), CQ::kSmemBytes, stream>>>(mq, mk, mv, mdo, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

int launch_backward(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, int BH, int Lq, int Lk, int D,
                    float scale, int causal, float* workspace, int* err, cudaStream_t stream,
                    const Dropout& dr) {
  if (D == 64 && dr.on)
    return launch_bwd_d<64, true>(q, k, v, o, dout, lse, dq, dk, dv, BH, Lq, Lk, scale, causal, workspace, err,
                                  stream, dr);
  if (D == 64)
    return launch_bwd_d<64, false>(q, k, v, o, dout, lse, dq, dk, dv, BH, Lq, Lk, scale, causal, workspace, err,
                                   stream, dr);
  if (D == 128 && dr.on)
    return launch_bwd_d<128, true>(q, k, v, o, dout, lse, dq, dk, dv, BH, Lq, Lk, scale, causal, workspace, err,
                                   stream, dr);
  if (D == 128)
    return launch_bwd_d<128, false>(q, k, v, o, dout, lse, dq, dk, dv, BH, Lq, Lk, scale, causal, workspace, err,
                                    stream, dr);
  return -2;
}

}  // namespace fa
