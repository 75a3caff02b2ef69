// fa_decode_sm103.cu - single-query (Lq == 1) attention: split-K/V + combine.
//
// With one query row per head a tensor-core tile would be 1/128 full and the
// work is a pure stream over K and V (about 1 flop per byte), so it runs on
// CUDA cores and is sized for HBM bandwidth:
//
//   fa_decode_split_kernel  grid = B*H*n_split CTAs of 256 threads.  CTA
//     (head, split) streams keys [split*chunk, (split+1)*chunk) of that head.
//     A group of D/8 lanes owns one key at a time (16 bytes of K and of V per
//     lane, coalesced 128/256-byte rows); each lane keeps several keys' K and
//     V in flight.  The dot product is reduced with warp shuffles, then the
//     group applies the guide's recurrence for its keys ("Expand: why
//     multiplying by exp(d1 - d2) fixes it" / "Expand: the correction for the
//     output O", NTU Hung-yi Lee ML 2026 Guide, quidproquo.cc): new max,
//     rescale of the running denominator and output by 2^(m_old - m_new),
//     add the new terms.  The CTA's groups are merged the same way through
//     shared memory and the split writes (m, l, unnormalised O) in fp32.
//   fa_decode_combine_kernel  one CTA per head merges the n_split partials
//     with the same rescale identity (M = max m_s, l = sum l_s 2^(m_s - M),
//     O = sum O_s 2^(m_s - M) / l) and writes O (bf16) and LSE (fp32).
// Exponentials are base 2: x = q.k * scale * log2(e).
//
// The same kernels serve a paged key/value cache (fa_fwd_decode_paged): keys
// and values of sequence b live in pages of page_size positions, [num_pages,
// page_size, H, D], listed in order by row b of a page table; sequence b has
// seq_lens[b] positions.  A split then covers positions [split*chunk, ...) of
// its sequence, looks the pages up through the table (staged in shared memory,
// every page id bounds-checked), and splits past the sequence's end leave an
// empty partial (m = -inf, l = 0) that the combine weighs with zero.
#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kUnroll = 4;  // keys per group kept in flight
constexpr int kCombThreads = 256;
constexpr float kLn2 = 0.69314718055994530942f;

struct DecParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  float* lse;
  float* part_o;   // [n_split][BH][D]
  float* part_ml;  // [n_split][BH][2]  (m in log2 units, l)
  int BH, Lk, n_split, chunk;
  float scale_log2;
  // paged cache only
  const int* block_table;  // [B][max_pages]
  const int* seq_lens;     // [B]
  int* err;                // device error word: a page id out of range
  int H, max_pages, num_pages, page_shift;
};
constexpr int kMaxPagesPerSplit = 2048;   // page-table entries one split stages

__device__ __forceinline__ uint4 ld_stream16(const void* ptr) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(ptr));
  return r;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D, bool PAGED>
__global__ void __launch_bounds__(kDecThreads) fa_decode_split_kernel(const DecParams p) {
  constexpr int G = D / 8;             // lanes per key
  constexpr int GPW = 32 / G;          // key groups per warp
  constexpr int NG = kDecWarps * GPW;  // key groups per CTA
  __shared__ float sm_m[NG], sm_l[NG];
  __shared__ float sm_acc[NG][D];
  __shared__ int sm_page[PAGED ? kMaxPagesPerSplit : 1];

  const int split = int(blockIdx.x) % p.n_split;
  const int bh = int(blockIdx.x) / p.n_split;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = warp * GPW + lane / G;  // key group of this lane
  const int li = lane % G;               // this lane covers dims [8*li, 8*li + 8)

  // query slice, pre-multiplied by scale*log2(e)
  float qf[8];
  {
    const uint4 qw = *reinterpret_cast<const uint4*>(p.q + size_t(bh) * D + 8 * li);
    const uint32_t w[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qf[2 * e] = bf_lo(w[e]) * p.scale_log2;
      qf[2 * e + 1] = bf_hi(w[e]) * p.scale_log2;
    }
  }

  const int kbeg = split * p.chunk;
  int kend;
  const __nv_bfloat16* kp;
  const __nv_bfloat16* vp;
  if constexpr (PAGED) {
    // this sequence's length, clamped to what its page-table row can address
    const int b = bh / p.H;
    const int len = min(max(p.seq_lens[b], 0), p.max_pages << p.page_shift);
    kend = min(kbeg + p.chunk, len);
    // page ids of positions [kbeg, kend), checked against the cache size
    const int pg0 = kbeg >> p.page_shift;
    const int npg = kend > kbeg ? ((kend - 1) >> p.page_shift) - pg0 + 1 : 0;
    for (int i = threadIdx.x; i < npg; i += kDecThreads) {
      int pg = p.block_table[size_t(b) * p.max_pages + pg0 + i];
      if (pg < 0 || pg >= p.num_pages) {  // record it; the page's keys stay unread
        if (atomicCAS(p.err, 0, FA_ERR_INVALID_ARG) == 0) atomicExch(p.err + 1, kSitePageTable);
        pg = -1;
      }
      sm_page[i] = pg;
    }
    __syncthreads();
    const int h = bh - b * p.H;
    kp = p.k + size_t(h) * D + 8 * li;   // + (page * page_size + offset) * H * D
    vp = p.v + size_t(h) * D + 8 * li;
  } else {
    const size_t head = size_t(bh) * size_t(p.Lk) * D;
    kp = p.k + head + 8 * li;
    vp = p.v + head + 8 * li;
    kend = min(kbeg + p.chunk, p.Lk);
  }

  float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;

  // the loop bound is uniform over the CTA, so every lane takes part in the shuffles
  for (int base = kbeg; base < kend; base += NG * kUnroll) {
    uint4 kr[kUnroll], vr[kUnroll];
    bool valid[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int key = base + u * NG + gi;
      valid[u] = key < kend;
      size_t row = size_t(key);
      if constexpr (PAGED) {
        if (valid[u]) {
          const int pg = sm_page[(key >> p.page_shift) - (kbeg >> p.page_shift)];
          valid[u] = pg >= 0;
          row = (size_t(pg) << p.page_shift) + (key & ((1 << p.page_shift) - 1));
          row *= size_t(p.H);
        }
      }
      if (valid[u]) {
        kr[u] = ld_stream16(kp + row * D);
        vr[u] = ld_stream16(vp + row * D);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t w[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
      float d0 = 0.f, d1 = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        d0 = fmaf(qf[2 * e], bf_lo(w[e]), d0);
        d1 = fmaf(qf[2 * e + 1], bf_hi(w[e]), d1);
      }
      float d = d0 + d1;
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      x[u] = valid[u] ? d : -INFINITY;
    }
    float mx = x[0];
#pragma unroll
    for (int u = 1; u < kUnroll; ++u) mx = fmaxf(mx, x[u]);
    const float m_new = fmaxf(m, mx);
    const float m_safe = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = ex2_approx(m - m_safe);
    l *= alpha;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float pu = ex2_approx(x[u] - m_safe);
      l += pu;
      const uint32_t w[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] = fmaf(pu, bf_lo(w[e]), acc[2 * e]);
        acc[2 * e + 1] = fmaf(pu, bf_hi(w[e]), acc[2 * e + 1]);
      }
    }
    m = m_new;
  }

  // merge the CTA's key groups
  if (li == 0) {
    sm_m[gi] = m;
    sm_l[gi] = l;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) sm_acc[gi][8 * li + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    const int d = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int g2 = 0; g2 < NG; ++g2) M = fmaxf(M, sm_m[g2]);
    const float M_safe = (M == -INFINITY) ? 0.f : M;
    float od = 0.f, L = 0.f;
#pragma unroll
    for (int g2 = 0; g2 < NG; ++g2) {
      const float w = ex2_approx(sm_m[g2] - M_safe);
      od = fmaf(sm_acc[g2][d], w, od);
      L = fmaf(sm_l[g2], w, L);
    }
    const size_t slot = size_t(split) * p.BH + bh;
    p.part_o[slot * D + d] = od;
    if (d == 0) {
      p.part_ml[slot * 2 + 0] = M;
      p.part_ml[slot * 2 + 1] = L;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kCombThreads) fa_decode_combine_kernel(const DecParams p) {
  // one CTA per head: warp w folds splits w, w + 8, ... (lanes over the D
  // output dims, several splits' loads in flight), then the warps' partial
  // sums are folded through shared memory
  constexpr int E = D / 32;  // output dims per lane
  constexpr int W = kCombThreads / 32;
  __shared__ float red_m[W], red_l[W];
  __shared__ float red_acc[W][D];
  const int bh = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  float m = -INFINITY;
  for (int s = threadIdx.x; s < p.n_split; s += kCombThreads)
    m = fmaxf(m, p.part_ml[(size_t(s) * p.BH + bh) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) red_m[warp] = m;
  __syncthreads();
  float M = red_m[0];
#pragma unroll
  for (int w = 1; w < W; ++w) M = fmaxf(M, red_m[w]);
  const float M_safe = (M == -INFINITY) ? 0.f : M;

  float acc[E], L = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int s = warp; s < p.n_split; s += W) {
    const size_t slot = size_t(s) * p.BH + bh;
    const float ms = p.part_ml[slot * 2 + 0];
    const float ls = p.part_ml[slot * 2 + 1];
    const float w = ex2_approx(ms - M_safe);
    L = fmaf(ls, w, L);
    const float* po = p.part_o + slot * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(po[e], w, acc[e]);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) red_acc[warp][lane * E + e] = acc[e];
  if (lane == 0) red_l[warp] = L;
  __syncthreads();
  if (threadIdx.x < D / 2) {
    const int d = 2 * threadIdx.x;
    float L_tot = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      L_tot += red_l[w];
      o0 += red_acc[w][d];
      o1 += red_acc[w][d + 1];
    }
    // an empty row (a paged sequence of length 0) has L_tot = 0: O = 0, LSE = -inf
    const float inv = L_tot > 0.f ? 1.f / L_tot : 0.f;
    *reinterpret_cast<uint32_t*>(p.o + size_t(bh) * D + d) = pack_bf16x2(o0 * inv, o1 * inv);
    if (threadIdx.x == 0 && p.lse != nullptr)
      p.lse[bh] = L_tot > 0.f ? (M + __log2f(L_tot)) * kLn2 : -INFINITY;
  }
}

template <int D, bool PAGED>
int launch(const DecParams& p, cudaStream_t stream) {
  const long long nblk = (long long)p.BH * p.n_split;
  if (nblk > 0x7fffffffLL) return -2;
  fa_decode_split_kernel<D, PAGED><<<dim3(unsigned(nblk)), dim3(kDecThreads), 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return -4;
  fa_decode_combine_kernel<D><<<dim3(unsigned(p.BH)), dim3(kCombThreads), 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

int launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int Lk,
                  int D, float scale, int n_split, float* workspace, cudaStream_t stream) {
  DecParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.BH = BH;
  p.Lk = Lk;
  p.n_split = n_split;
  p.chunk = (Lk + n_split - 1) / n_split;
  p.part_o = workspace;
  p.part_ml = workspace + size_t(n_split) * BH * D;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.block_table = nullptr;
  p.seq_lens = nullptr;
  p.err = nullptr;
  p.H = 1;
  p.max_pages = 0;
  p.num_pages = 0;
  p.page_shift = 0;
  if (D == 64) return launch<64, false>(p, stream);
  if (D == 128) return launch<128, false>(p, stream);
  return -2;
}

int launch_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                        const int* block_table, const int* seq_lens, void* o, float* lse, int B,
                        int H, int D, int num_pages, int page_size, int max_pages, float scale,
                        int n_split, float* workspace, int* err, cudaStream_t stream) {
  DecParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k_cache);
  p.v = static_cast<const __nv_bfloat16*>(v_cache);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.BH = B * H;
  const long long max_len = (long long)max_pages * page_size;
  p.Lk = int(max_len);
  p.n_split = n_split;
  p.chunk = int((max_len + n_split - 1) / n_split);
  if ((p.chunk + page_size - 1) / page_size + 1 > kMaxPagesPerSplit) return -2;
  p.part_o = workspace;
  p.part_ml = workspace + size_t(n_split) * p.BH * D;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.err = err;
  p.H = H;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  int shift = 0;
  while ((1 << shift) < page_size) ++shift;
  p.page_shift = shift;
  if (D == 64) return launch<64, true>(p, stream);
  if (D == 128) return launch<128, true>(p, stream);
  return -2;
}

}  // namespace fa
