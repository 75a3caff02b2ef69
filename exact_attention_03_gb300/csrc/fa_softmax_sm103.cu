// fa_softmax_sm103.cu - row softmax in two reads (fa_softmax_rows).
//
// "NTU Hung-yi Lee ML 2026 Guide: Faster Generation, Part 1: Flash Attention"
// (quidproquo.cc), "Expand: why multiplying by exp(d1 - d2) fixes it": a row's
// maximum and denominator can be found in one read, chunk by chunk, keeping a
// running maximum d and a running sum s that is multiplied by exp(d_old -
// d_new) whenever the maximum grows; a second read then writes the weights
// exp(a_i - Amax) / S.  This file is that two-read softmax as an operation of
// its own over the rows of a matrix:
//
//   read 1: every thread keeps (d, s) over the groups of 4 elements (16 in
//           the one-warp-per-row kernel) it reads, one rescale per group; then
//           the pairs of a warp, and of the warps of a CTA, are merged with the
//           same identity (d = max, s = s1 exp(d1 - d) + s2 exp(d2 - d));
//   read 2: y_i = exp(a_i - d) / s, written once.
//
// A row of up to kWarpCols columns is one warp's (8 rows per CTA); a longer row
// is one CTA's (256 threads).  A longer row that is 16-byte aligned, has a
// multiple of 4 columns and at most kSmemCols of them is copied whole into
// shared memory by one bulk copy, the next row's copy running while the CTA
// works on this one (two row buffers per CTA, several CTAs per SM): both reads
// then come from shared memory, and the bytes in flight per SM are whole rows
// instead of one vector per thread.  Exponentials are base 2: the running maximum is
// kept as D = d log2 e (rounded once), every term as 2^(a log2 e - D) (one fused
// multiply-add) and every rescale as 2^(D_old - D_new), so that all terms of a
// row share one reference.  Rows are independent; the grid walks them in
// strides.
#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

#include <cmath>
#include <cstdint>

namespace fa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpCols = 2048;
constexpr int kSmemCols = 16384;   // two rows of 64 KB: one CTA per SM at the most
constexpr int kSmemThreads = 256;  // threads of the shared-memory kernel
constexpr int kSmemMisc = 16 + 8 * kSmemThreads / 32 + 16;   // barriers, the warps' (D, s) pairs, abort flag
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

// (D, s) after adding the values v[0..n): D = running maximum times log2 e,
// s = sum of 2^(a log2 e - D); one rescale of s for the group
__device__ __forceinline__ void online_group(float& D, float& s, const float* v, int n) {
  float mx = v[0];
  for (int i = 1; i < n; ++i) mx = fmaxf(mx, v[i]);
  const float Dn = fmaxf(D, mx * kLog2e);
  if (Dn == -INFINITY) return;  // every value so far is -inf
  float add = 0.f;
  for (int i = 0; i < n; ++i) add += ex2_approx(fmaf(v[i], kLog2e, -Dn));
  s = s * ex2_approx(D - Dn) + add;
  D = Dn;
}

// merge of two partial (D, s) pairs
__device__ __forceinline__ void merge(float& D, float& s, float D2, float s2) {
  const float Dn = fmaxf(D, D2);
  if (Dn == -INFINITY) return;  // both empty
  s = s * ex2_approx(D - Dn) + s2 * ex2_approx(D2 - Dn);
  D = Dn;
}

// read 1 over this thread's share of a row: vector loads when the row is
// 16-byte aligned, scalar loads otherwise; with UNROLL, four loads in flight
// per thread and one rescale per 16 values (the one-warp-per-row kernel,
// whose rows give each thread few loads)
template <bool UNROLL>
__device__ __forceinline__ void scan(const float* row, int cols, int t, int nt, float& d, float& s) {
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
    const int n4 = cols >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    int i = t;
    if constexpr (UNROLL)
    for (; i + 3 * nt < n4; i += 4 * nt) {
      const float4 a = __ldg(r4 + i), b = __ldg(r4 + i + nt), c = __ldg(r4 + i + 2 * nt),
                   e = __ldg(r4 + i + 3 * nt);
      const float v[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, e.x, e.y, e.z, e.w};
      online_group(d, s, v, 16);
    }
    for (; i < n4; i += nt) {
      const float4 v4 = __ldg(r4 + i);
      const float v[4] = {v4.x, v4.y, v4.z, v4.w};
      online_group(d, s, v, 4);
    }
    for (int i = (n4 << 2) + t; i < cols; i += nt) online_group(d, s, row + i, 1);
  } else {
    for (int i = t; i < cols; i += nt) {
      const float v = __ldg(row + i);
      online_group(d, s, &v, 1);
    }
  }
}

// read 2: y = 2^(a log2 e - D) / s (a row without any finite value gives 0)
template <bool UNROLL>
__device__ __forceinline__ void write_row(const float* row, float* out, int cols, int t, int nt,
                                          float D, float s) {
  const bool empty = !(s > 0.f);
  const float inv = empty ? 0.f : 1.f / s;
  const float ds = empty ? 0.f : D;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
    const int n4 = cols >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    float4* o4 = reinterpret_cast<float4*>(out);
    auto weights = [&](const float4 v) {
      return make_float4(ex2_approx(fmaf(v.x, kLog2e, -ds)) * inv, ex2_approx(fmaf(v.y, kLog2e, -ds)) * inv,
                         ex2_approx(fmaf(v.z, kLog2e, -ds)) * inv, ex2_approx(fmaf(v.w, kLog2e, -ds)) * inv);
    };
    int i = t;
    if constexpr (UNROLL)
    for (; i + 3 * nt < n4; i += 4 * nt) {
      const float4 a = __ldg(r4 + i), b = __ldg(r4 + i + nt), c = __ldg(r4 + i + 2 * nt),
                   e = __ldg(r4 + i + 3 * nt);
      o4[i] = weights(a);
      o4[i + nt] = weights(b);
      o4[i + 2 * nt] = weights(c);
      o4[i + 3 * nt] = weights(e);
    }
    for (; i < n4; i += nt) o4[i] = weights(__ldg(r4 + i));
    for (int i = (n4 << 2) + t; i < cols; i += nt) out[i] = ex2_approx(fmaf(row[i], kLog2e, -ds)) * inv;
  } else {
    for (int i = t; i < cols; i += nt) out[i] = ex2_approx(fmaf(__ldg(row + i), kLog2e, -ds)) * inv;
  }
}

__device__ __forceinline__ void warp_merge(float& d, float& s) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float d2 = __shfl_xor_sync(0xffffffffu, d, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    merge(d, s, d2, s2);
  }
}

// rows of up to kWarpCols columns: one warp per row
__global__ void __launch_bounds__(kThreads) softmax_rows_warp(const float* x, float* y, float* lse,
                                                              long long rows, int cols) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (kThreads / 32);
  for (long long r = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
    const float* row = x + r * cols;
    float d = -INFINITY, s = 0.f;
    scan<true>(row, cols, lane, 32, d, s);
    warp_merge(d, s);
    write_row<true>(row, y + r * cols, cols, lane, 32, d, s);
    if (lse != nullptr && lane == 0) lse[r] = (s > 0.f) ? (d + __log2f(s)) * kLn2 : -INFINITY;
  }
}

// longer rows: one CTA per row
__global__ void __launch_bounds__(kThreads) softmax_rows_cta(const float* x, float* y, float* lse,
                                                             long long rows, int cols) {
  __shared__ float sd[kThreads / 32], ss[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const float* row = x + r * cols;
    float d = -INFINITY, s = 0.f;
    scan<false>(row, cols, threadIdx.x, kThreads, d, s);
    warp_merge(d, s);
    if (lane == 0) {
      sd[warp] = d;
      ss[warp] = s;
    }
    __syncthreads();
    d = sd[0];
    s = ss[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) merge(d, s, sd[w], ss[w]);
    write_row<false>(row, y + r * cols, cols, threadIdx.x, kThreads, d, s);
    if (lse != nullptr && threadIdx.x == 0) lse[r] = (s > 0.f) ? (d + __log2f(s)) * kLn2 : -INFINITY;
    __syncthreads();  // sd/ss are rewritten for the next row
  }
}

// 1-D bulk copy global -> shared, completing `bytes` on `bar` (both addresses
// 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void bulk_row(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// longer rows through shared memory: one CTA per row, its rows in strides of
// the grid, row k of the CTA in buffer k mod 2 (cols a multiple of 4, x
// 16-byte aligned; y needs only 4-byte alignment)
__global__ void __launch_bounds__(kSmemThreads) softmax_rows_smem(const float* x, float* y, float* lse,
                                                              long long rows, int cols, int* err) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* const buf0 = reinterpret_cast<float*>(smem);
  auto buf = [&](int b) { return buf0 + size_t(b) * cols; };
  uint8_t* misc = smem + size_t(2) * cols * sizeof(float);
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);          // [2]
  float* sd = reinterpret_cast<float*>(misc + 16);              // [kSmemThreads / 32]
  float* ss = sd + kSmemThreads / 32;                           // [kSmemThreads / 32]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ss + kSmemThreads / 32);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t bytes = uint32_t(cols) * 4u;
  int issued = 0;   // copies issued (thread 0)
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&full[0]), 1);
    mbar_init(smem_u32(&full[1]), 1);
    *abort_flag = 0;
    fence_mbar_init();
    if ((long long)blockIdx.x < rows) {
      mbar_arrive_expect_tx(smem_u32(&full[0]), bytes);
      bulk_row(smem_u32(buf(0)), x + (long long)blockIdx.x * cols, bytes, smem_u32(&full[0]));
      issued = 1;
    }
  }
  __syncthreads();
  int k = 0;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x, ++k) {
    const int b = k & 1;
    // the next row's copy into the other buffer, whose last row every thread
    // finished with before the previous iteration's closing barrier
    if (threadIdx.x == 0 && r + gridDim.x < rows) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // after the generic reads of the buffer
      mbar_arrive_expect_tx(smem_u32(&full[b ^ 1]), bytes);
      bulk_row(smem_u32(buf(b ^ 1)), x + (r + gridDim.x) * cols, bytes, smem_u32(&full[b ^ 1]));
      ++issued;
    }
    // every thread waits (bounded); the CTA leaves together if any gave up
    const bool landed = mbar_wait(smem_u32(&full[b]), (k >> 1) & 1, abort_flag, err, kSiteSoftmaxS);
    if (__syncthreads_or(!landed)) break;
    const float4* r4 = reinterpret_cast<const float4*>(buf(b));
    const int n4 = cols >> 2;
    // read 1
    float d = -INFINITY, s = 0.f;
    for (int i = threadIdx.x; i < n4; i += kSmemThreads) {
      const float4 v4 = r4[i];
      const float v[4] = {v4.x, v4.y, v4.z, v4.w};
      online_group(d, s, v, 4);
    }
    warp_merge(d, s);
    if (lane == 0) {
      sd[warp] = d;
      ss[warp] = s;
    }
    __syncthreads();
    d = sd[0];
    s = ss[0];
#pragma unroll
    for (int w = 1; w < kSmemThreads / 32; ++w) merge(d, s, sd[w], ss[w]);
    // read 2: y = 2^(a log2 e - D) / s
    const bool empty = !(s > 0.f);
    const float inv = empty ? 0.f : 1.f / s;
    const float ds = empty ? 0.f : d;
    float* out = y + r * cols;
    if ((reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
      float4* o4 = reinterpret_cast<float4*>(out);
      for (int i = threadIdx.x; i < n4; i += kSmemThreads) {
        const float4 v = r4[i];
        o4[i] = make_float4(ex2_approx(fmaf(v.x, kLog2e, -ds)) * inv, ex2_approx(fmaf(v.y, kLog2e, -ds)) * inv,
                            ex2_approx(fmaf(v.z, kLog2e, -ds)) * inv, ex2_approx(fmaf(v.w, kLog2e, -ds)) * inv);
      }
    } else {
      const float* rv = buf(b);
      for (int i = threadIdx.x; i < cols; i += kSmemThreads) out[i] = ex2_approx(fmaf(rv[i], kLog2e, -ds)) * inv;
    }
    if (lse != nullptr && threadIdx.x == 0) lse[r] = empty ? -INFINITY : (d + __log2f(s)) * kLn2;
    __syncthreads();  // the buffer, sd and ss are rewritten for the CTA's row after next / next row
  }
  // every copy this CTA issued has landed before it exits (a CTA that gave up
  // on an error may still have one in flight)
  if (threadIdx.x == 0) {
    for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) {
      const uint64_t t0 = globaltimer_ns();
      for (uint32_t it = 0; it < (1u << 24) && !mbar_try_wait(smem_u32(&full[j & 1]), uint32_t((j >> 1) & 1)); ++it)
        if (globaltimer_ns() - t0 > 50000000ull) break;   // 50 ms
    }
  }
}

}  // namespace
}  // namespace fa

extern "C" int fa_softmax_rows(const float* x, float* y, float* lse, long long rows, int cols,
                               void* stream) {
  if (x == nullptr || y == nullptr) return FA_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0) return FA_ERR_INVALID_ARG;
  if (rows > (1LL << 40) / cols) return FA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) & 3u) != 0 || (reinterpret_cast<uintptr_t>(y) & 3u) != 0 ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
    return FA_ERR_MISALIGNED;
  int sms = 0;
  if (fa::num_sms_of_current_device(&sms) != FA_OK) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cols <= fa::kWarpCols) {
    const long long want = (rows + fa::kThreads / 32 - 1) / (fa::kThreads / 32);
    const long long grid = want < 16LL * sms ? want : 16LL * sms;
    fa::softmax_rows_warp<<<dim3(unsigned(grid)), dim3(fa::kThreads), 0, s>>>(x, y, lse, rows, cols);
  } else if (cols <= fa::kSmemCols && (cols & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    int* err = fa::error_word_ptr(dev);
    if (err == nullptr) return FA_ERR_CUDA;
    const int smem = 2 * cols * 4 + fa::kSmemMisc;
    // CTAs per SM by shared memory: 228 KB per SM, 1 KB reserved per CTA
    int per_sm = 233472 / (smem + 1024);
    if (per_sm > 8) per_sm = 8;
    const long long grid = rows < (long long)per_sm * sms ? rows : (long long)per_sm * sms;
    if (cudaFuncSetAttribute(fa::softmax_rows_smem, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return FA_ERR_CUDA;
    fa::softmax_rows_smem<<<dim3(unsigned(grid)), dim3(fa::kSmemThreads), smem, s>>>(x, y, lse, rows, cols, err);
  } else {
    const long long grid = rows < 8LL * sms ? rows : 8LL * sms;
    fa::softmax_rows_cta<<<dim3(unsigned(grid)), dim3(fa::kThreads), 0, s>>>(x, y, lse, rows, cols);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
