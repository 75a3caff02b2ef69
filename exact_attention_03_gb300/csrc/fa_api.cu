// fa_api.cu - the C ABI declared in include/fa.h: argument checks, TMA
// tensor maps, dispatch to the prefill / single-query kernels, the device
// error word and the bounded-wait self-test.
#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

#include <cmath>
#include <cstdint>
#include <mutex>

namespace fa {

// [0] status of the first device-side wait that gave up (0 = none), [1] its site.
__device__ int g_device_error[2];

constexpr int kMaxDevices = 64;

int* error_word_ptr(int dev) {
  static std::mutex mu;
  static int* cached[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(ptr);
  }
  return cached[dev];
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The library's stream-ordered workspace pool on device `dev`.  Its release
// threshold is the maximum, so memory freed at the end of a call stays in the
// pool for the next one instead of being unmapped at the next synchronisation.
cudaMemPool_t workspace_pool(int dev) {
  static std::mutex mu;
  static cudaMemPool_t pools[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (pools[dev] == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t keep = UINT64_MAX;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return nullptr;
    }
    pools[dev] = pool;
  }
  return pools[dev];
}

__global__ void wait_selftest_kernel(int* err, unsigned long long limit_ns) {
  __shared__ alignas(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the wait must give up after limit_ns
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, err, kSiteSelftest, limit_ns);
}

}  // namespace

int workspace_alloc(void** ptr, size_t bytes, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  cudaMemPool_t pool = workspace_pool(dev);
  if (pool == nullptr) return FA_ERR_CUDA;
  return cudaMallocFromPoolAsync(ptr, bytes, pool, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int workspace_free(void* ptr, cudaStream_t stream) {
  return cudaFreeAsync(ptr, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int make_tensor_map_bf16(CUtensorMap* map, const void* ptr, int BH, int L, int D) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return FA_ERR_CUDA;
  // [BH, L, D] seen as {64 columns, L rows, D/64 column blocks, BH heads}: a box
  // {64, 128, D/64, 1} is one 128-row tile, stored in shared memory as D/64
  // blocks of 128 rows x 128 bytes (the 128-byte swizzle works per block).
  const cuuint64_t dims[4] = {64, cuuint64_t(L), cuuint64_t(D / 64), cuuint64_t(BH)};
  const cuuint64_t strides[3] = {cuuint64_t(D) * 2, 128, cuuint64_t(L) * cuuint64_t(D) * 2};
  const cuuint32_t box[4] = {64, 128, cuuint32_t(D / 64), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Prefill / general path: head dimension 64 (fa_prefill_d64x1_sm103.cu, or
// fa_prefill_d64_sm103.cu with dropout) or 128 (fa_prefill_d128_sm103.cu).
int launch_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int Lq, int Lk, int D, float scale, int causal, cudaStream_t stream, int* err,
                   const Dropout& dr) {
  if (D == 64) return launch_prefill_d64(q, k, v, o, lse, B, H, Lq, Lk, scale, causal, stream, err, dr);
  if (D == 128) return launch_prefill_d128(q, k, v, o, lse, B, H, Lq, Lk, scale, causal, stream, err, dr);
  return -2;
}

// The dropout contract of fa_fwd_dropout / fa_bwd_dropout: t = floor(256 p
// + 1/2) in double precision (p in [0, 1), t <= 255), keep_scale =
// 256 / (256 - t), the 64-bit seed split into the Philox key words.
int make_dropout(float p_drop, unsigned long long seed, unsigned int offset, Dropout* dr) {
  if (!std::isfinite(p_drop) || !(p_drop >= 0.f) || !(p_drop < 1.f)) return FA_ERR_INVALID_ARG;
  const double tt = std::floor(double(p_drop) * 256.0 + 0.5);
  if (tt > 255.0) return FA_ERR_INVALID_ARG;
  dr->on = 1;
  dr->seed_lo = uint32_t(seed & 0xffffffffull);
  dr->seed_hi = uint32_t(seed >> 32);
  dr->offset = offset;
  dr->t = uint32_t(tt);
  dr->keep_scale = float(256.0 / (256.0 - tt));
  return FA_OK;
}

int num_sms_of_current_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace fa

extern "C" {

int fa_abi_version(void) { return FA_ABI_VERSION; }

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "success";
    case FA_ERR_INVALID_ARG: return "invalid argument (null pointer, non-positive size or bad scale)";
    case FA_ERR_UNSUPPORTED: return "unsupported problem (head dim not 64/128, causal with Lq != Lk, or size limit)";
    case FA_ERR_MISALIGNED: return "misaligned pointer (q/k/v/o need 16 bytes, lse 4 bytes)";
    case FA_ERR_CUDA: return "CUDA runtime or driver call failed";
    case FA_ERR_TIMEOUT: return "a device-side wait gave up (timeout)";
    default: return "unknown fa_status";
  }
}

int fa_decode_num_splits(int BH, int Lk, int num_sms) {
  if (BH <= 0 || Lk <= 0 || num_sms <= 0) return FA_ERR_INVALID_ARG;
  // about 2048 keys (1 MB of K+V at D = 128) per CTA, at least ~32 CTAs per SM
  // in total, at least 64 keys per split, at most 4096 splits
  long long n = (Lk + 2047LL) / 2048;
  const long long fill = (32LL * num_sms + BH - 1) / BH;
  if (fill > n) n = fill;
  const long long max_by_len = Lk / 64 > 0 ? Lk / 64 : 1;
  if (n > max_by_len) n = max_by_len;
  if (n > 4096) n = 4096;
  if (n < 1) n = 1;
  // no empty split: recompute from the chunk length
  const long long chunk = (Lk + n - 1) / n;
  n = (Lk + chunk - 1) / chunk;
  return int(n);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Lq,
           int Lk, int D, float scale, int causal, void* stream) {
  // ---- host-side checks, before any CUDA call
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Lq <= 0 || Lk <= 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (causal && Lq != Lk) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (!fa::aligned(q, 16) || !fa::aligned(k, 16) || !fa::aligned(v, 16) || !fa::aligned(o, 16))
    return FA_ERR_MISALIGNED;
  if (lse != nullptr && !fa::aligned(lse, 4)) return FA_ERR_MISALIGNED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  int* err = fa::error_word_ptr(dev);
  if (err == nullptr) return FA_ERR_CUDA;

  if (Lq == 1 && !causal) {
    int sms = 0;
    if (fa::num_sms_of_current_device(&sms) != FA_OK) return FA_ERR_CUDA;
    const int n_split = fa_decode_num_splits(int(BH), Lk, sms);
    const size_t ws_bytes = size_t(n_split) * size_t(BH) * size_t(D + 2) * sizeof(float);
    void* ws = nullptr;
    if (fa::workspace_alloc(&ws, ws_bytes, s) != FA_OK) return FA_ERR_CUDA;
    const int st = fa::launch_decode(q, k, v, o, lse, int(BH), Lk, D, scale, n_split,
                                     static_cast<float*>(ws), s);
    const bool freed = fa::workspace_free(ws, s) == FA_OK;
    if (st != FA_OK) return st;
    return freed ? FA_OK : FA_ERR_CUDA;
  }
  return fa::launch_prefill(q, k, v, o, lse, B, H, Lq, Lk, D, scale, causal, s, err);
}

int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int Lq, int Lk, int D, float scale, int causal, float p_drop,
                   unsigned long long seed, unsigned int offset, void* stream) {
  // ---- host-side checks, before any CUDA call
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Lq <= 0 || Lk <= 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  fa::Dropout dr;
  if (fa::make_dropout(p_drop, seed, offset, &dr) != FA_OK) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (causal && Lq != Lk) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (!fa::aligned(q, 16) || !fa::aligned(k, 16) || !fa::aligned(v, 16) || !fa::aligned(o, 16))
    return FA_ERR_MISALIGNED;
  if (lse != nullptr && !fa::aligned(lse, 4)) return FA_ERR_MISALIGNED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  int* err = fa::error_word_ptr(dev);
  if (err == nullptr) return FA_ERR_CUDA;
  return fa::launch_prefill(q, k, v, o, lse, B, H, Lq, Lk, D, scale, causal, s, err, dr);
}

int fa_last_device_error(void* stream, int* site) {
  if (site != nullptr) *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpyFromSymbol(h, fa::g_device_error, sizeof(h)) != cudaSuccess) return FA_ERR_CUDA;
  if (h[0] != 0) {
    const int zero[2] = {0, 0};
    if (cudaMemcpyToSymbol(fa::g_device_error, zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (site != nullptr) *site = h[1];
  return h[0];  // FA_OK, FA_ERR_TIMEOUT, or FA_ERR_INVALID_ARG (a page id out of range)
}

}  // extern "C"

namespace {

int bwd_common(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
               void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int D, float scale, int causal,
               void* stream, const fa::Dropout& dr) {
  // ---- host-side checks, before any CUDA call
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || dout == nullptr ||
      lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr)
    return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Lq <= 0 || Lk <= 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (causal && Lq != Lk) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  for (const void* ptr : {q, k, v, o, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                          static_cast<const void*>(dv)})
    if (!fa::aligned(ptr, 16)) return FA_ERR_MISALIGNED;
  if (!fa::aligned(lse, 4)) return FA_ERR_MISALIGNED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  int* err = fa::error_word_ptr(dev);
  if (err == nullptr) return FA_ERR_CUDA;
  const size_t lq_pad = (size_t(Lq) + 127) / 128 * 128;
  const size_t ws_bytes = 2 * size_t(BH) * lq_pad * sizeof(float);
  void* ws = nullptr;
  if (fa::workspace_alloc(&ws, ws_bytes, s) != FA_OK) return FA_ERR_CUDA;
  const int st = fa::launch_backward(q, k, v, o, dout, lse, dq, dk, dv, int(BH), Lq, Lk, D, scale,
                                     causal, static_cast<float*>(ws), err, s, dr);
  const bool freed = fa::workspace_free(ws, s) == FA_OK;
  if (st == -2) return FA_ERR_UNSUPPORTED;
  if (st != 0) return FA_ERR_CUDA;
  return freed ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int D,
           float scale, int causal, void* stream) {
  return bwd_common(q, k, v, o, dout, lse, dq, dk, dv, B, H, Lq, Lk, D, scale, causal, stream, fa::Dropout());
}

int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk, int D,
                   float scale, int causal, float p_drop, unsigned long long seed, unsigned int offset,
                   void* stream) {
  fa::Dropout dr;
  if (fa::make_dropout(p_drop, seed, offset, &dr) != FA_OK) return FA_ERR_INVALID_ARG;
  return bwd_common(q, k, v, o, dout, lse, dq, dk, dv, B, H, Lq, Lk, D, scale, causal, stream, dr);
}

int fa_fwd_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                        const int* block_table, const int* seq_lens, void* o, float* lse, int B,
                        int H, int D, int num_pages, int page_size, int max_pages_per_seq,
                        float scale, void* stream) {
  // ---- host-side checks, before any CUDA call
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr ||
      seq_lens == nullptr || o == nullptr)
    return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || D <= 0 || num_pages <= 0 || page_size <= 0 || max_pages_per_seq <= 0)
    return FA_ERR_INVALID_ARG;
  if ((page_size & (page_size - 1)) != 0 || page_size > 65536) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  const long long max_len = (long long)max_pages_per_seq * page_size;
  if (BH > 0x7fffffffLL || max_len > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (!fa::aligned(q, 16) || !fa::aligned(k_cache, 16) || !fa::aligned(v_cache, 16) ||
      !fa::aligned(o, 16))
    return FA_ERR_MISALIGNED;
  if (!fa::aligned(block_table, 4) || !fa::aligned(seq_lens, 4) ||
      (lse != nullptr && !fa::aligned(lse, 4)))
    return FA_ERR_MISALIGNED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  int* err = fa::error_word_ptr(dev);
  if (err == nullptr) return FA_ERR_CUDA;
  int sms = 0;
  if (fa::num_sms_of_current_device(&sms) != FA_OK) return FA_ERR_CUDA;
  // splits sized for the longest sequence the page table can address; a split
  // stages at most 2048 page ids, which short pages can require more splits for
  long long n_split = fa_decode_num_splits(int(BH), int(max_len), sms);
  const long long per_split = 2046LL * page_size;
  if (n_split < (max_len + per_split - 1) / per_split) n_split = (max_len + per_split - 1) / per_split;
  const size_t ws_bytes = size_t(n_split) * size_t(BH) * size_t(D + 2) * sizeof(float);
  void* ws = nullptr;
  if (fa::workspace_alloc(&ws, ws_bytes, s) != FA_OK) return FA_ERR_CUDA;
  const int st = fa::launch_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, H,
                                         D, num_pages, page_size, max_pages_per_seq, scale,
                                         int(n_split), static_cast<float*>(ws), err, s);
  const bool freed = fa::workspace_free(ws, s) == FA_OK;
  if (st == -2) return FA_ERR_UNSUPPORTED;
  if (st != 0) return FA_ERR_CUDA;
  return freed ? FA_OK : FA_ERR_CUDA;
}

int fa_wait_selftest(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 10000000) return FA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  int* err = fa::error_word_ptr(dev);
  if (err == nullptr) return FA_ERR_CUDA;
  // start from a clear error word so the wait runs to its own limit
  const int cleared = fa_last_device_error(stream, nullptr);
  if (cleared == FA_ERR_CUDA) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fa::wait_selftest_kernel<<<1, 32, 0, s>>>(err, (unsigned long long)limit_us * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  return fa_last_device_error(stream, nullptr);
}

}  // extern "C"
