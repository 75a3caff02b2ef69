// fa_decode_noalloc.cu - single-query attention that allocates no memory.
//
// fa_fwd runs the single-query (Lq == 1) path with a split-K/V workspace it
// allocates stream-ordered for every call.  Some callers cannot allocate while
// they run: an engine that plans all device memory before serving and treats
// any allocation during a request as an error, a plugin that must stay inside
// a memory budget owned by its host framework, or a latency-critical loop in
// which a memory-pool growth (a driver call) would be a stall.
// fa_fwd_decode_noalloc serves them: it runs the same split-K/V and combine
// kernels, but their workspace is a fixed-size array in device memory that
// the library reserves when it is loaded (kScratchFloats floats, 4 MiB, held
// on every GPU that loads the library until the process exits).
#include "fa.h"
#include "fa_internal.h"

#include <cmath>
#include <cstdint>
#include <mutex>

namespace fa {
namespace {

// (n_split x B x H) partial rows of D + 2 floats live here.  Every call
// overwrites every slot it reads, so nothing needs clearing between calls.
constexpr size_t kScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;

// Device address of g_decode_scratch on the current device, looked up once per
// device (the host-side name is only a stand-in for the device array).
float* scratch_ptr(int dev) {
  static std::mutex mu;
  static float* cached[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<float*>(ptr);
  }
  return cached[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace fa

extern "C" int fa_decode_noalloc_max_floats(void) { return int(fa::kScratchFloats); }

extern "C" int fa_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                     float* lse, int B, int H, int Lk, int D, float scale,
                                     void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Lk <= 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  const long long row_floats = BH * (D + 2);  // one split's partial results
  if (row_floats > (long long)fa::kScratchFloats) return FA_ERR_UNSUPPORTED;
  if (!fa::aligned(q, 16) || !fa::aligned(k, 16) || !fa::aligned(v, 16) || !fa::aligned(o, 16))
    return FA_ERR_MISALIGNED;
  if (lse != nullptr && !fa::aligned(lse, 4)) return FA_ERR_MISALIGNED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  float* scratch = fa::scratch_ptr(dev);
  if (scratch == nullptr) return FA_ERR_CUDA;
  int sms = 0;
  if (fa::num_sms_of_current_device(&sms) != FA_OK) return FA_ERR_CUDA;

  // as many splits as fa_fwd would use, but no more than the scratch holds
  long long n = fa_decode_num_splits(int(BH), Lk, sms);
  const long long cap = (long long)fa::kScratchFloats / row_floats;
  if (n > cap) n = cap;
  const long long chunk = (Lk + n - 1) / n;
  n = (Lk + chunk - 1) / chunk;  // no empty split
  return fa::launch_decode(q, k, v, o, lse, int(BH), Lk, D, scale, int(n), scratch,
                           static_cast<cudaStream_t>(stream));
}
