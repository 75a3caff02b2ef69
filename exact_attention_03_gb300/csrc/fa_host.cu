// fa_host.cu - attention on host buffers, with the host<->device copies
// overlapped with the kernels (fa_fwd_host).
//
// Heads are independent problems, so one call is split into chunks of
// consecutive heads (the [B, H, L, D] layout keeps a chunk contiguous) and run
// as a three-stage pipeline: the copies of chunk i+1 into the device run while
// chunk i is computed and the output of chunk i-1 is copied back.  The two
// copy directions use separate copy engines.  Chunks are computed on two
// streams in turn, so that the kernel of one chunk fills the SMs the previous
// chunk's kernel leaves idle (a chunk of a few heads is often less than one
// full wave of CTAs).  The device memory is a ring of three chunk slots kept
// per device across calls, and chunks are numbered across calls, so that
// chunk g uses slot g mod 3 whichever call it belongs to.  Events (one per
// slot and stage) order the stages:
//   copy-in g    after compute g-3 (its input slot is free)
//   compute g    after copy-in g and after copy-out g-3 (its output slot is free)
//   copy-out g   after compute g
// The caller's stream waits for the last copy-out (copy-outs run in order on
// one stream).  fa_fwd_host returns when the outputs are in host memory;
// fa_fwd_host_async returns once the work is queued (complete when `stream`
// reaches that point), so that the copy-in of the next call runs while this
// call computes.  The ring grows (after the work in flight has finished) when
// a call needs larger slots.
#include "fa.h"
#include "fa_internal.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

namespace fa {
namespace {

constexpr int kMaxChunks = 8;
constexpr int kSlots = 3;      // chunk slots of device memory
constexpr int kCompStreams = 2;
constexpr long long kMinChunkBytes = 8ll << 20;   // below this a chunk's copy is latency-bound
constexpr int kMaxDevices = 64;

// per-device copy streams, events and slot ring, created once; queueing a
// call takes the mutex because calls share them
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp[kCompStreams] = {};
  cudaEvent_t in_done[kSlots] = {}, comp_done[kSlots] = {}, out_done[kSlots] = {};
  uint8_t* ring = nullptr;          // kSlots slots of slot_cap bytes
  size_t slot_cap = 0;
  unsigned long long next = 0;      // number of the next chunk
};

HostPipe* host_pipe(int dev) {
  static HostPipe pipes[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  return &pipes[dev];
}

bool init_pipe(HostPipe& p) {
  if (p.ready) return true;
  if (cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) != cudaSuccess) return false;
  for (int i = 0; i < kCompStreams; ++i)
    if (cudaStreamCreateWithFlags(&p.comp[i], cudaStreamNonBlocking) != cudaSuccess) return false;
  for (int i = 0; i < kSlots; ++i)
    if (cudaEventCreateWithFlags(&p.in_done[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.comp_done[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.out_done[i], cudaEventDisableTiming) != cudaSuccess)
      return false;
  p.ready = true;
  return true;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// a ring whose slots hold `slot_bytes`; a larger one is allocated only after
// every chunk in flight has finished with the old one
bool ensure_ring(HostPipe& p, size_t slot_bytes) {
  if (p.ring != nullptr && p.slot_cap >= slot_bytes) return true;
  for (int i = 0; i < kSlots; ++i)
    if (cudaEventSynchronize(p.out_done[i]) != cudaSuccess || cudaEventSynchronize(p.comp_done[i]) != cudaSuccess)
      return false;
  if (cudaStreamSynchronize(p.h2d) != cudaSuccess || cudaStreamSynchronize(p.d2h) != cudaSuccess) return false;
  for (int i = 0; i < kCompStreams; ++i)
    if (cudaStreamSynchronize(p.comp[i]) != cudaSuccess) return false;
  if (p.ring != nullptr && cudaFree(p.ring) != cudaSuccess) return false;
  p.ring = nullptr;
  p.slot_cap = 0;
  void* mem = nullptr;
  if (cudaMalloc(&mem, kSlots * slot_bytes) != cudaSuccess) return false;
  p.ring = static_cast<uint8_t*>(mem);
  p.slot_cap = slot_bytes;
  return true;
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_host_num_chunks(long long BH, long long bytes_per_head) {
  if (BH <= 0 || bytes_per_head <= 0) return 1;
  long long n = BH * bytes_per_head / fa::kMinChunkBytes;   // at least 8 MiB per chunk
  n = std::max(1ll, std::min<long long>(n, fa::kMaxChunks));
  n = std::min(n, BH);
  const long long hc = (BH + n - 1) / n;                      // heads per chunk
  return int((BH + hc - 1) / hc);
}

int fa_fwd_host_async(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                      int Lq, int Lk, int D, float scale, int causal, void* stream) {
  // ---- host-side checks (as fa_fwd), before any CUDA call
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Lq <= 0 || Lk <= 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (causal && Lq != Lk) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;

  const size_t qb = size_t(Lq) * D * 2, kb = size_t(Lk) * D * 2, lb = size_t(Lq) * 4;
  const int n = fa_host_num_chunks(BH, (long long)(2 * qb + 2 * kb + lb));
  const long long hc = (BH + n - 1) / n;
  // one slot: q, k, v, o, lse of hc heads, each part 256-byte aligned
  const size_t oq = 0, ok_ = fa::round_up(oq + hc * qb, 256), ov = fa::round_up(ok_ + hc * kb, 256),
               oo = fa::round_up(ov + hc * kb, 256), ol = fa::round_up(oo + hc * qb, 256),
               slot_bytes = fa::round_up(ol + hc * lb, 256);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  fa::HostPipe* pipe = fa::host_pipe(dev);
  if (pipe == nullptr) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(pipe->mu);
  if (!fa::init_pipe(*pipe)) return FA_ERR_CUDA;

  if (!fa::ensure_ring(*pipe, slot_bytes)) return FA_ERR_CUDA;
  const uint8_t* hq = static_cast<const uint8_t*>(q);
  const uint8_t* hk = static_cast<const uint8_t*>(k);
  const uint8_t* hv = static_cast<const uint8_t*>(v);
  uint8_t* ho = static_cast<uint8_t*>(o);
  uint8_t* hl = reinterpret_cast<uint8_t*>(lse);

  int st = FA_OK;
  auto ok = [&](cudaError_t e) {
    if (e != cudaSuccess && st == FA_OK) st = FA_ERR_CUDA;
    return st == FA_OK;
  };
  for (int i = 0; i < n && st == FA_OK; ++i) {
    const long long h0 = i * hc, nh = std::min(hc, BH - h0);
    const int e = int(pipe->next++ % fa::kSlots);   // slot of this chunk, and of chunk - 3
    uint8_t* slot = pipe->ring + size_t(e) * pipe->slot_cap;
    // copy-in once compute of chunk - 3 (of this or an earlier call) has
    // released the slot's inputs (an event never recorded is complete)
    if (!ok(cudaStreamWaitEvent(pipe->h2d, pipe->comp_done[e], 0))) break;
    if (!ok(cudaMemcpyAsync(slot + oq, hq + h0 * qb, nh * qb, cudaMemcpyHostToDevice, pipe->h2d)) ||
        !ok(cudaMemcpyAsync(slot + ok_, hk + h0 * kb, nh * kb, cudaMemcpyHostToDevice, pipe->h2d)) ||
        !ok(cudaMemcpyAsync(slot + ov, hv + h0 * kb, nh * kb, cudaMemcpyHostToDevice, pipe->h2d)) ||
        !ok(cudaEventRecord(pipe->in_done[e], pipe->h2d)))
      break;
    // compute (heads h0 .. h0+nh-1 as one batch) on the compute streams in
    // turn, once the copy-out of chunk - 3 has read the slot's outputs
    cudaStream_t cs = pipe->comp[(pipe->next - 1) % fa::kCompStreams];
    if (!ok(cudaStreamWaitEvent(cs, pipe->in_done[e], 0))) break;
    if (!ok(cudaStreamWaitEvent(cs, pipe->out_done[e], 0))) break;
    const int r = fa_fwd(slot + oq, slot + ok_, slot + ov, slot + oo,
                         lse != nullptr ? reinterpret_cast<float*>(slot + ol) : nullptr, 1, int(nh), Lq, Lk,
                         D, scale, causal, cs);
    if (r != FA_OK) {
      st = r;
      break;
    }
    if (!ok(cudaEventRecord(pipe->comp_done[e], cs))) break;
    // copy-out
    if (!ok(cudaStreamWaitEvent(pipe->d2h, pipe->comp_done[e], 0))) break;
    if (!ok(cudaMemcpyAsync(ho + h0 * qb, slot + oo, nh * qb, cudaMemcpyDeviceToHost, pipe->d2h))) break;
    if (lse != nullptr && !ok(cudaMemcpyAsync(hl + h0 * lb, slot + ol, nh * lb, cudaMemcpyDeviceToHost, pipe->d2h)))
      break;
    if (!ok(cudaEventRecord(pipe->out_done[e], pipe->d2h))) break;
  }
  if (st == FA_OK) {
    // the caller's stream reaches the end of this call once the last
    // copy-out has landed (copy-outs run in order on one stream)
    ok(cudaStreamWaitEvent(s, pipe->out_done[(pipe->next - 1) % fa::kSlots], 0));
  } else {
    // a failed call leaves nothing in flight
    cudaStreamSynchronize(pipe->h2d);
    for (int i = 0; i < fa::kCompStreams; ++i) cudaStreamSynchronize(pipe->comp[i]);
    cudaStreamSynchronize(pipe->d2h);
    cudaStreamSynchronize(s);
  }
  return st;
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Lq, int Lk, int D, float scale, int causal, void* stream) {
  const int st = fa_fwd_host_async(q, k, v, o, lse, B, H, Lq, Lk, D, scale, causal, stream);
  if (st != FA_OK) return st;
  return cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
