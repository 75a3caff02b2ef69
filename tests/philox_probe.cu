// philox_probe.cu - test-only probe: runs the attention library's device
// Philox-4x32-10 (exact_attention_03_gb300/csrc/philox.cuh) on counters and
// keys given by the host, so that a test can compare its words bit for bit
// with the CPU oracle's.  Built by tests/test_philox_gpu.py into _build/; not
// part of the library.
#include <cstdint>
#include <cuda_runtime.h>

#include "philox.cuh"

namespace {

// in: n records of 6 words (c0, c1, c2, c3, k0, k1); out: n records of 4 words
__global__ void philox_probe_kernel(const uint32_t* in, uint32_t* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* r = in + 6 * size_t(i);
  const uint4 w = fa::philox4x32_10(make_uint4(r[0], r[1], r[2], r[3]), r[4], r[5]);
  uint32_t* o = out + 4 * size_t(i);
  o[0] = w.x;
  o[1] = w.y;
  o[2] = w.z;
  o[3] = w.w;
}

}  // namespace

// Host buffers in and out; returns 0 or the CUDA error code.
extern "C" int philox_probe(const uint32_t* in_host, uint32_t* out_host, int n) {
  if (n <= 0 || in_host == nullptr || out_host == nullptr) return -1;
  uint32_t* d_in = nullptr;
  uint32_t* d_out = nullptr;
  cudaError_t e = cudaMalloc(&d_in, size_t(n) * 6 * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMalloc(&d_out, size_t(n) * 4 * sizeof(uint32_t));
  if (e == cudaSuccess)
    e = cudaMemcpy(d_in, in_host, size_t(n) * 6 * sizeof(uint32_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    philox_probe_kernel<<<(n + 127) / 128, 128>>>(d_in, d_out, n);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess)
    e = cudaMemcpy(out_host, d_out, size_t(n) * 4 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
  cudaFree(d_in);
  cudaFree(d_out);
  return int(e);
}
