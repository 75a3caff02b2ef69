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

// the paired form: records 2m and 2m+1 share record 2m's key
__global__ void philox_probe_x2_kernel(const uint32_t* in, uint32_t* out, int npairs) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= npairs) return;
  const uint32_t* r = in + 12 * size_t(m);
  uint4 a = make_uint4(r[0], r[1], r[2], r[3]);
  uint4 b = make_uint4(r[6], r[7], r[8], r[9]);
  fa::philox4x32_10_x2(a, b, r[4], r[5]);
  uint32_t* o = out + 8 * size_t(m);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// the row routines: record i's counter (x, i, bh, offset) through philox_row
__global__ void philox_probe_row_kernel(const uint32_t* in, uint32_t* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* r = in + 6 * size_t(i);
  const fa::PhiloxRow R = fa::philox_row(r[1], r[2], r[3], r[4], r[5]);
  const uint4 w = fa::philox4x32_10_row(r[0], R, fa::philox_round_keys(r[4], r[5]));
  uint32_t* o = out + 4 * size_t(i);
  o[0] = w.x; o[1] = w.y; o[2] = w.z; o[3] = w.w;
}

// records 2m and 2m+1 share words 1-3 and the key of record 2m
__global__ void philox_probe_row_x2_kernel(const uint32_t* in, uint32_t* out, int npairs) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= npairs) return;
  const uint32_t* r = in + 12 * size_t(m);
  const fa::PhiloxRow R = fa::philox_row(r[1], r[2], r[3], r[4], r[5]);
  uint4 a, b;
  fa::philox4x32_10_row_x2(r[0], r[6], R, fa::philox_round_keys(r[4], r[5]), a, b);
  uint32_t* o = out + 8 * size_t(m);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// the column routine: record i's counter (x, i, bh, offset) through philox_col
// (x, head, offset and key fixed per column of keys, the query row varying)
__global__ void philox_probe_col_kernel(const uint32_t* in, uint32_t* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* r = in + 6 * size_t(i);
  const fa::PhiloxCol C = fa::philox_col(r[0], r[2], r[3], r[4], r[5]);
  const uint4 w = fa::philox4x32_10_col(r[1], C, fa::philox_round_keys(r[4], r[5]));
  uint32_t* o = out + 4 * size_t(i);
  o[0] = w.x; o[1] = w.y; o[2] = w.z; o[3] = w.w;
}

// the keep masks of the dropout kernels: record i = (word, t, -, -, -, -);
// out = (mask of keys 0-1, mask of keys 2-3, -, -)
__global__ void keep_mask_probe_kernel(const uint32_t* in, uint32_t* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* r = in + 6 * size_t(i);
  const uint32_t t = r[1];
  const uint32_t keep = fa::dropout_keep_msb(r[0], (t & 0x7fu) * 0x01010101u, t >= 128u ? 0xffffffffu : 0u);
  uint32_t* o = out + 4 * size_t(i);
  o[0] = fa::dropout_pair_mask(keep, 0);
  o[1] = fa::dropout_pair_mask(keep, 1);
  o[2] = 0;
  o[3] = 0;
}

// the per-key keep masks: record i = (word, t, -, -, -, -); out = the 32-bit
// masks of keys 0, 1, 2, 3
__global__ void byte_mask_probe_kernel(const uint32_t* in, uint32_t* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* r = in + 6 * size_t(i);
  const uint32_t t = r[1];
  const uint32_t keep = fa::dropout_keep_msb(r[0], (t & 0x7fu) * 0x01010101u, t >= 128u ? 0xffffffffu : 0u);
  uint32_t* o = out + 4 * size_t(i);
  o[0] = fa::dropout_byte_mask(keep, 0);
  o[1] = fa::dropout_byte_mask(keep, 1);
  o[2] = fa::dropout_byte_mask(keep, 2);
  o[3] = fa::dropout_byte_mask(keep, 3);
}

}  // namespace

// Host buffers in and out; returns 0 or the CUDA error code.  mode: 0 = the
// single routine, 1 = the paired routine (n even; records 2m, 2m+1 under
// record 2m's key), 2 = the row routine, 3 = the paired row routine (records
// 2m, 2m+1 share words 1-3 and the key), 4 = the dropout keep masks, 5 = the
// column routine, 6 = the per-key keep masks.
extern "C" int philox_probe(const uint32_t* in_host, uint32_t* out_host, int n, int mode) {
  if (n <= 0 || in_host == nullptr || out_host == nullptr || mode < 0 || mode > 6) return -1;
  const bool pairs = (mode == 1 || mode == 3);
  if (pairs && (n & 1)) return -1;
  uint32_t* d_in = nullptr;
  uint32_t* d_out = nullptr;
  cudaError_t e = cudaMalloc(&d_in, size_t(n) * 6 * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMalloc(&d_out, size_t(n) * 4 * sizeof(uint32_t));
  if (e == cudaSuccess)
    e = cudaMemcpy(d_in, in_host, size_t(n) * 6 * sizeof(uint32_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    if (mode == 1)
      philox_probe_x2_kernel<<<(n / 2 + 127) / 128, 128>>>(d_in, d_out, n / 2);
    else if (mode == 3)
      philox_probe_row_x2_kernel<<<(n / 2 + 127) / 128, 128>>>(d_in, d_out, n / 2);
    else if (mode == 2)
      philox_probe_row_kernel<<<(n + 127) / 128, 128>>>(d_in, d_out, n);
    else if (mode == 6)
      byte_mask_probe_kernel<<<(n + 127) / 128, 128>>>(d_in, d_out, n);
    else if (mode == 5)
      philox_probe_col_kernel<<<(n + 127) / 128, 128>>>(d_in, d_out, n);
    else if (mode == 4)
      keep_mask_probe_kernel<<<(n + 127) / 128, 128>>>(d_in, d_out, n);
    else
      philox_probe_kernel<<<(n + 127) / 128, 128>>>(d_in, d_out, n);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess)
    e = cudaMemcpy(out_host, d_out, size_t(n) * 4 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
  cudaFree(d_in);
  cudaFree(d_out);
  return int(e);
}
