// fa_internal.h - host-side launchers shared between the C-ABI translation
// unit and the kernel translation units (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Wait-site identifiers recorded in the device error word when a bounded wait gives up.
enum WaitSite : int {
  kSiteNone = 0,
  kSiteProducerEmpty = 1,
  kSiteMmaQ = 2,
  kSiteMmaK = 3,
  kSiteMmaV = 4,
  kSiteMmaP = 5,
  kSiteSoftmaxS = 6,
  kSiteSoftmaxO = 7,
  kSiteSelftest = 8,
  kSiteMmaS = 9,
  kSiteSoftmaxGo = 10,
  kSitePageTable = 11,  // not a wait: a page id outside the paged cache (FA_ERR_INVALID_ARG)
};

// Dropout on the attention weights (fa_fwd_dropout); `on` = 0 is the plain
// forward.  Bits from the Philox contract in philox.cuh: a key is kept iff its
// byte >= t, and O is scaled by keep_scale = 256 / (256 - t).
struct Dropout {
  int on = 0;
  uint32_t seed_lo = 0, seed_hi = 0, offset = 0;
  uint32_t t = 0;
  float keep_scale = 1.f;
};

// The dropout contract from the C ABI's arguments (FA_OK or FA_ERR_INVALID_ARG).
int make_dropout(float p_drop, unsigned long long seed, unsigned int offset, Dropout* dr);

// Prefill / general path (any Lq, tcgen05 kernel).  Arguments already validated.
int launch_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int Lq, int Lk, int D, float scale, int causal, cudaStream_t stream, int* err,
                   const Dropout& dr = Dropout());

// Head dimension 64 (Lq >= 1): separate P buffer, one MMA issuer per query tile,
// the two query tiles' softmax groups half an iteration apart.  Runs the
// dropout forward itself and hands the plain forward to launch_prefill_d64x1.
int launch_prefill_d64(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int Lq, int Lk, float scale, int causal, cudaStream_t stream,
                       int* err, const Dropout& dr = Dropout());

// Head dimension 128: the weights P in tensor memory, one S buffer shared by
// the CTA's two query tiles, one MMA-issuing thread per query tile.
int launch_prefill_d128(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int Lq, int Lk, float scale, int causal, cudaStream_t stream,
                        int* err, const Dropout& dr = Dropout());

// Head dimension 64, one query tile per CTA and two CTAs per SM (twice the
// work units of launch_prefill_d64, each half the size).
int launch_prefill_d64x1(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int Lq, int Lk, float scale, int causal, cudaStream_t stream,
                         int* err, const Dropout& dr = Dropout());

// Single-query split-K/V path (Lq == 1).  Arguments already validated.
// `workspace` must hold n_split * B * H * (D + 2) floats.
int launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, int BH,
                  int Lk, int D, float scale, int n_split, float* workspace, cudaStream_t stream);

// Single-query attention over a paged cache (fa_fwd_decode_paged): arguments
// already validated; `workspace` holds n_split * B * H * (D + 2) floats; `err`
// is the device error word.  Returns 0, -2 (a split would need more than 2048
// page-table entries) or -4.
int launch_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                        const int* block_table, const int* seq_lens, void* o, float* lse, int B,
                        int H, int D, int num_pages, int page_size, int max_pages, float scale,
                        int n_split, float* workspace, int* err, cudaStream_t stream);

// Backward pass (fa_bwd): arguments already validated; `workspace` holds
// 2 * BH * roundup(Lq, 128) floats.  Returns 0, -2 or -4 (or a tensor-map error).
// With dr.on, the backward of fa_fwd_dropout's forward (the same keep bits).
int launch_backward(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, int BH, int Lq, int Lk, int D,
                    float scale, int causal, float* workspace, int* err, cudaStream_t stream,
                    const Dropout& dr = Dropout());

int num_sms_of_current_device(int* num_sms);

// The device error word of device `dev` ([0] status, [1] wait site), whose
// address the library looks up once per device; nullptr on failure.
int* error_word_ptr(int dev);

// Grid order for work in tiles of whole heads: heads in groups of `group`, all
// tiles of a group before the next group, so that the CTAs resident at one
// time share a few heads' K/V (or Q/dO) in L2 instead of streaming every
// head's from HBM; within a group, rank 0 of every head first, then rank 1,
// ... (rank 0 = the most work when causal).  A bijection of [0, BH * ntiles)
// onto (rank, bh).
struct TileOrder {
  int rank, bh;
};
__host__ __device__ inline TileOrder grouped_tile_order(long long block, int BH, int ntiles, int group) {
  const int full = BH / group * group;   // heads in whole groups
  const long long in_full = (long long)full * ntiles;
  TileOrder t;
  if (block < in_full) {
    const long long per = (long long)group * ntiles;
    const int grp = int(block / per);
    const int idx = int(block - grp * per);
    t.rank = idx / group;
    t.bh = grp * group + idx % group;
  } else {
    const int rest = BH - full;
    const int idx = int(block - in_full);
    t.rank = idx / rest;
    t.bh = full + idx % rest;
  }
  return t;
}
// Heads per group: as many as keep `bytes_per_head` of streamed tiles within
// FA_L2_GROUP_BUDGET_MB (default 24 MB; 24 to 48 MB measured best for
// causal 64K and the D = 64 sweep lengths, against one group of all heads),
// at least one.
#ifndef FA_L2_GROUP_BUDGET_MB
#define FA_L2_GROUP_BUDGET_MB 24
#endif
inline int l2_head_group(int BH, long long bytes_per_head) {
  const long long budget = (long long)FA_L2_GROUP_BUDGET_MB << 20;
  long long g = bytes_per_head > 0 ? budget / bytes_per_head : BH;
  if (g < 1) g = 1;
  if (g > BH) g = BH;
  return int(g);
}

// Workspace memory, stream-ordered on `stream`, from the library's pool of the
// current device (kept between calls).  Return FA_OK or FA_ERR_CUDA.
int workspace_alloc(void** ptr, size_t bytes, cudaStream_t stream);
int workspace_free(void* ptr, cudaStream_t stream);

// TMA tensor map over a [BH, L, D] bf16 tensor, viewed as {64, L, D/64, BH}: one
// box is a 128-row tile of one head (D/64 swizzled blocks of 128 rows x 128 B),
// rows past L read as zeros.  Returns 0 or FA_ERR_CUDA.
int make_tensor_map_bf16(CUtensorMap* map, const void* ptr, int BH, int L, int D);

}  // namespace fa
