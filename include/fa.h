/*
 * fa.h - C ABI of the GB300 (sm_103a) exact-attention library: the forward
 * pass (with optional dropout), single-query decode over a dense or paged
 * cache, the backward pass and a standalone row softmax.
 *
 * The library computes exact scaled-dot-product attention
 *
 *     O = softmax(scale * Q K^T [+ causal mask]) V,   LSE = ln sum_j exp(scale * q.k_j)
 *
 * in one pass over K/V tiles, with the online-softmax recurrence derived in
 * "NTU Hung-yi Lee ML 2026 Guide: Faster Generation, Part 1: Flash Attention"
 * (quidproquo.cc), sections "Mechanism: run with the wrong answer, then
 * correct it", "Expand: why multiplying by exp(d1 - d2) fixes it" and
 * "Expand: the correction for the output O": a running maximum d, a running
 * denominator s rescaled by exp(d_old - d_new), and a running output rescaled
 * the same way, so that the attention weights are never written to memory
 * ("Back to real models": no attention weights are returned).  The per-row
 * statistics m (max) and l (sum) are those of "6.3 FlashAttention"
 * (comfyai.app), "How FlashAttention Works"; LSE = m + ln l is exported as
 * their natural-log summary.
 *
 * Every entry point is a plain C function: pointers, sizes and a status
 * code.  No entry point takes or returns a PyTorch or C++ type.
 *
 * Per-device state: on first use on a device the library looks up the device
 * addresses of its own device arrays (the error word, the array of
 * fa_fwd_decode_noalloc) and creates its workspace pool, and keeps them until
 * the process exits.  They belong to the device's primary context, so the
 * library must not be used on a device after cudaDeviceReset (or any other
 * reset of that context) in the same process.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (returned by every entry point). */
typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1,  /* null pointer, non-positive size, non-finite or non-positive scale */
  FA_ERR_UNSUPPORTED = -2,  /* valid but not implemented: head dim not in {64,128}, causal with Lq != Lk, size limits */
  FA_ERR_MISALIGNED = -3,   /* q, k, v or o not 16-byte aligned, or lse not 4-byte aligned */
  FA_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed (no device, launch failure, ...) */
  FA_ERR_TIMEOUT = -5       /* a device-side wait gave up (reported by fa_last_device_error) */
} fa_status;

/*
 * fa_fwd - attention forward pass on the GPU.
 *
 * q     : device pointer, bf16, [B, H, Lq, D], contiguous (row-major, D fastest).
 * k, v  : device pointers, bf16, [B, H, Lk, D], contiguous.
 * o     : device pointer, bf16, [B, H, Lq, D], contiguous; written.
 * lse   : device pointer, fp32, [B, H, Lq]; written with the natural-log
 *         log-sum-exp of the scaled scores of each query row; may be NULL.
 * B, H  : batch size and number of heads (each head attends independently).
 * Lq, Lk: number of query and key/value positions (>= 1).
 * D     : head dimension, 64 or 128.
 * scale : score scale (typically 1/sqrt(D)); finite and > 0.
 * causal: 0 = every key visible; 1 = key j visible to query i iff j <= i
 *         (requires Lq == Lk).
 * stream: the cudaStream_t to enqueue on (NULL = legacy default stream).
 *
 * Ownership: the caller owns every buffer; the library keeps no pointer after
 * the call returns.  The single-query path (Lq == 1, non-causal) splits the
 * keys over many thread blocks and needs a workspace of
 * n_split * B * H * (D + 2) * 4 bytes, allocated and freed stream-ordered on
 * `stream` from a memory pool the library creates per device
 * (cudaMemPoolCreate; the pool keeps freed memory for later calls, so that a
 * call after a synchronisation does not map new memory, and lives until the
 * process ends).
 *
 * Errors: arguments are checked on the host before any CUDA call, and a bad
 * argument returns FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED / FA_ERR_MISALIGNED
 * without touching the GPU.  A failing CUDA call returns FA_ERR_CUDA.
 * Like any kernel launch the call is asynchronous: FA_OK means "enqueued".
 * Device-side waits are bounded; one that gives up records FA_ERR_TIMEOUT,
 * readable with fa_last_device_error.  q/k/v must not alias o or lse.
 * Thread safety: reentrant; calls on different streams may overlap.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int Lq, int Lk, int D, float scale, int causal,
           void* stream);

/*
 * fa_strerror - static, NUL-terminated description of a status code.
 * Never returns NULL; unknown codes give "unknown fa_status".
 */
const char* fa_strerror(int status);

/*
 * fa_last_device_error - synchronises `stream`, then reads and clears the
 * library's device error word on the current device.  Returns FA_OK when
 * nothing was recorded since the last call, FA_ERR_TIMEOUT when a device-side
 * wait gave up, FA_ERR_INVALID_ARG when fa_fwd_decode_paged met a page id
 * outside its cache (FA_ERR_CUDA if the synchronisation itself fails); the
 * first event recorded wins.  If `site` is not NULL it receives an identifier
 * of where it happened (0 when none).
 */
int fa_last_device_error(void* stream, int* site);

/*
 * fa_decode_num_splits - the number of key splits the single-query path uses
 * for a problem of B*H heads with Lk keys on a GPU with `num_sms` SMs
 * (host-only arithmetic; no CUDA call).  Returns >= 1, or FA_ERR_INVALID_ARG.
 */
int fa_decode_num_splits(int BH, int Lk, int num_sms);

/*
 * fa_wait_selftest - launches one block whose single thread waits on a
 * shared-memory barrier that nothing ever completes, with a wait limit of
 * `limit_us` microseconds (1..10,000,000).  The wait must give up, record
 * FA_ERR_TIMEOUT in the device error word and return.  The call synchronises
 * `stream` and returns what fa_last_device_error then reads (FA_ERR_TIMEOUT
 * when the bounded wait works).  It exercises the same bounded-wait routine
 * the attention kernels use, without faulting or hanging the GPU.
 */
int fa_wait_selftest(int limit_us, void* stream);

/*
 * fa_fwd_decode_noalloc - single-query attention (Lq = 1, non-causal) that
 * allocates no memory.  The pages describe no such variant; it exists for
 * callers that cannot allocate device memory while they run (an engine that
 * plans all memory before serving, a plugin inside a framework-owned memory
 * budget, a latency-critical loop where a memory-pool growth would stall).
 *
 * Arguments mean what they mean for fa_fwd with Lq = 1: q, o bf16 [B, H, 1, D],
 * k, v bf16 [B, H, Lk, D], lse fp32 [B, H, 1] (may be NULL), D in {64, 128},
 * finite scale > 0, all device pointers owned by the caller.
 *
 * Instead of a per-call workspace it uses one device array of
 * fa_decode_noalloc_max_floats() floats (4 MiB) that the library reserves on
 * every GPU that loads it, until the process exits.  B * H * (D + 2) must fit
 * in it (B * H <= 8065 at D = 128), else FA_ERR_UNSUPPORTED is returned before
 * any CUDA call; within that limit the number of key splits is capped so that
 * the partial results fit.  No cudaMalloc/cudaFree or allocating library call
 * is made.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * All calls share the array: calls whose kernels overlap on the GPU (other
 * streams, other host threads) race on it and must be serialised by the
 * caller.  The array keeps the last call's contents; every slot a call reads
 * is written by the same call first, so nothing needs clearing.  When the
 * split count fa_fwd would use fits in the array, the results are bit for bit
 * those of fa_fwd.  The cached address assumes the device's context is never
 * reset (see "Per-device state" above).
 * Errors: as fa_fwd.
 */
int fa_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int H, int Lk, int D, float scale, void* stream);

/* fa_decode_noalloc_max_floats - size, in floats, of fa_fwd_decode_noalloc's array. */
int fa_decode_noalloc_max_floats(void);

/*
 * fa_fwd_decode_paged - single-query attention (one query row per head,
 * non-causal) against a paged key/value cache with a length per sequence:
 * the decode step of generation over a cache that grows page by page.  The
 * lecture leaves the cache's layout to its next part; this one is the plainest
 * paged form.  For every sequence b and head h it computes what fa_fwd
 * computes for q[b, h] against the seq_lens[b] cached positions of that
 * sequence, in order:
 *   position p of sequence b sits in page block_table[b * max_pages_per_seq +
 *   p / page_size], row p % page_size of that page.
 *
 * q        : device, bf16, [B, H, D] (= [B, H, 1, D]), contiguous.
 * k_cache, v_cache : device, bf16, [num_pages, page_size, H, D], contiguous
 *            (within a page: position-major, then head, then D).
 * block_table : device, int32, [B, max_pages_per_seq]; entries past a
 *            sequence's last page are not read.  An entry that is read and is
 *            outside [0, num_pages) is recorded in the device error word
 *            (FA_ERR_INVALID_ARG, see fa_last_device_error) and that page's
 *            keys are left out; nothing is read out of bounds.
 * seq_lens : device, int32, [B]; values are clamped to
 *            [0, max_pages_per_seq * page_size].  A sequence of length 0 gets
 *            O = 0 and LSE = -inf.
 * o, lse   : bf16 [B, H, D] and fp32 [B, H] (lse may be NULL), written.
 * page_size: a power of two, 1 .. 65536.  D in {64, 128}; finite scale > 0.
 *
 * Workspace: n_split * B * H * (D + 2) * 4 bytes from the library's pool
 * (see fa_fwd), n_split as fa_decode_num_splits for Lk = max_pages_per_seq *
 * page_size, raised where one split would span more than 2046 pages.
 * Errors and asynchrony as for fa_fwd (q, k_cache, v_cache, o 16-byte aligned;
 * block_table, seq_lens, lse 4-byte aligned).
 */
int fa_fwd_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                        const int* block_table, const int* seq_lens, void* o, float* lse,
                        int B, int H, int D, int num_pages, int page_size,
                        int max_pages_per_seq, float scale, void* stream);

/*
 * fa_softmax_rows - softmax of every row of a matrix, in two reads: the guide's
 * "Expand: why multiplying by exp(d1 - d2) fixes it" (a running maximum d and
 * a running sum s rescaled by exp(d_old - d_new) find Amax and the denominator
 * in one read; a second read writes exp(a_i - Amax) / S).
 *
 * x    : device, fp32, [rows, cols], row-major; values finite or -inf.
 * y    : device, fp32, [rows, cols]; written with the row softmax of x (may be
 *        x itself: each element is read before it is written, in place).
 * lse  : device, fp32, [rows]; written with ln(sum_j exp(x_ij)) (may be NULL).
 *        A row of only -inf gets y = 0 and lse = -inf.
 * rows >= 1, cols >= 1, rows * cols <= 2^40.  4-byte aligned pointers (16-byte
 * aligned rows are read and written with vector accesses).
 * Errors and asynchrony as for fa_fwd.
 */
int fa_softmax_rows(const float* x, float* y, float* lse, long long rows, int cols,
                    void* stream);

/*
 * fa_bwd - attention backward pass with recomputation ("6.3 FlashAttention",
 * "A simple implementation w/ C++": the weights are not saved by the forward
 * pass but recomputed here).  Computes the gradients of <dout, O> with respect
 * to q, k and v, where O = softmax(scale q k^T [causal]) v is fa_fwd's output:
 * dv = P^T dout, dq = scale dS k, dk = scale dS^T q with
 * P = exp(scale q k^T - lse), dS = P * (dout v^T - rowsum(dout * O)).
 *
 * q, o, dout : device, bf16, [B, H, Lq, D]; k, v: [B, H, Lk, D] (contiguous).
 *              o is fa_fwd's output for these q, k, v, scale and causal flag.
 * lse        : device, fp32, [B, H, Lq]: fa_fwd's log-sum-exp (natural log).
 * dq, dk, dv : device, bf16, shaped like q, k, v; written.
 * Argument rules as for fa_fwd (D in {64, 128}, causal needs Lq == Lk; every
 * bf16 pointer 16-byte aligned, lse 4-byte aligned).  Workspace:
 * 2 * B * H * roundup(Lq, 128) * 4 bytes from the library's pool (see fa_fwd).
 * Errors and asynchrony as for fa_fwd.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk,
           int D, float scale, int causal, void* stream);

/*
 * fa_bwd_dropout - backward pass of fa_fwd_dropout: the gradients of
 * <dout, O> with respect to q, k and v, where O is fa_fwd_dropout's output for
 * the same q, k, v, scale, causal flag, p_drop, seed and offset.  The keep
 * bits are drawn again from the same contract (see fa_fwd_dropout), so no
 * mask is stored between the two passes.  With z the keep mask and
 * s = 256 / (256 - t):
 *   dv = s (P * z)^T dout,   dP = s z * (dout v^T),
 *   dS = P * (dP - rowsum(dout * O)),   dq = scale dS k,   dk = scale dS^T q
 * (P = exp(scale q k^T - lse); the gradient of a dropped weight is zero).
 *
 * Arguments as for fa_bwd (o and lse: fa_fwd_dropout's outputs) and
 * p_drop, seed, offset as for fa_fwd_dropout; p_drop = 0 gives fa_bwd's
 * results.  Errors and asynchrony as for fa_fwd.
 */
int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk,
                   int D, float scale, int causal, float p_drop, unsigned long long seed,
                   unsigned int offset, void* stream);

/*
 * fa_fwd_dropout - fa_fwd with dropout on the attention weights, fused into the
 * kernel ("6.3 FlashAttention", section "6.3.3 FlashAttention Forward
 * Process", "Kernel Fusion": scale -> mask -> softmax -> dropout -> matrix
 * product, all on one tile in on-chip memory).  The pages give no random
 * number contract; this library's is:
 *   t = floor(256 * p_drop + 0.5) (in double precision), 0 <= t <= 255;
 *   key j of query row i in head bh = b * H + h takes byte (j mod 4) of word
 *   ((j div 4) mod 4) of Philox-4x32-10 (Salmon et al., SC 2011) with
 *   counter (j div 16, i, bh, offset) and key (seed mod 2^32, seed div 2^32),
 *   and is kept iff that byte >= t;
 *   O = ((w * keep) v) * 256 / (256 - t), w = the softmax weights;
 *   lse = the undropped log-sum-exp (exactly fa_fwd's).
 * Same arguments and rules as fa_fwd, plus p_drop in [0, 1) with t <= 255
 * (else FA_ERR_INVALID_ARG), seed and offset.  Every shape, Lq == 1 included,
 * runs on the prefill kernels.  Errors and asynchrony as for fa_fwd.
 */
int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int Lq, int Lk, int D, float scale, int causal, float p_drop,
                   unsigned long long seed, unsigned int offset, void* stream);

/*
 * fa_fwd_host - fa_fwd on HOST buffers: q, k, v are read from and o, lse
 * written to host memory (page-locked memory gives the full copy bandwidth;
 * pageable memory works, slower).  The heads are split into up to 8 chunks of
 * consecutive heads (at least 8 MiB of copies each, fa_host_num_chunks), and
 * the copies of one chunk overlap the computation of the next: copy-in,
 * compute and copy-out run on internal streams (one per copy direction, and
 * two compute streams taken in turn, so that one chunk's kernel fills the SMs
 * the previous chunk's kernel leaves idle), ordered by events, over a ring of
 * three chunk slots of device memory the library keeps per device (grown when
 * a call needs larger slots, after the work in flight); `stream` waits for the
 * last copy-out.  The inputs are read as they are when the call is made (the
 * copy-in is not ordered after work queued earlier on `stream`).  Same
 * argument rules as fa_fwd (lse may be NULL; host pointers have no alignment
 * rule).  The call returns after the outputs are in host memory.  Calls on one
 * device share the internal streams (queueing a call takes a per-device lock).
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Lq, int Lk, int D, float scale, int causal, void* stream);

/*
 * fa_fwd_host_async - fa_fwd_host without the final synchronisation: returns
 * once the copies and kernels are queued; the outputs are in host memory when
 * `stream` has reached the point after this call (cudaStreamSynchronize, or an
 * event recorded on it).  The host buffers must stay valid until then.  The
 * copy-in of a following call runs while this call computes, so a sequence of
 * calls followed by one synchronisation overlaps their copies and kernels.
 */
int fa_fwd_host_async(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Lq, int Lk, int D, float scale, int causal, void* stream);

/* fa_host_num_chunks - the number of head chunks fa_fwd_host uses for BH heads
 * of bytes_per_head copied bytes each: min(8, BH, BH * bytes_per_head / 8 MiB),
 * at least 1, then rounded so that every chunk but the last has the same
 * number of heads. */
int fa_host_num_chunks(long long BH, long long bytes_per_head);

/* fa_abi_version - (major << 16) | minor of this header's ABI. */
int fa_abi_version(void);

#define FA_ABI_VERSION ((1 << 16) | 6)

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
