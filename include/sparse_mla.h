/*
 * sparse_mla.h -- C ABI of libsparse_mla.so, the token-sparse MLA attention
 * forward for GB300 (sm_103a).
 *
 * What the library computes.  Each query token t has h heads of 576-dim bf16
 * queries (512 latent + 64 rope dims) and its own list of `topk` int32 slot
 * indices into a paged compact latent KV cache (one KV head, 576 dims per
 * row).  For every head:
 *     s_j    = scale * <q[t,h,:], kv[idx[t,j], :]>            (all 576 dims)
 *     P      = softmax over the valid j (idx in [0, num_slots); -1 = invalid)
 *     O[t,h] = sum_j P_j * kv[idx[t,j], 0:512]                (V = latent part)
 *     LSE    = ln sum_j exp(s_j)                              (natural log, fp32)
 * An index list with no valid entry gives O = 0 and LSE = -inf.  Each list
 * entry is a separate softmax term (a slot listed twice counts twice).
 * sparse_mla_merge combines the (O, LSE) of lists split into parts, e.g. over
 * decode-context-parallel ranks, into the result of the whole lists,
 * sparse_mla_v_up applies the per-head value up-projection to O, and
 * sparse_mla_topk builds the index lists from per-position scores.
 *
 * Sources (page title, section):
 *   vLLM PR #60220 "FlashMLA sparse: stage fp8 mixed-batch q/out in the
 *   workspace" -- Claims: q is T x heads x 576 bf16, out is T x heads x 512 bf16
 *   and is passed in by the caller (out=); Details: the kernel returns lse and
 *   should not allocate per call (o_accum, q padding).
 *   vLLM PR #64510 "Enable existing native 8/16/32-head kernels in SM90 BF16
 *   sparse FlashMLA" -- Overview/Details: 8, 16 and 32 heads per rank run
 *   natively instead of being padded to 64; padding, when wanted, is the
 *   caller's (zero heads whose outputs are discarded).
 *   PR #55738 report, 功能与动机 (motivation): the "per-token top-k MQA kernel"
 *   is bound by the HBM traffic of its KV gather.
 *   vLLM PR #54951 "Shard long-context indexer prefill rows across TP" --
 *   Summary: the index lists are fixed-width int32.
 *
 * Conventions for every entry point below:
 *   - Device pointers belong to the caller.  The library allocates nothing per
 *     call.  With 8 or 16 heads, a launch that cuts token lists between CTAs at
 *     arbitrary points (only sparse_mla_fwd_ex with a split count that does not
 *     divide ceil(topk/32) does) merges the parts through a scratch buffer: one per
 *     (device, stream), allocated at the first call on that stream that needs it
 *     (or a larger one), cleared once, and reused.  Calls on one stream are
 *     ordered and share it; a stream capture needs one uncaptured call of the
 *     same size on that stream first (otherwise SMLA_ERR_INVALID_ARG).  A
 *     stream's scratch stays allocated until the process exits (it is keyed by
 *     the stream handle, so a program that creates many short-lived streams
 *     for such calls keeps one buffer for each).
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).
 *   - A non-OK return means nothing was launched.  Device-side failures (a
 *     bounded wait inside the kernel that ran out; in checked mode, list
 *     entries out of range) are recorded in a device error word and reported
 *     by sparse_mla_sync_status().  After a launch that timed out, call
 *     sparse_mla_sync_status() before any further call on the device: a
 *     launch that gave up part-way may leave merge-scratch barrier words
 *     mid-count, and sparse_mla_sync_status() is what clears them.
 *   - sparse_mla_last_error() gives a message for the last non-OK return of
 *     the calling host thread.
 */
#ifndef SPARSE_MLA_H_
#define SPARSE_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMLA_D_QK 576          /* query/key dims: 512 latent + 64 rope */
#define SMLA_D_V 512           /* value/output dims: the latent part */
#define SMLA_BF16_ROW_BYTES 1152
#define SMLA_FP8_ROW_BYTES 656 /* 512 x e4m3 | 4 x fp32 tile scales | 64 x bf16 rope */

typedef enum smla_status {
    SMLA_OK = 0,
    SMLA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or scale */
    SMLA_ERR_UNSUPPORTED = 2,  /* head count or KV format this build does not run */
    SMLA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
    SMLA_ERR_TIMEOUT = 4,      /* a bounded wait inside a kernel gave up */
    SMLA_ERR_INDEX_RANGE = 5   /* checked mode: a list entry other than -1 was outside
                                  [0, num_slots) (it was masked) */
} smla_status;

typedef enum smla_kv_format {
    SMLA_KV_BF16 = 0,          /* rows of 576 bf16 (1152 bytes) */
    SMLA_KV_FP8 = 1            /* rows of 656 bytes: 512 e4m3 latent values, then
                                  4 fp32 scales (one per 128 latent values), then
                                  64 bf16 rope values; latent[d] = e4m3[d] * scale[d/128] */
} smla_kv_format;

/*
 * sparse_mla_fwd -- the forward pass.
 *   q          device, [T, h, 576] bf16, contiguous, 16-byte aligned
 *   kv_cache   device, [num_slots, 576] bf16 (SMLA_KV_BF16) or [num_slots] rows
 *              of 656 bytes (SMLA_KV_FP8), contiguous, 16-byte aligned
 *   indices    device, [T, topk] int32, contiguous, 4-byte aligned; entries
 *              outside [0, num_slots) (-1 by convention) are masked out
 *   T          query tokens (T = 0 is a no-op that returns SMLA_OK)
 *   h          heads per token: 8, 16, 32 or 64, all run natively
 *   topk       list length, >= 1
 *   num_slots  rows in the cache, 1 .. 2^31-1
 *   scale      softmax scale applied to the logits, finite
 *   out        device, [T, h, 512] bf16, written (caller-owned)
 *   lse        device, [T, h] fp32, written (caller-owned)
 * Returns SMLA_OK once the kernel is queued.
 */
smla_status sparse_mla_fwd(const void* q, const void* kv_cache, const int32_t* indices,
                           int32_t T, int32_t h, int32_t topk, int64_t num_slots,
                           int32_t kv_format, float scale, void* out, float* lse,
                           void* stream);

/*
 * sparse_mla_fwd_ex -- sparse_mla_fwd with an explicit split count.
 * splits = 0 lets the library choose (what sparse_mla_fwd does); other values
 * than 0, 1, 2, 4, 8 are SMLA_ERR_INVALID_ARG.
 *   h = 32, 64: each token's list is split over `splits` CTAs of one
 *     thread-block cluster and merged on chip by log-sum-exp weights.
 *   h = 8, 16: the T x ceil(topk/32) row blocks are cut into T * splits equal
 *     contiguous ranges, one per CTA.  When splits divides ceil(topk/32) each
 *     list falls into `splits` whole parts, one thread-block cluster per token,
 *     merged on chip; otherwise the cuts fall anywhere (at most one CTA per SM)
 *     and the parts of a cut list are merged through the scratch after a
 *     grid-wide barrier (cooperative launch), in CTA order.
 * Results agree with any other split count up to fp32 rounding, and repeated
 * calls with the same arguments give identical bytes.
 */
smla_status sparse_mla_fwd_ex(const void* q, const void* kv_cache, const int32_t* indices,
                              int32_t T, int32_t h, int32_t topk, int64_t num_slots,
                              int32_t kv_format, float scale, void* out, float* lse,
                              int32_t splits, void* stream);

/*
 * sparse_mla_fwd_checked -- sparse_mla_fwd_ex in checked mode.  Every list entry
 * outside [0, num_slots) is masked exactly as in sparse_mla_fwd_ex (outputs are
 * identical byte for byte); in addition, an entry other than -1 that is out of
 * range (>= num_slots, or negative and not -1) sets a bit in the device error
 * word, which the next sparse_mla_sync_status() returns as SMLA_ERR_INDEX_RANGE
 * and clears.  -1 is the list padding and never counts.  No trap and no fault:
 * the check is a vote over the entries the producer warps already hold, one
 * atomic per warp that met a bad entry.  The index lists are fixed-width int32
 * (vLLM PR #54951, Summary) with -1 for an unused entry; the checked mode is
 * the device-side range check that stands in for a memory checker.  Arguments
 * as sparse_mla_fwd_ex.
 */
smla_status sparse_mla_fwd_checked(const void* q, const void* kv_cache, const int32_t* indices,
                                   int32_t T, int32_t h, int32_t topk, int64_t num_slots,
                                   int32_t kv_format, float scale, void* out, float* lse,
                                   int32_t splits, void* stream);

/*
 * sparse_mla_fwd_noalloc -- sparse_mla_fwd_ex with the merge scratch taken from
 * a fixed array inside the library (file scope, about 10 MiB per device,
 * enough for 16 heads on up to 160 CTAs) instead of a per-stream buffer, so it
 * never allocates device memory.  The pages describe no counterpart; it exists
 * for callers that must not allocate at all (e.g. under a memory pool).
 *   - The array's address is looked up, and its barrier words cleared, at the
 *     first call on each device; that call synchronises the device and must
 *     not be inside a stream capture (SMLA_ERR_INVALID_ARG).  Later calls,
 *     captured or not, only launch.
 *   - Every call on a device uses the same array: calls that may overlap in
 *     time (different streams without ordering) race on it and must not be
 *     issued.  Launches that cut no list do not touch it.
 *   - A launch that would need more scratch than the array holds returns
 *     SMLA_ERR_UNSUPPORTED and launches nothing.
 * Arguments, results and errors are otherwise those of sparse_mla_fwd_ex.
 */
smla_status sparse_mla_fwd_noalloc(const void* q, const void* kv_cache, const int32_t* indices,
                                   int32_t T, int32_t h, int32_t topk, int64_t num_slots,
                                   int32_t kv_format, float scale, void* out, float* lse,
                                   int32_t splits, void* stream);

/*
 * sparse_mla_merge -- merge the partial results of token lists that were split
 * into parts (the DCP merge: with decode context parallelism each rank runs the
 * forward over its part of every list; vLLM PR #60220, Details: out and lse are
 * "consumed by the v_up projection or the DCP merge"; vLLM PR #64510, Details:
 * heads gathered by DCP).  The pages do not write the merge; it is the exact
 * combination of softmax results over disjoint parts of one list.  Per row
 * (token, head), with O_p and LSE_p what sparse_mla_fwd returns for part p:
 *     M = max_p LSE_p,  LSE = M + ln sum_p exp(LSE_p - M),
 *     O = sum_p exp(LSE_p - LSE) * O_p
 * A part with LSE_p = -inf (an empty part) weighs nothing; a row whose parts
 * are all empty gets O = 0, LSE = -inf.  fp32 arithmetic, O rounded to bf16.
 *   o_parts    device, [n_parts, T, h, 512] bf16, contiguous, 16-byte aligned
 *   lse_parts  device, [n_parts, T, h] fp32 natural-log LSE, 4-byte aligned
 *   n_parts    1 .. 16
 *   T, h       rows = T * h (any h >= 1); T = 0 is a no-op
 *   out        device, [T, h, 512] bf16, caller-owned, 16-byte aligned; must
 *              not overlap o_parts
 *   lse        device, [T, h] fp32, caller-owned, 4-byte aligned
 * Allocates nothing; asynchronous on `stream`.  Errors: SMLA_ERR_INVALID_ARG for
 * a bad n_parts, T, h, null pointer or alignment (nothing is launched);
 * SMLA_ERR_CUDA if the launch fails.
 */
smla_status sparse_mla_merge(const void* o_parts, const float* lse_parts, int32_t n_parts, int32_t T,
                             int32_t h, void* out, float* lse, void* stream);

/*
 * sparse_mla_v_up -- the v_up projection of the attention output: per head, the
 * 512-dim latent output through that head's value up-projection (the output
 * "is consumed by the v_up projection": vLLM PR #60220, Details; v_head_dim 128
 * (DeepSeek-V3.2) or 256 (GLM-5) at kv_lora_rank 512: PR #55738 report, the
 * `_is_masked_mha_available` geometry table):
 *     y[t, h, n] = sum_{k < 512} o[t, h, k] * w[h, n, k]
 * fp32 accumulation on the tcgen05 tensor cores, y rounded to bf16.
 *   o     device, [T, h, 512] bf16 (what sparse_mla_fwd returns), 16-byte aligned
 *   w     device, [h, v, 512] bf16: row n of head h holds the 512 weights of
 *         output n (the pages give no layout); 16-byte aligned
 *   v     128 or 256 (others: SMLA_ERR_UNSUPPORTED)
 *   y     device, [T, h, v] bf16, caller-owned, 16-byte aligned
 * T = 0 is a no-op.  Allocates nothing; asynchronous on `stream`.  Errors:
 * SMLA_ERR_INVALID_ARG for a bad T or h, a null pointer or misalignment;
 * SMLA_ERR_CUDA if a tensor map or the launch fails; a bounded wait that ran out
 * is reported by sparse_mla_sync_status().
 */
smla_status sparse_mla_v_up(const void* o, const void* w, int32_t T, int32_t h, int32_t v, void* y,
                            void* stream);

/*
 * sparse_mla_topk -- the index lists from per-position scores: the step before
 * the attention.  The indexer scores every position of a token's causal history
 * and keeps the top k as a fixed-width int32 list in which only the set matters
 * (vLLM PR #54951, Summary and Additional checks); the pages do not give the
 * scoring, so the scores are the input.  Row t keeps the topk positions with the
 * largest scores among [0, lengths[t]) (ties to the lower position), in
 * ascending position order, each mapped to its cache slot
 * block_table[p / 64] * 64 + p % 64 (block_table NULL: the position itself),
 * and pads with -1 when lengths[t] < topk.  Exact (a radix select), so results
 * are reproducible bit for bit.
 *   scores       device, [T, S] fp32 (no NaN), row-major, 4-byte aligned
 *   lengths      device, [T] int32; values outside [0, S] are clamped
 *   block_table  device, [ceil(S / 64)] int32 of one sequence, or NULL
 *   indices      device, [T, topk] int32, caller-owned: sparse_mla_fwd's input
 * One call serves the rows of one sequence (one block table): a mixed batch of
 * several sequences takes one call per sequence, each on that sequence's rows
 * of scores, lengths and indices.
 * T = 0 is a no-op.  Allocates nothing; asynchronous on `stream`.  Errors:
 * SMLA_ERR_INVALID_ARG for bad sizes (S < 1, topk outside [1, 2^20]), a null
 * pointer or misalignment; SMLA_ERR_CUDA if the launch fails.
 */
smla_status sparse_mla_topk(const float* scores, int32_t T, int64_t S, const int32_t* lengths, int32_t topk,
                            const int32_t* block_table, int32_t* indices, void* stream);

/*
 * sparse_mla_scatter_mask -- the masked dense route's first step: the index
 * lists of one request scattered into a bit mask.  PR #55738 report, 实现拆解
 * (implementation breakdown) items 2 and 5: short prefills run a scatter of the
 * top-k lists (_scatter_topk_single_req) and a dense attention with a mask
 * instead of the per-token gather.  The report gives no layout; here row t of
 * the mask has W = ceil(S / 32) uint32 words and bit s % 32 of word s / 32 is
 * set iff position s appears in indices[t, :].  Entries outside [0, S) (-1 by
 * convention) set nothing; a repeated position sets its bit once (the mask
 * holds a set, where sparse_mla_fwd weighs every list entry).
 *   indices   device, [T, topk] int32 positions of the request, 4-byte aligned
 *   S         positions in the request, 1 .. 2^20
 *   mask      device, [T, W] uint32, caller-owned, 16-byte aligned; every word
 *             is written
 * T = 0 is a no-op.  Allocates nothing; asynchronous on `stream`.  Errors:
 * SMLA_ERR_INVALID_ARG for bad sizes, a null pointer or misalignment;
 * SMLA_ERR_CUDA if the launch fails.
 */
smla_status sparse_mla_scatter_mask(const int32_t* indices, int32_t T, int32_t topk, int64_t S, uint32_t* mask,
                                    void* stream);

/*
 * sparse_mla_masked_mha -- the masked dense route's attention: multi-head
 * attention of T query tokens over the request's S positions with per-head
 * K and V, in which the mask alone decides which positions each token attends
 * to (the FA4 mask_mod attention of the same report).  Per token t and head h:
 *     s_j = scale * <q[t,h,:], k[j,h,:]>   for the positions j set in mask[t]
 *     O[t,h] = softmax(s) . v[:,h,:],   LSE[t,h] = ln sum_j exp(s_j)
 * A row with no bit set gives O = 0 and LSE = -inf.  Head dims follow the
 * report's `_is_masked_mha_available` geometry table: q/k 192 (128 nope + 64
 * rope, DeepSeek-V3.2) or 256 (192 + 64, GLM-5; 256 + 0, the NoPE layout),
 * v 128 or 256.  bf16 in, fp32 softmax and accumulation on the tcgen05 tensor
 * cores, O rounded to bf16.
 *   q      device, [T, h, dqk] bf16, 16-byte aligned
 *   k      device, [S, h, dqk] bf16, 16-byte aligned
 *   v      device, [S, h, dv] bf16, 16-byte aligned
 *   mask   device, [T, ceil(S / 32)] uint32 as sparse_mla_scatter_mask writes
 *          it, 4-byte aligned
 *   S      1 .. 65536;  h >= 1;  dqk 192 or 256;  dv 128 or 256
 *   out    device, [T, h, dv] bf16, caller-owned;  lse  device, [T, h] fp32
 * T = 0 is a no-op.  Allocates nothing; asynchronous on `stream`.  Errors:
 * SMLA_ERR_UNSUPPORTED for other head dims, SMLA_ERR_INVALID_ARG for bad sizes,
 * scale, a null pointer or misalignment; SMLA_ERR_CUDA if a tensor map or the
 * launch fails; a bounded wait that ran out is reported by
 * sparse_mla_sync_status().
 */
smla_status sparse_mla_masked_mha(const void* q, const void* k, const void* v, const uint32_t* mask, int32_t T,
                                  int64_t S, int32_t h, int32_t dqk, int32_t dv, float scale, void* out, float* lse,
                                  void* stream);

/*
 * sparse_mla_fwd_host -- the same forward pass taking HOST buffers for the
 * per-step inputs and outputs, for callers whose q/indices live in host memory.
 * It queues on `stream`: copies of q_host and indices_host into `workspace`,
 * the kernel, and copies of out/lse back into out_host/lse_host.  The KV cache
 * stays a device pointer (it is state resident on the GPU).  Host buffers
 * should be pinned for the copies to be asynchronous; the results are in
 * out_host/lse_host once the stream has been synchronised.
 *   workspace        device, at least sparse_mla_host_workspace_bytes(T,h,topk)
 *                    bytes, 256-byte aligned, caller-owned
 */
size_t sparse_mla_host_workspace_bytes(int32_t T, int32_t h, int32_t topk);
smla_status sparse_mla_fwd_host(const void* q_host, const void* kv_cache,
                                const int32_t* indices_host, int32_t T, int32_t h,
                                int32_t topk, int64_t num_slots, int32_t kv_format,
                                float scale, void* out_host, float* lse_host,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * sparse_mla_fwd_host_packed -- sparse_mla_fwd_host with the per-step inputs in
 * one host buffer and the outputs in another, so each call queues exactly one
 * host-to-device copy, the kernel and one device-to-host copy on `stream`.
 *   in_host    host, in_bytes: q ([T, h, 576] bf16) at offset 0, indices
 *              ([T, topk] int32) at indices_offset
 *   out_host   host, out_bytes: out ([T, h, 512] bf16) at offset 0, lse ([T, h]
 *              fp32) at lse_offset
 *   workspace  device, at least sparse_mla_host_workspace_bytes(T, h, topk)
 *              bytes, 256-byte aligned, caller-owned
 * sparse_mla_host_io_layout gives the sizes and offsets (the gaps are padding to
 * 256 bytes, never read or written by the kernel).  Pinned host buffers make the
 * copies asynchronous; the results are in out_host once `stream` has been
 * synchronised.  Calls on different streams with their own workspaces may
 * overlap one step's copies with another's kernel.
 */
smla_status sparse_mla_host_io_layout(int32_t T, int32_t h, int32_t topk, size_t* in_bytes,
                                      size_t* indices_offset, size_t* out_bytes, size_t* lse_offset);
smla_status sparse_mla_fwd_host_packed(const void* in_host, const void* kv_cache, int32_t T, int32_t h,
                                       int32_t topk, int64_t num_slots, int32_t kv_format, float scale,
                                       void* out_host, void* workspace, size_t workspace_bytes,
                                       void* stream);

/*
 * sparse_mla_sync_status -- synchronise `stream`, then read and clear the
 * device error word of the current device.  Returns SMLA_ERR_TIMEOUT if a
 * kernel gave up on a bounded wait since the last call (the device is then
 * synchronised and the barrier words of every merge scratch on it cleared),
 * else SMLA_ERR_INDEX_RANGE if a sparse_mla_fwd_checked launch met a list
 * entry other than -1 outside [0, num_slots), SMLA_ERR_CUDA if the
 * synchronisation failed, SMLA_OK otherwise.  The word is per device, so a
 * report covers every launch on the device since the last read.  Not for the
 * hot path.
 */
smla_status sparse_mla_sync_status(void* stream);

/*
 * sparse_mla_launch_info -- how sparse_mla_fwd would launch (T, h, topk):
 * split count, CTAs in the grid, dynamic shared memory per CTA in bytes and
 * kernel launches per call.  Any output pointer may be NULL.
 */
smla_status sparse_mla_launch_info(int32_t T, int32_t h, int32_t topk, int32_t kv_format,
                                   int32_t* splits, int32_t* ctas, int32_t* smem_bytes,
                                   int32_t* launches);

/* Message for the calling thread's last non-OK return ("" if none).  The
 * pointer is to a thread-local buffer owned by the library: valid until the
 * next non-OK return on the same thread; the caller copies it if it keeps it. */
const char* sparse_mla_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t sparse_mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MLA_H_ */
