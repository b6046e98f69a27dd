/*
 * inkling_attn.h -- C ABI of libinkling_attn.so: paged prefill and decode attention
 * with a per-token relative-position bias, grouped-query heads, and sliding-window or
 * full-causal masking, for NVIDIA GB300 (sm_103a).
 *
 * The operation is the attention of the RoPE-free hybrid model described in
 * "Support Inkling-NVFP4 model" (TensorRT-LLM PR #17062):
 *   - section "Architecture": position enters only through a learned bias per
 *     (query token, head, relative distance) added to the scores before the softmax;
 *     local layers attend over a 512-key sliding window (16 KV heads), global layers
 *     are full causal (8 KV heads);
 *   - section "Implementation", row attention_backend/inkling_triton.py: paged prefill
 *     and decode kernels apply the bias as a score modifier; rel_logits has a static
 *     shape so decode can be captured in a CUDA graph;
 *   - review of _build_rel_logits: the bias tensor is [tokens, heads, rel_extent] fp32.
 * and in "Inkling attn backend cleanup fake registry" (TensorRT-LLM PR #17860):
 *   - commit on GQA input checks: query head h reads KV head h / (Hq / Hkv); a
 *     non-divisible head pair is an error;
 *   - commit moving attention into the backend: per-layer scalars sm_scale,
 *     rel_extent, window_left (-1 on global layers);
 *   - commits on borrowing the base page table: key k lives in page
 *     block_table[b][k / page_size] (a positional table), and k < seq_len bounds every
 *     access, so entries past a sequence's own blocks are never read.
 *
 * Definition (exact; the kernels compute it in fp32 with bf16 inputs):
 *   sequence b has L_b = seq_lens[b] keys; its n_b new query tokens are the last n_b
 *   positions, so new token i sits at p = L_b - n_b + i.
 *   visible keys:  0 <= k <= p, and p - k <= window - 1 when window > 0
 *   s_k = sm_scale * <q[t,h,:], K[k,h/G,:]> + rel_logits[t, h, min(p - k, E - 1)]
 *   out[t,h,:] = sum_k softmax(s)_k * V[k,h/G,:]          (bf16, round to nearest even)
 *
 * Conventions for every entry point:
 *   - Pointers named "device" must point to GPU memory of the current device; the
 *     caller owns every buffer.  Calls never allocate, free or synchronise: they enqueue
 *     kernels on `stream` (a cudaStream_t; NULL = legacy default stream) and return.
 *   - Host-side validation reads only the scalars and pointer values.  On failure the
 *     call returns an error code and launches nothing.
 *   - Device-side problems (a page id outside [0, num_pages) for a key that must be
 *     read, more new tokens than history, a bounded wait that ran out) never fault:
 *     the kernel skips the access, treats the affected keys as masked, and ORs a bit
 *     into the sticky error word in the workspace (INK_DEVERR_*), which
 *     inkling_attn_read_device_error() returns.
 *   - Keys that sit in a loaded page but are not visible get weight exactly 0 and
 *     their V rows are zeroed before use, so any bit pattern (NaN included) may sit
 *     there.  Pages that hold no visible key are never read.
 *   - A sequence with seq_lens[b] == 0 writes zeros to its output rows.
 */
#ifndef INKLING_ATTN_H
#define INKLING_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  INK_OK = 0,
  INK_ERR_NULL_PTR = 1,        /* a required pointer is NULL */
  INK_ERR_BAD_SHAPE = 2,       /* Hq % Hkv != 0, head_dim not 64/128, non-positive sizes */
  INK_ERR_BAD_PAGE_SIZE = 3,   /* page_size not a power of two in [8, 2^20] */
  INK_ERR_WORKSPACE = 4,       /* workspace smaller than inkling_attn_workspace_bytes() */
  INK_ERR_ALIGNMENT = 5,       /* q/k/v/out not 16-byte aligned, or index arrays not 4-byte */
  INK_ERR_CUDA = 6,            /* a CUDA runtime call failed (launch, attribute, ...) */
  INK_ERR_TOO_LARGE = 7        /* an index would overflow the 32-bit coordinates used */
} ink_status_t;

/* Sticky device error bits (see inkling_attn_read_device_error). */
#define INK_DEVERR_PAGE_OUT_OF_RANGE 0x1u  /* block_table entry outside [0, num_pages) */
#define INK_DEVERR_QLEN_EXCEEDS_KV   0x2u  /* cu_q_lens gives more new tokens than seq_lens */
#define INK_DEVERR_WAIT_TIMEOUT      0x4u  /* a bounded wait on a copy ran out */
#define INK_DEVERR_QLEN_EXCEEDS_MAX  0x8u  /* a sequence has more new tokens than max_q_len */
#define INK_DEVERR_BAD_ROWS          0x10u /* cu_q_lens names rows outside [0, total_q) */

/* Per-call shape and layer scalars.  All sizes are element counts. */
typedef struct {
  int32_t num_seqs;           /* B */
  int32_t num_q_heads;        /* Hq */
  int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0 */
  int32_t head_dim;           /* D: 64 or 128 */
  int32_t page_size;          /* P: power of two, >= 8 */
  int32_t max_pages_per_seq;  /* row stride of block_table */
  int32_t num_pages;          /* pages in each K/V pool */
  int32_t rel_extent;         /* E >= 1: distances >= E-1 use bucket E-1 */
  int32_t window;             /* > 0: keys at distances 0..window-1; <= 0: full causal */
  float sm_scale;             /* multiplies q.k only; the bias is added unscaled */
} ink_attn_params_t;

/*
 * Bytes of device workspace a call needs.  is_decode != 0 sizes it for
 * inkling_attn_decode (split-K partials and tickets), else for inkling_attn_prefill.
 * Returns 0 if the parameters are invalid.  A buffer sized for decode also serves
 * prefill with the same params.
 */
size_t inkling_attn_workspace_bytes(const ink_attn_params_t* params, int is_decode);

/*
 * Zero a workspace (error word and split-K tickets) on `stream`.  Must be called once
 * after allocating a workspace and before its first use; the kernels leave the tickets
 * at zero when they finish, so later calls need no re-initialisation.
 */
ink_status_t inkling_attn_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Paged prefill (context phase), any number of new tokens per sequence.
 *   q          device, bf16 [total_q, Hq, D], rows packed by sequence
 *   cu_q_lens  device, int32 [B+1], cu_q_lens[0] = 0, non-decreasing; n_b = cu[b+1]-cu[b]
 *   max_q_len  host int >= every n_b (sizes the grid; larger n_b set INK_DEVERR_QLEN_EXCEEDS_MAX)
 *   total_q    host int = cu_q_lens[B], the number of rows of q, rel_logits and out (bounds
 *              the tensor-memory copies of q; rows past it are never read)
 *   k_cache, v_cache  device, bf16 [num_pages, Hkv, P, D]; the step's K/V must already
 *              be written (new tokens are the last n_b of seq_lens[b])
 *   block_table device, int32 [B, max_pages_per_seq], positional page ids
 *   seq_lens   device, int32 [B], KV length including the new tokens
 *   rel_logits device, fp32 [total_q, Hq, E]
 *   out        device, bf16 [total_q, Hq, D]
 *   workspace  device, >= inkling_attn_workspace_bytes(params, 0), initialised once
 * q and out must be 16-byte aligned; when both are 32-byte aligned the kernels move their
 * rows in 256-bit loads and stores (the same results, fewer memory requests).
 */
ink_status_t inkling_attn_prefill(const ink_attn_params_t* params, const void* q,
                                  const int32_t* cu_q_lens, int32_t max_q_len, int32_t total_q,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, const int32_t* seq_lens,
                                  const float* rel_logits, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * inkling_attn_prefill with the bias in bf16: rel_logits_bf16 is bf16 [total_q, Hq, E]
 * (same layout as rel_logits), every other argument and result as for
 * inkling_attn_prefill.  The review of _build_rel_logits in "Support Inkling-NVFP4 model"
 * (TensorRT-LLM PR #17062) suggests producing the bias in bf16 where the kernel can take
 * it: on long prompts the fp32 bias is the largest input of the call, and bf16 halves it.
 * The bias enters the scores as exactly the bf16 values given (widened to fp32); the
 * rest of the arithmetic is unchanged.
 *   Requirements beyond inkling_attn_prefill: E a multiple of 8 (else INK_ERR_BAD_SHAPE)
 *   and rel_logits_bf16 16-byte aligned (else INK_ERR_ALIGNMENT).
 */
ink_status_t inkling_attn_prefill_bf16bias(const ink_attn_params_t* params, const void* q,
                                           const int32_t* cu_q_lens, int32_t max_q_len, int32_t total_q,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_table, const int32_t* seq_lens,
                                           const void* rel_logits_bf16, void* out, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * inkling_attn_prefill with the bias given in low-rank form: the kernel computes each bias
 * tile itself, so the [total_q, Hq, E] bias tensor is never built or read.  "Support
 * Inkling-NVFP4 model" (TensorRT-LLM PR #17062), review of _build_rel_logits: a layer's
 * bias is the product over d_rel of a per-(token, head) vector r and the layer's
 * projection rel_logits_proj [d_rel, E]:
 *     rel[t, h, e] = sum_c r[t, h, c] * rel_logits_proj[c, e]
 *   r           device, bf16 [total_q, Hq, d_rel], 16-byte aligned
 *   rel_proj_t  device, bf16 [E, d_rel]: rel_logits_proj transposed (bucket-major, so each
 *               bucket's d_rel coefficients are contiguous), 16-byte aligned
 *   d_rel       a multiple of 8 in [8, 64] (else INK_ERR_BAD_SHAPE); the pages do not give it.
 *               The bias products run with K = 64; columns past d_rel are zeros.
 * The products are summed in fp32 from the bf16 operands (tensor-core MMA for the buckets
 * of a tile, a plain fp32 dot product for the clamped bucket E - 1) and the tile's bias
 * values are kept in fp16 until they are added to the fp32 scores (relative rounding
 * 2^-11); the rest of the arithmetic is that of inkling_attn_prefill.  Every other
 * argument and result as for inkling_attn_prefill.
 */
ink_status_t inkling_attn_prefill_lowrank_bias(const ink_attn_params_t* params, const void* q,
                                               const int32_t* cu_q_lens, int32_t max_q_len, int32_t total_q,
                                               const void* k_cache, const void* v_cache,
                                               const int32_t* block_table, const int32_t* seq_lens,
                                               const void* r, const void* rel_proj_t, int32_t d_rel, void* out,
                                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Paged decode: one new token per sequence (row b of q is sequence b, at p = L_b - 1).
 *   q          device, bf16 [B, Hq, D]
 *   rel_logits device, fp32 [B, Hq, E]
 *   out        device, bf16 [B, Hq, D]
 *   workspace  device, >= inkling_attn_workspace_bytes(params, 1), initialised once.
 *              Calls that share a workspace must not overlap on the GPU (the split-K
 *              partials and tickets live there).
 * Other arguments as for prefill.  Stream-ordered, no allocation, no host sync: the
 * call can be captured in a CUDA graph.
 */
ink_status_t inkling_attn_decode(const ink_attn_params_t* params, const void* q,
                                 const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 const float* rel_logits, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * inkling_attn_decode without a workspace argument, for callers that cannot allocate
 * device memory: for example a plugin whose host framework owns every device buffer
 * and hands out only fixed-size tensors, or a serving loop that must not grow its
 * memory after start-up.  Such a caller has no way to create the workspace that
 * inkling_attn_decode needs.  The pages this library follows have no counterpart to
 * this entry point.
 *   - Scratch: a 64 MiB device array inside the library, held by every GPU that loads
 *     it until the process exits.  A call whose workspace need
 *     (inkling_attn_workspace_bytes(params, 1)) exceeds 64 MiB returns
 *     INK_ERR_WORKSPACE and launches nothing.
 *   - The call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     routine.  It clears the array's error word and split-K tickets on `stream`
 *     (cudaMemsetAsync), then runs the same kernel as inkling_attn_decode.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  Make that first call before any
 *     stream capture.
 *   - All calls on a device share the array, which keeps the last call's contents.
 *     Calls that overlap on the GPU (different streams, no ordering between them) race
 *     on it and give wrong results.  Device-side error bits are kept in the array and
 *     not reported.
 * Other arguments and results as for inkling_attn_decode.
 */
ink_status_t inkling_attn_decode_noalloc(const ink_attn_params_t* params, const void* q,
                                         const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         const float* rel_logits, void* out, void* stream);

/*
 * The step's K/V write: causal short convolution of the new K and V rows, written into
 * the paged caches, and the convolution state carried to the next step.
 * "Support Inkling-NVFP4 model" (TensorRT-LLM PR #17062), section "Architecture": every
 * attention layer runs a causal short convolution over K and over V, with per-request
 * state between steps.  "Inkling attn backend cleanup fake registry" (TensorRT-LLM PR
 * #17860): the state is a window of kernel_size - 1 past inputs per request, carried with
 * the request; the backend itself writes the step's K/V into the paged cache through the
 * block table.  Neither page gives the kernel size, a bias or an activation: the
 * convolution here is depthwise (one filter per channel), without bias or activation.
 * For request b with n_b = cu_q_lens[b+1] - cu_q_lens[b] new rows and L_b = seq_lens[b]
 * (history including them), new row i sits at position p = L_b - n_b + i, and for each
 * channel c = (g, d) of K (and likewise of V)
 *     y[p, c] = sum_{j=0}^{ks-1} w_k[g, d, j] * x[p - (ks-1) + j, c]
 * where x at the ks - 1 positions before the first new row is state_k_in[b] (oldest
 * first).  y is computed in fp32 and stored rounded to bf16 (nearest even) at
 * k_cache[block_table[b][p / P], g, p % P, :].  state_k_out[b] receives the last ks - 1
 * rows of (state_k_in[b], new rows of b), unconvolved.
 *   k_new, v_new          device, bf16 [total_q, Hkv, D], rows packed by request
 *   cu_q_lens             device, int32 [B+1], cu_q_lens[0] = 0, cu_q_lens[B] = total_q
 *   seq_lens, block_table device, as for inkling_attn_prefill
 *   w_k, w_v              device, fp32 [Hkv, D, kernel_size] (a depthwise Conv1d weight over
 *                         the Hkv*D channels), 16-byte aligned
 *   kernel_size           1..8 (else INK_ERR_BAD_SHAPE); 1 stores x * w unshifted
 *   state_*_in/out        device, bf16 [B, kernel_size - 1, Hkv, D]; unused (may be NULL)
 *                         when kernel_size == 1.  Outputs must not overlap inputs; a fresh
 *                         request passes zero rows.
 *   k_cache, v_cache      device, bf16 [num_pages, Hkv, P, D]; only the slots of the step's
 *                         positions are written
 *   workspace             device, >= inkling_attn_workspace_bytes(params, 0) (error word)
 * Only num_seqs, num_kv_heads, head_dim, page_size, max_pages_per_seq and num_pages of
 * params are used; the rest must still be valid.  Device-side checks: a request with
 * n_b > L_b (INK_DEVERR_QLEN_EXCEEDS_KV) or a page id outside [0, num_pages)
 * (INK_DEVERR_PAGE_OUT_OF_RANGE) has those rows skipped; rows named outside [0, total_q)
 * set INK_DEVERR_BAD_ROWS.  Stream-ordered, no allocation: capturable in a CUDA graph.
 */
ink_status_t inkling_attn_kv_conv_write(const ink_attn_params_t* params, const void* k_new,
                                        const void* v_new, const int32_t* cu_q_lens, int32_t total_q,
                                        const int32_t* seq_lens, const int32_t* block_table,
                                        const float* w_k, const float* w_v, int32_t kernel_size,
                                        const void* state_k_in, const void* state_v_in,
                                        void* state_k_out, void* state_v_out, void* k_cache,
                                        void* v_cache, void* workspace, size_t workspace_bytes,
                                        void* stream);

/*
 * Synchronise `stream`, copy the sticky device error word (INK_DEVERR_* bits) to
 * *err_out, and clear it when `clear` is non-zero.  This is the only entry point that
 * blocks the host.
 */
ink_status_t inkling_attn_read_device_error(void* workspace, size_t workspace_bytes,
                                            void* stream, uint32_t* err_out, int clear);

/* Static, human-readable name of a status code. */
const char* inkling_attn_status_string(ink_status_t status);

/* ABI version of the library (major * 100 + minor). */
int32_t inkling_attn_version(void);

/*
 * Time limit, in nanoseconds, of one pipeline wait inside every kernel launched after this
 * call (process-wide; the default is 2 000 000 000, larger values are clamped to it).  A
 * wait that runs out sets INK_DEVERR_WAIT_TIMEOUT in the workspace error word; the kernel
 * then stops issuing work, waits (up to 2 s each) for the copies and tensor-core
 * operations it has already issued, and returns, leaving the device usable.  0 makes every
 * wait that finds its data not yet ready give up at once: a way for tests to drive the
 * timeout path without a fault.  Failure detection by status, not by fault, follows the
 * epoch-checked "ready" flag of "Inkling attn backend cleanup fake registry" (TensorRT-LLM
 * PR #17860), where stale decode metadata is detected rather than read.  Not for use in
 * production: launches in flight keep the limit they were launched with.
 */
void inkling_attn_set_wait_limit_ns(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* INKLING_ATTN_H */
